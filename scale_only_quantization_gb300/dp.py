"""Data-parallel helpers for running the layer on several GPUs, one process per GPU.

In data-parallel scale-only QAD each rank runs the layer on its own tokens and the
scale gradients are averaged over the data-parallel group before the optimizer step
(AngelSlim mcore_qad walkthrough, nxmr.cn/news/131691, section 二.5: scale gradients
are averaged over the DP x CP group; MoE experts use the expert-data-parallel group).
"""
import torch
import torch.distributed as dist


def world(group=None):
    return dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1


def average_scale_grads(grads, group=None):
    """In-place mean of each scale-gradient tensor over the ranks of `group`."""
    n = world(group)
    if n == 1:
        return grads
    for g in grads:
        dist.all_reduce(g, op=dist.ReduceOp.SUM, group=group)
        g.div_(n)
    return grads


def max_over_ranks(value, device="cpu", group=None):
    """The largest of one float per rank (step times are reported as the slowest rank's)."""
    if world(group) == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
