"""Data-parallel host logic on two CPU ranks over gloo: the scale-gradient average and the
max-over-ranks step time that the multi-GPU benchmark uses."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from scale_only_quantization_gb300 import dp
    g = torch.Generator().manual_seed(100 + rank)
    ds13 = torch.randn((4, 8, 16), generator=g)
    ds2 = torch.randn((4, 16, 8), generator=g)
    mine = (ds13.clone(), ds2.clone())
    dp.average_scale_grads([ds13, ds2])
    t = dp.max_over_ranks(1.5 + rank)
    out[rank] = (mine, (ds13, ds2), t)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_scale_grad_average_and_max_time():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    (m0, a0, t0), (m1, a1, t1) = out[0], out[1]
    for i in range(2):
        want = (m0[i] + m1[i]) / 2
        assert torch.allclose(a0[i], want, rtol=0, atol=1e-6)
        assert torch.equal(a0[i], a1[i])
    assert t0 == t1 == 2.5


def test_single_process_is_a_no_op():
    from scale_only_quantization_gb300 import dp
    x = torch.ones(3)
    dp.average_scale_grads([x])
    assert torch.equal(x, torch.ones(3)) and dp.max_over_ranks(3.0) == 3.0
