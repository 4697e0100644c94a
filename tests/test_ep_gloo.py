"""Expert-parallel exchange on CPU ranks over gloo, against one process computing the whole layer.

The ranks run scale_only_quantization_gb300.ep.ExpertParallelMoE with the fp64 oracle as the
expert backend (the CUDA backend needs one GPU per rank).  Each rank owns E / EP experts and
its own tokens; one process runs the oracle layer on the tokens of all ranks of an
expert-parallel group, concatenated in rank order, with every expert.  The routed rows each
owner receives must be, expert by expert, the rows that single process groups for it (bit
exact); out, dx and dprobs of every token and the scale gradients of every expert must equal
the single process's, and with expert-data-parallel replicas the scale gradients are the mean
over the replicas (the walkthrough's section 二.5 averaging; its section 二.4: experts split
only by expert parallelism).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

E, D, F, K, T = 8, 32, 16, 2, 24


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _weights(fmt=0):
    import synth
    cfg = synth.workload("tiny_nvfp4", E=E, d=D, F=F, topk=K, T=T, fmt=fmt)
    return synth.make_inputs(cfg, seed=0, device="cpu")


def _tokens(rank, skew=False):
    import synth
    cfg = synth.workload("tiny_nvfp4", E=E, d=D, F=F, topk=K, T=T)
    inp = synth.make_inputs(cfg, seed=100 + rank, device="cpu", with_weights=False)
    if skew:  # every pair to experts 0..E/2-1 (rank 0's with EP = 2): rank 1 receives nothing
        idx = inp["topk_idx"] % (E // 2)
        idx[:, 1] = torch.where(idx[:, 1] == idx[:, 0], (idx[:, 0] + 1) % (E // 2), idx[:, 1])
        inp["topk_idx"] = idx.contiguous()
    elif rank % 2 == 1:  # an invalid index and a repeated expert: both pairs are dropped
        inp["topk_idx"][3, 1] = E + 5
        inp["topk_idx"][5, 1] = inp["topk_idx"][5, 0]
    return inp


class OracleExperts:
    """The ExpertParallelMoE backend protocol on the fp64 oracle (tests only)."""

    def __init__(self, fmt, w13, s13, w2, s2):
        self.fmt, self.w13, self.s13, self.w2, self.s2 = fmt, w13, s13, w2, s2

    @staticmethod
    def _bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    @staticmethod
    def _bf16(values):
        from oracle import quant as OQ
        return torch.from_numpy(OQ.f64_to_bf16_bits(values).view(np.int16).copy()).view(torch.bfloat16)

    def forward(self, x_rows, local_expert):
        from oracle import moe as OM
        n = x_rows.shape[0]
        self.ones = np.ones((n, 1))
        self.fwd = OM.moe_forward(self.fmt, self._bits(x_rows), local_expert.numpy().reshape(n, 1).astype(np.int64),
                                  self.ones, self.w13, self.s13, self.w2, self.s2)
        return self._bf16(self.fwd["out"])

    def dgrad(self, dout_rows, p_rows):
        from oracle import moe as OM
        self.bwd = OM.moe_dgrad(self._bits(dout_rows), p_rows.numpy().astype(np.float64).reshape(-1, 1), self.fwd)
        return self._bf16(self.bwd["dx"]), torch.from_numpy(self.bwd["dprobs"].reshape(-1).copy())

    def scalegrad(self):
        from oracle import moe as OM
        ds13, ds2 = OM.moe_scalegrad(self.fmt, self.fwd, self.bwd, self.w13, self.s13, self.w2, self.s2)
        return torch.from_numpy(ds13), torch.from_numpy(ds2)

    def combine(self, rows, row_of, p):
        from oracle import moe as OM
        from oracle import quant as OQ
        ro = row_of.numpy().astype(np.int64)
        pw = np.ones(ro.shape) if p is None else p.numpy().astype(np.float64)
        return self._bf16(OM.combine(OQ.bf16_to_f64(self._bits(rows)), pw, ro))


def _rank_main(rank, world, ep, port, out, skew=False, fmt=0):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from scale_only_quantization_gb300 import ep as EP
    edp = world // ep
    ep_groups = [dist.new_group(list(range(i * ep, (i + 1) * ep))) for i in range(edp)]
    edp_groups = [dist.new_group(list(range(j, world, ep))) for j in range(ep)]
    my_ep, my_pos = rank // ep, rank % ep
    w = _weights(fmt)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    e_loc = E // ep
    lo = my_pos * e_loc
    backend = OracleExperts(w["fmt"], bits(w["w13"])[lo:lo + e_loc], w["s13"].numpy()[lo:lo + e_loc],
                            bits(w["w2"])[lo:lo + e_loc], w["s2"].numpy()[lo:lo + e_loc])
    layer = EP.ExpertParallelMoE(backend, E, group=ep_groups[my_ep],
                                 expert_dp_group=edp_groups[my_pos] if edp > 1 else None)
    tok = _tokens(rank, skew)
    o = layer.forward(tok["x"], tok["topk_idx"], tok["topk_w"])
    dx, dprobs = layer.backward(tok["dout"])
    ds13, ds2 = layer.scale_grads()

    # which global (token, slot) pairs reached this rank, in arrival order: the same exchange
    # applied to the pairs' global ids
    plan = layer.plan
    gid = (my_pos * T * K + plan["order"]).to(torch.int64)  # token numbering of the group's concatenation
    arrived = EP.exchange(gid, plan["send_counts"], plan["recv_counts"], ep_groups[my_ep]).numpy()
    rows_in_expert_order = arrived[backend.fwd["route"]["row_token"]]
    out[rank] = dict(out=bits(o).copy(), dx=bits(dx).copy(), dprobs=dprobs.numpy().copy(), ds13=ds13.numpy().copy(),
                     ds2=ds2.numpy().copy(), rows=rows_in_expert_order, counts=backend.fwd["route"]["counts"].copy())
    dist.barrier()
    dist.destroy_process_group()


def _single_process(ranks, skew=False, fmt=0):
    """The oracle layer on the tokens of `ranks` concatenated, with every expert."""
    from oracle import moe as OM
    w = _weights(fmt)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    toks = [_tokens(r, skew) for r in ranks]
    x = np.concatenate([bits(t["x"]) for t in toks])
    idx = np.concatenate([t["topk_idx"].numpy() for t in toks]).astype(np.int64)
    p = np.concatenate([t["topk_w"].numpy() for t in toks]).astype(np.float64)
    dout = np.concatenate([bits(t["dout"]) for t in toks])
    fwd = OM.moe_forward(w["fmt"], x, idx, p, bits(w["w13"]), w["s13"].numpy(), bits(w["w2"]), w["s2"].numpy())
    bwd = OM.moe_dgrad(dout, p, fwd)
    ds13, ds2 = OM.moe_scalegrad(w["fmt"], fwd, bwd, bits(w["w13"]), w["s13"].numpy(), bits(w["w2"]),
                                 w["s2"].numpy())
    return fwd, bwd, ds13, ds2


def _bf16_bits(v):
    from oracle import quant as OQ
    return OQ.f64_to_bf16_bits(v)


@pytest.mark.parametrize("world, ep, skew, fmt", [(2, 2, False, 0), (4, 4, False, 0), (4, 2, False, 0),
                                                   (2, 2, True, 0), (2, 2, False, 6)],
                         ids=["ep2", "ep4", "ep2-edp2", "ep2-owner-without-rows", "ep2-deployed-nvfp4"])
def test_expert_parallel_exchange_matches_one_process(world, ep, skew, fmt):
    """fmt 6 (deployed nvfp4 scales): the weights' tensor scale is per expert matrix and the
    activations' per row, so the split must leave every bit unchanged too."""
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, ep, port, out, skew, fmt), nprocs=world, start_method="spawn",
                       join=True)
    edp = world // ep
    e_loc = E // ep
    refs = [_single_process(list(range(i * ep, (i + 1) * ep)), skew, fmt) for i in range(edp)]
    if skew:
        assert int(np.sum(out[1]["counts"])) == 0  # rank 1 owned experts nobody was routed to
    for rank in range(world):
        r = out[rank]
        my_ep, my_pos = rank // ep, rank % ep
        fwd, bwd, ds13, ds2 = refs[my_ep]
        sl = slice(my_pos * T, (my_pos + 1) * T)
        # outputs and input gradients of this rank's tokens: bit for bit
        assert np.array_equal(r["out"], _bf16_bits(fwd["out"][sl]).reshape(T, D))
        assert np.array_equal(r["dx"], _bf16_bits(bwd["dx"][sl]).reshape(T, D))
        assert np.allclose(r["dprobs"], bwd["dprobs"][sl], rtol=1e-12, atol=0)
        # the rows each owned expert received, in the single process's order for that expert
        rt = fwd["route"]
        for el in range(e_loc):
            e = my_pos * e_loc + el
            lo, hi = rt["offsets"][e], rt["offsets"][e + 1]
            want = rt["row_token"][lo:hi] * K + rt["row_slot"][lo:hi]
            got_lo = int(np.sum(r["counts"][:el]))
            got = r["rows"][got_lo:got_lo + r["counts"][el]]
            assert np.array_equal(got, want), (rank, e)
        # scale gradients of the owned experts: the mean over the expert-data-parallel replicas
        mean13 = sum(ref[2] for ref in refs) / edp
        mean2 = sum(ref[3] for ref in refs) / edp
        own = slice(my_pos * e_loc, (my_pos + 1) * e_loc)
        assert np.allclose(r["ds13"], mean13[own], rtol=1e-12, atol=1e-300)
        assert np.allclose(r["ds2"], mean2[own], rtol=1e-12, atol=1e-300)


def test_plan_groups_pairs_by_owner_and_drops_invalid_ones():
    from scale_only_quantization_gb300 import ep as EP
    idx = torch.tensor([[0, 5], [7, 7], [3, 9], [4, 1]], dtype=torch.int32)
    plan = EP.make_plan(idx, 8, 2)
    # owners: experts 0-3 -> rank 0, 4-7 -> rank 1; (1,1) repeats expert 7, (2,1) is out of range
    assert plan["order"].tolist() == [0, 4, 7, 1, 2, 6]
    assert plan["send_counts"] == [3, 3]
    assert plan["local_expert"].tolist() == [0, 3, 1, 1, 3, 0]
    assert plan["row_of"].tolist() == [[0, 1], [2, -1], [4, -1], [6, 7]]
    with pytest.raises(ValueError):
        EP.make_plan(idx, 8, 3)
