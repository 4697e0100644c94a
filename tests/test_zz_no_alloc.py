"""The routing entry point that allocates nothing (qad_route_permute_noalloc).

It exists for callers that cannot allocate device memory (inside a CUDA-graph stream
capture, or under a runtime that owns all device memory and passes a plugin only its
inputs and outputs): its scratch is a fixed device array inside the library.  Its maps
must equal, bit for bit, those the layer's own forward builds in its workspace, on two
calls in a row (the second must not see the first one's leftovers: the first call has
invalid indices and sets error bits, the second is clean).  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import scale_only_quantization_gb300 as Q
import synth


def _rmax(T, k, E):
    return (T * k + 127 * E + 127) // 128 * 128


def test_sizes_beyond_the_scratch_are_rejected_before_launch():
    from scale_only_quantization_gb300 import build
    build.build()
    L = Q.lib()
    P = ctypes.c_void_p
    big_e = Q.QAD_NOALLOC_MAX_EXPERTS + 1
    assert L.qad_route_permute_noalloc(P(16), 4, 2, big_e, P(16), P(16), P(16), P(16), P(16), P(16),
                                       None) == Q.QAD_ERR_SCRATCH_LIMIT
    T = Q.QAD_NOALLOC_MAX_PAIRS // 8 + 1
    assert L.qad_route_permute_noalloc(P(16), T, 8, 128, P(16), P(16), P(16), P(16), P(16), P(16),
                                       None) == Q.QAD_ERR_SCRATCH_LIMIT
    assert "scratch" in Q.status_string(Q.QAD_ERR_SCRATCH_LIMIT)


@pytest.mark.gpu
def test_noalloc_routing_equals_layer_routing_on_two_calls():
    from gpu_util import Run
    from scale_only_quantization_gb300 import build
    build.build()
    base = synth.make_inputs(synth.workload("tiny_nvfp4", E=8, T=700), seed=5, device="cuda")
    T, k, E = 700, 2, 8
    rng = np.random.default_rng(9)
    good = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    bad = good.copy()
    bad[3] = [E + 2, 1]       # out of range
    bad[40] = [5, 5]          # repeated expert
    Rmax = _rmax(T, k, E)
    for idx in (bad, good):
        inp = dict(base)
        inp["topk_idx"] = torch.as_tensor(idx, dtype=torch.int32, device="cuda").contiguous()
        run = Run(inp)                                      # the layer's own routing, in its workspace
        ref = run.routing()
        out = dict(row_token=torch.full((Rmax,), -99, dtype=torch.int32, device="cuda"),
                   row_slot=torch.full((Rmax,), -99, dtype=torch.int32, device="cuda"),
                   row_of=torch.full((T * k,), -99, dtype=torch.int32, device="cuda"),
                   offsets=torch.full((E + 1,), -99, dtype=torch.int32, device="cuda"),
                   counts=torch.full((E,), -99, dtype=torch.int32, device="cuda"),
                   header=torch.full((4,), -99, dtype=torch.int32, device="cuda"))
        Q.qad_route_permute_noalloc(inp["topk_idx"], T, k, E, out["row_token"], out["row_slot"], out["row_of"],
                                    out["offsets"], out["counts"], out["header"])
        torch.cuda.synchronize()
        hdr = out["header"].cpu().numpy()
        assert np.array_equal(hdr, ref["hdr"][:4]), (hdr, ref["hdr"][:4])
        rpad = int(hdr[2])
        assert np.array_equal(out["row_token"][:rpad].cpu().numpy(), ref["row_token"])
        assert np.array_equal(out["row_slot"][:rpad].cpu().numpy(), ref["row_slot"])
        assert np.array_equal(out["row_of"].cpu().numpy().reshape(T, k), ref["row_of"])
        assert np.array_equal(out["offsets"].cpu().numpy(), ref["offs"])
        assert np.array_equal(out["counts"].cpu().numpy(), ref["counts"])
        want_err = (Q.QAD_DEV_BAD_INDEX | Q.QAD_DEV_DUP_INDEX) if idx is bad else 0
        assert int(hdr[0]) == want_err
