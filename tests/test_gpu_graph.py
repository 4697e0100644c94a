"""The whole step (forward, dgrad, scale gradient) captured in one CUDA graph.

Every call only enqueues work on the caller's stream (plus an internal side stream that
forks from it and joins back with events) and allocates nothing, so a caller can capture a
training step once and replay it.  The replay must give the eager run's bits, and since the
routing maps and the GEMM tile lists are built on the device, one captured graph serves new
inputs of the same shape, new routing included, written into the captured buffers.
"""
import pytest
import torch

import scale_only_quantization_gb300 as Q
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from scale_only_quantization_gb300 import build
    build.build()
    Q.lib()


def _buffers(inp, s):
    T, d, k = inp["T"], inp["d"], inp["topk"]
    nan = float("nan")
    return dict(
        ws=torch.empty(Q.qad_moe_workspace_bytes(s), dtype=torch.uint8, device="cuda"),
        out=torch.full((T, d), nan, dtype=torch.bfloat16, device="cuda"),
        dx=torch.full((T, d), nan, dtype=torch.bfloat16, device="cuda"),
        dprobs=torch.full((T, k), nan, dtype=torch.float32, device="cuda"),
        ds13=torch.full_like(inp["s13"], nan),
        ds2=torch.full_like(inp["s2"], nan),
    )


def _step(s, inp, b):
    Q.qad_moe_fwd(s, inp["x"], inp["topk_idx"], inp["topk_w"], inp["w13"], inp["s13"], inp["w2"], inp["s2"],
                  b["out"], b["ws"])
    Q.qad_moe_bwd_dgrad(s, inp["dout"], inp["topk_w"], inp["w13"], inp["s13"], inp["w2"], inp["s2"], b["dx"],
                        b["dprobs"], b["ws"])
    Q.qad_moe_bwd_scalegrad(s, inp["w13"], inp["s13"], inp["w2"], inp["s2"], b["ds13"], b["ds2"], 0, b["ws"])


def _same_bits(a, b):
    for name in ("out", "dx", "dprobs", "ds13", "ds2"):
        x, y = a[name], b[name]
        iv = torch.int16 if x.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(x.view(iv), y.view(iv)), name


INPUTS = ("x", "dout", "topk_idx", "topk_w", "w13", "s13", "w2", "s2")


@pytest.mark.parametrize("fmt, flags", [
    (Q.QAD_FMT_NVFP4, 0),
    (Q.QAD_FMT_NVFP4, Q.QAD_FLAG_RECOMPUTE),
    (Q.QAD_FMT_FP8_ROW, Q.QAD_FLAG_NATIVE_FP8),
    (Q.QAD_FMT_NVFP4_E4M3, 0),
])
def test_step_captured_in_a_cuda_graph_replays_bit_identically(fmt, flags):
    cfg = synth.workload("tiny_nvfp4", fmt=fmt, T=1536, E=8)
    inp = synth.make_inputs(cfg, seed=3, device="cuda")
    s = Q.shape(inp["T"], inp["d"], inp["F"], inp["E"], inp["topk"], inp["fmt"], flags)

    eager = _buffers(inp, s)
    _step(s, inp, eager)
    torch.cuda.synchronize()
    assert Q.qad_check_device_error(eager["ws"]) == 0

    static = _buffers(inp, s)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # one warm-up run outside the capture
        _step(s, inp, static)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(s, inp, static)
    for name in ("out", "dx", "dprobs", "ds13", "ds2"):
        static[name].fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert Q.qad_check_device_error(static["ws"]) == 0
    _same_bits(eager, static)

    # new values, new routing: written into the captured inputs, replayed
    new = synth.make_inputs(cfg, seed=4, device="cuda")
    assert not torch.equal(new["topk_idx"], inp["topk_idx"])
    for name in INPUTS:
        inp[name].copy_(new[name])
    graph.replay()
    fresh = _buffers(new, s)
    _step(s, new, fresh)
    torch.cuda.synchronize()
    assert Q.qad_check_device_error(static["ws"]) == 0
    _same_bits(fresh, static)
