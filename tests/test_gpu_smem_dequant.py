"""QAD_FLAG_SMEM_DEQUANT on the GPU: the grouped GEMMs fake-quantize their weight tiles in
shared memory instead of reading a materialised fake-quant copy (AngelSlim mcore_qad
walkthrough, section 二.4: the stacked experts are fake-quantized and consumed by one grouped
GEMM).

The converted tiles (dumped with QAD_FLAG_DEQUANT_DUMP) must equal the oracle's fake-quant
bit for bit, and since the GEMMs then contract the same values in the same order, every
output and gradient must equal the materialised-copy run's bit for bit.
"""
import numpy as np
import pytest
import torch

import scale_only_quantization_gb300 as Q
from oracle import quant as OQ
import synth

from gpu_util import Run, bits, host_inputs

pytestmark = pytest.mark.gpu

FMTS = [Q.QAD_FMT_NVFP4, Q.QAD_FMT_INT4_G128, Q.QAD_FMT_FP8_ROW, Q.QAD_FMT_NVFP4A16, Q.QAD_FMT_W8A8,
        Q.QAD_FMT_W4AFP8, Q.QAD_FMT_NVFP4_E4M3]
DQ = Q.QAD_FLAG_SMEM_DEQUANT


@pytest.fixture(scope="module", autouse=True)
def _built():
    from scale_only_quantization_gb300 import build
    build.build()
    Q.lib()


def _same(a, b):
    assert a.error == 0 and b.error == 0
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.dx.view(torch.int16), b.dx.view(torch.int16))
    assert torch.equal(a.dprobs, b.dprobs)
    assert torch.equal(a.ds13, b.ds13) and torch.equal(a.ds2, b.ds2)


def _dumps_match_oracle(run, host):
    inp = run.inp
    E, d, F, fmt = inp["E"], inp["d"], inp["F"], inp["fmt"]
    w13h = bits(run.view("W13_HAT", torch.bfloat16)).reshape(E, 2 * F, d)
    w2h = bits(run.view("W2_HAT", torch.bfloat16)).reshape(E, d, F)
    want13 = OQ.f64_to_bf16_bits(OQ.fakequant_weight(fmt, host["w13"], host["s13"]))
    want2 = OQ.f64_to_bf16_bits(OQ.fakequant_weight(fmt, host["w2"], host["s2"]))
    bad13 = int(np.count_nonzero(w13h != want13))
    bad2 = int(np.count_nonzero(w2h != want2))
    assert bad13 == 0 and bad2 == 0, "converted tiles differ from the oracle: %d of W13, %d of W2" % (bad13, bad2)


def _tiny(fmt, **over):
    return synth.make_inputs(synth.workload("tiny_nvfp4", fmt=fmt, **over), seed=0, device="cuda")


@pytest.mark.parametrize("fmt", FMTS)
def test_dequantized_tiles_are_bit_exact_and_outputs_identical(fmt):
    inp = _tiny(fmt)
    a = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    b = Run(inp, flags=DQ | Q.QAD_FLAG_DEQUANT_DUMP | Q.QAD_FLAG_STASH_H, zero_ws=True)
    _dumps_match_oracle(b, host_inputs(inp))
    _same(a, b)
    assert b.view("H_HAT", torch.bfloat16).numel() == a.view("H_HAT", torch.bfloat16).numel()


@pytest.mark.parametrize("fmt", [Q.QAD_FMT_NVFP4, Q.QAD_FMT_INT4_G128, Q.QAD_FMT_FP8_ROW, Q.QAD_FMT_NVFP4_E4M3])
def test_every_dequantizing_gemm_converts_every_tile(fmt):
    """The forward's GEMMs (fc1, fc2) and the input-gradient GEMMs (dgrad fc2, dgrad fc1) each
    write the values they converted: after clearing the dump between the calls, the dgrad call
    alone must rebuild both weights completely."""
    inp = _tiny(fmt)
    host = host_inputs(inp)
    T, d, F, E, k = inp["T"], inp["d"], inp["F"], inp["E"], inp["topk"]
    s = Q.shape(T, d, F, E, k, fmt, DQ | Q.QAD_FLAG_DEQUANT_DUMP)
    ws = torch.zeros(Q.qad_moe_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty_like(out)
    Q.qad_moe_fwd(s, inp["x"], inp["topk_idx"], inp["topk_w"], inp["w13"], inp["s13"], inp["w2"], inp["s2"], out, ws)

    class _R:
        pass

    r = _R()
    r.inp = inp
    r.view = lambda name, dt: Q.workspace_view(ws, s, name, dt)
    torch.cuda.synchronize()
    _dumps_match_oracle(r, host)
    r.view("W13_HAT", torch.bfloat16).zero_()
    r.view("W2_HAT", torch.bfloat16).zero_()
    Q.qad_moe_bwd_dgrad(s, inp["dout"], inp["topk_w"], inp["w13"], inp["s13"], inp["w2"], inp["s2"], dx, None, ws)
    assert Q.qad_check_device_error(ws) == 0
    _dumps_match_oracle(r, host)


def test_uneven_shapes_and_ragged_routing_identical():
    """d = 768, F = 384 (128-column tiles for the F-sized GEMMs, so both converter layouts of the
    K-major and MN-major weight tiles at two widths), top-3, T = 333, E = 6."""
    inp = synth.make_inputs(synth.workload("tiny_nvfp4", E=6, d=768, F=384, topk=3, T=333), seed=9, device="cuda")
    a = Run(inp, flags=0)
    b = Run(inp, flags=DQ | Q.QAD_FLAG_DEQUANT_DUMP, zero_ws=True)
    _dumps_match_oracle(b, host_inputs(inp))
    _same(a, b)


def test_empty_and_single_row_experts_identical():
    base = synth.make_inputs(synth.workload("tiny_nvfp4", E=8, T=300), seed=1, device="cuda")
    rng = np.random.default_rng(3)
    idx = np.stack([rng.choice([0, 3, 5], 2, replace=False) for _ in range(300)])
    idx[17] = [6, 0]
    inp = dict(base)
    inp["topk_idx"] = torch.as_tensor(idx, dtype=torch.int32, device="cuda").contiguous()
    a = Run(inp, flags=0)
    b = Run(inp, flags=DQ)
    _same(a, b)


def test_with_recompute_identical():
    inp = _tiny(Q.QAD_FMT_NVFP4)
    a = Run(inp, flags=0)
    b = Run(inp, flags=DQ | Q.QAD_FLAG_RECOMPUTE)
    _same(a, b)


def test_full_size_identical_to_the_materialised_copy():
    """qwen3_30b_a3b_nvfp4 (E = 128, d = 2048, F = 768, top-8, 16384 tokens), in the launch
    configuration the benchmark times: every output bit equal, in a workspace without the two
    weight copies."""
    inp = synth.make_inputs(synth.workload("qwen3_30b_a3b_nvfp4"), seed=5, device="cuda")
    a = Run(inp, flags=0)
    ref = [t.clone() for t in (a.out, a.dx, a.dprobs, a.ds13, a.ds2)]
    nb_a = a.ws.numel()
    del a
    torch.cuda.empty_cache()
    b = Run(inp, flags=DQ)
    assert b.error == 0
    E, d, F = inp["E"], inp["d"], inp["F"]
    assert nb_a - b.ws.numel() >= 2 * 3 * E * F * d
    for x, y in zip(ref, (b.out, b.dx, b.dprobs, b.ds13, b.ds2)):
        assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x.view(torch.int16),
                           y.view(torch.int32) if y.dtype == torch.float32 else y.view(torch.int16))
