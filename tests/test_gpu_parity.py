"""GPU parity of the CUDA path against the fp64 oracle, through the C ABI (small cases).

Protocol (stage by stage, "teacher forced"): quantized values and routing maps are
compared bit for bit; each floating-point stage is compared with the oracle applied to
the GPU's own bf16 output of the previous stage, within the tolerances of gpu_util.
The activation quantizer is discontinuous, so a one-ulp difference in H may move one
FP4 code; the end-to-end comparison from raw inputs only reports how many moved.
"""
import numpy as np
import pytest
import torch

import scale_only_quantization_gb300 as Q
from oracle import moe as OM
from oracle import quant as OQ
import synth

from gpu_util import (E2E_REL_L2, Run, assert_close, assert_scale_grad, bits, e4m3_values, host_inputs, rel_l2,
                      unpadded_row_of, vals)

pytestmark = pytest.mark.gpu

FMTS = [Q.QAD_FMT_NVFP4, Q.QAD_FMT_INT4_G128, Q.QAD_FMT_FP8_ROW, Q.QAD_FMT_NVFP4A16, Q.QAD_FMT_W8A8,
        Q.QAD_FMT_W4AFP8, Q.QAD_FMT_NVFP4_E4M3]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from scale_only_quantization_gb300 import build
    build.build()
    Q.lib()


# ------------------------------------------------------------------------------ weight fake-quant

def _special_weights(E, N, K, fmt, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = torch.randn((E, N, K), generator=g, device="cuda") * 0.02
    w[0, 0, :8] = torch.tensor([0.5, -0.5, 0.0, -0.0, 1e-30, -1e-30, 3.0, -3.0], device="cuda")
    w[0, 1, :] = 0.0                                   # all-zero rows -> zero scales
    w[-1, -1, ::7] *= 40.0                             # outliers inside their block
    w[0, 3, :] *= 2.0 ** -12                           # a row of tiny scales (deployed E4M3: subnormal)
    w = w.to(torch.bfloat16)
    s = synth.init_scales(w, fmt, g)
    s[0, 2] *= 0.25                                    # clipped weights
    return w.contiguous(), s.contiguous()


@pytest.mark.parametrize("fmt", FMTS)
# the last shape has more 16-element chunks (277,560) than two passes of the persistent grid's
# threads over them (3 CTAs x 256 threads x 152 SMs = 116,736 per pass), and not a multiple of
# that: every thread runs several iterations of its load-ahead loop and the last ones are ragged
@pytest.mark.parametrize("E,N,K", [(3, 64, 512), (1, 5, 256), (2, 128, 2048), (5, 771, 1152)])
def test_fakequant_bit_exact(fmt, E, N, K):
    w, s = _special_weights(E, N, K, fmt, seed=100 + fmt)
    out = torch.empty_like(w)
    if fmt == Q.QAD_FMT_NVFP4_E4M3:
        # the deployed scales, then the plain nvfp4 fake-quant with them (the header's recipe)
        with pytest.raises(Q.QADError):
            Q.qad_fakequant_fwd(fmt, w, s, out, E, N, K)
        sq = torch.empty_like(s)
        Q.qad_nvfp4_deploy_scales(s, sq, E, s[0].numel())
        Q.qad_fakequant_fwd(Q.QAD_FMT_NVFP4, w, sq, out, E, N, K)
    else:
        Q.qad_fakequant_fwd(fmt, w, s, out, E, N, K)
    torch.cuda.synchronize()
    want = OQ.f64_to_bf16_bits(OQ.fakequant_weight(fmt, bits(w), synth.to_numpy(s)))
    got = bits(out)
    bad = np.count_nonzero(got != want)
    assert bad == 0, "%d of %d fake-quant outputs differ" % (bad, got.size)


def test_fakequant_empty_is_a_no_op():
    Q.qad_fakequant_fwd(0, None, None, None, 0, 16, 64)


# ------------------------------------------------------------------------------ routing

def _check_routing(run, host):
    rt = run.routing()
    ref = OM.route(host["topk_idx"], run.inp["E"])
    real = rt["real"]
    assert np.array_equal(rt["row_token"][real], ref["row_token"])
    assert np.array_equal(rt["row_slot"][real], ref["row_slot"])
    assert np.array_equal(rt["counts"], ref["counts"])
    padded = (ref["counts"] + 127) // 128 * 128
    assert np.array_equal(rt["offs"], np.concatenate([[0], np.cumsum(padded)]))
    assert np.array_equal(unpadded_row_of(rt), ref["row_of"])
    assert rt["hdr"][0] == ref["error"] == run.error
    assert rt["rpad"] == padded.sum() and rt["hdr"][1] == padded.sum() // 128
    return rt, ref


# ------------------------------------------------------------------------------ the layer, stage by stage

def _codes(run, name, n_rows, cols, rows=None):
    t = run.view(name, torch.uint8).cpu().numpy()[: n_rows * cols].reshape(n_rows, cols)
    return e4m3_values(t if rows is None else t[rows])


def _stagewise(run, host, check_h=True, factored=False):
    """Teacher-forced comparison of every stage; returns the GPU stages for further use.

    factored: the native fp8 forward (QAD_FLAG_NATIVE_FP8) -- the E4M3 codes and row scales
    are checked bit for bit and fc1 / fc2 against the oracle's scale-factored GEMMs."""
    inp = run.inp
    fmt, T, d, F, E, k = inp["fmt"], inp["T"], inp["d"], inp["F"], inp["E"], inp["topk"]
    rt, ref = _check_routing(run, host)
    real, off = rt["real"], ref["offsets"]
    row_of = ref["row_of"]
    p = host["topk_w"].astype(np.float64)

    # fake-quantized weights (bit exact)
    w13h_b = bits(run.view("W13_HAT", torch.bfloat16)).reshape(E, 2 * F, d)
    w2h_b = bits(run.view("W2_HAT", torch.bfloat16)).reshape(E, d, F)
    assert np.array_equal(w13h_b, OQ.f64_to_bf16_bits(OQ.fakequant_weight(fmt, host["w13"], host["s13"])))
    assert np.array_equal(w2h_b, OQ.f64_to_bf16_bits(OQ.fakequant_weight(fmt, host["w2"], host["s2"])))
    w13h, w2h = OQ.bf16_to_f64(w13h_b), OQ.bf16_to_f64(w2h_b)

    # A1 = AQ(x) gathered (bit exact); padding rows are zero
    a1_all = run.rows("A1", d)
    a1 = a1_all[real]
    want_a1 = OQ.fakequant_act(fmt, OQ.bf16_to_f64(host["x"]))[ref["row_token"]]
    assert np.array_equal(OQ.f64_to_bf16_bits(a1), OQ.f64_to_bf16_bits(want_a1))
    assert np.all(a1_all[~real] == 0)

    # Z1 = A1 . W13_hat^T
    z1_all = run.rows("Z1", 2 * F)
    z1 = z1_all[real]
    x64 = OQ.bf16_to_f64(host["x"])
    if factored:
        qw13 = _codes(run, "W13_CODES", E * 2 * F, d).reshape(E, 2 * F, d)
        s13 = host["s13"].astype(np.float64)
        assert np.array_equal(qw13 * s13, OQ.fakequant_weight_factored(fmt, host["w13"], host["s13"]))
        qw2 = _codes(run, "W2_CODES", E * d, F).reshape(E, d, F)
        assert np.array_equal(qw2 * host["s2"].astype(np.float64),
                              OQ.fakequant_weight_factored(fmt, host["w2"], host["s2"]))
        sa = synth.to_numpy(run.view("A_SCALE", torch.float32)).astype(np.float64)
        assert np.array_equal(sa, OQ.act_scale(fmt, x64)[:, 0])
        qa = _codes(run, "A1_CODES", rt["rpad"], d)
        assert np.array_equal(qa[real] * sa[ref["row_token"]][:, None],
                              OQ.fakequant_act_factored(fmt, x64)[ref["row_token"]])
        assert np.all(qa[~real] == 0)
        want_z1 = OM.grouped_gemm_nt(OQ.fakequant_act_factored(fmt, x64)[ref["row_token"]],
                                     OQ.fakequant_weight_factored(fmt, host["w13"], host["s13"]), off)
    else:
        want_z1 = OM.grouped_gemm_nt(a1, w13h, off)
    assert_close(z1, want_z1, "Z1")
    assert np.all(z1_all[~real] == 0)

    # H and H_hat = AQ(H): bit exact given the GPU's H
    hh = run.rows("H_HAT", F)[real]
    if check_h:
        h = run.rows("H", F)[real]
        assert_close(h, OM.swiglu(z1), "H")
        assert np.array_equal(OQ.f64_to_bf16_bits(hh), OQ.f64_to_bf16_bits(OQ.fakequant_act(fmt, h)))

    # Y = H_hat . W2_hat^T, out = sum_j p Y
    y = run.rows("Y", d)[real]
    if factored:
        h = run.rows("H", F)[real]
        sh = synth.to_numpy(run.view("H_SCALE", torch.float32)).astype(np.float64)[: rt["rpad"]][real]
        assert np.array_equal(sh, OQ.act_scale(fmt, h)[:, 0])
        qh = _codes(run, "H_CODES", rt["rpad"], F)[real]
        assert np.array_equal(qh * sh[:, None], OQ.fakequant_act_factored(fmt, h))
        want_y = OM.grouped_gemm_nt(OQ.fakequant_act_factored(fmt, h),
                                    OQ.fakequant_weight_factored(fmt, host["w2"], host["s2"]), off)
    else:
        want_y = OM.grouped_gemm_nt(hh, w2h, off)
    assert_close(y, want_y, "Y")
    out = vals(run.out)
    assert_close(out, OM.combine(y, p, row_of), "out")

    # dY = bf16(fp32(p * dout)) (bit exact), padding rows zero
    dy_all = run.rows("DY", d)
    dy = dy_all[real]
    dout = OQ.bf16_to_f64(host["dout"])
    want_dy = OQ.round_bf16(OQ.round_f32(dout[ref["row_token"]] * p[ref["row_token"], ref["row_slot"]][:, None]))
    assert np.array_equal(OQ.f64_to_bf16_bits(dy), OQ.f64_to_bf16_bits(want_dy))
    assert np.all(dy_all[~real] == 0)

    # dZ1 = SwiGLU'(dY . W2_hat) given the GPU's Z1
    dz1 = run.rows("DZ1", 2 * F)[real]
    assert_close(dz1, OM.swiglu_bwd(OM.grouped_gemm_nn(dy, w2h, off), z1), "dZ1")
    da1 = run.rows("DA1", d)[real]
    assert_close(da1, OM.grouped_gemm_nn(dz1, w13h, off), "dA1")
    assert_close(vals(run.dx), OM.combine(da1, np.ones((T, k)), row_of), "dx")
    if run.dprobs is not None:
        dp = np.zeros((T, k))
        for j in range(k):
            r = row_of[:, j]
            ok = r >= 0
            dp[ok, j] = np.einsum("td,td->t", dout[ok], y[r[ok]])
        assert_close(synth.to_numpy(run.dprobs).astype(np.float64), dp, "dprobs")

    # scale gradients from the GPU's stored operands
    dw2 = OM.grouped_wgrad(dy, hh, off, E)
    dw13 = OM.grouped_wgrad(dz1, a1, off, E)
    ds2 = OQ.scale_grad_from_wgrad(fmt, dw2, host["w2"], host["s2"])
    ds13 = OQ.scale_grad_from_wgrad(fmt, dw13, host["w13"], host["s13"])
    assert_scale_grad(synth.to_numpy(run.ds2), ds2.reshape(host["s2"].shape), "ds2")
    assert_scale_grad(synth.to_numpy(run.ds13), ds13.reshape(host["s13"].shape), "ds13")
    return dict(y=y, ds2=ds2, ds13=ds13)


def _tiny(fmt, **over):
    cfg = synth.workload("tiny_nvfp4", fmt=fmt, **over)
    return synth.make_inputs(cfg, seed=0, device="cuda")


@pytest.mark.parametrize("fmt", FMTS)
def test_layer_stagewise_tiny(fmt):
    inp = _tiny(fmt)
    host = host_inputs(inp)
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    assert run.error == 0
    _stagewise(run, host)

    # end to end from raw inputs: report moved activation codes, check the outputs loosely
    fwd = OM.moe_forward(fmt, host["x"], host["topk_idx"], host["topk_w"], host["w13"], host["s13"], host["w2"],
                         host["s2"])
    rt = run.routing()
    hh_gpu = run.rows("H_HAT", inp["F"])[rt["real"]]
    moved = int(np.count_nonzero(OQ.f64_to_bf16_bits(hh_gpu) != OQ.f64_to_bf16_bits(fwd["hh"])))
    print("fmt %d: %d of %d H_hat codes differ end to end" % (fmt, moved, hh_gpu.size))
    assert moved <= 0.01 * hh_gpu.size
    # out and dx end to end: relative L2 <= 1e-3 (a moved code shifts one element by about one
    # grid step of its block; a quantizer applied to the wrong tensor moves the whole output)
    bwd = OM.moe_dgrad(host["dout"], host["topk_w"], fwd)
    assert rel_l2(vals(run.out), fwd["out"]) <= E2E_REL_L2
    assert rel_l2(vals(run.dx), bwd["dx"]) <= E2E_REL_L2


def test_stash_h_flag_off_matches_on():
    inp = _tiny(Q.QAD_FMT_NVFP4)
    a = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    b = Run(inp, flags=0)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.dx.view(torch.int16), b.dx.view(torch.int16))
    assert torch.equal(a.ds13, b.ds13) and torch.equal(a.ds2, b.ds2)


def test_native_fp8_forward_stagewise_tiny():
    """QAD_FLAG_NATIVE_FP8: fc1 and fc2 contract E4M3 codes on the fp8 tensor path and apply the
    row scales to the sums; every stage against the oracle's scale-factored forward."""
    inp = _tiny(Q.QAD_FMT_FP8_ROW)
    host = host_inputs(inp)
    run = Run(inp, flags=Q.QAD_FLAG_NATIVE_FP8 | Q.QAD_FLAG_STASH_H)
    assert run.error == 0
    _stagewise(run, host, factored=True)
    # the end-to-end output stays close to the rounded reading's
    fwd = OM.moe_forward(Q.QAD_FMT_FP8_ROW, host["x"], host["topk_idx"], host["topk_w"], host["w13"], host["s13"],
                         host["w2"], host["s2"], factored=True)
    assert rel_l2(vals(run.out), fwd["out"]) <= E2E_REL_L2
    assert rel_l2(vals(run.dx), OM.moe_dgrad(host["dout"], host["topk_w"], fwd)["dx"]) <= E2E_REL_L2


def test_native_fp8_flag_rejected_for_other_formats():
    for fmt in (Q.QAD_FMT_NVFP4, Q.QAD_FMT_W8A8):
        assert Q.qad_moe_workspace_bytes(Q.shape(512, 256, 128, 4, 2, fmt, Q.QAD_FLAG_NATIVE_FP8)) == 0
    assert Q.qad_moe_workspace_bytes(
        Q.shape(512, 256, 128, 4, 2, Q.QAD_FMT_FP8_ROW, Q.QAD_FLAG_NATIVE_FP8 | Q.QAD_FLAG_NO_QUANT)) == 0


def test_native_fp8_recompute_is_bit_identical():
    inp = _tiny(Q.QAD_FMT_FP8_ROW)
    a = Run(inp, flags=Q.QAD_FLAG_NATIVE_FP8)
    b = Run(inp, flags=Q.QAD_FLAG_NATIVE_FP8 | Q.QAD_FLAG_RECOMPUTE)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.dx.view(torch.int16), b.dx.view(torch.int16))
    assert torch.equal(a.ds13, b.ds13) and torch.equal(a.ds2, b.ds2)


@pytest.mark.parametrize("fmt", [Q.QAD_FMT_NVFP4, Q.QAD_FMT_FP8_ROW, Q.QAD_FMT_INT4_G128])
def test_recompute_matches_stash_bit_for_bit(fmt):
    """QAD_FLAG_RECOMPUTE drops the Z1 stash and reruns fc1 in the dgrad call: the same
    mainloop over the same tiles, so every output and gradient is identical bit for bit."""
    inp = _tiny(fmt)
    a = Run(inp, flags=0)
    b = Run(inp, flags=Q.QAD_FLAG_RECOMPUTE)
    assert a.error == 0 and b.error == 0
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.dx.view(torch.int16), b.dx.view(torch.int16))
    assert torch.equal(a.dprobs, b.dprobs)
    assert torch.equal(a.ds13, b.ds13) and torch.equal(a.ds2, b.ds2)
    F = inp["F"]
    assert np.array_equal(a.rows_bits("Z1", 2 * F), b.rows_bits("Z1", 2 * F))
    assert np.array_equal(a.rows_bits("DZ1", 2 * F), b.rows_bits("DZ1", 2 * F))


def test_runs_are_deterministic():
    inp = _tiny(Q.QAD_FMT_NVFP4)
    a, b = Run(inp), Run(inp)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.dx.view(torch.int16), b.dx.view(torch.int16))
    assert torch.equal(a.dprobs, b.dprobs)
    assert torch.equal(a.ds13, b.ds13) and torch.equal(a.ds2, b.ds2)


@pytest.mark.parametrize("fmt", [Q.QAD_FMT_NVFP4, Q.QAD_FMT_INT4_G128, Q.QAD_FMT_FP8_ROW])
def test_weights_only_16_byte_aligned_give_identical_results(fmt):
    """The scale-gradient epilogue reads W with 256-bit loads when W is 32-byte aligned and
    with 16-byte loads otherwise (the ABI asks for 16): both give the same bits."""
    inp = _tiny(fmt)
    a = Run(inp)
    moved = dict(inp)
    for name in ("w13", "w2"):
        buf = torch.empty(inp[name].numel() + 8, dtype=torch.bfloat16, device="cuda")
        assert buf.data_ptr() % 32 == 0
        v = buf[8:].view(inp[name].shape)  # 16 bytes past a 32-byte boundary
        v.copy_(inp[name])
        assert v.data_ptr() % 32 == 16
        moved[name] = v
    b = Run(moved)
    assert a.error == 0 and b.error == 0
    assert torch.equal(a.ds13, b.ds13) and torch.equal(a.ds2, b.ds2)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.dx.view(torch.int16), b.dx.view(torch.int16))


@pytest.mark.parametrize("fmt", FMTS)
def test_scalegrad_accumulate_adds(fmt):
    inp = _tiny(fmt)
    a = Run(inp)
    base = (torch.full_like(inp["s13"], 0.5), torch.full_like(inp["s2"], -0.25))
    b = Run(inp, accumulate=1, ds_init=base)
    assert torch.allclose(b.ds13, a.ds13 + 0.5, rtol=0, atol=1e-6 * float(a.ds13.abs().max()) + 1e-6)
    assert torch.allclose(b.ds2, a.ds2 - 0.25, rtol=0, atol=1e-6 * float(a.ds2.abs().max()) + 1e-6)


# ------------------------------------------------------------------------------ edge cases

def _custom_routing(inp, idx):
    inp = dict(inp)
    T, k = idx.shape
    g = torch.Generator(device="cuda").manual_seed(7)
    inp["topk_idx"] = torch.as_tensor(idx, dtype=torch.int32, device="cuda").contiguous()
    inp["topk_w"] = torch.softmax(torch.randn((T, k), generator=g, device="cuda"), 1).contiguous()
    inp["x"] = inp["x"][:T].contiguous()
    inp["dout"] = inp["dout"][:T].contiguous()
    inp["T"], inp["topk"] = T, k
    return inp


def test_empty_experts_single_row_expert_and_small_batch():
    base = synth.make_inputs(synth.workload("tiny_nvfp4", E=8, T=300), seed=1, device="cuda")
    rng = np.random.default_rng(3)
    T, k = 300, 2
    idx = np.stack([rng.choice([0, 3, 5], 2, replace=False) for _ in range(T)])
    idx[17] = [6, 0]                                  # expert 6 gets exactly one row
    inp = _custom_routing(base, idx)
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    assert run.error == 0
    res = _stagewise(run, host_inputs(inp))
    # experts that received no rows get a zero scale gradient
    for e in (1, 2, 4, 7):
        assert np.all(synth.to_numpy(run.ds13)[e] == 0) and np.all(synth.to_numpy(run.ds2)[e] == 0)
    assert np.count_nonzero(synth.to_numpy(run.ds13)[6]) > 0


@pytest.mark.parametrize("E, topk, T", [
    (1024, 32, 96),   # the largest expert count and top-k the layout accepts; most experts empty
    (1, 1, 700),      # a dense layer: one expert, every token routed to it (ragged last tile)
    (4, 1, 513),      # top-1 routing
])
def test_extreme_expert_counts_and_top_k(E, topk, T):
    inp = synth.make_inputs(synth.workload("tiny_nvfp4", E=E, topk=topk, T=T), seed=4, device="cuda")
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    assert run.error == 0
    _stagewise(run, host_inputs(inp))


@pytest.mark.parametrize("fmt", [Q.QAD_FMT_NVFP4, Q.QAD_FMT_FP8_ROW])
def test_layer_stagewise_uneven_shapes(fmt):
    """d = 768 (not a multiple of 512: a partial row chunk in the token scatters, six 128-wide
    K stages in fc1), F = 384 (128-column tiles for the F-sized GEMMs, 2F = 768), top-3,
    T = 333 (ragged), E = 6."""
    inp = synth.make_inputs(synth.workload("tiny_nvfp4", fmt=fmt, E=6, d=768, F=384, topk=3, T=333), seed=9,
                            device="cuda")
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    assert run.error == 0
    _stagewise(run, host_inputs(inp))


def test_fewer_rows_than_one_tile():
    base = synth.make_inputs(synth.workload("tiny_nvfp4"), seed=2, device="cuda")
    idx = np.array([[1, 2], [2, 3], [0, 1], [3, 0], [1, 3]])
    inp = _custom_routing(base, idx)
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    _stagewise(run, host_inputs(inp))


def test_zero_tokens():
    base = synth.make_inputs(synth.workload("tiny_nvfp4"), seed=3, device="cuda")
    inp = _custom_routing(base, np.zeros((0, 2), dtype=np.int64))
    run = Run(inp)
    assert run.error == 0
    assert torch.all(run.ds13 == 0) and torch.all(run.ds2 == 0)


def test_invalid_routing_indices_are_dropped_and_flagged():
    base = synth.make_inputs(synth.workload("tiny_nvfp4"), seed=4, device="cuda")
    rng = np.random.default_rng(5)
    idx = np.stack([rng.permutation(4)[:2] for _ in range(512)])
    idx[3] = [9, 1]            # out of range
    idx[10] = [2, 2]           # repeated expert
    idx[11] = [-1, -7]         # negative
    inp = _custom_routing(base, idx)
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    assert run.error == (Q.QAD_DEV_BAD_INDEX | Q.QAD_DEV_DUP_INDEX)
    _stagewise(run, host_inputs(inp))
    dp = synth.to_numpy(run.dprobs)
    assert dp[3, 0] == 0 and dp[10, 1] == 0 and np.all(dp[11] == 0)


def test_outputs_stay_inside_their_buffers():
    """Guard bands around every output keep their sentinel values."""
    inp = _tiny(Q.QAD_FMT_NVFP4)
    T, d, k = inp["T"], inp["d"], inp["topk"]
    G = 256
    s = Q.shape(T, d, inp["F"], inp["E"], k, 0)
    ws = torch.empty(Q.qad_moe_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    big_out = torch.full((T * d + 2 * G,), 7.0, dtype=torch.bfloat16, device="cuda")
    big_dx = torch.full((T * d + 2 * G,), 7.0, dtype=torch.bfloat16, device="cuda")
    big_dp = torch.full((T * k + 2 * G,), 7.0, dtype=torch.float32, device="cuda")
    n13, n2 = inp["s13"].numel(), inp["s2"].numel()
    big13 = torch.full((n13 + 2 * G,), 7.0, dtype=torch.float32, device="cuda")
    big2 = torch.full((n2 + 2 * G,), 7.0, dtype=torch.float32, device="cuda")
    Q.qad_moe_fwd(s, inp["x"], inp["topk_idx"], inp["topk_w"], inp["w13"], inp["s13"], inp["w2"], inp["s2"],
                  big_out[G:G + T * d], ws)
    Q.qad_moe_bwd_dgrad(s, inp["dout"], inp["topk_w"], inp["w13"], inp["s13"], inp["w2"], inp["s2"],
                        big_dx[G:G + T * d], big_dp[G:G + T * k], ws)
    Q.qad_moe_bwd_scalegrad(s, inp["w13"], inp["s13"], inp["w2"], inp["s2"], big13[G:G + n13], big2[G:G + n2], 0, ws)
    torch.cuda.synchronize()
    for t, n in ((big_out, T * d), (big_dx, T * d), (big_dp, T * k), (big13, n13), (big2, n2)):
        assert torch.all(t[:G] == 7.0) and torch.all(t[G + n:] == 7.0)
        assert torch.all(torch.isfinite(t[G:G + n].float()))


# ------------------------------------------------------------------------------ the quotient

def _quotient_cases(n, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = torch.randn(n, generator=g, device="cuda") * torch.exp2(torch.randint(-40, 12, (n,), generator=g,
                                                                              device="cuda").float())
    w = w.to(torch.bfloat16).float()
    s = torch.rand(n, generator=g, device="cuda") * torch.exp2(torch.randint(-30, 4, (n,), generator=g,
                                                                            device="cuda").float())
    # hard cases: all-ones mantissas, powers of two, exact multiples, signed zeros, tiny/huge
    ones = torch.tensor([1.9999999, 1.0, 1.5, 1.9999998], device="cuda")
    m = 1 << 16
    s[:m] = ones[torch.arange(m, device="cuda") % 4] * torch.exp2(torch.randint(-20, 4, (m,), generator=g,
                                                                                device="cuda").float())
    w[m:2 * m] = s[m:2 * m] * torch.randint(-8, 8, (m,), generator=g, device="cuda").float()
    w[2 * m:2 * m + 8] = torch.tensor([0.0, -0.0, 3e38, -3e38, 1e-38, -1e-38, 6.0, -0.5], device="cuda")
    s[2 * m:2 * m + 8] = torch.tensor([0.25, 0.25, 1e-3, 1e-3, 0.5, 2e-38, 1.0, 0.0], device="cuda")
    s[2 * m + 8:2 * m + 12] = torch.tensor([1e-40, 3e-39, 0.0, 1e-45], device="cuda")   # subnormal / zero scales
    # the activation case: |w| <= amax, s = amax / Qmax
    k = 1 << 20
    amax = torch.rand(k, generator=g, device="cuda") * 10.0 + 1e-3
    w[3 * m:3 * m + k] = ((torch.rand(k, generator=g, device="cuda") * 2 - 1) * amax).to(torch.bfloat16).float()
    s[3 * m:3 * m + k] = amax.to(torch.bfloat16).float() / 6.0
    return w, s


@pytest.mark.parametrize("mode", [0, 1])
def test_reciprocal_quotient_matches_cuda_division(mode):
    """The quantizers' x = w / s (correctly rounded reciprocal + one FMA correction) equals
    CUDA's IEEE division bit for bit, on hard cases and 32M random pairs; the block-guarded
    form (mode 1) wherever 2^-11 <= |x| <= 2^100, and below that it still rounds to zero on
    every grid."""
    n = 1 << 25
    w, s = _quotient_cases(n, 11 + mode)
    fast = torch.empty_like(w)
    ieee = torch.empty_like(w)
    Q.qad_debug_quotient(w, s, fast, ieee, n, mode)
    torch.cuda.synchronize()
    same = fast.view(torch.int32) == ieee.view(torch.int32)
    if mode == 1:
        # contract of the block-guarded form: exact for 2^-11 <= |x| <= 2^100 (its callers
        # never produce larger quotients: activations have |x| <= amax / s ~ Qmax, and the
        # scale-gradient reduction re-runs a block whose sum is not finite with mode 0's form)
        small = ieee.abs() < 2.0 ** -11
        assert bool((fast[small].abs() < 2.0 ** -10).all())
        same = same | small | (ieee.abs() > 2.0 ** 100)
    assert bool(same.all()), "%d mismatches, e.g. w=%r s=%r" % (int((~same).sum()), w[~same][:3].tolist(),
                                                                s[~same][:3].tolist())
    nz = s != 0
    torch_div = w[nz] / s[nz]
    assert torch.equal(ieee[nz].view(torch.int32), torch_div.view(torch.int32))


# ------------------------------------------------------------------------------ teacher pass

@pytest.mark.parametrize("fmt", [Q.QAD_FMT_NVFP4, Q.QAD_FMT_FP8_ROW])
def test_teacher_pass_without_quantizers(fmt):
    """QAD_FLAG_NO_QUANT: the same layer with both quantizers off (the self-distillation
    teacher) against the oracle with quant=False, stage by stage."""
    inp = _tiny(fmt)
    host = host_inputs(inp)
    s = Q.shape(inp["T"], inp["d"], inp["F"], inp["E"], inp["topk"], fmt, Q.QAD_FLAG_NO_QUANT | Q.QAD_FLAG_STASH_H)
    ws = torch.empty(Q.qad_moe_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    T, d, k, F, E = inp["T"], inp["d"], inp["topk"], inp["F"], inp["E"]
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty_like(out)
    dprobs = torch.empty((T, k), dtype=torch.float32, device="cuda")
    Q.qad_moe_fwd(s, inp["x"], inp["topk_idx"], inp["topk_w"], inp["w13"], inp["s13"], inp["w2"], inp["s2"], out, ws)
    Q.qad_moe_bwd_dgrad(s, inp["dout"], inp["topk_w"], inp["w13"], inp["s13"], inp["w2"], inp["s2"], dx, dprobs, ws)
    assert Q.qad_check_device_error(ws) == 0
    with pytest.raises(Q.QADError):
        Q.qad_moe_bwd_scalegrad(s, inp["w13"], inp["s13"], inp["w2"], inp["s2"], torch.empty_like(inp["s13"]),
                                torch.empty_like(inp["s2"]), 0, ws)
    ref = OM.route(host["topk_idx"], E)
    off, row_of = ref["offsets"], ref["row_of"]
    token = Q.workspace_view(ws, s, "ROW_TOKEN", torch.int32).cpu().numpy()
    real = token[:int(Q.workspace_view(ws, s, "HEADER", torch.int32)[2])] >= 0
    rpad = real.size

    def rows(name, cols):
        return vals(Q.workspace_view(ws, s, name, torch.bfloat16)[:rpad * cols].view(rpad, cols))[real]

    w13, w2 = OQ.bf16_to_f64(host["w13"]), OQ.bf16_to_f64(host["w2"])
    a1 = rows("A1", d)
    assert np.array_equal(a1, OQ.bf16_to_f64(host["x"])[ref["row_token"]])      # no activation quant
    z1 = rows("Z1", 2 * F)
    assert_close(z1, OM.grouped_gemm_nt(a1, w13, off), "teacher Z1")
    h, hh = rows("H", F), rows("H_HAT", F)
    assert np.array_equal(h, hh)                                                   # H_hat = H
    y = rows("Y", d)
    assert_close(y, OM.grouped_gemm_nt(hh, w2, off), "teacher Y")
    p = host["topk_w"].astype(np.float64)
    assert_close(vals(out), OM.combine(y, p, row_of), "teacher out")
    fwd = OM.moe_forward(fmt, host["x"], host["topk_idx"], host["topk_w"], host["w13"], host["s13"], host["w2"],
                         host["s2"], quant=False)
    assert rel_l2(vals(out), fwd["out"]) <= E2E_REL_L2                             # end to end, no codes to move
    dz1 = rows("DZ1", 2 * F)
    da1 = rows("DA1", d)
    assert_close(da1, OM.grouped_gemm_nn(dz1, w13, off), "teacher dA1")
    assert_close(vals(dx), OM.combine(da1, np.ones((T, k)), row_of), "teacher dx")


# ------------------------------------------------------------------------------ failure path

def test_bounded_wait_reports_timeout_and_leaves_the_context_usable():
    """The GEMMs' bounded mbarrier wait, on a barrier nothing arrives on with a ~0.5 ms budget,
    gives up and raises QAD_DEV_TIMEOUT; the device keeps working afterwards."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q.qad_debug_wait_timeout(err, 1_000_000)
    torch.cuda.synchronize()
    assert int(err.item()) == Q.QAD_DEV_TIMEOUT
    # the context is intact: a normal call still runs and is still bit exact
    w, s = _special_weights(1, 8, 256, Q.QAD_FMT_NVFP4, seed=5)
    out = torch.empty_like(w)
    Q.qad_fakequant_fwd(Q.QAD_FMT_NVFP4, w, s, out, 1, 8, 256)
    torch.cuda.synchronize()
    want = OQ.f64_to_bf16_bits(OQ.fakequant_weight(Q.QAD_FMT_NVFP4, bits(w), synth.to_numpy(s)))
    assert np.array_equal(bits(out), want)


# ------------------------------------------------------------------------------ shapes that are not whole tiles

@pytest.mark.parametrize("fmt, d, F", [
    (Q.QAD_FMT_NVFP4, 272, 144), (Q.QAD_FMT_FP8_ROW, 272, 144), (Q.QAD_FMT_NVFP4A16, 272, 144),
    (Q.QAD_FMT_W8A8, 272, 144), (Q.QAD_FMT_NVFP4_E4M3, 272, 144),
    # the row quantizer of H with 16 lanes per row (F <= 768), 32 lanes and 3 blocks per lane
    # (F <= 1536), 32 lanes and 4 blocks (F <= 2048)
    (Q.QAD_FMT_NVFP4_E4M3, 256, 1040), (Q.QAD_FMT_FP8_ROW, 256, 1536), (Q.QAD_FMT_W8A8, 272, 2032),
    # INT4 weights need multiples of 128 (group-128 scales along d and F): 384 is not a whole 256 tile
    (Q.QAD_FMT_INT4_G128, 384, 384), (Q.QAD_FMT_W4AFP8, 384, 384)])
def test_layer_stagewise_partial_tiles(fmt, d, F):
    """d and F that are multiples of 16 but not of the GEMM tiles: the last N tiles of fc1
    (2 x 128 gate/up rows), fc2, both input-gradient GEMMs and the scale-gradient GEMMs are
    partial, the last K blocks are partial (zero-filled by the tensor maps), the scale-gradient
    tiles past the weight's rows or columns take the masked path, and nvfp4 scale rows are not
    16-byte aligned (F / 16 = 9).  Every stage against the oracle, as for whole tiles."""
    inp = synth.make_inputs(synth.workload("tiny_nvfp4", fmt=fmt, E=5, d=d, F=F, topk=3, T=301), seed=12,
                            device="cuda")
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    assert run.error == 0
    _stagewise(run, host_inputs(inp))


@pytest.mark.parametrize("fmt", [Q.QAD_FMT_NVFP4, Q.QAD_FMT_FP8_ROW, Q.QAD_FMT_NVFP4_E4M3])
def test_layer_stagewise_gpt_oss_like_width(fmt):
    """A layer as wide as GPT-OSS's experts (d = F = 2880: 11.25 tiles of 256 columns).  With the
    per-row activation grids (fp8, deployed nvfp4) the H rows (2880 > 2048 columns) take the
    row quantizer's two-pass form instead of the register-held one."""
    E, T = (16, 1024) if fmt == Q.QAD_FMT_NVFP4 else (8, 384)  # the oracle's GEMMs dominate the test's time
    inp = synth.make_inputs(synth.workload("tiny_nvfp4", fmt=fmt, E=E, d=2880, F=2880, topk=4, T=T), seed=13,
                            device="cuda")
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    assert run.error == 0
    _stagewise(run, host_inputs(inp))


# ------------------------------------------------------------------------------ a seeded sweep of small shapes

def _sweep_cases(n=16, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        fmt = int(rng.choice(FMTS))
        mult = 128 if fmt in (Q.QAD_FMT_INT4_G128, Q.QAD_FMT_W4AFP8) else 16
        d = int(mult * rng.integers(1, 1024 // mult + 1))
        F = int(mult * rng.integers(1, 640 // mult + 1))
        E = int(rng.integers(1, 12))
        k = int(rng.integers(1, min(E, 6) + 1))
        T = int(rng.integers(1, 400))
        flags = int(rng.choice([0, Q.QAD_FLAG_RECOMPUTE]))
        cases.append((i, fmt, d, F, E, k, T, flags))
    return cases


@pytest.mark.parametrize("case", _sweep_cases(), ids=lambda c: "case%d" % c[0])
def test_layer_stagewise_random_shapes(case):
    """Random small layers (seeded): any format, d and F any multiple of 16 (128 for INT4 weights)
    up to 1024 / 640, 1-11 experts, top-1..6, 1-399 tokens, with and without recompute -- every
    stage against the oracle."""
    _, fmt, d, F, E, k, T, flags = case
    inp = synth.make_inputs(synth.workload("tiny_nvfp4", fmt=fmt, E=E, d=d, F=F, topk=k, T=T), seed=case[0],
                            device="cuda")
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    assert run.error == 0
    _stagewise(run, host_inputs(inp))
    if flags & Q.QAD_FLAG_RECOMPUTE:  # recompute reuses Y's region for Z1: compare with the stashing run
        b = Run(inp, flags=Q.QAD_FLAG_RECOMPUTE)
        assert b.error == 0
        assert torch.equal(run.out.view(torch.int16), b.out.view(torch.int16))
        assert torch.equal(run.dx.view(torch.int16), b.dx.view(torch.int16))
        assert torch.equal(run.ds13, b.ds13) and torch.equal(run.ds2, b.ds2)
