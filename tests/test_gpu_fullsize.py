"""GPU parity at the full workload sizes, in the launch configuration the benchmark times.

The oracle cannot run a whole Qwen3-30B-A3B-shaped layer in seconds, so these tests
check, against the oracle: the complete routing maps (bit exact); the fake-quantized
weights of sampled experts (bit exact); every stage of sampled routed rows of sampled
experts (teacher forced, as in test_gpu_parity); out / dx / dprobs / dY / A1 of sampled
tokens; and the full scale gradients of sampled experts.
"""
import numpy as np
import pytest
import torch

import scale_only_quantization_gb300 as Q
from oracle import moe as OM
from oracle import quant as OQ
import synth

from gpu_util import Run, assert_close, assert_scale_grad, bits, host_inputs, unpadded_row_of, vals

pytestmark = pytest.mark.gpu

WORKLOADS = ["qwen3_30b_a3b_nvfp4", "qwen3_30b_a3b_w4a16", "qwen3_30b_a3b_fp8", "large_nvfp4",
             # the remaining formats of the support matrix on the same Qwen3-30B-A3B shapes
             "qwen3_30b_a3b_nvfp4:3", "qwen3_30b_a3b_nvfp4:4", "qwen3_30b_a3b_nvfp4:5",
             # nvfp4 with deployed (E4M3-rounded) block scales
             "qwen3_30b_a3b_nvfp4:6",
             # fp8 with the forward GEMMs on the fp8 tensor path (scales applied to the sums)
             "qwen3_30b_a3b_fp8+native"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from scale_only_quantization_gb300 import build
    build.build()
    Q.lib()


def _rows(run, name, cols, idx):
    t = run.view(name, torch.bfloat16)
    n = t.numel() // cols
    sel = t.view(n, cols)[torch.as_tensor(idx, dtype=torch.long, device=t.device)]
    return vals(sel)


def _expert_w(run, name, e, n, k):
    return OQ.bf16_to_f64(bits(run.view(name, torch.bfloat16).view(-1, n, k)[e]))


@pytest.mark.parametrize("name", WORKLOADS)
def test_full_size_sampled(name):
    name, _, native = name.partition("+")
    base, _, fmt_override = name.partition(":")
    cfg = synth.workload(base, **({"fmt": int(fmt_override)} if fmt_override else {}))
    inp = synth.make_inputs(cfg, seed=0, device="cuda")
    fmt, T, d, F, E, k = inp["fmt"], inp["T"], inp["d"], inp["F"], inp["E"], inp["topk"]
    factored = native == "native"
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H | (Q.QAD_FLAG_NATIVE_FP8 if factored else 0))
    assert run.error == 0
    rng = np.random.default_rng(0)

    # routing maps, complete
    idx = synth.to_numpy(inp["topk_idx"])
    ref = OM.route(idx, E)
    rt = run.routing()
    real = rt["real"]
    assert np.array_equal(rt["row_token"][real], ref["row_token"])
    assert np.array_equal(rt["row_slot"][real], ref["row_slot"])
    assert np.array_equal(unpadded_row_of(rt), ref["row_of"])
    assert np.array_equal(rt["counts"], ref["counts"])
    offs = rt["offs"]

    # two sampled experts (one of them the most loaded), full weights and scale gradients
    experts = sorted({int(np.argmax(ref["counts"])), int(rng.integers(E))})
    p = synth.to_numpy(inp["topk_w"]).astype(np.float64)
    for e in experts:
        w13_e = bits(inp["w13"][e])
        w2_e = bits(inp["w2"][e])
        s13_e = synth.to_numpy(inp["s13"][e])
        s2_e = synth.to_numpy(inp["s2"][e])
        w13h = _expert_w(run, "W13_HAT", e, 2 * F, d)
        w2h = _expert_w(run, "W2_HAT", e, d, F)
        assert np.array_equal(OQ.f64_to_bf16_bits(w13h), OQ.f64_to_bf16_bits(OQ.fakequant_weight(fmt, w13_e, s13_e)))
        assert np.array_equal(OQ.f64_to_bf16_bits(w2h), OQ.f64_to_bf16_bits(OQ.fakequant_weight(fmt, w2_e, s2_e)))
        n_e = int(rt["counts"][e])
        rows_e = np.arange(offs[e], offs[e] + n_e)
        a1 = _rows(run, "A1", d, rows_e)
        dz1 = _rows(run, "DZ1", 2 * F, rows_e)
        hh = _rows(run, "H_HAT", F, rows_e)
        dy = _rows(run, "DY", d, rows_e)
        ds13 = OQ.scale_grad_from_wgrad(fmt, dz1.T @ a1, w13_e, s13_e)
        ds2 = OQ.scale_grad_from_wgrad(fmt, dy.T @ hh, w2_e, s2_e)
        assert_scale_grad(synth.to_numpy(run.ds13[e]), ds13.reshape(s13_e.shape), "ds13[%d]" % e)
        assert_scale_grad(synth.to_numpy(run.ds2[e]), ds2.reshape(s2_e.shape), "ds2[%d]" % e)

        # every stage of 48 sampled rows of this expert, teacher forced
        pick = rows_e[rng.choice(n_e, size=min(48, n_e), replace=False)] if n_e else rows_e
        if pick.size == 0:
            continue
        toks, slots = rt["row_token"][pick], rt["row_slot"][pick]
        x = OQ.bf16_to_f64(bits(inp["x"][torch.as_tensor(toks, device="cuda")]))
        dout = OQ.bf16_to_f64(bits(inp["dout"][torch.as_tensor(toks, device="cuda")]))
        a1 = _rows(run, "A1", d, pick)
        assert np.array_equal(OQ.f64_to_bf16_bits(a1), OQ.f64_to_bf16_bits(OQ.fakequant_act(fmt, x)))
        z1 = _rows(run, "Z1", 2 * F, pick)
        if factored:
            want_z1 = OQ.fakequant_act_factored(fmt, x) @ OQ.fakequant_weight_factored(fmt, w13_e, s13_e).T
        else:
            want_z1 = a1 @ w13h.T
        assert_close(z1, want_z1, "Z1 rows e%d" % e)
        h = _rows(run, "H", F, pick)
        assert_close(h, OM.swiglu(z1), "H rows e%d" % e)
        hh = _rows(run, "H_HAT", F, pick)
        assert np.array_equal(OQ.f64_to_bf16_bits(hh), OQ.f64_to_bf16_bits(OQ.fakequant_act(fmt, h)))
        y = _rows(run, "Y", d, pick)
        if factored:
            want_y = OQ.fakequant_act_factored(fmt, h) @ OQ.fakequant_weight_factored(fmt, w2_e, s2_e).T
        else:
            want_y = hh @ w2h.T
        assert_close(y, want_y, "Y rows e%d" % e)
        dy = _rows(run, "DY", d, pick)
        want_dy = OQ.round_bf16(OQ.round_f32(dout * p[toks, slots][:, None]))
        assert np.array_equal(OQ.f64_to_bf16_bits(dy), OQ.f64_to_bf16_bits(want_dy))
        dz1 = _rows(run, "DZ1", 2 * F, pick)
        assert_close(dz1, OM.swiglu_bwd(dy @ w2h, z1), "dZ1 rows e%d" % e)
        da1 = _rows(run, "DA1", d, pick)
        assert_close(da1, dz1 @ w13h, "dA1 rows e%d" % e)

    # 64 sampled tokens: combine, input gradient and routing-weight gradient
    toks = rng.choice(T, size=64, replace=False)
    ro = rt["row_of"][toks]
    ys = _rows(run, "Y", d, np.maximum(ro, 0).reshape(-1)).reshape(64, k, d)
    das = _rows(run, "DA1", d, np.maximum(ro, 0).reshape(-1)).reshape(64, k, d)
    dout = OQ.bf16_to_f64(bits(inp["dout"][torch.as_tensor(toks, device="cuda")]))
    out_ref = np.einsum("tj,tjd->td", p[toks], ys)
    dx_ref = das.sum(axis=1)
    dp_ref = np.einsum("td,tjd->tj", dout, ys)
    sel = torch.as_tensor(toks, device="cuda")
    assert_close(vals(run.out[sel]), out_ref, "out (sampled tokens)")
    assert_close(vals(run.dx[sel]), dx_ref, "dx (sampled tokens)")
    assert_close(synth.to_numpy(run.dprobs[sel]).astype(np.float64), dp_ref, "dprobs (sampled tokens)")
    # padding rows stay zero in the operands the scale-gradient GEMMs contract over
    pad = np.nonzero(~real)[0][:256]
    if pad.size:
        for nm, cols in (("A1", d), ("DY", d), ("H_HAT", F), ("DZ1", 2 * F)):
            assert np.all(_rows(run, nm, cols, pad) == 0), nm


def test_recompute_matches_stash_at_full_size():
    """qwen3_30b_a3b_nvfp4 with QAD_FLAG_RECOMPUTE: outputs and scale gradients equal the
    stashing run's bit for bit, in a workspace smaller by the Z1 region."""
    inp = synth.make_inputs(synth.workload("qwen3_30b_a3b_nvfp4"), seed=11, device="cuda")
    a = Run(inp, flags=0)
    out, dx, dprobs, ds13, ds2 = a.out.clone(), a.dx.clone(), a.dprobs.clone(), a.ds13.clone(), a.ds2.clone()
    nb_a = a.ws.numel()
    del a
    torch.cuda.empty_cache()
    b = Run(inp, flags=Q.QAD_FLAG_RECOMPUTE)
    assert b.error == 0
    assert b.ws.numel() < nb_a
    assert torch.equal(out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(dx.view(torch.int16), b.dx.view(torch.int16))
    assert torch.equal(dprobs, b.dprobs)
    assert torch.equal(ds13, b.ds13) and torch.equal(ds2, b.ds2)
