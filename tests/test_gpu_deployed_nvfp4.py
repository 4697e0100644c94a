"""nvfp4 with deployed block scales (QAD_FMT_NVFP4_E4M3) on the GPU, against the oracle.

The compressed-tensors NVFP4 layout (AngelSlim mcore_qad walkthrough, section 三: the QAD
format names map to the deployment side's layout) stores each 16-element block scale as an
E4M3 number times one fp32 scale of the tensor.  Checked here: the deployed weight scales
bit for bit (zero matrices, negative scales, scales in E4M3's subnormal range and below it),
the layer stage by stage on activations whose blocks span the E4M3 range (blocks far below
their row's largest come out as zeros), and the deployed-scale regions of the workspace.
"""
import numpy as np
import pytest
import torch

import scale_only_quantization_gb300 as Q
from oracle import quant as OQ
import synth

from gpu_util import Run, host_inputs
from test_gpu_parity import _stagewise

pytestmark = pytest.mark.gpu

FMT = Q.QAD_FMT_NVFP4_E4M3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from scale_only_quantization_gb300 import build
    build.build()
    Q.lib()


def _scales(n_mat, per, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    s = torch.exp(torch.randn((n_mat, per), generator=g, device="cuda") * 1.5 - 5.0)
    if n_mat > 1:
        s[1] = 0.0                                      # an all-zero matrix
    s[0, : min(per, 8)] *= -1.0                         # negative scales keep their sign
    s[0, min(per, 8): min(per, 16)] = 0.0               # zero blocks
    s[-1, :: 5] *= 2.0 ** -12                           # E4M3 subnormal range and below
    s[-1, 1] = s[-1].abs().max() * 7.0                  # the matrix maximum, far above the rest
    return s.float().contiguous()


@pytest.mark.parametrize("n_mat, per", [(3, 4), (5, 1000), (2, 1536 * 128), (128, 2048 * 48 // 16)])
def test_deploy_scales_bit_exact(n_mat, per):
    s = _scales(n_mat, per, seed=per)
    sq = torch.full_like(s, float("nan"))
    Q.qad_nvfp4_deploy_scales(s, sq, n_mat, per)
    torch.cuda.synchronize()
    want = OQ.deploy_scales(synth.to_numpy(s).astype(np.float64), axes=-1)
    got = synth.to_numpy(sq).astype(np.float64)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))
    # in place gives the same bits
    s2 = s.clone()
    Q.qad_nvfp4_deploy_scales(s2, s2, n_mat, per)
    torch.cuda.synchronize()
    assert torch.equal(s2.view(torch.int32), sq.view(torch.int32))


def _structured(seed, **over):
    """tiny_nvfp4 shapes in format 6, with activation blocks spread over the E4M3 range: per token,
    a few blocks scaled by 2^-6 (subnormal block scales), 2^-9 (near E4M3's smallest) and 2^-12
    (below it: flushed to zero), and one tie of the E4M3 rounding."""
    inp = synth.make_inputs(synth.workload("tiny_nvfp4", fmt=FMT, **over), seed=seed, device="cuda")
    x = inp["x"].float()
    T, d = x.shape
    nb = d // 16
    rng = np.random.default_rng(seed)
    xb = x.view(T, nb, 16)
    for t in range(T):
        b = rng.choice(nb, 4, replace=False)
        xb[t, b[0]] *= 2.0 ** -6
        xb[t, b[1]] *= 2.0 ** -9
        xb[t, b[2]] *= 2.0 ** -12
    # token 0: the row maximum fixes g = 2^-10 (block amax 6 * 448 * 2^-10) and block 1's scale
    # sits on the E4M3 tie 13.5 -> 14 (amax 6 * 13.5 * 2^-10)
    xb[0].mul_(0.0)
    xb[0, 0, 0] = 6 * 448 * 2.0 ** -10
    xb[0, 1, 3] = -6 * 13.5 * 2.0 ** -10
    xb[0, 2, :] = 0.01
    inp["x"] = x.to(torch.bfloat16).contiguous()
    return inp


def test_layer_stagewise_with_deployed_scales():
    inp = _structured(seed=3)
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    assert run.error == 0
    host = host_inputs(inp)
    _stagewise(run, host)
    E, d, F = inp["E"], inp["d"], inp["F"]
    s13q = synth.to_numpy(run.view("S13_DEPLOYED", torch.float32)).astype(np.float64).reshape(E, 2 * F, d // 16)
    s2q = synth.to_numpy(run.view("S2_DEPLOYED", torch.float32)).astype(np.float64).reshape(E, d, F // 16)
    assert np.array_equal(s13q, OQ.effective_weight_scales(FMT, host["s13"]))
    assert np.array_equal(s2q, OQ.effective_weight_scales(FMT, host["s2"]))
    # the structured token: the tie block's scale is 14 * 2^-10, its largest element comes back as
    # 6 * 14 * 2^-10 (E2M1 rounds 6 * 13.5 / 14 to 6), and the 2^-12 blocks are zeros
    xq = run.view("XQ", torch.bfloat16).view(inp["T"], d).float().cpu().numpy()
    assert xq[0, 16 + 3] == -6 * 14 * 2.0 ** -10
    assert xq[0, 0] == 6 * 448 * 2.0 ** -10


def test_deployed_layer_uneven_shapes_and_dequant_in_gemm():
    inp = _structured(seed=4, E=6, d=768, F=384, topk=3, T=333)
    a = Run(inp, flags=0)
    assert a.error == 0
    _stagewise(a, host_inputs(inp), check_h=False)
    b = Run(inp, flags=Q.QAD_FLAG_SMEM_DEQUANT)
    assert b.error == 0
    for x, y in ((a.out, b.out), (a.dx, b.dx)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert torch.equal(a.ds13, b.ds13) and torch.equal(a.ds2, b.ds2)


def test_deployed_recompute_is_bit_identical():
    inp = _structured(seed=5)
    a = Run(inp, flags=0)
    b = Run(inp, flags=Q.QAD_FLAG_RECOMPUTE)
    for x, y in ((a.out, b.out), (a.dx, b.dx)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert torch.equal(a.ds13, b.ds13) and torch.equal(a.ds2, b.ds2)


def test_deployed_layer_with_a_zero_matrix_and_negative_scales():
    """An expert whose w13 scales are all zero (its tensor scale is 0, so every deployed scale is 0
    and its fake-quantized gate/up weights are signed zeros) and a few negative w2 scales (rounded
    as their magnitude, sign kept): the layer stage by stage against the oracle, and the deployed
    scale views."""
    inp = _structured(seed=6)
    inp["s13"][1].zero_()
    inp["s2"][2, :5, :3] *= -1.0
    run = Run(inp, flags=Q.QAD_FLAG_STASH_H)
    assert run.error == 0
    host = host_inputs(inp)
    _stagewise(run, host)
    E, d, F = inp["E"], inp["d"], inp["F"]
    s13q = synth.to_numpy(run.view("S13_DEPLOYED", torch.float32)).astype(np.float64).reshape(E, 2 * F, d // 16)
    s2q = synth.to_numpy(run.view("S2_DEPLOYED", torch.float32)).astype(np.float64).reshape(E, d, F // 16)
    assert np.all(s13q[1] == 0)
    assert np.array_equal(s13q, OQ.effective_weight_scales(FMT, host["s13"]))
    assert np.array_equal(s2q, OQ.effective_weight_scales(FMT, host["s2"]))
    assert np.all(s2q[2, :5, :3] < 0)
