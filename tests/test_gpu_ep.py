"""The expert-parallel pieces on one GPU: the combine step the C ABI exposes for the exchange
(qad_moe_combine) against the oracle, and the expert-parallel layer with the CUDA backend on one
rank (the exchange is then the identity) against the layer's own calls, bit for bit: the owner
sees the same rows per expert in the same order."""
import numpy as np
import pytest
import torch

import scale_only_quantization_gb300 as Q
from scale_only_quantization_gb300 import ep as EP
from oracle import moe as OM
import synth

from gpu_util import Run, assert_close, vals

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from scale_only_quantization_gb300 import build
    build.build()
    Q.lib()


@pytest.mark.parametrize("T, k, d", [(300, 8, 2048), (77, 3, 784), (5, 1, 16)])
def test_combine_against_the_oracle(T, k, d):
    g = torch.Generator(device="cuda").manual_seed(T + k)
    n_rows = T * k + 13
    rows = (torch.randn((n_rows, d), generator=g, device="cuda")).to(torch.bfloat16)
    perm = torch.randperm(n_rows, generator=g, device="cuda")[: T * k].to(torch.int32).view(T, k)
    row_of = torch.where(torch.rand((T, k), generator=g, device="cuda") < 0.1, -1, perm).to(torch.int32).contiguous()
    p = torch.softmax(torch.randn((T, k), generator=g, device="cuda"), 1).contiguous()
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty_like(out)
    Q.qad_moe_combine(rows, row_of, p, out, T, k, d)
    Q.qad_moe_combine(rows, row_of, None, dx, T, k, d)
    torch.cuda.synchronize()
    ro = synth.to_numpy(row_of).astype(np.int64)
    r64 = vals(rows)
    assert_close(vals(out), OM.combine(r64, synth.to_numpy(p).astype(np.float64), ro), "combine")
    assert_close(vals(dx), OM.combine(r64, np.ones((T, k)), ro), "combine (weight 1)")


@pytest.mark.parametrize("fmt, name", [(Q.QAD_FMT_NVFP4, "tiny_nvfp4"), (Q.QAD_FMT_FP8_ROW, "tiny_nvfp4"),
                                       (Q.QAD_FMT_NVFP4_E4M3, "tiny_nvfp4"),
                                       (Q.QAD_FMT_NVFP4, "qwen3_30b_a3b_nvfp4")])
def test_single_rank_expert_parallel_layer_equals_the_layer(fmt, name):
    inp = synth.make_inputs(synth.workload(name, fmt=fmt), seed=3, device="cuda")
    inp["topk_idx"][7, 1] = inp["E"] + 2            # dropped pairs travel nowhere
    inp["topk_idx"][9, 1] = inp["topk_idx"][9, 0]
    ref = Run(inp)
    layer = EP.ExpertParallelMoE(EP.CudaExperts(inp["w13"], inp["s13"], inp["w2"], inp["s2"], fmt), inp["E"])
    out = layer.forward(inp["x"], inp["topk_idx"], inp["topk_w"])
    dx, dprobs = layer.backward(inp["dout"])
    ds13, ds2 = layer.scale_grads()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.out.view(torch.int16))
    assert torch.equal(dx.view(torch.int16), ref.dx.view(torch.int16))
    assert torch.equal(dprobs, ref.dprobs)
    assert torch.equal(ds13, ref.ds13) and torch.equal(ds2, ref.ds2)


def test_cuda_experts_with_no_received_rows():
    """An owner that receives no pairs (every token routed elsewhere) runs the layer calls on zero
    rows: empty outputs, and scale gradients of exactly zero for its experts."""
    inp = synth.make_inputs(synth.workload("tiny_nvfp4"), seed=5, device="cuda")
    be = EP.CudaExperts(inp["w13"], inp["s13"], inp["w2"], inp["s2"], inp["fmt"])
    d = inp["d"]
    y = be.forward(torch.empty((0, d), dtype=torch.bfloat16, device="cuda"),
                   torch.empty((0,), dtype=torch.int32, device="cuda"))
    da, dp = be.dgrad(torch.empty((0, d), dtype=torch.bfloat16, device="cuda"),
                      torch.empty((0,), dtype=torch.float32, device="cuda"))
    ds13, ds2 = be.scalegrad()
    torch.cuda.synchronize()
    assert y.shape == (0, d) and da.shape == (0, d) and dp.shape == (0,)
    assert torch.count_nonzero(ds13) == 0 and torch.count_nonzero(ds2) == 0
