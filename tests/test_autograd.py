"""The torch.autograd view of the layer (scale_only_quantization_gb300.autograd).

Its gradients must be exactly the C-ABI calls' results: dx for x, dprobs for the routing
weights, ds13 / ds2 for the scales, nothing for the frozen weights and the indices.
"""
import pytest
import torch

import scale_only_quantization_gb300 as Q
from scale_only_quantization_gb300.autograd import QADMoE
import synth


def test_module_holds_frozen_weights_and_learnable_scales():
    inp = synth.make_inputs(synth.workload("tiny_nvfp4"), seed=0, device="cpu")
    m = QADMoE(inp["w13"], inp["s13"], inp["w2"], inp["s2"], Q.QAD_FMT_NVFP4)
    assert sorted(n for n, _ in m.named_parameters()) == ["s13", "s2"]
    assert sorted(n for n, _ in m.named_buffers()) == ["w13", "w2"]


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", [Q.QAD_FMT_NVFP4, Q.QAD_FMT_FP8_ROW, Q.QAD_FMT_NVFP4_E4M3])
def test_autograd_gradients_equal_the_abi_calls(fmt):
    from gpu_util import Run
    from scale_only_quantization_gb300 import build
    build.build()
    inp = synth.make_inputs(synth.workload("tiny_nvfp4", fmt=fmt), seed=3, device="cuda")
    ref = Run(inp)
    m = QADMoE(inp["w13"], inp["s13"], inp["w2"], inp["s2"], fmt)
    x = inp["x"].clone().requires_grad_(True)
    p = inp["topk_w"].clone().requires_grad_(True)
    out = m(x, inp["topk_idx"], p)
    out.backward(inp["dout"])
    torch.cuda.synchronize()
    assert torch.equal(out.detach().view(torch.int16), ref.out.view(torch.int16))
    assert torch.equal(x.grad.view(torch.int16), ref.dx.view(torch.int16))
    assert torch.equal(p.grad, ref.dprobs)
    assert torch.equal(m.s13.grad, ref.ds13) and torch.equal(m.s2.grad, ref.ds2)
    assert m.w13.grad is None and m.w2.grad is None
