"""The layer as a torch.autograd.Function and an nn.Module, over the C ABI.

Scale-only QAD ("MCoreQAD Backend", opening section; AngelSlim mcore_qad walkthrough,
nxmr.cn/news/131691, sections 二.3-二.4): the routed-expert weights are frozen, the forward
sees their fake-quantized copies, and the quantizer scales are the only trainable
parameters.  So the backward returns no gradient for the weights or the routing indices,
dx for the hidden states, dprobs for the routing weights (their gradient reaches the router)
and ds13 / ds2 for the scales.

Marshalling only: the forward is qad_moe_fwd, the backward qad_moe_bwd_dgrad followed by
qad_moe_bwd_scalegrad, all on torch's current stream.  The workspace, which carries the
stashed stages from the forward to the backward, lives in the autograd context.
"""
import torch

from . import (qad_moe_bwd_dgrad, qad_moe_bwd_scalegrad, qad_moe_fwd, qad_moe_workspace_bytes, shape)


class QADMoEFunction(torch.autograd.Function):
    """out = MoE(x; topk_idx, topk_w, W13_hat(s13), W2_hat(s2)).

    x [T, d] bf16; topk_idx [T, k] int32; topk_w [T, k] fp32; w13 [E, 2F, d] bf16 (gate rows,
    then up rows); s13 fp32 [E, 2F, d / B]; w2 [E, d, F] bf16; s2 fp32 [E, d, F / B]; fmt a
    qad_fmt; flags QAD_FLAG_* bits.  All tensors contiguous on the current CUDA device.
    """

    @staticmethod
    def forward(ctx, x, topk_idx, topk_w, w13, s13, w2, s2, fmt, flags):
        T, d = x.shape
        E, two_f, _ = w13.shape
        k = topk_idx.shape[1]
        s = shape(T, d, two_f // 2, E, k, fmt, flags)
        ws = torch.empty(qad_moe_workspace_bytes(s), dtype=torch.uint8, device=x.device)
        out = torch.empty_like(x)
        qad_moe_fwd(s, x, topk_idx, topk_w, w13, s13, w2, s2, out, ws)
        ctx.save_for_backward(topk_w, w13, s13, w2, s2)
        ctx.layer_shape = s
        ctx.ws = ws
        ctx.mark_non_differentiable(topk_idx)
        return out

    @staticmethod
    def backward(ctx, dout):
        topk_w, w13, s13, w2, s2 = ctx.saved_tensors
        s, ws = ctx.layer_shape, ctx.ws
        dout = dout.contiguous()
        dx = torch.empty_like(dout)
        dprobs = torch.empty_like(topk_w) if ctx.needs_input_grad[2] else None
        qad_moe_bwd_dgrad(s, dout, topk_w, w13, s13, w2, s2, dx, dprobs, ws)
        ds13 = ds2 = None
        if ctx.needs_input_grad[4] or ctx.needs_input_grad[6]:
            ds13 = torch.empty_like(s13)
            ds2 = torch.empty_like(s2)
            qad_moe_bwd_scalegrad(s, w13, s13, w2, s2, ds13, ds2, 0, ws)
        ctx.ws = None
        return (dx if ctx.needs_input_grad[0] else None, None, dprobs, None, ds13, None, ds2, None, None)


class QADMoE(torch.nn.Module):
    """The routed experts of one MoE layer: frozen bf16 weights (buffers) and learnable fp32
    scales (parameters), initialised by the caller."""

    def __init__(self, w13, s13, w2, s2, fmt, flags=0):
        super().__init__()
        self.register_buffer("w13", w13.contiguous())
        self.register_buffer("w2", w2.contiguous())
        self.s13 = torch.nn.Parameter(s13.contiguous())
        self.s2 = torch.nn.Parameter(s2.contiguous())
        self.fmt = int(fmt)
        self.flags = int(flags)

    def forward(self, x, topk_idx, topk_w):
        return QADMoEFunction.apply(x.contiguous(), topk_idx.contiguous(), topk_w.contiguous(), self.w13, self.s13,
                                    self.w2, self.s2, self.fmt, self.flags)
