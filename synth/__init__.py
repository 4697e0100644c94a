"""Seeded synthetic inputs for one MoE layer (shared by the tests, the bench and smoke()).

This module draws random numbers and nothing else: it holds none of the quantizer,
GEMM or gradient arithmetic of the method.  The initial weight scales are drawn
here because they are an input of the layer (the learnable parameters' starting
value), following the initialisation rule "block amax / Qmax x (1 + U(-0.1, 0.1))".

Workloads, named by what they are:

  tiny_nvfp4            E=4,   d=256,  F=128,  top-2, 512 tokens, nvfp4 W4A4
  qwen3_30b_a3b_nvfp4   E=128, d=2048, F=768,  top-8, 16384 tokens (8 x 2048), nvfp4
  qwen3_30b_a3b_w4a16   same shapes, INT4 group-128 weights, bf16 activations
  qwen3_30b_a3b_fp8     same shapes, fp8 W8A8 per-row, Zipf(1.2) expert popularity
  large_nvfp4           E=256, d=4096, F=1536, top-8, 32768 tokens, nvfp4, 0.1% outliers
  qwen3_30b_a3b_nvfp4_deployed  the nvfp4 shapes with deployed (E4M3-rounded) block scales

Any workload can be run in another format with workload(name, fmt=...): 3 nvfp4a16,
4 w8a8, 5 w4afp8, 6 nvfp4 with deployed (E4M3-rounded) block scales.

The MoE-layer shapes follow the Qwen3-MoE model family that the pages support
("MCoreQAD Backend", Support Matrix) and its example run (seq_len 2048, micro-batch
8); the hidden states are N(0, 1) stand-ins for the pages' random-token inputs.
"""
import math

import torch

FMT_NVFP4, FMT_INT4_G128, FMT_FP8_ROW, FMT_NVFP4A16, FMT_W8A8, FMT_W4AFP8, FMT_NVFP4_E4M3 = 0, 1, 2, 3, 4, 5, 6

WORKLOADS = {
    "tiny_nvfp4": dict(E=4, d=256, F=128, topk=2, T=512, fmt=FMT_NVFP4, routing="uniform", outliers=0.0),
    "qwen3_30b_a3b_nvfp4": dict(E=128, d=2048, F=768, topk=8, T=16384, fmt=FMT_NVFP4, routing="uniform",
                                outliers=0.0),
    "qwen3_30b_a3b_w4a16": dict(E=128, d=2048, F=768, topk=8, T=16384, fmt=FMT_INT4_G128, routing="uniform",
                                outliers=0.0),
    "qwen3_30b_a3b_fp8": dict(E=128, d=2048, F=768, topk=8, T=16384, fmt=FMT_FP8_ROW, routing="zipf",
                              outliers=0.0),
    "large_nvfp4": dict(E=256, d=4096, F=1536, topk=8, T=32768, fmt=FMT_NVFP4, routing="uniform",
                        outliers=0.001),
    "qwen3_30b_a3b_nvfp4_deployed": dict(E=128, d=2048, F=768, topk=8, T=16384, fmt=FMT_NVFP4_E4M3,
                                         routing="uniform", outliers=0.0),
}

# elements per weight scale along K (absent: one per row), and the divisor that turns a
# block amax into a scale
_BLOCK = {FMT_NVFP4: 16, FMT_INT4_G128: 128, FMT_NVFP4A16: 16, FMT_W4AFP8: 128, FMT_NVFP4_E4M3: 16}
_QMAX = {FMT_NVFP4: 6.0, FMT_INT4_G128: 7.0, FMT_FP8_ROW: 448.0, FMT_NVFP4A16: 6.0, FMT_W8A8: 127.0,
         FMT_W4AFP8: 7.0, FMT_NVFP4_E4M3: 6.0}


def workload(name, **override):
    cfg = dict(WORKLOADS[name])
    cfg.update(override)
    cfg["name"] = name
    return cfg


def scale_block(fmt, K):
    return _BLOCK.get(fmt, K)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def init_scales(w, fmt, g):
    """fp32 scales [E, N, K / B]: block amax of |W| / Qmax, times (1 + U(-0.1, 0.1))."""
    E, N, K = w.shape
    B = scale_block(fmt, K)
    amax = w.float().abs().reshape(E, N, K // B, B).amax(dim=-1)
    jitter = 1.0 + (torch.rand(amax.shape, generator=g, device=w.device) * 0.2 - 0.1)
    return (amax / _QMAX[fmt] * jitter).float().contiguous()


def _weights(shape, outliers, g, device):
    w = torch.randn(shape, generator=g, device=device) * 0.02
    if outliers > 0:
        n = w.numel()
        m = max(1, int(round(outliers * n)))
        pos = torch.randint(0, n, (m,), generator=g, device=device)
        sign = torch.randint(0, 2, (m,), generator=g, device=device).float() * 2 - 1
        w.view(-1)[pos] = 0.5 * sign
    return w.to(torch.bfloat16).contiguous()


def _routing(T, E, k, kind, g, device):
    if kind == "uniform":
        keys = torch.rand((T, E), generator=g, device=device)
    else:  # Zipf(1.2) popularity over a random order of experts; Gumbel-top-k = sampling w/o replacement
        rank = torch.randperm(E, generator=g, device=device).float() + 1.0
        logp = -1.2 * torch.log(rank)
        u = torch.rand((T, E), generator=g, device=device).clamp_min(1e-20)
        keys = logp[None, :] - torch.log(-torch.log(u))
    idx = torch.topk(keys, k, dim=1).indices.to(torch.int32).contiguous()
    logits = torch.randn((T, k), generator=g, device=device)
    p = torch.softmax(logits, dim=1).float().contiguous()
    return idx, p


def make_inputs(cfg, seed=0, device="cpu", with_weights=True):
    """All inputs of one fwd + bwd step of the layer, as torch tensors on `device`.

    x, dout: bf16 [T, d] ~ N(0, 1);  topk_idx int32 [T, k] (k distinct experts per token);
    topk_w fp32 [T, k] (softmax of N(0, 1));  w13 bf16 [E, 2F, d], w2 bf16 [E, d, F]
    ~ N(0, 0.02);  s13 fp32 [E, 2F, d/B], s2 fp32 [E, d, F/B].
    """
    E, d, F, k, T = cfg["E"], cfg["d"], cfg["F"], cfg["topk"], cfg["T"]
    fmt = cfg["fmt"]
    g = _gen(seed, device)
    out = dict(fmt=fmt, E=E, d=d, F=F, topk=k, T=T)
    if with_weights:
        out["w13"] = _weights((E, 2 * F, d), cfg.get("outliers", 0.0), g, device)
        out["w2"] = _weights((E, d, F), cfg.get("outliers", 0.0), g, device)
        out["s13"] = init_scales(out["w13"], fmt, g)
        out["s2"] = init_scales(out["w2"], fmt, g)
    out["x"] = torch.randn((T, d), generator=g, device=device).to(torch.bfloat16).contiguous()
    out["dout"] = torch.randn((T, d), generator=g, device=device).to(torch.bfloat16).contiguous()
    out["topk_idx"], out["topk_w"] = _routing(T, E, k, cfg.get("routing", "uniform"), g, device)
    return out


def random_bf16(shape, seed=0, std=1.0, device="cpu"):
    g = _gen(seed, device)
    return (torch.randn(shape, generator=g, device=device) * std).to(torch.bfloat16).contiguous()


def to_numpy_bits(t):
    """bf16 tensor -> NumPy uint16 bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def to_numpy(t):
    return t.detach().cpu().contiguous().numpy()


def routed_rows_per_expert(topk_idx, E):
    return torch.bincount(topk_idx.reshape(-1).long(), minlength=E)


def tokens_to_flops(cfg):
    """Algorithmic fwd + bwd FLOPs of the layer: 3 x (2 R 2F d + 2 R d F), R = T k."""
    R = cfg["T"] * cfg["topk"]
    return 3 * (2 * R * 2 * cfg["F"] * cfg["d"] + 2 * R * cfg["d"] * cfg["F"])


__all__ = ["WORKLOADS", "workload", "make_inputs", "random_bf16", "to_numpy_bits", "to_numpy",
           "scale_block", "init_scales", "tokens_to_flops", "math"]
