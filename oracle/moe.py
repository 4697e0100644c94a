"""One MoE layer of scale-only QAD, forward and backward, in fp64 (test infrastructure only).

Sources, by page and section:

* AngelSlim mcore_qad walkthrough (nxmr.cn/news/131691), section 二.4: the routed
  experts of a layer are held as 3D-stacked weights, fake-quantized as a whole in one
  vectorised pass, and all experts run as ONE grouped GEMM over the token-routed rows
  (experts are split only by expert parallelism, ETP = 1, so each expert's [N, K]
  matrix is whole).
* Same article, section 二.3: the weight is quantize->dequantize(W; s), the input of
  each quantized matmul is fake-quantized first, the router is not quantized.
* "MCoreQAD Backend" (mcore_qad.md), opening section: BF16 weights frozen, only the
  quantizer scales receive gradients.

Readings taken where the pages are silent (each one is listed in the design notes):

* The routed-expert FFN is SwiGLU with the fused first weight [E, 2F, d]: rows [0, F)
  are the gate, rows [F, 2F) the up projection; H = silu(gate) * up.
* Routing indices and weights are inputs; the routing weight p multiplies the expert
  output in the combine (out = sum_j p_j * Y_j), so dY = p * dout.
* The (token, slot) pairs are grouped by expert, stably: order by (expert, token, slot).
  An index outside [0, E) or a repeat of an earlier slot's expert in the same token is
  dropped and flagged.
* Values are rounded to bf16 where a GPU implementation stores them: Z1, H, H_hat, Y,
  dY, dZ1, dA1, out, dx.  GEMMs, SwiGLU and sums are exact fp64 otherwise.  The fc2
  input gradient dH is consumed by the SwiGLU backward without being stored.
* Straight-through estimator for both quantizers: the gradient passes the fake-quant
  unchanged to its input; for the weight the scale gradient uses the LSQ factor
  (oracle.quant.lsq_factor).  Activation scales are detached.

``quant=False`` replaces every quantizer by the identity (the self-distillation
teacher pass of "MCoreQAD Backend", opening section) and ``round_bf16=False`` drops the
bf16 storage roundings; both together make the layer a smooth function, which the
finite-difference pins use.
"""
import numpy as np

from . import quant as Q

ERR_BAD_INDEX = 1   # a routing index outside [0, E)
ERR_DUP_INDEX = 2   # a token routed twice to the same expert


# --------------------------------------------------------------------------------------
# Routing permutation
# --------------------------------------------------------------------------------------

def route(topk_idx, E):
    """Group the T*k (token, slot) pairs by expert, keeping (token, slot) order inside.

    Returns a dict:
      row_token[R], row_slot[R]  -- the pair behind routed row r (R = valid pairs),
      row_of[T, k]               -- the row of pair (t, j), or -1 if it was dropped,
      counts[E], offsets[E + 1]  -- rows per expert and their exclusive prefix sum,
      error                      -- ERR_* bits for dropped pairs.
    """
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, k = idx.shape
    valid = (idx >= 0) & (idx < E)
    error = 0 if valid.all() else ERR_BAD_INDEX
    for j in range(1, k):
        dup = np.zeros(T, dtype=bool)
        for jj in range(j):
            dup |= idx[:, jj] == idx[:, j]
        dup &= valid[:, j]
        if dup.any():
            error |= ERR_DUP_INDEX
        valid[:, j] &= ~dup
    flat = np.where(valid, idx, -1).reshape(-1)
    row_token, row_slot, counts = [], [], np.zeros(E, dtype=np.int64)
    for e in range(E):
        pairs = np.nonzero(flat == e)[0]          # ascending pair index = (token, slot) order
        counts[e] = pairs.size
        row_token.append(pairs // k)
        row_slot.append(pairs % k)
    row_token = np.concatenate(row_token) if E else np.zeros(0, np.int64)
    row_slot = np.concatenate(row_slot) if E else np.zeros(0, np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    row_of = -np.ones((T, k), dtype=np.int64)
    row_of[row_token, row_slot] = np.arange(row_token.size)
    return dict(row_token=row_token, row_slot=row_slot, row_of=row_of,
                counts=counts, offsets=offsets, error=error)


# --------------------------------------------------------------------------------------
# Stages
# --------------------------------------------------------------------------------------

def grouped_gemm_nt(a, w, offsets):
    """out[r] = a[r] @ w[e].T for the rows r of expert e (w: [E, N, K], a: [R, K])."""
    E, N, _ = w.shape
    out = np.zeros((a.shape[0], N))
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            out[lo:hi] = a[lo:hi] @ w[e].T
    return out


def grouped_gemm_nn(a, w, offsets):
    """out[r] = a[r] @ w[e] for the rows r of expert e (w: [E, N, K], a: [R, N])."""
    E, _, K = w.shape
    out = np.zeros((a.shape[0], K))
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            out[lo:hi] = a[lo:hi] @ w[e]
    return out


def grouped_wgrad(dz, a, offsets, E):
    """dW[e] = dz[rows of e].T @ a[rows of e]: the weight gradient, [E, N, K]."""
    out = np.zeros((E, dz.shape[1], a.shape[1]))
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            out[e] = dz[lo:hi].T @ a[lo:hi]
    return out


def _sigmoid(g):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-g))


def swiglu(z1):
    """H = silu(gate) * up with gate = z1[:, :F], up = z1[:, F:]."""
    F = z1.shape[1] // 2
    g, u = z1[:, :F], z1[:, F:]
    return g * _sigmoid(g) * u


def swiglu_bwd(dh, z1):
    """dZ1 = [dgate, dup] for H = silu(gate) * up.

    d silu(g)/dg = sig(g) * (1 + g * (1 - sig(g))).
    """
    F = z1.shape[1] // 2
    g, u = z1[:, :F], z1[:, F:]
    sg = _sigmoid(g)
    dg = dh * u * sg * (1.0 + g * (1.0 - sg))
    du = dh * g * sg
    return np.concatenate([dg, du], axis=1)


def combine(y, p, row_of):
    """out[t] = sum_{j = 0..k-1} p[t, j] * y[row_of[t, j]] (dropped pairs contribute 0)."""
    T, k = row_of.shape
    out = np.zeros((T, y.shape[1]))
    for j in range(k):
        r = row_of[:, j]
        ok = r >= 0
        out[ok] += p[ok, j][:, None] * y[r[ok]]
    return out


# --------------------------------------------------------------------------------------
# The layer
# --------------------------------------------------------------------------------------

def _maybe_round(x, on):
    return Q.round_bf16(x) if on else x


def _values(a):
    """bf16 bit patterns (uint16) -> fp64 values; fp64 arrays pass through unchanged."""
    a = np.asarray(a)
    return Q.bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def moe_forward(fmt, x_bits, topk_idx, topk_w, w13_bits, s13, w2_bits, s2,
                quant=True, round_bf16=True, factored=False):
    """Forward of one MoE layer; returns out (fp64 on the bf16 grid) and the stash.

    factored=True (per-row scaled formats): the two forward GEMMs contract the quantization
    codes and apply the per-row weight and activation scales to the sum, i.e. they use
    q * s unrounded (the scales leave the contraction exactly in real arithmetic); the
    Ŵ13, Ŵ2, Â1 and Ĥ kept for the backward are the rounded fake-quant values as usual.
    """
    E = w13_bits.shape[0]
    rt = route(topk_idx, E)
    off = rt["offsets"]
    p = np.asarray(topk_w, dtype=np.float64)
    x = _values(x_bits)
    if quant:
        w13h = Q.fakequant_weight(fmt, w13_bits, s13)
        w2h = Q.fakequant_weight(fmt, w2_bits, s2)
        a1 = Q.fakequant_act(fmt, x)[rt["row_token"]]
    else:
        w13h, w2h = _values(w13_bits), _values(w2_bits)
        a1 = x[rt["row_token"]]
    if quant and factored:
        a1f = Q.fakequant_act_factored(fmt, x)[rt["row_token"]]
        z1 = _maybe_round(grouped_gemm_nt(a1f, Q.fakequant_weight_factored(fmt, w13_bits, s13), off), round_bf16)
    else:
        z1 = _maybe_round(grouped_gemm_nt(a1, w13h, off), round_bf16)
    h = _maybe_round(swiglu(z1), round_bf16)
    hh = Q.fakequant_act(fmt, h) if quant else h
    if quant and factored:
        y = _maybe_round(grouped_gemm_nt(Q.fakequant_act_factored(fmt, h),
                                         Q.fakequant_weight_factored(fmt, w2_bits, s2), off), round_bf16)
    else:
        y = _maybe_round(grouped_gemm_nt(hh, w2h, off), round_bf16)
    out = _maybe_round(combine(y, p, rt["row_of"]), round_bf16)
    return dict(out=out, route=rt, w13h=w13h, w2h=w2h, a1=a1, z1=z1, h=h, hh=hh, y=y)


def moe_dgrad(dout_bits, topk_w, fwd, round_bf16=True):
    """Input gradient dx [T, d] and routing-weight gradient dprobs [T, k].

    dY = bf16(fp32(p * dout)); dH = dY @ W2_hat[e]; dZ1 = SwiGLU backward; dA1 = dZ1 @
    W13_hat[e]; dx[t] = sum_j dA1[row_of[t, j]] (straight through the activation
    fake-quant); dprobs[t, j] = <dout[t], Y[row_of[t, j]]>.
    """
    rt = fwd["route"]
    off, row_of = rt["offsets"], rt["row_of"]
    p = np.asarray(topk_w, dtype=np.float64)
    dout = _values(dout_bits)
    prow = p[rt["row_token"], rt["row_slot"]][:, None]
    dy = dout[rt["row_token"]] * prow
    if round_bf16:
        dy = Q.round_bf16(Q.round_f32(dy))
    dh = grouped_gemm_nn(dy, fwd["w2h"], off)
    dz1 = _maybe_round(swiglu_bwd(dh, fwd["z1"]), round_bf16)
    da1 = _maybe_round(grouped_gemm_nn(dz1, fwd["w13h"], off), round_bf16)
    T, k = row_of.shape
    dx = _maybe_round(combine(da1, np.ones((T, k)), row_of), round_bf16)
    dprobs = np.zeros((T, k))
    for j in range(k):
        r = row_of[:, j]
        ok = r >= 0
        dprobs[ok, j] = np.einsum("td,td->t", dout[ok], fwd["y"][r[ok]])
    return dict(dx=dx, dprobs=dprobs, dy=dy, dh=dh, dz1=dz1, da1=da1)


def moe_weight_grads(fwd, bwd):
    """Gradients with respect to the fake-quantized weights (never stored by the GPU path)."""
    E = fwd["w13h"].shape[0]
    off = fwd["route"]["offsets"]
    dw2 = grouped_wgrad(bwd["dy"], fwd["hh"], off, E)
    dw13 = grouped_wgrad(bwd["dz1"], fwd["a1"], off, E)
    return dw13, dw2


def moe_scalegrad(fmt, fwd, bwd, w13_bits, s13, w2_bits, s2):
    """Scale gradients ds13 [E, 2F, d/B], ds2 [E, d, F/B]: block sums of dW * phi."""
    dw13, dw2 = moe_weight_grads(fwd, bwd)
    ds13 = Q.scale_grad_from_wgrad(fmt, dw13, w13_bits, s13)
    ds2 = Q.scale_grad_from_wgrad(fmt, dw2, w2_bits, s2)
    return ds13, ds2
