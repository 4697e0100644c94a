"""Quantizer arithmetic of the oracle (fp64 NumPy; test infrastructure only).

Sources, by page and section:

* AngelSlim mcore_qad walkthrough (nxmr.cn/news/131691), section 二.3: the weight
  seen by the matmul is quantize->dequantize(W; s) with s the trainable quantity;
  activations are fake-quantized by a pre-hook before each quantized matmul.
* Same article, section 三, and "MCoreQAD Backend" (mcore_qad.md), "Support Matrix":
  the formats nvfp4 (FP4 E2M1 weights and activations), w4a16 (INT4 weights,
  BF16 activations) and fp8 (E4M3 weights and activations).

The pages never write the quantizer formulas down.  The readings used here:

* E2M1 grid {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6} (OCP Microscaling Formats
  v1.0, E2M1 element type), round to nearest with ties to the even code
  (IEEE 754 roundTiesToEven), saturating at +-6.
* E4M3 ("fn" variant: max finite 448, subnormals spaced 2^-9), ties to even,
  saturating at +-448.
* INT4 symmetric grid {-8, ..., 7}: round half to even, then clamp.
* INT8 (w8a8) grid {-128, ..., 127}: round half to even, then clamp; scales amax/127.
* The weight scale is one fp32 number per block of B consecutive elements along K
  (B = 16 for nvfp4, 128 for INT4 group-128, B = K for fp8 per output row), not
  itself rounded to a narrower format (formats 0-5; format 6 below rounds it).
* x = fp32(w / s) is an IEEE fp32 division; the dequantized product q(x)*s is
  rounded to fp32 and then to bf16.  Division of two fp32 values done in fp64 and
  rounded once to fp32 equals the IEEE fp32 quotient (53 >= 2*24 + 2), so these
  steps are bit-exact while everything else runs in fp64.
* s == 0 (an all-zero block) gives x = +-0 (the sign of w), output +-0 and a zero
  LSQ factor.
* nvfp4 with deployed scales (format 6): the compressed-tensors NVFP4 layout that the
  format names map to (walkthrough, section 三) keeps each 16-element block's scale as an E4M3
  number times an fp32 scale of the whole tensor.  Weights: the learnable fp32 block scale s is
  used as s_q = fp32(e4m3(fp32(s / g)) * g), with g = fp32(max |s| / 448) over each expert matrix
  (the largest block scale becomes E4M3's 448; gate and up share one g, as the fused gate-up
  matrix of a deployed expert stores one); activations: the dynamic block scale
  fp32(amax / 6) is rounded the same way under g = fp32(max of the row's block scales / 448).
  g = 0 (an all-zero matrix or row) gives s_q = 0.  The gradient reaches s straight through the
  E4M3 rounding; g is treated as a constant.
* The LSQ straight-through factor (Esser et al., "Learned Step Size
  Quantization", 2019) is phi = q(x) - x inside the CLOSED clip range and the
  violated bound outside it.  No 1/sqrt(N*Qp) gradient scale is applied.

Parity pins for every function here live in tests/test_oracle_pins.py.
"""
import numpy as np

FMT_NVFP4 = 0       # nvfp4 W4A4: E2M1, block 16 along K, activations block-16 amax/6
FMT_INT4_G128 = 1   # w4a16: INT4, group 128 along K, activations left in bf16
FMT_FP8_ROW = 2     # fp8 W8A8: E4M3, one scale per output row, activations per-row amax/448
FMT_NVFP4A16 = 3    # nvfp4a16: E2M1 weights as nvfp4, activations left in bf16
FMT_W8A8 = 4        # w8a8: INT8 weights, one scale per output row, activations per-row amax/127
FMT_W4AFP8 = 5      # w4afp8: INT4 weights as w4a16, activations E4M3 per-row amax/448
FMT_NVFP4_E4M3 = 6  # nvfp4 with deployed scales: E4M3 block scales under an fp32 per-matrix / per-row scale
FORMATS = (FMT_NVFP4, FMT_INT4_G128, FMT_FP8_ROW, FMT_NVFP4A16, FMT_W8A8, FMT_W4AFP8, FMT_NVFP4_E4M3)

# element grids ("quantizer kinds") and what each format uses for weights / activations
Q_E2M1, Q_INT4, Q_E4M3, Q_INT8 = "e2m1", "int4", "e4m3", "int8"
Q_E2M1G = "e2m1g"  # E2M1 elements, E4M3 block scales under an fp32 scale of the row (activations)
WEIGHT_Q = {FMT_NVFP4: Q_E2M1, FMT_INT4_G128: Q_INT4, FMT_FP8_ROW: Q_E4M3, FMT_NVFP4A16: Q_E2M1,
            FMT_W8A8: Q_INT8, FMT_W4AFP8: Q_INT4, FMT_NVFP4_E4M3: Q_E2M1}
ACT_Q = {FMT_NVFP4: Q_E2M1, FMT_INT4_G128: None, FMT_FP8_ROW: Q_E4M3, FMT_NVFP4A16: None,
         FMT_W8A8: Q_INT8, FMT_W4AFP8: Q_E4M3, FMT_NVFP4_E4M3: Q_E2M1G}
# per quantizer kind: (lower clip bound, upper clip bound), the divisor that turns an amax
# into a scale, and the block of consecutive K elements sharing a scale (None = a whole row)
Q_CLIP = {Q_E2M1: (-6.0, 6.0), Q_INT4: (-8.0, 7.0), Q_E4M3: (-448.0, 448.0), Q_INT8: (-128.0, 127.0),
          Q_E2M1G: (-6.0, 6.0)}
Q_AMAX_DIV = {Q_E2M1: 6.0, Q_INT4: 7.0, Q_E4M3: 448.0, Q_INT8: 127.0, Q_E2M1G: 6.0}
Q_BLOCK = {Q_E2M1: 16, Q_INT4: 128, Q_E4M3: None, Q_INT8: None, Q_E2M1G: 16}
E4M3_MAX = 448.0

CLIP = {f: Q_CLIP[WEIGHT_Q[f]] for f in FORMATS}
AMAX_DIV = {f: Q_AMAX_DIV[WEIGHT_Q[f]] for f in FORMATS}


def weight_block(fmt, K):
    """Elements of K that share one weight scale."""
    b = Q_BLOCK[WEIGHT_Q[fmt]]
    return K if b is None else b


# --------------------------------------------------------------------------------------
# bf16 / fp32 storage
# --------------------------------------------------------------------------------------

def bf16_to_f64(bits):
    """uint16 bf16 bit patterns -> exact fp64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_bf16(x):
    """Round fp64 (or fp32) values ONCE to the nearest bf16 (ties to even).

    bf16 keeps 8 significant bits and fp32's exponent range (normal floor 2^-126,
    subnormal spacing 2^-133); values that round to 2^128 or beyond become inf.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # |x| = m * 2^e with 0.5 <= m < 1
    qexp = np.maximum(e - 8, -133)            # spacing of bf16 numbers near x
    r = np.ldexp(np.rint(np.ldexp(x, -qexp)), qexp)
    r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, x), r)
    return np.where(np.isfinite(x), r, x)


def f64_to_bf16_bits(x):
    """fp64 values -> bf16 bit patterns (rounding once, ties to even)."""
    r = round_bf16(x).astype(np.float32)     # exact: r already lies on the bf16 grid
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def round_f32(x):
    """Round fp64 values once to fp32 (NumPy's cast is round-to-nearest-even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# --------------------------------------------------------------------------------------
# Element quantizers q(x): values on the format's grid, as fp64
# --------------------------------------------------------------------------------------

def e2m1_decode(code):
    """4-bit E2M1 code (sign, 2 exponent bits, 1 mantissa bit, bias 1) -> value."""
    code = np.asarray(code, dtype=np.int64)
    sign = np.where(code & 8, -1.0, 1.0)
    ex = (code >> 1) & 3
    man = code & 1
    mag = np.where(ex == 0, 0.5 * man, (1.0 + 0.5 * man) * np.ldexp(1.0, ex - 1))
    return sign * mag


def q_e2m1(x):
    """Round to the E2M1 grid, ties to even code, saturating at +-6.

    For |x| the decision points are the midpoints between neighbouring grid values:
    0.25 (0|0.5), 0.75 (0.5|1), 1.25 (1|1.5), 1.75 (1.5|2), 2.5 (2|3), 3.5 (3|4), 5 (4|6).
    At a midpoint the result is the neighbour whose mantissa bit is 0 (0, 1, 2, 4 are
    even; 0.5, 1.5, 3, 6 are odd), so 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2,
    3.5->4, 5->4.  Anything above 5 rounds to 6 (satfinite).  The sign is kept, so a
    negative input that rounds to zero gives -0.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    mag = np.select(
        [a <= 0.25, a < 0.75, a <= 1.25, a < 1.75, a <= 2.5, a < 3.5, a <= 5.0],
        [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0],
        default=6.0)
    return np.copysign(mag, x)


def q_e4m3(x):
    """Round to the E4M3 (fn) grid, ties to even, saturating at +-448.

    Normal binades [2^e, 2^(e+1)) for e >= -6 hold 8 values spaced 2^(e-3); below
    2^-6 the subnormals are spaced 2^-9.  Scaling by a power of two is exact, so
    rint(|x| / spacing) * spacing is the tie-to-even rounding on that binade; a
    result that carries to 2^(e+1) is still on the grid.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                       # a = m * 2^e, 0.5 <= m < 1 -> binade e-1
    binade = np.maximum(e - 1, -6)
    spacing = np.ldexp(1.0, binade - 3)
    mag = np.minimum(np.rint(a / spacing) * spacing, 448.0)
    mag = np.where(a == 0, 0.0, mag)
    return np.copysign(mag, x)


def q_int4(x):
    """Round half to even to an integer, then clamp to the INT4 range [-8, 7]."""
    x = np.asarray(x, dtype=np.float64)
    return np.clip(np.rint(x), -8.0, 7.0)


def q_int8(x):
    """Round half to even to an integer, then clamp to the INT8 range [-128, 127]."""
    x = np.asarray(x, dtype=np.float64)
    return np.clip(np.rint(x), -128.0, 127.0)


Q_FUNC = {Q_E2M1: q_e2m1, Q_INT4: q_int4, Q_E4M3: q_e4m3, Q_INT8: q_int8, Q_E2M1G: q_e2m1}


def q_fmt(fmt, x):
    """The weight quantizer of format `fmt`."""
    return Q_FUNC[WEIGHT_Q[fmt]](x)


# --------------------------------------------------------------------------------------
# Fake quantization
# --------------------------------------------------------------------------------------

def _quotient(w, s):
    """x = fp32(w / s) with IEEE fp32 rounding; s == 0 gives +-0 with w's sign."""
    with np.errstate(divide="ignore", invalid="ignore"):
        x = round_f32(w / np.where(s == 0, 1.0, s))
    return np.where(s == 0, np.copysign(0.0, w), x)


def _dequant(qx, s):
    """bf16(fp32(q * s)): the product rounded to fp32, then to bf16."""
    return round_bf16(round_f32(qx * s))


def deploy_scales(scale, axes):
    """Block scales as deployed NVFP4 holds them: s_q = fp32(e4m3(fp32(s / g)) * g) with
    g = fp32(max |s| / 448) over `axes` (a matrix, or a row); g = 0 gives s_q = 0.  (The
    magnitude: a learnable scale is not constrained to stay positive, and a negative one is
    rounded as its magnitude with the sign kept.)"""
    s = np.asarray(scale, dtype=np.float64)
    g = round_f32(np.abs(s).max(axis=axes, keepdims=True) / E4M3_MAX)
    safe = np.where(g == 0, 1.0, g)
    sq = round_f32(q_e4m3(round_f32(s / safe)) * g)
    return np.where(g == 0, 0.0, sq)


def effective_weight_scales(fmt, scale):
    """The scales the weight quantizer uses: the learnable ones, or their deployed rounding
    (format 6, one fp32 g per matrix: the last two axes)."""
    s = np.asarray(scale, dtype=np.float64)
    return deploy_scales(s, axes=(-2, -1)) if fmt == FMT_NVFP4_E4M3 else s


def weight_quotient(fmt, w_bits, scale):
    """x = fp32(W / s) for stacked weights [..., N, K] and scales [..., N, K / B]."""
    w = bf16_to_f64(w_bits)
    K = w.shape[-1]
    s = np.repeat(effective_weight_scales(fmt, scale), weight_block(fmt, K), axis=-1)
    return w, s, _quotient(w, s)


def fakequant_weight(fmt, w_bits, scale):
    """W_hat = bf16(fp32(q(fp32(W / s)) * s)), element by element (section 二.3/二.4).

    w_bits: uint16 bf16 [..., N, K]; scale: fp32 [..., N, K / B].  Returns fp64 values
    that all lie on the bf16 grid.
    """
    _, s, x = weight_quotient(fmt, w_bits, scale)
    return _dequant(q_fmt(fmt, x), s)


def fakequant_weight_factored(fmt, w_bits, scale):
    """q(fp32(W / s)) * s in fp64, the product not rounded: the weight a GEMM applies when its
    per-row scale is factored out of the contraction and multiplied into the accumulator
    (native low-precision MMA on the codes q).  The codes are those of fakequant_weight, so
    rounding this to fp32 and then bf16 gives fakequant_weight exactly."""
    _, s, x = weight_quotient(fmt, w_bits, scale)
    return q_fmt(fmt, x) * s


def fakequant_act_factored(fmt, a):
    """q(fp32(a / s_a)) * s_a in fp64, not rounded (see fakequant_weight_factored)."""
    a = np.asarray(a, dtype=np.float64)
    kind = ACT_Q[fmt]
    if kind is None:
        return a.copy()
    s = act_scale(fmt, a)
    return Q_FUNC[kind](_quotient(a, s)) * s


def act_scale(fmt, a):
    """Dynamic activation scale per block along the last axis (detached, not learnable).

    E2M1 (nvfp4): one scale per 16 elements, fp32(amax / 6); with deployed scales (format 6)
    those block scales are then rounded as deploy_scales does, under one g per row.  E4M3 (fp8,
    w4afp8): one per row, fp32(amax / 448).  INT8 (w8a8): one per row, fp32(amax / 127).
    Returns the scale broadcast to a's shape.
    """
    a = np.asarray(a, dtype=np.float64)
    kind = ACT_Q[fmt]
    if kind is None:
        raise ValueError("format has no activation quantizer")
    div = Q_AMAX_DIV[kind]
    if Q_BLOCK[kind] == 16:
        blocks = a.reshape(a.shape[:-1] + (a.shape[-1] // 16, 16))
        amax = np.abs(blocks).max(axis=-1)
        sb = round_f32(amax / div)
        if kind == Q_E2M1G:
            sb = deploy_scales(sb, axes=-1)
        return np.repeat(sb, 16, axis=-1)
    amax = np.abs(a).max(axis=-1, keepdims=True)
    return np.broadcast_to(round_f32(amax / div), a.shape)


def fakequant_act(fmt, a):
    """Activation fake-quant a_hat = bf16(fp32(q(fp32(a / s_a)) * s_a)); identity without one."""
    a = np.asarray(a, dtype=np.float64)
    kind = ACT_Q[fmt]
    if kind is None:
        return a.copy()
    s = act_scale(fmt, a)
    return _dequant(Q_FUNC[kind](_quotient(a, s)), s)


def lsq_factor(fmt, x):
    """LSQ straight-through derivative of s*q(w/s) with respect to s, given x = fp32(w/s).

    Inside the closed clip range [lo, hi] it is q(x) - x; below it lo, above it hi.
    """
    lo, hi = CLIP[fmt]
    x = np.asarray(x, dtype=np.float64)
    return np.where(x < lo, lo, np.where(x > hi, hi, q_fmt(fmt, x) - x))


def scale_grad_from_wgrad(fmt, dw, w_bits, scale):
    """g_s[..., n, b] = sum over k in block b of dW[..., n, k] * phi(W[..., n, k], s[..., n, b])."""
    _, _, x = weight_quotient(fmt, w_bits, scale)
    prod = np.asarray(dw, dtype=np.float64) * lsq_factor(fmt, x)
    K = prod.shape[-1]
    B = weight_block(fmt, K)
    return prod.reshape(prod.shape[:-1] + (K // B, B)).sum(axis=-1)
