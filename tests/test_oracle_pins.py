"""Pins of the oracle against facts fixed outside it (CPU only).

Each test checks the oracle against something it does not itself contain: golden
values worked by hand from a format's definition (tests/golden/, cited there), a
library routine (torch's float8_e4m3fn cast, NumPy's stable argsort, torch's silu),
brute-force enumeration of a grid, autograd of the straight-through definition,
or central finite differences.
"""
import os

import numpy as np
import pytest
import torch

from oracle import moe as M
from oracle import quant as Q

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _f32_sweep(lo, hi, n, rng):
    """Random fp32 values in [lo, hi] plus the fp32 neighbours of every quarter-integer and grid point."""
    x = rng.uniform(lo, hi, n).astype(np.float32)
    marks = np.arange(lo * 64, hi * 64 + 1) / 64.0
    m32 = marks.astype(np.float32)
    near = np.concatenate([m32, np.nextafter(m32, np.float32(np.inf)), np.nextafter(m32, np.float32(-np.inf))])
    return np.concatenate([x, near, -x, -near]).astype(np.float64)


def _brute_nearest(x, grid, even):
    """Nearest grid value to each x; ties go to the value whose `even` flag is set."""
    grid = np.asarray(grid, dtype=np.float64)
    even = np.asarray(even, dtype=bool)
    dist = np.abs(x[:, None] - grid[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    pick_even = cand & even[None, :]
    use = np.where(pick_even.any(axis=1, keepdims=True), pick_even, cand)
    return grid[np.argmax(use, axis=1)]


# ------------------------------------------------------------------------------ E2M1

def test_e2m1_decode_matches_spec_table():
    rows = _rows("e2m1_grid.txt")
    codes = np.array([int(r[0]) for r in rows])
    want = np.array([float(r[1]) for r in rows])
    got = Q.e2m1_decode(codes)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_e2m1_tie_table():
    rows = _rows("e2m1_ties.txt")
    x = np.array([float.fromhex(r[0]) for r in rows])
    want = np.array([float(r[1]) for r in rows])
    got = Q.q_e2m1(x)
    assert np.array_equal(got, want), list(zip(x, got, want))
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_e2m1_bruteforce_nearest_even_code():
    rng = np.random.default_rng(1)
    x = _f32_sweep(-8.0, 8.0, 20000, rng)
    codes = np.arange(16)
    grid = Q.e2m1_decode(codes)
    even = (codes & 1) == 0
    want = _brute_nearest(np.abs(x), grid[:8], even[:8]) * np.where(np.signbit(x), -1.0, 1.0)
    got = Q.q_e2m1(x)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(x))


# ------------------------------------------------------------------------------ E4M3

def _e4m3_positive_grid():
    vals, even = [], []
    for code in range(0x7F):          # 0x7F is NaN in the fn variant
        ex, man = code >> 3, code & 7
        vals.append(man * 2.0 ** -9 if ex == 0 else (1 + man / 8) * 2.0 ** (ex - 7))
        even.append(man % 2 == 0)
    return np.array(vals), np.array(even)


def test_e4m3_golden_points():
    rows = _rows("e4m3_points.txt")
    x = np.array([float.fromhex(r[0]) for r in rows])
    want = np.array([float.fromhex(r[1]) for r in rows])
    got = Q.q_e4m3(x)
    assert np.array_equal(got, want), list(zip(x, got, want))
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_e4m3_matches_torch_cast_inside_range():
    rng = np.random.default_rng(2)
    x = np.concatenate([_f32_sweep(-8.0, 8.0, 20000, rng),
                        rng.uniform(-448, 448, 20000).astype(np.float32).astype(np.float64),
                        (rng.standard_normal(20000) * 1e-3).astype(np.float32).astype(np.float64)])
    x = x[np.abs(x) <= 448]
    lib = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(Q.q_e4m3(x), lib)


def test_e4m3_bruteforce_with_saturation():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-600, 600, 5000), rng.standard_normal(5000) * 0.01]).astype(np.float32)
    x = x.astype(np.float64)
    grid, even = _e4m3_positive_grid()
    want = _brute_nearest(np.abs(x), grid, even) * np.where(np.signbit(x), -1.0, 1.0)
    assert np.array_equal(Q.q_e4m3(x), want)


# ------------------------------------------------------------------------------ INT4

def test_int4_bruteforce_nearest_even():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.uniform(-12, 12, 20000), np.arange(-24, 25) / 2.0])
    grid = np.arange(-8, 8, dtype=np.float64)
    want = _brute_nearest(x, grid, grid % 2 == 0)
    assert np.array_equal(Q.q_int4(x), want)


def test_int8_bruteforce_nearest_even():
    rng = np.random.default_rng(40)
    x = np.concatenate([rng.uniform(-140, 140, 20000), np.arange(-280, 281) / 2.0])
    grid = np.arange(-128, 128, dtype=np.float64)
    want = _brute_nearest(x, grid, grid % 2 == 0)
    assert np.array_equal(Q.q_int8(x), want)


def _grid(fmt):
    """The weight grid of a format, enumerated (not computed by the quantizer)."""
    kind = Q.WEIGHT_Q[fmt]
    if kind == Q.Q_E2M1:
        return Q.e2m1_decode(np.arange(16))
    if kind == Q.Q_INT4:
        return np.arange(-8, 8, dtype=np.float64)
    if kind == Q.Q_INT8:
        return np.arange(-128, 128, dtype=np.float64)
    pos, _ = _e4m3_positive_grid()
    return np.concatenate([pos, -pos])


# ------------------------------------------------------------------------------ bf16 rounding

def test_round_bf16_fp32_inputs_match_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.integers(-30, 30, 50000),
                        [0.0, -0.0, 3.0e38, -3.0e38, 1e-40]]).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(Q.round_bf16(x.astype(np.float64)), lib)


def test_round_bf16_fp64_is_single_rounding():
    rng = np.random.default_rng(6)
    x = rng.standard_normal(50000) * 10.0 ** rng.integers(-20, 20, 50000)
    got = Q.round_bf16(x)
    # the three bf16 numbers around the truncation of fp32(x)
    t = (x.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000))
    cands = []
    for dlt in (-1, 0, 1):
        c = (t.astype(np.int64) + dlt * 0x10000).astype(np.uint32).view(np.float32).astype(np.float64)
        cands.append(c)
    cands = np.stack(cands, 1)
    dist = np.abs(cands - x[:, None])
    best = dist.min(1, keepdims=True)
    tie_even = (dist == best) & (((cands.astype(np.float32).view(np.uint32) >> 16) & 1) == 0)
    use = np.where(tie_even.any(1, keepdims=True), tie_even, dist == best)
    want = cands[np.arange(x.size), np.argmax(use, 1)]
    assert np.array_equal(got, want)


# ------------------------------------------------------------------------------ fake quant

def _weights(fmt, E=2, N=8, K=256, seed=7, outliers=True):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn((E, N, K), generator=g) * 0.02
    if outliers:
        w[0, 0, :5] = torch.tensor([0.5, -0.5, 0.0, -0.0, 1e-30])
        w[1, 1, :16] = 0.0                       # an all-zero block -> zero scale
    w = w.to(torch.bfloat16)
    B = Q.weight_block(fmt, K)
    amax = w.float().abs().reshape(E, N, K // B, B).amax(-1)
    s = (amax / Q.AMAX_DIV[fmt] * (1 + (torch.rand(amax.shape, generator=g) * 0.2 - 0.1))).float()
    bits = w.view(torch.int16).numpy().view(np.uint16)
    return bits, s.numpy()


@pytest.mark.parametrize("fmt", Q.FORMATS)
def test_fakequant_idempotent(fmt):
    bits, s = _weights(fmt)
    w1 = Q.fakequant_weight(fmt, bits, s)
    w2 = Q.fakequant_weight(fmt, Q.f64_to_bf16_bits(w1), s)
    assert np.array_equal(Q.f64_to_bf16_bits(w1), Q.f64_to_bf16_bits(w2))
    assert np.all(np.isfinite(w1))


@pytest.mark.parametrize("fmt", Q.FORMATS)
def test_fakequant_outputs_lie_on_scaled_grid(fmt):
    bits, s = _weights(fmt, N=4, K=128)
    what = Q.fakequant_weight(fmt, bits, s)
    K = bits.shape[-1]
    # the scales the quantizer uses (format 6: the deployed E4M3 rounding of s)
    sf = np.repeat(Q.effective_weight_scales(fmt, s), Q.weight_block(fmt, K), axis=-1)
    grid = _grid(fmt)
    # every output equals bf16(fp32(g * s)) for some g of the grid (enumerated, not computed by q)
    cand = Q.round_bf16(Q.round_f32(grid[None, :] * sf.reshape(-1)[:, None]))
    hit = (cand == what.reshape(-1)[:, None]).any(axis=1)
    assert hit.all()


def test_fakequant_zero_scale_block_gives_signed_zero():
    bits, s = _weights(Q.FMT_NVFP4)
    assert s[1, 1, 0] == 0
    what = Q.fakequant_weight(Q.FMT_NVFP4, bits, s)
    blk = what[1, 1, :16]
    assert np.all(blk == 0)
    w = Q.bf16_to_f64(bits)[1, 1, :16]
    assert np.array_equal(np.signbit(blk), np.signbit(w))


@pytest.mark.parametrize("fmt", [f for f in Q.FORMATS if Q.ACT_Q[f] is not None])
def test_act_fakequant_properties(fmt):
    rng = np.random.default_rng(8)
    a = Q.round_bf16(rng.standard_normal((6, 64)))
    a[2, :16] = 0.0
    ah = Q.fakequant_act(fmt, a)
    assert np.all(np.isfinite(ah))
    assert np.all(ah[2, :16] == 0)
    # the block maximum maps to the top of the grid, so it is kept to bf16 accuracy
    blk = 16 if Q.ACT_Q[fmt] == Q.Q_E2M1 else 64
    ab = np.abs(a).reshape(6, -1, blk)
    hb = np.abs(ah).reshape(6, -1, blk)
    i = ab.argmax(-1)
    amax = np.take_along_axis(ab, i[..., None], -1)[..., 0]
    hmax = np.take_along_axis(hb, i[..., None], -1)[..., 0]
    assert np.allclose(hmax, amax, rtol=2 ** -7, atol=0)
    # the block maximum divided by its scale is the top of the grid (up to the fp32 scale rounding)
    s_a = np.take_along_axis(Q.act_scale(fmt, a).reshape(6, -1, blk), i[..., None], -1)[..., 0]
    top = Q.Q_CLIP[Q.ACT_Q[fmt]][1]
    nz = amax > 0
    assert np.allclose(amax[nz] / s_a[nz], top, rtol=1e-6, atol=0)
    # idempotent up to the dynamic scale being recomputed from the quantized block
    assert np.array_equal(Q.fakequant_act(fmt, ah), ah)


@pytest.mark.parametrize("fmt", [f for f in Q.FORMATS if Q.ACT_Q[f] is None])
def test_weight_only_formats_leave_activations_alone(fmt):
    a = Q.round_bf16(np.random.default_rng(9).standard_normal((3, 256)))
    assert np.array_equal(Q.fakequant_act(fmt, a), a)


# ------------------------------------------------------------------------------ LSQ factor

@pytest.mark.parametrize("fmt", Q.FORMATS)
def test_scale_grad_zero_for_weights_on_grid_points(fmt):
    E, N, K = 2, 4, 256
    B = Q.weight_block(fmt, K)
    rng = np.random.default_rng(10)
    grid = _grid(fmt)
    s = 2.0 ** rng.integers(-8, -2, (E, N, K // B))        # powers of two: g * s exact in bf16
    if fmt == Q.FMT_NVFP4_E4M3:
        # deployed scales: with each matrix's largest scale 448 * 2^-12 the per-matrix fp32
        # scale is 2^-12 exactly and every power of two in [2^-8, 2^-4] is an E4M3 number
        # times it, so the deployed rounding leaves s unchanged (448 * 2^-12 * grid is exact in bf16)
        s = 2.0 ** rng.integers(-8, -3, (E, N, K // B))
        s[:, 0, 0] = 448.0 * 2.0 ** -12
        assert np.array_equal(Q.effective_weight_scales(fmt, s), s)
    g = rng.choice(grid, (E, N, K))
    lo, hi = Q.CLIP[fmt]
    g[0, 0, 0], g[0, 0, 1] = lo, hi                         # the clip bounds themselves (closed range)
    w = g * np.repeat(s, B, -1)
    bits = Q.f64_to_bf16_bits(w)
    assert np.array_equal(Q.bf16_to_f64(bits), w)
    dw = rng.standard_normal((E, N, K))
    ds = Q.scale_grad_from_wgrad(fmt, dw, bits, s.astype(np.float32))
    assert np.all(ds == 0.0)


@pytest.mark.parametrize("fmt", Q.FORMATS)
def test_lsq_factor_structure(fmt):
    lo, hi = Q.CLIP[fmt]
    rng = np.random.default_rng(11)
    x = Q.round_f32(rng.uniform(2 * lo, 2 * hi, 20000))
    phi = Q.lsq_factor(fmt, x)
    inside = (x >= lo) & (x <= hi)
    assert np.all(phi[x < lo] == lo) and np.all(phi[x > hi] == hi)
    # inside the range x + phi is the quantized value: on the grid and the nearest grid point
    grid = _grid(fmt)
    xin, qin = x[inside], x[inside] + phi[inside]
    assert np.isin(qin, grid).all()
    nearest = np.abs(xin[:, None] - grid[None, :]).min(1)
    assert np.allclose(np.abs(phi[inside]), nearest, rtol=0, atol=1e-12)


def _ste_fakequant_torch(fmt, w, s):
    """s * q_ste(w / s) with autograd: inside the clip range the rounding residual is
    detached (straight-through), outside the clamp has zero slope."""
    lo, hi = Q.CLIP[fmt]
    xd = w / s
    x = xd + (xd.float().double() - xd).detach()          # the fp32 quotient, same slope
    kind = Q.WEIGHT_Q[fmt]
    if kind == Q.Q_E4M3:
        qx = x.detach().float().to(torch.float8_e4m3fn).double()
    elif kind in (Q.Q_INT4, Q.Q_INT8):
        qx = torch.round(x.detach())                       # half to even
    else:
        grid = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64)
        a = x.detach().abs().clamp(max=6.0)
        d = (a[..., None] - grid).abs()
        best = d.min(-1, keepdim=True).values
        evenmask = torch.tensor([1, 0, 1, 0, 1, 0, 1, 0], dtype=torch.bool)
        tie = (d == best) & evenmask
        use = torch.where(tie.any(-1, keepdim=True), tie, d == best)
        qx = grid[use.float().argmax(-1)] * torch.sign(x.detach())
    inside = (x >= lo) & (x <= hi)
    xq = torch.where(inside, x + (qx - x).detach(), x.clamp(lo, hi))
    return s * xq


@pytest.mark.parametrize("fmt", Q.FORMATS)
def test_scale_grad_matches_autograd_of_ste_definition(fmt):
    bits, s = _weights(fmt, E=2, N=4, K=256, seed=12)
    s = s * np.float32(0.7)                                 # push some weights past the clip bound
    s = s.astype(np.float32)
    K = bits.shape[-1]
    B = Q.weight_block(fmt, K)
    rng = np.random.default_rng(13)
    dw = rng.standard_normal(bits.shape)
    w_t = torch.from_numpy(Q.bf16_to_f64(bits))
    s_t = torch.from_numpy(s.astype(np.float64)).requires_grad_(True)
    s_used = s_t
    if fmt == Q.FMT_NVFP4_E4M3:
        # the deployed rounding of the scale, passed straight through: the forward sees
        # s_q = fp32(e4m3(fp32(s / g)) * g), computed here with torch's float8_e4m3fn cast, and
        # the gradient reaches s unchanged (g a constant)
        s32 = torch.from_numpy(s.astype(np.float32))
        g = (s32.abs().amax(dim=(-2, -1), keepdim=True) / 448.0)
        sq = ((s32 / g).to(torch.float8_e4m3fn).float() * g).double()
        s_used = s_t + (sq - s_t).detach()
    s_full = s_used.repeat_interleave(B, dim=-1)
    safe = torch.where(s_full == 0, torch.ones_like(s_full), s_full)
    what = _ste_fakequant_torch(fmt, w_t, safe)
    what = torch.where(s_full == 0, torch.zeros_like(what), what)
    (what * torch.from_numpy(dw)).sum().backward()
    want = s_t.grad.numpy()
    got = Q.scale_grad_from_wgrad(fmt, dw, bits, s)
    # autograd's slope uses the fp64 quotient w/s, the oracle's the fp32 one: they differ
    # by ~1e-7 relative; a dropped term or a wrong sign would differ by O(1)
    assert np.allclose(got, want, rtol=1e-5, atol=1e-5)


# ------------------------------------------------------------------------------ routing

def test_route_matches_stable_argsort():
    rng = np.random.default_rng(14)
    T, E, k = 300, 7, 3
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    rt = M.route(idx, E)
    order = np.argsort(idx.reshape(-1), kind="stable")
    assert np.array_equal(rt["row_token"] * k + rt["row_slot"], order)
    assert np.array_equal(rt["counts"], np.bincount(idx.reshape(-1), minlength=E))
    assert rt["error"] == 0


def test_route_hand_worked_example_with_invalid_pairs():
    rows = _rows("route_small.txt")
    idx = np.array([[int(v) for v in r[1:]] for r in rows if r[0] == "idx"])
    want_rows = [(int(r[1]), int(r[2])) for r in rows if r[0] == "row"]
    counts = [int(v) for r in rows if r[0] == "counts" for v in r[1:]]
    err = [int(r[1]) for r in rows if r[0] == "error"][0]
    rt = M.route(idx, 3)
    assert list(zip(rt["row_token"], rt["row_slot"])) == want_rows
    assert list(rt["counts"]) == counts
    assert rt["error"] == err
    assert rt["row_of"][3, 0] == -1 and rt["row_of"][2, 1] == -1


# ------------------------------------------------------------------------------ grouped GEMM

def test_grouped_gemm_against_triple_loops():
    rng = np.random.default_rng(15)
    counts = [0, 1, 5]
    off = np.concatenate([[0], np.cumsum(counts)])
    R, E, N, K = off[-1], 3, 4, 6
    a = rng.standard_normal((R, K))
    w = rng.standard_normal((E, N, K))
    b = rng.standard_normal((R, N))
    nt = M.grouped_gemm_nt(a, w, off)
    nn = M.grouped_gemm_nn(b, w, off)
    wg = M.grouped_wgrad(b, a, off, E)
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            for n in range(N):
                assert abs(nt[r, n] - sum(a[r, kk] * w[e, n, kk] for kk in range(K))) < 1e-12
            for kk in range(K):
                assert abs(nn[r, kk] - sum(b[r, n] * w[e, n, kk] for n in range(N))) < 1e-12
        for n in range(N):
            for kk in range(K):
                want = sum(b[r, n] * a[r, kk] for r in range(off[e], off[e + 1]))
                assert abs(wg[e, n, kk] - want) < 1e-12


# ------------------------------------------------------------------------------ the layer

def _layer(T=24, E=3, d=32, F=16, k=2, seed=16):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, d), generator=g, dtype=torch.float64)
    w13 = torch.randn((E, 2 * F, d), generator=g, dtype=torch.float64) * 0.3
    w2 = torch.randn((E, d, F), generator=g, dtype=torch.float64) * 0.3
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).numpy()
    p = torch.softmax(torch.randn((T, k), generator=g, dtype=torch.float64), 1).numpy()
    dout = torch.randn((T, d), generator=g, dtype=torch.float64).numpy()
    return x.numpy(), w13.numpy(), w2.numpy(), idx, p, dout


def _fwd(x, w13, w2, idx, p):
    return M.moe_forward(Q.FMT_NVFP4, x, idx, p, w13, None, w2, None, quant=False, round_bf16=False)


def test_dense_special_case_matches_torch_swiglu_mlp():
    x, w13, w2, _, _, _ = _layer(E=1, k=1)
    T = x.shape[0]
    out = _fwd(x, w13, w2, np.zeros((T, 1), np.int64), np.ones((T, 1)))["out"]
    xt = torch.from_numpy(x)
    F_ = w2.shape[2]
    gate = xt @ torch.from_numpy(w13[0, :F_]).T
    up = xt @ torch.from_numpy(w13[0, F_:]).T
    want = (torch.nn.functional.silu(gate) * up) @ torch.from_numpy(w2[0]).T
    assert np.allclose(out, want.numpy(), rtol=1e-12, atol=1e-12)


def test_finite_differences_of_the_ste_free_layer():
    x, w13, w2, idx, p, dout = _layer()
    fwd = _fwd(x, w13, w2, idx, p)
    bwd = M.moe_dgrad(dout, p, fwd, round_bf16=False)
    dw13, dw2 = M.moe_weight_grads(fwd, bwd)

    def loss(x_, w13_, w2_, p_):
        return float((_fwd(x_, w13_, w2_, idx, p_)["out"] * dout).sum())

    h = 1e-6
    rng = np.random.default_rng(17)
    for arr, grad, name in ((x, bwd["dx"], "x"), (w13, dw13, "w13"), (w2, dw2, "w2"), (p, bwd["dprobs"], "p")):
        for _ in range(6):
            i = tuple(rng.integers(0, s) for s in arr.shape)
            args = {"x": x, "w13": w13, "w2": w2, "p": p}
            plus = {kk: v.copy() for kk, v in args.items()}
            minus = {kk: v.copy() for kk, v in args.items()}
            plus[name][i] += h
            minus[name][i] -= h
            fd = (loss(plus["x"], plus["w13"], plus["w2"], plus["p"])
                  - loss(minus["x"], minus["w13"], minus["w2"], minus["p"])) / (2 * h)
            assert abs(fd - grad[i]) <= 1e-6 * max(1.0, abs(fd)), (name, i, fd, grad[i])


# ---------------------------------------------------------------- scale-factored forward
# Per-row scaled formats: the forward GEMMs may contract the codes and apply the weight-row
# and activation-row scales to the sum (native low-precision MMA).  The pins tie that
# reading to the rounded fake-quant one.

def _bits(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _row_layer(fmt, T=40, E=3, d=64, F=32, k=2, seed=21, pow2=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, d), generator=g).clamp(-1.7, 1.7)
    w13 = torch.randn((E, 2 * F, d), generator=g) * 0.05
    w2 = torch.randn((E, d, F), generator=g) * 0.05
    qmax = Q.AMAX_DIV[fmt]
    if pow2:
        # every row's amax is qmax * 2^-8, so the dynamic scale fp32(amax / qmax) is 2^-8 exactly,
        # and the weight scales are powers of two: q * s is then exact in bf16
        x = x * (qmax / 448.0)
        x[:, 0] = torch.where(torch.rand(T, generator=g) < 0.5, -1.0, 1.0) * qmax * 2.0 ** -8
    def scales(w):
        amax = w.to(torch.bfloat16).float().abs().amax(-1, keepdim=True)
        s = amax / qmax
        if pow2:
            return torch.exp2(torch.round(torch.log2(s))).numpy()
        return (s * (1 + (torch.rand(s.shape, generator=g) * 0.2 - 0.1))).numpy()
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).numpy()
    p = torch.softmax(torch.randn((T, k), generator=g), 1).numpy()
    return dict(x=_bits(x), w13=_bits(w13), w2=_bits(w2), s13=scales(w13), s2=scales(w2), idx=idx, p=p)


@pytest.mark.parametrize("fmt", [Q.FMT_FP8_ROW, Q.FMT_W8A8])
def test_factored_values_round_to_the_fake_quant_values(fmt):
    L = _row_layer(fmt)
    wf = Q.fakequant_weight_factored(fmt, L["w13"], L["s13"])
    assert np.array_equal(Q.f64_to_bf16_bits(Q.round_bf16(Q.round_f32(wf))),
                          Q.f64_to_bf16_bits(Q.fakequant_weight(fmt, L["w13"], L["s13"])))
    x = Q.bf16_to_f64(L["x"])
    af = Q.fakequant_act_factored(fmt, x)
    assert np.array_equal(Q.round_bf16(Q.round_f32(af)), Q.fakequant_act(fmt, x))
    # the unrounded product is within the fp32-then-bf16 rounding of the stored value
    for f, r in ((wf, Q.fakequant_weight(fmt, L["w13"], L["s13"])), (af, Q.fakequant_act(fmt, x))):
        assert np.all(np.abs(f - r) <= 2.0 ** -8 * np.abs(f) + 1e-300)


@pytest.mark.parametrize("fmt", [Q.FMT_FP8_ROW, Q.FMT_W8A8])
def test_factored_fc1_equals_rounded_fc1_for_power_of_two_scales(fmt):
    L = _row_layer(fmt, pow2=True)
    args = (fmt, L["x"], L["idx"], L["p"], L["w13"], L["s13"], L["w2"], L["s2"])
    a = M.moe_forward(*args, factored=False)
    b = M.moe_forward(*args, factored=True)
    assert np.array_equal(a["z1"], b["z1"]) and np.array_equal(a["h"], b["h"])
    assert np.array_equal(a["hh"], b["hh"])
    # with random scales the two readings differ, by about the bf16 rounding of q * s
    L = _row_layer(fmt)
    args = (fmt, L["x"], L["idx"], L["p"], L["w13"], L["s13"], L["w2"], L["s2"])
    a = M.moe_forward(*args, factored=False, round_bf16=False)
    b = M.moe_forward(*args, factored=True, round_bf16=False)
    rms = np.sqrt(np.mean(a["z1"] ** 2))
    assert 0 < np.abs(a["z1"] - b["z1"]).max() < 2e-2 * rms


def test_factored_fc1_is_the_scaled_integer_code_product():
    """E4M3 values are multiples of 2^-9, so the code contraction is an exact integer dot
    product; fc1's unrounded output must be s_a[row] * s_w[n] times it (rows in the oracle's
    expert-grouped order, W13 rows as output columns)."""
    fmt = Q.FMT_FP8_ROW
    L = _row_layer(fmt)
    out = M.moe_forward(fmt, L["x"], L["idx"], L["p"], L["w13"], L["s13"], L["w2"], L["s2"],
                        factored=True, round_bf16=False)
    rt = out["route"]
    x = Q.bf16_to_f64(L["x"])
    sa = Q.round_f32(np.abs(x).max(axis=1) / 448.0)                        # [T]
    qa = np.rint(Q.q_e4m3(Q.round_f32(x / sa[:, None])) * 512).astype(np.int64)
    w = Q.bf16_to_f64(L["w13"])
    sw = L["s13"][..., 0].astype(np.float64)                               # [E, 2F]
    qw = np.rint(Q.q_e4m3(Q.round_f32(w / sw[..., None])) * 512).astype(np.int64)
    off = rt["offsets"]
    for e in range(w.shape[0]):
        rows = range(off[e], off[e + 1])
        toks = rt["row_token"][off[e]:off[e + 1]]
        want = (qa[toks] @ qw[e].T).astype(np.float64) / 2.0 ** 18 * sa[toks][:, None] * sw[e][None, :]
        got = out["z1"][off[e]:off[e + 1]]
        # fp64 rounding of the oracle's sum only (cancellation makes the error absolute)
        assert np.abs(got - want).max() <= 1e-12 * np.abs(want).max(), e


# ------------------------------------------------------------------------------ quantizer placement (hand-worked)

def _bf16_bits_of(values):
    return Q.f64_to_bf16_bits(np.asarray(values, dtype=np.float64))


def test_quantizer_placement_hand_worked_case():
    """nvfp4, one expert, one token, d = F = 16, p = 0.5: every stage worked out by hand.

    x = [6, 1.25, 0...]: block amax 6, s_a = 1, and 1.25 is a tie that rounds to the even
    code 1, so A1 = [6, 1, 0...] (the activation quantizer sits on fc1's input).
    Gate rows are [12, 0...] with s = 2 (12 / 2 = 6 on the grid): every gate is 6 * 12 = 72,
    and silu(72) = 72 exactly in fp64 (exp(-72) vanishes beside 1).  Up row i is [w_i, c_i, 0...]
    with a power-of-two scale that keeps it on the grid, so u_i = 6 w_i + c_i and H_i = 72 u_i.
    H's block amax is 72 * 36 = 2592, s_H = 432, and H_i / s_H = u_i / 6:
      u:      36   18   9    4.5   2.25   1.125  30   15   10.5  -18   0...
      H/s_H:  6    3    1.5  0.75  0.375  0.1875 5    2.5  1.75  -3    0
      code:   6    3    1.5  1     0.5    0      4    2    2     -3    0   (0.75, 5, 2.5, 1.75: ties to even)
      H_hat:  2592 1296 648  432   216    0      1728 864  864   -1296 0
    W2 is the identity (s = 1/4: 1 / 0.25 = 4 on the grid), so Y = H_hat and out = 0.5 H_hat.
    Had fc2 read H instead of H_hat, out[3] would be 162, not 216; had the activation
    quantizer been skipped on x, u_6 = 24 + 7.5 and H_hat_6 = 2592, not 1728."""
    d = F = 16
    x = np.zeros((1, d))
    x[0, :2] = [6.0, 1.25]
    w_up = [6, 3, 1.5, 0.75, 0.375, 0.1875, 4, 2, 1.5, -3] + [0] * 6
    c_up = [0, 0, 0, 0, 0, 0, 6, 3, 1.5, 0] + [0] * 6
    s_up = [1, 1, 1, 0.5, 0.25, 0.125, 1, 1, 1, 1] + [1] * 6
    w13 = np.zeros((1, 2 * F, d))
    s13 = np.ones((1, 2 * F, 1))
    w13[0, :F, 0] = 12.0
    s13[0, :F, 0] = 2.0
    w13[0, F:, 0] = w_up
    w13[0, F:, 1] = c_up
    s13[0, F:, 0] = s_up
    w2 = np.eye(d, F)[None]
    s2 = np.full((1, d, 1), 0.25)
    fwd = M.moe_forward(Q.FMT_NVFP4, _bf16_bits_of(x), np.zeros((1, 1), np.int64), np.array([[0.5]]),
                        _bf16_bits_of(w13), s13.astype(np.float32), _bf16_bits_of(w2), s2.astype(np.float32))
    a1 = np.zeros(d)
    a1[:2] = [6.0, 1.0]
    assert np.array_equal(fwd["a1"][0], a1)
    assert np.array_equal(fwd["w13h"], w13) and np.array_equal(fwd["w2h"], w2)
    u = np.array([36, 18, 9, 4.5, 2.25, 1.125, 30, 15, 10.5, -18] + [0] * 6)
    assert np.array_equal(fwd["z1"][0], np.concatenate([np.full(F, 72.0), u]))
    assert np.array_equal(fwd["h"][0], 72.0 * u)
    hh = np.array([2592, 1296, 648, 432, 216, 0, 1728, 864, 864, -1296] + [0] * 6, dtype=np.float64)
    assert np.array_equal(fwd["hh"][0], hh)
    assert np.array_equal(fwd["y"][0], hh)
    assert np.array_equal(fwd["out"][0], 0.5 * hh)

    # backward, straight through the activation quantizer: dout = 2 everywhere, so dY = 1 and dH = 1
    # (identity W2); at g = 72, sigmoid = 1 exactly, so dgate = dH * u and dup = dH * 72
    bwd = M.moe_dgrad(_bf16_bits_of(np.full((1, d), 2.0)), np.array([[0.5]]), fwd)
    assert np.array_equal(bwd["dy"][0], np.ones(d))
    assert np.array_equal(bwd["dz1"][0], np.concatenate([u, np.full(F, 72.0)]))
    # dA1[0] = 12 * sum(u) + 72 * sum(w_up) = 1300.5 + 1174.5 = 2475 -> bf16 (spacing 16) 2480;
    # dA1[1] = 72 * sum(c_up) = 756
    da1 = np.zeros(d)
    da1[:2] = [2480.0, 756.0]
    assert np.array_equal(bwd["da1"][0], da1) and np.array_equal(bwd["dx"][0], da1)


# ------------------------------------------------------------------------------ the fp32 quotient, bit by bit

def test_quotient_is_the_correctly_rounded_fp32_value():
    """oracle.quant._quotient(w, s) against exact rational arithmetic: the result is the fp32
    value nearest to w / s (ties to the even significand), on random pairs and on hard cases
    (scales with all-ones significands, powers of two, quotients at fp32 midpoints, results in
    fp32's subnormal range)."""
    from fractions import Fraction
    rng = np.random.default_rng(7)
    w = Q.bf16_to_f64(rng.integers(0, 1 << 16, 3000, dtype=np.uint32).astype(np.uint16))
    w = w[np.isfinite(w) & (np.abs(w) < 2.0 ** 100)]                                 # quotients stay finite
    s = rng.uniform(2.0 ** -20, 2.0 ** 4, 3000).astype(np.float32).astype(np.float64)
    ones = np.float32(np.nextafter(np.float32(2.0), np.float32(0.0)))          # 2 - 2^-23
    hard_s = [float(ones) * 2.0 ** e for e in range(-30, 10, 3)] + [2.0 ** e for e in range(-40, 20, 7)]
    hard_w = [1.0, 3.0, -5.0, 0.0078125, 1.5, 65280.0, -0.0]
    mid = []
    for k in range(40):  # w = s * (a fp32 midpoint): s = 2^-k exact, w/s has 25 significant bits
        m = (np.float64(np.float32(1.0 + k / 64.0)) + 2.0 ** -24) * 2.0 ** (k % 5)
        mid.append((m * 2.0 ** -k, 2.0 ** -k))
    pairs = list(zip(w, s)) + [(a, b) for a in hard_w for b in hard_s] + mid
    pairs += [(1.0, 2.0 ** 100), (-3.0, 2.0 ** 120), (2.0 ** -120, 3.0)]                  # subnormal results
    ws = np.array([p[0] for p in pairs])
    ss = np.array([p[1] for p in pairs])
    got = Q._quotient(ws, ss)
    for a, b, x in zip(ws, ss, got):
        if b == 0:
            continue
        q = Fraction(float(a)) / Fraction(float(b))
        x32 = np.float32(x)
        assert float(x32) == x, (a, b, x)                                            # lies on the fp32 grid
        err = abs(Fraction(float(x)) - q)
        for nb in (np.nextafter(x32, np.float32(np.inf)), np.nextafter(x32, np.float32(-np.inf))):
            if not np.isfinite(nb):
                continue
            e2 = abs(Fraction(float(nb)) - q)
            assert err <= e2, (a, b, x)                                              # nearest
            if err == e2:                                                            # a tie: even significand
                assert int(x32.view(np.uint32)) % 2 == 0, (a, b, x)
        if q == 0:
            assert np.signbit(x) == np.signbit(a)


# ------------------------------------------------------------------------------ deployed nvfp4 scales

def _deployed_rows():
    rows = _rows("nvfp4_deployed_scales.txt")
    return [tuple(float.fromhex(c) for c in r) for r in rows]


def test_deployed_scales_golden_weights():
    rows = _deployed_rows()
    v = np.array([r[0] for r in rows])
    want = np.array([r[1] for r in rows]) * 2.0 ** -10
    # one matrix [2, n] holding the blocks' scales (the 448 row fixes g = 2^-10), and the same
    # blocks split over two matrices of one stack: each matrix gets its own g
    s = np.stack([v, v[::-1]]) * 2.0 ** -10
    assert np.array_equal(Q.deploy_scales(s, axes=(-2, -1)), np.stack([want, want[::-1]]))
    stack = np.stack([s, 2.0 * s])[:, :, :]
    got = Q.effective_weight_scales(Q.FMT_NVFP4_E4M3, stack)
    assert np.array_equal(got[0], np.stack([want, want[::-1]]))
    assert np.array_equal(got[1], 2.0 * np.stack([want, want[::-1]]))
    # other formats use the learnable scales as they are
    assert np.array_equal(Q.effective_weight_scales(Q.FMT_NVFP4, stack), stack)


def test_deployed_scales_golden_activations():
    rows = _deployed_rows()
    n = len(rows)
    rng = np.random.default_rng(30)
    a = np.zeros((2, 16 * n))
    for b, (v, _, _) in enumerate(rows):
        amax = 6.0 * v * 2.0 ** -10
        blk = rng.uniform(-1, 1, 16) * amax * 0.9
        blk[(5 * b) % 16] = amax if b % 2 == 0 else -amax
        a[0, 16 * b:16 * b + 16] = blk
    a = Q.round_bf16(a)
    a[1] = a[0, ::-1]                                   # the same blocks, reversed: same scales
    assert np.array_equal(np.abs(a[0]).reshape(n, 16).max(-1), np.array([6.0 * r[0] * 2.0 ** -10 for r in rows]))
    s_a = Q.act_scale(Q.FMT_NVFP4_E4M3, a)
    want = np.repeat(np.array([r[1] for r in rows]) * 2.0 ** -10, 16)
    assert np.array_equal(s_a[0], want)
    assert np.array_equal(s_a[1], want[::-1])
    ah = Q.fakequant_act(Q.FMT_NVFP4_E4M3, a)
    top = np.abs(ah[0]).reshape(n, 16).max(-1)
    assert np.array_equal(top, np.array([r[2] for r in rows]) * 2.0 ** -10)
    # a block whose scale underflows E4M3 comes back as zeros
    for b, (v, e, _) in enumerate(rows):
        if e == 0:
            assert np.all(ah[0, 16 * b:16 * b + 16] == 0)


def test_deploy_scales_bruteforce_and_torch_cast():
    rng = np.random.default_rng(31)
    E, N, nb = 3, 24, 8
    s = (rng.lognormal(-5, 1.5, (E, N, nb))).astype(np.float32)
    s[0, 0, :3] = 0.0                                   # zero blocks
    s[1] = s[1] * np.float32(1e-30)                     # tiny scales: g far below 1
    s[2, 5, 2] = s[2].max() * np.float32(3.0)           # one outlier block: most others go subnormal
    s[2, 7, :4] *= np.float32(-1.0)                     # negative scales: rounded as their magnitude
    got = Q.deploy_scales(s.astype(np.float64), axes=(-2, -1))
    # torch: the same two fp32 steps with the float8_e4m3fn cast
    st = torch.from_numpy(s)
    g = st.abs().amax(dim=(-2, -1), keepdim=True) / 448.0
    want_t = ((st / g).to(torch.float8_e4m3fn).float() * g).double().numpy()
    assert np.array_equal(got, want_t)
    # brute force: s_q / g is the E4M3 value nearest fp32(s / g), ties to the even mantissa
    g64 = g.double().numpy()
    ratio = (st / g).double().numpy()
    grid, even = _e4m3_positive_grid()
    near = _brute_nearest(np.abs(ratio).reshape(-1), grid, even).reshape(ratio.shape) * np.sign(ratio)
    assert np.array_equal(got, Q.round_f32(near * g64))
    # the largest scale of each matrix is kept to fp32 accuracy; zeros stay zero
    for e in range(E):
        i = np.unravel_index(np.argmax(np.abs(s[e])), s[e].shape)
        assert abs(got[e][i] - s[e][i]) <= 2.0 ** -22 * s[e][i]
    assert np.all(got[0, 0, :3] == 0)
    # the negative ones are the magnitude's rounding, negated
    assert np.all(got[2, 7, :4] < 0)
    # rounding is monotone in s within a matrix
    for e in range(E):
        o = np.argsort(s[e].reshape(-1), kind="stable")
        assert np.all(np.diff(got[e].reshape(-1)[o]) >= 0)


def test_deploy_scales_all_zero_matrix_and_row():
    z = np.zeros((2, 4, 3))
    z[1, 2, 1] = 0.25
    got = Q.deploy_scales(z, axes=(-2, -1))
    assert np.all(got[0] == 0)
    assert got[1, 2, 1] == 0.25 and np.count_nonzero(got[1]) == 1
    a = np.zeros((2, 32))
    a[1, 3] = 1.5
    s_a = Q.act_scale(Q.FMT_NVFP4_E4M3, a)
    assert np.all(s_a[0] == 0) and np.all(s_a[1, 16:] == 0)
    assert np.all(s_a[1, :16] == Q.round_f32(Q.round_f32(Q.round_f32(1.5 / 6.0) / 448.0) * 448.0))
    assert np.array_equal(Q.fakequant_act(Q.FMT_NVFP4_E4M3, a)[1, 3], 1.5)


def test_deployed_activation_scales_against_torch_cast():
    """Format 6 activations: per 16-block fp32(amax / 6), rounded as deployed NVFP4 stores it under
    one fp32 scale per row (the row's largest block scale / 448), the E4M3 rounding done by torch's
    float8_e4m3fn cast; rows spanning many binades, a zero block and a zero row included."""
    rng = np.random.default_rng(32)
    a = rng.standard_normal((7, 256)) * 2.0 ** rng.integers(-20, 4, (7, 16)).repeat(16, axis=1)
    a[2, 32:48] = 0.0
    a[5] = 0.0
    a = Q.round_bf16(a)
    got = Q.act_scale(Q.FMT_NVFP4_E4M3, a)[:, ::16]
    at = torch.from_numpy(a).float()
    sb = at.abs().reshape(7, 16, 16).amax(-1) / 6.0
    g = sb.amax(-1, keepdim=True) / 448.0
    safe = torch.where(g == 0, torch.ones_like(g), g)
    sq = ((sb / safe).to(torch.float8_e4m3fn).float() * g)
    want = torch.where(g == 0, torch.zeros_like(sq), sq).double().numpy()
    assert np.array_equal(got, want)
    assert np.all(got[5] == 0) and got[2, 2] == 0
