"""The C ABI library loads without a GPU, exports every function include/qad.h declares,
and rejects bad arguments on the host before touching CUDA (CPU only)."""
import ctypes
import os
import re

import pytest

import scale_only_quantization_gb300 as Q
from scale_only_quantization_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return Q.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "qad.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qad_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_layer_calls():
    names = _declared()
    for n in ("qad_fakequant_fwd", "qad_moe_fwd", "qad_moe_bwd_dgrad", "qad_moe_bwd_scalegrad"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(Q.EXPORTS) == _declared()


def test_workspace_size_and_views(lib):
    s = Q.shape(512, 256, 128, 4, 2, Q.QAD_FMT_NVFP4)
    ws = Q.qad_moe_workspace_bytes(s)
    assert ws > 0 and ws % 1024 == 0
    off, n = Q.qad_moe_debug_view(s, "W13_HAT")
    assert off % 1024 == 0 and n == 4 * 256 * 256
    off2, n2 = Q.qad_moe_debug_view(s, "ROW_TOKEN")
    Rmax = (512 * 2 + 127 * 4 + 127) // 128 * 128
    assert n2 == Rmax
    for v in range(len(Q.VIEWS)):
        o, k = Q.qad_moe_debug_view(s, v)
        assert o + k <= ws


_ELEM = dict(HEADER=4, OFFSETS=4, COUNTS=4, ROW_TOKEN=4, ROW_SLOT=4, ROW_OF=4, W13_HAT=2, W2_HAT=2, A1=2, Z1=2,
             H=2, H_HAT=2, Y=2, DY=2, DZ1=2, DA1=2, XQ=2, W13_CODES=1, W2_CODES=1, A1_CODES=1, H_CODES=1,
             A_SCALE=4, H_SCALE=4, S13_DEPLOYED=4, S2_DEPLOYED=4)
_ALL_FMTS = [Q.QAD_FMT_NVFP4, Q.QAD_FMT_INT4_G128, Q.QAD_FMT_FP8_ROW, Q.QAD_FMT_NVFP4A16, Q.QAD_FMT_W8A8,
             Q.QAD_FMT_W4AFP8, Q.QAD_FMT_NVFP4_E4M3]


def _layouts():
    for T, d, F, E, k in [(0, 256, 128, 4, 2), (1, 256, 128, 1, 1), (7, 512, 384, 3, 3), (512, 256, 128, 4, 2),
                          (4096, 2048, 768, 32, 8), (16384, 2048, 768, 128, 8), (1000, 256, 1024, 16, 4)]:
        for fmt in _ALL_FMTS:
            flag_sets = [0, Q.QAD_FLAG_STASH_H, Q.QAD_FLAG_RECOMPUTE, Q.QAD_FLAG_NO_QUANT, Q.QAD_FLAG_SMEM_DEQUANT,
                         Q.QAD_FLAG_SMEM_DEQUANT | Q.QAD_FLAG_DEQUANT_DUMP,
                         Q.QAD_FLAG_SMEM_DEQUANT | Q.QAD_FLAG_RECOMPUTE]
            if fmt == Q.QAD_FMT_FP8_ROW:
                flag_sets += [Q.QAD_FLAG_NATIVE_FP8, Q.QAD_FLAG_NATIVE_FP8 | Q.QAD_FLAG_RECOMPUTE]
            for flags in flag_sets:
                yield T, d, F, E, k, fmt, flags


def test_workspace_views_lie_inside_and_do_not_overlap(lib):
    """Every stage view is 1 KB aligned, lies inside the workspace in bytes, and no two views share
    bytes except Z1 and Y under QAD_FLAG_RECOMPUTE when Y's rows hold Z1's (d >= 2F)."""
    n_cases = 0
    for T, d, F, E, k, fmt, flags in _layouts():
        s = Q.shape(T, d, F, E, k, fmt, flags)
        ws = Q.qad_moe_workspace_bytes(s)
        assert ws > 0 and ws % 1024 == 0
        spans = []
        for name in Q.VIEWS:
            off, n = Q.qad_moe_debug_view(s, name)
            assert n >= 0
            if n == 0:
                continue
            assert off % 1024 == 0, (name, off)
            end = off + n * _ELEM[name]
            assert end <= ws, (name, off, n, ws)
            spans.append((off, end, name))
        spans.sort()
        aliased = (flags & Q.QAD_FLAG_RECOMPUTE) and d >= 2 * F
        for (a0, a1, an), (b0, b1, bn) in zip(spans, spans[1:]):
            if b0 < a1:
                assert aliased and {an, bn} == {"Z1", "Y"}, (an, bn, T, d, F, E, k, fmt, flags)
        names = [n for _, _, n in spans]
        if flags & Q.QAD_FLAG_NATIVE_FP8:
            per_token = {"A_SCALE"} if T > 0 else set()  # one activation scale per token
            assert {"W13_CODES", "W2_CODES", "A1_CODES", "H_CODES", "H_SCALE"} | per_token <= set(names)
        else:
            assert not {"W13_CODES", "W2_CODES", "A1_CODES", "H_CODES", "A_SCALE", "H_SCALE"} & set(names)
        n_cases += 1
    assert n_cases > 150


@pytest.mark.parametrize("bad, status", [
    (dict(d=200), Q.QAD_ERR_UNSUPPORTED),          # not a multiple of 16
    (dict(d=272, fmt=1), Q.QAD_ERR_UNSUPPORTED),   # INT4 weights: multiples of 128
    (dict(F=104), Q.QAD_ERR_UNSUPPORTED),
    (dict(topk=5, E=4), Q.QAD_ERR_UNSUPPORTED),
    (dict(E=2000), Q.QAD_ERR_UNSUPPORTED),
    (dict(fmt=7), Q.QAD_ERR_INVALID_ARG),
    (dict(T=-1), Q.QAD_ERR_INVALID_ARG),
])
def test_bad_shapes_rejected_on_host(lib, bad, status):
    kw = dict(T=512, d=256, F=128, E=4, topk=2, fmt=0)
    kw.update(bad)
    s = Q.shape(**kw)
    assert Q.qad_moe_workspace_bytes(s) == 0
    rc = lib.qad_moe_fwd(ctypes.byref(s), None, None, None, None, None, None, None, None, None, 0, None)
    assert rc == status


def test_null_and_misaligned_pointers_rejected_before_launch(lib):
    s = Q.shape(512, 256, 128, 4, 2, Q.QAD_FMT_NVFP4)
    P = ctypes.c_void_p
    assert lib.qad_moe_fwd(ctypes.byref(s), None, None, None, None, None, None, None, None, None, 0,
                           None) == Q.QAD_ERR_INVALID_ARG
    ws = P(1 << 20)
    need = Q.qad_moe_workspace_bytes(s)
    assert lib.qad_moe_fwd(ctypes.byref(s), P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16), ws,
                           need - 1, None) == Q.QAD_ERR_WORKSPACE
    assert lib.qad_moe_fwd(ctypes.byref(s), P(8), P(16), P(16), P(16), P(16), P(16), P(16), P(16), ws, need,
                           None) == Q.QAD_ERR_INVALID_ARG
    assert lib.qad_fakequant_fwd(0, P(16), P(16), P(16), 1, 4, 24, None) == Q.QAD_ERR_UNSUPPORTED
    assert lib.qad_fakequant_fwd(1, P(16), P(16), P(16), 1, 4, 64, None) == Q.QAD_ERR_UNSUPPORTED
    assert lib.qad_fakequant_fwd(0, P(16), P(16), P(17), 1, 4, 64, None) == Q.QAD_ERR_INVALID_ARG
    assert lib.qad_fakequant_fwd(0, None, None, None, 0, 4, 64, None) == Q.QAD_OK   # empty: nothing to do


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5):
        assert Q.status_string(st)
    assert Q.qad_kernel_name(4) == "gemm_fc1_swiglu_aq"


def test_recompute_flag_shares_z1_with_y(lib):
    """QAD_FLAG_RECOMPUTE: Z1 is not kept between the calls, so when d >= 2F it lives in Y's
    region and the workspace is smaller by exactly that region; unknown flag bits are rejected."""
    T, d, F, E, k = 512, 256, 128, 4, 2
    Rmax = (T * k + 127 * E + 127) // 128 * 128
    s0 = Q.shape(T, d, F, E, k, Q.QAD_FMT_NVFP4)
    s1 = Q.shape(T, d, F, E, k, Q.QAD_FMT_NVFP4, Q.QAD_FLAG_RECOMPUTE)
    assert Q.qad_moe_workspace_bytes(s0) - Q.qad_moe_workspace_bytes(s1) == 2 * Rmax * 2 * F
    assert Q.qad_moe_debug_view(s1, "Z1")[0] == Q.qad_moe_debug_view(s1, "Y")[0]
    assert Q.qad_moe_debug_view(s0, "Z1")[0] != Q.qad_moe_debug_view(s0, "Y")[0]
    # d < 2F: Y is too small to hold Z1, nothing is shared
    s2 = Q.shape(T, d, 256, E, k, Q.QAD_FMT_NVFP4, Q.QAD_FLAG_RECOMPUTE)
    s3 = Q.shape(T, d, 256, E, k, Q.QAD_FMT_NVFP4)
    assert Q.qad_moe_workspace_bytes(s2) == Q.qad_moe_workspace_bytes(s3)
    assert Q.qad_moe_workspace_bytes(Q.shape(T, d, F, E, k, Q.QAD_FMT_NVFP4, 8)) == 0


def test_native_fp8_flag_adds_codes_and_row_scales(lib):
    T, d, F, E, k = 512, 256, 128, 4, 2
    Rmax = (T * k + 127 * E + 127) // 128 * 128
    base = Q.shape(T, d, F, E, k, Q.QAD_FMT_FP8_ROW)
    nat = Q.shape(T, d, F, E, k, Q.QAD_FMT_FP8_ROW, Q.QAD_FLAG_NATIVE_FP8)
    up = lambda n: (n + 1023) // 1024 * 1024
    extra = up(E * 2 * F * d) + up(E * d * F) + up(Rmax * d) + up(Rmax * F) + up(4 * T) + up(4 * Rmax)
    assert Q.qad_moe_workspace_bytes(nat) - Q.qad_moe_workspace_bytes(base) == extra
    for name, n in (("W13_CODES", E * 2 * F * d), ("W2_CODES", E * d * F), ("A1_CODES", Rmax * d),
                    ("H_CODES", Rmax * F), ("A_SCALE", T), ("H_SCALE", Rmax)):
        assert Q.qad_moe_debug_view(nat, name)[1] == n
        assert Q.qad_moe_debug_view(base, name)[1] == 0
    for fmt in (Q.QAD_FMT_NVFP4, Q.QAD_FMT_INT4_G128, Q.QAD_FMT_W8A8, Q.QAD_FMT_W4AFP8):
        assert Q.qad_moe_workspace_bytes(Q.shape(T, d, F, E, k, fmt, Q.QAD_FLAG_NATIVE_FP8)) == 0


def _enum(prefix):
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "qad.h")).read(), flags=re.S)
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(%s[A-Z0-9_]+)\s*=\s*(-?\d+)" % prefix, text)}


def test_binding_constants_match_the_header(lib):
    views = _enum("QAD_VIEW_")
    count = views.pop("QAD_VIEW_COUNT")
    assert count == len(Q.VIEWS)
    assert {"QAD_VIEW_" + n: i for i, n in enumerate(Q.VIEWS)} == views
    kernels = _enum("QAD_K_")
    assert kernels.pop("QAD_K_COUNT") == Q.KERNELS
    assert sorted(kernels.values()) == list(range(Q.KERNELS))
    assert len({Q.qad_kernel_name(i) for i in range(Q.KERNELS)}) == Q.KERNELS
    flags = _enum("QAD_FLAG_")
    assert flags == {"QAD_FLAG_STASH_H": Q.QAD_FLAG_STASH_H, "QAD_FLAG_NO_QUANT": Q.QAD_FLAG_NO_QUANT,
                     "QAD_FLAG_RECOMPUTE": Q.QAD_FLAG_RECOMPUTE, "QAD_FLAG_NATIVE_FP8": Q.QAD_FLAG_NATIVE_FP8,
                     "QAD_FLAG_SMEM_DEQUANT": Q.QAD_FLAG_SMEM_DEQUANT,
                     "QAD_FLAG_DEQUANT_DUMP": Q.QAD_FLAG_DEQUANT_DUMP}
    fmts = _enum("QAD_FMT_")
    assert fmts == {"QAD_FMT_NVFP4": 0, "QAD_FMT_INT4_G128": 1, "QAD_FMT_FP8_ROW": 2, "QAD_FMT_NVFP4A16": 3,
                    "QAD_FMT_W8A8": 4, "QAD_FMT_W4AFP8": 5, "QAD_FMT_NVFP4_E4M3": 6}
    assert Q.QAD_FMT_NVFP4_E4M3 == 6


def test_smem_dequant_flag_drops_the_weight_copies(lib):
    """QAD_FLAG_SMEM_DEQUANT: no W13_hat / W2_hat regions (E * 3F * d bf16 less), unless
    QAD_FLAG_DEQUANT_DUMP keeps them for testing; invalid with the teacher pass, the native fp8
    path, or the dump flag alone."""
    T, d, F, E, k = 16384, 2048, 768, 128, 8
    for fmt in _ALL_FMTS:
        base = Q.qad_moe_workspace_bytes(Q.shape(T, d, F, E, k, fmt))
        dq = Q.qad_moe_workspace_bytes(Q.shape(T, d, F, E, k, fmt, Q.QAD_FLAG_SMEM_DEQUANT))
        dump = Q.qad_moe_workspace_bytes(
            Q.shape(T, d, F, E, k, fmt, Q.QAD_FLAG_SMEM_DEQUANT | Q.QAD_FLAG_DEQUANT_DUMP))
        assert base - dq >= 2 * E * 3 * F * d and dump == base
        s = Q.shape(T, d, F, E, k, fmt, Q.QAD_FLAG_SMEM_DEQUANT)
        assert Q.qad_moe_debug_view(s, "W13_HAT")[1] == 0 and Q.qad_moe_debug_view(s, "W2_HAT")[1] == 0
    for flags in (Q.QAD_FLAG_SMEM_DEQUANT | Q.QAD_FLAG_NO_QUANT, Q.QAD_FLAG_DEQUANT_DUMP,
                  Q.QAD_FLAG_SMEM_DEQUANT | Q.QAD_FLAG_NATIVE_FP8):
        assert Q.qad_moe_workspace_bytes(Q.shape(T, d, F, E, k, Q.QAD_FMT_FP8_ROW, flags)) == 0


def test_combine_rejects_bad_arguments_before_launch(lib):
    """qad_moe_combine: d % 16, 1 <= topk <= 32, T >= 0 and 16-byte aligned pointers are checked on
    the host (no GPU is touched); T = 0 is a no-op."""
    P = 1 << 20  # a 16-byte aligned stand-in address; nothing is launched for invalid arguments
    assert lib.qad_moe_combine(P, P, P, P, 4, 2, 24, None) == Q.QAD_ERR_INVALID_ARG      # d % 16
    assert lib.qad_moe_combine(P, P, P, P, 4, 33, 32, None) == Q.QAD_ERR_INVALID_ARG     # topk > 32
    assert lib.qad_moe_combine(P + 4, P, P, P, 4, 2, 32, None) == Q.QAD_ERR_INVALID_ARG  # misaligned
    assert lib.qad_moe_combine(None, P, P, P, 4, 2, 32, None) == Q.QAD_ERR_INVALID_ARG
    assert lib.qad_moe_combine(None, None, None, None, 0, 2, 32, None) == Q.QAD_OK
    assert lib.qad_moe_combine(P, P, P, P, -1, 2, 32, None) == Q.QAD_ERR_INVALID_ARG


def test_shape_contract(lib):
    """d and F: multiples of 16, of 128 for the INT4 formats; the E4M3 tensor path and the in-GEMM
    dequant keep whole tiles (d % 256, F % 128).  Others are refused on the host."""
    ok = lambda T, d, F, fmt, flags=0: Q.qad_moe_workspace_bytes(Q.shape(T, d, F, 4, 2, fmt, flags)) > 0  # noqa
    for fmt in (Q.QAD_FMT_NVFP4, Q.QAD_FMT_FP8_ROW, Q.QAD_FMT_NVFP4A16, Q.QAD_FMT_W8A8, Q.QAD_FMT_NVFP4_E4M3):
        assert ok(64, 272, 144, fmt) and ok(64, 2880, 2880, fmt) and ok(64, 16, 16, fmt)
        assert not ok(64, 264, 144, fmt) and not ok(64, 272, 136, fmt)
    for fmt in (Q.QAD_FMT_INT4_G128, Q.QAD_FMT_W4AFP8):
        assert ok(64, 384, 384, fmt) and ok(64, 128, 128, fmt)
        assert not ok(64, 272, 384, fmt) and not ok(64, 384, 144, fmt)
    assert not ok(64, 272, 144, Q.QAD_FMT_FP8_ROW, Q.QAD_FLAG_NATIVE_FP8)
    assert ok(64, 512, 256, Q.QAD_FMT_FP8_ROW, Q.QAD_FLAG_NATIVE_FP8)
    assert not ok(64, 2880, 2880, Q.QAD_FMT_NVFP4, Q.QAD_FLAG_SMEM_DEQUANT)
    s = Q.shape(64, 264, 144, 4, 2, Q.QAD_FMT_NVFP4)
    ws = ctypes.c_void_p(1 << 20)
    assert lib.qad_moe_fwd(ctypes.byref(s), None, None, None, None, None, None, None, None, ws, 1 << 30,
                           None) == Q.QAD_ERR_UNSUPPORTED


def test_deployed_nvfp4_layout_and_host_checks(lib):
    """QAD_FMT_NVFP4_E4M3 keeps the deployed weight scales in the workspace (E * 2F * d / 16 and
    E * d * F / 16 fp32 more than nvfp4); the deploy entry point checks its sizes and pointers on
    the host, and the standalone fake-quant refuses the format (it needs the deployed scales)."""
    T, d, F, E, k = 512, 256, 128, 4, 2
    up = lambda n: (n + 1023) // 1024 * 1024  # noqa: E731
    base = Q.qad_moe_workspace_bytes(Q.shape(T, d, F, E, k, Q.QAD_FMT_NVFP4))
    dep = Q.shape(T, d, F, E, k, Q.QAD_FMT_NVFP4_E4M3)
    # the deployed scales, and 2E matrix amax words plus 2E (g, 1/g) pairs
    assert Q.qad_moe_workspace_bytes(dep) - base == up(4 * E * 2 * F * d // 16) + up(4 * E * d * F // 16) + up(24 * E)
    assert Q.qad_moe_debug_view(dep, "S13_DEPLOYED")[1] == E * 2 * F * d // 16
    assert Q.qad_moe_debug_view(dep, "S2_DEPLOYED")[1] == E * d * F // 16
    assert Q.qad_moe_debug_view(Q.shape(T, d, F, E, k, Q.QAD_FMT_NVFP4), "S13_DEPLOYED")[1] == 0
    P = 1 << 20  # a 16-byte aligned stand-in address; nothing is launched for these
    assert lib.qad_nvfp4_deploy_scales(P, P, 4, 6, None) == Q.QAD_ERR_INVALID_ARG      # per_mat % 4
    assert lib.qad_nvfp4_deploy_scales(P, P, -1, 8, None) == Q.QAD_ERR_INVALID_ARG
    assert lib.qad_nvfp4_deploy_scales(P, P, 4, 0, None) == Q.QAD_ERR_INVALID_ARG
    assert lib.qad_nvfp4_deploy_scales(P + 4, P, 4, 8, None) == Q.QAD_ERR_INVALID_ARG  # misaligned
    assert lib.qad_nvfp4_deploy_scales(None, P, 4, 8, None) == Q.QAD_ERR_INVALID_ARG
    assert lib.qad_nvfp4_deploy_scales(None, None, 0, 8, None) == Q.QAD_OK
    assert lib.qad_fakequant_fwd(Q.QAD_FMT_NVFP4_E4M3, P, P, P, 1, 16, 64, None) == Q.QAD_ERR_UNSUPPORTED
    assert lib.qad_fakequant_fwd(7, P, P, P, 1, 16, 64, None) == Q.QAD_ERR_INVALID_ARG
