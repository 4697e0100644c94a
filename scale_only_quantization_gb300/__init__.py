"""Python binding of the scale-only QAD MoE library (libqad_gb300.so, sm_103a).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
Each function below has the name and argument order of the C entry point in
include/qad.h; tensors are torch tensors on the current CUDA device (their data pointers
are passed), the stream defaults to torch's current stream, and a non-zero status
raises QADError.  There is no CPU fallback: if the library is not built the functions
raise.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqad_gb300.so")

QAD_OK, QAD_ERR_INVALID_ARG, QAD_ERR_UNSUPPORTED, QAD_ERR_WORKSPACE, QAD_ERR_CUDA, QAD_ERR_DEVICE = 0, -1, -2, -3, -4, -5
QAD_ERR_SCRATCH_LIMIT = -6
QAD_NOALLOC_MAX_EXPERTS, QAD_NOALLOC_MAX_PAIRS = 256, 262144
QAD_FMT_NVFP4, QAD_FMT_INT4_G128, QAD_FMT_FP8_ROW, QAD_FMT_NVFP4A16, QAD_FMT_W8A8, QAD_FMT_W4AFP8 = range(6)
QAD_FMT_NVFP4_E4M3 = 6
QAD_DEV_BAD_INDEX, QAD_DEV_DUP_INDEX, QAD_DEV_TIMEOUT = 1, 2, 4
QAD_FLAG_STASH_H, QAD_FLAG_NO_QUANT, QAD_FLAG_RECOMPUTE, QAD_FLAG_NATIVE_FP8 = 1, 2, 4, 8
QAD_FLAG_SMEM_DEQUANT, QAD_FLAG_DEQUANT_DUMP = 16, 32
VIEWS = ["HEADER", "OFFSETS", "COUNTS", "ROW_TOKEN", "ROW_SLOT", "ROW_OF", "W13_HAT", "W2_HAT", "A1", "Z1", "H",
         "H_HAT", "Y", "DY", "DZ1", "DA1", "XQ", "W13_CODES", "W2_CODES", "A1_CODES", "H_CODES", "A_SCALE",
         "H_SCALE", "S13_DEPLOYED", "S2_DEPLOYED"]
VIEW = {n: i for i, n in enumerate(VIEWS)}
KERNELS = 16

EXPORTS = ["qad_fakequant_fwd", "qad_moe_workspace_bytes", "qad_moe_fwd", "qad_moe_bwd_dgrad",
           "qad_moe_bwd_scalegrad", "qad_check_device_error", "qad_status_string", "qad_moe_debug_view",
           "qad_profile_enable", "qad_profile_reset", "qad_profile_read", "qad_kernel_name", "qad_launch_count",
           "qad_debug_quotient", "qad_route_permute_noalloc", "qad_debug_wait_timeout", "qad_moe_combine",
           "qad_nvfp4_deploy_scales"]


class QADError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


class MoEShape(ctypes.Structure):
    """qad_moe_shape: T tokens, hidden d, expert FFN F, E experts, top-k, format, flags."""
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int64), ("F", ctypes.c_int64), ("E", ctypes.c_int64),
                ("topk", ctypes.c_int32), ("fmt", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SHAPE = ctypes.POINTER(MoEShape)


def lib():
    """Load libqad_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libqad_gb300.so is not built: run `python -m scale_only_quantization_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "qad_fakequant_fwd": (ctypes.c_int, [ctypes.c_int, _P, _P, _P, _I64, _I64, _I64, _P]),
            "qad_moe_workspace_bytes": (ctypes.c_size_t, [_SHAPE]),
            "qad_moe_fwd": (ctypes.c_int, [_SHAPE, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
            "qad_moe_bwd_dgrad": (ctypes.c_int, [_SHAPE, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
            "qad_moe_bwd_scalegrad": (ctypes.c_int, [_SHAPE, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P,
                                                     ctypes.c_size_t, _P]),
            "qad_check_device_error": (ctypes.c_int, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
            "qad_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "qad_moe_debug_view": (ctypes.c_int, [_SHAPE, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t),
                                                  ctypes.POINTER(ctypes.c_int64)]),
            "qad_profile_enable": (ctypes.c_int, [ctypes.c_int]),
            "qad_profile_reset": (ctypes.c_int, []),
            "qad_profile_read": (ctypes.c_int, [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int64),
                                                ctypes.c_int]),
            "qad_kernel_name": (ctypes.c_char_p, [ctypes.c_int]),
            "qad_launch_count": (ctypes.c_int64, []),
            "qad_debug_quotient": (ctypes.c_int, [_P, _P, _P, _P, _I64, ctypes.c_int32, _P]),
            "qad_debug_wait_timeout": (ctypes.c_int, [_P, _I64, _P]),
            "qad_route_permute_noalloc": (ctypes.c_int, [_P, _I64, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P,
                                                         _P, _P, _P]),
            "qad_moe_combine": (ctypes.c_int, [_P, _P, _P, _P, _I64, ctypes.c_int32, _I64, _P]),
            "qad_nvfp4_deploy_scales": (ctypes.c_int, [_P, _P, _I64, _I64, _P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def status_string(status):
    return lib().qad_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc, where):
    if rc != QAD_OK:
        raise QADError(rc, where)
    return rc


def shape(T, d, F, E, topk, fmt, flags=0):
    return MoEShape(int(T), int(d), int(F), int(E), int(topk), int(fmt), int(flags), 0)


def qad_fakequant_fwd(fmt, w, scale, w_hat, E, N, K, stream=None):
    return _check(lib().qad_fakequant_fwd(int(fmt), _ptr(w), _ptr(scale), _ptr(w_hat), int(E), int(N), int(K),
                                          _stream(stream)), "qad_fakequant_fwd")


def qad_nvfp4_deploy_scales(s, s_q, n_mat, per_mat, stream=None):
    return _check(lib().qad_nvfp4_deploy_scales(_ptr(s), _ptr(s_q), int(n_mat), int(per_mat), _stream(stream)),
                  "qad_nvfp4_deploy_scales")


def qad_moe_workspace_bytes(s):
    return int(lib().qad_moe_workspace_bytes(ctypes.byref(s)))


def qad_moe_fwd(s, x, topk_idx, topk_w, w13, s13, w2, s2, out, ws, stream=None):
    return _check(lib().qad_moe_fwd(ctypes.byref(s), _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(w13), _ptr(s13),
                                    _ptr(w2), _ptr(s2), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                    _stream(stream)), "qad_moe_fwd")


def qad_moe_bwd_dgrad(s, dout, topk_w, w13, s13, w2, s2, dx, dprobs, ws, stream=None):
    return _check(lib().qad_moe_bwd_dgrad(ctypes.byref(s), _ptr(dout), _ptr(topk_w), _ptr(w13), _ptr(s13), _ptr(w2),
                                          _ptr(s2), _ptr(dx), _ptr(dprobs), _ptr(ws),
                                          ws.numel() * ws.element_size(), _stream(stream)), "qad_moe_bwd_dgrad")


def qad_moe_bwd_scalegrad(s, w13, s13, w2, s2, ds13, ds2, accumulate, ws, stream=None):
    return _check(lib().qad_moe_bwd_scalegrad(ctypes.byref(s), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), _ptr(ds13),
                                              _ptr(ds2), int(accumulate), _ptr(ws), ws.numel() * ws.element_size(),
                                              _stream(stream)), "qad_moe_bwd_scalegrad")


def qad_check_device_error(ws, stream=None):
    """Returns the device error word (0 = none); synchronises the stream."""
    code = ctypes.c_int32(0)
    rc = lib().qad_check_device_error(_ptr(ws), _stream(stream), ctypes.byref(code))
    if rc not in (QAD_OK, QAD_ERR_DEVICE):
        raise QADError(rc, "qad_check_device_error")
    return int(code.value)


def qad_moe_debug_view(s, which):
    """(byte offset, element count) of workspace region `which` (a VIEWS name or index)."""
    off, n = ctypes.c_size_t(0), ctypes.c_int64(0)
    w = VIEW[which] if isinstance(which, str) else int(which)
    _check(lib().qad_moe_debug_view(ctypes.byref(s), w, ctypes.byref(off), ctypes.byref(n)), "qad_moe_debug_view")
    return int(off.value), int(n.value)


def qad_profile_enable(on):
    return _check(lib().qad_profile_enable(int(bool(on))), "qad_profile_enable")


def qad_profile_reset():
    return _check(lib().qad_profile_reset(), "qad_profile_reset")


def qad_profile_read():
    """{kernel name: (total ms, launches)} since the last reset; synchronises the device."""
    ms = (ctypes.c_float * KERNELS)()
    n = (ctypes.c_int64 * KERNELS)()
    _check(lib().qad_profile_read(ms, n, KERNELS), "qad_profile_read")
    return {lib().qad_kernel_name(i).decode(): (float(ms[i]), int(n[i])) for i in range(KERNELS)}


def qad_kernel_name(i):
    return lib().qad_kernel_name(int(i)).decode()


def qad_launch_count():
    return int(lib().qad_launch_count())


def qad_debug_quotient(w, s, x_fast, x_ieee, n, mode=0, stream=None):
    return _check(lib().qad_debug_quotient(_ptr(w), _ptr(s), _ptr(x_fast), _ptr(x_ieee), int(n), int(mode),
                                           _stream(stream)), "qad_debug_quotient")


def qad_route_permute_noalloc(topk_idx, T, topk, E, row_token, row_slot, row_of, offsets, counts, header,
                              stream=None):
    """Routing maps without any device allocation by the library (see include/qad.h)."""
    return _check(lib().qad_route_permute_noalloc(_ptr(topk_idx), int(T), int(topk), int(E), _ptr(row_token),
                                                  _ptr(row_slot), _ptr(row_of), _ptr(offsets), _ptr(counts),
                                                  _ptr(header), _stream(stream)), "qad_route_permute_noalloc")


def qad_moe_combine(rows, row_of, p, out, T, topk, d, stream=None):
    return _check(lib().qad_moe_combine(_ptr(rows), _ptr(row_of), _ptr(p), _ptr(out), int(T), int(topk), int(d),
                                        _stream(stream)), "qad_moe_combine")


def qad_debug_wait_timeout(err_word, budget_cycles, stream=None):
    return _check(lib().qad_debug_wait_timeout(_ptr(err_word), int(budget_cycles), _stream(stream)),
                  "qad_debug_wait_timeout")


def workspace_view(ws, s, which, dtype):
    """A torch view of workspace region `which` with element type `dtype` (flat)."""
    import torch
    off, n = qad_moe_debug_view(s, which)
    itemsize = torch.tensor([], dtype=dtype).element_size()
    return ws.view(torch.uint8)[off: off + n * itemsize].view(dtype)
