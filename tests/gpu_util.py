"""Helpers of the GPU parity tests: run the layer through the C ABI, pull workspace
stages back to the host, and the tolerance rules.

Tolerances: floating-point layer outputs and input gradients must satisfy
|gpu - oracle| <= 2e-2 * RMS(oracle) + 2^-8 * |oracle| element by element: the stated
2e-2 x RMS bound on the arithmetic, plus the rounding of each stored bf16 value
(at most half a bf16 ulp, i.e. 2^-8 of its magnitude), which on its own exceeds
2e-2 x RMS for any element larger than ~5 x RMS.  Scale gradients: relative L2 <= 1e-2.
Quantized values (fake-quant weights/activations), routing maps and the bf16(p * dout)
rows are compared bit for bit.  A tolerance check compares the GPU's stored bf16 value
with the oracle's value BEFORE the oracle's own final bf16 rounding: the GPU rounds an
fp32 sum and the oracle an fp64 one, so near a rounding midpoint the two stored values
may legitimately differ by one bf16 ulp, which for an element far above the RMS exceeds
2e-2 x RMS on its own.
"""
import numpy as np
import torch

import scale_only_quantization_gb300 as Q
from oracle import moe as OM
from oracle import quant as OQ
import synth

MAXABS_REL = 2e-2
BF16_HALF_ULP_REL = 2.0 ** -8
SCALE_REL_L2 = 1e-2


def bits(t):
    return synth.to_numpy_bits(t)


def vals(t):
    """bf16 tensor -> fp64 NumPy values (host copy)."""
    return OQ.bf16_to_f64(bits(t))


E2E_REL_L2 = 1e-3  # end-to-end (oracle from the raw inputs) relative L2 bound of out and dx


def rel_l2(gpu, ref):
    """||gpu - ref||_2 / ||ref||_2 over all elements."""
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    return float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30))


def assert_close(gpu, ref, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.isfinite(gpu)), what
    diff = np.abs(gpu - ref)
    excess = diff - (MAXABS_REL * rms + BF16_HALF_ULP_REL * np.abs(ref))
    i = int(np.argmax(excess))
    assert excess.flat[i] <= 1e-30, "%s: |err| %.3e at |ref| %.3e exceeds %.1e x rms %.3e + 2^-8 |ref|" % (
        what, diff.flat[i], abs(ref.flat[i]), MAXABS_REL, rms)
    return float(diff.max()) / max(rms, 1e-30)


def assert_scale_grad(gpu, ref, what):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    nrm = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(gpu - ref)) / max(nrm, 1e-30)
    if nrm == 0.0:
        assert np.all(gpu == 0.0), what
        return 0.0
    assert rel <= SCALE_REL_L2, "%s: relative L2 error %.3e > %.1e" % (what, rel, SCALE_REL_L2)
    return rel


class Run:
    """One fwd + dgrad + scalegrad of the layer through the C ABI, on `inp` (synth dict)."""

    def __init__(self, inp, flags=0, accumulate=0, ds_init=None, dprobs=True, zero_ws=False):
        self.inp = inp
        dev = inp["x"].device
        self.s = Q.shape(inp["T"], inp["d"], inp["F"], inp["E"], inp["topk"], inp["fmt"], flags)
        nb = Q.qad_moe_workspace_bytes(self.s)
        assert nb > 0
        self.ws = (torch.zeros if zero_ws else torch.empty)(nb, dtype=torch.uint8, device=dev)
        T, d, k = inp["T"], inp["d"], inp["topk"]
        self.out = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device=dev)
        self.dx = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device=dev)
        self.dprobs = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev) if dprobs else None
        if ds_init is None:
            self.ds13 = torch.full_like(inp["s13"], float("nan"))
            self.ds2 = torch.full_like(inp["s2"], float("nan"))
        else:
            self.ds13, self.ds2 = ds_init[0].clone(), ds_init[1].clone()
        Q.qad_moe_fwd(self.s, inp["x"], inp["topk_idx"], inp["topk_w"], inp["w13"], inp["s13"], inp["w2"], inp["s2"],
                      self.out, self.ws)
        Q.qad_moe_bwd_dgrad(self.s, inp["dout"], inp["topk_w"], inp["w13"], inp["s13"], inp["w2"], inp["s2"], self.dx,
                            self.dprobs, self.ws)
        Q.qad_moe_bwd_scalegrad(self.s, inp["w13"], inp["s13"], inp["w2"], inp["s2"], self.ds13, self.ds2, accumulate,
                                self.ws)
        self.error = Q.qad_check_device_error(self.ws)
        torch.cuda.synchronize()

    def view(self, name, dtype):
        return Q.workspace_view(self.ws, self.s, name, dtype)

    def routing(self):
        """Padded row maps on the host, and the mask of real (non-padding) rows."""
        T, k, E = self.inp["T"], self.inp["topk"], self.inp["E"]
        hdr = self.view("HEADER", torch.int32).cpu().numpy()
        rpad = int(hdr[2])
        row_token = self.view("ROW_TOKEN", torch.int32)[:rpad].cpu().numpy().astype(np.int64)
        row_slot = self.view("ROW_SLOT", torch.int32)[:rpad].cpu().numpy().astype(np.int64)
        row_of = self.view("ROW_OF", torch.int32).cpu().numpy().astype(np.int64).reshape(T, k)
        offs = self.view("OFFSETS", torch.int32).cpu().numpy().astype(np.int64)
        counts = self.view("COUNTS", torch.int32).cpu().numpy().astype(np.int64)
        return dict(hdr=hdr, rpad=rpad, row_token=row_token, row_slot=row_slot, row_of=row_of, offs=offs,
                    counts=counts, real=row_token >= 0)

    def rows(self, name, cols):
        """Stage `name` as fp64 [rpad, cols] (padded row order)."""
        rt = self.routing()
        t = self.view(name, torch.bfloat16)[: rt["rpad"] * cols].view(rt["rpad"], cols)
        return vals(t)

    def rows_bits(self, name, cols):
        rt = self.routing()
        t = self.view(name, torch.bfloat16)[: rt["rpad"] * cols].view(rt["rpad"], cols)
        return bits(t)


def e4m3_values(codes):
    """E4M3 (fn) code bytes -> fp64 values (torch's float8_e4m3fn decoding)."""
    t = torch.as_tensor(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def unpadded_row_of(rt):
    """Map padded row indices in row_of to the oracle's unpadded numbering."""
    real = rt["real"]
    idx = np.cumsum(real) - 1
    ro = rt["row_of"]
    return np.where(ro >= 0, idx[np.maximum(ro, 0)], -1)


def host_inputs(inp):
    """The synth tensors as the oracle's NumPy inputs."""
    return dict(fmt=inp["fmt"], x=bits(inp["x"]), dout=bits(inp["dout"]), topk_idx=synth.to_numpy(inp["topk_idx"]),
                topk_w=synth.to_numpy(inp["topk_w"]), w13=bits(inp["w13"]), w2=bits(inp["w2"]),
                s13=synth.to_numpy(inp["s13"]), s2=synth.to_numpy(inp["s2"]))
