"""Benchmark of one scale-only QAD MoE layer step (fwd + input grad + scale grad) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole path over one batch: qad_moe_fwd, qad_moe_bwd_dgrad and
qad_moe_bwd_scalegrad through the C ABI.  `value` is tokens/s with inputs resident in HBM;
`e2e` adds, every step, the host->device copy of the step's activations and routing from
pinned memory and the device->host read of out, dx, dprobs and the scale gradients,
double-buffered as an input pipeline would run them (inputs up on one copy stream, results
down on another, both beside the compute).  Every step streams far more than the 129 MB L2
(weights alone are 1.2 GB at the default workload), so no explicit flush is used.

Roofline fractions of the GEMMs are taken against the measured bf16 peak of the clock
regime the timed region ran in: the burst figure when the sampled median SM clock sat at
its maximum with no power cap, the sustained one otherwise; both fractions are printed.
`configs` holds a short timed run of every other workload on the same box.

Under torchrun each rank runs its own replica on its own batch (weak scaling) and the
scale gradients are averaged over ranks, as data-parallel training does.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

DEFAULT_WORKLOAD = "qwen3_30b_a3b_nvfp4"
METRIC = "MoE-layer fwd+bwd tokens/s (nvfp4, 1 GB300); % HBM / tensor-core roofline"
FMT_NAME = {0: "nvfp4", 1: "w4a16", 2: "fp8", 3: "nvfp4a16", 4: "w8a8", 5: "w4afp8", 6: "nvfp4_e4m3_scales"}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(pk["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "10"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # the sampler is running (its first line is in) before the timed region starts, so a
            # region of a few tens of milliseconds still gets several samples
            t0 = time.time()
            while not self.lines and time.time() - t0 < 2.0 and self.proc.poll() is None:
                time.sleep(0.005)
            self.lines.clear()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, *others):
        """Median SM clock, maximum and active throttle reasons over this sampler's lines and
        those of `others` (the other timed regions of the same run)."""
        sm, mx, reasons = [], None, set()
        lines = list(self.lines)
        for o in others:
            lines += o.lines
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_per_launch(cfg, native_fp8=False):
    """FLOPs per GEMM launch (routed rows only) and bytes per weight-fake-quant launch (with
    native fp8 the fake-quant also writes one E4M3 code byte per element)."""
    R = cfg["T"] * cfg["topk"]
    d, F, E = cfg["d"], cfg["F"], cfg["E"]
    fc1 = 2.0 * R * 2 * F * d
    fc2 = 2.0 * R * d * F
    # format 6 (deployed nvfp4): the fake-quant pass also writes each deployed fp32 block scale
    bpe = {0: 2 + 4.0 / 16 + 2, 1: 2 + 4.0 / 128 + 2, 2: None, 3: 2 + 4.0 / 16 + 2, 4: None,
           5: 2 + 4.0 / 128 + 2, 6: 2 + 2 * 4.0 / 16 + 2}[cfg["fmt"]]
    n13, n2 = E * 2 * F * d, E * d * F
    if bpe is None:  # one fp32 scale per row
        per_el = 5.0 if native_fp8 else 4.0
        fq = (per_el * n13 + 4 * E * 2 * F + per_el * n2 + 4 * E * d) / 2
    else:
        fq = bpe * (n13 + n2) / 2  # average of the two launches
    alg = {"gemm_fc1_swiglu_aq": ("tensor", fc1), "gemm_fc2": ("tensor", fc2),
           "gemm_dgrad_fc2_swiglu_bwd": ("tensor", fc2), "gemm_dgrad_fc1": ("tensor", fc1),
           "gemm_wgrad_fc2_scalegrad": ("tensor", fc2), "gemm_wgrad_fc1_scalegrad": ("tensor", fc1),
           "fakequant_w": ("hbm", fq)}
    if cfg["fmt"] == 6:  # the matrices' tensor scales: every fp32 block scale read once
        alg["deploy_scales"] = ("hbm", 4.0 * (n13 + n2) / 16)
    return alg


def side_stream_bytes(cfg):
    """Bytes per step that the routing and the token scatter move on the library's side stream
    while the weight fake-quant runs: the routing indices read and the pair-to-row maps written
    (int32), every token row read once and written to each of its routed rows (bf16)."""
    T, k, d = cfg["T"], cfg["topk"], cfg["d"]
    R = T * k
    return 4.0 * R + 4.0 * 3 * R + 2.0 * T * d + 2.0 * R * d


def _traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.txt), or None
    when the kernel's sources have changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    import hashlib
    for ln in open(path):
        f = ln.split()
        if len(f) < 4 or ln.startswith("#") or f[0] != kernel or f[1] != workload:
            continue
        files, want = f[3].split(":")
        h = hashlib.sha256()
        for name in files.split("+"):
            src = os.path.join(ROOT, "scale_only_quantization_gb300", "csrc", name)
            if not os.path.exists(src):
                return None
            h.update(open(src, "rb").read())
        return float(f[2]) if h.hexdigest()[:16] == want else None
    return None


NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s the fake-quant target is stated against (nominal HBM3e)


def tensor_peak(clocks, tf_burst, tf_sust):
    """The measured bf16 peak that matches the run's clock regime: the burst figure when the
    median SM clock under load sat at the maximum and no power cap was active (or when no
    clock was sampled: the larger peak, so no fraction is overstated), else the sustained one."""
    sm, mx, reasons = clocks.get("sm_mhz"), clocks.get("sm_max_mhz"), clocks.get("reasons") or []
    if sm is None or not mx:
        return tf_burst, "bf16_tflops (burst; clocks not sampled)"
    if sm >= 0.97 * mx and "sw_power_cap" not in reasons:
        return tf_burst, "bf16_tflops (burst: median SM clock %.0f of %.0f MHz, no power cap)" % (sm, mx)
    return tf_sust, "bf16_tflops_sustained (median SM clock %.0f of %.0f MHz, reasons %s)" % (
        sm, mx, ",".join(reasons) or "none")


def kernel_table(prof, steps, alg, peak, tf_burst, tf_sust, hbm, f8_kernels=(), side_bytes=None):
    """Per kernel: time per launch, launches per step, share of the step's serial kernel time,
    and for the GEMMs and the weight fake-quant the achieved rate against the peaks.  With
    `side_bytes` (bytes per step of the side-stream kernels that start beside the fake-quant), the
    fake-quant entry also gives the rate of the whole memory phase: its own bytes and those over
    the phase's time, the longer of the fake-quant launches and the side-stream launches (both
    start at the fork; the GEMMs wait for both)."""
    kernels = {}
    for name, (tot, n) in prof.items():
        if n == 0:
            continue
        entry = {"ms_per_launch": tot / n, "launches_per_step": n / steps, "share": None}
        if name in ("route_permute", "gather_rows"):
            # on the library's side stream beside the weight fake-quant: wall time while sharing the GPU
            entry["overlapped_with"] = "fakequant_w"
        if name in alg:
            bound, amount = alg[name]
            per_s = amount / (tot / n / 1e3)
            if bound == "tensor":
                m = 2 if name in f8_kernels else 1  # E4M3 x E4M3: nominal fp8 / bf16 ratio
                entry.update(achieved_tflops=per_s / 1e12, frac=per_s / 1e12 / (m * peak),
                             frac_of_burst=per_s / 1e12 / (m * tf_burst),
                             frac_of_sustained=per_s / 1e12 / (m * tf_sust))
            else:
                entry.update(achieved_gbs=per_s / 1e9, frac=per_s / 1e9 / hbm,
                             frac_of_nominal_8tbs=per_s / 1e9 / NOMINAL_HBM_GBS)
        kernels[name] = entry
    fq = kernels.get("fakequant_w")
    if fq is not None and side_bytes and "fakequant_w" in alg and any(
            "overlapped_with" in v for v in kernels.values()):
        n = fq["launches_per_step"]
        moved = alg["fakequant_w"][1] * n + side_bytes
        side_ms = sum(v["ms_per_launch"] * v["launches_per_step"] for v in kernels.values() if "overlapped_with" in v)
        phase_ms = max(fq["ms_per_launch"] * n, side_ms)
        rate = moved / (phase_ms / 1e3) / 1e9
        fq["with_side_stream"] = {"bytes_per_step": moved, "phase_ms": phase_ms, "achieved_gbs": rate,
                                  "frac": rate / hbm}
    total_ms = sum(v["ms_per_launch"] * v["launches_per_step"] for v in kernels.values() if "overlapped_with" not in v)
    for v in kernels.values():
        if "overlapped_with" not in v:
            v["share"] = v["ms_per_launch"] * v["launches_per_step"] / total_ms if total_ms else None
    return kernels


class Layer:
    """One MoE layer's buffers on the device and its fwd + dgrad + scalegrad step (C ABI)."""

    def __init__(self, Q, inp, flags, dev):
        self.Q, self.inp = Q, inp
        T, d, F, E, k, fmt = inp["T"], inp["d"], inp["F"], inp["E"], inp["topk"], inp["fmt"]
        self.s = Q.shape(T, d, F, E, k, fmt, flags)
        nb = Q.qad_moe_workspace_bytes(self.s)
        if nb == 0:
            raise RuntimeError("shape not supported: %r" % ((T, d, F, E, k, fmt, flags),))
        self.ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        self.outs = self.new_outputs()

    def new_outputs(self):
        inp = self.inp
        out = torch.empty((inp["T"], inp["d"]), dtype=torch.bfloat16, device=self.ws.device)
        return (out, torch.empty_like(out), torch.empty((inp["T"], inp["topk"]), dtype=torch.float32,
                                                         device=self.ws.device),
                torch.empty_like(inp["s13"]), torch.empty_like(inp["s2"]))

    def fwd(self, stream, x, idx, p, outs):
        inp = self.inp
        self.Q.qad_moe_fwd(self.s, x, idx, p, inp["w13"], inp["s13"], inp["w2"], inp["s2"], outs[0], self.ws, stream)

    def dgrad(self, stream, p, dout, outs):
        inp = self.inp
        self.Q.qad_moe_bwd_dgrad(self.s, dout, p, inp["w13"], inp["s13"], inp["w2"], inp["s2"], outs[1], outs[2],
                                 self.ws, stream)

    def scalegrad(self, stream, outs, average=None):
        inp = self.inp
        self.Q.qad_moe_bwd_scalegrad(self.s, inp["w13"], inp["s13"], inp["w2"], inp["s2"], outs[3], outs[4], 0,
                                     self.ws, stream)
        if average is not None:
            average([outs[3], outs[4]])

    def step(self, stream, x, idx, p, dout, outs=None, average=None):
        outs = outs if outs is not None else self.outs
        self.fwd(stream, x, idx, p, outs)
        self.dgrad(stream, p, dout, outs)
        self.scalegrad(stream, outs, average)


def timed_steps(Q, layer, stream, dev, steps, warmup, barrier, local, average=None):
    """Warm-up, then `steps` device-resident steps timed with CUDA events on the launching
    stream, the library's per-kernel events on, clocks sampled.  Returns (ms per step, kernel
    profile, library launches in the timed region, clock sampler)."""
    inp = layer.inp
    args_dev = (inp["x"], inp["topk_idx"], inp["topk_w"], inp["dout"])
    for _ in range(warmup):
        layer.step(stream, *args_dev, average=average)
    err = Q.qad_check_device_error(layer.ws, stream)
    if err:
        raise RuntimeError("device error word %d after warm-up" % err)
    barrier()
    Q.qad_profile_reset()
    Q.qad_profile_enable(True)
    n0 = Q.qad_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        barrier()
        e0.record(stream)
        for _ in range(steps):
            layer.step(stream, *args_dev, average=average)
        e1.record(stream)
        barrier()
    launches = Q.qad_launch_count() - n0
    ms = e0.elapsed_time(e1) / steps
    prof = Q.qad_profile_read()
    Q.qad_profile_enable(False)
    return ms, prof, launches, clk


def e2e_steps(layer, stream, dev, steps, warmup, barrier, local, average=None, host_in=None, results=None):
    """The same step end to end through the public calls: every step copies its inputs (x,
    topk_idx, topk_w, dout) from pinned host memory and reads its results (out, dx, dprobs,
    ds13, ds2) back to pinned host memory.  Double-buffered as an input pipeline runs it: one
    copy stream moves step i+1's inputs to the device while the compute stream runs step i (the
    forward's inputs first, dout after them: the forward waits only for its own), and a second
    copy stream moves each result down as soon as the call that writes it has finished (out after
    the forward, dx and dprobs after the input gradient, the scale gradients after the last
    call), so the two directions of the host link run at the same time and a short run's first
    and last steps wait for as few bytes as possible.  Returns (ms per step, H2D bytes, D2H
    bytes, clocks).  `host_in` (two lists of pinned x, topk_idx, topk_w, dout) replaces the
    layer's own inputs in the two buffers (step i uses buffer i % 2); with `results` (a list)
    the two buffers' host results are appended to it after the run."""
    inp = layer.inp
    args_dev = (inp["x"], inp["topk_idx"], inp["topk_w"], inp["dout"])
    if host_in is None:
        host_in = [[a.cpu().pin_memory() for a in args_dev] for _ in range(2)]
    dev_in = [[torch.empty_like(a) for a in args_dev] for _ in range(2)]
    dev_out = [layer.new_outputs() for _ in range(2)]
    host_out = [[torch.empty(a.shape, dtype=a.dtype, pin_memory=True) for a in dev_out[0]] for _ in range(2)]
    h2d = sum(a.numel() * a.element_size() for a in host_in[0])
    d2h = sum(a.numel() * a.element_size() for a in host_out[0])
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {name: [torch.cuda.Event() for _ in range(2)]
          for name in ("in_fwd", "in_bwd", "fwd", "dgrad", "done", "out", "dx", "ds")}

    def copy(dsts, srcs):
        for dst, src in zip(dsts, srcs):
            dst.copy_(src, non_blocking=True)

    def inputs_up(b):
        with torch.cuda.stream(up):
            copy(dev_in[b][:3], host_in[b][:3])  # x, topk_idx, topk_w: the forward's inputs
            ev["in_fwd"][b].record(up)
            copy(dev_in[b][3:], host_in[b][3:])  # dout
            ev["in_bwd"][b].record(up)

    def run(n):
        up.wait_stream(stream)
        down.wait_stream(stream)
        inputs_up(0)
        for i in range(n):
            b = i % 2
            x, idx, p, dout = dev_in[b]
            outs = dev_out[b]
            stream.wait_event(ev["in_fwd"][b])
            if i >= 2:
                stream.wait_event(ev["out"][b])  # step i-2's out has left dev_out[b]
            layer.fwd(stream, x, idx, p, outs)
            ev["fwd"][b].record(stream)
            stream.wait_event(ev["in_bwd"][b])
            if i >= 2:
                stream.wait_event(ev["dx"][b])
            layer.dgrad(stream, p, dout, outs)
            ev["dgrad"][b].record(stream)
            if i >= 2:
                stream.wait_event(ev["ds"][b])
            layer.scalegrad(stream, outs, average)
            ev["done"][b].record(stream)
            if i + 1 < n:
                nb = (i + 1) % 2
                if i >= 1:
                    up.wait_event(ev["dgrad"][nb])  # step i-1 has finished reading dev_in[nb]
                inputs_up(nb)
            with torch.cuda.stream(down):
                down.wait_event(ev["fwd"][b])
                copy(host_out[b][:1], outs[:1])
                ev["out"][b].record(down)
                down.wait_event(ev["dgrad"][b])
                copy(host_out[b][1:3], outs[1:3])
                ev["dx"][b].record(down)
                down.wait_event(ev["done"][b])
                copy(host_out[b][3:], outs[3:])
                ev["ds"][b].record(down)
        stream.wait_stream(up)
        stream.wait_stream(down)

    run(max(3, warmup))
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        barrier()
        e0.record(stream)
        run(steps)
        e1.record(stream)
        barrier()
    if results is not None:
        results.extend(host_out)
    return e0.elapsed_time(e1) / steps, h2d, d2h, clk


def dominant_roofline(kernels, alg, peak, peak_name, hbm, peak_src, f8_kernels, workload):
    dom = max((nm for nm in kernels if nm in alg), key=lambda nm: kernels[nm]["share"])
    bound, amount = alg[dom]
    dur = kernels[dom]["ms_per_launch"] / 1e3
    if bound == "tensor":
        m = 2 if dom in f8_kernels else 1
        roof = {"bound": "tensor", "kernel": dom, "achieved": amount / dur / 1e12, "peak": m * peak,
                "unit": "TFLOP/s",
                "peak_source": peak_src + " " + peak_name + (" x 2 (nominal fp8 / bf16)" if m == 2 else ""),
                "frac_of_burst": kernels[dom]["frac_of_burst"],
                "frac_of_sustained": kernels[dom]["frac_of_sustained"]}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": amount / dur / 1e9, "peak": hbm, "unit": "GB/s",
                "peak_source": peak_src + " hbm_gbs", "frac_of_nominal_8tbs": amount / dur / 1e9 / NOMINAL_HBM_GBS}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = _traffic(dom, workload)
    return roof


def run_ours(args):
    import scale_only_quantization_gb300 as Q
    from scale_only_quantization_gb300 import build as B
    from scale_only_quantization_gb300 import dp
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    Q.lib()
    over = {}
    if args.tokens:
        over["T"] = args.tokens
    if args.experts:
        over["E"] = args.experts
    cfg = synth.workload(args.workload, **over)
    inp = synth.make_inputs(cfg, seed=rank, device=dev)
    T, d, F, E, k, fmt = inp["T"], inp["d"], inp["F"], inp["E"], inp["topk"], inp["fmt"]
    flags = ((Q.QAD_FLAG_RECOMPUTE if args.recompute else 0) | (Q.QAD_FLAG_NATIVE_FP8 if args.native_fp8 else 0) |
             (Q.QAD_FLAG_SMEM_DEQUANT if args.smem_dequant else 0))
    stream = torch.cuda.current_stream(dev)
    average = dp.average_scale_grads if world > 1 else None

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    layer = Layer(Q, inp, flags, dev)

    # ---- device-resident timed region (kernel timing on, clocks sampled)
    ms, prof, launches, clk = timed_steps(Q, layer, stream, dev, args.steps, args.warmup, barrier, local, average)
    ms = dp.max_over_ranks(ms, device=dev)

    # ---- end to end through the public API with pinned host buffers
    ms_e2e, h2d, d2h, clk_e2e = e2e_steps(layer, stream, dev, args.steps, args.warmup, barrier, local, average)
    ms_e2e = dp.max_over_ranks(ms_e2e, device=dev)

    # ---- roofline of the dominant kernel (largest share of the timed region), against the
    # measured peak of the clock regime the timed region ran in
    hbm, tf_burst, tf_sust, peak_src = _peaks()
    clocks = clk.summary()
    peak, peak_name = tensor_peak(clocks, tf_burst, tf_sust)
    alg = algorithmic_per_launch(cfg, native_fp8=args.native_fp8)
    f8_kernels = ("gemm_fc1_swiglu_aq", "gemm_fc2") if args.native_fp8 else ()
    kernels = kernel_table(prof, args.steps, alg, peak, tf_burst, tf_sust, hbm, f8_kernels,
                           side_bytes=side_stream_bytes(cfg))
    roof = dominant_roofline(kernels, alg, peak, peak_name, hbm, peak_src, f8_kernels, args.workload)
    flops_step = synth.tokens_to_flops(cfg)
    step_tf = flops_step / (ms / 1e3) / 1e12

    line = {
        "metric": METRIC, "value": T * world / (ms / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16+e4m3" if args.native_fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload + ("" if not over else "_T%d_E%d" % (T, E)),
                   "format": FMT_NAME[fmt], "E": E, "d": d, "F": F, "topk": k,
                   "tokens_per_gpu": T, "global_batch": T * world, "parallelism": "dp%d" % world,
                   "activations": "recompute" if args.recompute else "stash",
                   "forward_gemms": "e4m3 codes, scales on the sums" if args.native_fp8 else "bf16 fake-quant",
                   "weight_fake_quant": ("in the GEMMs' shared memory" if args.smem_dequant
                                         else "one pass into a bf16 copy"),
                   "workspace_gb": layer.ws.numel() / 1e9,
                   "l2": "inputs larger than L2 (weights %.2f GB streamed per pass), no flush" %
                         (2 * 3 * E * F * d / 1e9)},
        "step_tflops": step_tf,
        "step_tensor_frac": step_tf / peak,
        "step_tensor_frac_of_burst": step_tf / tf_burst,
        "step_tensor_frac_of_sustained": step_tf / tf_sust,
        "roofline": roof,
        "kernels": kernels,
        "gpu_launches": int(launches),
        "clocks": clocks,
        "e2e": {"value": T * world / (ms_e2e / 1e3), "unit": "tokens/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "link_gbs": (h2d + d2h) / (ms_e2e / 1e3) / 1e9, "clocks": clk_e2e.summary(),
                "note": "pinned host buffers; step i+1's inputs go up on one copy stream (the forward's first, "
                        "dout after them) while step i computes, and each of step i's results comes down on "
                        "another as soon as the call that writes it has finished"},
    }
    del layer
    torch.cuda.empty_cache()
    if not args.no_ab and not args.native_fp8:
        # the other way of fake-quantizing the weights, same workload, same box
        ab_flags = flags ^ Q.QAD_FLAG_SMEM_DEQUANT
        lab = Layer(Q, inp, ab_flags, dev)
        ms_ab, prof_ab, _, clk_ab = timed_steps(Q, lab, stream, dev, args.steps, args.warmup, barrier, local, average)
        ms_ab = dp.max_over_ranks(ms_ab, device=dev)
        k_ab = kernel_table(prof_ab, args.steps, alg, peak, tf_burst, tf_sust, hbm)
        line["ab_weight_fake_quant"] = {
            "mode": "in the GEMMs' shared memory" if ab_flags & Q.QAD_FLAG_SMEM_DEQUANT else "one pass into a bf16 copy",
            "value": T * world / (ms_ab / 1e3), "unit": "tokens/s", "ms_per_step": ms_ab,
            "workspace_gb": lab.ws.numel() / 1e9, "clocks": clk_ab.summary(),
            "kernels": {nm: {kk: v[kk] for kk in ("ms_per_launch", "launches_per_step", "frac") if kk in v}
                        for nm, v in k_ab.items()}}
        del lab
        torch.cuda.empty_cache()
    if world == 1 and not args.no_configs and not over:
        line["configs"] = other_configs(Q, args, dev, stream, barrier, local, tf_burst, tf_sust, hbm, peak_src)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def other_configs(Q, args, dev, stream, barrier, local, tf_burst, tf_sust, hbm, peak_src):
    """A short timed run of every other workload (same step, default flags): tokens/s, ms per
    step, and the dominant kernel against the peak of that run's own clock regime.  The fp8
    workloads run once more with the forward GEMMs on the E4M3 tensor path (QAD_FLAG_NATIVE_FP8,
    key suffix "+native_fp8")."""
    res = {}
    runs = []
    for name in sorted(synth.WORKLOADS):
        if name != args.workload:
            runs.append((name, name, 0))
        if synth.WORKLOADS[name]["fmt"] == synth.FMT_FP8_ROW and not args.native_fp8:
            runs.append((name + "+native_fp8", name, Q.QAD_FLAG_NATIVE_FP8))
    for key, name, flags in runs:
        cfg = synth.workload(name)
        inp = synth.make_inputs(cfg, seed=0, device=dev)
        layer = Layer(Q, inp, flags, dev)
        native = (flags & Q.QAD_FLAG_NATIVE_FP8) != 0
        ms, prof, launches, clk = timed_steps(Q, layer, stream, dev, args.config_steps, 3, barrier, local)
        clocks = clk.summary()
        peak, peak_name = tensor_peak(clocks, tf_burst, tf_sust)
        alg = algorithmic_per_launch(cfg, native_fp8=native)
        f8_kernels = ("gemm_fc1_swiglu_aq", "gemm_fc2") if native else ()
        kernels = kernel_table(prof, args.config_steps, alg, peak, tf_burst, tf_sust, hbm, f8_kernels,
                               side_bytes=side_stream_bytes(cfg))
        roof = dominant_roofline(kernels, alg, peak, peak_name, hbm, peak_src, f8_kernels, name)
        step_tf = synth.tokens_to_flops(cfg) / (ms / 1e3) / 1e12
        res[key] = {"value": cfg["T"] / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
                     "steps": args.config_steps, "format": FMT_NAME[cfg["fmt"]],
                     "routing": cfg.get("routing", "uniform"), "step_tflops": step_tf,
                     "step_tensor_frac": step_tf / peak, "gpu_launches": int(launches),
                     "roofline": {kk: roof[kk] for kk in ("kernel", "bound", "achieved", "unit", "frac",
                                                          "peak_source")},
                     "clocks": clocks}
        del layer, inp
        torch.cuda.empty_cache()
    return res


def _oracle_sample(cfg, host, n_experts):
    """The oracle's fwd + dgrad + scalegrad restricted to experts [0, n_experts): pairs routed
    elsewhere are dropped.  Returns (routed pairs processed, seconds)."""
    from oracle import moe as OM
    idx = host["topk_idx"]
    keep = (idx >= 0) & (idx < n_experts)
    toks = np.nonzero(keep.any(axis=1))[0]
    sub_idx = np.where(keep[toks], idx[toks], -1)
    p = host["topk_w"][toks]
    E = n_experts
    t0 = time.perf_counter()
    fwd = OM.moe_forward(cfg["fmt"], host["x"][toks], sub_idx, p, host["w13"][:E], host["s13"][:E], host["w2"][:E],
                         host["s2"][:E])
    bwd = OM.moe_dgrad(host["dout"][toks], p, fwd)
    OM.moe_scalegrad(cfg["fmt"], fwd, bwd, host["w13"][:E], host["s13"][:E], host["w2"][:E], host["s2"][:E])
    return int(keep.sum()), time.perf_counter() - t0


def _host_inputs(inp, n_experts):
    to_bits = synth.to_numpy_bits
    return {"x": to_bits(inp["x"]), "dout": to_bits(inp["dout"]), "topk_idx": synth.to_numpy(inp["topk_idx"]),
            "topk_w": synth.to_numpy(inp["topk_w"]), "w13": to_bits(inp["w13"][:n_experts]),
            "w2": to_bits(inp["w2"][:n_experts]), "s13": synth.to_numpy(inp["s13"][:n_experts]),
            "s2": synth.to_numpy(inp["s2"][:n_experts])}


def cpu_baseline(cfg, inp, budget_s=15.0):
    """Time the oracle as it stands on this host's cores on a bounded sample: the experts
    [0, n) with every pair routed to them, n grown until ~budget_s of work."""
    n, pairs, secs = 1, 0, 0.0
    host = _host_inputs(inp, min(cfg["E"], 64))
    while True:
        pr, dt = _oracle_sample(cfg, host, n)
        pairs, secs = pr, dt
        if dt * 2 > budget_s or n * 2 > min(cfg["E"], 64):
            break
        n *= 2
    return {"value": pairs / cfg["topk"] / secs, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": "fp64 NumPy oracle, fwd+dgrad+scalegrad of experts 0..%d (%d routed rows = %.0f token-"
                      "equivalents) of %s; %.1f s" % (n - 1, pairs, pairs / cfg["topk"], cfg["name"], secs)}


def run_reference(args):
    world, rank, local = _dist()
    if rank != 0:
        return
    cfg = synth.workload(args.workload)
    inp = synth.make_inputs(cfg, seed=0, device="cpu")
    host = _host_inputs(inp, min(cfg["E"], 64))
    n = 4 if cfg["E"] >= 4 else cfg["E"]
    for _ in range(args.warmup):
        _oracle_sample(cfg, host, 1)
    tot_pairs, tot_s = 0, 0.0
    for _ in range(args.steps):
        pr, dt = _oracle_sample(cfg, host, n)
        tot_pairs += pr
        tot_s += dt
    value = tot_pairs / cfg["topk"] / tot_s
    ms = tot_s / args.steps * 1e3
    sample = ("fp64 NumPy oracle on the host cores, each step fwd+dgrad+scalegrad of experts 0..%d (all pairs "
              "routed to them) of %s" % (n - 1, cfg["name"]))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "format": FMT_NAME[cfg["fmt"]], "E": cfg["E"], "d": cfg["d"],
                   "F": cfg["F"], "topk": cfg["topk"], "tokens_per_gpu": cfg["T"], "parallelism": "none (CPU)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the short timed runs of the other workloads (the `configs` key)")
    ap.add_argument("--config-steps", type=int, default=20, help="timed steps of each other workload")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (small cases for profiler captures)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override the workload's expert count (small cases for profiler captures)")
    ap.add_argument("--recompute", action="store_true",
                    help="QAD_FLAG_RECOMPUTE: recompute fc1's Z1 in the backward instead of stashing it")
    ap.add_argument("--smem-dequant", action="store_true",
                    help="QAD_FLAG_SMEM_DEQUANT: the GEMMs fake-quantize weight tiles in shared memory")
    ap.add_argument("--no-ab", action="store_true",
                    help="skip timing the other weight fake-quant mode (the `ab_weight_fake_quant` key)")
    ap.add_argument("--native-fp8", action="store_true",
                    help="QAD_FLAG_NATIVE_FP8 (fp8 workloads): forward GEMMs on the E4M3 tensor path")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
