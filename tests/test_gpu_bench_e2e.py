"""The benchmark's end-to-end pipeline gives the results of the public calls.

The end-to-end timing double-buffers the inputs and results through pinned host memory on two
copy streams and waits on events per call (the forward's inputs, dout, each result as soon as the
call writing it has finished).  With different inputs in the two buffers, the results that come
back to the host after the run must be, bit for bit, those of plain calls on the same inputs: a
missing wait (a call reading inputs that have not arrived, or a result read back before it was
written or after the next step overwrote it) shows up as a mismatch.
"""
import importlib.util
import os

import pytest
import torch

import scale_only_quantization_gb300 as Q
import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from scale_only_quantization_gb300 import build
    build.build()
    Q.lib()


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("steps", [5, 6])
def test_end_to_end_pipeline_returns_each_buffers_results(steps):
    b = _bench()
    dev = torch.device("cuda", 0)
    cfg = synth.workload("tiny_nvfp4", T=1536, E=8)
    inp = [synth.make_inputs(cfg, seed=s, device=dev) for s in (21, 22)]
    layer = b.Layer(Q, inp[0], 0, dev)
    stream = torch.cuda.current_stream(dev)
    names = ("x", "topk_idx", "topk_w", "dout")
    host_in = [[inp[k][n].cpu().pin_memory() for n in names] for k in (0, 1)]
    results = []
    b.e2e_steps(layer, stream, dev, steps, 3, torch.cuda.synchronize, 0, host_in=host_in, results=results)
    torch.cuda.synchronize()
    assert Q.qad_check_device_error(layer.ws) == 0
    for k in (0, 1):
        outs = layer.new_outputs()
        layer.step(stream, *(inp[k][n] for n in names), outs=outs)
        torch.cuda.synchronize()
        for name, want, got in zip(("out", "dx", "dprobs", "ds13", "ds2"), outs, results[k]):
            iv = torch.int16 if want.dtype == torch.bfloat16 else torch.int32
            assert torch.equal(want.cpu().view(iv), got.view(iv)), (k, name)
