"""Oracle for the scale-only QAD MoE-layer path: plain, slow, fp64 NumPy.

This package is TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it. The CUDA library never calls it,
and it shares no code, table or helper with the CUDA sources.

What it computes follows these passages:

* "MCoreQAD Backend" (AngelSlim docs, mcore_qad.md), opening section: the BF16
  weights are frozen, fake quantization is applied, and only the quantizer scales
  are optimised.
* AngelSlim mcore_qad walkthrough article (nxmr.cn/news/131691), section 二.3: the
  weight returns quantize->dequantize(W; s) with gradients flowing to s; the input of
  each quantized matmul is fake-quantized before the matmul; the router stays
  high precision.  Section 二.4: expert weights are stacked [E, N, K], fake-quantized
  in one vectorised pass and consumed by one grouped GEMM.  Section 三: the format
  names nvfp4 / w4a16 / fp8 (W8A8).

Where the pages leave the arithmetic open (grids, rounding, the scale layout, the
LSQ factor, SwiGLU order, where the routing weight applies) the oracle takes the
plain readings listed in the repository's design notes; each function says which.

Modules:
  quant  -- bf16/fp32 rounding, the E2M1 / E4M3 / INT4 quantizers, weight and
            activation fake-quant, the LSQ straight-through factor.
  moe    -- routing permutation, forward, input-gradient and scale-gradient of one
            MoE layer, one expert at a time.
"""
from . import quant, moe  # noqa: F401
