// Device helpers shared by the kernels of the scale-only QAD MoE library (sm_103a).
//
// Quantizer readings (the pages name the formats but print no formula).  Element grids:
//   E2M1 - {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6}, round to nearest even, saturating
//          (PTX cvt.rn.satfinite.e2m1x2.f32); weight scale per 16 along K, activations
//          per 16 with amax / 6;
//   INT4 - {-8..7}: rintf (half to even) then clamp; weight scale per 128 along K;
//   E4M3 - max 448, round to nearest even, saturating (cvt.rn.satfinite.e4m3x2.f32);
//          weight scale per output row, activations per row with amax / 448;
//   INT8 - {-128..127}: rintf then clamp; weight scale per output row, activations per row
//          with amax / 127.
// Formats: nvfp4 = E2M1/E2M1, w4a16 = INT4/bf16, fp8 = E4M3/E4M3, nvfp4a16 = E2M1/bf16,
// w8a8 = INT8/INT8, w4afp8 = INT4/E4M3 (weights/activations).
// x = w / s is the IEEE fp32 quotient (__fdiv_rn); the dequantized value is
// bf16(fp32(q(x) * s)); s == 0 gives x = +-0 with the sign of w.
// Formats: "MCoreQAD Backend" (mcore_qad.md), Support Matrix; AngelSlim mcore_qad
// walkthrough (nxmr.cn/news/131691), sections 二.3 and 三.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qad.h"

namespace qad {

// element grids ("quantizer kinds"); kQE2M1G: E2M1 elements whose per-16 block scales are
// rounded to E4M3 under one fp32 scale of the row (deployed nvfp4 activations)
constexpr int kQNone = -1, kQE2M1 = 0, kQInt4 = 1, kQE4M3 = 2, kQInt8 = 3, kQE2M1G = 4;

// weight and activation grids of each public format (qad_fmt)
__host__ __device__ constexpr int weight_kind(int fmt) {
  return fmt == QAD_FMT_NVFP4 || fmt == QAD_FMT_NVFP4A16 || fmt == QAD_FMT_NVFP4_E4M3 ? kQE2M1
         : fmt == QAD_FMT_INT4_G128 || fmt == QAD_FMT_W4AFP8                         ? kQInt4
         : fmt == QAD_FMT_FP8_ROW                                                    ? kQE4M3
                                                                                     : kQInt8;
}
__host__ __device__ constexpr int act_kind(int fmt) {
  return fmt == QAD_FMT_NVFP4                              ? kQE2M1
         : fmt == QAD_FMT_FP8_ROW || fmt == QAD_FMT_W4AFP8 ? kQE4M3
         : fmt == QAD_FMT_W8A8                             ? kQInt8
         : fmt == QAD_FMT_NVFP4_E4M3                       ? kQE2M1G
                                                           : kQNone;
}
// a scale per whole row (E4M3, INT8) rather than per block along K
__host__ __device__ constexpr bool row_scaled(int kind) { return kind == kQE4M3 || kind == kQInt8; }
// an activation grid whose scales depend on the whole row (the per-row grids, and the E2M1
// blocks under a row scale): the fc1 epilogue cannot apply it tile by tile
__host__ __device__ constexpr bool act_needs_row(int kind) { return row_scaled(kind) || kind == kQE2M1G; }

// ---------------------------------------------------------------------------------- bf16

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// 8 bf16 in a uint4 <-> 8 floats
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  f[0] = bf16lo(u.x); f[1] = bf16hi(u.x); f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
  f[4] = bf16lo(u.z); f[5] = bf16hi(u.z); f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
}
__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
}

// ---------------------------------------------------------------------------------- f32x2
// Blackwell's packed fp32 arithmetic: two independent lanes per instruction, each rounded
// to nearest even exactly as the scalar instruction would.
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2unpack(uint64_t v) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return make_float2(a, b);
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---------------------------------------------------------------------------------- quantizers

// E2M1 rounding of two values; returns the decoded grid values (exact in fp32).
__device__ __forceinline__ float2 q_e2m1x2(float a, float b) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2) : "f"(a), "f"(b));
  __half2 h = *reinterpret_cast<__half2*>(&h2);   // low half <- a, high half <- b
  return make_float2(__low2float(h), __high2float(h));
}

// E4M3 rounding of two values; returns the decoded grid values (exact in fp32).
__device__ __forceinline__ float2 q_e4m3x2(float a, float b) {
  uint16_t p;
  uint32_t h2;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(p) : "f"(a), "f"(b));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(p));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return make_float2(__low2float(h), __high2float(h));
}

__device__ __forceinline__ float q_int4(float x) { return fminf(fmaxf(rintf(x), -8.0f), 7.0f); }
__device__ __forceinline__ float q_int8(float x) { return fminf(fmaxf(rintf(x), -128.0f), 127.0f); }

template <int QK>
__device__ __forceinline__ float2 q_pair_raw(float a, float b) {
  if constexpr (QK == kQE2M1) {
    return q_e2m1x2(a, b);
  } else if constexpr (QK == kQE4M3) {
    return q_e4m3x2(a, b);
  } else if constexpr (QK == kQInt4) {
    return make_float2(q_int4(a), q_int4(b));
  } else {
    return make_float2(q_int8(a), q_int8(b));
  }
}

template <int QK>
__device__ __forceinline__ float2 q_pair(float a, float b) {
  const float2 r = q_pair_raw<QK>(a, b);
  // the grid value keeps the sign of its input, also when it rounds to zero
  return make_float2(copysignf(r.x, a), copysignf(r.y, b));
}

template <int QK> struct Clip;
template <> struct Clip<kQE2M1> { static constexpr float lo = -6.0f, hi = 6.0f; };
template <> struct Clip<kQInt4> { static constexpr float lo = -8.0f, hi = 7.0f; };
template <> struct Clip<kQE4M3> { static constexpr float lo = -448.0f, hi = 448.0f; };
template <> struct Clip<kQInt8> { static constexpr float lo = -128.0f, hi = 127.0f; };

// x = fp32(w / s); s == 0 -> +-0 with the sign of w (IEEE division, the reference path)
__device__ __forceinline__ float quotient(float w, float s) {
  return s == 0.0f ? copysignf(0.0f, w) : __fdiv_rn(w, s);
}

// One 32-byte sector (16 bf16) of read-only global memory with a 256-bit load that allocates no
// L1 line (ptr 32-byte aligned).  Used where a warp's load touches 32 different rows.
__device__ __forceinline__ void ld_nc_256(const void* ptr, uint4& lo, uint4& hi) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
               : "l"(ptr));
}

// x = fp32(w / s) from r = RN(1 / s) (computed once by the caller for many w): Markstein's
// correction, with the range guards of quotients<N> below; outside them the IEEE division.
__device__ __forceinline__ float quotient_r(float w, float s, float r) {
  const float q = __fmul_rn(w, r);
  const float e = __fmaf_rn(-q, s, w);
  const float x = copysignf(__fmaf_rn(e, r, q), w);
  const float aw = fabsf(w);
  const bool ok = s >= 1.17549435e-38f && s <= 0x1p20f && (aw >= 0x1p-80f || aw == 0.0f) && fabsf(x) <= 3.0e38f;
  return ok ? x : quotient(w, s);
}

// Deployed nvfp4 block scale: s_q = fp32(e4m3(fp32(s / g)) * g), E4M3 rounding to nearest even
// with saturation at 448 (cvt.rn.satfinite), exact decode; g = 0 gives 0.  The sign of s is kept.
__device__ __forceinline__ float deployed_scale(float s, float g) {
  if (g == 0.0f) return 0.0f;
  return __fmul_rn(q_e4m3x2(__fdiv_rn(s, g), 0.0f).x, g);
}
// the same from r = RN(1 / g), for many scales under one g
__device__ __forceinline__ float deployed_scale_r(float s, float g, float r) {
  if (g == 0.0f) return 0.0f;
  return __fmul_rn(q_e4m3x2(quotient_r(s, g, r), 0.0f).x, g);
}
// the tensor scale g = fp32(amax / 448) of a set of block scales whose largest magnitude is amax
__device__ __forceinline__ float deploy_tensor_scale(float amax) { return __fdiv_rn(amax, 448.0f); }


// The same correctly rounded quotients from r = RN(1 / s), without a division per element.
// Markstein's theorem (P. Markstein, "IA-64 and Elementary Functions", 2000; also
// Cornea, Golliver and Markstein 1999): if r is the correctly rounded reciprocal of s and
// q approximates w / s within one ulp, the remainder e = w - s q is exact (one FMA) and
// RN(q + e r) is the correctly rounded quotient; q = RN(w r) is within one ulp.  The
// theorem needs the remainder and the quotient in the normal range.  With s in
// [2^-126, 2^20] and |w| >= 2^-80 the remainder (>= 2^-46 |w| when non-zero) and the
// quotient (>= 2^-100) are normal; w = +-0 gives +-0 (sign restored below); an overflow
// is checked.  If any element of the block falls outside, the whole block is recomputed
// with the division (rare: tiny non-zero weights or extreme scales).  The GPU tests
// compare the result with CUDA's own division bit for bit.
template <int N>
__device__ __forceinline__ void quotients(const float* w, float s, float* x) {
  const float r = __frcp_rn(s);
  bool ok = s >= 1.17549435e-38f && s <= 0x1p20f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float q = __fmul_rn(w[i], r);
    const float e = __fmaf_rn(-q, s, w[i]);
    const float xi = copysignf(__fmaf_rn(e, r, q), w[i]);
    const float aw = fabsf(w[i]);
    ok = ok && (aw >= 0x1p-80f || aw == 0.0f) && fabsf(xi) <= 3.0e38f;
    x[i] = xi;
  }
  if (__builtin_expect(!ok, 0)) {
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = quotient(w[i], s);
  }
}

// Quotients for a block whose scale lies in [2^-60, 2^60] (the caller checks, and falls back
// to quotients<N> otherwise), without per-element guards.  Exactness is only needed where x
// can change a quantization decision: every grid's smallest decision point is >= 2^-10, and
// for |x| >= 2^-11 with such a scale, w, q and the remainder (a multiple of
// ulp(s) ulp(q) >= 2^-117) are normal, so Markstein's theorem gives the correctly rounded
// quotient; smaller |x| may be off by a subnormal quantum but rounds to zero on every grid
// either way.  The caller must also rule out an overflowing quotient (finite activations
// with s = amax / Qmax never overflow; the LSQ reduction checks its block sum).
template <int N>
__device__ __forceinline__ void quotients_unguarded(const float* w, float s, float* x) {
  const float r = __frcp_rn(s);
  const uint64_t r2 = f2pack(r, r), ns2 = f2pack(-s, -s);
#pragma unroll
  for (int i = 0; i + 1 < N; i += 2) {  // q = w r, e = w - q s, x = q + e r, two lanes at a time
    const uint64_t w2 = f2pack(w[i], w[i + 1]);
    const uint64_t q2 = f2mul(w2, r2);
    const uint64_t e2 = f2fma(q2, ns2, w2);
    const float2 x2 = f2unpack(f2fma(e2, r2, q2));
    x[i] = x2.x;
    x[i + 1] = x2.y;
  }
  if constexpr (N & 1) {
    const float q = __fmul_rn(w[N - 1], r);
    const float e = __fmaf_rn(-q, s, w[N - 1]);
    x[N - 1] = __fmaf_rn(e, r, q);
  }
}
__device__ __forceinline__ bool scale_in_fast_range(float s) { return s >= 0x1p-60f && s <= 0x1p60f; }

// Quotients x = fp32(v / s) of n activation values sharing the dynamic scale s = fp32(amax /
// Qmax): |x| <= amax / s stays near Qmax, so no overflow is possible; the sign of a zero
// result is v's.
template <int N>
__device__ __forceinline__ void act_quotients(const float* v, float s, float* x) {
  if (scale_in_fast_range(s)) {
    quotients_unguarded<N>(v, s, x);
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = copysignf(x[i], v[i]);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = quotient(v[i], s);
  }
}

// Quotients of n weights sharing scale s.  Weights are arbitrary, so besides the block's
// scale range the quotients are checked for overflow through one NaN/inf-propagating sum (an
// overflowing fast quotient gives inf or NaN); a block that fails is recomputed with the
// per-element guarded form.
template <int N>
__device__ __forceinline__ void weight_quotients(const float* v, float s, float* x) {
  bool fast = scale_in_fast_range(s);
  if (fast) {
    quotients_unguarded<N>(v, s, x);
    float probe = 0.0f;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      x[i] = copysignf(x[i], v[i]);
      probe += x[i] * 0.0f;  // 0 unless some x is inf or NaN
    }
    fast = probe == 0.0f;
  }
  if (!fast) quotients<N>(v, s, x);
}

// Activation fake-quant of n values sharing the dynamic scale s, in place.
template <int QK, int N>
__device__ __forceinline__ void fakequant_act_inplace(float* v, float s) {
  float x[N];
  act_quotients<N>(v, s, x);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float2 q = q_pair<QK>(x[i], x[i + 1]);
    v[i] = round_bf16(__fmul_rn(q.x, s));
    v[i + 1] = round_bf16(__fmul_rn(q.y, s));
  }
}

// Fake-quantize n (even) values that share scale s, in place: v <- bf16(fp32(q(v / s) * s)).
template <int QK, int N>
__device__ __forceinline__ void fakequant_inplace(float* v, float s) {
  float x[N];
  weight_quotients<N>(v, s, x);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float2 q = q_pair<QK>(x[i], x[i + 1]);
    v[i] = round_bf16(__fmul_rn(q.x, s));
    v[i + 1] = round_bf16(__fmul_rn(q.y, s));
  }
}

// Weight fake-quant of 16 weights packed as bf16 pairs (w[i]: element 2i in the low half,
// 2i + 1 in the high half) sharing scale s, returning packed bf16 results: the same bits as
// unpack8 -> fakequant_inplace<QK, 16> -> pack8, with fewer conversion instructions (they
// issue at a fraction of the fp32 rate).  For a scale in [2^-60, 2^16) and finite quotients:
//  - x = fp32(w / s) from the reciprocal and one FMA correction, as quotients_unguarded;
//  - E2M1 / E4M3: the saturating conversion to the 4- / 8-bit code and back to f16 (two
//    instructions per pair); an f16 magnitude shifted left by 13 bits is the fp32 bit pattern
//    of |q| * 2^-112 (every grid value is a normal f16 or zero), and s * 2^112 is exact, so
//    their fp32 product is RN(|q| s), the same rounding of the same real number;
//  - INT4 / INT8: clamp to the clip range, then round to the nearest integer (ties to even) by
//    adding and subtracting 1.5 * 2^23 (exact for |x| <= 2^22), equal to clamping rint(x);
//  - one bf16x2 conversion of the products; the sign is w's (a zero result keeps w's sign,
//    as fakequant_inplace's copysign does).
// Other scales, or a non-finite quotient, take fakequant_inplace itself.
template <int QK>
__device__ __forceinline__ void fakequant16_packed(const uint32_t (&w)[8], float s, uint32_t (&out)[8]) {
  if (s >= 0x1p-60f && s < 0x1p16f) {
    const float r = __frcp_rn(s);
    const uint64_t r2 = f2pack(r, r), ns2 = f2pack(-s, -s), zero2 = f2pack(0.0f, 0.0f);
    const float sc = (QK == kQE2M1 || QK == kQE4M3) ? s * 0x1p112f : s;
    const uint64_t sc2 = f2pack(sc, sc);
    uint64_t probe = zero2;
    uint32_t res[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint64_t w2 = f2pack(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
      const uint64_t q2 = f2mul(w2, r2);
      const uint64_t e2 = f2fma(q2, ns2, w2);
      const uint64_t x2 = f2fma(e2, r2, q2);
      probe = f2fma(x2, zero2, probe);  // stays 0 unless a quotient is inf or NaN
      const float2 x = f2unpack(x2);
      uint64_t m2;
      if constexpr (QK == kQE2M1 || QK == kQE4M3) {
        uint32_t h2;
        if constexpr (QK == kQE2M1) {
          asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
              : "=r"(h2) : "f"(x.x), "f"(x.y));
        } else {
          uint16_t c;
          asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(c) : "f"(x.x), "f"(x.y));
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
        }
        const uint32_t la = (h2 << 13) & 0x0FFFE000u, lb = (h2 >> 3) & 0x0FFFE000u;
        m2 = f2mul(f2pack(__uint_as_float(la), __uint_as_float(lb)), sc2);
      } else {
        const uint64_t big2 = f2pack(12582912.0f, 12582912.0f);  // 1.5 * 2^23
        const float ta = fminf(fmaxf(x.x, Clip<QK>::lo), Clip<QK>::hi);
        const float tb = fminf(fmaxf(x.y, Clip<QK>::lo), Clip<QK>::hi);
        const uint64_t q = f2sub(f2add(f2pack(ta, tb), big2), big2);
        m2 = f2mul(q, sc2);
      }
      const float2 m = f2unpack(m2);
      res[i] = pack_bf16(m.x, m.y) | (w[i] & 0x80008000u);
    }
    if (f2unpack(probe).x == 0.0f && f2unpack(probe).y == 0.0f) {
#pragma unroll
      for (int i = 0; i < 8; ++i) out[i] = res[i];
      return;
    }
  }
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16lo(w[i]);
    v[2 * i + 1] = bf16hi(w[i]);
  }
  fakequant_inplace<QK, 16>(v, s);
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
}

// E4M3 codes of a pair (a in the low byte, b in the high byte) and their grid values, signed
// as q_pair<kQE4M3> signs them.
__device__ __forceinline__ uint16_t e4m3_codes2(float a, float b, float2* q) {
  uint16_t p;
  uint32_t h2;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(p) : "f"(a), "f"(b));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(p));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  *q = make_float2(copysignf(__low2float(h), a), copysignf(__high2float(h), b));
  return p;
}

// E4M3 fake-quant of N (a multiple of 4) values sharing scale s, in place, also returning
// their codes (byte i of the N / 4 words = code of value i): the quotients and grid values
// of fakequant_inplace (ACT = false) or fakequant_act_inplace (ACT = true).
template <int N, bool ACT>
__device__ __forceinline__ void fakequant_e4m3_codes(float* v, float s, uint32_t* codes) {
  float x[N];
  if constexpr (ACT) act_quotients<N>(v, s, x);
  else weight_quotients<N>(v, s, x);
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    float2 q0, q1;
    const uint32_t c0 = e4m3_codes2(x[i], x[i + 1], &q0);
    const uint32_t c1 = e4m3_codes2(x[i + 2], x[i + 3], &q1);
    codes[i / 4] = c0 | (c1 << 16);
    v[i] = round_bf16(__fmul_rn(q0.x, s));
    v[i + 1] = round_bf16(__fmul_rn(q0.y, s));
    v[i + 2] = round_bf16(__fmul_rn(q1.x, s));
    v[i + 3] = round_bf16(__fmul_rn(q1.y, s));
  }
}

// LSQ straight-through factor phi(x): q(x) - x inside the closed clip range, else the
// violated bound.  q saturates (E2M1, E4M3) or clamps (INT4) to exactly that bound
// outside the range, so phi = q(x) - (x inside ? x : 0).  The sign of a zero q does not
// matter here, so the grid value is used as the conversion returns it.
template <int QK>
__device__ __forceinline__ float2 lsq_pair(float xa, float xb) {
  const float2 q = q_pair_raw<QK>(xa, xb);
  float ia, ib;
  if constexpr (QK == kQInt4 || QK == kQInt8) {
    ia = (xa >= Clip<QK>::lo && xa <= Clip<QK>::hi) ? xa : 0.0f;
    ib = (xb >= Clip<QK>::lo && xb <= Clip<QK>::hi) ? xb : 0.0f;
  } else {  // symmetric clip range
    ia = fabsf(xa) <= Clip<QK>::hi ? xa : 0.0f;
    ib = fabsf(xb) <= Clip<QK>::hi ? xb : 0.0f;
  }
  return make_float2(q.x - ia, q.y - ib);
}

// ---------------------------------------------------------------------------------- misc

// sigmoid(g) = 1 / (1 + exp(-g)) from CUDA's fast exponential and the hardware's approximate
// reciprocal (exp(-g) = inf gives 0).  Used only where the result is compared with the
// oracle by tolerance.
__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float sigmoid_f(float g) { return rcp_approx(1.0f + __expf(-g)); }
__device__ __forceinline__ float silu_f(float g) { return __fmul_rn(g, sigmoid_f(g)); }

// sigmoid of two lanes: the exponentials by the intrinsic, the +1 in packed fp32.
__device__ __forceinline__ uint64_t sigmoid2(uint64_t g2) {
  const float2 g = f2unpack(g2);
  const float2 d = f2unpack(f2add(f2pack(__expf(-g.x), __expf(-g.y)), f2pack(1.0f, 1.0f)));
  return f2pack(rcp_approx(d.x), rcp_approx(d.y));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace qad
