// Memory-bound kernels of the scale-only QAD MoE path: weight fake-quant (optionally with
// E4M3 codes), routing permutation, the per-token activation fake-quant and scatter to the
// routed rows, the per-row activation fake-quant of H, combine, the per-token dY scatter,
// the scale-gradient reduction, and the quotient self-check.
//
// Weight fake-quant: the whole stacked expert weight is fake-quantized in one vectorised
// pass (AngelSlim mcore_qad walkthrough, nxmr.cn/news/131691, section 二.4); the weight a
// matmul sees is quantize->dequantize(W; s) (section 二.3).  Activations are fake-quantized
// before each quantized matmul with a dynamic (detached) scale (section 二.3).  The routed
// rows are grouped by expert for one grouped GEMM (section 二.4); routing indices and
// weights come from the unquantized router and are inputs here.
#include "common.cuh"
#include "internal.h"

namespace qad {

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }

int grid_for(int64_t items, int threads, int per_sm) {
  int64_t want = (items + threads - 1) / threads;
  int64_t cap = (int64_t)num_sms() * per_sm;
  if (want > cap) want = cap;
  return want < 1 ? 1 : (int)want;
}

// ------------------------------------------------------------------------- weight fake-quant

// One thread per 16 consecutive elements of a row (16 | K, and every scale block is a
// whole number of 16-element chunks).  `cps` = chunks per scale (1, 8 or K / 16).  CODES
// (E4M3 only): also write each element's E4M3 code byte to `codes` (same layout as w).
template <int QK, bool CODES = false>
__device__ __forceinline__ void fakequant_chunk(const uint4& u0, const uint4& u1, float sc, uint4* out, uint4* codes,
                                                uint64_t c) {
  if constexpr (CODES) {
    float v[16];
    unpack8(u0, v);
    unpack8(u1, v + 8);
    uint32_t cw[4];
    fakequant_e4m3_codes<16, false>(v, sc, cw);
    st_stream(codes + c, make_uint4(cw[0], cw[1], cw[2], cw[3]));
    st_stream(out + 2 * c, pack8(v));
    st_stream(out + 2 * c + 1, pack8(v + 8));
  } else {
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    uint32_t o[8];
    fakequant16_packed<QK>(w, sc, o);
    st_stream(out + 2 * c, make_uint4(o[0], o[1], o[2], o[3]));
    st_stream(out + 2 * c + 1, make_uint4(o[4], o[5], o[6], o[7]));
  }
}

// DEPLOY (deployed nvfp4, one scale per chunk): the chunk's scale is first rounded as deployed
// NVFP4 stores it, s_q = fp32(e4m3(fp32(s / g)) * g) with gr[m] = (g, RN(1 / g)) of its matrix
// m = c / cpm, and s_q is also written to sq[c] (the backward calls read it).
__device__ __forceinline__ float deploy_chunk(float s, const float2* __restrict__ gr, uint32_t cpm,
                                              float* __restrict__ sq, uint64_t c) {
  const float2 g = __ldg(gr + (uint32_t)c / cpm);
  const float v = deployed_scale_r(s, g.x, g.y);
  sq[c] = v;
  return v;
}

// A persistent grid of three 256-thread CTAs per SM (the registers of three fit; see the
// launchers): with the next two chunks of each thread loaded ahead of the current two, ~96 KB
// of weights per SM are in flight, which the memory system needs to run near its copy rate
// (with one pair per thread at a time and eight CTAs per SM the pass ran ~10% slower).
template <int QK, bool CODES = false, bool DEPLOY = false>
__global__ void __launch_bounds__(256, 3) fakequant_kernel(const uint4* __restrict__ w, const float* __restrict__ s,
                                                           uint4* __restrict__ out, uint64_t nchunks, uint32_t cps,
                                                           uint4* __restrict__ codes = nullptr,
                                                           const float2* __restrict__ gr = nullptr, uint32_t cpm = 1,
                                                           float* __restrict__ sq = nullptr) {
  static_assert(!DEPLOY || (QK == kQE2M1 && !CODES), "deployed scales: nvfp4 weights, one scale per chunk");
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint64_t c = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // two chunks (64 bytes) per thread per iteration, and the next iteration's two chunks loaded
  // before this one's arithmetic: 128 bytes of weights per thread in flight
  auto load = [&](uint64_t cc, uint4& x0, uint4& x1, float& sc) {
    x0 = ld_stream(w + 2 * cc);
    x1 = ld_stream(w + 2 * cc + 1);
    sc = __ldg(s + (cps == 1 ? cc : cc / cps));
  };
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
  uint4 a0 = z4, a1 = z4, b0 = z4, b1 = z4;
  float sa = 0.0f, sb = 0.0f;
  if (c < nchunks) load(c, a0, a1, sa);
  if (c + stride < nchunks) load(c + stride, b0, b1, sb);
  for (; c < nchunks; c += 2 * stride) {
    const uint64_t c2 = c + stride, n = c + 2 * stride;
    uint4 na0 = z4, na1 = z4, nb0 = z4, nb1 = z4;
    float nsa = 0.0f, nsb = 0.0f;
    if (n < nchunks) load(n, na0, na1, nsa);
    if (n + stride < nchunks) load(n + stride, nb0, nb1, nsb);
    if constexpr (DEPLOY) sa = deploy_chunk(sa, gr, cpm, sq, c);
    fakequant_chunk<QK, CODES>(a0, a1, sa, out, codes, c);
    if (c2 < nchunks) {
      if constexpr (DEPLOY) sb = deploy_chunk(sb, gr, cpm, sq, c2);
      fakequant_chunk<QK, CODES>(b0, b1, sb, out, codes, c2);
    }
    a0 = na0; a1 = na1; b0 = nb0; b1 = nb1;
    sa = nsa; sb = nsb;
  }
}

// ------------------------------------------------------------------------- routing

// Expert of pair i = t * k + j, or -1 when the pair is dropped (index outside [0, E), or
// the same expert as an earlier slot of the token); sets error bits in *err.
__device__ __forceinline__ int pair_expert(const int32_t* __restrict__ idx, int64_t i, int k, int E, int* err) {
  const int64_t t = i / k;
  const int j = (int)(i - t * k);
  const int e = idx[i];
  if (e < 0 || e >= E) {
    *err |= QAD_DEV_BAD_INDEX;
    return -1;
  }
  for (int jj = 0; jj < j; ++jj)
    if (idx[t * k + jj] == e) {
      *err |= QAD_DEV_DUP_INDEX;
      return -1;
    }
  return e;
}

__global__ void __launch_bounds__(256) route_hist_kernel(const int32_t* __restrict__ idx, int64_t R, int k, int E,
                                                         int32_t* __restrict__ chunk_counts, int32_t* hdr) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  int err = 0;
  const int64_t base = (int64_t)blockIdx.x * kRouteChunk;
  for (int i = threadIdx.x; i < kRouteChunk; i += blockDim.x) {
    const int64_t g = base + i;
    if (g < R) {
      const int e = pair_expert(idx, g, k, E, &err);
      if (e >= 0) atomicAdd(&hist[e], 1);
    }
  }
  if (err) atomicOr(&hdr[HDR_ERR], err);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// One block of 1024 threads.  Each expert gets G = 1024 / (E rounded up to a power of two)
// threads, each of which sums the expert's counts over a contiguous range of chunks; the
// ranges' exclusive prefixes give each chunk's first row for the expert.  Produces per-expert
// counts, padded offsets (multiples of 128 rows), the chunk bases, the expert of every
// 128-row tile, and marks padding rows with token -1.
__global__ void __launch_bounds__(1024) route_scan_kernel(int64_t nchunks, int E, const int32_t* __restrict__ chunk_counts,
                                                          int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offs, int32_t* __restrict__ mtile_expert,
                                                          int32_t* __restrict__ row_token, int32_t* __restrict__ row_slot,
                                                          int32_t* hdr) {
  __shared__ int32_t part[1024];  // each thread's sum over its chunk range
  __shared__ int32_t tot[1024];   // per-expert totals
  __shared__ int32_t eoff[1024];  // per-expert padded offsets
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t valid_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int ep = 1;
  while (ep < E) ep <<= 1;
  const int G = 1024 / ep;
  const int e = tid / G, g = tid - (tid / G) * G;
  const int64_t per = (nchunks + G - 1) / G;
  const int64_t c0 = min(nchunks, (int64_t)g * per), c1 = min(nchunks, c0 + per);
  int32_t sum = 0;
  if (e < E) {
#pragma unroll 8
    for (int64_t c = c0; c < c1; ++c) sum += chunk_counts[c * E + e];
  }
  part[tid] = sum;
  __syncthreads();
  int32_t before = 0;  // the expert's rows in the chunks before this thread's range
  if (e < E) {
    for (int h = e * G; h < tid; ++h) before += part[h];
    if (g == G - 1) tot[e] = before + sum;
  }
  __syncthreads();
  // exclusive scan over experts of the padded totals (thread x: expert x)
  const int32_t total = tid < E ? tot[tid] : 0;
  const int32_t padded = (total + kTileRows - 1) / kTileRows * kTileRows;
  int32_t v = padded, nv = total;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) nv += __shfl_xor_sync(0xffffffffu, nv, o);
  if (lane == 31) warp_tot[w] = v;
  if (lane == 0) valid_tot[w] = nv;
  __syncthreads();
  if (w == 0) {
    int32_t t = warp_tot[lane], sv = valid_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
    warp_tot[lane] = t;
    if (lane == 0) valid_tot[0] = sv;
  }
  __syncthreads();
  if (tid < E) {
    const int32_t incl = v + (w > 0 ? warp_tot[w - 1] : 0);
    eoff[tid] = incl - padded;
    counts[tid] = total;
    offs[tid] = incl - padded;
    if (tid == E - 1) {
      offs[E] = incl;
      hdr[HDR_NMTILES] = incl / kTileRows;
      hdr[HDR_RPAD] = incl;
      hdr[HDR_NVALID] = valid_tot[0];
    }
  }
  __syncthreads();
  if (e < E) {
    int32_t run = eoff[e] + before;
#pragma unroll 8
    for (int64_t c = c0; c < c1; ++c) {
      const int32_t n = chunk_counts[c * E + e];
      chunk_base[c * E + e] = run;
      run += n;
    }
    const int32_t ex = eoff[e], t = tot[e];
    const int32_t end = ex + (t + kTileRows - 1) / kTileRows * kTileRows;
    for (int32_t r = ex + t + g; r < end; r += G) {
      row_token[r] = -1;
      row_slot[r] = -1;
    }
    for (int32_t mb = ex / kTileRows + g; mb < end / kTileRows; mb += G) mtile_expert[mb] = e;
  }
}

// One block of 1024 threads per chunk of 1024 pairs, one pair per thread.  A pair's row is its
// chunk's first row for the expert plus the number of earlier pairs of the chunk with that
// expert: the pairs' experts and their ranks within each warp (match_any) are found in
// parallel, then the warps take their turns in order to add the earlier warps' counts.
static_assert(kRouteChunk == 1024, "route_scatter_kernel maps one chunk to one 1024-thread block");
__global__ void __launch_bounds__(1024) route_scatter_kernel(const int32_t* __restrict__ idx, int64_t R, int k, int E,
                                                             const int32_t* __restrict__ chunk_base,
                                                             int32_t* __restrict__ row_token,
                                                             int32_t* __restrict__ row_slot,
                                                             int32_t* __restrict__ row_of) {
  extern __shared__ int32_t sm[];
  int32_t* seen = sm;      // [E] pairs of the chunk placed so far, per expert
  int32_t* base = sm + E;  // [E] the chunk's first row per expert
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int64_t chunk = blockIdx.x;
  for (int e = tid; e < E; e += blockDim.x) {
    seen[e] = 0;
    base[e] = chunk_base[chunk * E + e];
  }
  const int64_t gi = chunk * kRouteChunk + tid;
  int err = 0;
  const int e = gi < R ? pair_expert(idx, gi, k, E, &err) : -1;
  const int key = e >= 0 ? e : -1 - lane;  // unmatched keys for dropped pairs
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const int before = __popc(peers & ((1u << lane) - 1u));
  __syncthreads();
  int pos = -1;
  for (int turn = 0; turn < 32; ++turn) {
    if (w == turn) {
      if (e >= 0) pos = base[e] + seen[e] + before;
      __syncwarp();
      if (e >= 0 && before == 0) seen[e] += __popc(peers);
    }
    __syncthreads();
  }
  if (gi < R) {
    row_of[gi] = pos;
    if (pos >= 0) {
      const int64_t t = gi / k;
      row_token[pos] = (int32_t)t;
      row_slot[pos] = (int32_t)(gi - t * k);
    }
  }
}

// ------------------------------------------------------------------------- activations

// E4M3 / INT8: one warp per row, scale fp32(row amax / 448) or fp32(row amax / 127).  CODES
// (E4M3): also the code bytes of the row (8 bytes per 8 elements) and the row's scale.
template <int QK, bool CODES = false>
__global__ void __launch_bounds__(256) act_quant_row_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                            int64_t rows, int64_t cols, const int32_t* dev_rows,
                                                            uint2* __restrict__ codes = nullptr,
                                                            float* __restrict__ row_scale = nullptr) {
  const int64_t nrows = dev_rows ? (int64_t)*dev_rows : rows;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t c8 = cols / 8;
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; r < nrows; r += warps) {
    const uint4* src = in + r * c8;
    float amax = 0.0f;
    for (int64_t c = lane; c < c8; c += 32) {
      float v[8];
      unpack8(src[c], v);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
    amax = warp_max(amax);
    const float s = __fdiv_rn(amax, QK == kQE4M3 ? 448.0f : 127.0f);
    if constexpr (CODES) {
      if (lane == 0) row_scale[r] = s;
    }
    for (int64_t c = lane; c < c8; c += 32) {
      float v[8];
      unpack8(src[c], v);
      if constexpr (CODES) {
        uint32_t cw[2];
        fakequant_e4m3_codes<8, true>(v, s, cw);
        codes[r * c8 + c] = make_uint2(cw[0], cw[1]);
      } else {
        fakequant_act_inplace<QK, 8>(v, s);
      }
      out[r * c8 + c] = pack8(v);
    }
  }
}

// Activation fake-quant of rows of at most LPR * 16 * NB elements (the per-row grids E4M3 /
// INT8, and kQE2M1G), LPR lanes per row (a warp takes 32 / LPR rows at once), the row held in
// registers between the amax and the quantization: sub-lane l of a row holds its 16-element
// blocks l, l + LPR, ... (one 256-bit load each).  CODES (E4M3): also the row's code bytes and
// scale.
template <int AQ, int LPR, int NB, bool CODES = false>
__global__ void __launch_bounds__(256) act_quant_row_reg_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                                int64_t rows, int64_t cols, const int32_t* dev_rows,
                                                                uint4* __restrict__ codes = nullptr,
                                                                float* __restrict__ row_scale = nullptr) {
  constexpr int RPW = 32 / LPR;  // rows per warp at once
  const int64_t nrows = dev_rows ? (int64_t)*dev_rows : rows;
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR;
  const int64_t groups = (int64_t)gridDim.x * (blockDim.x / 32) * RPW;
  const int nb = (int)(cols / 16);
  for (int64_t r0 = ((int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * RPW; r0 < nrows; r0 += groups) {
    const int64_t r = r0 + lane / LPR;
    const bool live = r < nrows;  // the warp stays together for the shuffles; dead rows load nothing
    const uint4* src = in + r * nb * 2;
    uint4 v[NB][2];
    float bmax[NB];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int b = sub + LPR * i;
      bmax[i] = 0.0f;
      if (live && b < nb) {
        ld_nc_256(src + 2 * b, v[i][0], v[i][1]);
        float f[16];
        unpack8(v[i][0], f);
        unpack8(v[i][1], f + 8);
#pragma unroll
        for (int e = 0; e < 16; ++e) bmax[i] = fmaxf(bmax[i], fabsf(f[e]));
        amax = fmaxf(amax, bmax[i]);
      }
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    float s_row, r_g = 0.0f;
    if constexpr (AQ == kQE2M1G) {
      s_row = deploy_tensor_scale(__fdiv_rn(amax, 6.0f));  // the row's tensor scale g
      r_g = s_row == 0.0f ? 0.0f : __frcp_rn(s_row);
    } else {
      s_row = __fdiv_rn(amax, AQ == kQE4M3 ? 448.0f : 127.0f);
    }
    if constexpr (CODES) {
      if (live && sub == 0) row_scale[r] = s_row;
    }
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int b = sub + LPR * i;
      if (live && b < nb) {
        float f[16];
        unpack8(v[i][0], f);
        unpack8(v[i][1], f + 8);
        if constexpr (AQ == kQE2M1G) {
          fakequant_act_inplace<kQE2M1, 16>(f, deployed_scale_r(__fdiv_rn(bmax[i], 6.0f), s_row, r_g));
        } else if constexpr (CODES) {
          uint32_t cw[4];
          fakequant_e4m3_codes<16, true>(f, s_row, cw);
          codes[r * nb + b] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        } else {
          fakequant_act_inplace<AQ, 16>(f, s_row);
        }
        out[r * nb * 2 + 2 * b] = pack8(f);
        out[r * nb * 2 + 2 * b + 1] = pack8(f + 8);
      }
    }
  }
}

// Deployed-nvfp4 activations (kQE2M1G): one warp per row.  The row's tensor scale g =
// fp32(fp32(row amax / 6) / 448) (the largest of the row's block scales fp32(block amax / 6),
// divided by 448: fp32 rounding is monotone, so it is the block scale of the row amax); then
// each 16-element block is fake-quantized on E2M1 with s_q = fp32(e4m3(fp32(sb / g)) * g),
// sb = fp32(block amax / 6).
__global__ void __launch_bounds__(256) act_quant_row_e2m1g_kernel(const uint4* __restrict__ in,
                                                                  uint4* __restrict__ out, int64_t rows,
                                                                  int64_t cols, const int32_t* dev_rows) {
  const int64_t nrows = dev_rows ? (int64_t)*dev_rows : rows;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t c16 = cols / 16;
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; r < nrows; r += warps) {
    const uint4* src = in + r * c16 * 2;
    float amax = 0.0f;
    for (int64_t c = lane; c < c16; c += 32) {
      float v[16];
      unpack8(src[2 * c], v);
      unpack8(src[2 * c + 1], v + 8);
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
    const float g = deploy_tensor_scale(__fdiv_rn(warp_max(amax), 6.0f));
    for (int64_t c = lane; c < c16; c += 32) {
      float v[16];
      unpack8(src[2 * c], v);
      unpack8(src[2 * c + 1], v + 8);
      float bmax = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
      fakequant_act_inplace<kQE2M1, 16>(v, deployed_scale(__fdiv_rn(bmax, 6.0f), g));
      out[r * c16 * 2 + 2 * c] = pack8(v);
      out[r * c16 * 2 + 2 * c + 1] = pack8(v + 8);
    }
  }
}

// Deployed nvfp4 weight scales, one CTA per matrix of `per_mat` scales (two tensors in one
// launch: blocks [0, a.n_mat) take tensor a, the rest tensor b).  Pass 1: the matrix's largest
// |s| (block reduction); g = fp32(amax / 448).  Pass 2: s_q = fp32(e4m3(fp32(s / g)) * g), written
// in place or to another buffer (plain loads: the buffers may be the same).
struct DeployJob {
  const float* s;
  float* sq;
  int64_t n_mat, per_mat;
};

__global__ void __launch_bounds__(1024) deploy_scales_kernel(DeployJob a, DeployJob b) {
  __shared__ float red[32];
  const bool second = blockIdx.x >= a.n_mat;
  const float* s = second ? b.s : a.s;
  float* sq = second ? b.sq : a.sq;
  const int64_t per = second ? b.per_mat : a.per_mat;
  const int64_t m = second ? (int64_t)blockIdx.x - a.n_mat : (int64_t)blockIdx.x;
  const float4* src = reinterpret_cast<const float4*>(s + m * per);
  float4* dst = reinterpret_cast<float4*>(sq + m * per);
  const int64_t n4 = per / 4;
  float amax = 0.0f;
#pragma unroll 4
  for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 v = src[i];
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.0f;
    v = warp_max(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float g = deploy_tensor_scale(red[0]);
  const float r = g == 0.0f ? 0.0f : __frcp_rn(g);
#pragma unroll 4
  for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 v = src[i];
    dst[i] = make_float4(deployed_scale_r(v.x, g, r), deployed_scale_r(v.y, g, r), deployed_scale_r(v.z, g, r),
                         deployed_scale_r(v.w, g, r));
  }
}

// The same in parallel over many CTAs, for the layer calls (their workspace holds the
// per-matrix words): grid (parts, matrices of a then b).  deploy_amax_kernel: each CTA's slice
// max |s|, combined per matrix with atomicMax on the bit patterns (non-negative floats order as
// their bits; amax_bits zeroed first); deploy_g_kernel: gr[m] = (g, RN(1 / g)), g = fp32(amax /
// 448); deploy_round_kernel: s_q for every scale (the fake-quant pass does the same inline).
__device__ __forceinline__ void deploy_job(const DeployJob& a, const DeployJob& b, int m_all, const float** s,
                                           float** sq, int64_t* per) {
  const bool second = m_all >= a.n_mat;
  const int64_t m = second ? m_all - a.n_mat : m_all;
  *per = second ? b.per_mat : a.per_mat;
  *s = (second ? b.s : a.s) + m * *per;
  float* base = second ? b.sq : a.sq;
  *sq = base ? base + m * *per : nullptr;
}

__global__ void __launch_bounds__(256) deploy_amax_kernel(DeployJob a, DeployJob b, uint32_t* __restrict__ amax_bits) {
  __shared__ float red[8];
  const float* s;
  float* sq;
  int64_t per;
  deploy_job(a, b, (int)blockIdx.y, &s, &sq, &per);
  const int64_t n4 = per / 4;
  const int64_t slice = (n4 + gridDim.x - 1) / gridDim.x;
  const int64_t lo = (int64_t)blockIdx.x * slice, hi = lo + slice < n4 ? lo + slice : n4;
  const float4* src = reinterpret_cast<const float4*>(s);
  float amax = 0.0f;
#pragma unroll 4
  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    const float4 v = __ldg(src + i);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = red[0];
    for (int i = 1; i < (int)(blockDim.x / 32); ++i) v = fmaxf(v, red[i]);
    if (lo < hi) atomicMax(amax_bits + blockIdx.y, __float_as_uint(v));
  }
}

__global__ void deploy_g_kernel(const uint32_t* __restrict__ amax_bits, float2* __restrict__ gr, int n) {
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m < n) {
    const float g = deploy_tensor_scale(__uint_as_float(amax_bits[m]));
    gr[m] = make_float2(g, g == 0.0f ? 0.0f : __frcp_rn(g));
  }
}

__global__ void __launch_bounds__(256) deploy_round_kernel(DeployJob a, DeployJob b, const float2* __restrict__ gr) {
  const float* s;
  float* sq;
  int64_t per;
  deploy_job(a, b, (int)blockIdx.y, &s, &sq, &per);
  const float2 g = gr[blockIdx.y];
  const float4* src = reinterpret_cast<const float4*>(s);
  float4* dst = reinterpret_cast<float4*>(sq);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < per / 4; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = __ldg(src + i);
    dst[i] = make_float4(deployed_scale_r(v.x, g.x, g.y), deployed_scale_r(v.y, g.x, g.y),
                         deployed_scale_r(v.z, g.x, g.y), deployed_scale_r(v.w, g.x, g.y));
  }
}

// Zero the padding rows (row_token < 0) of a routed-row buffer below *dev_rpad: each warp
// tests 32 rows at a time and clears the padding ones (c16 16-byte chunks per row).
__device__ __forceinline__ void zero_pad_rows(uint4* __restrict__ dst, const int32_t* __restrict__ row_token,
                                              int64_t c16, const int32_t* dev_rpad, int64_t w0, int64_t warps,
                                              int lane) {
  if (!dev_rpad) return;  // rows without padding (the exchange pieces of an expert-parallel split)
  const int64_t rpad = *dev_rpad;
  for (int64_t g = w0; g * 32 < rpad; g += warps) {
    const int64_t r = g * 32 + lane;
    const bool pad = r < rpad && __ldg(row_token + r) < 0;
    unsigned m = __ballot_sync(0xffffffffu, pad);
    while (m) {
      const int i = __ffs(m) - 1;
      m &= m - 1;
      uint4* d = dst + (g * 32 + i) * c16;
      for (int64_t c = lane; c < c16; c += 32) d[c] = make_uint4(0, 0, 0, 0);
    }
  }
}

constexpr int kScatterNB = 4;  // 16-element blocks per lane per pass over a row chunk
constexpr int kStageChunk = 32 * kScatterNB * 2;  // 16-byte units of one staged row chunk (4 KB)
constexpr int kDyScatterSmem = 8 * 2 * kStageChunk * 16;  // two staged chunks per warp, 8 warps

__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"((uint32_t)__cvta_generic_to_shared(src_smem)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_one() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_done() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_smem_to_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Forward gather, one warp per token: the token's row of x is read once, fake-quantized on
// the activation grid (E2M1 per 16-element block with scale fp32(block amax / 6); E4M3 /
// INT8 per row with fp32(row amax / 448) / fp32(row amax / 127); or not at all), written to
// xq (when the grid quantizes) and to each routed row of the token; then the padding rows
// are zeroed.  Lane l holds the 16-element blocks l, l + 32, ... of a 128 x 16-element
// chunk of the row.  The quantized chunk is staged in the warp's 4 KB of shared memory and
// lane j < k copies it to routed row j with one bulk copy (plain per-thread stores of the
// same rows ran at two thirds of the speed).  CODES (E4M3): each routed row also gets the
// E4M3 code bytes of its elements in a1q (16 bytes per block, staged and bulk-copied the same
// way) and sa_tok[t] the token's scale.
template <int AQ, bool CODES = false>
__global__ void __launch_bounds__(256) scatter_tokens_kernel(const uint4* __restrict__ x, uint4* __restrict__ xq,
                                                             uint4* __restrict__ a1, const int32_t* __restrict__ row_of,
                                                             const int32_t* __restrict__ row_token, int64_t T, int k,
                                                             int64_t nblk, const int32_t* dev_rpad,
                                                             uint4* __restrict__ a1q = nullptr,
                                                             float* __restrict__ sa_tok = nullptr) {
  constexpr int NB = kScatterNB;
  __shared__ __align__(128) uint4 stage_all[8][kStageChunk];
  __shared__ __align__(128) uint4 cstage_all[CODES ? 8 : 1][CODES ? kStageChunk / 2 : 1];
  const int lane = threadIdx.x & 31;
  uint4* stage = stage_all[threadIdx.x / 32];
  uint4* cstage = cstage_all[CODES ? threadIdx.x / 32 : 0];
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  for (int64_t t = w0; t < T; t += warps) {
    const int32_t my_row = lane < k ? __ldg(row_of + t * k + lane) : -1;
    const uint4* src = x + t * nblk * 2;
    float s_row = 0.0f;  // the row's scale (E4M3, INT8) or tensor scale g (kQE2M1G)
    if constexpr (AQ == kQE4M3 || AQ == kQInt8 || AQ == kQE2M1G) {
      float amax = 0.0f;
      for (int64_t b = lane; b < nblk; b += 32) {
        float f[16];
        unpack8(__ldg(src + 2 * b), f);
        unpack8(__ldg(src + 2 * b + 1), f + 8);
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
      }
      if constexpr (AQ == kQE2M1G)
        s_row = deploy_tensor_scale(__fdiv_rn(warp_max(amax), 6.0f));
      else
        s_row = __fdiv_rn(warp_max(amax), AQ == kQE4M3 ? 448.0f : 127.0f);
      if constexpr (CODES) {
        if (lane == 0) sa_tok[t] = s_row;
      }
    }
    for (int64_t b0 = 0; b0 < nblk; b0 += 32 * NB) {
      uint4 v[NB][2];
      uint4 cd[CODES ? NB : 1];
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const int64_t b = b0 + 32 * i + lane;
        if (b < nblk) {
          v[i][0] = __ldg(src + 2 * b);
          v[i][1] = __ldg(src + 2 * b + 1);
        }
      }
      if constexpr (AQ != kQNone) {
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int64_t b = b0 + 32 * i + lane;
          if (b < nblk) {
            float f[16];
            unpack8(v[i][0], f);
            unpack8(v[i][1], f + 8);
            float sc = s_row;
            if constexpr (AQ == kQE2M1 || AQ == kQE2M1G) {
              float amax = 0.0f;
#pragma unroll
              for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(f[e]));
              sc = __fdiv_rn(amax, 6.0f);
              if constexpr (AQ == kQE2M1G) sc = deployed_scale(sc, s_row);
            }
            if constexpr (CODES) {
              uint32_t cw[4];
              fakequant_e4m3_codes<16, true>(f, sc, cw);
              cd[i] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            } else {
              fakequant_act_inplace<AQ == kQE2M1G ? kQE2M1 : AQ, 16>(f, sc);
            }
            v[i][0] = pack8(f);
            v[i][1] = pack8(f + 8);
            uint4* o = xq + t * nblk * 2 + 2 * b;
            o[0] = v[i][0];
            o[1] = v[i][1];
          }
        }
      }
      if (lane < k) bulk_wait_read_all();  // the previous chunk's copies have read the stage
      __syncwarp();
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const int64_t b = b0 + 32 * i + lane;
        if (b < nblk) {
          stage[2 * (32 * i + lane)] = v[i][0];
          stage[2 * (32 * i + lane) + 1] = v[i][1];
          if constexpr (CODES) cstage[32 * i + lane] = cd[i];
        }
      }
      fence_smem_to_async();
      __syncwarp();
      if (lane < k) {
        const int64_t nb_here = nblk - b0 < 32 * NB ? nblk - b0 : 32 * NB;
        if (my_row >= 0) {
          bulk_store(a1 + (int64_t)my_row * nblk * 2 + 2 * b0, stage, (uint32_t)(nb_here * 32));
          if constexpr (CODES) bulk_store(a1q + (int64_t)my_row * nblk + b0, cstage, (uint32_t)(nb_here * 16));
        }
        bulk_commit_group();
      }
    }
  }
  if (lane < k) bulk_wait_done();
  zero_pad_rows(a1, row_token, nblk * 2, dev_rpad, w0, warps, lane);
  if constexpr (CODES) zero_pad_rows(a1q, row_token, nblk, dev_rpad, w0, warps, lane);
}

// ------------------------------------------------------------------------- combine

// one warp per token; fixed slot order j = 0..k-1, fp32 sums.  KC > 0 fixes k at compile time
// so that the k row loads of a column chunk are all in flight together.
template <int KC>
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ row_of,
                                                      const float* __restrict__ p, uint4* __restrict__ out, int64_t T,
                                                      int k_rt, int64_t c8) {
  const int k = KC > 0 ? KC : k_rt;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; t < T; t += warps) {
    if constexpr (KC > 0) {
      int32_t rows[KC];
      float pw[KC];
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        rows[j] = __ldg(row_of + t * KC + j);
        pw[j] = p ? __ldg(p + t * KC + j) : 1.0f;
      }
      for (int64_t c = lane; c < c8; c += 32) {
        uint4 v[KC];
#pragma unroll
        for (int j = 0; j < KC; ++j) v[j] = rows[j] >= 0 ? __ldg(y + (int64_t)rows[j] * c8 + c) : make_uint4(0, 0, 0, 0);
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < KC; ++j) {
          if (rows[j] < 0) continue;
          float f[8];
          unpack8(v[j], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(pw[j], f[i], acc[i]);
        }
        out[t * c8 + c] = pack8(acc);
      }
    } else {
      for (int64_t c = lane; c < c8; c += 32) {
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int j = 0; j < k; ++j) {
          const int32_t r = __ldg(row_of + t * k + j);
          if (r < 0) continue;
          const float pj = p ? __ldg(p + t * k + j) : 1.0f;
          float v[8];
          unpack8(__ldg(y + (int64_t)r * c8 + c), v);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(pj, v[i], acc[i]);
        }
        out[t * c8 + c] = pack8(acc);
      }
    }
  }
}

// Backward gather, one warp per token: for each routed row r of the token (slot j),
// dy[r] = bf16(fp32(p[t, j] * dout[t])) and dprobs[t, j] = <dout[t], y[r]> (fp32, each lane
// over its blocks in order, then a warp sum; 0 for a dropped pair); dout[t] is read from
// memory once and from L1 for the later slots.  Each scaled row chunk is staged in one of
// the warp's two 4 KB buffers (dynamic shared memory, kDyScatterSmem per block) and lane 0
// writes it with one bulk copy.  Then the padding rows of dy are zeroed.
__global__ void __launch_bounds__(256) dy_scatter_kernel(const uint4* __restrict__ dout, const float* __restrict__ p,
                                                         const int32_t* __restrict__ row_of,
                                                         const int32_t* __restrict__ row_token,
                                                         const uint4* __restrict__ y, uint4* __restrict__ dy,
                                                         float* __restrict__ dprobs, int64_t T, int k, int64_t nblk,
                                                         const int32_t* dev_rpad) {
  constexpr int NB = kScatterNB;
  extern __shared__ __align__(128) uint4 dy_stage[];
  const int lane = threadIdx.x & 31;
  uint4* stage0 = dy_stage + (threadIdx.x / 32) * 2 * kStageChunk;
  uint32_t buf = 0;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  for (int64_t t = w0; t < T; t += warps) {
    const int32_t my_row = lane < k ? __ldg(row_of + t * k + lane) : -1;
    const float my_p = lane < k ? __ldg(p + t * k + lane) : 0.0f;
    const uint4* g = dout + t * nblk * 2;
    for (int j = 0; j < k; ++j) {
      const int32_t r = __shfl_sync(0xffffffffu, my_row, j);
      const float pj = __shfl_sync(0xffffffffu, my_p, j);
      float dot = 0.0f;
      if (r >= 0) {
        const uint4* yr = y + (int64_t)r * nblk * 2;
        for (int64_t b0 = 0; b0 < nblk; b0 += 32 * NB) {
          uint4 gv[NB][2], yv[NB][2];
#pragma unroll
          for (int i = 0; i < NB; ++i) {
            const int64_t b = b0 + 32 * i + lane;
            if (b < nblk) {
              gv[i][0] = __ldg(g + 2 * b);
              gv[i][1] = __ldg(g + 2 * b + 1);
              if (dprobs) {
                yv[i][0] = __ldcs(yr + 2 * b);
                yv[i][1] = __ldcs(yr + 2 * b + 1);
              }
            }
          }
          uint4* stg = stage0 + buf * kStageChunk;
          if (lane == 0) bulk_wait_read_one();  // the copy issued from this buffer last time has read it
          __syncwarp();
#pragma unroll
          for (int i = 0; i < NB; ++i) {
            const int64_t b = b0 + 32 * i + lane;
            if (b < nblk) {
              float f[16];
              unpack8(gv[i][0], f);
              unpack8(gv[i][1], f + 8);
              if (dprobs) {
                float yf[16];
                unpack8(yv[i][0], yf);
                unpack8(yv[i][1], yf + 8);
#pragma unroll
                for (int e = 0; e < 16; ++e) dot = fmaf(f[e], yf[e], dot);
              }
#pragma unroll
              for (int e = 0; e < 16; ++e) f[e] = __fmul_rn(pj, f[e]);
              stg[2 * (32 * i + lane)] = pack8(f);
              stg[2 * (32 * i + lane) + 1] = pack8(f + 8);
            }
          }
          fence_smem_to_async();
          __syncwarp();
          if (lane == 0) {
            const int64_t nb_here = nblk - b0 < 32 * NB ? nblk - b0 : 32 * NB;
            bulk_store(dy + (int64_t)r * nblk * 2 + 2 * b0, stg, (uint32_t)(nb_here * 32));
            bulk_commit_group();
          }
          buf ^= 1u;
        }
      }
      if (dprobs) {
        dot = warp_sum(dot);
        if (lane == 0) dprobs[t * k + j] = dot;
      }
    }
  }
  if (lane == 0) bulk_wait_done();
  zero_pad_rows(dy, row_token, nblk * 2, dev_rpad, w0, warps, lane);
}

__global__ void __launch_bounds__(256) scale_reduce_kernel(const float* __restrict__ part, float* __restrict__ ds,
                                                           int64_t n, int nparts, int accumulate) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float acc = accumulate ? ds[i] : 0.0f;
    for (int j = 0; j < nparts; ++j) acc += part[i * nparts + j];
    ds[i] = acc;
  }
}

__global__ void __launch_bounds__(256) quotient_check_kernel(const float* __restrict__ w, const float* __restrict__ s,
                                                             float* __restrict__ fast, float* __restrict__ ieee,
                                                             int64_t n, int mode) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float wi = w[i], si = s[i];
    float x;
    if (mode == 1 && scale_in_fast_range(si)) {
      quotients_unguarded<1>(&wi, si, &x);
    } else {
      quotients<1>(&wi, si, &x);
    }
    fast[i] = x;
    ieee[i] = quotient(wi, si);
  }
}

}  // namespace

cudaError_t launch_quotient_check(const float* w, const float* s, float* fast, float* ieee, int64_t n, int mode,
                                  cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  quotient_check_kernel<<<grid_for(n, 256, 8), 256, 0, st>>>(w, s, fast, ieee, n, mode);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------- launchers

cudaError_t launch_fakequant(int fmt, const void* w, const float* s, void* out, int64_t rows, int64_t K,
                             cudaStream_t st, void* codes) {
  const uint64_t nchunks = (uint64_t)rows * (uint64_t)(K / 16);
  if (nchunks == 0) return cudaSuccess;
  const int grid = grid_for((int64_t)nchunks, 256, 3);
  const uint4* wi = static_cast<const uint4*>(w);
  uint4* o = static_cast<uint4*>(out);
  prof_begin(QAD_K_FAKEQUANT, st);
  switch (weight_kind(fmt)) {
    case kQE2M1: fakequant_kernel<kQE2M1><<<grid, 256, 0, st>>>(wi, s, o, nchunks, 1u); break;
    case kQInt4: fakequant_kernel<kQInt4><<<grid, 256, 0, st>>>(wi, s, o, nchunks, 8u); break;
    case kQE4M3:
      if (codes)
        fakequant_kernel<kQE4M3, true><<<grid, 256, 0, st>>>(wi, s, o, nchunks, (uint32_t)(K / 16),
                                                             static_cast<uint4*>(codes));
      else
        fakequant_kernel<kQE4M3><<<grid, 256, 0, st>>>(wi, s, o, nchunks, (uint32_t)(K / 16));
      break;
    default: fakequant_kernel<kQInt8><<<grid, 256, 0, st>>>(wi, s, o, nchunks, (uint32_t)(K / 16)); break;
  }
  prof_end(QAD_K_FAKEQUANT, st);
  return cudaGetLastError();
}

cudaError_t launch_deploy_scales(const float* s_a, float* sq_a, int64_t n_a, int64_t per_a, const float* s_b,
                                 float* sq_b, int64_t n_b, int64_t per_b, cudaStream_t st) {
  if (n_a + n_b == 0) return cudaSuccess;
  if (n_a + n_b > 0x7fffffff) return cudaErrorInvalidValue;
  prof_begin(QAD_K_DEPLOY_SCALES, st);
  deploy_scales_kernel<<<(unsigned)(n_a + n_b), 1024, 0, st>>>(DeployJob{s_a, sq_a, n_a, per_a},
                                                               DeployJob{s_b, sq_b, n_b, per_b});
  prof_end(QAD_K_DEPLOY_SCALES, st);
  return cudaGetLastError();
}

cudaError_t launch_deploy_tensor_scales(const float* s_a, int64_t n_a, int64_t per_a, const float* s_b, int64_t n_b,
                                        int64_t per_b, uint32_t* amax_bits, float2* gr, cudaStream_t st) {
  const int64_t n = n_a + n_b;
  if (n == 0) return cudaSuccess;
  if (n > 65535) return cudaErrorInvalidValue;
  prof_begin(QAD_K_DEPLOY_SCALES, st);
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t) * (size_t)n, st);
  if (e != cudaSuccess) return e;
  const int64_t per4 = (per_a > per_b ? per_a : per_b) / 4;
  const int parts = (int)((per4 + 2047) / 2048);  // ~8 float4 per thread of a 256-thread CTA
  deploy_amax_kernel<<<dim3((unsigned)(parts > 0 ? parts : 1), (unsigned)n), 256, 0, st>>>(
      DeployJob{s_a, nullptr, n_a, per_a}, DeployJob{s_b, nullptr, n_b, per_b}, amax_bits);
  deploy_g_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(amax_bits, gr, (int)n);
  prof_end(QAD_K_DEPLOY_SCALES, st);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_deploy_round(const float* s_a, float* sq_a, int64_t n_a, int64_t per_a, const float* s_b,
                                float* sq_b, int64_t n_b, int64_t per_b, const float2* gr, cudaStream_t st) {
  const int64_t n = n_a + n_b;
  if (n == 0) return cudaSuccess;
  if (n > 65535) return cudaErrorInvalidValue;
  prof_begin(QAD_K_DEPLOY_SCALES, st);
  const int64_t per4 = (per_a > per_b ? per_a : per_b) / 4;
  const int64_t want = (per4 + 1023) / 1024;  // ~4 float4 per thread
  deploy_round_kernel<<<dim3((unsigned)(want > 0 ? want : 1), (unsigned)n), 256, 0, st>>>(
      DeployJob{s_a, sq_a, n_a, per_a}, DeployJob{s_b, sq_b, n_b, per_b}, gr);
  prof_end(QAD_K_DEPLOY_SCALES, st);
  return cudaGetLastError();
}

cudaError_t launch_fakequant_deployed(const void* w, const float* s, void* out, int64_t rows, int64_t K,
                                      int64_t rows_per_mat, const float2* gr, float* sq, cudaStream_t st) {
  const uint64_t nchunks = (uint64_t)rows * (uint64_t)(K / 16);
  if (nchunks == 0) return cudaSuccess;
  if (nchunks >= (1ull << 32) || rows_per_mat <= 0) return cudaErrorInvalidValue;  // 32-bit chunk -> matrix map
  const int grid = grid_for((int64_t)nchunks, 256, 3);
  prof_begin(QAD_K_FAKEQUANT, st);
  fakequant_kernel<kQE2M1, false, true><<<grid, 256, 0, st>>>(static_cast<const uint4*>(w), s,
                                                              static_cast<uint4*>(out), nchunks, 1u, nullptr, gr,
                                                              (uint32_t)(rows_per_mat * (K / 16)), sq);
  prof_end(QAD_K_FAKEQUANT, st);
  return cudaGetLastError();
}

cudaError_t launch_route(const int32_t* idx, const Layout& L, uint8_t* ws, cudaStream_t st) {
  return launch_route_ptrs(idx, L.R, (int)L.k, (int)L.E, L.nchunks, reinterpret_cast<int32_t*>(ws + L.header),
                           reinterpret_cast<int32_t*>(ws + L.chunk_counts), reinterpret_cast<int32_t*>(ws + L.chunk_base),
                           reinterpret_cast<int32_t*>(ws + L.counts), reinterpret_cast<int32_t*>(ws + L.offs),
                           reinterpret_cast<int32_t*>(ws + L.mtile_expert), reinterpret_cast<int32_t*>(ws + L.row_token),
                           reinterpret_cast<int32_t*>(ws + L.row_slot), reinterpret_cast<int32_t*>(ws + L.row_of), st);
}

cudaError_t launch_route_ptrs(const int32_t* idx, int64_t R, int k, int E, int64_t nchunks, int32_t* hdr,
                              int32_t* chunk_counts, int32_t* chunk_base, int32_t* counts, int32_t* offs,
                              int32_t* mtile_expert, int32_t* row_token, int32_t* row_slot, int32_t* row_of,
                              cudaStream_t st) {
  prof_begin(QAD_K_ROUTE, st);
  if (nchunks > 0) {
    route_hist_kernel<<<(unsigned)nchunks, 256, E * sizeof(int32_t), st>>>(idx, R, k, E, chunk_counts, hdr);
  }
  route_scan_kernel<<<1, 1024, 0, st>>>(nchunks, E, chunk_counts, chunk_base, counts, offs, mtile_expert, row_token,
                                        row_slot, hdr);
  if (nchunks > 0) {
    route_scatter_kernel<<<(unsigned)nchunks, kRouteChunk, 2 * E * sizeof(int32_t), st>>>(idx, R, k, E, chunk_base,
                                                                                         row_token, row_slot, row_of);
  }
  prof_end(QAD_K_ROUTE, st);
  if (nchunks > 0) note_launches(2);
  return cudaGetLastError();
}

namespace {
template <int LPR, int NB>
void act_quant_rows_reg(int kind, const uint4* in, uint4* out, int64_t rows, int64_t cols, const int32_t* dev_rows,
                        uint4* codes, float* row_scale, cudaStream_t st) {
  const int grid = grid_for((rows * LPR + 31) / 32 * 32, 256, 8);
  if (kind == kQE2M1G)
    act_quant_row_reg_kernel<kQE2M1G, LPR, NB><<<grid, 256, 0, st>>>(in, out, rows, cols, dev_rows);
  else if (kind == kQE4M3 && codes)
    act_quant_row_reg_kernel<kQE4M3, LPR, NB, true><<<grid, 256, 0, st>>>(in, out, rows, cols, dev_rows, codes,
                                                                          row_scale);
  else if (kind == kQE4M3)
    act_quant_row_reg_kernel<kQE4M3, LPR, NB><<<grid, 256, 0, st>>>(in, out, rows, cols, dev_rows);
  else
    act_quant_row_reg_kernel<kQInt8, LPR, NB><<<grid, 256, 0, st>>>(in, out, rows, cols, dev_rows);
}
}  // namespace

cudaError_t launch_act_quant_rows(int kind, const void* in, void* out, int64_t rows, int64_t cols,
                                  const int32_t* dev_rows, cudaStream_t st, void* codes, float* row_scale) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (kind != kQE4M3 && kind != kQInt8 && kind != kQE2M1G) return cudaErrorInvalidValue;
  if (kind == kQE2M1G && (cols % 16 || codes)) return cudaErrorInvalidValue;
  prof_begin(QAD_K_ACT_QUANT, st);
  const int grid = grid_for(rows * 32, 256, 8);
  const uint4* src = static_cast<const uint4*>(in);
  uint4* dst = static_cast<uint4*>(out);
  const int64_t nb = cols / 16;
  uint4* cd = static_cast<uint4*>(codes);
  if (cols % 16 == 0 && nb <= 128) {
    // rows of up to 2048 elements stay in registers between the row amax and the quantization;
    // up to 768 elements two rows per warp (16 lanes each), so each warp has more loads in flight
    if (nb <= 48)
      act_quant_rows_reg<16, 3>(kind, src, dst, rows, cols, dev_rows, cd, row_scale, st);
    else if (nb <= 96)
      act_quant_rows_reg<32, 3>(kind, src, dst, rows, cols, dev_rows, cd, row_scale, st);
    else
      act_quant_rows_reg<32, 4>(kind, src, dst, rows, cols, dev_rows, cd, row_scale, st);
  } else if (kind == kQE2M1G) {
    act_quant_row_e2m1g_kernel<<<grid, 256, 0, st>>>(src, dst, rows, cols, dev_rows);
  } else if (kind == kQE4M3 && codes) {
    act_quant_row_kernel<kQE4M3, true><<<grid, 256, 0, st>>>(src, dst, rows, cols, dev_rows,
                                                            static_cast<uint2*>(codes), row_scale);
  } else if (kind == kQE4M3) {
    act_quant_row_kernel<kQE4M3><<<grid, 256, 0, st>>>(src, dst, rows, cols, dev_rows);
  } else {
    act_quant_row_kernel<kQInt8><<<grid, 256, 0, st>>>(src, dst, rows, cols, dev_rows);
  }
  prof_end(QAD_K_ACT_QUANT, st);
  return cudaGetLastError();
}

cudaError_t launch_scatter_tokens(int aq, const void* x, void* xq, void* a1, const int32_t* row_of,
                                  const int32_t* row_token, int64_t T, int k, int64_t d, const int32_t* dev_rpad,
                                  cudaStream_t st, void* a1q, float* sa_tok) {
  if (T == 0) return cudaSuccess;
  prof_begin(QAD_K_GATHER, st);
  const int grid = grid_for(T * 32, 256, 8);
  const uint4* xs = static_cast<const uint4*>(x);
  uint4* q = static_cast<uint4*>(xq);
  uint4* a = static_cast<uint4*>(a1);
  const int64_t nblk = d / 16;
  if (aq == kQE2M1) scatter_tokens_kernel<kQE2M1><<<grid, 256, 0, st>>>(xs, q, a, row_of, row_token, T, k, nblk, dev_rpad);
  else if (aq == kQE2M1G)
    scatter_tokens_kernel<kQE2M1G><<<grid, 256, 0, st>>>(xs, q, a, row_of, row_token, T, k, nblk, dev_rpad);
  else if (aq == kQE4M3 && a1q)
    scatter_tokens_kernel<kQE4M3, true><<<grid, 256, 0, st>>>(xs, q, a, row_of, row_token, T, k, nblk, dev_rpad,
                                                              static_cast<uint4*>(a1q), sa_tok);
  else if (aq == kQE4M3) scatter_tokens_kernel<kQE4M3><<<grid, 256, 0, st>>>(xs, q, a, row_of, row_token, T, k, nblk, dev_rpad);
  else if (aq == kQInt8) scatter_tokens_kernel<kQInt8><<<grid, 256, 0, st>>>(xs, q, a, row_of, row_token, T, k, nblk, dev_rpad);
  else scatter_tokens_kernel<kQNone><<<grid, 256, 0, st>>>(xs, q, a, row_of, row_token, T, k, nblk, dev_rpad);
  prof_end(QAD_K_GATHER, st);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y, const int32_t* row_of, const float* p, void* out, int64_t T, int k,
                           int64_t d, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int id = p ? QAD_K_COMBINE : QAD_K_DX_COMBINE;
  prof_begin(id, st);
  const int grid = grid_for(T * 32, 256, 8);
  const uint4* yy = static_cast<const uint4*>(y);
  uint4* o = static_cast<uint4*>(out);
  if (k == 8) combine_kernel<8><<<grid, 256, 0, st>>>(yy, row_of, p, o, T, k, d / 8);
  else if (k == 2) combine_kernel<2><<<grid, 256, 0, st>>>(yy, row_of, p, o, T, k, d / 8);
  else if (k == 4) combine_kernel<4><<<grid, 256, 0, st>>>(yy, row_of, p, o, T, k, d / 8);
  else combine_kernel<0><<<grid, 256, 0, st>>>(yy, row_of, p, o, T, k, d / 8);
  prof_end(id, st);
  return cudaGetLastError();
}

cudaError_t launch_dy_scatter(const void* dout, const float* p, const int32_t* row_of, const int32_t* row_token,
                              const void* y, void* dy, float* dprobs, int64_t T, int k, int64_t d,
                              const int32_t* dev_rpad, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(dy_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kDyScatterSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  prof_begin(QAD_K_DY_GATHER, st);
  dy_scatter_kernel<<<grid_for(T * 32, 256, 8), 256, kDyScatterSmem, st>>>(
      static_cast<const uint4*>(dout), p, row_of, row_token, static_cast<const uint4*>(y), static_cast<uint4*>(dy),
      dprobs, T, k, d / 16, dev_rpad);
  prof_end(QAD_K_DY_GATHER, st);
  return cudaGetLastError();
}

cudaError_t launch_scale_reduce(const float* part, float* ds, int64_t n, int nparts, int accumulate,
                                cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  prof_begin(QAD_K_SCALE_REDUCE, st);
  scale_reduce_kernel<<<grid_for(n, 256, 8), 256, 0, st>>>(part, ds, n, nparts, accumulate);
  prof_end(QAD_K_SCALE_REDUCE, st);
  return cudaGetLastError();
}

}  // namespace qad
