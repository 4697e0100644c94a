// Internal interfaces of the scale-only QAD MoE library: workspace layout and launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/qad.h"

namespace qad {

constexpr int kTileRows = 128;     // rows per GEMM tile; every expert's rows are padded to a multiple
constexpr int kRouteChunk = 1024;  // (token, slot) pairs per routing chunk

// Byte offsets of the workspace regions (each 1024-byte aligned).
struct Layout {
  int64_t T, d, F, E, k, R, Rmax, nchunks;
  size_t header, counts, offs, chunk_counts, chunk_base, mtile_expert, ptile_row0, ptile_expert, wg_order, row_token,
      row_slot, row_of;
  size_t xq, w13h, w2h, a1, z1, h, hh, y, dy, dz1, da1, part13, part2;
  // QAD_FLAG_NATIVE_FP8: E4M3 codes of W13, W2, A1 and H, per-token activation scales and
  // per-row H scales (all 0 otherwise)
  bool native_fp8;
  bool w_copies;  // the W13_hat / W2_hat regions exist (not with QAD_FLAG_SMEM_DEQUANT unless dumped)
  size_t w13q, w2q, a1q, hq, sa_tok, sh_row;
  // QAD_FMT_NVFP4_E4M3: the deployed weight scales (0 otherwise)
  bool deployed;
  size_t s13q, s2q, deploy_tmp;  // deploy_tmp: 2E words of matrix amax bits, then 2E (g, 1/g) pairs
  size_t total;
};

// Header words (int32) at the start of the workspace
enum { HDR_ERR = 0, HDR_NMTILES = 1, HDR_RPAD = 2, HDR_NVALID = 3, HDR_NPTILES = 4 };

// Returns a negative qad_status for an unsupported or invalid shape.
int layout_of(const qad_moe_shape& s, Layout* L);

// Profiler / launch accounting (api.cu)
void prof_begin(int kernel_id, cudaStream_t st);
void prof_end(int kernel_id, cudaStream_t st);
void note_launches(int n);  // extra kernels launched inside one profiled region
int num_sms();

// ---- kernels (each returns the launch's cudaError_t) ----
// codes (E4M3 weights only, may be null): the E4M3 code byte of every element, [rows, K]
cudaError_t launch_fakequant(int fmt, const void* w, const float* s, void* out, int64_t rows, int64_t K,
                             cudaStream_t st, void* codes = nullptr);
// deployed nvfp4 weight scales of two tensors in one launch (n_b may be 0): for each of the
// n matrices of `per` scales (per % 4 == 0, 16-byte aligned), s_q = fp32(e4m3(fp32(s / g)) * g),
// g = fp32(max |s| / 448) of that matrix; s_q may alias s
cudaError_t launch_deploy_scales(const float* s_a, float* sq_a, int64_t n_a, int64_t per_a, const float* s_b,
                                 float* sq_b, int64_t n_b, int64_t per_b, cudaStream_t st);
// the same for the layer calls, in parallel: gr[m] = (g, RN(1 / g)) of each of the n_a + n_b
// (<= 65535) matrices (amax_bits: n_a + n_b words of scratch), then s_q either by
// launch_deploy_round or inside the weight fake-quant (launch_fakequant_deployed: nvfp4, writes
// s_q to sq besides w_hat; rows_per_mat rows of K per matrix)
cudaError_t launch_deploy_tensor_scales(const float* s_a, int64_t n_a, int64_t per_a, const float* s_b, int64_t n_b,
                                        int64_t per_b, uint32_t* amax_bits, float2* gr, cudaStream_t st);
cudaError_t launch_deploy_round(const float* s_a, float* sq_a, int64_t n_a, int64_t per_a, const float* s_b,
                                float* sq_b, int64_t n_b, int64_t per_b, const float2* gr, cudaStream_t st);
cudaError_t launch_fakequant_deployed(const void* w, const float* s, void* out, int64_t rows, int64_t K,
                                      int64_t rows_per_mat, const float2* gr, float* sq, cudaStream_t st);
cudaError_t launch_route(const int32_t* idx, const Layout& L, uint8_t* ws, cudaStream_t st);
// the same three routing kernels on explicit buffers (hdr: int32[64], zeroed by the caller;
// chunk_counts / chunk_base: int32[nchunks * E]; mtile_expert: int32[Rmax / 128])
cudaError_t launch_route_ptrs(const int32_t* idx, int64_t R, int k, int E, int64_t nchunks, int32_t* hdr,
                              int32_t* chunk_counts, int32_t* chunk_base, int32_t* counts, int32_t* offs,
                              int32_t* mtile_expert, int32_t* row_token, int32_t* row_slot, int32_t* row_of,
                              cudaStream_t st);
// out[r, :] = AQ(in[r, :]) with activation grid `kind` (kQE4M3 / kQInt8: per row; kQE2M1G: per
// 16 under a row scale) for r < rows (or < *dev_rows when dev_rows != nullptr)
cudaError_t launch_act_quant_rows(int kind, const void* in, void* out, int64_t rows, int64_t cols,
                                  const int32_t* dev_rows, cudaStream_t st, void* codes = nullptr,
                                  float* row_scale = nullptr);
// Per token t: xq[t] = AQ(x[t]) (aq != kQNone) and a1[row_of[t, j]] = AQ(x[t]) for its routed
// rows; the padding rows (row_token < 0) below *dev_rpad are zeroed
cudaError_t launch_scatter_tokens(int aq, const void* x, void* xq, void* a1, const int32_t* row_of,
                                  const int32_t* row_token, int64_t T, int k, int64_t d, const int32_t* dev_rpad,
                                  cudaStream_t st, void* a1q = nullptr, float* sa_tok = nullptr);
// out[t, :] = bf16(sum_j p[t, j] * y[row_of[t, j], :]) (p == nullptr: weight 1)
cudaError_t launch_combine(const void* y, const int32_t* row_of, const float* p, void* out, int64_t T, int k,
                           int64_t d, cudaStream_t st);
// dy[row_of[t, j]] = bf16(p[t, j] * dout[t]); dprobs[t, j] = <dout[t], y[row_of[t, j]]> (0 for a
// dropped pair; dprobs may be null); the padding rows of dy below *dev_rpad are zeroed
cudaError_t launch_dy_scatter(const void* dout, const float* p, const int32_t* row_of, const int32_t* row_token,
                              const void* y, void* dy, float* dprobs, int64_t T, int k, int64_t d,
                              const int32_t* dev_rpad, cudaStream_t st);
// ds[i] = (accumulate ? ds[i] : 0) + sum_j part[i * nparts + j]
cudaError_t launch_scale_reduce(const float* part, float* ds, int64_t n, int nparts, int accumulate,
                                cudaStream_t st);

// fast[i] = the quantizers' reciprocal-based quotient of w[i] / s[i] (mode 0: per-element
// guarded form; mode 1: the block-guarded form), ieee[i] = IEEE division
cudaError_t launch_quotient_check(const float* w, const float* s, float* fast, float* ieee, int64_t n, int mode,
                                  cudaStream_t st);

// ---- grouped GEMMs (gemm.cu) ----
// the GEMMs' bounded mbarrier wait on a barrier nothing arrives on; sets QAD_DEV_TIMEOUT in *err
cudaError_t launch_wait_selftest(int32_t* err, int64_t budget_cycles, cudaStream_t st);
struct GemmCtx {
  const Layout* L;
  uint8_t* ws;
  int wq, aq;  // weight grid (LSQ factor) and activation grid of the fc1 epilogue (kQNone: none)
  int flags;
  cudaStream_t st;
  const void* w13h;  // the weights the GEMMs read: the fake-quantized copies in the workspace,
  const void* w2h;   // or the caller's raw weights for the unquantized teacher pass
  const float* s13;  // the caller's weight scales (read by the native fp8 forward epilogues and,
  const float* s2;   // with dq, by the GEMMs' shared-memory dequant)
  // QAD_FLAG_SMEM_DEQUANT: w13h / w2h are the caller's raw weights and the row-mode GEMMs
  // fake-quantize each weight tile in shared memory; dump13 / dump2 (QAD_FLAG_DEQUANT_DUMP,
  // else null) receive the converted values, laid out like the weights
  bool dq;
  void* dump13;
  void* dump2;
};
cudaError_t gemm_prepare(const GemmCtx& c);     // pair-tile table of the row-mode GEMMs (after routing)
// fc1 epilogue modes: everything; everything but Z1 (recompute, forward); only Z1 (recompute,
// backward: the same mainloop, so the same Z1 bits)
enum { kFc1Full = 0, kFc1NoZ1 = 1, kFc1Z1Only = 2 };
cudaError_t gemm_fc1(const GemmCtx& c, int mode);  // Z1, H, H_hat  <- A1 . W13_hat^T (+ SwiGLU, AQ)
cudaError_t gemm_fc2(const GemmCtx& c);         // Y <- H_hat . W2_hat^T
cudaError_t gemm_dgrad_fc2(const GemmCtx& c);   // dZ1 <- SwiGLU'(dY . W2_hat)
cudaError_t gemm_dgrad_fc1(const GemmCtx& c);   // dA1 <- dZ1 . W13_hat
cudaError_t gemm_wgrad_fc2(const GemmCtx& c, const void* w2, const float* s2, float* ds2, int accumulate);
cudaError_t gemm_wgrad_fc1(const GemmCtx& c, const void* w13, const float* s13, float* ds13, int accumulate);

}  // namespace qad
