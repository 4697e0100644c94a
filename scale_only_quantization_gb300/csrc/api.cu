// C ABI of the scale-only QAD MoE library: argument checks, workspace layout, the call
// sequences of the forward / input-gradient / scale-gradient passes, and kernel timing.
//
// The passes follow the AngelSlim mcore_qad walkthrough (nxmr.cn/news/131691): weights
// fake-quantized as quantize->dequantize(W; s) with gradients reaching only s, activations
// fake-quantized before each quantized matmul, router unquantized (section 二.3); the
// whole expert stack fake-quantized in one pass and every expert run as one grouped GEMM
// (section 二.4).
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace qad {

namespace {

constexpr size_t kAlign = 1024;
size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------- profiler

struct Pending {
  int id;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_free_events;
double g_ms[QAD_K_COUNT];
int64_t g_launches[QAD_K_COUNT];
std::atomic<int64_t> g_launch_total{0};
thread_local Pending t_open = {-1, nullptr, nullptr};

cudaEvent_t take_event() {
  if (!g_free_events.empty()) {
    cudaEvent_t e = g_free_events.back();
    g_free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

int g_sms[64] = {0};

}  // namespace

int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!g_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return g_sms[dev];
}

void prof_begin(int id, cudaStream_t st) {
  g_launch_total.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) return;
  t_open.id = id;
  t_open.a = take_event();
  t_open.b = take_event();
  cudaEventRecord(t_open.a, st);
}

void note_launches(int n) { g_launch_total.fetch_add(n, std::memory_order_relaxed); }

void prof_end(int id, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on || t_open.id != id || !t_open.a) return;
  cudaEventRecord(t_open.b, st);
  g_pending.push_back(t_open);
  t_open = {-1, nullptr, nullptr};
}

int layout_of(const qad_moe_shape& s, Layout* L) {
  if (s.T < 0 || s.d <= 0 || s.F <= 0 || s.E <= 0 || s.topk <= 0) return QAD_ERR_INVALID_ARG;
  if (s.fmt < QAD_FMT_NVFP4 || s.fmt > QAD_FMT_NVFP4_E4M3) return QAD_ERR_INVALID_ARG;
  if (s.reserved != 0 || (s.flags & ~(QAD_FLAG_STASH_H | QAD_FLAG_NO_QUANT | QAD_FLAG_RECOMPUTE |
                                       QAD_FLAG_NATIVE_FP8 | QAD_FLAG_SMEM_DEQUANT | QAD_FLAG_DEQUANT_DUMP)))
    return QAD_ERR_INVALID_ARG;
  if ((s.flags & QAD_FLAG_NATIVE_FP8) && (s.fmt != QAD_FMT_FP8_ROW || (s.flags & QAD_FLAG_NO_QUANT)))
    return QAD_ERR_INVALID_ARG;
  const bool dq = (s.flags & QAD_FLAG_SMEM_DEQUANT) != 0;
  if (dq && (s.flags & (QAD_FLAG_NO_QUANT | QAD_FLAG_NATIVE_FP8))) return QAD_ERR_INVALID_ARG;
  if ((s.flags & QAD_FLAG_DEQUANT_DUMP) && !dq) return QAD_ERR_INVALID_ARG;
  // d and F: multiples of 16 (the scale blocks, activation blocks and 32-byte row sectors), of 128
  // for the INT4 formats (their group-128 scales run along both d and F); the E4M3 tensor path and
  // the in-GEMM dequant take only whole 256 x 128 tiles (d % 256 == 0, F % 128 == 0)
  const int64_t mult = weight_kind(s.fmt) == kQInt4 ? 128 : 16;
  if (s.d % mult || s.F % mult) return QAD_ERR_UNSUPPORTED;
  if ((s.flags & (QAD_FLAG_NATIVE_FP8 | QAD_FLAG_SMEM_DEQUANT)) && (s.d % 256 || s.F % 128)) return QAD_ERR_UNSUPPORTED;
  if (s.E > 1024 || s.topk > 32 || s.topk > s.E) return QAD_ERR_UNSUPPORTED;
  const int64_t R = s.T * (int64_t)s.topk;
  const int64_t Rmax = (R + (int64_t)(kTileRows - 1) * s.E + kTileRows - 1) / kTileRows * kTileRows;
  if (Rmax >= (int64_t(1) << 31) || s.E * 2 * s.F >= (int64_t(1) << 31) || s.E * s.d >= (int64_t(1) << 31))
    return QAD_ERR_UNSUPPORTED;
  L->T = s.T; L->d = s.d; L->F = s.F; L->E = s.E; L->k = s.topk; L->R = R; L->Rmax = Rmax;
  L->nchunks = (R + kRouteChunk - 1) / kRouteChunk;
  const int64_t d = s.d, F = s.F, E = s.E;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = up(o + bytes); return at; };
  L->header = take(256);
  L->counts = take(4 * E);
  L->offs = take(4 * (E + 1));
  L->chunk_counts = take(4 * (size_t)(L->nchunks * E));
  L->chunk_base = take(4 * (size_t)(L->nchunks * E));
  L->mtile_expert = take(4 * (size_t)(Rmax / kTileRows));
  L->ptile_row0 = take(4 * (size_t)(Rmax / kTileRows));
  L->ptile_expert = take(4 * (size_t)(Rmax / kTileRows));
  L->wg_order = take(4 * (size_t)E);
  L->row_token = take(4 * (size_t)Rmax);
  L->row_slot = take(4 * (size_t)Rmax);
  L->row_of = take(4 * (size_t)R);
  L->xq = take(2 * (size_t)(s.T * d));
  // the fake-quantized weight copies (not with QAD_FLAG_SMEM_DEQUANT, unless dumped)
  const bool copies = !dq || (s.flags & QAD_FLAG_DEQUANT_DUMP);
  L->w13h = take(copies ? 2 * (size_t)(E * 2 * F * d) : 0);
  L->w2h = take(copies ? 2 * (size_t)(E * d * F) : 0);
  L->w_copies = copies;
  L->a1 = take(2 * (size_t)(Rmax * d));
  // with QAD_FLAG_RECOMPUTE (and d >= 2F) Z1 lives in Y's region: it only exists between the
  // dgrad call's recompute and its SwiGLU backward, after Y has been read for dprobs
  const bool z1_in_y = (s.flags & QAD_FLAG_RECOMPUTE) && d >= 2 * F;
  L->z1 = z1_in_y ? 0 : take(2 * (size_t)(Rmax * 2 * F));
  L->h = take(2 * (size_t)(Rmax * F));
  L->hh = take(2 * (size_t)(Rmax * F));
  L->y = take(2 * (size_t)(Rmax * d));
  if (z1_in_y) L->z1 = L->y;
  L->dy = take(2 * (size_t)(Rmax * d));
  L->dz1 = take(2 * (size_t)(Rmax * 2 * F));
  L->da1 = take(2 * (size_t)(Rmax * d));
  L->part13 = take(4 * (size_t)(E * 2 * F * ((d + 127) / 128) * 2));
  L->part2 = take(4 * (size_t)(E * d * ((F + 127) / 128) * 2));
  L->native_fp8 = (s.flags & QAD_FLAG_NATIVE_FP8) != 0;
  L->w13q = L->w2q = L->a1q = L->hq = L->sa_tok = L->sh_row = 0;
  if (L->native_fp8) {
    L->w13q = take((size_t)(E * 2 * F * d));
    L->w2q = take((size_t)(E * d * F));
    L->a1q = take((size_t)(Rmax * d));
    L->hq = take((size_t)(Rmax * F));
    L->sa_tok = take(4 * (size_t)(s.T > 0 ? s.T : 1));
    L->sh_row = take(4 * (size_t)Rmax);
  }
  L->deployed = s.fmt == QAD_FMT_NVFP4_E4M3;
  L->s13q = L->deployed ? take(4 * (size_t)(E * 2 * F * (d / 16))) : 0;
  L->s2q = L->deployed ? take(4 * (size_t)(E * d * (F / 16))) : 0;
  L->deploy_tmp = L->deployed ? take(4 * (size_t)(2 * E) + 8 * (size_t)(2 * E)) : 0;
  L->total = o;
  return QAD_OK;
}

}  // namespace qad

using namespace qad;

namespace {

int to_status(cudaError_t e) { return e == cudaSuccess ? QAD_OK : QAD_ERR_CUDA; }

#define QAD_TRY(expr)                     \
  do {                                    \
    cudaError_t e_ = (expr);              \
    if (e_ != cudaSuccess) return QAD_ERR_CUDA; \
  } while (0)

int check_layer(const qad_moe_shape* s, void* ws, size_t ws_bytes, Layout* L) {
  if (!s) return QAD_ERR_INVALID_ARG;
  const int rc = layout_of(*s, L);
  if (rc != QAD_OK) return rc;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return QAD_ERR_INVALID_ARG;
  if (ws_bytes < L->total) return QAD_ERR_WORKSPACE;
  return QAD_OK;
}

bool ok_ptr(const void* p) { return p && aligned16(p); }

// GEMM context of one call.  With QAD_FLAG_NO_QUANT the GEMMs read the caller's raw weights
// and the fc1 epilogue applies no activation quantizer; otherwise they read the
// fake-quantized copies the forward wrote.
GemmCtx gemm_ctx(const Layout& L, uint8_t* wsb, const qad_moe_shape& s, const void* w13, const void* w2,
                 cudaStream_t st) {
  const bool no_quant = (s.flags & QAD_FLAG_NO_QUANT) != 0;
  const bool dq = (s.flags & QAD_FLAG_SMEM_DEQUANT) != 0;
  const bool dump = (s.flags & QAD_FLAG_DEQUANT_DUMP) != 0;
  GemmCtx c;
  c.L = &L;
  c.ws = wsb;
  c.wq = weight_kind(s.fmt);
  c.aq = no_quant ? kQNone : act_kind(s.fmt);
  c.flags = s.flags;
  c.st = st;
  c.w13h = (no_quant || dq) ? w13 : static_cast<const void*>(wsb + L.w13h);
  c.w2h = (no_quant || dq) ? w2 : static_cast<const void*>(wsb + L.w2h);
  c.s13 = nullptr;
  c.s2 = nullptr;
  c.dq = dq;
  c.dump13 = dump ? static_cast<void*>(wsb + L.w13h) : nullptr;
  c.dump2 = dump ? static_cast<void*>(wsb + L.w2h) : nullptr;
  return c;
}

}  // namespace

extern "C" {

const char* qad_status_string(int status) {
  switch (status) {
    case QAD_OK: return "ok";
    case QAD_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size or flag)";
    case QAD_ERR_UNSUPPORTED:
      return "unsupported shape (needs d, F multiples of 16 -- of 128 for INT4 weights, d % 256 == 0 and F % 128 == 0 "
             "with the E4M3 tensor path or the in-GEMM dequant --, topk <= min(E, 32), E <= 1024)";
    case QAD_ERR_WORKSPACE: return "workspace smaller than qad_moe_workspace_bytes()";
    case QAD_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
    case QAD_ERR_DEVICE: return "device error word set (bad or repeated routing index, or a pipeline timeout)";
    case QAD_ERR_SCRATCH_LIMIT: return "problem larger than the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

int qad_fakequant_fwd(int fmt, const void* w, const float* scale, void* w_hat, int64_t E, int64_t N, int64_t K,
                      qad_stream_t stream) {
  if (fmt < QAD_FMT_NVFP4 || fmt > QAD_FMT_NVFP4_E4M3) return QAD_ERR_INVALID_ARG;
  if (fmt == QAD_FMT_NVFP4_E4M3) return QAD_ERR_UNSUPPORTED;  // deploy the scales, then QAD_FMT_NVFP4
  if (E < 0 || N < 0 || K <= 0) return QAD_ERR_INVALID_ARG;
  if (K % 16 || (weight_kind(fmt) == kQInt4 && K % 128)) return QAD_ERR_UNSUPPORTED;
  if (E * N == 0) return QAD_OK;
  if (!ok_ptr(w) || !ok_ptr(scale) || !ok_ptr(w_hat)) return QAD_ERR_INVALID_ARG;
  return to_status(launch_fakequant(fmt, w, scale, w_hat, E * N, K, reinterpret_cast<cudaStream_t>(stream)));
}

int qad_nvfp4_deploy_scales(const float* s, float* s_q, int64_t n_mat, int64_t per_mat, qad_stream_t stream) {
  if (n_mat < 0 || per_mat <= 0 || per_mat % 4 || n_mat > 0x7fffffff) return QAD_ERR_INVALID_ARG;
  if (n_mat == 0) return QAD_OK;
  if (!ok_ptr(s) || !ok_ptr(s_q)) return QAD_ERR_INVALID_ARG;
  return to_status(launch_deploy_scales(s, s_q, n_mat, per_mat, nullptr, nullptr, 0, 0,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

size_t qad_moe_workspace_bytes(const qad_moe_shape* s) {
  if (!s) return 0;
  Layout L;
  return layout_of(*s, &L) == QAD_OK ? L.total : 0;
}

namespace qad {
namespace {
// Per-device side stream and events of the forward's fork / join: the routing kernels
// (latency-bound, a few tens of microseconds) run beside the HBM-bound weight fake-quant.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[64];

cudaError_t side_stream(SideStream** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  SideStream& ss = g_side[dev];
  if (!ss.s) {
    if ((e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &ss;
  return cudaSuccess;
}
}  // namespace
}  // namespace qad

int qad_moe_fwd(const qad_moe_shape* s, const void* x, const int32_t* topk_idx, const float* topk_w,
                const void* w13, const float* s13, const void* w2, const float* s2, void* out, void* ws,
                size_t ws_bytes, qad_stream_t stream) {
  Layout L;
  int rc = check_layer(s, ws, ws_bytes, &L);
  if (rc != QAD_OK) return rc;
  if (L.T > 0 && (!ok_ptr(x) || !ok_ptr(topk_idx) || !ok_ptr(topk_w) || !ok_ptr(out))) return QAD_ERR_INVALID_ARG;
  if (!ok_ptr(w13) || !ok_ptr(s13) || !ok_ptr(w2) || !ok_ptr(s2)) return QAD_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  int32_t* hdr = reinterpret_cast<int32_t*>(wsb + L.header);
  const int32_t* rpad = hdr + HDR_RPAD;
  const int fmt = s->fmt;
  const bool no_quant = (s->flags & QAD_FLAG_NO_QUANT) != 0;
  QAD_TRY(cudaMemsetAsync(hdr, 0, 256, st));
  const bool f8 = L.native_fp8;  // E4M3 codes for the fp8 tensor path as well
  const int32_t* row_token = reinterpret_cast<const int32_t*>(wsb + L.row_token);
  GemmCtx c = gemm_ctx(L, wsb, *s, w13, w2, st);
  // deployed nvfp4: every consumer of the weight scales (the fake-quant pass or the in-GEMM
  // dequant here, the dequant and the LSQ epilogues in the backward calls) reads s_q
  const bool deploy = L.deployed && !no_quant;
  const float* s13u = deploy ? reinterpret_cast<const float*>(wsb + L.s13q) : s13;
  const float* s2u = deploy ? reinterpret_cast<const float*>(wsb + L.s2q) : s2;
  c.s13 = s13u;
  c.s2 = s2u;
  {
    // routing and the activation gather on the side stream, the weight fake-quant on the
    // caller's: the latency-bound routing hides under the fake-quant, and the two HBM-bound
    // passes share the memory system; joined before the GEMMs
    std::lock_guard<std::mutex> lk(g_side_mu);
    SideStream* ss = nullptr;
    QAD_TRY(side_stream(&ss));
    QAD_TRY(cudaEventRecord(ss->fork, st));
    QAD_TRY(cudaStreamWaitEvent(ss->s, ss->fork, 0));
    QAD_TRY(launch_route(topk_idx, L, wsb, ss->s));
    QAD_TRY(launch_scatter_tokens(c.aq, x, wsb + L.xq, wsb + L.a1, reinterpret_cast<const int32_t*>(wsb + L.row_of),
                                  row_token, L.T, (int)L.k, L.d, rpad, ss->s, f8 ? wsb + L.a1q : nullptr,
                                  f8 ? reinterpret_cast<float*>(wsb + L.sa_tok) : nullptr));
    QAD_TRY(cudaEventRecord(ss->join, ss->s));
    if (deploy) {
      // the tensor scale of each expert matrix; the deployed block scales are then made by the
      // weight fake-quant pass itself (or, with the in-GEMM dequant, by a rounding pass)
      uint32_t* amax_bits = reinterpret_cast<uint32_t*>(wsb + L.deploy_tmp);
      const float2* gr = reinterpret_cast<const float2*>(wsb + L.deploy_tmp + 4 * 2 * L.E);
      QAD_TRY(launch_deploy_tensor_scales(s13, L.E, 2 * L.F * (L.d / 16), s2, L.E, L.d * (L.F / 16), amax_bits,
                                          const_cast<float2*>(gr), st));
      if (c.dq) {
        QAD_TRY(launch_deploy_round(s13, const_cast<float*>(s13u), L.E, 2 * L.F * (L.d / 16), s2,
                                    const_cast<float*>(s2u), L.E, L.d * (L.F / 16), gr, st));
      } else {
        QAD_TRY(launch_fakequant_deployed(w13, s13, wsb + L.w13h, L.E * 2 * L.F, L.d, 2 * L.F, gr,
                                          const_cast<float*>(s13u), st));
        QAD_TRY(launch_fakequant_deployed(w2, s2, wsb + L.w2h, L.E * L.d, L.F, L.d, gr + L.E, const_cast<float*>(s2u),
                                          st));
      }
    } else if (!no_quant && !c.dq) {  // with QAD_FLAG_SMEM_DEQUANT the GEMMs fake-quantize the weights themselves
      QAD_TRY(launch_fakequant(fmt, w13, s13u, wsb + L.w13h, L.E * 2 * L.F, L.d, st, f8 ? wsb + L.w13q : nullptr));
      QAD_TRY(launch_fakequant(fmt, w2, s2u, wsb + L.w2h, L.E * L.d, L.F, st, f8 ? wsb + L.w2q : nullptr));
    }
    QAD_TRY(cudaStreamWaitEvent(st, ss->join, 0));
  }
  QAD_TRY(gemm_prepare(c));
  QAD_TRY(gemm_fc1(c, (s->flags & QAD_FLAG_RECOMPUTE) ? kFc1NoZ1 : kFc1Full));
  if (act_needs_row(c.aq))
    QAD_TRY(launch_act_quant_rows(c.aq, wsb + L.h, wsb + L.hh, L.Rmax, L.F, rpad, st, f8 ? wsb + L.hq : nullptr,
                                  f8 ? reinterpret_cast<float*>(wsb + L.sh_row) : nullptr));
  QAD_TRY(gemm_fc2(c));
  QAD_TRY(launch_combine(wsb + L.y, reinterpret_cast<const int32_t*>(wsb + L.row_of), topk_w, out, L.T, (int)L.k,
                         L.d, st));
  return QAD_OK;
}

int qad_moe_bwd_dgrad(const qad_moe_shape* s, const void* dout, const float* topk_w, const void* w13,
                      const float* s13, const void* w2, const float* s2, void* dx, float* dprobs, void* ws,
                      size_t ws_bytes, qad_stream_t stream) {
  Layout L;
  int rc = check_layer(s, ws, ws_bytes, &L);
  if (rc != QAD_OK) return rc;
  if (L.T > 0 && (!ok_ptr(dout) || !ok_ptr(topk_w) || !ok_ptr(dx))) return QAD_ERR_INVALID_ARG;
  if (dprobs && !ok_ptr(dprobs)) return QAD_ERR_INVALID_ARG;
  if (!ok_ptr(w13) || !ok_ptr(s13) || !ok_ptr(w2) || !ok_ptr(s2)) return QAD_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  int32_t* hdr = reinterpret_cast<int32_t*>(wsb + L.header);
  const int32_t* rpad = hdr + HDR_RPAD;
  QAD_TRY(launch_dy_scatter(dout, topk_w, reinterpret_cast<const int32_t*>(wsb + L.row_of),
                            reinterpret_cast<const int32_t*>(wsb + L.row_token), wsb + L.y, wsb + L.dy, dprobs, L.T,
                            (int)L.k, L.d, rpad, st));
  GemmCtx c = gemm_ctx(L, wsb, *s, w13, w2, st);
  const bool deploy = L.deployed && !(s->flags & QAD_FLAG_NO_QUANT);  // the forward's s_q
  c.s13 = deploy ? reinterpret_cast<const float*>(wsb + L.s13q) : s13;
  c.s2 = deploy ? reinterpret_cast<const float*>(wsb + L.s2q) : s2;
  if (s->flags & QAD_FLAG_RECOMPUTE) QAD_TRY(gemm_fc1(c, kFc1Z1Only));  // Z1 again, after Y's last use
  QAD_TRY(gemm_dgrad_fc2(c));
  QAD_TRY(gemm_dgrad_fc1(c));
  QAD_TRY(launch_combine(wsb + L.da1, reinterpret_cast<const int32_t*>(wsb + L.row_of), nullptr, dx, L.T, (int)L.k,
                         L.d, st));
  return QAD_OK;
}

int qad_moe_bwd_scalegrad(const qad_moe_shape* s, const void* w13, const float* s13, const void* w2, const float* s2,
                          float* ds13, float* ds2, int accumulate, void* ws, size_t ws_bytes, qad_stream_t stream) {
  Layout L;
  int rc = check_layer(s, ws, ws_bytes, &L);
  if (rc != QAD_OK) return rc;
  if (!ok_ptr(w13) || !ok_ptr(s13) || !ok_ptr(w2) || !ok_ptr(s2) || !ok_ptr(ds13) || !ok_ptr(ds2))
    return QAD_ERR_INVALID_ARG;
  if (s->flags & QAD_FLAG_NO_QUANT) return QAD_ERR_INVALID_ARG;  // no scales without quantizers
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  GemmCtx c = gemm_ctx(L, wsb, *s, w13, w2, st);
  // deployed nvfp4: the LSQ factor is taken at the forward's s_q, and the gradient reaches s
  // straight through the E4M3 rounding (ds13 / ds2 are the gradients of s_q)
  const float* s13u = L.deployed ? reinterpret_cast<const float*>(wsb + L.s13q) : s13;
  const float* s2u = L.deployed ? reinterpret_cast<const float*>(wsb + L.s2q) : s2;
  QAD_TRY(gemm_wgrad_fc2(c, w2, s2u, ds2, accumulate ? 1 : 0));
  QAD_TRY(gemm_wgrad_fc1(c, w13, s13u, ds13, accumulate ? 1 : 0));
  return QAD_OK;
}

int qad_moe_combine(const void* rows, const int32_t* row_of, const float* p, void* out, int64_t T, int32_t topk,
                    int64_t d, qad_stream_t stream) {
  if (T < 0 || d <= 0 || d % 16 || topk < 1 || topk > 32) return QAD_ERR_INVALID_ARG;
  if (T == 0) return QAD_OK;
  if (!ok_ptr(rows) || !ok_ptr(row_of) || !ok_ptr(out) || (p && !ok_ptr(p))) return QAD_ERR_INVALID_ARG;
  return to_status(launch_combine(rows, row_of, p, out, T, topk, d, reinterpret_cast<cudaStream_t>(stream)));
}

int qad_check_device_error(void* ws, qad_stream_t stream, int32_t* code) {
  if (!ws) return QAD_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess) return QAD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return QAD_ERR_CUDA;
  if (code) *code = v;
  return v == 0 ? QAD_OK : QAD_ERR_DEVICE;
}

int qad_moe_debug_view(const qad_moe_shape* s, int which, size_t* byte_offset, int64_t* numel) {
  if (!s || !byte_offset || !numel) return QAD_ERR_INVALID_ARG;
  Layout L;
  const int rc = layout_of(*s, &L);
  if (rc != QAD_OK) return rc;
  const int64_t d = L.d, F = L.F, E = L.E, Rm = L.Rmax;
  size_t off = 0;
  int64_t n = 0;
  switch (which) {
    case QAD_VIEW_HEADER: off = L.header; n = 64; break;
    case QAD_VIEW_OFFSETS: off = L.offs; n = E + 1; break;
    case QAD_VIEW_COUNTS: off = L.counts; n = E; break;
    case QAD_VIEW_ROW_TOKEN: off = L.row_token; n = Rm; break;
    case QAD_VIEW_ROW_SLOT: off = L.row_slot; n = Rm; break;
    case QAD_VIEW_ROW_OF: off = L.row_of; n = L.R; break;
    case QAD_VIEW_W13_HAT: off = L.w13h; n = L.w_copies ? E * 2 * F * d : 0; break;
    case QAD_VIEW_W2_HAT: off = L.w2h; n = L.w_copies ? E * d * F : 0; break;
    case QAD_VIEW_A1: off = L.a1; n = Rm * d; break;
    case QAD_VIEW_Z1: off = L.z1; n = Rm * 2 * F; break;
    case QAD_VIEW_H: off = L.h; n = Rm * F; break;
    case QAD_VIEW_H_HAT: off = L.hh; n = Rm * F; break;
    case QAD_VIEW_Y: off = L.y; n = Rm * d; break;
    case QAD_VIEW_DY: off = L.dy; n = Rm * d; break;
    case QAD_VIEW_DZ1: off = L.dz1; n = Rm * 2 * F; break;
    case QAD_VIEW_DA1: off = L.da1; n = Rm * d; break;
    case QAD_VIEW_XQ: off = L.xq; n = L.T * d; break;
    case QAD_VIEW_W13_CODES: off = L.w13q; n = L.native_fp8 ? E * 2 * F * d : 0; break;
    case QAD_VIEW_W2_CODES: off = L.w2q; n = L.native_fp8 ? E * d * F : 0; break;
    case QAD_VIEW_A1_CODES: off = L.a1q; n = L.native_fp8 ? Rm * d : 0; break;
    case QAD_VIEW_H_CODES: off = L.hq; n = L.native_fp8 ? Rm * F : 0; break;
    case QAD_VIEW_A_SCALE: off = L.sa_tok; n = L.native_fp8 ? L.T : 0; break;
    case QAD_VIEW_H_SCALE: off = L.sh_row; n = L.native_fp8 ? Rm : 0; break;
    case QAD_VIEW_S13_DEPLOYED: off = L.s13q; n = L.deployed ? E * 2 * F * (d / 16) : 0; break;
    case QAD_VIEW_S2_DEPLOYED: off = L.s2q; n = L.deployed ? E * d * (F / 16) : 0; break;
    default: return QAD_ERR_INVALID_ARG;
  }
  *byte_offset = off;
  *numel = n;
  return QAD_OK;
}

int qad_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
  return QAD_OK;
}

int qad_profile_reset(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return QAD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& pe : g_pending) {
    g_free_events.push_back(pe.a);
    g_free_events.push_back(pe.b);
  }
  g_pending.clear();
  memset(g_ms, 0, sizeof(g_ms));
  memset(g_launches, 0, sizeof(g_launches));
  return QAD_OK;
}

int qad_profile_read(float* ms, int64_t* launches, int n) {
  if (cudaDeviceSynchronize() != cudaSuccess) return QAD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& pe : g_pending) {
    float t = 0.0f;
    if (cudaEventElapsedTime(&t, pe.a, pe.b) == cudaSuccess && pe.id >= 0 && pe.id < QAD_K_COUNT) {
      g_ms[pe.id] += t;
      g_launches[pe.id] += 1;
    }
    g_free_events.push_back(pe.a);
    g_free_events.push_back(pe.b);
  }
  g_pending.clear();
  for (int i = 0; i < n && i < QAD_K_COUNT; ++i) {
    if (ms) ms[i] = (float)g_ms[i];
    if (launches) launches[i] = g_launches[i];
  }
  return QAD_OK;
}

const char* qad_kernel_name(int id) {
  static const char* names[QAD_K_COUNT] = {"fakequant_w", "route_permute", "act_quant", "gather_rows",
                                           "gemm_fc1_swiglu_aq", "gemm_fc2", "combine", "dy_gather",
                                           "gemm_dgrad_fc2_swiglu_bwd", "gemm_dgrad_fc1", "dx_combine",
                                           "gemm_wgrad_fc2_scalegrad", "gemm_wgrad_fc1_scalegrad", "scale_reduce",
                                           "gemm_fc1_recompute", "deploy_scales"};
  return (id >= 0 && id < QAD_K_COUNT) ? names[id] : "unknown";
}

int64_t qad_launch_count(void) { return g_launch_total.load(); }

int qad_debug_wait_timeout(int32_t* err_word, int64_t budget_cycles, qad_stream_t stream) {
  if (!err_word || budget_cycles < 0 || budget_cycles > 2000000000LL) return QAD_ERR_INVALID_ARG;
  return to_status(launch_wait_selftest(err_word, budget_cycles, reinterpret_cast<cudaStream_t>(stream)));
}

int qad_debug_quotient(const float* w, const float* s, float* x_fast, float* x_ieee, int64_t n, int32_t mode,
                       qad_stream_t stream) {
  if (n < 0 || mode < 0 || mode > 1) return QAD_ERR_INVALID_ARG;
  if (n == 0) return QAD_OK;
  if (!w || !s || !x_fast || !x_ieee) return QAD_ERR_INVALID_ARG;
  return to_status(launch_quotient_check(w, s, x_fast, x_ieee, n, mode, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
