// Routing permutation for callers that cannot allocate device memory.
//
// qad_moe_fwd keeps the routing scratch (per-chunk expert histograms, each chunk's first
// row per expert, the expert of every 128-row tile, a small header) in the caller's
// workspace.  Some callers have no workspace to give: code that runs while a stream is
// being captured into a CUDA graph and may not call cudaMalloc, or a runtime that owns
// all device memory and hands a plugin only its inputs and outputs.  For them this file
// keeps that scratch in one file-scope device array of fixed size, so the entry point
// needs nothing but its inputs and outputs.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace qad {
namespace {

constexpr int kMaxE = QAD_NOALLOC_MAX_EXPERTS;
constexpr int64_t kMaxPairs = QAD_NOALLOC_MAX_PAIRS;
constexpr int64_t kMaxChunks = (kMaxPairs + kRouteChunk - 1) / kRouteChunk;
constexpr int64_t kMaxRows = (kMaxPairs + (int64_t)(kTileRows - 1) * kMaxE + kTileRows - 1) / kTileRows * kTileRows;
constexpr int64_t kHdrInts = 64;
constexpr int64_t kChunkInts = kMaxChunks * kMaxE;
constexpr int64_t kTileInts = kMaxRows / kTileRows;
constexpr int64_t kScratchInts = kHdrInts + 2 * kChunkInts + kTileInts;

// The scratch: header | chunk histograms | chunk first rows | tile experts (534 KB).
// Every GPU that loads the library holds one copy until the process exits.
static __device__ __align__(256) int32_t g_route_scratch[kScratchInts];

constexpr int kMaxDevices = 64;
int32_t* g_scratch_dev[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device (with that
// device current) and cached.
int scratch_on_current_device(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QAD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return QAD_ERR_CUDA;
    g_scratch_dev[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_dev[dev];
  return QAD_OK;
}

}  // namespace
}  // namespace qad

extern "C" int qad_route_permute_noalloc(const int32_t* topk_idx, int64_t T, int32_t topk, int32_t E,
                                         int32_t* row_token, int32_t* row_slot, int32_t* row_of, int32_t* offsets,
                                         int32_t* counts, int32_t* header, qad_stream_t stream) {
  using namespace qad;
  if (T < 0 || topk <= 0 || E <= 0 || topk > 32 || topk > E) return QAD_ERR_INVALID_ARG;
  const int64_t R = T * (int64_t)topk;
  if (E > kMaxE || R > kMaxPairs) return QAD_ERR_SCRATCH_LIMIT;
  if (!row_token || !row_slot || !offsets || !counts || !header) return QAD_ERR_INVALID_ARG;
  if (R > 0 && (!topk_idx || !row_of)) return QAD_ERR_INVALID_ARG;
  int32_t* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != QAD_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t* hdr = scratch;
  int32_t* chunk_counts = hdr + kHdrInts;
  int32_t* chunk_base = chunk_counts + kChunkInts;
  int32_t* mtile_expert = chunk_base + kChunkInts;
  const int64_t nchunks = (R + kRouteChunk - 1) / kRouteChunk;
  // the header keeps the previous call's error bits and counters: clear it first
  if (cudaMemsetAsync(hdr, 0, kHdrInts * sizeof(int32_t), st) != cudaSuccess) return QAD_ERR_CUDA;
  if (launch_route_ptrs(topk_idx, R, topk, E, nchunks, hdr, chunk_counts, chunk_base, counts, offsets, mtile_expert,
                        row_token, row_slot, row_of, st) != cudaSuccess)
    return QAD_ERR_CUDA;
  if (cudaMemcpyAsync(header, hdr, 4 * sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return QAD_ERR_CUDA;
  return QAD_OK;
}
