// Grouped GEMMs of the scale-only QAD MoE layer on the 5th-generation tensor cores.
//
// "All experts in one grouped GEMM over the token-routed rows" (AngelSlim mcore_qad
// walkthrough, nxmr.cn/news/131691, section 二.4).  One persistent kernel template serves
// the six GEMMs of a fwd + bwd step:
//
//   fc1    Z1 = A1 . W13_hat[e]^T   epilogue: bf16 Z1, SwiGLU, activation fake-quant -> H_hat
//   fc2    Y  = H_hat . W2_hat[e]^T  epilogue: bf16 store
//   dgrad  dH = dY . W2_hat[e]       epilogue: SwiGLU backward -> dZ1 (dH never stored)
//   dgrad  dA1 = dZ1 . W13_hat[e]    epilogue: bf16 store
//   wgrad  dW2 = dY_e^T . H_hat_e    epilogue: x LSQ factor, per-block sums -> ds2 (dW never stored)
//   wgrad  dW13 = dZ1_e^T . A1_e     epilogue: same -> ds13
//
// With E4M3 operands (F8) the forward GEMMs run tcgen05 kind::f8f6f4 on the quantization
// codes and the epilogues multiply each fp32 sum by its activation-row and weight-row scale.
//
// Rows of each expert are padded to a multiple of 128 (zero rows), so a 128-row half tile
// never straddles two experts and a wgrad contraction runs over whole 128-row blocks.
//
// The MMAs run on SM pairs (a cluster of two CTAs, tcgen05 cta_group::2): one
// 256 x BN x 16 MMA issued by the pair's leader reads the 256 rows of A from the two CTAs'
// shared memory (128 each) and the BN columns of B from both (BN/2 each), and writes each
// CTA's 128 rows of the accumulator into that CTA's tensor memory.  Each SM therefore
// loads only half of the B tile: a third fewer operand bytes per FLOP than a one-SM
// 128 x BN tile, which matters because these GEMMs are limited by L2-to-SM bandwidth.
// A row-mode pair tile is two consecutive 128-row blocks of one expert; when an expert
// has an odd number of blocks the second CTA's half of its last tile is dead (computed,
// not stored).
//
// Per CTA (persistent over the pair's tiles): warp 0 issues TMA loads (128B-swizzled
// tiles) into a ring of stages holding one or two 128-byte K atoms per operand row (ATOMS);
// the pair's TMA bytes complete on the leader's "full" barrier; warp 1 of each CTA owns the pair's tensor memory allocation and, in the
// leader, one thread issues the MMAs and commits to both CTAs' "empty" (ring slot free)
// and "full accumulator" barriers at once (multicast); warps 2-9 read their CTA's
// accumulator (two TMEM buffers, so the next tile's MMAs overlap this epilogue) with
// tcgen05.ld and run the fused epilogue, then arrive on the leader's "empty accumulator"
// barrier.  A warp may only read the 32 TMEM lanes of its quadrant (warp id mod 4), so
// each quadrant has two warps, one per column half.  Every wait is bounded: on expiry the CTA
// raises QAD_DEV_TIMEOUT in the workspace error word, drains what it issued and exits.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace qad {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // bf16 K elements in one 128-byte swizzle atom row
// Pipeline stages hold ATOMS 128-byte K atoms per operand row.  Two atoms (8 MMAs per stage)
// halve the per-stage barrier and commit work of the single producer and MMA threads at the
// same bytes of lookahead; measured per GEMM, two atoms help fc1 and the two wgrad GEMMs
// (5-7%) and cost fc2 and the two dgrad GEMMs 1-3%, which keep one.
__host__ __device__ constexpr int bke_of(bool f8, int atoms) { return atoms * (f8 ? 128 : BK); }  // K per stage
constexpr int kAtomsFc1 = 2, kAtomsFc2 = 1, kAtomsDgrad = 1, kAtomsWgrad = 2;
constexpr int kThreads = 320;       // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2-9 epilogue
constexpr int kEpiThreads = 256;
// With the weight operand dequantized in shared memory (DQ), warps 10-13 are converters: they
// fake-quantize each B stage in place after its TMA load and before the MMAs read it.
constexpr int kConvWarps = 4;
constexpr int kConvThreads = 32 * kConvWarps;
__host__ __device__ constexpr int threads_of(bool dq) { return kThreads + (dq ? kConvThreads : 0); }
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz

enum { EPI_FC1 = 0, EPI_STORE = 1, EPI_SWIGLU_BWD = 2, EPI_SCALEGRAD = 3 };

struct Params {
  int32_t* hdr;                 // workspace header ([HDR_ERR], [HDR_NPTILES])
  const int32_t* ptile_row0;    // first row of each row-mode pair tile
  const int32_t* ptile_expert;  // expert of each row-mode pair tile
  const int32_t* wg_order;      // wgrad: experts by decreasing padded row count (tile order)
  const int32_t* poff;          // padded expert offsets [E + 1]
  int E;
  int wgrad;                    // 0: output rows grouped by expert; 1: contraction over an expert's rows
  int n_ntiles;                 // tiles along the GEMM's N
  int n_mtiles_w;               // wgrad: pair tiles along the GEMM's M (weight rows / 256)
  int num_kb;                   // rows mode: K / 64
  int b_rows;                   // rows of the B tensor map per expert
  int F;                        // expert FFN width (fc1 / SwiGLU epilogues)
  int wq, aq, flags;  // weight grid (LSQ), activation grid of the fc1 epilogue (kQNone: none)
  int fc1_mode;       // kFc1Full, kFc1NoZ1 or kFc1Z1Only
  int n_total;        // the GEMM's N (output columns): store tiles past it are skipped
  // E4M3 operands (native fp8): the epilogue multiplies the fp32 sum of row r, column n by
  // row_scale[row_tok ? row_tok[r] : r] * col_scale[e * b_rows + weight row of n]
  const float* row_scale;
  const int32_t* row_tok;
  const float* col_scale;
  __nv_bfloat16* out3; int64_t ld_out2;  // FC1: H, kept besides H_hat with QAD_FLAG_STASH_H
  // (the tiles the epilogues produce are written through the kernel's store tensor maps)
  const __nv_bfloat16* aux; int64_t ld_aux;  // SWIGLU_BWD: Z1
  const __nv_bfloat16* w;  const float* s;   // SCALEGRAD: raw weights [E, Mw, Kw] and scales
  int64_t w_rows, w_cols;
  int w_vec32;  // w is 32-byte aligned: its sectors are read with 256-bit loads
  int s_vec4;   // E2M1 scale rows are 16-byte aligned (w_cols % 64 == 0): 4 scales per vector access
  float* ds; float* part; int accumulate;
  // DQ: the B operand is the raw bf16 weight [E, dq_rows, dq_cols] with scales dq_s; the
  // converters apply bf16(fp32(q(fp32(w / s)) * s)) (grid p.wq) to each B stage in shared
  // memory.  dq_dump (debug, may be null): the converted values are also written there, laid
  // out like the weight.
  const float* dq_s;
  int64_t dq_rows, dq_cols;
  __nv_bfloat16* dq_dump;
};

template <int BN, int ATOMS> struct Cfg {
  static constexpr int A_ATOM = BM * 128;                  // this CTA's 128 rows of A, one atom
  static constexpr int B_ATOM = (BN / 2) * 128;            // this CTA's half of B, one atom
  static constexpr int A_BYTES = ATOMS * A_ATOM;
  static constexpr int B_BYTES = ATOMS * B_ATOM;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (192 * 1024) / STAGE;  // BN = 256: 6 (one atom) or 3; BN = 128: 8 or 4
  static constexpr int RING = STAGES * STAGE;
  static constexpr int SMEM = RING + 512 + 1024;  // + barriers, + alignment slack
  static constexpr int TMEM_COLS = 2 * BN;
};

// Shared memory that the epilogues stage their bf16 outputs in for TMA stores: 4 KB per
// epilogue warp.  The plain store uses it as two 32-row x 32-column boxes (64-byte swizzle),
// the fc1 and SwiGLU-backward epilogues as a ring of four 32-row x 16-column boxes
// (32-byte swizzle).  The scale-gradient epilogue writes no tiles.
constexpr int kStageBox = 32 * 32 * 2;
constexpr int kStageWarp = 4096;
template <int EPI> __host__ __device__ constexpr int staging_bytes() {
  return EPI == EPI_SCALEGRAD ? 0 : (kEpiThreads / 32) * kStageWarp;
}
template <int BN, int EPI, int ATOMS> __host__ __device__ constexpr int smem_bytes() {
  return Cfg<BN, ATOMS>::SMEM + staging_bytes<EPI>();
}

// ---------------------------------------------------------------------------------- PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// The same test with acquire semantics at cluster scope: the phase was completed by release
// arrivals from threads of both CTAs of the pair whose shared-memory writes must be visible.
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, "
      "1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait for the phase with parity `parity` of barrier `bar`: gives up after `budget`
// clock cycles (or as soon as another role of the CTA gave up), raising QAD_DEV_TIMEOUT.
// The first tries are inline: the producer and MMA-issuer threads wait once per k-block, and
// a function call there (with its stack frame) measurably slows every GEMM.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                           long long budget) {
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      *abort_flag = 1;
      atomicOr(err, QAD_DEV_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                          long long budget = kWaitCycles) {
#pragma unroll 1
  for (int i = 0; i < 4; ++i)
    if (mbar_try(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, err, budget);
}

// Bounded wait with cluster-scope acquire (see mbar_try_cluster); the slow path ends with one
// more acquiring test, so a phase it saw complete is also acquired.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err) {
#pragma unroll 1
  for (int i = 0; i < 4; ++i)
    if (mbar_try_cluster(bar, parity)) return true;
  if (!mbar_wait_slow(bar, parity, abort_flag, err, kWaitCycles)) return false;
  return mbar_try_cluster(bar, parity);
}

// Self-check of the timeout path: one thread waits, with the GEMMs' own bounded-wait routine,
// on a barrier that nothing ever arrives on.  It must give up after `budget` cycles and
// raise QAD_DEV_TIMEOUT in *err; nothing faults or hangs.
__global__ void wait_selftest_kernel(int32_t* err, long long budget) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, err, budget);
}

// TMA tile load into this CTA's shared memory; the bytes complete on `bar`, a shared::cluster
// address that may be the pair leader's barrier (cta_group::2).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// TMA tile load into this CTA's shared memory completing on one of its own barriers
__device__ __forceinline__ void tma_load_2d_local(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// TMA tile store from this CTA's shared memory (bulk-group completion, tracked per thread)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N of this thread's bulk groups still read shared memory
template <int N> __device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// wait until all of this thread's bulk groups have completed (writes done)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// make this thread's shared-memory writes visible to the TMA (async proxy)
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Arrive on a barrier of either CTA of the pair.  Relaxed: it only tells the MMA issuer that
// this warp's tensor-memory reads are complete (tcgen05.wait::ld has returned); it must not
// wait for the epilogue's global stores to become visible, which release semantics would.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// Arrive with release semantics at cluster scope: the arriving warp's shared-memory writes
// (already ordered before the tensor cores' reads by fence.proxy.async) become visible to
// the thread that acquires the phase.
__device__ __forceinline__ void mbar_arrive_release_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start >> 4 in [0,14), leading byte offset
// >> 4 in [16,30), stride byte offset >> 4 in [32,46), the fixed 0b001 in [46,49),
// base offset 0 (tiles are 1024-byte aligned), swizzle mode 2 = 128-byte in [61,64).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor: D fp32 (bits 4-5 = 1); A and B types in bits 7-9 and 10-12 (kind::f16:
// bf16 = 1; kind::f8f6f4: E4M3 = 0); A/B major in bits 15/16 (0 = K-major, 1 = MN-major),
// N >> 3 in [17,23), M >> 4 in [24,29); M = 256 for the pair.
template <int N, bool A_MN, bool B_MN, bool F8 = false>
__host__ __device__ constexpr uint32_t instr_desc() {
  return (1u << 4) | (F8 ? 0u : ((1u << 7) | (1u << 10))) | ((A_MN ? 1u : 0u) << 15) | ((B_MN ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)((2 * BM) >> 4) << 24);
}

// One pair MMA, 256 x N x 16 (bf16) or 256 x N x 32 (E4M3: kind::f8f6f4); both read 32 bytes
// of K per operand row.
template <bool F8>
__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  if constexpr (F8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}
// arrive on the barrier at offset `bar` in every CTA of `mask` once the MMAs issued so far are done
__device__ __forceinline__ void mma_commit(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"(mask)
               : "memory");
}

// tcgen05.ld is asynchronous until tcgen05.wait::ld: the loads of the next chunk are issued
// before the current chunk is processed.  The wait takes the destination registers as
// in/out operands so the compiler keeps them untouched until the data has landed.

// 32 consecutive fp32 columns of this thread's TMEM lane (issue only)
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
// 16 consecutive fp32 columns (issue only)
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]) :: "memory");
}
__device__ __forceinline__ void tmem_wait16(uint32_t (&a)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]) :: "memory");
}
__device__ __forceinline__ void tmem_wait16x2(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15]) :: "memory");
}


// ---------------------------------------------------------------------------------- tiles

struct Tile {
  int e, mb, nb, nkb, r0;
  int64_t row_base;  // first output row of this CTA's 128-row half (rows mode) / weight row (wgrad)
  bool live;         // false for the dead second half of an expert's odd last block
};

__device__ __forceinline__ int tile_count(const Params& p) {
  return p.wgrad ? p.E * p.n_mtiles_w * p.n_ntiles : p.hdr[HDR_NPTILES] * p.n_ntiles;
}

__device__ __forceinline__ Tile tile_of(const Params& p, int t, uint32_t rank, int bke) {
  Tile ti;
  if (p.wgrad) {
    const int per_e = p.n_mtiles_w * p.n_ntiles;
    const int k = t / per_e;
    ti.e = __ldg(p.wg_order + k);
    const int rem = t - k * per_e;
    ti.mb = rem / p.n_ntiles;
    ti.nb = rem - ti.mb * p.n_ntiles;
    ti.r0 = __ldg(p.poff + ti.e);
    ti.nkb = (__ldg(p.poff + ti.e + 1) - ti.r0) / bke;
    ti.row_base = (int64_t)ti.mb * (2 * BM) + (int64_t)rank * BM;
    ti.live = true;
  } else {
    const int pt = t / p.n_ntiles;
    ti.mb = pt;
    ti.nb = t - pt * p.n_ntiles;
    ti.e = __ldg(p.ptile_expert + pt);
    ti.r0 = __ldg(p.ptile_row0 + pt) + (int)rank * BM;
    ti.nkb = p.num_kb;
    ti.row_base = ti.r0;
    ti.live = ti.r0 < __ldg(p.poff + ti.e + 1);
  }
  return ti;
}

// ---------------------------------------------------------------------------------- epilogues

// A warp's ring of four 1 KB staging boxes, each 32 rows x 16 bf16 columns in the 32-byte
// swizzle (thread = row; its two 16-byte chunks c at c ^ ((row >> 2) & 1), which keeps the
// shared-memory writes free of bank conflicts).  Every box is its own bulk group, so a slot
// is rewritten once the store issued from it four boxes earlier has read it.
struct BoxRing {
  uint32_t base;  // this warp's 4 KB
  uint32_t slot;
};
__device__ __forceinline__ void store_box16(BoxRing& ring, const CUtensorMap* tm, int lane, const float* v, int x,
                                            int y) {
  const uint32_t box = ring.base + ring.slot * 1024u;
  if (lane == 0) bulk_wait_read<3>();
  __syncwarp();
  const uint32_t row = (uint32_t)lane * 32u, sw = ((uint32_t)lane >> 2) & 1u;
  st_shared_v4(box + row + (sw << 4), pack8(v));
  st_shared_v4(box + row + ((sw ^ 1u) << 4), pack8(v + 8));
  fence_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tm, box, x, y);
    bulk_commit();
  }
  ring.slot = (ring.slot + 1u) & 3u;
}

// Z1 (bf16; not with kFc1NoZ1) and H = bf16(silu(gate) * up) (not with kFc1Z1Only) for 64 of the tile's 128 FFN columns (this warp's
// half), 16 at a time (one activation-quant block); H_hat = AQ(H) for the E2M1 (per 16)
// activation grid, = H without activation quant; the per-row grids (E4M3, INT8) need the
// row amax over all F columns, so H goes to the H buffer and a separate pass quantizes it.
template <int BN, bool F8>
__device__ __forceinline__ void epi_fc1(const Params& p, const CUtensorMap* tm_z1, const CUtensorMap* tm_h,
                                        const Tile& ti, uint32_t tbase, int q, int lane, int half, BoxRing& ring) {
  const int row_in_tile = q * 32 + lane;
  const int64_t row = ti.row_base + row_in_tile;
  const int y = (int)ti.row_base + 32 * q;
  __nv_bfloat16* hrow = p.out3 + row * p.ld_out2;
  const bool row_aq = act_needs_row(p.aq);
  // tm_h is the H_hat map, or the H map for the per-row activation grids (whose H_hat is
  // made by a separate pass); with QAD_FLAG_STASH_H and a per-block grid H is also kept.
  const bool extra_h = (p.flags & QAD_FLAG_STASH_H) && !row_aq;
  const int c0 = 64 * half;  // first of this warp's 64 columns within the tile's 128
  float rs = 1.0f;
  if constexpr (F8) {
    const int32_t tok = p.row_tok ? __ldg(p.row_tok + row) : (int32_t)row;
    rs = tok >= 0 ? __ldg(p.row_scale + tok) : 0.0f;
  }
  // 16-column steps of this warp that lie inside F (all 4 unless F % 128 != 0 in the last tile);
  // the same for the whole warp, so the warp-wide TMEM loads stay uniform
  int nsteps = (p.F - (ti.nb * 128 + c0)) / 16;
  nsteps = nsteps < 0 ? 0 : (nsteps > 4 ? 4 : nsteps);
  if (nsteps == 0) return;
  uint32_t g[16], u[16], gn[16], un[16];
  tmem_ld16_issue(tbase + c0, g);
  tmem_ld16_issue(tbase + 128 + c0, u);
  tmem_wait16x2(g, u);
#pragma unroll 1
  for (int j = 0; j < nsteps; ++j) {
    const int cc = c0 + 16 * j;
    if (j + 1 < nsteps) {
      tmem_ld16_issue(tbase + cc + 16, gn);
      tmem_ld16_issue(tbase + 128 + cc + 16, un);
    }
    const int f0 = ti.nb * 128 + cc;
    float gv[16], uv[16], h[16];
    if constexpr (F8) {
      const float4* cg = reinterpret_cast<const float4*>(p.col_scale + (int64_t)ti.e * p.b_rows + f0);
      const float4* cu = reinterpret_cast<const float4*>(p.col_scale + (int64_t)ti.e * p.b_rows + p.F + f0);
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        const float4 a = __ldg(cg + i4), b = __ldg(cu + i4);
        const float sa[4] = {a.x, a.y, a.z, a.w}, sb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          gv[4 * i4 + i] = round_bf16(__fmul_rn(__uint_as_float(g[4 * i4 + i]), __fmul_rn(rs, sa[i])));
          uv[4 * i4 + i] = round_bf16(__fmul_rn(__uint_as_float(u[4 * i4 + i]), __fmul_rn(rs, sb[i])));
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        gv[i] = round_bf16(__uint_as_float(g[i]));
        uv[i] = round_bf16(__uint_as_float(u[i]));
      }
    }
    if (p.fc1_mode != kFc1NoZ1) {
      store_box16(ring, tm_z1, lane, gv, f0, y);
      store_box16(ring, tm_z1, lane, uv, p.F + f0, y);
    }
    if (p.fc1_mode != kFc1Z1Only) {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {  // H = silu(g) u, two lanes at a time
      const uint64_t g2 = f2pack(gv[i], gv[i + 1]);
      const float2 hv = f2unpack(f2mul(f2mul(g2, sigmoid2(g2)), f2pack(uv[i], uv[i + 1])));
      h[i] = round_bf16(hv.x);
      h[i + 1] = round_bf16(hv.y);
    }
    if (extra_h) {
      uint4* hs = reinterpret_cast<uint4*>(hrow + f0);
      hs[0] = pack8(h);
      hs[1] = pack8(h + 8);
    }
    if (p.aq == kQE2M1) {
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(h[i]));
      fakequant_act_inplace<kQE2M1, 16>(h, __fdiv_rn(amax, 6.0f));
    }
    store_box16(ring, tm_h, lane, h, f0, y);
    }
    if (j + 1 < nsteps) {
      tmem_wait16x2(gn, un);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        g[i] = gn[i];
        u[i] = un[i];
      }
    }
  }
}

// bf16 store of this warp's 32 rows x BN/2 columns: its TMEM loads are issued in batches of
// BATCH 32-column chunks (all at once unless the register budget is tight), one wait per batch;
// each 32-column chunk is written into one of the warp's two staging boxes
// (thread = row, 16-byte chunk c of the 64-byte row at position c ^ ((row >> 1) & 3), the
// 64-byte swizzle, which also keeps the shared-memory writes free of bank conflicts) and
// one lane stores the box with TMA.  A box is rewritten only after the TMA store issued
// from it two chunks earlier has read it.
template <int BN, bool F8, int BATCH>
__device__ __forceinline__ void epi_store_batch(const Params& p, const CUtensorMap* tmC, const Tile& ti,
                                                uint32_t tbase, int q, int lane, int c0, int y,
                                                uint32_t stage_base, uint32_t& buf) {
  constexpr int NH = BATCH;
  uint32_t r[NH][32];
#pragma unroll
  for (int c = 0; c < NH; ++c) tmem_ld32_issue(tbase + 32 * (c0 + c), r[c]);
#pragma unroll
  for (int c = 0; c < NH; ++c) tmem_wait32(r[c]);
  const uint32_t row_addr = (uint32_t)lane * 64u;
  const uint32_t sw = ((uint32_t)lane >> 1) & 3u;
  float rs = 1.0f;
  if constexpr (F8) {
    const int64_t row = ti.row_base + 32 * q + lane;
    const int32_t tok = p.row_tok ? __ldg(p.row_tok + row) : (int32_t)row;
    rs = tok >= 0 ? __ldg(p.row_scale + tok) : 0.0f;
  }
#pragma unroll
  for (int c = 0; c < NH; ++c) {
    // a 32-column box that starts past N is not stored (one that straddles it is cut by the
    // tensor map's extent)
    if (ti.nb * BN + 32 * (c0 + c) >= p.n_total) continue;
    if constexpr (F8) {
      const float4* cs =
          reinterpret_cast<const float4*>(p.col_scale + (int64_t)ti.e * p.b_rows + ti.nb * BN + 32 * (c0 + c));
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4) {
        const float4 a = __ldg(cs + i4);
        const float sc[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          r[c][4 * i4 + i] = __float_as_uint(__fmul_rn(__uint_as_float(r[c][4 * i4 + i]), __fmul_rn(rs, sc[i])));
      }
    }
    const uint32_t box = stage_base + buf * kStageBox;
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[c][8 * ch + i]);
      st_shared_v4(box + row_addr + ((((uint32_t)ch) ^ sw) << 4), pack8(v));
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmC, box, ti.nb * BN + 32 * (c0 + c), y);
      bulk_commit();
    }
    buf ^= 1u;
  }
}

template <int BN, bool F8, int BATCH = BN / 64>
__device__ __forceinline__ void epi_store(const Params& p, const CUtensorMap* tmC, const Tile& ti, uint32_t tbase,
                                          int q, int lane, int half, uint32_t stage_base, uint32_t& buf) {
  constexpr int NH = BN / 64;  // 32-column chunks per half: 4 or 2
  static_assert(NH % BATCH == 0, "batches of whole chunks");
  const int c0 = half * NH;
  const int y = (int)ti.row_base + 32 * q;
#pragma unroll
  for (int b0 = 0; b0 < NH; b0 += BATCH)
    epi_store_batch<BN, F8, BATCH>(p, tmC, ti, tbase, q, lane, c0 + b0, y, stage_base, buf);
}


// This thread's Z1 row and first column in a tile of the SwiGLU-backward epilogue.
struct Z1Cursor {
  const __nv_bfloat16* row;
  int f_first;
};
template <int BN>
__device__ __forceinline__ Z1Cursor z1_cursor(const Params& p, const Tile& ti, int q, int lane, int half) {
  const int64_t row = ti.row_base + q * 32 + lane;
  return {p.aux + row * p.ld_aux, ti.nb * BN + half * (BN / 2)};
}
// Z1 of 16-column step `step`: the 32-byte gate sector and the 32-byte up sector of this
// thread's row, each with one 256-bit load that allocates no L1 line.  A warp's load touches
// 32 rows, i.e. 32 lines, and L1 shares the SM with the 225 KB of shared memory this kernel
// takes: with 16-byte loads through L1 the line allocations throttled the loads and the
// kernel ran ~11% slower.  Alignment: Z1 rows are 4F bytes apart (F % 128 == 0) from a
// 256-byte aligned region, and the columns start at multiples of 16 elements.
__device__ __forceinline__ void z1_load(const Params& p, const Z1Cursor& c, int step, uint4 (&slot)[4]) {
  ld_nc_256(c.row + c.f_first + 16 * step, slot[0], slot[1]);
  ld_nc_256(c.row + p.F + c.f_first + 16 * step, slot[2], slot[3]);
}

// dZ1 = [dH * up * sig(g) * (1 + g (1 - sig(g))), dH * g * sig(g)] from the stored bf16 Z1,
// 16 columns at a time.  The Z1 loads run three steps ahead in a 4-slot register ring that
// carries over from tile to tile: the last steps of a tile load the first steps of the
// thread's next tile (`next`, when `next_ok`), so a tile only waits for memory at the start
// when nothing was prefetched for it (`prefetched` false: first tile, or after a dead one).
// The TMEM loads run one step ahead.
template <int BN>
__device__ __forceinline__ void epi_swiglu_bwd(const Params& p, const CUtensorMap* tm_dz1, const Tile& ti,
                                               uint32_t tbase, int q, int lane, int half, BoxRing& ring,
                                               uint4 (&z)[4][4], bool prefetched, bool next_ok,
                                               const Z1Cursor& next) {
  const int y = (int)ti.row_base + 32 * q;
  constexpr int STEPS = BN / 32;  // 16-column steps per half
  constexpr int AHEAD = 3;
  static_assert(STEPS % 4 == 0, "the Z1 ring's slots must line up from tile to tile");
  const int col0 = half * (BN / 2);
  const Z1Cursor cur = z1_cursor<BN>(p, ti, q, lane, half);
  const int f_first = cur.f_first;
  uint32_t r[16], rn[16];
  if (!prefetched) {
#pragma unroll
    for (int s = 0; s < AHEAD && s < STEPS; ++s) z1_load(p, cur, s, z[s % 4]);
  }
  tmem_ld16_issue(tbase + col0, r);
  tmem_wait16(r);
#pragma unroll
  for (int j = 0; j < STEPS; ++j) {
    const int f0 = f_first + 16 * j;
    if (j + AHEAD < STEPS) z1_load(p, cur, j + AHEAD, z[(j + AHEAD) % 4]);
    else if (next_ok) z1_load(p, next, j + AHEAD - STEPS, z[(j + AHEAD) % 4]);
    if (j + 1 < STEPS) tmem_ld16_issue(tbase + col0 + 16 * (j + 1), rn);
    float g[16], u[16];
    unpack8(z[j % 4][0], g);
    unpack8(z[j % 4][1], g + 8);
    unpack8(z[j % 4][2], u);
    unpack8(z[j % 4][3], u + 8);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {  // two lanes at a time
      const uint64_t one2 = f2pack(1.0f, 1.0f);
      const uint64_t g2 = f2pack(g[i], g[i + 1]);
      const uint64_t sg2 = sigmoid2(g2);
      const uint64_t t2 = f2mul(f2pack(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), sg2);  // dh sig
      const uint64_t inner2 = f2fma(g2, f2sub(one2, sg2), one2);                                   // 1 + g (1 - sig)
      const float2 dgv = f2unpack(f2mul(f2mul(t2, f2pack(u[i], u[i + 1])), inner2));
      const float2 duv = f2unpack(f2mul(t2, g2));
      g[i] = dgv.x;
      g[i + 1] = dgv.y;
      u[i] = duv.x;
      u[i + 1] = duv.y;
    }
    if (f0 < p.F) {  // steps past F (the last tile when F % BN != 0) read and compute, but store nothing
      store_box16(ring, tm_dz1, lane, g, f0, y);
      store_box16(ring, tm_dz1, lane, u, p.F + f0, y);
    }
    if (j + 1 < STEPS) {
      tmem_wait16(rn);
#pragma unroll
      for (int i = 0; i < 16; ++i) r[i] = rn[i];
    }
  }
}

// ds[e, n, b] (+)= sum_{kappa in b} dW[n, kappa] * phi(W[e, n, kappa], s[e, n, b]), 16
// columns at a time.  The half-row's scales are loaded once up front, W runs two steps
// ahead of the arithmetic, and the TMEM accumulator one step.  nvfp4 blocks (16) are
// written as vectors at the end; INT4 groups (128, when a column half holds a whole
// group) are written directly; otherwise (fp8's whole-row block, INT4 with 128-column
// tiles) each column half writes its partial sum to
// part[ds_index * parts + (tile in block) * 2 + half] and a reduction kernel adds the
// parts in a fixed order.
// 16 weights (one 32-byte sector of a W row): one 256-bit load that allocates no L1 line
// when W is 32-byte aligned (rows are multiples of 32 bytes apart and the columns start at
// multiples of 16), else two 16-byte loads.  A warp's load touches 32 rows of W; the wide
// form made the two scale-gradient GEMMs 2-3% faster.
__device__ __forceinline__ void w_load(const __nv_bfloat16* ptr, bool vec32, uint4 (&v)[2]) {
  if (vec32) {
    ld_nc_256(ptr, v[0], v[1]);
  } else {
    v[0] = __ldg(reinterpret_cast<const uint4*>(ptr));
    v[1] = __ldg(reinterpret_cast<const uint4*>(ptr) + 1);
  }
}

template <int QK>
__device__ __forceinline__ float lsq_block_sum(const uint32_t (&acc)[16], const uint4 (&wraw)[2], float sc) {
  float wv[16], x[16];
  unpack8(wraw[0], wv);
  unpack8(wraw[1], wv + 8);
  float t = 0.0f;
  if (scale_in_fast_range(sc)) {
    quotients_unguarded<16>(wv, sc, x);
    uint64_t t2 = f2pack(0.0f, 0.0f);  // two partial sums, one per lane
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const float2 q = q_pair_raw<QK>(x[i], x[i + 1]);
      float ia, ib;  // x inside the closed clip range, else 0 (q is then the violated bound)
      if constexpr (QK == kQInt4 || QK == kQInt8) {
        ia = (x[i] >= Clip<QK>::lo && x[i] <= Clip<QK>::hi) ? x[i] : 0.0f;
        ib = (x[i + 1] >= Clip<QK>::lo && x[i + 1] <= Clip<QK>::hi) ? x[i + 1] : 0.0f;
      } else {
        ia = fabsf(x[i]) <= Clip<QK>::hi ? x[i] : 0.0f;
        ib = fabsf(x[i + 1]) <= Clip<QK>::hi ? x[i + 1] : 0.0f;
      }
      const uint64_t ph2 = f2sub(f2pack(q.x, q.y), f2pack(ia, ib));
      t2 = f2fma(f2pack(__uint_as_float(acc[i]), __uint_as_float(acc[i + 1])), ph2, t2);
    }
    const float2 tt = f2unpack(t2);
    t = tt.x + tt.y;
  }
  if (!scale_in_fast_range(sc) || !isfinite(t)) {  // rare: extreme scale or an overflowing quotient
    quotients<16>(wv, sc, x);
    t = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const float2 ph = lsq_pair<QK>(x[i], x[i + 1]);
      t = fmaf(__uint_as_float(acc[i]), ph.x, t);
      t = fmaf(__uint_as_float(acc[i + 1]), ph.y, t);
    }
  }
  return t;
}

// A tile that reaches past the weight (rows % 256 or cols % BN != 0, or nvfp4 scale rows that
// are not 16-byte aligned) takes this plain loop instead: every accumulator column is still read
// (the TMEM loads are warp-wide), but W, the scales and ds are touched only inside the weight, one
// 16-column step at a time -- few registers, no software pipelining; only edge tiles run it.
template <int BN, int QK>
__device__ __forceinline__ void epi_scalegrad_edge(const Params& p, const Tile& ti, uint32_t tbase, int row_in_tile,
                                                   int half) {
  constexpr int STEPS = BN / 32;
  const int64_t n = ti.row_base + row_in_tile;
  const int64_t wrow = (int64_t)ti.e * p.w_rows + n;
  const int col0 = half * (BN / 2);
  const int64_t k_first = (int64_t)ti.nb * BN + col0;
  int nvalid = n < p.w_rows ? (int)((p.w_cols - k_first) / 16) : 0;
  nvalid = nvalid < 0 ? 0 : (nvalid > STEPS ? STEPS : nvalid);
  const bool have_acc = ti.nkb > 0;
  const bool vec32 = p.w_vec32 != 0;
  float sum = 0.0f;
#pragma unroll 1
  for (int j = 0; j < STEPS; ++j) {
    uint32_t r[16];
    if (have_acc) {
      tmem_ld16_issue(tbase + col0 + 16 * j, r);
      tmem_wait16(r);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) r[i] = 0u;
    }
    if (j >= nvalid) continue;
    uint4 wq[2];
    w_load(p.w + wrow * p.w_cols + k_first + 16 * j, vec32, wq);
    const int64_t k = k_first + 16 * j;
    float sc;
    if constexpr (QK == kQE2M1) sc = __ldg(p.s + wrow * (p.w_cols / 16) + k / 16);
    else if constexpr (QK == kQInt4) sc = __ldg(p.s + wrow * (p.w_cols / 128) + k / 128);
    else sc = __ldg(p.s + wrow);
    const float t = lsq_block_sum<QK>(r, wq, sc);
    if constexpr (QK == kQE2M1) {
      float* dst = p.ds + wrow * (p.w_cols / 16) + k / 16;
      *dst = p.accumulate ? *dst + t : t;
    } else {
      sum += t;
    }
  }
  if constexpr (QK != kQE2M1) {
    if (n >= p.w_rows) return;
    if constexpr ((QK == kQInt4) && (BN == 256)) {
      if (nvalid == 0) return;  // a half past the weight's last 128-column group
      float* dst = p.ds + wrow * (p.w_cols / 128) + k_first / 128;
      *dst = p.accumulate ? *dst + sum : sum;
    } else {
      // every part of a scale block is written (0 for a half past the weight), so the reduction
      // adds a fixed number of parts in a fixed order
      const int64_t B = (QK == kQInt4) ? 128 : p.w_cols;
      const int tiles_per_block = (int)((B + BN - 1) / BN);
      const int64_t ds_index = wrow * (p.w_cols / B) + ((int64_t)ti.nb * BN) / B;
      p.part[ds_index * (2 * tiles_per_block) + (ti.nb % tiles_per_block) * 2 + half] = sum;
    }
  }
}

template <int BN, int QK>
__device__ __forceinline__ void epi_scalegrad_fmt(const Params& p, const Tile& ti, uint32_t tbase, int row_in_tile,
                                                  int half) {
  constexpr int STEPS = BN / 32;  // 16-column steps per half (= nvfp4 scales per half)
  const int64_t n = ti.row_base + row_in_tile;
  const int64_t wrow = (int64_t)ti.e * p.w_rows + n;
  const int col0 = half * (BN / 2);
  const int64_t k_first = (int64_t)ti.nb * BN + col0;
  const __nv_bfloat16* wr = p.w + wrow * p.w_cols + k_first;
  constexpr bool kDirectGroups = (QK == kQInt4) && (BN == 256);
  const bool have_acc = ti.nkb > 0;

  // scales of this half row
  float sv[STEPS];
  float* ds_row = nullptr;
  if constexpr (QK == kQE2M1) {
    const int64_t sidx = wrow * (p.w_cols / 16) + k_first / 16;  // a multiple of 4
    ds_row = p.ds + sidx;
    const float4* sp = reinterpret_cast<const float4*>(p.s + sidx);
#pragma unroll
    for (int i = 0; i < STEPS / 4; ++i) {
      const float4 v4 = __ldg(sp + i);
      sv[4 * i] = v4.x; sv[4 * i + 1] = v4.y; sv[4 * i + 2] = v4.z; sv[4 * i + 3] = v4.w;
    }
  } else {
    const float sc = (QK == kQInt4) ? __ldg(p.s + wrow * (p.w_cols / 128) + k_first / 128) : __ldg(p.s + wrow);
#pragma unroll
    for (int i = 0; i < STEPS; ++i) sv[i] = sc;
  }

  uint32_t r[16], rn[16];
  uint4 wq[3][2];
  const bool vec32 = p.w_vec32 != 0;
  w_load(wr, vec32, wq[0]);
  if (STEPS > 1) w_load(wr + 16, vec32, wq[1]);
  if (have_acc) {
    tmem_ld16_issue(tbase + col0, r);
    tmem_wait16(r);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = 0u;
  }
  float tsum[STEPS];
#pragma unroll
  for (int j = 0; j < STEPS; ++j) {
    if (j + 2 < STEPS) w_load(wr + 16 * (j + 2), vec32, wq[(j + 2) % 3]);
    if (have_acc && j + 1 < STEPS) tmem_ld16_issue(tbase + col0 + 16 * (j + 1), rn);
    tsum[j] = lsq_block_sum<QK>(r, wq[j % 3], sv[j]);
    if (j + 1 < STEPS && have_acc) {
      tmem_wait16(rn);
#pragma unroll
      for (int i = 0; i < 16; ++i) r[i] = rn[i];
    }
  }

  if constexpr (QK == kQE2M1) {
    float4* dv = reinterpret_cast<float4*>(ds_row);
#pragma unroll
    for (int i = 0; i < STEPS / 4; ++i) {
      float4 o = make_float4(tsum[4 * i], tsum[4 * i + 1], tsum[4 * i + 2], tsum[4 * i + 3]);
      if (p.accumulate) {
        const float4 old = dv[i];
        o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
      }
      dv[i] = o;
    }
  } else {
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < STEPS; ++j) sum += tsum[j];
    if constexpr (kDirectGroups) {
      float* dst = p.ds + wrow * (p.w_cols / 128) + k_first / 128;
      *dst = p.accumulate ? *dst + sum : sum;
    } else {
      // every part of a scale block is written (0 for a half past the weight), so the reduction
      // adds a fixed number of parts in a fixed order
      const int64_t B = (QK == kQInt4) ? 128 : p.w_cols;  // elements per scale
      const int tiles_per_block = (int)((B + BN - 1) / BN);
      const int64_t ds_index = wrow * (p.w_cols / B) + ((int64_t)ti.nb * BN) / B;
      p.part[ds_index * (2 * tiles_per_block) + (ti.nb % tiles_per_block) * 2 + half] = sum;
    }
  }
}

template <int BN, int QK>
__device__ __forceinline__ void scalegrad_tile(const Params& p, const Tile& ti, uint32_t tbase, int row_in_tile,
                                               int half) {
  const bool inside = p.s_vec4 && (int64_t)(ti.mb + 1) * (2 * BM) <= p.w_rows &&
                      (int64_t)(ti.nb + 1) * BN <= p.w_cols;  // the same for every thread of the tile
  if (inside) epi_scalegrad_fmt<BN, QK>(p, ti, tbase, row_in_tile, half);
  else epi_scalegrad_edge<BN, QK>(p, ti, tbase, row_in_tile, half);
}

template <int BN>
__device__ __forceinline__ void run_scalegrad(const Params& p, const Tile& ti, uint32_t tbase, int row_in_tile,
                                             int half) {
  if (p.wq == kQE2M1) scalegrad_tile<BN, kQE2M1>(p, ti, tbase, row_in_tile, half);
  else if (p.wq == kQInt4) scalegrad_tile<BN, kQInt4>(p, ti, tbase, row_in_tile, half);
  else if (p.wq == kQE4M3) scalegrad_tile<BN, kQE4M3>(p, ti, tbase, row_in_tile, half);
  else scalegrad_tile<BN, kQInt8>(p, ti, tbase, row_in_tile, half);
}

// ---------------------------------------------------------------------------------- B-operand dequant

// Elements sharing one weight scale along a weight row: 16 (E2M1), 128 (INT4), the whole row.
__device__ __forceinline__ int64_t dq_block(int wq, int64_t cols) {
  return wq == kQE2M1 ? 16 : wq == kQInt4 ? 128 : cols;
}

// One B stage of this CTA, converted in place by the 128 converter threads.  The stage holds NB
// boxes of R rows x 64 bf16 (128-byte rows, 128-byte swizzle: 16-byte chunk c of row r sits at
// chunk position c ^ (r & 7)).  K-major B (forward GEMMs): box = 128-byte K atom, row = weight
// row b_row0 + r, columns k0 + 64 box + [0, 64).  MN-major B (input-gradient GEMMs): box = 64
// weight columns n0 + 64 box + [0, 64), row = weight row k0 + r.  A unit is 16 elements (chunks
// 2m and 2m + 1 of a row, one E2M1 scale block); consecutive threads take consecutive rows of
// the same m, so every quarter-warp's 16-byte accesses fall in distinct bank groups.  Each unit
// is fake-quantized with the routine of the standalone pass (fakequant16_packed), so the MMA
// reads exactly the values qad_fakequant_fwd writes.
template <int NB, int R, bool B_MN>
struct DqStage {
  static constexpr int UNITS = NB * R * 4;
  static constexpr int PER = UNITS / kConvThreads;
  static constexpr int BATCH = PER < 4 ? PER : 4;  // units whose loads are issued together
  static_assert(PER * kConvThreads == UNITS && PER % BATCH == 0, "units per stage must split evenly");
  struct Unit {
    int box, r, m;
    int64_t wrow, wcol;
  };
  __device__ __forceinline__ static Unit unit(int tid, int i, int64_t b_row0, int64_t k0, int64_t n0) {
    Unit x;
    const int u = tid + i * kConvThreads;
    x.m = u / (NB * R);
    const int rid = u - x.m * (NB * R);
    x.box = rid / R;
    x.r = rid - x.box * R;
    if constexpr (B_MN) {
      x.wrow = k0 + x.r;
      x.wcol = n0 + 64 * x.box + 16 * x.m;
    } else {
      x.wrow = b_row0 + x.r;
      x.wcol = k0 + 64 * x.box + 16 * x.m;
    }
    return x;
  }
  // the scales of this thread's units (issued early: their latency hides behind the previous stage)
  __device__ __forceinline__ static void scales(const Params& p, int tid, int e, int64_t b_row0, int64_t k0,
                                                int64_t n0, float (&sc)[PER]) {
    const int64_t blk = dq_block(p.wq, p.dq_cols);
    const int64_t s_pitch = p.dq_cols / blk;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const Unit x = unit(tid, i, b_row0, k0, n0);
      sc[i] = __ldg(p.dq_s + ((int64_t)e * p.dq_rows + x.wrow) * s_pitch + x.wcol / blk);
    }
  }
  // sb: the stage's B half in shared memory (generic pointer: ordinary accesses, ordered after the
  // barrier wait and before the proxy fence that follows)
  template <int QK, int BOX_BYTES>
  __device__ __forceinline__ static void convert(const Params& p, uint8_t* sb, int tid, int e, int64_t b_row0,
                                                 int64_t k0, int64_t n0, const float (&sc)[PER]) {
#pragma unroll
    for (int i0 = 0; i0 < PER; i0 += BATCH) {
      uint4* c0[BATCH];
      uint4* c1[BATCH];
      uint32_t w[BATCH][8];
#pragma unroll
      for (int j = 0; j < BATCH; ++j) {
        const Unit x = unit(tid, i0 + j, b_row0, k0, n0);
        uint8_t* row = sb + x.box * BOX_BYTES + x.r * 128;
        c0[j] = reinterpret_cast<uint4*>(row + (((2 * x.m) ^ (x.r & 7)) << 4));
        c1[j] = reinterpret_cast<uint4*>(row + (((2 * x.m + 1) ^ (x.r & 7)) << 4));
        const uint4 lo = *c0[j], hi = *c1[j];
        w[j][0] = lo.x; w[j][1] = lo.y; w[j][2] = lo.z; w[j][3] = lo.w;
        w[j][4] = hi.x; w[j][5] = hi.y; w[j][6] = hi.z; w[j][7] = hi.w;
      }
#pragma unroll
      for (int j = 0; j < BATCH; ++j) {
        uint32_t o[8];
        fakequant16_packed<QK>(w[j], sc[i0 + j], o);
        const uint4 lo = make_uint4(o[0], o[1], o[2], o[3]), hi = make_uint4(o[4], o[5], o[6], o[7]);
        *c0[j] = lo;
        *c1[j] = hi;
        if (p.dq_dump) {
          const Unit x = unit(tid, i0 + j, b_row0, k0, n0);
          uint4* d = reinterpret_cast<uint4*>(p.dq_dump + ((int64_t)e * p.dq_rows + x.wrow) * p.dq_cols + x.wcol);
          d[0] = lo;
          d[1] = hi;
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------------- kernel

template <int BN, bool A_MN, bool B_MN, int EPI, bool F8, int ATOMS, bool DQ>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(threads_of(DQ), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                        const Params p) {
  using C = Cfg<BN, ATOMS>;
  constexpr int STAGES = C::STAGES;
  static_assert(!F8 || (!A_MN && !B_MN), "E4M3 operands are K-major (forward GEMMs)");
  static_assert(!DQ || (!F8 && !A_MN), "the dequantized weight is the bf16 B operand of a row-mode GEMM");
  constexpr uint32_t IDESC = instr_desc<BN, A_MN, B_MN, F8>();
  constexpr int BKE = bke_of(F8, ATOMS);  // K elements per stage
  constexpr int AKE = F8 ? 128 : BK;  // K elements per 128-byte atom row
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t a_ring = smem_u32(smem);
  const uint32_t b_ring = a_ring + STAGES * C::A_BYTES;
  const uint32_t stage_out = a_ring + C::RING;  // EPI_STORE: the epilogue warps' staging boxes
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::RING + staging_bytes<EPI>());
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // DQ: this CTA's raw B bytes of a stage have landed (local) / both CTAs' B halves of the stage
  // are converted (the leader's, one arrival per converter warp of either CTA)
  auto bfull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 6 + s); };
  auto bconv_bar = [&](int s) { return bar0 + 8u * (3 * STAGES + 6 + s); };
  int32_t* err = p.hdr + HDR_ERR;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0 = the pair's leader, which issues the MMAs
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * (kEpiThreads / 32));  // one arrival per epilogue warp of either CTA
    }
    mbar_init(drain_bar, 1);
    if constexpr (DQ) {
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(bfull_bar(s), 1);
        mbar_init(bconv_bar(s), 2 * kConvWarps);
      }
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"((uint32_t)C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tile_count(p);
  const int first = (int)cluster_id(), step = (int)cluster_count();

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_parity = 0;  // stages with a load in flight, and its phase parity
    bool ok = true;
    const int half_n = (int)rank * (BN / 2);
    // TMA loads of this CTA's A tile and half of the B tile for k-block kb of tile ti into
    // shared memory, completing on `fb` (DQ: the B half on this CTA's own barrier `bb`)
    auto operand_tiles = [&](const Tile& ti, int kb, uint32_t sa, uint32_t sb, uint32_t fb, uint32_t bb) {
      auto box = [&](uint32_t dst, const CUtensorMap* tm, int x, int y) {
        if (DQ && tm == &tmB) tma_load_2d_local(dst, tm, x, y, bb);
        else tma_load_2d(dst, tm, x, y, fb);
      };
      // K-major operands: one box {64 bf16 | 128 E4M3, rows} per 128-byte K atom; MN-major
      // operands: one box {64, BKE K rows} per 64 columns of M or N
      if (!p.wgrad) {
#pragma unroll
        for (int a = 0; a < ATOMS; ++a) box(sa + a * C::A_ATOM, &tmA, kb * BKE + a * AKE, ti.r0);
        if constexpr (!B_MN) {
#pragma unroll
          for (int a = 0; a < ATOMS; ++a) {
            if constexpr (EPI == EPI_FC1) {
              // leader: the 128 gate rows of the tile, peer: the matching 128 up rows
              box(sb + a * C::B_ATOM, &tmB, kb * BKE + a * AKE, ti.e * p.b_rows + (int)rank * p.F + ti.nb * 128);
            } else {
              box(sb + a * C::B_ATOM, &tmB, kb * BKE + a * AKE, ti.e * p.b_rows + ti.nb * BN + half_n);
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < BN / 128; ++i)
            box(sb + i * BKE * 128, &tmB, ti.nb * BN + half_n + i * 64, ti.e * p.b_rows + kb * BKE);
        }
      } else {
        const int y = ti.r0 + kb * BKE;
#pragma unroll
        for (int i = 0; i < 2; ++i) box(sa + i * BKE * 128, &tmA, ti.mb * 2 * BM + (int)rank * BM + i * 64, y);
#pragma unroll
        for (int i = 0; i < BN / 128; ++i) box(sb + i * BKE * 128, &tmB, ti.nb * BN + half_n + i * 64, y);
      }
    };
    for (int t = first; ok && t < total; t += step) {
      const Tile ti = tile_of(p, t, rank, BKE);
      for (int kb = 0; kb < ti.nkb; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, err)) {
          ok = false;
          break;
        }
        if constexpr (DQ) {
          if (leader) mbar_expect_tx(full_bar(stage), 2 * C::A_BYTES);  // both CTAs' A bytes
          mbar_expect_tx(bfull_bar(stage), C::B_BYTES);                 // this CTA's raw B bytes
        } else {
          if (leader) mbar_expect_tx(full_bar(stage), 2 * C::STAGE);  // both CTAs' bytes
        }
        const uint32_t fb = peer_addr(full_bar(stage), 0);          // the leader's barrier
        operand_tiles(ti, kb, a_ring + stage * C::A_BYTES, b_ring + stage * C::B_BYTES, fb, bfull_bar(stage));
        armed |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (*abort_flag) {
      // let every load of the pair land before the CTA releases its shared memory (the B halves
      // of DQ stages land on each CTA's own barrier)
      int32_t dummy = 0;
      for (int s = 0; s < STAGES; ++s)
        if (armed & (1u << s)) {
          volatile int zero = 0;
          if (leader) mbar_wait(full_bar(s), (armed_parity >> s) & 1u, &zero, &dummy);
          if (DQ) mbar_wait(bfull_bar(s), (armed_parity >> s) & 1u, &zero, &dummy);
        }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------------ MMA issuer (leader)
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    int acc = 0;
    bool ok = true;
    for (int t = first; ok && t < total; t += step) {
      const Tile ti = tile_of(p, t, rank, BKE);
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, err)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < ti.nkb; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag, err)) {
          ok = false;
          break;
        }
        if (DQ && !mbar_wait_cluster(bconv_bar(stage), phase, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = a_ring + stage * C::A_BYTES;
        const uint32_t sb = b_ring + stage * C::B_BYTES;
#pragma unroll
        for (int k = 0; k < ATOMS * 4; ++k) {  // each MMA reads 32 bytes of K per row
          const uint64_t ad = A_MN ? smem_desc(sa + k * 2048, BKE * 128, 1024)
                                   : smem_desc(sa + (k / 4) * C::A_ATOM + (k % 4) * 32, 16, 1024);
          const uint64_t bd = B_MN ? smem_desc(sb + k * 2048, BKE * 128, 1024)
                                   : smem_desc(sb + (k / 4) * C::B_ATOM + (k % 4) * 32, 16, 1024);
          mma_issue<F8>(d_tmem, ad, bd, IDESC, (kb | k) != 0 ? 1u : 0u);
        }
        mma_commit(empty_bar(stage), 3);  // frees the slot in both CTAs
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit(tfull_bar(acc), 3);  // both CTAs' accumulators are ready
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // every MMA issued has finished before tensor memory and shared memory are released
    mma_commit(drain_bar, 1);
    volatile int zero = 0;
    int32_t dummy = 0;
    mbar_wait(drain_bar, 0, &zero, &dummy);
  } else if (DQ && warp >= 2 + kEpiThreads / 32) {
    // ------------------------------------------------------------------ B converters (DQ, both CTAs)
    // Each stage's raw weight half is fake-quantized in place once this CTA's TMA bytes have
    // landed; then every converter warp of both CTAs arrives on the leader's bconv barrier,
    // which the MMA issuer waits on besides the A bytes.  The scales of the next stage are
    // loaded while the current one is converted.
    constexpr int NB = B_MN ? BN / 128 : ATOMS;
    constexpr int R = B_MN ? BKE : BN / 2;
    constexpr int BOX_BYTES = B_MN ? BKE * 128 : C::B_ATOM;
    using S = DqStage<NB, R, B_MN>;
    const int tid = threadIdx.x - kThreads;
    const int half_n = (int)rank * (BN / 2);
    auto b_row0 = [&](const Tile& ti) -> int64_t {
      return EPI == EPI_FC1 ? (int64_t)rank * p.F + (int64_t)ti.nb * 128 : (int64_t)ti.nb * BN + half_n;
    };
    auto n0_of = [&](const Tile& ti) -> int64_t { return (int64_t)ti.nb * BN + half_n; };
    int stage = 0;
    uint32_t phase = 0;
    int t = first;
    if (t < total) {
      Tile ti = tile_of(p, t, rank, BKE);
      int kb = 0;
      float sc[S::PER];
      S::scales(p, tid, ti.e, b_row0(ti), (int64_t)kb * BKE, n0_of(ti), sc);
      while (true) {
        int t2 = t, kb2 = kb + 1;
        Tile ti2 = ti;
        if (kb2 == ti.nkb) {
          t2 = t + step;
          kb2 = 0;
          if (t2 < total) ti2 = tile_of(p, t2, rank, BKE);
        }
        const bool more = t2 < total;
        float sc2[S::PER];
        if (more) S::scales(p, tid, ti2.e, b_row0(ti2), (int64_t)kb2 * BKE, n0_of(ti2), sc2);
        const bool got = mbar_wait(bfull_bar(stage), phase, abort_flag, err);
        if (!__all_sync(0xffffffffu, got)) break;
        uint8_t* sb = smem + (b_ring - a_ring) + stage * C::B_BYTES;
        const int64_t k0 = (int64_t)kb * BKE, br = b_row0(ti), n0 = n0_of(ti);
        if (p.wq == kQE2M1) S::template convert<kQE2M1, BOX_BYTES>(p, sb, tid, ti.e, br, k0, n0, sc);
        else if (p.wq == kQInt4) S::template convert<kQInt4, BOX_BYTES>(p, sb, tid, ti.e, br, k0, n0, sc);
        else if (p.wq == kQE4M3) S::template convert<kQE4M3, BOX_BYTES>(p, sb, tid, ti.e, br, k0, n0, sc);
        else S::template convert<kQInt8, BOX_BYTES>(p, sb, tid, ti.e, br, k0, n0, sc);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor-core reads
        __syncwarp();
        if (lane == 0) mbar_arrive_release_cluster(peer_addr(bconv_bar(stage), 0));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (!more) break;
        t = t2;
        kb = kb2;
        ti = ti2;
#pragma unroll
        for (int i = 0; i < S::PER; ++i) sc[i] = sc2[i];
      }
    }
  } else if (warp >= 2 && warp < 2 + kEpiThreads / 32) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;            // TMEM lane quadrant this warp may read
    const int half = (warp - 2) >> 2;  // which half of the tile's columns it handles
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t buf = 0;
    const uint32_t my_stage = stage_out + (uint32_t)(warp - 2) * (uint32_t)kStageWarp;
    BoxRing ring{my_stage, 0u};
    uint4 zr[4][4];          // SwiGLU backward: Z1 ring carried from tile to tile
    bool prefetched = false;  // the ring holds the first steps of the current tile
    if constexpr (EPI != EPI_SCALEGRAD) tma_prefetch_desc(&tmC);
    if constexpr (EPI == EPI_FC1) tma_prefetch_desc(&tmD);
    for (int t = first; t < total; t += step) {
      const Tile ti = tile_of(p, t, rank, BKE);
      const bool got = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, err);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (ti.live) {
        if constexpr (EPI == EPI_STORE)  // DQ: the converters' warps leave 128 registers: half the chunks at a time
          epi_store<BN, F8, (DQ ? BN / 128 : BN / 64)>(p, &tmC, ti, tbase, q, lane, half, my_stage, buf);
        else if constexpr (EPI == EPI_FC1) epi_fc1<BN, F8>(p, &tmC, &tmD, ti, tbase, q, lane, half, ring);
        else if constexpr (EPI == EPI_SWIGLU_BWD) {
          bool next_ok = false;
          Z1Cursor next{nullptr, 0};
          if (t + step < total) {
            const Tile tn = tile_of(p, t + step, rank, BKE);
            next_ok = tn.live;
            next = z1_cursor<BN>(p, tn, q, lane, half);
          }
          epi_swiglu_bwd<BN>(p, &tmC, ti, tbase, q, lane, half, ring, zr, prefetched, next_ok, next);
          prefetched = next_ok;
        }
        else run_scalegrad<BN>(p, ti, tbase, row_in_tile, half);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(peer_addr(tempty_bar(acc), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if constexpr (EPI != EPI_SCALEGRAD) {
      if (lane == 0) bulk_wait_all();  // the staged tiles are in global memory before the CTA exits
    }
  }

  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal its barriers or read its TMEM
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"((uint32_t)C::TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2D bf16 tensor [outer, inner] (row-major, `ld` elements per row), box {64, box_rows}, 128B swizzle
bool make_tmap(CUtensorMap* tm, const void* base, int64_t inner, int64_t outer, int64_t ld, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1u, 1u};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D byte tensor [outer, inner] (E4M3 codes, `ld` bytes per row), box {128, box_rows}, 128B swizzle
bool make_tmap_u8(CUtensorMap* tm, const void* base, int64_t inner, int64_t outer, int64_t ld, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld};
  cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1u, 1u};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output map of a staged epilogue: [outer, inner] bf16, box {cols, 32} with cols = 32 (64-byte
// swizzle) or 16 (32-byte swizzle)
bool make_store_tmap(CUtensorMap* tm, void* base, int64_t inner, int64_t outer, int64_t ld, int cols = 32) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)cols, 32u};
  cuuint32_t es[2] = {1u, 1u};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool A_MN, bool B_MN, int EPI, int ATOMS, bool F8 = false, bool DQ = false>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& td,
                   const Params& p, int64_t max_tiles, int kid, cudaStream_t st) {
  auto kern = grouped_gemm_kernel<BN, A_MN, B_MN, EPI, F8, ATOMS, DQ>;
  constexpr int kThreadsK = threads_of(DQ);
  constexpr int SMEM = smem_bytes<BN, EPI, ATOMS>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  static int max_pairs[64] = {0};  // per device (one instantiation of this function per kernel)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!max_pairs[dev]) {
    // SM pairs that can hold one CTA each at the same time (persistent grid)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    cfg.blockDim = dim3(kThreadsK, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    max_pairs[dev] = n;
  }
  int64_t pairs = max_tiles < max_pairs[dev] ? max_tiles : max_pairs[dev];
  if (pairs < 1) return cudaSuccess;
  prof_begin(kid, st);
  kern<<<(unsigned)(2 * pairs), kThreadsK, SMEM, st>>>(ta, tb, tc, td, p);
  prof_end(kid, st);
  return cudaGetLastError();
}

// Row-mode pair tiles: expert e with m_e padded 128-row blocks gets ceil(m_e / 2) tiles of two
// consecutive blocks starting at row offs[e] + 256 i.  One block of 1024 threads, one
// expert per thread (E <= 1024), exclusive scan of the tile counts.  Also the order in which
// the wgrad GEMMs visit the experts: by decreasing padded row count (ties by index), so that
// the persistent CTAs, which take tiles round-robin, start with the longest ones (with skewed
// routing the index order left the busiest CTA with ~1.8x the mean work).
__global__ void __launch_bounds__(1024) pair_tiles_kernel(const int32_t* __restrict__ offs, int E,
                                                          int32_t* __restrict__ row0, int32_t* __restrict__ expert,
                                                          int32_t* __restrict__ wg_order, int32_t* hdr) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t rows_of[1024];
  const int e = threadIdx.x, lane = e & 31, w = e >> 5;
  const int32_t start = e < E ? offs[e] : 0;
  const int32_t blocks = e < E ? (offs[e + 1] - start) / BM : 0;
  const int32_t n = (blocks + 1) / 2;
  if (e < E) rows_of[e] = blocks;
  int32_t v = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += x;
  }
  if (lane == 31) warp_tot[w] = v;
  __syncthreads();
  if (w == 0) {
    int32_t t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t x = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += x;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  const int32_t incl = v + (w > 0 ? warp_tot[w - 1] : 0);
  const int32_t excl = incl - n;
  for (int32_t i = 0; i < n; ++i) {
    row0[excl + i] = start + 2 * BM * i;
    expert[excl + i] = e;
  }
  if (e == E - 1) hdr[HDR_NPTILES] = incl;
  __syncthreads();
  if (e < E) {  // rank of expert e in decreasing row count, ties by index
    int32_t rank = 0;
    for (int f = 0; f < E; ++f) {
      const int32_t bf = rows_of[f];
      rank += (bf > blocks || (bf == blocks && f < e)) ? 1 : 0;
    }
    wg_order[rank] = e;
  }
}

template <typename T>
T* at(uint8_t* ws, size_t off) {
  return reinterpret_cast<T*>(ws + off);
}

Params base_params(const GemmCtx& c) {
  const Layout& L = *c.L;
  Params p = {};
  p.hdr = at<int32_t>(c.ws, L.header);
  p.ptile_row0 = at<int32_t>(c.ws, L.ptile_row0);
  p.ptile_expert = at<int32_t>(c.ws, L.ptile_expert);
  p.wg_order = at<int32_t>(c.ws, L.wg_order);
  p.poff = at<int32_t>(c.ws, L.offs);
  p.E = (int)L.E;
  p.F = (int)L.F;
  p.wq = c.wq;
  p.aq = c.aq;
  p.flags = c.flags;
  return p;
}

inline int pick_bn(int64_t n) { return n % 256 == 0 ? 256 : 128; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The weight operand of this GEMM is dequantized in shared memory: raw weight [E, rows, cols]
// with scales s (grid p.wq)
void set_dq(Params& p, const float* s, int64_t rows, int64_t cols, void* dump) {
  p.dq_s = s;
  p.dq_rows = rows;
  p.dq_cols = cols;
  p.dq_dump = static_cast<__nv_bfloat16*>(dump);
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t* err, int64_t budget_cycles, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, (long long)budget_cycles);
  return cudaGetLastError();
}

cudaError_t gemm_prepare(const GemmCtx& c) {
  const Layout& L = *c.L;
  pair_tiles_kernel<<<1, 1024, 0, c.st>>>(at<int32_t>(c.ws, L.offs), (int)L.E, at<int32_t>(c.ws, L.ptile_row0),
                                          at<int32_t>(c.ws, L.ptile_expert), at<int32_t>(c.ws, L.wg_order),
                                          at<int32_t>(c.ws, L.header));
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t gemm_fc1(const GemmCtx& c, int mode) {
  const Layout& L = *c.L;
  Params p = base_params(c);
  p.fc1_mode = mode;
  const bool f8 = L.native_fp8;
  CUtensorMap ta, tb;
  if (f8) {
    if (!make_tmap_u8(&ta, c.ws + L.a1q, L.d, L.Rmax, L.d, 128)) return cudaErrorInvalidValue;
    if (!make_tmap_u8(&tb, c.ws + L.w13q, L.d, L.E * 2 * L.F, L.d, 128)) return cudaErrorInvalidValue;
    p.row_scale = at<float>(c.ws, L.sa_tok);
    p.row_tok = at<int32_t>(c.ws, L.row_token);
    p.col_scale = c.s13;
  } else {
    if (!make_tmap(&ta, c.ws + L.a1, L.d, L.Rmax, L.d, 128)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb, c.w13h, L.d, L.E * 2 * L.F, L.d, 128)) return cudaErrorInvalidValue;
  }
  p.n_ntiles = (int)cdiv(L.F, 128);
  p.num_kb = (int)cdiv(L.d, bke_of(f8, f8 ? 1 : kAtomsFc1));
  p.b_rows = (int)(2 * L.F);
  p.ld_out2 = L.F;
  p.out3 = at<__nv_bfloat16>(c.ws, L.h);
  CUtensorMap tz, th;
  if (!make_store_tmap(&tz, c.ws + L.z1, 2 * L.F, L.Rmax, 2 * L.F, 16)) return cudaErrorInvalidValue;
  if (!make_store_tmap(&th, c.ws + (act_needs_row(c.aq) ? L.h : L.hh), L.F, L.Rmax, L.F, 16)) return cudaErrorInvalidValue;
  const int kid = mode == kFc1Z1Only ? QAD_K_GEMM_FC1_RECOMPUTE : QAD_K_GEMM_FC1;
  const int64_t tiles = (L.Rmax / BM) * (int64_t)p.n_ntiles;
  if (c.dq) {
    set_dq(p, c.s13, 2 * L.F, L.d, c.dump13);
    return launch<256, false, false, EPI_FC1, kAtomsFc1, false, true>(ta, tb, tz, th, p, tiles, kid, c.st);
  }
  return f8 ? launch<256, false, false, EPI_FC1, 1, true>(ta, tb, tz, th, p, tiles, kid, c.st)
            : launch<256, false, false, EPI_FC1, kAtomsFc1>(ta, tb, tz, th, p, tiles, kid, c.st);
}

cudaError_t gemm_fc2(const GemmCtx& c) {
  const Layout& L = *c.L;
  Params p = base_params(c);
  CUtensorMap ta, tb;
  const int bn = pick_bn(L.d);
  const bool f8 = L.native_fp8 && bn == 256;
  if (L.native_fp8 && !f8) return cudaErrorInvalidValue;  // d % 256 == 0 is a layout precondition
  if (f8) {
    if (!make_tmap_u8(&ta, c.ws + L.hq, L.F, L.Rmax, L.F, 128)) return cudaErrorInvalidValue;
    if (!make_tmap_u8(&tb, c.ws + L.w2q, L.F, L.E * L.d, L.F, bn / 2)) return cudaErrorInvalidValue;
    p.row_scale = at<float>(c.ws, L.sh_row);
    p.row_tok = nullptr;
    p.col_scale = c.s2;
  } else {
    if (!make_tmap(&ta, c.ws + L.hh, L.F, L.Rmax, L.F, 128)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb, c.w2h, L.F, L.E * L.d, L.F, bn / 2)) return cudaErrorInvalidValue;
  }
  p.n_ntiles = (int)cdiv(L.d, bn);
  p.num_kb = (int)cdiv(L.F, bke_of(f8, f8 ? 1 : kAtomsFc2));
  p.n_total = (int)L.d;
  p.b_rows = (int)L.d;
  CUtensorMap tc;
  if (!make_store_tmap(&tc, c.ws + L.y, L.d, L.Rmax, L.d)) return cudaErrorInvalidValue;
  const int64_t tiles = (L.Rmax / BM) * (int64_t)p.n_ntiles;
  if (f8) return launch<256, false, false, EPI_STORE, 1, true>(ta, tb, tc, tc, p, tiles, QAD_K_GEMM_FC2, c.st);
  if (c.dq) {
    set_dq(p, c.s2, L.d, L.F, c.dump2);
    return bn == 256
               ? launch<256, false, false, EPI_STORE, kAtomsFc2, false, true>(ta, tb, tc, tc, p, tiles, QAD_K_GEMM_FC2,
                                                                             c.st)
               : launch<128, false, false, EPI_STORE, kAtomsFc2, false, true>(ta, tb, tc, tc, p, tiles, QAD_K_GEMM_FC2,
                                                                             c.st);
  }
  return bn == 256 ? launch<256, false, false, EPI_STORE, kAtomsFc2>(ta, tb, tc, tc, p, tiles, QAD_K_GEMM_FC2, c.st)
                   : launch<128, false, false, EPI_STORE, kAtomsFc2>(ta, tb, tc, tc, p, tiles, QAD_K_GEMM_FC2, c.st);
}

cudaError_t gemm_dgrad_fc2(const GemmCtx& c) {
  const Layout& L = *c.L;
  Params p = base_params(c);
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, c.ws + L.dy, L.d, L.Rmax, L.d, 128)) return cudaErrorInvalidValue;
  // W2_hat viewed as [E * d (GEMM K), F (GEMM N)], N contiguous
  if (!make_tmap(&tb, c.w2h, L.F, L.E * L.d, L.F, bke_of(false, kAtomsDgrad))) return cudaErrorInvalidValue;
  const int bn = pick_bn(L.F);
  p.n_ntiles = (int)cdiv(L.F, bn);
  p.num_kb = (int)cdiv(L.d, bke_of(false, kAtomsDgrad));
  p.n_total = (int)L.F;
  p.b_rows = (int)L.d;
  p.aux = at<__nv_bfloat16>(c.ws, L.z1);
  p.ld_aux = 2 * L.F;
  CUtensorMap tz;
  if (!make_store_tmap(&tz, c.ws + L.dz1, 2 * L.F, L.Rmax, 2 * L.F, 16)) return cudaErrorInvalidValue;
  const int64_t tiles = (L.Rmax / BM) * (int64_t)p.n_ntiles;
  if (c.dq) {
    set_dq(p, c.s2, L.d, L.F, c.dump2);
    return bn == 256 ? launch<256, false, true, EPI_SWIGLU_BWD, kAtomsDgrad, false, true>(ta, tb, tz, tz, p, tiles,
                                                                                         QAD_K_GEMM_DGRAD_FC2, c.st)
                     : launch<128, false, true, EPI_SWIGLU_BWD, kAtomsDgrad, false, true>(ta, tb, tz, tz, p, tiles,
                                                                                         QAD_K_GEMM_DGRAD_FC2, c.st);
  }
  return bn == 256
             ? launch<256, false, true, EPI_SWIGLU_BWD, kAtomsDgrad>(ta, tb, tz, tz, p, tiles, QAD_K_GEMM_DGRAD_FC2, c.st)
             : launch<128, false, true, EPI_SWIGLU_BWD, kAtomsDgrad>(ta, tb, tz, tz, p, tiles, QAD_K_GEMM_DGRAD_FC2, c.st);
}

cudaError_t gemm_dgrad_fc1(const GemmCtx& c) {
  const Layout& L = *c.L;
  Params p = base_params(c);
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, c.ws + L.dz1, 2 * L.F, L.Rmax, 2 * L.F, 128)) return cudaErrorInvalidValue;
  // W13_hat viewed as [E * 2F (GEMM K), d (GEMM N)], N contiguous
  if (!make_tmap(&tb, c.w13h, L.d, L.E * 2 * L.F, L.d, bke_of(false, kAtomsDgrad))) return cudaErrorInvalidValue;
  const int bn = pick_bn(L.d);
  p.n_ntiles = (int)cdiv(L.d, bn);
  p.num_kb = (int)cdiv(2 * L.F, bke_of(false, kAtomsDgrad));
  p.n_total = (int)L.d;
  p.b_rows = (int)(2 * L.F);
  CUtensorMap tc;
  if (!make_store_tmap(&tc, c.ws + L.da1, L.d, L.Rmax, L.d)) return cudaErrorInvalidValue;
  const int64_t tiles = (L.Rmax / BM) * (int64_t)p.n_ntiles;
  if (c.dq) {
    set_dq(p, c.s13, 2 * L.F, L.d, c.dump13);
    return bn == 256 ? launch<256, false, true, EPI_STORE, kAtomsDgrad, false, true>(ta, tb, tc, tc, p, tiles,
                                                                                    QAD_K_GEMM_DGRAD_FC1, c.st)
                     : launch<128, false, true, EPI_STORE, kAtomsDgrad, false, true>(ta, tb, tc, tc, p, tiles,
                                                                                    QAD_K_GEMM_DGRAD_FC1, c.st);
  }
  return bn == 256
             ? launch<256, false, true, EPI_STORE, kAtomsDgrad>(ta, tb, tc, tc, p, tiles, QAD_K_GEMM_DGRAD_FC1, c.st)
             : launch<128, false, true, EPI_STORE, kAtomsDgrad>(ta, tb, tc, tc, p, tiles, QAD_K_GEMM_DGRAD_FC1, c.st);
}

namespace {
cudaError_t wgrad(const GemmCtx& c, size_t a_off, int64_t m_w, size_t b_off, int64_t k_w, const void* w,
                  const float* s, float* ds, size_t part_off, int accumulate, int kid) {
  const Layout& L = *c.L;
  Params p = base_params(c);
  CUtensorMap ta, tb;
  // A = dZ [Rmax, Mw] (M contiguous), B = A_hat [Rmax, Kw] (N contiguous)
  if (!make_tmap(&ta, c.ws + a_off, m_w, L.Rmax, m_w, bke_of(false, kAtomsWgrad))) return cudaErrorInvalidValue;
  if (!make_tmap(&tb, c.ws + b_off, k_w, L.Rmax, k_w, bke_of(false, kAtomsWgrad))) return cudaErrorInvalidValue;
  const int bn = pick_bn(k_w);
  p.wgrad = 1;
  p.n_mtiles_w = (int)cdiv(m_w, 2 * BM);
  p.n_ntiles = (int)cdiv(k_w, bn);
  p.s_vec4 = (k_w % 64) == 0;
  p.w = static_cast<const __nv_bfloat16*>(w);
  p.w_vec32 = (reinterpret_cast<uintptr_t>(w) & 31u) == 0;
  p.s = s;
  p.w_rows = m_w;
  p.w_cols = k_w;
  p.ds = ds;
  p.part = at<float>(c.ws, part_off);
  p.accumulate = accumulate;
  const int64_t tiles = L.E * p.n_mtiles_w * p.n_ntiles;
  cudaError_t e = bn == 256 ? launch<256, true, true, EPI_SCALEGRAD, kAtomsWgrad>(ta, tb, ta, ta, p, tiles, kid, c.st)
                            : launch<128, true, true, EPI_SCALEGRAD, kAtomsWgrad>(ta, tb, ta, ta, p, tiles, kid, c.st);
  if (e != cudaSuccess) return e;
  if (row_scaled(c.wq) || (c.wq == kQInt4 && bn == 128)) {
    const int64_t B = c.wq == kQInt4 ? 128 : k_w;  // elements per scale
    return launch_scale_reduce(p.part, ds, L.E * m_w * (k_w / B), (int)(2 * cdiv(B, bn)), accumulate, c.st);
  }
  return cudaSuccess;
}
}  // namespace

cudaError_t gemm_wgrad_fc2(const GemmCtx& c, const void* w2, const float* s2, float* ds2, int accumulate) {
  const Layout& L = *c.L;
  return wgrad(c, L.dy, L.d, L.hh, L.F, w2, s2, ds2, L.part2, accumulate, QAD_K_GEMM_WGRAD_FC2);
}

cudaError_t gemm_wgrad_fc1(const GemmCtx& c, const void* w13, const float* s13, float* ds13, int accumulate) {
  const Layout& L = *c.L;
  return wgrad(c, L.dz1, 2 * L.F, L.a1, L.d, w13, s13, ds13, L.part13, accumulate, QAD_K_GEMM_WGRAD_FC1);
}

}  // namespace qad
