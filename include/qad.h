/*
 * qad.h -- C ABI of the scale-only QAD MoE-layer library for one GB300 (sm_103a).
 *
 * What the library computes.  Scale-only quantization-aware training/distillation
 * keeps the BF16 weights frozen, fake-quantizes them (quantize then dequantize) and
 * optimises only the quantizer scales ("MCoreQAD Backend", mcore_qad.md, opening
 * section).  The weight a matmul sees is quantize->dequantize(W; s) with gradients
 * reaching s, and each quantized matmul's input is fake-quantized first (AngelSlim
 * mcore_qad walkthrough, nxmr.cn/news/131691, section 二.3).  The routed experts of a
 * MoE layer are 3D-stacked, fake-quantized in one pass and run as one grouped GEMM
 * (same article, section 二.4).  Formats: nvfp4 (W4A4), w4a16 (INT4) and fp8 (W8A8)
 * ("MCoreQAD Backend", Support Matrix; article section 三).
 *
 * Layer (per token t, routed to k distinct experts j with weights p[t, j]):
 *   A1  = AQ(x[t])                                  activation fake-quant
 *   Z1  = A1 . W13_hat[e]^T          [2F]           rows [0, F) gate, [F, 2F) up
 *   H   = silu(gate) * up;  H_hat = AQ(H)           [F]
 *   Y   = H_hat . W2_hat[e]^T        [d]
 *   out = sum_j p[t, j] * Y_j                       [d]
 * W_hat = bf16(fp32(q(fp32(W / s)) * s)) element by element, s broadcast over its block.
 * Backward: straight-through estimator for both quantizers; the weights get no
 * gradient; the scale gradient is
 *   ds[e, n, b] = sum_{kappa in block b} dW_hat[e, n, kappa] * phi(W[e, n, kappa], s[e, n, b])
 * with the LSQ factor phi = q(x) - x inside the closed clip range, the clip bound
 * outside it (x = fp32(W / s)).
 *
 * Conventions for every call:
 *   - pointers are DEVICE pointers unless stated; bf16 tensors are passed as void*;
 *     every pointer must be 16-byte aligned;
 *   - every call is asynchronous on `stream` and allocates nothing; the caller owns
 *     all memory, including the workspace;
 *   - a call returns QAD_OK, or a negative qad_status BEFORE launching anything when
 *     an argument is invalid; CUDA launch failures return QAD_ERR_CUDA;
 *   - problems found on the device (a routing index out of range or repeated within a
 *     token, a pipeline wait that timed out) set bits in the workspace's device error
 *     word, which qad_check_device_error() reads; no kernel traps or aborts.
 */
#ifndef QAD_H_
#define QAD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* qad_stream_t; /* the same type as cudaStream_t; NULL = legacy stream */

typedef enum {
  QAD_OK = 0,
  QAD_ERR_INVALID_ARG = -1, /* null/misaligned pointer, bad size, bad flag */
  QAD_ERR_UNSUPPORTED = -2, /* shape outside the supported set (divisibility, limits) */
  QAD_ERR_WORKSPACE = -3,   /* workspace smaller than qad_moe_workspace_bytes() */
  QAD_ERR_CUDA = -4,        /* a CUDA runtime call or kernel launch failed */
  QAD_ERR_DEVICE = -5,      /* the device error word is non-zero (see QAD_DEV_*) */
  QAD_ERR_SCRATCH_LIMIT = -6 /* larger than the fixed scratch of qad_route_permute_noalloc */
} qad_status;

/* Formats: the pages' names ("MCoreQAD Backend", Support Matrix: nvfp4, nvfp4a16, w4a16,
 * w8a8, fp8, w4afp8).  The element grids, scale granularity and activation scales are
 * readings of those names (the pages give no formula). */
typedef enum {
  QAD_FMT_NVFP4 = 0,     /* nvfp4 W4A4: E2M1 weights, one fp32 scale per 16 along K;
                            activations E2M1 with dynamic per-16 scale amax/6 */
  QAD_FMT_INT4_G128 = 1, /* w4a16: INT4 {-8..7} weights, one fp32 scale per 128 along K;
                            activations stay bf16 */
  QAD_FMT_FP8_ROW = 2,   /* fp8 W8A8: E4M3 weights, one fp32 scale per output row;
                            activations E4M3 with dynamic per-row scale amax/448 */
  QAD_FMT_NVFP4A16 = 3,  /* nvfp4a16: E2M1 weights as nvfp4; activations stay bf16 */
  QAD_FMT_W8A8 = 4,      /* w8a8: INT8 {-128..127} weights, one fp32 scale per output row;
                            activations INT8 with dynamic per-row scale amax/127 */
  QAD_FMT_W4AFP8 = 5,    /* w4afp8: INT4 weights as w4a16; activations E4M3 per row, amax/448 */
  QAD_FMT_NVFP4_E4M3 = 6 /* nvfp4 with deployed block scales: as nvfp4, but every block scale is
                            used as the compressed-tensors NVFP4 layout stores it (AngelSlim
                            mcore_qad walkthrough, section 三: the format names map to the
                            deployment side's layout), an E4M3 number times one fp32 scale g of
                            the tensor: s_q = fp32(e4m3(fp32(s / g)) * g) (round to nearest even,
                            saturating).  Weights: g = fp32(max |s| / 448) over each expert's w13
                            (gate and up share it) and each expert's w2, see
                            qad_nvfp4_deploy_scales; the scale gradient reaches s straight through
                            the rounding.  Activations: the dynamic per-16 scale fp32(amax / 6) is
                            rounded the same way with g = fp32(max over the row's blocks / 448)
                            per row.  A block whose s_q is 0 comes out as signed zeros. */
} qad_fmt;

/* Bits of the device error word */
enum {
  QAD_DEV_BAD_INDEX = 1, /* a topk index outside [0, E): that (token, slot) pair is dropped */
  QAD_DEV_DUP_INDEX = 2, /* a token names the same expert twice: the later slot is dropped */
  QAD_DEV_TIMEOUT = 4    /* a bounded pipeline wait expired; outputs of that call are invalid */
};

/* qad_moe_shape.flags */
enum {
  QAD_FLAG_STASH_H = 1,  /* also store the un-quantized SwiGLU output H in the workspace */
  QAD_FLAG_NO_QUANT = 2, /* quantizers off: the self-distillation teacher pass ("MCoreQAD
                            Backend", opening section: the same frozen model with quantization
                            disabled supplies the teacher logits).  qad_moe_fwd and
                            qad_moe_bwd_dgrad then use the raw bf16 weights and bf16
                            activations; the scales are not read (pass any valid pointer)
                            and qad_moe_bwd_scalegrad returns QAD_ERR_INVALID_ARG. */
  QAD_FLAG_RECOMPUTE = 4, /* recompute instead of stash ("MCoreQAD Backend", performance notes:
                            full activation recomputation for large models): qad_moe_fwd does
                            not keep the fc1 output Z1, and qad_moe_bwd_dgrad recomputes it
                            (one more fc1 GEMM, identical values) before its SwiGLU backward.
                            When d >= 2F, Z1 then shares the workspace region of Y (Y is no
                            longer needed once the dgrad call has used it for dprobs), so
                            qad_moe_workspace_bytes is smaller by about 4·Rmax·F bytes.  The
                            fwd, dgrad and scalegrad calls of one step must use the same flags. */
  QAD_FLAG_NATIVE_FP8 = 8, /* fp8 format (QAD_FMT_FP8_ROW) only: the forward GEMMs contract the
                            E4M3 codes on the fp8 tensor path (tcgen05 kind::f8f6f4) and apply
                            the per-row weight and activation scales to the fp32 sums -- the
                            scales leave the contraction exactly ("MCoreQAD Backend", Support
                            Matrix: fp8 W8A8 per-channel/per-token), so q*s is not rounded to
                            bf16 before the products.  Also writes the codes and row scales to
                            the workspace; the backward is unchanged (bf16 fake-quant copies).
                            Any other format, or QAD_FLAG_NO_QUANT, gives QAD_ERR_INVALID_ARG. */
  QAD_FLAG_SMEM_DEQUANT = 16, /* the fake-quantized weights are never materialised (AngelSlim
                            mcore_qad walkthrough, section 二.4: the stacked experts are
                            fake-quantized and consumed by one grouped GEMM): instead of one
                            fake-quant pass writing W13_hat and W2_hat to the workspace, the four
                            GEMMs that read them (fc1, fc2 and the two input-gradient GEMMs) load
                            tiles of the raw bf16 weights and fake-quantize each tile in shared
                            memory before the tensor cores read it, with the same arithmetic and
                            hence the same bits.  The workspace loses the two weight copies
                            (E * 3 * F * d * 2 bytes).  Not with QAD_FLAG_NO_QUANT or
                            QAD_FLAG_NATIVE_FP8 (QAD_ERR_INVALID_ARG).  All three calls of a step
                            must pass it. */
  QAD_FLAG_DEQUANT_DUMP = 32 /* testing aid for QAD_FLAG_SMEM_DEQUANT (required with it): the
                            workspace keeps the W13_hat / W2_hat regions and every GEMM that
                            dequantizes a weight tile in shared memory also writes the values it
                            converted there, so they can be compared with qad_fakequant_fwd. */
};

/* Shape of one MoE layer. T tokens, hidden d, expert FFN width F, E experts, top-k. */
typedef struct {
  int64_t T, d, F, E;
  int32_t topk;
  int32_t fmt;   /* qad_fmt */
  int32_t flags; /* QAD_FLAG_* */
  int32_t reserved; /* must be 0 */
} qad_moe_shape;

/*
 * Weight fake-quant of a stack of E matrices [N, K] (article section 二.3/二.4: the whole
 * expert stack in one vectorised pass).
 *   w      bf16 [E, N, K] row-major (read only)
 *   scale  fp32 [E, N, K / B] with B = 16 (E2M1 formats), 128 (INT4 formats), K (fp8, w8a8)
 *   w_hat  bf16 [E, N, K] (written; may not overlap w)
 * Requires K % 16 == 0 (K % 128 == 0 for the INT4 formats), scales >= 0 and finite.
 * Output is bit-exact: w_hat = bf16(fp32(q(fp32(w / s)) * s)).
 * QAD_FMT_NVFP4_E4M3 returns QAD_ERR_UNSUPPORTED: round the scales with
 * qad_nvfp4_deploy_scales and call this with QAD_FMT_NVFP4 and the rounded scales (the same
 * arithmetic, which is what the layer calls do).
 */
int qad_fakequant_fwd(int fmt, const void* w, const float* scale, void* w_hat,
                      int64_t E, int64_t N, int64_t K, qad_stream_t stream);

/*
 * The block scales of QAD_FMT_NVFP4_E4M3 weights as deployed NVFP4 stores them (AngelSlim
 * mcore_qad walkthrough, section 三): for each of the n_mat matrices of per_mat consecutive
 * scales, g = fp32(max |s| / 448) and s_q[i] = fp32(e4m3(fp32(s[i] / g)) * g) (E4M3 "fn":
 * round to nearest even, saturating at 448); g = 0 (an all-zero matrix) gives s_q = 0.
 *   s    fp32 [n_mat, per_mat] (read)          s_q fp32 [n_mat, per_mat] (written; may be s)
 * Requires per_mat % 4 == 0 and 16-byte aligned pointers; n_mat == 0 does nothing.
 */
int qad_nvfp4_deploy_scales(const float* s, float* s_q, int64_t n_mat, int64_t per_mat, qad_stream_t stream);

/* Bytes of workspace the three layer calls need for this shape; 0 if the shape is
 * not supported.  Host-only, no CUDA call. */
size_t qad_moe_workspace_bytes(const qad_moe_shape* s);

/*
 * Forward of one MoE layer.
 *   x        bf16 [T, d]        topk_idx int32 [T, topk]     topk_w fp32 [T, topk]
 *   w13      bf16 [E, 2F, d]    s13 fp32 [E, 2F, d / B]      (rows [0,F) gate, [F,2F) up)
 *   w2       bf16 [E, d, F]     s2  fp32 [E, d, F / B]
 *   out      bf16 [T, d] (written)
 *   ws       workspace (256-byte aligned) of ws_bytes >= qad_moe_workspace_bytes(s); it keeps what the
 *            backward calls need (routing maps, fake-quantized weights, activations, and for
 *            QAD_FMT_NVFP4_E4M3 the deployed weight scales, which the backward calls use in place
 *            of s13 / s2 -- they must still be passed).
 * Supported: d and F multiples of 16 (multiples of 128 for the INT4 formats, whose group-128
 * scales run along both; d % 256 == 0 and F % 128 == 0 with QAD_FLAG_NATIVE_FP8 or
 * QAD_FLAG_SMEM_DEQUANT), 1 <= topk <= min(E, 32), 1 <= E <= 1024, T * topk < 2^31; other shapes
 * return QAD_ERR_UNSUPPORTED before any launch.  The error word is cleared at the start of this
 * call.
 */
int qad_moe_fwd(const qad_moe_shape* s, const void* x, const int32_t* topk_idx, const float* topk_w,
                const void* w13, const float* s13, const void* w2, const float* s2,
                void* out, void* ws, size_t ws_bytes, qad_stream_t stream);

/*
 * Input gradient of the layer (straight-through both quantizers).
 *   dout   bf16 [T, d]; topk_w as in the forward; w13/s13/w2/s2 as in the forward
 *   dx     bf16 [T, d] (written)
 *   dprobs fp32 [T, topk] (written, may be NULL): dL/dtopk_w[t, j] = <dout[t], Y_j>
 * Must follow qad_moe_fwd on the same workspace, inputs and stream.
 */
int qad_moe_bwd_dgrad(const qad_moe_shape* s, const void* dout, const float* topk_w,
                      const void* w13, const float* s13, const void* w2, const float* s2,
                      void* dx, float* dprobs, void* ws, size_t ws_bytes, qad_stream_t stream);

/*
 * Scale gradients (the only trainable parameters).
 *   ds13 fp32 [E, 2F, d / B], ds2 fp32 [E, d, F / B]: overwritten, or added to when
 *   accumulate != 0.
 * The weight gradient is reduced into the scale gradient inside the GEMM epilogue and
 * never stored.  Must follow qad_moe_bwd_dgrad on the same workspace and stream.
 * The epilogue reads w13 / w2 row by row: with 32-byte aligned weights (as PyTorch's
 * allocations are) one 256-bit load per 16 weights, with 16-byte aligned ones two 16-byte
 * loads; the results are the same bits.
 */
int qad_moe_bwd_scalegrad(const qad_moe_shape* s, const void* w13, const float* s13,
                          const void* w2, const float* s2, float* ds13, float* ds2,
                          int accumulate, void* ws, size_t ws_bytes, qad_stream_t stream);

/*
 * The layer's combine step on rows the caller holds: out[t] = bf16(sum_{j = 0..topk-1} p[t, j] *
 * rows[row_of[t, j]]), fp32 sums in slot order; p NULL means weight 1; a pair with row_of < 0 is
 * skipped.  It serves an expert-parallel split (AngelSlim mcore_qad walkthrough, section 二.4:
 * experts are split across ranks only by expert parallelism, ETP = 1): a rank sends each routed
 * (token, slot) pair to the rank that owns its expert, that rank runs the layer on the received
 * rows with top-1 routing (weight 1 in the forward, the pair's weight in the input-gradient call),
 * so its output rows are the expert outputs Y and its input-gradient rows are dA1; the rows come
 * back in pair order and this call forms out (with p) and dx (weight 1) exactly as qad_moe_fwd /
 * qad_moe_bwd_dgrad would on one GPU.
 *   rows bf16 [n_rows, d]; row_of int32 [T, topk]; p fp32 [T, topk] or NULL; out bf16 [T, d]
 * Requires d % 16 == 0, 1 <= topk <= 32, 16-byte aligned pointers, and every row_of entry -1 or
 * in [0, n_rows) (the caller builds row_of; it is not checked on the device).
 */
int qad_moe_combine(const void* rows, const int32_t* row_of, const float* p, void* out, int64_t T, int32_t topk,
                    int64_t d, qad_stream_t stream);

/* Synchronises `stream`, copies the device error word of `ws` into *code (host
 * pointer, may be NULL) and returns QAD_OK if it is zero, QAD_ERR_DEVICE otherwise. */
int qad_check_device_error(void* ws, qad_stream_t stream, int32_t* code);

/* Static English text for a qad_status value. */
const char* qad_status_string(int status);

/* Views into the workspace for stage-by-stage testing.  Writes the byte offset of
 * region `which` from the workspace base and its element count.  Host-only. */
enum {
  QAD_VIEW_HEADER = 0,     /* int32[64]: [0] error word, [1] routed-row tiles, [2] padded rows */
  QAD_VIEW_OFFSETS = 1,    /* int32 [E + 1]: first padded row of each expert (multiples of 128) */
  QAD_VIEW_COUNTS = 2,     /* int32 [E]: routed rows per expert */
  QAD_VIEW_ROW_TOKEN = 3,  /* int32 [Rmax]: token of each padded row, -1 for padding */
  QAD_VIEW_ROW_SLOT = 4,   /* int32 [Rmax]: top-k slot of each padded row, -1 for padding */
  QAD_VIEW_ROW_OF = 5,     /* int32 [T * topk]: padded row of each pair, -1 if dropped */
  QAD_VIEW_W13_HAT = 6,    /* bf16 [E, 2F, d] */
  QAD_VIEW_W2_HAT = 7,     /* bf16 [E, d, F] */
  QAD_VIEW_A1 = 8,         /* bf16 [Rmax, d] */
  QAD_VIEW_Z1 = 9,         /* bf16 [Rmax, 2F] */
  QAD_VIEW_H = 10,         /* bf16 [Rmax, F] (QAD_FLAG_STASH_H, or per-row activation grids) */
  QAD_VIEW_H_HAT = 11,     /* bf16 [Rmax, F] */
  QAD_VIEW_Y = 12,         /* bf16 [Rmax, d] */
  QAD_VIEW_DY = 13,        /* bf16 [Rmax, d] */
  QAD_VIEW_DZ1 = 14,       /* bf16 [Rmax, 2F] */
  QAD_VIEW_DA1 = 15,       /* bf16 [Rmax, d] */
  QAD_VIEW_XQ = 16,        /* bf16 [T, d]: AQ(x) per token */
  /* QAD_FLAG_NATIVE_FP8 only (count 0 otherwise): */
  QAD_VIEW_W13_CODES = 17, /* uint8 [E, 2F, d]: E4M3 codes of W13 */
  QAD_VIEW_W2_CODES = 18,  /* uint8 [E, d, F] */
  QAD_VIEW_A1_CODES = 19,  /* uint8 [Rmax, d]: E4M3 codes of the routed activation rows */
  QAD_VIEW_H_CODES = 20,   /* uint8 [Rmax, F] */
  QAD_VIEW_A_SCALE = 21,   /* fp32 [T]: activation scale fp32(row amax / 448) of each token */
  QAD_VIEW_H_SCALE = 22,   /* fp32 [Rmax]: the same for each row of H */
  /* QAD_FMT_NVFP4_E4M3 only (count 0 otherwise): the deployed weight scales the forward made */
  QAD_VIEW_S13_DEPLOYED = 23, /* fp32 [E, 2F, d / 16] */
  QAD_VIEW_S2_DEPLOYED = 24,  /* fp32 [E, d, F / 16] */
  QAD_VIEW_COUNT = 25
};
int qad_moe_debug_view(const qad_moe_shape* s, int which, size_t* byte_offset, int64_t* numel);

/*
 * Kernel timing.  While enabled, every kernel launch of the library is bracketed by
 * CUDA events on its stream.  qad_profile_read() synchronises the device and returns,
 * per kernel id, the summed milliseconds and the launch count since the last reset.
 * qad_launch_count() counts all launches of the library, enabled or not.
 */
enum {
  QAD_K_FAKEQUANT = 0, QAD_K_ROUTE = 1, QAD_K_ACT_QUANT = 2, QAD_K_GATHER = 3,
  QAD_K_GEMM_FC1 = 4, QAD_K_GEMM_FC2 = 5, QAD_K_COMBINE = 6, QAD_K_DY_GATHER = 7,
  QAD_K_GEMM_DGRAD_FC2 = 8, QAD_K_GEMM_DGRAD_FC1 = 9, QAD_K_DX_COMBINE = 10,
  QAD_K_GEMM_WGRAD_FC2 = 11, QAD_K_GEMM_WGRAD_FC1 = 12, QAD_K_SCALE_REDUCE = 13,
  QAD_K_GEMM_FC1_RECOMPUTE = 14, /* QAD_FLAG_RECOMPUTE: fc1 again in the dgrad call (Z1 only) */
  QAD_K_DEPLOY_SCALES = 15,      /* QAD_FMT_NVFP4_E4M3: the deployed weight scales */
  QAD_K_COUNT = 16
};
int qad_profile_enable(int on);
int qad_profile_reset(void);
int qad_profile_read(float* ms, int64_t* launches, int n);
const char* qad_kernel_name(int id);
int64_t qad_launch_count(void);

/*
 * Routing permutation that allocates nothing (the pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory, e.g. code running inside
 * a CUDA-graph stream capture where cudaMalloc is not allowed, or a runtime that owns all
 * device memory and gives a plugin only its inputs and outputs).
 *
 * Computes the same maps as the routing step of qad_moe_fwd: the T * topk (token, slot)
 * pairs grouped by expert in (token, slot) order, each expert's rows padded to a
 * multiple of 128; out-of-range or repeated indices are dropped and flagged.
 *   topk_idx  int32 [T, topk]                        (read)
 *   row_token int32 [Rmax], row_slot int32 [Rmax]     token / slot of each padded row, -1 = padding,
 *             Rmax = round_up(T * topk + 127 * E, 128); only the first header[2] are written
 *   row_of    int32 [T * topk]                        padded row of each pair, -1 if dropped
 *   offsets   int32 [E + 1]                           first padded row of each expert
 *   counts    int32 [E]                               routed rows per expert
 *   header    int32 [4]                               device error word (QAD_DEV_*), 128-row
 *                                                     tiles, padded rows, routed rows
 * All pointers are device pointers to int32 data and need only 4-byte alignment (unlike the
 * layer calls' 16 bytes: these kernels read and write single int32 values); nothing is
 * allocated.  The library's own scratch for this call is a file-scope device array of
 * 534 KB per GPU (held until the process exits), sized for E <= QAD_NOALLOC_MAX_EXPERTS and
 * T * topk <= QAD_NOALLOC_MAX_PAIRS; larger problems return QAD_ERR_SCRATCH_LIMIT before
 * anything is launched.  The first call on a device looks up the scratch's device address
 * (cudaGetSymbolAddress) and keeps it for the life of the process, so make that first call
 * before any stream capture, and do not call cudaDeviceReset on a device between calls (a
 * reset unloads the library's device code with the array; its address may change).  Every
 * call shares the one scratch array: calls whose execution overlaps on the GPU (different
 * streams, or different host threads) race and give undefined results; the header is
 * cleared at the start of each call.  Null pointers and sizes outside the limits return
 * QAD_ERR_INVALID_ARG / QAD_ERR_SCRATCH_LIMIT.
 */
enum { QAD_NOALLOC_MAX_EXPERTS = 256, QAD_NOALLOC_MAX_PAIRS = 262144 };
int qad_route_permute_noalloc(const int32_t* topk_idx, int64_t T, int32_t topk, int32_t E,
                              int32_t* row_token, int32_t* row_slot, int32_t* row_of, int32_t* offsets,
                              int32_t* counts, int32_t* header, qad_stream_t stream);

/*
 * Self-check of the failure path (not an operation of the method).  Every pipeline wait of
 * the GEMM kernels is bounded; when one expires the kernel sets QAD_DEV_TIMEOUT in the
 * workspace error word, drains what it issued and returns instead of hanging.  This
 * launches one warp that runs that same bounded-wait routine on a barrier nothing ever
 * arrives on, with a budget of `budget_cycles` SM clock cycles (<= 2e9), and ORs
 * QAD_DEV_TIMEOUT into *err_word (device int32) when it gives up.
 */
int qad_debug_wait_timeout(int32_t* err_word, int64_t budget_cycles, qad_stream_t stream);

/*
 * Self-check of the division inside the quantizers (not an operation of the method).
 * The kernels compute x = fp32(w / s) from the correctly rounded reciprocal of s and one
 * FMA correction (Markstein's theorem) instead of a division per element.  For each i
 * this writes x_ieee[i] (CUDA's IEEE division) and x_fast[i]:
 *   mode 0: the per-element guarded form used for weights -- must equal x_ieee bit for bit;
 *   mode 1: the form used for activations and the scale-gradient factor, which checks only
 *           the block's scale (in [2^-60, 2^60], else mode 0's form) -- must equal x_ieee
 *           bit for bit wherever 2^-11 <= |x| <= 2^100, and round to zero on every grid
 *           below (its callers never produce larger quotients: see the kernels).
 * w, s, x_fast, x_ieee: fp32 [n], device pointers.
 */
int qad_debug_quotient(const float* w, const float* s, float* x_fast, float* x_ieee, int64_t n,
                       int32_t mode, qad_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QAD_H_ */
