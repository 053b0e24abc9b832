/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) MoE-layer hot path.
 *
 *   router GEMM -> top-K routing -> permute -> grouped SwiGLU expert GEMM
 *   -> weighted unpermute / combine
 *
 * Pages the operations come from (titles shortened):
 *   [dispatch] "vLLM CPU MoE: dynamic GEMM dispatch beyond a fixed threshold"
 *              (vllm PR #50949), sections "1. gemm.h", "2. moe_fp8.cpp"
 *   [router]   "vLLM MiniMax-M2 MoE gate optimisation: fused FP32 kernel"
 *              (vllm PR #38445), sections "1. Python layer", "2. CUDA kernel"
 *   [shared]   "vLLM fused shared-expert gate GEMM path on ROCm"
 *              (vllm PR #54185), section "code analysis"
 *   [permute]  "vLLM MoE permute optimisation: buffer pre-allocation"
 *              (vllm PR #43014), sections "1. C++ kernel level", "2. Python layer"
 *   [routing]  "FlashInfer MoE routing optimisation" (flashinfer PR #4152),
 *              sections "1. routing_custom.cu", "2. routing_common.cu"
 *
 * Conventions for every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  Inputs are
 *     const and never written.  The library never allocates device memory,
 *     never frees, never synchronises: all work is queued on `stream`
 *     (a cudaStream_t; NULL = legacy default stream).  Caller scratch and
 *     workspace follow [permute] "1. C++ kernel level": buffers are allocated
 *     once by the caller and reused on every call.
 *   - Layouts are dense row-major with the last index contiguous.
 *   - bf16 tensors are IEEE bfloat16; FP8 weights are OCP e4m3 ("fn") codes
 *     with one fp32 scale per 128 x 128 block (the last block of a dimension
 *     may be narrower); scales are laid out [E][ceil(rows/128)][ceil(cols/128)].
 *     MXFP4 weights ([dispatch] introduction: FP8 and MXFP4 experts) follow
 *     OCP Microscaling: [E][rows][cols/2] bytes, each two E2M1 codes (sign, 2
 *     exponent bits with bias 1, 1 mantissa bit), element 2i in the low
 *     nibble; one UE8M0 scale byte s (value 2^(s-127), s < 255) per 32
 *     consecutive elements of a row, laid out [E][rows][cols/32] (uint8, passed
 *     through the scale pointers); rows must hold whole 32-element blocks.
 *   - Errors found on the host (null pointer, bad size, misalignment, short
 *     scratch) return a status != MOE_OK before anything is queued.  A failed
 *     launch returns MOE_ERR_CUDA.  Errors found by a kernel (an expert id out
 *     of range, a bounded wait that ran out) are written to *dev_status, a
 *     device int32 the caller zeroes; the first error written wins.  The
 *     caller reads it whenever it chooses.
 *   - Alignment: bf16 activation/weight pointers 16-byte aligned, fp32 and
 *     int32 pointers 4-byte aligned, scratch/workspace 256-byte aligned.
 *   - Sizes: 1 <= K <= E <= 1024, H % 16 == 0, I % 16 == 0, T >= 0
 *     (T == 0 is a no-op that returns MOE_OK).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, size out of range */
  MOE_ERR_UNSUPPORTED = 2,   /* combination the kernels do not implement */
  MOE_ERR_WORKSPACE = 3,     /* scratch / workspace too small */
  MOE_ERR_MISALIGNED = 4,    /* pointer alignment rule broken */
  MOE_ERR_CUDA = 5,          /* a CUDA call or launch failed */
  MOE_ERR_DEVICE_STATUS = 6  /* reserved for callers that fold *dev_status in */
} moe_status_t;

/* codes a kernel writes to *dev_status */
#define MOE_DEV_OK 0
#define MOE_DEV_BAD_EXPERT_ID 1  /* permute saw an id outside [0, E) */
#define MOE_DEV_WAIT_TIMEOUT 2   /* a bounded wait inside the expert GEMM ran out */

typedef enum {
  MOE_SCORE_SOFTMAX_RENORM = 0,      /* softmax over E, top-K, weights sum to 1 */
  MOE_SCORE_SIGMOID_BIAS_SCALED = 1  /* key sigmoid(l)+bias, weights scale*s/sum s */
} moe_score_mode_t;

typedef enum {
  MOE_W_BF16 = 0,          /* expert weights bf16 */
  MOE_W_FP8E4M3_B128 = 1,  /* expert weights e4m3 + fp32 128x128 block scales */
  MOE_W_MXFP4 = 2,         /* expert weights MXFP4: e2m1 pairs + a UE8M0 scale per 32 */
  MOE_W8A8_FP8E4M3_B128 = 3 /* weights as MOE_W_FP8E4M3_B128; activations quantised (W8A8) */
} moe_wdtype_t;

/* How the grouped GEMM picks a kernel variant for each expert block. */
typedef enum {
  MOE_DISPATCH_PER_BLOCK = 0,  /* from the block's own m_size ([dispatch] after) */
  MOE_DISPATCH_GLOBAL_AVG = 1, /* from max(1, R/E) for every block ([dispatch] before) */
  MOE_DISPATCH_SIMT = 2,       /* every block on the CUDA-core kernel (cross-check) */
  MOE_DISPATCH_ONE_LAUNCH = 3, /* moe_layer only: every batch of T <= 16 as one launch (see
                                  moe_layer); blocks otherwise as MOE_DISPATCH_PER_BLOCK */
  MOE_DISPATCH_GEMV = 4        /* moe_layer only: batches of T <= 4 with the expert GEMMs as
                                  CUDA-core matrix-vector products (see moe_layer);
                                  otherwise as MOE_DISPATCH_PER_BLOCK */
} moe_dispatch_t;

/* Variant codes reported per expert block. */
#define MOE_VARIANT_SKIP 0    /* m_size == 0: no work */
#define MOE_VARIANT_SKINNY 1  /* small block: narrow token tile */
#define MOE_VARIANT_TILE 2    /* large block: wide tensor-core tile */
#define MOE_VARIANT_SIMT 3    /* CUDA-core kernel (MOE_DISPATCH_SIMT) */
#define MOE_VARIANT_WIDE 4    /* FP8, m_size >= MOE_WIDE_MIN_ROWS: 256-row token tiles */
#define MOE_WIDE_MIN_ROWS 129

typedef struct {
  int T_max;           /* largest T the workspace must hold */
  int H;               /* hidden size */
  int E;               /* routed experts */
  int K;               /* experts per token */
  int I;               /* routed expert intermediate size */
  int has_shared;      /* 1: gate has E+1 rows, row E gates a shared expert */
  int I_shared;        /* shared expert intermediate size (has_shared) */
  int mode;            /* moe_score_mode_t */
  float routed_scale;  /* ScaledSumNormalize factor (mode 1); ignored in mode 0 */
  int wdtype;          /* moe_wdtype_t of the routed experts */
  int m_skinny;        /* blocks with m_size <= m_skinny use the skinny variant;
                          -1 = library default (moe_default_m_skinny()) */
  int dispatch;        /* moe_dispatch_t */
} moe_config_t;

typedef struct {
  const float* wg;         /* [G, H] fp32 gate weight, G = E + has_shared */
  const float* gate_bias;  /* [G] fp32 added to the logits, or NULL */
  const float* sel_bias;   /* [E] fp32 selection bias (mode 1), or NULL = 0 */
  const void* w1;          /* [E, I, H] gate projection (bf16 or e4m3) */
  const void* w3;          /* [E, I, H] up projection */
  const void* w2;          /* [E, H, I] down projection */
  const float* s1;         /* FP8 block scales (fp32) or MXFP4 scale bytes (uint8,
                              cast) of w1 / w3 / w2, else NULL */
  const float* s3;
  const float* s2;
  const void* sw1;         /* shared expert bf16 [I_shared, H], or NULL */
  const void* sw3;         /* [I_shared, H] */
  const void* sw2;         /* [H, I_shared] */
} moe_weights_t;

/* Text for a status code (static storage). */
const char* moe_status_string(moe_status_t status);

/* Default skinny/tile threshold on m_size used when m_skinny == -1. */
int moe_default_m_skinny(void);

/*
 * Variant a block of m_size rows takes, as the grouped GEMM decides it on the
 * device ([dispatch] "2. moe_fp8.cpp": m_size = offsets[e+1] - offsets[e], a
 * block with m_size == 0 returns at once, the kernel is chosen per block;
 * "1. gemm.h": the large-tile kernel is used above a small-M threshold).
 * R = total rows, E = number of blocks (used by MOE_DISPATCH_GLOBAL_AVG, which
 * decides from max(1, R / E) for every non-empty block).  The large-tile side
 * is split once more on the GPU for FP8 weights (wdtype): blocks of more than
 * 128 rows take 256-row token tiles (MOE_VARIANT_WIDE), so each dequantised
 * weight tile serves twice the tokens; otherwise 128-row tiles.
 * Host-callable copy of the device predicate; returns a MOE_VARIANT_* code.
 */
int moe_block_variant(int64_t m_size, int64_t R, int E, int m_skinny, int dispatch, int wdtype);

/*
 * R: router (gate) GEMM.   logits[t, g] = sum_h fp32(x[t, h]) * wg[g, h] (+ gate_bias[g])
 * [router] "2. CUDA kernel": bf16 activations are loaded 8 at a time (16 bytes)
 * and widened to fp32 in registers, so no fp32 copy of x is written; the
 * products accumulate in fp32 on the CUDA cores.  [shared] "code analysis":
 * with a fused shared-expert gate, G = E + 1.
 *   x         [T, H] bf16, 16-byte aligned, H % 8 == 0
 *   wg        [G, H] fp32 (nn.Linear layout), 16-byte aligned
 *   gate_bias [G] fp32 or NULL
 *   logits    [T, G] fp32 output
 * Deterministic: the summation order depends only on (T, H, G).
 */
moe_status_t moe_router_gemm(const void* x, const float* wg, const float* gate_bias,
                             float* logits, int T, int H, int G, moe_stream_t stream);

/* Scratch bytes moe_router_gemm_tc needs for (H, G): 3 * G * H bf16, rounded up. */
moe_status_t moe_router_tc_scratch_bytes(int H, int G, size_t* bytes);

/*
 * R on the tensor cores, for prefill-sized batches.  Same operation and
 * arguments as moe_router_gemm, computed to fp32 accuracy from bf16 MMAs:
 * [router] "2. CUDA kernel" keeps the gate in fp32 with bf16 activations;
 * the bf16 activations are exact MMA operands, and the fp32 weight is split
 * exactly into three bf16 parts (hi = bf16(w), mid = bf16(w - hi),
 * lo = bf16(w - hi - mid)) whose products with x are exact in fp32 and
 * accumulate in one fp32 TMEM accumulator.  |error| stays within a few fp32
 * roundings of sum_h |x_h w_h|.
 *   scratch    >= moe_router_tc_scratch_bytes(H, G), 256-byte aligned; the
 *              split weight is written there on every call (two launches:
 *              split, then the GEMM), so wg may change between calls
 *   dev_status optional int32 device word: MOE_DEV_WAIT_TIMEOUT when a
 *              pipeline wait gave up (the logits are then undefined)
 * Deterministic: the split-K partials are summed in a fixed order.
 * moe_layer uses this path for T >= 64 and moe_router_gemm below that.
 */
moe_status_t moe_router_gemm_tc(const void* x, const float* wg, const float* gate_bias,
                                float* logits, int T, int H, int G, void* scratch,
                                size_t scratch_bytes, int32_t* dev_status, moe_stream_t stream);

/*
 * K: top-K routing, one warp per token.  [routing] "1. routing_custom.cu":
 * every lane keeps its own sorted top-K candidates (from the experts it
 * reads) and the warp merges the lane heads K times with shuffles; "2.
 * routing_common.cu": E = 896 has its own tier (28 experts per lane) instead
 * of running as 1024.
 *   mode MOE_SCORE_SOFTMAX_RENORM: select the K largest logits among columns
 *     [0, E); weights = softmax over the selected logits (sum 1).
 *   mode MOE_SCORE_SIGMOID_BIAS_SCALED: s = sigmoid(l) in a fixed float32
 *     formula (Cody-Waite exp + degree-7 Taylor, each step one correctly
 *     rounded operation), key = s + sel_bias[e]; select the K largest keys;
 *     weights = scale * s / sum_selected s.
 *   Equal keys: the lower expert index wins.  Outputs are in selection order
 *   (key descending).
 *   logits       [T, ld_logits] fp32, ld_logits >= E
 *   sel_bias     [E] fp32 or NULL (mode 1 only)
 *   ids          [T, K] int32 output;  weights [T, K] fp32 output
 *   shared_gate  [T] fp32 output sigmoid(logits[t, E]) or NULL (needs
 *                ld_logits >= E + 1)
 */
moe_status_t moe_topk_route(const float* logits, int ld_logits, const float* sel_bias,
                            int T, int E, int K, int mode, float scale,
                            int32_t* ids, float* weights, float* shared_gate,
                            moe_stream_t stream);

/* Scratch bytes moe_permute needs for (T, E, K). */
moe_status_t moe_permute_scratch_bytes(int T, int E, int K, size_t* bytes);

/*
 * P: permute.  Replica f = t*K + k of token t, routed to expert e = ids[f],
 * goes to row offsets[e] + (number of replicas f' < f routed to e): a stable
 * counting sort ([permute] "1. C++ kernel level" permutes the replicas into
 * expert order; [dispatch] "2. moe_fp8.cpp" reads each block's size as
 * offsets[e+1] - offsets[e]).  Done as a per-chunk histogram, a scan and a
 * stable scatter (warp match + popcount), then a row gather.
 *   x            [T, H] bf16 (may be NULL when xp is NULL)
 *   ids          [T, K] int32 in [0, E); an id outside it sets
 *                MOE_DEV_BAD_EXPERT_ID and that replica is dropped
 *                (flat_to_row = -1)
 *   offsets      [E + 1] int32 output, offsets[0] = 0
 *   row_to_flat  [T*K] int32 output;  flat_to_row [T*K] int32 output
 *   xp           [T*K, H] bf16 output, xp[row] = x[row_to_flat[row] / K];
 *                NULL skips the gather
 *   scratch      >= moe_permute_scratch_bytes(T, E, K) bytes, 256-byte aligned
 */
moe_status_t moe_permute(const void* x, const int32_t* ids, int T, int H, int E, int K,
                         int32_t* offsets, int32_t* row_to_flat, int32_t* flat_to_row,
                         void* xp, void* scratch, size_t scratch_bytes,
                         int32_t* dev_status, moe_stream_t stream);

/*
 * moe_permute without caller scratch (the pages have no counterpart; this is a
 * convenience of this library).  For callers that cannot allocate device
 * memory at all -- e.g. code whose device memory is owned entirely by a fixed
 * pool or arena set up at start-up, or hooks that are not allowed to call
 * cudaMalloc -- and so have no scratch buffer to pass.  Same arguments,
 * results and errors as moe_permute, minus scratch / scratch_bytes.
 *   - The scratch is a fixed array of MOE_PERMUTE_STATIC_SCRATCH_BYTES inside
 *     the library, held on every GPU that loads the library until the process
 *     exits.  It holds one int32 count per expert for every chunk of 256
 *     replicas, so sizes whose moe_permute_scratch_bytes(T, E, K) exceeds it
 *     return MOE_ERR_WORKSPACE before anything is queued: the largest accepted
 *     T*K is 255 chunks (65280 replicas) at E = 1024, 292 chunks (74752) at
 *     E = 896, 511 chunks (130816) at E = 512 and 2047 chunks (524032) at
 *     E = 128.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it with the device's current context;
 *     a call that finds another context (after cudaDeviceReset) looks it up
 *     again.  Make the first call on a device, and the first after a reset,
 *     before any stream capture.  No cudaMalloc, cudaFree or allocating
 *     routine is called.
 *   - Every call shares the array and it keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls whose kernels may overlap
 *     on the GPU -- on different streams without ordering, or from different
 *     host threads -- race on it: order them on one stream.
 */
#define MOE_PERMUTE_STATIC_SCRATCH_BYTES (1u << 20)
moe_status_t moe_permute_static(const void* x, const int32_t* ids, int T, int H, int E, int K,
                                int32_t* offsets, int32_t* row_to_flat, int32_t* flat_to_row,
                                void* xp, int32_t* dev_status, moe_stream_t stream);

/* Scratch bytes moe_grouped_gemm needs for R rows in E_blocks blocks (every
 * weight format but MOE_W8A8_FP8E4M3_B128). */
moe_status_t moe_grouped_gemm_scratch_bytes(int R, int E_blocks, size_t* bytes);
/* Scratch bytes for any weight format: as above, plus for
 * MOE_W8A8_FP8E4M3_B128 the e4m3 copies of xp and hact with their scales. */
moe_status_t moe_grouped_gemm_scratch_bytes_ex(int R, int E_blocks, int H, int I, int wdtype,
                                               size_t* bytes);

/*
 * G1 + G2: grouped SwiGLU expert GEMM over expert-contiguous row blocks.
 *   for every block e with m_e = offsets[e+1] - offsets[e] > 0, rows r in it:
 *     hact[r] = bf16( silu(xp[r] . W1[e]^T) * (xp[r] . W3[e]^T) )   (fp32 accumulate)
 *     y[r]    = bf16( hact[r] . W2[e]^T )
 * The kernel variant is chosen on the device for each block from its own m_e
 * (moe_block_variant), never from a global average unless dispatch asks for
 * it ([dispatch] "2. moe_fp8.cpp").  Every variant runs tcgen05 tensor-core
 * MMAs fed by TMA with TMEM accumulators: the skinny variant uses a 16-row
 * token tile, the tile variant a 128-row one and the wide variant (FP8) a
 * 256-row one.  W8A16 FP8 weights need H, I <= 8192.
 *   xp        [R, H] bf16, 16-byte aligned
 *   offsets   [E_blocks + 1] int32 (device), or NULL for one block [0, R)
 *   w1, w3    [E_blocks, I, H]; w2 [E_blocks, H, I]; bf16 or e4m3 per wdtype
 *   s1, s3    [E_blocks, ceil(I/128), ceil(H/128)] fp32; s2 [E_blocks, ceil(H/128), ceil(I/128)]
 *             (FP8 weights, W8A16 or W8A8); MXFP4: uint8 scale bytes
 *             [E_blocks, rows, cols/32] cast to these pointers; bf16: NULL
 *   hact      [R, I] bf16 output;  y [R, H] bf16 output (rows outside every
 *             block are left untouched)
 *   block_variant  [E_blocks] int32 output of MOE_VARIANT_* codes, or NULL
 *   scratch   >= moe_grouped_gemm_scratch_bytes_ex(R, E_blocks, H, I, wdtype),
 *             256-byte aligned
 * W8A8 (wdtype MOE_W8A8_FP8E4M3_B128; the pages fix FP8 weights, not the
 * activations): both GEMMs' activations are quantised to e4m3 with one fp32
 * scale per row and 128 columns -- s = amax / 448 (IEEE fp32 division, 0 for
 * an all-zero block), code = e4m3(v / s) rounded to nearest even, saturated
 * at 448 -- xp before G1, and the bf16 hact (as stored) before G2; the
 * products run as kind::f8f6f4 MMAs, each 128-wide K block scaled by the
 * weight block scale times the row's activation scale and summed in fp32.
 * Every non-empty block takes one kernel with 128-row token tiles (variant
 * MOE_VARIANT_TILE; a prefill option: no skinny variant), dispatch
 * MOE_DISPATCH_PER_BLOCK or MOE_DISPATCH_GLOBAL_AVG (MOE_DISPATCH_SIMT:
 * MOE_ERR_UNSUPPORTED).
 */
moe_status_t moe_grouped_gemm(const void* xp, const int32_t* offsets, int E_blocks, int R,
                              int H, int I, int wdtype,
                              const void* w1, const void* w3, const void* w2,
                              const float* s1, const float* s3, const float* s2,
                              void* hact, void* y, int m_skinny, int dispatch,
                              int32_t* block_variant, void* scratch, size_t scratch_bytes,
                              int32_t* dev_status, moe_stream_t stream);

/*
 * U: weighted unpermute / combine ([permute] introduction: the inverse of
 * permute that returns expert outputs to token order and combines them).
 *   out[t] = bf16( sum_{k=0..K-1} weights[t,k] * y[flat_to_row[t*K+k]]
 *                  + shared_gate[t] * shared_y[t] )
 *   summed in fp32 in k order, one rounding to bf16 at the end.  A replica
 *   with flat_to_row < 0 contributes nothing.
 *   y [T*K, H] bf16; flat_to_row [T*K] int32; weights [T, K] fp32
 *   shared_y [T, H] bf16 and shared_gate [T] fp32: both or neither (NULL)
 *   out [T, H] bf16 output
 */
moe_status_t moe_unpermute(const void* y, const int32_t* flat_to_row, const float* weights,
                           int T, int K, int H, const void* shared_y,
                           const float* shared_gate, void* out, moe_stream_t stream);

/* Workspace bytes moe_layer needs for cfg (sized for cfg->T_max). */
moe_status_t moe_workspace_bytes(const moe_config_t* cfg, size_t* bytes);

/*
 * The whole layer on one stream, no host synchronisation:
 *   R -> K -> P -> G1/G2 (+ shared expert) -> U.
 *   x    [T, H] bf16 input, out [T, H] bf16 output, T <= cfg->T_max
 *   workspace  >= moe_workspace_bytes(cfg), 256-byte aligned; holds every
 *              intermediate (logits, ids, weights, offsets, permuted rows,
 *              expert activations and outputs, plans).  Its `sync` region
 *              (moe_workspace_layout: from `sync` up to `logits`; completion
 *              counters) must be zero before the first call -- e.g. zero the
 *              whole workspace once after allocating it; every call leaves it
 *              zero again.
 * Small batches ([router] "why" 1: at low concurrency launches and round trips
 * between them set the time; [permute] performance table):
 *   - T <= 4 with bf16, W8A16 FP8 or MXFP4 experts, cfg->dispatch
 *     MOE_DISPATCH_GEMV, or MOE_DISPATCH_PER_BLOCK with T <= 2 (MXFP4: T = 1;
 *     where it measured fastest): G1 and G2 as CUDA-core matrix-vector products (a
 *     warp streams whole weight rows, no K split; the shared expert in the
 *     same two launches; [dispatch] "1. gemm.h": tiny blocks skip the tiled
 *     GEMM), then the combine; blocks report the skinny variant.  Where
 *     T * K <= 32 and E <= 128 (or K <= 16 and E <= 4096 / T rounded up to a
 *     power of two) the first launch computes only the logits and every G1
 *     CTA routes the batch itself (top-K, permutation and plan, CTA 0 writing
 *     them to the workspace); otherwise the fused routing launch comes first;
 *   - the whole layer -- router, top-K, permute, G1/G2, shared expert and the
 *     combine -- runs as ONE cooperative launch of one CTA per SM (bf16 expert
 *     weights, T <= 16) when cfg->dispatch is MOE_DISPATCH_ONE_LAUNCH, or,
 *     under MOE_DISPATCH_PER_BLOCK, where it measured faster than the
 *     multi-launch path: a shared expert with 3 <= T <= 4, or E <= 128 with
 *     4 <= T <= 8;
 *   - otherwise for T <= 32 the router, top-K, permute and the GEMM plan run
 *     as one fused launch, followed by the GEMM and combine launches.
 * The results are those of the separate steps (same routing and permutation
 * bit for bit, the same arithmetic up to the order of fp32 sums).
 */
moe_status_t moe_layer(const moe_config_t* cfg, int T, const void* x, const moe_weights_t* w,
                       void* out, void* workspace, size_t workspace_bytes,
                       int32_t* dev_status, moe_stream_t stream);

/*
 * Byte offsets of the intermediates inside a moe_layer workspace, for callers
 * that inspect them (tests, profilers).  Filled for cfg and T_max.
 */
typedef struct {
  size_t logits, ids, weights, shared_gate, offsets, row_to_flat, flat_to_row,
      xp, hact, y, shared_hact, shared_y, block_variant, permute_scratch, gemm_scratch,
      shared_gemm_scratch, sync, splitk, router_split, total;
} moe_workspace_layout_t;

moe_status_t moe_workspace_layout(const moe_config_t* cfg, moe_workspace_layout_t* layout);

/*
 * Self-test of the library's bounded cross-CTA wait (the one the grouped
 * GEMM's single-launch G1+G2 path uses for a G2 tile's dependency on G1): one
 * thread waits until the device int32 *counter >= target, reading it with GPU
 * acquire loads, for at most limit_us microseconds; if the wait runs out it
 * writes MOE_DEV_WAIT_TIMEOUT into *dev_status (first error wins) and
 * returns, leaving the context usable.  Lets a caller check that a stuck
 * dependency ends in a status word, not a hang.  counter and dev_status are
 * device pointers owned by the caller; 0 < limit_us <= 10^7, else
 * MOE_ERR_INVALID_ARG.  Asynchronous on `stream`, not ordered by programmatic
 * dependent launch (it waits for the stream's earlier work).
 */
moe_status_t moe_bounded_wait_check(const int32_t* counter, int target, int limit_us,
                                    int32_t* dev_status, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
