// The whole MoE layer for a small batch (T <= 16 tokens) in ONE launch.
//
// "vLLM MiniMax-M2 MoE gate optimisation: fused FP32 kernel" (vllm PR
// #38445), "why" 1: at low concurrency the launches and the fp32 round trip
// between them, not the arithmetic, set the time; "vLLM MoE permute
// optimisation: buffer pre-allocation" (vllm PR #43014), performance table:
// the smallest batches gain most from removing per-call overhead.  Here the
// router, top-K, permute, both expert GEMMs (and the shared expert) and the
// combine share one persistent, cooperative launch of one CTA per SM:
//
//   1. router: CTA c computes gate rows c, c + grid, ... for every token
//      (16-byte bf16 vectors widened to fp32, fixed-order block reduction)
//      and counts itself done in a global word;
//   2. every CTA waits (bounded) until all have counted, then routes every
//      token itself (warp top-K, logits read through L2), permutes the
//      replicas (stable counting sort) and lists the active experts ("slots",
//      ascending expert index; a shared expert is one more slot holding every
//      token).  No CTA routes for another, so nothing waits on a serial step;
//   3. the weight streams.  G1 is split into (slot, 128-feature block) pairs
//      of ceil(H/64) 64-wide K steps, G2 likewise over H-feature blocks; the
//      steps of each phase are cut into one contiguous, equal share per CTA,
//      so every SM streams the same number of weight bytes.  Operand B is the
//      token rows themselves (x for G1: all T rows, the epilogue keeps the
//      slot's tokens; hact rows of the slot for G2), 16 rows per MMA
//      (tcgen05, M = 128 weight rows, N = 16, fp32 accumulators in TMEM);
//   4. a pair cut over several CTAs is summed by the last of them to arrive
//      (a count per pair and lane quarter), in CTA order, so the result is
//      deterministic; a G1 pair's reducer stores its hact columns and counts
//      them ready;
//   5. G2 needs the hact that G1 stores: its W2 tiles (two K steps per
//      stage) are loaded ahead, as they do not depend on G1, and once the
//      ring holds nothing else the producer waits (bounded, once) until every
//      G1 pair is stored, then adds the hact tiles;
//   6. combine: every stored y block counts itself for each of its tokens;
//      the block that completes a token's K (+1 shared) contributions sums
//      them in k order and stores that part of out.
// The last CTA to finish clears the counters for the next call.  Every wait is
// bounded: one that runs out writes MOE_DEV_WAIT_TIMEOUT to dev_status and the
// CTA drains its copies and MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"
#include "tmap.h"
#include "topk_group.cuh"
#include "topk_warp.cuh"

namespace {

using namespace moe_ptx;
using namespace moe_route;

constexpr int kThreads = 256;           // the working warps
constexpr int kWarps = kThreads / 32;
constexpr int kBlock = kThreads + 32;   // plus one warp that warms the instruction cache
constexpr int kBM = 128;                         // weight rows per MMA (output features)
constexpr int kBK = 64;                          // K per stage: one 128-byte swizzle row
constexpr int kBN = 16;                          // token columns per MMA
constexpr int kMaxT = kDecodeMaxT;               // tokens
constexpr int kMaxR = kMaxT * 32;                // replicas (K <= 32)
constexpr int kMaxE = 1024;
constexpr int kWBytes = kBM * kBK * 2;           // one bf16 weight tile
constexpr int kBBytes = kBN * kBK * 2;           // one token tile
// a stage holds one G1 step (W1, W3 and x tiles) or two consecutive G2 steps
// of one pair (two W2 tiles and their hact tiles)
constexpr int kStageBytes = 2 * kWBytes + 2 * kBBytes;
constexpr int kStages = 5;
constexpr int kAcc = 4;                          // accumulator sets in TMEM
constexpr int kAccCols = 2 * kBN;                // W1 (or W2) columns, then W3 columns
constexpr int kTmemCols = 128;
constexpr int kEpiWarp0 = 2;                     // warps 2..5 read the accumulators
constexpr int kPieceFloats = kBN * 32 * 2;       // per lane quarter: 16 columns x 32 lanes x (g, u)
constexpr uint64_t kWaitLimitNs = 2000000000ull; // 2 s
constexpr size_t kDynSmem = 1024 + (size_t)kStages * kStageBytes;
static_assert(kMaxT <= kBN, "every token is one MMA column");
static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte alignment");

struct Params {
  const __nv_bfloat16* x;
  const float* wg;
  const float* gate_bias;
  const float* sel_bias;
  int T, H, G, E, K, I, Is, mode, has_shared;
  float scale;
  float* logits;
  int32_t* ids;
  float* weights;
  float* shared_gate;
  int32_t* offsets;
  int32_t* row_to_flat;
  int32_t* flat_to_row;
  int32_t* block_variant;
  __nv_bfloat16* hact;
  __nv_bfloat16* y;
  __nv_bfloat16* sh_hact;
  __nv_bfloat16* sh_y;
  __nv_bfloat16* out;
  float* part;        // [2 phases][kDecodeMaxGrid][2][4][kPieceFloats] partial sums of cut pairs
  uint32_t* sync;     // [0] router count, [1] exit count, [2] stored G1 quarters, then cnt1, cnt2, comb
  int P1max, P2max;   // pair capacities of the counter arrays
  int32_t* dev_status;
  int m_skinny, dispatch, wdtype;
  int route_kind;
};

struct Maps {
  CUtensorMap w1, w3, w2;  // routed experts [E][I][H], [E][I][H], [E][H][I]
  CUtensorMap x;           // [T][H]
  CUtensorMap h;           // hact [R][I]
  CUtensorMap sw1, sw3, sw2, hs;  // shared expert [I_s][H] x2, [H][I_s]; shared hact [T][I_s]
};

MOE_DEVICE float silu_f(float g) { return g / (1.f + __expf(-g)); }

MOE_DEVICE uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// wait until *p >= target (GPU-scope acquire); bounded
MOE_DEVICE bool wait_geq(const uint32_t* p, uint32_t target, const volatile int* abort) {
  if (ld_acquire_u32(p) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1; i < (1u << 30); ++i) {
    if (i > 4096) __nanosleep(64);  // spin first: the waits here are short
    if (ld_acquire_u32(p) >= target) return true;
    if ((i & 15) == 0) {
      if (abort && *abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
  return false;
}

// GPU-scope atomics carrying the ordering themselves (no separate fence): a
// release add publishes the writes that happen before it -- the lane's own,
// and the warp's when a __syncwarp precedes it; an acq_rel add also acquires
// what earlier releases on the word published.
MOE_DEVICE uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
MOE_DEVICE void red_add_release(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// one contiguous global -> shared copy on the TMA engine (16-byte aligned,
// size a multiple of 16), completing on an mbarrier's transaction count
MOE_DEVICE void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

MOE_DEVICE void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

MOE_DEVICE void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// take back `bytes` of expected transactions that will never be issued, so
// the stage's phase completes once the copies that were issued have landed
MOE_DEVICE void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// ---------------------------------------------------------------- top-K of one token
// One warp; ids/weights go to shared memory.  kind picks the list shape
// (as the fused routing launches choose it from E and K).
template <int NPL, int LK>
MOE_DEVICE void route_warp(const float* row, const Params& p, int32_t* ids, float* w) {
  warp_topk<NPL, LK, true>(row, p.sel_bias, p.E, p.K, p.mode, p.scale, ids, w, nullptr);
}

template <int NPL, int LK, bool kVec>
MOE_DEVICE void route_group(const float* row, const Params& p, int32_t* ids, float* w,
                            int32_t* s_ids) {
  float l[NPL];
  group_load<32, NPL, kVec, true>(row, true, p.E, l);
  group_route<32, NPL, LK, kVec, true>(l, row, true, 1, p.sel_bias, p.E, p.K, p.mode, p.scale,
                                       ids, w, nullptr, s_ids);
}

__device__ __noinline__ void route_token(int kind, const float* row, const Params& p,
                                         int32_t* ids, float* w, int32_t* s_ids) {
  switch (kind) {
    case 0: route_warp<1, 1>(row, p, ids, w); break;
    case 1: route_warp<2, 2>(row, p, ids, w); break;
    case 2: route_warp<4, 2>(row, p, ids, w); break;
    case 3: route_warp<4, 4>(row, p, ids, w); break;
#define MOE_DL_GROUP(base, VEC)                                      \
    case base + 0: route_group<8, 4, VEC>(row, p, ids, w, s_ids); break;  \
    case base + 1: route_group<8, 8, VEC>(row, p, ids, w, s_ids); break;  \
    case base + 2: route_group<16, 4, VEC>(row, p, ids, w, s_ids); break; \
    case base + 3: route_group<16, 8, VEC>(row, p, ids, w, s_ids); break; \
    case base + 4: route_group<28, 4, VEC>(row, p, ids, w, s_ids); break; \
    case base + 5: route_group<28, 8, VEC>(row, p, ids, w, s_ids); break; \
    case base + 6: route_group<32, 4, VEC>(row, p, ids, w, s_ids); break; \
    case base + 7: route_group<32, 8, VEC>(row, p, ids, w, s_ids); break;
    MOE_DL_GROUP(4, false)
    MOE_DL_GROUP(12, true)
#undef MOE_DL_GROUP
    default: break;
  }
}

// Large E at very small T: "FlashInfer MoE routing optimisation" (flashinfer
// PR #4152), lessons 2 -- for E = 512-1024 and K = 9-16 worker warps each take
// a partition of the experts and warp 0 merges their picks.  Here P warps
// route one token: warp q picks the top min(K, n) of experts [q*EP, q*EP + n)
// with warp_topk (every expert of a lane fits its list), then one warp
// merges the P partitions' picks.  The merge keeps the same order (larger
// key first, lower expert index first among equal keys), so the K picks are
// those of a single warp over all E, bit for bit.
template <int NPL>
MOE_DEVICE void route_part_npl(const float* row, const Params& p, int base, int n, int kp,
                               int32_t* cand, float* wscratch) {
  warp_topk<NPL, NPL, true>(row + base, p.sel_bias ? p.sel_bias + base : nullptr, n, kp, p.mode,
                            p.scale, cand, wscratch, nullptr);
  __syncwarp();
  if (lane_id() < kp) cand[lane_id()] += base;  // partition-local -> expert id
  __syncwarp();
}

__device__ __noinline__ void route_part(const float* row, const Params& p, int base, int n,
                                        int kp, int32_t* cand, float* wscratch) {
  const int npl = moe_cdiv(n, 32);
  if (npl <= 1) route_part_npl<1>(row, p, base, n, kp, cand, wscratch);
  else if (npl <= 2) route_part_npl<2>(row, p, base, n, kp, cand, wscratch);
  else if (npl <= 4) route_part_npl<4>(row, p, base, n, kp, cand, wscratch);
  else if (npl <= 8) route_part_npl<8>(row, p, base, n, kp, cand, wscratch);
  else route_part_npl<16>(row, p, base, n, kp, cand, wscratch);
}

// One warp: the token's top K among the partitions' picks (partition q's
// kp picks at cand[q * 32 ..], the last partition's kp_last; at most 128 in
// all), weights as warp_topk.
__device__ __noinline__ void route_merge(const float* row, const Params& p, const int32_t* cand,
                                         int P, int kp, int kp_last, int32_t* ids_out,
                                         float* w_out) {
  const int lane = lane_id(), K = p.K;
  const int nc = (P - 1) * kp + kp_last;
  constexpr int kL = 4;  // candidates per lane
  uint32_t lk[kL];
  int li[kL];
#pragma unroll
  for (int s = 0; s < kL; ++s) { lk[s] = 0u; li[s] = 0x7fffffff; }
#pragma unroll
  for (int s = 0; s < kL; ++s) {
    const int i = lane + 32 * s;
    if (i < nc) {
      const int q = min(i / kp, P - 1);
      const int e = cand[q * 32 + (i - q * kp)];
      const float l = __ldcg(row + e);
      const float key = p.mode == MOE_SCORE_SIGMOID_BIAS_SCALED
                            ? __fadd_rn(sigmoid_key(l), p.sel_bias ? __ldg(p.sel_bias + e) : 0.f)
                            : l;
      uint32_t nk = order_key(key);
      int ni = e;
#pragma unroll
      for (int q = 0; q < kL; ++q) {
        const bool b = better(nk, ni, lk[q], li[q]);
        const uint32_t tk = lk[q];
        const int ti = li[q];
        lk[q] = b ? nk : tk;
        li[q] = b ? ni : ti;
        nk = b ? tk : nk;
        ni = b ? ti : ni;
      }
    }
  }
  int my_id = -1;
  for (int r = 0; r < K; ++r) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, lk[0]);
    const uint32_t mi = __reduce_min_sync(0xffffffffu, lk[0] == m ? (uint32_t)li[0] : 0xffffffffu);
    if (li[0] == (int)mi) {
#pragma unroll
      for (int q = 0; q < kL - 1; ++q) { lk[q] = lk[q + 1]; li[q] = li[q + 1]; }
      lk[kL - 1] = 0u;
      li[kL - 1] = 0x7fffffff;
    }
    if (lane == r) my_id = (int)mi;
  }
  float v = 0.f;
  if (p.mode == MOE_SCORE_SOFTMAX_RENORM) {
    const float l = lane < K ? __ldcg(row + my_id) : 0.f;
    const float m = __shfl_sync(0xffffffffu, l, 0);  // the first pick is the largest
    v = lane < K ? expf(l - m) : 0.f;
  } else {
    v = lane < K ? sigmoid_key(__ldcg(row + my_id)) : 0.f;
  }
  float sum = v;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < K) {
    ids_out[lane] = my_id;
    w_out[lane] = p.mode == MOE_SCORE_SOFTMAX_RENORM ? v / sum : p.scale * v / sum;
  }
}

// ---------------------------------------------------------------- schedule
// Pairs and steps, identical in every CTA (computed from the shared plan).
//   G1 pair p: routed slot j = p / nb1r, block p % nb1r (p < n_r * nb1r), then
//              the shared slot's nb1s blocks; nk1 = ceil(H/64) steps each
//   G2 pair p: slot j = p / nb2, block p % nb2; routed pairs have nk2r =
//              ceil(I/64) steps, the shared slot's nk2s = ceil(I_s/64)
// A phase's S steps are cut into shares of ceil(S / grid) consecutive steps:
// CTA c takes [c * chunk, (c + 1) * chunk) (clipped to S), so every CTA that
// owns a step owns a full share except the last one, and empty shares come
// only after every non-empty one (a pair's pieces are consecutive CTAs).
struct Sched {
  int n_r, nb1r, nb1s, nk1, nb2, nk2r, nk2s;
  long long P1, S1, P2, S2, S2r, chunk1, chunk2;

  MOE_DEVICE long long lo(long long S, long long chunk, int c) const {
    return min(S, (long long)c * chunk);
  }
  MOE_DEVICE int cta_of(long long chunk, long long s) const { return (int)(s / chunk); }
  MOE_DEVICE int pair_of(int phase, long long s) const {
    if (phase == 1) return (int)(s / nk1);
    if (s < S2r) return (int)(s / nk2r);
    return n_r * nb2 + (int)((s - S2r) / nk2s);
  }
  MOE_DEVICE long long first_step(int phase, int pair) const {
    if (phase == 1) return (long long)pair * nk1;
    if (pair < n_r * nb2) return (long long)pair * nk2r;
    return S2r + (long long)(pair - n_r * nb2) * nk2s;
  }
  MOE_DEVICE int nk_of(int phase, int pair) const {
    return phase == 1 ? nk1 : (pair < n_r * nb2 ? nk2r : nk2s);
  }
  MOE_DEVICE int slot1(int pair) const { return pair < n_r * nb1r ? pair / nb1r : n_r; }
  MOE_DEVICE int blk1(int pair) const { return pair < n_r * nb1r ? pair % nb1r : pair - n_r * nb1r; }
};

// A maximal run of one CTA's steps inside one pair.
struct Piece {
  int pair, k0, k1;  // steps [k0, k1) of the pair
  bool full;         // the whole pair: no partial sums
};

MOE_DEVICE Piece piece_at(const Sched& s, int phase, long long cur, long long end,
                          long long cta_lo) {
  Piece pc;
  pc.pair = s.pair_of(phase, cur);
  const long long f = s.first_step(phase, pc.pair);
  const int nk = s.nk_of(phase, pc.pair);
  pc.k0 = (int)(cur - f);
  pc.k1 = (int)min((long long)nk, end - f);
  pc.full = pc.k0 == 0 && pc.k1 == nk;
  return pc;
}

// ---------------------------------------------------------------- the kernel
// named barrier of the working warps only (the warm-up warp is elsewhere)
MOE_DEVICE void bar_workers() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

__global__ void __launch_bounds__(kBlock, 1)
decode_layer_kernel(const Params p, const __grid_constant__ Maps maps) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float red[kWarps][kMaxT];
  __shared__ int32_t ids_s[kMaxR];
  __shared__ float w_s[kMaxR];
  __shared__ int32_t f2r_s[kMaxR];
  __shared__ int32_t r2f_s[kMaxR];
  __shared__ int32_t mask_s[kMaxE];
  __shared__ int32_t wtot_s[kWarps][2];
  __shared__ int32_t off_s[kMaxE + 1];
  __shared__ int4 slot_s[kMaxR + 1];  // {expert (-1: shared), first row, rows, token mask}
  __shared__ float gsh_s[kMaxT];
  __shared__ int32_t sids_s[kWarps][32];
  __shared__ float wsc_s[kWarps][32];
  __shared__ int32_t warm_i[2][32];
  __shared__ float warm_f[32];
  __shared__ int n_slots_s;
  __shared__ alignas(8) uint64_t bars[2 * kStages + 2 * kAcc + 2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_s;
  __shared__ int last_s;

  const int tid = threadIdx.x, warp = warp_id(), lane = lane_id();
  const bool worker = tid < kThreads;
  const int T = p.T, H = p.H, G = p.G, E = p.E, K = p.K;
  const int R = T * K;
  const int grid = (int)gridDim.x, c = (int)blockIdx.x;
  uint32_t* router_ctr = p.sync;
  uint32_t* exit_ctr = p.sync + 1;
  uint32_t* g1_done = p.sync + 2;
  uint32_t* cnt1 = p.sync + 64;
  uint32_t* cnt2 = cnt1 + 4 * (size_t)p.P1max;
  uint32_t* comb = cnt2 + 4 * (size_t)p.P2max;
  volatile int* abort_flag = &abort_s;
  auto fail = [&]() {
    moe_set_status(p.dev_status, MOE_DEV_WAIT_TIMEOUT);
    *abort_flag = 1;
  };

  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto acc_full = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
  auto acc_empty = [&](int a) { return bar0 + 8u * (2 * kStages + kAcc + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 2 * kAcc);
  const uint32_t router_bar = drain_bar + 8u;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < kAcc; ++a) {
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), 32 * 4);
    }
    mbar_init(drain_bar, 1);
    mbar_init(router_bar, 1);
    abort_s = 0;
    n_slots_s = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.w1);
    prefetch_tmap(&maps.w3);
    prefetch_tmap(&maps.w2);
    prefetch_tmap(&maps.x);
    prefetch_tmap(&maps.h);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
    tmem_relinquish();
  }

  __syncthreads();  // barriers initialised
  // ---------------- 1. router rows c, c + grid, ... for every token
  // The CTA's rows are worked on together (wpr warps per row, rows_pp rows
  // per pass).  When they fit in the stage ring (idle until the GEMMs), one
  // thread brings them in with bulk copies, all in flight at once.
  // partitions per token for the routing (a power of two, P * T <= kWarps)
  // when E is large
  int P = 1;
  if (E > 128)
    while (2 * P * T <= kWarps && 2 * P * min(K, moe_cdiv(E, 2 * P)) <= 128) P *= 2;
  if (!worker) {
    // The routing code runs once per call on every SM, first thing after the
    // router; its first execution pays for fetching the instructions.  This
    // warp runs the same code on whatever the logits buffer holds (nothing is
    // kept) while the router waits on memory, so the real route finds it
    // fetched.
    const float* row = p.logits;
    if (P > 1) {
      const int n = min(moe_cdiv(E, P), E), kp = min(K, n);
      route_part(row, p, 0, n, kp, warm_i[0], warm_f);
      route_merge(row, p, warm_i[0], 1, kp, kp, warm_i[1], warm_f);
    } else {
      route_token(p.route_kind, row, p, warm_i[1], warm_f, warm_i[0]);
    }
  } else {
    const int nrows = c < G ? (G - c + grid - 1) / grid : 0;
    const size_t row_bytes = (size_t)H * sizeof(float);
    const bool bulk = nrows > 0 && (size_t)nrows * row_bytes <= (size_t)kStages * kStageBytes;
    const float* wrows = reinterpret_cast<const float*>(smem);
    if (bulk) {
      if (tid == 0) {
        mbar_arrive_expect_tx(router_bar, (uint32_t)(nrows * row_bytes));
        for (int r = 0; r < nrows; ++r)
          bulk_load(sbase + (uint32_t)(r * row_bytes), p.wg + (size_t)(c + grid * r) * H,
                    (uint32_t)row_bytes, router_bar);
      }
      if (!mbar_wait_bounded(router_bar, 0, abort_flag, kWaitLimitNs)) fail();
    }
    int wpr = kWarps;
    while (wpr > 1 && wpr * nrows > kWarps) wpr >>= 1;
    const int rows_pp = kWarps / wpr;
    const int sub = warp % wpr;
    for (int r0 = 0; r0 < nrows; r0 += rows_pp) {
      const int r = r0 + warp / wpr;
      const int g = c + grid * r;
      float acc[kMaxT];
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) acc[t] = 0.f;
      if (r < nrows) {
#pragma unroll 2
        for (int h = (sub * 32 + lane) * 8; h < H; h += wpr * 256) {
          float4 a, b;
          if (bulk) {
            const float4* wp = reinterpret_cast<const float4*>(wrows + (size_t)r * H + h);
            a = wp[0];
            b = wp[1];
          } else {
            const float4* wp = reinterpret_cast<const float4*>(p.wg + (size_t)g * H + h);
            a = __ldg(wp);
            b = __ldg(wp + 1);
          }
          const float wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
          for (int t = 0; t < kMaxT; ++t) {
            if (t < T) {
              const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)t * H + h));
              float xf[8];
              bf16x8_to_f32(v, xf);
#pragma unroll
              for (int i = 0; i < 8; ++i) acc[t] = fmaf(wv[i], xf[i], acc[t]);
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) {
        float v = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[warp][t] = v;
      }
      bar_workers();
      // one thread per (row, token) adds the row's warps in order
      if (sub == 0 && lane < T && r < nrows) {
        float sum = 0.f;
        for (int q = 0; q < wpr; ++q) sum += red[warp + q][lane];
        p.logits[(size_t)lane * G + g] = sum + (p.gate_bias ? p.gate_bias[g] : 0.f);
      }
      bar_workers();
    }
    bar_workers();
  }
  if (tid == 0) {
    __threadfence();
    atomicAdd(router_ctr, 1u);
    if (!wait_geq(router_ctr, (uint32_t)grid, abort_flag)) fail();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // ---------------- 2. every CTA routes every token and plans
  {
    if (!*abort_flag && P > 1) {
      const int t = warp / P, q = warp % P;
      const int ep = moe_cdiv(E, P);
      const int base = q * ep, n = min(ep, E - base);
      if (worker && t < T && n > 0)
        route_part(p.logits + (size_t)t * G, p, base, n, min(K, n), sids_s[warp], wsc_s[warp]);
      __syncthreads();
      if (warp < T) {
        // token `warp`: its partitions' picks are in sids_s[warp * P + q]
        const int kp = min(K, ep), kp_last = min(K, E - (P - 1) * ep);
        route_merge(p.logits + (size_t)warp * G, p, sids_s[warp * P], P, kp, kp_last,
                    ids_s + warp * K, w_s + warp * K);
      }
    } else if (!*abort_flag && worker) {
      for (int t = warp; t < T; t += kWarps) {
        const float* row = p.logits + (size_t)t * G;
        route_token(p.route_kind, row, p, ids_s + t * K, w_s + t * K, sids_s[warp]);
      }
    }
    if (!*abort_flag && worker && p.has_shared && lane == 0)
      for (int t = warp; t < T; t += kWarps) gsh_s[t] = sigmoid_key(__ldcg(p.logits + (size_t)t * G + E));
  }
  __syncthreads();
  // plan: mask_s[e] = the tokens that picked expert e.  Every token picks an
  // expert at most once, so the stable counting sort of the flat replica
  // index t*K + k puts token t's replica of e at row offsets[e] + (tokens
  // before t in mask_s[e]); the slots are the experts with a non-empty mask
  if (worker)
    for (int e = tid; e < E; e += kThreads) mask_s[e] = 0;
  __syncthreads();
  if (!*abort_flag && worker)
    for (int f = tid; f < R; f += kThreads) atomicOr(&mask_s[ids_s[f]], 1 << (f / K));
  __syncthreads();
  {
    // two-level scan of the per-expert counts (warp w owns a run of experts;
    // the warm-up warp owns none)
    const int per_w = (E + kWarps - 1) / kWarps, per_l = (per_w + 31) / 32;
    const int wend = worker ? min(E, warp * per_w + per_w) : 0;
    const int e0 = min(wend, warp * per_w + lane * per_l), e1 = min(wend, e0 + per_l);
    int sum = 0, nz = 0;
    for (int e = e0; e < e1; ++e) {
      const int m = __popc(mask_s[e]);
      sum += m;
      nz += m > 0;
    }
    int isum = sum, inz = nz;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, isum, o);
      const int b = __shfl_up_sync(0xffffffffu, inz, o);
      if (lane >= o) {
        isum += a;
        inz += b;
      }
    }
    if (lane == 31 && worker) {
      wtot_s[warp][0] = isum;
      wtot_s[warp][1] = inz;
    }
    __syncthreads();
    int run = isum - sum, slot = inz - nz;
    for (int q = 0; q < warp && worker; ++q) {
      run += wtot_s[q][0];
      slot += wtot_s[q][1];
    }
    for (int e = e0; e < e1; ++e) {
      const int mask = mask_s[e], m = __popc(mask);
      off_s[e] = run;
      if (m > 0) slot_s[slot++] = make_int4(e, run, m, mask);
      run += m;
    }
    if (warp == kWarps - 1 && lane == 31) {
      int tr = 0, ts = 0;
      for (int q = 0; q < kWarps; ++q) {
        tr += wtot_s[q][0];
        ts += wtot_s[q][1];
      }
      off_s[E] = tr;
      n_slots_s = ts;
      if (p.has_shared) slot_s[ts] = make_int4(-1, 0, T, (1 << T) - 1);
    }
  }
  __syncthreads();
  if (!*abort_flag && worker)
    for (int f = tid; f < R; f += kThreads) {
      const int e = ids_s[f], t = f / K;
      const int row = off_s[e] + __popc(mask_s[e] & ((1 << t) - 1));
      r2f_s[row] = f;
      f2r_s[f] = row;
    }
  __syncthreads();
  if (c == 0 && !*abort_flag && worker) {
    // the routing results for the caller
    for (int f = tid; f < R; f += kThreads) {
      p.ids[f] = ids_s[f];
      p.weights[f] = w_s[f];
      p.row_to_flat[f] = r2f_s[f];
      p.flat_to_row[f] = f2r_s[f];
    }
    for (int e = tid; e <= E; e += kThreads) p.offsets[e] = off_s[e];
    for (int e = tid; e < E; e += kThreads)
      if (p.block_variant)
        p.block_variant[e] = moe_variant_of(off_s[e + 1] - off_s[e], R, E, p.m_skinny,
                                            p.dispatch, p.wdtype);
    if (p.has_shared && tid < T) p.shared_gate[tid] = gsh_s[tid];
  }

  // ---------------- 3-6. the expert GEMMs and the combine
  Sched s;
  s.n_r = n_slots_s;
  s.nb1r = moe_cdiv(p.I, kBM);
  s.nb1s = p.has_shared ? moe_cdiv(p.Is, kBM) : 0;
  s.nk1 = moe_cdiv(H, kBK);
  s.nb2 = moe_cdiv(H, kBM);
  s.nk2r = moe_cdiv(p.I, kBK);
  s.nk2s = p.has_shared ? moe_cdiv(p.Is, kBK) : 1;
  s.P1 = (long long)s.n_r * s.nb1r + s.nb1s;
  s.S1 = s.P1 * s.nk1;
  s.S2r = (long long)s.n_r * s.nb2 * s.nk2r;
  s.P2 = (long long)(s.n_r + p.has_shared) * s.nb2;
  s.S2 = s.S2r + (p.has_shared ? (long long)s.nb2 * s.nk2s : 0);
  s.chunk1 = s.S1 > 0 ? (s.S1 + grid - 1) / grid : 1;
  s.chunk2 = s.S2 > 0 ? (s.S2 + grid - 1) / grid : 1;
  const long long lo1 = s.lo(s.S1, s.chunk1, c), hi1 = s.lo(s.S1, s.chunk1, c + 1);
  const long long lo2 = s.lo(s.S2, s.chunk2, c), hi2 = s.lo(s.S2, s.chunk2, c + 1);
  const int Kt = K + p.has_shared;  // contributions per token and feature block

  if (*abort_flag) {
    // routing never completed: no GEMM work
  } else if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0, pend_tx = 0;
      bool ok = true;
      auto take = [&]() -> bool {
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, kWaitLimitNs)) return false;
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        return true;
      };
      auto advance = [&]() {
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      };
      // the router read the ring through the generic proxy
      fence_proxy_async_smem();
      // G1: weights and x rows together
      for (long long st = lo1; st < hi1 && ok; ++st) {
        const int pr = s.pair_of(1, st);
        const int k = (int)(st - s.first_step(1, pr));
        const int j = s.slot1(pr), nb = s.blk1(pr);
        const bool sh = j == s.n_r;
        if (!take()) { fail(); ok = false; break; }
        const uint32_t d = sbase + stage * kStageBytes;
        mbar_arrive_expect_tx(full_bar(stage), 2 * kWBytes + kBBytes);
        const int e = sh ? 0 : slot_s[j].x;
        tma_load_3d(d, sh ? &maps.sw1 : &maps.w1, full_bar(stage), k * kBK, nb * kBM, e);
        tma_load_3d(d + kWBytes, sh ? &maps.sw3 : &maps.w3, full_bar(stage), k * kBK, nb * kBM, e);
        tma_load_3d(d + 2 * kWBytes, &maps.x, full_bar(stage), k * kBK, 0, 0);
        advance();
      }
      // G2: stages of up to two K steps of one pair.  Their W2 tiles do not
      // depend on G1 and are issued first; the hact tiles follow once every
      // G1 pair is stored (one bounded wait, taken when the ring holds
      // nothing but such stages, or at the end).
      struct Pend { int stage, j, k, n; };
      Pend pend[kStages];
      int npend = 0;
      bool g1_ready = false;
      auto issue_acts = [&](const Pend& g) {
        const uint32_t d = sbase + g.stage * kStageBytes + 2 * kWBytes;
        for (int u = 0; u < g.n; ++u) {
          if (g.j == s.n_r)
            tma_load_3d(d + u * kBBytes, &maps.hs, full_bar(g.stage), (g.k + u) * kBK, 0, 0);
          else
            tma_load_3d(d + u * kBBytes, &maps.h, full_bar(g.stage), (g.k + u) * kBK,
                        slot_s[g.j].y, 0);
        }
        pend_tx &= ~(1u << g.stage);
      };
      auto wait_g1 = [&]() -> bool {
        if (!wait_geq(g1_done, 4u * (uint32_t)s.P1, abort_flag)) return false;
        fence_proxy_async_global();
        g1_ready = true;
        for (int i = 0; i < npend; ++i) issue_acts(pend[i]);
        npend = 0;
        return true;
      };
      for (long long cur = lo2; cur < hi2 && ok;) {
        const Piece pc = piece_at(s, 2, cur, hi2, lo2);
        cur = s.first_step(2, pc.pair) + pc.k1;
        const int j = pc.pair / s.nb2, nb = pc.pair % s.nb2;
        const bool sh = j == s.n_r;
        for (int k = pc.k0; k < pc.k1 && ok; k += 2) {
          const int n = min(2, pc.k1 - k);
          if (!g1_ready && npend == kStages && !wait_g1()) { fail(); ok = false; break; }
          if (!take()) { fail(); ok = false; break; }
          mbar_arrive_expect_tx(full_bar(stage), n * (kWBytes + kBBytes));
          pend_tx |= 1u << stage;
          for (int u = 0; u < n; ++u)
            tma_load_3d(sbase + stage * kStageBytes + u * kWBytes, sh ? &maps.sw2 : &maps.w2,
                        full_bar(stage), (k + u) * kBK, nb * kBM, sh ? 0 : slot_s[j].x);
          const Pend g = {stage, j, k, n};
          if (g1_ready) issue_acts(g);
          else pend[npend++] = g;
          advance();
        }
      }
      if (ok && !g1_ready && npend > 0 && !wait_g1()) { fail(); ok = false; }
      // stages whose hact tile will never come: take those bytes back so the
      // drain below sees every issued copy land
      for (int i = 0; i < npend; ++i)
        if (pend_tx & (1u << pend[i].stage))
          mbar_complete_tx(full_bar(pend[i].stage), pend[i].n * kBBytes);
      for (int st = 0; st < kStages; ++st)
        if (armed & (1u << st))
          if (!mbar_wait_bounded(full_bar(st), (armed_par >> st) & 1u, nullptr, kWaitLimitNs)) fail();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN);
      int stage = 0;
      uint32_t phase = 0, npc = 0;
      bool ok = true, issued = false;
      for (int ph = 1; ph <= 2 && ok; ++ph) {
        const long long lo = ph == 1 ? lo1 : lo2, hi = ph == 1 ? hi1 : hi2;
        for (long long cur = lo; cur < hi && ok; ++npc) {
          const Piece pc = piece_at(s, ph, cur, hi, lo);
          cur = s.first_step(ph, pc.pair) + pc.k1;
          const int a = (int)(npc % kAcc);
          if (!mbar_wait_bounded(acc_empty(a), ((npc / kAcc) & 1u) ^ 1u, abort_flag, kWaitLimitNs)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dacc = tmem + a * kAccCols;
          const int per = ph == 1 ? 1 : 2;  // K steps per stage
          for (int k = pc.k0; k < pc.k1; k += per) {
            if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, kWaitLimitNs)) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st = sbase + stage * kStageBytes;
            const int n = min(per, pc.k1 - k);
            for (int u = 0; u < n; ++u) {
              const uint32_t wa = ph == 1 ? st : st + u * kWBytes;
              const uint32_t bt = st + 2 * kWBytes + u * kBBytes;
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk) {
                const uint32_t accum = (k + u > pc.k0 || kk > 0) ? 1u : 0u;
                const uint64_t bdesc = sdesc_k128_sw128(bt + kk * 32);
                tc_mma_f16(dacc, sdesc_k128_sw128(wa + kk * 32), bdesc, kIdesc, accum);
                if (ph == 1)
                  tc_mma_f16(dacc + kBN, sdesc_k128_sw128(st + kWBytes + kk * 32), bdesc, kIdesc,
                             accum);
              }
            }
            issued = true;
            tc_commit(empty_bar(stage));
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          tc_commit(acc_full(a));
        }
      }
      if (issued) {
        tc_commit(drain_bar);
        if (!mbar_wait_bounded(drain_bar, 0, nullptr, kWaitLimitNs)) fail();
      }
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ---------------- epilogue: TMEM lane quarter q = 32 output features
    const int q = warp & 3;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t npc = 0;
    bool ok = true;
    for (int ph = 1; ph <= 2 && ok; ++ph) {
      const long long lo = ph == 1 ? lo1 : lo2, hi = ph == 1 ? hi1 : hi2;
      const long long chunk = ph == 1 ? s.chunk1 : s.chunk2;
      float* part_ph = p.part + (size_t)(ph - 1) * kDecodeMaxGrid * 2 * 4 * kPieceFloats;
      for (long long cur = lo; cur < hi; ++npc) {
        const Piece pc = piece_at(s, ph, cur, hi, lo);
        cur = s.first_step(ph, pc.pair) + pc.k1;
        const int a = (int)(npc % kAcc);
        // A cut pair is summed by its first CTA (c0), in CTA order.  The
        // other pieces are the first pieces of their CTAs, done early: c0
        // waits for them and reads their partial sums before its own
        // accumulator is ready, so only its own finish remains on the path.
        const long long f = s.first_step(ph, pc.pair);
        const int c0 = s.cta_of(chunk, f), c1 = s.cta_of(chunk, f + s.nk_of(ph, pc.pair) - 1);
        uint32_t* pflag = (ph == 1 ? cnt1 : cnt2) + (size_t)pc.pair * 4 + q;
        float og[16], ou[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) { og[i] = 0.f; ou[i] = 0.f; }
        if (!pc.full && c == c0) {
          if (lane == 0 && !wait_geq(pflag, (uint32_t)(c1 - c0), abort_flag)) fail();
          __syncwarp();  // lane 0 acquired the other pieces' stores
          for (int cc = c0 + 1; cc <= c1; ++cc) {
            const float* pp = part_ph + ((size_t)(cc * 2) * 4 + q) * kPieceFloats;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              og[i] += __ldcg(pp + i * 32 + lane);
              if (ph == 1) ou[i] += __ldcg(pp + 512 + i * 32 + lane);
            }
          }
          if (lane == 0) *pflag = 0u;  // ready for the next call
        }
        if (!mbar_wait_bounded(acc_full(a), (npc / kAcc) & 1u, abort_flag, kWaitLimitNs)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t gr[16], ur[16];
        tc_ld_32x32b_x16(t_lane + a * kAccCols, gr);
        if (ph == 1) tc_ld_32x32b_x16(t_lane + a * kAccCols + kBN, ur);
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(acc_empty(a));
        float g[16], u[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          g[i] = __uint_as_float(gr[i]);
          u[i] = ph == 1 ? __uint_as_float(ur[i]) : 0.f;
        }
        if (!pc.full && c != c0) {
          // a later piece of a cut pair (the first piece of this CTA): store
          // the partial sums for c0 and count them
          float* mine = part_ph + ((size_t)(c * 2) * 4 + q) * kPieceFloats;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            mine[i * 32 + lane] = g[i];
            if (ph == 1) mine[512 + i * 32 + lane] = u[i];
          }
          __syncwarp();
          if (lane == 0) red_add_release(pflag, 1u);
          continue;
        }
        if (!pc.full) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            g[i] += og[i];
            u[i] += ou[i];
          }
        }
        if (ph == 1) {
          // hact columns of this pair: the slot's tokens (MMA column = token)
          const int j = s.slot1(pc.pair), nb = s.blk1(pc.pair);
          const int4 sl = slot_s[j];
          const bool sh = j == s.n_r;
          const int I_j = sh ? p.Is : p.I;
          const int n = nb * kBM + q * 32 + lane;
          __nv_bfloat16* dst = sh ? p.sh_hact : p.hact;
          if (n < I_j) {
#pragma unroll
            for (int t = 0; t < kBN; ++t) {
              if ((sl.w >> t) & 1) {
                const int i = __popc(sl.w & ((1 << t) - 1));
                dst[(size_t)(sl.y + i) * I_j + n] = __float2bfloat16_rn(silu_f(g[t]) * u[t]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) red_add_release(g1_done, 1u);
        } else {
          // y columns of this pair: MMA column i = the slot's i-th row
          const int j = pc.pair / s.nb2, nb = pc.pair % s.nb2;
          const int4 sl = slot_s[j];
          const bool sh = j == s.n_r;
          const int n = nb * kBM + q * 32 + lane;
          __nv_bfloat16* dst = sh ? p.sh_y : p.y;
          if (n < H) {
#pragma unroll
            for (int i = 0; i < kBN; ++i)
              if (i < sl.z) dst[(size_t)(sl.y + i) * H + n] = __float2bfloat16_rn(g[i]);
          }
          __syncwarp();
          // count this block for each of the slot's tokens (lane i for the
          // slot's i-th row); the block that completes a token's Kt
          // contributions combines them
          bool due = false;
          int tok = 0;
          if (lane < sl.z) {
            tok = sh ? lane : r2f_s[sl.y + lane] / K;
            due = atom_add_acq_rel(comb + ((size_t)tok * s.nb2 + nb) * 4 + q, 1u) ==
                  (uint32_t)(Kt - 1);
          }
          uint32_t todo = __ballot_sync(0xffffffffu, due);
          __syncwarp();  // the counting lanes acquired the other blocks' y stores
          while (todo) {
            const int i = __ffs(todo) - 1;
            todo &= todo - 1u;
            const int t = __shfl_sync(0xffffffffu, tok, i);
            if (n < H) {
              float yv[32];
#pragma unroll
              for (int k = 0; k < 32; ++k)
                yv[k] = k < K ? __bfloat162float(__ldcg(p.y + (size_t)f2r_s[t * K + k] * H + n))
                              : 0.f;
              float acc = 0.f;
#pragma unroll
              for (int k = 0; k < 32; ++k)
                if (k < K) acc = fmaf(w_s[t * K + k], yv[k], acc);
              if (p.has_shared)
                acc = fmaf(gsh_s[t], __bfloat162float(__ldcg(p.sh_y + (size_t)t * H + n)), acc);
              p.out[(size_t)t * H + n] = __float2bfloat16_rn(acc);
            }
            if (lane == i) comb[((size_t)t * s.nb2 + nb) * 4 + q] = 0u;  // ready for the next call
          }
        }
      }
    }
  }

  // ---------------- the last CTA out clears the call's counters
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0) {
    __threadfence();
    last_s = atomicAdd(exit_ctr, 1u) == (uint32_t)grid - 1;
  }
  __syncthreads();
  if (last_s) {
    // every other CTA has counted itself out, after all of its waits
    __threadfence();
    if (p.dev_status && *reinterpret_cast<volatile int32_t*>(p.dev_status) != 0) {
      // a wait gave up somewhere: pieces may have been left uncounted
      const size_t n = 4 * ((size_t)p.P1max + p.P2max) + 4 * (size_t)kMaxT * moe_cdiv(H, kBM);
      for (size_t i = tid; i < n && worker; i += kThreads) cnt1[i] = 0u;
    }
    if (tid == 0) {
      *router_ctr = 0u;
      *g1_done = 0u;
      *exit_ctr = 0u;
    }
  }
}

// route_kind for E and K (the list shapes the fused routing launches use)
int route_kind_of(int E, int K, int G, bool logits_aligned) {
  if (E <= 128) {
    const int npl = moe_cdiv(E, 32);
    if (npl <= 1) return 0;
    if (npl <= 2) return 1;
    return K <= 2 ? 2 : 3;
  }
  const bool vec = E % 4 == 0 && G % 4 == 0 && logits_aligned;
  const int npl = vec ? 4 * moe_cdiv(E, 128) : moe_cdiv(E, 32);
  const int ni = npl <= 8 ? 0 : npl <= 16 ? 1 : npl <= 28 ? 2 : 3;
  return (vec ? 12 : 4) + 2 * ni + (K <= 8 ? 0 : 1);
}

// one CTA per SM of the current device
int decode_grid() {
  static std::atomic<int> n[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int v = n[dev].load(std::memory_order_relaxed);
  if (!v) {
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

}  // namespace

// ---------------------------------------------------------------- host side
size_t decode_layer_sync_words(int T_max, int E, int K, int H, int I, int Is, int has_shared) {
  const int t = T_max < kMaxT ? T_max : kMaxT;
  const int slots = (t * K < E ? t * K : E) + (has_shared ? 1 : 0);
  const int nb1 = moe_cdiv(I > Is ? I : Is, kBM);
  const size_t P1 = (size_t)slots * nb1, P2 = (size_t)slots * moe_cdiv(H, kBM);
  return 64 + 4 * P1 + 4 * P2 + 4 * (size_t)kMaxT * moe_cdiv(H, kBM);
}

size_t decode_layer_part_bytes() {
  return 2 * (size_t)kDecodeMaxGrid * 2 * 4 * kPieceFloats * sizeof(float);
}

bool decode_layer_supported(int T, int E, int K, int H, int I, int Is, int has_shared, int wdtype,
                            int dispatch, int m_skinny) {
  if (T < 1 || T > kMaxT || wdtype != MOE_W_BF16) return false;
  if (dispatch != MOE_DISPATCH_PER_BLOCK && dispatch != MOE_DISPATCH_ONE_LAUNCH) return false;
  if (m_skinny < T || K > 32 || E > kMaxE) return false;
  if (H % 16 != 0 || I % 16 != 0 || (has_shared && Is % 16 != 0)) return false;
  const int g = decode_grid();
  return g > 0 && g <= kDecodeMaxGrid;
}

cudaError_t launch_decode_layer(const DecodeLayerArgs& a, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = moe_raise_smem(decode_layer_kernel, kDynSmem, smem_set);
  if (e != cudaSuccess) return e;
  const int grid = decode_grid();
  if (grid <= 0 || grid > kDecodeMaxGrid) return cudaErrorInvalidConfiguration;
  Params p;
  p.x = static_cast<const __nv_bfloat16*>(a.x);
  p.wg = a.wg;
  p.gate_bias = a.gate_bias;
  p.sel_bias = a.sel_bias;
  p.T = a.T; p.H = a.H; p.G = a.G; p.E = a.E; p.K = a.K; p.I = a.I; p.Is = a.Is;
  p.mode = a.mode; p.has_shared = a.has_shared; p.scale = a.scale;
  p.logits = a.logits; p.ids = a.ids; p.weights = a.weights; p.shared_gate = a.shared_gate;
  p.offsets = a.offsets; p.row_to_flat = a.row_to_flat; p.flat_to_row = a.flat_to_row;
  p.block_variant = a.block_variant;
  p.hact = static_cast<__nv_bfloat16*>(a.hact);
  p.y = static_cast<__nv_bfloat16*>(a.y);
  p.sh_hact = static_cast<__nv_bfloat16*>(a.sh_hact);
  p.sh_y = static_cast<__nv_bfloat16*>(a.sh_y);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.part = a.part;
  p.sync = a.sync;
  const int t = a.T_max < kMaxT ? a.T_max : kMaxT;
  const int slots = (t * a.K < a.E ? t * a.K : a.E) + (a.has_shared ? 1 : 0);
  p.P1max = slots * moe_cdiv(a.I > a.Is ? a.I : a.Is, kBM);
  p.P2max = slots * moe_cdiv(a.H, kBM);
  p.dev_status = a.dev_status;
  p.m_skinny = a.m_skinny < 0 ? MOE_DEFAULT_M_SKINNY : a.m_skinny;
  p.dispatch = a.dispatch;
  p.wdtype = a.wdtype;
  p.route_kind = route_kind_of(a.E, a.K, a.G, (reinterpret_cast<uintptr_t>(a.logits) & 15) == 0);

  Maps m;
  memset(&m, 0, sizeof(m));
  const int R = a.T * a.K;
  bool ok = moe_tmap::bf16_map_3d(&m.w1, a.w1, a.H, a.I, a.E, kBK, kBM) &&
            moe_tmap::bf16_map_3d(&m.w3, a.w3, a.H, a.I, a.E, kBK, kBM) &&
            moe_tmap::bf16_map_3d(&m.w2, a.w2, a.I, a.H, a.E, kBK, kBM) &&
            moe_tmap::bf16_map_3d(&m.x, a.x, a.H, a.T, 1, kBK, kBN) &&
            moe_tmap::bf16_map_3d(&m.h, a.hact, a.I, R, 1, kBK, kBN);
  if (ok && a.has_shared)
    ok = moe_tmap::bf16_map_3d(&m.sw1, a.sw1, a.H, a.Is, 1, kBK, kBM) &&
         moe_tmap::bf16_map_3d(&m.sw3, a.sw3, a.H, a.Is, 1, kBK, kBM) &&
         moe_tmap::bf16_map_3d(&m.sw2, a.sw2, a.Is, a.H, 1, kBK, kBM) &&
         moe_tmap::bf16_map_3d(&m.hs, a.sh_hact, a.Is, a.T, 1, kBK, kBN);
  if (!ok) return cudaErrorInvalidValue;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kBlock);
  cfg.dynamicSmemBytes = kDynSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: CTAs wait on each other
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel, p, m);
}
