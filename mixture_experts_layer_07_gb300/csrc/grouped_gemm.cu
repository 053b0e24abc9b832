// G1 + G2: grouped SwiGLU expert GEMM over expert-contiguous row blocks.
//
//   hact[r] = bf16( silu(xp[r] . W1[e]^T) * (xp[r] . W3[e]^T) )     (G1, N = I, K = H)
//   y[r]    = bf16( hact[r] . W2[e]^T )                             (G2, N = H, K = I)
//
// Kernel choice per expert block, on the device.  "vLLM CPU MoE: dynamic GEMM
// dispatch beyond a fixed threshold" (vllm PR #50949), "2. moe_fp8.cpp":
// the variant used to be fixed for all experts from the global average
// avg_M = max(1, M*topk/E); it is now chosen inside the per-expert loop from
// that block's own m_size = offsets[mb+1] - offsets[mb], and a block with
// m_size == 0 returns at once; "1. gemm.h": the high-throughput kernel is
// taken above a small-M threshold.  Here a one-CTA plan kernel reads the
// offsets on the device (the host never learns m_size, so nothing syncs),
// applies that predicate per block and writes two work lists:
//   skinny -- blocks with m_size <= m_skinny, 16-row token tiles
//   tile   -- larger blocks, 128-row token tiles
//   wide   -- FP8 weights only: blocks of more than 128 rows, 256-row token
//             tiles, so each dequantised weight tile serves twice the tokens
// All lists run on the same tensor-core kernel template, instantiated for the
// three token-tile widths, so small blocks do not pay for a wide tile.
//
// Tensor-core kernel (sm_100 family: tcgen05 + TMEM + TMA), "swap-AB" form:
// the MMA's M side is 128 rows of the expert weight (output features), its N
// side is the token tile, so even a one-token block fills the 128-row MMA and
// the accumulator's TMEM lane is the output feature -- the epilogue's thread
// i owns feature i and walks the tokens, and the 32 threads of a warp store
// 32 consecutive features of one token row.
//   warp 0     TMA producer: weight tiles [128 x 64] (W1 and W3 for G1) and
//              the activation tile [BN x 64], 128-byte swizzled, into a ring
//              of stages guarded by full/empty mbarriers
//   warp 1     allocates TMEM, one thread issues tcgen05.mma (K = 16 per
//              instruction, 4 per stage) and commits each stage back to the
//              producer and the finished accumulator to the epilogue
//   warps 2-9  epilogue: tcgen05.ld the fp32 accumulators (TMEM lanes are
//              split by warp % 4, token columns between the two warps of a
//              lane quarter), SwiGLU, bf16 store masked to the block
// Persistent: one CTA per SM walks (item, 128-feature block) work units.
// Every mbarrier wait is bounded; a wait that runs out sets
// MOE_DEV_WAIT_TIMEOUT, the CTA drains its own in-flight copies and MMAs
// (again bounded), frees its TMEM and returns.
//
// A CUDA-core kernel (MOE_DISPATCH_SIMT) runs the same work list with plain
// FMA, bf16 or e4m3 weights; it is the cross-check of the tensor-core path.
#include <cuda.h>
#include <cuda_fp8.h>
#include <string.h>

#include "common.cuh"
#include "mxfp4.cuh"
#include "internal.h"
#include "plan.cuh"
#include "sm100_ptx.cuh"

namespace {

using namespace moe_mx;

using namespace moe_ptx;
using namespace moe_plan;

constexpr int kBM = 128;  // weight rows per MMA (output features)
constexpr int kBK = 64;   // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------- plan
__global__ void __launch_bounds__(1024)
gemm_plan_kernel(const int32_t* __restrict__ offsets, int E_blocks, int R, int m_skinny,
                 int dispatch, int wdtype, int32_t* __restrict__ counts, PlanOut out,
                 int32_t* __restrict__ block_variant) {
  pdl_wait();
  pdl_trigger();
  plan_experts<1024>(offsets, E_blocks, R, m_skinny, dispatch, wdtype, counts, out, block_variant);
}

// ---------------------------------------------------------------- tensor cores
// WQ: the expert weights' storage (a MOE_W_* code).  0: bf16, read by the MMA
// as TMA lands it.  1 (FP8): e4m3 with one fp32 scale per 128 x 128 block.
// TMA brings the e4m3 tile [128 rows x 64 K] in unswizzled; a converter
// warpgroup turns it into bf16 (e4m3 -> f16 is exact, times the block's scale,
// rounded once to bf16) written straight into the 128-byte-swizzled K-major
// layout the MMA reads, in a small ring of its own.  The 128-row weight tile
// is exactly one scale row block and a 64-wide K stage lies inside one scale
// column block, so each converted tile needs a single scale.  2 (MXFP4): the
// tile is [128 rows x 32 bytes] of e2m1 pairs and each 32 elements of a row
// carry their own power-of-two scale; the converters turn every element into
// bf16 exactly (an e2m1 value times a power of two has at most two significant
// bits), so the MMA sees the stored weights themselves.
template <int BN, bool SWIGLU, int WQ>
struct TcCfg {
  static constexpr int kMaxScaleCols = 64;  // FP8: K up to 8192 (64 scale columns of 128)
  static constexpr int kNA = SWIGLU ? 2 : 1;
  static constexpr int kABytes = kBM * kBK * 2;             // bf16 weight tile
  static constexpr int kQBytes = WQ == 2 ? kBM * kBK / 2 : kBM * kBK;  // e4m3 / e2m1-pair tile
  static constexpr int kBBytes = BN * kBK * 2;              // bf16 activation tile
  static constexpr int kStageBytes = kNA * (WQ ? kQBytes : kABytes) + kBBytes;
  static constexpr int kConvStages = WQ ? 2 : 0;
  static constexpr int kConvBytes = kNA * kABytes;
  static constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, splitting the token columns
  static constexpr int kEpiBytes = kEpiWarps * 16 * 32 * 2;  // per warp: 16 tokens x 32 features
  static constexpr int kStagesRaw =
      (216 * 1024 - kEpiBytes - kConvStages * kConvBytes) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static constexpr int kAccCols = kNA * BN;                  // columns of one accumulator set
  static constexpr int kAccStages = 2 * kAccCols <= 512 ? 2 : 1;
  static constexpr int kTmemNeed = kAccStages * kAccCols;
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64
                                 : kTmemNeed <= 128 ? 128 : kTmemNeed <= 256 ? 256 : 512;
  static constexpr int kScaleBufs = WQ ? 3 : 0;  // per-unit scale rows, reused every 3 units
  // work-unit queue: warp 0 takes units (its first is blockIdx.x, the rest
  // from the launch's atomic counter) and hands each to the other roles
  static constexpr int kQ = 8;
  static constexpr int kQConsumers = 1 + kEpiWarps + (WQ ? 8 : 0);  // MMA thread + warps
  static constexpr int kNumBars =
      2 * kStages + 2 * kAccStages + 1 + 2 * kConvStages + kScaleBufs + 2 * kQ;
  static constexpr int kBarBytes =
      kNumBars * 8 + 16 + kScaleBufs * 2 * kMaxScaleCols * 4 + kQ * 4 + BN * 4;
  static constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes +
                                       (size_t)kConvStages * kConvBytes + kEpiBytes + kBarBytes;
  static constexpr int kConvThreads = WQ ? 256 : 0;  // eight converter warps
  static constexpr int kConvWarp0 = 2 + kEpiWarps;        // first converter warp
  // G1 (SwiGLU) only: one more warp that, in gather mode, copies the tile's
  // rows straight from x (small batches: a few rows per tile)
  static constexpr int kGatherWarp = kConvWarp0 + kConvThreads / 32;
  static constexpr int kThreads = 64 + 32 * kEpiWarps + kConvThreads + (SWIGLU ? 32 : 0);
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, BN);
  static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
  static_assert(kTmemNeed <= 512, "TMEM holds 512 columns");
  static_assert(kStages >= 2, "pipeline needs two stages");
  static_assert(kSmemBytes <= 232448, "227 KB of shared memory per CTA");
};

MOE_DEVICE float silu_f(float g) { return g / (1.f + __expf(-g)); }

// generic-proxy global writes (made visible to this thread) -> later TMA reads
MOE_DEVICE void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// wait until *p >= target (acquire, GPU scope); bounded like the mbarrier waits
MOE_DEVICE bool wait_count_geq(const int32_t* p, int target, const volatile int* abort,
                               uint64_t limit_ns) {
  auto ld = [&]() {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
  };
  if (ld() >= target) return true;
  const uint64_t t0 = moe_ptx::globaltimer_ns();
  for (uint32_t i = 1; i < (1u << 30); ++i) {
    __nanosleep(64);
    if (ld() >= target) return true;
    if ((i & 15) == 0) {
      if (abort && *abort) return false;
      if (moe_ptx::globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
  return false;
}

// one thread waits (bounded) until *counter >= target and reports
// MOE_DEV_WAIT_TIMEOUT if the wait runs out: the wait the fused G1+G2 launch
// uses for its cross-CTA dependency, on its own
__global__ void __launch_bounds__(32)
bounded_wait_kernel(const int32_t* counter, int target, uint64_t limit_ns, int32_t* dev_status) {
  if (threadIdx.x == 0 && !wait_count_geq(counter, target, nullptr, limit_ns))
    moe_set_status(dev_status, MOE_DEV_WAIT_TIMEOUT);
}

MOE_DEVICE void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// two e4m3 codes (low byte first) -> two bf16 of code * scale, packed low first
MOE_DEVICE uint32_t e4m3x2_to_bf16x2(uint32_t two, float sc) {
  const __half2_raw hr =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  return pack_bf16x2(f.x * sc, f.y * sc);
}


// FUSED (G1 layout, SWIGLU = true): one persistent launch runs the list's G1
// units and then its G2 units (W2 = tm_w2, activations hact = tm_h, output
// y = out2, N2 x K2).  A G2 unit of token tile i starts loading only after
// all G1 units of tile i have stored their hact rows: each G1 epilogue warp
// fences its stores and bumps done[i]; the G2 producer waits (bounded) for
// nblk x 8 and fences the generic-proxy writes for its TMA reads.  So the
// CTAs that finish G1 early start G2 work instead of idling, and the launch
// boundary between the two disappears.
// The kernel body for one work list, run by CTAs cta = 0..ncta-1 of a group
// (the whole grid, or one of the two groups of the two-list launch below).
template <int BN, bool SWIGLU, int WQ, bool FUSED>
MOE_DEVICE void gemm_tc_body(const CUtensorMap& tm_wa, const CUtensorMap& tm_wb,
                             const CUtensorMap& tm_act, const float* __restrict__ sa,
                             const float* __restrict__ sb, int32_t* __restrict__ counts, int list,
                             const int4* __restrict__ items, int N, int Kdim,
                             __nv_bfloat16* __restrict__ out, int ksplit, int R,
                             float* __restrict__ part, int32_t* dev_status,
                             const CUtensorMap& tm_w2, const CUtensorMap& tm_h,
                             const float* __restrict__ s2, int N2, int K2,
                             __nv_bfloat16* __restrict__ out2, int32_t* __restrict__ done,
                             const __nv_bfloat16* __restrict__ gx,
                             const int32_t* __restrict__ grows, int gk, int ksplit2,
                             float* __restrict__ part2, int32_t* __restrict__ scnt1,
                             int32_t* __restrict__ scnt2, const int cta, const int ncta) {
  using C = TcCfg<BN, SWIGLU, WQ>;
  static_assert(!FUSED || SWIGLU, "the fused launch uses the G1 layout");
  // gather mode (G1, small batches): the gather warp copies each tile's rows
  // from x -- row r of the expert-ordered layout is token grows[r] / gk -- so
  // the permuted copy of the activations is not needed
  const bool gat = SWIGLU && gx != nullptr;
  const int nblk = (N + kBM - 1) / kBM;
  const int total1 = counts[list] * nblk * ksplit;
  const int nblk2 = FUSED ? (N2 + kBM - 1) / kBM : 1;
  const int ks2 = FUSED ? ksplit2 : 1;
  const int total = FUSED ? total1 + counts[list] * nblk2 * ks2 : total1;
  if (cta >= total) return;
  const int nk = (Kdim + kBK - 1) / kBK;
  const int nk2 = FUSED ? (K2 + kBK - 1) / kBK : 0;
  // work unit w -> (item, 128-feature block nb, K slice ks); with ksplit > 1
  // each slice writes fp32 partial sums to part[ks][row][feature] instead of
  // the finished output, and the last slice to finish (counted in scnt)
  // reduces the slices in order (or, without scnt, a finalize kernel does).
  // FUSED: units total1.. are the G2 units (ksplit2 slices, partials in part2).
  const int kbs = (nk + ksplit - 1) / ksplit;
  const int kbs2 = FUSED ? (nk2 + ks2 - 1) / ks2 : 1;
  struct Unit { int4 it; int nb, kb_lo, kb_hi, ks, idx; bool g1; };
  auto unit_of = [&](int w) {
    Unit u;
    if (FUSED && w >= total1) {
      const int w2 = w - total1;
      u.idx = w2 / (nblk2 * ks2);
      u.nb = (w2 / ks2) % nblk2;
      u.ks = w2 % ks2;
      u.kb_lo = u.ks * kbs2;
      u.kb_hi = min(nk2, u.kb_lo + kbs2);
      u.g1 = false;
    } else {
      u.idx = w / (nblk * ksplit);
      u.nb = (w / ksplit) % nblk;
      u.ks = w % ksplit;
      u.kb_lo = u.ks * kbs;
      u.kb_hi = min(nk, u.kb_lo + kbs);
      u.g1 = SWIGLU;
    }
    u.it = items[u.idx];
    return u;
  };

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  uint8_t* conv = smem + (size_t)C::kStages * C::kStageBytes;
  const uint32_t cbase = smem_u32(conv);
  uint16_t* epi = reinterpret_cast<uint16_t*>(conv + (size_t)C::kConvStages * C::kConvBytes);
  uint8_t* bar_area = reinterpret_cast<uint8_t*>(epi) + C::kEpiBytes;
  const uint32_t bar0 = smem_u32(bar_area);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::kStages + s); };
  auto acc_full = [&](uint32_t a) { return bar0 + 8u * (2 * C::kStages + a); };
  auto acc_empty = [&](uint32_t a) { return bar0 + 8u * (2 * C::kStages + C::kAccStages + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C::kStages + 2 * C::kAccStages);
  auto conv_full = [&](int c) { return drain_bar + 8u * (1 + c); };
  auto conv_empty = [&](int c) { return drain_bar + 8u * (1 + C::kConvStages + c); };
  auto scale_bar = [&](int b) { return drain_bar + 8u * (1 + 2 * C::kConvStages + b); };
  auto uq_full = [&](int q) {
    return drain_bar + 8u * (1 + 2 * C::kConvStages + C::kScaleBufs + q);
  };
  auto uq_empty = [&](int q) {
    return drain_bar + 8u * (1 + 2 * C::kConvStages + C::kScaleBufs + C::kQ + q);
  };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* scale_rows = reinterpret_cast<float*>(tmem_slot + 4);  // FP8: [3][2][kMaxScaleCols]
  volatile int32_t* uq = reinterpret_cast<volatile int32_t*>(scale_rows + C::kScaleBufs * 2 * C::kMaxScaleCols);
  int32_t* tok_s = const_cast<int32_t*>(uq + C::kQ);  // gather mode: token of each tile row
  int32_t* sched = counts + kSchedBase + 2 * list + (SWIGLU ? 0 : 1);

  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    // gather mode: a stage is full after the weight bytes (expect_tx) and the
    // gather warp's arrival once its row copies have landed
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), gat ? 2 : 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < C::kAccStages; ++a) {
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), 32 * C::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    for (int c = 0; c < C::kConvStages; ++c) {
      mbar_init(conv_full(c), C::kConvThreads);
      mbar_init(conv_empty(c), 1);
    }
    for (int b = 0; b < C::kScaleBufs; ++b) mbar_init(scale_bar(b), C::kConvThreads);
    for (int q = 0; q < C::kQ; ++q) {
      mbar_init(uq_full(q), 1);
      mbar_init(uq_empty(q), C::kQConsumers + (gat ? 1 : 0));
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_wa);
    if (SWIGLU) prefetch_tmap(&tm_wb);
    if (!gat) prefetch_tmap(&tm_act);
    if (FUSED) {
      prefetch_tmap(&tm_w2);
      prefetch_tmap(&tm_h);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    moe_set_status(dev_status, MOE_DEV_WAIT_TIMEOUT);
    *abort_flag = 1;
  };
  // accumulator set and the parity of its barriers for the i-th unit of this CTA
  auto acc_set = [](uint32_t i) { return C::kAccStages == 2 ? (i & 1u) : 0u; };
  auto acc_par = [](uint32_t i) { return (C::kAccStages == 2 ? (i >> 1) : i) & 1u; };
  constexpr int kWeightBytes = WQ ? C::kQBytes : C::kABytes;
  constexpr int kWx = WQ == 2 ? kBK / 2 : kBK;  // a stage's K step in the weight map's units
  // next work unit from the queue (every consumer sees every unit, in order);
  // `arrive` frees the entry (one arrival per consuming warp or thread).
  // total (or more) ends the walk; -1 means the wait gave up.
  auto pop_unit = [&](uint32_t& q, uint32_t& qph, bool arrive) {
    int w = -1;
    if (mbar_wait_bounded(uq_full(q), qph, abort_flag, kWaitLimitNs)) w = uq[q];
    if (arrive) mbar_arrive(uq_empty(q));
    if (++q == C::kQ) { q = 0; qph ^= 1u; }
    return w;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0, q = 0, qph = 0;
      bool ok = true;
      int w = cta;  // first unit; later ones come from the launch's counter
      for (;;) {
        // hand the unit (or the end mark) to the other roles
        if (!mbar_wait_bounded(uq_empty(q), qph ^ 1u, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
        uq[q] = ok ? w : total;
        mbar_arrive(uq_full(q));
        if (++q == C::kQ) { q = 0; qph ^= 1u; }
        if (!ok || w >= total) break;
        const Unit u = unit_of(w);
        const int4 it = u.it;
        const int nb = u.nb;
        int kb0 = u.kb_lo;
        if (FUSED && !u.g1) {
          // The unit's first weight tiles do not depend on G1: start them into
          // free stages now (transaction bytes only, no arrival, so a stage
          // cannot complete early), then wait for this tile's hact rows --
          // every G1 unit of the tile stored and counted -- and add the
          // activation tiles with the arrival.
          int npre = 0;
          uint32_t pre_par = 0;
          for (int kb = u.kb_lo; kb < u.kb_hi && npre < C::kStages; ++kb, ++npre) {
            if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, kWaitLimitNs)) {
              fail();
              ok = false;
              break;
            }
            mbar_expect_tx(full_bar(stage), kWeightBytes);
            tma_load_3d(sbase + stage * C::kStageBytes, &tm_w2, full_bar(stage), kb * kWx, nb * kBM,
                        it.x);
            pre_par |= phase << npre;
            if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
          }
          if (ok && !wait_count_geq(done + u.idx, nblk * C::kEpiWarps, abort_flag, kWaitLimitNs)) {
            fail();
            ok = false;
          }
          fence_proxy_async_global();
          for (int i = 0; i < npre; ++i) {
            const int s_i = (stage + C::kStages - npre + i) % C::kStages;
            if (ok) {
              mbar_arrive_expect_tx(full_bar(s_i), C::kBBytes);
              tma_load_2d(sbase + s_i * C::kStageBytes + C::kNA * kWeightBytes, &tm_h, full_bar(s_i),
                          (u.kb_lo + i) * kBK, it.y);
            } else {
              mbar_arrive(full_bar(s_i));  // the weight bytes alone complete it: drainable
            }
            armed |= 1u << s_i;
            armed_parity = (armed_parity & ~(1u << s_i)) | (((pre_par >> i) & 1u) << s_i);
          }
          kb0 = u.kb_lo + npre;
        }
        const CUtensorMap* wmap = (FUSED && !u.g1) ? &tm_w2 : &tm_wa;
        const CUtensorMap* amap = (FUSED && !u.g1) ? &tm_h : &tm_act;
        const uint32_t stage_bytes = u.g1 ? C::kStageBytes : kWeightBytes + C::kBBytes;
        for (int kb = kb0; kb < u.kb_hi && ok; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            fail();
            ok = false;
            break;
          }
          const uint32_t st = sbase + stage * C::kStageBytes;
          mbar_arrive_expect_tx(full_bar(stage), gat && u.g1 ? C::kNA * kWeightBytes : stage_bytes);
          tma_load_3d(st, wmap, full_bar(stage), kb * kWx, nb * kBM, it.x);
          if (u.g1) tma_load_3d(st + kWeightBytes, &tm_wb, full_bar(stage), kb * kWx, nb * kBM, it.x);
          if (!(gat && u.g1))
            tma_load_2d(st + C::kNA * kWeightBytes, amap, full_bar(stage), kb * kBK, it.y);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        // the next unit: taken once this one's loads are issued, so a CTA that
        // drew short units takes more (the group's first units are its CTA ids)
        if (ok) w = ncta + atomicAdd(sched, 1);
      }
      // every copy this thread started has landed before the CTA moves on
      for (int s = 0; s < C::kStages; ++s)
        if (armed & (1u << s))
          if (!mbar_wait_bounded(full_bar(s), (armed_parity >> s) & 1u, nullptr, kWaitLimitNs)) fail();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int stage = 0, cs = 0;
      uint32_t phase = 0, cphase = 0, unit = 0, q = 0, qph = 0;
      bool ok = true, issued = false;
      for (;; ++unit) {
        const int w = pop_unit(q, qph, true);
        if (w < 0) fail();
        if (w < 0 || w >= total) break;
        const uint32_t a = acc_set(unit);
        if (!mbar_wait_bounded(acc_empty(a), acc_par(unit) ^ 1u, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + a * C::kAccCols;
        const Unit u = unit_of(w);
        for (int kb = u.kb_lo; kb < u.kb_hi; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, kWaitLimitNs) ||
              (WQ && !mbar_wait_bounded(conv_full(cs), cphase, abort_flag, kWaitLimitNs))) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + stage * C::kStageBytes;
          const uint32_t wa_s = WQ ? cbase + cs * C::kConvBytes : st;
          const uint32_t wb_s = wa_s + C::kABytes;
          const uint32_t sx = st + C::kNA * kWeightBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t acc = (kb > u.kb_lo || kk > 0) ? 1u : 0u;
            const uint64_t bdesc = sdesc_k128_sw128(sx + kk * 32);
            tc_mma_f16(d, sdesc_k128_sw128(wa_s + kk * 32), bdesc, C::kIdesc, acc);
            if (u.g1) tc_mma_f16(d + BN, sdesc_k128_sw128(wb_s + kk * 32), bdesc, C::kIdesc, acc);
          }
          issued = true;
          tc_commit(empty_bar(stage));
          if (WQ) {
            tc_commit(conv_empty(cs));
            if (++cs == C::kConvStages) { cs = 0; cphase ^= 1u; }
          }
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(acc_full(a));
      }
      if (issued) {
        // all MMAs of this thread complete before TMEM is released
        tc_commit(drain_bar);
        if (!mbar_wait_bounded(drain_bar, 0, nullptr, kWaitLimitNs)) fail();
      }
    }
  } else if (warp < C::kConvWarp0) {
    // ---------------- epilogue, warps 2..9
    // TMEM lane quarter = warp % 4 = 32 output features; the two warps of a
    // quarter take alternate 16-token chunks.  Each chunk is staged in shared
    // memory and written back as 16-byte row segments.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint16_t* stg = epi + (warp - 2) * (16 * 32);
    uint32_t unit = 0, q = 0, qph = 0;
    for (;; ++unit) {
      const int w = pop_unit(q, qph, false);
      __syncwarp();
      if (lane == 0) mbar_arrive(uq_empty((q + C::kQ - 1) % C::kQ));
      if (w < 0) fail();
      if (w < 0 || w >= total) break;
      const Unit un = unit_of(w);
      const int4 it = un.it;
      const int nb = un.nb;
      const uint32_t a = acc_set(unit);
      if (!mbar_wait_bounded(acc_full(a), acc_par(unit), abort_flag, kWaitLimitNs)) {
        fail();
        break;
      }
      tc_fence_after();
      const uint32_t tacc = t_lane + a * C::kAccCols;
      const int m = it.z;
      const bool sw = un.g1;  // SwiGLU of the gate and up accumulators
      const int Nu = sw || !FUSED ? N : N2;
      __nv_bfloat16* outu = sw || !FUSED ? out : out2;
      const int ksu = sw || !FUSED ? ksplit : ks2;  // K slices of this unit's GEMM
      float* partu = sw || !FUSED ? part : part2;
      int32_t* scntu = sw || !FUSED ? scnt1 : scnt2;
      for (int c0 = 16 * half; c0 < BN && c0 < m; c0 += 32) {
        uint32_t g[16], u[16];
        tc_ld_32x32b_x16(tacc + c0, g);
        if (sw) tc_ld_32x32b_x16(tacc + BN + c0, u);
        tc_wait_ld();
        if (ksu > 1) {
          // fp32 partials of this K slice: row-major [ks][R][Npart], Npart = N or 2N
          const int n = nb * kBM + quarter * 32 + lane;
          const int np = sw ? 2 * Nu : Nu;
          float* pr = partu + ((size_t)un.ks * R + it.y + c0) * np;
          const bool empty = un.kb_lo >= un.kb_hi;  // no K left for this slice
          if (n < Nu) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (c0 + j < m) {
                pr[(size_t)j * np + n] = empty ? 0.f : __uint_as_float(g[j]);
                if (sw) pr[(size_t)j * np + Nu + n] = empty ? 0.f : __uint_as_float(u[j]);
              }
            }
          }
          continue;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float gv = __uint_as_float(g[j]);
          const float v = sw ? silu_f(gv) * __uint_as_float(u[j]) : gv;
          stg[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        }
        __syncwarp();
        // 16 token rows x 64 bytes: lane -> (row lane/4 (+8), 16-byte chunk lane%4)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = (lane >> 2) + 8 * i;
          const int n0 = nb * kBM + quarter * 32 + (lane & 3) * 8;
          if (c0 + r < m && n0 < Nu) {
            const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 32 + (lane & 3) * 8);
            *reinterpret_cast<uint4*>(outu + (size_t)(it.y + c0 + r) * Nu + n0) = v;
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      mbar_arrive(acc_empty(a));
      if (ksu > 1 && scntu) {
        // K slices: every epilogue warp of every slice counts itself once its
        // partials are stored; the last one reduces the unit's slices in slice
        // order (deterministic) and stores the bf16 rows
        __threadfence();
        __syncwarp();
        int32_t* cnt = scntu + (size_t)un.idx * (sw || !FUSED ? nblk : nblk2) + nb;
        int old = 0;
        if (lane == 0) old = atomicAdd(cnt, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == ksu * C::kEpiWarps - 1) {
          __threadfence();
          const int np = sw ? 2 * Nu : Nu;
          const int n = nb * kBM + lane * 4;
          for (int r = 0; r < m && n < Nu; ++r) {
            float4 gs = make_float4(0.f, 0.f, 0.f, 0.f), us = gs;
            for (int q = 0; q < ksu; ++q) {
              const float* pr = partu + ((size_t)q * R + it.y + r) * np + n;
              const float4 a4 = __ldcg(reinterpret_cast<const float4*>(pr));
              gs.x += a4.x; gs.y += a4.y; gs.z += a4.z; gs.w += a4.w;
              if (sw) {
                const float4 b4 = __ldcg(reinterpret_cast<const float4*>(pr + Nu));
                us.x += b4.x; us.y += b4.y; us.z += b4.z; us.w += b4.w;
              }
            }
            if (sw) {
              gs.x = silu_f(gs.x) * us.x; gs.y = silu_f(gs.y) * us.y;
              gs.z = silu_f(gs.z) * us.z; gs.w = silu_f(gs.w) * us.w;
            }
            uint2 o;
            o.x = pack_bf16x2(gs.x, gs.y);
            o.y = pack_bf16x2(gs.z, gs.w);
            *reinterpret_cast<uint2*>(outu + (size_t)(it.y + r) * Nu + n) = o;
          }
          __syncwarp();
          if (lane == 0) *cnt = 0;  // ready for the next call
          if (FUSED && sw) {
            // the whole 128-feature block of the tile's hact rows is stored
            __threadfence();
            __syncwarp();
            if (lane == 0) atomicAdd(done + un.idx, C::kEpiWarps);
          }
        }
      } else if (FUSED && sw) {
        // this warp's share of the tile's hact rows is stored: count it
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(done + un.idx, 1);
      }
    }
  } else if (SWIGLU && warp == C::kGatherWarp) {
    if (gat) {
      // ---------------- activation rows from x (gather mode)
      // 16-byte cp.async into the 128-byte-swizzled layout the MMA reads
      // (chunk c of row r at chunk c ^ (r % 8), as a swizzled TMA box would
      // land), only the unit's m valid rows (the rest of the tile only feeds
      // token columns the epilogue never stores).  A stage's copies are known
      // complete kLag stages later (cp.async.wait_group), or at the end of the
      // unit; then every lane fences them for the tensor core and lane 0
      // arrives on the stage.
      constexpr int kLag = C::kStages - 1;
      int stage = 0, issued = 0;
      uint32_t phase = 0, q = 0, qph = 0;
      bool ok = true;
      for (;;) {
        const int w = pop_unit(q, qph, false);
        __syncwarp();
        if (lane == 0) mbar_arrive(uq_empty((q + C::kQ - 1) % C::kQ));
        if (w < 0) fail();
        if (w < 0 || w >= total || !ok) break;
        const Unit u = unit_of(w);
        const int4 it = u.it;
        // G2 units of a fused launch bring their rows by TMA: no copies, but
        // the warp still arrives on their stages
        const int m = u.g1 ? (it.z < BN ? it.z : BN) : 0;
        __syncwarp();
        for (int r = lane; r < m; r += 32) tok_s[r] = __ldg(grows + it.y + r) / gk;
        __syncwarp();
        for (int kb = u.kb_lo; kb < u.kb_hi; ++kb) {
          int good = 1;
          if (lane == 0)
            good = mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, kWaitLimitNs);
          if (!__shfl_sync(0xffffffffu, good, 0)) {
            if (lane == 0) fail();
            ok = false;
            break;
          }
          const uint32_t sx = sbase + stage * C::kStageBytes + C::kNA * kWeightBytes;
          for (int i = lane; i < m * 8; i += 32) {
            const int r = i >> 3, ch = i & 7;
            const int k0 = kb * kBK + ch * 8;
            const int nbytes = k0 < Kdim ? 16 : 0;
            cp_async_16(sx + r * 128 + ((ch ^ (r & 7)) << 4),
                        gx + (size_t)tok_s[r] * Kdim + (nbytes ? k0 : 0), nbytes);
          }
          cp_async_commit();
          if (++issued > kLag) {
            cp_async_wait<kLag>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(full_bar((stage + C::kStages - kLag) % C::kStages));
            --issued;
          }
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        // settle the unit before waiting for the next one: the next unit may
        // only be handed out once this one is done (a fused launch's G2 unit
        // waits for G1 results), so no arrival may stay owed across the wait
        cp_async_wait<0>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
          for (int j = issued; j > 0; --j) mbar_arrive(full_bar((stage + C::kStages - j) % C::kStages));
        issued = 0;
      }
      // after a failure: the stages still owed their arrival, so that warp 0
      // can drain its weight copies
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0)
        for (int j = issued; j > 0; --j) mbar_arrive(full_bar((stage + C::kStages - j) % C::kStages));
    }
  } else if (WQ && warp < C::kConvWarp0 + C::kConvThreads / 32) {
    // ---------------- e4m3 / e2m1 -> bf16 converters, warps 10..17
    // FP8: at the start of each work unit the converters stage that unit's row
    // of block scales (one per 128-wide K block) in shared memory, so the
    // per-stage scale is a shared-memory read, not a global load.  Rows rotate
    // through three buffers: a converter can run at most two stages ahead of
    // the slowest one, so a buffer is never rewritten while still being read.
    // MXFP4: a converter owns one row and 32 K elements of each stage (one
    // scale byte per matrix) and decodes the e2m1 codes with integer bit
    // placement and one bf16 multiply (e2m1x8_to_bf16).
    const int ct = threadIdx.x - 32 * C::kConvWarp0;
    int stage = 0, cs = 0;
    uint32_t phase = 0, cphase = 0, unit = 0, q = 0, qph = 0;
    bool ok = true;
    for (;; ++unit) {
      const int w = pop_unit(q, qph, false);
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(uq_empty((q + C::kQ - 1) % C::kQ));
      if (w < 0) fail();
      if (w < 0 || w >= total || !ok) break;
      const Unit un = unit_of(w);
      const int4 it = un.it;
      const int nb = un.nb;
      const int buf = (int)(unit % 3u);
      float* scale_row = scale_rows + buf * 2 * C::kMaxScaleCols;
      // the unit's matrices: W1 and W3 (G1) or W2 (G2 of a fused launch)
      const bool g1 = un.g1;
      const int Nm = g1 || !FUSED ? N : N2, Km = g1 || !FUSED ? Kdim : K2;
      if (WQ == 1) {
        const int rb = (Nm + 127) / 128;
        const int cb = (Km + 127) / 128;
        const float* s_a = g1 || !FUSED ? sa : s2;
        const size_t row = ((size_t)it.x * rb + nb) * cb;
        for (int c = ct; c < cb; c += C::kConvThreads) {
          scale_row[c] = __ldg(s_a + row + c);
          scale_row[C::kMaxScaleCols + c] = g1 ? __ldg(sb + row + c) : 0.f;
        }
        mbar_arrive(scale_bar(buf));
        if (!mbar_wait_bounded(scale_bar(buf), (unit / 3u) & 1u, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
      }
      // MXFP4: this thread's row of the tile and its 32-element half of each
      // stage.  Its scale bytes (one per stage and matrix) are fetched eight
      // stages ahead into registers: the rows of a tile span more cache lines
      // than L1 keeps next to the pipeline's shared memory, so a load issued
      // at the stage that needs it would wait on L2 every stage.
      const int r4 = ct >> 1, j4 = ct & 1;
      const int n4 = nb * kBM + r4, kcb = Km / 32;
      const uint8_t* srow[2] = {
          reinterpret_cast<const uint8_t*>(g1 || !FUSED ? sa : s2) + ((size_t)it.x * Nm + n4) * kcb,
          reinterpret_cast<const uint8_t*>(sb) + ((size_t)it.x * Nm + n4) * kcb};
      uint32_t pend[2][8], win[2][2];
      auto fetch = [&](int kb0) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int kblk = 2 * (kb0 + i) + j4;
            pend[t][i] = (WQ == 2 && (t == 0 || g1) && n4 < Nm && kb0 + i < un.kb_hi && kblk < kcb)
                             ? (uint32_t)__ldg(srow[t] + kblk) : 0u;
          }
      };
      if (WQ == 2) fetch(un.kb_lo);
      for (int kb = un.kb_lo; kb < un.kb_hi; ++kb) {
        if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, kWaitLimitNs) ||
            !mbar_wait_bounded(conv_empty(cs), cphase ^ 1u, abort_flag, kWaitLimitNs)) {
          fail();
          ok = false;
          break;
        }
        const int sc = (kb * kBK) / 128;
        const int wi = (kb - un.kb_lo) & 7;
        if (WQ == 2 && wi == 0) {
          // the window's scale bytes (loaded a window ago) -> packed words;
          // then the next window's loads
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            win[t][0] = pend[t][0] | pend[t][1] << 8 | pend[t][2] << 16 | pend[t][3] << 24;
            win[t][1] = pend[t][4] | pend[t][5] << 8 | pend[t][6] << 16 | pend[t][7] << 24;
          }
          fetch(kb + 8);
        }
#pragma unroll
        for (int t = 0; t < C::kNA; ++t) {
          if (t > 0 && !g1) break;
          if (WQ == 2) {
            // 16 bytes = 32 e2m1 codes of row r4, K kb*64 + 32*j4 .. +31, times
            // their block's power of two (rows and blocks past the matrix: TMA
            // reads zero codes; a zero scale byte keeps them zero)
            const uint32_t sbyte = ((wi < 4 ? win[t][0] : win[t][1]) >> (8 * (wi & 3))) & 0xFFu;
            uint32_t m1, m2;
            mx_multipliers(sbyte, m1, m2);
            const bool big = sbyte > 128u;
            const uint8_t* src = smem + (size_t)stage * C::kStageBytes + t * C::kQBytes;
            uint8_t* dst = conv + (size_t)cs * C::kConvBytes + t * C::kABytes;
            const uint4 v = *reinterpret_cast<const uint4*>(src + r4 * (kBK / 2) + j4 * 16);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint4 o;
              e2m1x8_to_bf16(wv[c], m1, m2, big, &o.x);
              // 8 bf16 = 16-byte chunk 4*j4 + c of row r4, 128-byte swizzled
              *reinterpret_cast<uint4*>(dst + r4 * 128 + (((4 * j4 + c) ^ (r4 & 7)) << 4)) = o;
            }
            continue;
          }
          const float scl = scale_row[t * C::kMaxScaleCols + sc];
          const uint8_t* src = smem + (size_t)stage * C::kStageBytes + t * C::kQBytes;
          uint8_t* dst = conv + (size_t)cs * C::kConvBytes + t * C::kABytes;
#pragma unroll
          for (int i = 0; i < 512 / C::kConvThreads; ++i) {
            const int q = ct + C::kConvThreads * i;  // 16-byte e4m3 chunk: row q/4, K 16*(q%4)..+15
            const int r = q >> 2, j = q & 3;
            const uint4 v = *reinterpret_cast<const uint4*>(src + r * kBK + j * 16);
            uint4 lo, hi;
            lo.x = e4m3x2_to_bf16x2(v.x & 0xFFFFu, scl);
            lo.y = e4m3x2_to_bf16x2(v.x >> 16, scl);
            lo.z = e4m3x2_to_bf16x2(v.y & 0xFFFFu, scl);
            lo.w = e4m3x2_to_bf16x2(v.y >> 16, scl);
            hi.x = e4m3x2_to_bf16x2(v.z & 0xFFFFu, scl);
            hi.y = e4m3x2_to_bf16x2(v.z >> 16, scl);
            hi.z = e4m3x2_to_bf16x2(v.w & 0xFFFFu, scl);
            hi.w = e4m3x2_to_bf16x2(v.w >> 16, scl);
            // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r % 8)
            *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * j) ^ (r & 7)) << 4)) = lo;
            *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * j + 1) ^ (r & 7)) << 4)) = hi;
          }
        }
        fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
        mbar_arrive(conv_full(cs));
        if (++cs == C::kConvStages) { cs = 0; cphase ^= 1u; }
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN, bool SWIGLU, int WQ, bool FUSED>
__global__ void __launch_bounds__(TcCfg<BN, SWIGLU, WQ>::kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_wa, const __grid_constant__ CUtensorMap tm_wb,
               const __grid_constant__ CUtensorMap tm_act, const float* __restrict__ sa,
               const float* __restrict__ sb, int32_t* __restrict__ counts, int list,
               const int4* __restrict__ items, int N, int Kdim, __nv_bfloat16* __restrict__ out,
               int ksplit, int R, float* __restrict__ part, int32_t* dev_status,
               const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_h,
               const float* __restrict__ s2, int N2, int K2, __nv_bfloat16* __restrict__ out2,
               int32_t* __restrict__ done, const __nv_bfloat16* __restrict__ gx,
               const int32_t* __restrict__ grows, int gk, int ksplit2,
               float* __restrict__ part2, int32_t* __restrict__ scnt1,
               int32_t* __restrict__ scnt2) {
  pdl_wait();
  pdl_trigger();
  gemm_tc_body<BN, SWIGLU, WQ, FUSED>(tm_wa, tm_wb, tm_act, sa, sb, counts, list, items, N, Kdim,
                                        out, ksplit, R, part, dev_status, tm_w2, tm_h, s2, N2, K2,
                                        out2, done, gx, grows, gk, ksplit2, part2, scnt1, scnt2,
                                        (int)blockIdx.x, (int)gridDim.x);
}

// The skinny and the tile list in ONE launch: the grid splits into two CTA
// groups in proportion to each list's work units (read on the device from the
// plan's counts), each group walking its own list with its
// own token-tile width and pipeline -- both variants run side by side instead
// of one launch after the other, each block still on the variant its own
// m_size chose.
struct DualMaps {
  CUtensorMap act[2];  // per list: G1 activations (xp) or, for G2, hact
  CUtensorMap h[2];    // FUSED: hact per list
};

template <bool SWIGLU, int WQ, bool FUSED>
__global__ void __launch_bounds__(TcCfg<kBnSkinny, SWIGLU, WQ>::kThreads, 1)
gemm_tc_dual_kernel(const __grid_constant__ CUtensorMap tm_wa,
                    const __grid_constant__ CUtensorMap tm_wb, const __grid_constant__ DualMaps maps,
                    const float* __restrict__ sa, const float* __restrict__ sb,
                    int32_t* __restrict__ counts, const int4* __restrict__ items0,
                    const int4* __restrict__ items1, int N, int Kdim,
                    __nv_bfloat16* __restrict__ out, int R, int32_t* dev_status,
                    const __grid_constant__ CUtensorMap tm_w2, const float* __restrict__ s2,
                    int N2, int K2, __nv_bfloat16* __restrict__ out2,
                    int32_t* __restrict__ done0, int32_t* __restrict__ done1,
                    const __nv_bfloat16* __restrict__ gx, const int32_t* __restrict__ grows,
                    int gk) {
  using C0 = TcCfg<kBnSkinny, SWIGLU, WQ>;
  using C1 = TcCfg<kBnTile, SWIGLU, WQ>;
  static_assert(C0::kThreads == C1::kThreads, "one block size for both groups");
  pdl_wait();
  pdl_trigger();
  // a unit of either list streams the same weight tile, which dominates its
  // time: split by unit count
  const long long b0 = counts[0];
  const long long b1 = counts[1];
  const int g = (int)gridDim.x;
  int s0 = b0 + b1 > 0 ? (int)((b0 * g + (b0 + b1) / 2) / (b0 + b1)) : 0;
  if (b0 > 0 && s0 < 1) s0 = 1;
  if (b1 > 0 && s0 > g - 1) s0 = g - 1;
  if ((int)blockIdx.x < s0)
    gemm_tc_body<kBnSkinny, SWIGLU, WQ, FUSED>(
        tm_wa, tm_wb, maps.act[0], sa, sb, counts, 0, items0, N, Kdim, out, 1, R, nullptr,
        dev_status, tm_w2, maps.h[0], s2, N2, K2, out2, done0, gx, grows, gk, 1, nullptr, nullptr,
        nullptr, (int)blockIdx.x, s0);
  else
    gemm_tc_body<kBnTile, SWIGLU, WQ, FUSED>(
        tm_wa, tm_wb, maps.act[1], sa, sb, counts, 1, items1, N, Kdim, out, 1, R, nullptr,
        dev_status, tm_w2, maps.h[1], s2, N2, K2, out2, done1, gx, grows, gk, 1, nullptr, nullptr,
        nullptr, (int)blockIdx.x - s0, g - s0);
}

// ---------------------------------------------------------------- CUDA cores
// One CTA = one skinny item (<= 16 rows) x 64 output features, 256 threads:
// thread = feature (tid % 64) x 4 rows (tid / 64).  Weights and activations
// are staged per 64-wide K chunk in shared memory as fp32.
constexpr int kSimtN = 64;
constexpr int kSimtK = 64;

template <int WQ>
MOE_DEVICE float load_w(const void* w, const float* s, int e, int n, int k, int N, int Kdim) {
  const size_t idx = ((size_t)e * N + n) * Kdim + k;
  if (WQ == MOE_W_MXFP4) {
    // element k of the row: byte k/2, low nibble for even k; scale k/32
    const uint8_t byte = static_cast<const uint8_t*>(w)[idx / 2];
    const int c = (k & 1) ? byte >> 4 : byte & 15, ex = (c >> 1) & 3, m = c & 1;
    const float mag = ex == 0 ? 0.5f * m : (1.f + 0.5f * m) * (float)(1 << (ex - 1));
    const uint32_t sb = reinterpret_cast<const uint8_t*>(s)[((size_t)e * N + n) * (Kdim / 32) + k / 32];
    const float sc = sb ? __uint_as_float(sb << 23) : __uint_as_float(0x00400000u);
    return ((c & 8) ? -mag : mag) * sc;
  }
  if (WQ == MOE_W_FP8E4M3_B128) {
    const uint8_t code = static_cast<const uint8_t*>(w)[idx];
    const __half_raw hr = __nv_cvt_fp8_to_halfraw(code, __NV_E4M3);
    const int rb = (N + 127) / 128, cb = (Kdim + 127) / 128;
    const float sc = s[((size_t)e * rb + n / 128) * cb + k / 128];
    return __half2float(__half(hr)) * sc;
  } else {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(w)[idx]);
  }
}

template <bool SWIGLU, int WQ>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const __nv_bfloat16* __restrict__ act, const void* __restrict__ wa,
                 const void* __restrict__ wb, const float* __restrict__ sa,
                 const float* __restrict__ sb, const int32_t* __restrict__ counts, int list,
                 const int4* __restrict__ items, int N, int Kdim, __nv_bfloat16* __restrict__ out) {
  __shared__ float As[kBnSkinny][kSimtK];
  __shared__ float Wa[kSimtN][kSimtK + 1];
  __shared__ float Wb[SWIGLU ? kSimtN : 1][kSimtK + 1];
  pdl_wait();
  pdl_trigger();
  const int n_items = counts[list];
  for (int item = blockIdx.y; item < n_items; item += gridDim.y) {
  const int4 it = items[item];
  const int e = it.x, r0 = it.y, m = it.z;
  const int n0 = blockIdx.x * kSimtN;
  const int tid = threadIdx.x, fl = tid % kSimtN, tg = tid / kSimtN;
  float ga[4] = {0.f, 0.f, 0.f, 0.f}, gb[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < Kdim; k0 += kSimtK) {
    for (int i = tid; i < kBnSkinny * kSimtK; i += 256) {
      const int r = i / kSimtK, k = k0 + i % kSimtK;
      As[r][i % kSimtK] = (r < m && k < Kdim) ? __bfloat162float(act[(size_t)(r0 + r) * Kdim + k]) : 0.f;
    }
    for (int i = tid; i < kSimtN * kSimtK; i += 256) {
      const int r = i / kSimtK, k = k0 + i % kSimtK, n = n0 + r;
      const bool in = n < N && k < Kdim;
      Wa[r][i % kSimtK] = in ? load_w<WQ>(wa, sa, e, n, k, N, Kdim) : 0.f;
      if (SWIGLU) Wb[r][i % kSimtK] = in ? load_w<WQ>(wb, sb, e, n, k, N, Kdim) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < kSimtK; ++k) {
      const float w1 = Wa[fl][k];
      const float w3 = SWIGLU ? Wb[fl][k] : 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = As[tg * 4 + i][k];
        ga[i] = fmaf(a, w1, ga[i]);
        if (SWIGLU) gb[i] = fmaf(a, w3, gb[i]);
      }
    }
    __syncthreads();
  }
  const int n = n0 + fl;
  if (n < N) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = tg * 4 + i;
      if (r < m) {
        const float v = SWIGLU ? silu_f(ga[i]) * gb[i] : ga[i];
        out[(size_t)(r0 + r) * N + n] = __float2bfloat16_rn(v);
      }
    }
  }
  }
}

// ---------------------------------------------------------------- split-K finalize
// out[r][n] = bf16( silu(sum_ks g) * sum_ks u )  (SwiGLU)  or  bf16( sum_ks p )
// with the K slices summed in slice order; 4 features per thread.
template <bool SWIGLU>
__global__ void __launch_bounds__(256)
splitk_finalize_kernel(const float* __restrict__ part, int ksplit, int R, int N,
                       __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int np = SWIGLU ? 2 * N : N;
  const int n4 = N / 4;
  const long long total = (long long)R * n4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / n4), n = (int)(i % n4) * 4;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    for (int ks = 0; ks < ksplit; ++ks) {
      const float* pr = part + ((size_t)ks * R + r) * np;
      const float4 a = *reinterpret_cast<const float4*>(pr + n);
      g.x += a.x; g.y += a.y; g.z += a.z; g.w += a.w;
      if (SWIGLU) {
        const float4 b = *reinterpret_cast<const float4*>(pr + N + n);
        u.x += b.x; u.y += b.y; u.z += b.z; u.w += b.w;
      }
    }
    float4 v = g;
    if (SWIGLU) {
      v.x = silu_f(g.x) * u.x; v.y = silu_f(g.y) * u.y;
      v.z = silu_f(g.z) * u.z; v.w = silu_f(g.w) * u.w;
    }
    uint2 o;
    o.x = pack_bf16x2(v.x, v.y);
    o.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2*>(out + (size_t)r * N + n) = o;
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [E][N][Kdim] weights, a box of 64 K elements x 128 rows (N) x 1: bf16 in the
// 128-byte swizzle the MMA reads, or e4m3 bytes / e2m1 byte pairs (32 bytes a
// row) unswizzled (the converters re-lay them out).  wq: a MOE_W_* code.
bool make_weight_map(CUtensorMap* m, const void* w, int E, int N, int Kdim, int wq) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const bool bytes = wq != MOE_W_BF16;
  const cuuint64_t row = wq == MOE_W_MXFP4 ? (cuuint64_t)Kdim / 2
                       : (cuuint64_t)Kdim * (wq == MOE_W_BF16 ? 2 : 1);  // bytes per row
  cuuint64_t dims[3] = {bytes ? row : (cuuint64_t)Kdim, (cuuint64_t)N, (cuuint64_t)E};
  cuuint64_t strides[2] = {row, (cuuint64_t)N * row};
  cuuint32_t box[3] = {wq == MOE_W_MXFP4 ? (cuuint32_t)kBK / 2 : (cuuint32_t)kBK, kBM, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void*>(w), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             bytes ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [R][Kdim] bf16 activations, box 64 (K) x bn (rows)
bool make_act_map(CUtensorMap* m, const void* a, int R, int Kdim, int bn) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)Kdim, (cuuint64_t)R};
  cuuint64_t strides[1] = {(cuuint64_t)Kdim * 2};
  cuuint32_t box[2] = {kBK, (cuuint32_t)bn};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() { return moe_num_sms(); }

// One launch of the tensor-core kernel over a list.  FUSED: the list's G1
// and G2 units in one persistent launch (w2/h/s2/N2/K2/out2/done describe G2;
// ksplit must be 1).
template <int BN, bool SWIGLU, int WQ, bool FUSED = false>
cudaError_t run_tc(const CUtensorMap& wa, const CUtensorMap& wb, const CUtensorMap& act,
                   const float* sa, const float* sb, int32_t* counts, int list,
                   const int4* items, int cap, int N, int Kdim, void* out, int32_t* dev_status,
                   cudaStream_t stream, int ksplit = 1, int R = 0, float* part = nullptr,
                   const CUtensorMap* w2 = nullptr, const CUtensorMap* h = nullptr,
                   const float* s2 = nullptr, int N2 = 0, int K2 = 0, void* out2 = nullptr,
                   int32_t* done = nullptr, const void* gx = nullptr,
                   const int32_t* grows = nullptr, int gk = 0, int ksplit2 = 1,
                   float* part2 = nullptr, int32_t* scnt1 = nullptr, int32_t* scnt2 = nullptr) {
  using C = TcCfg<BN, SWIGLU, WQ>;
  static std::atomic<unsigned long long> smem_set{0};  // devices whose limit is raised
  {
    cudaError_t e = moe_raise_smem(gemm_tc_kernel<BN, SWIGLU, WQ, FUSED>, C::kSmemBytes, smem_set);
    if (e != cudaSuccess) return e;
  }
  const long long work =
      (long long)cap * (moe_cdiv(N, kBM) * ksplit + (FUSED ? moe_cdiv(N2, kBM) * ksplit2 : 0));
  const int grid = (int)(work < num_sms() ? work : num_sms());
  if (grid <= 0) return cudaSuccess;
  cudaError_t e = moe_launch(gemm_tc_kernel<BN, SWIGLU, WQ, FUSED>, dim3(grid),
                             dim3(C::kThreads), C::kSmemBytes, stream, 1, wa, wb, act, sa, sb,
                             counts, list, items, N, Kdim, static_cast<__nv_bfloat16*>(out),
                             ksplit, R, part, dev_status, FUSED ? *w2 : wa, FUSED ? *h : act, s2,
                             N2, K2, static_cast<__nv_bfloat16*>(out2), done,
                             static_cast<const __nv_bfloat16*>(gx), grows, gk, ksplit2, part2,
                             scnt1, scnt2);
  // K slices are reduced in the kernel by their last slice when counters are
  // given, else by a finalize launch
  if (e != cudaSuccess || ksplit <= 1 || scnt1) return e;
  const long long n = (long long)R * (N / 4);
  const int fgrid = (int)((n + 255) / 256 < 4 * num_sms() ? (n + 255) / 256 : 4 * num_sms());
  return moe_launch(splitk_finalize_kernel<SWIGLU>, dim3(fgrid), dim3(256), 0, stream, 1,
                    (const float*)part, ksplit, R, N, static_cast<__nv_bfloat16*>(out));
}

// Both lists (skinny, tile) in one launch of two CTA groups.  FUSED: each
// group runs its list's G1 and G2 units (act = xp maps, h = hact maps).
template <bool SWIGLU, int WQ, bool FUSED>
cudaError_t run_tc_dual(const CUtensorMap& wa, const CUtensorMap& wb, const DualMaps& maps,
                        const float* sa, const float* sb, const PlanView& pv, int N, int Kdim,
                        void* out, int R, int32_t* dev_status, cudaStream_t stream,
                        const CUtensorMap& w2, const float* s2, int N2, int K2, void* out2,
                        const void* gx = nullptr, const int32_t* grows = nullptr, int gk = 0) {
  using C0 = TcCfg<kBnSkinny, SWIGLU, WQ>;
  using C1 = TcCfg<kBnTile, SWIGLU, WQ>;
  const size_t smem = C0::kSmemBytes > C1::kSmemBytes ? C0::kSmemBytes : C1::kSmemBytes;
  static std::atomic<unsigned long long> smem_set{0};  // devices whose limit is raised
  {
    cudaError_t e = moe_raise_smem(gemm_tc_dual_kernel<SWIGLU, WQ, FUSED>, smem, smem_set);
    if (e != cudaSuccess) return e;
  }
  const int grid = num_sms();
  return moe_launch(gemm_tc_dual_kernel<SWIGLU, WQ, FUSED>, dim3(grid), dim3(C0::kThreads), smem,
                    stream, 1, wa, wb, maps, sa, sb, pv.counts, (const int4*)pv.items[0],
                    (const int4*)pv.items[1], N, Kdim, static_cast<__nv_bfloat16*>(out), R,
                    dev_status, w2, s2, N2, K2, static_cast<__nv_bfloat16*>(out2), pv.done[0],
                    pv.done[1], static_cast<const __nv_bfloat16*>(gx), grows, gk);
}

// K slices for the skinny variant.  The persistent grid walks units x slices
// in waves of one unit per SM, and a wave lasts as long as its longest slice,
// so the time is about waves(s) x (K steps per slice + a fixed cost per unit
// for pipeline fill and epilogue, ~2 K steps).  s = 1..kMaxKSplit minimising
// that (ties to the smaller s), slices at least 2 K steps long; 1 = no split.
constexpr int kMaxKSplit = 8;
int pick_ksplit(long long units, int Kdim) {
  const int nk = (Kdim + kBK - 1) / kBK;
  const long long sms = num_sms();
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= kMaxKSplit; ++s) {
    const int kbs = (nk + s - 1) / s;
    if (s > 1 && kbs < 2) break;
    const long long waves = (units * s + sms - 1) / sms;
    const long long cost = waves * (kbs + 2);
    if (best_cost < 0 || cost < best_cost) { best = s; best_cost = cost; }
  }
  return best;
}

template <int WQ>
cudaError_t run_tc_all(const void* xp, int R, int E_blocks, int H, int I, const void* w1,
                       const void* w3, const void* w2, const float* s1, const float* s3,
                       const float* s2, void* hact, void* y, const PlanView& pv,
                       int32_t* dev_status, cudaStream_t stream, const bool (&any)[kLists],
                       float* splitk_buf, size_t splitk_bytes, const void* gx,
                       const int32_t* grows, int gk, int32_t* split_cnt) {
  // split-K only when every block is skinny (all rows then belong to skinny
  // items, which the finalize kernel rewrites) and the buffer holds the slices
  int ks1 = 1, ks2 = 1;
  if (splitk_buf && any[0] && !any[1] && !any[2]) {
    const long long blocks = R < E_blocks ? R : E_blocks;
    ks1 = pick_ksplit(blocks * moe_cdiv(I, kBM), H);
    ks2 = pick_ksplit(blocks * moe_cdiv(H, kBM), I);
    if ((size_t)ks1 * R * 2 * I * sizeof(float) > splitk_bytes) ks1 = 1;
    if ((size_t)ks2 * R * H * sizeof(float) > splitk_bytes) ks2 = 1;
    if (I % 4 || H % 4) ks1 = ks2 = 1;
  }
  // One fused G1+G2 launch per list pays off while the G1 units are few (its
  // last wave is a large share of the G1 time): mean rows per block <= 64, and
  // G2 not much larger than G1 (H <= 3 I).  Otherwise G2 prefers its own
  // deeper pipeline: in the fused layout a G2 stage occupies a G1-sized slot,
  // so its own launch keeps half again as many stages in flight.
  // (Measured: qwen3-30b-a3b shape T=256 264 -> 254 us and gpt-oss-20b shape
  // T=512 427 -> 415 us fused; the H = 4 I shared-gate shape at T=1024 went
  // 630 -> 655 us fused.)
  const bool fuse = (long long)R <= 64LL * E_blocks && H <= 3 * I && !gx;
  CUtensorMap m_w1, m_w3, m_w2, m_x[kLists], m_h[kLists];
  memset(m_x, 0, sizeof(m_x));  // gather mode: G1 reads x rows itself, no activation map
  if (!make_weight_map(&m_w1, w1, E_blocks, I, H, WQ) ||
      !make_weight_map(&m_w3, w3, E_blocks, I, H, WQ) ||
      !make_weight_map(&m_w2, w2, E_blocks, H, I, WQ))
    return cudaErrorInvalidValue;
  for (int l = 0; l < kLists; ++l)
    if (any[l] && ((!gx && !make_act_map(&m_x[l], xp, R, H, list_bn(l))) ||
                   !make_act_map(&m_h[l], hact, R, I, list_bn(l))))
      return cudaErrorInvalidValue;
  cudaError_t err = cudaSuccess;
  if (split_cnt && splitk_buf && any[0] && !any[1] && !any[2]) {
    // small batches, every block skinny: the K slices of each unit are
    // reduced in the kernel by the slice that finishes last (no finalize
    // launch); G2 reuses the slice buffer once G1 is done with it.  (One
    // launch for G1 and G2 together measured no faster here: G2 units wait for
    // G1 results, and in the shared layout a G2 stage occupies a G1-sized slot.)
    int32_t* c1 = split_cnt;
    int32_t* c2 = split_cnt + (size_t)pv.cap[0] * moe_cdiv(I, kBM);
    err = run_tc<kBnSkinny, true, WQ>(m_w1, m_w3, m_x[0], s1, s3, pv.counts, 0, pv.items[0],
                                        pv.cap[0], I, H, hact, dev_status, stream, ks1, R,
                                        splitk_buf, nullptr, nullptr, nullptr, 0, 0, nullptr,
                                        nullptr, gx, grows, gk, 1, nullptr, c1, nullptr);
    if (err != cudaSuccess) return err;
    return run_tc<kBnSkinny, false, WQ>(m_w2, m_w2, m_h[0], s2, s2, pv.counts, 0, pv.items[0],
                                          pv.cap[0], H, I, y, dev_status, stream, ks2, R,
                                          splitk_buf, nullptr, nullptr, nullptr, 0, 0, nullptr,
                                          nullptr, nullptr, nullptr, 0, 1, nullptr, c2, nullptr);
  }
  if (any[0] && any[1] && !any[2] && ks1 == 1 && ks2 == 1) {
    // skinny and tile blocks both present: one launch per phase (or one in
    // all, fused) in which the two lists run side by side
    DualMaps mx, mh;
    for (int l = 0; l < 2; ++l) {
      mx.act[l] = m_x[l];
      mx.h[l] = m_h[l];
      mh.act[l] = m_h[l];
      mh.h[l] = m_h[l];
    }
    if (fuse)
      return run_tc_dual<true, WQ, true>(m_w1, m_w3, mx, s1, s3, pv, I, H, hact, R, dev_status,
                                           stream, m_w2, s2, H, I, y);
    err = run_tc_dual<true, WQ, false>(m_w1, m_w3, mx, s1, s3, pv, I, H, hact, R, dev_status,
                                         stream, m_w2, s2, 0, 0, nullptr, gx, grows, gk);
    if (err != cudaSuccess) return err;
    return run_tc_dual<false, WQ, false>(m_w2, m_w2, mh, s2, s2, pv, H, I, y, R, dev_status,
                                           stream, m_w2, s2, 0, 0, nullptr);
  }
  // G1 (SwiGLU, N = I, K = H) for every list, then G2 (N = H, K = I)
  if (any[0] && err == cudaSuccess)
    err = run_tc<kBnSkinny, true, WQ>(m_w1, m_w3, m_x[0], s1, s3, pv.counts, 0, pv.items[0],
                                        pv.cap[0], I, H, hact, dev_status, stream, ks1, R,
                                        splitk_buf, nullptr, nullptr, nullptr, 0, 0, nullptr,
                                        nullptr, gx, grows, gk);
  if (fuse) {
    // tile and wide lists: G1 and G2 in one persistent launch each
    if (any[1] && err == cudaSuccess)
      err = run_tc<kBnTile, true, WQ, true>(m_w1, m_w3, m_x[1], s1, s3, pv.counts, 1,
                                              pv.items[1], pv.cap[1], I, H, hact, dev_status,
                                              stream, 1, R, nullptr, &m_w2, &m_h[1], s2, H, I, y,
                                              pv.done[1]);
    if (any[2] && err == cudaSuccess)
      err = run_tc<kBnWide, true, WQ, true>(m_w1, m_w3, m_x[2], s1, s3, pv.counts, 2,
                                              pv.items[2], pv.cap[2], I, H, hact, dev_status,
                                              stream, 1, R, nullptr, &m_w2, &m_h[2], s2, H, I, y,
                                              pv.done[2]);
  } else {
    if (any[1] && err == cudaSuccess)
      err = run_tc<kBnTile, true, WQ>(m_w1, m_w3, m_x[1], s1, s3, pv.counts, 1, pv.items[1],
                                        pv.cap[1], I, H, hact, dev_status, stream, 1, R, nullptr,
                                        nullptr, nullptr, nullptr, 0, 0, nullptr, nullptr, gx,
                                        grows, gk);
    if (any[2] && err == cudaSuccess)
      err = run_tc<kBnWide, true, WQ>(m_w1, m_w3, m_x[2], s1, s3, pv.counts, 2, pv.items[2],
                                        pv.cap[2], I, H, hact, dev_status, stream, 1, R, nullptr,
                                        nullptr, nullptr, nullptr, 0, 0, nullptr, nullptr, gx,
                                        grows, gk);
    if (any[1] && err == cudaSuccess)
      err = run_tc<kBnTile, false, WQ>(m_w2, m_w2, m_h[1], s2, s2, pv.counts, 1, pv.items[1],
                                         pv.cap[1], H, I, y, dev_status, stream);
    if (any[2] && err == cudaSuccess)
      err = run_tc<kBnWide, false, WQ>(m_w2, m_w2, m_h[2], s2, s2, pv.counts, 2, pv.items[2],
                                         pv.cap[2], H, I, y, dev_status, stream);
  }
  if (any[0] && err == cudaSuccess)
    err = run_tc<kBnSkinny, false, WQ>(m_w2, m_w2, m_h[0], s2, s2, pv.counts, 0, pv.items[0],
                                         pv.cap[0], H, I, y, dev_status, stream, ks2, R,
                                         splitk_buf);

  return err;
}

template <bool SWIGLU>
cudaError_t run_simt(int wq, const void* act, const void* wa, const void* wb, const float* sa,
                     const float* sb, const int32_t* counts, const int4* items, int cap, int N,
                     int Kdim, void* out, cudaStream_t stream) {
  if (cap <= 0) return cudaSuccess;
  dim3 grid(moe_cdiv(N, kSimtN), cap < 32768 ? cap : 32768);
  const __nv_bfloat16* a = static_cast<const __nv_bfloat16*>(act);
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  if (wq == MOE_W_MXFP4)
    return moe_launch(gemm_simt_kernel<SWIGLU, MOE_W_MXFP4>, grid, dim3(256), 0, stream, 1, a, wa,
                      wb, sa, sb, counts, 0, items, N, Kdim, o);
  if (wq == MOE_W_FP8E4M3_B128)
    return moe_launch(gemm_simt_kernel<SWIGLU, MOE_W_FP8E4M3_B128>, grid, dim3(256), 0, stream, 1,
                      a, wa, wb, sa, sb, counts, 0, items, N, Kdim, o);
  return moe_launch(gemm_simt_kernel<SWIGLU, MOE_W_BF16>, grid, dim3(256), 0, stream, 1, a, wa, wb,
                    sa, sb, counts, 0, items, N, Kdim, o);
}

}  // namespace

cudaError_t launch_bounded_wait_check(const int32_t* counter, int target, uint64_t limit_ns,
                                      int32_t* dev_status, cudaStream_t stream) {
  // a plain launch: it reads caller memory that earlier stream work may write
  bounded_wait_kernel<<<1, 32, 0, stream>>>(counter, target, limit_ns, dev_status);
  return cudaGetLastError();
}

size_t grouped_gemm_scratch_bytes(int R, int E_blocks) { return plan_bytes(R, E_blocks); }

size_t grouped_gemm_scratch_bytes_ex(int R, int E_blocks, int H, int I, int wdtype) {
  return plan_bytes(R, E_blocks) +
         (wdtype == MOE_W8A8_FP8E4M3_B128 ? w8a8_act_bytes(R, H, I) : 0);
}

size_t grouped_gemm_split_counter_bytes(int R, int E_blocks, int H, int I) {
  const size_t cap0 = (size_t)moe_cdiv(R, kBnSkinny) + E_blocks;
  return moe_align_up(cap0 * (moe_cdiv(I, kBM) + moe_cdiv(H, kBM)) * sizeof(int32_t), 256);
}

size_t grouped_gemm_splitk_bytes(int R, int H, int I) {
  const size_t w = (size_t)(2 * I > H ? 2 * I : H);
  return moe_align_up((size_t)kMaxKSplit * R * w * sizeof(float), 256);
}

int grouped_gemm_check(int H, int I, int wdtype) {
  if (H % 16 != 0 || I % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (wdtype != MOE_W_BF16 && wdtype != MOE_W_FP8E4M3_B128 && wdtype != MOE_W_MXFP4 &&
      wdtype != MOE_W8A8_FP8E4M3_B128)
    return MOE_ERR_UNSUPPORTED;
  // MXFP4: whole 32-element scale blocks along every row
  if (wdtype == MOE_W_MXFP4 && (H % 32 != 0 || I % 32 != 0)) return MOE_ERR_INVALID_ARG;
  // FP8: each work unit stages its row of 128-wide K-block scales (<= 64)
  if (wdtype == MOE_W_FP8E4M3_B128 && (H > 8192 || I > 8192)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

cudaError_t launch_grouped_gemm(const void* xp, const int32_t* offsets, int E_blocks, int R,
                                int H, int I, int wdtype, const void* w1, const void* w3,
                                const void* w2, const float* s1, const float* s3,
                                const float* s2, void* hact, void* y, int m_skinny,
                                int dispatch, int32_t* block_variant, void* scratch,
                                int32_t* dev_status, cudaStream_t stream, int max_rows,
                                bool plan_ready, float* splitk_buf, size_t splitk_bytes,
                                const void* gather_x, const int32_t* gather_rows, int gather_k,
                                int32_t* split_cnt) {
  if (m_skinny < 0) m_skinny = MOE_DEFAULT_M_SKINNY;
  const bool conv = wdtype != MOE_W_BF16;  // weights converted in the kernel (FP8, MXFP4)
  const bool simt = dispatch == MOE_DISPATCH_SIMT;
  PlanView pv = plan_view(scratch, R, E_blocks);
  PlanOut po = plan_out(pv);
  cudaError_t err = cudaSuccess;
  if (!plan_ready)
    err = moe_launch(gemm_plan_kernel, dim3(1), dim3(1024), 0, stream, 1, offsets, E_blocks, R,
                     m_skinny, dispatch, wdtype, pv.counts, po, block_variant);
  if (err != cudaSuccess || R == 0) return err;

  if (wdtype == MOE_W8A8_FP8E4M3_B128) {
    if (simt || gather_x) return cudaErrorInvalidValue;  // W8A8 reads xp, tensor cores only
    return launch_w8a8(xp, R, E_blocks, H, I, w1, w3, w2, s1, s3, s2, hact, y, pv.counts,
                       pv.items[1], static_cast<char*>(scratch) + plan_bytes(R, E_blocks),
                       dev_status, stream);
  }
  if (simt && gather_x) return cudaErrorInvalidValue;  // the CUDA-core path reads xp only
  if (simt) {
    err = run_simt<true>(wdtype, xp, w1, w3, s1, s3, pv.counts, pv.items[0], pv.cap[0], I, H,
                         hact, stream);
    if (err != cudaSuccess) return err;
    return run_simt<false>(wdtype, hact, w2, nullptr, s2, nullptr, pv.counts, pv.items[0],
                           pv.cap[0], H, I, y, stream);
  }
  // Which lists can be non-empty, from what the host knows without reading
  // the offsets: no block holds more than max_rows rows (moe_layer passes T:
  // a token picks distinct experts), and under the global average every block
  // takes the same variant.  An empty list's launch is skipped.
  if (max_rows < 0 || max_rows > R) max_rows = R;
  bool any[kLists];
  if (dispatch == MOE_DISPATCH_GLOBAL_AVG) {
    const int v = moe_variant_of(1, R, E_blocks, m_skinny, dispatch, wdtype);
    any[0] = v == MOE_VARIANT_SKINNY;
    any[1] = v == MOE_VARIANT_TILE;
    any[2] = v == MOE_VARIANT_WIDE;
  } else {
    any[0] = true;
    any[1] = max_rows > m_skinny;
    any[2] = conv && max_rows > m_skinny && max_rows >= MOE_WIDE_MIN_ROWS;
  }
  if (wdtype == MOE_W_MXFP4)
    return run_tc_all<MOE_W_MXFP4>(xp, R, E_blocks, H, I, w1, w3, w2, s1, s3, s2, hact, y, pv,
                                   dev_status, stream, any, splitk_buf, splitk_bytes, gather_x,
                                   gather_rows, gather_k, split_cnt);
  if (wdtype == MOE_W_FP8E4M3_B128)
    return run_tc_all<MOE_W_FP8E4M3_B128>(xp, R, E_blocks, H, I, w1, w3, w2, s1, s3, s2, hact, y,
                                          pv, dev_status, stream, any, splitk_buf, splitk_bytes,
                                          gather_x, gather_rows, gather_k, split_cnt);
  return run_tc_all<MOE_W_BF16>(xp, R, E_blocks, H, I, w1, w3, w2, s1, s3, s2, hact, y, pv,
                                dev_status, stream, any, splitk_buf, splitk_bytes, gather_x,
                                gather_rows, gather_k, split_cnt);
}
