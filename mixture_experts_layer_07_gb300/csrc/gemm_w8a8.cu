// W8A8 expert GEMMs: FP8 e4m3 weights (fp32 scale per 128 x 128 block) times
// activations quantised to e4m3 with one fp32 scale per (row, 128 columns),
// on the tcgen05 tensor cores with kind::f8f6f4 MMAs.
//
// "vLLM CPU MoE: dynamic GEMM dispatch beyond a fixed threshold" (vllm PR
// #50949), introduction: the MoE path serves FP8 expert weights.  The pages
// fix no activation format; this option quantises both GEMMs' activations:
//   xq, sx = quant(xp)            (per row and 128 columns of H)
//   hact   = bf16(silu(g) * u),   g, u = dequant(xq) . dequant(W1 | W3)^T
//   hq, sh = quant(hact)          (per row and 128 columns of I)
//   y      = bf16(dequant(hq) . dequant(W2)^T)
// quant: s = amax / 448 (fp32, IEEE division; 0 for an all-zero block),
// code = e4m3(v / s) rounded to nearest even and saturated at 448.
//
// A stage holds one 128-wide K block, which is one scale block of both
// operands, so a stage's product is exact in the MMA's fp32 accumulator up to
// the two scales.  The MMA writes each stage's product into a fresh TMEM
// tile (four tiles in rotation); the epilogue warps read it back, multiply by
// the weight scale times the column's activation scale and add it into fp32
// accumulators held in registers (packed two-wide FMAs), then release the
// tile.  After the last stage they apply SwiGLU (G1) and store bf16 rows.
//
// Token tiles: G1 64 tokens (its two 64-column products -- W1 and W3 -- fill
// one 128-column TMEM tile), G2 128 tokens.  Work units are (tile-list item,
// 64-token half (G1), 128-feature block), dealt to the persistent CTAs in a
// fixed stride; every role walks the same sequence.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace {

using namespace moe_ptx;

constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, splitting the tile's token columns
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint64_t kWaitNs = 2000000000ull;  // every wait gives up after 2 s
constexpr int kQuantWarps = 8;

// D fp32, A and B e4m3, both K-major (kind::f8f6f4 instruction descriptor)
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                                 // D format: f32
         | (0u << 7)                               // A format: e4m3
         | (0u << 10)                              // B format: e4m3
         | (static_cast<uint32_t>(N >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);  // M / 16
}

// D(tmem) (+)= A(smem) * B(smem)^T, 8-bit inputs, K = 32 per instruction
MOE_DEVICE void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// two fp32 FMAs in one instruction: (a.x*b.x + c.x, a.y*b.y + c.y)
MOE_DEVICE float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long*>(&a)),
        "l"(*reinterpret_cast<unsigned long long*>(&b)),
        "l"(*reinterpret_cast<unsigned long long*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}

constexpr int kSets = 4;  // TMEM product tiles in flight between the MMA and the epilogue

template <bool G1>
struct W8Cfg {
  static constexpr int BN = G1 ? 64 : 128;     // token columns of a unit
  static constexpr int kNA = G1 ? 2 : 1;       // weight matrices of a unit (W1, W3 | W2)
  static constexpr int kABytes = 128 * 128;    // e4m3 weight tile: 128 rows x 128 K
  static constexpr int kBBytes = BN * 128;     // e4m3 activation tile
  static constexpr int kStageBytes = kNA * kABytes + kBBytes;
  static constexpr int kSetCols = kNA * BN;    // TMEM columns of one stage's products
  static constexpr int kTmemCols = kSets * kSetCols;
  static constexpr int kCols = BN / (kEpiWarps / 4);  // token columns of one epilogue warp
  static constexpr int kXs = kCols < 32 ? 1 : kCols / 32;  // activation scales per lane and stage
  static constexpr int kScPer = G1 ? 2 * kCols : kCols;    // per warp: column scales of a stage
  static constexpr int kStgBytes = kEpiWarps * kCols * 32 * 2;  // store staging: kCols rows x 32 bf16
  static constexpr int kScBytes = kEpiWarps * 2 * kScPer * 4;  // two scale rows per warp
  static constexpr int kStagesRaw = (220 * 1024 - kStgBytes - kScBytes - 2048) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static constexpr int kNumBars = 2 * kStages + 2 * kSets + 1;  // full/empty, tile full/empty, drain
  static constexpr size_t kSmemBytes =
      1024 + (size_t)kStages * kStageBytes + kStgBytes + kScBytes + kNumBars * 8 + 16;
  static constexpr uint32_t kIdesc = idesc_e4m3_f32(128, BN);
  static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
  static_assert(kStages >= 2, "pipeline needs two stages");
  static_assert(kTmemCols <= 512, "TMEM holds 512 columns");
  static_assert(kSmemBytes <= 232448, "227 KB of shared memory per CTA");
};

// ---------------------------------------------------------------- quantiser
// One warp per (row, 128-column block); lane l holds columns 4l .. 4l + 3.
__global__ void __launch_bounds__(32 * kQuantWarps)
quant_e4m3_kernel(const __nv_bfloat16* __restrict__ a, long long R, int C,
                  uint8_t* __restrict__ q, float* __restrict__ s) {
  pdl_wait();
  pdl_trigger();
  const int KB = (C + 127) / 128;
  const long long wid = (long long)blockIdx.x * kQuantWarps + warp_id();
  if (wid >= R * KB) return;
  const long long r = wid / KB;
  const int b = (int)(wid % KB), lane = lane_id();
  const int c0 = b * 128 + 4 * lane;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (c0 < C) {  // C % 16 == 0: a lane's four columns are all inside or all outside
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(a + r * C + c0));
    v[0] = bf16_lo(raw.x);
    v[1] = bf16_hi(raw.x);
    v[2] = bf16_lo(raw.y);
    v[3] = bf16_hi(raw.y);
  }
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  // non-negative floats order like their bit patterns
  m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
  const float sc = __fdiv_rn(m, 448.f);
  uint32_t packed = 0;
  if (sc > 0.f) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      packed |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(v[j], sc), __NV_SATFINITE, __NV_E4M3)
                << (8 * j);
  }
  if (c0 < C) *reinterpret_cast<uint32_t*>(q + r * C + c0) = packed;
  if (lane == 0) s[r * KB + b] = sc;
}

// ---------------------------------------------------------------- the GEMM
// G1: out = hact [R][N] (N = I), Kdim = H, wa/wb = W1/W3; G2: out = y, wa = W2.
// swa/swb: the weights' block scales [E][ceil(N/128)][ceil(Kdim/128)];
// sact: the activations' scales [R][ceil(Kdim/128)].  items: the plan's tile
// list ({expert, first row, rows, -}, rows <= 128), counts[1] of them.
template <bool G1>
__global__ void __launch_bounds__(kThreads, 1)
w8a8_gemm_kernel(const __grid_constant__ CUtensorMap tm_wa,
                 const __grid_constant__ CUtensorMap tm_wb,
                 const __grid_constant__ CUtensorMap tm_act, const float* __restrict__ swa,
                 const float* __restrict__ swb, const float* __restrict__ sact,
                 const int32_t* __restrict__ counts, const int4* __restrict__ items, int N,
                 int Kdim, int R, __nv_bfloat16* __restrict__ out, int32_t* dev_status) {
  using C = W8Cfg<G1>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint16_t* stg_all = reinterpret_cast<uint16_t*>(smem + (size_t)C::kStages * C::kStageBytes);
  float* sc_all = reinterpret_cast<float*>(smem + (size_t)C::kStages * C::kStageBytes + C::kStgBytes);
  uint8_t* bar_area = smem + (size_t)C::kStages * C::kStageBytes + C::kStgBytes + C::kScBytes;
  const uint32_t bars = smem_u32(bar_area);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (C::kStages + s); };
  auto tfull_bar = [&](int t) { return bars + 8u * (2 * C::kStages + t); };
  auto tempty_bar = [&](int t) { return bars + 8u * (2 * C::kStages + kSets + t); };
  const uint32_t drain_bar = bars + 8u * (2 * C::kStages + 2 * kSets);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t sbase = smem_u32(smem);
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int t = 0; t < kSets; ++t) {
      mbar_init(tfull_bar(t), 1);
      mbar_init(tempty_bar(t), kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_wa);
    if (G1) prefetch_tmap(&tm_wb);
    prefetch_tmap(&tm_act);
  }
  // the plan, the activations and their scales come from earlier launches
  pdl_wait();
  pdl_trigger();
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
  const int nblk = (N + 127) / 128;
  const int KB = (Kdim + 127) / 128;
  constexpr int kHalves = G1 ? 2 : 1;
  const int total = counts[1] * kHalves * nblk;
  struct Unit { int4 it; int nb, row0, m; };
  auto unit_of = [&](int w) {
    Unit u;
    u.it = __ldg(items + w / (kHalves * nblk));
    u.nb = w % nblk;
    const int hf = (w / nblk) % kHalves;
    u.row0 = u.it.y + hf * C::BN;
    const int left = u.it.z - hf * C::BN;
    u.m = left < C::BN ? left : C::BN;  // <= 0: an empty half, skipped by every role
    return u;
  };

  if (warp == 0) {
    // ---------------- TMA producer (one thread)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const Unit u = unit_of(w);
        if (u.m <= 0) continue;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, kWaitNs)) {
            fail();
            ok = false;
            break;
          }
          const uint32_t st = sbase + stage * C::kStageBytes;
          mbar_arrive_expect_tx(full_bar(stage), C::kStageBytes);
          tma_load_3d(st, &tm_wa, full_bar(stage), kb * 128, u.nb * 128, u.it.x);
          if (G1) tma_load_3d(st + C::kABytes, &tm_wb, full_bar(stage), kb * 128, u.nb * 128, u.it.x);
          tma_load_2d(st + C::kNA * C::kABytes, &tm_act, full_bar(stage), kb * 128, u.row0);
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (one thread)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, g = 0;
      bool ok = true, issued = false;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const Unit u = unit_of(w);
        if (u.m <= 0) continue;
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const uint32_t t = g % kSets, tpar = (g / kSets) & 1u;
          if (!mbar_wait_bounded(tempty_bar(t), tpar ^ 1u, abort_flag, kWaitNs) ||
              !mbar_wait_bounded(full_bar(stage), phase, abort_flag, kWaitNs)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + stage * C::kStageBytes;
          const uint32_t sx = st + C::kNA * C::kABytes;
          const uint32_t d = tmem + t * C::kSetCols;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 32 e4m3 = 32 bytes of K per MMA
            const uint64_t bdesc = sdesc_k128_sw128(sx + kk * 32);
            tc_mma_f8(d, sdesc_k128_sw128(st + kk * 32), bdesc, C::kIdesc, kk > 0 ? 1u : 0u);
            if (G1)
              tc_mma_f8(d + C::BN, sdesc_k128_sw128(st + C::kABytes + kk * 32), bdesc, C::kIdesc,
                        kk > 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit(empty_bar(stage));
          tc_commit(tfull_bar(t));
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (issued) {
        // every MMA of this thread completes before TMEM is released
        tc_commit(drain_bar);
        if (!mbar_wait_bounded(drain_bar, 0, nullptr, kWaitNs)) fail();
      }
    }
  } else {
    // ---------------- epilogue warps: TMEM lane quarter = 32 output features;
    // the kEpiWarps / 4 warps of a quarter split the tile's token columns
    const int quarter = warp & 3;
    const int c_off = ((warp - 2) >> 2) * C::kCols;
    uint16_t* stg = stg_all + (warp - 2) * (C::kCols * 32);
    float* sc = sc_all + (warp - 2) * 2 * C::kScPer;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int NB = nblk;
    // a stage's scales: lane j holds the activation scales of columns
    // c_off + j (+ 32 ...), every lane the weight block scale(s); loaded two
    // stages ahead (even and odd stages in their own registers)
    struct Sc { float xs[C::kXs], wa, wb; };
    uint32_t g = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const Unit u = unit_of(w);
      if (u.m <= 0) continue;
      __align__(8) float acc_a[C::kCols];
      __align__(8) float acc_b[G1 ? C::kCols : 2];
#pragma unroll
      for (int j = 0; j < C::kCols; ++j) acc_a[j] = 0.f;
#pragma unroll
      for (int j = 0; j < (G1 ? C::kCols : 2); ++j) acc_b[j] = 0.f;
      const float* sw_a = swa + ((size_t)u.it.x * NB + u.nb) * KB;
      const float* sw_b = G1 ? swb + ((size_t)u.it.x * NB + u.nb) * KB : nullptr;
      bool col_in[C::kXs];
      const float* sx_row[C::kXs];
#pragma unroll
      for (int x = 0; x < C::kXs; ++x) {
        const int col = c_off + 32 * x + lane;
        col_in[x] = 32 * x + lane < C::kCols && col < u.m && u.row0 + col < R;
        sx_row[x] = sact + (size_t)(col_in[x] ? u.row0 + col : 0) * KB;
      }
      auto load = [&](int kb, Sc& v) {
        if (kb < KB) {
          v.wa = __ldg(sw_a + kb);
          v.wb = G1 ? __ldg(sw_b + kb) : 0.f;
#pragma unroll
          for (int x = 0; x < C::kXs; ++x)  // columns past the unit's rows: 0
            v.xs[x] = col_in[x] ? __ldg(sx_row[x] + kb) : 0.f;
        }
      };
      // Stage kb's scale row goes to buffer kb & 1 of sc, so the next stage's
      // row is written while this stage's FMAs still read it.
      auto put_sc = [&](int kb, const Sc& v) {
        float* d = sc + (kb & 1) * C::kScPer;
        __syncwarp();
#pragma unroll
        for (int x = 0; x < C::kXs; ++x) {
          if (32 * x + lane < C::kCols) {
            d[32 * x + lane] = v.xs[x] * v.wa;
            if (G1) d[C::kCols + 32 * x + lane] = v.xs[x] * v.wb;
          }
        }
        __syncwarp();
      };
      // TMEM loads of the 16-column chunk c0 of product tile t (G1: gate and up)
      auto issue = [&](uint32_t t, int c0, uint32_t (&pa)[16], uint32_t (&pb)[16]) {
        const uint32_t ta = t_lane + t * C::kSetCols + c_off + c0;
        tc_ld_32x32b_x16(ta, pa);
        if (G1) tc_ld_32x32b_x16(ta + C::BN, pb);
      };
      // acc += product chunk x its columns' scales (two-wide FMAs)
      auto fma_chunk = [&](const float* sr, int c0, const uint32_t (&pa)[16],
                           const uint32_t (&pb)[16]) {
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const float4 s4 = *reinterpret_cast<const float4*>(sr + c0 + j);
          float2* aa = reinterpret_cast<float2*>(&acc_a[c0 + j]);
          aa[0] = ffma2(make_float2(__uint_as_float(pa[j]), __uint_as_float(pa[j + 1])),
                        make_float2(s4.x, s4.y), aa[0]);
          aa[1] = ffma2(make_float2(__uint_as_float(pa[j + 2]), __uint_as_float(pa[j + 3])),
                        make_float2(s4.z, s4.w), aa[1]);
          if (G1) {
            const float4 u4 = *reinterpret_cast<const float4*>(sr + C::kCols + c0 + j);
            float2* bb = reinterpret_cast<float2*>(&acc_b[c0 + j]);
            bb[0] = ffma2(make_float2(__uint_as_float(pb[j]), __uint_as_float(pb[j + 1])),
                          make_float2(u4.x, u4.y), bb[0]);
            bb[1] = ffma2(make_float2(__uint_as_float(pb[j + 2]), __uint_as_float(pb[j + 3])),
                          make_float2(u4.z, u4.w), bb[1]);
          }
        }
      };
      // Software pipeline over 16-column chunks: each chunk's TMEM load is
      // issued before the previous chunk's FMAs (the first chunk of the next
      // stage included), so the loads' latency hides behind the arithmetic.
      // Even chunks land in (a0, a1), odd ones in (b0, b1).
      constexpr int nC = C::kCols / 16;
      static_assert(nC % 2 == 0, "chunks alternate between two register sets");
      uint32_t a0[16], a1[16], b0[16], b1[16];
      Sc even{}, odd{};
      load(0, even);
      load(1, odd);
      put_sc(0, even);
      if (!mbar_wait_bounded(tfull_bar(g % kSets), (g / kSets) & 1u, abort_flag, kWaitNs)) {
        ok = false;
      } else {
        tc_fence_after();
        issue(g % kSets, 0, a0, a1);
      }
      for (int kb = 0; kb < KB && ok; ++kb, ++g) {
        const uint32_t t = g % kSets;
        const float* sr = sc + (kb & 1) * C::kScPer;
#pragma unroll
        for (int c = 0; c < nC; ++c) {
          tc_wait_ld();  // chunk c is in registers
          if (c == nC - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(t));  // the tile may take a later stage
          }
          if (c + 1 < nC) {
            if ((c + 1) & 1) issue(t, 16 * (c + 1), b0, b1);
            else issue(t, 16 * (c + 1), a0, a1);
          } else if (kb + 1 < KB) {
            put_sc(kb + 1, (kb & 1) ? even : odd);
            const uint32_t g1 = g + 1;
            if (!mbar_wait_bounded(tfull_bar(g1 % kSets), (g1 / kSets) & 1u, abort_flag,
                                   kWaitNs)) {
              ok = false;
            } else {
              tc_fence_after();
              issue(g1 % kSets, 0, a0, a1);
            }
          }
          if (c & 1) fma_chunk(sr, 16 * c, b0, b1);
          else fma_chunk(sr, 16 * c, a0, a1);
        }
        // the struct of this stage's parity is free: stage kb + 2's scales
        if (kb & 1) load(kb + 2, odd);
        else load(kb + 2, even);
      }
      if (!ok) {
        fail();
        break;
      }
      // bf16 rows: feature nb*128 + quarter*32 + lane of tokens row0 + c_off + j
#pragma unroll
      for (int j = 0; j < C::kCols; ++j) {
        const float a = acc_a[j];
        const float v = G1 ? (a / (1.f + __expf(-a))) * acc_b[j] : a;
        stg[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      }
      __syncwarp();
      // kCols token rows x 64 bytes: lane -> (row lane/4 + 8i, 16-byte chunk lane%4)
#pragma unroll
      for (int i = 0; i < C::kCols / 8; ++i) {
        const int r = (lane >> 2) + 8 * i;
        const int cc = c_off + r;
        const int n0 = u.nb * 128 + quarter * 32 + (lane & 3) * 8;
        if (cc < u.m && n0 < N) {
          const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 32 + (lane & 3) * 8);
          *reinterpret_cast<uint4*>(out + (size_t)(u.row0 + cc) * N + n0) = v;
        }
      }
      __syncwarp();
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

// [E][N][Kdim] e4m3 weights, box 128 (K bytes) x 128 rows, 128-byte swizzle
bool w8_weight_map(CUtensorMap* m, const void* w, int E, int N, int Kdim) {
  moe_tmap::EncodeTiledFn enc = moe_tmap::encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)Kdim, (cuuint64_t)N, (cuuint64_t)E};
  cuuint64_t strides[2] = {(cuuint64_t)Kdim, (cuuint64_t)N * Kdim};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(w), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [R][Kdim] e4m3 activations, box 128 (K bytes) x bn rows, 128-byte swizzle
bool w8_act_map(CUtensorMap* m, const void* a, int R, int Kdim, int bn) {
  moe_tmap::EncodeTiledFn enc = moe_tmap::encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)Kdim, (cuuint64_t)R};
  cuuint64_t strides[1] = {(cuuint64_t)Kdim};
  cuuint32_t box[2] = {128, (cuuint32_t)bn};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_quant(const void* a, int R, int C, uint8_t* q, float* s, cudaStream_t stream) {
  const long long warps = (long long)R * ((C + 127) / 128);
  const long long grid = (warps + kQuantWarps - 1) / kQuantWarps;
  return moe_launch(quant_e4m3_kernel, dim3((unsigned)grid), dim3(32 * kQuantWarps), 0, stream, 1,
                    static_cast<const __nv_bfloat16*>(a), (long long)R, C, q, s);
}

template <bool G1>
cudaError_t launch_gemm(const CUtensorMap& wa, const CUtensorMap& wb, const CUtensorMap& act,
                        const float* swa, const float* swb, const float* sact,
                        const int32_t* counts, const int4* items, int N, int Kdim, int R,
                        void* out, int32_t* dev_status, cudaStream_t stream) {
  using C = W8Cfg<G1>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = moe_raise_smem(w8a8_gemm_kernel<G1>, C::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  return moe_launch(w8a8_gemm_kernel<G1>, dim3(moe_num_sms()), dim3(kThreads), C::kSmemBytes,
                    stream, 1, wa, wb, act, swa, swb, sact, counts, items, N, Kdim, R,
                    static_cast<__nv_bfloat16*>(out), dev_status);
}

}  // namespace

size_t w8a8_act_bytes(int R, int H, int I) {
  const size_t r = (size_t)(R > 0 ? R : 0);
  return moe_align_up(r * H, 256) + moe_align_up(r * moe_cdiv(H, 128) * 4, 256) +
         moe_align_up(r * I, 256) + moe_align_up(r * moe_cdiv(I, 128) * 4, 256);
}

cudaError_t launch_w8a8(const void* xp, int R, int E_blocks, int H, int I, const void* w1,
                        const void* w3, const void* w2, const float* s1, const float* s3,
                        const float* s2, void* hact, void* y, const int32_t* counts,
                        const int4* tile_items, void* act_scratch, int32_t* dev_status,
                        cudaStream_t stream) {
  if (R <= 0) return cudaSuccess;
  char* p = static_cast<char*>(act_scratch);
  uint8_t* xq = reinterpret_cast<uint8_t*>(p);
  p += moe_align_up((size_t)R * H, 256);
  float* sx = reinterpret_cast<float*>(p);
  p += moe_align_up((size_t)R * moe_cdiv(H, 128) * 4, 256);
  uint8_t* hq = reinterpret_cast<uint8_t*>(p);
  p += moe_align_up((size_t)R * I, 256);
  float* sh = reinterpret_cast<float*>(p);

  CUtensorMap m_w1, m_w3, m_w2, m_x, m_h;
  if (!w8_weight_map(&m_w1, w1, E_blocks, I, H) || !w8_weight_map(&m_w3, w3, E_blocks, I, H) ||
      !w8_weight_map(&m_w2, w2, E_blocks, H, I) || !w8_act_map(&m_x, xq, R, H, W8Cfg<true>::BN) ||
      !w8_act_map(&m_h, hq, R, I, W8Cfg<false>::BN))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_quant(xp, R, H, xq, sx, stream);
  if (e != cudaSuccess) return e;
  e = launch_gemm<true>(m_w1, m_w3, m_x, s1, s3, sx, counts, tile_items, I, H, R, hact,
                        dev_status, stream);
  if (e != cudaSuccess) return e;
  e = launch_quant(hact, R, I, hq, sh, stream);
  if (e != cudaSuccess) return e;
  return launch_gemm<false>(m_w2, m_w2, m_h, s2, nullptr, sh, counts, tile_items, H, I, R, y,
                            dev_status, stream);
}
