// Decode batches (a few tokens) on the CUDA cores: G1 and G2 as matrix-vector
// products.
//
// "vLLM CPU MoE: dynamic GEMM dispatch beyond a fixed threshold" (vllm PR
// #50949), "1. gemm.h": a block of very few rows is not worth a tiled GEMM
// kernel (TinyGEMM there).  With at most four tokens, every weight element is
// used by at most four tokens of its expert: the work is a stream of the
// active experts' weights through HBM, with one FMA per weight and token.
// Tensor-core tiles would pad the token dimension to 16 and split K across
// CTAs to reach every SM, with a cross-CTA reduction after each GEMM; here a
// warp owns whole weight rows instead, so nothing is reduced across warps
// (every warp streams a whole row: many independent rows in flight per SM):
//
//   G1 (gemv_g1_kernel): a warp per (expert block, feature f): streams rows f
//      of W1 and W3 once, dots them with the block's token rows (x, staged in
//      shared memory; the permuted copy xp is not needed) and writes
//      hact = bf16(silu(g) * u).  The shared expert's features are more
//      units of the same launch (all T tokens, weights sw1 / sw3).  Where
//      gemv_routes holds (T * K <= 32; E <= 128, or K <= 16 and E <= 4096/T')
//      the launch before G1 computes only the logits: every G1 CTA routes
//      the batch itself (gemv_route: top-K per token, the stable permutation
//      and the skinny plan in shared memory), which replaces the routing
//      launch's serial tail (completion count, then top-K, permute and plan
//      in its last CTA: ~6 us of a 38 us layer at T = 1, 128 experts; ~10 us
//      at 512 experts).
//   G2 (gemv_g2_kernel): CTA units of (expert block, 64 output features): the
//      block's hact rows staged in shared memory, each warp streams W2 rows
//      four at a time (two for T = 4) -> y (bf16); the shared expert's rows
//      likewise -> shared_y.  At T <= 2 (gemv_g2_t1_kernel, gemv_g2w_kernel)
//      warp units of 4 W2 rows instead, the block's hact rows read with the
//      weights (no staging or barrier; every warp busy: T = 2, GPT-OSS-20B
//      FP8 80.1 -> 71.3 us; T = 1, Qwen3-30B-A3B shape 34.4 ->
//      32.2 us, shared-gate shape 42.6 -> 37.8).  Then the combine kernel.
// Each warp keeps 16 row vectors per lane in flight (G1: two rows, 8 each;
// G2: four rows, 4 each, or two, 8 each) before it uses any, so a
// 2-CTA-per-SM grid holds up to ~128 KB of weights in flight per SM.
//
// Measured and not kept (Qwen3-30B-A3B shape, L2 flushed): a G2 warp per
// (token, feature) running the token's K picks in turn with the combine fused
// in (K dependent row loads per warp), and feeding the rows by bulk copies on
// the TMA engine into per-warp shared-memory slot rings (T = 1: 52.9 us
// against 38.5); bulk L2
// prefetches of each warp's next units' rows (T = 1 38.5 -> 40.6, T = 2
// 53 -> 65); G2 issuing each warp's first W2 batch before the hact staging
// barrier (T = 2 50.9 -> 54.9); G1 fed by a per-lane cp.async ring instead of
// register batches (T = 1 34.3 -> 36.5); the combine folded into the T = 1 G2
// through per-row-group arrival counters (32.4 -> 32.6: a fence and an atomic
// per warp unit cost more than the combine launch); the T = 1 G2 taking the
// plan from a flag G1's CTA 0 sets and sending its first units' W2 rows to L2
// before its grid dependency (30.7 -> 32.7 us); the row batches split into two
// alternating halves, the next requested before the current one is summed
// (T = 1 31.8 -> 32.5, T = 2 51.5 -> 54.2: less in flight at each unit's
// start, and that depth is what this latency-bound path lives on).
//
// Weights bf16, e4m3 with fp32 128 x 128 block scales (the W8A16 format), or
// MXFP4 (e2m1 with a UE8M0 byte per 32 weights of a row): each weight is
// widened to fp32 exactly: the e4m3 code times its block scale, the e2m1
// code times 2^(scale byte - 127) (exact unless it overflows fp32, as a bf16
// weight would).
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"
#include "gemv_route.cuh"
#include "topk_warp.cuh"

namespace {

using moe_gemv_route::gemv_route;
using moe_gemv_route::RouteSmem;

constexpr int kWarps = 8;      // per CTA
static_assert(kWarps == moe_gemv_route::kRouteWarps, "the routing prologue's warps");
constexpr size_t kMaxSmem = 200 * 1024;  // the staged token rows: T * H bf16 at most

MOE_DEVICE float silu(float g) { return g / (1.f + __expf(-g)); }

// A weight vector's scale: the fp32 block scale (e4m3), or 2^(byte - 127)
// of its UE8M0 byte (e2m1)
struct WScale {
  float f;
};

// weights per 16-byte vector: bf16 8, e4m3 16, e2m1 32
template <int WQ>
constexpr int per_vec() { return WQ == 0 ? 8 : WQ == 1 ? 16 : 32; }

// 8 weights (part p of a 16-byte vector) as floats: bf16; e4m3 codes times
// the block scale; e2m1 codes times 2^(scale byte - 127), exact
template <int WQ>
MOE_DEVICE void weights8(const uint4& v, int part, const WScale& sc, float* f) {
  if (WQ == 0) {
    bf16x8_to_f32(v, f);
  } else if (WQ == 1) {
    const uint32_t w[2] = {part ? v.z : v.x, part ? v.w : v.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
            static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * h)) & 0xFFFFu), __NV_E4M3);
        const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        f[4 * i + 2 * h] = p.x * sc.f;
        f[4 * i + 2 * h + 1] = p.y * sc.f;
      }
    }
  } else {
    // byte i holds elements 2i (low nibble) and 2i + 1; each e2m1 value is
    // exact in f16, and times the power of two sc.f exact in fp32
    const uint32_t w = part == 0 ? v.x : part == 1 ? v.y : part == 2 ? v.z : v.w;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2_raw hr = __nv_cvt_fp4x2_to_halfraw2(
          static_cast<__nv_fp4x2_storage_t>((w >> (8 * i)) & 0xFFu), __NV_E2M1);
      const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      f[2 * i] = p.x * sc.f;
      f[2 * i + 1] = p.y * sc.f;
    }
  }
}

// 2^(b - 127) for a UE8M0 scale byte b below 255, as an fp32 (b = 0: the
// subnormal 2^-127)
MOE_DEVICE float ue8m0_to_f32(uint32_t b) {
  return __uint_as_float(b ? b << 23 : 0x00400000u);
}

// Dot products of nr <= NR weight rows (row i at byte r0 + i * rs; bf16;
// e4m3 with its fp32 block-scale row at byte s0 + i * ss, one scale per 128
// weights; e2m1 with its UE8M0 scale row at byte s0 + i * ss, one byte per
// 32 weights) of length n with up to MT activation rows, lane-strided 16-byte
// vectors; per-lane partial sums in acc[i][j] (row i, token j), each summed in
// element order.  Every lane loads KB vectors of each row (NR * KB in flight)
// before it uses any.  act(j, e0, a) loads 8 activations of token j from
// element e0.  WQ: 0 bf16, 1 e4m3, 2 e2m1 (per_vec weights per vector).
template <int WQ, int MT, int NR, int KB, typename Act>
MOE_DEVICE void rows_dot(const void* r0, ptrdiff_t rs, const void* s0, ptrdiff_t ss, int nr,
                         int n, int m, Act act, float (&acc)[NR][MT]) {
  constexpr int kPer = per_vec<WQ>();
  const int lane = lane_id();
  const int nv = n / kPer;
  for (int v0 = lane; v0 < nv; v0 += 32 * KB) {
    uint4 vv[NR][KB];
#pragma unroll
    for (int i = 0; i < NR; ++i) {
#pragma unroll
      for (int q = 0; q < KB; ++q) {
        const int v = v0 + 32 * q;
        const uint4* row = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(r0) + i * rs);
        vv[i][q] = (i < nr && v < nv) ? __ldcs(row + v) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int q = 0; q < KB; ++q) {
      const int v = v0 + 32 * q;
      if (v >= nv) break;
      WScale sc[NR];
#pragma unroll
      for (int i = 0; i < NR; ++i) {
        const uint8_t* srow = static_cast<const uint8_t*>(s0) + i * ss;
        sc[i].f = 1.f;
        if (WQ == 1 && i < nr) sc[i].f = __ldg(reinterpret_cast<const float*>(srow) + (kPer * v) / 128);
        if (WQ == 2 && i < nr) sc[i].f = ue8m0_to_f32(__ldg(srow + v));
      }
      if constexpr (NR <= 2 && kPer <= 16) {
        // the rows' weights once, each token's activations once per 8
        float w[NR][kPer];
#pragma unroll
        for (int i = 0; i < NR; ++i)
#pragma unroll
          for (int p = 0; p < kPer; p += 8)
            if (i < nr) weights8<WQ>(vv[i][q], p / 8, sc[i], &w[i][p]);
#pragma unroll
        for (int j = 0; j < MT; ++j) {
          if (j < m) {
#pragma unroll
            for (int p = 0; p < kPer; p += 8) {
              float a[8];
              act(j, kPer * v + p, a);
#pragma unroll
              for (int i = 0; i < NR; ++i) {
                if (i < nr) {
#pragma unroll
                  for (int c = 0; c < 8; ++c) acc[i][j] = fmaf(w[i][p + c], a[c], acc[i][j]);
                }
              }
            }
          }
        }
      } else {
        // four rows, or e2m1: every token's 8 activations once, each row's
        // 8 weights once per 8
#pragma unroll
        for (int p = 0; p < kPer; p += 8) {
          float a[MT][8];
#pragma unroll
          for (int j = 0; j < MT; ++j)
            if (j < m) act(j, kPer * v + p, a[j]);
#pragma unroll
          for (int i = 0; i < NR; ++i) {
            if (i < nr) {
              float w[8];
              weights8<WQ>(vv[i][q], p / 8, sc[i], w);
#pragma unroll
              for (int j = 0; j < MT; ++j) {
                if (j < m) {
#pragma unroll
                  for (int c = 0; c < 8; ++c) acc[i][j] = fmaf(w[c], a[j][c], acc[i][j]);
                }
              }
            }
          }
        }
      }
    }
  }
}

// sum over the warp, the same value (lane 0's) in every lane
MOE_DEVICE float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return __shfl_sync(0xffffffffu, v, 0);
}

// G1.  units: n_items * I routed (items = the plan's skinny list) + Is shared;
// MT >= the rows of any block (the batch size T).  kRoute: the CTA routes the
// batch first (gemv_route) and takes items and rows from that.
template <int WQ, int MT, bool kRoute>
__global__ void __launch_bounds__(32 * kWarps, 2)
gemv_g1_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, int I, int K,
               const int32_t* __restrict__ counts, const int4* __restrict__ items,
               const int32_t* __restrict__ row_to_flat, const void* __restrict__ w1,
               const void* __restrict__ w3, const float* __restrict__ s1,
               const float* __restrict__ s3, __nv_bfloat16* __restrict__ hact, int Is,
               const __nv_bfloat16* __restrict__ sw1, const __nv_bfloat16* __restrict__ sw3,
               __nv_bfloat16* __restrict__ shared_hact, int wdtype, GemvRoute rt) {
  extern __shared__ uint4 xs[];  // the T token rows, H bf16 each
  __shared__ RouteSmem rs;
  pdl_wait();
  pdl_trigger();
  const int H8 = H / 8;
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
  // threads from.. copy the token rows, four 16-byte loads in flight each
  auto stage = [&](int from) {
    const int n = T * H8, nt = (int)blockDim.x - from;
    for (int i = (int)threadIdx.x - from; i >= 0 && i < n; i += 4 * nt) {
      uint4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = i + k * nt < n ? __ldg(x4 + i + k * nt) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (i + k * nt < n) xs[i + k * nt] = v[k];
    }
  };
  if (kRoute)
    gemv_route(rt, T, K, wdtype, rs, stage);  // stages the rows beside the routing
  else
    stage(0);
  __syncthreads();
  const int lane = lane_id();
  const int n_items = kRoute ? rs.n_items : counts[0];
  const long long routed = (long long)n_items * I;
  const long long total = routed + Is;
  const int KBh = (H + 127) / 128, NBi = (I + 127) / 128;
  for (long long u = (long long)blockIdx.x * kWarps + warp_id(); u < total;
       u += (long long)gridDim.x * kWarps) {
    int tok[MT];
    int m, f, e = 0;
    const void *ra, *rb;
    const uint8_t *sa = nullptr, *sb = nullptr;  // the rows' scales (bytes)
    __nv_bfloat16* dst;
    int ld_dst, row0;
    if (u < routed) {
      // {expert, first row, rows, -}
      const int4 it = kRoute ? rs.items[u / I] : __ldg(items + u / I);
      f = (int)(u % I);
      e = it.x;
      m = it.z < MT ? it.z : MT;
#pragma unroll
      for (int j = 0; j < MT; ++j)
        tok[j] = j < m ? (kRoute ? rs.r2f[it.y + j] : __ldg(row_to_flat + it.y + j)) / K : 0;
      const size_t row = (size_t)e * I + f;
      const size_t wrow = (size_t)H * 16 / per_vec<WQ>();  // bytes of a weight row
      ra = static_cast<const uint8_t*>(w1) + row * wrow;
      rb = static_cast<const uint8_t*>(w3) + row * wrow;
      if (WQ == 1) {  // fp32 128 x 128 block scales
        sa = reinterpret_cast<const uint8_t*>(s1 + ((size_t)e * NBi + f / 128) * KBh);
        sb = reinterpret_cast<const uint8_t*>(s3 + ((size_t)e * NBi + f / 128) * KBh);
      } else if (WQ == 2) {  // a UE8M0 byte per 32 weights of the row
        sa = reinterpret_cast<const uint8_t*>(s1) + row * (H / 32);
        sb = reinterpret_cast<const uint8_t*>(s3) + row * (H / 32);
      }
      dst = hact;
      ld_dst = I;
      row0 = it.y;
    } else {
      f = (int)(u - routed);
      m = T;
#pragma unroll
      for (int j = 0; j < MT; ++j) tok[j] = j;
      ra = sw1 + (size_t)f * H;
      rb = sw3 + (size_t)f * H;
      dst = shared_hact;
      ld_dst = Is;
      row0 = 0;
    }
    auto act = [&](int j, int e0, float* a) {
      bf16x8_to_f32(xs[(tok[j] * H + e0) / 8], a);
    };
    float acc[2][MT];  // gate (W1) and up (W3) partial sums per token
#pragma unroll
    for (int j = 0; j < MT; ++j) acc[0][j] = acc[1][j] = 0.f;
    // row b and its scales at a fixed distance from row a
    const ptrdiff_t rs = static_cast<const uint8_t*>(rb) - static_cast<const uint8_t*>(ra);
    if (WQ && u < routed)
      rows_dot<WQ, MT, 2, 8>(ra, rs, sa, sb - sa, 2, H, m, act, acc);
    else
      rows_dot<0, MT, 2, 8>(ra, rs, nullptr, 0, 2, H, m, act, acc);
    float hv = 0.f;
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      if (j < m) {  // m is the same in every lane
        const float gs = warp_sum(acc[0][j]), us = warp_sum(acc[1][j]);
        if (lane == j) hv = silu(gs) * us;
      }
    }
    if (lane < m) dst[(size_t)(row0 + lane) * ld_dst + f] = __float2bfloat16_rn(hv);
  }
}

// G2.  CTA units: (expert block, 64 output features) routed, then (64 output
// features) of the shared expert.  The CTA stages the block's hact rows (the
// shared expert: all T shared_hact rows) in shared memory once; each warp
// then streams 8 rows of W2, four at a time (two for four tokens), dotted
// with the staged rows.
constexpr int kG2Rows = 64;
// W2 rows a warp streams at once, and vectors per lane and row in a batch
// (16 in flight per lane); four tokens keep two rows (registers)
template <int MT>
constexpr int g2_per() { return MT <= 2 ? 4 : 2; }
template <int WQ, int MT>
__global__ void __launch_bounds__(32 * kWarps, 2)
gemv_g2_kernel(const __nv_bfloat16* __restrict__ hact, int T, int H, int I,
               const int32_t* __restrict__ counts, const int4* __restrict__ items,
               const void* __restrict__ w2, const float* __restrict__ s2,
               __nv_bfloat16* __restrict__ y, int Is, const __nv_bfloat16* __restrict__ shared_hact,
               const __nv_bfloat16* __restrict__ sw2, __nv_bfloat16* __restrict__ shared_y) {
  extern __shared__ uint4 hs[];  // up to MT rows of n (I or Is) bf16
  pdl_wait();
  pdl_trigger();
  const int lane = lane_id(), warp = warp_id();
  const int nhb = (H + kG2Rows - 1) / kG2Rows;
  const int routed = counts[0] * nhb;
  const int total = routed + (Is > 0 ? nhb : 0);
  const int KBi = (I + 127) / 128, NBh = (H + 127) / 128;
  for (int u = blockIdx.x; u < total; u += gridDim.x) {
    const bool sh = u >= routed;
    const int hb = sh ? u - routed : u % nhb;
    int4 it = make_int4(0, 0, T, 0);
    if (!sh) it = __ldg(items + u / nhb);  // {expert, first row, rows, -}
    const int m = it.z < MT ? it.z : MT;
    const int n = sh ? Is : I;
    const __nv_bfloat16* src = sh ? shared_hact : hact + (size_t)it.y * I;
    __syncthreads();  // the previous unit's rows are no longer read
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    for (int i = threadIdx.x; i < m * n / 8; i += blockDim.x) hs[i] = __ldg(s4 + i);
    __syncthreads();
    auto act = [&](int j, int e0, float* a) { bf16x8_to_f32(hs[(j * n + e0) / 8], a); };
    __nv_bfloat16* dst = sh ? shared_y : y + (size_t)it.y * H;
    constexpr int kG2Per = g2_per<MT>(), kG2Batch = 16 / kG2Per;
    for (int r = warp * kG2Per; r < kG2Rows; r += kG2Per * kWarps) {
      const int h0 = hb * kG2Rows + r;
      if (h0 >= H) break;
      const int nr = H - h0 < kG2Per ? H - h0 : kG2Per;  // the same in every lane
      // nr consecutive rows h0.. (h0 % 4 == 0: e4m3, one 128-row scale
      // block; e2m1, a scale row per weight row)
      const void* r0;
      ptrdiff_t rs, ss = 0;
      const void* s0 = nullptr;
      if (sh) {
        r0 = sw2 + (size_t)h0 * Is;
        rs = (ptrdiff_t)Is * 2;
      } else if (WQ == 1) {
        r0 = static_cast<const uint8_t*>(w2) + ((size_t)it.x * H + h0) * I;
        rs = I;
        s0 = s2 + ((size_t)it.x * NBh + h0 / 128) * KBi;
      } else if (WQ == 2) {
        r0 = static_cast<const uint8_t*>(w2) + ((size_t)it.x * H + h0) * (I / 2);
        rs = I / 2;
        s0 = reinterpret_cast<const uint8_t*>(s2) + ((size_t)it.x * H + h0) * (I / 32);
        ss = I / 32;
      } else {
        r0 = static_cast<const __nv_bfloat16*>(w2) + ((size_t)it.x * H + h0) * I;
        rs = (ptrdiff_t)I * 2;
      }
      float acc[kG2Per][MT];
#pragma unroll
      for (int i = 0; i < kG2Per; ++i)
#pragma unroll
        for (int j = 0; j < MT; ++j) acc[i][j] = 0.f;
      if (sh)
        rows_dot<0, MT, kG2Per, kG2Batch>(r0, rs, nullptr, 0, nr, Is, m, act, acc);
      else
        rows_dot<WQ, MT, kG2Per, kG2Batch>(r0, rs, s0, ss, nr, I, m, act, acc);
      float v[kG2Per];
#pragma unroll
      for (int i = 0; i < kG2Per; ++i) {
        v[i] = 0.f;
#pragma unroll
        for (int j = 0; j < MT; ++j) {
          if (i < nr && j < m) {
            const float sum = warp_sum(acc[i][j]);
            if (lane == j) v[i] = sum;
          }
        }
      }
      if (lane < m) {
#pragma unroll
        for (int i = 0; i < kG2Per; ++i)
          if (i < nr) dst[(size_t)lane * H + h0 + i] = __float2bfloat16_rn(v[i]);
      }
    }
  }
}

// G2 for one token (T = 1; every expert block is one row): warp units of 4
// consecutive W2 rows of a block (then of the shared expert).  Each lane
// loads its vectors of the 4 rows and the matching vectors of the block's
// hact row together (no staging, no barrier), KB per row in flight; the sums
// run in the element order of gemv_g2_kernel.
template <int WQ>
__global__ void __launch_bounds__(32 * kWarps, 2)
gemv_g2_t1_kernel(const __nv_bfloat16* __restrict__ hact, int H, int I,
                  const int32_t* __restrict__ counts, const int4* __restrict__ items,
                  const void* __restrict__ w2, const float* __restrict__ s2,
                  __nv_bfloat16* __restrict__ y, int Is,
                  const __nv_bfloat16* __restrict__ shared_hact,
                  const __nv_bfloat16* __restrict__ sw2, __nv_bfloat16* __restrict__ shared_y) {
  constexpr int kRows = 4;
  constexpr int kPerR = per_vec<WQ>();
  pdl_wait();
  pdl_trigger();
  const int lane = lane_id();
  const int ng = H / kRows;  // row groups per block
  const long long routed = (long long)counts[0] * ng;
  const long long total = routed + (Is > 0 ? ng : 0);
  const int KBi = (I + 127) / 128, NBh = (H + 127) / 128;
  for (long long u = (long long)blockIdx.x * kWarps + warp_id(); u < total;
       u += (long long)gridDim.x * kWarps) {
    const bool sh = u >= routed;
    const int h0 = kRows * (int)(sh ? u - routed : u % ng);
    float acc[kRows] = {0.f, 0.f, 0.f, 0.f};
    __nv_bfloat16* dst;
    if (sh) {
      // bf16 rows of Is, the shared expert's hact row
      const int nv = Is / 8;
      const uint4* hrow = reinterpret_cast<const uint4*>(shared_hact);
      for (int v0 = lane; v0 < nv; v0 += 32 * 4) {
        uint4 vv[kRows][4], hv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int v = v0 + 32 * q;
          hv[q] = v < nv ? __ldg(hrow + v) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int i = 0; i < kRows; ++i)
            vv[i][q] = v < nv ? __ldcs(reinterpret_cast<const uint4*>(sw2 + (size_t)(h0 + i) * Is) + v)
                              : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (v0 + 32 * q >= nv) break;
          float a[8];
          bf16x8_to_f32(hv[q], a);
#pragma unroll
          for (int i = 0; i < kRows; ++i) {
            float w[8];
            bf16x8_to_f32(vv[i][q], w);
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[i] = fmaf(w[c], a[c], acc[i]);
          }
        }
      }
      dst = shared_y;
    } else {
      const int4 it = __ldg(items + u / ng);  // {expert, first row, rows = 1, -}
      const size_t rowb = (size_t)I * 16 / kPerR;  // bytes of a W2 row
      const uint8_t* r0 = static_cast<const uint8_t*>(w2) + ((size_t)it.x * H + h0) * rowb;
      const uint4* hrow = reinterpret_cast<const uint4*>(hact + (size_t)it.y * I);
      const int nv = I / kPerR;
      constexpr int KB = WQ == 2 ? 2 : 4;  // weight vectors per lane and row in a batch
      for (int v0 = lane; v0 < nv; v0 += 32 * KB) {
        uint4 vv[kRows][KB], hv[KB][kPerR / 8];
#pragma unroll
        for (int q = 0; q < KB; ++q) {
          const int v = v0 + 32 * q;
#pragma unroll
          for (int p = 0; p < kPerR / 8; ++p)
            hv[q][p] = v < nv ? __ldg(hrow + (size_t)v * (kPerR / 8) + p) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int i = 0; i < kRows; ++i)
            vv[i][q] = v < nv ? __ldcs(reinterpret_cast<const uint4*>(r0 + i * rowb) + v)
                              : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < KB; ++q) {
          const int v = v0 + 32 * q;
          if (v >= nv) break;
          WScale sc[kRows];
#pragma unroll
          for (int i = 0; i < kRows; ++i) {
            sc[i].f = 1.f;
            if (WQ == 1)  // h0 % 4 == 0: the 4 rows share a 128-row scale block
              sc[i].f = __ldg(s2 + ((size_t)it.x * NBh + h0 / 128) * KBi + (16 * v) / 128);
            if (WQ == 2)
              sc[i].f = ue8m0_to_f32(__ldg(reinterpret_cast<const uint8_t*>(s2) +
                                           ((size_t)it.x * H + h0 + i) * (I / 32) + v));
          }
#pragma unroll
          for (int p = 0; p < kPerR; p += 8) {
            float a[8];
            bf16x8_to_f32(hv[q][p / 8], a);
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
              float w[8];
              weights8<WQ>(vv[i][q], p / 8, sc[i], w);
#pragma unroll
              for (int c = 0; c < 8; ++c) acc[i] = fmaf(w[c], a[c], acc[i]);
            }
          }
        }
      }
      dst = y + (size_t)it.y * H;
    }
    float out = 0.f;
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const float sum = warp_sum(acc[i]);
      if (lane == i) out = sum;
    }
    if (lane < kRows) dst[h0 + lane] = __float2bfloat16_rn(out);
  }
}

// G2 for two tokens (MT = 2; an expert block has one or two rows): the
// T = 1 kernel's warp units of 4 consecutive W2 rows with up to MT hact rows
// per block (the one-token instance measured ~2 us slower than the kernel
// above at the Qwen3-30B-A3B shape, so T = 1 keeps its own).  Each lane loads its vectors of the 4 rows and the matching
// vectors of the block's hact rows together (no staging, no barrier), KB per
// row in flight; the sums run in the element order of gemv_g2_kernel.
template <int WQ, int MT>
constexpr int g2w_batch() {
  // hact registers grow with the tokens and the weights per vector
  return (per_vec<WQ>() / 8) * MT <= 2 ? 4 : ((per_vec<WQ>() / 8) * MT <= 4 ? 2 : 1);
}

template <int WQ, int MT>
__global__ void __launch_bounds__(32 * kWarps, 2)
gemv_g2w_kernel(const __nv_bfloat16* __restrict__ hact, int T, int H, int I,
                const int32_t* __restrict__ counts, const int4* __restrict__ items,
                const void* __restrict__ w2, const float* __restrict__ s2,
                __nv_bfloat16* __restrict__ y, int Is,
                const __nv_bfloat16* __restrict__ shared_hact,
                const __nv_bfloat16* __restrict__ sw2, __nv_bfloat16* __restrict__ shared_y) {
  constexpr int kRows = 4;
  constexpr int kPerR = per_vec<WQ>();
  pdl_wait();
  pdl_trigger();
  const int lane = lane_id();
  const int ng = H / kRows;  // row groups per block
  const long long routed = (long long)counts[0] * ng;
  const long long total = routed + (Is > 0 ? ng : 0);
  const int KBi = (I + 127) / 128, NBh = (H + 127) / 128;
  for (long long u = (long long)blockIdx.x * kWarps + warp_id(); u < total;
       u += (long long)gridDim.x * kWarps) {
    const bool sh = u >= routed;
    const int h0 = kRows * (int)(sh ? u - routed : u % ng);
    float acc[kRows][MT];
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < MT; ++j) acc[i][j] = 0.f;
    __nv_bfloat16* dst;
    int m;
    if (sh) {
      // bf16 rows of Is, the shared expert's hact rows (all T tokens)
      m = T < MT ? T : MT;
      const int nv = Is / 8;
      for (int v0 = lane; v0 < nv; v0 += 32 * 4) {
        uint4 vv[kRows][4], hv[4][MT];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int v = v0 + 32 * q;
#pragma unroll
          for (int j = 0; j < MT; ++j)
            hv[q][j] = (v < nv && j < m)
                           ? __ldg(reinterpret_cast<const uint4*>(shared_hact + (size_t)j * Is) + v)
                           : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int i = 0; i < kRows; ++i)
            vv[i][q] = v < nv ? __ldcs(reinterpret_cast<const uint4*>(sw2 + (size_t)(h0 + i) * Is) + v)
                              : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (v0 + 32 * q >= nv) break;
          float a[MT][8];
#pragma unroll
          for (int j = 0; j < MT; ++j) bf16x8_to_f32(hv[q][j], a[j]);
#pragma unroll
          for (int i = 0; i < kRows; ++i) {
            float w[8];
            bf16x8_to_f32(vv[i][q], w);
#pragma unroll
            for (int j = 0; j < MT; ++j)
              if (j < m) {
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[i][j] = fmaf(w[c], a[j][c], acc[i][j]);
              }
          }
        }
      }
      dst = shared_y;
    } else {
      const int4 it = __ldg(items + u / ng);  // {expert, first row, rows, -}
      m = it.z < MT ? it.z : MT;
      const size_t rowb = (size_t)I * 16 / kPerR;  // bytes of a W2 row
      const uint8_t* r0 = static_cast<const uint8_t*>(w2) + ((size_t)it.x * H + h0) * rowb;
      const uint4* hrow = reinterpret_cast<const uint4*>(hact + (size_t)it.y * I);
      const int nv = I / kPerR, hstride = I / 8;  // hact row stride in 16-byte vectors
      constexpr int KB = g2w_batch<WQ, MT>();  // weight vectors per lane and row in a batch
      for (int v0 = lane; v0 < nv; v0 += 32 * KB) {
        uint4 vv[kRows][KB], hv[KB][kPerR / 8][MT];
#pragma unroll
        for (int q = 0; q < KB; ++q) {
          const int v = v0 + 32 * q;
#pragma unroll
          for (int p = 0; p < kPerR / 8; ++p)
#pragma unroll
            for (int j = 0; j < MT; ++j)
              hv[q][p][j] = (v < nv && j < m)
                                ? __ldg(hrow + (size_t)j * hstride + (size_t)v * (kPerR / 8) + p)
                                : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int i = 0; i < kRows; ++i)
            vv[i][q] = v < nv ? __ldcs(reinterpret_cast<const uint4*>(r0 + i * rowb) + v)
                              : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < KB; ++q) {
          const int v = v0 + 32 * q;
          if (v >= nv) break;
          WScale sc[kRows];
#pragma unroll
          for (int i = 0; i < kRows; ++i) {
            sc[i].f = 1.f;
            if (WQ == 1)  // h0 % 4 == 0: the 4 rows share a 128-row scale block
              sc[i].f = __ldg(s2 + ((size_t)it.x * NBh + h0 / 128) * KBi + (16 * v) / 128);
            if (WQ == 2)
              sc[i].f = ue8m0_to_f32(__ldg(reinterpret_cast<const uint8_t*>(s2) +
                                           ((size_t)it.x * H + h0 + i) * (I / 32) + v));
          }
#pragma unroll
          for (int p = 0; p < kPerR; p += 8) {
            float a[MT][8];
#pragma unroll
            for (int j = 0; j < MT; ++j) bf16x8_to_f32(hv[q][p / 8][j], a[j]);
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
              float w[8];
              weights8<WQ>(vv[i][q], p / 8, sc[i], w);
#pragma unroll
              for (int j = 0; j < MT; ++j)
                if (j < m) {
#pragma unroll
                  for (int c = 0; c < 8; ++c) acc[i][j] = fmaf(w[c], a[j][c], acc[i][j]);
                }
            }
          }
        }
      }
      dst = y + (size_t)it.y * H;
    }
    // lane i + 4 j: row h0 + i of token j
    float out = 0.f;
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        if (j < m) {
          const float sum = warp_sum(acc[i][j]);
          if (lane == i + kRows * j) out = sum;
        }
      }
    if (lane < kRows * m) dst[(size_t)(lane / kRows) * H + h0 + lane % kRows] = __float2bfloat16_rn(out);
  }
}

// CTAs that stay resident together (a grid-stride loop shares the units):
// the kernel's occupancy at this shared-memory size, cached per device for
// the last size asked
template <typename Kern>
int gemv_grid(Kern kernel, size_t smem) {
  static std::atomic<unsigned long long> last[64];  // smem << 8 | CTAs per SM
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  const unsigned long long c = last[dev].load(std::memory_order_relaxed);
  int per_sm = (c >> 8) == smem ? (int)(c & 0xFF) : 0;
  if (!per_sm) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 32 * kWarps, smem) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    if (per_sm > 255) per_sm = 255;
    last[dev].store(((unsigned long long)smem << 8) | (unsigned)per_sm, std::memory_order_relaxed);
  }
  return moe_num_sms() * per_sm;
}

template <int WQ, int MT, bool kRoute>
cudaError_t launch_g1(const GemvArgs& a, cudaStream_t stream) {
  // the limit is raised once, to the largest size a call may stage
  static std::atomic<unsigned long long> set{0};
  const cudaError_t e = moe_raise_smem(gemv_g1_kernel<WQ, MT, kRoute>, kMaxSmem, set);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)a.T * a.H * 2;
  return moe_launch(gemv_g1_kernel<WQ, MT, kRoute>,
                    dim3(gemv_grid(gemv_g1_kernel<WQ, MT, kRoute>, smem)), dim3(32 * kWarps), smem,
                    stream, 1, static_cast<const __nv_bfloat16*>(a.x), a.T, a.H, a.I, a.K,
                    a.counts, a.items, a.row_to_flat, a.w1, a.w3, a.s1, a.s3,
                    static_cast<__nv_bfloat16*>(a.hact), a.Is,
                    static_cast<const __nv_bfloat16*>(a.sw1),
                    static_cast<const __nv_bfloat16*>(a.sw3),
                    static_cast<__nv_bfloat16*>(a.shared_hact), a.wdtype, a.rt);
}

template <int WQ, int MT>
cudaError_t launch_wq(const GemvArgs& a, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if constexpr (MT > 2) {
    // the limit is raised once, to the largest size a call may stage
    static std::atomic<unsigned long long> set2{0};
    e = moe_raise_smem(gemv_g2_kernel<WQ, MT>, kMaxSmem, set2);
    if (e != cudaSuccess) return e;
  }
  e = a.route ? launch_g1<WQ, MT, true>(a, stream) : launch_g1<WQ, MT, false>(a, stream);
  if (e != cudaSuccess) return e;
  if constexpr (MT <= 2) {
    // one or two tokens: warp units of 4 W2 rows, hact read with the weights
    if constexpr (MT == 1)
      e = moe_launch(gemv_g2_t1_kernel<WQ>, dim3(gemv_grid(gemv_g2_t1_kernel<WQ>, 0)),
                     dim3(32 * kWarps), 0, stream, 1, static_cast<const __nv_bfloat16*>(a.hact),
                     a.H, a.I, a.counts, a.items, a.w2, a.s2, static_cast<__nv_bfloat16*>(a.y),
                     a.Is, static_cast<const __nv_bfloat16*>(a.shared_hact),
                     static_cast<const __nv_bfloat16*>(a.sw2),
                     static_cast<__nv_bfloat16*>(a.shared_y));
    else
      e = moe_launch(gemv_g2w_kernel<WQ, MT>, dim3(gemv_grid(gemv_g2w_kernel<WQ, MT>, 0)),
                     dim3(32 * kWarps), 0, stream, 1, static_cast<const __nv_bfloat16*>(a.hact),
                     a.T, a.H, a.I, a.counts, a.items, a.w2, a.s2,
                     static_cast<__nv_bfloat16*>(a.y), a.Is,
                     static_cast<const __nv_bfloat16*>(a.shared_hact),
                     static_cast<const __nv_bfloat16*>(a.sw2),
                     static_cast<__nv_bfloat16*>(a.shared_y));
    if (e != cudaSuccess) return e;
    return launch_unpermute(a.y, a.flat_to_row, a.weights, a.T, a.K, a.H,
                            a.Is > 0 ? a.shared_y : nullptr, a.Is > 0 ? a.shared_gate : nullptr,
                            a.out, stream);
  } else {
    const size_t smem2 = (size_t)a.T * (a.I > a.Is ? a.I : a.Is) * 2;
    e = moe_launch(gemv_g2_kernel<WQ, MT>, dim3(gemv_grid(gemv_g2_kernel<WQ, MT>, smem2)),
                   dim3(32 * kWarps), smem2, stream, 1, static_cast<const __nv_bfloat16*>(a.hact),
                   a.T, a.H, a.I, a.counts, a.items, a.w2, a.s2, static_cast<__nv_bfloat16*>(a.y),
                   a.Is, static_cast<const __nv_bfloat16*>(a.shared_hact),
                   static_cast<const __nv_bfloat16*>(a.sw2),
                   static_cast<__nv_bfloat16*>(a.shared_y));
    if (e != cudaSuccess) return e;
    return launch_unpermute(a.y, a.flat_to_row, a.weights, a.T, a.K, a.H,
                            a.Is > 0 ? a.shared_y : nullptr, a.Is > 0 ? a.shared_gate : nullptr,
                            a.out, stream);
  }
}

template <int WQ>
cudaError_t launch_t(const GemvArgs& a, cudaStream_t stream) {
  if (a.T == 1) return launch_wq<WQ, 1>(a, stream);
  if (a.T == 2) return launch_wq<WQ, 2>(a, stream);
  return launch_wq<WQ, 4>(a, stream);
}

}  // namespace

bool gemv_supported(int T, int H, int I, int Is, int wdtype, int m_skinny) {
  const int n = I > Is ? I : Is;
  return T >= 1 && T <= kGemvMaxT && T <= m_skinny && (size_t)T * H * 2 <= kMaxSmem &&
         (size_t)T * n * 2 <= kMaxSmem &&
         (wdtype == MOE_W_BF16 || wdtype == MOE_W_FP8E4M3_B128 || wdtype == MOE_W_MXFP4);
}

bool gemv_routes(int T, int E, int K) {
  if (T < 1 || T > kGemvMaxT || E < 1 || K < 1 || T * K > 32) return false;
  if (E <= 128) return true;
  // slices of 16 candidates per lane, picks of at most 16 per slice
  const int slices = kWarps / (T == 1 ? 1 : T == 2 ? 2 : 4);
  return K <= 16 && E <= 32 * 16 * slices;
}

cudaError_t launch_gemv_layer(const GemvArgs& a, cudaStream_t stream) {
  if (a.route && !gemv_routes(a.T, a.rt.E, a.K)) return cudaErrorInvalidValue;
  if (a.wdtype == MOE_W_FP8E4M3_B128) return launch_t<1>(a, stream);
  if (a.wdtype == MOE_W_MXFP4) return launch_t<2>(a, stream);
  return launch_t<0>(a, stream);
}
