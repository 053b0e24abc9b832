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
//      units of the same launch (all T tokens, weights sw1 / sw3).
//   G2 (gemv_g2_kernel): CTA units of (expert block, 64 output features): the
//      block's hact rows staged in shared memory, each warp streams W2 rows
//      two at a time -> y (bf16); the shared expert's rows likewise ->
//      shared_y.  Then the combine kernel.
// Each warp keeps 16 row vectors per lane in flight (two rows, 8 each) before
// it uses any, so a 2-CTA-per-SM grid holds ~128 KB of weights in flight per
// SM.  Measured and not kept (Qwen3-30B-A3B shape, T = 1, L2 flushed): a G2
// warp per (token, feature) running the token's K picks in turn with the
// combine fused in (K dependent row loads per warp), and feeding the rows by
// bulk copies on the TMA engine into per-warp shared-memory slot rings
// (52.9 us against 38.5).
//
// Weights bf16 or e4m3 with fp32 128 x 128 block scales (the W8A16 format);
// each weight is widened to fp32 exactly and times its block scale.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"

namespace {

constexpr int kWarps = 8;      // per CTA
constexpr int kMaxTok = kGemvMaxT;
constexpr size_t kMaxSmem = 200 * 1024;  // the staged token rows: T * H bf16 at most

MOE_DEVICE float silu(float g) { return g / (1.f + __expf(-g)); }

// 16 e4m3 codes (a 16-byte vector) -> 16 floats times the block scale
MOE_DEVICE void e4m3x16_to_f32(const uint4& v, float s, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
          static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * h)) & 0xFFFFu), __NV_E4M3);
      const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      f[4 * i + 2 * h] = p.x * s;
      f[4 * i + 2 * h + 1] = p.y * s;
    }
  }
}

// Dot products of one or two weight rows (bf16, or e4m3 with block scales;
// `two`: rb/sb too) of length n with up to MT activation rows, lane-strided;
// per-lane partial sums in ga[j] (row a) and gb[j] (row b).  Loads go out in
// batches of 8 vectors per lane and row (16 in flight per lane for two rows)
// before any of them is used.  act(j, e0, a) loads 8 activations of token j
// from element e0.  WQ: 0 bf16 (8 weights per 16-byte vector), 1 e4m3 (16).
template <int WQ, int MT, typename Act>
MOE_DEVICE void row_dots(const void* ra, const void* rb, const float* sa, const float* sb,
                         bool two, int n, int m, Act act, float (&ga)[MT], float (&gb)[MT]) {
  constexpr int kPer = WQ ? 16 : 8;  // weights per 16-byte vector
  constexpr int kB = 8;              // vectors per lane and row in one batch
  const int lane = lane_id();
  const uint4* a4 = static_cast<const uint4*>(ra);
  const uint4* b4 = static_cast<const uint4*>(rb);
  const int nv = n / kPer;
  for (int v0 = lane; v0 < nv; v0 += 32 * kB) {
    uint4 va[kB], vb[kB];
#pragma unroll
    for (int q = 0; q < kB; ++q) {
      const int v = v0 + 32 * q;
      va[q] = v < nv ? __ldcs(a4 + v) : make_uint4(0u, 0u, 0u, 0u);
      vb[q] = (two && v < nv) ? __ldcs(b4 + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < kB; ++q) {
      const int v = v0 + 32 * q;
      if (v >= nv) break;
      float wa[kPer], wb[kPer];
      if (WQ) {
        e4m3x16_to_f32(va[q], __ldg(sa + (kPer * v) / 128), wa);
        if (two) e4m3x16_to_f32(vb[q], __ldg(sb + (kPer * v) / 128), wb);
      } else {
        bf16x8_to_f32(va[q], wa);
        if (two) bf16x8_to_f32(vb[q], wb);
      }
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        if (j < m) {
#pragma unroll
          for (int p = 0; p < kPer; p += 8) {
            float a[8];
            act(j, kPer * v + p, a);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              ga[j] = fmaf(wa[p + c], a[c], ga[j]);
              if (two) gb[j] = fmaf(wb[p + c], a[c], gb[j]);
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
// MT >= the rows of any block (the batch size T).
template <int WQ, int MT>
__global__ void __launch_bounds__(32 * kWarps, 2)
gemv_g1_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, int I, int K,
               const int32_t* __restrict__ counts, const int4* __restrict__ items,
               const int32_t* __restrict__ row_to_flat, const void* __restrict__ w1,
               const void* __restrict__ w3, const float* __restrict__ s1,
               const float* __restrict__ s3, __nv_bfloat16* __restrict__ hact, int Is,
               const __nv_bfloat16* __restrict__ sw1, const __nv_bfloat16* __restrict__ sw3,
               __nv_bfloat16* __restrict__ shared_hact) {
  extern __shared__ uint4 xs[];  // the T token rows, H bf16 each
  pdl_wait();
  pdl_trigger();
  const int H8 = H / 8;
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
  for (int i = threadIdx.x; i < T * H8; i += blockDim.x) xs[i] = __ldg(x4 + i);
  __syncthreads();
  const int lane = lane_id();
  const int n_items = counts[0];
  const long long routed = (long long)n_items * I;
  const long long total = routed + Is;
  const int KBh = (H + 127) / 128, NBi = (I + 127) / 128;
  for (long long u = (long long)blockIdx.x * kWarps + warp_id(); u < total;
       u += (long long)gridDim.x * kWarps) {
    int tok[MT];
    int m, f, e = 0;
    const void *ra, *rb;
    const float *sa = nullptr, *sb = nullptr;
    __nv_bfloat16* dst;
    int ld_dst, row0;
    if (u < routed) {
      const int4 it = __ldg(items + u / I);  // {expert, first row, rows, -}
      f = (int)(u % I);
      e = it.x;
      m = it.z < MT ? it.z : MT;
#pragma unroll
      for (int j = 0; j < MT; ++j) tok[j] = j < m ? __ldg(row_to_flat + it.y + j) / K : 0;
      const size_t row = (size_t)e * I + f;
      ra = WQ ? (const void*)(static_cast<const uint8_t*>(w1) + row * H)
              : (const void*)(static_cast<const __nv_bfloat16*>(w1) + row * H);
      rb = WQ ? (const void*)(static_cast<const uint8_t*>(w3) + row * H)
              : (const void*)(static_cast<const __nv_bfloat16*>(w3) + row * H);
      if (WQ) {
        sa = s1 + ((size_t)e * NBi + f / 128) * KBh;
        sb = s3 + ((size_t)e * NBi + f / 128) * KBh;
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
    float g[MT], up[MT];
#pragma unroll
    for (int j = 0; j < MT; ++j) g[j] = up[j] = 0.f;
    if (WQ && u < routed)
      row_dots<1, MT>(ra, rb, sa, sb, true, H, m, act, g, up);
    else
      row_dots<0, MT>(ra, rb, nullptr, nullptr, true, H, m, act, g, up);
    float hv = 0.f;
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      if (j < m) {  // m is the same in every lane
        const float gs = warp_sum(g[j]), us = warp_sum(up[j]);
        if (lane == j) hv = silu(gs) * us;
      }
    }
    if (lane < m) dst[(size_t)(row0 + lane) * ld_dst + f] = __float2bfloat16_rn(hv);
  }
}

// G2.  CTA units: (expert block, 64 output features) routed, then (64 output
// features) of the shared expert.  The CTA stages the block's hact rows (the
// shared expert: all T shared_hact rows) in shared memory once; each warp
// then streams 8 rows of W2, two at a time, dotted with the staged rows.
constexpr int kG2Rows = 64;
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
    for (int r = warp * 2; r < kG2Rows; r += 2 * kWarps) {
      const int h0 = hb * kG2Rows + r;
      if (h0 >= H) break;
      const bool two = h0 + 1 < H;
      float a0[MT], a1[MT];
#pragma unroll
      for (int j = 0; j < MT; ++j) a0[j] = a1[j] = 0.f;
      if (sh) {
        row_dots<0, MT>(sw2 + (size_t)h0 * Is, sw2 + (size_t)(h0 + (two ? 1 : 0)) * Is, nullptr,
                        nullptr, two, Is, m, act, a0, a1);
      } else if (WQ) {
        const uint8_t* w = static_cast<const uint8_t*>(w2) + ((size_t)it.x * H + h0) * I;
        const float* sr = s2 + ((size_t)it.x * NBh + h0 / 128) * KBi;
        const float* sr1 = s2 + ((size_t)it.x * NBh + (h0 + 1) / 128) * KBi;
        row_dots<1, MT>(w, w + (two ? I : 0), sr, two ? sr1 : sr, two, I, m, act, a0, a1);
      } else {
        const __nv_bfloat16* w =
            static_cast<const __nv_bfloat16*>(w2) + ((size_t)it.x * H + h0) * I;
        row_dots<0, MT>(w, w + (two ? I : 0), nullptr, nullptr, two, I, m, act, a0, a1);
      }
      float v0 = 0.f, v1 = 0.f;
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        if (j < m) {
          const float s0 = warp_sum(a0[j]);
          const float s1 = two ? warp_sum(a1[j]) : 0.f;
          if (lane == j) {
            v0 = s0;
            v1 = s1;
          }
        }
      }
      if (lane < m) {
        dst[(size_t)lane * H + h0] = __float2bfloat16_rn(v0);
        if (two) dst[(size_t)lane * H + h0 + 1] = __float2bfloat16_rn(v1);
      }
    }
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

template <int WQ, int MT>
cudaError_t launch_wq(const GemvArgs& a, cudaStream_t stream) {
  // the limits are raised once, to the largest sizes a call may stage
  static std::atomic<unsigned long long> set1{0}, set2{0};
  cudaError_t e = moe_raise_smem(gemv_g1_kernel<WQ, MT>, kMaxSmem, set1);
  if (e != cudaSuccess) return e;
  e = moe_raise_smem(gemv_g2_kernel<WQ, MT>, kMaxSmem, set2);
  if (e != cudaSuccess) return e;
  const size_t smem1 = (size_t)a.T * a.H * 2;
  e = moe_launch(gemv_g1_kernel<WQ, MT>, dim3(gemv_grid(gemv_g1_kernel<WQ, MT>, smem1)),
                 dim3(32 * kWarps), smem1, stream, 1,
                 static_cast<const __nv_bfloat16*>(a.x), a.T, a.H, a.I, a.K, a.counts, a.items,
                 a.row_to_flat, a.w1, a.w3, a.s1, a.s3, static_cast<__nv_bfloat16*>(a.hact), a.Is,
                 static_cast<const __nv_bfloat16*>(a.sw1), static_cast<const __nv_bfloat16*>(a.sw3),
                 static_cast<__nv_bfloat16*>(a.shared_hact));
  if (e != cudaSuccess) return e;
  const size_t smem2 = (size_t)a.T * (a.I > a.Is ? a.I : a.Is) * 2;
  e = moe_launch(gemv_g2_kernel<WQ, MT>, dim3(gemv_grid(gemv_g2_kernel<WQ, MT>, smem2)),
                 dim3(32 * kWarps), smem2, stream, 1, static_cast<const __nv_bfloat16*>(a.hact),
                 a.T, a.H, a.I, a.counts, a.items, a.w2, a.s2, static_cast<__nv_bfloat16*>(a.y),
                 a.Is, static_cast<const __nv_bfloat16*>(a.shared_hact),
                 static_cast<const __nv_bfloat16*>(a.sw2), static_cast<__nv_bfloat16*>(a.shared_y));
  if (e != cudaSuccess) return e;
  return launch_unpermute(a.y, a.flat_to_row, a.weights, a.T, a.K, a.H,
                          a.Is > 0 ? a.shared_y : nullptr, a.Is > 0 ? a.shared_gate : nullptr,
                          a.out, stream);
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
         (wdtype == MOE_W_BF16 || wdtype == MOE_W_FP8E4M3_B128);
}

cudaError_t launch_gemv_layer(const GemvArgs& a, cudaStream_t stream) {
  if (a.wdtype == MOE_W_FP8E4M3_B128) return launch_t<1>(a, stream);
  return launch_t<0>(a, stream);
}
