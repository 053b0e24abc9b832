// R: router (gate) GEMM, logits[t, g] = sum_h fp32(x[t, h]) * wg[g, h] (+ bias[g]).
//
// "vLLM MiniMax-M2 MoE gate optimisation: fused FP32 kernel" (vllm PR #38445),
// "2. CUDA kernel": instead of casting the bf16 hidden states to an fp32 copy
// and running an fp32 GEMM (up to three kernels), one kernel loads 8 bf16 at a
// time as one 16-byte vector, widens them to fp32 in registers and feeds the
// fp32 dot products directly.  The accumulation is fp32 on the CUDA cores:
// the gate must stay in fp32 precision, so tensor cores (tf32) are not used.
//
// Two kernels:
//  * decode (T <= 16): bound by reading wg once (4*G*H bytes).  A CTA owns ROWS
//    gate rows; its 256 threads split H in 8-element chunks, accumulate all
//    tokens of an 8-token group, and reduce across the block in a fixed tree.
//  * prefill (T > 16): FP32-FMA bound (2*T*G*H flops).  A 64x64 output tile per
//    CTA, bf16 tile widened while it is staged into shared memory, 4x4
//    register micro-tile per thread.
// Both are deterministic: the order of the sums depends only on the sizes.
#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kSmallThreads = 256;
constexpr int kSmallTok = 8;

template <int ROWS>
__global__ void __launch_bounds__(kSmallThreads)
router_small_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ wg,
                    const float* __restrict__ bias, float* __restrict__ logits, int T, int H,
                    int G) {
  __shared__ float red[kSmallThreads / 32][ROWS * kSmallTok];
  const int g0 = blockIdx.x * ROWS;
  const int tid = threadIdx.x;
  for (int t0 = 0; t0 < T; t0 += kSmallTok) {
    float acc[ROWS][kSmallTok];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
      for (int j = 0; j < kSmallTok; ++j) acc[r][j] = 0.f;

    for (int h = tid * 8; h < H; h += kSmallThreads * 8) {
      float w[ROWS][8];
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        if (g0 + r < G) {
          const float4* p = reinterpret_cast<const float4*>(wg + (size_t)(g0 + r) * H + h);
          float4 a = __ldg(p), b = __ldg(p + 1);
          w[r][0] = a.x; w[r][1] = a.y; w[r][2] = a.z; w[r][3] = a.w;
          w[r][4] = b.x; w[r][5] = b.y; w[r][6] = b.z; w[r][7] = b.w;
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) w[r][i] = 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < kSmallTok; ++j) {
        if (t0 + j < T) {
          uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + j) * H + h));
          float xf[8];
          bf16x8_to_f32(v, xf);
#pragma unroll
          for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[r][j] = fmaf(w[r][i], xf[i], acc[r][j]);
        }
      }
    }
    // block reduction, fixed order: butterfly inside the warp, then warps 0..7
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
      for (int j = 0; j < kSmallTok; ++j) {
        float v = acc[r][j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane_id() == 0) red[warp_id()][r * kSmallTok + j] = v;
      }
    __syncthreads();
    if (tid < ROWS * kSmallTok) {
      const int r = tid / kSmallTok, j = tid % kSmallTok;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kSmallThreads / 32; ++w) s += red[w][tid];
      if (g0 + r < G && t0 + j < T) {
        if (bias) s += bias[g0 + r];
        logits[(size_t)(t0 + j) * G + g0 + r] = s;
      }
    }
    __syncthreads();
  }
}

constexpr int kBM = 64;  // tokens per tile
constexpr int kBN = 64;  // gate rows per tile
constexpr int kBK = 32;  // H per stage

__global__ void __launch_bounds__(256)
router_tiled_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ wg,
                    const float* __restrict__ bias, float* __restrict__ logits, int T, int H,
                    int G) {
  // transposed tiles, padded so the transposing stores are conflict free
  __shared__ float xs[kBK][kBM + 1];
  __shared__ float ws[kBK][kBN + 1];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  const int ty = tid / 16, tx = tid % 16;  // token m = ty + 16 i, gate n = tx + 16 j
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  // x tile: 64 rows x 32 bf16 = 256 uint4, one per thread
  const int xr = tid / 4, xc = (tid % 4) * 8;
  for (int k0 = 0; k0 < H; k0 += kBK) {
    {
      float f[8];
      if (m0 + xr < T && k0 + xc < H) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(m0 + xr) * H + k0 + xc));
        bf16x8_to_f32(v, f);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[xc + i][xr] = f[i];
    }
    // wg tile: 64 rows x 32 fp32 = 512 float4, two per thread
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int idx = tid + q * 256;
      const int wr = idx / 8, wc = (idx % 8) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (n0 + wr < G && k0 + wc < H)
        v = __ldg(reinterpret_cast<const float4*>(wg + (size_t)(n0 + wr) * H + k0 + wc));
      ws[wc + 0][wr] = v.x; ws[wc + 1][wr] = v.y; ws[wc + 2][wr] = v.z; ws[wc + 3][wr] = v.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < kBK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[k][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[k][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n < G) logits[(size_t)m * G + n] = acc[i][j] + (bias ? bias[n] : 0.f);
    }
  }
}

}  // namespace

cudaError_t launch_router_gemm(const void* x, const float* wg, const float* gate_bias,
                               float* logits, int T, int H, int G, cudaStream_t stream) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (T <= 16) {
    if (G <= 256) {
      router_small_kernel<1><<<G, kSmallThreads, 0, stream>>>(xb, wg, gate_bias, logits, T, H, G);
    } else if (G <= 512) {
      router_small_kernel<2><<<moe_cdiv(G, 2), kSmallThreads, 0, stream>>>(xb, wg, gate_bias,
                                                                          logits, T, H, G);
    } else {
      router_small_kernel<4><<<moe_cdiv(G, 4), kSmallThreads, 0, stream>>>(xb, wg, gate_bias,
                                                                          logits, T, H, G);
    }
  } else {
    dim3 grid(moe_cdiv(G, kBN), moe_cdiv(T, kBM));
    router_tiled_kernel<<<grid, 256, 0, stream>>>(xb, wg, gate_bias, logits, T, H, G);
  }
  return cudaGetLastError();
}
