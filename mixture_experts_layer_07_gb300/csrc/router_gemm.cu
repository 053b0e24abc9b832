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
//  * decode (T <= 32): bound by reading wg once (4*G*H bytes).  A CTA owns ROWS
//    gate rows; its 256 threads split H in 8-element chunks, accumulate all
//    tokens of an 8-token group, and reduce across the block in a fixed tree.
//  * prefill (T > 32): FP32-FMA bound (2*T*G*H flops).  64x64 output tiles,
//    the bf16 tile widened while it is staged into shared memory, an 8x4
//    register micro-tile per thread, and H split across the CTAs of a
//    thread-block cluster (reduced through distributed shared memory) so that
//    small T x G still fills the GPU.
// Both are deterministic: the order of the sums depends only on the sizes.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kSmallThreads = 256;
constexpr int kSmallTok = 8;
constexpr int kSmallMaxT = 32;  // up to here the gate-weight stream dominates

template <int ROWS>
__global__ void __launch_bounds__(kSmallThreads)
router_small_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ wg,
                    const float* __restrict__ bias, float* __restrict__ logits, int T, int H,
                    int G) {
  __shared__ float red[kSmallThreads / 32][ROWS * kSmallTok];
  pdl_wait();
  pdl_trigger();
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
constexpr int kTiledThreads = 128;

// One CTA computes a 64x64 logit tile over its slice of H; the `splits` CTAs
// of a thread-block cluster take consecutive slices and the partial tiles are
// summed through distributed shared memory in rank order (deterministic, no
// global scratch, no atomics).  Thread (ty, tx) owns tokens 8ty..8ty+7 and
// gate rows 4tx..4tx+3; operands are staged transposed so that each k step is
// two 16-byte loads of x (a broadcast across the warp) and one of wg.
__global__ void __launch_bounds__(kTiledThreads)
router_cluster_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ wg,
                      const float* __restrict__ bias, float* __restrict__ logits, int T, int H,
                      int G, int kchunk) {
  __shared__ __align__(16) float xs[kBK][kBM + 4];
  __shared__ __align__(16) float ws[kBK][kBN + 4];
  __shared__ __align__(16) float part[kBM][kBN + 4];
  pdl_wait();
  pdl_trigger();
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int splits = (int)cluster.num_blocks();
  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  const int k_lo = rank * kchunk;
  const int k_hi = min(H, k_lo + kchunk);

  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  uint4 xr[2];
  float4 wr[4];
  auto load = [&](int k0) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {  // 64 rows x 32 bf16 = 256 vectors
      const int idx = tid + q * kTiledThreads;
      const int r = idx / 4, c = (idx % 4) * 8;
      xr[q] = (m0 + r < T && k0 + c < k_hi)
                  ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)(m0 + r) * H + k0 + c))
                  : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // 64 rows x 32 fp32 = 512 vectors
      const int idx = tid + q * kTiledThreads;
      const int r = idx / 8, c = (idx % 8) * 4;
      wr[q] = (n0 + r < G && k0 + c < k_hi)
                  ? __ldg(reinterpret_cast<const float4*>(wg + (size_t)(n0 + r) * H + k0 + c))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto stage = [&]() {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int idx = tid + q * kTiledThreads;
      const int r = idx / 4, c = (idx % 4) * 8;
      float f[8];
      bf16x8_to_f32(xr[q], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[c + i][r] = f[i];
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = tid + q * kTiledThreads;
      const int r = idx / 8, c = (idx % 8) * 4;
      ws[c + 0][r] = wr[q].x; ws[c + 1][r] = wr[q].y; ws[c + 2][r] = wr[q].z; ws[c + 3][r] = wr[q].w;
    }
  };

  if (k_lo < k_hi) load(k_lo);
  for (int k0 = k_lo; k0 < k_hi; k0 += kBK) {
    stage();
    __syncthreads();
    if (k0 + kBK < k_hi) load(k0 + kBK);  // next tile's loads overlap this tile's math
#pragma unroll 8
    for (int k = 0; k < kBK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&xs[k][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&xs[k][ty * 8 + 4]);
      const float4 b = *reinterpret_cast<const float4*>(&ws[k][tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
    *reinterpret_cast<float4*>(&part[ty * 8 + i][tx * 4]) =
        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  cluster.sync();
  // rank r sums rows [r*64/splits, (r+1)*64/splits) of the tile over the cluster
  const int rows = kBM / splits;
  for (int e = tid; e < rows * kBN; e += kTiledThreads) {
    const int r = rank * rows + e / kBN, c = e % kBN;
    float sum = 0.f;
    for (int q = 0; q < splits; ++q) sum += cluster.map_shared_rank(&part[r][c], q)[0];
    const int m = m0 + r, n = n0 + c;
    if (m < T && n < G) logits[(size_t)m * G + n] = sum + (bias ? bias[n] : 0.f);
  }
  cluster.sync();  // keep this CTA's partial tile alive until every rank has read it
}

int num_sms_router() { return moe_num_sms(); }

}  // namespace

cudaError_t launch_router_gemm(const void* x, const float* wg, const float* gate_bias,
                               float* logits, int T, int H, int G, cudaStream_t stream) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (T <= kSmallMaxT) {
    if (G <= 256) {
      return moe_launch(router_small_kernel<1>, dim3(G), dim3(kSmallThreads), 0, stream, 1, xb, wg,
                        gate_bias, logits, T, H, G);
    } else if (G <= 512) {
      return moe_launch(router_small_kernel<2>, dim3(moe_cdiv(G, 2)), dim3(kSmallThreads), 0,
                        stream, 1, xb, wg, gate_bias, logits, T, H, G);
    } else {
      return moe_launch(router_small_kernel<4>, dim3(moe_cdiv(G, 4)), dim3(kSmallThreads), 0,
                        stream, 1, xb, wg, gate_bias, logits, T, H, G);
    }
  } else {
    // split H over a cluster until there are about two CTAs per SM
    const int tiles = moe_cdiv(G, kBN) * moe_cdiv(T, kBM);
    int splits = 1;
    while (splits < 8 && tiles * splits < 2 * num_sms_router() && H / (splits * 2) >= 2 * kBK)
      splits *= 2;
    const int kchunk = moe_cdiv(moe_cdiv(H, splits), kBK) * kBK;
    return moe_launch(router_cluster_kernel, dim3(moe_cdiv(G, kBN), moe_cdiv(T, kBM), splits),
                      dim3(kTiledThreads), 0, stream, splits, xb, wg, gate_bias, logits, T, H, G,
                      kchunk);
  }
  return cudaGetLastError();
}
