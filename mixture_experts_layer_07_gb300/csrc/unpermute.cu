// U: weighted unpermute / combine.
//
// "vLLM MoE permute optimisation: buffer pre-allocation" (vllm PR #43014),
// introduction: unpermute is the inverse of permute; it brings every expert
// output row back to its token and combines the K rows of a token.  Fused
// here into one gather-multiply-add pass:
//   out[t] = bf16( sum_{k=0..K-1} w[t,k] * y[flat_to_row[t*K+k]] + g[t] * sh[t] )
// with fp32 sums in k order and one rounding at the end.  Each thread owns 8
// consecutive columns (one 16-byte vector per source row); a CTA covers one
// token and 1024 columns.
#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads)
unpermute_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ flat_to_row,
                 const float* __restrict__ weights, int K, int H8,
                 const uint4* __restrict__ shared_y, const float* __restrict__ shared_gate,
                 uint4* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int c = blockIdx.y * kThreads + threadIdx.x;
  if (c >= H8) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  // K sources in groups of 8: all row indices, then all 16-byte vectors in
  // flight together, then the fp32 sums in k order
  for (int k0 = 0; k0 < K; k0 += 8) {
    int rows[8];
    float wk[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      rows[j] = k0 + j < K ? __ldg(flat_to_row + (size_t)t * K + k0 + j) : -1;
      wk[j] = k0 + j < K ? __ldg(weights + (size_t)t * K + k0 + j) : 0.f;
    }
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      v[j] = rows[j] >= 0 ? __ldg(y + (size_t)rows[j] * H8 + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (rows[j] < 0) continue;
      float f[8];
      bf16x8_to_f32(v[j], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wk[j], f[i], acc[i]);
    }
  }
  if (shared_y) {
    const float g = __ldg(shared_gate + t);
    float f[8];
    bf16x8_to_f32(__ldg(shared_y + (size_t)t * H8 + c), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, f[i], acc[i]);
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  out[(size_t)t * H8 + c] = o;
}

}  // namespace

cudaError_t launch_unpermute(const void* y, const int32_t* flat_to_row, const float* weights,
                             int T, int K, int H, const void* shared_y, const float* shared_gate,
                             void* out, cudaStream_t stream) {
  const int H8 = H / 8;
  dim3 grid(T, moe_cdiv(H8, kThreads));
  return moe_launch(unpermute_kernel, grid, dim3(kThreads), 0, stream, 1,
                    static_cast<const uint4*>(y), flat_to_row, weights, K, H8,
                    static_cast<const uint4*>(shared_y), shared_gate, static_cast<uint4*>(out));
}
