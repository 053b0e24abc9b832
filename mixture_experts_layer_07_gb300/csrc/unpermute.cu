// U: weighted unpermute / combine.
//
// "vLLM MoE permute optimisation: buffer pre-allocation" (vllm PR #43014),
// introduction: unpermute is the inverse of permute; it brings every expert
// output row back to its token and combines the K rows of a token.  Fused
// here into one gather-multiply-add pass:
//   out[t] = bf16( sum_{k=0..K-1} w[t,k] * y[flat_to_row[t*K+k]] + g[t] * sh[t] )
// with fp32 sums in k order and one rounding at the end.  Each thread owns 8
// consecutive columns of a token (one 16-byte vector per source row).
#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kThreads = 128;
constexpr int kCtasPerSm = 16;

// Each thread owns 16-byte output vectors (token t, columns 8c..8c+7), taken
// grid-stride over all T*H/8 of them so one wave of threads shares the work
// evenly (consecutive threads on consecutive vectors of a row).
__global__ void __launch_bounds__(kThreads)
unpermute_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ flat_to_row,
                 const float* __restrict__ weights, int T, int K, int H8,
                 const uint4* __restrict__ shared_y, const float* __restrict__ shared_gate,
                 uint4* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const long long n = (long long)T * H8;
  for (long long i = blockIdx.x * (long long)kThreads + threadIdx.x; i < n;
       i += (long long)gridDim.x * kThreads) {
    const int t = (int)(i / H8), c = (int)(i % H8);
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
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
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(wk[j], f[q], acc[q]);
      }
    }
    if (shared_y) {
      const float g = __ldg(shared_gate + t);
      float f[8];
      bf16x8_to_f32(__ldg(shared_y + i), f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(g, f[q], acc[q]);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    out[i] = o;
  }
}

}  // namespace

cudaError_t launch_unpermute(const void* y, const int32_t* flat_to_row, const float* weights,
                             int T, int K, int H, const void* shared_y, const float* shared_gate,
                             void* out, cudaStream_t stream) {
  const int sms = moe_num_sms();
  const int H8 = H / 8;
  const long long n = (long long)T * H8;
  const long long need = (n + kThreads - 1) / kThreads;
  const int grid = (int)(need < (long long)kCtasPerSm * sms ? need : (long long)kCtasPerSm * sms);
  return moe_launch(unpermute_kernel, dim3(grid > 0 ? grid : 1), dim3(kThreads), 0, stream, 1,
                    static_cast<const uint4*>(y), flat_to_row, weights, T, K, H8,
                    static_cast<const uint4*>(shared_y), shared_gate, static_cast<uint4*>(out));
}
