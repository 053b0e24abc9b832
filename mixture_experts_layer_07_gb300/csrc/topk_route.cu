// K: top-K expert selection.
//
// "FlashInfer MoE routing optimisation" (flashinfer PR #4152):
//  * "1. routing_custom.cu" -- instead of warp 0 holding K-sized score arrays
//    and doing all the sorting, every lane keeps its own candidates, so the
//    register cost is spread over the lanes.  Here a group of 8, 16 or 32
//    lanes routes one token (group_topk, topk_group.cuh): lane-owned sorted
//    candidate lists, K rounds of a group arg-max over the list heads, the
//    winning lane pops its head.  With E <= 128 a warp routes four tokens at
//    once, so each merge round serves four tokens.
//  * "2. routing_common.cu" -- E = 896 gets its own tier (28 experts per lane)
//    rather than running as the 1024 tier.
//
// Scores: mode 0 selects on the raw logit (softmax is monotone) and weights the
// selected experts by the softmax over their logits.  Mode 1 (SigmoidBias +
// ScaledSumNormalize, named in the same page's "performance" section) selects
// on sigmoid(l) + bias and weights by scale * sigmoid(l) / sum.  The sigmoid is
// a fixed float32 formula (topk_warp.cuh) so that the selection is
// reproducible bit for bit.  Ties: the lower expert index wins.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "topk_group.cuh"
#include "topk_thread.cuh"
#include "topk_warp.cuh"

namespace {

using namespace moe_route;

constexpr int kThreads = 256;

int sm_count() { return moe_num_sms(); }

// GS lanes per token, 32/GS tokens per warp (group_load + group_route in
// topk_group.cuh)
template <int GS, int NPL, int LK, bool kVec>
__global__ void __launch_bounds__(kThreads, 5)
topk_kernel(const float* __restrict__ logits, int ld, const float* __restrict__ sel_bias, int T,
            int E, int K, int mode, float scale, int32_t* __restrict__ ids,
            float* __restrict__ weights, float* __restrict__ shared_gate) {
  extern __shared__ int32_t s_slots[];  // [warp][group][K]
  pdl_wait();
  pdl_trigger();
  constexpr int kGroups = 32 / GS;
  const int g = lane_id() / GS;
  const int tb = (blockIdx.x * (blockDim.x / 32) + warp_id()) * kGroups;  // the warp's first token
  if (tb >= T) return;  // the whole warp
  const int t = tb + g;
  const bool valid = t < T;
  const int nvalid = T - tb < kGroups ? T - tb : kGroups;
  const float* row = logits + (size_t)(valid ? t : 0) * ld;
  float l[NPL];
  group_load<GS, NPL, kVec>(row, valid, E, l);
  group_route<GS, NPL, LK, kVec>(l, row, valid, nvalid, sel_bias, E, K, mode, scale,
                                 ids + (size_t)t * K, weights + (size_t)t * K, nullptr,
                                 s_slots + (warp_id() * kGroups + g) * K);
  if (shared_gate && valid && (lane_id() & (GS - 1)) == 0)
    shared_gate[t] = sigmoid_key(__ldg(row + E));
}

template <int GS, int NPL, int LK, bool kVec>
cudaError_t launch_kernel(const float* logits, int ld, const float* sel_bias, int T, int E, int K,
                          int mode, float scale, int32_t* ids, float* weights,
                          float* shared_gate, cudaStream_t stream) {
  // small batches get 64-thread CTAs so that more SMs take part
  const int threads = moe_cdiv(T, kThreads / GS) >= 2 * sm_count() ? kThreads : 64;
  const int tpc = threads / GS;
  const dim3 grid(moe_cdiv(T, tpc)), block(threads);
  const size_t smem = (size_t)tpc * K * sizeof(int32_t);
  return moe_launch(topk_kernel<GS, NPL, LK, kVec>, grid, block, smem, stream, 1, logits, ld,
                    sel_bias, T, E, K, mode, scale, ids, weights, shared_gate);
}

template <int GS, int NPL, bool kVec>
cudaError_t launch_tier(const float* logits, int ld, const float* sel_bias, int T, int E, int K,
                        int mode, float scale, int32_t* ids, float* weights, float* shared_gate,
                        cudaStream_t stream) {
  // lists of 4 for K <= 8, else 8 (refills keep either exact)
  constexpr int kLK8 = NPL >= 8 ? 8 : NPL;
  if (K <= 8)
    return launch_kernel<GS, NPL, 4, kVec>(logits, ld, sel_bias, T, E, K, mode, scale, ids,
                                           weights, shared_gate, stream);
  return launch_kernel<GS, NPL, kLK8, kVec>(logits, ld, sel_bias, T, E, K, mode, scale, ids,
                                            weights, shared_gate, stream);
}

// Small batches with E <= 128: one warp per token (warp_topk), whose
// per-token latency is shorter than a group's (4 experts per lane instead of
// 16); the group kernel wins once there are tokens enough to fill the GPU.
constexpr long long kGroupMinT = 32768;

template <int NPL, int LK>
__global__ void __launch_bounds__(128)
topk_warp_kernel(const float* __restrict__ logits, int ld, const float* __restrict__ sel_bias,
                 int T, int E, int K, int mode, float scale, int32_t* __restrict__ ids,
                 float* __restrict__ weights, float* __restrict__ shared_gate) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * (blockDim.x / 32) + warp_id();
  if (t >= T) return;
  const float* row = logits + (size_t)t * ld;
  warp_topk<NPL, LK>(row, sel_bias, E, K, mode, scale, ids + (size_t)t * K, weights + (size_t)t * K);
  if (shared_gate && lane_id() == 0) shared_gate[t] = sigmoid_key(__ldg(row + E));
}

template <int NPL>
cudaError_t launch_warp(const float* logits, int ld, const float* sel_bias, int T, int E, int K,
                        int mode, float scale, int32_t* ids, float* weights, float* shared_gate,
                        cudaStream_t stream) {
  constexpr int kWarps = 4;
  const dim3 grid(moe_cdiv(T, kWarps)), block(32 * kWarps);
  // list length = min(K tier, experts per lane)
#define MOE_TOPK_LAUNCH(KT)                                                                  \
  return moe_launch(topk_warp_kernel<NPL, (KT < NPL ? KT : NPL)>, grid, block, 0, stream, 1, \
                    logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate)
  if (K <= 2) MOE_TOPK_LAUNCH(2);
  if (K <= 4) MOE_TOPK_LAUNCH(4);
  if (K <= 8) MOE_TOPK_LAUNCH(8);
  if (K <= 16) MOE_TOPK_LAUNCH(16);
  MOE_TOPK_LAUNCH(32);
#undef MOE_TOPK_LAUNCH
}

// ---------------------------------------------------------------- thread per token
// Large batches with E <= 128: one thread routes one token (thread_topk,
// topk_thread.cuh).  A thread reading its own 512-byte row would make every
// warp load touch 32 lines, so each warp first copies its 32 rows into shared
// memory with row-contiguous (coalesced) loads, rows padded by 16 bytes so
// the threads' own-row reads fall in distinct banks.
constexpr int kThreadWarps = 2;
template <int NV, int KT, bool kVec>
__global__ void __launch_bounds__(32 * kThreadWarps)
topk_thread_kernel(const float* __restrict__ logits, int ld, const float* __restrict__ sel_bias,
                   int T, int E, int K, int mode, float scale, int32_t* __restrict__ ids,
                   float* __restrict__ weights, float* __restrict__ shared_gate) {
  constexpr int kRow = 4 * NV + 4;  // floats per staged row
  __shared__ __align__(16) float rows[kThreadWarps][32][kRow];
  pdl_wait();
  pdl_trigger();
  const int warp = warp_id(), lane = lane_id();
  const int t0 = (blockIdx.x * kThreadWarps + warp) * 32;
  if (t0 >= T) return;  // the whole warp
  float (*mine)[kRow] = rows[warp];
  if constexpr (kVec) {
    // 32 / NV rows per load instruction, one float4 per lane
    constexpr int kRowsPer = 32 / NV;
    const int rr = lane / NV, v = lane % NV;
#pragma unroll 4
    for (int r0 = 0; r0 < 32; r0 += kRowsPer) {
      const int r = r0 + rr;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t0 + r < T && 4 * v < E)
        f = __ldg(reinterpret_cast<const float4*>(logits + (size_t)(t0 + r) * ld + 4 * v));
      *reinterpret_cast<float4*>(&mine[r][4 * v]) = f;
    }
  } else {
    for (int r = 0; r < 32 && t0 + r < T; ++r)
      for (int e = lane; e < E; e += 32) mine[r][e] = __ldg(logits + (size_t)(t0 + r) * ld + e);
  }
  __syncwarp();
  const int t = t0 + lane;
  if (t < T) {
    thread_topk<NV, KT, kVec, true>(mine[lane], sel_bias, E, K, mode, scale, ids + (size_t)t * K,
                                    weights + (size_t)t * K);
    if (shared_gate) shared_gate[t] = sigmoid_key(__ldg(logits + (size_t)t * ld + E));
  }
}

template <int NV, bool kVec>
cudaError_t launch_thread_nv(const float* logits, int ld, const float* sel_bias, int T, int E,
                             int K, int mode, float scale, int32_t* ids, float* weights,
                             float* shared_gate, cudaStream_t stream) {
  const dim3 grid(moe_cdiv(T, 32 * kThreadWarps)), block(32 * kThreadWarps);
#define MOE_TOPK_THREAD(KT)                                                                   \
  return moe_launch(topk_thread_kernel<NV, KT, kVec>, grid, block, 0, stream, 1, logits, ld, \
                    sel_bias, T, E, K, mode, scale, ids, weights, shared_gate)
  if (K <= 2) MOE_TOPK_THREAD(2);
  if (K <= 4) MOE_TOPK_THREAD(4);
  if (K <= 8) MOE_TOPK_THREAD(8);
  if (K <= 16) MOE_TOPK_THREAD(16);
  MOE_TOPK_THREAD(32);
#undef MOE_TOPK_THREAD
}

// list length (K rounded up to a power of two) no larger than E, so that
// every group of the bound holds an expert
bool thread_route_fits(int E, int K) {
  int kt = 2;
  while (kt < K) kt *= 2;
  return E <= 128 && kt <= E && K <= 32;
}

template <bool kVec>
cudaError_t launch_thread(const float* logits, int ld, const float* sel_bias, int T, int E, int K,
                          int mode, float scale, int32_t* ids, float* weights, float* shared_gate,
                          cudaStream_t stream) {
  if (E <= 32)
    return launch_thread_nv<8, kVec>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights,
                                     shared_gate, stream);
  if (E <= 64)
    return launch_thread_nv<16, kVec>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights,
                                      shared_gate, stream);
  return launch_thread_nv<32, kVec>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights,
                                    shared_gate, stream);
}

template <bool kVec>
cudaError_t launch_vec(const float* logits, int ld, const float* sel_bias, int T, int E, int K,
                       int mode, float scale, int32_t* ids, float* weights, float* shared_gate,
                       cudaStream_t stream) {
#define MOE_TOPK_TIER(GS, NPL)                                                                    \
  return launch_tier<GS, NPL, kVec>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, \
                                    shared_gate, stream)
  if (E <= 32) MOE_TOPK_TIER(8, 4);
  if (E <= 64) MOE_TOPK_TIER(8, 8);
  if (E <= 128) MOE_TOPK_TIER(8, 16);
  if (E <= 256) MOE_TOPK_TIER(16, 16);
  if (E <= 512) MOE_TOPK_TIER(32, 16);
  if (E <= 896) MOE_TOPK_TIER(32, 28);  // E = 896 as its own tier, not padded to 1024
  MOE_TOPK_TIER(32, 32);
#undef MOE_TOPK_TIER
}

}  // namespace

cudaError_t launch_topk_route(const float* logits, int ld, const float* sel_bias, int T, int E,
                              int K, int mode, float scale, int32_t* ids, float* weights,
                              float* shared_gate, cudaStream_t stream) {
  if (E <= 128 && T < kGroupMinT) {
    const int npl = moe_cdiv(E, 32);
    if (npl <= 1) return launch_warp<1>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate, stream);
    if (npl <= 2) return launch_warp<2>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate, stream);
    return launch_warp<4>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate, stream);
  }
  // float4 rows when every row starts on a 16-byte boundary and E fills whole vectors
  const bool vec = E % 4 == 0 && ld % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
  if (thread_route_fits(E, K)) {
    if (vec)
      return launch_thread<true>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights,
                                 shared_gate, stream);
    return launch_thread<false>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights,
                                shared_gate, stream);
  }
  if (vec)
    return launch_vec<true>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate,
                            stream);
  return launch_vec<false>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate,
                           stream);
}
