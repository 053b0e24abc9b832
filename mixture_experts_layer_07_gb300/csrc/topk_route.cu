// K: top-K expert selection, one warp per token.
//
// "FlashInfer MoE routing optimisation" (flashinfer PR #4152):
//  * "1. routing_custom.cu" -- instead of warp 0 holding K-sized score arrays
//    and doing all the sorting, every lane keeps its own top-K candidates, so
//    the register cost is spread over the warp.  Here lane l reads experts
//    l, l+32, l+64, ... (coalesced), keeps a sorted list of its best
//    min(K, experts-per-lane) candidates in registers, and the warp then takes
//    K rounds of an arg-max over the lanes' list heads (two warp reductions,
//    redux.sync, per round); the winning lane pops its head.
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
#include "topk_warp.cuh"

namespace {

using namespace moe_route;

template <int NPL, int LK>
__global__ void __launch_bounds__(128)
topk_kernel(const float* __restrict__ logits, int ld, const float* __restrict__ sel_bias, int T,
            int E, int K, int mode, float scale, int32_t* __restrict__ ids,
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
cudaError_t launch_npl(const float* logits, int ld, const float* sel_bias, int T, int E, int K,
                       int mode, float scale, int32_t* ids, float* weights, float* shared_gate,
                       cudaStream_t stream) {
  constexpr int kWarps = 4;
  dim3 grid(moe_cdiv(T, kWarps)), block(32 * kWarps);
  // list length = min(K tier, experts per lane)
#define MOE_TOPK_LAUNCH(KT)                                                                 \
  return moe_launch(topk_kernel<NPL, (KT < NPL ? KT : NPL)>, grid, block, 0, stream, 1, logits, \
                    ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate)
  if (K <= 2) MOE_TOPK_LAUNCH(2);
  if (K <= 4) MOE_TOPK_LAUNCH(4);
  if (K <= 8) MOE_TOPK_LAUNCH(8);
  if (K <= 16) MOE_TOPK_LAUNCH(16);
  MOE_TOPK_LAUNCH(32);
#undef MOE_TOPK_LAUNCH
}

}  // namespace

cudaError_t launch_topk_route(const float* logits, int ld, const float* sel_bias, int T, int E,
                              int K, int mode, float scale, int32_t* ids, float* weights,
                              float* shared_gate, cudaStream_t stream) {
  const int npl = moe_cdiv(E, 32);
  if (npl <= 1) return launch_npl<1>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate, stream);
  if (npl <= 2) return launch_npl<2>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate, stream);
  if (npl <= 4) return launch_npl<4>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate, stream);
  if (npl <= 8) return launch_npl<8>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate, stream);
  if (npl <= 16) return launch_npl<16>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate, stream);
  if (npl <= 28) return launch_npl<28>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate, stream);
  return launch_npl<32>(logits, ld, sel_bias, T, E, K, mode, scale, ids, weights, shared_gate, stream);
}
