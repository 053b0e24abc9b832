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
// a fixed float32 formula so that the selection is reproducible bit for bit:
//   exp(z): n = rint(z*log2e); r = (z - n*ln2_hi) - n*ln2_lo (Cody-Waite);
//           p = degree-7 Taylor polynomial of e^r (Horner); exp = p * 2^n
//   sigmoid(l) = 1 / (1 + exp(-l)), with 0 for -l > 88 and 1 for -l < -87
// each step a single correctly rounded float32 operation (__f*_rn, never
// contracted to an FMA).  Ties: the lower expert index wins.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace {

// float32 constants of the formula above, each the float32 nearest the value
// named (ln2_hi keeps 15 significant bits so n * ln2_hi is exact)
__device__ __constant__ float kLog2e = 0x1.715476p+0f;     // log2(e)
__device__ __constant__ float kLn2Hi = 0x1.62e4p-1f;       // 0.693145751953125
__device__ __constant__ float kLn2Lo = 0x1.7f7d1cp-20f;    // ln2 - ln2_hi
__device__ __constant__ float kTaylor[8] = {
    0x1.a01a02p-13f,  // 1/5040
    0x1.6c16c2p-10f,  // 1/720
    0x1.111112p-7f,   // 1/120
    0x1.555556p-5f,   // 1/24
    0x1.555556p-3f,   // 1/6
    0x1p-1f,          // 1/2
    0x1p+0f,          // 1
    0x1p+0f};         // 1

MOE_DEVICE float sigmoid_key(float l) {
  const float z = -l;
  if (z > 88.f) return 0.f;
  if (z < -87.f) return 1.f;
  const float n = rintf(__fmul_rn(z, kLog2e));
  float r = __fsub_rn(z, __fmul_rn(n, kLn2Hi));
  r = __fsub_rn(r, __fmul_rn(n, kLn2Lo));
  float p = kTaylor[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) p = __fadd_rn(__fmul_rn(p, r), kTaylor[i]);
  const float two_n = __int_as_float(((int)n + 127) << 23);
  const float e = __fmul_rn(p, two_n);
  return __fdiv_rn(1.f, __fadd_rn(1.f, e));
}

// Keys are compared as unsigned integers: the map below is monotone on
// floats (negative below positive, larger magnitude further out) once -0 is
// folded to +0 (an fp32 add of +0), so equal floats give equal keys.
MOE_DEVICE uint32_t order_key(float k) {
  const uint32_t b = __float_as_uint(__fadd_rn(k, 0.f));
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// strict total order: larger key first, lower index first among equal keys
MOE_DEVICE bool better(uint32_t ka, int ia, uint32_t kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

template <int NPL, int LK>
__global__ void __launch_bounds__(128)
topk_kernel(const float* __restrict__ logits, int ld, const float* __restrict__ sel_bias, int T,
            int E, int K, int mode, float scale, int32_t* __restrict__ ids,
            float* __restrict__ weights, float* __restrict__ shared_gate) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * (blockDim.x / 32) + warp_id();
  if (t >= T) return;
  const int lane = lane_id();
  const float* row = logits + (size_t)t * ld;

  // lane-owned sorted candidate list (keys as ordered u32, empty slots lowest)
  uint32_t lk[LK];
  int li[LK];
#pragma unroll
  for (int s = 0; s < LK; ++s) { lk[s] = 0u; li[s] = 0x7fffffff; }

#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = j * 32 + lane;
    if (e < E) {
      const float l = __ldg(row + e);
      float key = l;
      if (mode == MOE_SCORE_SIGMOID_BIAS_SCALED)
        key = __fadd_rn(sigmoid_key(l), sel_bias ? __ldg(sel_bias + e) : 0.f);
      const uint32_t ku = order_key(key);
      if (better(ku, e, lk[LK - 1], li[LK - 1])) {
        uint32_t nk = ku;
        int ni = e;
#pragma unroll
        for (int s = 0; s < LK; ++s) {
          const bool b = better(nk, ni, lk[s], li[s]);
          const uint32_t tk = lk[s];
          const int ti = li[s];
          lk[s] = b ? nk : tk;
          li[s] = b ? ni : ti;
          nk = b ? tk : nk;
          ni = b ? ti : ni;
        }
      }
    }
  }

  // K merge rounds over the lanes' heads: the largest head key by one warp
  // max-reduction, then the lowest expert index among heads with that key by
  // one min-reduction; the owning lane pops its head.
  int my_id = -1;
  for (int r = 0; r < K; ++r) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, lk[0]);
    const uint32_t mi = __reduce_min_sync(0xffffffffu, lk[0] == m ? (uint32_t)li[0] : 0xffffffffu);
    if (li[0] == (int)mi) {
#pragma unroll
      for (int s = 0; s < LK - 1; ++s) { lk[s] = lk[s + 1]; li[s] = li[s + 1]; }
      lk[LK - 1] = 0u;
      li[LK - 1] = 0x7fffffff;
    }
    if (lane == r) my_id = (int)mi;
  }

  float v = 0.f;
  if (mode == MOE_SCORE_SOFTMAX_RENORM) {
    const float l = lane < K ? __ldg(row + my_id) : 0.f;
    const float m = __shfl_sync(0xffffffffu, l, 0);  // the first pick is the largest
    v = lane < K ? expf(l - m) : 0.f;
  } else {
    v = lane < K ? sigmoid_key(__ldg(row + my_id)) : 0.f;
  }
  float sum = v;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < K) {
    const float w = mode == MOE_SCORE_SOFTMAX_RENORM ? v / sum : scale * v / sum;
    ids[(size_t)t * K + lane] = my_id;
    weights[(size_t)t * K + lane] = w;
  }
  if (shared_gate && lane == 0) shared_gate[t] = sigmoid_key(__ldg(row + E));
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
