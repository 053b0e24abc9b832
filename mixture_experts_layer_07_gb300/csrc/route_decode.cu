// Fused decode routing: router GEMM, top-K, permute and the grouped-GEMM plan
// in ONE launch for small batches (T <= 32).
//
// "vLLM MiniMax-M2 MoE gate optimisation: fused FP32 kernel" (vllm PR #38445),
// "why" 1: at low concurrency launch overhead outweighs the work, so the
// cast and the GEMM became one kernel; "vLLM MoE permute optimisation: buffer
// pre-allocation" (vllm PR #43014): small batches pay most for per-call
// overhead.  Here the steps up to the expert GEMM share one launch:
//   1. every CTA computes one gate row g for all T tokens (fp32 dot products
//      from 16-byte bf16 vectors, fixed-order block reduction) -> logits
//   2. each CTA, after its stores, fences and bumps a completion counter; the
//      CTA that sees the last count (no CTA ever waits) then
//   3. routes every token (warp top-K, logits read through L2; for E > 128
//      the shorter-list group route of topk_group.cuh),
//   4. permutes the T*K replicas in one CTA (shared-memory counters),
//   5. plans the grouped GEMM (per-block variant and work lists),
//   6. and resets the counter to zero for the next call.
// The results are those of the separate kernels: same sums for the logits
// (the decode router's order), same selection, same stable permutation.
#include "common.cuh"
#include "internal.h"
#include "permute_block.cuh"
#include "plan.cuh"
#include "topk_group.cuh"
#include "topk_warp.cuh"

namespace {

using namespace moe_route;
using namespace moe_plan;

constexpr int kThreads = 256;
constexpr int kTok = 8;  // tokens accumulated together
constexpr int kWarps = kThreads / 32;

// kGroup (E > 128): the token's route is group_route over the whole warp
// (lists of 4 or 8 with refill instead of K-long lists: a shorter chain per
// token); kVec: float4 logit rows
template <int NPL, int LK, bool kGroup, bool kVec>
__global__ void __launch_bounds__(kThreads)
route_decode_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ wg,
                    const float* __restrict__ gate_bias, float* __restrict__ logits, int T, int H,
                    int G, const float* __restrict__ sel_bias, int E, int K, int mode, float scale,
                    int32_t* __restrict__ ids, float* __restrict__ weights,
                    float* __restrict__ shared_gate, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ row_to_flat, int32_t* __restrict__ flat_to_row,
                    int32_t* dev_status, int m_skinny, int dispatch, int wdtype,
                    int32_t* __restrict__ plan_counts, PlanOut plan_out,
                    int32_t* __restrict__ block_variant, unsigned int* done_ctr) {
  extern __shared__ int32_t sm[];  // [kWarps][E] counters, [E + 1] offsets, [T*K] ids
  __shared__ float red[kWarps][kTok];
  __shared__ int is_last;
  pdl_wait();
  pdl_trigger();
  const int g = blockIdx.x, tid = threadIdx.x, warp = warp_id(), lane = lane_id();

  // 1. gate row g for every token
  for (int t0 = 0; t0 < T; t0 += kTok) {
    float acc[kTok];
#pragma unroll
    for (int j = 0; j < kTok; ++j) acc[j] = 0.f;
    for (int h = tid * 8; h < H; h += kThreads * 8) {
      const float4* p = reinterpret_cast<const float4*>(wg + (size_t)g * H + h);
      const float4 a = __ldg(p), b = __ldg(p + 1);
      const float w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int j = 0; j < kTok; ++j) {
        if (t0 + j < T) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + j) * H + h));
          float xf[8];
          bf16x8_to_f32(v, xf);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[j] = fmaf(w[i], xf[i], acc[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kTok; ++j) {
      float v = acc[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[warp][j] = v;
    }
    __syncthreads();
    if (tid < kTok && t0 + tid < T) {
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < kWarps; ++q) s += red[q][tid];
      logits[(size_t)(t0 + tid) * G + g] = s + (gate_bias ? gate_bias[g] : 0.f);
    }
    __syncthreads();
  }

  // 2. the last CTA to finish takes the rest
  if (tid == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(done_ctr, 1u);
    is_last = prev == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  int32_t* cnt = sm;
  int32_t* off_s = sm + kWarps * E;
  int32_t* ids_s = off_s + E + 1;
  // 3. top-K, one warp per token
  for (int t = warp; t < T; t += kWarps) {
    const float* row = logits + (size_t)t * G;
    if constexpr (kGroup) {
      float l[NPL];
      group_load<32, NPL, kVec, true>(row, true, E, l);
      group_route<32, NPL, LK, kVec, true>(l, row, true, 1, sel_bias, E, K, mode, scale,
                                           ids + (size_t)t * K, weights + (size_t)t * K, nullptr,
                                           ids_s + t * K);
    } else {
      warp_topk<NPL, LK, true>(row, sel_bias, E, K, mode, scale, ids + (size_t)t * K,
                               weights + (size_t)t * K, ids_s + t * K);
    }
    if (shared_gate && lane == 0) shared_gate[t] = sigmoid_key(__ldcg(row + E));
  }
  __syncthreads();
  // 4. permute
  moe_permute_block::permute_block<kWarps>(ids_s, T * K, E, offsets, off_s, row_to_flat,
                                           flat_to_row, dev_status, cnt);
  // 5. plan
  plan_experts<kThreads>(off_s, E, T * K, m_skinny, dispatch, wdtype, plan_counts, plan_out,
                         block_variant);
  // 6. ready for the next call
  if (tid == 0) *done_ctr = 0u;
}

template <int NPL, int LK, bool kGroup, bool kVec>
cudaError_t launch_one(const RouteDecodeArgs& a, cudaStream_t stream) {
  const size_t smem = ((size_t)(kWarps + 1) * a.E + 1 + (size_t)a.T * a.K) * sizeof(int32_t);
  const PlanView pv = plan_view(a.gemm_scratch, a.T * a.K, a.E);
  PlanOut po = plan_out(pv);
  const int m_skinny = a.m_skinny < 0 ? MOE_DEFAULT_M_SKINNY : a.m_skinny;
  return moe_launch(route_decode_kernel<NPL, LK, kGroup, kVec>, dim3(a.G), dim3(kThreads), smem,
                    stream, 1, static_cast<const __nv_bfloat16*>(a.x), a.wg, a.gate_bias,
                    a.logits, a.T, a.H, a.G, a.sel_bias, a.E, a.K, a.mode, a.scale, a.ids,
                    a.weights, a.shared_gate, a.offsets, a.row_to_flat, a.flat_to_row,
                    a.dev_status, m_skinny, a.dispatch, a.wdtype, pv.counts, po, a.block_variant,
                    a.done_ctr);
}

// E <= 128: one warp per token, lists of min(K tier, experts per lane)
template <int NPL>
cudaError_t launch_warp(const RouteDecodeArgs& a, cudaStream_t stream) {
#define MOE_RD_LAUNCH(KT) return launch_one<NPL, (KT < NPL ? KT : NPL), false, false>(a, stream)
  if (a.K <= 2) MOE_RD_LAUNCH(2);
  if (a.K <= 4) MOE_RD_LAUNCH(4);
  if (a.K <= 8) MOE_RD_LAUNCH(8);
  if (a.K <= 16) MOE_RD_LAUNCH(16);
  MOE_RD_LAUNCH(32);
#undef MOE_RD_LAUNCH
}

// E > 128: group_route over the warp, lists of 4 (K <= 8) or 8
template <int NPL, bool kVec>
cudaError_t launch_group(const RouteDecodeArgs& a, cudaStream_t stream) {
  if (a.K <= 8) return launch_one<NPL, 4, true, kVec>(a, stream);
  return launch_one<NPL, 8, true, kVec>(a, stream);
}

template <bool kVec>
cudaError_t launch_group_tier(const RouteDecodeArgs& a, cudaStream_t stream) {
  // experts per lane: whole float4s of 4 * 32 experts per step (kVec) or
  // one expert per 32 (scalar)
  const int npl = kVec ? 4 * moe_cdiv(a.E, 128) : moe_cdiv(a.E, 32);
  if (npl <= 8) return launch_group<8, kVec>(a, stream);
  if (npl <= 16) return launch_group<16, kVec>(a, stream);
  if (npl <= 28) return launch_group<28, kVec>(a, stream);
  return launch_group<32, kVec>(a, stream);
}

}  // namespace

cudaError_t launch_route_decode(const RouteDecodeArgs& a, cudaStream_t stream) {
  if (a.E > 128) {
    const bool vec = a.E % 4 == 0 && a.G % 4 == 0 &&
                     (reinterpret_cast<uintptr_t>(a.logits) & 15) == 0;
    return vec ? launch_group_tier<true>(a, stream) : launch_group_tier<false>(a, stream);
  }
  const int npl = moe_cdiv(a.E, 32);
  if (npl <= 1) return launch_warp<1>(a, stream);
  if (npl <= 2) return launch_warp<2>(a, stream);
  return launch_warp<4>(a, stream);
}
