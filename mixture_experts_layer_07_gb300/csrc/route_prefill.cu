// Fused routing for batches above the decode range: top-K, the per-chunk
// expert histograms of the permute, and -- in whichever CTA finishes last --
// the scan to offsets and the grouped-GEMM plan, in ONE launch; a second
// kernel then places every replica (the stable scatter).
//
// "FlashInfer MoE routing optimisation" (flashinfer PR #4152), "1.
// routing_custom.cu": one warp per token keeps lane-owned top-K candidates
// (topk_warp.cuh; for E > 128 the shorter-list group route of
// topk_group.cuh).  "vLLM MoE permute optimisation: buffer pre-allocation"
// (vllm PR #43014), introduction and "1. C++ kernel level": the permute's
// counts, offsets and rows live in caller-owned scratch; here the expert
// histogram of each chunk of tokens is taken right where its ids are chosen,
// so the ids are not read back, and the launches of the separate count, scan
// and plan kernels disappear:
//   1. warp w of CTA c routes tokens c*TPC + w + 32*i (TPC tokens per CTA)
//   2. the CTA histograms its TPC*K replicas in shared memory and writes
//      counts[c][0..E)
//   3. every CTA fences its counts and bumps a completion counter; the CTA
//      that sees the last count (no CTA waits) turns counts into per-chunk
//      exclusive bases in place, writes offsets[E+1], runs the plan of the
//      grouped GEMM (plan.cuh), and resets the counter to zero
//   4. scatter: a warp per chunk walks its replicas in order, 32 at a time;
//      lanes with the same expert find each other with __match_any_sync, so
//      row = offsets[e] + base[c][e] + running count + rank among equal lanes
// The result is the multi-kernel path's, bit for bit (same selection, same
// unique stable permutation, same plan).
#include "common.cuh"
#include "internal.h"
#include "plan.cuh"
#include "topk_group.cuh"
#include "topk_warp.cuh"

namespace {

using namespace moe_route;
using namespace moe_plan;

constexpr int kWarps = 32;  // one token per warp at a time
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxChunks = 1024;  // tokens per CTA grow with T beyond 32 x this

inline int tokens_per_cta(int T) {
  const int tpw = moe_cdiv(T, kWarps * kMaxChunks);  // tokens per warp
  return kWarps * (tpw > 0 ? tpw : 1);
}

// kGroup (E > 128): each token's route is group_route over the whole warp
// (lists of 4 or 8 with refill: a shorter chain per token); kVec: float4 rows
template <int NPL, int LK, bool kGroup, bool kVec>
__global__ void __launch_bounds__(kThreads)
route_prefill_kernel(const float* __restrict__ logits, int ld, const float* __restrict__ sel_bias,
                     int T, int E, int K, int mode, float scale, int32_t* __restrict__ ids,
                     float* __restrict__ weights, float* __restrict__ shared_gate, int tpc,
                     int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int m_skinny,
                     int dispatch, int wdtype, int32_t* __restrict__ plan_counts,
                     PlanOut plan_out, int32_t* __restrict__ block_variant,
                     unsigned int* done_ctr) {
  extern __shared__ int32_t sm[];  // ids [tpc*K], hist [E], off [E + 1], totals [E]
  __shared__ int is_last;
  __shared__ int32_t warp_sum[kWarps];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = warp_id(), lane = lane_id();
  const int c = blockIdx.x, nchunks = gridDim.x;
  const int t0 = c * tpc;
  const int ntok = min(tpc, T - t0);
  int32_t* ids_s = sm;
  int32_t* hist = ids_s + (size_t)tpc * K;
  int32_t* off_s = hist + E;
  int32_t* tot_s = off_s + E + 1;
  for (int e = tid; e < E; e += kThreads) hist[e] = 0;

  // 1. top-K
  for (int i = warp; i < ntok; i += kWarps) {
    const int t = t0 + i;
    const float* row = logits + (size_t)t * ld;
    if constexpr (kGroup) {
      float l[NPL];
      group_load<32, NPL, kVec>(row, true, E, l);
      group_route<32, NPL, LK, kVec>(l, row, true, 1, sel_bias, E, K, mode, scale,
                                     ids + (size_t)t * K, weights + (size_t)t * K, nullptr,
                                     ids_s + i * K);
    } else {
      warp_topk<NPL, LK>(row, sel_bias, E, K, mode, scale, ids + (size_t)t * K,
                         weights + (size_t)t * K, ids_s + i * K);
    }
    if (shared_gate && lane == 0) shared_gate[t] = sigmoid_key(__ldg(row + E));
  }
  __syncthreads();
  // 2. this chunk's histogram
  for (int i = tid; i < ntok * K; i += kThreads) {
    const int e = ids_s[i];
    if ((unsigned)e < (unsigned)E) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kThreads) counts[(size_t)c * E + e] = hist[e];
  __threadfence();
  __syncthreads();
  // 3. the last CTA to finish scans and plans
  if (tid == 0) is_last = atomicAdd(done_ctr, 1u) == (unsigned)nchunks - 1u;
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // counts[c][e] -> exclusive prefix over chunks, in place.  tpe consecutive
  // lanes share an expert, each summing a contiguous run of chunks; a shuffle
  // scan over the tpe lanes joins the runs.
  int tpe = 1;
  while (tpe < 32 && tpe * E < kThreads) tpe *= 2;
  const int per_pass = kThreads / tpe;
  const int seg = moe_cdiv(nchunks, tpe);
  const int sub = tid % tpe;
  constexpr int kV = 8;  // chunk counts a thread keeps in registers
  for (int e0 = 0; e0 < E; e0 += per_pass) {
    const int e = e0 + tid / tpe;
    const bool on = e < E;
    const int c_lo = min(nchunks, sub * seg), c_hi = min(nchunks, c_lo + seg);
    int32_t v[kV];
    int32_t run = 0;
    if (seg <= kV) {
      // one round trip: the thread's whole run of chunks in flight at once
#pragma unroll
      for (int j = 0; j < kV; ++j)
        v[j] = (on && c_lo + j < c_hi) ? __ldcg(counts + (size_t)(c_lo + j) * E + e) : 0;
#pragma unroll
      for (int j = 0; j < kV; ++j) run += v[j];
    } else {
      for (int cb = c_lo; cb < c_hi; cb += kV) {
#pragma unroll
        for (int j = 0; j < kV; ++j)
          v[j] = (on && cb + j < c_hi) ? __ldcg(counts + (size_t)(cb + j) * E + e) : 0;
#pragma unroll
        for (int j = 0; j < kV; ++j) run += v[j];
      }
    }
    // exclusive scan of the runs over the expert's tpe lanes
    int32_t incl = run;
    for (int o = 1; o < tpe; o <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, incl, o, tpe);
      if (sub >= o) incl += n;
    }
    int32_t base = incl - run;
    if (on && sub == tpe - 1) tot_s[e] = incl;
    if (seg <= kV) {
#pragma unroll
      for (int j = 0; j < kV; ++j) {
        if (on && c_lo + j < c_hi) counts[(size_t)(c_lo + j) * E + e] = base;
        base += v[j];
      }
    } else {
      for (int cb = c_lo; cb < c_hi; cb += kV) {
#pragma unroll
        for (int j = 0; j < kV; ++j)
          v[j] = (on && cb + j < c_hi) ? __ldcg(counts + (size_t)(cb + j) * E + e) : 0;
#pragma unroll
        for (int j = 0; j < kV; ++j) {
          if (on && cb + j < c_hi) counts[(size_t)(cb + j) * E + e] = base;
          base += v[j];
        }
      }
    }
  }
  __syncthreads();
  // offsets: exclusive scan of the expert totals (E <= kThreads: one pass)
  {
    const int e = tid;
    const int32_t mine = e < E ? tot_s[e] : 0;
    int32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int32_t v = warp_sum[lane];
      int32_t sc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xffffffffu, sc, o);
        if (lane >= o) sc += n;
      }
      warp_sum[lane] = sc - v;
    }
    __syncthreads();
    const int32_t excl = incl - mine + warp_sum[warp];
    if (e < E) {
      off_s[e] = excl;
      offsets[e] = excl;
    }
    if (e == E - 1) {
      off_s[E] = excl + mine;
      offsets[E] = excl + mine;
    }
  }
  __syncthreads();
  plan_experts<kThreads>(off_s, E, T * K, m_skinny, dispatch, wdtype, plan_counts, plan_out,
                         block_variant);
  if (tid == 0) *done_ctr = 0u;
}

constexpr int kScatterWarps = 8;

__global__ void __launch_bounds__(32 * kScatterWarps)
route_scatter_kernel(const int32_t* __restrict__ ids, int R, int E, int chunk_reps, int nchunks,
                     const int32_t* __restrict__ bases, const int32_t* __restrict__ offsets,
                     int32_t* __restrict__ row_to_flat, int32_t* __restrict__ flat_to_row) {
  extern __shared__ int32_t cnt_all[];  // [kScatterWarps][E]
  pdl_wait();
  pdl_trigger();
  const int w = warp_id(), lane = lane_id();
  const int c = blockIdx.x * kScatterWarps + w;
  if (c >= nchunks) return;
  int32_t* cnt = cnt_all + w * E;
  for (int e = lane; e < E; e += 32) cnt[e] = __ldg(offsets + e) + __ldg(bases + (size_t)c * E + e);
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
  const int f0 = c * chunk_reps, f1 = min(R, f0 + chunk_reps);
  constexpr int kBatch = 8;
  for (int fb = f0; fb < f1; fb += 32 * kBatch) {
    int v[kBatch];  // 256 ids in flight, then placed 32 at a time in order
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int f = fb + i * 32 + lane;
      v[i] = f < f1 ? __ldg(ids + f) : -1;
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int f = fb + i * 32 + lane;
      const int e = (unsigned)v[i] < (unsigned)E ? v[i] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & lt_mask);
      const int leader = __ffs(peers) - 1;
      int base = 0;
      if (e >= 0) base = cnt[e];
      __syncwarp();
      if (e >= 0 && lane == leader) cnt[e] = base + __popc(peers);
      __syncwarp();
      if (f < f1) {
        if (e >= 0) {
          const int row = base + rank;
          row_to_flat[row] = f;
          flat_to_row[f] = row;
        } else {
          flat_to_row[f] = -1;
        }
      }
    }
  }
}

size_t prefill_smem(int tpc, int E, int K) {
  return ((size_t)tpc * K + 3 * (size_t)E + 1) * sizeof(int32_t);
}

template <int NPL, int LK, bool kGroup, bool kVec>
cudaError_t launch_one(const RoutePrefillArgs& a, int tpc, int nchunks, cudaStream_t stream) {
  const size_t smem = prefill_smem(tpc, a.E, a.K);
  PlanView pv = plan_view(a.gemm_scratch, a.T * a.K, a.E);
  PlanOut po = plan_out(pv);
  const int m_skinny = a.m_skinny < 0 ? MOE_DEFAULT_M_SKINNY : a.m_skinny;
  auto kern = route_prefill_kernel<NPL, LK, kGroup, kVec>;
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return moe_launch(kern, dim3(nchunks), dim3(kThreads), smem, stream, 1, a.logits, a.ld,
                    a.sel_bias, a.T, a.E, a.K, a.mode, a.scale, a.ids, a.weights, a.shared_gate,
                    tpc, a.counts, a.offsets, m_skinny, a.dispatch, a.wdtype, pv.counts, po,
                    a.block_variant, a.done_ctr);
}

// E <= 128: one warp per token, lists of min(K tier, experts per lane)
template <int NPL>
cudaError_t launch_warp(const RoutePrefillArgs& a, int tpc, int nchunks, cudaStream_t stream) {
#define MOE_RP_LAUNCH(KT) \
  return launch_one<NPL, (KT < NPL ? KT : NPL), false, false>(a, tpc, nchunks, stream)
  if (a.K <= 2) MOE_RP_LAUNCH(2);
  if (a.K <= 4) MOE_RP_LAUNCH(4);
  if (a.K <= 8) MOE_RP_LAUNCH(8);
  if (a.K <= 16) MOE_RP_LAUNCH(16);
  MOE_RP_LAUNCH(32);
#undef MOE_RP_LAUNCH
}

// E > 128: group_route over the warp, lists of 4 (K <= 8) or 8
template <int NPL, bool kVec>
cudaError_t launch_group(const RoutePrefillArgs& a, int tpc, int nchunks, cudaStream_t stream) {
  if (a.K <= 8) return launch_one<NPL, 4, true, kVec>(a, tpc, nchunks, stream);
  return launch_one<NPL, 8, true, kVec>(a, tpc, nchunks, stream);
}

template <bool kVec>
cudaError_t launch_group_tier(const RoutePrefillArgs& a, int tpc, int nchunks,
                              cudaStream_t stream) {
  // experts per lane: whole float4s of 4 * 32 experts per step (kVec) or
  // one expert per 32 (scalar)
  const int npl = kVec ? 4 * moe_cdiv(a.E, 128) : moe_cdiv(a.E, 32);
  if (npl <= 8) return launch_group<8, kVec>(a, tpc, nchunks, stream);
  if (npl <= 16) return launch_group<16, kVec>(a, tpc, nchunks, stream);
  if (npl <= 28) return launch_group<28, kVec>(a, tpc, nchunks, stream);
  return launch_group<32, kVec>(a, tpc, nchunks, stream);
}

}  // namespace

bool route_prefill_fits(int T, int E, int K) {
  return E <= kThreads && prefill_smem(tokens_per_cta(T), E, K) <= 200 * 1024;
}

size_t route_prefill_scratch_bytes(int T, int E) {
  // the most chunks any batch of at most T tokens uses
  const int nchunks = min(kMaxChunks, moe_cdiv(T, kWarps));
  return moe_align_up((size_t)nchunks * E * sizeof(int32_t), 256);
}

cudaError_t launch_route_prefill(const RoutePrefillArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  const int tpc = tokens_per_cta(a.T);
  const int nchunks = moe_cdiv(a.T, tpc);
  cudaError_t e;
  if (a.E > 128) {
    const bool vec = a.E % 4 == 0 && a.ld % 4 == 0 &&
                     (reinterpret_cast<uintptr_t>(a.logits) & 15) == 0;
    e = vec ? launch_group_tier<true>(a, tpc, nchunks, stream)
            : launch_group_tier<false>(a, tpc, nchunks, stream);
  } else {
    const int npl = moe_cdiv(a.E, 32);
    e = npl <= 1   ? launch_warp<1>(a, tpc, nchunks, stream)
        : npl <= 2 ? launch_warp<2>(a, tpc, nchunks, stream)
                   : launch_warp<4>(a, tpc, nchunks, stream);
  }
  if (e != cudaSuccess) return e;
  const int R = a.T * a.K;
  const size_t smem = (size_t)kScatterWarps * a.E * sizeof(int32_t);
  return moe_launch(route_scatter_kernel, dim3(moe_cdiv(nchunks, kScatterWarps)),
                    dim3(32 * kScatterWarps), smem, stream, 1, (const int32_t*)a.ids, R, a.E,
                    tpc * a.K, nchunks, (const int32_t*)a.counts, (const int32_t*)a.offsets,
                    a.row_to_flat, a.flat_to_row);
}
