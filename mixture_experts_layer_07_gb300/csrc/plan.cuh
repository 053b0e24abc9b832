// Device-side plan of the grouped expert GEMM: for every expert block its
// m_size from the offsets, the kernel variant chosen from it (per block), and
// the work lists the GEMM kernels walk.  Shared by the standalone plan kernel
// and the fused decode routing kernel.
#pragma once

#include "common.cuh"

namespace moe_plan {

constexpr int kBnSkinny = 16;
constexpr int kBnTile = 128;
constexpr int kBnWide = 256;
constexpr int kLists = 3;  // skinny, tile, wide
__host__ __device__ constexpr int list_bn(int l) { return l == 0 ? kBnSkinny : l == 1 ? kBnTile : kBnWide; }
// scratch layout: counts[kLists] and the GEMM launches' work counters
// (counts[kSchedBase + 2*list + {0: G1, 1: G2}], zeroed by every plan) in a
// 256-byte head, then one int4 item list per variant
constexpr int kSchedBase = 8;
struct PlanView {
  int32_t* counts;          // items per list
  int4* items[kLists];      // {block, first row, rows, 0}
  int32_t* done[kLists];    // per item: finished G1 epilogue warps (fused launch)
  int cap[kLists];
};

// bytes of the plan for R rows in E_blocks blocks (the layout plan_view reads)
inline size_t plan_bytes(int R, int E_blocks) {
  size_t b = 256;
  for (int l = 0; l < kLists; ++l) {
    const size_t cap = (size_t)moe_cdiv(R, list_bn(l)) + E_blocks;
    b += moe_align_up(cap * sizeof(int4), 256) + moe_align_up(cap * sizeof(int32_t), 256);
  }
  return b;
}

inline PlanView plan_view(void* scratch, int R, int E_blocks) {
  PlanView v;
  char* p = static_cast<char*>(scratch);
  v.counts = reinterpret_cast<int32_t*>(p);
  size_t off = 256;
  for (int l = 0; l < kLists; ++l) {
    v.cap[l] = moe_cdiv(R, list_bn(l)) + E_blocks;
    v.items[l] = reinterpret_cast<int4*>(p + off);
    off += moe_align_up((size_t)v.cap[l] * sizeof(int4), 256);
    v.done[l] = reinterpret_cast<int32_t*>(p + off);
    off += moe_align_up((size_t)v.cap[l] * sizeof(int32_t), 256);
  }
  return v;
}

struct PlanOut {
  int4* items[kLists];
  int32_t* done[kLists];
};

inline PlanOut plan_out(const PlanView& v) {
  PlanOut o;
  for (int l = 0; l < kLists; ++l) {
    o.items[l] = v.items[l];
    o.done[l] = v.done[l];
  }
  return o;
}

// Plan for E_blocks blocks by one CTA of NT threads (NT a multiple of 32, at
// most 1024).  offsets == nullptr: a single block [0, R).
template <int NT>
MOE_DEVICE void plan_experts(const int32_t* offsets, int E_blocks, int R, int m_skinny,
                             int dispatch, int wdtype, int32_t* __restrict__ counts,
                             const PlanOut& out, int32_t* __restrict__ block_variant) {
  __shared__ int wsum[kLists][32];
  __shared__ int carry[kLists];
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  constexpr int kWarps = NT / 32;
  if (tid < kLists) carry[tid] = 0;
  __syncthreads();
  for (int base = 0; base < E_blocks; base += NT) {
    const int e = base + tid;
    int lo = 0, m = 0;
    if (e < E_blocks) {
      lo = offsets ? offsets[e] : 0;
      m = (offsets ? offsets[e + 1] : R) - lo;
    }
    const int v = e < E_blocks ? moe_variant_of(m, R, E_blocks, m_skinny, dispatch, wdtype)
                               : MOE_VARIANT_SKIP;
    const int list = (v == MOE_VARIANT_SKINNY || v == MOE_VARIANT_SIMT) ? 0
                   : v == MOE_VARIANT_TILE ? 1 : v == MOE_VARIANT_WIDE ? 2 : -1;
    int n[kLists], incl[kLists];
#pragma unroll
    for (int l = 0; l < kLists; ++l) {
      n[l] = (l == list) ? moe_cdiv(m, list_bn(l)) : 0;
      incl[l] = n[l];
    }
    // block-wide exclusive scans of the per-list item counts
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
      for (int l = 0; l < kLists; ++l) {
        const int a = __shfl_up_sync(0xffffffffu, incl[l], o);
        if (lane >= o) incl[l] += a;
      }
    }
    if (lane == 31) {
#pragma unroll
      for (int l = 0; l < kLists; ++l) wsum[l][warp] = incl[l];
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int l = 0; l < kLists; ++l) {
        const int a = lane < kWarps ? wsum[l][lane] : 0;
        int sc = a;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int x = __shfl_up_sync(0xffffffffu, sc, o);
          if (lane >= o) sc += x;
        }
        if (lane < kWarps) wsum[l][lane] = sc - a;
      }
    }
    __syncthreads();
    if (list >= 0) {
      const int bn = list_bn(list);
      const int pos = carry[list] + wsum[list][warp] + incl[list] - n[list];
      for (int i = 0; i < n[list]; ++i) {
        out.items[list][pos + i] = make_int4(e, lo + i * bn, min(bn, m - i * bn), 0);
        out.done[list][pos + i] = 0;
      }
    }
    if (block_variant && e < E_blocks) block_variant[e] = v;
    __syncthreads();
    if (tid == NT - 1) {
#pragma unroll
      for (int l = 0; l < kLists; ++l) carry[l] += wsum[l][kWarps - 1] + incl[l];
    }
    __syncthreads();
  }
  if (tid < kLists) counts[tid] = carry[tid];
  if (tid < 2 * kLists) counts[kSchedBase + tid] = 0;
}

}  // namespace moe_plan
