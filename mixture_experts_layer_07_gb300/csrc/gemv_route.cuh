// The batch's routing inside one CTA of the matrix-vector decode path (G1's
// prologue in gemv_decode.cu): top-K per token, the stable permutation of the
// replicas and the skinny plan, in shared memory, CTA 0 also writing them to
// the workspace.  A header so that the host emulation of the SIMT primitives
// (tests/host_emu) can run it lane by lane against a stable sort.
#pragma once

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"
#include "topk_warp.cuh"

namespace moe_gemv_route {

// The batch's routing inside a G1 CTA (kRoute).  E <= 128: warps 0..T-1
// route one token each from the logits (warp_topk, the selection and weights
// of the routing kernels).  E > 128: each token's experts are split over
// S = 8 / T' warps (T' = T rounded up to a power of two) in lane-strided
// slices; every warp picks its slice's K best (key, expert) pairs, then one
// warp per token picks the K best of those S * K candidates -- the exact
// top-K under the same order (larger key first, lower expert first among
// equal keys) -- and turns them into weights by the formula warp_topk uses.
// Then warp 0 sorts the R = T*K <= 32 replicas stably by expert with lane
// ballots: replica f (lane f, expert e) goes to row (replicas with a smaller
// expert) + (earlier replicas with expert e), the counting-sort permutation
// of the permute stage; each expert's first replica writes its skinny item
// {e, first row, rows, 0} at (experts below e that occur).  CTA 0 writes
// everything the later launches and the workspace hold: ids, weights, shared
// gate, offsets, both permutation maps, per-expert variant and the plan
// (every occurring expert is skinny: m <= T <= m_skinny).
constexpr int kRouteWarps = 8;  // the warps of a routing CTA
constexpr int kRouteSlicesMax = kRouteWarps;
struct RouteSmem {
  int32_t ids[32];
  float w[32];
  int4 items[32];
  int32_t r2f[32];
  uint32_t ck[kGemvMaxT][kRouteSlicesMax * 16];  // E > 128: the slices' picks
  int32_t ci[kGemvMaxT][kRouteSlicesMax * 16];
  int n_items;
};

// A warp's K best candidates: lane l holds keys ck[j] (0: none) of distinct
// experts ci[j], j < N.  Each lane first sorts its candidates into a list
// (larger key first, lower expert first among equal keys: warp_topk's
// order); then K rounds: the warp's largest head key by one max-reduction,
// the lowest expert among heads at that key by one min-reduction, and the
// owning lane pops its head.  Lane r < K ends with pick r.
template <int N>
MOE_DEVICE void warp_pick(int K, const uint32_t (&ck)[N], const int (&ci)[N], uint32_t& my_key,
                          int& my_id) {
  using moe_route::better;
  const int lane = lane_id();
  uint32_t lk[N];
  int li[N];
#pragma unroll
  for (int s = 0; s < N; ++s) {
    lk[s] = 0u;
    li[s] = 0x7fffffff;
  }
#pragma unroll
  for (int j = 0; j < N; ++j) {
    if (ck[j] != 0u) {
      uint32_t nk = ck[j];
      int ni = ci[j];
#pragma unroll
      for (int s = 0; s < N; ++s) {
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
  my_id = -1;
  my_key = 0u;
  for (int r = 0; r < K; ++r) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, lk[0]);
    const uint32_t mi = __reduce_min_sync(0xffffffffu, lk[0] == m ? (uint32_t)li[0] : 0xffffffffu);
    if (li[0] == (int)mi) {
#pragma unroll
      for (int s = 0; s < N - 1; ++s) {
        lk[s] = lk[s + 1];
        li[s] = li[s + 1];
      }
      lk[N - 1] = 0u;
      li[N - 1] = 0x7fffffff;
    }
    if (lane == r) {
      my_id = (int)mi;
      my_key = m;
    }
  }
}

// One slice of a token's experts (sl*32 + lane + 32*S*j, j < N, below E):
// keys as warp_topk forms them, the slice's K best by warp_pick
template <int N>
MOE_DEVICE void slice_pick(const GemvRoute& rt, const float* row, int sl, int S, int K,
                           uint32_t& my_key, int& my_id) {
  const int lane = lane_id();
  float l[N];
  uint32_t ck[N];
  int ci[N];
#pragma unroll
  for (int j = 0; j < N; ++j) {  // every load first
    ci[j] = sl * 32 + lane + j * 32 * S;
    l[j] = ci[j] < rt.E ? __ldcg(row + ci[j]) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < N; ++j) {
    ck[j] = 0u;
    if (ci[j] < rt.E) {
      float key = l[j];
      if (rt.mode == MOE_SCORE_SIGMOID_BIAS_SCALED)
        key = __fadd_rn(moe_route::sigmoid_key(l[j]), rt.sel_bias ? __ldg(rt.sel_bias + ci[j]) : 0.f);
      ck[j] = moe_route::order_key(key);
    }
  }
  warp_pick<N>(K, ck, ci, my_key, my_id);
}

// the weights of the K picks (lane r: pick r) by warp_topk's formula; ids and
// weights to ids_out / w_out, the ids also to ids_copy (nullable)
MOE_DEVICE void pick_weights(uint32_t my_key, int my_id, const float* row, int K, int mode,
                             float scale, int32_t* ids_out, float* w_out, int32_t* ids_copy) {
  const int lane = lane_id();
  float v;
  if (mode == MOE_SCORE_SOFTMAX_RENORM) {
    const float l = lane < K ? moe_route::key_float(my_key) : 0.f;
    const float m = __shfl_sync(0xffffffffu, l, 0);  // the first pick is the largest
    v = lane < K ? expf(l - m) : 0.f;
  } else {
    v = lane < K ? moe_route::sigmoid_key(__ldcg(row + my_id)) : 0.f;
  }
  float sum = v;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < K) {
    ids_out[lane] = my_id;
    w_out[lane] = mode == MOE_SCORE_SOFTMAX_RENORM ? v / sum : scale * v / sum;
    if (ids_copy) ids_copy[lane] = my_id;
  }
}

// stage(from): threads from.. of the CTA stage the token rows
template <typename Stage>
MOE_DEVICE void gemv_route(const GemvRoute& rt, int T, int K, int wdtype, RouteSmem& rs,
                           Stage stage) {
  const int warp = warp_id(), lane = lane_id();
  const bool cta0 = blockIdx.x == 0;
  if (rt.E <= 128) {
    if (warp < T) {
      const float* row = rt.logits + (size_t)warp * rt.G;
      if (cta0)
        moe_route::warp_topk<4, 4, true>(row, rt.sel_bias, rt.E, K, rt.mode, rt.scale,
                                         rt.ids + (size_t)warp * K,
                                         rt.weights + (size_t)warp * K, rs.ids + warp * K);
      else
        moe_route::warp_topk<4, 4, true>(row, rt.sel_bias, rt.E, K, rt.mode, rt.scale,
                                         rs.ids + warp * K, rs.w + warp * K);
    } else {
      stage(32 * T);
    }
  } else {
    const int S = kRouteWarps / (T == 1 ? 1 : T == 2 ? 2 : 4);
    const int t = warp / S, sl = warp % S;
    if (t < T) {
      const float* row = rt.logits + (size_t)t * rt.G;
      // candidates per lane: the largest count of any slice, rounded up
      const int npl = (rt.E + 32 * S - 1) / (32 * S);
      uint32_t mk;
      int mi;
      if (npl <= 2)
        slice_pick<2>(rt, row, sl, S, K, mk, mi);
      else if (npl <= 4)
        slice_pick<4>(rt, row, sl, S, K, mk, mi);
      else if (npl <= 8)
        slice_pick<8>(rt, row, sl, S, K, mk, mi);
      else
        slice_pick<16>(rt, row, sl, S, K, mk, mi);
      if (lane < K) {
        rs.ck[t][sl * K + lane] = mk;
        rs.ci[t][sl * K + lane] = mi;
      }
    }
    stage(0);
    __syncthreads();
    if (warp < T) {
      const float* row = rt.logits + (size_t)warp * rt.G;
      const int n = S * K;  // at most 128
      uint32_t ck[4];
      int ci[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = j * 32 + lane;
        ck[j] = c < n ? rs.ck[warp][c] : 0u;
        ci[j] = c < n ? rs.ci[warp][c] : 0x7fffffff;
      }
      uint32_t mk;
      int mi;
      warp_pick<4>(K, ck, ci, mk, mi);
      if (cta0)
        pick_weights(mk, mi, row, K, rt.mode, rt.scale, rt.ids + (size_t)warp * K,
                     rt.weights + (size_t)warp * K, rs.ids + warp * K);
      else
        pick_weights(mk, mi, row, K, rt.mode, rt.scale, rs.ids + warp * K, rs.w + warp * K,
                     nullptr);
    }
  }
  if (cta0 && rt.shared_gate && warp < T && lane == 0)
    rt.shared_gate[warp] = moe_route::sigmoid_key(__ldcg(rt.logits + (size_t)warp * rt.G + rt.E));
  __syncthreads();
  const int R = T * K;
  if (warp != 0) {
    // CTA 0's other warps: the offsets and the per-expert variants
    if (cta0) {
      for (int x = (int)threadIdx.x - 32; x <= rt.E; x += (int)blockDim.x - 32) {
        int lt = 0, eq = 0;
        for (int g = 0; g < R; ++g) {
          const int eg = rs.ids[g];
          lt += eg < x;
          eq += eg == x;
        }
        rt.offsets[x] = lt;
        if (x < rt.E)
          rt.block_variant[x] = moe_variant_of(eq, R, rt.E, rt.m_skinny, rt.dispatch, wdtype);
      }
    }
    return;
  }
  const int e = lane < R ? rs.ids[lane] : 0x7fffffff;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  const bool lead = lane < R && rank == 0;
  const unsigned leads = __ballot_sync(0xffffffffu, lead);
  int less = 0, idx = 0;
  for (int g = 0; g < R; ++g) {
    const int eg = __shfl_sync(0xffffffffu, e, g);
    less += eg < e;
    idx += (eg < e) && ((leads >> g) & 1u);
  }
  const int row = less + rank;
  if (lane < R) {
    rs.r2f[row] = lane;
    if (cta0) {
      rt.row_to_flat[row] = lane;
      rt.flat_to_row[lane] = row;
    }
  }
  if (lead) {
    const int4 it = make_int4(e, less, __popc(peers), 0);
    rs.items[idx] = it;
    if (cta0) {
      rt.plan_items[idx] = it;
      rt.plan_done[idx] = 0;
    }
  }
  if (lane == 0) rs.n_items = __popc(leads);
  if (cta0) {
    if (lane < moe_plan::kLists) rt.plan_counts[lane] = lane == 0 ? __popc(leads) : 0;
    if (lane < 2 * moe_plan::kLists) rt.plan_counts[moe_plan::kSchedBase + lane] = 0;
  }
}

}  // namespace moe_gemv_route
