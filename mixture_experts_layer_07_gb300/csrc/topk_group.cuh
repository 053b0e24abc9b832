// Group top-K routing: GS lanes (8, 16 or 32) route one token, so a warp
// routes 32/GS tokens at once.  Same selection rule and weights as
// warp_topk (topk_warp.cuh): keys as order-mapped u32, larger key first,
// lower expert index first among equal keys; mode 0 weights are the softmax
// over the selected logits, mode 1 weights scale * s / sum s.
//
// "FlashInfer MoE routing optimisation" (flashinfer PR #4152), "1.
// routing_custom.cu": the candidates stay lane-owned and are merged by lane
// reductions.  What changes against one warp per token: with E <= 128 a warp
// spends most of a one-token route on K merge rounds whose cost does not
// depend on how many lanes take part, so here each round serves 32/GS tokens.
//   * Lane q of a group owns the experts of its 16-byte vectors
//     (4q + 4*GS*j + c, c < 4) -- coalesced float4 loads -- or, when the rows
//     are not 16-byte aligned, experts q + GS*p.  Either way a lane's experts
//     rise with its position p.
//   * Each lane keeps a sorted list of its best LK (key, expert) pairs,
//     built by stable insertion in p order (strictly larger keys move up).
//   * A round: group max of the list heads (shuffle butterfly, or one
//     redux.sync for a whole warp); the single lane holding it pops it.  One
//     warp-wide count of the lanes at their group's max tells whether two
//     heads are equal somewhere; only then (rare) a second reduction picks the
//     lowest expert index among them.
//   * A lane whose list runs dry while it still owns unpicked experts
//     rebuilds its list from the experts after the one it popped last
//     (key order), so LK can stay far below K.
// Key 0 marks an empty slot: order_key maps no float to 0.
#pragma once

#include "topk_warp.cuh"

namespace moe_route {

template <int GS>
MOE_DEVICE uint32_t group_max_u32(uint32_t v) {
  if constexpr (GS == 32) {
    return __reduce_max_sync(0xffffffffu, v);
  } else {
#pragma unroll
    for (int d = 1; d < GS; d <<= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, d));
    return v;
  }
}

template <int GS>
MOE_DEVICE uint32_t group_min_u32(uint32_t v) {
  if constexpr (GS == 32) {
    return __reduce_min_sync(0xffffffffu, v);
  } else {
#pragma unroll
    for (int d = 1; d < GS; d <<= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, d));
    return v;
  }
}

template <int GS>
MOE_DEVICE float group_sum_f32(float v) {
#pragma unroll
  for (int d = 1; d < GS; d <<= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Insert (nk, ne) into the sorted list (lk, le) of length LK: larger keys
// first; an equal key goes behind the entries already there (callers insert
// in rising expert order).  The entries from the insertion slot on move down
// one slot, the last drops out.  Key 0 never enters.
template <int LK>
MOE_DEVICE void list_insert(uint32_t (&lk)[LK], uint32_t (&le)[LK], uint32_t nk, uint32_t ne) {
  bool b[LK];  // nk belongs at or above slot s (rising with s: the list is sorted)
#pragma unroll
  for (int s = 0; s < LK; ++s) b[s] = nk > lk[s];
#pragma unroll
  for (int s = LK - 1; s > 0; --s) {
    lk[s] = b[s] ? (b[s - 1] ? lk[s - 1] : nk) : lk[s];
    le[s] = b[s] ? (b[s - 1] ? le[s - 1] : ne) : le[s];
  }
  lk[0] = b[0] ? nk : lk[0];
  le[0] = b[0] ? ne : le[0];
}

// This lane's logits of the token at `row` (lane q holds the experts
// expert_of(q, p), p < NPL); zeros beyond E or when !valid.  kVec: rows are
// 16-byte aligned and E is a multiple of 4 (float4 loads).
template <int GS, bool kVec>
MOE_DEVICE int group_expert_of(int q, int p) {
  return kVec ? (p >> 2) * (4 * GS) + 4 * q + (p & 3) : p * GS + q;
}

template <int GS, int NPL, bool kVec, bool kL2Only = false>
MOE_DEVICE void group_load(const float* __restrict__ row, bool valid, int E, float (&l)[NPL]) {
  static_assert(!kVec || NPL % 4 == 0, "vector lanes own whole float4s");
  const int q = lane_id() & (GS - 1);
  if constexpr (kVec) {
#pragma unroll
    for (int v = 0; v < NPL / 4; ++v) {
      const int e0 = group_expert_of<GS, true>(q, 4 * v);
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (valid && e0 < E) {
        const float4* p = reinterpret_cast<const float4*>(row + e0);
        f = kL2Only ? __ldcg(p) : __ldg(p);
      }
      l[4 * v] = f.x;
      l[4 * v + 1] = f.y;
      l[4 * v + 2] = f.z;
      l[4 * v + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int p = 0; p < NPL; ++p) {
      const int e = group_expert_of<GS, false>(q, p);
      l[p] = 0.f;
      if (valid && e < E) l[p] = kL2Only ? __ldcg(row + e) : __ldg(row + e);
    }
  }
}

// One group of GS lanes routes one token from the logits group_load gave
// (`l`; `row` is read again only for the K selected experts' weights).
// Every lane of the warp calls this; groups with valid == false take part in
// the warp's shuffles and write nothing.  nvalid: how many groups of this
// warp have valid == true.  s_ids: K shared-memory slots of this group.
template <int GS, int NPL, int LK, bool kVec, bool kL2Only = false>
MOE_DEVICE void group_route(const float (&l)[NPL], const float* __restrict__ row, bool valid,
                            int nvalid, const float* __restrict__ sel_bias, int E, int K, int mode,
                            float scale, int32_t* __restrict__ ids_out,
                            float* __restrict__ w_out, int32_t* __restrict__ ids_copy,
                            int32_t* s_ids) {
  static_assert(GS == 8 || GS == 16 || GS == 32, "group size");
  static_assert(LK >= 2 && LK <= NPL, "list no longer than the lane's experts");
  const int q = lane_id() & (GS - 1);
  auto expert_of = [&](int p) -> uint32_t { return (uint32_t)group_expert_of<GS, kVec>(q, p); };

  // ---- keys of this lane's experts (0 beyond E or for an invalid token)
  uint32_t kk[NPL];
#pragma unroll
  for (int p = 0; p < NPL; ++p) {
    const int e = (int)expert_of(p);
    float key = l[p];
    if (mode == MOE_SCORE_SIGMOID_BIAS_SCALED && valid && e < E)
      key = __fadd_rn(sigmoid_key(key), sel_bias ? __ldg(sel_bias + e) : 0.f);
    kk[p] = (valid && e < E) ? order_key(key) : 0u;
  }

  // ---- this lane's best LK, sorted
  uint32_t lk[LK], le[LK];
#pragma unroll
  for (int s = 0; s < LK; ++s) { lk[s] = 0u; le[s] = 0u; }
#pragma unroll
  for (int p = 0; p < NPL; ++p) list_insert<LK>(lk, le, kk[p], expert_of(p));

  // ---- K rounds over the group's list heads
  for (int r = 0; r < K; ++r) {
    const uint32_t hk = lk[0];
    const uint32_t m = group_max_u32<GS>(hk);
    const bool top = hk == m && hk != 0u;
    bool win = top;
    // every valid group has exactly one top lane unless two heads are equal
    if (__reduce_add_sync(0xffffffffu, top ? 1u : 0u) != (unsigned)nvalid) {
      // equal heads in some group: the lowest expert index among them
      const uint32_t mi = group_min_u32<GS>(top ? le[0] : 0xffffffffu);
      win = top && le[0] == mi;
    }
    const uint32_t pk = lk[0], pe = le[0];
    if (win) {
      s_ids[r] = (int32_t)pe;
#pragma unroll
      for (int s = 0; s < LK - 1; ++s) { lk[s] = lk[s + 1]; le[s] = le[s + 1]; }
      lk[LK - 1] = 0u;
      le[LK - 1] = 0u;
    }
    if constexpr (NPL > LK) {
      // a lane that popped its last listed entry rebuilds the list from the
      // experts after that entry in key order (none left: it stays empty)
      const bool refill = win && lk[0] == 0u;
      if (__any_sync(0xffffffffu, refill) && refill) {
#pragma unroll
        for (int p = 0; p < NPL; ++p) {
          const uint32_t e = expert_of(p);
          const bool after = kk[p] < pk || (kk[p] == pk && e > pe);
          list_insert<LK>(lk, le, after ? kk[p] : 0u, e);
        }
      }
    }
  }
  __syncwarp();

  // ---- weights: lane q takes slots q, q + GS, ... (at most 4 with K <= 32)
  float v[4];
  int id[4];
  float local = 0.f;
  float m0 = 0.f;
  if (valid && mode == MOE_SCORE_SOFTMAX_RENORM) {
    const int i0 = s_ids[0];  // the first pick holds the largest logit
    m0 = kL2Only ? __ldcg(row + i0) : __ldg(row + i0);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = q + i * GS;
    v[i] = 0.f;
    id[i] = 0;
    if (valid && r < K) {
      id[i] = s_ids[r];
      const float x = kL2Only ? __ldcg(row + id[i]) : __ldg(row + id[i]);
      v[i] = mode == MOE_SCORE_SOFTMAX_RENORM ? expf(x - m0) : sigmoid_key(x);
      local += v[i];
    }
  }
  const float sum = group_sum_f32<GS>(local);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = q + i * GS;
    if (valid && r < K) {
      ids_out[r] = id[i];
      w_out[r] = mode == MOE_SCORE_SOFTMAX_RENORM ? v[i] / sum : scale * v[i] / sum;
      if (ids_copy) ids_copy[r] = id[i];
    }
  }
  __syncwarp();  // s_ids is reused by the group's next token
}

}  // namespace moe_route
