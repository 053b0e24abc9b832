// Thread-per-token top-K for E <= 128 (large batches).  Same selection and
// weights as warp_topk / group_route (topk_warp.cuh, topk_group.cuh): larger
// key first, lower expert index first among equal keys; mode 0 weights are the
// softmax over the selected logits, mode 1 weights scale * s / sum s.
//
// "FlashInfer MoE routing optimisation" (flashinfer PR #4152), "why" 1: the
// lane-owned lists spread the top-K registers over a warp.  With a token's
// <= 128 keys in one thread's registers, most of that work can be skipped:
//   * tau = the KT-th largest of the 2 KT group maxima (expert e in group
//     e % 2KT; KT groups and their least maximum where 2 KT groups would not
//     fit the row).  The KT largest group maxima are KT distinct experts with
//     keys >= tau, so at least KT >= K keys are >= tau, and every expert of
//     the top K has a key >= tau.  (For random logits, E = 128, K = 8: about
//     10 candidates a token and 15 for the warp's slowest lane, against 20
//     and 39 with the least of 8 group maxima.)
//   * only the experts with key >= tau (a bit mask: for random logits a few
//     times K of them) are inserted, in rising expert order, into a sorted
//     list of KT (strictly larger keys move up, so among equal keys the lower
//     expert index stays first) -- the same K picks, bit for bit.
// A token whose keys tie heavily simply has more candidates (all of them at
// worst); the result does not change.
#pragma once

#include "topk_warp.cuh"

namespace moe_route {

// N values sorted into descending order in place (bitonic network, N a power
// of two; NaN-free inputs)
template <int N>
MOE_DEVICE void sort_desc(float (&v)[N]) {
#pragma unroll
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const float x = v[i], y = v[l];
          const bool down = (i & k) == 0;  // this block ends up descending
          v[i] = down ? fmaxf(x, y) : fminf(x, y);
          v[l] = down ? fminf(x, y) : fmaxf(x, y);
        }
      }
    }
  }
}

// NV float4 vectors of logits per row (E <= 4 NV); KT >= K list entries, KT a
// power of two with KT <= E; kVec: the row is 16-byte aligned and E % 4 == 0.
// kShared: `row` is a copy in shared memory (plain loads), else global memory
// (read-only loads).
template <int NV, int KT, bool kVec, bool kShared = false>
MOE_DEVICE void thread_topk(const float* __restrict__ row, const float* __restrict__ sel_bias,
                            int E, int K, int mode, float scale, int32_t* __restrict__ ids_out,
                            float* __restrict__ w_out) {
  auto ld = [&](int i) { return kShared ? row[i] : __ldg(row + i); };
  constexpr int kN = 4 * NV;   // experts a row may hold
  constexpr int kW = kN / 32;  // candidate mask words
  static_assert(kN % 32 == 0, "whole mask words");
  const float kNegInf = -__int_as_float(0x7f800000);
  float key[kN];
  if constexpr (kVec) {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      float4 f = make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
      if (4 * v < E)
        f = kShared ? *reinterpret_cast<const float4*>(row + 4 * v)
                    : __ldg(reinterpret_cast<const float4*>(row + 4 * v));
      key[4 * v] = f.x;
      key[4 * v + 1] = f.y;
      key[4 * v + 2] = f.z;
      key[4 * v + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kN; ++i) key[i] = i < E ? ld(i) : kNegInf;
  }
  auto sel_key = [&](float l, int e) {
    return __fadd_rn(sigmoid_key(l), sel_bias ? __ldg(sel_bias + e) : 0.f);
  };
  if (mode == MOE_SCORE_SIGMOID_BIAS_SCALED) {
#pragma unroll
    for (int i = 0; i < kN; ++i)
      if (i < E) key[i] = sel_key(key[i], i);
  }
  // the bound: with 2 KT groups, the KT-th largest of their maxima (KT
  // distinct experts reach it, so every top-K key does); with KT groups (2 KT
  // would leave groups of under one row's worth), the least maximum
  constexpr int kG = 2 * KT <= kN ? 2 * KT : KT;
  float gmax[kG];
#pragma unroll
  for (int g = 0; g < kG; ++g) gmax[g] = kNegInf;
#pragma unroll
  for (int i = 0; i < kN; ++i) gmax[i % kG] = fmaxf(gmax[i % kG], key[i]);
  float tau;
  if constexpr (kG == 2 * KT) {
    // each half sorted descending; the half-cleaner max(a_i, b_{KT-1-i})
    // keeps the KT largest of the union, the least of which is tau
    float a[KT], b[KT];
#pragma unroll
    for (int g = 0; g < KT; ++g) {
      a[g] = gmax[g];
      b[g] = gmax[KT + g];
    }
    sort_desc<KT>(a);
    sort_desc<KT>(b);
    tau = fmaxf(a[0], b[KT - 1]);
#pragma unroll
    for (int g = 1; g < KT; ++g) tau = fminf(tau, fmaxf(a[g], b[KT - 1 - g]));
  } else {
    tau = gmax[0];
#pragma unroll
    for (int g = 1; g < kG; ++g) tau = fminf(tau, gmax[g]);
  }
  uint32_t cand[kW];
#pragma unroll
  for (int w = 0; w < kW; ++w) cand[w] = 0u;
#pragma unroll
  for (int i = 0; i < kN; ++i)
    if (i < E && key[i] >= tau) cand[i / 32] |= 1u << (i % 32);

  // the candidates, in rising expert order, into a sorted list of KT
  float lk[KT];
  int li[KT];
#pragma unroll
  for (int s = 0; s < KT; ++s) {
    lk[s] = kNegInf;
    li[s] = 0x7fffffff;
  }
#pragma unroll
  for (int w = 0; w < kW; ++w) {
    uint32_t m = cand[w];
    while (m) {
      const int e = 32 * w + __ffs(m) - 1;
      m &= m - 1u;
      const float l = ld(e);
      const float k = mode == MOE_SCORE_SIGMOID_BIAS_SCALED ? sel_key(l, e) : l;
      bool b[KT];  // k belongs at or above slot s (rising with s: the list is sorted)
#pragma unroll
      for (int s = 0; s < KT; ++s) b[s] = k > lk[s];
#pragma unroll
      for (int s = KT - 1; s > 0; --s) {
        lk[s] = b[s] ? (b[s - 1] ? lk[s - 1] : k) : lk[s];
        li[s] = b[s] ? (b[s - 1] ? li[s - 1] : e) : li[s];
      }
      lk[0] = b[0] ? k : lk[0];
      li[0] = b[0] ? e : li[0];
    }
  }

  // fewer than K candidates cannot happen for finite keys; should NaN logits
  // (outside the contract) leave a slot empty, it reads expert 0, never
  // past the row
#pragma unroll
  for (int s = 0; s < KT; ++s) li[s] = (unsigned)li[s] < (unsigned)E ? li[s] : 0;
  // weights over the K picks, summed in pick order
  float v[KT];
  float sum = 0.f;
  const float m0 = ld(li[0]);  // the first pick holds the largest logit (mode 0)
#pragma unroll
  for (int s = 0; s < KT; ++s) {
    v[s] = 0.f;
    if (s < K) {
      const float l = ld(li[s]);
      v[s] = mode == MOE_SCORE_SOFTMAX_RENORM ? expf(l - m0) : sigmoid_key(l);
      sum += v[s];
    }
  }
#pragma unroll
  for (int s = 0; s < KT; ++s) {
    if (s < K) {
      ids_out[s] = li[s];
      w_out[s] = mode == MOE_SCORE_SOFTMAX_RENORM ? v[s] / sum : scale * v[s] / sum;
    }
  }
}

}  // namespace moe_route
