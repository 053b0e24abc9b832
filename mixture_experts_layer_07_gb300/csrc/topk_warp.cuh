// Warp-level top-K routing shared by the routing kernels (method and sources
// in topk_route.cu).  The sigmoid used as the selection key is one fixed
// float32 formula, each step a single correctly rounded operation (never
// contracted to an FMA):
//   exp(z): n = rint(z*log2e); r = (z - n*ln2_hi) - n*ln2_lo (Cody-Waite);
//           p = degree-7 Taylor polynomial of e^r (Horner); exp = p * 2^n
//   sigmoid(l) = 1 / (1 + exp(-l)), with 0 for -l > 88 and 1 for -l < -87
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe_route {

// float32 constants of the formula above, each the float32 nearest the value
// named (ln2_hi keeps 15 significant bits so n * ln2_hi is exact)
static __device__ __constant__ float kLog2e = 0x1.715476p+0f;     // log2(e)
static __device__ __constant__ float kLn2Hi = 0x1.62e4p-1f;       // 0.693145751953125
static __device__ __constant__ float kLn2Lo = 0x1.7f7d1cp-20f;    // ln2 - ln2_hi
static __device__ __constant__ float kTaylor[8] = {
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

// Keys are compared as unsigned integers: non-negative floats map to
// bits + 2^31, negative floats to 2^32 - bits (two's complement negation).
// The map is monotone (larger magnitude further out), -0 and +0 both land on
// 2^31, and no float (not even a NaN pattern) maps to 0, so 0 can mark an
// empty slot.
MOE_DEVICE uint32_t order_key(float k) {
  const uint32_t b = __float_as_uint(k);
  return (b & 0x80000000u) ? 0u - b : (b | 0x80000000u);
}

// the float whose order_key is k (exact inverse; -0 comes back as +0)
MOE_DEVICE float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : 0u - k);
}

// strict total order: larger key first, lower index first among equal keys
MOE_DEVICE bool better(uint32_t ka, int ia, uint32_t kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// One warp routes one token: `row` holds the token's logits (at least E of
// them); writes ids[0..K) and weights[0..K).  Every lane of the warp calls it.
// kL2Only: read the logits through L2 only (they were written earlier in the
// same kernel by other CTAs); ids_copy (nullable) receives the ids as well.
template <int NPL, int LK, bool kL2Only = false>
MOE_DEVICE void warp_topk(const float* __restrict__ row, const float* __restrict__ sel_bias,
                          int E, int K, int mode, float scale, int32_t* __restrict__ ids_out,
                          float* __restrict__ w_out, int32_t* ids_copy = nullptr) {
  auto ld = [&](int i) { return kL2Only ? __ldcg(row + i) : __ldg(row + i); };
  const int lane = lane_id();

  // lane-owned sorted candidate list (keys as ordered u32, empty slots lowest)
  uint32_t lk[LK];
  int li[LK];
#pragma unroll
  for (int s = 0; s < LK; ++s) { lk[s] = 0u; li[s] = 0x7fffffff; }

#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = j * 32 + lane;
    if (e < E) {
      const float l = ld(e);
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
  uint32_t my_key = 0u;
  for (int r = 0; r < K; ++r) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, lk[0]);
    const uint32_t mi = __reduce_min_sync(0xffffffffu, lk[0] == m ? (uint32_t)li[0] : 0xffffffffu);
    if (li[0] == (int)mi) {
#pragma unroll
      for (int s = 0; s < LK - 1; ++s) { lk[s] = lk[s + 1]; li[s] = li[s + 1]; }
      lk[LK - 1] = 0u;
      li[LK - 1] = 0x7fffffff;
    }
    if (lane == r) {
      my_id = (int)mi;
      my_key = m;
    }
  }

  float v = 0.f;
  if (mode == MOE_SCORE_SOFTMAX_RENORM) {
    // a pick's key is its logit (mode 0): no second read of the row
    const float l = lane < K ? key_float(my_key) : 0.f;
    const float m = __shfl_sync(0xffffffffu, l, 0);  // the first pick is the largest
    v = lane < K ? expf(l - m) : 0.f;
  } else {
    v = lane < K ? sigmoid_key(ld(my_id)) : 0.f;
  }
  float sum = v;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < K) {
    const float w = mode == MOE_SCORE_SOFTMAX_RENORM ? v / sum : scale * v / sum;
    ids_out[lane] = my_id;
    w_out[lane] = w;
    if (ids_copy) ids_copy[lane] = my_id;
  }
}

}  // namespace moe_route
