// Host emulation of the top-K device code (topk_group.cuh, topk_warp.cuh).
//
// One warp is 32 host threads (simt_emu.h): every warp-collective intrinsic
// the routing code uses (shuffle, redux, ballot, any, syncwarp) is a write to
// a shared slot array between two barriers, so the threads run the device
// source itself, lane by lane, on the CPU.  The selection is checked against a
// stable sort of the same keys (larger first, lower expert index first among
// equal keys), for float4 and scalar rows, groups of 8, 16 and 32 lanes,
// random, tie-heavy and "one lane owns every pick" logits, both score modes;
// and the one-warp-per-token route (warp_topk) on random and tie-heavy rows.
// Exit status 0 when every token matches.
#include <cstdio>
#include <numeric>
#include <random>

#include "simt_emu.h"
#include "topk_group.cuh"

using namespace moe_route;

// one warp routes tokens t0 .. t0 + 32/GS - 1
template <int GS, int NPL, int LK, bool kVec>
void run_warp(const float* logits, int ld, const float* bias, int T, int E, int K, int mode,
              int t0, int32_t* ids, float* w) {
  std::vector<int32_t> slots(32 * K);
  emu_run_cta(32, [&]() {
    const int g = simt_emu::lane / GS;
    const int t = t0 + g;
    const bool valid = t < T;
    const int nvalid = std::min(T - t0, 32 / GS);
    const float* row = logits + (size_t)(valid ? t : 0) * ld;
    float l[NPL];
    group_load<GS, NPL, kVec>(row, valid, E, l);
    group_route<GS, NPL, LK, kVec>(l, row, valid, nvalid, bias, E, K, mode, 2.5f,
                                   ids + (size_t)t * K, w + (size_t)t * K, nullptr,
                                   slots.data() + g * K);
  });
}

// pattern 0: normal logits; 1: values from {-1, 0, 1} (ties decided by index);
// 2: +20 on the experts lane 0 of each group owns (that lane supplies every
// pick); 3: as 2 with every other logit 0, so lane 0's experts all tie and
// its list rebuilds across equal keys
template <int GS, int NPL, int LK, bool kVec>
int check(int E, int K, int G, int T, int mode, int pattern, unsigned seed) {
  std::mt19937 rng(seed);
  std::normal_distribution<float> nd(0.f, 1.f);
  std::vector<float> lg((size_t)T * G), bias(E);
  for (auto& v : lg) v = pattern == 1 ? (float)((int)(rng() % 3) - 1) : pattern == 3 ? 0.f : nd(rng);
  for (auto& v : bias) v = mode ? 0.3f * nd(rng) : 0.f;
  if (pattern >= 2)
    for (int t = 0; t < T; ++t)
      for (int e = 0; e < E; ++e)
        if (kVec ? ((e % (4 * GS)) / 4 == 0) : (e % GS == 0)) lg[(size_t)t * G + e] += 20.f;
  std::vector<int32_t> ids((size_t)T * K, -1);
  std::vector<float> w((size_t)T * K);
  for (int t0 = 0; t0 < T; t0 += 32 / GS)
    run_warp<GS, NPL, LK, kVec>(lg.data(), G, mode ? bias.data() : nullptr, T, E, K, mode, t0,
                                ids.data(), w.data());
  int bad = 0;
  for (int t = 0; t < T; ++t) {
    const float* r = lg.data() + (size_t)t * G;
    std::vector<float> key(E);
    for (int e = 0; e < E; ++e) key[e] = mode ? __fadd_rn(sigmoid_key(r[e]), bias[e]) : r[e];
    std::vector<int> idx(E);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return key[a] > key[b]; });
    float wsum = 0.f;
    for (int k = 0; k < K; ++k) {
      if (ids[(size_t)t * K + k] != idx[k]) {
        if (!bad) printf("  token %d pick %d: %d, expected %d\n", t, k, ids[(size_t)t * K + k], idx[k]);
        ++bad;
        break;
      }
      wsum += w[(size_t)t * K + k];
    }
    if (std::fabs(wsum - (mode ? 2.5f : 1.f)) > 1e-5f * K) ++bad;
  }
  printf("GS=%d NPL=%d LK=%d vec=%d E=%d K=%d G=%d mode=%d pattern=%d: %d of %d tokens wrong\n",
         GS, NPL, LK, (int)kVec, E, K, G, mode, pattern, bad, T);
  return bad;
}

// the one-warp-per-token route (warp_topk, topk_warp.cuh) on the same inputs
template <int NPL, int LK>
int check_warp(int E, int K, int G, int T, int mode, int pattern, unsigned seed) {
  std::mt19937 rng(seed);
  std::normal_distribution<float> nd(0.f, 1.f);
  std::vector<float> lg((size_t)T * G), bias(E);
  for (auto& v : lg) v = pattern == 1 ? (float)((int)(rng() % 3) - 1) : nd(rng);
  for (auto& v : bias) v = mode ? 0.3f * nd(rng) : 0.f;
  std::vector<int32_t> ids((size_t)T * K, -1);
  std::vector<float> w((size_t)T * K);
  for (int t = 0; t < T; ++t)
    emu_run_cta(32, [&]() {
      warp_topk<NPL, LK>(lg.data() + (size_t)t * G, mode ? bias.data() : nullptr, E, K, mode,
                         2.5f, ids.data() + (size_t)t * K, w.data() + (size_t)t * K);
    });
  int bad = 0;
  for (int t = 0; t < T; ++t) {
    const float* r = lg.data() + (size_t)t * G;
    std::vector<float> key(E);
    for (int e = 0; e < E; ++e) key[e] = mode ? __fadd_rn(sigmoid_key(r[e]), bias[e]) : r[e];
    std::vector<int> idx(E);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return key[a] > key[b]; });
    for (int k = 0; k < K; ++k)
      if (ids[(size_t)t * K + k] != idx[k]) { ++bad; break; }
  }
  printf("warp NPL=%d LK=%d E=%d K=%d mode=%d pattern=%d: %d of %d tokens wrong\n", NPL, LK, E,
         K, mode, pattern, bad, T);
  return bad;
}

int main() {
  int bad = 0;
  for (int pat = 0; pat < 4; ++pat) {
    bad += check<8, 16, 4, true>(128, 8, 128, 16, 0, pat, 11 + pat);
    bad += check<8, 16, 4, false>(128, 8, 129, 16, 1, pat, 21 + pat);
    bad += check<8, 4, 4, true>(32, 4, 32, 16, 0, pat, 31 + pat);
    bad += check<16, 16, 8, false>(256, 16, 257, 8, 1, pat, 41 + pat);
    bad += check<32, 16, 8, false>(512, 10, 513, 8, 0, pat, 51 + pat);
    bad += check<32, 28, 8, true>(896, 16, 896, 4, 1, pat, 61 + pat);
  }
  for (int pat = 0; pat < 2; ++pat) {
    bad += check_warp<4, 4>(128, 8, 128, 8, 0, pat, 71 + pat);
    bad += check_warp<1, 1>(8, 2, 8, 8, 1, pat, 81 + pat);
    bad += check_warp<16, 10>(512, 10, 513, 4, 0, pat, 91 + pat);
    bad += check_warp<28, 16>(896, 16, 896, 2, 1, pat, 101 + pat);
  }
  printf("%s\n", bad ? "FAIL" : "OK");
  return bad != 0;
}
