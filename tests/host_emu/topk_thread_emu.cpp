// Host run of the thread-per-token top-K (csrc/topk_thread.cuh): the device
// routine compiled for the CPU (rows read as global and as shared-memory
// copies), one token at a time, checked against a stable
// sort of the same keys (larger first, lower expert index first among equal
// keys) for every (E, K) shape it serves, float4 and scalar rows, both score
// modes, and random, tie-heavy, all-equal and "top experts in one bound
// group" logits (for both groupings the bound may use).  Exit status 0 when every token matches.
#include <cstdio>
#include <numeric>
#include <random>

#include "simt_emu.h"
#include "topk_thread.cuh"

using namespace moe_route;

template <int NV, int KT, bool kVec, bool kShared>
int check(int E, int K, int T, int mode, int pattern, unsigned seed) {
  std::mt19937 rng(seed);
  std::normal_distribution<float> nd(0.f, 1.f);
  const int ld = kVec ? (E + 3) / 4 * 4 : E + 1;
  std::vector<float> lg((size_t)T * ld + 4, 0.f), bias(E);
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      float v = nd(rng);
      if (pattern == 1) v = (float)((int)(rng() % 3) - 1);
      if (pattern == 2) v = 0.f;
      if (pattern == 3 && e % KT == 0) v += 20.f;  // every pick from bound group 0
      if (pattern == 4 && e % (2 * KT) == 0) v += 20.f;  // ... of the 2 KT grouping
      lg[(size_t)t * ld + e] = v;
    }
  for (auto& v : bias) v = mode ? 0.3f * nd(rng) : 0.f;
  int bad = 0;
  std::vector<int32_t> ids(K);
  std::vector<float> w(K);
  for (int t = 0; t < T; ++t) {
    const float* row = lg.data() + (size_t)t * ld;
    thread_topk<NV, KT, kVec, kShared>(row, mode ? bias.data() : nullptr, E, K, mode, 2.5f,
                                       ids.data(), w.data());
    std::vector<float> key(E);
    for (int e = 0; e < E; ++e)
      key[e] = mode ? __fadd_rn(sigmoid_key(row[e]), bias[e]) : row[e];
    std::vector<int> ord(E);
    std::iota(ord.begin(), ord.end(), 0);
    std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return key[a] > key[b]; });
    double sw = 0.0;
    for (int k = 0; k < K; ++k) {
      if (ids[k] != ord[k]) ++bad;
      sw += w[k];
    }
    const double want = mode ? 2.5 : 1.0;
    if (std::abs(sw - want) > 1e-5 * want) ++bad;
  }
  if (bad)
    std::printf("MISMATCH NV=%d KT=%d vec=%d E=%d K=%d mode=%d pattern=%d: %d\n", NV, KT, kVec, E,
                K, mode, pattern, bad);
  return bad;
}

template <int NV, int KT, bool kVec>
int sweep(int E, int K) {
  int bad = 0;
  for (int mode = 0; mode < 2; ++mode)
    for (int pattern = 0; pattern < 5; ++pattern)
      bad += check<NV, KT, kVec, false>(E, K, 300, mode, pattern, 1000u * E + 10u * K + pattern) +
             check<NV, KT, kVec, true>(E, K, 100, mode, pattern, 7u * E + 3u * K + pattern);
  return bad;
}

int main() {
  int bad = 0;
  bad += sweep<32, 8, true>(128, 8);
  bad += sweep<32, 8, false>(128, 8);
  bad += sweep<32, 8, true>(100, 7);
  bad += sweep<32, 8, false>(97, 5);
  bad += sweep<8, 4, true>(32, 4);
  bad += sweep<8, 4, false>(33 - 1, 3);
  bad += sweep<16, 8, true>(64, 6);
  bad += sweep<16, 32, true>(64, 32);
  bad += sweep<8, 8, true>(8, 8);
  bad += sweep<8, 2, false>(8, 2);
  bad += sweep<32, 16, true>(128, 16);
  bad += sweep<32, 32, false>(128, 32);
  std::printf("%s\n", bad ? "FAIL" : "OK");
  return bad ? 1 : 0;
}
