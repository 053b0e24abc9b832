// Host run of the matrix-vector decode path's in-CTA routing
// (csrc/gemv_route.cuh): one CTA of 8 warps routes a batch of T <= 4 tokens
// from its logits, as CTA 0 (which also writes the workspace) and as another
// CTA (shared memory only).  Checked against plain host definitions: the K
// picks of every token = the first K of a stable sort of its keys (larger
// first, lower expert first among equal keys); weights that sum to 1 (or to
// the scale) and follow the pick order; offsets, row_to_flat and flat_to_row
// = the stable counting sort of the T*K replicas by expert; the skinny plan =
// one item {expert, first row, rows, 0} per occurring expert in rising order;
// the per-expert variants = moe_variant_of of each expert's row count.  Both
// paths (E <= 128: a warp per token; E > 128: slices over 8 / T' warps, then
// a merge), both score modes, random and tie-heavy logits.  Exit status 0
// when everything matches.
#include <cstdio>
#include <numeric>
#include <random>
#include "simt_emu.h"
#include "common.cuh"
#define blockIdx emu_block_idx
#define blockDim emu_block_dim
#include "gemv_route.cuh"
using namespace moe_gemv_route;

int check(int T, int E, int K, int mode, int pattern, unsigned seed) {
  std::mt19937 rng(seed);
  std::normal_distribution<float> nd(0.f, 1.f);
  const int G = E + 1;  // one more column: the shared gate
  std::vector<float> lg((size_t)T * G), bias(E);
  for (auto& v : lg) v = pattern ? (float)((int)(rng() % 5) - 2) : nd(rng);
  for (auto& v : bias) v = mode ? 0.3f * nd(rng) : 0.f;
  const int R = T * K;
  int bad = 0;
  for (int cta = 0; cta < 2; ++cta) {
    std::vector<int32_t> ids(R, -7), r2f(R, -7), f2r(R, -7), off(E + 1, -7), bv(E, -7);
    std::vector<float> w(R, -7.f), sg(T, -7.f);
    std::vector<int32_t> counts(16, -7), done(64, -7);
    std::vector<int4> items(64, make_int4(-7, -7, -7, -7));
    GemvRoute rt{};
    rt.logits = lg.data(); rt.G = G; rt.E = E; rt.mode = mode; rt.scale = 2.5f;
    rt.sel_bias = mode ? bias.data() : nullptr; rt.ids = ids.data(); rt.weights = w.data();
    rt.shared_gate = sg.data(); rt.offsets = off.data(); rt.row_to_flat = r2f.data();
    rt.flat_to_row = f2r.data(); rt.block_variant = bv.data(); rt.plan_counts = counts.data();
    rt.plan_items = items.data(); rt.plan_done = done.data(); rt.m_skinny = 16;
    rt.dispatch = MOE_DISPATCH_PER_BLOCK;
    static RouteSmem rs;
    emu_block_idx = {(unsigned)cta, 0, 0};
    emu_run_cta(32 * kRouteWarps, [&]() {
      gemv_route(rt, T, K, MOE_W_BF16, rs, [](int) {});
      __syncthreads();
    });
    // the expected picks and permutation
    std::vector<int32_t> want(R);
    for (int t = 0; t < T; ++t) {
      std::vector<float> key(E);
      for (int e = 0; e < E; ++e) {
        const float l = lg[(size_t)t * G + e];
        key[e] = mode ? __fadd_rn(moe_route::sigmoid_key(l), bias[e]) : l;
      }
      std::vector<int> ord(E);
      std::iota(ord.begin(), ord.end(), 0);
      std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return key[a] > key[b]; });
      for (int k = 0; k < K; ++k) want[t * K + k] = ord[k];
    }
    std::vector<int32_t> w_off(E + 1, 0), w_r2f(R), w_f2r(R);
    for (int f = 0; f < R; ++f) ++w_off[want[f] + 1];
    for (int e = 0; e < E; ++e) w_off[e + 1] += w_off[e];
    std::vector<int32_t> fill(w_off.begin(), w_off.end() - 1);
    for (int f = 0; f < R; ++f) {
      const int row = fill[want[f]]++;
      w_r2f[row] = f;
      w_f2r[f] = row;
    }
    // shared memory, every CTA
    for (int f = 0; f < R; ++f) bad += rs.ids[f] != want[f];
    for (int r = 0; r < R; ++r) bad += rs.r2f[r] != w_r2f[r];
    int n_items = 0;
    for (int e = 0; e < E; ++e) {
      const int m = w_off[e + 1] - w_off[e];
      if (!m) continue;
      const int4 it = rs.items[n_items];
      bad += it.x != e || it.y != w_off[e] || it.z != m || it.w != 0;
      if (cta == 0) {
        const int4 g = items[n_items];
        bad += g.x != e || g.y != w_off[e] || g.z != m || g.w != 0 || done[n_items] != 0;
      }
      ++n_items;
    }
    bad += rs.n_items != n_items;
    if (cta == 0) {
      // the workspace
      for (int f = 0; f < R; ++f) bad += ids[f] != want[f] || f2r[f] != w_f2r[f];
      for (int r = 0; r < R; ++r) bad += r2f[r] != w_r2f[r];
      for (int e = 0; e <= E; ++e) bad += off[e] != w_off[e];
      for (int e = 0; e < E; ++e)
        bad += bv[e] != moe_variant_of(w_off[e + 1] - w_off[e], R, E, 16, MOE_DISPATCH_PER_BLOCK,
                                       MOE_W_BF16);
      bad += counts[0] != n_items || counts[1] != 0 || counts[2] != 0;
      for (int i = 0; i < 6; ++i) bad += counts[moe_plan::kSchedBase + i] != 0;
      for (int t = 0; t < T; ++t) {
        double sw = 0.0, prev = 1e30;
        for (int k = 0; k < K; ++k) {
          sw += w[t * K + k];
          if (mode == MOE_SCORE_SOFTMAX_RENORM && w[t * K + k] > prev * (1 + 1e-6)) ++bad;
          prev = w[t * K + k];
        }
        const double target = mode ? 2.5 : 1.0;
        if (std::abs(sw - target) > 1e-5 * target) ++bad;
        const float sg_want = moe_route::sigmoid_key(lg[(size_t)t * G + E]);
        bad += sg[t] != sg_want;
      }
    } else {
      bad += ids[0] != -7 || off[0] != -7 || counts[0] != -7;  // CTA > 0 writes nothing
    }
  }
  if (bad) std::printf("MISMATCH T=%d E=%d K=%d mode=%d pattern=%d: %d\n", T, E, K, mode, pattern, bad);
  return bad;
}

int main() {
  int bad = 0;
  const int shapes[][3] = {{1, 128, 8}, {2, 128, 8}, {4, 128, 8}, {3, 8, 2}, {4, 32, 4},
                           {1, 512, 10}, {2, 512, 10}, {3, 512, 10}, {1, 896, 16},
                           {2, 896, 16}, {2, 300, 5}, {3, 257, 7}, {4, 1024, 8}, {1, 4096, 16}};
  unsigned seed = 1;
  for (const auto& sh : shapes)
    for (int mode = 0; mode < 2; ++mode)
      for (int pattern = 0; pattern < 2; ++pattern)
        bad += check(sh[0], sh[1], sh[2], mode, pattern, seed++);
  std::printf("%s\n", bad ? "FAIL" : "OK");
  return bad ? 1 : 0;
}
