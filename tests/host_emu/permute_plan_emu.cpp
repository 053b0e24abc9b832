// Host emulation of the one-CTA permute (permute_block.cuh) and the grouped
// GEMM plan (plan.cuh) that the fused routing launches run, on a CTA of 256
// threads (simt_emu.h).  The permute is checked against a stable counting
// sort (offsets = prefix sum of the expert histogram; replica f = t*K + k
// goes to row offsets[e] + number of earlier replicas of e); out-of-range ids
// must raise the device status and map to row -1.  The plan is checked
// against the lists it must hold: for every block, in block order, its
// token tiles of the width of the list its variant picks (skinny 16, tile
// 128, wide 256 rows), each {block, first row, rows}; its done words zero.
// Exit status 0 when everything matches.
#include <cstdio>
#include <random>

#include "simt_emu.h"
#include "permute_block.cuh"
#include "plan.cuh"

int check(int R, int E, int wdtype, int skew, unsigned seed, bool bad_ids) {
  std::mt19937 rng(seed);
  std::vector<int32_t> ids(R);
  for (auto& v : ids) v = skew ? (rng() % 4 == 0 ? (int)(rng() % E) : (int)(rng() % std::max(1, E / 16)))
                               : (int)(rng() % E);
  if (bad_ids) { ids[R / 3] = E; ids[R / 2] = -2; }
  constexpr int kWarps = 8, kThreads = 256;
  std::vector<int32_t> offsets(E + 1, -7), off_s(E + 1), r2f(R, -7), f2r(R, -7), cnt(kWarps * E);
  int32_t status = 0;
  // the plan's scratch, laid out as plan_view lays it out
  std::vector<uint8_t> scratch(moe_plan::plan_bytes(R, E) + 256);
  void* sp = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(scratch.data()) + 255) & ~uintptr_t(255));
  const moe_plan::PlanView pv = moe_plan::plan_view(sp, R, E);
  for (int l = 0; l < moe_plan::kLists; ++l)
    for (int i = 0; i < pv.cap[l]; ++i) pv.done[l][i] = 99;
  const moe_plan::PlanOut po = moe_plan::plan_out(pv);
  std::vector<int32_t> bvar(E, -7);
  emu_run_cta(kThreads, [&]() {
    moe_permute_block::permute_block<kWarps>(ids.data(), R, E, offsets.data(), off_s.data(),
                                             r2f.data(), f2r.data(), &status, cnt.data());
    moe_plan::plan_experts<kThreads>(off_s.data(), E, R, MOE_DEFAULT_M_SKINNY, 0, wdtype,
                                     pv.counts, po, bvar.data());
  });
  int bad = 0;
  // permute
  std::vector<int32_t> hist(E, 0), want_off(E + 1, 0), run(E, 0);
  for (int f = 0; f < R; ++f)
    if (ids[f] >= 0 && ids[f] < E) ++hist[ids[f]];
  for (int e = 0; e < E; ++e) want_off[e + 1] = want_off[e] + hist[e];
  for (int e = 0; e <= E; ++e) bad += offsets[e] != want_off[e] || off_s[e] != want_off[e];
  for (int f = 0; f < R; ++f) {
    const int e = ids[f];
    if (e < 0 || e >= E) { bad += f2r[f] != -1; continue; }
    const int row = want_off[e] + run[e]++;
    bad += f2r[f] != row || r2f[row] != f;
  }
  bad += bad_ids ? status != MOE_DEV_BAD_EXPERT_ID : status != 0;
  const int pbad = bad;
  // plan
  std::vector<std::vector<int4>> want(moe_plan::kLists);
  for (int e = 0; e < E; ++e) {
    const int m = want_off[e + 1] - want_off[e];
    const int v = moe_variant_of(m, want_off[E], E, MOE_DEFAULT_M_SKINNY, 0, wdtype);
    bad += bvar[e] != v;
    const int l = v == MOE_VARIANT_SKINNY ? 0 : v == MOE_VARIANT_TILE ? 1 : v == MOE_VARIANT_WIDE ? 2 : -1;
    if (l < 0) continue;
    const int bn = moe_plan::list_bn(l);
    for (int i = 0; i * bn < m; ++i) want[l].push_back(make_int4(e, want_off[e] + i * bn, std::min(bn, m - i * bn), 0));
  }
  for (int l = 0; l < moe_plan::kLists; ++l) {
    bad += pv.counts[l] != (int)want[l].size();
    for (size_t i = 0; i < want[l].size() && i < (size_t)pv.cap[l]; ++i) {
      const int4 a = pv.items[l][i], b = want[l][i];
      bad += a.x != b.x || a.y != b.y || a.z != b.z || a.w != b.w;
      bad += pv.done[l][i] != 0;
    }
    bad += pv.counts[moe_plan::kSchedBase + 2 * l] != 0 || pv.counts[moe_plan::kSchedBase + 2 * l + 1] != 0;
  }
  printf("R=%d E=%d wdtype=%d skew=%d bad_ids=%d: permute %d wrong, plan %d wrong\n", R, E, wdtype,
         skew, (int)bad_ids, pbad, bad - pbad);
  return bad;
}

int main() {
  int bad = 0;
  bad += check(8, 128, 0, 0, 1, false);        // T=1, K=8 (decode)
  bad += check(32 * 8, 128, 0, 0, 2, false);   // T=32, K=8
  bad += check(4 * 10, 513, 0, 0, 3, false);   // shared-gate shape blocks
  bad += check(2 * 16, 896, 0, 0, 4, false);
  bad += check(256 * 8, 128, 0, 1, 5, false);  // concentrated: tile lists
  bad += check(4096, 32, 1, 1, 6, false);      // FP8: wide lists above 128 rows
  bad += check(777, 40, 0, 0, 7, true);        // out-of-range ids flagged
  bad += check(1, 8, 0, 0, 8, false);
  printf("%s\n", bad ? "FAIL" : "OK");
  return bad != 0;
}
