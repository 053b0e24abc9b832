// Stable permute of up to a few thousand replicas by ONE CTA of NW warps,
// every counter in shared memory (used by the fused permute kernel and by the
// fused decode routing kernel).
//   warp w owns the contiguous replica range [w*span, (w+1)*span)
//   1. per-warp histogram cnt[w][e] (one leader per distinct expert per step,
//      found with __match_any_sync: no atomics)
//   2. scan over warps per expert, then over experts -> offsets[E+1]
//   3. each warp walks its range again in order, 32 replicas per step: row =
//      offsets[e] + warp base + running count + rank among equal lanes
// Replica f = t*K + k goes to row offsets[e] + (number of f' < f with the same
// expert), exactly the multi-CTA path's result.
#pragma once

#include "common.cuh"

namespace moe_permute_block {

// ids: R expert ids (global or shared memory).  cnt: shared [NW][E];
// off_s: shared [E + 1] (filled with the offsets).  offsets: global [E + 1].
template <int NW>
MOE_DEVICE void permute_block(const int32_t* ids, int R, int E, int32_t* __restrict__ offsets,
                              int32_t* off_s, int32_t* __restrict__ row_to_flat,
                              int32_t* __restrict__ flat_to_row, int32_t* dev_status,
                              int32_t* cnt) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t pass_tot;
  const int w = warp_id(), lane = lane_id();
  const int span = ((R + NW - 1) / NW + 31) / 32 * 32;
  const int f0 = w * span, f1 = min(R, f0 + span);
  const unsigned lt_mask = (1u << lane) - 1u;
  int32_t* mine = cnt + w * E;
  for (int e = lane; e < E; e += 32) mine[e] = 0;
  __syncwarp();
  // ids of this warp's range are read 8 steps (256 replicas) at a time, all
  // loads in flight together, then processed step by step
  constexpr int kBatch = 8;
  auto load_batch = [&](int fb, int (&v)[kBatch]) {
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int f = fb + i * 32 + lane;
      v[i] = f < f1 ? ids[f] : -1;
    }
  };
  // 1. per-warp histogram
  for (int fb = f0; fb < f1; fb += 32 * kBatch) {
    int v[kBatch];
    load_batch(fb, v);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      int e = v[i];
      if (fb + i * 32 + lane < f1 && (e < 0 || e >= E)) {
        moe_set_status(dev_status, MOE_DEV_BAD_EXPERT_ID);
        e = -1;
      }
      if (e >= E) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && (peers & lt_mask) == 0) mine[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  // 2. scan: over warps per expert (thread e, loop), then over experts
  int32_t tot_last = 0;
  for (int e0 = 0; e0 < E; e0 += 32 * NW) {
    const int e = e0 + threadIdx.x;
    int32_t tot = 0;
    if (e < E) {
      for (int q = 0; q < NW; ++q) {
        const int32_t v = cnt[q * E + e];
        cnt[q * E + e] = tot;
        tot += v;
      }
    }
    int32_t incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    if (w == 0) {
      const int32_t v = lane < NW ? warp_tot[lane] : 0;
      int32_t sc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xffffffffu, sc, o);
        if (lane >= o) sc += n;
      }
      if (lane < NW) warp_tot[lane] = sc - v;
      if (lane == NW - 1) pass_tot = sc;
    }
    __syncthreads();
    if (e < E) {
      const int32_t ex = tot_last + incl - tot + warp_tot[w];
      off_s[e] = ex;
      offsets[e] = ex;
    }
    tot_last += pass_tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    off_s[E] = tot_last;
    offsets[E] = tot_last;
  }
  __syncthreads();
  // 3. stable scatter
  for (int fb = f0; fb < f1; fb += 32 * kBatch) {
    int v[kBatch];
    load_batch(fb, v);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int f = fb + i * 32 + lane;
      const int ee = (v[i] >= 0 && v[i] < E) ? v[i] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, ee);
      int base = 0;
      if (ee >= 0) base = off_s[ee] + mine[ee];
      __syncwarp();
      if (ee >= 0 && (peers & lt_mask) == 0) mine[ee] += __popc(peers);
      __syncwarp();
      if (f < f1) {
        if (ee >= 0) {
          const int row = base + __popc(peers & lt_mask);
          row_to_flat[row] = f;
          flat_to_row[f] = row;
        } else {
          flat_to_row[f] = -1;
        }
      }
    }
  }
  __syncthreads();
}

}  // namespace moe_permute_block
