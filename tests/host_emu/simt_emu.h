// Host emulation of the SIMT primitives the routing device code uses, for
// CPU tests of that code.  A CTA of N threads is N std::threads; the threads
// of a warp (32 consecutive ones) meet at a warp barrier in every warp
// collective (shuffle, redux, ballot, any, match, syncwarp), all N at a CTA
// barrier in __syncthreads.  Device keywords become plain host C++ and
// __shared__ variables become statics shared by the CTA's threads; only one
// CTA runs at a time.  Include this before the device headers under test.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <barrier>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <memory>
#include <mutex>
#include <thread>
#include <vector>

#undef __device__
#define __device__
#undef __constant__
#define __constant__
#undef __shared__
#define __shared__ static
#undef __forceinline__
#define __forceinline__ inline

namespace simt_emu {
inline std::barrier<>* warp_bar[32];
inline std::barrier<>* cta_bar;
inline uint64_t slot[32][32];
inline thread_local int lane, warp;
}  // namespace simt_emu

struct EmuDim { unsigned x, y, z; };
inline thread_local EmuDim emu_thread_idx;
#undef threadIdx
#define threadIdx emu_thread_idx
// the CTA being run (one at a time; set emu_block_idx before emu_run_cta) and
// its size.  A program whose device code reads blockIdx / blockDim defines
// them as these after including common.cuh (whose launch helper names a
// cudaLaunchConfig_t member blockDim).
inline EmuDim emu_block_idx = {0, 0, 0};
inline EmuDim emu_block_dim = {0, 1, 1};

// run fn on one CTA of n threads (n a multiple of 32, at most 1024)
inline void emu_run_cta(int n, const std::function<void()>& fn) {
  using namespace simt_emu;
  std::vector<std::unique_ptr<std::barrier<>>> wb;
  for (int w = 0; w < n / 32; ++w) {
    wb.emplace_back(new std::barrier<>(32));
    warp_bar[w] = wb.back().get();
  }
  std::barrier<> cb(n);
  cta_bar = &cb;
  emu_block_dim = {(unsigned)n, 1, 1};
  std::vector<std::thread> th;
  for (int i = 0; i < n; ++i)
    th.emplace_back([&, i]() {
      lane = i & 31;
      warp = i >> 5;
      emu_thread_idx = {(unsigned)i, 0, 0};
      fn();
    });
  for (auto& t : th) t.join();
}

inline void __syncthreads() { simt_emu::cta_bar->arrive_and_wait(); }
inline void __syncwarp(unsigned = 0xffffffffu) { simt_emu::warp_bar[simt_emu::warp]->arrive_and_wait(); }

// every lane posts v; returns the 32 posted values of this warp
inline void emu_post(uint64_t v, uint64_t (&all)[32]) {
  using namespace simt_emu;
  slot[warp][lane] = v;
  warp_bar[warp]->arrive_and_wait();
  std::memcpy(all, slot[warp], sizeof(all));
  warp_bar[warp]->arrive_and_wait();
}
template <class T> uint64_t emu_bits(T v) { uint64_t u = 0; std::memcpy(&u, &v, sizeof(T)); return u; }
template <class T> T emu_val(uint64_t u) { T v; std::memcpy(&v, &u, sizeof(T)); return v; }

template <class T> T __shfl_xor_sync(unsigned, T v, int d) {
  uint64_t a[32]; emu_post(emu_bits(v), a); return emu_val<T>(a[simt_emu::lane ^ d]);
}
template <class T> T __shfl_sync(unsigned, T v, int s) {
  uint64_t a[32]; emu_post(emu_bits(v), a); return emu_val<T>(a[s & 31]);
}
template <class T> T __shfl_up_sync(unsigned, T v, int d) {
  uint64_t a[32]; emu_post(emu_bits(v), a);
  return simt_emu::lane >= d ? emu_val<T>(a[simt_emu::lane - d]) : v;
}
inline uint32_t __reduce_max_sync(unsigned, uint32_t v) {
  uint64_t a[32]; emu_post(v, a); uint32_t r = 0; for (auto x : a) r = std::max<uint32_t>(r, (uint32_t)x); return r;
}
inline uint32_t __reduce_min_sync(unsigned, uint32_t v) {
  uint64_t a[32]; emu_post(v, a); uint32_t r = ~0u; for (auto x : a) r = std::min<uint32_t>(r, (uint32_t)x); return r;
}
inline uint32_t __reduce_add_sync(unsigned, uint32_t v) {
  uint64_t a[32]; emu_post(v, a); uint32_t r = 0; for (auto x : a) r += (uint32_t)x; return r;
}
inline unsigned __ballot_sync(unsigned, int p) {
  uint64_t a[32]; emu_post(p ? 1 : 0, a); unsigned m = 0;
  for (int i = 0; i < 32; ++i) if (a[i]) m |= 1u << i; return m;
}
inline int __any_sync(unsigned m, int p) { return __ballot_sync(m, p) != 0; }
template <class T> unsigned __match_any_sync(unsigned, T v) {
  uint64_t a[32]; emu_post(emu_bits(v), a); unsigned m = 0;
  for (int i = 0; i < 32; ++i) if (a[i] == a[simt_emu::lane]) m |= 1u << i; return m;
}
inline int __popc(unsigned v) { return __builtin_popcount(v); }
inline int __ffs(unsigned v) { return __builtin_ffs((int)v); }
template <class T> T __ldg(const T* p) { return *p; }
template <class T> T __ldcg(const T* p) { return *p; }
inline uint32_t __float_as_uint(float f) { return emu_val<uint32_t>(emu_bits(f)); }
inline float __uint_as_float(uint32_t u) { return emu_val<float>(u); }
inline float __int_as_float(int u) { return emu_val<float>((uint32_t)u); }
// single IEEE operations, round to nearest (what the _rn intrinsics are)
inline float __fadd_rn(float a, float b) { volatile float r = a + b; return r; }
inline float __fsub_rn(float a, float b) { volatile float r = a - b; return r; }
inline float __fmul_rn(float a, float b) { volatile float r = a * b; return r; }
inline float __fdiv_rn(float a, float b) { volatile float r = a / b; return r; }
template <class T> T max(T a, T b) { return a > b ? a : b; }
template <class T> T min(T a, T b) { return a < b ? a : b; }
inline int atomicCAS(int* p, int c, int v) {
  static std::mutex m;
  std::lock_guard<std::mutex> g(m);
  const int o = *p; if (o == c) *p = v; return o;
}
