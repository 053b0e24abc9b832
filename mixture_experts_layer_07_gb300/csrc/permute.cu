// P: stable permute of token replicas into expert-contiguous row blocks.
//
// "vLLM MoE permute optimisation: buffer pre-allocation" (vllm PR #43014),
// "1. C++ kernel level": the permute works in caller-owned scratch that is
// allocated once and reused instead of being allocated on every call.  The
// block boundaries are the per-expert offsets whose differences are the
// m_size of "vLLM CPU MoE: dynamic GEMM dispatch" (vllm PR #50949),
// "2. moe_fp8.cpp".
//
// Replica f = t*K + k goes to row offsets[e] + rank, rank = number of
// replicas f' < f with the same expert, so the result is unique and the
// kernels need no sort and no cross-CTA waits:
//   1. count   one warp per 256-replica chunk: per-chunk expert histogram
//   2. scan    one CTA: a warp per expert scans its chunk counts; then an
//              exclusive scan over experts gives offsets[E+1]
//   3. scatter one warp per chunk, 32 replicas per step in order: lanes with
//              the same expert find each other with __match_any_sync, the
//              rank is the running count plus the popcount of lower lanes
//   4. copy    xp[flat_to_row[t*K+k]] = x[t]: each row of x is read once and
//              written to its token's K rows, 16-byte vectors
#include "common.cuh"
#include "internal.h"
#include "permute_block.cuh"

namespace {

constexpr int kChunk = 256;        // replicas per warp chunk
constexpr int kWarpsPerCta = 8;

// scratch: int32 counts[E][nchunks] (turned into per-chunk bases by the scan)
inline int num_chunks(int R) { return moe_cdiv(R, kChunk); }

__global__ void __launch_bounds__(32 * kWarpsPerCta)
permute_count_kernel(const int32_t* __restrict__ ids, int R, int E, int nchunks,
                     int32_t* __restrict__ counts, int32_t* dev_status) {
  extern __shared__ int32_t hist[];  // [kWarpsPerCta][E]
  pdl_wait();
  pdl_trigger();
  const int w = warp_id(), lane = lane_id();
  const int chunk = blockIdx.x * kWarpsPerCta + w;
  int32_t* h = hist + w * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  if (chunk < nchunks) {
    const int f0 = chunk * kChunk;
    int v[kChunk / 32];  // all of the chunk's ids in flight at once
#pragma unroll
    for (int i = 0; i < kChunk / 32; ++i) {
      const int f = f0 + i * 32 + lane;
      v[i] = f < R ? __ldg(ids + f) : E;
    }
#pragma unroll
    for (int i = 0; i < kChunk / 32; ++i) {
      const int e = v[i];
      if (e >= 0 && e < E) atomicAdd(&h[e], 1);
      else if (f0 + i * 32 + lane < R) moe_set_status(dev_status, MOE_DEV_BAD_EXPERT_ID);
    }
    __syncwarp();
    for (int e = lane; e < E; e += 32) counts[(size_t)e * nchunks + chunk] = h[e];
  }
}

// counts[e][c] -> exclusive prefix over chunks (in place), one warp per expert
// (32 chunks per step, warp scan), then an exclusive scan of the per-expert
// totals over the block gives offsets[E+1].
__global__ void __launch_bounds__(1024)
permute_scan_kernel(int32_t* __restrict__ counts, int E, int nchunks,
                    int32_t* __restrict__ offsets) {
  __shared__ int32_t tot[1024];
  __shared__ int32_t warp_tot[32];
  pdl_wait();
  pdl_trigger();
  const int lane = lane_id(), warp = warp_id();
  constexpr int kB = 8;  // 8 x 32 chunk counts loaded before they are scanned
  for (int e = warp; e < E; e += 32) {
    int32_t* row = counts + (size_t)e * nchunks;
    int32_t run = 0;
    for (int c0 = 0; c0 < nchunks; c0 += 32 * kB) {
      int32_t v[kB];
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int c = c0 + b * 32 + lane;
        v[b] = c < nchunks ? row[c] : 0;
      }
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int c = c0 + b * 32 + lane;
        int32_t incl = v[b];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t n = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += n;
        }
        if (c < nchunks) row[c] = run + incl - v[b];
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (lane == 0) tot[e] = run;
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int32_t mine = e < E ? tot[e] : 0;
  int32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int32_t v = warp_tot[lane];
    int32_t sc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, sc, o);
      if (lane >= o) sc += n;
    }
    warp_tot[lane] = sc - v;
  }
  __syncthreads();
  const int32_t excl = incl - mine + warp_tot[warp];
  if (e < E) offsets[e] = excl;
  if (e == E - 1) offsets[E] = excl + mine;
}

__global__ void __launch_bounds__(32 * kWarpsPerCta)
permute_scatter_kernel(const int32_t* __restrict__ ids, int R, int E, int nchunks,
                       const int32_t* __restrict__ bases, const int32_t* __restrict__ offsets,
                       int32_t* __restrict__ row_to_flat, int32_t* __restrict__ flat_to_row) {
  extern __shared__ int32_t cnt_all[];  // [kWarpsPerCta][E]
  pdl_wait();
  pdl_trigger();
  const int w = warp_id(), lane = lane_id();
  const int chunk = blockIdx.x * kWarpsPerCta + w;
  if (chunk >= nchunks) return;
  int32_t* cnt = cnt_all + w * E;
  for (int e = lane; e < E; e += 32) cnt[e] = offsets[e] + bases[(size_t)e * nchunks + chunk];
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
  const int f0 = chunk * kChunk;
  int v[kChunk / 32];  // all of the chunk's ids in flight at once
#pragma unroll
  for (int i = 0; i < kChunk / 32; ++i) {
    const int f = f0 + i * 32 + lane;
    v[i] = f < R ? __ldg(ids + f) : -1;
  }
#pragma unroll
  for (int i = 0; i < kChunk / 32; ++i) {
    const int f = f0 + i * 32 + lane;
    const int e = (v[i] >= 0 && v[i] < E) ? v[i] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    const int leader = __ffs(peers) - 1;
    int base = 0;
    if (e >= 0) base = cnt[e];
    __syncwarp();
    if (e >= 0 && lane == leader) cnt[e] = base + __popc(peers);
    __syncwarp();
    if (f < R) {
      if (e >= 0) {
        const int row = base + rank;
        row_to_flat[row] = f;
        flat_to_row[f] = row;
      } else {
        flat_to_row[f] = -1;
      }
    }
  }
}

// Small problems (R <= kFusedMaxR replicas, the decode regime): count, scan
// and stable scatter in ONE CTA (permute_block.cuh) -- one launch instead of
// three, and no global scratch.
constexpr int kFusedWarps = 32;
// Above this many replicas the multi-CTA path (count, scan, scatter) wins: one
// CTA cannot keep enough loads and stores in flight.
constexpr int kFusedMaxR = 4096;

__global__ void __launch_bounds__(32 * kFusedWarps)
permute_fused_kernel(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ offsets,
                     int32_t* __restrict__ row_to_flat, int32_t* __restrict__ flat_to_row,
                     int32_t* dev_status) {
  extern __shared__ int32_t sm[];  // [kFusedWarps][E] counters, then [E + 1] offsets
  pdl_wait();
  pdl_trigger();
  moe_permute_block::permute_block<kFusedWarps>(ids, R, E, offsets, sm + kFusedWarps * E,
                                                 row_to_flat, flat_to_row, dev_status, sm);
}

// xp[flat_to_row[t*K+k]] = x[t]: one warp per token reads each 16-byte vector
// of x[t] once and writes it to the token's K rows (reading x once instead of
// once per replica), 8 vectors per lane in flight.
__global__ void __launch_bounds__(256)
permute_copy_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ flat_to_row, int T,
                    int K, int H8, uint4* __restrict__ xp) {
  pdl_wait();
  pdl_trigger();
  const int lane = lane_id();
  for (int t = blockIdx.x * 8 + warp_id(); t < T; t += gridDim.x * 8) {
    const int myrow = lane < K ? __ldg(flat_to_row + (size_t)t * K + lane) : -1;
    const uint4* src = x + (size_t)t * H8;
    for (int c0 = 0; c0 < H8; c0 += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = c0 + j * 32 + lane;
        if (c < H8) v[j] = __ldg(src + c);
      }
      for (int k = 0; k < K; ++k) {
        const int r = __shfl_sync(0xffffffffu, myrow, k);
        if (r < 0) continue;
        uint4* dst = xp + (size_t)r * H8;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c = c0 + j * 32 + lane;
          if (c < H8) dst[c] = v[j];
        }
      }
    }
  }
}

}  // namespace

namespace {

cudaError_t launch_copy(const void* x, const int32_t* flat_to_row, int T, int K, int H, void* xp,
                        cudaStream_t stream) {
  const int grid = moe_cdiv(T, 8) < 152 * 16 ? moe_cdiv(T, 8) : 152 * 16;
  return moe_launch(permute_copy_kernel, dim3(grid), dim3(256), 0, stream, 1,
                    static_cast<const uint4*>(x), flat_to_row, T, K, H / 8,
                    static_cast<uint4*>(xp));
}

}  // namespace

cudaError_t launch_permute_copy(const void* x, const int32_t* flat_to_row, int T, int K, int H,
                                void* xp, cudaStream_t stream) {
  return launch_copy(x, flat_to_row, T, K, H, xp, stream);
}

size_t permute_scratch_bytes(int T, int E, int K) {
  const int R = T * K;
  return moe_align_up((size_t)num_chunks(R) * E * sizeof(int32_t) + 256, 256);
}

cudaError_t launch_permute(const void* x, const int32_t* ids, int T, int H, int E, int K,
                           int32_t* offsets, int32_t* row_to_flat, int32_t* flat_to_row,
                           void* xp, void* scratch, int32_t* dev_status, cudaStream_t stream) {
  const int R = T * K;
  const int nch = num_chunks(R);
  int32_t* counts = static_cast<int32_t*>(scratch);
  const size_t smem = (size_t)kWarpsPerCta * E * sizeof(int32_t);
  const int ctas = moe_cdiv(nch, kWarpsPerCta);
  const size_t fused_smem = ((size_t)(kFusedWarps + 1) * E + 1) * sizeof(int32_t);
  if (R > 0 && R <= kFusedMaxR && fused_smem <= 200 * 1024) {
    static std::atomic<unsigned long long> smem_set{0};  // devices whose limit is raised
    cudaError_t e = moe_raise_smem(permute_fused_kernel, 200 * 1024, smem_set);
    if (e != cudaSuccess) return e;
    e = moe_launch(permute_fused_kernel, dim3(1), dim3(32 * kFusedWarps), fused_smem,
                               stream, 1, ids, R, E, offsets, row_to_flat, flat_to_row, dev_status);
    if (e != cudaSuccess || !xp) return e;
    return launch_copy(x, flat_to_row, T, K, H, xp, stream);
  }
  cudaError_t e = cudaSuccess;
  if (R > 0) {
    e = moe_launch(permute_count_kernel, dim3(ctas), dim3(32 * kWarpsPerCta), smem, stream, 1, ids,
                   R, E, nch, counts, dev_status);
    if (e != cudaSuccess) return e;
  }
  e = moe_launch(permute_scan_kernel, dim3(1), dim3(1024), 0, stream, 1, counts, E, nch, offsets);
  if (e != cudaSuccess || R == 0) return e;
  e = moe_launch(permute_scatter_kernel, dim3(ctas), dim3(32 * kWarpsPerCta), smem, stream, 1, ids,
                 R, E, nch, (const int32_t*)counts, (const int32_t*)offsets, row_to_flat,
                 flat_to_row);
  if (e != cudaSuccess || !xp) return e;
  return launch_copy(x, flat_to_row, T, K, H, xp, stream);
}

// ---------------------------------------------------------------- static scratch
// A variant of moe_permute for callers that may not allocate device memory at
// all: its per-chunk counts live in a fixed array compiled into this library,
// so the caller passes only inputs and outputs.  The array is shared by every
// call on a device and keeps the previous call's contents; the count kernel
// overwrites every entry it later reads, so nothing needs clearing.  Two calls
// whose kernels overlap on the GPU (different streams, no ordering) race on it.
#include <cuda.h>

#include <mutex>

static __device__ __align__(256) unsigned char g_permute_static_scratch[MOE_PERMUTE_STATIC_SCRATCH_BYTES];

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The CUDA context current on this thread, to tell a cached address from a stale one.
CUcontext current_context() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  CUcontext c = nullptr;
  if (fn) fn(&c);
  return c;
}

// Device address of the array on the current device (in host code the symbol
// is only a host-side stand-in).  Looked up with that device current and
// cached per device together with the context it belongs to: after a
// cudaDeviceReset the device gets a new context, the module is loaded again
// and the array may sit elsewhere, so a changed context means a new lookup.
void* static_scratch_address(cudaError_t* err) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  static CUcontext ctx_of[64] = {nullptr};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  const CUcontext ctx = current_context();  // null before the runtime binds one
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || !ctx || ctx_of[dev] != ctx) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_permute_static_scratch);  // binds the context
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
    ctx_of[dev] = current_context();
  }
  return addr[dev];
}

bool unaligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

}  // namespace

extern "C" moe_status_t moe_permute_static(const void* x, const int32_t* ids, int T, int H, int E,
                                           int K, int32_t* offsets, int32_t* row_to_flat,
                                           int32_t* flat_to_row, void* xp, int32_t* dev_status,
                                           moe_stream_t stream) {
  if (T < 0 || H <= 0 || H % 16 != 0 || E <= 0 || E > 1024 || K <= 0 || K > E || K > 32)
    return MOE_ERR_INVALID_ARG;
  if (!offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !row_to_flat || !flat_to_row || (xp && !x))) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * K > 0x3fffffff) return MOE_ERR_INVALID_ARG;
  if (permute_scratch_bytes(T, E, K) > (size_t)MOE_PERMUTE_STATIC_SCRATCH_BYTES)
    return MOE_ERR_WORKSPACE;
  if (unaligned(offsets, 4) || (ids && unaligned(ids, 4)) ||
      (row_to_flat && unaligned(row_to_flat, 4)) || (flat_to_row && unaligned(flat_to_row, 4)) ||
      (xp && (unaligned(xp, 16) || unaligned(x, 16))))
    return MOE_ERR_MISALIGNED;
  cudaError_t err;
  void* scratch = static_scratch_address(&err);
  if (!scratch) return MOE_ERR_CUDA;
  err = launch_permute(x, ids, T, H, E, K, offsets, row_to_flat, flat_to_row, xp, scratch,
                       dev_status, stream);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
