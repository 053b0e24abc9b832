// Shared device helpers of the MoE-layer library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "moe_gb300.h"

#define MOE_DEVICE __device__ __forceinline__

// Skinny/tile threshold on m_size used when the caller passes -1.  The
// skinny variant's token tile is 16 rows, so blocks that fit one skinny tile
// take it.
#define MOE_DEFAULT_M_SKINNY 16

// Variant predicate shared by the host mirror and the plan kernel.
//   m_size == 0                      -> skip (no work for the block)
//   dispatch SIMT                    -> CUDA-core kernel
//   m (per block, or max(1, R/E))    -> skinny if m <= m_skinny, else wide if
//                                       FP8 weights and m >= MOE_WIDE_MIN_ROWS,
//                                       else tile
__host__ __device__ __forceinline__ int moe_variant_of(int64_t m_size, int64_t R, int E,
                                                      int m_skinny, int dispatch, int wdtype) {
  if (m_size <= 0) return MOE_VARIANT_SKIP;
  // W8A8: one kernel takes every block, in 128-row token tiles
  if (wdtype == MOE_W8A8_FP8E4M3_B128) return MOE_VARIANT_TILE;
  if (dispatch == MOE_DISPATCH_SIMT) return MOE_VARIANT_SIMT;
  int64_t m = m_size;
  if (dispatch == MOE_DISPATCH_GLOBAL_AVG) {
    int64_t avg = E > 0 ? R / E : R;
    m = avg < 1 ? 1 : avg;
  }
  if (m <= (int64_t)m_skinny) return MOE_VARIANT_SKINNY;
  // 256-row token tiles pay off where each weight tile is dequantised (FP8,
  // MXFP4): the conversion is amortised over twice the tokens
  return (wdtype != MOE_W_BF16 && m >= MOE_WIDE_MIN_ROWS) ? MOE_VARIANT_WIDE : MOE_VARIANT_TILE;
}

// SM count of the current device, cached per device (148 if the query fails)
inline int moe_num_sms() {
  static std::atomic<int> n[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int v = n[dev].load(std::memory_order_relaxed);
  if (!v) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    n[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// First error wins.
MOE_DEVICE void moe_set_status(int32_t* dev_status, int32_t code) {
  if (dev_status) atomicCAS(dev_status, 0, code);
}

MOE_DEVICE float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
MOE_DEVICE float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// 8 bf16 packed in a uint4 -> 8 fp32 (exact widening)
MOE_DEVICE void bf16x8_to_f32(const uint4& v, float* f) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

MOE_DEVICE uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

MOE_DEVICE int lane_id() { return threadIdx.x & 31; }
MOE_DEVICE int warp_id() { return threadIdx.x >> 5; }

static inline size_t moe_align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
__host__ __device__ static inline int moe_cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Programmatic dependent launch.  Every kernel of the layer is launched with
// programmatic stream serialisation: the next kernel's grid may be scheduled
// while this one runs, and each kernel waits here for its predecessor's
// completion (and memory) before reading anything the predecessor wrote.
MOE_DEVICE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEVICE void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// cudaLaunchKernelEx with programmatic stream serialisation (and an optional
// cluster of `cluster_z` CTAs along z).
template <typename... KArgs, typename... Args>
static inline cudaError_t moe_launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t stream, int cluster_z, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_z > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = cluster_z;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device.  The attribute belongs to the (function, device) pair, so a process
// that launches on several GPUs must set it on each: `done` holds one bit per
// device index already set (devices past 63 set it on every launch).  Setting
// it twice is harmless, so two host threads racing here only repeat the call.
template <typename... KArgs>
static inline cudaError_t moe_raise_smem(void (*kernel)(KArgs...), size_t bytes,
                                         std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}
