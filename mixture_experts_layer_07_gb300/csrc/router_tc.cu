// R on the tensor cores for prefill batches (T > 32): logits = x . Wg^T + bias
// with fp32 accuracy from bf16 MMAs.
//
// "vLLM MiniMax-M2 MoE gate optimisation: fused FP32 kernel" (vllm PR #38445):
// the gate must be computed in fp32 from bf16 activations.  At decode sizes
// that is the CUDA-core kernel of router_gemm.cu; at prefill sizes the product
// is a dense contraction bound by the FP32 pipes, so here it runs on tcgen05:
//   * x is bf16, so every x element is exact as an MMA operand;
//   * Wg (fp32) is split exactly into three bf16 parts, hi = bf16(w),
//     mid = bf16(w - hi), lo = bf16(w - hi - mid), which together carry the
//     24 significant bits of w (the remainder is below 2^-24 |w|);
//   * each bf16 x bf16 product is exact in fp32, and the three partial
//     products accumulate in fp32 in one TMEM accumulator
//     (3 MMAs per 16-wide K step).
// The error is a few fp32 roundings of the running sums, far inside the
// 1e-5 bound relative to sum |x w|.
//
// Tiling (non-swapped): a CTA owns 128*MT tokens x 128 gate rows; A = x tiles
// (TMA, 128-byte swizzle), B = the three split weight tiles (one 3-D TMA map
// over [3][G][H]); warp 0 issues TMA, warp 1 the MMAs, warps 2-5 read the
// accumulator.  When tiles are few, H is split across the CTAs of a cluster
// and the fp32 partial tiles are summed through distributed shared memory in
// rank order (deterministic, no global scratch).  Bounded waits as in the
// expert GEMM.
#include <cooperative_groups.h>
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace {

using namespace moe_ptx;

constexpr int kBK = 64;
constexpr int kTile = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------- split
__global__ void __launch_bounds__(256)
router_split_kernel(const float4* __restrict__ wg, long long n4, uint2* __restrict__ hi,
                    uint2* __restrict__ mid, uint2* __restrict__ lo) {
  pdl_wait();
  pdl_trigger();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 w = __ldg(wg + i);
    const float v[4] = {w.x, w.y, w.z, w.w};
    uint32_t h[4], m[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat16 bh = __float2bfloat16_rn(v[j]);
      const float r1 = __fsub_rn(v[j], __bfloat162float(bh));
      const __nv_bfloat16 bm = __float2bfloat16_rn(r1);
      const float r2 = __fsub_rn(r1, __bfloat162float(bm));
      const __nv_bfloat16 bl = __float2bfloat16_rn(r2);
      h[j] = __bfloat16_as_ushort(bh);
      m[j] = __bfloat16_as_ushort(bm);
      l[j] = __bfloat16_as_ushort(bl);
    }
    hi[i] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    mid[i] = make_uint2(m[0] | (m[1] << 16), m[2] | (m[3] << 16));
    lo[i] = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
  }
}

// ---------------------------------------------------------------- GEMM
template <int MT>
struct RtCfg {
  static constexpr int kABytes = kTile * kBK * 2;      // one 128-token x tile
  static constexpr int kBBytes = kTile * kBK * 2;      // one 128-gate weight part tile
  static constexpr int kStageBytes = MT * kABytes + 3 * kBBytes;
  static constexpr int kStages = (200 * 1024) / kStageBytes > 4 ? 4 : (200 * 1024) / kStageBytes;
  static constexpr int kPitch = kTile + 4;              // fp32 partial tile row pitch
  static constexpr int kPartBytes = MT * kTile * kPitch * 4;
  static constexpr int kMainBytes = kStages * kStageBytes > kPartBytes ? kStages * kStageBytes
                                                                        : kPartBytes;
  static constexpr int kBarBytes = (2 * kStages + 2) * 8 + 16;
  static constexpr size_t kSmemBytes = 1024 + (size_t)kMainBytes + kBarBytes;
  static constexpr int kTmemCols = MT * kTile;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kTile, kTile);
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kStages >= 2, "two stages");
  static_assert(kSmemBytes <= 232448, "shared memory");
};

template <int MT>
__global__ void __launch_bounds__(192, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                 const float* __restrict__ bias, float* __restrict__ logits, int T, int H, int G,
                 int kchunk, int32_t* dev_status) {
  using C = RtCfg<MT>;
  namespace cg = cooperative_groups;
  pdl_wait();
  pdl_trigger();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int splits = (int)cluster.num_blocks();
  const int n0 = blockIdx.x * kTile;
  const int m0 = blockIdx.y * kTile * MT;
  const int k_lo = rank * kchunk;
  const int k_hi = min(H, k_lo + kchunk);
  const int nk = k_hi > k_lo ? (k_hi - k_lo + kBK - 1) / kBK : 0;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  uint8_t* bar_area = smem + C::kMainBytes;
  const uint32_t bar0 = smem_u32(bar_area);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::kStages + s); };
  const uint32_t acc_full = bar0 + 8u * (2 * C::kStages);
  const uint32_t drain_bar = acc_full + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * (2 * C::kStages + 2));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* part = reinterpret_cast<float*>(smem);  // reused after the main loop

  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) { mbar_init(full_bar(s), 1); mbar_init(empty_bar(s), 1); }
    mbar_init(acc_full, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    moe_set_status(dev_status, MOE_DEV_WAIT_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
        const uint32_t st = sbase + stage * C::kStageBytes;
        const int k = k_lo + kb * kBK;
        mbar_arrive_expect_tx(full_bar(stage), C::kStageBytes);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
          tma_load_2d(st + mt * C::kABytes, &tm_x, full_bar(stage), k, m0 + mt * kTile);
#pragma unroll
        for (int p = 0; p < 3; ++p)
          tma_load_3d(st + MT * C::kABytes + p * C::kBBytes, &tm_w, full_bar(stage), k, n0, p);
        armed |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
      }
      for (int s = 0; s < C::kStages; ++s)
        if (armed & (1u << s))
          if (!mbar_wait_bounded(full_bar(s), (armed_parity >> s) & 1u, nullptr, kWaitLimitNs)) fail();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: 3 split parts per 16-wide K step, one accumulator
      int stage = 0;
      uint32_t phase = 0;
      bool issued = false;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t st = sbase + stage * C::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint64_t adesc = sdesc_k128_sw128(st + mt * C::kABytes + kk * 32);
#pragma unroll
            for (int p = 0; p < 3; ++p) {
              const uint32_t acc = (kb > 0 || kk > 0 || p > 0) ? 1u : 0u;
              tc_mma_f16(tmem + mt * kTile,
                         adesc, sdesc_k128_sw128(st + MT * C::kABytes + p * C::kBBytes + kk * 32),
                         C::kIdesc, acc);
            }
          }
        }
        issued = true;
        tc_commit(empty_bar(stage));
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
      }
      tc_commit(acc_full);  // also when nothing was issued: the epilogue then writes zeros
      if (issued) {
        tc_commit(drain_bar);
        if (!mbar_wait_bounded(drain_bar, 0, nullptr, kWaitLimitNs)) fail();
      }
    }
  } else {
    // ---------------- epilogue: thread = token row (TMEM lane), 32 gates per load
    const int quarter = warp & 3;
    const bool ok = mbar_wait_bounded(acc_full, 0, abort_flag, kWaitLimitNs);
    if (!ok) fail();
    tc_fence_after();
    const int r = quarter * 32 + lane;
    for (int mt = 0; mt < MT; ++mt) {
      for (int c0 = 0; c0 < kTile; c0 += 16) {
        uint32_t v[16];
        tc_ld_32x32b_x16(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + mt * kTile + c0, v);
        tc_wait_ld();
        float* dst = part + (size_t)(mt * kTile + r) * C::kPitch + c0;
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<float4*>(dst + j) =
              (ok && nk > 0) ? make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                           __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  // All of this CTA's smem is free for `part` only after the producer's copies
  // landed and the MMAs retired (both waited on above), so the epilogue's
  // writes into the reused stage memory cannot race them.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  cluster.sync();
  // rank r sums its share of the tile's rows over the cluster, in rank order
  const int rows = MT * kTile;
  const int per = (rows + splits - 1) / splits;
  const int r_lo = rank * per, r_hi = min(rows, r_lo + per);
  for (int e = threadIdx.x; e < (r_hi - r_lo) * (kTile / 4); e += blockDim.x) {
    const int rr = r_lo + e / (kTile / 4), c = (e % (kTile / 4)) * 4;
    // all ranks' partials in flight at once, then summed in rank order
    float4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < splits)
        v[q] = *reinterpret_cast<const float4*>(
            cluster.map_shared_rank(part + (size_t)rr * C::kPitch + c, q));
    float4 s = v[0];
#pragma unroll
    for (int q = 1; q < 8; ++q)
      if (q < splits) { s.x += v[q].x; s.y += v[q].y; s.z += v[q].z; s.w += v[q].w; }
    const int m = m0 + rr, n = n0 + c;
    if (m < T) {
      const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (n + j < G) logits[(size_t)m * G + n + j] = sv[j] + (bias ? bias[n + j] : 0.f);
    }
  }
  cluster.sync();
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  return dev;
}

// per device: SM counts (and cluster occupancies below) differ between GPUs
int sm_count() {
  static std::atomic<int> n[64];
  const int dev = current_device();
  int v = n[dev].load(std::memory_order_relaxed);
  if (!v) {
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    v = v > 0 ? v : 148;
    n[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// clusters of `splits` CTAs of this kernel that fit on the GPU at once
// (with one CTA per SM the GPC layout, not the SM count, decides)
template <int MT>
int max_active_clusters(int splits) {
  static std::atomic<int> cache_all[64][9];
  std::atomic<int>* cache = cache_all[current_device()];
  if (!cache[splits].load(std::memory_order_relaxed)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, splits);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = RtCfg<MT>::kSmemBytes;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = splits;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, router_tc_kernel<MT>, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = sm_count() / (2 * splits);  // conservative
    }
    cache[splits].store(n > 0 ? n : 1, std::memory_order_relaxed);
  }
  return cache[splits].load(std::memory_order_relaxed);
}

template <int MT>
cudaError_t run(const CUtensorMap& mx, const CUtensorMap& mw, const float* bias, float* logits,
                int T, int H, int G, int32_t* dev_status, cudaStream_t stream) {
  using C = RtCfg<MT>;
  static std::atomic<unsigned long long> smem_set{0};  // devices whose limit is raised
  {
    cudaError_t e = moe_raise_smem(router_tc_kernel<MT>, C::kSmemBytes, smem_set);
    if (e != cudaSuccess) return e;
  }
  const int tiles = moe_cdiv(G, kTile) * moe_cdiv(T, kTile * MT);
  // split H over a cluster while all clusters still run in one wave and every
  // rank keeps at least two 64-wide K steps
  int splits = 1;
  while (splits < 8 && tiles <= max_active_clusters<MT>(2 * splits) &&
         H / (2 * splits) >= 2 * kBK)
    splits *= 2;
  const int kchunk = moe_cdiv(moe_cdiv(H, splits), kBK) * kBK;
  return moe_launch(router_tc_kernel<MT>, dim3(moe_cdiv(G, kTile), moe_cdiv(T, kTile * MT), splits),
                    dim3(192), C::kSmemBytes, stream, splits, mx, mw, bias, logits, T, H, G,
                    kchunk, dev_status);
}

}  // namespace

size_t router_tc_scratch_bytes(int H, int G) {
  return moe_align_up((size_t)3 * G * H * 2, 256);
}

cudaError_t launch_router_tc(const void* x, const float* wg, const float* gate_bias, float* logits,
                             int T, int H, int G, void* scratch, int32_t* dev_status,
                             cudaStream_t stream) {
  // 1. exact three-way bf16 split of the gate weight
  const long long n4 = (long long)G * H / 4;
  __nv_bfloat16* hi = static_cast<__nv_bfloat16*>(scratch);
  __nv_bfloat16* mid = hi + (size_t)G * H;
  __nv_bfloat16* lo = mid + (size_t)G * H;
  const int sgrid = (int)((n4 + 255) / 256 < 4 * sm_count() ? (n4 + 255) / 256 : 4 * sm_count());
  cudaError_t e = moe_launch(router_split_kernel, dim3(sgrid), dim3(256), 0, stream, 1,
                             reinterpret_cast<const float4*>(wg), n4, reinterpret_cast<uint2*>(hi),
                             reinterpret_cast<uint2*>(mid), reinterpret_cast<uint2*>(lo));
  if (e != cudaSuccess) return e;
  // 2. tensor maps: x [T][H] bf16, parts [3][G][H] bf16, 64 x 128 boxes, 128-byte swizzle
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorInvalidValue;
  CUtensorMap mx, mw;
  {
    cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    cuuint32_t box[2] = {kBK, kTile};
    cuuint32_t es[2] = {1, 1};
    if (enc(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)G, 3};
    cuuint64_t strides[2] = {(cuuint64_t)H * 2, (cuuint64_t)G * H * 2};
    cuuint32_t box[3] = {kBK, kTile, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, hi, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // 3. the GEMM: two 128-token halves per CTA when there are tokens enough
  if (T >= 2 * kTile * sm_count() / 4)
    return run<2>(mx, mw, gate_bias, logits, T, H, G, dev_status, stream);
  return run<1>(mx, mw, gate_bias, logits, T, H, G, dev_status, stream);
}
