// C ABI of the MoE-layer library: argument checks, workspace layout, launches.
// Every entry point validates on the host first (nothing is queued when a
// check fails), then queues kernels on the caller's stream and returns.  No
// allocation, no synchronisation -- the caller-scratch convention of "vLLM MoE
// permute optimisation: buffer pre-allocation" (vllm PR #43014), "1. C++
// kernel level": scratch is allocated once by the owner and reused, and each
// reused buffer's size is checked before use.
#include <stdio.h>

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"

namespace {

bool misaligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status_t check_dims(int T, int H, int E, int K) {
  if (T < 0 || H <= 0 || E <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || K > E || K > 32) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t check_cfg(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  moe_status_t s = check_dims(c->T_max, c->H, c->E, c->K);
  if (s != MOE_OK) return s;
  if (c->I <= 0 || c->I % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (c->mode != MOE_SCORE_SOFTMAX_RENORM && c->mode != MOE_SCORE_SIGMOID_BIAS_SCALED)
    return MOE_ERR_INVALID_ARG;
  if (c->wdtype != MOE_W_BF16 && c->wdtype != MOE_W_FP8E4M3_B128 && c->wdtype != MOE_W_MXFP4 &&
      c->wdtype != MOE_W8A8_FP8E4M3_B128)
    return MOE_ERR_UNSUPPORTED;
  if (c->wdtype == MOE_W8A8_FP8E4M3_B128 &&
      (c->dispatch == MOE_DISPATCH_SIMT || c->dispatch == MOE_DISPATCH_ONE_LAUNCH ||
       c->dispatch == MOE_DISPATCH_GEMV))
    return MOE_ERR_UNSUPPORTED;
  if (c->wdtype == MOE_W_MXFP4 && (c->H % 32 != 0 || c->I % 32 != 0)) return MOE_ERR_INVALID_ARG;
  if (c->dispatch < MOE_DISPATCH_PER_BLOCK || c->dispatch > MOE_DISPATCH_GEMV)
    return MOE_ERR_INVALID_ARG;
  if (c->m_skinny < -1) return MOE_ERR_INVALID_ARG;
  if (c->has_shared && (c->I_shared <= 0 || c->I_shared % 16 != 0)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)c->T_max * c->K > 0x7fffffff / 2) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// byte offset of the one-launch small-batch layer's counters inside `sync`
// (after the fused routing's 256 bytes and the K-slice counters)
size_t decode_sync_offset(const moe_config_t* c) {
  const int ms = c->m_skinny < 0 ? MOE_DEFAULT_M_SKINNY : c->m_skinny;
  const int tsp = c->T_max < ms ? c->T_max : ms;
  return 256 + moe_align_up(grouped_gemm_split_counter_bytes(tsp * c->K, c->E, c->H, c->I), 256);
}

// Whether moe_layer runs this batch as one launch (decode_layer.cu): always
// under MOE_DISPATCH_ONE_LAUNCH; under MOE_DISPATCH_PER_BLOCK where it measured
// faster than the multi-launch path on one GB300 (L2 flushed before each call):
// with a shared expert up to T = 4 (512 experts, K = 10: T=1 58 vs 82 us), and
// with E <= 128 from T = 4 to 8 (128 experts, K = 8: about even).  Elsewhere the
// split-K reductions at the phase boundaries cost more than the launches they
// save (128 experts at T = 1: 53 vs 44 us).
// The CUDA-core matrix-vector decode path (gemv_decode.cu): forced by
// MOE_DISPATCH_GEMV, taken under MOE_DISPATCH_PER_BLOCK where it measured
// faster than the tensor-core paths (L2 flushed): T <= 2 for bf16 and FP8
// weights, T = 1 for MXFP4 (T = 1: Qwen3-30B-A3B shape 33.4 vs 44.7 us,
// GPT-OSS-20B FP8 54.3 vs 65.8, shared-gate 42.6 vs 86.7, 896 experts 241.3
// vs 280.2); at T = 3, 4 the tensor-core paths were faster (e.g. 71.3 vs
// 79.5 us).
bool use_gemv(const moe_config_t* c, int T) {
  const int ms = c->m_skinny < 0 ? MOE_DEFAULT_M_SKINNY : c->m_skinny;
  if (!gemv_supported(T, c->H, c->I, c->has_shared ? c->I_shared : 0, c->wdtype, ms))
    return false;
  if (c->dispatch == MOE_DISPATCH_GEMV) return true;
  // MXFP4 (GPT-OSS-20B shape): T = 1 58.4 vs 66.8 us, T = 2 86.9 vs 85.3
  return c->dispatch == MOE_DISPATCH_PER_BLOCK && T <= (c->wdtype == MOE_W_MXFP4 ? 1 : 2);
}

bool one_launch(const moe_config_t* c, int T) {
  if (c->dispatch == MOE_DISPATCH_ONE_LAUNCH) return true;
  if (c->dispatch != MOE_DISPATCH_PER_BLOCK) return false;
  return (c->has_shared && T <= 4) || (c->E <= 128 && T >= 4 && T <= 8);
}

void layout_of(const moe_config_t* c, moe_workspace_layout_t* L) {
  const int G = c->E + (c->has_shared ? 1 : 0);
  const size_t Tm = (size_t)c->T_max, R = Tm * c->K;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = moe_align_up(off + bytes, 256);
    return o;
  };
  // zero before the first call, zero again after every call: completion
  // counters of the fused routing launches (first 256 bytes) and of the
  // in-kernel reduction of K slices in the small-batch GEMM launch
  // and of the one-launch small-batch layer (decode_sync_offset on)
  {
    const int ms0 = c->m_skinny < 0 ? MOE_DEFAULT_M_SKINNY : c->m_skinny;
    const int tsp = c->T_max < ms0 ? c->T_max : ms0;
    L->sync = take(decode_sync_offset(c) +
                   4 * decode_layer_sync_words(c->T_max, c->E, c->K, c->H, c->I,
                                               c->has_shared ? c->I_shared : 0, c->has_shared));
    (void)tsp;
  }
  L->logits = take(Tm * G * 4);
  L->ids = take(R * 4);
  L->weights = take(R * 4);
  L->shared_gate = take(Tm * 4);
  L->offsets = take((size_t)(c->E + 1) * 4);
  L->row_to_flat = take(R * 4);
  L->flat_to_row = take(R * 4);
  L->xp = take(R * c->H * 2);
  L->hact = take(R * c->I * 2);
  L->y = take(R * c->H * 2);
  L->shared_hact = take(c->has_shared ? Tm * c->I_shared * 2 : 0);
  L->shared_y = take(c->has_shared ? Tm * c->H * 2 : 0);
  L->block_variant = take((size_t)c->E * 4);
  // the permute's chunk counts: moe_layer's fused routing (T > 32) or the
  // stand-alone permute, whichever needs more
  const size_t pb = permute_scratch_bytes(c->T_max, c->E, c->K);
  const size_t rb = route_prefill_scratch_bytes(c->T_max, c->E);
  L->permute_scratch = take(pb > rb ? pb : rb);
  L->gemm_scratch = take(grouped_gemm_scratch_bytes_ex((int)R, c->E, c->H, c->I, c->wdtype));
  L->shared_gemm_scratch = take(c->has_shared ? grouped_gemm_scratch_bytes(c->T_max, 1) : 0);
  // split-K slices for small batches (all blocks skinny: T <= m_skinny)
  const int ms = c->m_skinny < 0 ? MOE_DEFAULT_M_SKINNY : c->m_skinny;
  const int t_split = c->T_max < ms ? c->T_max : ms;
  // the three bf16 parts of the gate weight for the tensor-core router
  L->router_split = take(c->T_max >= kRouterTcMinT ? router_tc_scratch_bytes(c->H, G) : 0);
  // split-K slices for small batches (all blocks skinny: T <= m_skinny), or
  // the one-launch layer's partial sums (the two never run in one call); last
  const size_t sk = grouped_gemm_splitk_bytes(t_split * c->K, c->H, c->I);
  const size_t dp = decode_layer_part_bytes();
  L->splitk = take(sk > dp ? sk : dp);
  L->total = off;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported combination";
    case MOE_ERR_WORKSPACE: return "scratch or workspace too small";
    case MOE_ERR_MISALIGNED: return "misaligned pointer";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_STATUS: return "device status error";
  }
  return "unknown status";
}

int moe_default_m_skinny(void) { return MOE_DEFAULT_M_SKINNY; }

int moe_block_variant(int64_t m_size, int64_t R, int E, int m_skinny, int dispatch, int wdtype) {
  if (m_skinny < 0) m_skinny = MOE_DEFAULT_M_SKINNY;
  return moe_variant_of(m_size, R, E, m_skinny, dispatch, wdtype);
}

moe_status_t moe_router_gemm(const void* x, const float* wg, const float* gate_bias,
                             float* logits, int T, int H, int G, moe_stream_t stream) {
  if (T < 0 || H <= 0 || G <= 0 || H % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !wg || !logits) return MOE_ERR_INVALID_ARG;
  if (misaligned(x, 16) || misaligned(wg, 16) || misaligned(logits, 4) ||
      (gate_bias && misaligned(gate_bias, 4)))
    return MOE_ERR_MISALIGNED;
  return cuda_status(launch_router_gemm(x, wg, gate_bias, logits, T, H, G, stream));
}

moe_status_t moe_router_tc_scratch_bytes(int H, int G, size_t* bytes) {
  if (!bytes || H <= 0 || G <= 0 || H % 8 != 0) return MOE_ERR_INVALID_ARG;
  *bytes = router_tc_scratch_bytes(H, G);
  return MOE_OK;
}

moe_status_t moe_router_gemm_tc(const void* x, const float* wg, const float* gate_bias,
                                float* logits, int T, int H, int G, void* scratch,
                                size_t scratch_bytes, int32_t* dev_status, moe_stream_t stream) {
  if (T < 0 || H <= 0 || G <= 0 || H % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !wg || !logits || !scratch) return MOE_ERR_INVALID_ARG;
  if (scratch_bytes < router_tc_scratch_bytes(H, G)) return MOE_ERR_WORKSPACE;
  if (misaligned(x, 16) || misaligned(wg, 16) || misaligned(logits, 4) ||
      misaligned(scratch, 256) || (gate_bias && misaligned(gate_bias, 4)))
    return MOE_ERR_MISALIGNED;
  return cuda_status(
      launch_router_tc(x, wg, gate_bias, logits, T, H, G, scratch, dev_status, stream));
}

moe_status_t moe_topk_route(const float* logits, int ld_logits, const float* sel_bias, int T,
                            int E, int K, int mode, float scale, int32_t* ids, float* weights,
                            float* shared_gate, moe_stream_t stream) {
  if (T < 0 || E <= 0 || E > 1024 || K <= 0 || K > E || K > 32) return MOE_ERR_INVALID_ARG;
  if (ld_logits < E || (shared_gate && ld_logits < E + 1)) return MOE_ERR_INVALID_ARG;
  if (mode != MOE_SCORE_SOFTMAX_RENORM && mode != MOE_SCORE_SIGMOID_BIAS_SCALED)
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !ids || !weights) return MOE_ERR_INVALID_ARG;
  if (misaligned(logits, 4) || misaligned(ids, 4) || misaligned(weights, 4) ||
      (sel_bias && misaligned(sel_bias, 4)) || (shared_gate && misaligned(shared_gate, 4)))
    return MOE_ERR_MISALIGNED;
  return cuda_status(launch_topk_route(logits, ld_logits, sel_bias, T, E, K, mode, scale, ids,
                                       weights, shared_gate, stream));
}

moe_status_t moe_permute_scratch_bytes(int T, int E, int K, size_t* bytes) {
  if (!bytes || T < 0 || E <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  *bytes = permute_scratch_bytes(T, E, K);
  return MOE_OK;
}

moe_status_t moe_permute(const void* x, const int32_t* ids, int T, int H, int E, int K,
                         int32_t* offsets, int32_t* row_to_flat, int32_t* flat_to_row, void* xp,
                         void* scratch, size_t scratch_bytes, int32_t* dev_status,
                         moe_stream_t stream) {
  moe_status_t s = check_dims(T, H, E, K);
  if (s != MOE_OK) return s;
  if (!offsets || !scratch) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !row_to_flat || !flat_to_row || (xp && !x))) return MOE_ERR_INVALID_ARG;
  if (scratch_bytes < permute_scratch_bytes(T, E, K)) return MOE_ERR_WORKSPACE;
  if (misaligned(scratch, 256) || misaligned(offsets, 4) || (ids && misaligned(ids, 4)) ||
      (row_to_flat && misaligned(row_to_flat, 4)) || (flat_to_row && misaligned(flat_to_row, 4)) ||
      (xp && (misaligned(xp, 16) || misaligned(x, 16))))
    return MOE_ERR_MISALIGNED;
  return cuda_status(launch_permute(x, ids, T, H, E, K, offsets, row_to_flat, flat_to_row, xp,
                                    scratch, dev_status, stream));
}

moe_status_t moe_grouped_gemm_scratch_bytes(int R, int E_blocks, size_t* bytes) {
  if (!bytes || R < 0 || E_blocks <= 0) return MOE_ERR_INVALID_ARG;
  *bytes = grouped_gemm_scratch_bytes(R, E_blocks);
  return MOE_OK;
}

moe_status_t moe_grouped_gemm_scratch_bytes_ex(int R, int E_blocks, int H, int I, int wdtype,
                                               size_t* bytes) {
  if (!bytes || R < 0 || E_blocks <= 0 || H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
  *bytes = grouped_gemm_scratch_bytes_ex(R, E_blocks, H, I, wdtype);
  return MOE_OK;
}

moe_status_t moe_grouped_gemm(const void* xp, const int32_t* offsets, int E_blocks, int R, int H,
                              int I, int wdtype, const void* w1, const void* w3, const void* w2,
                              const float* s1, const float* s3, const float* s2, void* hact,
                              void* y, int m_skinny, int dispatch, int32_t* block_variant,
                              void* scratch, size_t scratch_bytes, int32_t* dev_status,
                              moe_stream_t stream) {
  if (E_blocks <= 0 || R < 0 || m_skinny < -1) return MOE_ERR_INVALID_ARG;
  if (dispatch < MOE_DISPATCH_PER_BLOCK || dispatch > MOE_DISPATCH_SIMT) return MOE_ERR_INVALID_ARG;
  const int chk = grouped_gemm_check(H, I, wdtype);
  if (chk != MOE_OK) return (moe_status_t)chk;
  if (!w1 || !w3 || !w2 || !scratch) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!xp || !hact || !y)) return MOE_ERR_INVALID_ARG;
  if (wdtype != MOE_W_BF16 && (!s1 || !s3 || !s2)) return MOE_ERR_INVALID_ARG;
  if (wdtype == MOE_W8A8_FP8E4M3_B128 && dispatch == MOE_DISPATCH_SIMT) return MOE_ERR_UNSUPPORTED;
  if (scratch_bytes < grouped_gemm_scratch_bytes_ex(R, E_blocks, H, I, wdtype))
    return MOE_ERR_WORKSPACE;
  if (misaligned(scratch, 256) || misaligned(w1, 16) || misaligned(w3, 16) || misaligned(w2, 16) ||
      (xp && misaligned(xp, 16)) || (hact && misaligned(hact, 16)) || (y && misaligned(y, 16)) ||
      (offsets && misaligned(offsets, 4)) || (block_variant && misaligned(block_variant, 4)))
    return MOE_ERR_MISALIGNED;
  return cuda_status(launch_grouped_gemm(xp, offsets, E_blocks, R, H, I, wdtype, w1, w3, w2, s1,
                                         s3, s2, hact, y, m_skinny, dispatch, block_variant,
                                         scratch, dev_status, stream));
}

moe_status_t moe_unpermute(const void* y, const int32_t* flat_to_row, const float* weights, int T,
                           int K, int H, const void* shared_y, const float* shared_gate,
                           void* out, moe_stream_t stream) {
  if (T < 0 || K <= 0 || H <= 0 || H % 8 != 0) return MOE_ERR_INVALID_ARG;
  if ((shared_y == nullptr) != (shared_gate == nullptr)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y || !flat_to_row || !weights || !out) return MOE_ERR_INVALID_ARG;
  if (misaligned(y, 16) || misaligned(out, 16) || misaligned(flat_to_row, 4) ||
      misaligned(weights, 4) || (shared_y && (misaligned(shared_y, 16) || misaligned(shared_gate, 4))))
    return MOE_ERR_MISALIGNED;
  return cuda_status(
      launch_unpermute(y, flat_to_row, weights, T, K, H, shared_y, shared_gate, out, stream));
}

moe_status_t moe_workspace_layout(const moe_config_t* cfg, moe_workspace_layout_t* layout) {
  const moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!layout) return MOE_ERR_INVALID_ARG;
  layout_of(cfg, layout);
  return MOE_OK;
}

moe_status_t moe_workspace_bytes(const moe_config_t* cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  moe_workspace_layout_t L;
  const moe_status_t s = moe_workspace_layout(cfg, &L);
  if (s != MOE_OK) return s;
  *bytes = L.total;
  return MOE_OK;
}

moe_status_t moe_layer(const moe_config_t* cfg, int T, const void* x, const moe_weights_t* w,
                       void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                       moe_stream_t stream) {
  moe_status_t s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (T < 0 || T > cfg->T_max) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w || !out || !workspace || !w->wg || !w->w1 || !w->w3 || !w->w2)
    return MOE_ERR_INVALID_ARG;
  if (cfg->wdtype != MOE_W_BF16 && (!w->s1 || !w->s3 || !w->s2)) return MOE_ERR_INVALID_ARG;
  if (cfg->has_shared && (!w->sw1 || !w->sw3 || !w->sw2)) return MOE_ERR_INVALID_ARG;
  moe_workspace_layout_t L;
  layout_of(cfg, &L);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (misaligned(workspace, 256) || misaligned(x, 16) || misaligned(out, 16) ||
      misaligned(w->wg, 16) || misaligned(w->w1, 16) || misaligned(w->w3, 16) ||
      misaligned(w->w2, 16) ||
      (cfg->has_shared && (misaligned(w->sw1, 16) || misaligned(w->sw3, 16) || misaligned(w->sw2, 16))))
    return MOE_ERR_MISALIGNED;

  char* ws = static_cast<char*>(workspace);
  float* logits = reinterpret_cast<float*>(ws + L.logits);
  int32_t* ids = reinterpret_cast<int32_t*>(ws + L.ids);
  float* wts = reinterpret_cast<float*>(ws + L.weights);
  float* gsh = reinterpret_cast<float*>(ws + L.shared_gate);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  int32_t* r2f = reinterpret_cast<int32_t*>(ws + L.row_to_flat);
  int32_t* f2r = reinterpret_cast<int32_t*>(ws + L.flat_to_row);
  void* xp = ws + L.xp;
  void* hact = ws + L.hact;
  void* y = ws + L.y;
  const int E = cfg->E, K = cfg->K, H = cfg->H;
  const int G = E + (cfg->has_shared ? 1 : 0);
  const int R = T * K;

  int32_t* bvar = reinterpret_cast<int32_t*>(ws + L.block_variant);
  const int Is = cfg->has_shared ? cfg->I_shared : 0;
  const bool gemv = use_gemv(cfg, T);
  if (one_launch(cfg, T) && !gemv &&
      decode_layer_supported(T, E, K, H, cfg->I, Is, cfg->has_shared, cfg->wdtype, cfg->dispatch,
                             cfg->m_skinny < 0 ? MOE_DEFAULT_M_SKINNY : cfg->m_skinny)) {
    // small batch: the whole layer in one launch
    DecodeLayerArgs a;
    a.x = x; a.wg = w->wg; a.gate_bias = w->gate_bias; a.sel_bias = w->sel_bias;
    a.T = T; a.T_max = cfg->T_max; a.H = H; a.G = G; a.E = E; a.K = K; a.I = cfg->I; a.Is = Is;
    a.mode = cfg->mode; a.has_shared = cfg->has_shared; a.scale = cfg->routed_scale;
    a.w1 = w->w1; a.w3 = w->w3; a.w2 = w->w2; a.sw1 = w->sw1; a.sw3 = w->sw3; a.sw2 = w->sw2;
    a.logits = logits; a.ids = ids; a.weights = wts; a.shared_gate = gsh;
    a.offsets = offsets; a.row_to_flat = r2f; a.flat_to_row = f2r; a.block_variant = bvar;
    a.hact = hact; a.y = y; a.sh_hact = ws + L.shared_hact; a.sh_y = ws + L.shared_y; a.out = out;
    a.part = reinterpret_cast<float*>(ws + L.splitk);
    a.sync = reinterpret_cast<uint32_t*>(ws + L.sync + decode_sync_offset(cfg));
    a.dev_status = dev_status;
    a.m_skinny = cfg->m_skinny; a.dispatch = cfg->dispatch; a.wdtype = cfg->wdtype;
    return cuda_status(launch_decode_layer(a, stream));
  }
  const bool decode = T <= kRouteDecodeMaxT;
  bool planned = true;  // the grouped-GEMM plan was written by the routing launch
  cudaError_t e;
  // the matrix-vector path where G1's CTAs can route the batch themselves
  // (gemv_routes): the logits alone here
  const bool gemv_route = decode && gemv && gemv_routes(T, E, K);
  if (gemv_route) {
    e = launch_router_gemm(x, w->wg, w->gate_bias, logits, T, H, G, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else if (decode) {
    // small batch: router + top-K + permute + GEMM plan in one launch
    RouteDecodeArgs a;
    a.x = x; a.wg = w->wg; a.gate_bias = w->gate_bias; a.logits = logits;
    a.T = T; a.H = H; a.G = G; a.sel_bias = w->sel_bias; a.E = E; a.K = K;
    a.mode = cfg->mode; a.scale = cfg->routed_scale; a.ids = ids; a.weights = wts;
    a.shared_gate = cfg->has_shared ? gsh : nullptr; a.offsets = offsets;
    a.row_to_flat = r2f; a.flat_to_row = f2r; a.dev_status = dev_status;
    a.m_skinny = cfg->m_skinny; a.dispatch = cfg->dispatch; a.wdtype = cfg->wdtype;
    a.gemm_scratch = ws + L.gemm_scratch; a.block_variant = bvar;
    a.done_ctr = reinterpret_cast<unsigned int*>(ws + L.sync);
    e = launch_route_decode(a, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (decode) {
    if (gemv) {
      // the expert GEMMs as matrix-vector products, then the combine
      const moe_plan::PlanView pv = moe_plan::plan_view(ws + L.gemm_scratch, R, E);
      GemvArgs g{};
      g.x = x; g.T = T; g.H = H; g.I = cfg->I; g.K = K; g.Is = Is; g.wdtype = cfg->wdtype;
      g.counts = pv.counts; g.items = pv.items[0];
      g.row_to_flat = r2f; g.flat_to_row = f2r; g.ids = ids; g.weights = wts;
      g.w1 = w->w1; g.w3 = w->w3; g.w2 = w->w2; g.s1 = w->s1; g.s3 = w->s3; g.s2 = w->s2;
      g.hact = hact; g.y = y; g.sw1 = w->sw1; g.sw3 = w->sw3; g.sw2 = w->sw2;
      g.shared_hact = ws + L.shared_hact; g.shared_y = ws + L.shared_y;
      g.shared_gate = cfg->has_shared ? gsh : nullptr; g.out = out;
      g.route = gemv_route;
      if (gemv_route) {
        GemvRoute& rt = g.rt;
        rt.logits = logits; rt.G = G; rt.E = E; rt.mode = cfg->mode;
        rt.scale = cfg->routed_scale; rt.sel_bias = w->sel_bias; rt.ids = ids; rt.weights = wts;
        rt.shared_gate = cfg->has_shared ? gsh : nullptr; rt.offsets = offsets;
        rt.row_to_flat = r2f; rt.flat_to_row = f2r; rt.block_variant = bvar;
        rt.plan_counts = pv.counts; rt.plan_items = pv.items[0]; rt.plan_done = pv.done[0];
        rt.m_skinny = cfg->m_skinny < 0 ? MOE_DEFAULT_M_SKINNY : cfg->m_skinny;
        rt.dispatch = cfg->dispatch;
      }
      return cuda_status(launch_gemv_layer(g, stream));
    }
  } else {
    e = T >= kRouterTcMinT
            ? launch_router_tc(x, w->wg, w->gate_bias, logits, T, H, G, ws + L.router_split,
                               dev_status, stream)
            : launch_router_gemm(x, w->wg, w->gate_bias, logits, T, H, G, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (route_prefill_fits(T, E, K)) {
      // top-K + chunk histograms + (last CTA) offsets and GEMM plan, then the
      // stable scatter
      RoutePrefillArgs a;
      a.logits = logits; a.ld = G; a.sel_bias = w->sel_bias; a.T = T; a.E = E; a.K = K;
      a.mode = cfg->mode; a.scale = cfg->routed_scale; a.ids = ids; a.weights = wts;
      a.shared_gate = cfg->has_shared ? gsh : nullptr;
      a.counts = reinterpret_cast<int32_t*>(ws + L.permute_scratch); a.offsets = offsets;
      a.row_to_flat = r2f; a.flat_to_row = f2r;
      a.m_skinny = cfg->m_skinny; a.dispatch = cfg->dispatch; a.wdtype = cfg->wdtype;
      a.gemm_scratch = ws + L.gemm_scratch; a.block_variant = bvar;
      a.done_ctr = reinterpret_cast<unsigned int*>(ws + L.sync + 64);
      e = launch_route_prefill(a, stream);
    } else {
      // very large batches (the fused routing's shared memory would not
      // fit): top-K, the multi-kernel permute, and the GEMM's own plan
      e = launch_topk_route(logits, G, w->sel_bias, T, E, K, cfg->mode, cfg->routed_scale, ids,
                            wts, cfg->has_shared ? gsh : nullptr, stream);
      if (e != cudaSuccess) return MOE_ERR_CUDA;
      e = launch_permute(x, ids, T, H, E, K, offsets, r2f, f2r, nullptr, ws + L.permute_scratch,
                         dev_status, stream);
      planned = false;
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  // the permuted activations: each row of x written to its token's K rows --
  // except for small batches on the tensor cores, where G1 copies its few
  // rows per tile straight from x itself
  // (not with FP8 weights: there a stage must also pass the converter warps,
  // and tying the row copies' completion to the pipeline's progress stalled
  // it -- gpt-oss-20b shape T=32: 217 -> 308 us)
  const bool gather = decode && cfg->dispatch != MOE_DISPATCH_SIMT &&
                      cfg->wdtype == MOE_W_BF16;
  if (!gather) {
    e = launch_permute_copy(x, f2r, T, K, H, xp, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  e = launch_grouped_gemm(xp, offsets, E, R, H, cfg->I, cfg->wdtype, w->w1, w->w3, w->w2, w->s1,
                          w->s3, w->s2, hact, y, cfg->m_skinny, cfg->dispatch, bvar,
                          ws + L.gemm_scratch, dev_status, stream, /*max_rows=*/T,
                          /*plan_ready=*/planned, reinterpret_cast<float*>(ws + L.splitk),
                          L.total - L.splitk, gather ? x : nullptr, gather ? r2f : nullptr, K,
                          reinterpret_cast<int32_t*>(ws + L.sync + 256));
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  void* sh_y = nullptr;
  if (cfg->has_shared) {
    sh_y = ws + L.shared_y;
    e = launch_grouped_gemm(x, nullptr, 1, T, H, cfg->I_shared, MOE_W_BF16, w->sw1, w->sw3, w->sw2,
                            nullptr, nullptr, nullptr, ws + L.shared_hact, sh_y, cfg->m_skinny,
                            cfg->dispatch, nullptr, ws + L.shared_gemm_scratch, dev_status, stream,
                            /*max_rows=*/T);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  e = launch_unpermute(y, f2r, wts, T, K, H, sh_y, cfg->has_shared ? gsh : nullptr, out, stream);
  return cuda_status(e);
}

}  // extern "C"

moe_status_t moe_bounded_wait_check(const int32_t* counter, int target, int limit_us,
                                    int32_t* dev_status, moe_stream_t stream) {
  if (!counter || !dev_status || limit_us <= 0 || limit_us > 10000000) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_bounded_wait_check(counter, target, (uint64_t)limit_us * 1000,
                                               dev_status, static_cast<cudaStream_t>(stream)));
}
