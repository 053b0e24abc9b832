// Launchers shared between the C-ABI layer and the kernel translation units.
// Every launcher queues work on `stream` and returns cudaGetLastError().
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

cudaError_t launch_router_gemm(const void* x, const float* wg, const float* gate_bias,
                               float* logits, int T, int H, int G, cudaStream_t stream);

// Router on the tensor cores (exact three-way bf16 split of wg, three MMAs per
// K step into one fp32 accumulator); scratch holds the split parts.
constexpr int kRouterTcMinT = 64;  // moe_layer uses it from this batch size on
size_t router_tc_scratch_bytes(int H, int G);
cudaError_t launch_router_tc(const void* x, const float* wg, const float* gate_bias,
                             float* logits, int T, int H, int G, void* scratch,
                             int32_t* dev_status, cudaStream_t stream);

cudaError_t launch_topk_route(const float* logits, int ld, const float* sel_bias, int T, int E,
                              int K, int mode, float scale, int32_t* ids, float* weights,
                              float* shared_gate, cudaStream_t stream);

size_t permute_scratch_bytes(int T, int E, int K);
cudaError_t launch_permute(const void* x, const int32_t* ids, int T, int H, int E, int K,
                           int32_t* offsets, int32_t* row_to_flat, int32_t* flat_to_row,
                           void* xp, void* scratch, int32_t* dev_status, cudaStream_t stream);

size_t grouped_gemm_scratch_bytes(int R, int E_blocks);
// scratch of a grouped-GEMM call: the plan, plus for W8A8 the quantised
// activations (w8a8_act_bytes) right after it
size_t grouped_gemm_scratch_bytes_ex(int R, int E_blocks, int H, int I, int wdtype);
// W8A8 expert GEMMs (gemm_w8a8.cu): e4m3 copies of xp and hact with their
// per-(row, 128 columns) scales live in act_scratch (w8a8_act_bytes of it);
// the plan's tile list (every non-empty block, 128-row items) drives both GEMMs
size_t w8a8_act_bytes(int R, int H, int I);
cudaError_t launch_w8a8(const void* xp, int R, int E_blocks, int H, int I, const void* w1,
                        const void* w3, const void* w2, const float* s1, const float* s3,
                        const float* s2, void* hact, void* y, const int32_t* counts,
                        const int4* tile_items, void* act_scratch, int32_t* dev_status,
                        cudaStream_t stream);
int grouped_gemm_check(int H, int I, int wdtype);  // 0 ok, else a moe_status_t
// plan_ready: the plan in `scratch` was already written (by the fused decode
// routing kernel); only the GEMM kernels are launched.
cudaError_t launch_grouped_gemm(const void* xp, const int32_t* offsets, int E_blocks, int R,
                                int H, int I, int wdtype, const void* w1, const void* w3,
                                const void* w2, const float* s1, const float* s3,
                                const float* s2, void* hact, void* y, int m_skinny,
                                int dispatch, int32_t* block_variant, void* scratch,
                                int32_t* dev_status, cudaStream_t stream, int max_rows = -1,
                                bool plan_ready = false, float* splitk_buf = nullptr,
                                size_t splitk_bytes = 0, const void* gather_x = nullptr,
                                const int32_t* gather_rows = nullptr, int gather_k = 0,
                                int32_t* split_cnt = nullptr);
// zero-initialised counters for the in-kernel reduction of K slices in the
// small-batch launch (every call leaves them zero again)
size_t grouped_gemm_split_counter_bytes(int R, int E_blocks, int H, int I);
// fp32 bytes for split-K slices of the skinny variant in moe_layer's decode
// regime (at most 4 slices of R x max(2I, H) partial sums)
size_t grouped_gemm_splitk_bytes(int R, int H, int I);

// xp[flat_to_row[t*K+k]] = x[t] (the permute's copy step alone)
// one bounded wait (the fused GEMM's cross-CTA wait) on *counter >= target
cudaError_t launch_bounded_wait_check(const int32_t* counter, int target, uint64_t limit_ns,
                                      int32_t* dev_status, cudaStream_t stream);
cudaError_t launch_permute_copy(const void* x, const int32_t* flat_to_row, int T, int K, int H,
                                void* xp, cudaStream_t stream);

// Fused decode routing (T <= kRouteDecodeMaxT): router + top-K + permute +
// grouped-GEMM plan in one launch.  done_ctr must be zero before the launch
// and is zero again after it.
constexpr int kRouteDecodeMaxT = 32;
// Decode batches on the CUDA cores (gemv_decode.cu): G1 and G2 as
// matrix-vector products over the plan's skinny list (x rows gathered through
// row_to_flat), the shared expert riding in both launches, then the combine.
constexpr int kGemvMaxT = 4;
// The routing that G1's CTAs run themselves (gemv_routes): every CTA routes
// the batch from the logits, CTA 0 writes the results below for the later
// launches and the workspace.
struct GemvRoute {
  const float* logits;  // [T][G]
  int G, E, mode;
  float scale;
  const float* sel_bias;
  int32_t* ids;
  float *weights, *shared_gate;  // shared_gate nullable
  int32_t *offsets, *row_to_flat, *flat_to_row, *block_variant;
  int32_t* plan_counts;  // the plan head, its skinny list and done flags
  int4* plan_items;
  int32_t* plan_done;
  int m_skinny, dispatch;
};
struct GemvArgs {
  const void* x;
  int T, H, I, K, Is, wdtype;
  const int32_t* counts;  // the plan's list counts; items: its skinny list
  const int4* items;
  const int32_t *row_to_flat, *flat_to_row, *ids;
  const float* weights;
  const void *w1, *w3, *w2;
  const float *s1, *s3, *s2;
  void *hact, *y;
  const void *sw1, *sw3, *sw2;
  void *shared_hact, *shared_y;
  const float* shared_gate;
  void* out;
  bool route;  // G1 routes the batch itself (rt), after the logits-only router
  GemvRoute rt;
};
bool gemv_supported(int T, int H, int I, int Is, int wdtype, int m_skinny);
// G1 can route the batch itself: T * K <= 32, and E <= 128 or (K <= 16 and
// E <= 4096 / T', T' = T rounded up to a power of two)
bool gemv_routes(int T, int E, int K);
cudaError_t launch_gemv_layer(const GemvArgs& a, cudaStream_t stream);

struct RouteDecodeArgs {
  const void* x;
  const float* wg;
  const float* gate_bias;
  float* logits;
  int T, H, G;
  const float* sel_bias;
  int E, K, mode;
  float scale;
  int32_t* ids;
  float* weights;
  float* shared_gate;
  int32_t* offsets;
  int32_t* row_to_flat;
  int32_t* flat_to_row;
  int32_t* dev_status;
  int m_skinny, dispatch, wdtype;
  void* gemm_scratch;  // plan written here (grouped-GEMM scratch layout for R = T*K)
  int32_t* block_variant;
  unsigned int* done_ctr;
};
cudaError_t launch_route_decode(const RouteDecodeArgs& args, cudaStream_t stream);

// Fused routing above the decode range: top-K + per-chunk expert histograms +
// (last CTA) scan to offsets and the grouped-GEMM plan, then the stable
// scatter -- two launches in all.  done_ctr must be zero before the launch and
// is zero again after it.  counts: route_prefill_scratch_bytes(T, E) bytes.
struct RoutePrefillArgs {
  const float* logits;
  int ld;
  const float* sel_bias;
  int T, E, K, mode;
  float scale;
  int32_t* ids;
  float* weights;
  float* shared_gate;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_to_flat;
  int32_t* flat_to_row;
  int m_skinny, dispatch, wdtype;
  void* gemm_scratch;  // plan written here (grouped-GEMM scratch layout for R = T*K)
  int32_t* block_variant;
  unsigned int* done_ctr;
};
bool route_prefill_fits(int T, int E, int K);  // shared memory and E limits
size_t route_prefill_scratch_bytes(int T, int E);
cudaError_t launch_route_prefill(const RoutePrefillArgs& args, cudaStream_t stream);

cudaError_t launch_unpermute(const void* y, const int32_t* flat_to_row, const float* weights,
                             int T, int K, int H, const void* shared_y, const float* shared_gate,
                             void* out, cudaStream_t stream);

// The whole layer for small batches in one cooperative launch (decode_layer.cu):
// router, top-K, permute, G1/G2 (+ shared expert) and combine.  The sync
// words must be zero before the launch and are zero again after it.
constexpr int kDecodeMaxT = 16;      // tokens the kernel takes
constexpr int kDecodeMaxGrid = 256;  // SMs it can use (one CTA each)
struct DecodeLayerArgs {
  const void* x;
  const float* wg;
  const float* gate_bias;
  const float* sel_bias;
  int T, T_max, H, G, E, K, I, Is, mode, has_shared;
  float scale;
  const void* w1;
  const void* w3;
  const void* w2;
  const void* sw1;
  const void* sw3;
  const void* sw2;
  float* logits;
  int32_t* ids;
  float* weights;
  float* shared_gate;
  int32_t* offsets;
  int32_t* row_to_flat;
  int32_t* flat_to_row;
  int32_t* block_variant;
  void* hact;
  void* y;
  void* sh_hact;
  void* sh_y;
  void* out;
  float* part;     // decode_layer_part_bytes()
  uint32_t* sync;  // decode_layer_sync_words(...) words
  int32_t* dev_status;
  int m_skinny, dispatch, wdtype;
};
size_t decode_layer_sync_words(int T_max, int E, int K, int H, int I, int Is, int has_shared);
size_t decode_layer_part_bytes();
bool decode_layer_supported(int T, int E, int K, int H, int I, int Is, int has_shared, int wdtype,
                            int dispatch, int m_skinny);
cudaError_t launch_decode_layer(const DecodeLayerArgs& args, cudaStream_t stream);
