// Host-side declarations shared by the library's translation units: the
// kernel launchers each .cu file exports to the C-ABI layer (api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace ep {

// Kernel launch through cudaLaunchKernelEx (one code path for every kernel).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Dynamic shared-memory limit of a kernel: the device's opt-in maximum less
// the kernel's static shared memory -- the same value whatever handle asks,
// so no later call lowers it under an earlier one.  Fails (without touching
// the attribute) if `needed` bytes do not fit under it; *limit (if given)
// receives the limit.
inline cudaError_t set_dynamic_smem_limit(const void* kernel, size_t needed, size_t optin, size_t* limit = nullptr) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  const size_t lim = optin > fa.sharedSizeBytes ? optin - fa.sharedSizeBytes : 0;
  if (limit) *limit = lim;
  if (needed > lim) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(lim));
}

struct RouteParams;  // routing.cuh

struct LowLatencyOutPtrs {
  int* recv_count;  // [E] or null
  int* ll_idx;      // [T][k]
  int* ll_slot;     // [T][k]
  int M;
};

struct LayoutOutPtrs {
  int2* dst;
  int* idx32;
  int* recv_per_rank;
  int* rank_offset;
  int* recv_per_expert;
  int* num_tokens_per_rank;
  int* num_tokens_per_expert;
  uint8_t* is_token_in_rank;
};

void launch_layout(const RouteParams& p, const LayoutOutPtrs& out, size_t smem, cudaStream_t stream);
cudaError_t configure_layout(size_t needed, size_t optin, size_t* limit = nullptr);
// token-per-lane layout (R <= 64)
constexpr int kLayoutTokenChunk = 256;
void launch_layout_tokens(const RouteParams& p, const LayoutOutPtrs& out, cudaStream_t stream);
size_t layout_tokens_smem(int R, int E, int CT, int kmax);
cudaError_t configure_layout_tokens(size_t needed, size_t optin);

// Normal dispatch: one warp per token, persistent grid.
struct DispatchArgs {
  const uint16_t* x;           // [T][H] bf16
  const float* topk_weights;   // [T][k] or null
  const int2* dst;             // [T][kmax]
  const int* idx32;            // [T][k]
  const int* rank_offset;      // [R+1]
  void* recv_x;                // [cap][H] bf16 or e4m3
  float* recv_scales;          // [cap][H/128]
  int* recv_src_idx;           // [cap] or null
  int* recv_topk_idx;          // [cap][k] or null
  float* recv_topk_weights;    // [cap][k] or null
  long long cap;
  int T, H, k, kmax, El;
  int* err;
};
void launch_dispatch(const DispatchArgs& a, bool fp8, int blocks, cudaStream_t stream);
int dispatch_threads();
const void* dispatch_kernel(bool fp8);

// combine: one warp per (token, 1024-channel part), every receive layout.
enum : int { kSrcRanks = 0, kSrcLowLatency = 1, kSrcExpertMajor = 2 };
struct CombineArgs {
  const void* y;               // rows [.][H]: bf16, or e4m3 bytes with y_scales
  const float* y_scales;       // [y_rows][H/128] (e4m3 rows)
  uint16_t* out;               // [T][H]
  long long y_rows;
  int T, H, k, kmax, R, E;
  // rank-major (normal) rows
  const int2* dst;             // [T][kmax]
  const int* rank_offset;      // [R+1]
  const float* recv_topk_weights;  // [y_rows][k] or null
  float* combined_topk_weights;    // [T][k] (with recv_topk_weights)
  // low-latency / expert-major rows: per (token, k) entry its expert id and
  // its slot inside the expert
  const int* ent_idx;          // [T][k]
  const int* ent_slot;         // [T][k]
  const float* topk_weights;   // [T][k] (low latency)
  int M;                       // low latency: rows per expert
  const int* expert_offset;    // expert-major: [E+1] first row of each expert
  int* err;
};
void launch_combine(const CombineArgs& a, int src, bool fp8, int blocks, cudaStream_t stream);
size_t combine_smem_bytes(int src, int R, int E);
int combine_threads();
const void* combine_kernel(int src, bool fp8);

// Control words shared by the row-moving kernels (the handle's
// fused_barrier array): [0] grid-barrier arrivals, [1] launch generation,
// [2] row-claim counter, [3] blocks finished, [4 + b] block b's "destinations
// published" word of the fused kernel (= generation + 1 once written).  The
// last block to finish a launch resets [0], [2], [3] and (fused kernel)
// advances [1].
constexpr int kCtlClaim = 2, kCtlDone = 3, kCtlPub = 4;
// Tokens per row claim: as few as the claim counter and the claim's latency
// allow.  (1) One atomic on one address completes about every 3.5 ns, so the
// claims must come at most about every 8 ns over a launch that moves its
// bytes at ~6 TB/s: a token moving b bytes takes b / 6000 ns of the GPU's
// time, hence at least ceil(48000 / b) tokens per claim.  (2) With blocks > 0
// (the rank-major fused kernel, whose tokens are the quickest to move): a
// producer claims one claim ahead, and a claim's round trip (~1.5 us under
// load) must not outlast moving the claim's tokens at the block's share of
// the rate, 6 TB/s / blocks: at least ceil(9e6 / (blocks * b)) tokens.  Rows
// of the V3 shape move 53-90 KB a token: one per claim on 152 SMs (fused V3
// FP8 dispatch 89.0 -> 86.6 us against two, four slower still); on 24 SMs
// the rank-major fused dispatch takes six (312 -> 260 us against one), 64
// SMs two (130 -> 116 us), while the same rule made the low-latency kernel
// 1 % slower on 24 SMs and the cached-layout BF16 dispatch 15 % slower on 64
// (rate-only for them); 512-channel rows move ~5 KB: ten per claim (one per
// claim caps 81 920 tokens at ~330 us, the counter's rate).
long long row_bytes_per_token(int H, int k, int kmax, bool fp8, int mode);
inline int claim_tokens_for(long long bytes_per_token, int blocks) {
  if (bytes_per_token <= 0) return 1;
  long long c = (48000 + bytes_per_token - 1) / bytes_per_token;
  if (blocks > 0) {
    const long long per = static_cast<long long>(blocks) * bytes_per_token;
    const long long by_latency = (9000000 + per - 1) / per;
    if (by_latency > c) c = by_latency;
  }
  return c < 1 ? 1 : (c > 64 ? 64 : static_cast<int>(c));
}
// Rows a fused-kernel producer streams in, in the rank-major mode, before its
// own block's prefixes are final: more would queue ahead of the routing's
// dependent loads.
constexpr int kRouteStages = 2;

// TMA bulk-copy scatter (dispatch row movement), persistent: one block per
// SM, one producer warp and up to kScatterMaxConsumers consumer warps.
constexpr int kScatterMaxConsumers = 8;
struct ScatterArgs {
  const uint16_t* x;           // [T][H] bf16
  int T, H, k, kmax, El, R, E;
  // normal destinations
  const int2* dst;             // [T][kmax]
  const int* rank_offset;      // [R+1]
  long long cap;
  const int* idx32;            // [T][k]
  const float* topk_weights;   // [T][k] or null
  int* recv_src_idx;
  int* recv_topk_idx;
  float* recv_topk_weights;
  // low-latency destinations
  const int* ll_idx;           // [T][k]
  const int* ll_slot;          // [T][k]
  int M;
  int* recv_src_info;
  // expert-major destinations (ll_idx / ll_slot above are the entries'
  // expert and slot in the expert; recv_src_idx is the row's source token)
  const int* expert_offset;    // [E+1]
  const int* expert_count;     // [E]
  float* recv_weights;         // [cap] or null
  long long scales_ld;         // scales stored [G][scales_ld]
  // outputs
  void* recv_x;
  float* recv_scales;
  unsigned* ctl;               // control words (row claims)
  int claim_tokens;            // tokens per claim (claim_tokens_for)
  int* err;
};
// NS row stages and NC consumer warps that fit `smem_limit` (NS = 0: the
// rows are too long for the bulk-copy staging).
void scatter_config(int H, int R, int E, bool fp8, int mode, size_t smem_limit, int* NS, int* NC);
size_t scatter_smem_bytes(int H, int R, int E, bool fp8, int mode, int NS, int NC);
cudaError_t configure_scatter(size_t optin);
void launch_scatter(const ScatterArgs& a, bool fp8, int mode, int blocks, int NS, int NC, cudaStream_t stream);

// Fused routing + dispatch (cooperative launch, one block per SM).
constexpr int kFusedMaxItems = 4096;  // (token, k) entries a block may own
// Per-entry fused routing counts every entry in every block (no grid
// barrier) when the batch has at most this many (token, k) entries.
constexpr long long kFusedRedundantEntries = 16384;

struct FusedArgs {
  const void* topk_idx;        // [T][k] int64, or int32 if ids32
  int ids32;
  int redundant;               // small batch: every block counts every entry, no grid barrier
  int own_first;               // own tokens a block streams before claiming others' (>= tokens per block: no claims)
  int claim_tokens;            // tokens per claim (claim_tokens_for)
  const uint16_t* x;
  const float* topk_weights;
  int T, R, E, El, k, kp_log2, kmax, H, M;
  uint16_t* agg;      // per-block counts [blocks][R+E] (normal) or [blocks][E], rows padded to 8
  unsigned* barrier;  // [4 + blocks] control words: grid barrier, row claims, published flags
  int* err;
  // normal mode: the handle's layout state and the dispatch outputs
  int2* dst;
  int* idx32;
  int* recv_per_rank;
  int* rank_offset;
  int* recv_per_expert;
  long long cap;
  int* recv_src_idx;
  int* recv_topk_idx;
  float* recv_topk_weights;
  // low-latency and expert-major modes: per entry expert id and slot in
  // the expert (the handle's state); per expert rows filled
  int* ll_idx;
  int* ll_slot;
  int* recv_count;
  int* recv_src_info;
  // expert-major mode: group alignment, the handle's group offsets [E+1],
  // per-row top-k weight, scales stored [G][scales_ld] (recv_src_idx above
  // is the per-row source token)
  int align;
  int* expert_offset;
  float* recv_weights;
  long long scales_ld;
  // rows
  void* recv_x;
  float* recv_scales;
};
void fused_config(int mode, bool fp8, int T, int R, int E, int k, int kmax, int H, int sms, size_t smem_limit,
                  int* blocks, int* NS, int* NC, int* own_first);
cudaError_t configure_fused(size_t optin);
cudaError_t launch_fused(const FusedArgs& a, bool fp8, int mode, int blocks, int NS, int NC, cudaStream_t stream);

// Low-latency routing only (slots, counts); the rows move with k_scatter.
void launch_ll_route(const RouteParams& p, const LowLatencyOutPtrs& o, size_t smem, cudaStream_t stream);
cudaError_t configure_ll_route(size_t needed, size_t optin);
// Expert-major group offsets [E+1] from per-expert counts (one block).
void launch_em_offsets(const int* count, int E, int align, int* offset, cudaStream_t stream);

// Fused low-latency dispatch: routing phase + per-chunk scatter.
struct LowLatencyOut {
  const uint16_t* x;
  void* recv_x;                // [E][M][H]
  float* recv_scales;          // [E][M][H/128]
  int* recv_src_info;          // [E][M] or null
  int* recv_count;             // [E] or null
  int* ll_idx;                 // [T][k]
  int* ll_slot;                // [T][k]
  int H, M;
};
void launch_ll_dispatch(const RouteParams& p, const LowLatencyOut& o, bool fp8, size_t smem,
                        cudaStream_t stream);
cudaError_t configure_ll_dispatch(size_t needed, size_t optin);

}  // namespace ep
