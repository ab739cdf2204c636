// The C ABI declared in include/ep.h: handle lifecycle, argument checks,
// launch configuration and the device status latch.  Every step of the
// computation runs in this library's kernels; there is no host fallback.
#include <climits>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "ep.h"
#include "ep_internal.h"
#include "routing.cuh"

struct ep_handle {
  int R, E, k, H, max_tpr, El, kmax, kp_log2;
  int Tmax;
  int ids32;  // top-k ids are int32 (else int64)
  int device, num_sms;
  // routing configuration
  int layout_CT, ll_CT;
  size_t layout_smem, ll_smem, layout_tokens_smem;
  int layout_cmax, ll_cmax;
  // occupancy (blocks per SM) of the persistent kernels
  int occ_dispatch[2], occ_combine[4];  // combine: rank-major bf16, rank-major e4m3, low latency, expert-major
  // TMA scatter: row stages and consumer warps per block for
  // [fp8][rank-major, low latency, expert-major]; 0 stages = rows too long,
  // the register-resident kernels are used instead (none for expert-major)
  int scatter_ns[2][3], scatter_nc[2][3];
  size_t ll_route_smem;
  // state
  int T_layout;  // tokens of the last layout, -1 before the first
  int T_ll;      // tokens of the last low-latency dispatch, -1 before the first
  int T_em;      // tokens of the last expert-major layout, -1 before the first
  bool debug;
  // device arena
  void* arena;
  int2* dst;
  int* idx32;
  int* rank_offset;
  int* recv_per_rank;
  int* recv_per_expert;
  int* ll_idx;
  int* ll_slot;
  unsigned long long* layout_flags;
  unsigned long long* ll_flags;
  unsigned long long* em_flags;
  unsigned long long* tickets;  // [0] layout, [1] low latency, [2] expert-major: (epoch << 32) | next chunk id
  // expert-major layout: per entry expert id and slot inside the expert,
  // per expert count and group offset
  int* em_idx;
  int* em_slot;
  int* em_count;
  int* em_offset;
  uint16_t* fused_agg;          // [num_sms][R+E padded to 8] per-block counts of the fused kernel
  unsigned* fused_barrier;      // [4 + num_sms] its control words (barrier, row claims, published flags)
  size_t smem_optin;
  int* err;
  // pinned host mirror: err, then R + E + R+1 counts
  int* host;
};

namespace ep {

// A flag word that no code writes: the self-check's flag wait never sees its
// epoch and gives up.
__device__ unsigned long long g_never_set_flag;

// One thread waits on the flag above, then on a fresh mbarrier that nobody
// arrives at; both waits are the bounded ones of the real kernels.
__global__ void k_wait_timeout_check(int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  (void)flag_wait(&g_never_set_flag, 1u, 1u, err);
  mbar_init(&bar, 1);
  mbar_init_fence();
  (void)mbar_wait(&bar, 0u, err);
}

void launch_wait_timeout_check(int* err, cudaStream_t stream) { k_wait_timeout_check<<<1, 32, 0, stream>>>(err); }

}  // namespace ep

namespace {

using ep::RouteParams;

ep_status_t cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return EP_OK;
  if (std::getenv("EP_DEBUG")) std::fprintf(stderr, "[ep] %s: %s\n", what, cudaGetErrorString(e));
  return EP_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int ceil_div(int a, int b) { return (a + b - 1) / b; }

bool ids_aligned(const ep_handle* h, const void* topk_idx) {
  return !topk_idx || (h->ids32 ? aligned4(topk_idx) : aligned8(topk_idx));
}

// EP_NUM_TOPK_IDX_BITS: 64 (default) or 32; anything else is an error (-1).
int ids32_from_env() {
  const char* v = std::getenv("EP_NUM_TOPK_IDX_BITS");
  if (!v || !*v) return 0;
  if (std::strcmp(v, "64") == 0) return 0;
  if (std::strcmp(v, "32") == 0) return 1;
  return -1;
}

ep_status_t check_device(const ep_handle* h) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess) return EP_ERR_CUDA;
  return d == h->device ? EP_OK : EP_ERR_INVALID_ARG;
}

int grid_for(const ep_handle* h, int occ, int num_sms, int T, int warps_per_block) {
  int sms = num_sms <= 0 ? h->num_sms : (num_sms < h->num_sms ? num_sms : h->num_sms);
  int blocks = sms * (occ > 0 ? occ : 1);
  int need = ceil_div(T, warps_per_block);
  if (need < blocks) blocks = need;
  return blocks > 0 ? blocks : 1;
}

RouteParams route_params(ep_handle* h, const void* topk_idx, int T, int CT,
                         unsigned long long* flags, unsigned long long* ticket) {
  RouteParams p;
  p.topk_idx = topk_idx;
  p.ids32 = h->ids32;
  p.T = T;
  p.R = h->R;
  p.E = h->E;
  p.El = h->El;
  p.k = h->k;
  p.kp_log2 = h->kp_log2;
  p.kmax = h->kmax;
  p.tpr = T / h->R;
  p.CT = CT;
  p.cps = ceil_div(p.tpr, CT);
  p.C = h->R * p.cps;
  p.flags = flags;
  p.ticket = ticket;
  p.err = h->err;
  return p;
}

// Rank-major batches of at most this many (token, k) entries count every
// token in every block instead of meeting at the fused kernel's grid barrier.
constexpr long long kFusedRedundantRankEntries = 4096;

int sms_for(const ep_handle* h, int num_sms) {
  return num_sms <= 0 ? h->num_sms : (num_sms < h->num_sms ? num_sms : h->num_sms);
}

ep::FusedArgs fused_args(ep_handle* h, const void* topk_idx, const uint16_t* x, const float* w, int T) {
  ep::FusedArgs f{};
  f.topk_idx = topk_idx;
  f.ids32 = h->ids32;
  f.redundant = static_cast<long long>(T) * h->k <= ep::kFusedRedundantEntries ? 1 : 0;  // rank-major: reset by the caller
  f.x = x;
  f.topk_weights = w;
  f.T = T;
  f.R = h->R;
  f.E = h->E;
  f.El = h->El;
  f.k = h->k;
  f.kp_log2 = h->kp_log2;
  f.kmax = h->kmax;
  f.H = h->H;
  f.barrier = h->fused_barrier;
  f.err = h->err;
  return f;
}

}  // namespace

extern "C" {

const char* ep_status_str(ep_status_t s) {
  switch (s) {
    case EP_OK: return "EP_OK";
    case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
    case EP_ERR_CUDA: return "EP_ERR_CUDA";
    case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY";
    case EP_ERR_BAD_EXPERT: return "EP_ERR_BAD_EXPERT";
    case EP_ERR_TIMEOUT: return "EP_ERR_TIMEOUT";
    case EP_ERR_STATE: return "EP_ERR_STATE";
  }
  return "EP_ERR_UNKNOWN";
}

ep_status_t ep_handle_create(int R, int E, int k, int H, int max_tpr, ep_handle_t* out) {
  if (!out) return EP_ERR_INVALID_ARG;
  *out = nullptr;
  if (R < 1 || R > 1024 || E < 1 || E > 4096 || E % R != 0 || k < 1 || k > 32 || H < 128 ||
      H % 128 != 0 || max_tpr < 1)
    return EP_ERR_INVALID_ARG;
  if (static_cast<long long>(R) * max_tpr > (1LL << 30)) return EP_ERR_INVALID_ARG;

  ep_handle* h = new (std::nothrow) ep_handle();
  if (!h) return EP_ERR_CUDA;
  h->R = R;
  h->E = E;
  h->k = k;
  h->H = H;
  h->max_tpr = max_tpr;
  h->El = E / R;
  h->kmax = k < R ? k : R;
  int kp = 1, lg = 0;
  while (kp < k) kp <<= 1, ++lg;
  h->kp_log2 = lg;
  h->Tmax = R * max_tpr;
  h->ids32 = ids32_from_env();
  if (h->ids32 < 0) {
    delete h;
    return EP_ERR_INVALID_ARG;
  }
  h->T_layout = -1;
  h->T_ll = -1;
  h->T_em = -1;
  h->debug = std::getenv("EP_DEBUG") != nullptr;

  ep_status_t st = EP_OK;
  cudaDeviceProp prop;
  if ((st = cuda_status(cudaGetDevice(&h->device), "cudaGetDevice")) != EP_OK ||
      (st = cuda_status(cudaGetDeviceProperties(&prop, h->device), "cudaGetDeviceProperties")) != EP_OK) {
    delete h;
    return st;
  }
  h->num_sms = prop.multiProcessorCount;

  // routing chunks: 2048 (token, k) items per layout block (1024 when the
  // per-block tables would not fit), 8 tokens per fused low-latency block
  const int NKl = R + E, NKll = E;
  int items = ep::kRouteMaxItems;
  while (items > 1024 &&
         ep::route_smem_bytes(NKl, items, items >> lg, h->kmax) > static_cast<size_t>(prop.sharedMemPerBlockOptin))
    items >>= 1;
  h->layout_CT = items >> lg;
  h->ll_CT = 8;
  h->layout_smem = ep::route_smem_bytes(NKl, h->layout_CT << lg, h->layout_CT, h->kmax);
  h->ll_smem = ep::route_smem_bytes(NKll, h->ll_CT << lg, h->ll_CT, h->kmax);
  if (h->layout_smem > static_cast<size_t>(prop.sharedMemPerBlockOptin) ||
      h->ll_smem + 1024 > static_cast<size_t>(prop.sharedMemPerBlockOptin)) {
    delete h;
    return EP_ERR_INVALID_ARG;
  }
  h->layout_cmax = R * ceil_div(max_tpr, h->layout_CT < ep::kLayoutTokenChunk ? h->layout_CT : ep::kLayoutTokenChunk);
  h->layout_tokens_smem = ep::layout_tokens_smem(R, E, ep::kLayoutTokenChunk, h->kmax);
  h->ll_cmax = R * ceil_div(max_tpr, h->ll_CT);

  // one device arena for all metadata
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off += (bytes + 255) & ~static_cast<size_t>(255);
    return at;
  };
  const size_t o_dst = take(sizeof(int2) * static_cast<size_t>(h->Tmax) * h->kmax);
  const size_t o_idx = take(sizeof(int) * static_cast<size_t>(h->Tmax) * k);
  const size_t o_off = take(sizeof(int) * (R + 1));
  const size_t o_rpr = take(sizeof(int) * R);
  const size_t o_rpe = take(sizeof(int) * E);
  const size_t o_llidx = take(sizeof(int) * static_cast<size_t>(h->Tmax) * k);
  const size_t o_llslot = take(sizeof(int) * static_cast<size_t>(h->Tmax) * k);
  const size_t o_lf = take(sizeof(unsigned long long) * static_cast<size_t>(h->layout_cmax) * NKl);
  const size_t o_llf = take(sizeof(unsigned long long) * static_cast<size_t>(h->ll_cmax) * NKll);
  const size_t o_emf = take(sizeof(unsigned long long) * static_cast<size_t>(h->ll_cmax) * NKll);
  const size_t o_tk = take(sizeof(unsigned long long) * 3);
  const size_t o_emidx = take(sizeof(int) * static_cast<size_t>(h->Tmax) * k);
  const size_t o_emslot = take(sizeof(int) * static_cast<size_t>(h->Tmax) * k);
  const size_t o_emcnt = take(sizeof(int) * E);
  const size_t o_emoff = take(sizeof(int) * (E + 1));
  const size_t o_fagg = take(sizeof(uint16_t) * static_cast<size_t>(h->num_sms) * ((R + E + 7) & ~7));
  const size_t o_fbar = take(sizeof(unsigned) * (4 + static_cast<size_t>(h->num_sms)));
  const size_t o_err = take(sizeof(int));
  if ((st = cuda_status(cudaMalloc(&h->arena, off), "cudaMalloc")) != EP_OK) {
    delete h;
    return st;
  }
  char* base = static_cast<char*>(h->arena);
  h->dst = reinterpret_cast<int2*>(base + o_dst);
  h->idx32 = reinterpret_cast<int*>(base + o_idx);
  h->rank_offset = reinterpret_cast<int*>(base + o_off);
  h->recv_per_rank = reinterpret_cast<int*>(base + o_rpr);
  h->recv_per_expert = reinterpret_cast<int*>(base + o_rpe);
  h->ll_idx = reinterpret_cast<int*>(base + o_llidx);
  h->ll_slot = reinterpret_cast<int*>(base + o_llslot);
  h->layout_flags = reinterpret_cast<unsigned long long*>(base + o_lf);
  h->ll_flags = reinterpret_cast<unsigned long long*>(base + o_llf);
  h->em_flags = reinterpret_cast<unsigned long long*>(base + o_emf);
  h->tickets = reinterpret_cast<unsigned long long*>(base + o_tk);
  h->em_idx = reinterpret_cast<int*>(base + o_emidx);
  h->em_slot = reinterpret_cast<int*>(base + o_emslot);
  h->em_count = reinterpret_cast<int*>(base + o_emcnt);
  h->em_offset = reinterpret_cast<int*>(base + o_emoff);
  h->fused_agg = reinterpret_cast<uint16_t*>(base + o_fagg);
  h->fused_barrier = reinterpret_cast<unsigned*>(base + o_fbar);
  h->err = reinterpret_cast<int*>(base + o_err);
  // zero everything once (latch, look-back words); tickets start at epoch 1,
  // so no look-back word ever matches before it is written
  const unsigned long long first_ticket[3] = {1ull << 32, 1ull << 32, 1ull << 32};
  if ((st = cuda_status(cudaMemset(h->arena, 0, off), "cudaMemset")) != EP_OK ||
      (st = cuda_status(cudaMemcpy(h->tickets, first_ticket, sizeof(first_ticket), cudaMemcpyHostToDevice),
                        "cudaMemcpy")) != EP_OK ||
      (st = cuda_status(cudaMallocHost(&h->host, sizeof(int) * (2 + 2 * R + 2 * E + 2)), "cudaMallocHost")) != EP_OK) {
    cudaFree(h->arena);
    delete h;
    return st;
  }
  // low-latency routing runs on layout-sized chunks (its look-back words fit
  // in the space sized for the fused kernel's smaller chunks)
  h->ll_route_smem = ep::route_smem_bytes(NKll, h->layout_CT << lg, h->layout_CT, h->kmax);
  const size_t optin = static_cast<size_t>(prop.sharedMemPerBlockOptin);
  h->smem_optin = optin;
  for (int f = 0; f < 2; ++f)
    for (int m = 0; m < 3; ++m) ep::scatter_config(H, R, E, f == 1, m, optin, &h->scatter_ns[f][m], &h->scatter_nc[f][m]);
  // every kernel's dynamic shared-memory limit is set from the device's
  // opt-in maximum, the same value for every handle (a per-handle size would
  // let a later, smaller handle lower it under an earlier, larger one); a
  // handle whose sizes do not fit under it is refused
  if ((st = cuda_status(ep::configure_layout(h->layout_smem, optin), "configure_layout")) != EP_OK ||
      (st = cuda_status(ep::configure_ll_dispatch(h->ll_smem, optin), "configure_ll_dispatch")) != EP_OK ||
      (st = cuda_status(ep::configure_ll_route(h->ll_route_smem, optin), "configure_ll_route")) != EP_OK ||
      (st = cuda_status(ep::configure_layout_tokens(R <= 64 ? h->layout_tokens_smem : 0, optin),
                        "configure_layout_tokens")) != EP_OK ||
      (st = cuda_status(ep::configure_scatter(optin), "configure_scatter")) != EP_OK ||
      (st = cuda_status(ep::configure_fused(optin), "configure_fused")) != EP_OK) {
    ep_handle_destroy(h);
    return st;
  }
  for (int m = 0; m < 2; ++m) {
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, ep::dispatch_kernel(m == 1), ep::dispatch_threads(), 0);
    h->occ_dispatch[m] = occ > 0 ? occ : 1;
  }
  for (int m = 0; m < 4; ++m) {
    const int src = m < 2 ? ep::kSrcRanks : m == 2 ? ep::kSrcLowLatency : ep::kSrcExpertMajor;
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, ep::combine_kernel(src, m == 1), ep::combine_threads(),
                                                  ep::combine_smem_bytes(src, R, E));
    h->occ_combine[m] = occ > 0 ? occ : 1;
  }
  if (h->debug)
    std::fprintf(stderr,
                 "[ep] handle R=%d E=%d k=%d H=%d max_tokens_per_rank=%d on device %d (%d SMs); "
                 "layout chunk %d tokens (%zu B smem), ll chunk %d tokens (%zu B smem); "
                 "blocks/SM dispatch bf16 %d fp8 %d, combine %d ll-combine %d; scatter stages/consumers bf16 %d/%d "
                 "fp8 %d/%d; arena %zu B\n",
                 R, E, k, H, max_tpr, h->device, h->num_sms, h->layout_CT, h->layout_smem, h->ll_CT,
                 h->ll_smem, h->occ_dispatch[0], h->occ_dispatch[1], h->occ_combine[0], h->occ_combine[1],
                 h->scatter_ns[0][0], h->scatter_nc[0][0], h->scatter_ns[1][0], h->scatter_nc[1][0], off);
  *out = h;
  return EP_OK;
}

ep_status_t ep_handle_destroy(ep_handle_t h) {
  if (!h) return EP_OK;
  if (h->arena) cudaFree(h->arena);
  if (h->host) cudaFreeHost(h->host);
  delete h;
  return EP_OK;
}

ep_status_t ep_get_dispatch_layout(ep_handle_t h, const void* topk_idx, int T, int* num_tokens_per_rank,
                                   int* num_tokens_per_expert, uint8_t* is_token_in_rank, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  if (T < 0 || T % h->R != 0 || T > h->Tmax || (T > 0 && !topk_idx)) return EP_ERR_INVALID_ARG;
  if (!ids_aligned(h, topk_idx) || (num_tokens_per_rank && !aligned4(num_tokens_per_rank)) ||
      (num_tokens_per_expert && !aligned4(num_tokens_per_expert)))
    return EP_ERR_INVALID_ARG;
  ep_status_t st = check_device(h);
  if (st != EP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    // nothing to route: every count is zero
    cudaError_t e = cudaMemsetAsync(h->rank_offset, 0, sizeof(int) * (h->R + 1), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->recv_per_rank, 0, sizeof(int) * h->R, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->recv_per_expert, 0, sizeof(int) * h->E, s);
    if (e == cudaSuccess && num_tokens_per_rank)
      e = cudaMemsetAsync(num_tokens_per_rank, 0, sizeof(int) * h->R * h->R, s);
    if (e == cudaSuccess && num_tokens_per_expert)
      e = cudaMemsetAsync(num_tokens_per_expert, 0, sizeof(int) * static_cast<size_t>(h->R) * h->E, s);
    if ((st = cuda_status(e, "layout memset")) != EP_OK) return st;
    h->T_layout = 0;
    return EP_OK;
  }
  ep::LayoutOutPtrs o{h->dst, h->idx32, h->recv_per_rank, h->rank_offset, h->recv_per_expert,
                      num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank};
  // R <= 64: one lane per token (rank masks); otherwise one lane per (token, k) entry
  const bool by_token = h->R <= 64;
  RouteParams p = route_params(h, topk_idx, T, by_token ? ep::kLayoutTokenChunk : h->layout_CT, h->layout_flags,
                               h->tickets + 0);
  if (by_token)
    ep::launch_layout_tokens(p, o, s);
  else
    ep::launch_layout(p, o, h->layout_smem, s);
  if ((st = cuda_status(cudaGetLastError(), "k_layout launch")) != EP_OK) return st;
  if (h->debug) std::fprintf(stderr, "[ep] layout T=%d: %d blocks x %d threads\n", T, p.C, ep::kRouteThreads);
  h->T_layout = T;
  return EP_OK;
}

ep_status_t ep_get_num_recv(ep_handle_t h, int* num_recv_tokens_per_rank, int* num_recv_tokens_per_expert,
                            int* rank_offset, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  if (h->T_layout < 0) return EP_ERR_STATE;
  ep_status_t st = check_device(h);
  if (st != EP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* hp = h->host;
  cudaError_t e = cudaMemcpyAsync(hp, h->err, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(hp + 1, h->recv_per_rank, sizeof(int) * h->R, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(hp + 1 + h->R, h->recv_per_expert, sizeof(int) * h->E, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(hp + 1 + h->R + h->E, h->rank_offset, sizeof(int) * (h->R + 1), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if ((st = cuda_status(e, "ep_get_num_recv")) != EP_OK) return st;
  if (num_recv_tokens_per_rank) std::memcpy(num_recv_tokens_per_rank, hp + 1, sizeof(int) * h->R);
  if (num_recv_tokens_per_expert) std::memcpy(num_recv_tokens_per_expert, hp + 1 + h->R, sizeof(int) * h->E);
  if (rank_offset) std::memcpy(rank_offset, hp + 1 + h->R + h->E, sizeof(int) * (h->R + 1));
  return static_cast<ep_status_t>(hp[0]);
}

ep_status_t ep_dispatch(ep_handle_t h, const void* x, const float* topk_weights, ep_dtype_t dtype, void* recv_x,
                        float* recv_scales, int64_t cap, int* recv_src_idx, int* recv_topk_idx,
                        float* recv_topk_weights, int num_sms, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  if (h->T_layout < 0) return EP_ERR_STATE;
  if (dtype != EP_BF16 && dtype != EP_FP8_E4M3) return EP_ERR_INVALID_ARG;
  const bool fp8 = dtype == EP_FP8_E4M3;
  const int T = h->T_layout;
  if (cap < 0 || (cap > 0 && !recv_x) || (fp8 && cap > 0 && !recv_scales) || (T > 0 && !x))
    return EP_ERR_INVALID_ARG;
  if (recv_topk_weights && !topk_weights) return EP_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (recv_x && !aligned16(recv_x)) || (fp8 && recv_scales && !aligned4(recv_scales)) ||
      (topk_weights && !aligned4(topk_weights)) || (recv_src_idx && !aligned4(recv_src_idx)) ||
      (recv_topk_idx && !aligned4(recv_topk_idx)) || (recv_topk_weights && !aligned4(recv_topk_weights)))
    return EP_ERR_INVALID_ARG;
  ep_status_t st = check_device(h);
  if (st != EP_OK) return st;
  if (T == 0) return EP_OK;
  const int sns = h->scatter_ns[fp8 ? 1 : 0][ep::kSrcRanks], snc = h->scatter_nc[fp8 ? 1 : 0][ep::kSrcRanks];
  if (sns > 0) {
    ep::ScatterArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.T = T;
    a.H = h->H;
    a.k = h->k;
    a.kmax = h->kmax;
    a.El = h->El;
    a.R = h->R;
    a.E = h->E;
    a.dst = h->dst;
    a.rank_offset = h->rank_offset;
    a.cap = cap;
    a.idx32 = h->idx32;
    a.topk_weights = topk_weights;
    a.recv_src_idx = recv_src_idx;
    a.recv_topk_idx = recv_topk_idx;
    a.recv_topk_weights = recv_topk_weights;
    a.recv_x = recv_x;
    a.recv_scales = recv_scales;
    a.ctl = h->fused_barrier;
    a.err = h->err;
    const int blocks = grid_for(h, 1, num_sms, T, 1);
    ep::launch_scatter(a, fp8, ep::kSrcRanks, blocks, sns, snc, reinterpret_cast<cudaStream_t>(stream));
    if (h->debug)
      std::fprintf(stderr, "[ep] dispatch %s T=%d: TMA scatter %d blocks, %d stages, %d consumers\n",
                   fp8 ? "fp8" : "bf16", T, blocks, sns, snc);
    return cuda_status(cudaGetLastError(), "k_scatter launch");
  }
  ep::DispatchArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.topk_weights = topk_weights;
  a.dst = h->dst;
  a.idx32 = h->idx32;
  a.rank_offset = h->rank_offset;
  a.recv_x = recv_x;
  a.recv_scales = recv_scales;
  a.recv_src_idx = recv_src_idx;
  a.recv_topk_idx = recv_topk_idx;
  a.recv_topk_weights = recv_topk_weights;
  a.cap = cap;
  a.T = T;
  a.H = h->H;
  a.k = h->k;
  a.kmax = h->kmax;
  a.El = h->El;
  a.err = h->err;
  const int blocks = grid_for(h, h->occ_dispatch[fp8 ? 1 : 0], num_sms, T, ep::dispatch_threads() / 32);
  ep::launch_dispatch(a, fp8, blocks, reinterpret_cast<cudaStream_t>(stream));
  if (h->debug) std::fprintf(stderr, "[ep] dispatch %s T=%d: %d blocks\n", fp8 ? "fp8" : "bf16", T, blocks);
  return cuda_status(cudaGetLastError(), "k_dispatch launch");
}

ep_status_t ep_layout_and_dispatch(ep_handle_t h, const void* topk_idx, int T, const void* x,
                                   const float* topk_weights, ep_dtype_t dtype, void* recv_x, float* recv_scales,
                                   int64_t cap, int* recv_src_idx, int* recv_topk_idx, float* recv_topk_weights,
                                   int num_sms, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  if (dtype != EP_BF16 && dtype != EP_FP8_E4M3) return EP_ERR_INVALID_ARG;
  const bool fp8 = dtype == EP_FP8_E4M3;
  if (T < 0 || T % h->R != 0 || T > h->Tmax || (T > 0 && (!topk_idx || !x)) || cap < 0 ||
      (cap > 0 && !recv_x) || (fp8 && cap > 0 && !recv_scales))
    return EP_ERR_INVALID_ARG;
  if (recv_topk_weights && !topk_weights) return EP_ERR_INVALID_ARG;
  if (!ids_aligned(h, topk_idx) || (x && !aligned16(x)) || (recv_x && !aligned16(recv_x)) ||
      (fp8 && recv_scales && !aligned4(recv_scales)) || (topk_weights && !aligned4(topk_weights)) ||
      (recv_src_idx && !aligned4(recv_src_idx)) || (recv_topk_idx && !aligned4(recv_topk_idx)) ||
      (recv_topk_weights && !aligned4(recv_topk_weights)))
    return EP_ERR_INVALID_ARG;
  ep_status_t st = check_device(h);
  if (st != EP_OK) return st;
  int fblocks = 0, fns = 0, fnc = 0, fown = 0;
  if (static_cast<long long>(T) * h->kmax < (1LL << 31))
    ep::fused_config(ep::kSrcRanks, fp8, T, h->R, h->E, h->k, h->kmax, h->H, sms_for(h, num_sms), h->smem_optin,
                     &fblocks, &fns, &fnc, &fown);
  if (fblocks == 0) {
    // the general path: layout kernel, then the scatter
    if ((st = ep_get_dispatch_layout(h, topk_idx, T, nullptr, nullptr, nullptr, stream)) != EP_OK) return st;
    return ep_dispatch(h, x, topk_weights, dtype, recv_x, recv_scales, cap, recv_src_idx, recv_topk_idx,
                       recv_topk_weights, num_sms, stream);
  }
  ep::FusedArgs f = fused_args(h, topk_idx, static_cast<const uint16_t*>(x), topk_weights, T);
  f.redundant = static_cast<long long>(T) * h->k <= kFusedRedundantRankEntries ? 1 : 0;
  f.own_first = fown;
  f.agg = h->fused_agg;
  f.dst = h->dst;
  f.idx32 = h->idx32;
  f.recv_per_rank = h->recv_per_rank;
  f.rank_offset = h->rank_offset;
  f.recv_per_expert = h->recv_per_expert;
  f.cap = cap;
  f.recv_src_idx = recv_src_idx;
  f.recv_topk_idx = recv_topk_idx;
  f.recv_topk_weights = recv_topk_weights;
  f.recv_x = recv_x;
  f.recv_scales = recv_scales;
  if ((st = cuda_status(ep::launch_fused(f, fp8, ep::kSrcRanks, fblocks, fns, fnc, reinterpret_cast<cudaStream_t>(stream)),
                        "k_route_scatter launch")) != EP_OK)
    return st;
  if (h->debug)
    std::fprintf(stderr, "[ep] layout+dispatch %s T=%d: fused, %d blocks, %d stages, %d consumers\n",
                 fp8 ? "fp8" : "bf16", T, fblocks, fns, fnc);
  h->T_layout = T;
  return EP_OK;
}

ep_status_t ep_combine_ex(ep_handle_t h, ep_dtype_t y_dtype, const void* y, const float* y_scales, int64_t y_rows,
                          const float* recv_topk_weights, void* out, float* combined_topk_weights, int num_sms,
                          ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  if (h->T_layout < 0) return EP_ERR_STATE;
  if (y_dtype != EP_BF16 && y_dtype != EP_FP8_E4M3) return EP_ERR_INVALID_ARG;
  const bool fp8 = y_dtype == EP_FP8_E4M3;
  const int T = h->T_layout;
  if (y_rows < 0 || (T > 0 && (!out || (y_rows > 0 && (!y || (fp8 && !y_scales)))))) return EP_ERR_INVALID_ARG;
  if ((recv_topk_weights != nullptr) != (combined_topk_weights != nullptr)) return EP_ERR_INVALID_ARG;
  if ((y && !aligned16(y)) || (out && !aligned16(out)) || (fp8 && y_scales && !aligned4(y_scales)) ||
      (recv_topk_weights && !aligned4(recv_topk_weights)) || (combined_topk_weights && !aligned4(combined_topk_weights)))
    return EP_ERR_INVALID_ARG;
  ep_status_t st = check_device(h);
  if (st != EP_OK) return st;
  if (T == 0) return EP_OK;
  ep::CombineArgs a{};
  a.y = y;
  a.y_scales = fp8 ? y_scales : nullptr;
  a.out = static_cast<uint16_t*>(out);
  a.y_rows = y_rows;
  a.T = T;
  a.H = h->H;
  a.k = h->k;
  a.kmax = h->kmax;
  a.R = h->R;
  a.E = h->E;
  a.dst = h->dst;
  a.rank_offset = h->rank_offset;
  a.recv_topk_weights = recv_topk_weights;
  a.combined_topk_weights = combined_topk_weights;
  a.err = h->err;
  const int blocks =
      grid_for(h, h->occ_combine[fp8 ? 1 : 0], num_sms, T * ((h->H + 1023) / 1024), ep::combine_threads() / 32);
  ep::launch_combine(a, ep::kSrcRanks, fp8, blocks, reinterpret_cast<cudaStream_t>(stream));
  if (h->debug) std::fprintf(stderr, "[ep] combine %s T=%d: %d blocks\n", fp8 ? "e4m3" : "bf16", T, blocks);
  return cuda_status(cudaGetLastError(), "k_combine launch");
}

ep_status_t ep_combine(ep_handle_t h, const void* y, int64_t y_rows, void* out, int num_sms, ep_stream_t stream) {
  return ep_combine_ex(h, EP_BF16, y, nullptr, y_rows, nullptr, out, nullptr, num_sms, stream);
}

ep_status_t ep_low_latency_dispatch(ep_handle_t h, const void* x, const void* topk_idx, int T, ep_dtype_t dtype,
                                    void* recv_x, float* recv_scales, int* recv_src_info, int* recv_count,
                                    int num_sms, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  if (dtype != EP_BF16 && dtype != EP_FP8_E4M3) return EP_ERR_INVALID_ARG;
  const bool fp8 = dtype == EP_FP8_E4M3;
  if (T < 0 || T % h->R != 0 || T > h->Tmax) return EP_ERR_INVALID_ARG;
  if (T > 0 && (!x || !topk_idx || !recv_x || (fp8 && !recv_scales))) return EP_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || !ids_aligned(h, topk_idx) || (recv_x && !aligned16(recv_x)) ||
      (fp8 && recv_scales && !aligned4(recv_scales)) || (recv_src_info && !aligned4(recv_src_info)) ||
      (recv_count && !aligned4(recv_count)))
    return EP_ERR_INVALID_ARG;
  ep_status_t st = check_device(h);
  if (st != EP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int M = h->Tmax;
  if (T == 0) {
    h->T_ll = 0;
    if (recv_count) return cuda_status(cudaMemsetAsync(recv_count, 0, sizeof(int) * h->E, s), "ll memset");
    return EP_OK;
  }
  int fblocks = 0, fns = 0, fnc = 0, own = 0;
  ep::fused_config(ep::kSrcLowLatency, fp8, T, h->R, h->E, h->k, h->kmax, h->H, sms_for(h, num_sms), h->smem_optin,
                   &fblocks, &fns, &fnc, &own);
  if (fblocks > 0) {
    // routing and row movement in one cooperative launch
    ep::FusedArgs f = fused_args(h, topk_idx, static_cast<const uint16_t*>(x), nullptr, T);
    f.M = M;
    f.own_first = own;
    f.agg = h->fused_agg;
    f.ll_idx = h->ll_idx;
    f.ll_slot = h->ll_slot;
    f.recv_count = recv_count;
    f.recv_src_info = recv_src_info;
    f.recv_x = recv_x;
    f.recv_scales = recv_scales;
    if ((st = cuda_status(ep::launch_fused(f, fp8, ep::kSrcLowLatency, fblocks, fns, fnc, s), "k_route_scatter(ll) launch")) !=
        EP_OK)
      return st;
    if (h->debug)
      std::fprintf(stderr, "[ep] ll dispatch T=%d: fused, %d blocks, %d stages, %d consumers, %d own tokens first\n", T,
                   fblocks, fns, fnc, own);
    h->T_ll = T;
    return EP_OK;
  }
  const int sns = h->scatter_ns[fp8 ? 1 : 0][ep::kSrcLowLatency], snc = h->scatter_nc[fp8 ? 1 : 0][ep::kSrcLowLatency];
  if (sns > 0) {
    // routing (slots, counts) on layout-sized chunks, then the TMA scatter
    RouteParams p = route_params(h, topk_idx, T, h->layout_CT, h->ll_flags, h->tickets + 1);
    ep::LowLatencyOutPtrs ro{recv_count, h->ll_idx, h->ll_slot, M};
    ep::launch_ll_route(p, ro, h->ll_route_smem, s);
    if ((st = cuda_status(cudaGetLastError(), "k_ll_route launch")) != EP_OK) return st;
    ep::ScatterArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.T = T;
    a.H = h->H;
    a.k = h->k;
    a.kmax = h->kmax;
    a.El = h->El;
    a.R = h->R;
    a.E = h->E;
    a.ll_idx = h->ll_idx;
    a.ll_slot = h->ll_slot;
    a.M = M;
    a.recv_src_info = recv_src_info;
    a.recv_x = recv_x;
    a.recv_scales = recv_scales;
    a.ctl = h->fused_barrier;
    a.err = h->err;
    const int blocks = grid_for(h, 1, num_sms, T, 1);
    ep::launch_scatter(a, fp8, ep::kSrcLowLatency, blocks, sns, snc, s);
    if ((st = cuda_status(cudaGetLastError(), "k_scatter(ll) launch")) != EP_OK) return st;
    if (h->debug)
      std::fprintf(stderr, "[ep] ll dispatch T=%d: route %d blocks, TMA scatter %d blocks, %d stages, %d consumers\n",
                   T, p.C, blocks, sns, snc);
    h->T_ll = T;
    return EP_OK;
  }
  RouteParams p = route_params(h, topk_idx, T, h->ll_CT, h->ll_flags, h->tickets + 1);
  ep::LowLatencyOut o;
  o.x = static_cast<const uint16_t*>(x);
  o.recv_x = recv_x;
  o.recv_scales = recv_scales;
  o.recv_src_info = recv_src_info;
  o.recv_count = recv_count;
  o.ll_idx = h->ll_idx;
  o.ll_slot = h->ll_slot;
  o.H = h->H;
  o.M = M;
  ep::launch_ll_dispatch(p, o, fp8, h->ll_smem, s);
  if ((st = cuda_status(cudaGetLastError(), "k_ll_dispatch launch")) != EP_OK) return st;
  if (h->debug) std::fprintf(stderr, "[ep] ll dispatch T=%d: %d blocks\n", T, p.C);
  h->T_ll = T;
  return EP_OK;
}

ep_status_t ep_low_latency_combine(ep_handle_t h, const void* y, const float* topk_weights, void* out, int num_sms,
                                   ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  if (h->T_ll < 0) return EP_ERR_STATE;
  const int T = h->T_ll;
  if (T > 0 && (!y || !topk_weights || !out)) return EP_ERR_INVALID_ARG;
  if ((y && !aligned16(y)) || (out && !aligned16(out)) || (topk_weights && !aligned4(topk_weights)))
    return EP_ERR_INVALID_ARG;
  ep_status_t st = check_device(h);
  if (st != EP_OK) return st;
  if (T == 0) return EP_OK;
  ep::CombineArgs a{};
  a.y = y;
  a.out = static_cast<uint16_t*>(out);
  a.y_rows = static_cast<long long>(h->E) * h->Tmax;
  a.T = T;
  a.H = h->H;
  a.k = h->k;
  a.kmax = h->kmax;
  a.ent_idx = h->ll_idx;
  a.ent_slot = h->ll_slot;
  a.topk_weights = topk_weights;
  a.M = h->Tmax;
  a.R = h->R;
  a.E = h->E;
  a.err = h->err;
  const int blocks = grid_for(h, h->occ_combine[2], num_sms, T * ((h->H + 1023) / 1024), ep::combine_threads() / 32);
  ep::launch_combine(a, ep::kSrcLowLatency, false, blocks, reinterpret_cast<cudaStream_t>(stream));
  if (h->debug) std::fprintf(stderr, "[ep] ll combine T=%d: %d blocks\n", T, blocks);
  return cuda_status(cudaGetLastError(), "k_combine(ll) launch");
}

// ---------------------------------------------------------------- expert-major

namespace {

ep_status_t em_check_outputs(const ep_handle* h, ep_dtype_t dtype, const float* topk_weights, void* recv_x,
                             float* recv_scales, int64_t scales_ld, int64_t cap, int* recv_src_idx,
                             float* recv_weights) {
  if (dtype != EP_BF16 && dtype != EP_FP8_E4M3) return EP_ERR_INVALID_ARG;
  const bool fp8 = dtype == EP_FP8_E4M3;
  if (cap < 0 || cap > (1LL << 31) - 1 || (cap > 0 && !recv_x)) return EP_ERR_INVALID_ARG;
  if (fp8 && cap > 0 && (!recv_scales || scales_ld < cap || scales_ld % 4 != 0)) return EP_ERR_INVALID_ARG;
  if (recv_weights && !topk_weights) return EP_ERR_INVALID_ARG;
  if ((recv_x && !aligned16(recv_x)) || (fp8 && recv_scales && !aligned16(recv_scales)) ||
      (topk_weights && !aligned4(topk_weights)) || (recv_src_idx && !aligned4(recv_src_idx)) ||
      (recv_weights && !aligned4(recv_weights)))
    return EP_ERR_INVALID_ARG;
  if (h->scatter_ns[fp8 ? 1 : 0][ep::kSrcExpertMajor] == 0) return EP_ERR_INVALID_ARG;  // rows too long to stage
  return EP_OK;
}

// The rows of the handle's expert-major layout through the TMA scatter.
ep_status_t em_scatter(ep_handle* h, const void* x, const float* topk_weights, bool fp8, void* recv_x,
                       float* recv_scales, int64_t scales_ld, int64_t cap, int* recv_src_idx, float* recv_weights,
                       int num_sms, cudaStream_t s) {
  const int T = h->T_em;
  ep::ScatterArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.T = T;
  a.H = h->H;
  a.k = h->k;
  a.kmax = h->kmax;
  a.El = h->El;
  a.R = h->R;
  a.E = h->E;
  a.cap = cap;
  a.topk_weights = topk_weights;
  a.ll_idx = h->em_idx;
  a.ll_slot = h->em_slot;
  a.expert_offset = h->em_offset;
  a.expert_count = h->em_count;
  a.recv_src_idx = recv_src_idx;
  a.recv_weights = recv_weights;
  a.scales_ld = scales_ld;
  a.recv_x = recv_x;
  a.recv_scales = recv_scales;
  a.ctl = h->fused_barrier;
  a.err = h->err;
  const int sns = h->scatter_ns[fp8 ? 1 : 0][ep::kSrcExpertMajor], snc = h->scatter_nc[fp8 ? 1 : 0][ep::kSrcExpertMajor];
  const int blocks = grid_for(h, 1, num_sms, T, 1);
  ep::launch_scatter(a, fp8, ep::kSrcExpertMajor, blocks, sns, snc, s);
  if (h->debug)
    std::fprintf(stderr, "[ep] em dispatch %s T=%d: TMA scatter %d blocks, %d stages, %d consumers\n",
                 fp8 ? "fp8" : "bf16", T, blocks, sns, snc);
  return cuda_status(cudaGetLastError(), "k_scatter(em) launch");
}

}  // namespace

ep_status_t ep_em_layout_and_dispatch(ep_handle_t h, const void* topk_idx, int T, const void* x,
                                      const float* topk_weights, ep_dtype_t dtype, int align, void* recv_x,
                                      float* recv_scales, int64_t scales_ld, int64_t cap, int* recv_src_idx,
                                      float* recv_weights, int num_sms, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  if (T < 0 || T % h->R != 0 || T > h->Tmax || (T > 0 && (!topk_idx || !x)) || align < 1 || align > (1 << 16))
    return EP_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * h->k + static_cast<long long>(h->E) * (align - 1) > (1LL << 31) - 1)
    return EP_ERR_INVALID_ARG;
  if (!ids_aligned(h, topk_idx) || (x && !aligned16(x))) return EP_ERR_INVALID_ARG;
  ep_status_t st = em_check_outputs(h, dtype, topk_weights, recv_x, recv_scales, scales_ld, cap, recv_src_idx,
                                    recv_weights);
  if (st != EP_OK) return st;
  if ((st = check_device(h)) != EP_OK) return st;
  const bool fp8 = dtype == EP_FP8_E4M3;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    cudaError_t e = cudaMemsetAsync(h->em_count, 0, sizeof(int) * h->E, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->em_offset, 0, sizeof(int) * (h->E + 1), s);
    if ((st = cuda_status(e, "em memset")) != EP_OK) return st;
    h->T_em = 0;
    return EP_OK;
  }
  int fblocks = 0, fns = 0, fnc = 0, fown = 0;
  ep::fused_config(ep::kSrcExpertMajor, fp8, T, h->R, h->E, h->k, h->kmax, h->H, sms_for(h, num_sms), h->smem_optin,
                   &fblocks, &fns, &fnc, &fown);
  if (fblocks > 0) {
    ep::FusedArgs f = fused_args(h, topk_idx, static_cast<const uint16_t*>(x), topk_weights, T);
    f.agg = h->fused_agg;
    f.own_first = fown;
    f.ll_idx = h->em_idx;
    f.ll_slot = h->em_slot;
    f.recv_count = h->em_count;
    f.align = align;
    f.expert_offset = h->em_offset;
    f.cap = cap;
    f.recv_src_idx = recv_src_idx;
    f.recv_weights = recv_weights;
    f.scales_ld = scales_ld;
    f.recv_x = recv_x;
    f.recv_scales = recv_scales;
    if ((st = cuda_status(ep::launch_fused(f, fp8, ep::kSrcExpertMajor, fblocks, fns, fnc, s),
                          "k_route_scatter(em) launch")) != EP_OK)
      return st;
    if (h->debug)
      std::fprintf(stderr, "[ep] em layout+dispatch T=%d: fused, %d blocks, %d stages, %d consumers\n", T, fblocks,
                   fns, fnc);
    h->T_em = T;
    return EP_OK;
  }
  // per-expert slots on layout-sized chunks, the group offsets, then the rows
  RouteParams p = route_params(h, topk_idx, T, h->layout_CT, h->em_flags, h->tickets + 2);
  ep::LowLatencyOutPtrs ro{h->em_count, h->em_idx, h->em_slot, INT_MAX};
  ep::launch_ll_route(p, ro, h->ll_route_smem, s);
  if ((st = cuda_status(cudaGetLastError(), "k_ll_route(em) launch")) != EP_OK) return st;
  ep::launch_em_offsets(h->em_count, h->E, align, h->em_offset, s);
  if ((st = cuda_status(cudaGetLastError(), "k_em_offsets launch")) != EP_OK) return st;
  h->T_em = T;
  return em_scatter(h, x, topk_weights, fp8, recv_x, recv_scales, scales_ld, cap, recv_src_idx, recv_weights,
                    num_sms, s);
}

ep_status_t ep_em_dispatch(ep_handle_t h, const void* x, const float* topk_weights, ep_dtype_t dtype, void* recv_x,
                           float* recv_scales, int64_t scales_ld, int64_t cap, int* recv_src_idx,
                           float* recv_weights, int num_sms, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  if (h->T_em < 0) return EP_ERR_STATE;
  const int T = h->T_em;
  if ((T > 0 && !x) || (x && !aligned16(x))) return EP_ERR_INVALID_ARG;
  ep_status_t st = em_check_outputs(h, dtype, topk_weights, recv_x, recv_scales, scales_ld, cap, recv_src_idx,
                                    recv_weights);
  if (st != EP_OK) return st;
  if ((st = check_device(h)) != EP_OK) return st;
  if (T == 0) return EP_OK;
  return em_scatter(h, x, topk_weights, dtype == EP_FP8_E4M3, recv_x, recv_scales, scales_ld, cap, recv_src_idx,
                    recv_weights, num_sms, reinterpret_cast<cudaStream_t>(stream));
}

ep_status_t ep_em_get_layout(ep_handle_t h, int* num_recv_tokens_per_expert, int* expert_offset, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  if (h->T_em < 0) return EP_ERR_STATE;
  ep_status_t st = check_device(h);
  if (st != EP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* hp = h->host;
  cudaError_t e = cudaMemcpyAsync(hp, h->err, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(hp + 1, h->em_count, sizeof(int) * h->E, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(hp + 1 + h->E, h->em_offset, sizeof(int) * (h->E + 1), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if ((st = cuda_status(e, "ep_em_get_layout")) != EP_OK) return st;
  if (num_recv_tokens_per_expert) std::memcpy(num_recv_tokens_per_expert, hp + 1, sizeof(int) * h->E);
  if (expert_offset) std::memcpy(expert_offset, hp + 1 + h->E, sizeof(int) * (h->E + 1));
  return static_cast<ep_status_t>(hp[0]);
}

ep_status_t ep_em_combine(ep_handle_t h, const void* y, int64_t y_rows, void* out, int num_sms, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  if (h->T_em < 0) return EP_ERR_STATE;
  const int T = h->T_em;
  if (y_rows < 0 || (T > 0 && (!out || (y_rows > 0 && !y)))) return EP_ERR_INVALID_ARG;
  if ((y && !aligned16(y)) || (out && !aligned16(out))) return EP_ERR_INVALID_ARG;
  ep_status_t st = check_device(h);
  if (st != EP_OK) return st;
  if (T == 0) return EP_OK;
  ep::CombineArgs a{};
  a.y = y;
  a.out = static_cast<uint16_t*>(out);
  a.y_rows = y_rows;
  a.T = T;
  a.H = h->H;
  a.k = h->k;
  a.kmax = h->kmax;
  a.R = h->R;
  a.E = h->E;
  a.ent_idx = h->em_idx;
  a.ent_slot = h->em_slot;
  a.expert_offset = h->em_offset;
  a.err = h->err;
  const int blocks = grid_for(h, h->occ_combine[3], num_sms, T * ((h->H + 1023) / 1024), ep::combine_threads() / 32);
  ep::launch_combine(a, ep::kSrcExpertMajor, false, blocks, reinterpret_cast<cudaStream_t>(stream));
  if (h->debug) std::fprintf(stderr, "[ep] em combine T=%d: %d blocks\n", T, blocks);
  return cuda_status(cudaGetLastError(), "k_combine(em) launch");
}

ep_status_t ep_get_buffer_size_hint(int R, int E, int k, int H, int max_tpr, ep_dtype_t dtype, ep_layout_t layout,
                                    int align, int64_t* rows, int64_t* bytes) {
  if (R < 1 || E < 1 || E % R != 0 || k < 1 || k > 32 || H < 128 || H % 128 != 0 || max_tpr < 1 ||
      (dtype != EP_BF16 && dtype != EP_FP8_E4M3) || (layout == EP_LAYOUT_EXPERT_MAJOR && align < 1))
    return EP_ERR_INVALID_ARG;
  const bool fp8 = dtype == EP_FP8_E4M3;
  const long long T = static_cast<long long>(R) * max_tpr;
  const long long G = H / 128;
  const long long row_bytes = fp8 ? H + 4 * G : 2LL * H;
  long long n = 0, b = 0;
  switch (layout) {
    case EP_LAYOUT_RANK_MAJOR:
      // at most min(k, R) destination ranks per token; per row the payload,
      // its scales, the source index and the k local ids and weights
      n = T * (k < R ? k : R);
      b = n * (row_bytes + 4 + 8LL * k);
      break;
    case EP_LAYOUT_LOW_LATENCY:
      // [E][M][H] with M = R * max_tokens_per_rank, plus src_info and counts
      n = static_cast<long long>(E) * T;
      b = n * (row_bytes + 4) + 4LL * E;
      break;
    case EP_LAYOUT_EXPERT_MAJOR: {
      // every entry unmasked, and each group padded by at most align - 1;
      // scales [G][ld] with ld = rows rounded up to 4
      n = T * k + static_cast<long long>(E) * (align - 1);
      const long long ld = (n + 3) / 4 * 4;
      b = n * (fp8 ? H : 2LL * H) + (fp8 ? 4 * G * ld : 0) + n * 8;
      break;
    }
    default:
      return EP_ERR_INVALID_ARG;
  }
  if (rows) *rows = n;
  if (bytes) *bytes = b;
  return EP_OK;
}

ep_status_t ep_handle_set_topk_idx_bits(ep_handle_t h, int bits) {
  if (!h || (bits != 32 && bits != 64)) return EP_ERR_INVALID_ARG;
  h->ids32 = bits == 32 ? 1 : 0;
  return EP_OK;
}

int ep_handle_topk_idx_bits(ep_handle_t h) { return !h ? 0 : h->ids32 ? 32 : 64; }

ep_status_t ep_check_wait_timeout(ep_handle_t h, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  ep_status_t st = check_device(h);
  if (st != EP_OK) return st;
  ep::launch_wait_timeout_check(h->err, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError(), "ep_check_wait_timeout launch");
}

ep_status_t ep_get_device_status(ep_handle_t h, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID_ARG;
  ep_status_t st = check_device(h);
  if (st != EP_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(h->host, h->err, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->err, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if ((st = cuda_status(e, "ep_get_device_status")) != EP_OK) return st;
  if (h->host[0] == EP_ERR_TIMEOUT) {
    // a wait gave up somewhere: start the fused kernel's control words afresh
    e = cudaMemsetAsync(h->fused_barrier, 0, sizeof(unsigned) * (4 + static_cast<size_t>(h->num_sms)), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if ((st = cuda_status(e, "ep_get_device_status reset")) != EP_OK) return st;
  }
  return static_cast<ep_status_t>(h->host[0]);
}

}  // extern "C"
