// ep_get_dispatch_layout_noalloc: the layout computation for callers that
// cannot allocate device memory.  It needs no handle: the cross-block scan
// state lives in a fixed, file-scope device array that the library owns, and
// every result goes to buffers the caller passes in.  The kernel is the same
// k_layout that ep_get_dispatch_layout launches.
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "ep.h"
#include "ep_internal.h"
#include "routing.cuh"

namespace {

// 1 MiB of scan state, shared by every call on a device and kept for the
// life of the process: word 0 = chunk ticket (with its epoch), word 1 = the
// fallback status latch, words [kFlagBase, kScratchWords) = look-back words.
constexpr int kScratchWords = 1 << 17;
constexpr int kFlagBase = 32;
static __device__ __align__(256) unsigned long long g_layout_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned long long* g_scratch_ptr[kMaxDevices] = {};
size_t g_smem_limit[kMaxDevices] = {};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Once per device, with that device current: the device address of the
// scratch array (its host-side name is only a stand-in), and the layout
// kernel's dynamic shared-memory limit (set from the opt-in maximum).
ep_status_t device_setup(int dev, unsigned long long** scratch, size_t* smem_limit) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_layout_scratch);
    if (e != cudaSuccess) {
      if (std::getenv("EP_DEBUG"))
        std::fprintf(stderr, "[ep] cudaGetSymbolAddress(layout scratch): %s\n", cudaGetErrorString(e));
      return EP_ERR_CUDA;
    }
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    // the layout kernel's shared-memory limit: the opt-in maximum, the value
    // handle creation also sets, so the two never lower it under each other
    size_t limit = 0;
    if (e == cudaSuccess) e = ep::configure_layout(0, static_cast<size_t>(optin), &limit);
    if (e != cudaSuccess) return EP_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<unsigned long long*>(p);
    g_smem_limit[dev] = limit;
  }
  *scratch = g_scratch_ptr[dev];
  *smem_limit = g_smem_limit[dev];
  return EP_OK;
}

}  // namespace

extern "C" ep_status_t ep_get_dispatch_layout_noalloc(int R, int E, int k, const int64_t* topk_idx, int T,
                                                      int* num_tokens_per_rank, int* num_tokens_per_expert,
                                                      uint8_t* is_token_in_rank, int* num_recv_tokens_per_rank,
                                                      int* num_recv_tokens_per_expert, int* rank_offset,
                                                      int* token_dest, int* topk_idx32, int* device_status,
                                                      ep_stream_t stream) {
  if (R < 1 || R > 1024 || E < 1 || E > 4096 || E % R != 0 || k < 1 || k > 32) return EP_ERR_INVALID_ARG;
  if (T < 0 || T % R != 0 || (T > 0 && (!topk_idx || !token_dest || !topk_idx32)) || !num_recv_tokens_per_rank ||
      !num_recv_tokens_per_expert || !rank_offset)
    return EP_ERR_INVALID_ARG;
  if ((topk_idx && !aligned(topk_idx, 8)) || (token_dest && !aligned(token_dest, 8)) ||
      (topk_idx32 && !aligned(topk_idx32, 4)) || (num_tokens_per_rank && !aligned(num_tokens_per_rank, 4)) ||
      (num_tokens_per_expert && !aligned(num_tokens_per_expert, 4)) || !aligned(num_recv_tokens_per_rank, 4) ||
      !aligned(num_recv_tokens_per_expert, 4) || !aligned(rank_offset, 4) ||
      (device_status && !aligned(device_status, 4)))
    return EP_ERR_INVALID_ARG;
  int lg = 0;
  while ((1 << lg) < k) ++lg;
  const int kmax = k < R ? k : R;
  const int CT = 1024 >> lg;
  const int tpr = T / R;
  const int cps = (tpr + CT - 1) / CT;
  const int C = R * cps;
  const int NK = R + E;
  if (static_cast<long long>(C) * NK > kScratchWords - kFlagBase) {
    if (std::getenv("EP_DEBUG"))
      std::fprintf(stderr, "[ep] layout_noalloc: %d chunks x %d columns exceed the %d-word scratch\n", C, NK,
                   kScratchWords - kFlagBase);
    return EP_ERR_INVALID_ARG;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return EP_ERR_CUDA;
  if (dev >= kMaxDevices) return EP_ERR_INVALID_ARG;
  unsigned long long* scratch = nullptr;
  size_t smem_limit = 0;
  ep_status_t st = device_setup(dev, &scratch, &smem_limit);
  if (st != EP_OK) return st;
  const size_t smem = ep::route_smem_bytes(NK, CT << lg, CT, kmax);
  if (smem > smem_limit) return EP_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (T == 0) {
    cudaError_t e = cudaMemsetAsync(num_recv_tokens_per_rank, 0, sizeof(int) * R, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(num_recv_tokens_per_expert, 0, sizeof(int) * E, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(rank_offset, 0, sizeof(int) * (R + 1), s);
    if (e == cudaSuccess && num_tokens_per_rank) e = cudaMemsetAsync(num_tokens_per_rank, 0, sizeof(int) * R * R, s);
    if (e == cudaSuccess && num_tokens_per_expert)
      e = cudaMemsetAsync(num_tokens_per_expert, 0, sizeof(int) * static_cast<size_t>(R) * E, s);
    return e == cudaSuccess ? EP_OK : EP_ERR_CUDA;
  }
  // Each call starts from cleared scan state: ticket (chunk 0, epoch 0), the
  // fallback latch and the look-back words this call uses.  All-zero words
  // never count as published.
  cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(unsigned long long) * (kFlagBase + static_cast<size_t>(C) * NK), s);
  if (e != cudaSuccess) return EP_ERR_CUDA;

  ep::RouteParams p;
  p.topk_idx = topk_idx;
  p.ids32 = 0;
  p.T = T;
  p.R = R;
  p.E = E;
  p.El = E / R;
  p.k = k;
  p.kp_log2 = lg;
  p.kmax = kmax;
  p.tpr = tpr;
  p.CT = CT;
  p.cps = cps;
  p.C = C;
  p.flags = scratch + kFlagBase;
  p.ticket = scratch;
  p.err = device_status ? device_status : reinterpret_cast<int*>(scratch + 1);
  ep::LayoutOutPtrs o{reinterpret_cast<int2*>(token_dest), topk_idx32, num_recv_tokens_per_rank, rank_offset,
                      num_recv_tokens_per_expert, num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank};
  ep::launch_layout(p, o, smem, s);
  e = cudaGetLastError();
  return e == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}
