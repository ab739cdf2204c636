// low_latency_dispatch on sm_103a, one launch: each block ranks the entries
// of a small chunk of tokens per expert (single-pass cross-block scan), then
// writes its tokens -- quantised once to FP8 or copied as BF16 -- into the
// expert-major receive buffer [E][M][H] ("Как DeepSeek разогнали обмен
// данными ..." (devtrends.ru), "Как это выглядит в коде":
// low_latency_dispatch(hidden_states, topk_idx, num_max_tokens, num_experts);
// "DeepEP 要約" (stakiran.github.io) section 3, decode: no host
// synchronisation, CUDA-graph compatible).
//
// Rows of expert e are filled in (source rank, token, k-index) order, so the
// result does not depend on block scheduling.
#include "ep_internal.h"
#include "routing.cuh"
#include "scatter.cuh"

namespace ep {

template <bool kFP8>
__global__ void __launch_bounds__(kRouteThreads) k_ll_dispatch(RouteParams p, LowLatencyOut o) {
  extern __shared__ int smem_raw[];
  __shared__ float sscale[kRouteWarps][kSeg * 4];
  const int NK = p.E;
  const int NI = p.CT << p.kp_log2;
  const RouteSmem s = route_smem_carve(smem_raw, NK, NI, p.CT, p.kmax);
  const RouteTicket tk = route_take_ticket(p, s);
  const int c = tk.chunk;
  const int src = c / p.cps;
  const int ci = c - src * p.cps;
  const int t0 = src * p.tpr + ci * p.CT;
  const int ct = min(p.CT, p.tpr - ci * p.CT);

  route_rank_chunk<false>(p, s, t0, ct, NK);
  route_lookback(p, s, c, tk.epoch, NK);

  const int kp = 1 << p.kp_log2;
  const int ipw = route_items_per_warp(NI);
  for (int i = threadIdx.x; i < NI; i += kRouteThreads) {
    const int tl = i >> p.kp_log2;
    const int j = i & (kp - 1);
    if (tl >= ct || j >= p.k) continue;
    const int t = t0 + tl;
    const int e = s.item_e[i];
    int slot = -1;
    if (e >= 0) {
      slot = s.excl[e] + s.cnt[(i / ipw) * NK + e] + s.item_le[i];
      if (slot >= o.M) {
        latch_error(p.err, kErrCapacity);
        slot = -1;
      }
    }
    o.ll_idx[static_cast<size_t>(t) * p.k + j] = e;
    o.ll_slot[static_cast<size_t>(t) * p.k + j] = slot;
    s.item_le[i] = slot;
  }
  if (c == p.C - 1 && o.recv_count) {
    for (int e = threadIdx.x; e < p.E; e += kRouteThreads) o.recv_count[e] = min(s.excl[e] + s.agg[e], o.M);
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int tl = warp; tl < ct; tl += kRouteWarps) {
    const int t = t0 + tl;
    long long row = -1;
    if (lane < p.k) {
      const int i = (tl << p.kp_log2) + lane;
      const int e = s.item_e[i];
      const int sl = s.item_le[i];
      if (e >= 0 && sl >= 0) row = static_cast<long long>(e) * o.M + sl;
    }
    const unsigned dmask = __ballot_sync(kFullMask, row >= 0);
    scatter_row<kFP8>(o.x + static_cast<size_t>(t) * o.H, o.H, dmask, row, o.recv_x, o.recv_scales,
                      sscale[warp], lane);
    if (o.recv_src_info && row >= 0) o.recv_src_info[row] = t;
  }
}

// Routing only: the same ranking as k_ll_dispatch on larger chunks, writing
// the slots and counts that k_scatter and the low-latency combine use.
__global__ void __launch_bounds__(kRouteThreads) k_ll_route(RouteParams p, LowLatencyOutPtrs o) {
  extern __shared__ int smem_raw[];
  const int NK = p.E;
  const int NI = p.CT << p.kp_log2;
  const RouteSmem s = route_smem_carve(smem_raw, NK, NI, p.CT, p.kmax);
  const RouteTicket tk = route_take_ticket(p, s);
  const int c = tk.chunk;
  const int src = c / p.cps;
  const int ci = c - src * p.cps;
  const int t0 = src * p.tpr + ci * p.CT;
  const int ct = min(p.CT, p.tpr - ci * p.CT);

  route_rank_chunk<false>(p, s, t0, ct, NK);
  route_lookback(p, s, c, tk.epoch, NK);

  const int kp = 1 << p.kp_log2;
  const int ipw = route_items_per_warp(NI);
  for (int i = threadIdx.x; i < NI; i += kRouteThreads) {
    const int tl = i >> p.kp_log2;
    const int j = i & (kp - 1);
    if (tl >= ct || j >= p.k) continue;
    const int t = t0 + tl;
    const int e = s.item_e[i];
    int slot = -1;
    if (e >= 0) {
      slot = s.excl[e] + s.cnt[(i / ipw) * NK + e] + s.item_le[i];
      if (slot >= o.M) {
        latch_error(p.err, kErrCapacity);
        slot = -1;
      }
    }
    o.ll_idx[static_cast<size_t>(t) * p.k + j] = e;
    o.ll_slot[static_cast<size_t>(t) * p.k + j] = slot;
  }
  if (c == p.C - 1 && o.recv_count) {
    for (int e = threadIdx.x; e < p.E; e += kRouteThreads) o.recv_count[e] = min(s.excl[e] + s.agg[e], o.M);
  }
}

void launch_ll_route(const RouteParams& p, const LowLatencyOutPtrs& o, size_t smem, cudaStream_t stream) {
  (void)launch_kernel(k_ll_route, dim3(p.C), dim3(kRouteThreads), smem, stream, p, o);
}

// Expert-major group offsets from the per-expert counts: offset[e] = sum over
// e' < e of count[e'] rounded up to a multiple of align; offset[E] = total.
// One block: each thread takes a contiguous run of experts, then a block scan.
constexpr int kEmOffsetThreads = 1024;
__global__ void __launch_bounds__(kEmOffsetThreads) k_em_offsets(const int* count, int E, int align, int* offset) {
  __shared__ int wsum[kEmOffsetThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (E + kEmOffsetThreads - 1) / kEmOffsetThreads;
  const int e0 = min(E, static_cast<int>(threadIdx.x) * per), e1 = min(E, e0 + per);
  int run = 0;
  for (int e = e0; e < e1; ++e) run += (count[e] + align - 1) / align * align;
  int inc = run;
  for (int d = 1; d < 32; d <<= 1) {
    const int u = __shfl_up_sync(kFullMask, inc, d);
    if (lane >= d) inc += u;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  int base = 0, total = 0;
  for (int w = 0; w < kEmOffsetThreads / 32; ++w) {
    if (w < warp) base += wsum[w];
    total += wsum[w];
  }
  int at = base + inc - run;
  for (int e = e0; e < e1; ++e) {
    offset[e] = at;
    at += (count[e] + align - 1) / align * align;
  }
  if (threadIdx.x == 0) offset[E] = total;
}

void launch_em_offsets(const int* count, int E, int align, int* offset, cudaStream_t stream) {
  (void)launch_kernel(k_em_offsets, dim3(1), dim3(kEmOffsetThreads), 0, stream, count, E, align, offset);
}

cudaError_t configure_ll_route(size_t needed, size_t optin) {
  return set_dynamic_smem_limit(reinterpret_cast<const void*>(k_ll_route), needed, optin);
}

void launch_ll_dispatch(const RouteParams& p, const LowLatencyOut& o, bool fp8, size_t smem,
                        cudaStream_t stream) {
  if (fp8)
    (void)launch_kernel(k_ll_dispatch<true>, dim3(p.C), dim3(kRouteThreads), smem, stream, p, o);
  else
    (void)launch_kernel(k_ll_dispatch<false>, dim3(p.C), dim3(kRouteThreads), smem, stream, p, o);
}

cudaError_t configure_ll_dispatch(size_t needed, size_t optin) {
  cudaError_t e = set_dynamic_smem_limit(reinterpret_cast<const void*>(k_ll_dispatch<true>), needed, optin);
  if (e != cudaSuccess) return e;
  return set_dynamic_smem_limit(reinterpret_cast<const void*>(k_ll_dispatch<false>), needed, optin);
}

}  // namespace ep
