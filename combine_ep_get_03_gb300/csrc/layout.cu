// get_dispatch_layout on sm_103a: one launch computes, from topk_idx, every
// token's destination ranks and its row inside each destination rank's
// receive region, the per-rank / per-expert counts and the region offsets
// ("DeepEP 要約" (stakiran.github.io) section 3, training forward;
// "Как DeepSeek разогнали обмен данными ..." (devtrends.ru), "Как это
// выглядит в коде": num_tokens_per_rank feeds dispatch).
//
// Row order inside rank r's region: (source rank, token) -- the order a
// deterministic scan yields.  Regions are packed in ascending rank.
#include "ep_internal.h"
#include "routing.cuh"

namespace ep {

struct LayoutOut {
  int2* dst;                   // [T][kmax] (rank, row in rank) ascending rank, (-1,-1) padded
  int* idx32;                  // [T][k] copy of topk_idx (int32)
  int* recv_per_rank;          // [R]
  int* rank_offset;            // [R+1]
  int* recv_per_expert;        // [E]
  int* num_tokens_per_rank;    // [R][R] or null
  int* num_tokens_per_expert;  // [R][E] or null
  uint8_t* is_token_in_rank;   // [T][R] or null
};

__global__ void __launch_bounds__(kRouteThreads) k_layout(RouteParams p, LayoutOut o) {
  extern __shared__ int smem_raw[];
  const int NK = p.R + p.E;
  const int NI = p.CT << p.kp_log2;
  const RouteSmem s = route_smem_carve(smem_raw, NK, NI, p.CT, p.kmax);
  const RouteTicket tk = route_take_ticket(p, s);
  const int c = tk.chunk;
  const int src = c / p.cps;
  const int ci = c - src * p.cps;
  const int t0 = src * p.tpr + ci * p.CT;
  const int ct = min(p.CT, p.tpr - ci * p.CT);

  route_rank_chunk<true>(p, s, t0, ct, NK);
  route_lookback(p, s, c, tk.epoch, NK);

  // per-item outputs: the token's destination list and the int32 id copy
  const int kp = 1 << p.kp_log2;
  const int ipw = route_items_per_warp(NI);
  for (int i = threadIdx.x; i < NI; i += kRouteThreads) {
    const int tl = i >> p.kp_log2;
    const int j = i & (kp - 1);
    if (tl >= ct || j >= p.k) continue;
    const int t = t0 + tl;
    o.idx32[static_cast<size_t>(t) * p.k + j] = s.item_e[i];
    const int r = s.item_r[i];
    if (r >= 0) {
      const int row = s.excl[r] + s.cnt[(i / ipw) * NK + r] + s.item_lr[i];
      o.dst[static_cast<size_t>(t) * p.kmax + s.item_pos[i]] = make_int2(r, row);
    }
    if (j < p.kmax && j >= s.tok_ndist[tl])
      o.dst[static_cast<size_t>(t) * p.kmax + j] = make_int2(-1, -1);
  }
  if (o.is_token_in_rank) {
    for (int q = threadIdx.x; q < ct * p.R; q += kRouteThreads) {
      const int tl = q / p.R;
      const int r = q - tl * p.R;
      uint8_t in = 0;
      for (int d = 0; d < s.tok_ndist[tl]; ++d) in |= (s.tok_rank[tl * p.kmax + d] == r);
      o.is_token_in_rank[static_cast<size_t>(t0 + tl) * p.R + r] = in;
    }
  }
  // per-source-rank counts: the source rank's last chunk subtracts the
  // inclusive prefix at the end of the previous source rank from its own
  if (ci == p.cps - 1 && (o.num_tokens_per_rank || o.num_tokens_per_expert)) {
    for (int col = threadIdx.x; col < NK; col += kRouteThreads) {
      uint32_t prev = 0;
      if (src > 0)
        prev = flag_value(flag_wait(p.flags + static_cast<size_t>(src * p.cps - 1) * NK + col, tk.epoch,
                                    kFlagInclusive, p.err));
      const int v = s.excl[col] + s.agg[col] - static_cast<int>(prev);
      if (col < p.R) {
        if (o.num_tokens_per_rank) o.num_tokens_per_rank[src * p.R + col] = v;
      } else if (o.num_tokens_per_expert) {
        o.num_tokens_per_expert[static_cast<size_t>(src) * p.E + (col - p.R)] = v;
      }
    }
  }
  // totals and region offsets: the last chunk holds the grand inclusive prefix
  if (c == p.C - 1) {
    for (int col = threadIdx.x; col < NK; col += kRouteThreads) {
      const int v = s.excl[col] + s.agg[col];
      if (col < p.R) {
        o.recv_per_rank[col] = v;
        s.agg[col] = v;  // reused below for the offsets
      } else {
        o.recv_per_expert[col - p.R] = v;
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {  // warp 0: exclusive scan over ranks
      const int lane = threadIdx.x;
      int carry = 0;
      for (int base = 0; base < p.R; base += 32) {
        const int r = base + lane;
        int v = r < p.R ? s.agg[r] : 0;
        int inc = v;
        for (int d = 1; d < 32; d <<= 1) {
          const int u = __shfl_up_sync(kFullMask, inc, d);
          if (lane >= d) inc += u;
        }
        if (r < p.R) o.rank_offset[r] = carry + inc - v;
        carry += __shfl_sync(kFullMask, inc, 31);
      }
      if (lane == 0) o.rank_offset[p.R] = carry;
    }
  }
}

void launch_layout(const RouteParams& p, const LayoutOutPtrs& out, size_t smem, cudaStream_t stream) {
  LayoutOut o;
  o.dst = out.dst;
  o.idx32 = out.idx32;
  o.recv_per_rank = out.recv_per_rank;
  o.rank_offset = out.rank_offset;
  o.recv_per_expert = out.recv_per_expert;
  o.num_tokens_per_rank = out.num_tokens_per_rank;
  o.num_tokens_per_expert = out.num_tokens_per_expert;
  o.is_token_in_rank = out.is_token_in_rank;
  k_layout<<<p.C, kRouteThreads, smem, stream>>>(p, o);
}

cudaError_t configure_layout(size_t smem) {
  return cudaFuncSetAttribute(k_layout, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

}  // namespace ep
