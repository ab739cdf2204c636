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

// ---------------------------------------------------------------------------
// Token-per-lane layout for R <= 64.  A lane holds one token: its destination
// ranks form a 64-bit mask, so the token's ascending rank list is the mask's
// set bits.  A rank's rows are numbered within a 32-token batch by one ballot
// per distinct rank present in the batch, carried across a warp's batches in
// registers (lane r holds the warp's running count for ranks r and r + 32),
// then across warps by a shared-memory prefix and across chunks by the
// look-back.  Expert counts are shared-memory atomic histograms (order-free
// integer sums).

struct TokenSmem {
  int* cnt;                 // [kRouteWarps][R] per-warp rank counts -> per-warp prefixes
  int* agg;                 // [NK] chunk totals: R rank columns, then E expert columns
  int* excl;                // [NK]
  unsigned long long* mask; // [CT] destination-rank mask of each token
  int* local;               // [CT][kmax] row of (token, k-th rank) within its warp
  int* misc;                // [4]
};

__host__ __device__ inline size_t layout_tokens_smem_bytes(int R, int E, int CT, int kmax) {
  const size_t ints = static_cast<size_t>(kRouteWarps) * R + 2 * (R + E) + static_cast<size_t>(CT) * kmax + 4;
  return ((ints * 4 + 7) & ~static_cast<size_t>(7)) + 8 * static_cast<size_t>(CT);
}

__global__ void __launch_bounds__(kRouteThreads) k_layout_tokens(RouteParams p, LayoutOut o) {
  extern __shared__ unsigned long long smem_u64[];
  const int R = p.R, E = p.E, NK = R + E, CT = p.CT, k = p.k, kmax = p.kmax;
  TokenSmem s;
  s.mask = smem_u64;
  s.cnt = reinterpret_cast<int*>(smem_u64 + CT);
  s.agg = s.cnt + kRouteWarps * R;
  s.excl = s.agg + NK;
  s.local = s.excl + NK;
  s.misc = s.local + CT * kmax;
  // ticket (shares the word format of the entry-per-lane kernel)
  RouteSmem rs;
  rs.agg = s.agg;
  rs.excl = s.excl;
  rs.misc = s.misc;
  const RouteTicket tk = route_take_ticket(p, rs);
  const int c = tk.chunk;
  const int src = c / p.cps;
  const int ci = c - src * p.cps;
  const int t0 = src * p.tpr + ci * CT;
  const int ct = min(CT, p.tpr - ci * CT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt = lanemask_lt();

  for (int i = threadIdx.x; i < E; i += kRouteThreads) s.agg[R + i] = 0;  // expert histogram
  __syncthreads();

  // phase 1: each warp ranks its run of tokens, 32 at a time
  const int tpw = ((CT + kRouteWarps - 1) / kRouteWarps + 31) & ~31;
  int run_lo = 0, run_hi = 0;  // this lane's running counts for ranks `lane` and `lane + 32`
  for (int b0 = warp * tpw; b0 < min(ct, (warp + 1) * tpw); b0 += 32) {  // warp-uniform
    const int tl = b0 + lane;
    const bool live = tl < ct && tl < (warp + 1) * tpw;
    unsigned long long m = 0;
    if (live) {
      const long long ids = static_cast<long long>(t0 + tl) * k;
      for (int j0 = 0; j0 < k; j0 += 8) {
        long long v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = j0 + j < k ? load_topk_id(p.topk_idx, ids + j0 + j, p.ids32) : -1;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j0 + j >= k) break;
          long long e = v[j];
          if (e < -1 || e >= E) {
            latch_error(p.err, kErrBadExpert);
            e = -1;
          }
          o.idx32[static_cast<size_t>(t0 + tl) * k + j0 + j] = static_cast<int>(e);
          if (e >= 0) {
            m |= 1ull << (static_cast<int>(e) / p.El);
            atomicAdd(s.agg + R + static_cast<int>(e), 1);
          }
        }
      }
      s.mask[tl] = m;
    }
    unsigned long long present = static_cast<unsigned long long>(__reduce_or_sync(kFullMask, static_cast<unsigned>(m))) |
                                 (static_cast<unsigned long long>(__reduce_or_sync(kFullMask, static_cast<unsigned>(m >> 32))) << 32);
    while (present) {  // warp-uniform: ascending ranks present in this batch
      const int r = __ffsll(static_cast<long long>(present)) - 1;
      present &= present - 1;
      const bool has = (m >> r) & 1ull;
      const unsigned bal = __ballot_sync(kFullMask, has);
      const int base = __shfl_sync(kFullMask, r < 32 ? run_lo : run_hi, r & 31);
      if (has) s.local[tl * kmax + __popcll(m & ((1ull << r) - 1ull))] = base + __popc(bal & lt);
      if (lane == (r & 31)) {
        if (r < 32) run_lo += __popc(bal);
        else run_hi += __popc(bal);
      }
    }
  }
  if (lane < R) s.cnt[warp * R + lane] = run_lo;
  if (lane + 32 < R) s.cnt[warp * R + lane + 32] = run_hi;
  __syncthreads();
  // per rank column: exclusive prefix over warps and the chunk total
  for (int col = threadIdx.x; col < R; col += kRouteThreads) {
    int run = 0;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int v = s.cnt[w * R + col];
      s.cnt[w * R + col] = run;
      run += v;
    }
    s.agg[col] = run;
  }
  __syncthreads();

  route_lookback(p, rs, c, tk.epoch, NK);

  // outputs: each token's (rank, row) list in ascending rank, (-1,-1) padded
  for (int tl = threadIdx.x; tl < ct; tl += kRouteThreads) {
    const int t = t0 + tl;
    const int w = tl / tpw;
    unsigned long long m = s.mask[tl];
    int pos = 0;
    while (m) {
      const int r = __ffsll(static_cast<long long>(m)) - 1;
      m &= m - 1;
      const int row = s.excl[r] + s.cnt[w * R + r] + s.local[tl * kmax + pos];
      o.dst[static_cast<size_t>(t) * kmax + pos] = make_int2(r, row);
      ++pos;
    }
    for (; pos < kmax; ++pos) o.dst[static_cast<size_t>(t) * kmax + pos] = make_int2(-1, -1);
  }
  if (o.is_token_in_rank) {
    for (int q = threadIdx.x; q < ct * R; q += kRouteThreads) {
      const int tl = q / R;
      const int r = q - tl * R;
      o.is_token_in_rank[static_cast<size_t>(t0 + tl) * R + r] = static_cast<uint8_t>((s.mask[tl] >> r) & 1ull);
    }
  }
  // per-source-rank counts
  if (ci == p.cps - 1 && (o.num_tokens_per_rank || o.num_tokens_per_expert)) {
    for (int col = threadIdx.x; col < NK; col += kRouteThreads) {
      uint32_t prev = 0;  // inclusive prefix at the end of the previous source rank
      if (src > 0)
        prev = flag_value(flag_wait(p.flags + static_cast<size_t>(src * p.cps - 1) * NK + col, tk.epoch,
                                    kFlagInclusive, p.err));
      const int v = s.excl[col] + s.agg[col] - static_cast<int>(prev);
      if (col < R) {
        if (o.num_tokens_per_rank) o.num_tokens_per_rank[src * R + col] = v;
      } else if (o.num_tokens_per_expert) {
        o.num_tokens_per_expert[static_cast<size_t>(src) * E + (col - R)] = v;
      }
    }
  }
  // totals and region offsets
  if (c == p.C - 1) {
    for (int col = threadIdx.x; col < NK; col += kRouteThreads) {
      const int v = s.excl[col] + s.agg[col];
      if (col < R) {
        o.recv_per_rank[col] = v;
        s.agg[col] = v;
      } else {
        o.recv_per_expert[col - R] = v;
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      int v = lane < R ? s.agg[lane] : 0;
      int v2 = lane + 32 < R ? s.agg[lane + 32] : 0;
      int inc = v, inc2 = v2;
      for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(kFullMask, inc, d);
        const int u2 = __shfl_up_sync(kFullMask, inc2, d);
        if (lane >= d) {
          inc += u;
          inc2 += u2;
        }
      }
      const int carry = __shfl_sync(kFullMask, inc, 31);
      const int total2 = __shfl_sync(kFullMask, inc2, 31);
      if (lane < R) o.rank_offset[lane] = inc - v;
      if (lane + 32 < R) o.rank_offset[lane + 32] = carry + inc2 - v2;
      if (lane == 0) o.rank_offset[R] = carry + total2;
    }
  }
}

void launch_layout_tokens(const RouteParams& p, const LayoutOutPtrs& out, cudaStream_t stream) {
  LayoutOut o;
  o.dst = out.dst;
  o.idx32 = out.idx32;
  o.recv_per_rank = out.recv_per_rank;
  o.rank_offset = out.rank_offset;
  o.recv_per_expert = out.recv_per_expert;
  o.num_tokens_per_rank = out.num_tokens_per_rank;
  o.num_tokens_per_expert = out.num_tokens_per_expert;
  o.is_token_in_rank = out.is_token_in_rank;
  const size_t smem = layout_tokens_smem_bytes(p.R, p.E, p.CT, p.kmax);
  (void)launch_kernel(k_layout_tokens, dim3(p.C), dim3(kRouteThreads), smem, stream, p, o);
}

size_t layout_tokens_smem(int R, int E, int CT, int kmax) { return layout_tokens_smem_bytes(R, E, CT, kmax); }

cudaError_t configure_layout_tokens(size_t needed, size_t optin) {
  return set_dynamic_smem_limit(reinterpret_cast<const void*>(k_layout_tokens), needed, optin);
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
  (void)launch_kernel(k_layout, dim3(p.C), dim3(kRouteThreads), smem, stream, p, o);
}

cudaError_t configure_layout(size_t needed, size_t optin, size_t* limit) {
  return set_dynamic_smem_limit(reinterpret_cast<const void*>(k_layout), needed, optin, limit);
}

}  // namespace ep
