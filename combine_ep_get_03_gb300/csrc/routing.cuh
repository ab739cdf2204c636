// The routing phase shared by the layout kernel and the fused low-latency
// dispatch kernel: one thread block ranks the (token, k) entries of one chunk
// of tokens, and a single-pass cross-block scan (decoupled look-back with
// bounded waits) turns the chunk-local ranks into global ones.
//
// What is ranked (get_dispatch_layout and low_latency_dispatch in "DeepEP
// 要約" (stakiran.github.io) section 3; the vi.news.hada.io DeepEP article,
// "Mẫu sử dụng cho huấn luyện, prefill và decoding"):
//  * rank columns (layout only): each (token, destination rank) pair, once
//    per rank even when several of the token's experts live there; its row in
//    the rank's region is the number of pairs with the same rank that come
//    earlier in (source rank, token) order;
//  * expert columns: each unmasked (token, k) entry; its slot in the expert's
//    low-latency buffer is the number of entries with the same expert earlier
//    in (source rank, token, k) order.  The layout uses only the counts.
//
// Chunks never straddle a source rank, and chunk ids are handed out by an
// atomic ticket, so a block only ever waits for blocks that started before
// it: the scan finishes without any co-residency assumption.
//
// The ticket word also carries the call's epoch ([63:32] epoch, [31:0] next
// chunk id).  The block that draws the last chunk id advances the epoch and
// zeroes the id in one exchange; every other block has drawn its id -- and
// so read the epoch -- before that.  Because the epoch lives on the device,
// replays of a captured CUDA graph each get a fresh epoch.
#pragma once

#include "device_common.cuh"

namespace ep {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;

struct RouteParams {
  const void* topk_idx;     // [T][k], int64 or int32 (ids32)
  int ids32;
  int T, R, E, El, k;
  int kp_log2;              // lanes per token: the power of two >= k
  int kmax;                 // min(k, R): distinct ranks a token can reach
  int tpr;                  // tokens per source rank
  int CT;                   // tokens per chunk
  int cps;                  // chunks per source rank
  int C;                    // chunks in total = R * cps
  unsigned long long* flags;   // [C][NK] look-back words
  unsigned long long* ticket;  // [63:32] epoch, [31:0] next chunk id (0 between calls)
  int* err;
};

struct RouteTicket {
  int chunk;
  uint32_t epoch;  // 30-bit, never 0
};

// Shared-memory carve-up of one routing block (all int32).
struct RouteSmem {
  int* cnt;       // [kRouteWarps][NK]: per-warp counts, then per-warp prefixes
  int* agg;       // [NK] chunk totals
  int* excl;      // [NK] exclusive prefix of the chunk over earlier chunks
  int* item_e;    // [NI] expert id of item i (-1 = none)
  int* item_le;   // [NI] rank of the item among its warp's same-expert items
  int* item_r;    // [NI] destination rank if the item is the token's first entry for it, else -1
  int* item_lr;   // [NI] rank of that pair among its warp's same-rank pairs
  int* item_pos;  // [NI] position of that rank among the token's distinct ranks (ascending)
  int* tok_ndist; // [CT] number of distinct destination ranks of each token
  int* tok_rank;  // [CT][kmax] the token's distinct ranks, ascending
  int* misc;      // [4]: chunk id, epoch
};

__host__ __device__ inline size_t route_smem_bytes(int NK, int NI, int CT, int kmax) {
  return sizeof(int) * (static_cast<size_t>(kRouteWarps) * NK + 2 * NK + 5 * NI + CT + CT * kmax + 4);
}

__device__ inline RouteSmem route_smem_carve(int* base, int NK, int NI, int CT, int kmax) {
  RouteSmem s;
  s.cnt = base;
  s.agg = s.cnt + kRouteWarps * NK;
  s.excl = s.agg + NK;
  s.item_e = s.excl + NK;
  s.item_le = s.item_e + NI;
  s.item_r = s.item_le + NI;
  s.item_lr = s.item_r + NI;
  s.item_pos = s.item_lr + NI;
  s.tok_ndist = s.item_pos + NI;
  s.tok_rank = s.tok_ndist + CT;
  s.misc = s.tok_rank + CT * kmax;
  return s;
}

// Items are the chunk's (token, k) entries padded to 2^kp_log2 lanes per
// token; warp w owns items [w*ipw, (w+1)*ipw), so warps hold consecutive
// runs of tokens and lane order inside a warp is (token, k) order.
__device__ __forceinline__ int route_items_per_warp(int NI) {
  int per = (NI + kRouteWarps - 1) / kRouteWarps;
  return (per + 31) & ~31;
}

// Items per chunk are at most kRouteMaxItems, so a warp holds at most
// kRouteMaxBatches batches of 32 and can load all of its ids up front.
constexpr int kRouteMaxItems = 2048;
constexpr int kRouteMaxBatches = kRouteMaxItems / kRouteThreads;

// Phase 1: chunk-local ranking.  kRanks adds the rank columns (layout).
// Column layout: kRanks ? [R rank columns | E expert columns] : [E expert columns].
template <bool kRanks>
__device__ inline void route_rank_chunk(const RouteParams& p, const RouteSmem& s, int t0, int ct, int NK) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kp = 1 << p.kp_log2;
  const int NI = p.CT << p.kp_log2;
  const int ipw = route_items_per_warp(NI);
  const int colE = kRanks ? p.R : 0;
  const int begin = warp * ipw;
  const int end = min(NI, begin + ipw);
  // every id this warp ranks, requested before any is used
  long long pre[kRouteMaxBatches];
#pragma unroll
  for (int bb = 0; bb < kRouteMaxBatches; ++bb) {
    const int i = begin + bb * 32 + lane;
    const int tl = i >> p.kp_log2;
    const int j = i & (kp - 1);
    pre[bb] = (i < end && tl < ct && j < p.k) ? load_topk_id(p.topk_idx, static_cast<long long>(t0 + tl) * p.k + j, p.ids32) : -1;
  }
  for (int i = threadIdx.x; i < kRouteWarps * NK; i += kRouteThreads) s.cnt[i] = 0;
  __syncthreads();

  int* cntw = s.cnt + warp * NK;
  const unsigned lt = lanemask_lt();
  const int gbase = lane & ~(kp - 1);
  const unsigned gmask = (kp == 32 ? kFullMask : ((1u << kp) - 1u)) << gbase;
#pragma unroll
  for (int bb = 0; bb < kRouteMaxBatches; ++bb) {
    const int b = begin + bb * 32;
    if (b >= end) break;  // warp-uniform
    const int i = b + lane;
    const int tl = i >> p.kp_log2;
    const int j = i & (kp - 1);
    const bool in_chunk = i < end && tl < ct;
    long long v = pre[bb];
    if (v < -1 || v >= p.E) {
      latch_error(p.err, kErrBadExpert);
      v = -1;
    }
    const int e = static_cast<int>(v);
    // expert columns: rank among this warp's entries for the same expert
    const unsigned pe = __match_any_sync(kFullMask, e);
    int le = 0;
    if (e >= 0) le = cntw[colE + e] + __popc(pe & lt);
    __syncwarp();
    if (e >= 0 && lane == __ffs(pe) - 1) cntw[colE + e] += __popc(pe);
    __syncwarp();
    if (in_chunk) {
      s.item_e[i] = e;
      s.item_le[i] = le;
    }
    if (kRanks) {
      const int r = e >= 0 ? e / p.El : -1;
      // the token's first entry for rank r represents the (token, r) pair
      const unsigned ptr = __match_any_sync(kFullMask, r >= 0 ? (lane >> p.kp_log2) * p.R + r : -1);
      const bool first = r >= 0 && lane == __ffs(ptr) - 1;
      const int keyr = first ? r : -1;
      const unsigned pr = __match_any_sync(kFullMask, keyr);
      int lr = 0;
      if (first) lr = cntw[r] + __popc(pr & lt);
      __syncwarp();
      if (first && lane == __ffs(pr) - 1) cntw[r] += __popc(pr);
      __syncwarp();
      // ascending position among the token's distinct ranks
      int pos = 0;
      for (int jj = 0; jj < kp; ++jj) {
        const int rr = __shfl_sync(kFullMask, keyr, gbase + jj);
        pos += (rr >= 0 && rr < r) ? 1 : 0;
      }
      const int ndist = __popc(__ballot_sync(kFullMask, first) & gmask);
      if (in_chunk) {
        s.item_r[i] = keyr;
        s.item_lr[i] = lr;
        s.item_pos[i] = pos;
        if (j == 0) s.tok_ndist[tl] = ndist;
        if (first) s.tok_rank[tl * p.kmax + pos] = r;
      }
    }
  }
  __syncthreads();
  // per column: exclusive prefix over warps (in place) and the chunk total
  for (int c = threadIdx.x; c < NK; c += kRouteThreads) {
    int run = 0;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int v = s.cnt[w * NK + c];
      s.cnt[w * NK + c] = run;
      run += v;
    }
    s.agg[c] = run;
  }
  __syncthreads();
}

// Phase 2: publish the chunk totals, then look back over earlier chunks for
// each column's exclusive prefix, then publish the inclusive prefix.
//
// The look-back reads a window of kLookbackWindow predecessors with
// independent loads and walks it from the nearest one, adding counts until it
// meets an inclusive prefix.  Chunks publish at nearly the same moment, so
// part of a window is often read just before it is written; the unread tail
// of the window is then reloaded as a batch (one memory round trip per retry,
// not one per predecessor).  Retries are bounded: after kSpinLimit the block
// latches kErrTimeout and stops looking back.
constexpr int kLookbackWindow = 32;

__device__ inline void route_lookback(const RouteParams& p, const RouteSmem& s, int c, uint32_t epoch, int NK) {
  unsigned long long* mine = p.flags + static_cast<size_t>(c) * NK;
  for (int col = threadIdx.x; col < NK; col += kRouteThreads)
    flag_store(mine + col, make_flag(epoch, c == 0 ? kFlagInclusive : kFlagAggregate,
                                     static_cast<uint32_t>(s.agg[col])));
  for (int col = threadIdx.x; col < NK; col += kRouteThreads) {
    uint32_t ex = 0;
    if (c > 0) {
      bool done = false;
      int retries = 0;
      for (int q = c - 1; q >= 0 && !done; q -= kLookbackWindow) {
        const int n = min(kLookbackWindow, q + 1);
        unsigned long long w[kLookbackWindow];
#pragma unroll
        for (int j = 0; j < kLookbackWindow; ++j)
          w[j] = j < n ? flag_load(p.flags + static_cast<size_t>(q - j) * NK + col) : 0ull;
        int first = 0;  // entries before `first` are already added
        while (true) {
          int stale = -1;
#pragma unroll
          for (int j = 0; j < kLookbackWindow; ++j) {
            if (j < first || j >= n || done || stale >= 0) continue;
            const unsigned long long v = w[j];
            if (flag_epoch(v) != epoch || flag_state(v) < kFlagAggregate) {
              stale = j;
            } else {
              ex += flag_value(v);
              if (flag_state(v) == kFlagInclusive) done = true;
            }
          }
          if (done || stale < 0) break;
          if (++retries > kSpinLimit) {
            latch_error(p.err, kErrTimeout);
            done = true;
            break;
          }
          first = stale;
          if (retries > 8) __nanosleep(32);
#pragma unroll
          for (int j = 0; j < kLookbackWindow; ++j)
            if (j >= first && j < n) w[j] = flag_load(p.flags + static_cast<size_t>(q - j) * NK + col);
        }
      }
      flag_store(mine + col, make_flag(epoch, kFlagInclusive, ex + static_cast<uint32_t>(s.agg[col])));
    }
    s.excl[col] = static_cast<int>(ex);
  }
  __syncthreads();
}

// Chunk id and epoch from the ticket word.  The block that draws the last
// id writes back (epoch + 1, id 0) for the next call.
__device__ __forceinline__ RouteTicket route_take_ticket(const RouteParams& p, const RouteSmem& s) {
  if (threadIdx.x == 0) {
    const unsigned long long w = atomicAdd(p.ticket, 1ull);
    const int c = static_cast<int>(static_cast<uint32_t>(w));
    const uint32_t epoch = static_cast<uint32_t>(w >> 32);
    if (c == p.C - 1) {
      uint32_t next = (epoch + 1) & ((1u << 30) - 1);
      if (next == 0) next = 1;
      atomicExch(p.ticket, static_cast<unsigned long long>(next) << 32);
    }
    s.misc[0] = c;
    s.misc[1] = static_cast<int>(epoch);
  }
  __syncthreads();
  return RouteTicket{s.misc[0], static_cast<uint32_t>(s.misc[1])};
}

}  // namespace ep
