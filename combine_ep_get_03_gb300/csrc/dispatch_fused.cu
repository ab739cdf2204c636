// Routing and dispatch in one cooperative launch on sm_103a (get_dispatch_layout
// + dispatch, and low_latency_dispatch, of "DeepEP 要約" (stakiran.github.io)
// section 3).
//
// One persistent block per SM: a producer warp and NC consumer warps.
//
// Routing.  Each block owns a contiguous run of tokens and ranks them:
//   normal       -- per (token, destination rank): one lane per token, the
//                   token's ranks as a 64-bit mask (R <= 64), one ballot per
//                   distinct rank in a 32-token batch; expert counts by
//                   shared-memory atomics;
//   low latency / expert-major -- per (token, k) entry and expert:
//                   __match_any_sync within a 32-entry batch, per-warp running
//                   counts in shared memory.
// Each block writes its counts (uint16), all blocks meet at one bounded grid
// barrier (co-residency guaranteed by the cooperative launch), and each block
// sums its predecessors' counts into exclusive prefixes.  Small batches skip
// the barrier and count the ids themselves: in the low-latency mode (up to
// kFusedRedundantEntries entries) each block counts the entries of the tokens
// before its own (16-byte id loads), and the block owning the last token
// writes the per-expert totals; in the expert-major mode every block counts
// every entry (each needs the totals for the group offsets); in the
// rank-major mode (its own instantiation, kRedRanks, so that the large-batch
// code is untouched, up to the host's smaller limit) every block counts every
// token's ranks and experts (tiny shape: 20.4 -> 16.2 us as graph replays).
// The block then writes its tokens' destinations and publishes them (a
// per-block word set to the launch's generation + 1).
//
// Rows.  The row movement is not tied to the routing's token runs.  Each
// block first streams a quarter ring of its own tokens (the first NS / 4 of
// its run): their destinations are in its shared-memory tables as soon as
// its prefixes are final, so its consumers start on them without waiting for
// any other block or reading anything back from L2 (a quarter ring beat a
// full one by 0.8 us on each V3-shaped fused dispatch, one token and half a
// ring came in between).  Then the producer claims the remaining tokens from
// one global counter, claim_tokens_for(bytes a token moves) at a time (one
// at the V3 shape) (position c of the claims names position
// F0 + c mod (tpb - F0) of block c / (tpb - F0), F0 the tokens each block
// moves first), one claim ahead, so that an SM that moves rows faster
// takes more of them (the SMs of one GB300 do not all stream at the same
// rate); a consumer reads a claimed token's destinations from global memory
// once the owning block has published them.  In the rank-major mode the
// producer streams only the first kRouteStages rows before the block's
// prefixes are final: a full ring of row loads from every SM queues ahead of
// the routing's dependent loads and delays it.  The per-entry modes keep the
// full ring (their consumers start with eight stores a row).  Consumers
// quantise / store a row exactly as k_scatter does.  Per-expert totals, which
// nothing waits for, are formed after the rows.
//
// Own rows.  A low-latency batch small enough for the counting above, whose
// tokens per block fit a block's stage ring at once, moves only each block's
// own tokens (decode shape, 7 tokens per SM: each consumer warp takes one
// token), with no claims at all.
//
// Rows and slots come out identical to the separate routing kernels: (source
// rank, token) order per rank, (source rank, token, k) order per expert.  The
// expert-major ("GEMM") layout of the V2 release notes in "DeepSeek công bố
// thư viện mã nguồn mở DeepEP ..." (vi.news.hada.io, "Những thay đổi chính của
// bản phát hành V2") packs those per-expert slots one expert after another,
// each expert's group starting at a multiple of the alignment; every block
// forms the group offsets itself from the totals.
#include <climits>

#include "ep_internal.h"
#include "scatter_common.cuh"

namespace ep {

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" : : "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_release_add_u32(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" : : "l"(p), "r"(v) : "memory");
}

// Grid-wide barrier among the consumer warps of all blocks, on word 0 (the
// arrival count, zero when the launch starts).  The block's writes are ordered
// before thread 32's fence by the block barrier, the fence before its
// releasing arrival; every block then polls the count itself until all nblocks
// have arrived, so the last arrival is seen one L2 round trip after it lands.
// The last block to finish the kernel resets the count (every block has passed
// the barrier by then).  Bounded: gives up after kSpinLimit polls (latched
// kErrTimeout).
__device__ inline void grid_sync(unsigned* words, unsigned nblocks, int* err, int nthreads) {
  consumer_sync(nthreads);
  if (threadIdx.x == 32) {
    __threadfence();
    red_release_add_u32(words, 1u);
    int it = 0;
    while (ld_acquire_u32(words) < nblocks) {
      if (++it > kSpinLimit) {
        latch_error(err, kErrTimeout);
        break;
      }
      if (it > 16) __nanosleep(32);
    }
    __threadfence();
  }
  consumer_sync(nthreads);
}

__host__ __device__ inline int fused_tokens_per_block(int T, int nb) { return (T + nb - 1) / nb; }

// The per-block counts (FusedArgs::agg) are uint16 -- a block owns at most
// kFusedMaxItems (token, k) entries -- in rows of agg_ld(NK) entries (a
// multiple of 8, so a row is a whole number of 16-byte words).
__host__ __device__ inline int agg_ld(int NK) { return (NK + 7) & ~7; }

// Column `col` of the per-block counts summed over every block (off the
// critical path: loads issued 32 at a time).
__device__ __forceinline__ int column_total(const uint16_t* agg, int ld, int col, int nb) {
  int all = 0;
  for (int q0 = 0; q0 < nb; q0 += 32) {
    int v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = q0 + j < nb ? __ldcg(agg + static_cast<size_t>(q0 + j) * ld + col) : 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) all += v[j];
  }
  return all;
}

// Columns [0, ncols) of the per-block counts: excl[c] = the sum over blocks
// q < b and, if `all` is given, all[c] = the sum over every block.  A thread
// loads 8 columns at a time (one 16-byte word per block row); tpc threads
// share an 8-column group (a power of two up to 32, so they sit in one warp)
// and issue their loads 16 words at a time before adding any, then one
// shuffle reduction: a group costs about one L2 round trip per 16 * tpc
// blocks.
__device__ inline void column_sums_par(const uint16_t* agg, int ld, int ncols, int nb, int b, int* excl, int* all,
                                       int nct, int ct) {
  const int oct = (ncols + 7) >> 3;
  int tpc = 32;
  while (tpc > 1 && tpc * oct > nct) tpc >>= 1;
  const int groups = nct / tpc;
  const int sub = ct & (tpc - 1);
  const int qend = all ? nb : b;
  for (int c0 = 0; c0 < oct; c0 += groups) {  // the same trip count in every thread
    const int c = c0 + ct / tpc;
    const bool valid = c < oct;
    int e[8], s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = s[i] = 0;
    if (valid) {
      for (int q0 = sub; q0 < qend; q0 += 16 * tpc) {
        uint4 v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int q = q0 + j * tpc;
          v[j] = q < qend ? __ldcg(reinterpret_cast<const uint4*>(agg + static_cast<size_t>(q) * ld) + c)
                          : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const bool before = q0 + j * tpc < b;
          const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int lo = static_cast<int>(w[i] & 0xffffu), hi = static_cast<int>(w[i] >> 16);
            s[2 * i] += lo;
            s[2 * i + 1] += hi;
            if (before) {
              e[2 * i] += lo;
              e[2 * i + 1] += hi;
            }
          }
        }
      }
    }
    for (int d = tpc >> 1; d >= 1; d >>= 1)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        e[i] += __shfl_xor_sync(kFullMask, e[i], d);
        s[i] += __shfl_xor_sync(kFullMask, s[i], d);
      }
    if (valid && sub == 0)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int col = 8 * c + i;
        if (col < ncols) {
          excl[col] = e[i];
          if (all) all[col] = s[i];
        }
      }
  }
}

// Adds 1 to hist[e] for every id e in [0, E) among the first n ids of the
// top-k table, with 16-byte loads where the table's alignment allows (the
// ids are never written while the kernel runs).  Called by the consumer
// threads (ct of nct).
__device__ inline void count_ids_prefix(const void* ids, int ids32, long long n, int E, int* hist, int ct, int nct) {
  auto add = [&](long long e) {
    if (e >= 0 && e < E) atomicAdd(hist + e, 1);
  };
  const bool vec = (reinterpret_cast<uintptr_t>(ids) & 15) == 0;
  if (vec && !ids32) {
    const longlong2* v = static_cast<const longlong2*>(ids);
    const long long nq = n >> 1;
    for (long long q0 = ct; q0 < nq; q0 += 8LL * nct) {
      longlong2 w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const long long q = q0 + static_cast<long long>(j) * nct;
        w[j] = q < nq ? __ldg(v + q) : make_longlong2(-1, -1);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        add(w[j].x);
        add(w[j].y);
      }
    }
    if ((n & 1) && ct == 0) add(static_cast<const long long*>(ids)[n - 1]);
  } else if (vec) {
    const int4* v = static_cast<const int4*>(ids);
    const long long nq = n >> 2;
    for (long long q0 = ct; q0 < nq; q0 += 8LL * nct) {
      int4 w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const long long q = q0 + static_cast<long long>(j) * nct;
        w[j] = q < nq ? __ldg(v + q) : make_int4(-1, -1, -1, -1);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        add(w[j].x);
        add(w[j].y);
        add(w[j].z);
        add(w[j].w);
      }
    }
    for (long long i = (nq << 2) + ct; i < n; i += nct) add(static_cast<const int*>(ids)[i]);
  } else {
    for (long long i0 = ct; i0 < n; i0 += 16LL * nct) {
      long long v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const long long i = i0 + static_cast<long long>(j) * nct;
        v[j] = i < n ? load_topk_id(ids, i, ids32) : -1;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) add(v[j]);
    }
  }
}

// Routing tables in shared memory (int32 unless noted).
__host__ __device__ inline size_t fused_route_bytes(int mode, int R, int E, int kmax, int kp, int tpb, int nc) {
  if (mode == kSrcRanks)
    return 8 * static_cast<size_t>(tpb)                        // token rank masks (u64)
           + 4 * static_cast<size_t>(tpb) * kmax               // local rows
           + 8 * static_cast<size_t>(tpb) * kp                 // own tokens' ids and weights
           + 4 * (static_cast<size_t>(nc) * R + E + 3 * (R + 1) + 4);
  const size_t ni = static_cast<size_t>(tpb) * kp;
  const size_t em = 2 * static_cast<size_t>(E) + 1 + 32;  // totals, group offsets, scan scratch
  return 8 * ni + 4 * (static_cast<size_t>(nc) * E + E + 4 + em);
}

// Exclusive scan of one value per consumer thread (in thread order) over
// the block's consumer threads; `wsum` holds NC ints.  Returns the thread's
// exclusive prefix and the total in *total.
__device__ inline int consumer_exclusive_scan(int v, int* wsum, int nct, int* total) {
  const int lane = threadIdx.x & 31;
  const int cw = (threadIdx.x >> 5) - 1;
  int inc = v;
  for (int d = 1; d < 32; d <<= 1) {
    const int u = __shfl_up_sync(kFullMask, inc, d);
    if (lane >= d) inc += u;
  }
  if (lane == 31) wsum[cw] = inc;
  consumer_sync(nct);
  int base = 0, all = 0;
  for (int w = 0; w < nct / 32; ++w) {
    const int s = wsum[w];
    if (w < cw) base += s;
    all += s;
  }
  consumer_sync(nct);
  *total = all;
  return base + inc - v;
}

__host__ __device__ inline size_t fused_smem_bytes(int mode, bool fp8, int R, int E, int kmax, int kp, int tpb,
                                                   int nc, int ns, int H) {
  const size_t route = (fused_route_bytes(mode, R, E, kmax, kp, tpb, nc) + 127) & ~static_cast<size_t>(127);
  const size_t qb = static_cast<size_t>(H) + ((4 * static_cast<size_t>(H / 128) + 15) & ~15ull);
  return route + 16 * static_cast<size_t>(ns) + 16 + ((4 * static_cast<size_t>(ns) + 4 + 15) & ~15ull) +
         static_cast<size_t>(ns) * 2 * H + (fp8 ? nc * qb : 0);
}

template <bool kFP8, int kMode, bool kRedRanks = false>
__global__ void __launch_bounds__((kScatterMaxConsumers + 1) * 32, 1) k_route_scatter(FusedArgs a, int NS) {
  constexpr bool kLL = kMode != kSrcRanks;        // per-entry routing (low latency, expert-major)
  constexpr bool kEM = kMode == kSrcExpertMajor;  // packed expert groups
  // rank-major batch small enough for every block to count every token
  static_assert(!kRedRanks || !kLL, "redundant rank counting is a rank-major variant");
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int NC = (blockDim.x >> 5) - 1;
  const int nct = NC * 32;  // consumer threads
  const int ct = threadIdx.x - 32;
  const int R = a.R, E = a.E, k = a.k, kmax = a.kmax, kp = 1 << a.kp_log2;
  const int H = a.H;
  const int G = H >> 7;
  const uint32_t row_bytes = 2u * static_cast<uint32_t>(H);
  const int nb = gridDim.x;
  const int b = blockIdx.x;
  const int tpb = fused_tokens_per_block(a.T, nb);
  const int t_begin = min(a.T, b * tpb);
  const int n_own = min(a.T, t_begin + tpb) - t_begin;
  // phase-1 partition of the block's tokens (rank-major: one lane per token)
  // and entries (per-entry modes) over the consumer warps, 32-aligned
  const int tpw = ((tpb + NC - 1) / NC + 31) & ~31;
  const int NI = tpb << a.kp_log2;
  const int ipw = (((NI + NC - 1) / NC) + 31) & ~31;

  // ---- shared memory carve-up
  unsigned char* p = smem;
  unsigned long long* tmask = nullptr;
  int *tlocal = nullptr, *cnt = nullptr, *hist = nullptr, *so = nullptr, *excl = nullptr, *tot = nullptr;
  int *item_e = nullptr, *item_slot = nullptr, *etot = nullptr, *eoff = nullptr, *wsum = nullptr;
  int* tids = nullptr;    // rank-major: the own tokens' ids [tpb][kp] (bad ids as -1)
  float* tw = nullptr;    // and their top-k weights [tpb][kp] (when rows carry metadata)
  if (!kLL) {
    tmask = reinterpret_cast<unsigned long long*>(p);
    p += 8 * static_cast<size_t>(tpb);
    tlocal = reinterpret_cast<int*>(p);
    p += 4 * static_cast<size_t>(tpb) * kmax;
    tids = reinterpret_cast<int*>(p);
    p += 4 * static_cast<size_t>(tpb) * kp;
    tw = reinterpret_cast<float*>(p);
    p += 4 * static_cast<size_t>(tpb) * kp;
    cnt = reinterpret_cast<int*>(p);   // [NC][R]
    hist = cnt + NC * R;               // [E]
    so = hist + E;                     // [R+1] rank_offset
    excl = so + (R + 1);               // [R+1]
    tot = excl + (R + 1);              // [R+1]
  } else {
    item_e = reinterpret_cast<int*>(p);
    item_slot = item_e + tpb * kp;
    cnt = item_slot + tpb * kp;        // [NC][E], then per-warp prefixes
    excl = cnt + NC * E;               // [E]
    etot = excl + E + 4;               // [E] totals
    eoff = etot + E;                   // [E+1] group offsets (expert-major)
    wsum = eoff + E + 1;               // [32] scan scratch
  }
  unsigned char* sbase = smem + ((fused_route_bytes(kMode, R, E, kmax, kp, tpb, NC) + 127) & ~static_cast<size_t>(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(sbase);
  uint64_t* empty = full + NS;
  uint64_t* routed = empty + NS;  // completes when this block has published its routing
  int* stage_tok = reinterpret_cast<int*>(routed + 2);  // token held by each stage (-1: no more)
  unsigned char* stage0 = reinterpret_cast<unsigned char*>(stage_tok) + ((4 * NS + 4 + 15) & ~15);
  unsigned char* qbuf0 = stage0 + static_cast<size_t>(NS) * row_bytes;
  auto stage = [&](int s) { return stage0 + static_cast<size_t>(s) * row_bytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init(routed, 1);
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == 0) {
    // producer: streams rows into the stages (rank-major: the first
    // kRouteStages from the first instruction on, the rest once this block's
    // prefixes are final); when the tokens run out it hands every consumer
    // warp a "no more" stage
    if (lane == 0) {
      // first the block's own tokens [t_begin, t_begin + F0) -- all of them
      // for small batches -- whose destinations its consumers read from
      // shared memory; then claims of the rest: claim c names position
      // F0 + c % rem of block c / rem (rem = tpb - F0 tokens per block),
      // a.claim_tokens at a time, one claim ahead
      unsigned* claim = a.barrier + kCtlClaim;
      const int F0 = min(a.own_first, tpb);
      const int rem = tpb - F0;
      const int cmax = ((a.T + tpb - 1) / tpb) * rem;  // claims that can name a token
      int i = 0;
      bool ok = true;
      auto put = [&](int t) -> bool {
        const int s = i % NS;
        if (!kLL && i == kRouteStages && !mbar_wait(routed, 0u, a.err)) return false;
        if (i >= NS && !mbar_wait(empty + s, static_cast<uint32_t>((i / NS - 1) & 1), a.err)) return false;
        stage_tok[s] = t;
        mbar_arrive_expect_tx(full + s, row_bytes);
        bulk_load(stage(s), a.x + static_cast<size_t>(t) * H, row_bytes, full + s);
        ++i;
        return true;
      };
      for (int tl = 0; ok && tl < min(F0, n_own); ++tl) ok = put(t_begin + tl);
      if (ok && rem > 0) {
        // one put() per pass of a single loop (an inner loop over a claim's
        // tokens compiled to a V3 fused dispatch 3.5 us slower)
        const int ct = a.claim_tokens;
        int c = static_cast<int>(atomicAdd(claim, static_cast<unsigned>(ct)));
        int end = min(c + ct, cmax);
        int next = c < cmax ? static_cast<int>(atomicAdd(claim, static_cast<unsigned>(ct))) : cmax;
        while (ok && c < cmax) {
          const int t = (c / rem) * tpb + F0 + c % rem;
          if (t < a.T) ok = put(t);
          if (++c == end) {  // this claim done: take the next, and claim one ahead again
            c = next;
            end = min(c + ct, cmax);
            if (c < cmax) next = static_cast<int>(atomicAdd(claim, static_cast<unsigned>(ct)));
          }
        }
      }
      for (int j = i; ok && j < i + NC; ++j) {
        const int s = j % NS;
        if (j >= NS && !mbar_wait(empty + s, static_cast<uint32_t>((j / NS - 1) & 1), a.err)) break;
        stage_tok[s] = -1;
        mbar_arrive(full + s);
      }
    }
    return;
  }

  const int cw = warp - 1;  // consumer warp
  // the grid barrier's generation: written last by the previous launch (a
  // relaxed load sees it), and it cannot change before this block has
  // finished; read here, off the block's start-up path, and first used when
  // the block publishes
  const unsigned gen = ld_relaxed_u32(a.barrier + 1);
  const unsigned lt = lanemask_lt();
  // rank-major rows carry source index / local ids / weights
  const bool meta = !kLL && (a.recv_src_idx || a.recv_topk_idx || a.recv_topk_weights);
  const bool w_own = meta && a.topk_weights;  // own tokens' weights kept in shared memory
  const bool vec8 = k == 8 && (reinterpret_cast<uintptr_t>(a.topk_idx) & 15) == 0 &&
                    (!w_own || (reinterpret_cast<uintptr_t>(a.topk_weights) & 15) == 0);
  // ---------------------------------------------------------------- phase 1: rank the block's tokens
  if (!kLL) {
    for (int i = ct; i < E; i += nct) hist[i] = 0;
    consumer_sync(nct);
    int run_lo = 0, run_hi = 0;
    for (int b0 = cw * tpw; b0 < min(n_own, (cw + 1) * tpw); b0 += 32) {  // warp-uniform
      const int tl = b0 + lane;
      const bool live = tl < n_own && tl < (cw + 1) * tpw;
      unsigned long long m = 0;
      if (live) {
        const int t = t_begin + tl;
        const long long ids = static_cast<long long>(t) * k;
        for (int j0 = 0; j0 < k; j0 += 8) {
          long long v[8];
          float wv[8];
          if (vec8) {
            if (a.ids32) {  // a token's eight int32 ids: two 16-byte loads
              const int4* p4 = reinterpret_cast<const int4*>(static_cast<const int*>(a.topk_idx) + ids);
              const int4 q0 = __ldg(p4), q1 = __ldg(p4 + 1);
              v[0] = q0.x; v[1] = q0.y; v[2] = q0.z; v[3] = q0.w;
              v[4] = q1.x; v[5] = q1.y; v[6] = q1.z; v[7] = q1.w;
            } else {
              const longlong2* p2 = reinterpret_cast<const longlong2*>(static_cast<const long long*>(a.topk_idx) + ids);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const longlong2 q = __ldg(p2 + j);
                v[2 * j] = q.x;
                v[2 * j + 1] = q.y;
              }
            }
            if (w_own) {
              const float4* w4 = reinterpret_cast<const float4*>(a.topk_weights + ids);
              const float4 w0 = __ldg(w4), w1 = __ldg(w4 + 1);
              wv[0] = w0.x; wv[1] = w0.y; wv[2] = w0.z; wv[3] = w0.w;
              wv[4] = w1.x; wv[5] = w1.y; wv[6] = w1.z; wv[7] = w1.w;
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) wv[j] = 0.0f;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              v[j] = j0 + j < k ? load_topk_id(a.topk_idx, ids + j0 + j, a.ids32) : -1;
              wv[j] = w_own && j0 + j < k ? a.topk_weights[ids + j0 + j] : 0.0f;
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (j0 + j >= k) break;
            long long e = v[j];
            if (e < -1 || e >= E) {
              latch_error(a.err, kErrBadExpert);
              e = -1;
            }
            a.idx32[static_cast<size_t>(t) * k + j0 + j] = static_cast<int>(e);
            tids[tl * kp + j0 + j] = static_cast<int>(e);
            tw[tl * kp + j0 + j] = wv[j];
            if (e >= 0) {
              m |= 1ull << (static_cast<int>(e) / a.El);
              if (!kRedRanks) atomicAdd(hist + static_cast<int>(e), 1);
            }
          }
        }
        tmask[tl] = m;
      }
      unsigned long long present =
          static_cast<unsigned long long>(__reduce_or_sync(kFullMask, static_cast<unsigned>(m))) |
          (static_cast<unsigned long long>(__reduce_or_sync(kFullMask, static_cast<unsigned>(m >> 32))) << 32);
      while (present) {  // warp-uniform: ascending ranks present in this batch
        const int r = __ffsll(static_cast<long long>(present)) - 1;
        present &= present - 1;
        const bool has = (m >> r) & 1ull;
        const unsigned bal = __ballot_sync(kFullMask, has);
        const int base = __shfl_sync(kFullMask, r < 32 ? run_lo : run_hi, r & 31);
        if (has) tlocal[tl * kmax + __popcll(m & ((1ull << r) - 1ull))] = base + __popc(bal & lt);
        if (lane == (r & 31)) {
          if (r < 32) run_lo += __popc(bal);
          else run_hi += __popc(bal);
        }
      }
    }
    if (lane < R) cnt[cw * R + lane] = run_lo;
    if (lane + 32 < R) cnt[cw * R + lane + 32] = run_hi;
    consumer_sync(nct);
    for (int col = ct; col < R; col += nct) {
      int run = 0;
      for (int w = 0; w < NC; ++w) {
        const int v = cnt[w * R + col];
        cnt[w * R + col] = run;
        run += v;
      }
      if (!kRedRanks) a.agg[static_cast<size_t>(b) * agg_ld(R + E) + col] = static_cast<uint16_t>(run);
    }
    if (!kRedRanks) {
      for (int e = ct; e < E; e += nct) a.agg[static_cast<size_t>(b) * agg_ld(R + E) + R + e] = static_cast<uint16_t>(hist[e]);
    } else {
      // a small batch: every block counts every token itself -- its
      // destination ranks (all tokens into tot, earlier ones into excl) and its
      // experts (into hist, here the per-expert totals) -- instead of meeting
      // the other blocks at the grid barrier
      for (int i = ct; i <= R; i += nct) excl[i] = tot[i] = 0;
      consumer_sync(nct);
      for (int t = ct; t < a.T; t += nct) {
        unsigned long long m = 0;
        for (int j0 = 0; j0 < k; j0 += 8) {
          long long v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            v[j] = j0 + j < k ? load_topk_id(a.topk_idx, static_cast<long long>(t) * k + j0 + j, a.ids32) : -1;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (v[j] >= 0 && v[j] < E) {
              m |= 1ull << (static_cast<int>(v[j]) / a.El);
              atomicAdd(hist + v[j], 1);
            }
          }
        }
        while (m) {
          const int r = __ffsll(static_cast<long long>(m)) - 1;
          m &= m - 1;
          atomicAdd(tot + r, 1);
          if (t < t_begin) atomicAdd(excl + r, 1);
        }
      }
    }
  } else {
    for (int i = ct; i < NC * E; i += nct) cnt[i] = 0;
    consumer_sync(nct);
    int* cntw = cnt + cw * E;
    const int w_end = min(NI, (cw + 1) * ipw);
    for (int g0 = cw * ipw; g0 < w_end; g0 += 8 * 32) {  // warp-uniform
      // up to 8 batches of 32 entries: every id load in flight before the
      // ranking, which runs batch by batch in order
      int ev[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = g0 + q * 32 + lane;
        const int tl = i >> a.kp_log2;
        const int j = i & (kp - 1);
        long long v = -1;
        if (i < w_end && tl < n_own && j < k) {
          v = load_topk_id(a.topk_idx, static_cast<long long>(t_begin + tl) * k + j, a.ids32);
          if (v < -1 || v >= E) {
            latch_error(a.err, kErrBadExpert);
            v = -1;
          }
        }
        ev[q] = static_cast<int>(v);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (g0 + q * 32 >= w_end) break;  // warp-uniform
        const int i = g0 + q * 32 + lane;
        const int e = ev[q];
        const unsigned pe = __match_any_sync(kFullMask, e);
        int le = 0;
        if (e >= 0) le = cntw[e] + __popc(pe & lt);
        __syncwarp();
        if (e >= 0 && lane == __ffs(pe) - 1) cntw[e] += __popc(pe);
        __syncwarp();
        if (i < NI) {
          item_e[i] = e;
          item_slot[i] = le;
        }
      }
    }
    consumer_sync(nct);
    for (int col = ct; col < E; col += nct) {
      int run = 0;
      for (int w = 0; w < NC; ++w) {
        const int v = cnt[w * E + col];
        cnt[w * E + col] = run;
        run += v;
      }
      if (!a.redundant) a.agg[static_cast<size_t>(b) * agg_ld(E) + col] = static_cast<uint16_t>(run);
      else if (!kEM) etot[col] = run;  // the block's own entries per expert
    }
    if (a.redundant && !kEM) {
      // small batches, low latency: every block with tokens counts the
      // entries of the tokens before its own (into excl) instead of meeting
      // the other blocks at the grid barrier; the block owning the last token
      // then has every expert's total (excl + its own entries)
      for (int e = ct; e < E; e += nct) excl[e] = 0;
      consumer_sync(nct);
      if (n_own > 0) count_ids_prefix(a.topk_idx, a.ids32, static_cast<long long>(t_begin) * k, E, excl, ct, nct);
    } else if (a.redundant) {
      // small batches, expert-major: every block counts every entry itself
      // (entries of earlier tokens into excl, all of them into etot: every
      // block needs the totals for the group offsets)
      for (int e = ct; e < E; e += nct) excl[e] = etot[e] = 0;
      consumer_sync(nct);
      const long long n_all = static_cast<long long>(a.T) * k, n_before = static_cast<long long>(t_begin) * k;
      for (long long i0 = ct; i0 < n_all; i0 += 16 * static_cast<long long>(nct)) {
        long long v[16];  // 16 independent loads in flight, then the counting
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const long long i = i0 + static_cast<long long>(j) * nct;
          v[j] = i < n_all ? load_topk_id(a.topk_idx, i, a.ids32) : -1;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (v[j] >= 0 && v[j] < E) {
            atomicAdd(etot + v[j], 1);
            if (i0 + static_cast<long long>(j) * nct < n_before) atomicAdd(excl + v[j], 1);
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- phase 2: prefixes over blocks
  const bool barrier = kLL ? !a.redundant : !kRedRanks;
  if (barrier) grid_sync(a.barrier, static_cast<unsigned>(nb), a.err, nct);
  else consumer_sync(nct);
  const int ld = agg_ld(kLL ? E : R + E);
  if (!kLL) {
    if (!kRedRanks) column_sums_par(a.agg, ld, R, nb, b, excl, tot, nct, ct);
    consumer_sync(nct);
    if (cw == 0) {  // exclusive scan of the rank totals -> region offsets
      const int v = lane < R ? tot[lane] : 0;
      const int v2 = lane + 32 < R ? tot[lane + 32] : 0;
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
      if (lane < R) so[lane] = inc - v;
      if (lane + 32 < R) so[lane + 32] = carry + inc2 - v2;
      if (lane == 0) so[R] = carry + total2;
      if (b == 0) {
        if (lane < R) {
          a.rank_offset[lane] = inc - v;
          a.recv_per_rank[lane] = v;
        }
        if (lane + 32 < R) {
          a.rank_offset[lane + 32] = carry + inc2 - v2;
          a.recv_per_rank[lane + 32] = v2;
        }
        if (lane == 0) a.rank_offset[R] = carry + total2;
      }
    }
    consumer_sync(nct);
  } else {
    if (!a.redundant) {
      column_sums_par(a.agg, ld, E, nb, b, excl, kEM ? etot : nullptr, nct, ct);
      consumer_sync(nct);
    }
    if (kEM) {
      // group offsets: each consumer thread takes a contiguous run of experts
      const int per = (E + nct - 1) / nct;
      const int e0 = min(E, ct * per), e1 = min(E, e0 + per);
      int run = 0;
      for (int e = e0; e < e1; ++e) run += (etot[e] + a.align - 1) / a.align * a.align;
      int total;
      int at = consumer_exclusive_scan(run, wsum, nct, &total);
      for (int e = e0; e < e1; ++e) {
        eoff[e] = at;
        at += (etot[e] + a.align - 1) / a.align * a.align;
      }
      if (ct == 0) eoff[E] = total;
      consumer_sync(nct);
    }
  }
  consumer_sync(nct);  // the prefixes are final: every own token's destinations are known here
  if (threadIdx.x == 32) mbar_arrive(routed);  // the producer may stream past kRouteStages rows (rank-major)

  // The own tokens' destinations for the handle and for the other blocks'
  // consumers: rank-major, each token's (rank, row-in-rank) list; per-entry
  // modes, each entry's expert and slot.
  auto write_own_destinations = [&]() {
    if (!kLL) {
      for (int tl = ct; tl < n_own; tl += nct) {
        const int t = t_begin + tl;
        const int w = tl / tpw;
        unsigned long long m = tmask[tl];
        int pos = 0;
        while (m) {
          const int r = __ffsll(static_cast<long long>(m)) - 1;
          m &= m - 1;
          const int in_rank = excl[r] + cnt[w * R + r] + tlocal[tl * kmax + pos];
          a.dst[static_cast<size_t>(t) * kmax + pos] = make_int2(r, in_rank);
          ++pos;
        }
        for (; pos < kmax; ++pos) a.dst[static_cast<size_t>(t) * kmax + pos] = make_int2(-1, -1);
      }
    } else {
      for (int i = ct; i < n_own * kp; i += nct) {
        const int tl = i >> a.kp_log2;
        const int j = i & (kp - 1);
        if (j >= k) continue;
        const int t = t_begin + tl;
        const int e = item_e[i];
        int slot = -1;
        if (e >= 0) {
          slot = excl[e] + cnt[(i / ipw) * E + e] + item_slot[i];
          if (!kEM && slot >= a.M) {
            latch_error(a.err, kErrCapacity);
            slot = -1;
          }
        }
        a.ll_idx[static_cast<size_t>(t) * k + j] = e;
        a.ll_slot[static_cast<size_t>(t) * k + j] = slot;
      }
    }
  };

  // ---------------------------------------------------------------- phase 3: move the rows
  unsigned char* qd = qbuf0 + static_cast<size_t>(cw) * (static_cast<size_t>(H) + ((4 * G + 15) & ~15));
  float* sd = reinterpret_cast<float*>(qd + H);
  bool first = true;
  int owner_ok = b;  // the owning block whose destinations were last seen published
  // ring item i (stage i % NS) of this consumer warp; false: no more items
  auto step = [&](int i) -> bool {
    const int s = i % NS;
    const bool landed = mbar_wait(full + s, static_cast<uint32_t>((i / NS) & 1), a.err);
    if (!__all_sync(kFullMask, landed)) return false;
    const int t = stage_tok[s];
    if (t >= a.T) latch_error(a.err, kErrState);  // never written by the producer: cannot happen
    if (t < 0 || t >= a.T) {  // no more rows
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
      return false;
    }
    // the owning block's destinations: published words, then plain L2 loads
    const int owner = t / tpb;
    bool have = true;
    if (owner != owner_ok) {
      int it = 0;
      while (ld_acquire_u32(a.barrier + kCtlPub + owner) != gen + 1) {
        if (++it > kSpinLimit) {
          latch_error(a.err, kErrTimeout);
          have = false;
          break;
        }
        if (it > 16) __nanosleep(64);
      }
      have = __all_sync(kFullMask, have);
      if (have) owner_ok = owner;
    }
    long long row = -1;
    int r = -1, e = -1;
    float w = 0.0f;
    if (!have) {
      // gave up waiting (latched): the token's rows are skipped
    } else if (!kLL) {
      if (owner == b) {
        // the block's own token: destinations from its shared-memory tables
        // (the values the routing phase published): the lane-th destination
        // rank in ascending order, its row in the rank's region
        const int tl = t - t_begin;
        if (lane < kmax) {
          unsigned long long m = tmask[tl];
          for (int q = 0; q < lane && m; ++q) m &= m - 1;
          if (m) {
            r = __ffsll(static_cast<long long>(m)) - 1;
            row = static_cast<long long>(so[r]) + excl[r] + cnt[(tl / tpw) * R + r] + tlocal[tl * kmax + lane];
          }
        }
        if (meta && lane < k) {
          e = tids[tl * kp + lane];
          w = tw[tl * kp + lane];
        }
      } else {
        if (lane < kmax) {
          const int2 d = __ldcg(a.dst + static_cast<size_t>(t) * kmax + lane);
          if (d.x >= 0) {
            r = d.x;
            row = static_cast<long long>(so[d.x]) + d.y;
          }
        }
        if (meta && lane < k) {
          e = __ldcg(a.idx32 + static_cast<size_t>(t) * k + lane);
          if (a.topk_weights) w = a.topk_weights[static_cast<size_t>(t) * k + lane];
        }
      }
      if (row >= a.cap) {
        latch_error(a.err, kErrCapacity);
        row = -1;
      }
    } else if (lane < k) {
      int ee, sl;
      if (owner == b) {
        // the block's own token: its entries' experts and slots from shared
        // memory (the values the routing phase published)
        const int it = ((t - t_begin) << a.kp_log2) + lane;
        ee = item_e[it];
        sl = ee >= 0 ? excl[ee] + cnt[(it / ipw) * E + ee] + item_slot[it] : -1;
        if (!kEM && sl >= a.M) sl = -1;  // over capacity (latched when published)
      } else {
        ee = __ldcg(a.ll_idx + static_cast<size_t>(t) * k + lane);
        sl = __ldcg(a.ll_slot + static_cast<size_t>(t) * k + lane);
      }
      if (ee >= 0 && sl >= 0) row = kEM ? static_cast<long long>(eoff[ee]) + sl : static_cast<long long>(ee) * a.M + sl;
      if (kEM && row >= a.cap) {
        latch_error(a.err, kErrCapacity);  // the row does not fit the receive buffer
        row = -1;
      }
      if (kEM && row >= 0 && a.recv_weights) w = a.topk_weights[static_cast<size_t>(t) * k + lane];
    }
    const unsigned dmask = __ballot_sync(kFullMask, row >= 0);
    if (kFP8) {
      if (!first) {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      }
      quantize_row_smem(stage(s), qd, sd, G, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
      unsigned m = dmask;
      while (m) {
        const int sl = __ffs(m) - 1;
        m &= m - 1;
        const long long rr = __shfl_sync(kFullMask, row, sl);
        if (lane == 0) bulk_store(static_cast<uint8_t*>(a.recv_x) + rr * H, qd, static_cast<uint32_t>(H));
        if (kEM)
          for (int g = lane; g < G; g += 32) st_keep(a.recv_scales + g * a.scales_ld + rr, sd[g]);
        else
          for (int g = lane; g < G; g += 32) a.recv_scales[rr * G + g] = sd[g];
      }
      if (lane == 0) bulk_commit();
    } else {
      unsigned m = dmask;
      while (m) {
        const int sl = __ffs(m) - 1;
        m &= m - 1;
        const long long rr = __shfl_sync(kFullMask, row, sl);
        if (lane == 0) bulk_store(static_cast<uint16_t*>(a.recv_x) + rr * H, stage(s), row_bytes);
      }
      if (lane == 0) {
        bulk_commit();
        bulk_wait_read<0>();
        mbar_arrive(empty + s);
      }
      __syncwarp();
    }
    first = false;
    if (meta) {
      unsigned m = dmask;
      while (m) {
        const int sl = __ffs(m) - 1;
        m &= m - 1;
        const long long rr = __shfl_sync(kFullMask, row, sl);
        const int rk = __shfl_sync(kFullMask, r, sl);
        if (lane == 0 && a.recv_src_idx) st_keep(a.recv_src_idx + rr, t);
        if (lane < k) {
          const bool here = e >= 0 && e / a.El == rk;
          if (a.recv_topk_idx) a.recv_topk_idx[rr * k + lane] = here ? e - rk * a.El : -1;
          if (a.recv_topk_weights) a.recv_topk_weights[rr * k + lane] = here ? w : 0.0f;
        }
      }
    } else if (kEM && row >= 0) {
      if (a.recv_src_idx) st_keep(a.recv_src_idx + row, t);
      if (a.recv_weights) st_keep(a.recv_weights + row, w);
    } else if (kLL && a.recv_src_info && row >= 0) {
      st_keep(a.recv_src_info + row, t);
    }
    return true;
  };
  // Publish this block's destinations (a consumer warp's first items are the
  // block's own tokens, whose destinations it reads from shared memory; the
  // other blocks need them for the tokens they claim), then move the rows in
  // ring order.
  write_own_destinations();
  consumer_sync(nct);
  if (threadIdx.x == 32) {  // this block's destinations are visible to every block
    __threadfence();
    st_release_u32(a.barrier + kCtlPub + b, gen + 1);
  }
  for (int i = cw; step(i); i += NC) {
  }
  if (kEM) {
    // padding rows of the groups this block owns (experts b, b + nb, ...):
    // no source token, weight 0; and the group offsets and counts
    for (int e = b; e < E; e += nb) {
      const long long end = min(static_cast<long long>(eoff[e + 1]), a.cap);
      for (long long rw = static_cast<long long>(eoff[e]) + etot[e] + ct; rw < end; rw += nct) {
        if (a.recv_src_idx) a.recv_src_idx[rw] = -1;
        if (a.recv_weights) a.recv_weights[rw] = 0.0f;
      }
      if (ct == 0) {
        a.expert_offset[e] = eoff[e];
        a.recv_count[e] = etot[e];
      }
    }
    if (b == 0 && ct == 0) a.expert_offset[E] = eoff[E];
  }
  // per-expert totals (outputs only, nothing above waits for them): block b
  // forms the totals of experts e = b, b + nb, ...
  if (kLL && !kEM && a.redundant) {
    if (n_own > 0 && t_begin + n_own == a.T && a.recv_count)
      for (int e = ct; e < E; e += nct) a.recv_count[e] = min(excl[e] + etot[e], a.M);
  } else {
    for (int e = b + ct * nb; !kEM && e < E; e += nct * nb) {
      const int all = kRedRanks ? hist[e] : column_total(a.agg, ld, (kLL ? 0 : R) + e, nb);
      if (kLL) {
        if (a.recv_count) a.recv_count[e] = min(all, a.M);
      } else {
        a.recv_per_expert[e] = all;
      }
    }
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
  // the last block to finish resets the claim counter for the next launch
  // (every claim of every block has returned by the time it counts itself)
  // and the grid barrier's count, and advances the generation that the
  // "published" words of the next launch are compared with
  consumer_sync(nct);
  if (threadIdx.x == 32 && atomicAdd(a.barrier + kCtlDone, 1u) == static_cast<unsigned>(nb) - 1) {
    atomicExch(a.barrier + kCtlClaim, 0u);
    atomicExch(a.barrier + kCtlDone, 0u);
    atomicExch(a.barrier, 0u);
    atomicAdd(a.barrier + 1, 1u);
  }
}

constexpr int kFusedMinStages = 8;

// Blocks, stages and consumers for the fused kernel, and how many of its own
// tokens each block streams before it claims others'; blocks = 0 when the
// kernel does not apply (R > 64 in normal mode, too many (token, k) entries
// per block, rows too long for two stages).  Each block first moves a quarter
// ring of its own tokens (their destinations are in its shared memory as soon
// as it has routed them).  A low-latency batch small enough for every block
// to count the entries itself moves only each block's own tokens when they
// fit its ring at once: then the most consumers whose ring still holds them
// all (one token per consumer where possible).
void fused_config(int mode, bool fp8, int T, int R, int E, int k, int kmax, int H, int sms, size_t smem_limit,
                  int* blocks, int* NS, int* NC, int* own_first) {
  *blocks = *NS = *NC = 0;
  if (own_first) *own_first = 0;
  if (T <= 0 || (mode == kSrcRanks && R > 64)) return;
  int kp = 1;
  while (kp < k) kp <<= 1;
  const int nb = sms;
  const int tpb = fused_tokens_per_block(T, nb);
  if (tpb * kp > kFusedMaxItems) return;
  const bool small = mode == kSrcLowLatency && static_cast<long long>(T) * k <= kFusedRedundantEntries;
  const int max_nc = fp8 ? kScatterMaxConsumers : 4;
  int own_ns = 0, own_nc = 0;
  for (int pass = 0; pass < 2 && *NS == 0; ++pass) {
    // first at least half the consumers (the quantiser's compute), then any
    for (int nc = max_nc; nc >= (pass == 0 ? (max_nc + 1) / 2 : 1); --nc) {
      const size_t fixed = fused_smem_bytes(mode, fp8, R, E, kmax, kp, tpb, nc, 0, H);
      if (fixed >= smem_limit) continue;
      int ns = static_cast<int>((smem_limit - fixed) / (20 + 2 * static_cast<size_t>(H)));
      if (ns > 32) ns = 32;
      while (ns >= 2 && fused_smem_bytes(mode, fp8, R, E, kmax, kp, tpb, nc, ns, H) > smem_limit) --ns;
      ns -= ns % nc;  // consumer c owns the stages s = c (mod nc), as in k_scatter
      // the most consumers whose ring has at least kFusedMinStages stages (the
      // quantiser's compute is spread over more warps: V3 shape, 8 consumers
      // x 8 stages beat 6 x 12 by 1-3 us); failing that, the most stages
      const bool enough = ns >= kFusedMinStages && *NS < kFusedMinStages;
      if (ns >= 2 && ns >= nc && (enough || (*NS < kFusedMinStages && ns > *NS))) {
        *NS = ns;
        *NC = nc;
      }
      if (small && own_ns == 0 && ns >= 2 && ns >= nc && ns >= tpb) {  // the most consumers that hold tpb
        own_ns = ns;
        own_nc = nc;
      }
    }
  }
  if (own_ns > 0) {
    *NS = own_ns;
    *NC = own_nc;
  }
  if (*NS > 0) {
    *blocks = nb;
    if (own_first) *own_first = own_ns > 0 ? tpb : min(max(*NS / 4, 1), tpb);
  }
}

cudaError_t configure_fused(size_t optin) {
  const void* ks[8] = {reinterpret_cast<const void*>(k_route_scatter<false, kSrcRanks>),
                       reinterpret_cast<const void*>(k_route_scatter<true, kSrcRanks>),
                       reinterpret_cast<const void*>(k_route_scatter<false, kSrcRanks, true>),
                       reinterpret_cast<const void*>(k_route_scatter<true, kSrcRanks, true>),
                       reinterpret_cast<const void*>(k_route_scatter<false, kSrcLowLatency>),
                       reinterpret_cast<const void*>(k_route_scatter<true, kSrcLowLatency>),
                       reinterpret_cast<const void*>(k_route_scatter<false, kSrcExpertMajor>),
                       reinterpret_cast<const void*>(k_route_scatter<true, kSrcExpertMajor>)};
  for (const void* kk : ks) {
    cudaError_t e = set_dynamic_smem_limit(kk, 0, optin);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_fused(const FusedArgs& args, bool fp8, int mode, int blocks, int NS, int NC, cudaStream_t stream) {
  FusedArgs a = args;
  a.claim_tokens =
      claim_tokens_for(row_bytes_per_token(a.H, a.k, a.kmax, fp8, mode), mode == kSrcRanks ? blocks : 0);
  int kp = 1;
  while (kp < a.k) kp <<= 1;
  const int tpb = fused_tokens_per_block(a.T, blocks);
  const size_t smem = fused_smem_bytes(mode, fp8, a.R, a.E, a.kmax, kp, tpb, NC, NS, a.H);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3((NC + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (mode == kSrcLowLatency)
    return fp8 ? cudaLaunchKernelEx(&cfg, k_route_scatter<true, kSrcLowLatency>, a, NS)
               : cudaLaunchKernelEx(&cfg, k_route_scatter<false, kSrcLowLatency>, a, NS);
  if (mode == kSrcExpertMajor)
    return fp8 ? cudaLaunchKernelEx(&cfg, k_route_scatter<true, kSrcExpertMajor>, a, NS)
               : cudaLaunchKernelEx(&cfg, k_route_scatter<false, kSrcExpertMajor>, a, NS);
  if (a.redundant)
    return fp8 ? cudaLaunchKernelEx(&cfg, k_route_scatter<true, kSrcRanks, true>, a, NS)
               : cudaLaunchKernelEx(&cfg, k_route_scatter<false, kSrcRanks, true>, a, NS);
  return fp8 ? cudaLaunchKernelEx(&cfg, k_route_scatter<true, kSrcRanks>, a, NS)
             : cudaLaunchKernelEx(&cfg, k_route_scatter<false, kSrcRanks>, a, NS);
}

}  // namespace ep
