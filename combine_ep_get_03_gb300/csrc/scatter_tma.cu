// Dispatch's row movement on sm_103a with TMA bulk copies ("DeepEP 要約"
// (stakiran.github.io) section 3: dispatch and low_latency_dispatch;
// "DeepSeek выпустила DeepEP V2.5" (aikraft.ru), "Технические детали и
// требования": FP8 dispatch).  A token row is read from HBM once by a bulk
// load into shared memory, quantised once to FP8 (or kept as BF16), and
// written to each destination by one bulk store per destination.
//
// HBM-bound.  One persistent block per SM: a producer warp keeps up to NS row
// loads in flight through a ring of stages, and NC consumer warps quantise
// and store, so both the bytes in flight and the quantisation warps are
// bounded by shared memory rather than registers.  The producer claims
// tokens one at a time from one global counter, so SMs that move rows
// faster take more of them (the SMs of one GB300 do not stream at one rate).
//
// Destinations:  normal  -- the handle's (rank, row-in-rank) list + the
//                           rank's region offset (the layout's output);
//                low latency -- expert e's row `slot` in [E][M][H];
//                expert-major -- row expert_offset[e] + slot of the packed
//                           expert groups; fp8 scales stored group-major
//                           [G][scales_ld]; padding rows of each group get
//                           source -1 and weight 0.
//
// FP8: a lane quantises whole 128-channel groups (quantize_row_smem), so a
// token row costs one warp-wide pair of divisions per 32 groups and no
// shuffles.
#include "ep_internal.h"
#include "scatter_common.cuh"

namespace ep {

// Block layout (dynamic shared memory):
//   [rank_offset: R+1 ints (normal) | expert_offset: E+1 ints (expert-major)]
//   [full[NS], empty[NS] mbarriers]
//   [NS row stages of 2H bytes][NC quantised-row buffers of H + scales (FP8)]
// Warp 0 is the producer: lane 0 streams claimed token rows into the stages
// with bulk loads (full[s] counts the bytes), item i into stage i % NS.
// Warps 1..NC are consumers: consumer c takes items c, c+NC, ...; it waits for
// its stage, quantises it into its own buffer (FP8) or stores straight from
// the stage (BF16), releases the stage (empty[s]) once nothing reads it any
// more, and bulk-stores the row to every destination.  NS is a multiple of
// NC, so consumer c is the only one to use stages s = c (mod NC): when it
// waits on a stage's parity for item i, it has itself consumed item i - NS
// of that stage, so the barrier cannot still be one phase behind (a parity
// wait would return at once on the phase before).
__host__ __device__ inline int scatter_head_ints(int mode, int R, int E) {
  return mode == kSrcRanks ? R + 1 : mode == kSrcExpertMajor ? E + 1 : 0;
}
__host__ __device__ inline size_t scatter_head_bytes(int n) { return (static_cast<size_t>(n) * 4 + 15) & ~15ull; }
__host__ __device__ inline size_t scatter_qbuf_bytes(int H) {
  return static_cast<size_t>(H) + ((4 * static_cast<size_t>(H / 128) + 15) & ~15ull);
}
__host__ __device__ inline size_t scatter_block_bytes(int H, int head_ints, bool fp8, int NS, int NC) {
  return scatter_head_bytes(head_ints) + 16 * static_cast<size_t>(NS) + ((4 * static_cast<size_t>(NS) + 15) & ~15ull) +
         static_cast<size_t>(NS) * 2 * static_cast<size_t>(H) + (fp8 ? static_cast<size_t>(NC) * scatter_qbuf_bytes(H) : 0);
}

template <bool kFP8, int kMode>
__global__ void __launch_bounds__((kScatterMaxConsumers + 1) * 32, 1) k_scatter(ScatterArgs a, int NS) {
  constexpr bool kLL = kMode != kSrcRanks;  // per-entry destinations
  constexpr bool kEM = kMode == kSrcExpertMajor;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int NC = (blockDim.x >> 5) - 1;
  const int H = a.H;
  const int G = H >> 7;
  const uint32_t row_bytes = 2u * static_cast<uint32_t>(H);
  int* so = reinterpret_cast<int*>(smem);  // rank_offset (normal) / expert_offset (expert-major)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + scatter_head_bytes(scatter_head_ints(kMode, a.R, a.E)));
  uint64_t* empty = full + NS;
  int* stage_tok = reinterpret_cast<int*>(empty + NS);  // token held by each stage (-1: no more)
  unsigned char* stage0 = reinterpret_cast<unsigned char*>(stage_tok) + ((4 * NS + 15) & ~15);
  unsigned char* qbuf0 = stage0 + static_cast<size_t>(NS) * row_bytes;
  auto stage = [&](int s) { return stage0 + static_cast<size_t>(s) * row_bytes; };

  if (!kLL)
    for (int r = threadIdx.x; r <= a.R; r += blockDim.x) so[r] = a.rank_offset[r];
  if (kEM) {
    for (int e = threadIdx.x; e <= a.E; e += blockDim.x) so[e] = a.expert_offset[e];
    // padding rows of the groups this block owns: no source token, weight 0
    for (int e = blockIdx.x; e < a.E; e += gridDim.x) {
      const long long end = min(static_cast<long long>(a.expert_offset[e + 1]), a.cap);
      for (long long rw = static_cast<long long>(a.expert_offset[e]) + a.expert_count[e] + threadIdx.x; rw < end;
           rw += blockDim.x) {
        if (a.recv_src_idx) a.recv_src_idx[rw] = -1;
        if (a.recv_weights) a.recv_weights[rw] = 0.0f;
      }
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == 0) {
    // producer: claims tokens a.claim_tokens at a time (one claim ahead); when
    // the claims run out it hands every consumer warp a "no more" stage
    if (lane == 0) {
      unsigned* claim = a.ctl + kCtlClaim;
      int base = static_cast<int>(atomicAdd(claim, static_cast<unsigned>(a.claim_tokens)));
      int next = base < a.T ? static_cast<int>(atomicAdd(claim, static_cast<unsigned>(a.claim_tokens))) : a.T;
      int i = 0;
      bool ok = true;
      while (ok && base < a.T) {
        for (int c = 0; c < a.claim_tokens && base + c < a.T; ++c, ++i) {
          const int s = i % NS;
          if (i >= NS && !mbar_wait(empty + s, static_cast<uint32_t>((i / NS - 1) & 1), a.err)) {
            ok = false;
            break;
          }
          stage_tok[s] = base + c;
          mbar_arrive_expect_tx(full + s, row_bytes);
          bulk_load(stage(s), a.x + static_cast<size_t>(base + c) * H, row_bytes, full + s);
        }
        base = next;
        if (base < a.T) next = static_cast<int>(atomicAdd(claim, static_cast<unsigned>(a.claim_tokens)));
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

  const int cc = warp - 1;  // consumer index
  unsigned char* qd = qbuf0 + static_cast<size_t>(cc) * scatter_qbuf_bytes(H);
  float* sd = reinterpret_cast<float*>(qd + H);
  const bool meta = !kLL && (a.recv_src_idx || a.recv_topk_idx || a.recv_topk_weights);
  bool first = true;
  for (int i = cc;; i += NC) {
    const int s = i % NS;
    const bool landed = mbar_wait(full + s, static_cast<uint32_t>((i / NS) & 1), a.err);
    if (!__all_sync(kFullMask, landed)) break;  // gave up (latched)
    const int t = stage_tok[s];
    if (t >= a.T) latch_error(a.err, kErrState);  // never written by the producer: cannot happen
    if (t < 0 || t >= a.T) {  // no more rows
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
      break;
    }
    // destinations of this token
    long long row = -1;
    int r = -1, e = -1;
    float w = 0.0f;
    if (!kLL) {
      if (lane < a.kmax) {
        const int2 d = a.dst[static_cast<size_t>(t) * a.kmax + lane];
        if (d.x >= 0) {
          r = d.x;
          row = static_cast<long long>(so[d.x]) + d.y;
          if (row >= a.cap) {
            latch_error(a.err, kErrCapacity);
            row = -1;
          }
        }
      }
      if (meta && lane < a.k) {
        e = a.idx32[static_cast<size_t>(t) * a.k + lane];
        if (a.topk_weights) w = a.topk_weights[static_cast<size_t>(t) * a.k + lane];
      }
    } else if (lane < a.k) {
      const int ee = a.ll_idx[static_cast<size_t>(t) * a.k + lane];
      const int ss = a.ll_slot[static_cast<size_t>(t) * a.k + lane];
      if (ee >= 0 && ss >= 0) row = kEM ? static_cast<long long>(so[ee]) + ss : static_cast<long long>(ee) * a.M + ss;
      if (kEM && row >= a.cap) {
        latch_error(a.err, kErrCapacity);
        row = -1;
      }
      if (kEM && row >= 0 && a.recv_weights) w = a.topk_weights[static_cast<size_t>(t) * a.k + lane];
    }
    const unsigned dmask = __ballot_sync(kFullMask, row >= 0);

    if (kFP8) {
      if (!first) {
        if (lane == 0) bulk_wait_read<0>();  // this consumer's previous stores have read its buffer
        __syncwarp();
      }
      quantize_row_smem(stage(s), qd, sd, G, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);  // the stage is free again
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
        bulk_wait_read<0>();  // the stores have read the stage
        mbar_arrive(empty + s);
      }
      __syncwarp();
    }
    first = false;
    // per-row metadata
    if (meta) {
      unsigned m = dmask;
      while (m) {
        const int sl = __ffs(m) - 1;
        m &= m - 1;
        const long long rr = __shfl_sync(kFullMask, row, sl);
        const int rk = __shfl_sync(kFullMask, r, sl);
        if (lane == 0 && a.recv_src_idx) st_keep(a.recv_src_idx + rr, t);
        if (lane < a.k) {
          const bool here = e >= 0 && e / a.El == rk;
          if (a.recv_topk_idx) a.recv_topk_idx[rr * a.k + lane] = here ? e - rk * a.El : -1;
          if (a.recv_topk_weights) a.recv_topk_weights[rr * a.k + lane] = here ? w : 0.0f;
        }
      }
    } else if (kEM && row >= 0) {
      if (a.recv_src_idx) st_keep(a.recv_src_idx + row, t);
      if (a.recv_weights) st_keep(a.recv_weights + row, w);
    } else if (kLL && a.recv_src_info && row >= 0) {
      st_keep(a.recv_src_info + row, t);
    }
  }
  if (lane == 0) bulk_wait_all();  // stores done before the block's shared memory goes away
  __syncwarp();
  // the last block to finish resets the claim counter for the next launch
  // (every claim of every block has returned by the time it counts itself)
  consumer_sync(NC * 32);
  if (threadIdx.x == 32 && atomicAdd(a.ctl + kCtlDone, 1u) == gridDim.x - 1) {
    atomicExch(a.ctl + kCtlClaim, 0u);
    atomicExch(a.ctl + kCtlDone, 0u);
  }
}

// Consumers and stages for a block: FP8 wants compute warps (8 consumers, the
// rest of shared memory as stages); BF16 only moves bytes: 2 consumers over
// at most 4 stages (V3-shaped BF16 dispatch 115.1 us, against 118.3 with 4
// consumers over all the stages that fit, 116.3 with 4 x 8, 116.5 with
// 3 x 3, 125-133 with 1 x 2, 1 x 4 or 2 x 2: fewer rows in flight per SM
// queue less in front of the HBM).  NS is a multiple of NC.  Fewer consumers
// if the rows are long; 0 if not even two stages fit.
void scatter_config(int H, int R, int E, bool fp8, int mode, size_t smem_limit, int* NS, int* NC) {
  *NS = 0;
  *NC = 0;
  const int max_nc = fp8 ? kScatterMaxConsumers : 2;
  const int max_ns = fp8 ? 32 : 4;
  for (int pass = 0; pass < 2 && *NS == 0; ++pass) {
    // first at least half the consumers (the quantiser's compute), then any
    for (int nc = max_nc; nc >= (pass == 0 ? (max_nc + 1) / 2 : 1); --nc) {
      const size_t fixed = scatter_block_bytes(H, scatter_head_ints(mode, R, E), fp8, 0, nc);
      if (fixed >= smem_limit) continue;
      int ns = static_cast<int>((smem_limit - fixed) / (20 + 2 * static_cast<size_t>(H)));
      if (ns > max_ns) ns = max_ns;
      while (ns >= 2 && scatter_block_bytes(H, scatter_head_ints(mode, R, E), fp8, ns, nc) > smem_limit) --ns;
      ns -= ns % nc;  // consumer c owns the stages s = c (mod nc): see the kernel
      if (ns >= 2 && ns >= nc && ns > *NS) {  // the most stages; more consumers on a tie
        *NS = ns;
        *NC = nc;
      }
    }
  }
}

size_t scatter_smem_bytes(int H, int R, int E, bool fp8, int mode, int NS, int NC) {
  return scatter_block_bytes(H, scatter_head_ints(mode, R, E), fp8, NS, NC);
}

cudaError_t configure_scatter(size_t optin) {
  const void* ks[6] = {reinterpret_cast<const void*>(k_scatter<false, kSrcRanks>),
                       reinterpret_cast<const void*>(k_scatter<true, kSrcRanks>),
                       reinterpret_cast<const void*>(k_scatter<false, kSrcLowLatency>),
                       reinterpret_cast<const void*>(k_scatter<true, kSrcLowLatency>),
                       reinterpret_cast<const void*>(k_scatter<false, kSrcExpertMajor>),
                       reinterpret_cast<const void*>(k_scatter<true, kSrcExpertMajor>)};
  for (const void* k : ks) {
    cudaError_t e = set_dynamic_smem_limit(k, 0, optin);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Bytes a token moves: its row read, and a row written per destination (at
// most kmax ranks, or k entries).
long long row_bytes_per_token(int H, int k, int kmax, bool fp8, int mode) {
  const long long out_row = fp8 ? static_cast<long long>(H) + 4LL * (H / 128) : 2LL * H;
  return 2LL * H + static_cast<long long>(mode == kSrcRanks ? kmax : k) * out_row;
}

void launch_scatter(const ScatterArgs& args, bool fp8, int mode, int blocks, int NS, int NC, cudaStream_t stream) {
  ScatterArgs a = args;
  a.claim_tokens = claim_tokens_for(row_bytes_per_token(a.H, a.k, a.kmax, fp8, mode), 0);
  const size_t smem = scatter_block_bytes(a.H, scatter_head_ints(mode, a.R, a.E), fp8, NS, NC);
  const dim3 grid(blocks), block((NC + 1) * 32);
  if (mode == kSrcLowLatency) {
    if (fp8)
      (void)launch_kernel(k_scatter<true, kSrcLowLatency>, grid, block, smem, stream, a, NS);
    else
      (void)launch_kernel(k_scatter<false, kSrcLowLatency>, grid, block, smem, stream, a, NS);
  } else if (mode == kSrcExpertMajor) {
    if (fp8)
      (void)launch_kernel(k_scatter<true, kSrcExpertMajor>, grid, block, smem, stream, a, NS);
    else
      (void)launch_kernel(k_scatter<false, kSrcExpertMajor>, grid, block, smem, stream, a, NS);
  } else {
    if (fp8)
      (void)launch_kernel(k_scatter<true, kSrcRanks>, grid, block, smem, stream, a, NS);
    else
      (void)launch_kernel(k_scatter<false, kSrcRanks>, grid, block, smem, stream, a, NS);
  }
}

}  // namespace ep
