// Dispatch's row movement on sm_103a with TMA bulk copies: each warp streams
// its tokens through shared memory -- a bulk load brings a token row in, the
// warp quantises it once to FP8 (or leaves BF16 as is), and one bulk store per
// destination writes it out ("DeepEP 要約" (stakiran.github.io) section 3:
// dispatch and low_latency_dispatch; "DeepSeek выпустила DeepEP V2.5"
// (aikraft.ru), "Технические детали и требования": FP8 dispatch).
//
// HBM-bound: the row is read once (2H bytes) and written once per
// destination.  The bytes in flight are bounded by shared memory, not by
// registers: every warp keeps its next rows' loads in flight while it
// quantises and stores the current one.
//
// Destinations:  normal  -- the handle's (rank, row-in-rank) list + the
//                           rank's region offset (the layout's output);
//                low latency -- expert e's row `slot` in [E][M][H].
//
// FP8: a lane quantises whole 128-channel groups (quantize_row_smem), so a
// token row costs one warp-wide pair of divisions per 32 groups and no
// shuffles.
#include "device_common.cuh"
#include "ep_internal.h"

namespace ep {

// Each warp's region starts with its mbarriers (8 bytes each), padded to 16.
constexpr size_t kScatterBarBytes = 32;
static_assert(8 * kScatterLoadsFp8 <= kScatterBarBytes && 8 * kScatterLoadsBf16 <= kScatterBarBytes,
              "every row buffer needs its own mbarrier inside the warp's barrier area");

__host__ __device__ inline size_t scatter_warp_bytes(int H, bool fp8) {
  const size_t G = static_cast<size_t>(H) / 128;
  if (fp8)
    return kScatterBarBytes + kScatterLoadsFp8 * 2 * static_cast<size_t>(H) +
           kScatterQBufs * (H + ((4 * G + 15) & ~15ull));
  return kScatterBarBytes + kScatterLoadsBf16 * 2 * static_cast<size_t>(H);
}

__host__ __device__ inline size_t scatter_head_bytes(int R) { return (static_cast<size_t>(R + 1) * 4 + 15) & ~15ull; }

// Largest |x| of 8 bf16 values, accumulated in packed form: with the sign
// bits cleared, bf16 values compare like their bit patterns, and max.bf16x2
// selects exactly.
__device__ __forceinline__ uint32_t absmax8_acc(uint32_t m, const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) asm("max.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(w[i] & 0x7fff7fffu));
  return m;
}

// 8 bf16 * inv -> 8 e4m3 bytes (two words): each product is one RN fp32
// multiply (two per packed mul.rn.f32x2), then one RN-even saturating
// conversion.
__device__ __forceinline__ uint2 quant8(const uint4& v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  unsigned long long iv;
  asm("mov.b64 %0, {%1, %1};" : "=l"(iv) : "f"(inv));
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    unsigned long long p, r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(bf16_lo(w[i])), "f"(bf16_hi(w[i])));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(p), "l"(iv));
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
    h[i] = pack_e4m3x2(lo, hi);
  }
  return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

// Quantise one token row (bf16 in shared memory) to e4m3 + one fp32 scale per
// 128 channels.  Lane l owns whole groups g = l, l+32, ...: it reads the
// group's 16 chunks of 16 bytes, takes their amax, computes
//   a = max(amax, 1e-4);  scale = a / 448;  inv = 448 / a   (IEEE RN divisions)
// and writes q = e4m3_rn_satfinite(x * inv).  The chunk order is rotated by
// the lane so that a warp's reads (16 B) and writes (8 B) spread evenly over
// the shared-memory banks.
__device__ __forceinline__ void quantize_row_smem(const unsigned char* x, unsigned char* q, float* scales, int G,
                                                  int lane) {
  for (int g0 = 0; g0 < G; g0 += 32) {
    const int g = g0 + lane;
    if (g < G) {
      const unsigned char* src = x + static_cast<size_t>(g) * 256;
      uint4 v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = lds128(src + (((j + lane) & 15) << 4));
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) m = absmax8_acc(m, v[j]);
      const float a = fmaxf(fmaxf(bf16_lo(m), bf16_hi(m)), 1e-4f);
      scales[g] = __fdiv_rn(a, 448.0f);
      const float inv = __fdiv_rn(448.0f, a);
      unsigned char* dst = q + static_cast<size_t>(g) * 128;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint2 o = quant8(v[j], inv);
        sts64(dst + (((j + lane) & 15) << 3), o.x, o.y);
      }
    }
  }
}

template <bool kFP8, bool kLL>
__global__ void __launch_bounds__(kScatterMaxWarps * 32, 1) k_scatter(ScatterArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int* so = reinterpret_cast<int*>(smem);  // rank_offset (normal mode)
  if (!kLL) {
    for (int r = threadIdx.x; r <= a.R; r += blockDim.x) so[r] = a.rank_offset[r];
    __syncthreads();
  }
  constexpr int NB = kFP8 ? kScatterLoadsFp8 : kScatterLoadsBf16;
  const int H = a.H;
  const int G = H >> 7;
  const uint32_t row_bytes = 2u * static_cast<uint32_t>(H);
  unsigned char* wb = smem + scatter_head_bytes(kLL ? 0 : a.R) + static_cast<size_t>(warp) * scatter_warp_bytes(H, kFP8);
  uint64_t* bar = reinterpret_cast<uint64_t*>(wb);
  unsigned char* xb0 = wb + kScatterBarBytes;
  unsigned char* qb0 = xb0 + static_cast<size_t>(NB) * row_bytes;
  const size_t qstride = static_cast<size_t>(H) + ((4 * G + 15) & ~15);
  auto xb = [&](int b) { return xb0 + static_cast<size_t>(b) * row_bytes; };
  auto qb = [&](int q) { return qb0 + static_cast<size_t>(q) * qstride; };
  auto sc = [&](int q) { return reinterpret_cast<float*>(qb(q) + H); };

  const int gw = blockIdx.x * nw + warp;
  const int total = gridDim.x * nw;
  const int n_my = gw < a.T ? (a.T - gw + total - 1) / total : 0;
  if (lane == 0) {
    for (int b = 0; b < NB; ++b) mbar_init(bar + b, 1);
    mbar_init_fence();
  }
  __syncwarp();
  auto issue_load = [&](int i, int b) {  // lane 0 only
    const int t = gw + i * total;
    mbar_arrive_expect_tx(bar + b, row_bytes);
    bulk_load(xb(b), a.x + static_cast<size_t>(t) * H, row_bytes, bar + b);
  };
  constexpr int ahead = kFP8 ? NB : NB - 1;
  if (lane == 0)
    for (int i = 0; i < ahead && i < n_my; ++i) issue_load(i, i);

  const bool meta = !kLL && (a.recv_src_idx || a.recv_topk_idx || a.recv_topk_weights);
  for (int i = 0; i < n_my; ++i) {
    const int t = gw + i * total;
    const int b = i % NB;
    // destinations of this token (overlaps the row load)
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
      if (ee >= 0 && ss >= 0) row = static_cast<long long>(ee) * a.M + ss;
    }
    const unsigned dmask = __ballot_sync(kFullMask, row >= 0);
    const bool landed = mbar_wait(bar + b, static_cast<uint32_t>((i / NB) & 1), a.err);
    if (!__all_sync(kFullMask, landed)) break;  // gave up (latched): stop this warp's tokens

    const unsigned char* src;
    if (kFP8) {
      const int q = i % kScatterQBufs;
      if (i >= kScatterQBufs) {
        if (lane == 0) bulk_wait_read<kScatterQBufs - 1>();  // qb(q)'s previous stores have read it
        __syncwarp();
      }
      unsigned char* qd = qb(q);
      float* sd = sc(q);
      quantize_row_smem(xb(b), qd, sd, G, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && i + NB < n_my) issue_load(i + NB, b);  // the row buffer is free again
      src = qd;
      unsigned m = dmask;
      while (m) {
        const int sl = __ffs(m) - 1;
        m &= m - 1;
        const long long rr = __shfl_sync(kFullMask, row, sl);
        if (lane == 0) bulk_store(static_cast<uint8_t*>(a.recv_x) + rr * H, src, static_cast<uint32_t>(H));
        for (int g = lane; g < G; g += 32) a.recv_scales[rr * G + g] = sd[g];
      }
      if (lane == 0) bulk_commit();
    } else {
      src = xb(b);
      unsigned m = dmask;
      while (m) {
        const int sl = __ffs(m) - 1;
        m &= m - 1;
        const long long rr = __shfl_sync(kFullMask, row, sl);
        if (lane == 0) bulk_store(static_cast<uint16_t*>(a.recv_x) + rr * H, src, row_bytes);
      }
      if (lane == 0) {
        bulk_commit();
        if (i + NB - 1 < n_my) {
          bulk_wait_read<1>();  // token i-1's stores have read the buffer reloaded next
          issue_load(i + NB - 1, (i + NB - 1) % NB);
        }
      }
      __syncwarp();
    }
    // per-row metadata
    if (meta) {
      unsigned m = dmask;
      while (m) {
        const int sl = __ffs(m) - 1;
        m &= m - 1;
        const long long rr = __shfl_sync(kFullMask, row, sl);
        const int rk = __shfl_sync(kFullMask, r, sl);
        if (lane == 0 && a.recv_src_idx) a.recv_src_idx[rr] = t;
        if (lane < a.k) {
          const bool here = e >= 0 && e / a.El == rk;
          if (a.recv_topk_idx) a.recv_topk_idx[rr * a.k + lane] = here ? e - rk * a.El : -1;
          if (a.recv_topk_weights) a.recv_topk_weights[rr * a.k + lane] = here ? w : 0.0f;
        }
      }
    } else if (kLL && a.recv_src_info && row >= 0) {
      a.recv_src_info[row] = t;
    }
  }
  if (lane == 0) bulk_wait_all();  // stores done before the block's shared memory goes away
  __syncwarp();
}

size_t scatter_smem_bytes(int H, int R, bool fp8, bool low_latency, int warps) {
  return scatter_head_bytes(low_latency ? 0 : R) + static_cast<size_t>(warps) * scatter_warp_bytes(H, fp8);
}

int scatter_warps_for(int H, int R, bool fp8, bool low_latency, size_t smem_limit) {
  int w = kScatterMaxWarps;
  while (w > 0 && scatter_smem_bytes(H, R, fp8, low_latency, w) > smem_limit) --w;
  return w;
}

cudaError_t configure_scatter(size_t smem_limit) {
  const void* ks[4] = {reinterpret_cast<const void*>(k_scatter<false, false>),
                       reinterpret_cast<const void*>(k_scatter<true, false>),
                       reinterpret_cast<const void*>(k_scatter<false, true>),
                       reinterpret_cast<const void*>(k_scatter<true, true>)};
  for (const void* k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_limit));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

void launch_scatter(const ScatterArgs& a, bool fp8, bool low_latency, int blocks, int warps, cudaStream_t stream) {
  const size_t smem = scatter_smem_bytes(a.H, a.R, fp8, low_latency, warps);
  const dim3 grid(blocks), block(warps * 32);
  if (low_latency) {
    if (fp8)
      k_scatter<true, true><<<grid, block, smem, stream>>>(a);
    else
      k_scatter<false, true><<<grid, block, smem, stream>>>(a);
  } else {
    if (fp8)
      k_scatter<true, false><<<grid, block, smem, stream>>>(a);
    else
      k_scatter<false, false><<<grid, block, smem, stream>>>(a);
  }
}

}  // namespace ep
