// combine on sm_103a, every receive layout -- "DeepEP 要約" (stakiran.github.io)
// section 3: combine(y, handle) and low_latency_combine; the vi.news.hada.io
// DeepEP article, "Mẫu sử dụng cho huấn luyện, prefill và decoding": combine
// reduces the expert outputs back to the originating rank, and its backward
// is a dispatch.
//
//  rank-major (normal):  out[t] = bf16( sum over t's destination ranks,
//                ascending, of v(row) ), from +0.0 with RN adds, where v is
//                the bf16 row widened, or an e4m3 row decoded and multiplied
//                by its 128-channel group's scale (one RN multiply).
//                Optionally also combined_w[t][j] = sum over the same rows,
//                same order, of recv_w[row][j] (the top-k weights' reduction
//                for the backward of the weights);
//  low latency:  out[t] = bf16( acc ), acc = fmaf(w_j, fp32(y[row_j]), acc)
//                over t's unmasked entries in ascending expert id (k-index
//                breaks ties), from +0.0;
//  expert-major: out[t] = bf16( sum of fp32(y[row_j]) ) over t's unmasked
//                entries in ascending expert id, from +0.0 with RN adds.
//
// HBM-bound gather-reduce.  Two blocks per SM (at most 128 registers a
// thread), three for the e4m3 input (at most 85): its dequantisation makes it
// latency-bound with fewer warps (148 us with one block, 101.6 with two, 92.9
// with three on the V3 shape).  Work is split into (token, 1024-channel part)
// items dealt round-robin to the warps of a persistent grid, so the last
// round leaves few warps idle.  A warp takes a part one slab at a time (512
// bf16 or 1024 e4m3 channels) and requests every source row of the slab
// before summing any, so up to kMaxSrc x 1 KB is in flight per warp; for
// bf16 sources it first asks L2 for the rest of each source's part (a bulk
// prefetch), which keeps tokens with few sources from starving HBM (combine
// 102.4 -> 99.3 us on the group-limited V3 shape, unchanged on uniform V3).
// e4m3 sources pass through a ring of three register buffers instead: the
// loads of the next two sources are in flight while one is decoded and
// summed (84.5 -> 82.0 us back to back on the V3 shape, against two-at-a-time
// batches with an L2 prefetch of the next two).  Per item, the sources are
// put in summation order through a 32-slot shared table per warp (one store
// and one load a lane, not a ballot per source), and a warp steps to its next
// item's (token, part) with a carry instead of a 64-bit division: 7 % fewer
// instructions in the issue-bound e4m3 combine (81.9 -> 75.5 us back to
// back), bf16 combine 120.5 -> 118.2 us.
#include <climits>

#include "device_common.cuh"
#include "ep_internal.h"

namespace ep {

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;
constexpr int kChunks = 2;   // 16-byte chunks per lane per slab
constexpr int kMaxSrc = 8;   // source rows loaded together
constexpr int kPartChannels = 1024;  // channels of one work item

// Four e4m3 codes (low byte first) -> four floats; exact (every e4m3 value
// is an f16 value, and every f16 value an f32 value).  The word is split into
// its 16-bit halves inside the asm, which saves a mask and a shift per pair
// (e4m3-input combine 92.3 -> 89.7 us on the V3 shape: it is issue-bound).
__device__ __forceinline__ void e4m3x4_to_float4(uint32_t w, float& f0, float& f1, float& f2, float& f3) {
  asm("{\n\t.reg .b16 lo, hi, a, b, c, d;\n\t.reg .b32 p0, p1;\n\t"
      "mov.b32 {lo, hi}, %4;\n\t"
      "cvt.rn.f16x2.e4m3x2 p0, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 p1, hi;\n\t"
      "mov.b32 {a, b}, p0;\n\t"
      "mov.b32 {c, d}, p1;\n\t"
      "cvt.f32.f16 %0, a;\n\t"
      "cvt.f32.f16 %1, b;\n\t"
      "cvt.f32.f16 %2, c;\n\t"
      "cvt.f32.f16 %3, d;\n\t}"
      : "=f"(f0), "=f"(f1), "=f"(f2), "=f"(f3)
      : "r"(w));
}

// (a0, a1) += (p0, p1) * s: two RN multiplies, then two RN adds.  Scalar
// intrinsics on purpose: a packed mul.rn.f32x2 followed by add.rn.f32x2 was
// measured to come out as a fused multiply-add (one rounding), which is not
// this sum; a packed multiply with scalar adds, or scalar multiplies with a
// packed add, keep both roundings but were no faster.
__device__ __forceinline__ void add_scaled2(float& a0, float& a1, float p0, float p1, float s) {
  a0 = __fadd_rn(a0, __fmul_rn(p0, s));
  a1 = __fadd_rn(a1, __fmul_rn(p1, s));
}

// One e4m3 source's slab in registers: kChunks 16-byte chunks of codes per
// lane and each chunk's 128-channel group scale.
struct E4m3Slab {
  uint4 q[kChunks];
  float s[kChunks];
};

// Loads the j-th source's slab (lane j of srow holds its row) when j < n.
// j and n are warp-uniform: the whole warp takes the shuffle or none of it.
__device__ __forceinline__ void load_e4m3_slab(E4m3Slab& b, const CombineArgs& a, long long srow, int j, int n,
                                               int h0, int h_end, int lane) {
  if (j >= n) return;
  const long long r = __shfl_sync(kFullMask, srow, j & 31);
  const uint8_t* yq = static_cast<const uint8_t*>(a.y) + r * a.H;
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int ch = h0 + (c * 32 + lane) * 16;
    b.q[c] = ch < h_end ? ld_stream(yq + ch) : make_uint4(0, 0, 0, 0);
    b.s[c] = ch < h_end ? __ldg(a.y_scales + r * (a.H >> 7) + (ch >> 7)) : 0.0f;
  }
}

// acc += decode(b) * scale, channel by channel, when j < n.
__device__ __forceinline__ void add_e4m3_slab(float (&acc)[kChunks][16], const E4m3Slab& b, int j, int n) {
  if (j >= n) return;
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const uint32_t q[4] = {b.q[c].x, b.q[c].y, b.q[c].z, b.q[c].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f0, f1, f2, f3;
      e4m3x4_to_float4(q[i], f0, f1, f2, f3);
      add_scaled2(acc[c][4 * i], acc[c][4 * i + 1], f0, f1, b.s[c]);
      add_scaled2(acc[c][4 * i + 2], acc[c][4 * i + 3], f2, f3, b.s[c]);
    }
  }
}

template <int kSrc, bool kFP8>
__global__ void __launch_bounds__(kCombineThreads, kFP8 ? 3 : 2) k_combine(CombineArgs a) {
  extern __shared__ int base_smem[];  // rank_offset [R+1] or expert_offset [E+1]
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nw = gridDim.x * kCombineWarps;
  const unsigned lt = lanemask_lt();
  if (kSrc == kSrcRanks) {
    for (int r = threadIdx.x; r <= a.R; r += kCombineThreads) base_smem[r] = a.rank_offset[r];
    __syncthreads();
  } else if (kSrc == kSrcExpertMajor) {
    for (int e = threadIdx.x; e <= a.E; e += kCombineThreads) base_smem[e] = a.expert_offset[e];
    __syncthreads();
  }
  // a warp's sources, compacted into summation order
  __shared__ long long s_row[kCombineWarps][32];
  __shared__ float s_w[kCombineWarps][32];
  // item i = (token i / parts, part i % parts); warp w takes items w, w + nw,
  // ..., stepping (token, part) by (dq, dr) with a carry instead of dividing
  const int parts = (a.H + kPartChannels - 1) / kPartChannels;
  const int first = blockIdx.x * kCombineWarps + warp;
  const int dq = nw / parts, dr = nw - dq * parts;
  int t = first / parts, part = first - t * parts;
  for (; t < a.T;) {
    long long row = -1;
    float w = 0.0f;
    int key = INT_MAX;
    if (kSrc == kSrcRanks) {
      if (lane < a.kmax) {
        const int2 d = a.dst[static_cast<size_t>(t) * a.kmax + lane];
        if (d.x >= 0) row = static_cast<long long>(base_smem[d.x]) + d.y;
      }
    } else if (lane < a.k) {
      const int e = a.ent_idx[static_cast<size_t>(t) * a.k + lane];
      const int s = a.ent_slot[static_cast<size_t>(t) * a.k + lane];
      if (e >= 0 && s >= 0) {
        row = kSrc == kSrcLowLatency ? static_cast<long long>(e) * a.M + s : static_cast<long long>(base_smem[e]) + s;
        if (kSrc == kSrcLowLatency) w = a.topk_weights[static_cast<size_t>(t) * a.k + lane];
        key = e;
      }
    }
    if (row >= a.y_rows) {
      latch_error(a.err, kErrCapacity);
      row = -1;
      key = INT_MAX;
    }
    const bool valid = row >= 0;
    const unsigned vmask = __ballot_sync(kFullMask, valid);
    const int n = __popc(vmask);
    // summation position of this lane's source
    int pos;
    if (kSrc == kSrcRanks) {
      pos = __popc(vmask & lt);  // the destination list is in ascending rank
    } else {
      pos = 0;
      for (int jj = 0; jj < a.k; ++jj) {
        const int kj = __shfl_sync(kFullMask, key, jj);
        pos += (kj < key || (kj == key && jj < lane)) ? 1 : 0;
      }
    }
    // lane s receives the s-th source's row (and weight); the valid lanes'
    // positions are distinct, so each slot below n is written once
    if (valid) {
      s_row[warp][pos] = row;
      if (kSrc == kSrcLowLatency) s_w[warp][pos] = w;
    }
    __syncwarp();
    const long long srow = lane < n ? s_row[warp][lane] : -1;
    const float sw = kSrc == kSrcLowLatency && lane < n ? s_w[warp][lane] : 0.0f;
    __syncwarp();  // read before the next item writes

    if (kSrc == kSrcRanks && a.recv_topk_weights && part == 0) {
      // the top-k weights, column `lane`, summed over the same rows in order
      float ws = 0.0f;
      for (int s = 0; s < n; ++s) {
        const long long r_ = __shfl_sync(kFullMask, srow, s);
        if (lane < a.k) ws = __fadd_rn(ws, a.recv_topk_weights[r_ * a.k + lane]);
      }
      if (lane < a.k) a.combined_topk_weights[static_cast<size_t>(t) * a.k + lane] = ws;
    }

    uint16_t* out = a.out + static_cast<size_t>(t) * a.H;
    const int h_end = min(a.H, (part + 1) * kPartChannels);
    constexpr int kLaneCh = kFP8 ? 16 : 8;  // channels per 16-byte chunk
    constexpr int kSlab = 32 * kChunks * kLaneCh;
    if (!kFP8 && part * kPartChannels + kSlab < h_end && lane < n) {
      // bf16 sources: lane s asks L2 for the rest of the s-th source row's
      // part while the first slab streams in (one bulk prefetch: 16-byte
      // aligned, since y is and H is a multiple of 128), so a token with few
      // sources still keeps enough bytes in flight
      const uint16_t* yb = static_cast<const uint16_t*>(a.y);
      const int h1 = part * kPartChannels + kSlab;
      prefetch_l2_bulk(yb + srow * a.H + h1, static_cast<uint32_t>(h_end - h1) * 2u);
    }
    for (int h0 = part * kPartChannels; h0 < h_end; h0 += 32 * kChunks * kLaneCh) {
      float acc[kChunks][kLaneCh];
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
#pragma unroll
        for (int i = 0; i < kLaneCh; ++i) acc[c][i] = 0.0f;
      if constexpr (kFP8) {
        // ring of three: sources j+1 and j+2 are loading while j is summed
        E4m3Slab b0, b1, b2;
        load_e4m3_slab(b0, a, srow, 0, n, h0, h_end, lane);
        load_e4m3_slab(b1, a, srow, 1, n, h0, h_end, lane);
        for (int j = 0; j < n; j += 3) {
          load_e4m3_slab(b2, a, srow, j + 2, n, h0, h_end, lane);
          add_e4m3_slab(acc, b0, j, n);
          if (j + 1 >= n) break;
          load_e4m3_slab(b0, a, srow, j + 3, n, h0, h_end, lane);
          add_e4m3_slab(acc, b1, j + 1, n);
          if (j + 2 >= n) break;
          load_e4m3_slab(b1, a, srow, j + 4, n, h0, h_end, lane);
          add_e4m3_slab(acc, b2, j + 2, n);
        }
      } else {
        // bf16 sources: all of a slab's source rows requested before any is summed
        for (int sb = 0; sb < n; sb += kMaxSrc) {
          uint4 v[kMaxSrc][kChunks];
#pragma unroll
          for (int s = 0; s < kMaxSrc; ++s) {
            const long long r_ = __shfl_sync(kFullMask, srow, (sb + s) & 31);
            if (sb + s < n) {
              const uint16_t* yb = static_cast<const uint16_t*>(a.y);
#pragma unroll
              for (int c = 0; c < kChunks; ++c) {
                const int ch = h0 + (c * 32 + lane) * kLaneCh;
                v[s][c] = ch < h_end ? ld_stream(yb + r_ * a.H + ch) : make_uint4(0, 0, 0, 0);
              }
            }
          }
#pragma unroll
          for (int s = 0; s < kMaxSrc; ++s) {
            const float ws = __shfl_sync(kFullMask, sw, (sb + s) & 31);
            if (sb + s < n) {
#pragma unroll
              for (int c = 0; c < kChunks; ++c) {
                const uint32_t q[4] = {v[s][c].x, v[s][c].y, v[s][c].z, v[s][c].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  if (kSrc == kSrcLowLatency) {
                    acc[c][2 * i] = __fmaf_rn(ws, bf16_lo(q[i]), acc[c][2 * i]);
                    acc[c][2 * i + 1] = __fmaf_rn(ws, bf16_hi(q[i]), acc[c][2 * i + 1]);
                  } else {
                    acc[c][2 * i] = __fadd_rn(acc[c][2 * i], bf16_lo(q[i]));
                    acc[c][2 * i + 1] = __fadd_rn(acc[c][2 * i + 1], bf16_hi(q[i]));
                  }
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const int ch = h0 + (c * 32 + lane) * kLaneCh;
        if (ch < h_end) {
#pragma unroll
          for (int half = 0; half < kLaneCh / 8; ++half) {
            const float* f = acc[c] + 8 * half;
            const uint4 o = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                                       pack_bf16x2(f[6], f[7]));
            st_na(out + ch + 8 * half, o);
          }
        }
      }
    }
    part += dr;
    t += dq;
    if (part >= parts) {
      part -= parts;
      ++t;
    }
  }
}

namespace {
const void* combine_fn(int src, bool fp8) {
  if (src == kSrcRanks)
    return fp8 ? reinterpret_cast<const void*>(k_combine<kSrcRanks, true>)
               : reinterpret_cast<const void*>(k_combine<kSrcRanks, false>);
  if (src == kSrcLowLatency) return reinterpret_cast<const void*>(k_combine<kSrcLowLatency, false>);
  return reinterpret_cast<const void*>(k_combine<kSrcExpertMajor, false>);
}
}  // namespace

size_t combine_smem_bytes(int src, int R, int E) {
  return src == kSrcRanks ? 4 * static_cast<size_t>(R + 1) : src == kSrcExpertMajor ? 4 * static_cast<size_t>(E + 1) : 0;
}

void launch_combine(const CombineArgs& a, int src, bool fp8, int blocks, cudaStream_t stream) {
  const size_t smem = combine_smem_bytes(src, a.R, a.E);
  if (src == kSrcRanks) {
    if (fp8)
      (void)launch_kernel(k_combine<kSrcRanks, true>, dim3(blocks), dim3(kCombineThreads), smem, stream, a);
    else
      (void)launch_kernel(k_combine<kSrcRanks, false>, dim3(blocks), dim3(kCombineThreads), smem, stream, a);
  } else if (src == kSrcLowLatency) {
    (void)launch_kernel(k_combine<kSrcLowLatency, false>, dim3(blocks), dim3(kCombineThreads), smem, stream, a);
  } else {
    (void)launch_kernel(k_combine<kSrcExpertMajor, false>, dim3(blocks), dim3(kCombineThreads), smem, stream, a);
  }
}

int combine_threads() { return kCombineThreads; }

const void* combine_kernel(int src, bool fp8) { return combine_fn(src, fp8); }

}  // namespace ep
