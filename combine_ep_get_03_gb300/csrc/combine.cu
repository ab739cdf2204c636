// combine on sm_103a, both modes -- "DeepEP 要約" (stakiran.github.io)
// section 3: combine(y, handle) and low_latency_combine; the vi.news.hada.io
// DeepEP article: combine reduces the expert outputs back to the
// originating rank.
//
//  normal:       out[t] = bf16( sum over t's destination ranks, ascending,
//                of fp32(y[row]) ), accumulated from +0.0 with RN adds;
//  low latency:  out[t] = bf16( acc ), acc = fmaf(w_j, fp32(y[row_j]), acc)
//                over t's unmasked entries in ascending expert id (k-index
//                breaks ties), from +0.0.
//
// HBM-bound gather-reduce.  Work is split into (token, 1024-channel part)
// items dealt round-robin to the warps of a persistent grid, so the last
// round leaves few warps idle.  A warp takes a part 512 channels at a time
// and requests every source row of the slab before summing any, so up to
// kMaxSrc x 1 KB is in flight per warp.
#include <climits>

#include "device_common.cuh"
#include "ep_internal.h"

namespace ep {

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;
constexpr int kChunks = 2;   // 16-byte chunks per lane per slab: slab = 32 * 2 * 8 = 512 channels
constexpr int kMaxSrc = 8;   // source rows loaded together
constexpr int kPartChannels = 1024;  // channels of one work item
constexpr int kMaxCachedRanks = 1024;

template <bool kLL>
__global__ void __launch_bounds__(kCombineThreads) k_combine(CombineArgs a) {
  __shared__ int so[kMaxCachedRanks + 1];  // rank_offset (normal mode)
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nw = gridDim.x * kCombineWarps;
  const unsigned lt = lanemask_lt();
  if (!kLL) {
    for (int r = threadIdx.x; r <= a.R; r += kCombineThreads) so[r] = a.rank_offset[r];
    __syncthreads();
  }
  const int parts = (a.H + kPartChannels - 1) / kPartChannels;
  const long long items = static_cast<long long>(a.T) * parts;
  for (long long item = blockIdx.x * kCombineWarps + warp; item < items; item += nw) {
    const int t = static_cast<int>(item / parts);
    const int part = static_cast<int>(item - static_cast<long long>(t) * parts);
    long long row = -1;
    float w = 0.0f;
    int key = INT_MAX;
    if (!kLL) {
      if (lane < a.kmax) {
        const int2 d = a.dst[static_cast<size_t>(t) * a.kmax + lane];
        if (d.x >= 0) row = static_cast<long long>(so[d.x]) + d.y;
      }
    } else if (lane < a.k) {
      const int e = a.ll_idx[static_cast<size_t>(t) * a.k + lane];
      const int s = a.ll_slot[static_cast<size_t>(t) * a.k + lane];
      if (e >= 0 && s >= 0) {
        row = static_cast<long long>(e) * a.M + s;
        w = a.topk_weights[static_cast<size_t>(t) * a.k + lane];
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
    if (!kLL) {
      pos = __popc(vmask & lt);  // the destination list is in ascending rank
    } else {
      pos = 0;
      for (int jj = 0; jj < a.k; ++jj) {
        const int kj = __shfl_sync(kFullMask, key, jj);
        pos += (kj < key || (kj == key && jj < lane)) ? 1 : 0;
      }
    }
    // lane s receives the s-th source's row (and weight)
    int from = 0;
    for (int s = 0; s < n; ++s) {
      const unsigned b = __ballot_sync(kFullMask, valid && pos == s);
      if (lane == s) from = __ffs(b) - 1;
    }
    const long long srow = __shfl_sync(kFullMask, row, from);
    const float sw = __shfl_sync(kFullMask, w, from);

    const uint16_t* y = a.y;
    uint16_t* out = a.out + static_cast<size_t>(t) * a.H;
    const int h_end = min(a.H, (part + 1) * kPartChannels);
    for (int h0 = part * kPartChannels; h0 < h_end; h0 += 32 * kChunks * 8) {
      float acc[kChunks][8];
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[c][i] = 0.0f;
      for (int sb = 0; sb < n; sb += kMaxSrc) {
        uint4 v[kMaxSrc][kChunks];
#pragma unroll
        for (int s = 0; s < kMaxSrc; ++s) {
          const long long r_ = __shfl_sync(kFullMask, srow, (sb + s) & 31);
          if (sb + s < n) {
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
              const int ch = h0 + (c * 32 + lane) * 8;
              v[s][c] = ch < h_end ? ld_stream(y + r_ * a.H + ch) : make_uint4(0, 0, 0, 0);
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
                if (kLL) {
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
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const int ch = h0 + (c * 32 + lane) * 8;
        if (ch < h_end) {
          const uint4 o = make_uint4(pack_bf16x2(acc[c][0], acc[c][1]), pack_bf16x2(acc[c][2], acc[c][3]),
                                     pack_bf16x2(acc[c][4], acc[c][5]), pack_bf16x2(acc[c][6], acc[c][7]));
          st_na(out + ch, o);
        }
      }
    }
  }
}

void launch_combine(const CombineArgs& a, bool low_latency, int blocks, cudaStream_t stream) {
  if (low_latency)
    (void)launch_kernel(k_combine<true>, dim3(blocks), dim3(kCombineThreads), 0, stream, a);
  else
    (void)launch_kernel(k_combine<false>, dim3(blocks), dim3(kCombineThreads), 0, stream, a);
}

int combine_threads() { return kCombineThreads; }

const void* combine_kernel(bool low_latency) {
  return low_latency ? reinterpret_cast<const void*>(k_combine<true>)
                     : reinterpret_cast<const void*>(k_combine<false>);
}

}  // namespace ep
