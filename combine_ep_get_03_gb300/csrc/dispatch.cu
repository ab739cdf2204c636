// dispatch, normal mode, on sm_103a: scatter each token to the receive rows
// the layout assigned it, BF16 copy or fused FP8 quantisation, plus the
// per-row metadata (source token, expert ids made local to the receiving
// rank, weights) -- "DeepEP 要約" (stakiran.github.io) section 3;
// "Как DeepSeek разогнали обмен данными ..." (devtrends.ru), "Как это
// выглядит в коде".
//
// HBM-bound: each token row is read once (2H bytes) and written once per
// destination rank.  One warp per token, persistent grid sized to the SMs
// the caller grants.
#include "ep_internal.h"
#include "scatter.cuh"

namespace ep {

constexpr int kDispatchThreads = 256;
constexpr int kDispatchWarps = kDispatchThreads / 32;

template <bool kFP8>
__global__ void __launch_bounds__(kDispatchThreads, 2) k_dispatch(DispatchArgs a) {
  __shared__ float sscale[kDispatchWarps][kSeg * 4];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nw = gridDim.x * kDispatchWarps;
  const bool meta = a.recv_src_idx || a.recv_topk_idx || a.recv_topk_weights;
  for (int t = blockIdx.x * kDispatchWarps + warp; t < a.T; t += nw) {
    long long row = -1;
    int r = -1;
    if (lane < a.kmax) {
      const int2 d = a.dst[static_cast<size_t>(t) * a.kmax + lane];
      if (d.x >= 0) {
        r = d.x;
        row = static_cast<long long>(a.rank_offset[d.x]) + d.y;
        if (row >= a.cap) {
          latch_error(a.err, kErrCapacity);
          row = -1;
        }
      }
    }
    int e = -1;
    float w = 0.0f;
    if (meta && lane < a.k) {
      e = a.idx32[static_cast<size_t>(t) * a.k + lane];
      if (a.topk_weights) w = a.topk_weights[static_cast<size_t>(t) * a.k + lane];
    }
    const unsigned dmask = __ballot_sync(kFullMask, row >= 0);
    scatter_row<kFP8>(a.x + static_cast<size_t>(t) * a.H, a.H, dmask, row, a.recv_x, a.recv_scales,
                      sscale[warp], lane);
    if (meta) {
      unsigned m = dmask;
      while (m) {
        const int sl = __ffs(m) - 1;
        m &= m - 1;
        const long long rrow = __shfl_sync(kFullMask, row, sl);
        const int rr = __shfl_sync(kFullMask, r, sl);
        if (lane == 0 && a.recv_src_idx) a.recv_src_idx[rrow] = t;
        if (lane < a.k) {
          const bool here = e >= 0 && e / a.El == rr;
          if (a.recv_topk_idx) a.recv_topk_idx[rrow * a.k + lane] = here ? e - rr * a.El : -1;
          if (a.recv_topk_weights) a.recv_topk_weights[rrow * a.k + lane] = here ? w : 0.0f;
        }
      }
    }
  }
}

void launch_dispatch(const DispatchArgs& a, bool fp8, int blocks, cudaStream_t stream) {
  if (fp8)
    (void)launch_kernel(k_dispatch<true>, dim3(blocks), dim3(kDispatchThreads), 0, stream, a);
  else
    (void)launch_kernel(k_dispatch<false>, dim3(blocks), dim3(kDispatchThreads), 0, stream, a);
}

int dispatch_threads() { return kDispatchThreads; }

const void* dispatch_kernel(bool fp8) {
  return fp8 ? reinterpret_cast<const void*>(k_dispatch<true>) : reinterpret_cast<const void*>(k_dispatch<false>);
}

}  // namespace ep
