// One warp moves one token row to all of its destination rows: the row is
// read from HBM once, optionally quantised to FP8 once, and stored to every
// destination ("DeepEP 要約" section 1: FP8 dispatch / BF16 combine; the
// per-token, per-128-channel scale is the workload's recipe).
//
// Lane mapping: pass `it` of a segment covers channels [it*512, it*512+512);
// lane l owns the 16 consecutive channels starting at it*512 + 16*l, i.e. two
// 16-byte bf16 loads and one 16-byte e4m3 store.  Eight consecutive lanes
// hold one 128-channel scale group, so a group's amax is three xor-shuffles.
// A segment keeps kSeg passes (4096 channels) in registers.
#pragma once

#include "device_common.cuh"

namespace ep {

constexpr int kSeg = 8;

// FP8 quantisation of 16 consecutive channels (a: channels 0-7, b: 8-15)
// whose 128-channel group spans this lane and its 7 neighbours.  Returns the
// e4m3 bytes; *scale_out gets the group's scale.
//   a = max(max |x|, 1e-4);  scale = a / 448;  q = e4m3_rn_satfinite(x * (448 / a))
// with one RN division each and one RN multiply per element.
__device__ __forceinline__ uint4 quantize16(const uint4& a, const uint4& b, float* scale_out) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  m = fmaxf(m, __shfl_xor_sync(kFullMask, m, 1));
  m = fmaxf(m, __shfl_xor_sync(kFullMask, m, 2));
  m = fmaxf(m, __shfl_xor_sync(kFullMask, m, 4));
  const float amax = fmaxf(m, 1e-4f);
  *scale_out = __fdiv_rn(amax, 448.0f);
  const float inv = __fdiv_rn(448.0f, amax);
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = pack_e4m3x2(__fmul_rn(bf16_lo(w[2 * i]), inv), __fmul_rn(bf16_hi(w[2 * i]), inv));
    const uint32_t hi =
        pack_e4m3x2(__fmul_rn(bf16_lo(w[2 * i + 1]), inv), __fmul_rn(bf16_hi(w[2 * i + 1]), inv));
    q[i] = lo | (hi << 16);
  }
  return make_uint4(q[0], q[1], q[2], q[3]);
}

// dmask: lanes whose `my_row` is a destination row (>= 0).  wscale: this
// warp's shared-memory staging area for kSeg*4 scales.
template <bool kFP8>
__device__ __forceinline__ void scatter_row(const uint16_t* __restrict__ xrow, int H, unsigned dmask,
                                            long long my_row, void* __restrict__ recv_x,
                                            float* __restrict__ recv_scales, float* wscale, int lane) {
  const int G = H >> 7;
  for (int seg = 0; seg < H; seg += kSeg * 512) {
    uint4 a[kSeg], b[kSeg];
#pragma unroll
    for (int it = 0; it < kSeg; ++it) {
      const int ch = seg + it * 512 + lane * 16;
      if (ch < H) {
        a[it] = ld_stream(xrow + ch);
        b[it] = ld_stream(xrow + ch + 8);
      } else {
        a[it] = make_uint4(0, 0, 0, 0);
        b[it] = make_uint4(0, 0, 0, 0);
      }
    }
    if (kFP8) {
      uint4 q[kSeg];
#pragma unroll
      for (int it = 0; it < kSeg; ++it) {
        if (seg + it * 512 < H) {  // warp-uniform
          float sc;
          q[it] = quantize16(a[it], b[it], &sc);
          if ((lane & 7) == 0) wscale[it * 4 + (lane >> 3)] = sc;
        }
      }
      __syncwarp();
      const int g0 = seg >> 7;
      const int ng = min(kSeg * 4, G - g0);
      unsigned m = dmask;
      while (m) {
        const int sl = __ffs(m) - 1;
        m &= m - 1;
        const long long row = __shfl_sync(kFullMask, my_row, sl);
        uint8_t* dst = static_cast<uint8_t*>(recv_x) + row * H;
#pragma unroll
        for (int it = 0; it < kSeg; ++it) {
          const int ch = seg + it * 512 + lane * 16;
          if (ch < H) st_na(dst + ch, q[it]);
        }
        if (lane < ng) recv_scales[row * G + g0 + lane] = wscale[lane];
      }
      __syncwarp();
    } else {
      unsigned m = dmask;
      while (m) {
        const int sl = __ffs(m) - 1;
        m &= m - 1;
        const long long row = __shfl_sync(kFullMask, my_row, sl);
        uint16_t* dst = static_cast<uint16_t*>(recv_x) + row * H;
#pragma unroll
        for (int it = 0; it < kSeg; ++it) {
          const int ch = seg + it * 512 + lane * 16;
          if (ch < H) {
            st_na(dst + ch, a[it]);
            st_na(dst + ch + 8, b[it]);
          }
        }
      }
    }
  }
}

}  // namespace ep
