// Row quantisation helpers shared by the TMA scatter kernels (k_scatter and
// the fused routing + scatter kernel).
#pragma once

#include "device_common.cuh"

namespace ep {

// Named barrier 1 among the consumer warps (warps 1..NC) of a block.
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" : : "r"(nthreads) : "memory");
}


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

}  // namespace ep
