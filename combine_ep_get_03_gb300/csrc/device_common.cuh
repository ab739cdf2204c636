// Device helpers shared by the sm_103a kernels: status latch, streaming
// 16-byte loads, bf16 / e4m3 conversions and the bounded single-pass
// cross-block scan ("decoupled look-back") flag protocol.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ep {

enum Status : int {
  kOk = 0,
  kErrInvalidArg = 1,
  kErrCuda = 2,
  kErrCapacity = 3,
  kErrBadExpert = 4,
  kErrTimeout = 5,
  kErrState = 6,
};

constexpr unsigned kFullMask = 0xffffffffu;

// First device-side condition wins; later ones are dropped.
__device__ __forceinline__ void latch_error(int* err, int code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// 16-byte load of data that no thread writes while the kernel runs: the
// non-coherent read-only path, no L1 allocation (each byte is used once),
// with a 256-byte L2 prefetch because whole rows are streamed.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// 16-byte store that is not kept in L1.
__device__ __forceinline__ void st_na(void* p, const uint4& v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};"
               :
               : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 -> packed e4m3x2, round to nearest even, saturating to +-448;
// `lo` lands in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------------ look-back
//
// One 64-bit word per (block, column): [63:34] call epoch, [33:32] state
// (1 = the block's own count is published, 2 = its inclusive prefix is),
// [31:0] value.  Words from an earlier call carry another epoch and read as
// "nothing published yet", so the array is never cleared.

constexpr uint32_t kFlagAggregate = 1;
constexpr uint32_t kFlagInclusive = 2;
constexpr int kSpinLimit = 1 << 22;  // ~0.5 s with the back-off below

__device__ __forceinline__ unsigned long long make_flag(uint32_t epoch, uint32_t state, uint32_t v) {
  return (static_cast<unsigned long long>(epoch) << 34) |
         (static_cast<unsigned long long>(state) << 32) | v;
}
__device__ __forceinline__ uint32_t flag_epoch(unsigned long long w) { return static_cast<uint32_t>(w >> 34); }
__device__ __forceinline__ uint32_t flag_state(unsigned long long w) { return static_cast<uint32_t>(w >> 32) & 3u; }
__device__ __forceinline__ uint32_t flag_value(unsigned long long w) { return static_cast<uint32_t>(w); }

__device__ __forceinline__ void flag_store(unsigned long long* p, unsigned long long w) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" : : "l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long flag_load(const unsigned long long* p) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}

// Wait until the word at p carries this epoch with at least `min_state`.
// Gives up after kSpinLimit polls: latches kErrTimeout and returns a word
// with state 0 (callers then treat the value as 0 and stop looking back).
__device__ __forceinline__ unsigned long long flag_wait(const unsigned long long* p, uint32_t epoch,
                                                        uint32_t min_state, int* err) {
  for (int it = 0; it < kSpinLimit; ++it) {
    unsigned long long w = flag_load(p);
    if (flag_epoch(w) == epoch && flag_state(w) >= min_state) return w;
    if (it >= 16) __nanosleep(it < 1024 ? 32 : 128);
  }
  latch_error(err, kErrTimeout);
  return 0ull;
}

}  // namespace ep
