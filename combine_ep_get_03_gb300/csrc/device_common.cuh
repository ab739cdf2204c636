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

// Asks L2 to fetch [p, p + bytes) (p 16-byte aligned, bytes a multiple of
// 16); nothing waits for it.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" : : "l"(p), "r"(bytes) : "memory");
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

// ------------------------------------------------------------------ bulk copies
//
// Untiled TMA ("bulk") copies between global and shared memory.  Sizes are
// multiples of 16 bytes and both addresses 16-byte aligned.  A load completes
// on an mbarrier (transaction bytes); stores are tracked per issuing thread
// in bulk groups.

namespace ep {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" : : "r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make the initialised barriers visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" : : : "memory");
}

__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" : : "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" : : "r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" : : "r"(smem_u32(bar)) : "memory");
}

// Bounded wait for the phase with parity `parity` to complete.  Returns
// false (and latches kErrTimeout) if it does not within the poll limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  const uint32_t addr = smem_u32(bar);
  for (int it = 0; it < kSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if (it >= 16) __nanosleep(64);
  }
  latch_error(err, kErrTimeout);
  return false;
}

// A 4-byte store that the L2 keeps ahead of streaming data (evict_last).
// For metadata scattered one word per row: the 32-byte sector of such a word
// is completed by other rows written much later, and a sector evicted half
// written costs the DRAM a read-modify-write.
__device__ __forceinline__ void st_keep(float* p, float v) {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" : : "l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep(int* p, int v) {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  asm volatile("st.global.L2::cache_hint.s32 [%0], %1, %2;" : : "l"(p), "r"(v), "l"(pol) : "memory");
}

// Expert id i of a top-k table held as int64 (ids32 == 0) or int32.
__device__ __forceinline__ long long load_topk_id(const void* topk_idx, long long i, int ids32) {
  return ids32 ? static_cast<long long>(static_cast<const int*>(topk_idx)[i])
               : static_cast<const long long*>(topk_idx)[i];
}

// global -> shared, completing `bytes` transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :
      : "r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// shared -> global, in the issuing thread's current bulk group.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               :
               : "l"(gmem_dst), "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" : : : "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" : : "n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" : : : "memory"); }

// Order this thread's generic-proxy shared-memory writes before later
// asynchronous-proxy (bulk copy) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" : : : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

__device__ __forceinline__ void sts64(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" : : "r"(smem_u32(p)), "r"(a), "r"(b) : "memory");
}

}  // namespace ep
