// TEST INFRASTRUCTURE ONLY -- the oracle spread over the host's cores.
//
// The same definitions as ep_oracle.cpp (included below, so every helper --
// the layout, the FP8 quantiser, the low-latency slots, the number formats --
// is that file's own code), with the outer loop of each row-moving step split
// into contiguous token ranges, one std::thread per range.  Nothing else
// changes: every output element is produced by the same sequence of IEEE
// operations as in the single-threaded functions, so the results are
// byte-identical (a test checks this).  The routing state (layout, slots) is
// formed once, single-threaded, before the threads start.
//
// Partitioning:
//   dispatch / low-latency dispatch -- by source token: a token's destination
//     rows belong to it alone, so the ranges write disjoint rows;
//   combine / low-latency combine   -- by output token.
//
// Used only by the benchmark's CPU-baseline leg and the tests; the product
// path never loads it.

#include <sched.h>

#include <thread>

#include "ep_oracle.cpp"

namespace {

// Runs body(i, t0, t1) for the i-th of `threads` contiguous ranges of [0, T),
// each on its own thread.  Returns the number of ranges.
template <typename Body>
int over_token_ranges(int T, int threads, Body body) {
  if (threads < 1) threads = 1;
  if (threads > T) threads = T > 0 ? T : 1;
  std::vector<std::thread> pool;
  pool.reserve(threads);
  for (int i = 0; i < threads; ++i) {
    const int t0 = static_cast<int>(static_cast<int64_t>(T) * i / threads);
    const int t1 = static_cast<int>(static_cast<int64_t>(T) * (i + 1) / threads);
    pool.emplace_back(body, i, t0, t1);
  }
  for (auto& th : pool) th.join();
  return threads;
}

int clamp_threads(int threads, int T) {
  if (threads < 1) threads = 1;
  if (threads > T) threads = T > 0 ? T : 1;
  return threads;
}

}  // namespace

extern "C" {

// Cores this process may run on (sched_getaffinity), at least 1.
int ref_threads_available() {
  cpu_set_t set;
  CPU_ZERO(&set);
  if (sched_getaffinity(0, sizeof(set), &set) != 0) return 1;
  const int n = CPU_COUNT(&set);
  return n > 0 ? n : 1;
}

int ref_threads_dispatch(int threads, int R, int E, int k, int T, int H, int fp8, const uint16_t* x,
                         const int64_t* topk_idx, const float* topk_weights, int64_t capacity_rows, void* recv_x,
                         float* recv_scales, int* recv_src_idx, int* recv_topk_idx, float* recv_topk_weights) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if (H <= 0 || H % 128 != 0) return kInvalidArg;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  Layout L;
  compute_layout(s, topk_idx, &L);
  const int G = H / 128;
  threads = clamp_threads(threads, T);
  std::vector<char> overflow(threads, 0);
  over_token_ranges(T, threads, [&](int me, int t0, int t1) {
    std::vector<uint8_t> q(H);
    std::vector<float> sc(G);
    for (int t = t0; t < t1; ++t) {
      const uint16_t* xt = x + static_cast<size_t>(t) * H;
      if (fp8) quantize_row(H, xt, q.data(), sc.data());
      for (int r = 0; r < R; ++r) {
        const int sl = L.slot[static_cast<size_t>(t) * R + r];
        if (sl < 0) continue;
        const int64_t row = static_cast<int64_t>(L.rank_offset[r]) + sl;
        if (row >= capacity_rows) {
          overflow[me] = 1;
          continue;
        }
        if (fp8) {
          std::memcpy(static_cast<uint8_t*>(recv_x) + row * H, q.data(), H);
          std::memcpy(recv_scales + row * G, sc.data(), G * sizeof(float));
        } else {
          std::memcpy(static_cast<uint16_t*>(recv_x) + row * H, xt, H * sizeof(uint16_t));
        }
        if (recv_src_idx) recv_src_idx[row] = t;
        for (int j = 0; j < k; ++j) {
          const int64_t e = topk_idx[static_cast<size_t>(t) * k + j];
          const bool local = e >= 0 && e / s.El == r;
          if (recv_topk_idx) recv_topk_idx[row * k + j] = local ? static_cast<int>(e - r * s.El) : -1;
          if (recv_topk_weights && topk_weights)
            recv_topk_weights[row * k + j] = local ? topk_weights[static_cast<size_t>(t) * k + j] : 0.0f;
        }
      }
    }
  });
  for (char o : overflow)
    if (o) return kCapacity;
  return kOk;
}

int ref_threads_combine_ex(int threads, int R, int E, int k, int T, int H, const int64_t* topk_idx, int y_fp8,
                           const void* y, const float* y_scales, int64_t y_rows, const float* recv_topk_weights,
                           uint16_t* out, float* combined_topk_weights) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if (H <= 0 || H % 128 != 0 || (y_fp8 && !y_scales)) return kInvalidArg;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  Layout L;
  compute_layout(s, topk_idx, &L);
  if (L.rank_offset[R] > y_rows) return kCapacity;
  over_token_ranges(T, clamp_threads(threads, T), [&](int, int t0, int t1) {
    for (int t = t0; t < t1; ++t) {
      for (int h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int r = 0; r < R; ++r) {  // ascending rank
          const int sl = L.slot[static_cast<size_t>(t) * R + r];
          if (sl < 0) continue;
          acc = acc + combine_input(y_fp8, y, y_scales, H, static_cast<int64_t>(L.rank_offset[r]) + sl, h);
        }
        out[static_cast<size_t>(t) * H + h] = float_to_bf16_bits_rn(acc);
      }
      if (!combined_topk_weights || !recv_topk_weights) continue;
      for (int j = 0; j < k; ++j) {
        float wsum = 0.0f;
        for (int r = 0; r < R; ++r) {
          const int sl = L.slot[static_cast<size_t>(t) * R + r];
          if (sl < 0) continue;
          wsum = wsum + recv_topk_weights[(static_cast<int64_t>(L.rank_offset[r]) + sl) * k + j];
        }
        combined_topk_weights[static_cast<size_t>(t) * k + j] = wsum;
      }
    }
  });
  return kOk;
}

int ref_threads_combine(int threads, int R, int E, int k, int T, int H, const int64_t* topk_idx, const uint16_t* y,
                        int64_t y_rows, uint16_t* out) {
  return ref_threads_combine_ex(threads, R, E, k, T, H, topk_idx, 0, y, nullptr, y_rows, nullptr, out, nullptr);
}

int ref_threads_ll_dispatch(int threads, int R, int E, int k, int T, int H, int M, int fp8, const uint16_t* x,
                            const int64_t* topk_idx, void* recv_x, float* recv_scales, int* recv_src_info,
                            int* recv_count, int* slot_out) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if (H <= 0 || H % 128 != 0 || M <= 0) return kInvalidArg;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  std::vector<int> slot, count;
  const bool overflow = ll_slots(s, topk_idx, M, &slot, &count);
  const int G = H / 128;
  over_token_ranges(T, clamp_threads(threads, T), [&](int, int t0, int t1) {
    std::vector<uint8_t> q(H);
    std::vector<float> sc(G);
    for (int t = t0; t < t1; ++t) {
      const uint16_t* xt = x + static_cast<size_t>(t) * H;
      if (fp8) quantize_row(H, xt, q.data(), sc.data());
      for (int j = 0; j < k; ++j) {
        const int64_t e = topk_idx[static_cast<size_t>(t) * k + j];
        const int sl = slot[static_cast<size_t>(t) * k + j];
        if (e < 0 || sl < 0) continue;
        const int64_t row = e * M + sl;
        if (fp8) {
          std::memcpy(static_cast<uint8_t*>(recv_x) + row * H, q.data(), H);
          std::memcpy(recv_scales + row * G, sc.data(), G * sizeof(float));
        } else {
          std::memcpy(static_cast<uint16_t*>(recv_x) + row * H, xt, H * sizeof(uint16_t));
        }
        if (recv_src_info) recv_src_info[row] = t;
      }
    }
  });
  if (recv_count)
    for (int e = 0; e < E; ++e) recv_count[e] = count[e] < M ? count[e] : M;
  if (slot_out) std::memcpy(slot_out, slot.data(), slot.size() * sizeof(int));
  return overflow ? kCapacity : kOk;
}

int ref_threads_ll_combine(int threads, int R, int E, int k, int T, int H, int M, const int64_t* topk_idx,
                           const float* topk_weights, const uint16_t* y, uint16_t* out) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if (H <= 0 || H % 128 != 0 || M <= 0) return kInvalidArg;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  std::vector<int> slot, count;
  ll_slots(s, topk_idx, M, &slot, &count);
  over_token_ranges(T, clamp_threads(threads, T), [&](int, int t0, int t1) {
    std::vector<int> order(k);
    for (int t = t0; t < t1; ++t) {
      // the token's entries in ascending expert id, equal ids in k-index order
      int n = 0;
      for (int j = 0; j < k; ++j) {
        const int64_t e = topk_idx[static_cast<size_t>(t) * k + j];
        if (e < 0 || slot[static_cast<size_t>(t) * k + j] < 0) continue;
        int at = n++;
        for (; at > 0 && topk_idx[static_cast<size_t>(t) * k + order[at - 1]] > e; --at) order[at] = order[at - 1];
        order[at] = j;
      }
      for (int h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int i = 0; i < n; ++i) {
          const size_t ent = static_cast<size_t>(t) * k + order[i];
          const int64_t row = topk_idx[ent] * M + slot[ent];
          acc = std::fmaf(topk_weights[ent], bf16_bits_to_float(y[row * H + h]), acc);
        }
        out[static_cast<size_t>(t) * H + h] = float_to_bf16_bits_rn(acc);
      }
    }
  });
  return kOk;
}

}  // extern "C"
