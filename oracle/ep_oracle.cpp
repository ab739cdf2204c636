// TEST INFRASTRUCTURE ONLY -- the oracle.
//
// A plain, slow, single-threaded CPU statement of what MoE expert-parallel
// dispatch and combine compute, used by the tests, by the package's smoke
// check and by the benchmark's CPU-baseline leg.  Nothing in the product path
// links, loads or calls this file.  It shares no code, header, table or
// helper with the CUDA library: every definition here is written out again
// from the pages and from the number formats, in the order the pages give.
//
// Sources (the pages are prose; they print no code for these operations and
// no worked values):
//  * "DeepEP 要約" (stakiran.github.io), section 3 "使うときの流れ":
//    forward = get_dispatch_layout -> dispatch(x, topk_idx, topk_weights)
//    -> expert compute -> combine(y, handle); backward reuses the handle;
//    decode uses low_latency_dispatch / low_latency_combine.
//  * "DeepSeek công bố thư viện mã nguồn mở DeepEP ..." (vi.news.hada.io),
//    section "Mẫu sử dụng cho huấn luyện, prefill và decoding": dispatch
//    routes each token to the experts of every rank; the handle keeps the
//    routing metadata and the per-expert receive counts; combine reduces the
//    expert outputs back to the originating rank.
//  * "Как DeepSeek разогнали обмен данными ..." (devtrends.ru), section
//    "Как это выглядит в коде": dispatch(x, topk_idx, topk_weights,
//    num_tokens_per_rank) and low_latency_dispatch(hidden_states, topk_idx,
//    num_max_tokens, num_experts).
//  * FP8 dispatch / BF16 combine: "DeepSeek выпустила DeepEP V2.5"
//    (aikraft.ru), "Технические детали и требования"; the per-token
//    per-128-channel scale granularity is the workload's stated recipe.
//
// Readings taken where the pages are silent (each is listed in the design
// notes):
//  (1) rank s owns tokens [s*T/R, (s+1)*T/R) and experts [r*E_l, (r+1)*E_l);
//  (2) a rank's receive rows are ordered by (source rank, source token);
//      the ranks' regions are packed one after another in ascending rank;
//  (3) FP8 group: a = max(max_i |x_i|, 1e-4); scale = a/448 (fp32, RN);
//      q_i = e4m3_rn_satfinite(x_i * (448/a)), with 448/a one RN division and
//      the product one RN multiply;
//  (4) normal combine is an unweighted fp32 sum over destination ranks in
//      ascending rank order starting from +0.0f, stored as bf16 (RN-even);
//  (5) low-latency slots are handed out in (source rank, token, k-index)
//      order; low-latency combine is acc = fmaf(w, y, acc) over the token's
//      entries in ascending expert id (k-index breaks ties), from +0.0f;
//  (6) an id of -1 is a masked entry; any other id outside [0, E) is an error;
//  (7) an e4m3 combine input is dequantised as decode(q) * scale (one RN
//      multiply, the scale of the row's 128-channel group) before the sum;
//      combine can also sum the receive-side per-row top-k weights back to
//      the source token, column by column, in the same ascending rank order;
//  (8) the expert-major ("GEMM") receive layout has one row per unmasked
//      (token, k-index) entry, grouped by ascending expert id, each expert's
//      group starting at a multiple of `align` rows; inside a group the
//      entries keep (source rank, token, k-index) order.  Its fp8 scales are
//      stored group-major, scales[g * ld + row], so that one group's scales
//      of consecutive rows are contiguous.  Its combine is the unweighted
//      fp32 sum of the token's rows in ascending expert id (k-index breaks
//      ties), from +0.0f.
//
// Compile with floating-point contraction off (-ffp-contract=off): every
// multiply and add below is meant as one IEEE-754 binary32 operation.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "ep_oracle.h"

namespace {

// ---------------------------------------------------------------- formats

// bfloat16 is the upper half of a binary32; widening is exact.
float bf16_bits_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// binary32 -> bfloat16, round to nearest, ties to even, on the 16 dropped
// bits.  Rounding up past the largest finite value yields infinity, as
// IEEE-754 round-to-nearest does.  NaN stays NaN.
uint16_t float_to_bf16_bits_rn(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  uint32_t keep = u >> 16;
  uint32_t dropped = u & 0xffffu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (keep & 1u))) keep += 1u;
  return static_cast<uint16_t>(keep);
}

// OCP 8-bit floating point, E4M3 ("FN" variant): 1 sign bit, 4 exponent
// bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN, so the
// largest finite magnitude is 1.75 * 2^8 = 448; subnormals (exponent field 0)
// are m * 2^-9.
double e4m3_magnitude(uint8_t code) {
  int e = (code >> 3) & 0xf;
  int m = code & 0x7;
  if (e == 0) return std::ldexp(static_cast<double>(m), -9);
  return std::ldexp(1.0 + m / 8.0, e - 7);
}

float e4m3_to_float(uint8_t code) {
  if ((code & 0x7f) == 0x7f) return std::nanf("");
  double v = e4m3_magnitude(code);
  return static_cast<float>((code & 0x80) ? -v : v);
}

// binary32 -> E4M3, round to nearest (ties to even) with saturation to +-448
// ("satfinite").  Worked in double, where every step below is exact: the
// quantum of the binade that holds |f| is 2^(max(floor(log2|f|), -6) - 3);
// |f| divided by that quantum is rounded to the nearest integer, ties to
// even; the rounded value is then re-encoded (rounding may carry it into the
// next binade, which the re-encoding handles).
uint8_t float_to_e4m3_satfinite(float f) {
  uint8_t sign = std::signbit(f) ? 0x80 : 0x00;
  if (std::isnan(f)) return static_cast<uint8_t>(sign | 0x7f);
  double a = std::fabs(static_cast<double>(f));
  if (a > 448.0) return static_cast<uint8_t>(sign | 0x7e);
  if (a == 0.0) return sign;
  int e2;
  std::frexp(a, &e2);                    // a = m * 2^e2 with m in [0.5, 1)
  int binade = e2 - 1;                   // floor(log2 a)
  if (binade < -6) binade = -6;          // below 2^-6 the spacing stays 2^-9
  int quantum_exp = binade - 3;
  double n = std::ldexp(a, -quantum_exp);  // exact
  double fl = std::floor(n);
  double frac = n - fl;
  double r = fl;
  if (frac > 0.5 || (frac == 0.5 && std::fmod(fl, 2.0) != 0.0)) r = fl + 1.0;
  double v = std::ldexp(r, quantum_exp);
  if (v > 448.0) return static_cast<uint8_t>(sign | 0x7e);
  if (v == 0.0) return sign;
  if (v < std::ldexp(1.0, -6)) {          // subnormal: v = m * 2^-9
    int m = static_cast<int>(std::ldexp(v, 9));
    return static_cast<uint8_t>(sign | m);
  }
  std::frexp(v, &e2);
  int ve = e2 - 1;                        // v = (1 + m/8) * 2^ve
  int m = static_cast<int>(std::ldexp(v, -ve) * 8.0) - 8;
  return static_cast<uint8_t>(sign | ((ve + 7) << 3) | m);
}

// ---------------------------------------------------------------- steps

constexpr int kOk = 0, kInvalidArg = 1, kCapacity = 3, kBadExpert = 4;

struct Shape {
  int R, E, k, T, El, tpr;  // tpr = tokens per source rank
};

int check_shape(int R, int E, int k, int T, Shape* s) {
  if (R <= 0 || E <= 0 || k <= 0 || T < 0) return kInvalidArg;
  if (E % R != 0 || T % R != 0) return kInvalidArg;
  s->R = R; s->E = E; s->k = k; s->T = T; s->El = E / R; s->tpr = T / R;
  return kOk;
}

int check_ids(const Shape& s, const int64_t* topk_idx) {
  for (int64_t i = 0; i < static_cast<int64_t>(s.T) * s.k; ++i) {
    int64_t e = topk_idx[i];
    if (e < -1 || e >= s.E) return kBadExpert;
  }
  return kOk;
}

// Routing layout (get_dispatch_layout): which ranks each token goes to, how
// many tokens each source rank sends to each rank and expert, and the row of
// each (token, rank) pair inside rank r's receive region.
struct Layout {
  std::vector<uint8_t> in_rank;          // [T][R]
  std::vector<int> slot;                 // [T][R], -1 if the token skips r
  std::vector<int> tokens_per_rank;      // [R src][R dst]
  std::vector<int> tokens_per_expert;    // [R src][E]
  std::vector<int> recv_per_rank;        // [R]
  std::vector<int> rank_offset;          // [R+1], exclusive prefix of recv_per_rank
  std::vector<int> recv_per_expert;      // [E]
};

void compute_layout(const Shape& s, const int64_t* topk_idx, Layout* L) {
  const int R = s.R, E = s.E, k = s.k, T = s.T;
  L->in_rank.assign(static_cast<size_t>(T) * R, 0);
  L->slot.assign(static_cast<size_t>(T) * R, -1);
  L->tokens_per_rank.assign(static_cast<size_t>(R) * R, 0);
  L->tokens_per_expert.assign(static_cast<size_t>(R) * E, 0);
  L->recv_per_rank.assign(R, 0);
  L->rank_offset.assign(R + 1, 0);
  L->recv_per_expert.assign(E, 0);

  // Which ranks a token is sent to: the owners of its (unmasked) experts; a
  // rank that owns several of the token's experts receives the token once.
  for (int t = 0; t < T; ++t) {
    int src = t / s.tpr;
    for (int j = 0; j < k; ++j) {
      int64_t e = topk_idx[static_cast<size_t>(t) * k + j];
      if (e < 0) continue;
      int r = static_cast<int>(e / s.El);
      L->in_rank[static_cast<size_t>(t) * R + r] = 1;
      L->tokens_per_expert[static_cast<size_t>(src) * E + e] += 1;
    }
  }
  for (int t = 0; t < T; ++t) {
    int src = t / s.tpr;
    for (int r = 0; r < R; ++r)
      if (L->in_rank[static_cast<size_t>(t) * R + r])
        L->tokens_per_rank[static_cast<size_t>(src) * R + r] += 1;
  }
  for (int src = 0; src < R; ++src) {
    for (int r = 0; r < R; ++r)
      L->recv_per_rank[r] += L->tokens_per_rank[static_cast<size_t>(src) * R + r];
    for (int e = 0; e < E; ++e)
      L->recv_per_expert[e] += L->tokens_per_expert[static_cast<size_t>(src) * E + e];
  }
  for (int r = 0; r < R; ++r) L->rank_offset[r + 1] = L->rank_offset[r] + L->recv_per_rank[r];

  // Slot of (t, r) in rank r's region: the tokens that earlier source ranks
  // send to r come first, then the earlier tokens of t's own source rank.
  for (int src = 0; src < R; ++src) {
    std::vector<int> running(R, 0);
    for (int r = 0; r < R; ++r)
      for (int p = 0; p < src; ++p) running[r] += L->tokens_per_rank[static_cast<size_t>(p) * R + r];
    for (int t = src * s.tpr; t < (src + 1) * s.tpr; ++t)
      for (int r = 0; r < R; ++r)
        if (L->in_rank[static_cast<size_t>(t) * R + r]) {
          L->slot[static_cast<size_t>(t) * R + r] = running[r];
          running[r] += 1;
        }
  }
}

// FP8 quantisation of one token row, one 128-channel group at a time.
void quantize_row(int H, const uint16_t* x, uint8_t* q, float* scales) {
  for (int g = 0; g < H / 128; ++g) {
    float amax = 0.0f;
    for (int i = 0; i < 128; ++i) {
      float v = std::fabs(bf16_bits_to_float(x[g * 128 + i]));
      if (v > amax) amax = v;
    }
    float a = amax > 1e-4f ? amax : 1e-4f;
    float scale = a / 448.0f;    // one RN division
    float inv = 448.0f / a;      // one RN division
    scales[g] = scale;
    for (int i = 0; i < 128; ++i) {
      float v = bf16_bits_to_float(x[g * 128 + i]) * inv;  // one RN multiply
      q[g * 128 + i] = float_to_e4m3_satfinite(v);
    }
  }
}

// Low-latency slot of every (token, k-index) entry: its position among the
// entries routed to the same expert, counted in (source rank, token, k-index)
// order.  Entries past the per-expert capacity M get no slot (-1).
bool ll_slots(const Shape& s, const int64_t* topk_idx, int M, std::vector<int>* slot,
              std::vector<int>* count) {
  bool overflow = false;
  slot->assign(static_cast<size_t>(s.T) * s.k, -1);
  count->assign(s.E, 0);
  for (int t = 0; t < s.T; ++t)
    for (int j = 0; j < s.k; ++j) {
      int64_t e = topk_idx[static_cast<size_t>(t) * s.k + j];
      if (e < 0) continue;
      int c = (*count)[e];
      (*count)[e] = c + 1;
      if (c < M) (*slot)[static_cast<size_t>(t) * s.k + j] = c;
      else overflow = true;
    }
  return overflow;
}

// Value of channel h of receive row `row` as fp32: a bf16 row widens
// exactly; an e4m3 row is decoded and multiplied by its group's scale.
float combine_input(int y_fp8, const void* y, const float* y_scales, int H, int64_t row, int h) {
  if (!y_fp8) return bf16_bits_to_float(static_cast<const uint16_t*>(y)[row * H + h]);
  float code_value = e4m3_to_float(static_cast<const uint8_t*>(y)[row * H + h]);
  return code_value * y_scales[row * (H / 128) + h / 128];  // one RN multiply
}

// Expert-major rows.  count[e] = entries routed to e; offset[e] = first row
// of expert e's group (each group rounded up to a multiple of align rows);
// row[t * k + j] = row of entry (t, j), or -1 if masked.  Entries are visited
// in (token, k-index) order, which is (source rank, token, k-index) order.
void em_rows(const Shape& s, const int64_t* topk_idx, int align, std::vector<int>* count,
             std::vector<int>* offset, std::vector<int>* row) {
  count->assign(s.E, 0);
  std::vector<int> rank_in_expert(static_cast<size_t>(s.T) * s.k, -1);
  for (int t = 0; t < s.T; ++t)
    for (int j = 0; j < s.k; ++j) {
      int64_t e = topk_idx[static_cast<size_t>(t) * s.k + j];
      if (e < 0) continue;
      rank_in_expert[static_cast<size_t>(t) * s.k + j] = (*count)[e];
      (*count)[e] += 1;
    }
  offset->assign(s.E + 1, 0);
  for (int e = 0; e < s.E; ++e) {
    int padded = ((*count)[e] + align - 1) / align * align;
    (*offset)[e + 1] = (*offset)[e] + padded;
  }
  row->assign(static_cast<size_t>(s.T) * s.k, -1);
  for (int t = 0; t < s.T; ++t)
    for (int j = 0; j < s.k; ++j) {
      size_t i = static_cast<size_t>(t) * s.k + j;
      if (rank_in_expert[i] >= 0) (*row)[i] = (*offset)[topk_idx[i]] + rank_in_expert[i];
    }
}

}  // namespace

extern "C" {

uint8_t ref_float_to_e4m3(float f) { return float_to_e4m3_satfinite(f); }
float ref_e4m3_to_float(uint8_t code) { return e4m3_to_float(code); }
uint16_t ref_float_to_bf16(float f) { return float_to_bf16_bits_rn(f); }

int ref_quantize_row(int H, const uint16_t* x, uint8_t* q, float* scales) {
  if (H <= 0 || H % 128 != 0) return kInvalidArg;
  quantize_row(H, x, q, scales);
  return kOk;
}

int ref_layout(int R, int E, int k, int T, const int64_t* topk_idx, int* num_tokens_per_rank,
               int* num_tokens_per_expert, uint8_t* is_token_in_rank, int* slot,
               int* num_recv_per_rank, int* rank_offset, int* num_recv_per_expert) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  Layout L;
  compute_layout(s, topk_idx, &L);
  auto put = [](int* dst, const std::vector<int>& v) {
    if (dst) std::memcpy(dst, v.data(), v.size() * sizeof(int));
  };
  put(num_tokens_per_rank, L.tokens_per_rank);
  put(num_tokens_per_expert, L.tokens_per_expert);
  put(slot, L.slot);
  put(num_recv_per_rank, L.recv_per_rank);
  put(rank_offset, L.rank_offset);
  put(num_recv_per_expert, L.recv_per_expert);
  if (is_token_in_rank) std::memcpy(is_token_in_rank, L.in_rank.data(), L.in_rank.size());
  return kOk;
}

int ref_dispatch(int R, int E, int k, int T, int H, int fp8, const uint16_t* x,
                 const int64_t* topk_idx, const float* topk_weights, int64_t capacity_rows,
                 void* recv_x, float* recv_scales, int* recv_src_idx, int* recv_topk_idx,
                 float* recv_topk_weights) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if (H <= 0 || H % 128 != 0) return kInvalidArg;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  Layout L;
  compute_layout(s, topk_idx, &L);
  const int G = H / 128;
  std::vector<uint8_t> q(H);
  std::vector<float> sc(G);
  bool overflow = false;
  for (int src = 0; src < R; ++src)
    for (int t = src * s.tpr; t < (src + 1) * s.tpr; ++t) {
      const uint16_t* xt = x + static_cast<size_t>(t) * H;
      if (fp8) quantize_row(H, xt, q.data(), sc.data());
      for (int r = 0; r < R; ++r) {
        int sl = L.slot[static_cast<size_t>(t) * R + r];
        if (sl < 0) continue;
        int64_t row = static_cast<int64_t>(L.rank_offset[r]) + sl;
        if (row >= capacity_rows) { overflow = true; continue; }
        if (fp8) {
          std::memcpy(static_cast<uint8_t*>(recv_x) + row * H, q.data(), H);
          std::memcpy(recv_scales + row * G, sc.data(), G * sizeof(float));
        } else {
          std::memcpy(static_cast<uint16_t*>(recv_x) + row * H, xt, H * sizeof(uint16_t));
        }
        if (recv_src_idx) recv_src_idx[row] = t;
        for (int j = 0; j < k; ++j) {
          int64_t e = topk_idx[static_cast<size_t>(t) * k + j];
          bool here = e >= 0 && e / s.El == r;
          if (recv_topk_idx) recv_topk_idx[row * k + j] = here ? static_cast<int>(e - r * s.El) : -1;
          if (recv_topk_weights && topk_weights)
            recv_topk_weights[row * k + j] = here ? topk_weights[static_cast<size_t>(t) * k + j] : 0.0f;
        }
      }
    }
  return overflow ? kCapacity : kOk;
}

int ref_combine_ex(int R, int E, int k, int T, int H, const int64_t* topk_idx, int y_fp8, const void* y,
                   const float* y_scales, int64_t y_rows, const float* recv_topk_weights, uint16_t* out,
                   float* combined_topk_weights) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if (H <= 0 || H % 128 != 0 || (y_fp8 && !y_scales)) return kInvalidArg;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  Layout L;
  compute_layout(s, topk_idx, &L);
  if (L.rank_offset[R] > y_rows) return kCapacity;
  for (int t = 0; t < T; ++t) {
    for (int h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int r = 0; r < R; ++r) {
        int sl = L.slot[static_cast<size_t>(t) * R + r];
        if (sl < 0) continue;
        int64_t row = static_cast<int64_t>(L.rank_offset[r]) + sl;
        acc = acc + combine_input(y_fp8, y, y_scales, H, row, h);  // one RN add
      }
      out[static_cast<size_t>(t) * H + h] = float_to_bf16_bits_rn(acc);
    }
    if (!combined_topk_weights || !recv_topk_weights) continue;
    for (int j = 0; j < k; ++j) {
      float wsum = 0.0f;
      for (int r = 0; r < R; ++r) {
        int sl = L.slot[static_cast<size_t>(t) * R + r];
        if (sl < 0) continue;
        int64_t row = static_cast<int64_t>(L.rank_offset[r]) + sl;
        wsum = wsum + recv_topk_weights[row * k + j];
      }
      combined_topk_weights[static_cast<size_t>(t) * k + j] = wsum;
    }
  }
  return kOk;
}

int ref_combine(int R, int E, int k, int T, int H, const int64_t* topk_idx, const uint16_t* y,
                int64_t y_rows, uint16_t* out) {
  return ref_combine_ex(R, E, k, T, H, topk_idx, 0, y, nullptr, y_rows, nullptr, out, nullptr);
}

int ref_ll_dispatch(int R, int E, int k, int T, int H, int M, int fp8, const uint16_t* x,
                    const int64_t* topk_idx, void* recv_x, float* recv_scales, int* recv_src_info,
                    int* recv_count, int* slot_out) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if (H <= 0 || H % 128 != 0 || M <= 0) return kInvalidArg;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  std::vector<int> slot, count;
  bool overflow = ll_slots(s, topk_idx, M, &slot, &count);
  const int G = H / 128;
  std::vector<uint8_t> q(H);
  std::vector<float> sc(G);
  for (int t = 0; t < T; ++t) {
    const uint16_t* xt = x + static_cast<size_t>(t) * H;
    if (fp8) quantize_row(H, xt, q.data(), sc.data());
    for (int j = 0; j < k; ++j) {
      int64_t e = topk_idx[static_cast<size_t>(t) * k + j];
      int sl = slot[static_cast<size_t>(t) * k + j];
      if (e < 0 || sl < 0) continue;
      int64_t row = e * M + sl;  // expert e = (rank e / E_l, local expert e % E_l)
      if (fp8) {
        std::memcpy(static_cast<uint8_t*>(recv_x) + row * H, q.data(), H);
        std::memcpy(recv_scales + row * G, sc.data(), G * sizeof(float));
      } else {
        std::memcpy(static_cast<uint16_t*>(recv_x) + row * H, xt, H * sizeof(uint16_t));
      }
      if (recv_src_info) recv_src_info[row] = t;
    }
  }
  if (recv_count)
    for (int e = 0; e < E; ++e) recv_count[e] = count[e] < M ? count[e] : M;
  if (slot_out) std::memcpy(slot_out, slot.data(), slot.size() * sizeof(int));
  return overflow ? kCapacity : kOk;
}

int ref_ll_combine(int R, int E, int k, int T, int H, int M, const int64_t* topk_idx,
                   const float* topk_weights, const uint16_t* y, uint16_t* out) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if (H <= 0 || H % 128 != 0 || M <= 0) return kInvalidArg;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  std::vector<int> slot, count;
  ll_slots(s, topk_idx, M, &slot, &count);
  std::vector<int> order(k);
  for (int t = 0; t < T; ++t) {
    // the token's entries in ascending expert id; equal ids keep k-index order
    int n = 0;
    for (int j = 0; j < k; ++j) {
      int64_t e = topk_idx[static_cast<size_t>(t) * k + j];
      if (e < 0 || slot[static_cast<size_t>(t) * k + j] < 0) continue;
      int pos = n++;
      while (pos > 0 && topk_idx[static_cast<size_t>(t) * k + order[pos - 1]] > e) {
        order[pos] = order[pos - 1];
        --pos;
      }
      order[pos] = j;
    }
    for (int h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int i = 0; i < n; ++i) {
        int j = order[i];
        int64_t e = topk_idx[static_cast<size_t>(t) * k + j];
        int64_t row = e * M + slot[static_cast<size_t>(t) * k + j];
        acc = std::fmaf(topk_weights[static_cast<size_t>(t) * k + j],
                        bf16_bits_to_float(y[row * H + h]), acc);
      }
      out[static_cast<size_t>(t) * H + h] = float_to_bf16_bits_rn(acc);
    }
  }
  return kOk;
}

int ref_em_layout(int R, int E, int k, int T, const int64_t* topk_idx, int align, int* num_recv_per_expert,
                  int* expert_offset, int* row_of) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if (align < 1) return kInvalidArg;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  std::vector<int> count, offset, row;
  em_rows(s, topk_idx, align, &count, &offset, &row);
  if (num_recv_per_expert) std::memcpy(num_recv_per_expert, count.data(), count.size() * sizeof(int));
  if (expert_offset) std::memcpy(expert_offset, offset.data(), offset.size() * sizeof(int));
  if (row_of) std::memcpy(row_of, row.data(), row.size() * sizeof(int));
  return kOk;
}

int ref_em_dispatch(int R, int E, int k, int T, int H, int fp8, const uint16_t* x, const int64_t* topk_idx,
                    const float* topk_weights, int align, int64_t capacity_rows, void* recv_x,
                    float* recv_scales, int64_t scales_ld, int* recv_src_idx, float* recv_weights) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if (H <= 0 || H % 128 != 0 || align < 1 || capacity_rows < 0) return kInvalidArg;
  if (fp8 && (!recv_scales || scales_ld < capacity_rows)) return kInvalidArg;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  std::vector<int> count, offset, row;
  em_rows(s, topk_idx, align, &count, &offset, &row);
  const int G = H / 128;
  // padding rows (and every row before the entries land): no source, weight 0
  const int64_t used = offset[E] < capacity_rows ? offset[E] : capacity_rows;
  for (int64_t i = 0; i < used; ++i) {
    if (recv_src_idx) recv_src_idx[i] = -1;
    if (recv_weights) recv_weights[i] = 0.0f;
  }
  std::vector<uint8_t> q(H);
  std::vector<float> sc(G);
  bool overflow = false;
  for (int t = 0; t < T; ++t) {
    const uint16_t* xt = x + static_cast<size_t>(t) * H;
    if (fp8) quantize_row(H, xt, q.data(), sc.data());
    for (int j = 0; j < k; ++j) {
      int64_t rw = row[static_cast<size_t>(t) * k + j];
      if (rw < 0) continue;
      if (rw >= capacity_rows) { overflow = true; continue; }
      if (fp8) {
        std::memcpy(static_cast<uint8_t*>(recv_x) + rw * H, q.data(), H);
        for (int g = 0; g < G; ++g) recv_scales[g * scales_ld + rw] = sc[g];
      } else {
        std::memcpy(static_cast<uint16_t*>(recv_x) + rw * H, xt, H * sizeof(uint16_t));
      }
      if (recv_src_idx) recv_src_idx[rw] = t;
      if (recv_weights && topk_weights) recv_weights[rw] = topk_weights[static_cast<size_t>(t) * k + j];
    }
  }
  return overflow ? kCapacity : kOk;
}

int ref_em_combine(int R, int E, int k, int T, int H, const int64_t* topk_idx, int align, const uint16_t* y,
                   int64_t y_rows, uint16_t* out) {
  Shape s;
  int st = check_shape(R, E, k, T, &s);
  if (st != kOk) return st;
  if (H <= 0 || H % 128 != 0 || align < 1) return kInvalidArg;
  if ((st = check_ids(s, topk_idx)) != kOk) return st;
  std::vector<int> count, offset, row;
  em_rows(s, topk_idx, align, &count, &offset, &row);
  if (offset[E] > y_rows) return kCapacity;
  std::vector<int> by_expert(k);
  for (int t = 0; t < T; ++t) {
    const int64_t* ids = topk_idx + static_cast<size_t>(t) * k;
    // unmasked k-indices sorted by expert id, stable (insertion sort)
    int n = 0;
    for (int j = 0; j < k; ++j) {
      if (ids[j] < 0) continue;
      int at = n++;
      for (; at > 0 && ids[by_expert[at - 1]] > ids[j]; --at) by_expert[at] = by_expert[at - 1];
      by_expert[at] = j;
    }
    for (int h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int i = 0; i < n; ++i) {
        int64_t rw = row[static_cast<size_t>(t) * k + by_expert[i]];
        acc = acc + bf16_bits_to_float(y[rw * H + h]);  // one RN add
      }
      out[static_cast<size_t>(t) * H + h] = float_to_bf16_bits_rn(acc);
    }
  }
  return kOk;
}

}  // extern "C"
