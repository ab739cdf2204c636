/* TEST INFRASTRUCTURE ONLY -- the oracle's C interface.
 *
 * Plain CPU definition of MoE expert-parallel dispatch / combine, called by
 * the tests (through ctypes), by the package smoke check and by the
 * benchmark's CPU-baseline leg.  Not part of the product; shares nothing with
 * the CUDA library's headers.
 *
 * Conventions: all buffers are host memory, row-major, owned by the caller.
 * x, y, out hold bfloat16 bit patterns (uint16).  T tokens are split evenly
 * over R source ranks; E experts evenly over R ranks (E_l = E / R each).
 * topk_idx is [T][k] int64 with -1 for a masked entry.  Return value:
 * 0 ok, 1 invalid argument, 3 capacity exceeded (rows beyond the capacity are
 * skipped), 4 an expert id outside [-1, E).
 */
#ifndef EP_ORACLE_H_
#define EP_ORACLE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* number formats */
uint8_t ref_float_to_e4m3(float f);      /* RN-even, saturating to +-448 */
float ref_e4m3_to_float(uint8_t code);
uint16_t ref_float_to_bf16(float f);     /* RN-even */
/* one token row -> H e4m3 bytes + H/128 fp32 scales */
int ref_quantize_row(int H, const uint16_t* x, uint8_t* q, float* scales);

/* get_dispatch_layout.  Every output may be NULL.
 * num_tokens_per_rank [R src][R dst], num_tokens_per_expert [R src][E],
 * is_token_in_rank [T][R] (0/1), slot [T][R] (row of (t, r) inside rank r's
 * region, -1 if absent), num_recv_per_rank [R], rank_offset [R+1] (start of
 * each rank's region in the packed receive buffer), num_recv_per_expert [E]. */
int ref_layout(int R, int E, int k, int T, const int64_t* topk_idx, int* num_tokens_per_rank,
               int* num_tokens_per_expert, uint8_t* is_token_in_rank, int* slot,
               int* num_recv_per_rank, int* rank_offset, int* num_recv_per_expert);

/* normal dispatch into the packed receive buffer of capacity_rows rows:
 * recv_x [rows][H] (e4m3 bytes if fp8 else bf16), recv_scales [rows][H/128]
 * (fp8 only), recv_src_idx [rows], recv_topk_idx [rows][k] (expert id local to
 * the receiving rank, else -1), recv_topk_weights [rows][k] (0 where -1).
 * topk_weights, recv_src_idx, recv_topk_idx, recv_topk_weights may be NULL. */
int ref_dispatch(int R, int E, int k, int T, int H, int fp8, const uint16_t* x,
                 const int64_t* topk_idx, const float* topk_weights, int64_t capacity_rows,
                 void* recv_x, float* recv_scales, int* recv_src_idx, int* recv_topk_idx,
                 float* recv_topk_weights);

/* normal combine: out [T][H] bf16 from y [y_rows][H] bf16 laid out like the
 * receive buffer. */
int ref_combine(int R, int E, int k, int T, int H, const int64_t* topk_idx, const uint16_t* y,
                int64_t y_rows, uint16_t* out);

/* normal combine, general form: y is bf16 (y_fp8 = 0) or e4m3 bytes with
 * fp32 scales y_scales [y_rows][H/128] (y_fp8 = 1), dequantised as
 * decode(q) * scale.  If recv_topk_weights [y_rows][k] and
 * combined_topk_weights [T][k] are both given, the per-row weights are also
 * summed back to the source token, column by column, in ascending rank
 * order.  ref_combine is this with bf16 y and no weights. */
int ref_combine_ex(int R, int E, int k, int T, int H, const int64_t* topk_idx, int y_fp8, const void* y,
                   const float* y_scales, int64_t y_rows, const float* recv_topk_weights, uint16_t* out,
                   float* combined_topk_weights);

/* low-latency dispatch into the expert-major buffer [E][M][H] (expert
 * e = rank e / E_l, local expert e % E_l): recv_scales [E][M][H/128] (fp8),
 * recv_src_info [E][M] (source token), recv_count [E], slot_out [T][k]
 * (row of the entry inside its expert, -1 if masked).  Any may be NULL
 * except recv_x. */
int ref_ll_dispatch(int R, int E, int k, int T, int H, int M, int fp8, const uint16_t* x,
                    const int64_t* topk_idx, void* recv_x, float* recv_scales, int* recv_src_info,
                    int* recv_count, int* slot_out);

/* low-latency combine: out [T][H] bf16 = weighted sum of y [E][M][H] bf16. */
int ref_ll_combine(int R, int E, int k, int T, int H, int M, const int64_t* topk_idx,
                   const float* topk_weights, const uint16_t* y, uint16_t* out);

/* expert-major ("GEMM") layout: num_recv_per_expert [E], expert_offset
 * [E+1] (first row of each expert's group; groups padded to multiples of
 * align rows), row_of [T][k] (row of each entry, -1 if masked).  Any output
 * may be NULL. */
int ref_em_layout(int R, int E, int k, int T, const int64_t* topk_idx, int align, int* num_recv_per_expert,
                  int* expert_offset, int* row_of);

/* expert-major dispatch: recv_x [capacity_rows][H] (e4m3 or bf16),
 * recv_scales [H/128][scales_ld] group-major (fp8 only, scales_ld >=
 * capacity_rows), recv_src_idx [rows] (source token, -1 on padding rows),
 * recv_weights [rows] (the entry's top-k weight, 0 on padding rows).
 * Padding rows' recv_x / recv_scales are not written.  topk_weights,
 * recv_src_idx, recv_weights may be NULL. */
int ref_em_dispatch(int R, int E, int k, int T, int H, int fp8, const uint16_t* x, const int64_t* topk_idx,
                    const float* topk_weights, int align, int64_t capacity_rows, void* recv_x,
                    float* recv_scales, int64_t scales_ld, int* recv_src_idx, float* recv_weights);

/* expert-major combine: out [T][H] bf16 = unweighted sum of the token's rows
 * of y [y_rows][H] bf16 in ascending expert id. */
int ref_em_combine(int R, int E, int k, int T, int H, const int64_t* topk_idx, int align, const uint16_t* y,
                   int64_t y_rows, uint16_t* out);

#ifdef __cplusplus
}
#endif

#endif /* EP_ORACLE_H_ */
