/*
 * moe_oracle.h -- CPU oracle for the MoE expert-parallel token pipeline.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library; the only thing both sides
 * share is the seeded input generator (workloads.py), which holds none of the
 * method's arithmetic.
 *
 * Every function is the plain definition of what a stage of the "EP Normal"
 * pipeline computes (UMDK/CAM analysis v2, section 2.1 "overall architecture",
 * sections 2.3-2.6 for the four stages).  Single-threaded, no blocking, no
 * reordering.  Build with -ffp-contract=off and without -ffast-math so that
 * each fp32 multiply and add rounds once, as the page's vector ops do.
 *
 * Notation (shared with the pages): R ranks, epr experts per rank, E = R*epr,
 * bs tokens per rank, k = top-k, H hidden size, T = R*bs tokens,
 * global token g = s*bs + t for source rank s and local token t,
 * dst(e) = e / epr.
 *
 * Return codes match the library's public status values by number:
 * 0 ok, 2 an expert id outside [0,E), 3 a destination row outside the
 * receive buffer, 1 an invalid argument.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes: 0 = bf16, 1 = fp16 (rows of 16-bit words). */

/* Number conversions, exported so tests can pin them against numpy/torch. */
void oracle_bf16_to_f32(const uint16_t* in, float* out, int64_t n);
void oracle_f16_to_f32(const uint16_t* in, float* out, int64_t n);
void oracle_f32_to_bf16(const float* in, uint16_t* out, int64_t n);
void oracle_f32_to_f16(const float* in, uint16_t* out, int64_t n);

/* Stage 1, dispatch layout (section 2.3).  topk_idx [R][bs][k].
 * count [R][E]: pairs of rank s routed to expert e.
 * rank_send [R][R]: pairs of rank s routed to any expert of rank r.
 * send_idx [R][bs][k]: index of the pair among the pairs of (s, e), in
 * (t, k) order.  An id outside [0,E) is not counted, gets send_idx -1, and
 * makes the call return 2. */
int oracle_layout(int R, int bs, int k, int epr, const int32_t* topk_idx,
                  int32_t* count, int32_t* rank_send, int32_t* send_idx);

/* Stage 2, notify (section 2.4).  count [R][E] (already "gathered").
 * put_offset [E][R]: exclusive prefix sum, per destination rank r, over the
 * (local expert j, source rank s) order; index e*R + s.
 * total_recv [R], rank_recv_base [R+1] (exclusive scan of total_recv; the
 * last entry is the number of rows), recv_per_expert [E], max_bs [1]. */
int oracle_notify(int R, int bs, int epr, const int32_t* count,
                  int32_t* put_offset, int32_t* total_recv,
                  int64_t* rank_recv_base, int32_t* recv_per_expert,
                  int32_t* max_bs);

/* Receive-buffer row of pair (g, kk) (section 2.6 addressing), or -1 when
 * the expert id is outside [0,E). */
int64_t oracle_dst_row(int R, int bs, int k, int epr, const int32_t* topk_idx,
                       const int32_t* send_idx, const int32_t* put_offset,
                       const int64_t* rank_recv_base, int64_t g, int kk);

/* oracle_dst_row for every pair: rows [T][k]. */
void oracle_dst_rows(int R, int bs, int k, int epr, const int32_t* topk_idx,
                     const int32_t* send_idx, const int32_t* put_offset,
                     const int64_t* rank_recv_base, int64_t* rows);

/* Bytes per receive row: quant -> align32(H) + 32, else H*2. */
int64_t oracle_row_bytes(int H, int quant);

/* Dynamic INT8 quantisation of one row (section 2.5 QuantProcess) into a
 * receive-row image of oracle_row_bytes(H,1) bytes. */
void oracle_quant_row(int H, int dtype, const uint16_t* xrow, uint8_t* out);

/* Stage 3, dispatch (section 2.5): every pair's row written into recv.
 * recv holds capacity_rows rows of oracle_row_bytes(H, quant) bytes.
 * Pairs with a bad id or a row >= capacity_rows are skipped (return 2/3). */
int oracle_dispatch(int R, int bs, int k, int epr, int H, int dtype, int quant,
                    const uint16_t* x, const int32_t* topk_idx,
                    const int32_t* send_idx, const int32_t* put_offset,
                    const int64_t* rank_recv_base, uint8_t* recv,
                    int64_t capacity_rows);

/* Dispatch restricted to the listed tokens: for each listed token and each
 * kk, the row image goes to rows_out[(i*k + kk) * row_bytes] and its row id
 * to row_ids[i*k + kk] (-1 for a bad id; the image is then left zero). */
int oracle_dispatch_tokens(int R, int bs, int k, int epr, int H, int dtype,
                           int quant, const uint16_t* x,
                           const int32_t* topk_idx, const int32_t* send_idx,
                           const int32_t* put_offset,
                           const int64_t* rank_recv_base,
                           const int64_t* tokens, int64_t ntok,
                           uint8_t* rows_out, int64_t* row_ids);

/* Stage 4, combine (section 2.6) for the listed tokens: out[i][h] =
 * RNE(sum over kk in order of fp32(y[row(g,kk)][h]) * w[g][kk]).
 * y has y_rows rows of H 16-bit words.  Pass tokens = NULL for all T tokens
 * (out is then [T][H]). */
int oracle_combine_tokens(int R, int bs, int k, int epr, int H, int dtype,
                          const uint16_t* y, int64_t y_rows,
                          const int32_t* topk_idx, const float* topk_weights,
                          const int32_t* send_idx, const int32_t* put_offset,
                          const int64_t* rank_recv_base,
                          const int64_t* tokens, int64_t ntok, uint16_t* out);

/* Token-level layout (section 2.3's per-rank receive count, read as distinct
 * tokens): in_rank[g][r] = 1
 * when token g routes at least one of its k pairs to an expert of rank r;
 * tokens_per_rank[s][r] = number of tokens of source rank s with
 * in_rank = 1.  Ids outside [0,E) are ignored (return 2). */
int oracle_token_layout(int R, int bs, int k, int epr, const int32_t* topk_idx,
                        int32_t* tokens_per_rank, uint8_t* in_rank);

/* exp in fp32 by Cody and Waite's two-constant range reduction
 * (x = n*ln2 + r, |r| <= ln2/2) and the degree-7 Taylor polynomial of e^r
 * in Horner form, scaled by 2^n; input clamped to [-87, 88].  Every step is
 * one fp32 operation rounded to nearest even; the two reduction steps and the
 * Horner steps are fused multiply-adds (one rounding each).  Exported for
 * pinning. */
void oracle_exp_f32(const float* in, float* out, int64_t n);

/* GMM1 epilogue of the fused deep MoE (section 4.8.1 PerTokenDequantSwiGLU,
 * section 8.7 "Cast + Dequant + SwiGLU + Quant"): for row m of the int32
 * accumulator acc [M][2I]:
 *   v = fp32(acc) (round to nearest) * weight_scale[col] * token_scale[m]
 *   a = v / (1 + exp(-v)) on the left half (columns j < I), right half b = v
 *   h[j] = a[j] * b[j + I]
 *   then the dispatch's dynamic INT8 quantisation of h: row image of
 *   align32(I) + 32 bytes (codes, zeros, fp32 1/scale at align32(I), zeros).
 * rows = NULL: all M rows, image i at out + i*row_bytes; else the listed
 * rows, image i for rows[i]. */
void oracle_swiglu_quant_rows(int64_t M, int I, const int32_t* acc,
                              const float* weight_scale,
                              const float* token_scale, const int64_t* rows,
                              int64_t nrows, uint8_t* out);

/* The same epilogue with Exp taken as the float nearest to e^x (libm's
 * double exp, rounded once to float) instead of oracle_exp_f32: the page
 * names the operation, not an algorithm for it, so this is the plainest
 * reading, written independently of any fast evaluation. */
void oracle_swiglu_quant_rows_libm(int64_t M, int I, const int32_t* acc,
                                   const float* weight_scale,
                                   const float* token_scale, const int64_t* rows,
                                   int64_t nrows, uint8_t* out);

/* Combine over INT8 expert outputs (the dequantisation the pipeline diagram
 * of section 2.1 adds to stage 4).  yq holds y_rows rows of oracle_row_bytes(H, 1) bytes laid
 * out like a dispatched INT8 row (H codes, fp32 1/scale at align32(H)).
 * Per element: t = float(q) * inv (one rounding), then the combine of
 * section 2.6: acc = acc + (t * w), RNE to the token dtype. */
int oracle_combine_quant_tokens(int R, int bs, int k, int epr, int H, int dtype,
                                const uint8_t* yq, int64_t y_rows,
                                const int32_t* topk_idx,
                                const float* topk_weights,
                                const int32_t* send_idx,
                                const int32_t* put_offset,
                                const int64_t* rank_recv_base,
                                const int64_t* tokens, int64_t ntok,
                                uint16_t* out);

/* Grouped INT8 GEMM of the fused deep MoE (section 4.3, GMM1 and GMM2:
 * INT8 x INT8 -> INT32).  Group g owns rows [group_off[g], group_off[g+1])
 * of a (int8 codes at byte 0 of rows lda bytes apart, K codes each) and
 * weight matrix b[g] (int8 [N][K], row n = output column n):
 * c[m][n] = sum_k a[m][k] * b[g][n][k], summed in int64 and stored as
 * int32.  With rows == NULL, a holds all M = group_off[G] rows and c is
 * [M][N]; else a holds nrows rows in list order (row i of a is global row
 * rows[i], which selects the group) and c[i][:] is its result.  Returns 1
 * (invalid) for a row outside [0, M) or a sum outside int32. */
int oracle_grouped_gemm_i8(int G, const int64_t* group_off, int K, int N,
                           const int8_t* a, int64_t lda, const int8_t* b,
                           const int64_t* rows, int64_t nrows, int32_t* c);

/* DeqCombine of the fused deep MoE (section 4.3, stage 3): expert-output
 * rows are int32 GMM2 accumulators acc2 [y_rows][H].  For token g and
 * k-slot kk (row = the dispatch row of (g, kk), e = its expert):
 * y = ((float)acc2[row][h] * weight_scale[e][h]) * row_scale[row], one
 * rounding each; then the combine of section 2.6: acc = acc + (y * w),
 * k in order, RNE to the token dtype.  With tokens == NULL acc2 and
 * row_scale are indexed by receive row; with a token list they hold the
 * ntok*k rows of the listed tokens in (token, k) order. */
int oracle_deq_combine_tokens(int R, int bs, int k, int epr, int H, int dtype,
                              const int32_t* acc2, int64_t y_rows,
                              const float* weight_scale, const float* row_scale,
                              const int32_t* topk_idx, const float* topk_weights,
                              const int32_t* send_idx, const int32_t* put_offset,
                              const int64_t* rank_recv_base,
                              const int64_t* tokens, int64_t ntok, uint16_t* out);

#ifdef __cplusplus
}
#endif
#endif
