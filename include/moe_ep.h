/*
 * moe_ep.h -- C ABI of libmoe_ep.so: the "EP Normal" MoE expert-parallel
 * token pipeline on one GB300 GPU (sm_103a).
 *
 * The pipeline is the one the UMDK/CAM deep-analysis page (v2) describes in
 * section 2 ("EP Normal" communication operators): (1) dispatch layout,
 * (2) notify dispatch, (3) dispatch with optional dynamic INT8 quantisation,
 * (4) combine (fp32 weighted sum).  The EP world of R ranks is modelled as R
 * logical ranks whose buffers are partitions of one GPU's HBM, so the
 * page's AllGather / shmem exchanges are ordinary global-memory traffic and
 * its BarrierAll / magic-counter protocol (section 2.7) is replaced by
 * stream order between the four calls.
 *
 * Entry points, in groups: the four stages (moe_dispatch_layout,
 * moe_notify_dispatch, moe_dispatch, moe_combine) and their size queries;
 * variants of them (moe_dispatch_layout_static, moe_dispatch_fused -- layout,
 * notify and dispatch in one launch -- and moe_combine_quant,
 * moe_token_layout); and the fused deep MoE of section 4 (moe_dispatch_expand,
 * moe_group_offsets, the grouped INT8 GEMMs on the tensor cores, the GMM1
 * epilogue moe_swiglu_quant*, moe_combine_f32 / moe_deq_combine).
 *
 * Notation: R ranks, epr experts per rank, E = R*epr experts, bs tokens per
 * rank, T = R*bs tokens, k experts per token, P = T*k (token, k) pairs,
 * H hidden size.  Token g = s*bs + t belongs to source rank s; expert e
 * belongs to rank e / epr.
 *
 * Conventions for every entry point:
 *  - All array arguments are DEVICE pointers, allocated and owned by the
 *    caller; the library allocates nothing and never synchronises.  Work is
 *    enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and returns immediately.
 *  - Global state: two things only.  The launchers remember each device's
 *    SM count and, per kernel, block size and shared-memory size, the
 *    occupancy they queried on first use (read-only device facts, behind a
 *    mutex; they change no result).  moe_dispatch_layout_static owns one
 *    device array (see there).  Nothing else outlives a call.
 *  - Host-checkable problems (NULL or misaligned pointers, sizes out of
 *    range) are reported synchronously by the return value and nothing is
 *    enqueued.  A failed launch returns MOE_ERR_CUDA.
 *  - Data-dependent problems found by a kernel (an expert id outside
 *    [0,E), a row outside the receive buffer, a wait that timed out) are
 *    written to *dev_status (an int32 in device memory that the caller sets
 *    to 0 beforehand; the first error code wins) after the kernel skips the
 *    offending writes.  Read it after the stream has been synchronised.
 *  - Results are deterministic: integer outputs are bit-exact functions of
 *    the inputs, and floating-point ones use a fixed operation order.
 */
#ifndef MOE_EP_H
#define MOE_EP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* bad size, NULL or misaligned pointer */
  MOE_ERR_EXPERT_ID = 2,   /* (device) an expert id outside [0, E) */
  MOE_ERR_CAPACITY = 3,    /* (device) a row outside the receive buffer */
  MOE_ERR_TIMEOUT = 4,     /* (device) a bounded wait gave up */
  MOE_ERR_CUDA = 5,        /* a CUDA launch or runtime call failed */
  MOE_ERR_WORKSPACE = 6    /* (device) the layout workspace was not zero-filled
                              before first use, or overlapping calls share it */
} moe_status;

typedef enum { MOE_BF16 = 0, MOE_FP16 = 1 } moe_dtype;

/* Limits.  R <= 384 is CAM_MAX_RANK_SIZE (comm_args.h, section 2.2.1). */
#define MOE_EP_MAX_RANKS 384
#define MOE_EP_MAX_EXPERTS 4096
#define MOE_EP_MAX_TOPK 64
#define MOE_EP_MAX_HIDDEN 65536

/* Problem shape (the page's CommArgs fields rankSize, expertNumPerRank,
 * topk, batchSize, hiddenSize; section 2.2.1).  Valid when
 * 1 <= R <= 384, epr >= 1, E = R*epr <= 4096, 1 <= k <= min(E, 64),
 * bs >= 0, T*k < 2^31, 8 <= H <= 65536 with H % 8 == 0, dtype a moe_dtype. */
typedef struct {
  int32_t R;
  int32_t bs;
  int32_t k;
  int32_t experts_per_rank;
  int32_t H;
  int32_t dtype;
} moe_shape;

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(int status);

/* Bytes per receive row.  quant != 0: H int8 codes, zeros up to the next
 * multiple of 32 bytes, the fp32 1/scale there, zeros to the end:
 * align32(H) + 32 bytes (the page stores 1/scale at hUBAlignSize, with
 * UB_ALIGN_SIZE = 32; section 2.5).  quant == 0: the row copied verbatim,
 * 2*H bytes.  Returns -1 for an invalid shape. */
int64_t moe_recv_row_bytes(const moe_shape* shape, int quant);

/* Bytes of device workspace moe_dispatch_layout needs (0 for an invalid
 * shape).  The workspace must be zero-filled once before its first use;
 * every call leaves it ready for the next one.  Calls that share a
 * workspace must not overlap on the GPU. */
size_t moe_layout_workspace_bytes(const moe_shape* shape);

/* (1) Dispatch layout -- moe_dispatch_layout_zb, section 2.3 (phase 1:
 * per-rank/expert token counts; phase 2: send index of every pair).
 *   topk_idx  int32 [R][bs][k]  expert id of each (token, k) pair (read)
 *   count     int32 [R][E]      pairs of source rank s routed to expert e
 *   rank_send int32 [R][R]      pairs of source rank s routed to rank r
 *   send_idx  int32 [R][bs][k]  position of the pair among the pairs of its
 *                               (source rank, expert), in (token, k) order
 *   workspace moe_layout_workspace_bytes() bytes, 16-byte aligned
 * An id outside [0,E) is not counted, gets send_idx -1, and sets
 * MOE_ERR_EXPERT_ID.  A layout wait that exceeds its bound (about 1 s)
 * sets MOE_ERR_TIMEOUT; a workspace in an unexpected state sets
 * MOE_ERR_WORKSPACE (the CTA that notices skips its tile).  One kernel
 * launch (none when T*k == 0: count and rank_send are then zeroed with
 * cudaMemsetAsync). */
moe_status moe_dispatch_layout(const moe_shape* shape, const int32_t* topk_idx,
                               int32_t* count, int32_t* rank_send,
                               int32_t* send_idx, void* workspace,
                               int32_t* dev_status, void* stream);

/* Size of the scratch array behind moe_dispatch_layout_static (4 MiB). */
#define MOE_EP_STATIC_LAYOUT_WS_BYTES (4u << 20)

/* moe_dispatch_layout for callers that cannot allocate device memory.  (The
 * paper has no counterpart: this is a convenience of this library.)
 *
 * Some callers have no way to call cudaMalloc: a plugin hosted by another
 * runtime is handed only its input and output buffers and no allocator,
 * and a serving loop whose device memory is reserved in full up front must
 * not allocate on its hot path (cudaMalloc can synchronise the device and
 * can fail under memory pressure).  This entry point takes the same
 * arguments as moe_dispatch_layout minus the workspace and gives the same
 * results.  The caller still passes (and owns) every input and output.
 *
 * Scratch: one file-scope device array of MOE_EP_STATIC_LAYOUT_WS_BYTES
 * bytes inside the library, which every GPU that loads the library holds
 * until the process exits.  A shape whose moe_layout_workspace_bytes()
 * exceeds that size is rejected with MOE_ERR_INVALID_ARG and nothing is
 * enqueued.  No call allocates or frees memory (no cudaMalloc, cudaFree or
 * allocating library routine).
 *
 * Every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress), so the current device must be the device of
 * `stream`.  The first call on each device is also the set-up: that lookup
 * loads the library's kernels onto the device, so make that first call
 * before any stream capture.  The address is not cached, so a call after
 * cudaDeviceReset finds the reloaded array.  Every call then clears the
 * part of the array it uses (cudaMemsetAsync on `stream`; needed only to
 * recover from an earlier call that timed out or overlapped another, but
 * always done) and launches the layout kernel on it: two operations on the
 * stream.  All calls share the one array, which keeps the last call's
 * contents: calls that overlap on the GPU (different streams, or several
 * host threads) race and must be serialised by the caller.  Returns
 * MOE_ERR_CUDA if the lookup or the clear fails. */
moe_status moe_dispatch_layout_static(const moe_shape* shape,
                                      const int32_t* topk_idx, int32_t* count,
                                      int32_t* rank_send, int32_t* send_idx,
                                      int32_t* dev_status, void* stream);

/* (1') Token-level layout -- section 2.3's per-rank receive count, counted
 * in distinct tokens: a token that routes several of its k
 * pairs to experts of the same rank counts once for that rank.
 *   topk_idx        int32 [R][bs][k] (read)
 *   tokens_per_rank int32 [R][R]  tokens of source rank s reaching rank r
 *   in_rank         uint8 [T][R]  1 if token g reaches rank r, else 0;
 *                                 4-byte aligned
 * Ids outside [0,E) are ignored and set MOE_ERR_EXPERT_ID.  A
 * cudaMemsetAsync of tokens_per_rank, then one launch. */
moe_status moe_token_layout(const moe_shape* shape, const int32_t* topk_idx,
                            int32_t* tokens_per_rank, uint8_t* in_rank,
                            int32_t* dev_status, void* stream);

/* (2) Notify -- moe_notify_dispatch_zb, section 2.4.  The AllGather of every
 * rank's tokenPerExpert is the identity (count is already the whole R x E
 * matrix); then BuildTotalRecvCount / BuildMaxBs / BuildTotalRecvTokens /
 * BuildRecvTokenPerExp.
 *   count           int32 [R][E]  from moe_dispatch_layout (read)
 *   put_offset      int32 [E][R]  put_offset[e*R + s]: exclusive prefix sum,
 *                                 per destination rank r = e/epr, of count
 *                                 walked expert by expert and, inside an
 *                                 expert, source rank by source rank (the
 *                                 index the combine reads, section 2.6)
 *   total_recv      int32 [R]     rows rank r receives
 *   rank_recv_base  int64 [R+1]   first row of rank r's partition;
 *                                 rank_recv_base[R] = total rows (= T*k
 *                                 when every id is valid)
 *   recv_per_expert int32 [E]     rows expert e receives
 *   max_bs          int32 [1]     tokens per rank (bs)
 * One launch when R <= 64; otherwise two: a per-destination-rank scan (one
 * warp per rank, spread over many SMs), then a one-CTA scan of the rank
 * totals. */
moe_status moe_notify_dispatch(const moe_shape* shape, const int32_t* count,
                               int32_t* put_offset, int32_t* total_recv,
                               int64_t* rank_recv_base,
                               int32_t* recv_per_expert, int32_t* max_bs,
                               int32_t* dev_status, void* stream);

/* (3) Dispatch -- moe_dispatch_normal_zb + QuantProcess, section 2.5.
 * Pair (g, k) with expert e goes to row
 *     rank_recv_base[e/epr] + put_offset[e*R + s] + send_idx[g][k]
 * of recv.  quant == 0 copies x[g] verbatim; quant != 0 writes the dynamic
 * INT8 image: scale = 127 / (max|x[g]| + 1e-12f) in fp32 (IEEE division),
 * q = round-half-even(x * scale), 1/scale after the codes (see
 * moe_recv_row_bytes).
 *   x          [T][H] bf16/fp16 (shape->dtype), 16-byte aligned (read)
 *   topk_idx, send_idx, put_offset, rank_recv_base: as above (read)
 *   recv       recv_capacity_rows rows of moe_recv_row_bytes(shape, quant)
 *              bytes, 16-byte aligned
 * A row >= recv_capacity_rows is skipped and sets MOE_ERR_CAPACITY; a bad
 * id is skipped and sets MOE_ERR_EXPERT_ID.  Rows no pair maps to are left
 * untouched.  One launch. */
moe_status moe_dispatch(const moe_shape* shape, const void* x,
                        const int32_t* topk_idx, const int32_t* send_idx,
                        const int32_t* put_offset,
                        const int64_t* rank_recv_base, int quant, void* recv,
                        int64_t recv_capacity_rows, int32_t* dev_status,
                        void* stream);

/* (4) Combine -- moe_combine_normal_zb ReadBufferAndWeightedSum, section 2.6.
 * For every token g and h: acc = 0.0f; for k = 0..K-1 in order:
 *     acc = acc + (float(expert_out[row(g,k)][h]) * topk_weights[g][k])
 * with each multiply and add rounded once (no FMA); out[g][h] = acc rounded
 * to nearest even in the token dtype.  row(g,k) is the dispatch row.
 *   expert_out   [expert_out_rows][H] bf16/fp16: the experts' outputs in the
 *                same row positions as the dispatched rows, 16-byte aligned
 *   topk_weights float [T][k] (read)
 *   out          [T][H] bf16/fp16, 16-byte aligned
 * A bad id or a row >= expert_out_rows contributes nothing and sets the
 * matching status.  One launch. */
moe_status moe_combine(const moe_shape* shape, const void* expert_out,
                       int64_t expert_out_rows, const int32_t* topk_idx,
                       const float* topk_weights, const int32_t* send_idx,
                       const int32_t* put_offset,
                       const int64_t* rank_recv_base, void* out,
                       int32_t* dev_status, void* stream);

/* Low-latency dispatch: stages (1), (2) and (3) in ONE launch, the way the
 * page's moe_dispatch_lowlatency_zb runs layout, count notify, prefix and
 * token output inside one kernel (section 3.2).  Same arguments and results
 * as moe_dispatch_layout + moe_notify_dispatch + moe_dispatch (bit for
 * bit), for small batches where three launches cost more than the work.
 * A problem that fits one SM's shared memory (R <= 32, T <= 256, T*k <=
 * 4096, R*E <= 8192, T*H*2 <= 64 KB) runs in one CTA with no grid barrier;
 * larger ones in one cooperative launch of persistent CTAs with grid
 * barriers between the phases (the one-CTA kernel leaves the workspace
 * untouched, so both kinds of call may share it).
 *   workspace  moe_fused_workspace_bytes() bytes, 16-byte aligned,
 *              zero-filled once before first use (each call leaves it ready;
 *              after MOE_ERR_TIMEOUT zero it again)
 * Calls sharing a workspace must not overlap on the GPU.  The cooperative
 * form is sized to fill the GPU, so do not run two such calls (or another
 * kernel whose CTAs wait on one another) at the same time on different
 * streams: their CTAs could not all be resident.  A grid-barrier wait that
 * exceeds about a second sets MOE_ERR_TIMEOUT. */
size_t moe_fused_workspace_bytes(const moe_shape* shape);
moe_status moe_dispatch_fused(const moe_shape* shape, const void* x,
                              const int32_t* topk_idx, int quant, int32_t* count,
                              int32_t* rank_send, int32_t* send_idx,
                              int32_t* put_offset, int32_t* total_recv,
                              int64_t* rank_recv_base, int32_t* recv_per_expert,
                              int32_t* max_bs, void* recv,
                              int64_t recv_capacity_rows, void* workspace,
                              int32_t* dev_status, void* stream);

/* GMM1 epilogue of the fused deep MoE, as a standalone pass over the grouped
 * GEMM's int32 output (section 4.8.1 PerTokenDequantSwiGLU; section 8.7
 * int32 sums cast, dequantised, SwiGLU, requantised to INT8).  Per row m:
 *   v = fp32(acc[m][c]) * weight_scale[c] * token_scale[m]   (c < 2I)
 *   h[j] = (v[j] / (1 + exp(-v[j]))) * v[I + j]                (j < I)
 * then h is quantised like moe_dispatch's INT8 rows (scale = 127/(max|h| +
 * 1e-12f), round half to even, 1/scale at byte align32(I)).  Each step is
 * one fp32 round-to-nearest operation; exp is Cody-Waite reduction plus a
 * degree-7 Taylor polynomial whose reduction and Horner steps are fused
 * multiply-adds (deterministic, within 1 ulp of exp).
 *   acc           int32 [M][2I], 16-byte aligned (gate half, then up half)
 *   weight_scale  fp32 [2I] per column, 16-byte aligned
 *   token_scale   fp32 [M] per row (e.g. the dispatched rows' 1/scale)
 *   out           [M][align32(I) + 32] bytes, 16-byte aligned
 * Valid when M >= 0 and 8 <= I <= 16384 with I % 8 == 0.  One launch. */
moe_status moe_swiglu_quant(const int32_t* acc, int64_t M, int32_t I,
                            const float* weight_scale, const float* token_scale,
                            void* out, int32_t* dev_status, void* stream);

/* (4') Combine over INT8 expert outputs -- the dequantisation the pipeline
 * diagram of section 2.1 adds to stage 4 (remote read, weighted sum).
 * Same gather and arithmetic as moe_combine, except that each expert-output
 * row is an INT8 row image in the layout moe_dispatch writes
 * (moe_recv_row_bytes(shape, 1) bytes: H int8 codes, fp32 1/scale at byte
 * align32(H)), dequantised element by element as float(q) * (1/scale) (one
 * fp32 rounding) before acc = acc + (y * w).  The page prints no dequant
 * code; that order is the reading taken.
 *   expert_out_q  [expert_out_rows][moe_recv_row_bytes(shape, 1)] bytes,
 *                 16-byte aligned
 *   other arguments as moe_combine.  One launch. */
moe_status moe_combine_quant(const moe_shape* shape, const void* expert_out_q,
                             int64_t expert_out_rows, const int32_t* topk_idx,
                             const float* topk_weights, const int32_t* send_idx,
                             const int32_t* put_offset,
                             const int64_t* rank_recv_base, void* out,
                             int32_t* dev_status, void* stream);

/* ---- fused deep MoE (section 4: dispatch -> GMM1 -> DeqSwigluQuant ->
 * GMM2 -> DeqCombine, section 4.3's three-stage pipeline) -----------------
 * On one GPU the stages are separate calls on one stream; expert e's rows
 * are contiguous in the receive buffer (rows group_off[e] ..
 * group_off[e+1]-1, group_off = exclusive prefix of recv_per_expert). */

/* group_off[g] = sum of group_rows[0..g-1] (int64 [G+1], the last entry is
 * the total).  Negative counts are read as 0 and set MOE_ERR_INVALID_ARG in
 * *dev_status.  1 <= G <= MOE_EP_MAX_EXPERTS.  One launch. */
moe_status moe_group_offsets(const int32_t* group_rows, int32_t G, int64_t* group_off,
                             int32_t* dev_status, void* stream);

/* INT8 codes -> bf16 (exact): out[r][j] = (bf16) codes[r * row_stride + j]
 * for j < K.  Feeds moe_grouped_gemm_i8 with the dispatched rows (row_stride
 * = moe_recv_row_bytes(shape, 1)), GMM1-epilogue rows (align32(I) + 32) or
 * INT8 weights (row_stride = K).
 *   codes  rows x row_stride bytes, 8-byte aligned, row_stride % 8 == 0
 *   out    bf16 [rows][K], 16-byte aligned
 * 8 <= K <= MOE_EP_MAX_HIDDEN, K % 8 == 0.  One launch. */
moe_status moe_codes_to_bf16(const void* codes, int64_t rows, int64_t row_stride, int32_t K,
                             void* out, void* stream);

/* Output-column tile of moe_grouped_gemm_i8. */
int32_t moe_gmm_block_n(void);

/* Grouped INT8 GEMM (section 4.3, GMM1 / GMM2: INT8 x INT8 -> INT32) on the
 * tensor cores.  Group g (an expert) owns the group_rows[g] consecutive rows
 * of a that follow the rows of groups 0..g-1, and weight matrix w[g]:
 *   c[m][n] = sum_{j<K} a[m][j] * w[g][n][j]        (exact int32)
 * Operands hold int8 values (-128..127) stored as bf16 (moe_codes_to_bf16):
 * GB300's tensor cores have no INT8 MMA, and with values of this range the
 * bf16 MMA with fp32 accumulation over K chunks of 1024 is exact, so c is
 * the integer GEMM bit for bit.
 *   a           bf16 [a_rows][K], 16-byte aligned; a_rows <= 2^31 - 1 (0: no-op)
 *   w           bf16 [G][N][K] (K-major), 16-byte aligned
 *   group_rows  int32 [G] device (e.g. recv_per_expert of moe_notify_dispatch)
 *   c           int32 [a_rows][N], 16-byte aligned; rows past the groups'
 *               total are not written
 * 8 <= K, N <= MOE_EP_MAX_HIDDEN with K % 8 == 0 and N % 8 == 0;
 * 1 <= G <= MOE_EP_MAX_EXPERTS.
 * Data-dependent errors: groups totalling more than a_rows rows ->
 * MOE_ERR_CAPACITY (nothing written); negative counts -> MOE_ERR_INVALID_ARG;
 * a pipeline wait that exceeds about a second -> MOE_ERR_TIMEOUT.  One
 * launch (one CTA per SM). */
moe_status moe_grouped_gemm_i8(const void* a, int64_t a_rows, int32_t K, const void* w,
                               int32_t G, int32_t N, const int32_t* group_rows, int32_t* c,
                               int32_t* dev_status, void* stream);

/* Stage 1 of the fused deep MoE (section 4.3's stage-1 outputs expand_x [M, h]
 * INT8 and dynamic_scale [M]): moe_dispatch's dynamic INT8 quantisation with the two
 * outputs as separate arrays laid out for the tensor-core GEMM: the codes of
 * each (token, k) pair's row written as bf16 values (exactly the int8 codes
 * moe_dispatch writes, -127..127), and that row's 1/scale into
 * dynamic_scale[row].  Row addressing, capacity and status as moe_dispatch.
 *   expand_x       bf16 [capacity_rows][H], 16-byte aligned
 *   dynamic_scale  fp32 [capacity_rows]
 * One launch. */
moe_status moe_dispatch_expand(const moe_shape* shape, const void* x,
                               const int32_t* topk_idx, const int32_t* send_idx,
                               const int32_t* put_offset, const int64_t* rank_recv_base,
                               void* expand_x, float* dynamic_scale,
                               int64_t capacity_rows, int32_t* dev_status, void* stream);

/* moe_swiglu_quant_grouped with the requantised codes written as bf16 values
 * (codes [M][I], exact) and each row's 1/scale to inv_scale[m], ready for the
 * GMM2 GEMM; the values are those of the INT8 row images.  One launch. */
moe_status moe_swiglu_quant_grouped_bf16(const int32_t* acc, int64_t M, int32_t I,
                                         const float* weight_scale, const int64_t* group_off,
                                         int32_t G, const void* token_scale,
                                         int64_t token_scale_stride, void* codes,
                                         float* inv_scale, int32_t* dev_status,
                                         void* stream);

/* moe_grouped_gemm_i8 with the GMM2 dequantisation of section 4.3 stage 3
 * (the int32 sums cast to fp32, times the weight scale, times the per-token scale) done
 * in the GEMM's epilogue registers: for row m of group g,
 *   y[m][n] = (fp32(c[m][n]) * col_scale[g][n]) * row_scale(m)
 * with each product rounded to nearest even, row_scale(m) the fp32 at byte
 * m * row_scale_stride of row_scale (the GMM1 epilogue rows' 1/scale).  y
 * feeds moe_combine_f32, which completes DeqCombine with the same results
 * as moe_deq_combine on c.
 *   col_scale  fp32 [G][N], 16-byte aligned
 *   y          fp32 [a_rows][N], 16-byte aligned
 * Other arguments and limits as moe_grouped_gemm_i8; row_scale_stride >= 4
 * and a multiple of 4.  One launch. */
moe_status moe_grouped_gemm_i8_dequant(const void* a, int64_t a_rows, int32_t K,
                                       const void* w, int32_t G, int32_t N,
                                       const int32_t* group_rows, const float* col_scale,
                                       const void* row_scale, int64_t row_scale_stride,
                                       float* y, int32_t* dev_status, void* stream);

/* GMM1 with its DeqSwiglu epilogue in the GEMM (section 4.3 stage 2; section
 * 4.8.1's Cast, x weight_scale, x per_token_scale, SwiGLU): the weights' gate
 * and up rows are interleaved (moe_interleave_gate_up: row 2j = gate j,
 * 2j + 1 = up j, column scales likewise), so every output tile holds whole
 * (gate, up) pairs, and for row m of group g
 *   gate = (fp32(c[m][2j]) * cs[g][2j]) * ts(m),  up likewise at 2j + 1,
 *   h[m][j] = (gate / (1 + exp(-gate))) * up
 * with the same operations as moe_swiglu_quant (exp: Cody-Waite + Taylor).
 * h (fp32 [a_rows][I], 16-byte aligned) then goes through
 * moe_quant_rows_bf16 for the requantisation, which needs whole rows.
 * Other arguments and limits as moe_grouped_gemm_i8 with N = 2I.  One launch. */
moe_status moe_grouped_gemm_i8_swiglu(const void* a, int64_t a_rows, int32_t K,
                                      const void* w_interleaved, int32_t G, int32_t I,
                                      const int32_t* group_rows,
                                      const float* col_scale_interleaved,
                                      const void* row_scale, int64_t row_scale_stride,
                                      float* h, int32_t* dev_status, void* stream);

/* Weight preparation for moe_grouped_gemm_i8_swiglu: w1 int8 [G][2I][K]
 * (rows 0..I-1 gate, I..2I-1 up) -> bf16 [G][2I][K] with row 2j = gate j and
 * row 2j + 1 = up j (exact); ws1 fp32 [G][2I] permuted the same way.  One
 * launch. */
moe_status moe_interleave_gate_up(const void* w1, const float* ws1, int32_t G, int32_t I,
                                  int32_t K, void* w1_interleaved,
                                  float* ws1_interleaved, void* stream);

/* The requantisation of the GMM1 epilogue on fp32 rows h [M][I]: per row,
 * scale = 127 / (max|h| + 1e-12f), codes = round half to even of h * scale
 * written as bf16 values [M][I] (exact), 1/scale to inv_scale[m].  With
 * group_off (int64 [G+1]) rows at or past group_off[G] are not written;
 * group_off may be NULL.  8 <= I <= 16384, I % 8 == 0.  One launch. */
moe_status moe_quant_rows_bf16(const float* h, int64_t M, int32_t I, const int64_t* group_off,
                               int32_t G, void* codes, float* inv_scale, void* stream);

/* Combine over fp32 expert outputs [expert_out_rows][H] (e.g. the output of
 * moe_grouped_gemm_i8_dequant): acc = acc + (y * w), k in order, acc from 0,
 * RNE to the token dtype (section 2.6's arithmetic).  Arguments as
 * moe_combine; expert_out 16-byte aligned.  One launch. */
moe_status moe_combine_f32(const moe_shape* shape, const float* expert_out,
                           int64_t expert_out_rows, const int32_t* topk_idx,
                           const float* topk_weights, const int32_t* send_idx,
                           const int32_t* put_offset, const int64_t* rank_recv_base,
                           void* out, int32_t* dev_status, void* stream);

/* GMM1 epilogue with per-expert weight scales (section 4.3 stage 2,
 * DeqSwigluQuant): as moe_swiglu_quant, except that row m uses
 * weight_scale + g*2I for the expert g with group_off[g] <= m <
 * group_off[g+1], and its token scale is the fp32 at byte
 * m * token_scale_stride of token_scale (the dispatched row image's 1/scale:
 * token_scale = recv + align32(H), stride moe_recv_row_bytes(shape, 1)).
 * Rows at or past group_off[G] are not written.
 *   weight_scale  fp32 [G][2I], 16-byte aligned
 *   group_off     int64 [G+1] (moe_group_offsets)
 * token_scale_stride >= 4 and a multiple of 4.  One launch. */
moe_status moe_swiglu_quant_grouped(const int32_t* acc, int64_t M, int32_t I,
                                    const float* weight_scale, const int64_t* group_off,
                                    int32_t G, const void* token_scale,
                                    int64_t token_scale_stride, void* out,
                                    int32_t* dev_status, void* stream);

/* DeqCombine (section 4.3, stage 3): combine over GMM2's int32 outputs.
 * For token g, slot k (row = its dispatch row, e = its expert):
 *   y = (fp32(expert_acc[row][h]) * weight_scale[e][h]) * row_scale(row)
 *   acc = acc + (y * topk_weights[g][k])     (k in order, acc starts at 0)
 * out[g][h] = acc rounded to nearest even in the token dtype; every step is
 * one fp32 rounding.  row_scale(row) is the fp32 at byte
 * row * row_scale_stride of row_scale (the GMM1 epilogue rows' 1/scale).
 *   expert_acc    int32 [expert_rows][H], 16-byte aligned
 *   weight_scale  fp32 [E][H], 16-byte aligned
 *   other arguments as moe_combine.  One launch. */
moe_status moe_deq_combine(const moe_shape* shape, const int32_t* expert_acc,
                           int64_t expert_rows, const float* weight_scale,
                           const void* row_scale, int64_t row_scale_stride,
                           const int32_t* topk_idx, const float* topk_weights,
                           const int32_t* send_idx, const int32_t* put_offset,
                           const int64_t* rank_recv_base, void* out, int32_t* dev_status,
                           void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_EP_H */
