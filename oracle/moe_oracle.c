/*
 * moe_oracle.c -- CPU oracle for the MoE expert-parallel token pipeline.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE (see moe_oracle.h).  Plain,
 * single-threaded definitions of the four stages of the "EP Normal" pipeline
 * on the UMDK/CAM analysis page (v2), section 2.  Compiled with
 * -ffp-contract=off and without -ffast-math: every fp32 multiply, add and
 * divide below rounds once, to nearest even.
 *
 * Where the page is silent the reading taken is stated next to the code:
 *  - send index: position of the pair among the pairs of its (source rank,
 *    expert), in (token, k) order, i.e. the stable order;
 *  - putOffset: exclusive prefix sum per destination rank over the
 *    (local expert, source rank) order, stored at index e*R + s, which is the
 *    index the combine code on the page reads (section 2.6);
 *  - receive rows of the R logical ranks are packed back to back: rank r's
 *    rows start at rank_recv_base[r];
 *  - quantised row layout: H int8 codes, zero pad to a 32-byte boundary,
 *    the fp32 1/scale there (UB_ALIGN_SIZE = 32 in comm_args.h, section
 *    2.2.1), zero pad to the row end; row = align32(H) + 32 bytes.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

enum { ST_OK = 0, ST_INVALID = 1, ST_EXPERT_ID = 2, ST_CAPACITY = 3 };

/* ---- number conversions -------------------------------------------------- */

static float bf16_bits_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16; /* bf16 is the top half of an fp32 */
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static float f16_bits_to_f32(uint16_t b) {
  _Float16 h;
  memcpy(&h, &b, 2);
  return (float)h; /* exact widening */
}

/* fp32 -> bf16, round to nearest, ties to even, on the bit pattern. */
static uint16_t f32_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
    return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays a (quiet) NaN */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* fp32 -> fp16 by the compiler's IEEE conversion (round to nearest even,
 * default rounding mode), subnormals and overflow included. */
static uint16_t f32_to_f16_bits(float f) {
  _Float16 h = (_Float16)f;
  uint16_t b;
  memcpy(&b, &h, 2);
  return b;
}

static float to_f32(int dtype, uint16_t b) {
  return dtype == 0 ? bf16_bits_to_f32(b) : f16_bits_to_f32(b);
}

static uint16_t from_f32(int dtype, float f) {
  return dtype == 0 ? f32_to_bf16_bits(f) : f32_to_f16_bits(f);
}

void oracle_bf16_to_f32(const uint16_t* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_bits_to_f32(in[i]);
}
void oracle_f16_to_f32(const uint16_t* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f16_bits_to_f32(in[i]);
}
void oracle_f32_to_bf16(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_bits(in[i]);
}
void oracle_f32_to_f16(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_f16_bits(in[i]);
}

/* ---- stage 1: dispatch layout (section 2.3) ------------------------------ */

int oracle_layout(int R, int bs, int k, int epr, const int32_t* topk_idx,
                  int32_t* count, int32_t* rank_send, int32_t* send_idx) {
  if (R < 1 || bs < 0 || k < 1 || epr < 1) return ST_INVALID;
  const int E = R * epr;
  int status = ST_OK;
  int32_t* cnt = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  if (!cnt) return ST_INVALID;
  for (int s = 0; s < R; ++s) {
    /* running count per expert for this source rank, pairs visited in
     * (token, k) order: the value before the increment is the send index */
    for (int e = 0; e < E; ++e) cnt[e] = 0;
    for (int t = 0; t < bs; ++t) {
      for (int kk = 0; kk < k; ++kk) {
        const int64_t p = ((int64_t)s * bs + t) * k + kk;
        const int32_t e = topk_idx[p];
        if (e < 0 || e >= E) {
          send_idx[p] = -1;
          status = ST_EXPERT_ID;
          continue;
        }
        send_idx[p] = cnt[e];
        cnt[e] += 1;
      }
    }
    for (int e = 0; e < E; ++e) count[(int64_t)s * E + e] = cnt[e];
    /* per destination rank: the sum over that rank's experts */
    for (int r = 0; r < R; ++r) {
      int32_t sum = 0;
      for (int j = 0; j < epr; ++j) sum += cnt[r * epr + j];
      rank_send[(int64_t)s * R + r] = sum;
    }
  }
  free(cnt);
  return status;
}

/* ---- stage 2: notify (section 2.4) --------------------------------------- */

int oracle_notify(int R, int bs, int epr, const int32_t* count,
                  int32_t* put_offset, int32_t* total_recv,
                  int64_t* rank_recv_base, int32_t* recv_per_expert,
                  int32_t* max_bs) {
  if (R < 1 || bs < 0 || epr < 1) return ST_INVALID;
  const int E = R * epr;
  /* The AllGather of every rank's tokenPerExpert is the identity here: the
   * R x E matrix is already whole.  putOffset is the exclusive prefix sum of
   * the counts a destination rank receives, walked expert by expert and,
   * within an expert, source rank by source rank. */
  for (int r = 0; r < R; ++r) {
    int32_t run = 0;
    for (int j = 0; j < epr; ++j) {
      const int e = r * epr + j;
      for (int s = 0; s < R; ++s) {
        put_offset[(int64_t)e * R + s] = run;
        run += count[(int64_t)s * E + e];
      }
    }
    total_recv[r] = run;
  }
  int64_t base = 0;
  for (int r = 0; r < R; ++r) {
    rank_recv_base[r] = base;
    base += total_recv[r];
  }
  rank_recv_base[R] = base;
  for (int e = 0; e < E; ++e) {
    int32_t sum = 0;
    for (int s = 0; s < R; ++s) sum += count[(int64_t)s * E + e];
    recv_per_expert[e] = sum;
  }
  /* every rank holds bs tokens (batchSize is one scalar in CommArgs) */
  max_bs[0] = bs;
  return ST_OK;
}

/* ---- row addressing (section 2.6) ---------------------------------------- */

int64_t oracle_dst_row(int R, int bs, int k, int epr, const int32_t* topk_idx,
                       const int32_t* send_idx, const int32_t* put_offset,
                       const int64_t* rank_recv_base, int64_t g, int kk) {
  const int E = R * epr;
  const int64_t p = g * k + kk;
  const int32_t e = topk_idx[p];
  if (e < 0 || e >= E) return -1;
  const int64_t s = g / bs;    /* source rank of the token */
  const int dst = e / epr;     /* rank that owns expert e */
  return rank_recv_base[dst] + (int64_t)put_offset[(int64_t)e * R + s] +
         (int64_t)send_idx[p];
}

void oracle_dst_rows(int R, int bs, int k, int epr, const int32_t* topk_idx,
                     const int32_t* send_idx, const int32_t* put_offset,
                     const int64_t* rank_recv_base, int64_t* rows) {
  const int64_t T = (int64_t)R * bs;
  for (int64_t g = 0; g < T; ++g)
    for (int kk = 0; kk < k; ++kk)
      rows[g * k + kk] = oracle_dst_row(R, bs, k, epr, topk_idx, send_idx,
                                        put_offset, rank_recv_base, g, kk);
}

int64_t oracle_row_bytes(int H, int quant) {
  if (quant) return (int64_t)((H + 31) / 32) * 32 + 32;
  return (int64_t)H * 2;
}

/* ---- stage 3: dispatch with optional INT8 quantisation (section 2.5) ----- */

void oracle_quant_row(int H, int dtype, const uint16_t* xrow, uint8_t* out) {
  const int64_t Sq = oracle_row_bytes(H, 1);
  const int64_t h_align = (int64_t)((H + 31) / 32) * 32;
  memset(out, 0, (size_t)Sq);
  /* 1. widen to fp32;  2. amax = max |x| */
  float amax = 0.0f;
  for (int h = 0; h < H; ++h) {
    const float a = fabsf(to_f32(dtype, xrow[h]));
    if (a > amax) amax = a;
  }
  /* scale = 127 / (amax + 1e-12), each step one fp32 rounding */
  const float denom = amax + 1e-12f;
  const float scale = 127.0f / denom;
  /* 3. x * scale, round half to even to an integer; |q| <= 127, so the
   *    page's later int16 and int8 casts change nothing */
  for (int h = 0; h < H; ++h) {
    const float v = to_f32(dtype, xrow[h]) * scale;
    const int q = (int)nearbyintf(v);
    out[h] = (uint8_t)(int8_t)q;
  }
  /* 4. 1/scale stored at the 32-byte-aligned end of the row */
  const float inv = 1.0f / scale;
  memcpy(out + h_align, &inv, 4);
}

static int dispatch_token(int R, int bs, int k, int epr, int H, int dtype,
                          int quant, const uint16_t* x,
                          const int32_t* topk_idx, const int32_t* send_idx,
                          const int32_t* put_offset,
                          const int64_t* rank_recv_base, int64_t g,
                          uint8_t* image, int64_t* rows) {
  const int64_t S = oracle_row_bytes(H, quant);
  const uint16_t* xrow = x + g * (int64_t)H;
  if (quant)
    oracle_quant_row(H, dtype, xrow, image);
  else
    memcpy(image, xrow, (size_t)S);
  int status = ST_OK;
  for (int kk = 0; kk < k; ++kk) {
    rows[kk] = oracle_dst_row(R, bs, k, epr, topk_idx, send_idx, put_offset,
                              rank_recv_base, g, kk);
    if (rows[kk] < 0) status = ST_EXPERT_ID;
  }
  return status;
}

int oracle_dispatch(int R, int bs, int k, int epr, int H, int dtype, int quant,
                    const uint16_t* x, const int32_t* topk_idx,
                    const int32_t* send_idx, const int32_t* put_offset,
                    const int64_t* rank_recv_base, uint8_t* recv,
                    int64_t capacity_rows) {
  const int64_t S = oracle_row_bytes(H, quant);
  const int64_t T = (int64_t)R * bs;
  uint8_t* image = (uint8_t*)malloc((size_t)S);
  int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)k);
  if (!image || !rows) {
    free(image);
    free(rows);
    return ST_INVALID;
  }
  int status = ST_OK;
  for (int64_t g = 0; g < T; ++g) {
    int st = dispatch_token(R, bs, k, epr, H, dtype, quant, x, topk_idx,
                            send_idx, put_offset, rank_recv_base, g, image,
                            rows);
    if (st && !status) status = st;
    for (int kk = 0; kk < k; ++kk) {
      if (rows[kk] < 0) continue;
      if (rows[kk] >= capacity_rows) {
        if (!status) status = ST_CAPACITY;
        continue;
      }
      memcpy(recv + rows[kk] * S, image, (size_t)S);
    }
  }
  free(image);
  free(rows);
  return status;
}

int oracle_dispatch_tokens(int R, int bs, int k, int epr, int H, int dtype,
                           int quant, const uint16_t* x,
                           const int32_t* topk_idx, const int32_t* send_idx,
                           const int32_t* put_offset,
                           const int64_t* rank_recv_base,
                           const int64_t* tokens, int64_t ntok,
                           uint8_t* rows_out, int64_t* row_ids) {
  const int64_t S = oracle_row_bytes(H, quant);
  uint8_t* image = (uint8_t*)malloc((size_t)S);
  if (!image) return ST_INVALID;
  int status = ST_OK;
  for (int64_t i = 0; i < ntok; ++i) {
    int st = dispatch_token(R, bs, k, epr, H, dtype, quant, x, topk_idx,
                            send_idx, put_offset, rank_recv_base, tokens[i],
                            image, row_ids + i * k);
    if (st && !status) status = st;
    for (int kk = 0; kk < k; ++kk) {
      uint8_t* dst = rows_out + (i * k + kk) * S;
      if (row_ids[i * k + kk] < 0)
        memset(dst, 0, (size_t)S);
      else
        memcpy(dst, image, (size_t)S);
    }
  }
  free(image);
  return status;
}

/* ---- stage 4: combine (section 2.6 ReadBufferAndWeightedSum) ------------- */

int oracle_combine_tokens(int R, int bs, int k, int epr, int H, int dtype,
                          const uint16_t* y, int64_t y_rows,
                          const int32_t* topk_idx, const float* topk_weights,
                          const int32_t* send_idx, const int32_t* put_offset,
                          const int64_t* rank_recv_base,
                          const int64_t* tokens, int64_t ntok, uint16_t* out) {
  const int64_t T = (int64_t)R * bs;
  if (!tokens) ntok = T;
  float* acc = (float*)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
  if (!acc) return ST_INVALID;
  int status = ST_OK;
  for (int64_t i = 0; i < ntok; ++i) {
    const int64_t g = tokens ? tokens[i] : i;
    /* accumulator starts at zero (Duplicate 0) */
    for (int h = 0; h < H; ++h) acc[h] = 0.0f;
    for (int kk = 0; kk < k; ++kk) {
      const int64_t row = oracle_dst_row(R, bs, k, epr, topk_idx, send_idx,
                                         put_offset, rank_recv_base, g, kk);
      if (row < 0) {
        if (!status) status = ST_EXPERT_ID;
        continue;
      }
      if (row >= y_rows) {
        if (!status) status = ST_CAPACITY;
        continue;
      }
      const float w = topk_weights[g * k + kk];
      const uint16_t* yrow = y + row * (int64_t)H;
      for (int h = 0; h < H; ++h) {
        /* Cast, then Muls (one rounding), then Add (one rounding) */
        const float prod = to_f32(dtype, yrow[h]) * w;
        acc[h] = acc[h] + prod;
      }
    }
    /* CAST_RINT back to the token dtype */
    for (int h = 0; h < H; ++h) out[i * (int64_t)H + h] = from_f32(dtype, acc[h]);
  }
  free(acc);
  return status;
}

/* ---- combine over INT8 expert outputs (section 2.1, stage 4 dequantised) - */

int oracle_combine_quant_tokens(int R, int bs, int k, int epr, int H, int dtype,
                                const uint8_t* yq, int64_t y_rows,
                                const int32_t* topk_idx,
                                const float* topk_weights,
                                const int32_t* send_idx,
                                const int32_t* put_offset,
                                const int64_t* rank_recv_base,
                                const int64_t* tokens, int64_t ntok,
                                uint16_t* out) {
  const int64_t T = (int64_t)R * bs;
  const int64_t S = oracle_row_bytes(H, 1);
  const int64_t h_align = (int64_t)((H + 31) / 32) * 32;
  if (!tokens) ntok = T;
  float* acc = (float*)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
  if (!acc) return ST_INVALID;
  int status = ST_OK;
  for (int64_t i = 0; i < ntok; ++i) {
    const int64_t g = tokens ? tokens[i] : i;
    for (int h = 0; h < H; ++h) acc[h] = 0.0f;
    for (int kk = 0; kk < k; ++kk) {
      const int64_t row = oracle_dst_row(R, bs, k, epr, topk_idx, send_idx,
                                         put_offset, rank_recv_base, g, kk);
      if (row < 0) {
        if (!status) status = ST_EXPERT_ID;
        continue;
      }
      if (row >= y_rows) {
        if (!status) status = ST_CAPACITY;
        continue;
      }
      const uint8_t* img = yq + row * S;
      float inv;
      memcpy(&inv, img + h_align, 4);
      const float w = topk_weights[g * k + kk];
      for (int h = 0; h < H; ++h) {
        const float t = (float)(int8_t)img[h] * inv;   /* dequantise */
        const float prod = t * w;                      /* Muls */
        acc[h] = acc[h] + prod;                        /* Add */
      }
    }
    for (int h = 0; h < H; ++h) out[i * (int64_t)H + h] = from_f32(dtype, acc[h]);
  }
  free(acc);
  return status;
}

/* ---- token-level layout (distinct tokens per destination rank) ----------- */

int oracle_token_layout(int R, int bs, int k, int epr, const int32_t* topk_idx,
                        int32_t* tokens_per_rank, uint8_t* in_rank) {
  if (R < 1 || bs < 0 || k < 1 || epr < 1) return ST_INVALID;
  const int E = R * epr;
  int status = ST_OK;
  for (int64_t i = 0; i < (int64_t)R * R; ++i) tokens_per_rank[i] = 0;
  for (int s = 0; s < R; ++s) {
    for (int t = 0; t < bs; ++t) {
      const int64_t g = (int64_t)s * bs + t;
      uint8_t* row = in_rank + g * R;
      for (int r = 0; r < R; ++r) row[r] = 0;
      for (int kk = 0; kk < k; ++kk) {
        const int32_t e = topk_idx[g * k + kk];
        if (e < 0 || e >= E) {
          status = ST_EXPERT_ID;
          continue;
        }
        row[e / epr] = 1;
      }
      for (int r = 0; r < R; ++r) tokens_per_rank[(int64_t)s * R + r] += row[r];
    }
  }
  return status;
}

/* ---- exp by Cody-Waite reduction + Taylor polynomial (fp32) -------------- */
/* e^x = 2^n * e^r with n = nearest integer to x / ln 2 and r = x - n ln 2,
 * |r| <= ln 2 / 2.  ln 2 is split into C1 = 0.693359375 (a few bits, so n*C1
 * is exact) and C2 = ln 2 - C1 (Cody and Waite).  e^r is the degree-7 Taylor
 * polynomial in Horner form.  Each reduction step and each Horner step is one
 * fused multiply-add (fmaf: a*b+c rounded once). */

static float exp_cw(float x) {
  if (x > 88.0f) x = 88.0f;
  if (x < -87.0f) x = -87.0f;
  const float t = x * 1.44269504f;           /* x / ln 2 */
  const float n = nearbyintf(t);             /* nearest integer, ties even */
  float r = fmaf(-n, 0.693359375f, x);       /* x - n*C1 */
  r = fmaf(-n, -2.12194440e-4f, r);          /* - n*C2 */
  float p = 1.98412698e-4f;                  /* 1/7! */
  p = fmaf(p, r, 1.38888889e-3f);            /* 1/6! */
  p = fmaf(p, r, 8.33333333e-3f);            /* 1/5! */
  p = fmaf(p, r, 4.16666667e-2f);            /* 1/4! */
  p = fmaf(p, r, 1.66666667e-1f);            /* 1/3! */
  p = fmaf(p, r, 0.5f);                      /* 1/2! */
  p = fmaf(p, r, 1.0f);                      /* 1/1! */
  p = fmaf(p, r, 1.0f);                      /* 1/0! */
  const int ni = (int)n;                     /* -126 .. 127 after the clamp */
  const uint32_t bits = (uint32_t)(ni + 127) << 23;
  float two_n;
  memcpy(&two_n, &bits, 4);
  return p * two_n;
}

void oracle_exp_f32(const float* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = exp_cw(in[i]);
}

/* ---- GMM1 epilogue: dequant, SwiGLU, requant (sections 4.8.1, 8.7) ------- */

/* The plain definition of Exp: the float nearest to e^x, through libm's
 * double exp (accurate far beyond fp32; the one rounding to float can round
 * twice only when e^x lies within 2^-29 ulp of a tie). */
static float exp_libm(float x) { return (float)exp((double)x); }

static void swiglu_quant_rows_with(float (*exp_fn)(float), int64_t M, int I,
                                   const int32_t* acc, const float* weight_scale,
                                   const float* token_scale, const int64_t* rows,
                                   int64_t nrows, uint8_t* out) {
  const int64_t S = oracle_row_bytes(I, 1);
  const int64_t i_align = (int64_t)((I + 31) / 32) * 32;
  float* h = (float*)malloc(sizeof(float) * (size_t)(I > 0 ? I : 1));
  if (!h) return;
  if (!rows) nrows = M;
  for (int64_t i = 0; i < nrows; ++i) {
    const int64_t m = rows ? rows[i] : i;
    const int32_t* a_row = acc + m * 2 * (int64_t)I;
    const float ts = token_scale[m];
    float amax = 0.0f;
    for (int j = 0; j < I; ++j) {
      /* 1. Cast (RINT)  2. x weight_scale (column)  3. x per-token scale */
      float gate = (float)a_row[j];
      gate = gate * weight_scale[j];
      gate = gate * ts;
      float up = (float)a_row[I + j];
      up = up * weight_scale[I + j];
      up = up * ts;
      /* 4. SwiGLU: Muls(-1), Exp, Adds(1), Div on the left half */
      const float e = exp_fn(-gate);
      const float d = e + 1.0f;
      const float sg = gate / d;
      h[j] = sg * up;
      const float ah = fabsf(h[j]);
      if (ah > amax) amax = ah;
    }
    /* 5. dynamic INT8 quantisation, as the dispatch's QuantProcess */
    uint8_t* img = out + i * S;
    memset(img, 0, (size_t)S);
    const float scale = 127.0f / (amax + 1e-12f);
    for (int j = 0; j < I; ++j) {
      const float v = h[j] * scale;
      img[j] = (uint8_t)(int8_t)(int)nearbyintf(v);
    }
    const float inv = 1.0f / scale;
    memcpy(img + i_align, &inv, 4);
  }
  free(h);
}

void oracle_swiglu_quant_rows(int64_t M, int I, const int32_t* acc,
                              const float* weight_scale,
                              const float* token_scale, const int64_t* rows,
                              int64_t nrows, uint8_t* out) {
  swiglu_quant_rows_with(exp_cw, M, I, acc, weight_scale, token_scale, rows, nrows, out);
}

void oracle_swiglu_quant_rows_libm(int64_t M, int I, const int32_t* acc,
                                   const float* weight_scale,
                                   const float* token_scale, const int64_t* rows,
                                   int64_t nrows, uint8_t* out) {
  swiglu_quant_rows_with(exp_libm, M, I, acc, weight_scale, token_scale, rows, nrows, out);
}

/* ---- fused deep MoE: grouped INT8 GEMM (sections 4.1, 4.3: GMM1 / GMM2,
 *      INT8 x INT8 -> INT32) ----------------------------------------------- */

int oracle_grouped_gemm_i8(int G, const int64_t* group_off, int K, int N,
                           const int8_t* a, int64_t lda, const int8_t* b,
                           const int64_t* rows, int64_t nrows, int32_t* c) {
  if (G < 1 || K < 0 || N < 1) return ST_INVALID;
  const int64_t M = group_off[G];
  if (!rows) nrows = M;
  for (int64_t i = 0; i < nrows; ++i) {
    const int64_t m = rows ? rows[i] : i;
    if (m < 0 || m >= M) return ST_INVALID;
    int g = 0;                                 /* the group that owns row m */
    while (!(group_off[g] <= m && m < group_off[g + 1])) ++g;
    const int8_t* arow = a + (rows ? i : m) * lda;
    for (int n = 0; n < N; ++n) {
      const int8_t* brow = b + ((int64_t)g * N + n) * K;
      int64_t acc = 0;
      for (int kk = 0; kk < K; ++kk) acc += (int64_t)arow[kk] * (int64_t)brow[kk];
      if (acc > INT32_MAX || acc < INT32_MIN) return ST_INVALID;
      c[i * (int64_t)N + n] = (int32_t)acc;
    }
  }
  return ST_OK;
}

/* ---- fused deep MoE: DeqCombine (section 4.3, stage 3) ------------------- */

int oracle_deq_combine_tokens(int R, int bs, int k, int epr, int H, int dtype,
                              const int32_t* acc2, int64_t y_rows,
                              const float* weight_scale, const float* row_scale,
                              const int32_t* topk_idx, const float* topk_weights,
                              const int32_t* send_idx, const int32_t* put_offset,
                              const int64_t* rank_recv_base,
                              const int64_t* tokens, int64_t ntok, uint16_t* out) {
  const int64_t T = (int64_t)R * bs;
  if (!tokens) ntok = T;
  float* acc = (float*)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
  if (!acc) return ST_INVALID;
  int status = ST_OK;
  for (int64_t i = 0; i < ntok; ++i) {
    const int64_t g = tokens ? tokens[i] : i;
    for (int h = 0; h < H; ++h) acc[h] = 0.0f;
    for (int kk = 0; kk < k; ++kk) {
      const int64_t row = oracle_dst_row(R, bs, k, epr, topk_idx, send_idx,
                                         put_offset, rank_recv_base, g, kk);
      if (row < 0) {
        if (!status) status = ST_EXPERT_ID;
        continue;
      }
      if (!tokens && row >= y_rows) {
        if (!status) status = ST_CAPACITY;
        continue;
      }
      const int32_t e = topk_idx[g * k + kk];
      const int64_t yr = tokens ? i * k + kk : row;  /* listed: (token, k) order */
      const int32_t* yrow = acc2 + yr * (int64_t)H;
      const float* ws = weight_scale + (int64_t)e * H;
      const float ts = row_scale[yr];
      const float w = topk_weights[g * k + kk];
      for (int h = 0; h < H; ++h) {
        /* Cast FP32 (RINT), x weight_scale (column), x per-token scale */
        float y = (float)yrow[h];
        y = y * ws[h];
        y = y * ts;
        const float prod = y * w;                      /* Muls by the score */
        acc[h] = acc[h] + prod;                        /* Add */
      }
    }
    for (int h = 0; h < H; ++h) out[i * (int64_t)H + h] = from_f32(dtype, acc[h]);
  }
  free(acc);
  return status;
}
