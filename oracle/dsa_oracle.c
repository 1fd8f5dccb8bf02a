/*
 * CPU oracle for DSA top-k sparse MLA attention over a paged FP8 (E4M3) KV
 * cache of 512-dim NoPE latent rows, and for the BF16 -> FP8 paged KV writer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the CUDA library computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load it; the library never does,
 * and it shares no code, header or table with the CUDA sources.
 *
 * Sources of each definition:
 *  - FP8 format: OCP 8-bit floating point specification, E4M3 ("FN") variant:
 *    bias 7, 3 mantissa bits, S.1111.111 is NaN, largest finite 448, no inf.
 *    The pages require exactly this flavour and reject E4M3FNUZ on CUDA
 *    (sgl-project/sglang pull 44012, "Modifications").
 *  - Raw 512-byte row: 512 unscaled E4M3 bytes (pull 44012, "Modifications",
 *    "Speed Tests and Profiling"; pull 44217 "[DSA] Support flashmla_sparse_q8
 *    prefill backend on CUDA", "Modifications").
 *  - Group-scaled 528-byte row: 512 E4M3 values then four FP32 scales, one per
 *    128-value group ("[DSA] Support group-scaled FP8 NoPE KV reads for CUDA
 *    TileLang", "Motivation").  Scale = amax(group)/448, values = e4m3(x/s).
 *  - 656-byte RoPE row: the group-scaled 528-byte row followed by the 64-dim
 *    BF16 RoPE part of the key (little-endian), so the query/key width is
 *    576 and the values stay the 512 latent dims ("[DSA] Support group-scaled
 *    FP8 NoPE KV reads for CUDA TileLang", Motivation: the 656-byte layout).
 *  - Sparse attention: per query token and head, softmax over the scaled dot
 *    products with the latent rows named by the token's top-k list; -1
 *    entries are masked (pull 44217, "Modifications": padding with -1); the
 *    output is the softmax-weighted sum of the same rows (MLA with the
 *    absorbed NoPE latent, kv_lora_rank = 512, RoPE dim 0) plus the log-sum-exp.
 *
 * Readings taken where the pages are silent, as they shape code here: LSE is
 * the natural log; duplicates count once per top-k slot; an all-masked token
 * gives O = 0, LSE = -inf; an index outside
 * the pool or the page table is masked and reported through an error bit;
 * a zero group gets scale 0 and zero bytes; an input that saturates maps to
 * +-448; a negative input that rounds to zero keeps its sign (0x80); a NaN
 * input (any payload) encodes as the FN NaN code 0x7F with its sign bit.
 *
 * Arithmetic: float64 throughout, except where the definition itself fixes
 * FP32 (the writer's scale amax/448 and the division x/s, which the format
 * stores as FP32; the FP8 query scale of the same form).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_D 512
#define ORACLE_GROUP 128
#define ORACLE_GROUPS 4
#define ORACLE_ROPE 64      /* RoPE dims of the 656-byte row */

/* error bits, same meaning as the library's device flag */
#define ORACLE_ERR_INDEX_RANGE 1
#define ORACLE_ERR_PAGE_RANGE 2

/* ---------------------------------------------------------------- FP8 codec */

/* OCP E4M3: sign s, exponent e (4 bits, bias 7), mantissa m (3 bits).
 * e == 0: subnormal m * 2^-9; otherwise (1 + m/8) * 2^(e-7); 0x7F/0xFF NaN. */
double oracle_e4m3_decode(uint8_t b) {
  int s = (b >> 7) & 1;
  int e = (b >> 3) & 0xF;
  int m = b & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* Saturating round-to-nearest-even encode by exhaustive search: the finite
 * non-negative code c in [0, 126] nearest to |x|; a tie goes to the even code
 * (the code's last bit is the mantissa's last bit).  |x| >= 448 (inf too)
 * gives 0x7E.  The sign bit is copied, so -0 and negative underflow give 0x80. */
uint8_t oracle_e4m3_encode_bruteforce(float x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 126; ++c) {
    double d = fabs(oracle_e4m3_decode((uint8_t)c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)(sign | best);
}

/* The same definition with the search done by bisection over the increasing
 * table of the 127 finite non-negative values (for bulk use; pinned to the
 * exhaustive search over every BF16 input). */
static double g_pos_values[127];
static pthread_once_t g_table_once = PTHREAD_ONCE_INIT;
static void build_table(void) {
  for (int c = 0; c <= 126; ++c) g_pos_values[c] = oracle_e4m3_decode((uint8_t)c);
}

uint8_t oracle_e4m3_encode(float x) {
  pthread_once(&g_table_once, build_table);
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int lo = 0, hi = 126; /* invariant: value[lo] <= a < value[hi] (a < 448) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (g_pos_values[mid] <= a) lo = mid; else hi = mid;
  }
  double dl = a - g_pos_values[lo], dh = g_pos_values[hi] - a;
  int c;
  if (dl < dh) c = lo;
  else if (dh < dl) c = hi;
  else c = (lo & 1) == 0 ? lo : hi;
  return (uint8_t)(sign | c);
}

float oracle_bf16_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static float le_f32(const uint8_t* p) {
  uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static void put_le_f32(uint8_t* p, float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  p[0] = (uint8_t)(u & 0xFF);
  p[1] = (uint8_t)((u >> 8) & 0xFF);
  p[2] = (uint8_t)((u >> 16) & 0xFF);
  p[3] = (uint8_t)((u >> 24) & 0xFF);
}

/* ------------------------------------------------------------------ writers */

/* Raw writer: pool[slot][d] = e4m3(float(x[i][d])), rows with slot < 0 skipped.
 * Returns the number of rows written, or -1 if a slot is >= pool_rows. */
int64_t oracle_kv_write_raw(const uint16_t* x, int64_t n_rows, const int64_t* slots,
                            uint8_t* pool, int64_t pool_rows) {
  int64_t written = 0;
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t s = slots[i];
    if (s < 0) continue;
    if (s >= pool_rows) return -1;
    uint8_t* row = pool + s * 512;
    for (int d = 0; d < ORACLE_D; ++d)
      row[d] = oracle_e4m3_encode(oracle_bf16_to_float(x[i * ORACLE_D + d]));
    ++written;
  }
  return written;
}

/* One group of 128 values: s = amax/448 in FP32; q = e4m3(x/s) with the FP32
 * quotient; amax == 0 gives s = 0 and zero bytes.  A NaN value encodes as
 * NaN with its own sign (the sign a division gives a NaN is left open by
 * IEEE 754, so it is not taken from the quotient); amax is over the values
 * that are not NaN. */
static float scaled_group(const float* v, uint8_t* q) {
  float amax = 0.0f;
  for (int i = 0; i < ORACLE_GROUP; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0f) {
    for (int i = 0; i < ORACLE_GROUP; ++i) q[i] = 0;
    return 0.0f;
  }
  float s = amax / 448.0f;
  for (int i = 0; i < ORACLE_GROUP; ++i) {
    q[i] = isnan(v[i]) ? oracle_e4m3_encode(v[i]) : oracle_e4m3_encode(v[i] / s);
  }
  return s;
}

/* The first 528 bytes of a group-scaled row from 512 BF16 values: 512 E4M3
 * bytes, then 4 little-endian FP32 scales at byte offsets 512 + 4g; group g
 * covers dims [128g, 128g + 128). */
static void scaled_row(const uint16_t* x, uint8_t* row) {
  float v[ORACLE_GROUP];
  for (int g = 0; g < ORACLE_GROUPS; ++g) {
    for (int j = 0; j < ORACLE_GROUP; ++j) v[j] = oracle_bf16_to_float(x[g * ORACLE_GROUP + j]);
    float sc = scaled_group(v, row + g * ORACLE_GROUP);
    put_le_f32(row + 512 + 4 * g, sc);
  }
}

/* Group-scaled writer: 528-byte rows. */
int64_t oracle_kv_write_scaled(const uint16_t* x, int64_t n_rows, const int64_t* slots,
                               uint8_t* pool, int64_t pool_rows) {
  int64_t written = 0;
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t s = slots[i];
    if (s < 0) continue;
    if (s >= pool_rows) return -1;
    scaled_row(x + i * ORACLE_D, pool + s * 528);
    ++written;
  }
  return written;
}

/* RoPE writer: x is [n_rows, 576] BF16; dims [0, 512) go through the group-
 * scaled writer, dims [512, 576) are stored as they are (BF16, little-endian)
 * at byte offsets 528 + 2j. */
int64_t oracle_kv_write_rope656(const uint16_t* x, int64_t n_rows, const int64_t* slots,
                                uint8_t* pool, int64_t pool_rows) {
  int64_t written = 0;
  const int W = ORACLE_D + ORACLE_ROPE;
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t s = slots[i];
    if (s < 0) continue;
    if (s >= pool_rows) return -1;
    uint8_t* row = pool + s * 656;
    scaled_row(x + i * W, row);
    for (int j = 0; j < ORACLE_ROPE; ++j) {
      uint16_t b = x[i * W + ORACLE_D + j];
      row[528 + 2 * j] = (uint8_t)(b & 0xFF);
      row[528 + 2 * j + 1] = (uint8_t)(b >> 8);
    }
    ++written;
  }
  return written;
}

/* FP8 query quantiser: per (token, head) vector of d values,
 * scale = amax/448 (FP32), q8 = e4m3(q/scale); amax == 0 gives scale 0, zeros.
 * NaN values as in the group-scaled writer: NaN with their own sign, left out
 * of amax. */
void oracle_quantize_q8(const uint16_t* q, int64_t n_vec, int d, uint8_t* q8, float* scale) {
  float* v = (float*)malloc(sizeof(float) * (size_t)d);
  for (int64_t i = 0; i < n_vec; ++i) {
    float amax = 0.0f;
    for (int j = 0; j < d; ++j) {
      v[j] = oracle_bf16_to_float(q[i * d + j]);
      float a = fabsf(v[j]);
      if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
      for (int j = 0; j < d; ++j) q8[i * d + j] = 0;
      scale[i] = 0.0f;
      continue;
    }
    float s = amax / 448.0f;
    for (int j = 0; j < d; ++j)
      q8[i * d + j] = isnan(v[j]) ? oracle_e4m3_encode(v[j]) : oracle_e4m3_encode(v[j] / s);
    scale[i] = s;
  }
  free(v);
}

/* ---------------------------------------------------------------- attention */

typedef struct {
  int q_kind;            /* 0: BF16 query, 1: E4M3 query + per-(t,h) FP32 scale */
  const void* q;         /* [T, H, 512] */
  const float* q_scale;  /* [T, H] when q_kind == 1 */
  int T, H;
  const uint8_t* pool;
  int64_t pool_rows;
  int layout;            /* 0: raw512, 1: scaled528, 2: rope656 */
  int DK;                /* query/key width: 512, or 576 with the RoPE part */
  const int32_t* page_table; /* [B, max_pages] or NULL: indices are physical rows */
  int B, max_pages, page_size;
  const int32_t* token_seq;  /* [T] or NULL: every token in sequence 0 */
  const int32_t* topk;       /* [T, K] */
  int K;
  double sm_scale;
  const int32_t* tokens;     /* which tokens to compute */
  int n_tokens;
  double* O;                 /* [n_tokens, H, 512] */
  double* LSE;               /* [n_tokens, H] */
  int next;                  /* shared work counter */
  pthread_mutex_t lock;
  int err;
} attn_job;

/* Resolve top-k entry -> physical row, or -1 when masked.  *err gets the bit. */
static int64_t resolve_row(const attn_job* J, int t, int32_t idx, int* err) {
  if (idx < 0) return -1;                         /* -1 sentinel (any negative) */
  if (J->page_table == NULL) {
    if ((int64_t)idx >= J->pool_rows) { *err |= ORACLE_ERR_INDEX_RANGE; return -1; }
    return idx;
  }
  int seq = J->token_seq ? J->token_seq[t] : 0;
  if (seq < 0 || seq >= J->B) { *err |= ORACLE_ERR_PAGE_RANGE; return -1; }
  int page = idx / J->page_size;
  int off = idx % J->page_size;
  if (page >= J->max_pages) { *err |= ORACLE_ERR_INDEX_RANGE; return -1; }
  int32_t phys = J->page_table[(int64_t)seq * J->max_pages + page];
  if (phys < 0) { *err |= ORACLE_ERR_PAGE_RANGE; return -1; }
  int64_t row = (int64_t)phys * J->page_size + off;
  if (row >= J->pool_rows) { *err |= ORACLE_ERR_PAGE_RANGE; return -1; }
  return row;
}

/* Dequantised key row in float64: the 512 latent dims, then (656-byte rows)
 * the 64 RoPE dims. */
static void dequant_row(const attn_job* J, int64_t row, double* k) {
  if (J->layout == 0) {
    const uint8_t* r = J->pool + row * 512;
    for (int d = 0; d < ORACLE_D; ++d) k[d] = oracle_e4m3_decode(r[d]);
  } else {
    const uint8_t* r = J->pool + row * (J->layout == 1 ? 528 : 656);
    for (int d = 0; d < ORACLE_D; ++d) {
      double s = (double)le_f32(r + 512 + 4 * (d / ORACLE_GROUP));
      k[d] = oracle_e4m3_decode(r[d]) * s;
    }
    if (J->layout == 2)
      for (int j = 0; j < ORACLE_ROPE; ++j)
        k[ORACLE_D + j] = (double)oracle_bf16_to_float((uint16_t)(r[528 + 2 * j] | (r[528 + 2 * j + 1] << 8)));
  }
}

static void attend_token(attn_job* J, int li, double* rows, double* q, double* s, int* err) {
  int t = J->tokens[li];
  const int32_t* idx = J->topk + (int64_t)t * J->K;
  int n = 0;
  for (int j = 0; j < J->K; ++j) {
    int64_t row = resolve_row(J, t, idx[j], err);
    if (row < 0) continue;
    dequant_row(J, row, rows + (int64_t)n * J->DK);
    ++n;
  }
  for (int h = 0; h < J->H; ++h) {
    double* o = J->O + ((int64_t)li * J->H + h) * ORACLE_D;
    int64_t qoff = ((int64_t)t * J->H + h) * J->DK;
    if (J->q_kind == 0) {
      const uint16_t* qb = (const uint16_t*)J->q + qoff;
      for (int d = 0; d < J->DK; ++d) q[d] = (double)oracle_bf16_to_float(qb[d]);
    } else {
      const uint8_t* q8 = (const uint8_t*)J->q + qoff;
      double sc = (double)J->q_scale[(int64_t)t * J->H + h];
      for (int d = 0; d < ORACLE_D; ++d) q[d] = oracle_e4m3_decode(q8[d]) * sc;
    }
    if (n == 0) {                                   /* all masked */
      for (int d = 0; d < ORACLE_D; ++d) o[d] = 0.0;
      J->LSE[(int64_t)li * J->H + h] = -INFINITY;
      continue;
    }
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
      const double* k = rows + (int64_t)j * J->DK;
      double dot = 0.0;
      for (int d = 0; d < J->DK; ++d) dot += q[d] * k[d];
      s[j] = J->sm_scale * dot;
      if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int j = 0; j < n; ++j) l += exp(s[j] - m);
    double lse = m + log(l);
    for (int d = 0; d < ORACLE_D; ++d) o[d] = 0.0;
    for (int j = 0; j < n; ++j) {
      double p = exp(s[j] - lse);
      const double* k = rows + (int64_t)j * J->DK;     /* values: the latent dims */
      for (int d = 0; d < ORACLE_D; ++d) o[d] += p * k[d];
    }
    J->LSE[(int64_t)li * J->H + h] = lse;
  }
}

static void* attn_worker(void* arg) {
  attn_job* J = (attn_job*)arg;
  double* rows = (double*)malloc(sizeof(double) * (size_t)J->K * J->DK);
  double* q = (double*)malloc(sizeof(double) * J->DK);
  double* s = (double*)malloc(sizeof(double) * (size_t)J->K);
  int err = 0;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int li = J->next++;
    pthread_mutex_unlock(&J->lock);
    if (li >= J->n_tokens) break;
    attend_token(J, li, rows, q, s, &err);
  }
  pthread_mutex_lock(&J->lock);
  J->err |= err;
  pthread_mutex_unlock(&J->lock);
  free(rows);
  free(q);
  free(s);
  return NULL;
}

/* O[li, h, :] and LSE[li, h] for each token tokens[li] (all tokens when
 * tokens == NULL).  Returns the OR of the error bits met. */
int oracle_sparse_attn(int q_kind, const void* q, const float* q_scale, int T, int H,
                       const uint8_t* pool, int64_t pool_rows, int layout,
                       const int32_t* page_table, int B, int max_pages, int page_size,
                       const int32_t* token_seq, const int32_t* topk, int K, double sm_scale,
                       const int32_t* tokens, int n_tokens, double* O, double* LSE,
                       int n_threads) {
  attn_job J;
  int32_t* all = NULL;
  memset(&J, 0, sizeof J);
  if (tokens == NULL) {
    all = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    for (int t = 0; t < T; ++t) all[t] = t;
    tokens = all;
    n_tokens = T;
  }
  J.q_kind = q_kind; J.q = q; J.q_scale = q_scale; J.T = T; J.H = H;
  J.pool = pool; J.pool_rows = pool_rows; J.layout = layout;
  J.DK = layout == 2 ? ORACLE_D + ORACLE_ROPE : ORACLE_D;
  J.page_table = page_table; J.B = B; J.max_pages = max_pages; J.page_size = page_size;
  J.token_seq = token_seq; J.topk = topk; J.K = K; J.sm_scale = sm_scale;
  J.tokens = tokens; J.n_tokens = n_tokens; J.O = O; J.LSE = LSE;
  pthread_mutex_init(&J.lock, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, attn_worker, &J);
  for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.lock);
  free(all);
  return J.err;
}

/* ------------------------------------------------ gather / dequantise reader */

/* BF16 bits of a finite float, rounded to nearest, ties to even. */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* The reader's BF16 workspace ("[DSA] Support group-scaled FP8 NoPE KV reads
 * for CUDA TileLang", Modifications, second bullet): when the top-k lists hold
 * fewer entries than the pool has physical rows, only the selected rows are
 * dequantised, one workspace row per top-k entry; otherwise the whole pool is
 * dequantised, one workspace row per physical row.  Either way the workspace
 * has min(pool_rows, T*K) rows, which bounds it at min(physical rows,
 * selected entries) * 1024 bytes for 512-wide BF16 rows.  The count is fixed
 * by the shapes alone (no data-dependent unique step, so nothing is read back
 * from the device to size it). */
int64_t oracle_gather_rows(int64_t pool_rows, int64_t n_selected) {
  return n_selected < pool_rows ? n_selected : pool_rows;
}

/* One physical row dequantised to BF16: the 512 latent dims
 * bf16_rne(fp32(e4m3(b_d) * s_g)) (raw rows: s = 1, exact), then for
 * 656-byte rows the 64 RoPE dims as stored (BF16 bits).  The FP32 product is
 * formed once (the exact product fits a double; the cast rounds it to the
 * nearest FP32), then rounded to BF16. */
static void dequant_row_bf16(const uint8_t* r, int layout, uint16_t* out) {
  for (int d = 0; d < ORACLE_D; ++d) {
    const int g = d / ORACLE_GROUP;                 /* the 128-dim group of d */
    double s = layout == 0 ? 1.0 : (double)le_f32(r + 512 + 4 * g);
    float v = (float)(oracle_e4m3_decode(r[d]) * s);
    out[d] = f32_to_bf16_rne(v);
  }
  if (layout == 2)
    for (int j = 0; j < ORACLE_ROPE; ++j)
      out[ORACLE_D + j] = (uint16_t)(((unsigned)r[528 + 2 * j + 1] << 8) | r[528 + 2 * j]);
}

/* The gather/dequantise reader that feeds BF16 consumers ("[DSA] Support
 * group-scaled FP8 NoPE KV reads for CUDA TileLang", Modifications: the full
 * and paged readers, the selected-row workspace with remapped indices and
 * kept masks; pull 44217, review thread: the paged gather with -1 padding).
 * Rows resolve as in the attention (same error bits).  out has
 * oracle_gather_rows(pool_rows, T*K) rows of W = 512 values (576 for
 * 656-byte rows, the RoPE dims appended).  For entry j of token t, e = t*K + j:
 *  - selected branch (T*K < pool_rows): out[e] = the entry's dequantised row
 *    and idx_out[e] = e;
 *  - full-pool branch (T*K >= pool_rows): out[r] = dequantised physical row r
 *    for every r, and idx_out[e] = the entry's physical row;
 *  - a masked entry gets idx_out[e] = -1 (in the selected branch its out row
 *    is left as it is).
 * So out[idx_out[e]] is entry e's row in both branches. */
int oracle_gather_dequant(const uint8_t* pool, int64_t pool_rows, int layout,
                          const int32_t* page_table, int B, int max_pages, int page_size,
                          const int32_t* token_seq, const int32_t* topk, int T, int K,
                          uint16_t* out, int32_t* idx_out) {
  attn_job J;
  memset(&J, 0, sizeof J);
  J.pool = pool; J.pool_rows = pool_rows; J.layout = layout;
  J.page_table = page_table; J.B = B; J.max_pages = max_pages; J.page_size = page_size;
  J.token_seq = token_seq;
  int err = 0;
  const int64_t R = layout == 0 ? 512 : layout == 1 ? 528 : 656;
  const int W = layout == 2 ? ORACLE_D + ORACLE_ROPE : ORACLE_D;
  const int64_t n_sel = (int64_t)T * K;
  const int full_pool = !(n_sel < pool_rows);
  if (full_pool)
    for (int64_t r = 0; r < pool_rows; ++r) dequant_row_bf16(pool + r * R, layout, out + r * W);
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < K; ++j) {
      const int64_t e = (int64_t)t * K + j;
      const int64_t row = resolve_row(&J, t, topk[e], &err);
      if (row < 0) {
        idx_out[e] = -1;
      } else if (full_pool) {
        idx_out[e] = (int32_t)row;
      } else {
        idx_out[e] = (int32_t)e;
        dequant_row_bf16(pool + row * R, layout, out + e * W);
      }
    }
  }
  return err;
}

/* ------------------------------------------------------- array conveniences */

void oracle_e4m3_encode_array(const float* x, int64_t n, uint8_t* out, int bruteforce) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = bruteforce ? oracle_e4m3_encode_bruteforce(x[i]) : oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t* b, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(b[i]);
}
