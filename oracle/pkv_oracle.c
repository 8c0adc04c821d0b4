/*
 * pkv_oracle.c — plain, slow, fp64 CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load this code. The product path never calls it, and
 * it shares no code, header, table or helper with the CUDA library.
 *
 * What it follows:
 *   - "--attention-backend" (SGLang manual, section "What an attention backend is"):
 *     a backend builds per-batch metadata (page tables, index buffers) and runs
 *     forward_extend for prefill and forward_decode for decode over the paged cache.
 *   - "[SGLang] Hybrid Attention: Dense-Sparse 동적 전환 전략", section
 *     "_select_backend: ForwardMode 기반 동적 전환": the ForwardMode truth table, and
 *     section "forward: 선형 어텐션까지 지원하는 범용 위임": save_kv_cache writes the
 *     step's K/V into the pool before attention.
 *   - The pages print no attention formula; the arithmetic below is the textbook
 *     definition of scaled dot-product attention, o = softmax(s) V with
 *     s_j = sm_scale * q . k_j, restricted to the keys a query row may see
 *     (bottom-right causal alignment), and lse = ln sum_j exp(s_j).
 *   - "--attention-backend", section "How SGLang picks a default": some models
 *     have K and V heads of different widths. q and k then have head_dim
 *     columns, v and the output head_dim_v; nothing else changes.
 *   - FP8 KV entries are OCP "E4M3FN" (bias 7, 3 mantissa bits, max 448, no
 *     infinities, NaN = S.1111.111), decoded bit by bit from that definition.
 *
 * Every floating-point step is done in double precision in the order the
 * definition states (one key after another); nothing is blocked or fused.
 *
 * Parity pins (checked by the CPU test suite): brute-force unpaged attention,
 * page-permutation invariance, page_size 1 vs 16, single key, uniform scores,
 * rows of weights summing to one, extend == stacked decodes, the LSE-merge
 * identity, the full E4M3 code table, metadata closed forms; for tree masks,
 * brute force and torch SDPA with the same mask, and a chain-shaped tree
 * reproducing the causal result exactly; for sinks, -inf sinks reproducing
 * the result without them exactly, torch SDPA with the sink as an extra key,
 * and the uniform-score closed form; for K and V of different widths, brute
 * force and torch SDPA with those widths, and zero-padded K/Q columns
 * reproducing the equal-width result exactly.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

/* KV pool element encodings */
#define ORACLE_KV_BF16 0
#define ORACLE_KV_FP8_E4M3 1

/* ForwardMode values and the two speculative attention modes. */
#define ORACLE_MODE_EXTEND 0
#define ORACLE_MODE_DECODE 1
#define ORACLE_MODE_IDLE 2
#define ORACLE_MODE_TARGET_VERIFY 3
#define ORACLE_MODE_DRAFT_EXTEND 4
#define ORACLE_SPEC_PREFILL 0
#define ORACLE_SPEC_DECODE 1
#define ORACLE_PATH_DECODE 0
#define ORACLE_PATH_EXTEND 1

/* ------------------------------------------------------------------------- */
/* Number formats                                                            */
/* ------------------------------------------------------------------------- */

/* A bfloat16 value is the upper half of an IEEE binary32; widening is exact. */
static float bf16_bits_to_float(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

double oracle_bf16_decode(uint16_t bits) { return (double)bf16_bits_to_float(bits); }

/* E4M3FN decode straight from the format definition:
 *   exponent field e (4 bits, bias 7), mantissa m (3 bits)
 *   e == 15 && m == 7      -> NaN
 *   e == 0                 -> (-1)^s * 2^(1-7) * (m / 8)       (subnormal)
 *   otherwise              -> (-1)^s * 2^(e-7) * (1 + m / 8)   (normal)      */
double oracle_e4m3_decode(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, 1 - 7);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Round half to even of a non-negative double that is exactly representable. */
static double round_half_even(double r) {
  double fl = floor(r);
  double diff = r - fl; /* exact: r and fl share the binade or fl is smaller */
  if (diff > 0.5) return fl + 1.0;
  if (diff < 0.5) return fl;
  return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* float -> E4M3FN, round to nearest even, saturating finite values (and
 * infinities) to +-448; NaN maps to the canonical NaN code 0x7F. */
uint8_t oracle_e4m3_encode(float xf) {
  if (isnan(xf)) return 0x7F;
  uint8_t sign = signbit(xf) ? 0x80 : 0x00;
  double a = fabs((double)xf);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E); /* 0x7E = 1.75 * 2^8 = 448 */
  if (a == 0.0) return sign;
  int e2;
  (void)frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1)  =>  floor(log2 a) = e2 - 1 */
  int E = e2 - 1;
  if (E < -6) E = -6; /* below 2^-6 the grid spacing stays 2^-9 (subnormals) */
  double quantum = ldexp(1.0, E - 3); /* 3 mantissa bits */
  double n = round_half_even(a / quantum); /* a / quantum is exact */
  if (n == 0.0) return sign;
  if (E == -6 && n < 8.0) return (uint8_t)(sign | (uint8_t)n); /* subnormal */
  if (n == 16.0) { /* rounded up into the next binade */
    E += 1;
    n = 8.0;
  }
  /* a < 448 keeps the result at or below 448 = code 0x7E */
  return (uint8_t)(sign | (uint8_t)(((E + 7) << 3) | ((int)n - 8)));
}

static double kv_value(const void* pool, int kv_dtype, int64_t elem, double scale) {
  if (kv_dtype == ORACLE_KV_BF16) return oracle_bf16_decode(((const uint16_t*)pool)[elem]) * scale;
  return oracle_e4m3_decode(((const uint8_t*)pool)[elem]) * scale;
}

/* ------------------------------------------------------------------------- */
/* ForwardMode dispatch                                                      */
/* ------------------------------------------------------------------------- */

/* HybridAttnBackend._select_backend: decode and idle always use the decode
 * backend; target-verify and draft-extend use the decode backend only when the
 * speculative attention mode is "decode", else the prefill backend; every other
 * mode (prefill / extend) uses the prefill backend. Returns -1 for a mode or
 * speculative setting outside the enumerations. */
int oracle_select_path(int mode, int spec_mode) {
  if (spec_mode != ORACLE_SPEC_PREFILL && spec_mode != ORACLE_SPEC_DECODE) return -1;
  if (mode == ORACLE_MODE_DECODE || mode == ORACLE_MODE_IDLE) return ORACLE_PATH_DECODE;
  if (mode == ORACLE_MODE_TARGET_VERIFY || mode == ORACLE_MODE_DRAFT_EXTEND)
    return spec_mode == ORACLE_SPEC_DECODE ? ORACLE_PATH_DECODE : ORACLE_PATH_EXTEND;
  if (mode == ORACLE_MODE_EXTEND) return ORACLE_PATH_EXTEND;
  return -1;
}

/* ------------------------------------------------------------------------- */
/* Per-batch metadata                                                        */
/* ------------------------------------------------------------------------- */

/* For request b with KV length L_b (tokens, including this step's new ones):
 *   num_pages_b        = ceil(L_b / page_size)
 *   kv_indptr[b+1]     = kv_indptr[b] + num_pages_b            (kv_indptr[0] = 0)
 *   kv_indices[...]    = page_table[b, 0 : num_pages_b]         (concatenated)
 *   kv_last_page_len_b = L_b - (num_pages_b - 1) * page_size    (0 when L_b == 0)
 *   qo_indptr[b+1]     = qo_indptr[b] + qo_len_b                (qo_len_b = 1 if qo_lens is NULL)
 * kv_indices must hold kv_indptr[bs] entries. */
int oracle_build_metadata(int bs, int page_size, const int32_t* seq_lens, const int32_t* qo_lens,
                          const int32_t* page_table, int64_t page_table_stride, int32_t* kv_indptr,
                          int32_t* kv_indices, int32_t* kv_last_page_len, int32_t* qo_indptr) {
  if (bs < 0 || page_size <= 0) return ORACLE_ERR_ARG;
  kv_indptr[0] = 0;
  qo_indptr[0] = 0;
  for (int b = 0; b < bs; ++b) {
    int32_t L = seq_lens[b];
    int32_t qo = qo_lens ? qo_lens[b] : 1;
    /* a request with L_b == 0 is graph padding: its query rows see no key */
    if (L < 0 || qo < 0 || (L > 0 && qo > L)) return ORACLE_ERR_ARG;
    int32_t np = (L + page_size - 1) / page_size;
    for (int32_t p = 0; p < np; ++p) kv_indices[kv_indptr[b] + p] = page_table[(int64_t)b * page_table_stride + p];
    kv_indptr[b + 1] = kv_indptr[b] + np;
    kv_last_page_len[b] = np > 0 ? L - (np - 1) * page_size : 0;
    qo_indptr[b + 1] = qo_indptr[b] + qo;
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* set_kv_buffer (save_kv_cache)                                             */
/* ------------------------------------------------------------------------- */

/* Pool layout: [slot][kv_head][width], slot = page * page_size + offset, with
 * width head_dim for the K pool and head_dim_v for the V pool (the two differ
 * for models whose K and V heads have different widths).
 * For each new token i: pool[loc[i], :, :] = new[i, :, :].
 * bf16 pool: the same bits. E4M3 pool: e4m3(float(new) * inv_scale), the
 * product taken in binary32 (one rounding), then rounded to E4M3FN. */
static void scatter_rows(int kv_dtype, void* pool, int64_t row, const int32_t* loc, const uint16_t* src_rows,
                         int n_tokens, float inv_scale) {
  for (int i = 0; i < n_tokens; ++i) {
    int64_t dst = (int64_t)loc[i] * row;
    int64_t src = (int64_t)i * row;
    for (int64_t e = 0; e < row; ++e) {
      if (kv_dtype == ORACLE_KV_BF16)
        ((uint16_t*)pool)[dst + e] = src_rows[src + e];
      else
        ((uint8_t*)pool)[dst + e] = oracle_e4m3_encode(bf16_bits_to_float(src_rows[src + e]) * inv_scale);
    }
  }
}

void oracle_set_kv_buffer(int kv_dtype, void* k_pool, void* v_pool, int num_kv_heads, int head_dim, int head_dim_v,
                          const int32_t* loc, const uint16_t* k_new, const uint16_t* v_new, int n_tokens,
                          float k_inv_scale, float v_inv_scale) {
  scatter_rows(kv_dtype, k_pool, (int64_t)num_kv_heads * head_dim, loc, k_new, n_tokens, k_inv_scale);
  scatter_rows(kv_dtype, v_pool, (int64_t)num_kv_heads * head_dim_v, loc, v_new, n_tokens, v_inv_scale);
}

/* ------------------------------------------------------------------------- */
/* LSE merge of partial attention results                                    */
/* ------------------------------------------------------------------------- */

/* Attention over a key set split into disjoint parts c, each giving o_c (its
 * own normalised output) and lse_c = ln sum_{j in c} exp(s_j):
 *   lse = ln sum_c exp(lse_c),   o = sum_c exp(lse_c - lse) * o_c.
 * Parts with lse_c = -inf hold no keys and contribute nothing. */
void oracle_lse_merge(int n_parts, int head_dim, const double* o_parts, const double* lse_parts, double* o_out,
                      double* lse_out) {
  double mx = -INFINITY;
  for (int c = 0; c < n_parts; ++c)
    if (lse_parts[c] > mx) mx = lse_parts[c];
  for (int d = 0; d < head_dim; ++d) o_out[d] = 0.0;
  if (mx == -INFINITY) {
    *lse_out = -INFINITY;
    return;
  }
  double z = 0.0;
  for (int c = 0; c < n_parts; ++c) z += exp(lse_parts[c] - mx);
  double lse = mx + log(z);
  for (int c = 0; c < n_parts; ++c) {
    if (lse_parts[c] == -INFINITY) continue;
    double w = exp(lse_parts[c] - lse);
    for (int d = 0; d < head_dim; ++d) o_out[d] += w * o_parts[(int64_t)c * head_dim + d];
  }
  *lse_out = lse;
}

/* ------------------------------------------------------------------------- */
/* Attention over the paged cache                                            */
/* ------------------------------------------------------------------------- */

typedef struct {
  int bs, num_q_heads, num_kv_heads, head_dim, head_dim_v, page_size, kv_dtype;
  const uint16_t* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* kv_last_page_len;
  const int32_t* qo_indptr;
  const uint64_t* tree_mask; /* NULL: chain drafts (bottom-right causal) */
  const double* sinks;       /* NULL, or one sink logit per query head */
  double sm_scale, k_scale, v_scale;
  int64_t n_rows; /* number of (token, q-head) rows to compute */
  const int32_t* row_token; /* NULL: every row in token-major order */
  const int32_t* row_head;
  double* out_o; /* [n_rows][head_dim_v] */
  double* out_lse; /* [n_rows] */
  int nthreads;
  int max_kv_len;
  int status;
} attn_job;


typedef struct {
  attn_job* job;
  int tid;
  int status;
} attn_worker;

static int kv_len_of(const attn_job* j, int b) {
  int np = j->kv_indptr[b + 1] - j->kv_indptr[b];
  return np > 0 ? (np - 1) * j->page_size + j->kv_last_page_len[b] : 0;
}

/* One output row: token t (global index into the packed query rows) and
 * query head h. Request b owns tokens qo_indptr[b] .. qo_indptr[b+1]-1; its
 * i-th new token sits at KV position P_b + i with P_b = L_b - qo_len_b, so it
 * sees keys 0 .. P_b + i (decode: qo_len 1, all L_b keys). With a tree mask
 * (speculative drafts with top-k above 1) the row sees every key before P_b
 * and, of the request's new tokens P_b + j with j <= i, those whose bit j is
 * set in tree_mask[t]: drafts are ordered with every ancestor before its
 * descendants, so bits above the row's own index are ignored. At most 64 new
 * tokens per request. GQA: query head h reads KV head h / (num_q_heads /
 * num_kv_heads). Scores contract the head_dim columns of q and k; the output
 * has the head_dim_v columns of v. With sinks, head h's sink logit joins the softmax as one
 * more score whose value vector is zero: it adds to the normaliser (and the
 * LSE) but not to o. */
static int key_visible(const uint64_t* tree_mask, uint64_t word, int p, int prefix, int limit) {
  if (p > limit) return 0;
  if (!tree_mask || p < prefix) return 1;
  return (int)((word >> (p - prefix)) & 1u);
}

static int attention_row(const attn_job* j, int t, int h, double* scores, double* qd, double* o, double* lse) {
  int D = j->head_dim, DV = j->head_dim_v;
  int b = 0;
  while (b < j->bs && j->qo_indptr[b + 1] <= t) ++b;
  if (b >= j->bs || t < j->qo_indptr[b]) return ORACLE_ERR_ARG;
  int i = t - j->qo_indptr[b];
  int qo_len = j->qo_indptr[b + 1] - j->qo_indptr[b];
  int L = kv_len_of(j, b);
  int prefix = L - qo_len;
  if (L > 0 && prefix < 0) return ORACLE_ERR_ARG;
  if (j->tree_mask && qo_len > 64) return ORACLE_ERR_ARG;
  int limit = L > 0 ? prefix + i : -1; /* last key position the row may see */
  uint64_t word = j->tree_mask ? j->tree_mask[t] : 0;
  int n_vis = 0;
  for (int p = 0; p <= limit; ++p) n_vis += key_visible(j->tree_mask, word, p, prefix, limit);
  int g = h / (j->num_q_heads / j->num_kv_heads);
  const uint16_t* qrow = j->q + ((int64_t)t * j->num_q_heads + h) * D;
  for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_decode(qrow[d]); /* the row's query, widened once */
  for (int d = 0; d < DV; ++d) o[d] = 0.0;
  double sink = j->sinks ? j->sinks[h] : -INFINITY;
  if (n_vis == 0) { /* no visible key: empty request (graph padding) or an empty mask row */
    *lse = sink; /* the sink alone (-inf without one); o stays zero */
    return ORACLE_OK;
  }
  /* scores s_j = sm_scale * sum_d q_d k_jd over the visible keys */
  double m = -INFINITY;
  for (int p = 0; p <= limit; ++p) {
    if (!key_visible(j->tree_mask, word, p, prefix, limit)) continue;
    int32_t page = j->kv_indices[j->kv_indptr[b] + p / j->page_size];
    int64_t slot = (int64_t)page * j->page_size + p % j->page_size;
    int64_t base = (slot * j->num_kv_heads + g) * D;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qd[d] * kv_value(j->k_pool, j->kv_dtype, base + d, j->k_scale);
    scores[p] = j->sm_scale * dot;
    if (scores[p] > m) m = scores[p];
  }
  if (sink > m) m = sink;
  /* softmax weights (the sink's term in the normaliser) and weighted sum of V */
  double z = sink > -INFINITY ? exp(sink - m) : 0.0;
  for (int p = 0; p <= limit; ++p)
    if (key_visible(j->tree_mask, word, p, prefix, limit)) z += exp(scores[p] - m);
  for (int p = 0; p <= limit; ++p) {
    if (!key_visible(j->tree_mask, word, p, prefix, limit)) continue;
    double w = exp(scores[p] - m) / z;
    int32_t page = j->kv_indices[j->kv_indptr[b] + p / j->page_size];
    int64_t slot = (int64_t)page * j->page_size + p % j->page_size;
    int64_t base = (slot * j->num_kv_heads + g) * DV;
    for (int d = 0; d < DV; ++d) o[d] += w * kv_value(j->v_pool, j->kv_dtype, base + d, j->v_scale);
  }
  *lse = m + log(z);
  return ORACLE_OK;
}

static void* attention_worker(void* arg) {
  attn_worker* w = (attn_worker*)arg;
  attn_job* j = w->job;
  double* scores = (double*)malloc(sizeof(double) * (size_t)(j->max_kv_len > 0 ? j->max_kv_len : 1));
  double* qd = (double*)malloc(sizeof(double) * (size_t)j->head_dim);
  if (!scores || !qd) {
    free(scores);
    free(qd);
    w->status = ORACLE_ERR_NOMEM;
    return NULL;
  }
  for (int64_t r = w->tid; r < j->n_rows; r += j->nthreads) {
    int t, h;
    if (j->row_token) {
      t = j->row_token[r];
      h = j->row_head[r];
    } else {
      t = (int)(r / j->num_q_heads);
      h = (int)(r % j->num_q_heads);
    }
    int st = attention_row(j, t, h, scores, qd, j->out_o + r * j->head_dim_v, j->out_lse + r);
    if (st != ORACLE_OK) w->status = st;
  }
  free(scores);
  free(qd);
  return NULL;
}

/* Attention for the requested rows. With row_token == NULL every row of the
 * batch is computed (n_rows must equal qo_indptr[bs] * num_q_heads) and the
 * outputs are laid out [token][q_head][head_dim_v] / [token][q_head]. Rows are
 * independent; threads take them round-robin. tree_mask: NULL, or one word
 * per query token; sinks: NULL, or one logit per query head (see
 * attention_row). */
int oracle_attention(int bs, int num_q_heads, int num_kv_heads, int head_dim, int head_dim_v, int page_size,
                     int kv_dtype,
                     const uint16_t* q, const void* k_pool, const void* v_pool, const int32_t* kv_indptr,
                     const int32_t* kv_indices, const int32_t* kv_last_page_len, const int32_t* qo_indptr,
                     const uint64_t* tree_mask, const double* sinks, double sm_scale, double k_scale, double v_scale, int64_t n_rows, const int32_t* row_token,
                     const int32_t* row_head, double* out_o, double* out_lse, int nthreads) {
  if (bs < 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || head_dim_v <= 0 ||
      page_size <= 0)
    return ORACLE_ERR_ARG;
  if (kv_dtype != ORACLE_KV_BF16 && kv_dtype != ORACLE_KV_FP8_E4M3) return ORACLE_ERR_ARG;
  if (nthreads < 1) nthreads = 1;
  attn_job job;
  memset(&job, 0, sizeof job);
  job.bs = bs;
  job.num_q_heads = num_q_heads;
  job.num_kv_heads = num_kv_heads;
  job.head_dim = head_dim;
  job.head_dim_v = head_dim_v;
  job.page_size = page_size;
  job.kv_dtype = kv_dtype;
  job.q = q;
  job.k_pool = k_pool;
  job.v_pool = v_pool;
  job.kv_indptr = kv_indptr;
  job.kv_indices = kv_indices;
  job.kv_last_page_len = kv_last_page_len;
  job.qo_indptr = qo_indptr;
  job.tree_mask = tree_mask;
  job.sinks = sinks;
  job.sm_scale = sm_scale;
  job.k_scale = k_scale;
  job.v_scale = v_scale;
  job.n_rows = n_rows;
  job.row_token = row_token;
  job.row_head = row_head;
  job.out_o = out_o;
  job.out_lse = out_lse;
  job.nthreads = nthreads;
  job.status = ORACLE_OK;
  if (!row_token && n_rows != (int64_t)qo_indptr[bs] * num_q_heads) return ORACLE_ERR_ARG;
  for (int b = 0; b < bs; ++b) {
    int L = kv_len_of(&job, b);
    if (L > job.max_kv_len) job.max_kv_len = L;
  }
  attn_worker* workers = (attn_worker*)calloc((size_t)nthreads, sizeof(attn_worker));
  pthread_t* threads = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!workers || !threads) {
    free(workers);
    free(threads);
    return ORACLE_ERR_NOMEM;
  }
  for (int i = 0; i < nthreads; ++i) {
    workers[i].job = &job;
    workers[i].tid = i;
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&threads[i], NULL, attention_worker, &workers[i]);
  attention_worker(&workers[0]);
  for (int i = 1; i < nthreads; ++i) pthread_join(threads[i], NULL);
  for (int i = 0; i < nthreads; ++i)
    if (workers[i].status != ORACLE_OK) job.status = workers[i].status;
  free(workers);
  free(threads);
  return job.status;
}

/* Bytes one pool (K or V) of one layer takes: slots * kv_heads * head_dim * elem. */
int64_t oracle_pool_bytes(int64_t num_slots, int num_kv_heads, int head_dim, int elem_bytes) {
  return num_slots * (int64_t)num_kv_heads * head_dim * elem_bytes;
}
