/*
 * fp64 CPU oracle for padding-free packed bidirectional attention.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the independent definition that the CUDA
 * library is checked against. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load it. It shares no code, header, table or helper
 * with the CUDA library, and the CUDA library never calls it.
 *
 * Sources (all on the page "Source code for gigl.nn.packed_attention"):
 *   - module docstring, "Data flow of a packed forward": pack_sequences turns
 *     lengths into flat_index and cu_seqlens; the packed buffer is
 *     grid.flatten()[flat_index]; every sequence attends only to itself.
 *   - module docstring, "Constraints": cu_seqlens is int32, so the token count
 *     must fit in int32.
 *   - module docstring, "Example": lengths [3, 1, 2] with max_seq_len 3 give
 *     flat_index [0, 1, 2, 3, 6, 7]; output shapes [6, 2, 8] and, with the
 *     first-token query, [3, 2, 8].
 *   - function _padded_packed_attention: the reference path. Tokens are laid out
 *     on a zero-padded [num_sequences, max_seq_len] grid, padded keys are masked,
 *     scaled-dot-product attention runs per sequence and head, outputs are
 *     unpadded; in first-token mode each sequence's query sits in its first row
 *     and only that row is kept.
 *   - function packed_attention: every sequence must hold at least one token.
 *   - custom op gigl::varlen_attention: returns the output and the log-sum-exp
 *     of the scaled scores (natural log).
 *
 * Readings where the pages leave a step open:
 *   - masking of padded keys: the pages add finfo.min/2 to their scores; since
 *     every row has at least one real key that bias sends their weight to exactly
 *     zero, so here padded keys are excluded from the softmax outright.
 *   - lengths above max_seq_len would alias the next grid row: rejected like 0.
 *   - scale is an explicit argument (the pages use SDPA's default 1/sqrt(d)).
 *   - log-sum-exp layout: [H, Nq] fp64, natural log, no row padding.
 *   - the backward is the analytic gradient of softmax attention (the pages
 *     hand it to aten's backward kernel, which computes the same gradient).
 *   - local (sliding-window) attention: the packed-encoders README lists a
 *     "local-64" mode for ModernBERT geometry and FlashAttention's
 *     sliding-window pruning without defining them. Read as: the key at
 *     position j of a sequence is visible from the query at position r of the
 *     same sequence iff r - window_left <= j <= r + window_right; a negative
 *     bound is unbounded, so (-1, -1) is full attention and local-64 is
 *     (64, 64). A first-token query sits at position 0. Invisible keys get a
 *     score of -inf, i.e. weight exactly zero.
 *
 * Everything is fp64, written as plain loops over the definition, with a
 * pthread pool over (sequence, head) pairs and no blocking or fusion.
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_OK 0
#define ORC_BAD_LENGTH 2
#define ORC_OVERFLOW 3
#define ORC_NO_MEMORY 4
#define ORC_INVALID 5

/* ------------------------------------------------------------------------- */
/* pack_sequences: "Data flow of a packed forward" and "Example".             */
/*   cu_seqlens[0] = 0, cu_seqlens[i+1] = cu_seqlens[i] + L_i                 */
/*   flat_index lists i*S + j for i ascending, then j ascending, j < L_i.     */
/* ------------------------------------------------------------------------- */
int orc_pack_sequences(const int32_t* lengths, int64_t B, int64_t S,
                       int64_t* flat_index, int32_t* cu_seqlens, int64_t* num_tokens) {
  if (B < 0 || S < 1) return ORC_INVALID;
  int64_t total = 0;
  for (int64_t i = 0; i < B; ++i) {
    if (lengths[i] < 1 || lengths[i] > S) return ORC_BAD_LENGTH;
    total += lengths[i];
  }
  if (total >= ((int64_t)1 << 31)) return ORC_OVERFLOW;
  *num_tokens = total;
  if (cu_seqlens) {
    cu_seqlens[0] = 0;
    for (int64_t i = 0; i < B; ++i) cu_seqlens[i + 1] = cu_seqlens[i] + lengths[i];
  }
  if (flat_index) {
    int64_t t = 0;
    for (int64_t i = 0; i < B; ++i)
      for (int64_t j = 0; j < lengths[i]; ++j) flat_index[t++] = i * S + j;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Batch-major packed rows (several documents per padded row), page            */
/* "nemo_automodel.components.models.common.packing":                         */
/*  - is_indexed_packed_mask: an indexed packing mask marks document i of a    */
/*    row (1-based) with i and padding with 0, e.g. [1,1,1,2,2,3,3,0,0].       */
/*  - flatten_packed_sequence_metadata: row-local token indices [B, S] and     */
/*    row-local cumulative lengths [B, M+1], both -1 padded, become one flat   */
/*    token stream (indices into the padded [B, S] layout) and flat            */
/*    cu_seqlens; inconsistent layouts, boundaries or token counts are errors. */
/* Readings: padding is trailing in both layouts; documents are non-empty and  */
/* numbered 1, 2, ... in order within a row; row-local boundaries start at 0,  */
/* increase strictly and end at the row's token count; row-local token indices */
/* lie in [0, S). Rows follow each other in the flat stream.                   */
/* ------------------------------------------------------------------------- */

/* ids: [B][S]. Outputs (nullable) flat_index [N] = i*S + j for every nonzero */
/* ids[i][j] in row-major order, cu [D+1] with a boundary wherever a document */
/* starts, and the totals N and D. */
int orc_pack_document_ids(const int32_t* ids, int64_t B, int64_t S, int64_t* flat_index,
                          int32_t* cu, int64_t* num_tokens, int64_t* num_docs) {
  if (B < 0 || S < 1) return ORC_INVALID;
  int64_t n = 0, d = 0;
  for (int64_t i = 0; i < B; ++i) {
    int32_t prev = 0;
    for (int64_t j = 0; j < S; ++j) {
      const int32_t id = ids[i * S + j];
      if (id < 0) return ORC_INVALID;
      if (id == 0) {                     /* padding: nothing may follow it */
        prev = -1;
        continue;
      }
      if (prev < 0) return ORC_INVALID;  /* a document after padding */
      if (id == prev + 1) {              /* a new document starts here */
        if (cu) cu[d] = (int32_t)n;
        ++d;
      } else if (id != prev) {
        return ORC_INVALID;              /* skipped or repeated document number */
      }
      if (flat_index) flat_index[n] = i * S + j;
      ++n;
      if (n >= ((int64_t)1 << 31)) return ORC_OVERFLOW;
      prev = id;
    }
  }
  if (cu) cu[d] = (int32_t)n;
  *num_tokens = n;
  *num_docs = d;
  return ORC_OK;
}

/* tok: [B][S] row-local token indices, -1 padded; row_cu: [B][M1] row-local  */
/* cumulative lengths, -1 padded. Outputs as above. */
int orc_flatten_packed_metadata(const int64_t* tok, const int32_t* row_cu, int64_t B, int64_t S,
                                int64_t M1, int64_t* flat_index, int32_t* cu,
                                int64_t* num_tokens, int64_t* num_docs) {
  if (B < 0 || S < 1 || M1 < 1) return ORC_INVALID;
  int64_t n = 0, d = 0;
  for (int64_t i = 0; i < B; ++i) {
    int64_t nb = 0;                       /* tokens of row i */
    for (int64_t j = 0; j < S; ++j) {
      const int64_t t = tok[i * S + j];
      if (t == -1) continue;
      if (t < 0 || t >= S || nb != j) return ORC_INVALID;  /* bad index, or padding not trailing */
      if (flat_index) flat_index[n + nb] = i * S + t;
      ++nb;
    }
    const int32_t* rc = row_cu + i * M1;
    if (rc[0] != 0) return ORC_INVALID;
    int64_t k = 1;
    for (; k < M1 && rc[k] != -1; ++k) {
      if (rc[k] <= rc[k - 1]) return ORC_INVALID;       /* empty or decreasing document */
      if (cu) cu[d] = (int32_t)(n + rc[k - 1]);
      ++d;
    }
    if (rc[k - 1] != nb) return ORC_INVALID;             /* boundaries disagree with tokens */
    for (; k < M1; ++k)
      if (rc[k] != -1) return ORC_INVALID;               /* padding not trailing */
    n += nb;
    if (n >= ((int64_t)1 << 31)) return ORC_OVERFLOW;
  }
  if (cu) cu[d] = (int32_t)n;
  *num_tokens = n;
  *num_docs = d;
  return ORC_OK;
}

/* grid.flatten()[flat_index]: packed row t is padded row flat_index[t]. */
void orc_gather_rows(const uint8_t* padded, const int64_t* flat_index, int64_t N,
                     int64_t row_bytes, uint8_t* packed) {
  for (int64_t t = 0; t < N; ++t)
    memcpy(packed + t * row_bytes, padded + flat_index[t] * row_bytes, (size_t)row_bytes);
}

/* to_dense_batch with fill value 0: padded row i*S+j holds packed row
 * cu_seqlens[i]+j when j < L_i, zeros otherwise. */
void orc_scatter_rows(const uint8_t* packed, const int32_t* cu_seqlens, int64_t B, int64_t S,
                      int64_t row_bytes, uint8_t* padded) {
  for (int64_t i = 0; i < B; ++i) {
    int64_t len = cu_seqlens[i + 1] - cu_seqlens[i];
    for (int64_t j = 0; j < S; ++j) {
      uint8_t* dst = padded + (i * S + j) * row_bytes;
      if (j < len)
        memcpy(dst, packed + ((int64_t)cu_seqlens[i] + j) * row_bytes, (size_t)row_bytes);
      else
        memset(dst, 0, (size_t)row_bytes);
    }
  }
}

/* ------------------------------------------------------------------------- */
/* A small pthread pool over (sequence, head) pairs.                          */
/* ------------------------------------------------------------------------- */
typedef void (*orc_task_fn)(void* ctx, int64_t item, double* scratch);

typedef struct {
  orc_task_fn fn;
  void* ctx;
  int64_t num_items;
  size_t scratch_doubles;
  atomic_llong next;
  atomic_int failed;
} orc_pool;

static void* orc_worker(void* arg) {
  orc_pool* pool = (orc_pool*)arg;
  double* scratch = (double*)malloc(pool->scratch_doubles * sizeof(double) + 64);
  if (!scratch) {
    atomic_store(&pool->failed, 1);
    return NULL;
  }
  for (;;) {
    int64_t item = atomic_fetch_add(&pool->next, 1);
    if (item >= pool->num_items) break;
    pool->fn(pool->ctx, item, scratch);
  }
  free(scratch);
  return NULL;
}

static int orc_run(orc_task_fn fn, void* ctx, int64_t num_items, size_t scratch_doubles,
                   int nthreads) {
  orc_pool pool;
  pool.fn = fn;
  pool.ctx = ctx;
  pool.num_items = num_items;
  pool.scratch_doubles = scratch_doubles;
  atomic_init(&pool.next, 0);
  atomic_init(&pool.failed, 0);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t threads[256];
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&threads[started], NULL, orc_worker, &pool) != 0) break;
    ++started;
  }
  orc_worker(&pool);
  for (int t = 0; t < started; ++t) pthread_join(threads[t], NULL);
  return atomic_load(&pool.failed) ? ORC_NO_MEMORY : ORC_OK;
}

/* Local-attention visibility of key position j from query position r. */
static int orc_visible(int64_t r, int64_t j, int64_t wl, int64_t wr) {
  return (wl < 0 || j >= r - wl) && (wr < 0 || j <= r + wr);
}

/* ------------------------------------------------------------------------- */
/* Forward on the padded grid (_padded_packed_attention).                     */
/* q: [Nq, H, D] with Nq = N (full) or B (first token). k, v: [N, H, D].      */
/* o: shaped like q. lse: [H, Nq].                                            */
/* ------------------------------------------------------------------------- */
typedef struct {
  const double *q, *k, *v;
  const int32_t* cu;
  int64_t B, S, H, D, Nq;
  double scale;
  int first_token;
  int64_t wl, wr;
  double *o, *lse;
} orc_fwd_ctx;

/* One (sequence i, head h): lay the sequence out as a zero-padded S-row slab of
 * this head (the padded grid of the reference path), then run masked softmax
 * attention for every real query row and unpad the result. */
static void orc_fwd_task(void* vctx, int64_t item, double* scratch) {
  orc_fwd_ctx* c = (orc_fwd_ctx*)vctx;
  const int64_t i = item / c->H, h = item % c->H;
  const int64_t S = c->S, D = c->D, H = c->H;
  const int64_t start = c->cu[i], len = (int64_t)c->cu[i + 1] - c->cu[i];
  double* Qp = scratch;           /* [S][D] */
  double* Kp = Qp + S * D;        /* [S][D] */
  double* Vp = Kp + S * D;        /* [S][D] */
  double* s = Vp + S * D;         /* [S] scores of one query row */
  memset(Qp, 0, sizeof(double) * (size_t)(3 * S * D));
  for (int64_t j = 0; j < len; ++j) {
    for (int64_t c2 = 0; c2 < D; ++c2) {
      Kp[j * D + c2] = c->k[((start + j) * H + h) * D + c2];
      Vp[j * D + c2] = c->v[((start + j) * H + h) * D + c2];
    }
  }
  /* First-token mode: the sequence's single query occupies its first row. */
  const int64_t num_rows = c->first_token ? 1 : len;
  for (int64_t r = 0; r < num_rows; ++r) {
    const int64_t qrow = c->first_token ? i : start + r;
    for (int64_t c2 = 0; c2 < D; ++c2) Qp[r * D + c2] = c->q[(qrow * H + h) * D + c2];
  }
  for (int64_t r = 0; r < num_rows; ++r) {
    const int64_t orow = c->first_token ? i : start + r;
    double m = -INFINITY;
    for (int64_t j = 0; j < S; ++j) {
      if (j >= len) continue; /* padded key: excluded from the softmax */
      double acc = 0.0;
      for (int64_t c2 = 0; c2 < D; ++c2) acc += Qp[r * D + c2] * Kp[j * D + c2];
      s[j] = orc_visible(r, j, c->wl, c->wr) ? c->scale * acc : -INFINITY;
      if (s[j] > m) m = s[j];
    }
    double z = 0.0;
    for (int64_t j = 0; j < len; ++j) {
      s[j] = exp(s[j] - m);
      z += s[j];
    }
    double* out = c->o + (orow * H + h) * D;
    for (int64_t c2 = 0; c2 < D; ++c2) {
      double acc = 0.0;
      for (int64_t j = 0; j < len; ++j) acc += s[j] * Vp[j * D + c2];
      out[c2] = acc / z;
    }
    if (c->lse) c->lse[h * c->Nq + orow] = m + log(z);
  }
}

int orc_attention_fwd_local(const double* q, const double* k, const double* v,
                            const int32_t* cu, int64_t B, int64_t S, int64_t H, int64_t D,
                            double scale, int first_token, int64_t window_left,
                            int64_t window_right, double* o, double* lse, int nthreads) {
  if (B < 0 || S < 1 || H < 1 || D < 1) return ORC_INVALID;
  for (int64_t i = 0; i < B; ++i) {
    int64_t len = (int64_t)cu[i + 1] - cu[i];
    if (len < 1 || len > S) return ORC_BAD_LENGTH;
  }
  orc_fwd_ctx ctx = {q, k, v, cu, B, S, H, D, first_token ? B : (B ? cu[B] : 0),
                     scale, first_token, window_left, window_right, o, lse};
  return orc_run(orc_fwd_task, &ctx, B * H, (size_t)(3 * S * D + S), nthreads);
}

int orc_attention_fwd(const double* q, const double* k, const double* v, const int32_t* cu,
                      int64_t B, int64_t S, int64_t H, int64_t D, double scale,
                      int first_token, double* o, double* lse, int nthreads) {
  return orc_attention_fwd_local(q, k, v, cu, B, S, H, D, scale, first_token, -1, -1, o, lse,
                                 nthreads);
}

/* ------------------------------------------------------------------------- */
/* Forward for chosen (row, head) pairs, read straight from the packed        */
/* buffers: for large inputs, where the whole output is too costly.          */
/* rows[r] is a packed token index (full mode) or a sequence index (first     */
/* token mode). o: [R, D], lse: [R].                                          */
/* ------------------------------------------------------------------------- */
typedef struct {
  const double *q, *k, *v;
  const int32_t* cu;
  int64_t B, H, D;
  double scale;
  int first_token;
  int64_t wl, wr;
  const int64_t *rows, *heads;
  double *o, *lse;
} orc_rows_ctx;

static int64_t orc_sequence_of(const int32_t* cu, int64_t B, int64_t t) {
  int64_t lo = 0, hi = B; /* find i with cu[i] <= t < cu[i+1] */
  while (hi - lo > 1) {
    int64_t mid = (lo + hi) / 2;
    if (cu[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

static void orc_rows_task(void* vctx, int64_t r, double* s) {
  orc_rows_ctx* c = (orc_rows_ctx*)vctx;
  const int64_t H = c->H, D = c->D, h = c->heads[r];
  const int64_t i = c->first_token ? c->rows[r] : orc_sequence_of(c->cu, c->B, c->rows[r]);
  const int64_t start = c->cu[i], len = (int64_t)c->cu[i + 1] - c->cu[i];
  const double* qv = c->q + (c->rows[r] * H + h) * D;
  const int64_t pos = c->first_token ? 0 : c->rows[r] - start; /* query position */
  double m = -INFINITY;
  for (int64_t j = 0; j < len; ++j) {
    const double* kv = c->k + ((start + j) * H + h) * D;
    double acc = 0.0;
    for (int64_t c2 = 0; c2 < D; ++c2) acc += qv[c2] * kv[c2];
    s[j] = orc_visible(pos, j, c->wl, c->wr) ? c->scale * acc : -INFINITY;
    if (s[j] > m) m = s[j];
  }
  double z = 0.0;
  for (int64_t j = 0; j < len; ++j) {
    s[j] = exp(s[j] - m);
    z += s[j];
  }
  for (int64_t c2 = 0; c2 < D; ++c2) {
    double acc = 0.0;
    for (int64_t j = 0; j < len; ++j) acc += s[j] * c->v[((start + j) * H + h) * D + c2];
    c->o[r * D + c2] = acc / z;
  }
  c->lse[r] = m + log(z);
}

int orc_attention_fwd_rows_local(const double* q, const double* k, const double* v,
                                 const int32_t* cu, int64_t B, int64_t H, int64_t D,
                                 double scale, int first_token, int64_t window_left,
                                 int64_t window_right, const int64_t* rows,
                                 const int64_t* heads, int64_t R, double* o, double* lse,
                                 int nthreads) {
  int64_t max_len = 0;
  for (int64_t i = 0; i < B; ++i) {
    int64_t len = (int64_t)cu[i + 1] - cu[i];
    if (len < 1) return ORC_BAD_LENGTH;
    if (len > max_len) max_len = len;
  }
  orc_rows_ctx ctx = {q, k, v, cu, B, H, D, scale, first_token, window_left, window_right,
                      rows, heads, o, lse};
  return orc_run(orc_rows_task, &ctx, R, (size_t)max_len, nthreads);
}

int orc_attention_fwd_rows(const double* q, const double* k, const double* v,
                           const int32_t* cu, int64_t B, int64_t H, int64_t D, double scale,
                           int first_token, const int64_t* rows, const int64_t* heads,
                           int64_t R, double* o, double* lse, int nthreads) {
  return orc_attention_fwd_rows_local(q, k, v, cu, B, H, D, scale, first_token, -1, -1, rows,
                                      heads, R, o, lse, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Backward: analytic gradient of softmax attention, per (sequence, head).    */
/* For each query row r, with P_r = softmax_j(scale * q_r . k_j):             */
/*   O_r   = sum_j P_rj v_j                                                   */
/*   Dlt_r = dO_r . O_r                                                       */
/*   dS_rj = P_rj * (dO_r . v_j - Dlt_r)                                      */
/*   dq_r  = scale * sum_j dS_rj k_j                                          */
/*   dk_j += scale * dS_rj q_r                                                */
/*   dv_j += P_rj dO_r                                                        */
/* Every (sequence, head) writes a disjoint slice of dq, dk, dv.              */
/* The backward op of page "Source code for gigl.nn.packed_attention"         */
/* (gigl::varlen_attention_backward) takes the forward's saved output; when   */
/* that output is given (out != NULL), Dlt_r = dO_r . out_r uses it as saved  */
/* (in bf16 it is O_r rounded), otherwise the exact O_r above.                */
/* ------------------------------------------------------------------------- */
typedef struct {
  const double *q, *k, *v, *dout;
  const int32_t* cu;
  int64_t B, H, D;
  double scale;
  int first_token;
  int64_t wl, wr;
  double *dq, *dk, *dv;
  const double* out; /* saved output [Nq][H][D] or NULL */
} orc_bwd_ctx;

static void orc_bwd_task(void* vctx, int64_t item, double* scratch) {
  orc_bwd_ctx* c = (orc_bwd_ctx*)vctx;
  const int64_t i = item / c->H, h = item % c->H;
  const int64_t H = c->H, D = c->D;
  const int64_t start = c->cu[i], len = (int64_t)c->cu[i + 1] - c->cu[i];
  double* p = scratch;       /* [len] */
  double* orow = p + len;    /* [D] */
  for (int64_t j = 0; j < len; ++j)
    for (int64_t c2 = 0; c2 < D; ++c2) {
      c->dk[((start + j) * H + h) * D + c2] = 0.0;
      c->dv[((start + j) * H + h) * D + c2] = 0.0;
    }
  const int64_t num_rows = c->first_token ? 1 : len;
  for (int64_t r = 0; r < num_rows; ++r) {
    const int64_t qrow = c->first_token ? i : start + r;
    const double* qv = c->q + (qrow * H + h) * D;
    const double* gv = c->dout + (qrow * H + h) * D;
    double m = -INFINITY;
    for (int64_t j = 0; j < len; ++j) {
      const double* kv = c->k + ((start + j) * H + h) * D;
      double acc = 0.0;
      for (int64_t c2 = 0; c2 < D; ++c2) acc += qv[c2] * kv[c2];
      p[j] = orc_visible(r, j, c->wl, c->wr) ? c->scale * acc : -INFINITY;
      if (p[j] > m) m = p[j];
    }
    double z = 0.0;
    for (int64_t j = 0; j < len; ++j) {
      p[j] = exp(p[j] - m);
      z += p[j];
    }
    for (int64_t j = 0; j < len; ++j) p[j] /= z;
    for (int64_t c2 = 0; c2 < D; ++c2) {
      double acc = 0.0;
      for (int64_t j = 0; j < len; ++j) acc += p[j] * c->v[((start + j) * H + h) * D + c2];
      orow[c2] = acc;
    }
    const double* ov = c->out ? c->out + (qrow * H + h) * D : orow;
    double delta = 0.0;
    for (int64_t c2 = 0; c2 < D; ++c2) delta += gv[c2] * ov[c2];
    double* dqv = c->dq + (qrow * H + h) * D;
    for (int64_t c2 = 0; c2 < D; ++c2) dqv[c2] = 0.0;
    for (int64_t j = 0; j < len; ++j) {
      const double* kv = c->k + ((start + j) * H + h) * D;
      const double* vv = c->v + ((start + j) * H + h) * D;
      double dp = 0.0;
      for (int64_t c2 = 0; c2 < D; ++c2) dp += gv[c2] * vv[c2];
      const double ds = p[j] * (dp - delta);
      double* dkv = c->dk + ((start + j) * H + h) * D;
      double* dvv = c->dv + ((start + j) * H + h) * D;
      for (int64_t c2 = 0; c2 < D; ++c2) {
        dqv[c2] += c->scale * ds * kv[c2];
        dkv[c2] += c->scale * ds * qv[c2];
        dvv[c2] += p[j] * gv[c2];
      }
    }
  }
}

int orc_attention_bwd_saved(const double* q, const double* k, const double* v,
                            const double* dout, const double* out, const int32_t* cu,
                            int64_t B, int64_t H, int64_t D, double scale, int first_token,
                            int64_t window_left, int64_t window_right, double* dq, double* dk,
                            double* dv, int nthreads) {
  int64_t max_len = 0;
  for (int64_t i = 0; i < B; ++i) {
    int64_t len = (int64_t)cu[i + 1] - cu[i];
    if (len < 1) return ORC_BAD_LENGTH;
    if (len > max_len) max_len = len;
  }
  orc_bwd_ctx ctx = {q, k, v, dout, cu, B, H, D, scale, first_token, window_left,
                     window_right, dq, dk, dv, out};
  return orc_run(orc_bwd_task, &ctx, B * H, (size_t)(max_len + D), nthreads);
}

int orc_attention_bwd_local(const double* q, const double* k, const double* v,
                            const double* dout, const int32_t* cu, int64_t B, int64_t H,
                            int64_t D, double scale, int first_token, int64_t window_left,
                            int64_t window_right, double* dq, double* dk, double* dv,
                            int nthreads) {
  return orc_attention_bwd_saved(q, k, v, dout, NULL, cu, B, H, D, scale, first_token,
                                 window_left, window_right, dq, dk, dv, nthreads);
}

int orc_attention_bwd(const double* q, const double* k, const double* v, const double* dout,
                      const int32_t* cu, int64_t B, int64_t H, int64_t D, double scale,
                      int first_token, double* dq, double* dk, double* dv, int nthreads) {
  return orc_attention_bwd_local(q, k, v, dout, cu, B, H, D, scale, first_token, -1, -1, dq, dk,
                                 dv, nthreads);
}

/* ------------------------------------------------------------------------- */
/* The packed encoder layer tail (page "packed-encoders 0.1.0": fused          */
/* LayerNorm / residual-LayerNorm / RoPE / GeGLU kernels on the flat token     */
/* buffer, with position ids that restart at every sequence - section "Fully  */
/* packed execution": position_ids = cat(arange(L_i))). The pages name the     */
/* operations and ModernBERT's split-half RoPE convention; the formulas are    */
/* ModernBERT's:                                                               */
/*   RoPE: for head_dim D and i < D/2, with a = pos * theta^(-2i/D),          */
/*         out[i] = x[i] cos a - x[i+D/2] sin a, out[i+D/2] = x[i+D/2] cos a + */
/*         x[i] sin a;                                                        */
/*   LayerNorm: y = (h - mean(h)) / sqrt(var(h) + eps) * w (+ b), biased var;  */
/*   residual-LayerNorm: h = x + residual (also returned), then LayerNorm;     */
/*   GeGLU: y[f] = gelu(x[f]) * x[F + f] with the exact (erf) GELU.            */
/* ------------------------------------------------------------------------- */

/* pos[t] = t - cu[i] for the sequence i holding token t. */
void orc_packed_positions(const int32_t* cu, int64_t B, int64_t* pos) {
  for (int64_t i = 0; i < B; ++i)
    for (int64_t t = cu[i]; t < cu[i + 1]; ++t) pos[t] = t - cu[i];
}

/* x: [N][H][D], rotated in place. */
void orc_rope(double* x, const int64_t* pos, int64_t N, int64_t H, int64_t D, double theta) {
  const int64_t half = D / 2;
  for (int64_t t = 0; t < N; ++t)
    for (int64_t h = 0; h < H; ++h) {
      double* v = x + (t * H + h) * D;
      for (int64_t i = 0; i < half; ++i) {
        const double a = (double)pos[t] * pow(theta, -2.0 * (double)i / (double)D);
        const double c = cos(a), s = sin(a);
        const double x1 = v[i], x2 = v[i + half];
        v[i] = x1 * c - x2 * s;
        v[i + half] = x2 * c + x1 * s;
      }
    }
}

/* x, residual (nullable), y, residual_out (nullable): [N][C]; w [C]; b [C] nullable. */
void orc_layernorm(const double* x, const double* residual, const double* w, const double* b,
                   int64_t N, int64_t C, double eps, double* y, double* residual_out) {
  for (int64_t t = 0; t < N; ++t) {
    const double* xr = x + t * C;
    double mean = 0.0;
    for (int64_t c = 0; c < C; ++c) mean += xr[c] + (residual ? residual[t * C + c] : 0.0);
    mean /= (double)C;
    double var = 0.0;
    for (int64_t c = 0; c < C; ++c) {
      const double d = xr[c] + (residual ? residual[t * C + c] : 0.0) - mean;
      var += d * d;
    }
    var /= (double)C;
    const double rstd = 1.0 / sqrt(var + eps);
    for (int64_t c = 0; c < C; ++c) {
      const double h = xr[c] + (residual ? residual[t * C + c] : 0.0);
      if (residual_out) residual_out[t * C + c] = h;
      y[t * C + c] = (h - mean) * rstd * w[c] + (b ? b[c] : 0.0);
    }
  }
}

/* x: [N][2F] -> y: [N][F]. */
void orc_geglu(const double* x, int64_t N, int64_t F, double* y) {
  for (int64_t t = 0; t < N; ++t)
    for (int64_t f = 0; f < F; ++f) {
      const double a = x[t * 2 * F + f], g = x[t * 2 * F + F + f];
      y[t * F + f] = 0.5 * a * (1.0 + erf(a / sqrt(2.0))) * g;
    }
}

int orc_hardware_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}
