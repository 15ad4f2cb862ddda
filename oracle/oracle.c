/*
 * oracle.c -- fp64 CPU oracle for banded + global sparse attention (forward).
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's shared library; the product library
 * (the CUDA path) never links, loads or calls it, and the two share no source,
 * header, table or helper.  It is deliberately slow and plain: every mask row is
 * materialised as an explicit byte array, and the softmax runs over exactly the
 * positions that row marks.
 *
 * What is computed, per head and per query row i (all arithmetic in double):
 *
 *   mask row      S_i  (byte array of length N, 1 = row i scores key j)
 *   scores        s_j  = scale * sum_d q[i][d] * k[j][d]            for j in S_i
 *   row maximum   m    = max_{j in S_i} s_j
 *   weights       e_j  = exp(s_j - m)
 *   output        o[i] = sum_{j in S_i} e_j * v[j]  /  sum_{j in S_i} e_j
 *   log-sum-exp   lse  = m + log(sum_{j in S_i} e_j)
 *
 * Sources:
 *  - Attention itself: "Unlimiformer: Long-Range Transformers with Unlimited
 *    Length Input", section 2.3 "Attention reformulation", Eq. (1):
 *    Attn(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V.  `scale` stands for 1/sqrt(d_k)
 *    and is a parameter.
 *  - Sparse attention as a mask: "GMAT: Global Memory Augmentation for
 *    Transformers", section "Global-Memory Augmented Transformers": only some
 *    entries of Q K^T are computed, the rest masked by an additive binary mask
 *    B in {0, -inf}.  Adding -inf before the softmax is the same as leaving the
 *    entry out of the sum, which is what this file does (no -inf arithmetic).
 *  - The Longformer pattern: the Ultralytics glossary page "Longformer",
 *    section "How the Longformer attention works" (three bullets: sliding
 *    window, dilated sliding window, global attention) and the mask-count
 *    example printed in that section.
 *  - The GMAT pattern: "GMAT", subsection "Global Memory" (M memory tokens
 *    prefixed to the L main tokens; main tokens use a sparse pattern among
 *    themselves and dense attention to memory; memory tokens attend to all M+L)
 *    and subsection "Chunked self-attention" (C x k chunks plus memory).
 *
 * Readings where the pages are silent or garbled (each one is also listed in
 * the design notes):
 *  - "within +-w/2" is inclusive with integer half-width floor(w/2), as the
 *    glossary example's `<= window // 2` comparison makes it.
 *  - Dilation d: keys j = i + t*d with |t| <= floor(w/2), i.e. |i-j| <= floor(w/2)*d
 *    and (i-j) divisible by d.  The glossary says dilation keeps the cost and
 *    widens the reach; this reading keeps w+1 keys per interior row.
 *  - Global set: a set (duplicates collapse); a global row scores every key,
 *    every row scores every global key, and a pair is counted once even when
 *    it is both in the band and global.
 *  - The band is clipped to [0, N): no padding positions exist.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_DTYPE_BF16 0 /* raw bfloat16 bit patterns (uint16) */
#define ORACLE_DTYPE_FP32 1
#define ORACLE_DTYPE_FP64 2

#define ORACLE_PATTERN_LONGFORMER 0 /* band (+dilation per head) + global set  */
#define ORACLE_PATTERN_GMAT_BAND 1  /* M memory tokens + band on the main part */
#define ORACLE_PATTERN_GMAT_CHUNK 2 /* M memory tokens + C-long chunks         */

/* ------------------------------------------------------------------------ */
/* Element access.  bf16 -> double and fp32 -> double are exact.             */

static double load_elem(const void *base, int dtype, int64_t idx) {
  if (dtype == ORACLE_DTYPE_BF16) {
    uint16_t bits = ((const uint16_t *)base)[idx];
    uint32_t wide = ((uint32_t)bits) << 16; /* bf16 is the top half of fp32 */
    float f;
    memcpy(&f, &wide, sizeof f);
    return (double)f;
  }
  if (dtype == ORACLE_DTYPE_FP32) return (double)((const float *)base)[idx];
  return ((const double *)base)[idx];
}

/* ------------------------------------------------------------------------ */
/* Global set: sort and drop duplicates.  Returns the set size, or -1 if an  */
/* index lies outside [0, N).                                                */

static int cmp_i32(const void *a, const void *b) {
  int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
  return (x > y) - (x < y);
}

int oracle_global_set(const int32_t *idx, int n, int N, int32_t *out) {
  int i, m = 0;
  int32_t *tmp;
  if (n <= 0) return 0;
  tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
  if (!tmp) return -1;
  for (i = 0; i < n; ++i) {
    if (idx[i] < 0 || idx[i] >= N) {
      free(tmp);
      return -1;
    }
    tmp[i] = idx[i];
  }
  qsort(tmp, (size_t)n, sizeof(int32_t), cmp_i32);
  for (i = 0; i < n; ++i)
    if (m == 0 || tmp[i] != out[m - 1]) out[m++] = tmp[i];
  free(tmp);
  return m;
}

/* ------------------------------------------------------------------------ */
/* Mask rows.  Each builder writes row[j] in {0,1} for j in [0, N).          */

/* Longformer: sliding window of half-width floor(w/2) in steps of `dilation`,
 * plus the global set in both directions. */
void oracle_mask_row_longformer(int N, int window, int dilation,
                                const int32_t *globals, int n_globals, int i,
                                uint8_t *row) {
  int j, g;
  int64_t half = window / 2; /* floor for w >= 0 */
  int row_is_global = 0;
  for (g = 0; g < n_globals; ++g)
    if (globals[g] == i) row_is_global = 1;
  for (j = 0; j < N; ++j) {
    int64_t diff = (int64_t)i - (int64_t)j;
    int64_t dist = diff < 0 ? -diff : diff;
    int in_band = (dist <= half * (int64_t)dilation) && (diff % dilation == 0);
    row[j] = (uint8_t)(in_band || row_is_global);
  }
  for (g = 0; g < n_globals; ++g) row[globals[g]] = 1;
}

/* GMAT with a band on the main sequence: positions [0, M) are memory, [M, N)
 * the main sequence.  Main-main pairs use the band |i-j| <= floor(w/2);
 * memory rows and memory columns are dense. */
void oracle_mask_row_gmat_band(int N, int M, int window, int i, uint8_t *row) {
  int j;
  int64_t half = window / 2;
  for (j = 0; j < N; ++j) {
    int row_mem = i < M, col_mem = j < M;
    int64_t diff = (int64_t)i - (int64_t)j;
    int64_t dist = diff < 0 ? -diff : diff;
    if (row_mem || col_mem)
      row[j] = 1;
    else
      row[j] = (uint8_t)(dist <= half);
  }
}

/* GMAT C x k chunked self-attention: main token at position p >= M belongs to
 * chunk (p - M) / C and scores the main tokens of its own chunk and all memory;
 * memory rows are dense. */
void oracle_mask_row_gmat_chunk(int N, int M, int C, int i, uint8_t *row) {
  int j;
  for (j = 0; j < N; ++j) {
    if (i < M || j < M)
      row[j] = 1;
    else
      row[j] = (uint8_t)(((i - M) / C) == ((j - M) / C));
  }
}

typedef struct {
  int pattern;
  int N;
  int window;
  const int32_t *dilation; /* per head (Longformer pattern), NULL = all 1 */
  const int32_t *globals;  /* sorted, unique */
  int n_globals;
  int M; /* memory tokens (GMAT patterns) */
  int C; /* chunk length (GMAT chunk pattern) */
} mask_spec;

static void build_row(const mask_spec *ms, int head, int i, uint8_t *row) {
  if (ms->pattern == ORACLE_PATTERN_LONGFORMER) {
    int d = ms->dilation ? ms->dilation[head] : 1;
    oracle_mask_row_longformer(ms->N, ms->window, d, ms->globals, ms->n_globals,
                               i, row);
  } else if (ms->pattern == ORACLE_PATTERN_GMAT_BAND) {
    oracle_mask_row_gmat_band(ms->N, ms->M, ms->window, i, row);
  } else {
    oracle_mask_row_gmat_chunk(ms->N, ms->M, ms->C, i, row);
  }
}

/* ------------------------------------------------------------------------ */
/* Pair counts: materialise every mask row and add up its ones.              */

typedef struct {
  const mask_spec *ms;
  int head;
  int row_begin, row_end;
  int64_t count;
} count_job;

static void *count_worker(void *arg) {
  count_job *job = (count_job *)arg;
  uint8_t *row = (uint8_t *)malloc((size_t)job->ms->N);
  int i, j;
  job->count = 0;
  if (!row) {
    job->count = -1;
    return NULL;
  }
  for (i = job->row_begin; i < job->row_end; ++i) {
    build_row(job->ms, job->head, i, row);
    for (j = 0; j < job->ms->N; ++j) job->count += row[j];
  }
  free(row);
  return NULL;
}

static int64_t count_head(const mask_spec *ms, int head, int threads) {
  count_job *jobs;
  pthread_t *tids;
  int t, per;
  int64_t total = 0;
  if (threads < 1) threads = 1;
  if (threads > ms->N) threads = ms->N;
  jobs = (count_job *)calloc((size_t)threads, sizeof(count_job));
  tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return -1;
  }
  per = (ms->N + threads - 1) / threads;
  for (t = 0; t < threads; ++t) {
    jobs[t].ms = ms;
    jobs[t].head = head;
    jobs[t].row_begin = t * per < ms->N ? t * per : ms->N;
    jobs[t].row_end = (t + 1) * per < ms->N ? (t + 1) * per : ms->N;
    pthread_create(&tids[t], NULL, count_worker, &jobs[t]);
  }
  for (t = 0; t < threads; ++t) {
    pthread_join(tids[t], NULL);
    if (jobs[t].count < 0) total = -1;
    if (total >= 0) total += jobs[t].count;
  }
  free(jobs);
  free(tids);
  return total;
}

/* Per-head pair counts for the Longformer pattern.  `globals` must already be
 * the sorted unique set.  Returns 0, or -1 on allocation failure. */
int oracle_count_pairs_longformer(int N, int window, const int32_t *dilation,
                                  int H, const int32_t *globals, int n_globals,
                                  int threads, int64_t *per_head) {
  mask_spec ms;
  int h;
  memset(&ms, 0, sizeof ms);
  ms.pattern = ORACLE_PATTERN_LONGFORMER;
  ms.N = N;
  ms.window = window;
  ms.dilation = dilation;
  ms.globals = globals;
  ms.n_globals = n_globals;
  for (h = 0; h < H; ++h) {
    per_head[h] = count_head(&ms, h, threads);
    if (per_head[h] < 0) return -1;
  }
  return 0;
}

int64_t oracle_count_pairs_gmat(int pattern, int N, int M, int window, int C,
                                int threads) {
  mask_spec ms;
  memset(&ms, 0, sizeof ms);
  ms.pattern = pattern;
  ms.N = N;
  ms.M = M;
  ms.window = window;
  ms.C = C;
  return count_head(&ms, 0, threads);
}

/* Full mask of one head, row-major N x N bytes (small N only). */
void oracle_mask_longformer(int N, int window, int dilation,
                            const int32_t *globals, int n_globals,
                            uint8_t *mask) {
  int i;
  for (i = 0; i < N; ++i)
    oracle_mask_row_longformer(N, window, dilation, globals, n_globals, i,
                               mask + (int64_t)i * N);
}

void oracle_mask_gmat(int pattern, int N, int M, int window, int C,
                      uint8_t *mask) {
  int i;
  for (i = 0; i < N; ++i) {
    if (pattern == ORACLE_PATTERN_GMAT_BAND)
      oracle_mask_row_gmat_band(N, M, window, i, mask + (int64_t)i * N);
    else
      oracle_mask_row_gmat_chunk(N, M, C, i, mask + (int64_t)i * N);
  }
}

/* ------------------------------------------------------------------------ */
/* Forward pass.                                                             */

typedef struct {
  const mask_spec *ms;
  const void *q, *k, *v;
  /* separate global projections (Longformer pattern), or NULL: a global row
   * then scores q_g . k_g over all keys and averages v_g */
  const void *qg, *kg, *vg;
  int dtype;
  int B, H, N, D;
  double scale;
  const int64_t *rows; /* flattened (b*H + h)*N + i, or NULL for all rows */
  int64_t n_rows;
  double *out; /* [n_rows][D] in the order of `rows` */
  double *lse; /* [n_rows] or NULL */
  int64_t begin, end;
  int status;
} fwd_job;

/* Is position i one of the Longformer pattern's global positions? */
static int is_global(const mask_spec *ms, int i) {
  int g;
  for (g = 0; g < ms->n_globals; ++g)
    if (ms->globals[g] == i) return 1;
  return 0;
}

static void *fwd_worker(void *arg) {
  fwd_job *job = (fwd_job *)arg;
  const mask_spec *ms = job->ms;
  int N = job->N, D = job->D;
  uint8_t *row = (uint8_t *)malloc((size_t)N);
  double *s = (double *)malloc(sizeof(double) * (size_t)N);
  double *qi = (double *)malloc(sizeof(double) * (size_t)D);
  int64_t r;
  job->status = 0;
  if (!row || !s || !qi) {
    job->status = -1;
    free(row);
    free(s);
    free(qi);
    return NULL;
  }
  for (r = job->begin; r < job->end; ++r) {
    int64_t flat = job->rows ? job->rows[r] : r;
    int64_t bh = flat / N;
    int i = (int)(flat % N);
    int head = (int)(bh % job->H);
    int64_t base = bh * (int64_t)N * D; /* start of this (b,h) slice */
    double m = -INFINITY, z = 0.0;
    double *o = job->out + r * (int64_t)D;
    int j, d;

    const void *qs = job->q, *ks = job->k, *vs = job->v;
    if (job->qg && is_global(ms, i)) {
      qs = job->qg;
      ks = job->kg;
      vs = job->vg;
    }
    build_row(ms, head, i, row);
    for (d = 0; d < D; ++d)
      qi[d] = load_elem(qs, job->dtype, base + (int64_t)i * D + d);

    /* scores over the masked set, and their maximum */
    for (j = 0; j < N; ++j) {
      double acc = 0.0;
      if (!row[j]) continue;
      for (d = 0; d < D; ++d)
        acc += qi[d] * load_elem(ks, job->dtype, base + (int64_t)j * D + d);
      s[j] = job->scale * acc;
      if (s[j] > m) m = s[j];
    }
    /* weights, normaliser and weighted sum of values */
    for (d = 0; d < D; ++d) o[d] = 0.0;
    for (j = 0; j < N; ++j) {
      double e;
      if (!row[j]) continue;
      e = exp(s[j] - m);
      z += e;
      for (d = 0; d < D; ++d)
        o[d] += e * load_elem(vs, job->dtype, base + (int64_t)j * D + d);
    }
    for (d = 0; d < D; ++d) o[d] /= z;
    if (job->lse) job->lse[r] = m + log(z);
  }
  free(row);
  free(s);
  free(qi);
  return NULL;
}

static int run_forward(const mask_spec *ms, const void *q, const void *k,
                       const void *v, const void *qg, const void *kg, const void *vg,
                       int dtype, int B, int H, int N, int D,
                       double scale, const int64_t *rows, int64_t n_rows,
                       double *out, double *lse, int threads) {
  fwd_job *jobs;
  pthread_t *tids;
  int64_t total = rows ? n_rows : (int64_t)B * H * N, per;
  int t, status = 0;
  if (threads < 1) threads = 1;
  if (total < threads) threads = total > 0 ? (int)total : 1;
  jobs = (fwd_job *)calloc((size_t)threads, sizeof(fwd_job));
  tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return -1;
  }
  per = (total + threads - 1) / threads;
  for (t = 0; t < threads; ++t) {
    fwd_job *job = &jobs[t];
    job->ms = ms;
    job->q = q;
    job->k = k;
    job->v = v;
    job->qg = qg;
    job->kg = kg;
    job->vg = vg;
    job->dtype = dtype;
    job->B = B;
    job->H = H;
    job->N = N;
    job->D = D;
    job->scale = scale;
    job->rows = rows;
    job->n_rows = total;
    job->out = out;
    job->lse = lse;
    job->begin = (int64_t)t * per < total ? (int64_t)t * per : total;
    job->end = (int64_t)(t + 1) * per < total ? (int64_t)(t + 1) * per : total;
    pthread_create(&tids[t], NULL, fwd_worker, job);
  }
  for (t = 0; t < threads; ++t) {
    pthread_join(tids[t], NULL);
    if (jobs[t].status) status = -1;
  }
  free(jobs);
  free(tids);
  return status;
}

/* Longformer pattern.  q, k, v: [B, H, N, D] contiguous in `dtype`.
 * `globals` must be the sorted unique set (see oracle_global_set).
 * rows == NULL computes every row into out[B*H*N][D]; otherwise only the listed
 * flattened rows, in order, into out[n_rows][D].  Returns 0 or -1. */
int oracle_forward_longformer(const void *q, const void *k, const void *v,
                              int dtype, int B, int H, int N, int D, int window,
                              const int32_t *dilation, const int32_t *globals,
                              int n_globals, double scale, const int64_t *rows,
                              int64_t n_rows, double *out, double *lse,
                              int threads) {
  mask_spec ms;
  memset(&ms, 0, sizeof ms);
  ms.pattern = ORACLE_PATTERN_LONGFORMER;
  ms.N = N;
  ms.window = window;
  ms.dilation = dilation;
  ms.globals = globals;
  ms.n_globals = n_globals;
  return run_forward(&ms, q, k, v, NULL, NULL, NULL, dtype, B, H, N, D, scale, rows,
                     n_rows, out, lse, threads);
}

/* Longformer pattern with separate global projections (Ultralytics glossary
 * "Longformer", section "How the Longformer attention works": global attention
 * uses its own query, key and value projections).  Reading taken: a global row
 * scores qg_i . kg_j over every key j and averages vg; every other row -- its
 * band keys and its global keys alike -- uses q, k, v, as in sa_forward.
 * qg, kg, vg: [B, H, N, D] like q, k, v (only the global rows of qg are read). */
int oracle_forward_longformer_global_proj(const void *q, const void *k, const void *v,
                                          const void *qg, const void *kg, const void *vg,
                                          int dtype, int B, int H, int N, int D, int window,
                                          const int32_t *dilation, const int32_t *globals,
                                          int n_globals, double scale, const int64_t *rows,
                                          int64_t n_rows, double *out, double *lse,
                                          int threads) {
  mask_spec ms;
  memset(&ms, 0, sizeof ms);
  ms.pattern = ORACLE_PATTERN_LONGFORMER;
  ms.N = N;
  ms.window = window;
  ms.dilation = dilation;
  ms.globals = globals;
  ms.n_globals = n_globals;
  return run_forward(&ms, q, k, v, qg, kg, vg, dtype, B, H, N, D, scale, rows, n_rows,
                     out, lse, threads);
}

/* GMAT patterns over the concatenated [memory; main] sequence of length N. */
int oracle_forward_gmat(const void *q, const void *k, const void *v, int dtype,
                        int B, int H, int N, int D, int pattern, int M,
                        int window, int C, double scale, const int64_t *rows,
                        int64_t n_rows, double *out, double *lse, int threads) {
  mask_spec ms;
  memset(&ms, 0, sizeof ms);
  ms.pattern = pattern;
  ms.N = N;
  ms.M = M;
  ms.window = window;
  ms.C = C;
  return run_forward(&ms, q, k, v, NULL, NULL, NULL, dtype, B, H, N, D, scale, rows,
                     n_rows, out, lse, threads);
}

/* ------------------------------------------------------------------------ */
/* Attention over per-query key lists ("Unlimiformer", section 2.2
 * "Retrieval-augmented Cross-Attention" and section 2.3 Eq. (1): each query
 * attends only to the keys its retrieval returned, with the standard
 * dot-product attention over that set).                                     */
/*
 * q: [B, H, Nq, D]; k, v: [B, H, Nk, D]; idx: int32 [B, H, Nq, K] -- row i of
 * head (b, h) scores exactly the keys listed in idx[b][h][i][0..K).  Readings
 * (the pages describe retrieval of a top-k set and say nothing of ragged or
 * repeated lists):
 *   - an entry outside [0, Nk) (e.g. -1) is padding and is skipped;
 *   - the list is a sum: an index listed twice is counted twice (a top-k list
 *     has no repeats, so nothing changes for retrieval output);
 *   - a row whose list has no valid entry has output 0 and log-sum-exp -inf.
 * Per row, in double:
 *   s_t = scale * q_i . k_{idx_t}  for each valid entry t,  m = max_t s_t,
 *   o_i = sum_t exp(s_t - m) v_{idx_t} / sum_t exp(s_t - m),
 *   lse_i = m + log(sum_t exp(s_t - m)).
 */
typedef struct {
  const void *q, *k, *v;
  const int32_t *idx;
  int dtype;
  int H, Nq, Nk, D, K;
  double scale;
  const int64_t *rows; /* flattened (b*H + h)*Nq + i, or NULL for all rows */
  double *out, *lse;
  int64_t begin, end;
  int status;
} gather_job;

/* Is list entry j a key of the head (not padding)? */
static int gather_valid(int j, int Nk) { return j >= 0 && j < Nk; }

static void *gather_worker(void *arg) {
  gather_job *job = (gather_job *)arg;
  int D = job->D, K = job->K;
  double *s = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
  double *qi = (double *)malloc(sizeof(double) * (size_t)D);
  int64_t r;
  job->status = 0;
  if (!s || !qi) {
    job->status = -1;
    free(s);
    free(qi);
    return NULL;
  }
  for (r = job->begin; r < job->end; ++r) {
    int64_t flat = job->rows ? job->rows[r] : r;
    int64_t bh = flat / job->Nq;
    int64_t qbase = flat * D;                    /* this query row */
    int64_t kbase = bh * (int64_t)job->Nk * D;   /* this head's keys and values */
    const int32_t *list = job->idx + flat * K;
    double top = -INFINITY, total = 0.0;
    double *o = job->out + r * (int64_t)D;
    int t, d, n_valid = 0;
    for (d = 0; d < D; ++d) qi[d] = load_elem(job->q, job->dtype, qbase + d);
    /* scores of the listed keys, and their maximum */
    for (t = 0; t < K; ++t) {
      double dot = 0.0;
      if (!gather_valid(list[t], job->Nk)) continue;
      for (d = 0; d < D; ++d)
        dot += qi[d] * load_elem(job->k, job->dtype, kbase + (int64_t)list[t] * D + d);
      s[t] = job->scale * dot;
      if (s[t] > top) top = s[t];
      ++n_valid;
    }
    for (d = 0; d < D; ++d) o[d] = 0.0;
    if (n_valid == 0) {
      if (job->lse) job->lse[r] = -INFINITY;
      continue;
    }
    /* weights, normaliser and weighted sum of the listed values */
    for (t = 0; t < K; ++t) {
      double w;
      if (!gather_valid(list[t], job->Nk)) continue;
      w = exp(s[t] - top);
      total += w;
      for (d = 0; d < D; ++d)
        o[d] += w * load_elem(job->v, job->dtype, kbase + (int64_t)list[t] * D + d);
    }
    for (d = 0; d < D; ++d) o[d] = o[d] / total;
    if (job->lse) job->lse[r] = top + log(total);
  }
  free(s);
  free(qi);
  return NULL;
}

/* rows == NULL computes every row into out[B*H*Nq][D]; otherwise only the
 * listed flattened rows, in order.  Returns 0 or -1. */
int oracle_forward_gather(const void *q, const void *k, const void *v, const int32_t *idx,
                          int dtype, int B, int H, int Nq, int Nk, int D, int K,
                          double scale, const int64_t *rows, int64_t n_rows, double *out,
                          double *lse, int threads) {
  gather_job *jobs;
  pthread_t *tids;
  int64_t total = rows ? n_rows : (int64_t)B * H * Nq, per;
  int t, status = 0;
  if (threads < 1) threads = 1;
  if (total < threads) threads = total > 0 ? (int)total : 1;
  jobs = (gather_job *)calloc((size_t)threads, sizeof(gather_job));
  tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return -1;
  }
  per = (total + threads - 1) / threads;
  for (t = 0; t < threads; ++t) {
    gather_job *job = &jobs[t];
    job->q = q;
    job->k = k;
    job->v = v;
    job->idx = idx;
    job->dtype = dtype;
    job->H = H;
    job->Nq = Nq;
    job->Nk = Nk;
    job->D = D;
    job->K = K;
    job->scale = scale;
    job->rows = rows;
    job->out = out;
    job->lse = lse;
    job->begin = (int64_t)t * per < total ? (int64_t)t * per : total;
    job->end = (int64_t)(t + 1) * per < total ? (int64_t)(t + 1) * per : total;
    pthread_create(&tids[t], NULL, gather_worker, job);
  }
  for (t = 0; t < threads; ++t) {
    pthread_join(tids[t], NULL);
    if (jobs[t].status) status = -1;
  }
  free(jobs);
  free(tids);
  return status;
}
