/*
 * unip_oracle.c -- plain, slow fp64 CPU oracle for packed / chunked prefill
 * attention with UniPrefill-style block selection.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA library; both sides only share the seeded
 * input generators.
 *
 * Conventions
 *   bf16 inputs are passed as their uint16 bit patterns and decoded exactly
 *   to double.  All arithmetic is double precision, one accumulator per sum,
 *   in index order.  Arrays are token-major ("THD"): q[N][Hq][D],
 *   k,v[N][Hkv][D]; paged cache [num_pages][page_size][Hkv][D];
 *   block_table[S][max_pages].
 *
 * Return value: 0 on success, a negative number when an input breaks the
 * stated layout (the oracle refuses rather than guesses).
 *
 * Sources (page titles as given on the pages):
 *   "Chunked Prefill" (Ultralytics glossary), section "Como funciona o
 *     pre-preenchimento segmentado": each chunk attends to the cached K/V of
 *     every earlier chunk plus its own tokens under a causal mask over
 *     absolute positions; the page's PyTorch example uses
 *     scaled_dot_product_attention, i.e. softmax(q k^T / sqrt(D)) v.
 *   same page, section "Tecnicas de servico relacionadas": PagedAttention
 *     keeps the KV cache in fixed-size pages.
 *   "Prepacking: A Simple Method for Fast Prefilling..." summary, sections
 *     "技术框架" / "关键设计": prompts packed into one sequence with a modified
 *     attention mask and positional encoding (block-diagonal causal mask,
 *     positions restarting per prompt).
 *   "[논문리뷰] UniPrefill ..." review, section 1 (Top-p token selection: the
 *     fewest blocks whose cumulative importance reaches p) and section 3
 *     (the sequence is split into blocks whose importance is estimated at a
 *     full-attention layer; dropped tokens leave every later sub-layer).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENOMEM (-2)

static double bf16_to_f64(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Segment holding token t: the s with cu[s] <= t < cu[s+1] (binary search). */
static int32_t segment_of(const int32_t *cu, int32_t S, int32_t t) {
  int32_t lo = 0, hi = S - 1;
  while (lo < hi) {
    int32_t mid = (lo + hi + 1) / 2;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  while (lo < S - 1 && cu[lo + 1] <= t) lo++;
  return lo;
}

static int check_segments(const int32_t *cu, int32_t S, const int32_t *pos, int32_t N) {
  if (S < 0 || N < 0 || cu[0] != 0 || cu[S] != N) return ORC_EINVAL;
  for (int32_t s = 0; s < S; s++) {
    if (cu[s + 1] < cu[s]) return ORC_EINVAL;
    if (cu[s + 1] > cu[s]) {
      int32_t p0 = pos[cu[s]];
      if (p0 < 0) return ORC_EINVAL;
      for (int32_t t = cu[s]; t < cu[s + 1]; t++)
        if (pos[t] != p0 + (t - cu[s])) return ORC_EINVAL;
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Attention                                                                  */
/* ------------------------------------------------------------------------ */
typedef struct {
  const uint16_t *q, *k, *v, *kc, *vc;
  const int32_t *cu, *pos, *bt, *rows;
  const int32_t *plen; /* compacted stream: explicit prefix length per segment (else NULL) */
  int32_t S, N, num_pages, page_size, max_pages, Hq, Hkv, D, n_rows;
  double scale;
  double *out, *lse;
  int64_t next, total;
  pthread_mutex_t lock;
  int err;
} attn_job_t;

static int64_t take_work(int64_t *next, pthread_mutex_t *lock, int64_t total) {
  pthread_mutex_lock(lock);
  int64_t w = *next;
  if (w < total) (*next)++;
  pthread_mutex_unlock(lock);
  return w < total ? w : -1;
}

/* Key (or value) vector number kk of segment s as seen from its queries:
 * kk <  P : cached prefix token kk, read through the segment's page table;
 * kk >= P : the segment's own token kk - P, read from the packed k / v. */
static const uint16_t *kv_row(const attn_job_t *J, int use_v, int32_t s, int32_t P, int32_t g, int64_t kk) {
  if (kk < P) {
    int32_t page = J->bt[(int64_t)s * J->max_pages + kk / J->page_size];
    int32_t slot = (int32_t)(kk % J->page_size);
    const uint16_t *base = use_v ? J->vc : J->kc;
    return base + (((int64_t)page * J->page_size + slot) * J->Hkv + g) * J->D;
  }
  const uint16_t *base = use_v ? J->v : J->k;
  return base + ((int64_t)(J->cu[s] + (kk - P)) * J->Hkv + g) * J->D;
}

static void *attn_worker(void *arg) {
  attn_job_t *J = (attn_job_t *)arg;
  double *sc = NULL, *acc = NULL;
  int64_t cap = 0;
  acc = (double *)malloc(sizeof(double) * (size_t)J->D);
  if (!acc) { J->err = ORC_ENOMEM; return NULL; }
  for (;;) {
    int64_t w = take_work(&J->next, &J->lock, J->total);
    if (w < 0) break;
    int32_t r = (int32_t)(w / J->Hq), h = (int32_t)(w % J->Hq);
    int32_t t = J->rows ? J->rows[r] : r;
    int32_t s = segment_of(J->cu, J->S, t);
    int32_t P = J->pos[J->cu[s]];
    int32_t i = t - J->cu[s];
    int32_t g = h / (J->Hq / J->Hkv);
    int64_t nk = (int64_t)P + i + 1; /* visible keys: whole prefix, own tokens 0..i */
    if (nk > cap) {
      free(sc);
      cap = nk;
      sc = (double *)malloc(sizeof(double) * (size_t)cap);
      if (!sc) { J->err = ORC_ENOMEM; free(acc); return NULL; }
    }
    const uint16_t *qr = J->q + ((int64_t)t * J->Hq + h) * J->D;
    double m = -INFINITY;
    for (int64_t kk = 0; kk < nk; kk++) {
      const uint16_t *kr = kv_row(J, 0, s, P, g, kk);
      double dot = 0.0;
      for (int32_t d = 0; d < J->D; d++) dot += bf16_to_f64(qr[d]) * bf16_to_f64(kr[d]);
      sc[kk] = dot * J->scale;
      if (sc[kk] > m) m = sc[kk];
    }
    double denom = 0.0;
    for (int32_t d = 0; d < J->D; d++) acc[d] = 0.0;
    for (int64_t kk = 0; kk < nk; kk++) {
      double e = exp(sc[kk] - m);
      denom += e;
      const uint16_t *vr = kv_row(J, 1, s, P, g, kk);
      for (int32_t d = 0; d < J->D; d++) acc[d] += e * bf16_to_f64(vr[d]);
    }
    double *o = J->out + ((int64_t)r * J->Hq + h) * J->D;
    for (int32_t d = 0; d < J->D; d++) o[d] = acc[d] / denom;
    if (J->lse) J->lse[(int64_t)r * J->Hq + h] = m + log(denom);
  }
  free(sc);
  free(acc);
  return NULL;
}

static int run_threads(void *(*fn)(void *), void *job, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) return ORC_ENOMEM;
  int started = 0;
  for (int i = 0; i < nthreads; i++) {
    if (pthread_create(&th[i], NULL, fn, job) != 0) break;
    started++;
  }
  if (started == 0) fn(job);
  for (int i = 0; i < started; i++) pthread_join(th[i], NULL);
  free(th);
  return ORC_OK;
}

/*
 * Causal attention of a packed (and possibly chunked) token stream.
 *
 * Segment s holds tokens cu[s] .. cu[s+1]-1 with contiguous positions; its
 * cached prefix length is P_s = pos[cu[s]].  Token t (segment-local index i,
 * position P_s + i) with query head h attends, with kv head g = h / (Hq/Hkv),
 * to the P_s prefix keys (from the pages named by block_table row s) and to
 * the segment's own tokens 0..i.  Tokens of other segments are never visible
 * (block-diagonal mask).  out = softmax(scale * q k^T) v, lse = natural-log
 * sum of exp of the scaled scores.
 *
 * rows (optional): token indices to evaluate; out is then [n_rows][Hq][D]
 * and lse [n_rows][Hq].  With rows == NULL every token is evaluated and
 * n_rows must equal N.
 */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const int32_t *cu_seqlens, int32_t num_segs,
                     const int32_t *positions, int32_t total_tokens,
                     const uint16_t *k_cache, const uint16_t *v_cache,
                     int32_t num_pages, int32_t page_size,
                     const int32_t *block_table, int32_t max_pages,
                     int32_t Hq, int32_t Hkv, int32_t D, double scale,
                     const int32_t *rows, int32_t n_rows,
                     double *out, double *lse, int32_t nthreads) {
  if (Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return ORC_EINVAL;
  if (check_segments(cu_seqlens, num_segs, positions, total_tokens)) return ORC_EINVAL;
  if (!rows && n_rows != total_tokens) return ORC_EINVAL;
  for (int32_t s = 0; s < num_segs; s++) {
    if (cu_seqlens[s + 1] == cu_seqlens[s]) continue;
    int32_t P = positions[cu_seqlens[s]];
    if (P == 0) continue;
    if (!k_cache || !v_cache || !block_table || page_size <= 0) return ORC_EINVAL;
    int32_t need = (P + page_size - 1) / page_size;
    if (need > max_pages) return ORC_EINVAL;
    for (int32_t p = 0; p < need; p++) {
      int32_t pg = block_table[(int64_t)s * max_pages + p];
      if (pg < 0 || pg >= num_pages) return ORC_EINVAL;
    }
  }
  if (rows)
    for (int32_t r = 0; r < n_rows; r++)
      if (rows[r] < 0 || rows[r] >= total_tokens) return ORC_EINVAL;
  attn_job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.kc = k_cache; J.vc = v_cache;
  J.cu = cu_seqlens; J.pos = positions; J.bt = block_table; J.rows = rows;
  J.S = num_segs; J.N = total_tokens; J.num_pages = num_pages; J.page_size = page_size;
  J.max_pages = max_pages; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.n_rows = n_rows;
  J.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)D);
  J.out = out; J.lse = lse; J.next = 0; J.total = (int64_t)n_rows * Hq;
  pthread_mutex_init(&J.lock, NULL);
  int rc = run_threads(attn_worker, &J, nthreads);
  pthread_mutex_destroy(&J.lock);
  return rc ? rc : J.err;
}

/*
 * Attention over a compacted stream (the UniPrefill review, section 3: the
 * tokens dropped by the selection leave every later sub-layer).  Segment s
 * holds its kept tokens cu[s] .. cu[s+1]-1 with their original positions,
 * increasing but possibly with gaps; its cached prefix (pages of block_table
 * row s) holds plen[s] tokens, which need not equal the first position (a
 * later layer's cache holds kept tokens only).  Token t with query head h
 * attends to the whole prefix and to the segment's own tokens u whose
 * position is at most t's (pos[u] <= pos[t]); the rest as oracle_attention.
 */
static void *attn_compacted_worker(void *arg) {
  attn_job_t *J = (attn_job_t *)arg;
  double *sc = NULL, *acc = NULL;
  int32_t *vis = NULL;
  int64_t cap = 0;
  acc = (double *)malloc(sizeof(double) * (size_t)J->D);
  vis = (int32_t *)malloc(sizeof(int32_t) * (size_t)(J->N > 0 ? J->N : 1));
  if (!acc || !vis) { J->err = ORC_ENOMEM; free(acc); free(vis); return NULL; }
  for (;;) {
    int64_t w = take_work(&J->next, &J->lock, J->total);
    if (w < 0) break;
    int32_t r = (int32_t)(w / J->Hq), h = (int32_t)(w % J->Hq);
    int32_t t = J->rows ? J->rows[r] : r;
    int32_t s = segment_of(J->cu, J->S, t);
    int32_t c0 = J->cu[s], n = J->cu[s + 1] - c0;
    int32_t P = J->plen[s];
    int32_t g = h / (J->Hq / J->Hkv);
    int32_t n_own = 0; /* own tokens at or before t's position */
    for (int32_t u = 0; u < n; u++)
      if (J->pos[c0 + u] <= J->pos[t]) vis[n_own++] = u;
    int64_t nk = (int64_t)P + n_own;
    if (nk > cap) {
      free(sc);
      cap = nk;
      sc = (double *)malloc(sizeof(double) * (size_t)cap);
      if (!sc) { J->err = ORC_ENOMEM; free(acc); free(vis); return NULL; }
    }
    const uint16_t *qr = J->q + ((int64_t)t * J->Hq + h) * J->D;
    double m = -INFINITY;
    for (int64_t kk = 0; kk < nk; kk++) {
      const uint16_t *kr = kv_row(J, 0, s, P, g, kk < P ? kk : (int64_t)P + vis[kk - P]);
      double dot = 0.0;
      for (int32_t d = 0; d < J->D; d++) dot += bf16_to_f64(qr[d]) * bf16_to_f64(kr[d]);
      sc[kk] = dot * J->scale;
      if (sc[kk] > m) m = sc[kk];
    }
    double denom = 0.0;
    for (int32_t d = 0; d < J->D; d++) acc[d] = 0.0;
    for (int64_t kk = 0; kk < nk; kk++) {
      double e = exp(sc[kk] - m);
      denom += e;
      const uint16_t *vr = kv_row(J, 1, s, P, g, kk < P ? kk : (int64_t)P + vis[kk - P]);
      for (int32_t d = 0; d < J->D; d++) acc[d] += e * bf16_to_f64(vr[d]);
    }
    double *o = J->out + ((int64_t)r * J->Hq + h) * J->D;
    for (int32_t d = 0; d < J->D; d++) o[d] = acc[d] / denom;
    if (J->lse) J->lse[(int64_t)r * J->Hq + h] = m + log(denom);
  }
  free(sc);
  free(acc);
  free(vis);
  return NULL;
}

int oracle_attention_compacted(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               const int32_t *cu_seqlens, int32_t num_segs,
                               const int32_t *positions, const int32_t *prefix_lens, int32_t total_tokens,
                               const uint16_t *k_cache, const uint16_t *v_cache,
                               int32_t num_pages, int32_t page_size,
                               const int32_t *block_table, int32_t max_pages,
                               int32_t Hq, int32_t Hkv, int32_t D, double scale,
                               const int32_t *rows, int32_t n_rows,
                               double *out, double *lse, int32_t nthreads) {
  if (Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || !prefix_lens) return ORC_EINVAL;
  if (num_segs < 0 || total_tokens < 0 || cu_seqlens[0] != 0 || cu_seqlens[num_segs] != total_tokens)
    return ORC_EINVAL;
  if (!rows && n_rows != total_tokens) return ORC_EINVAL;
  for (int32_t s = 0; s < num_segs; s++) {
    int32_t a = cu_seqlens[s], b = cu_seqlens[s + 1];
    if (b < a || prefix_lens[s] < 0) return ORC_EINVAL;
    for (int32_t t = a; t < b; t++) /* positions increase inside a segment */
      if (positions[t] < 0 || (t > a && positions[t] <= positions[t - 1])) return ORC_EINVAL;
    int32_t P = prefix_lens[s];
    if (P == 0 || a == b) continue;
    if (!k_cache || !v_cache || !block_table || page_size <= 0) return ORC_EINVAL;
    int32_t need = (P + page_size - 1) / page_size;
    if (need > max_pages) return ORC_EINVAL;
    for (int32_t p = 0; p < need; p++) {
      int32_t pg = block_table[(int64_t)s * max_pages + p];
      if (pg < 0 || pg >= num_pages) return ORC_EINVAL;
    }
  }
  if (rows)
    for (int32_t r = 0; r < n_rows; r++)
      if (rows[r] < 0 || rows[r] >= total_tokens) return ORC_EINVAL;
  attn_job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.kc = k_cache; J.vc = v_cache;
  J.cu = cu_seqlens; J.pos = positions; J.plen = prefix_lens; J.bt = block_table; J.rows = rows;
  J.S = num_segs; J.N = total_tokens; J.num_pages = num_pages; J.page_size = page_size;
  J.max_pages = max_pages; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.n_rows = n_rows;
  J.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)D);
  J.out = out; J.lse = lse; J.next = 0; J.total = (int64_t)n_rows * Hq;
  pthread_mutex_init(&J.lock, NULL);
  int rc = run_threads(attn_compacted_worker, &J, nthreads);
  pthread_mutex_destroy(&J.lock);
  return rc ? rc : J.err;
}

/* ------------------------------------------------------------------------ */
/* Block importance                                                           */
/* ------------------------------------------------------------------------ */
typedef struct {
  const uint16_t *q, *k;
  const double *lse;
  const int32_t *cu, *blk_cu, *seg_list;
  int32_t n_seg_list, Hq, Hkv, D, B;
  double scale;
  double *mass; /* [num_blocks_total][Hq] per-head block mass */
  int64_t next, total;
  pthread_mutex_t lock;
} imp_job_t;

static void *imp_worker(void *arg) {
  imp_job_t *J = (imp_job_t *)arg;
  for (;;) {
    int64_t w = take_work(&J->next, &J->lock, J->total);
    if (w < 0) break;
    int32_t s = J->seg_list[w / J->Hq], h = (int32_t)(w % J->Hq);
    int32_t c0 = J->cu[s], n = J->cu[s + 1] - J->cu[s];
    int32_t g = h / (J->Hq / J->Hkv);
    int32_t W = n < J->B ? n : J->B; /* scoring window: the last min(B, n) query rows */
    double *mass = J->mass + (int64_t)J->blk_cu[s] * J->Hq;
    for (int32_t i = n - W; i < n; i++) {
      const uint16_t *qr = J->q + ((int64_t)(c0 + i) * J->Hq + h) * J->D;
      double l = J->lse[(int64_t)(c0 + i) * J->Hq + h];
      for (int32_t j = 0; j <= i; j++) { /* the segment's own keys visible from row i */
        const uint16_t *kr = J->k + ((int64_t)(c0 + j) * J->Hkv + g) * J->D;
        double dot = 0.0;
        for (int32_t d = 0; d < J->D; d++) dot += bf16_to_f64(qr[d]) * bf16_to_f64(kr[d]);
        mass[(int64_t)(j / J->B) * J->Hq + h] += exp(dot * J->scale - l);
      }
    }
  }
  return NULL;
}

/*
 * Block importance of each selected segment (seg_mask[s] != 0, or all when
 * seg_mask is NULL).  Blocks are segment-local: block b covers local tokens
 * [b*B, min((b+1)*B, n)).  The scoring window is the last min(B, n) query
 * rows of the segment; each window row t and head h spreads the attention
 * probability exp(s_tj - lse_t) over the segment's own visible keys j, and a
 * block's mass is the sum over heads, window rows and its keys.  imp is the
 * mass divided by the segment's total mass.
 *
 * lse: [N][Hq] natural-log normalisers of the full attention rows (prefix
 * included); only window rows are read.
 * blk_cu (out, S+1): block offsets; unselected segments own zero blocks.
 * imp (out): one value per block, capacity imp_cap.
 */
int oracle_block_importance(const uint16_t *q, const uint16_t *k, const double *lse,
                            const int32_t *cu_seqlens, int32_t num_segs, int32_t total_tokens,
                            const uint8_t *seg_mask, int32_t block_size,
                            int32_t Hq, int32_t Hkv, int32_t D, double scale,
                            double *imp, int64_t imp_cap, int32_t *blk_cu, int32_t nthreads) {
  if (Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || block_size <= 0) return ORC_EINVAL;
  if (num_segs < 0 || cu_seqlens[0] != 0 || cu_seqlens[num_segs] != total_tokens) return ORC_EINVAL;
  int32_t *seg_list = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_segs + 1));
  if (!seg_list) return ORC_ENOMEM;
  int32_t n_list = 0;
  blk_cu[0] = 0;
  for (int32_t s = 0; s < num_segs; s++) {
    int32_t n = cu_seqlens[s + 1] - cu_seqlens[s];
    if (n < 0) { free(seg_list); return ORC_EINVAL; }
    int32_t nb = 0;
    if ((!seg_mask || seg_mask[s]) && n > 0) {
      nb = (n + block_size - 1) / block_size;
      seg_list[n_list++] = s;
    }
    blk_cu[s + 1] = blk_cu[s] + nb;
  }
  int64_t nblk = blk_cu[num_segs];
  if (nblk > imp_cap) { free(seg_list); return ORC_EINVAL; }
  double *mass = (double *)calloc((size_t)(nblk > 0 ? nblk : 1) * (size_t)Hq, sizeof(double));
  if (!mass) { free(seg_list); return ORC_ENOMEM; }
  imp_job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.lse = lse; J.cu = cu_seqlens; J.blk_cu = blk_cu; J.seg_list = seg_list;
  J.n_seg_list = n_list; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.B = block_size;
  J.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)D);
  J.mass = mass; J.next = 0; J.total = (int64_t)n_list * Hq;
  pthread_mutex_init(&J.lock, NULL);
  run_threads(imp_worker, &J, nthreads);
  pthread_mutex_destroy(&J.lock);
  for (int32_t li = 0; li < n_list; li++) {
    int32_t s = seg_list[li];
    double total = 0.0;
    for (int32_t b = blk_cu[s]; b < blk_cu[s + 1]; b++) {
      double m = 0.0;
      for (int32_t h = 0; h < Hq; h++) m += mass[(int64_t)b * Hq + h];
      imp[b] = m;
      total += m;
    }
    for (int32_t b = blk_cu[s]; b < blk_cu[s + 1]; b++) imp[b] = imp[b] / total;
  }
  free(mass);
  free(seg_list);
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Top-p block selection                                                      */
/* ------------------------------------------------------------------------ */
#define ORC_KEEP_FIRST 1u
#define ORC_KEEP_LAST 2u

typedef struct { uint32_t bits; int32_t idx; } rank_t;

/* Larger importance first; equal importance: lower block index first. */
static int rank_cmp(const void *a, const void *b) {
  const rank_t *x = (const rank_t *)a, *y = (const rank_t *)b;
  if (x->bits != y->bits) return x->bits > y->bits ? -1 : 1;
  return x->idx < y->idx ? -1 : (x->idx > y->idx ? 1 : 0);
}

/*
 * Top-p over each segment's blocks, on the float32 scores imp (as produced
 * by the importance step).  Steps, per segment with nb > 0 blocks:
 *   1. each score becomes a 32.32 fixed-point integer q_b = floor(imp_b * 2^32);
 *   2. T = sum of q_b (exact integer);
 *   3. threshold thr = p * T in double;
 *   4. forced set F = {first block, last block} (per flags); cum = sum over F;
 *   5. the other blocks are ranked by score, larger first, ties by lower index;
 *   6. while cum < thr, the next ranked block is added.
 * When T == 0 every block is kept.  Segments with nb == 0 are skipped.
 * keep[b] (out): 1 for kept blocks, 0 otherwise.
 */
int oracle_topp_select(const float *imp, const int32_t *blk_cu, int32_t num_segs,
                       double p, uint32_t flags, uint8_t *keep) {
  if (!(p >= 0.0 && p <= 1.0)) return ORC_EINVAL;
  for (int32_t s = 0; s < num_segs; s++) {
    int32_t b0 = blk_cu[s], nb = blk_cu[s + 1] - blk_cu[s];
    if (nb < 0) return ORC_EINVAL;
    if (nb == 0) continue;
    uint64_t *qv = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)nb);
    rank_t *rk = (rank_t *)malloc(sizeof(rank_t) * (size_t)nb);
    if (!qv || !rk) { free(qv); free(rk); return ORC_ENOMEM; }
    uint64_t T = 0;
    for (int32_t b = 0; b < nb; b++) {
      float f = imp[b0 + b];
      if (!(f >= 0.0f) || f > 1.0f) { free(qv); free(rk); return ORC_EINVAL; }
      if (f == 0.0f) f = 0.0f; /* -0 is the zero score */
      qv[b] = (uint64_t)floor((double)f * 4294967296.0);
      T += qv[b];
      keep[b0 + b] = 0;
    }
    if (T == 0) {
      for (int32_t b = 0; b < nb; b++) keep[b0 + b] = 1;
      free(qv); free(rk);
      continue;
    }
    double thr = p * (double)T;
    uint64_t cum = 0;
    if (flags & ORC_KEEP_FIRST) keep[b0] = 1;
    if (flags & ORC_KEEP_LAST) keep[b0 + nb - 1] = 1;
    int32_t R = 0;
    for (int32_t b = 0; b < nb; b++) {
      if (keep[b0 + b]) { cum += qv[b]; continue; }
      float f = imp[b0 + b];
      if (f == 0.0f) f = 0.0f; /* -0 ranks as the zero score */
      uint32_t bits;
      memcpy(&bits, &f, sizeof bits);
      rk[R].bits = bits;
      rk[R].idx = b;
      R++;
    }
    qsort(rk, (size_t)R, sizeof(rank_t), rank_cmp);
    for (int32_t r = 0; r < R && (double)cum < thr; r++) {
      keep[b0 + rk[r].idx] = 1;
      cum += qv[rk[r].idx];
    }
    free(qv);
    free(rk);
  }
  return ORC_OK;
}

/*
 * Compaction indices.  Kept tokens are listed segment by segment in their
 * original order: a token of a scored segment is kept when its block is kept;
 * every token of a segment with zero blocks (not scored) is kept.
 * gather_idx[i]: source token of kept row i; cu_kept: kept-token offsets per
 * segment; pos_kept: original positions; *n_kept: number of kept tokens.
 */
int oracle_index_build(const uint8_t *keep, const int32_t *blk_cu, const int32_t *cu_seqlens,
                       const int32_t *positions, int32_t num_segs, int32_t block_size,
                       int32_t *gather_idx, int32_t *cu_kept, int32_t *pos_kept, int32_t *n_kept) {
  if (block_size <= 0) return ORC_EINVAL;
  int32_t o = 0;
  cu_kept[0] = 0;
  for (int32_t s = 0; s < num_segs; s++) {
    int32_t c0 = cu_seqlens[s], n = cu_seqlens[s + 1] - cu_seqlens[s];
    int32_t nb = blk_cu[s + 1] - blk_cu[s];
    if (nb != 0 && nb != (n + block_size - 1) / block_size) return ORC_EINVAL;
    for (int32_t i = 0; i < n; i++) {
      if (nb == 0 || keep[blk_cu[s] + i / block_size]) {
        gather_idx[o] = c0 + i;
        pos_kept[o] = positions[c0 + i];
        o++;
      }
    }
    cu_kept[s + 1] = o;
  }
  *n_kept = o;
  return ORC_OK;
}

/* Row gather: out[i][:] = hidden[gather_idx[i]][:], bit for bit. */
int oracle_gather(const uint16_t *hidden, int64_t row_stride, int32_t d_model,
                  const int32_t *gather_idx, int32_t n_kept, int32_t n_rows_in, uint16_t *out) {
  for (int32_t i = 0; i < n_kept; i++) {
    int32_t src = gather_idx[i];
    if (src < 0 || src >= n_rows_in) return ORC_EINVAL;
    memcpy(out + (int64_t)i * d_model, hidden + (int64_t)src * row_stride,
           sizeof(uint16_t) * (size_t)d_model);
  }
  return ORC_OK;
}
