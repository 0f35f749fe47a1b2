/*
 * oracle.c -- plain fp64 CPU oracle for top-k block-sparse GQA attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; it shares no code, header or constant with the CUDA
 * path.  It is used by the tests (parity), by the package's smoke check and by
 * the benchmark's CPU-baseline leg.
 *
 * Every function is the plain definition written out in double precision, on
 * the exact stored input values widened to double.  No blocking, fusion or
 * reordering beyond the definitions.  Sources (web summaries of the papers):
 *
 *  - "How Much Dense Attention is Necessary? Oracle-Guided Sparse Prefill ..."
 *    Sec. 2.1: the dense attention distribution per query, aggregated over the
 *    query heads, ranks the keys; the top-k under a fixed budget form the
 *    support (shared by a block of consecutive queries when b_sel > 1), and
 *    attention is recomputed exactly, with the original q, k, v, on that
 *    support only.                              -> orc_mass, orc_select, orc_attend
 *  - "Faster Than Flash" Sec. 1 and 3: a small compressed sketch of the cache
 *    is scanned to estimate importance, and only the selected blocks are then
 *    loaded for exact attention; sink (initial) and local tokens dominate.
 *                                              -> orc_block_means, orc_*_scores
 *  - "Pulsar Attention" Phase 1: a fixed attention-sink prefix is kept.
 *  - "Pulsar Attention" Phase 2: per-shard partial softmaxes merge exactly
 *    (online softmax) -- the oracle computes each row in one piece.
 *
 * Readings where the pages are silent (listed with reasons in the design notes):
 * scale = 1/sqrt(d); sketch = mean of a block's valid key rows; sketch score of
 * a block = max over the group's query rows of scale * q . sketch; mass score =
 * sum over the group's rows of the per-block probability mass; ties go to the
 * lower block index; forced blocks = {0, last causal block} on top of the
 * budget; decode query t sits at cache position pos0 + t and is causal.
 *
 * Element-type codes for inputs: 0 = float32, 1 = bf16 bit patterns
 * (uint16), 2 = float64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double widen(const void* p, int dt, size_t i) {
  if (dt == 0) return (double)((const float*)p)[i];
  if (dt == 1) {
    uint32_t u = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
  }
  return ((const double*)p)[i];
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * Block sketch: the mean of the block's key rows ("Faster Than Flash" Sec. 1:
 * a compressed summary of the cache scanned in place of the keys; the statistic
 * itself is the mean, as the workload statement fixes).
 * K: [ngroups, Ls, d], rows j < L valid.  out: [ngroups, nb, d], nb = ceil(L/Bk).
 * A partial last block averages its valid rows only.
 */
void orc_block_means(const void* K, int dt, long ngroups, long L, long Ls, long d, long Bk,
                     double* out) {
  long nb = (L + Bk - 1) / Bk;
#pragma omp parallel for schedule(dynamic, 4)
  for (long u = 0; u < ngroups * nb; ++u) {
    long g = u / nb, b = u % nb;
    long j0 = b * Bk, j1 = j0 + Bk < L ? j0 + Bk : L;
    double* o = out + u * d;
    for (long c = 0; c < d; ++c) o[c] = 0.0;
    for (long j = j0; j < j1; ++j)
      for (long c = 0; c < d; ++c) o[c] += widen(K, dt, ((size_t)g * Ls + j) * d + c);
    for (long c = 0; c < d; ++c) o[c] /= (double)(j1 - j0);
  }
}

/* scale * q[b, t, h, :] . s[:] */
static double row_dot(const void* Q, int dt, long Tq, long Hq, long d, long b, long t, long h,
                      const double* s, double scale) {
  size_t base = (((size_t)b * Tq + t) * Hq + h) * d;
  double acc = 0.0;
  for (long c = 0; c < d; ++c) acc += widen(Q, dt, base + c) * s[c];
  return scale * acc;
}

/*
 * Decode sketch scores: s[g, b] = max over the group's query heads h and the
 * T query tokens t of scale * q[b, t, h, :] . sketch[g, b, :].
 * Q: [B, T, Hq, d]; sketch: [B*Hkv, nb, d]; out: [B*Hkv, nb].
 */
void orc_decode_scores(const void* Q, int dt, const double* sketch, long B, long T, long Hq,
                       long Hkv, long d, long nb, double scale, double* out) {
  long G = Hq / Hkv;
#pragma omp parallel for schedule(static)
  for (long u = 0; u < B * Hkv * nb; ++u) {
    long g = u / nb, blk = u % nb;
    long b = g / Hkv, kvh = g % Hkv;
    double best = -INFINITY;
    for (long t = 0; t < T; ++t)
      for (long hh = 0; hh < G; ++hh) {
        double s = row_dot(Q, dt, T, Hq, d, b, t, kvh * G + hh, sketch + ((size_t)g * nb + blk) * d, scale);
        if (s > best) best = s;
      }
    out[u] = best;
  }
}

/* last query row (exclusive end) of tile i, and the count of causal blocks */
static long tile_end(long i, long Qt, long Lq) { return (i + 1) * Qt < Lq ? (i + 1) * Qt : Lq; }

long orc_causal_blocks(long i, long Qt, long Bk, long Lq, long pos0) {
  long last = pos0 + tile_end(i, Qt, Lq) - 1; /* position of the tile's last query */
  return last / Bk + 1;
}

/*
 * Prefill sketch scores for selected (group, tile) units:
 * s[u, b] = max over the group's heads h and the tile's query rows t of
 * scale * q[b, t, h, :] . sketch[g, b, :] for causal blocks b (b*Bk <= the
 * tile's last query position), -inf otherwise.
 * units: [nunits, 2] = (g, i).  out: [nunits, nb].
 */
void orc_prefill_scores(const void* Q, int dt, const double* sketch, long B, long Lq, long Hq,
                        long Hkv, long d, long Qt, long Bk, long nb, double scale,
                        const long* units, long nunits, double* out) {
  long G = Hq / Hkv;
  (void)B;
#pragma omp parallel for schedule(dynamic, 1)
  for (long u = 0; u < nunits; ++u) {
    long g = units[2 * u], i = units[2 * u + 1];
    long b = g / Hkv, kvh = g % Hkv;
    long ncausal = orc_causal_blocks(i, Qt, Bk, Lq, 0);
    for (long blk = 0; blk < nb; ++blk) {
      double best = -INFINITY;
      if (blk < ncausal) {
        for (long t = i * Qt; t < tile_end(i, Qt, Lq); ++t)
          for (long hh = 0; hh < G; ++hh) {
            double s = row_dot(Q, dt, Lq, Hq, d, b, t, kvh * G + hh, sketch + ((size_t)g * nb + blk) * d, scale);
            if (s > best) best = s;
          }
      }
      out[u * nb + blk] = best;
    }
  }
}

typedef struct {
  double s;
  long b;
} cand_t;

/* order: higher score first; equal scores -> lower block index first */
static int cand_cmp(const void* x, const void* y) {
  const cand_t* a = (const cand_t*)x;
  const cand_t* c = (const cand_t*)y;
  if (a->s > c->s) return -1;
  if (a->s < c->s) return 1;
  return (a->b < c->b) ? -1 : (a->b > c->b);
}

static int long_cmp(const void* x, const void* y) {
  long a = *(const long*)x, b = *(const long*)y;
  return (a > b) - (a < b);
}

/*
 * Top-k selection with forced blocks ("How Much Dense Attention is
 * Necessary?" Sec. 2.1, top-k under a fixed budget; sink and local blocks
 * always kept as in "Pulsar Attention" Phase 1 and "Faster Than Flash" Sec. 2).
 * For unit u: valid blocks are [0, nvalid[u]); forced = {0, forced_hi[u]}
 * (deduplicated); the candidates are the other valid blocks, ranked by score
 * descending with ties to the lower index; the first min(budget[u], #candidates)
 * are kept.  Output: the union in ascending order in idx[u, 0:cnt[u]], the rest
 * of the row (up to kmax) filled with -1.  Returns 0, or -1 if kmax is too small.
 */
int orc_select(const double* scores, long nunits, long nb, const long* nvalid,
               const long* forced_hi, const long* budget, long kmax, int* idx, int* cnt) {
  int bad = 0;
  for (long u = 0; u < nunits; ++u) {
    long nv = nvalid[u];
    long f1 = forced_hi[u];
    cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)(nv > 0 ? nv : 1));
    long* sel = (long*)malloc(sizeof(long) * (size_t)(nv + 2));
    long nc = 0, ns = 0;
    for (long b = 0; b < nv; ++b) {
      if (b == 0 || b == f1) continue;
      c[nc].s = scores[u * nb + b];
      c[nc].b = b;
      ++nc;
    }
    qsort(c, (size_t)nc, sizeof(cand_t), cand_cmp);
    long take = budget[u] < nc ? budget[u] : nc;
    if (nv > 0) sel[ns++] = 0;
    if (f1 > 0 && f1 < nv) sel[ns++] = f1;
    for (long r = 0; r < take; ++r) sel[ns++] = c[r].b;
    qsort(sel, (size_t)ns, sizeof(long), long_cmp);
    if (ns > kmax) bad = 1;
    cnt[u] = (int)ns;
    for (long r = 0; r < kmax; ++r) idx[u * kmax + r] = r < ns ? (int)sel[r] : -1;
    free(c);
    free(sel);
  }
  return bad ? -1 : 0;
}

/*
 * Top-delta selection ("Faster Than Flash" Sec. 2: a key is kept when its score
 * is at least the pseudo-maximum minus delta, the pseudo-maximum being taken
 * over the sink and local-context keys only).  At block granularity: for unit
 * u with valid blocks [0, nvalid[u]) and forced blocks {0, forced_hi[u]}, the
 * pseudo-maximum is the larger score of the forced blocks; every other valid
 * block with score >= pseudo-max - delta is kept; if more than cap[u] qualify,
 * the cap[u] highest are kept (ties to the lower index).  Output as in
 * orc_select.  Returns 0, or -1 if kmax is too small.
 */
int orc_select_delta(const double* scores, long nunits, long nb, const long* nvalid, const long* forced_hi,
                     double delta, const long* cap, long kmax, int* idx, int* cnt) {
  int bad = 0;
  for (long u = 0; u < nunits; ++u) {
    long nv = nvalid[u];
    long f1 = forced_hi[u];
    double pmax = -INFINITY;
    if (nv > 0) pmax = scores[u * nb];
    if (f1 > 0 && f1 < nv && scores[u * nb + f1] > pmax) pmax = scores[u * nb + f1];
    const double thr = pmax - delta;
    cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)(nv > 0 ? nv : 1));
    long* sel = (long*)malloc(sizeof(long) * (size_t)(nv + 2));
    long nc = 0, ns = 0;
    for (long b = 0; b < nv; ++b) {
      if (b == 0 || b == f1) continue;
      if (scores[u * nb + b] >= thr) {
        c[nc].s = scores[u * nb + b];
        c[nc].b = b;
        ++nc;
      }
    }
    qsort(c, (size_t)nc, sizeof(cand_t), cand_cmp);
    long take = cap[u] < nc ? cap[u] : nc;
    if (nv > 0) sel[ns++] = 0;
    if (f1 > 0 && f1 < nv) sel[ns++] = f1;
    for (long r = 0; r < take; ++r) sel[ns++] = c[r].b;
    qsort(sel, (size_t)ns, sizeof(long), long_cmp);
    if (ns > kmax) bad = 1;
    cnt[u] = (int)ns;
    for (long r = 0; r < kmax; ++r) idx[u * kmax + r] = r < ns ? (int)sel[r] : -1;
    free(c);
    free(sel);
  }
  return bad ? -1 : 0;
}

/*
 * Exact softmax attention restricted to the selected blocks ("How Much Dense
 * Attention is Necessary?" Sec. 2.1: recompute with the original q, k, v on
 * the selected support only).
 * Q: [B, Tq, Hq, d]; K, V: [B, Hkv, Ls, d] with L valid rows.  Query row t of
 * any head sits at key position pos0 + t and sees keys j <= pos0 + t (causal).
 * Selection: unit (g, t / rows_per_sel) -> idx[(g*nsel + unit)*kmax ...],
 * cnt[...]; idx == NULL means every block (dense attention).
 * rows: [nrows, 3] = (b, t, h).  out: [nrows, d]; lse (optional): [nrows]
 * = log sum_j exp(logit_j) over the allowed keys.
 */
void orc_attend(const void* Q, const void* K, const void* V, int dt, long B, long Tq, long Hq,
                long Hkv, long d, long L, long Ls, long pos0, long Bk, double scale,
                const int* idx, const int* cnt, long kmax, long nsel, long rows_per_sel,
                const long* rows, long nrows, double* out, double* lse) {
  long G = Hq / Hkv;
  long nb = (L + Bk - 1) / Bk;
  (void)B;
#pragma omp parallel for schedule(dynamic, 1)
  for (long r = 0; r < nrows; ++r) {
    long b = rows[3 * r], t = rows[3 * r + 1], h = rows[3 * r + 2];
    long g = b * Hkv + h / G;
    long unit = g * nsel + t / rows_per_sel;
    long nblk = idx ? cnt[unit] : nb;
    long qpos = pos0 + t;
    size_t qbase = (((size_t)b * Tq + t) * Hq + h) * d;
    /* gather allowed key positions */
    long cap = nblk * Bk;
    long* keys = (long*)malloc(sizeof(long) * (size_t)(cap > 0 ? cap : 1));
    double* logit = (double*)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1));
    long nk = 0;
    for (long s = 0; s < nblk; ++s) {
      long blk = idx ? idx[unit * kmax + s] : s;
      for (long j = blk * Bk; j < (blk + 1) * Bk && j < L; ++j)
        if (j <= qpos) keys[nk++] = j;
    }
    double m = -INFINITY;
    for (long a = 0; a < nk; ++a) {
      size_t kb = ((size_t)g * Ls + keys[a]) * d;
      double acc = 0.0;
      for (long c = 0; c < d; ++c) acc += widen(Q, dt, qbase + c) * widen(K, dt, kb + c);
      logit[a] = scale * acc;
      if (logit[a] > m) m = logit[a];
    }
    double den = 0.0;
    double* o = out + r * d;
    for (long c = 0; c < d; ++c) o[c] = 0.0;
    for (long a = 0; a < nk; ++a) {
      double p = exp(logit[a] - m);
      den += p;
      size_t vb = ((size_t)g * Ls + keys[a]) * d;
      for (long c = 0; c < d; ++c) o[c] += p * widen(V, dt, vb + c);
    }
    for (long c = 0; c < d; ++c) o[c] = nk ? o[c] / den : 0.0;
    if (lse) lse[r] = nk ? m + log(den) : -INFINITY;
    free(keys);
    free(logit);
  }
}

/*
 * Exact attention mass per block ("How Much Dense Attention is Necessary?"
 * Sec. 2.1: the full dense attention distribution of each query, aggregated
 * over the query heads).  For unit (g, i):
 *   out[u, blk] = sum over the group's heads h and the tile's query rows t of
 *                 sum over keys j in block blk with j <= pos0 + t of P_{h,t}(j),
 * where P_{h,t} is the dense causal softmax of row (h, t) over all keys
 * j <= pos0 + t.  Non-causal blocks get 0.
 * units: [nunits, 2] = (g, i); out: [nunits, nb].
 */
void orc_mass(const void* Q, const void* K, int dt, long B, long Lq, long Hq, long Hkv, long d,
              long L, long Ls, long pos0, long Qt, long Bk, double scale, const long* units,
              long nunits, double* out) {
  long G = Hq / Hkv;
  long nb = (L + Bk - 1) / Bk;
  (void)B;
  for (long u = 0; u < nunits * nb; ++u) out[u] = 0.0;
  for (long u = 0; u < nunits; ++u) {
    long g = units[2 * u], i = units[2 * u + 1];
    long b = g / Hkv, kvh = g % Hkv;
    long t0 = i * Qt, t1 = tile_end(i, Qt, Lq);
    long nrow = (t1 - t0) * G;
    double* acc = (double*)calloc((size_t)nrow * nb, sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
    for (long rr = 0; rr < nrow; ++rr) {
      long t = t0 + rr / G, h = kvh * G + rr % G;
      long qpos = pos0 + t;
      long nk = qpos + 1 < L ? qpos + 1 : L;
      double* logit = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
      size_t qbase = (((size_t)b * Lq + t) * Hq + h) * d;
      double m = -INFINITY;
      for (long j = 0; j < nk; ++j) {
        size_t kb = ((size_t)g * Ls + j) * d;
        double a = 0.0;
        for (long c = 0; c < d; ++c) a += widen(Q, dt, qbase + c) * widen(K, dt, kb + c);
        logit[j] = scale * a;
        if (logit[j] > m) m = logit[j];
      }
      double den = 0.0;
      for (long j = 0; j < nk; ++j) den += exp(logit[j] - m);
      double* ar = acc + rr * nb;
      for (long j = 0; j < nk; ++j) ar[j / Bk] += exp(logit[j] - m) / den;
      free(logit);
    }
    for (long rr = 0; rr < nrow; ++rr)
      for (long blk = 0; blk < nb; ++blk) out[u * nb + blk] += acc[rr * nb + blk];
    free(acc);
  }
}
