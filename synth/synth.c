/*
 * synth.c -- seeded synthetic inputs for top-k block-sparse GQA attention.
 *
 * This file holds input construction only: a counter-based normal generator,
 * bf16 round-to-nearest-even packing, and the additive "plants" (needle keys,
 * a shared low-rank q/k component) that give the workloads their structure.
 * It contains none of the attention method's arithmetic (no sketch, score,
 * selection, softmax or mass).  Both the CUDA path and the CPU oracle are fed
 * the exact bits produced here.
 *
 * Generator definition (stated so that it can be re-implemented exactly):
 *   splitmix64(x):  z = x + 0x9E3779B97F4A7C15;
 *                   z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
 *                   z = (z ^ (z >> 27)) * 0x94D049BB133111EB;
 *                   return z ^ (z >> 31)
 *   stream key:     key = splitmix64(seed ^ splitmix64(stream))
 *   element i:      x  = splitmix64(key + (i >> 1))
 *                   u1 = ((x >> 32) + 0.5) / 2^32,  u2 = ((x & 0xFFFFFFFF) + 0.5) / 2^32
 *                   r  = sqrt(-2 ln u1)
 *                   z  = r cos(2 pi u2)  for even i,  r sin(2 pi u2) for odd i
 *   (Box-Muller transform on a splitmix64 counter stream.)
 *
 * Values are formed in double, rounded once to float (RNE) and, for bf16
 * tensors, once more to bf16 with round-to-nearest-even on the float bits.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define SY_PI 3.14159265358979323846

uint64_t sy_splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t sy_stream_key(uint64_t seed, uint64_t stream) {
  return sy_splitmix64(seed ^ sy_splitmix64(stream));
}

double sy_normal_at(uint64_t key, uint64_t i) {
  uint64_t x = sy_splitmix64(key + (i >> 1));
  double u1 = ((double)(x >> 32) + 0.5) * (1.0 / 4294967296.0);
  double u2 = ((double)(x & 0xFFFFFFFFull) + 0.5) * (1.0 / 4294967296.0);
  double r = sqrt(-2.0 * log(u1));
  return (i & 1) ? r * sin(2.0 * SY_PI * u2) : r * cos(2.0 * SY_PI * u2);
}

/* uniform 64-bit draw number i of a stream (used for needle placement) */
uint64_t sy_u64_at(uint64_t key, uint64_t i) { return sy_splitmix64(key + i); }

/* float -> bf16 bits, round to nearest even (NaN kept quiet). */
uint16_t sy_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

double sy_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static inline void store_val(void* out, int is_bf16, size_t i, double v) {
  float f = (float)v;
  if (is_bf16)
    ((uint16_t*)out)[i] = sy_f32_to_bf16(f);
  else
    ((float*)out)[i] = f;
}

static inline double load_val(const void* p, int is_bf16, size_t i) {
  if (is_bf16) return sy_bf16_to_f64(((const uint16_t*)p)[i]);
  return (double)((const float*)p)[i];
}

/* Plain N(0,1) tensor of n elements. */
void sy_fill_normal(void* out, int is_bf16, size_t n, uint64_t seed, uint64_t stream) {
  uint64_t key = sy_stream_key(seed, stream);
  long long nn = (long long)n;
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < nn; ++i) store_val(out, is_bf16, (size_t)i, sy_normal_at(key, (uint64_t)i));
}

/*
 * Queries, layout [B, Tq, Hq, d].  Optional low-rank plant: for every row
 * (b, t, h) with kv-head g = h / (Hq/Hkv), add gamma * U[b,g] c[b,t,h], where
 * U is [B*Hkv, d, r] (row-major over d then r) and c ~ N(0, I_r) is drawn from
 * stream (stream + 1).  Pass U = NULL for no plant.
 */
void sy_make_queries(void* out, int is_bf16, long B, long Tq, long Hq, long Hkv, long d,
                     uint64_t seed, uint64_t stream, const double* U, long r, double gamma) {
  uint64_t key = sy_stream_key(seed, stream);
  uint64_t ckey = sy_stream_key(seed, stream + 1);
  long G = Hq / Hkv;
  long long rows = (long long)B * Tq * Hq;
#pragma omp parallel for schedule(static)
  for (long long row = 0; row < rows; ++row) {
    long h = (long)(row % Hq);
    long b = (long)(row / ((long long)Tq * Hq));
    long g = b * Hkv + h / G;
    double c[16];
    if (U) {
      for (long a = 0; a < r; ++a) c[a] = sy_normal_at(ckey, (uint64_t)(row * r + a));
    }
    for (long e = 0; e < d; ++e) {
      size_t i = (size_t)row * d + e;
      double v = sy_normal_at(key, i);
      if (U) {
        double add = 0.0;
        for (long a = 0; a < r; ++a) add += U[(g * d + e) * r + a] * c[a];
        v += gamma * add;
      }
      store_val(out, is_bf16, i, v);
    }
  }
}

/*
 * Keys, layout [B, Hkv, L, d] (row stride d, group stride L*d).  Row j of
 * group g belongs to block j / Bk.  Additive terms:
 *   needle[g*nb + blk] != 0  ->  + alpha * qhat[g, :]
 *   U != NULL                ->  + gamma * U[g] e[g, blk]  with e ~ N(0, I_r)
 *                                 drawn from stream (stream + 1), shared by
 *                                 every key row of the block.
 */
void sy_make_keys(void* out, int is_bf16, long B, long Hkv, long L, long d, long Bk,
                  uint64_t seed, uint64_t stream, const uint8_t* needle, const double* qhat,
                  double alpha, const double* U, long r, double gamma) {
  uint64_t key = sy_stream_key(seed, stream);
  uint64_t ekey = sy_stream_key(seed, stream + 1);
  long nb = (L + Bk - 1) / Bk;
  long long rows = (long long)B * Hkv * L;
#pragma omp parallel for schedule(static)
  for (long long row = 0; row < rows; ++row) {
    long g = (long)(row / L);
    long j = (long)(row % L);
    long blk = j / Bk;
    int is_needle = needle && needle[g * nb + blk];
    double e[16];
    if (U) {
      for (long a = 0; a < r; ++a) e[a] = sy_normal_at(ekey, (uint64_t)((g * nb + blk) * r + a));
    }
    for (long c = 0; c < d; ++c) {
      size_t i = (size_t)row * d + c;
      double v = sy_normal_at(key, i);
      if (is_needle) v += alpha * qhat[g * d + c];
      if (U) {
        double add = 0.0;
        for (long a = 0; a < r; ++a) add += U[(g * d + c) * r + a] * e[a];
        v += gamma * add;
      }
      store_val(out, is_bf16, i, v);
    }
  }
}

/*
 * Needle direction per group: qhat_g = normalise( sum over the group's query
 * heads h and all Tq query rows t of q[b, t, h, :] ), from the stored
 * (already rounded) query values.  out: [B*Hkv, d].
 */
void sy_needle_direction(const void* q, int is_bf16, long B, long Tq, long Hq, long Hkv, long d,
                         double* out) {
  long G = Hq / Hkv;
  long ngroups = B * Hkv;
#pragma omp parallel for schedule(static)
  for (long g = 0; g < ngroups; ++g) {
    long b = g / Hkv, kvh = g % Hkv;
    double* acc = out + g * d;
    for (long c = 0; c < d; ++c) acc[c] = 0.0;
    for (long t = 0; t < Tq; ++t)
      for (long hh = 0; hh < G; ++hh) {
        long h = kvh * G + hh;
        size_t base = (((size_t)b * Tq + t) * Hq + h) * d;
        for (long c = 0; c < d; ++c) acc[c] += load_val(q, is_bf16, base + c);
      }
    double nrm = 0.0;
    for (long c = 0; c < d; ++c) nrm += acc[c] * acc[c];
    nrm = sqrt(nrm);
    if (nrm > 0)
      for (long c = 0; c < d; ++c) acc[c] /= nrm;
  }
}

/*
 * Needle blocks: for each group, `count` distinct blocks drawn uniformly from
 * [lo, hi] (inclusive) by uniform draws (rejecting repeats) from the u64
 * stream.  mask: [ngroups, nb] bytes, set to 1 for needle blocks.
 */
void sy_needle_blocks(uint8_t* mask, long ngroups, long nb, long lo, long hi, long count,
                      uint64_t seed, uint64_t stream) {
  memset(mask, 0, (size_t)ngroups * nb);
  long n = hi - lo + 1;
  if (n <= 0 || count <= 0) return;
  if (count > n) count = n;
  for (long g = 0; g < ngroups; ++g) {
    uint64_t key = sy_stream_key(seed, stream + (uint64_t)g);
    /* uniform draws with rejection of repeats, on the output bitmap */
    long chosen = 0;
    uint64_t draw = 0;
    while (chosen < count) {
      uint64_t x = sy_u64_at(key, draw++);
      long cand = lo + (long)(x % (uint64_t)n);
      if (!mask[g * nb + cand]) {
        mask[g * nb + cand] = 1;
        ++chosen;
      }
    }
  }
}

/*
 * Orthonormal basis per group for the low-rank plant: r Gaussian d-vectors
 * (stream `stream`), orthonormalised by modified Gram-Schmidt.  out: [ngroups, d, r].
 */
void sy_orthonormal_basis(double* out, long ngroups, long d, long r, uint64_t seed, uint64_t stream) {
  uint64_t key = sy_stream_key(seed, stream);
  for (long g = 0; g < ngroups; ++g) {
    double* U = out + g * d * r;
    for (long a = 0; a < r; ++a)
      for (long c = 0; c < d; ++c) U[c * r + a] = sy_normal_at(key, (uint64_t)((g * r + a) * d + c));
    for (long a = 0; a < r; ++a) {
      for (long p = 0; p < a; ++p) {
        double dot = 0.0;
        for (long c = 0; c < d; ++c) dot += U[c * r + a] * U[c * r + p];
        for (long c = 0; c < d; ++c) U[c * r + a] -= dot * U[c * r + p];
      }
      double nrm = 0.0;
      for (long c = 0; c < d; ++c) nrm += U[c * r + a] * U[c * r + a];
      nrm = sqrt(nrm);
      for (long c = 0; c < d; ++c) U[c * r + a] /= nrm;
    }
  }
}

int sy_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
