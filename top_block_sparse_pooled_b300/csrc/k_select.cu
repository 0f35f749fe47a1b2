// k_select.cu -- block scoring and deterministic top-k selection.
//
// "How Much Dense Attention is Necessary?" Sec. 2.1-2.2: score the candidate
// blocks, keep the top-k under a fixed budget, recompute attention on them.
// Sink block 0 and the local / diagonal block are always kept ("Pulsar
// Attention" Phase 1, "Faster Than Flash" Sec. 2) and do not count against
// the budget.  Ties go to the lower block index; the output is ascending.
//
// Top-delta (decode): the budget becomes the number of candidates that score at
// least max(sink score, local score) - delta, capped at k; the same exact
// top-k then picks exactly those candidates (they are the highest ones).
//
// Top-k is an exact MSB-first radix select on order-preserving 32-bit keys of
// the float32 scores (four 8-bit digit passes over 256-bin shared-memory
// histograms), followed by an index-ordered pass that admits ties at the
// threshold key lowest index first and writes the selection in ascending order.
#pragma once

#include <cstddef>
#include <type_traits>

#include "sa_ptx.cuh"

namespace sa {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

constexpr int kTopkMaxN = 16384;  // candidates per selection (blocks per sequence)

constexpr int kRankFinish = 64;  // rank the remaining keys once at most this many share the prefix


// 16-byte vector accesses: hist, live and cand are 16-byte aligned (the struct
// itself sits at a 16-byte aligned shared address).
constexpr int kHistBins = 2048;  // value-binned histogram of the top-k threshold search
constexpr int kHistCand = 256;   // keys of the threshold's bin ranked directly

struct TopkShared {
  alignas(16) uint32_t hist[kHistBins];  // radix passes use the first 4 x 256 as one histogram per pass
  uint32_t wdef[kSelWarps];  // per-warp count of selections decided without ties
  uint32_t weq[kSelWarps];   // per-warp count of candidates tied with the threshold key
  alignas(16) uint32_t live[kRankFinish];  // rank finish: the keys still sharing the threshold's prefix
  uint32_t nlive, fin_thr, fin_need;
  alignas(16) uint32_t cand[kHistCand];  // the threshold bin's keys (histogram search)
  uint32_t wmax[kSelWarps], wmin[kSelWarps];  // per-warp key range
  uint32_t bsel[4];                           // broadcast: bin, remaining, bin count, candidates gathered
};
static_assert(offsetof(TopkShared, hist) % 16 == 0 && offsetof(TopkShared, live) % 16 == 0 &&
                  offsetof(TopkShared, cand) % 16 == 0,
              "vector-accessed members must be 16-byte aligned");

// Shared-memory accesses by 32-bit shared-window address (explicit state space,
// so that no access falls back to generic addressing).
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float2 lds_f32x2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float4 lds_f32x4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint4 lds_u32x4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_u32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void red_add_shared(uint32_t a, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Barrier policies for the top-k functions: the whole CTA, or the first
// kSelThreads threads of a larger CTA (named barrier 1; the other warps of that
// CTA must not use barrier 1 meanwhile).
struct SyncCta {
  static __device__ __forceinline__ void sync() { __syncthreads(); }
};
struct SyncFirst256 {
  static __device__ __forceinline__ void sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
};

// Output pass shared by the threshold searches: given the threshold key thr
// of a by-key selection and the number need_eq of keys equal to it that are
// admitted (lowest indices first), write the selection.  Each warp owns a
// contiguous span of indices, counts its keys above the threshold and its ties,
// and after one barrier writes its selections at their ascending positions.
// The span is walked kOutBatch rounds of 32 indices at a time: the loads, key
// tests and ballots of a batch are independent, so their latencies overlap.
constexpr int kOutBatch = 8;

template <typename Sync, typename LoadF>
__device__ __forceinline__ void topk_output(LoadF score, int n, int take, bool by_key, uint32_t thr, uint32_t need_eq,
                                            int kmax, int32_t* __restrict__ idx_out, int32_t* __restrict__ cnt_out,
                                            uint32_t S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t wdef = S + static_cast<uint32_t>(offsetof(TopkShared, wdef));
  const uint32_t weq = S + static_cast<uint32_t>(offsetof(TopkShared, weq));
  const int last = n - 1;
  // classes of index b: `def` = kept regardless of ties, `eq` = tied with the threshold key
  auto classify = [&](int b, float v, bool& def, bool& eq) {
    def = false;
    eq = false;
    if (b >= n) return;
    if (b == 0 || b == last) {
      def = true;
    } else if (take > 0) {
      if (!by_key) {
        def = true;
      } else {
        const uint32_t key = float_key(v);
        def = key > thr;
        eq = key == thr;
      }
    }
  };
  const int span = ((n + kSelThreads - 1) / kSelThreads) * 32;  // indices per warp, a multiple of 32
  const int w0 = warp * span;
  // one batch: the ballots of kOutBatch rounds of 32 indices starting at base
  auto batch = [&](int base, uint32_t* db, uint32_t* eb) {
    float v[kOutBatch];
#pragma unroll
    for (int j = 0; j < kOutBatch; ++j) {
      const int b = base + 32 * j + lane;
      v[j] = (by_key && b < n && base + 32 * j < w0 + span) ? score(b) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kOutBatch; ++j) {
      bool d, e;
      const int b = base + 32 * j + lane;
      classify(base + 32 * j < w0 + span ? b : n, v[j], d, e);
      db[j] = __ballot_sync(0xFFFFFFFFu, d);
      eb[j] = __ballot_sync(0xFFFFFFFFu, e);
    }
  };
  uint32_t ndef = 0u, neq = 0u;
  for (int base = w0; base < w0 + span; base += 32 * kOutBatch) {
    uint32_t db[kOutBatch], eb[kOutBatch];
    batch(base, db, eb);
#pragma unroll
    for (int j = 0; j < kOutBatch; ++j) {
      ndef += __popc(db[j]);
      neq += __popc(eb[j]);
    }
  }
  if (lane == 0) {
    sts_u32(wdef + 4u * warp, ndef);
    sts_u32(weq + 4u * warp, neq);
  }
  Sync::sync();
  uint32_t def_before = 0u, eq_before = 0u, def_all = 0u, eq_all = 0u;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    const uint32_t a = lds_u32(wdef + 4u * w), e = lds_u32(weq + 4u * w);
    def_before += w < warp ? a : 0u;
    eq_before += w < warp ? e : 0u;
    def_all += a;
    eq_all += e;
  }
  const uint32_t total = def_all + min(eq_all, need_eq);
  uint32_t pos = def_before + min(eq_before, need_eq);
  uint32_t eq_seen = eq_before;
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = w0; base < w0 + span; base += 32 * kOutBatch) {
    uint32_t db[kOutBatch], eb[kOutBatch];
    batch(base, db, eb);
#pragma unroll
    for (int j = 0; j < kOutBatch; ++j) {
      // ties are admitted in index order while the budget for them lasts
      const bool sel = ((db[j] >> lane) & 1u) ||
                       (((eb[j] >> lane) & 1u) && eq_seen + static_cast<uint32_t>(__popc(eb[j] & lt)) < need_eq);
      const uint32_t sb = __ballot_sync(0xFFFFFFFFu, sel);
      if (sel) {
        const uint32_t at = pos + static_cast<uint32_t>(__popc(sb & lt));
        if (at < static_cast<uint32_t>(kmax)) idx_out[at] = base + 32 * j + lane;
      }
      pos += static_cast<uint32_t>(__popc(sb));
      eq_seen += static_cast<uint32_t>(__popc(eb[j]));
    }
  }
  for (int i = static_cast<int>(total) + tid; i < kmax; i += kSelThreads) idx_out[i] = -1;
  if (tid == 0) *cnt_out = static_cast<int32_t>(total);
}

// Select from scores score(0..n-1): the forced
// blocks are the first and the last (0 and n-1, one block when n == 1); the
// candidates are 1..n-2; keep min(budget, n-2) of them with the highest scores,
// ties to the lower index.  Writes idx_out[0:kmax] (ascending, -1 padded) and
// *cnt_out.  S: shared address of a TopkShared.  All kSelThreads threads call;
// every score is read six times (four digit passes, two output passes);
// six block barriers in all.
//
// Threshold: exact MSB-first radix select of the take-th largest order-preserving
// key (8-bit digit passes, each into its own 256-bin histogram; every warp then
// finds the digit itself, so a pass costs one barrier).  As soon as at most
// kRankFinish keys share the threshold's prefix, they are gathered and each
// counts the keys above and equal to it: the one with count-above < remaining <=
// count-above-or-equal is the threshold (two barriers instead of the remaining
// passes).  The selection is then written by topk_output.
template <typename Sync = SyncCta, typename LoadF>
__device__ __forceinline__ void block_topk_impl(LoadF score, int n, int budget, int kmax, int32_t* __restrict__ idx_out,
                                                int32_t* __restrict__ cnt_out, uint32_t S) {
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t hist = S + static_cast<uint32_t>(offsetof(TopkShared, hist));
  const uint32_t live = S + static_cast<uint32_t>(offsetof(TopkShared, live));
  const uint32_t nlive = S + static_cast<uint32_t>(offsetof(TopkShared, nlive));
  const uint32_t fin_thr = S + static_cast<uint32_t>(offsetof(TopkShared, fin_thr));
  const uint32_t fin_need = S + static_cast<uint32_t>(offsetof(TopkShared, fin_need));
  const int last = n - 1;                      // forced local / diagonal block
  const int ncand = n > 2 ? n - 2 : 0;         // candidates 1 .. n-2
  const int take = budget <= 0 ? 0 : (budget < ncand ? budget : ncand);
  const bool by_key = take > 0 && take < ncand;
  uint32_t thr = 0u, need_eq = 0u;
  if (by_key) {
    for (int i = tid; i < 4 * 256 / 4; i += kSelThreads)
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(hist + 16u * i), "r"(0u) : "memory");
    if (tid == 0) sts_u32(nlive, 0u);
    Sync::sync();
    uint32_t prefix = 0u, mask = 0u, remaining = static_cast<uint32_t>(take);
    for (int p = 0; p < 4; ++p) {
      const int shift = 24 - 8 * p;
      const uint32_t hp = hist + 1024u * p;
      for (int b = 1 + tid; b < last; b += kSelThreads) {
        const uint32_t key = float_key(score(b));
        if ((key & mask) == prefix) red_add_shared(hp + 4u * ((key >> shift) & 255u), 1u);
      }
      Sync::sync();
      // lane l holds digits 255-8l .. 248-8l (descending); the chosen digit is the
      // one where the count of keys above it stays below `remaining` and the count
      // including it reaches it (exactly one (lane, e) qualifies)
      const uint4 lo4 = lds_u32x4(hp + 4u * (248 - 8 * lane)), hi4 = lds_u32x4(hp + 4u * (252 - 8 * lane));
      const uint32_t c[8] = {hi4.w, hi4.z, hi4.y, hi4.x, lo4.w, lo4.z, lo4.y, lo4.x};
      uint32_t sum = 0u;
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += c[e];
      uint32_t inc = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
      }
      uint32_t run = inc - sum, hit = 0u, dsel = 0u, rem = 0u, ceq = 0u;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (hit == 0u && run < remaining && remaining <= run + c[e]) {
          hit = 1u;
          dsel = 255u - 8u * static_cast<uint32_t>(lane) - static_cast<uint32_t>(e);
          rem = remaining - run;
          ceq = c[e];
        }
        run += c[e];
      }
      const int src = (__ffs(__ballot_sync(0xFFFFFFFFu, hit != 0u)) - 1) & 31;
      dsel = __shfl_sync(0xFFFFFFFFu, dsel, src);
      rem = __shfl_sync(0xFFFFFFFFu, rem, src);
      ceq = __shfl_sync(0xFFFFFFFFu, ceq, src);
      prefix |= dsel << shift;
      mask |= 255u << shift;
      remaining = rem;
      if (p < 3 && ceq <= static_cast<uint32_t>(kRankFinish)) {
        // rank finish: gather the ceq keys that share the prefix (warp-aggregated slots) ...
        for (int base = 0; base < n; base += kSelThreads) {  // same trip count in every lane
          const int b = base + tid;
          const uint32_t key = (b >= 1 && b < last) ? float_key(score(b)) : 0u;
          const bool in = b >= 1 && b < last && (key & mask) == prefix;
          const uint32_t bal = __ballot_sync(0xFFFFFFFFu, in);
          uint32_t slot0 = 0u;
          if (lane == 0 && bal != 0u) {
            asm volatile("atom.shared.add.u32 %0, [%1], %2;" : "=r"(slot0) : "r"(nlive), "r"(__popc(bal)) : "memory");
          }
          slot0 = __shfl_sync(0xFFFFFFFFu, slot0, 0);
          if (in) sts_u32(live + 4u * (slot0 + __popc(bal & ((1u << lane) - 1u))), key);
        }
        Sync::sync();
        // ... and the key with count-above < remaining <= count-above-or-equal is the threshold
        if (tid < static_cast<int>(ceq)) {
          const uint32_t kt = lds_u32(live + 4u * tid);
          uint32_t above = 0u, same = 0u;
          for (uint32_t j0 = 0; j0 < ceq; j0 += 16) {  // sixteen keys per round: four loads, then compares
            uint4 x[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) x[v] = lds_u32x4(live + 4u * (j0 + 4u * v));
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint32_t xv[4] = {x[v].x, x[v].y, x[v].z, x[v].w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const bool ok = j0 + 4u * v + i < ceq;  // entries past ceq are stale
                above += (ok && xv[i] > kt) ? 1u : 0u;
                same += (ok && xv[i] == kt) ? 1u : 0u;
              }
            }
          }
          if (above < remaining && remaining <= above + same) {  // every such thread writes the same pair
            sts_u32(fin_thr, kt);
            sts_u32(fin_need, remaining - above);
          }
        }
        Sync::sync();
        prefix = lds_u32(fin_thr);
        remaining = lds_u32(fin_need);
        break;
      }
    }
    thr = prefix;
    need_eq = remaining;  // ties at the threshold key to admit, lowest indices first
  }
  topk_output<Sync>(score, n, take, by_key, thr, need_eq, kmax, idx_out, cnt_out, S);
}

// Inverse of float_key.
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The same selection as block_topk_impl, with the threshold found by value
// histograms instead of bit digits.  The keys inside a key interval [klo, khi]
// (at first all candidates) are binned by score, linearly over
// [score(klo), score(khi)] into kHistBins bins: the bin index is a monotone
// non-decreasing function of the score, so every bin is a key interval.  The
// bin that holds the remaining-th largest key of the interval is found by a
// descending prefix sum; its keys become the next interval, unless they are all
// equal (the threshold) or at most kHistCand of them, which are gathered and
// ranked directly (each counts the keys above and equal to it).  Value bins
// spread the keys evenly where they are dense, so the shared-memory atomics
// rarely collide; one histogram round usually suffices.  A key range whose
// width does not fit a float (infinite or non-finite scores) goes to the radix
// select.  All kSelThreads threads call; barriers are uniform.
template <typename Sync = SyncCta, typename LoadF>
__device__ __forceinline__ void block_topk_hist_impl(LoadF score, int n, int budget, int kmax,
                                                     int32_t* __restrict__ idx_out, int32_t* __restrict__ cnt_out,
                                                     uint32_t S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ncand = n > 2 ? n - 2 : 0;  // candidates 1 .. n-2
  const int take = budget <= 0 ? 0 : (budget < ncand ? budget : ncand);
  const bool by_key = take > 0 && take < ncand;
  if (!by_key) {
    topk_output<Sync>(score, n, take, false, 0u, 0u, kmax, idx_out, cnt_out, S);
    return;
  }
  const uint32_t hist = S + static_cast<uint32_t>(offsetof(TopkShared, hist));
  const uint32_t cand = S + static_cast<uint32_t>(offsetof(TopkShared, cand));
  const uint32_t wmax = S + static_cast<uint32_t>(offsetof(TopkShared, wmax));
  const uint32_t wmin = S + static_cast<uint32_t>(offsetof(TopkShared, wmin));
  const uint32_t bsel = S + static_cast<uint32_t>(offsetof(TopkShared, bsel));
  constexpr int kB = 8;  // loads in flight per thread
  // key range of the candidates; the histogram and the gather counter start at zero
  uint32_t kmx = 0u, kmn = 0xFFFFFFFFu;
  for (int b0 = 1 + tid; b0 < n - 1; b0 += kB * kSelThreads) {
    float v[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int b = b0 + j * kSelThreads;
      v[j] = b < n - 1 ? score(b) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kB; ++j)
      if (b0 + j * kSelThreads < n - 1) {
        const uint32_t k = float_key(v[j]);
        kmx = max(kmx, k);
        kmn = min(kmn, k);
      }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmx = max(kmx, __shfl_xor_sync(0xFFFFFFFFu, kmx, o));
    kmn = min(kmn, __shfl_xor_sync(0xFFFFFFFFu, kmn, o));
  }
  if (lane == 0) {
    sts_u32(wmax + 4u * warp, kmx);
    sts_u32(wmin + 4u * warp, kmn);
  }
  for (int i = tid; i < kHistBins / 4; i += kSelThreads)
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(hist + 16u * i), "r"(0u) : "memory");
  if (tid == 0) sts_u32(bsel + 12u, 0u);
  Sync::sync();
  uint32_t klo = 0xFFFFFFFFu, khi = 0u;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    khi = max(khi, lds_u32(wmax + 4u * w));
    klo = min(klo, lds_u32(wmin + 4u * w));
  }
  uint32_t remaining = static_cast<uint32_t>(take);
  uint32_t inside = static_cast<uint32_t>(ncand);  // keys in [klo, khi]
  uint32_t thr = 0u, need_eq = 0u;
  bool found = false, radix = false;
  // Gather the `inside` keys for which in(key, score) holds (slots by one atomic per warp and
  // batch; the order does not matter), then the key with count-above < remaining <=
  // count-above-or-equal is the threshold.  The gather counter is zero on entry.
  auto gather_rank = [&](auto in_set) {
    for (int base = 0; base < n; base += kB * kSelThreads) {  // same trip count in every lane
      uint32_t key[kB];
      bool in[kB];
      uint32_t bal[kB], tot = 0u;
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int b = base + j * kSelThreads + tid;
        const float v = (b >= 1 && b < n - 1) ? score(b) : 0.f;
        key[j] = float_key(v);
        in[j] = b >= 1 && b < n - 1 && in_set(key[j], v);
      }
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        bal[j] = __ballot_sync(0xFFFFFFFFu, in[j]);
        tot += static_cast<uint32_t>(__popc(bal[j]));
      }
      if (tot == 0u) continue;  // uniform in the warp
      uint32_t slot0 = 0u;
      if (lane == 0)
        asm volatile("atom.shared.add.u32 %0, [%1], %2;" : "=r"(slot0) : "r"(bsel + 12u), "r"(tot) : "memory");
      slot0 = __shfl_sync(0xFFFFFFFFu, slot0, 0);
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const uint32_t at = slot0 + static_cast<uint32_t>(__popc(bal[j] & ((1u << lane) - 1u)));
        if (in[j] && at < static_cast<uint32_t>(kHistCand)) sts_u32(cand + 4u * at, key[j]);
        slot0 += static_cast<uint32_t>(__popc(bal[j]));
      }
    }
    Sync::sync();
    if (tid < static_cast<int>(inside)) {
      const uint32_t kt = lds_u32(cand + 4u * tid);
      uint32_t above = 0u, same = 0u;
      for (uint32_t j0 = 0; j0 < inside; j0 += 16) {
        uint4 x[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) x[v] = lds_u32x4(cand + 4u * (j0 + 4u * v));
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t xv[4] = {x[v].x, x[v].y, x[v].z, x[v].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const bool ok = j0 + 4u * v + i < inside;  // entries past the count are stale
            above += (ok && xv[i] > kt) ? 1u : 0u;
            same += (ok && xv[i] == kt) ? 1u : 0u;
          }
        }
      }
      if (above < remaining && remaining <= above + same) {  // every such thread writes the same pair
        sts_u32(bsel, kt);
        sts_u32(bsel + 4u, remaining - above);
      }
    }
    Sync::sync();
    thr = lds_u32(bsel);
    need_eq = lds_u32(bsel + 4u);
    found = true;
  };
  // each round either ends the search or leaves a bin with fewer keys than the interval had
  for (int round = 0; round < 64 && !found && !radix; ++round) {
    if (klo == khi) {  // every key of the interval is the threshold
      thr = klo;
      need_eq = remaining;
      found = true;
      break;
    }
    const uint32_t lo = klo, hi = khi;
    if (inside <= static_cast<uint32_t>(kHistCand)) {
      gather_rank([&](uint32_t k, float) { return k >= lo && k <= hi; });
      break;
    }
    const float smin = key_float(klo), smax = key_float(khi);
    const float inv = static_cast<float>(kHistBins) / (smax - smin);
    if (!(inv > 0.f && inv < 3.0e38f && smax - smin < 3.0e38f)) {  // not a finite positive width
      radix = true;
      break;
    }
    auto bin_of = [smin, inv](float x) {
      const float f = (x - smin) * inv;
      return f >= static_cast<float>(kHistBins - 1) ? kHistBins - 1 : static_cast<int>(f);
    };
    for (int b0 = 1 + tid; b0 < n - 1; b0 += kB * kSelThreads) {
      float v[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int b = b0 + j * kSelThreads;
        v[j] = b < n - 1 ? score(b) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const uint32_t k = float_key(v[j]);
        if (b0 + j * kSelThreads < n - 1 && k >= klo && k <= khi)
          red_add_shared(hist + 4u * static_cast<uint32_t>(bin_of(v[j])), 1u);
      }
    }
    Sync::sync();
    // thread t holds bins kHistBins-1-8t .. kHistBins-8-8t (descending); a scan over the
    // threads finds the bin where the count of keys above it stays below `remaining` and
    // the count including it reaches it
    uint32_t c[8];
    {
      const uint4 hi4 = lds_u32x4(hist + 4u * (kHistBins - 4 - 8 * tid));
      const uint4 lo4 = lds_u32x4(hist + 4u * (kHistBins - 8 - 8 * tid));
      c[0] = hi4.w; c[1] = hi4.z; c[2] = hi4.y; c[3] = hi4.x;
      c[4] = lo4.w; c[5] = lo4.z; c[6] = lo4.y; c[7] = lo4.x;
      // clear them for a later round (every bin is read by its owner only)
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(hist + 4u * (kHistBins - 4 - 8 * tid)), "r"(0u)
                   : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(hist + 4u * (kHistBins - 8 - 8 * tid)), "r"(0u)
                   : "memory");
    }
    uint32_t sum = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) sum += c[e];
    uint32_t inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) sts_u32(wmax + 4u * warp, inc);  // warp totals (the key range is no longer needed)
    Sync::sync();
    uint32_t run = inc - sum;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) run += w < warp ? lds_u32(wmax + 4u * w) : 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (run < remaining && remaining <= run + c[e]) {  // exactly one (thread, e)
        sts_u32(bsel, static_cast<uint32_t>(kHistBins - 1 - 8 * tid - e));
        sts_u32(bsel + 4u, remaining - run);
        sts_u32(bsel + 8u, c[e]);
      }
      run += c[e];
    }
    if (tid == 0) sts_u32(bsel + 12u, 0u);
    Sync::sync();
    const int dsel = static_cast<int>(lds_u32(bsel));
    remaining = lds_u32(bsel + 4u);
    inside = lds_u32(bsel + 8u);
    if (inside <= static_cast<uint32_t>(kHistCand)) {  // the bin's keys, ranked directly
      gather_rank([&](uint32_t k, float v) { return k >= lo && k <= hi && bin_of(v) == dsel; });
      break;
    }
    // a crowded bin: its key range is the next interval
    uint32_t nlo = 0xFFFFFFFFu, nhi = 0u;
    for (int b0 = 1 + tid; b0 < n - 1; b0 += kB * kSelThreads) {
      float v[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int b = b0 + j * kSelThreads;
        v[j] = b < n - 1 ? score(b) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const uint32_t k = float_key(v[j]);
        if (b0 + j * kSelThreads < n - 1 && k >= klo && k <= khi && bin_of(v[j]) == dsel) {
          nhi = max(nhi, k);
          nlo = min(nlo, k);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      nhi = max(nhi, __shfl_xor_sync(0xFFFFFFFFu, nhi, o));
      nlo = min(nlo, __shfl_xor_sync(0xFFFFFFFFu, nlo, o));
    }
    if (lane == 0) {  // every warp read the warp totals before the last barrier
      sts_u32(wmax + 4u * warp, nhi);
      sts_u32(wmin + 4u * warp, nlo);
    }
    Sync::sync();
    klo = 0xFFFFFFFFu;
    khi = 0u;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
      khi = max(khi, lds_u32(wmax + 4u * w));
      klo = min(klo, lds_u32(wmin + 4u * w));
    }
    Sync::sync();  // the range words are read before a later round writes them
  }
  if (!found) {  // uniform: every thread took the same branches
    Sync::sync();
    block_topk_impl<Sync>(score, n, budget, kmax, idx_out, cnt_out, S);
    return;
  }
  topk_output<Sync>(score, n, take, true, thr, need_eq, kmax, idx_out, cnt_out, S);
}

// Register-resident selection for n <= 16 * kSelThreads candidates: the same
// selection as block_topk_impl (forced first and last index; the take highest
// keys among 1 .. n-2, ties to the lower index; ascending output).  Warp w owns
// the indices [32*M*w, 32*M*(w+1)); its lane l holds indices 32*M*w + 32*j + l,
// j < M, in registers (conflict-free loads, every score read once).
// Threshold: one value histogram (kHistBins linear bins over the candidates'
// key range, a monotone map) locates the bin b* of the take-th largest key.
// When all of b*'s keys are needed (the usual case: the bin holds one key), the
// selection is every key with a bin >= b*; otherwise b*'s keys (at most
// kHistCand) are gathered and ranked directly for the exact threshold key and
// the number of its ties to admit (lowest indices first).  Output: per-row
// ballots of the sure and the tied keys give each selected index its position
// from the warp's prefix counts.  Five barriers in the usual case (range,
// histogram, bin totals, bin choice, warp counts), seven with the bin ranked.
// Returns false (nothing written, every thread returning together) when the
// key range has no finite positive width or the threshold bin holds more than
// kHistCand keys; the caller then synchronises and runs the general selection.
template <int M, typename Sync, typename LoadF>
__device__ __forceinline__ bool block_topk_reg(LoadF score, int n, int budget, int kmax, int32_t* __restrict__ idx_out,
                                               int32_t* __restrict__ cnt_out, uint32_t S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t hist = S + static_cast<uint32_t>(offsetof(TopkShared, hist));
  const uint32_t cand = S + static_cast<uint32_t>(offsetof(TopkShared, cand));
  const uint32_t wmax = S + static_cast<uint32_t>(offsetof(TopkShared, wmax));
  const uint32_t wmin = S + static_cast<uint32_t>(offsetof(TopkShared, wmin));
  const uint32_t wdef = S + static_cast<uint32_t>(offsetof(TopkShared, wdef));
  const uint32_t weq = S + static_cast<uint32_t>(offsetof(TopkShared, weq));
  const uint32_t bsel = S + static_cast<uint32_t>(offsetof(TopkShared, bsel));
  const uint32_t fin_thr = S + static_cast<uint32_t>(offsetof(TopkShared, fin_thr));
  const uint32_t fin_need = S + static_cast<uint32_t>(offsetof(TopkShared, fin_need));
  const int last = n - 1;
  const int ncand = n > 2 ? n - 2 : 0;
  const int take = budget <= 0 ? 0 : (budget < ncand ? budget : ncand);
  const bool by_key = take > 0 && take < ncand;
  const int i0 = 32 * M * warp + lane;  // index of row j: i0 + 32 * j
  const uint32_t lt = (1u << lane) - 1u;
  float v[M];
  uint32_t key[M];
#pragma unroll
  for (int j = 0; j < M; ++j) {
    const int b = i0 + 32 * j;
    v[j] = (b >= 1 && b < last) ? score(b) : 0.f;
  }
  // selection rule: by bin (every key whose bin is >= b*) when the threshold bin is taken
  // whole, else by key (keys above thr, and the first need_eq keys equal to it)
  int bstar = 0;
  bool by_bin = false;
  uint32_t thr = 0u, need_eq = 0u;
  int bn[M];
#pragma unroll
  for (int j = 0; j < M; ++j) {
    key[j] = float_key(v[j]);
    bn[j] = 0;
  }
  if (by_key) {
    uint32_t kmx = 0u, kmn = 0xFFFFFFFFu;
#pragma unroll
    for (int j = 0; j < M; ++j) {
      const int b = i0 + 32 * j;
      if (b >= 1 && b < last) {
        kmx = max(kmx, key[j]);
        kmn = min(kmn, key[j]);
      }
    }
    kmx = __reduce_max_sync(0xFFFFFFFFu, kmx);
    kmn = __reduce_min_sync(0xFFFFFFFFu, kmn);
    if (lane == 0) {
      sts_u32(wmax + 4u * warp, kmx);
      sts_u32(wmin + 4u * warp, kmn);
    }
    for (int i = tid; i < kHistBins / 4; i += kSelThreads)
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(hist + 16u * i), "r"(0u) : "memory");
    if (tid == 0) sts_u32(bsel + 12u, 0u);
    Sync::sync();  // 1: key range, cleared histogram
    uint32_t klo = 0xFFFFFFFFu, khi = 0u;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
      khi = max(khi, lds_u32(wmax + 4u * w));
      klo = min(klo, lds_u32(wmin + 4u * w));
    }
    if (klo == khi) {  // every candidate has the threshold key
      thr = klo;
      need_eq = static_cast<uint32_t>(take);
    } else {
      const float smin = key_float(klo), smax = key_float(khi);
      const float inv = static_cast<float>(kHistBins) / (smax - smin);
      if (!(inv > 0.f && inv < 3.0e38f && smax - smin < 3.0e38f)) return false;  // uniform
#pragma unroll
      for (int j = 0; j < M; ++j) {
        const int b = i0 + 32 * j;
        // bin = floor((v - smin) * inv) clamped to the last bin: a monotone map of the score
        // (the floor by a round-down add of 2^23, whose low mantissa bits are then the integer)
        const float f = fminf((v[j] - smin) * inv, static_cast<float>(kHistBins - 1));
        bn[j] = __float_as_int(__fadd_rd(f, 8388608.0f)) - 0x4B000000;
        if (b >= 1 && b < last) red_add_shared(hist + 4u * static_cast<uint32_t>(bn[j]), 1u);
      }
      Sync::sync();  // 2: histogram
      // thread t holds bins kHistBins-1-8t .. kHistBins-8-8t (descending)
      uint32_t c[8];
      {
        const uint4 hi4 = lds_u32x4(hist + 4u * (kHistBins - 4 - 8 * tid));
        const uint4 lo4 = lds_u32x4(hist + 4u * (kHistBins - 8 - 8 * tid));
        c[0] = hi4.w; c[1] = hi4.z; c[2] = hi4.y; c[3] = hi4.x;
        c[4] = lo4.w; c[5] = lo4.z; c[6] = lo4.y; c[7] = lo4.x;
      }
      const uint32_t sum = ((c[0] + c[1]) + (c[2] + c[3])) + ((c[4] + c[5]) + (c[6] + c[7]));
      uint32_t inc = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) sts_u32(wdef + 4u * warp, inc);
      Sync::sync();  // 3: warp totals of the bins
      uint32_t run = inc - sum;
#pragma unroll
      for (int w = 0; w < kSelWarps; ++w) run += w < warp ? lds_u32(wdef + 4u * w) : 0u;
      const uint32_t remaining = static_cast<uint32_t>(take);
      if (run < remaining && remaining <= run + sum) {  // the threshold bin is one of this thread's
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (run < remaining && remaining <= run + c[e]) {
            sts_u32(bsel, static_cast<uint32_t>(kHistBins - 1 - 8 * tid - e));
            sts_u32(bsel + 4u, remaining - run);
            sts_u32(bsel + 8u, c[e]);
          }
          run += c[e];
        }
      }
      Sync::sync();  // 4: the bin
      bstar = static_cast<int>(lds_u32(bsel));
      const uint32_t rem = lds_u32(bsel + 4u), inside = lds_u32(bsel + 8u);
      if (rem >= inside) {
        by_bin = true;
      } else {  // only some of the bin's keys: rank them
        if (inside > static_cast<uint32_t>(kHistCand)) return false;  // uniform
        uint32_t bal[M], tot = 0u;
#pragma unroll
        for (int j = 0; j < M; ++j) {
          const int b = i0 + 32 * j;
          bal[j] = __ballot_sync(0xFFFFFFFFu, b >= 1 && b < last && bn[j] == bstar);
          tot += static_cast<uint32_t>(__popc(bal[j]));
        }
        // slots: one atomic per warp (the order of the gathered keys does not matter)
        uint32_t base = 0u;
        if (lane == 0 && tot > 0u)
          asm volatile("atom.shared.add.u32 %0, [%1], %2;" : "=r"(base) : "r"(bsel + 12u), "r"(tot) : "memory");
        base = __shfl_sync(0xFFFFFFFFu, base, 0);
#pragma unroll
        for (int j = 0; j < M; ++j) {
          if ((bal[j] >> lane) & 1u) sts_u32(cand + 4u * (base + static_cast<uint32_t>(__popc(bal[j] & lt))), key[j]);
          base += static_cast<uint32_t>(__popc(bal[j]));
        }
        Sync::sync();  // 5: gathered
        if (tid < static_cast<int>(inside)) {
          const uint32_t kt = lds_u32(cand + 4u * tid);
          uint32_t above = 0u, same = 0u;
          for (uint32_t j0 = 0; j0 < inside; j0 += 4) {
            const uint4 x = lds_u32x4(cand + 4u * j0);
            const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const bool ok = j0 + q < inside;  // entries past the count are stale
              above += (ok && xv[q] > kt) ? 1u : 0u;
              same += (ok && xv[q] == kt) ? 1u : 0u;
            }
          }
          if (above < rem && rem <= above + same) {  // every such thread writes the same pair
            sts_u32(fin_thr, kt);
            sts_u32(fin_need, rem - above);
          }
        }
        Sync::sync();  // 6: threshold key
        thr = lds_u32(fin_thr);
        need_eq = lds_u32(fin_need);
      }
    }
  }
  // ---- output: ballots of the sure and the tied keys per row; warp counts; positions
  uint32_t sb[M], tb[M], dw = 0u, ew = 0u;
#pragma unroll
  for (int j = 0; j < M; ++j) {
    const int b = i0 + 32 * j;
    bool sure = false, tie = false;
    if (b < n) {
      if (b == 0 || b == last) {
        sure = true;
      } else if (take > 0) {
        if (!by_key) {
          sure = true;
        } else if (by_bin) {
          sure = bn[j] >= bstar;
        } else {
          sure = key[j] > thr;
          tie = key[j] == thr;
        }
      }
    }
    sb[j] = __ballot_sync(0xFFFFFFFFu, sure);
    tb[j] = __ballot_sync(0xFFFFFFFFu, tie);
    dw += static_cast<uint32_t>(__popc(sb[j]));
    ew += static_cast<uint32_t>(__popc(tb[j]));
  }
  if (lane == 0) sts_u32(weq + 4u * warp, (dw << 16) | ew);
  Sync::sync();  // warp counts
  uint32_t dcum = 0u, ecum = 0u, dall = 0u, eall = 0u;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    const uint32_t x = lds_u32(weq + 4u * w);
    dcum += w < warp ? x >> 16 : 0u;
    ecum += w < warp ? x & 0xFFFFu : 0u;
    dall += x >> 16;
    eall += x & 0xFFFFu;
  }
  const uint32_t total = dall + min(eall, need_eq);
#pragma unroll
  for (int j = 0; j < M; ++j) {
    // selected before this index: the sure ones, and the ties while the budget for them lasts
    const uint32_t d_at = dcum + static_cast<uint32_t>(__popc(sb[j] & lt));
    const uint32_t e_at = ecum + static_cast<uint32_t>(__popc(tb[j] & lt));
    const bool sel = ((sb[j] >> lane) & 1u) || (((tb[j] >> lane) & 1u) && e_at < need_eq);
    const uint32_t at = d_at + min(e_at, need_eq);
    if (sel && at < static_cast<uint32_t>(kmax)) idx_out[at] = i0 + 32 * j;
    dcum += static_cast<uint32_t>(__popc(sb[j]));
    ecum += static_cast<uint32_t>(__popc(tb[j]));
  }
  for (int i = static_cast<int>(total) + tid; i < kmax; i += kSelThreads) idx_out[i] = -1;
  if (tid == 0) *cnt_out = static_cast<int32_t>(total);
  return true;
}

// scores at shared address sc
// Either threshold search gives the same selection; the digit passes are faster up to about a
// thousand candidates or for budgets of a sixteenth of them or more, the value histogram for
// small budgets over more candidates (measured on the B300: 512 candidates ~5.2k vs ~5.6k
// cycles, 4096 candidates with k = 80 ~18k vs ~15k, 16384 ~61k vs ~46k; per-query selections
// of 256 out of up to 4096 tokens ran 70.7 vs 88.1 us in all).
constexpr int kHistMinN = 1024;

template <typename Sync = SyncCta>
__device__ __forceinline__ void block_topk_fast(uint32_t sc, int n, int budget, int kmax, int32_t* __restrict__ idx_out,
                                                int32_t* __restrict__ cnt_out, uint32_t S) {
  auto score = [&](int b) { return lds_f32(sc + 4u * static_cast<uint32_t>(b)); };
  if (n <= 16 * kSelThreads) {
    bool done;
    if (n <= 2 * kSelThreads)
      done = block_topk_reg<2, Sync>(score, n, budget, kmax, idx_out, cnt_out, S);
    else if (n <= 4 * kSelThreads)
      done = block_topk_reg<4, Sync>(score, n, budget, kmax, idx_out, cnt_out, S);
    else if (n <= 8 * kSelThreads)
      done = block_topk_reg<8, Sync>(score, n, budget, kmax, idx_out, cnt_out, S);
    else
      done = block_topk_reg<16, Sync>(score, n, budget, kmax, idx_out, cnt_out, S);
    if (done) return;
    Sync::sync();  // every thread has left the register selection
  }
  if (n <= kHistMinN || 16LL * budget >= n)
    block_topk_impl<Sync>(score, n, budget, kmax, idx_out, cnt_out, S);
  else
    block_topk_hist_impl<Sync>(score, n, budget, kmax, idx_out, cnt_out, S);
}

// scores at shared address sc
__device__ __forceinline__ void block_topk(uint32_t sc, int n, int budget, int kmax, int32_t* __restrict__ idx_out,
                                           int32_t* __restrict__ cnt_out, uint32_t S) {
  block_topk_impl([&](int b) { return lds_f32(sc + 4u * static_cast<uint32_t>(b)); }, n, budget, kmax, idx_out,
                  cnt_out, S);
}

// --------------------------------------------------------------------------
// Decode selection.  grid (CS, groups), cluster (CS, 1, 1), kSelThreads.
// CTA rank r of group g's cluster scores blocks [r*per, r*per + per) of the
// group's sketch; the scores go straight into CTA rank 0's shared memory
// (distributed shared memory), and after one cluster barrier rank 0 runs the
// top-k over all nb scores.
//
// The sketch rows arrive by TMA in chunks of 64 rows (one mbarrier per chunk,
// 128-byte swizzle, one box per 32 columns), so scoring starts on the first
// chunk while the rest are in flight.  bf16 queries: the scores are a small
// matrix product S[row, r] = sketch[row, :] . q[r, :] on the tensor cores
// (mma.sync m16n8k16, fp32 accumulation), with the fp32 sketch split into
// three bf16 parts (hi, mid, lo: each the rounded remainder of the previous)
// so that the product keeps float32 accuracy while q (bf16) is exact; one warp
// per 16-row M tile, the max over the group's R rows taken from the
// accumulator fragments.  fp32 queries: one thread per row, FMA dot products.
constexpr int kSelTileRows = 256;  // rows staged per pass (at most 4 chunks)
constexpr int kSelChunkRows = 64;

// bytes of the staged query rows: bf16 rows (whole n8 tiles; rows past the
// group's R only feed accumulator columns that are never read), or fp32 rows
// with the scale folded in for fp32 queries
__host__ __device__ constexpr int sel_q_bytes(int D, int RMAX, bool bf16) {
  return bf16 ? ((RMAX + 7) / 8) * 8 * D * 2 : RMAX * D * 4;
}

// Shared layout (runtime): staged sketch chunks | q rows | gathered scores (rank 0) | top-k scratch |
// mbarriers (one per sketch chunk, then one for q)
struct SelDecodeLayout {
  int tile_bytes, q_bytes, nb;
  __host__ __device__ int q_off() const { return tile_bytes; }
  __host__ __device__ int all_off() const { return tile_bytes + q_bytes; }
  __host__ __device__ int topk_off() const { return all_off() + ((nb * 4 + 15) / 16) * 16; }
  __host__ __device__ int bar_off() const { return topk_off() + static_cast<int>(((sizeof(TopkShared) + 15) / 16) * 16); }
  __host__ __device__ int bytes() const { return bar_off() + 64 + 1024; }
};

// staged bytes for a pass of tile_rows rows with D fp32 columns
__host__ __device__ constexpr int sel_tile_bytes(int tile_rows, int D) {
  return ((tile_rows + kSelChunkRows - 1) / kSelChunkRows) * (D * 4 / 128) * kSelChunkRows * 128;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// c += a * b, m16n8k16, bf16 inputs, fp32 accumulators
__device__ __forceinline__ void sel_mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (x0, x1) = hi + mid + lo, each a bf16 pair (x0 in the low half), each part
// the bf16 rounding of what the previous parts leave (the remainders are exact
// in fp32), so the three carry 24 significant bits of each value.
__device__ __forceinline__ void split3_bf16(float x0, float x1, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  hi = pack_bf16x2(x0, x1);
  const float r0 = x0 - __uint_as_float(hi << 16), r1 = x1 - __uint_as_float(hi & 0xFFFF0000u);
  mid = pack_bf16x2(r0, r1);
  const float s0 = r0 - __uint_as_float(mid << 16), s1 = r1 - __uint_as_float(mid & 0xFFFF0000u);
  lo = pack_bf16x2(s0, s1);
}

// byte offset of fp32 column c (even) of staged row r in the chunked, swizzled tile
template <int D>
__device__ __forceinline__ uint32_t sel_tile_off(int r, int c) {
  constexpr int kBoxes = D * 4 / 128;
  const int rr = r & (kSelChunkRows - 1), cb = c & 31;
  return static_cast<uint32_t>((((r >> 6) * kBoxes + (c >> 5)) * kSelChunkRows + rr) * 128 +
                               ((((cb >> 2) ^ (rr & 7))) << 4) + (cb & 3) * 4);
}

// grid (CS, groups), cluster (CS, 1, 1), kSelThreads threads.
template <typename TE, int D, int RMAX>
__global__ void __launch_bounds__(kSelThreads) select_decode_kernel(
    const __grid_constant__ CUtensorMap sk_map, const TE* __restrict__ q, int T, int Hq, int Hkv, int nb,
    int nb_cap, float scale, int per, int tile_rows, int k, float* __restrict__ scores_out,
    int32_t* __restrict__ idx, int32_t* __restrict__ cnt, int kmax, int topdelta, float delta) {
  constexpr int kBoxes = D * 4 / 128;
  constexpr bool kTc = std::is_same<TE, __nv_bfloat16>::value;
  constexpr int NT = ((RMAX + 7) / 8) * 8;  // query rows padded to whole n8 tiles
  constexpr uint32_t kChunkBytes = kBoxes * kSelChunkRows * 128;
  extern __shared__ __align__(1024) uint8_t smem_sel_dec[];
  // 1024-byte aligned base (the 128-byte swizzle pattern repeats every 1024 bytes)
  uint8_t* smem = smem_sel_dec + ((1024u - (smem_u32(smem_sel_dec) & 1023u)) & 1023u);
  const SelDecodeLayout lay{sel_tile_bytes(tile_rows, D), sel_q_bytes(D, RMAX, kTc), nb};
  const uint32_t tile = smem_u32(smem);
  const uint32_t q_sh = tile + lay.q_off();
  const uint32_t all = tile + lay.all_off();     // rank 0: the group's nb scores
  const uint32_t topk_s = tile + lay.topk_off();  // TopkShared
  const uint32_t bar0 = tile + lay.bar_off();     // chunk c's mbarrier at bar0 + 8c

  cluster_arrive_relaxed();  // paired with the wait before the first remote store
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y;
  const uint32_t rank = cluster_ctarank();
  const int G = Hq / Hkv, R = G * T;
  const int b = g / Hkv, kvh = g % Hkv;
  const int b0 = static_cast<int>(rank) * per;
  const int b1 = min(nb, b0 + per);

  constexpr int kChunks = kSelTileRows / kSelChunkRows;
  const uint32_t qbar = bar0 + 8 * kChunks;
  pdl_launch_dependents();
  if (tid == 0) {
    prefetch_tmap(&sk_map);
#pragma unroll
    for (int c = 0; c <= kChunks; ++c) mbar_init(bar0 + 8 * c, 1);
    fence_mbar_init();
  }
  pdl_wait();  // the sketch and q may come from the previous kernel

  auto issue_pass = [&](int t0) {  // thread 0: the sketch chunks of the pass starting at row t0
    const int nch = (min(tile_rows, b1 - t0) + kSelChunkRows - 1) / kSelChunkRows;
    for (int c = 0; c < nch; ++c) {
      mbar_arrive_expect_tx(bar0 + 8 * c, kChunkBytes);
#pragma unroll
      for (int bx = 0; bx < kBoxes; ++bx)
        tma_g2s_2d(tile + (c * kBoxes + bx) * kSelChunkRows * 128, &sk_map, bx * 32,
                   g * nb_cap + t0 + c * kSelChunkRows, bar0 + 8 * c);
    }
  };
  // q rows of this group (row r = t * G + head; the G heads of a token are
  // contiguous): bf16 rows come in by bulk copies queued ahead of the sketch
  if constexpr (kTc) {
    if (tid == 0) {
      mbar_arrive_expect_tx(qbar, static_cast<uint32_t>(R * D * 2));
      for (int t = 0; t < T; ++t)
        bulk_g2s(q_sh + t * G * D * 2,
                 q + ((static_cast<size_t>(b) * T + t) * Hq + kvh * G) * D, G * D * 2, qbar);
      if (b0 < b1) issue_pass(b0);
    }
  } else {
    if (tid == 0 && b0 < b1) issue_pass(b0);
    for (int i = tid; i < RMAX * D; i += kSelThreads) {
      const int r = i / D, c = i % D;
      float v = 0.f;
      if (r < R) {
        const int t = r / G, hh = r % G;
        v = static_cast<float>(q[((static_cast<size_t>(b) * T + t) * Hq + kvh * G + hh) * D + c]) * scale;
      }
      sts_f32(q_sh + 4u * i, v);
    }
  }
  const uint32_t all0 = map_cluster(all, 0);  // rank 0's gather array
  __syncthreads();  // fp32 q staged
  cluster_wait();   // every CTA of the cluster is running: remote stores are safe
  bool ok = true;
  const int gq = lane >> 2, tq = lane & 3;
  // B fragments (q, k16 x n8, two bf16 along k per register) held in registers
  uint32_t bq[kTc ? NT / 8 : 1][kTc ? D / 16 : 1][2];
  if constexpr (kTc) {
    ok = mbar_wait(qbar, 0);
#pragma unroll
    for (int nt = 0; nt < NT / 8; ++nt) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t qb = q_sh + 2u * ((nt * 8 + gq) * D + ks * 16 + 2 * tq);
        bq[nt][ks][0] = lds_u32(qb);
        bq[nt][ks][1] = lds_u32(qb + 16u);
      }
    }
  }
  int pass = 0;
  for (int t0 = b0; t0 < b1; t0 += tile_rows, ++pass) {
    const int rows = min(tile_rows, b1 - t0);
    const int nch = (rows + kSelChunkRows - 1) / kSelChunkRows;
    const uint32_t parity = static_cast<uint32_t>(pass & 1);
    if (tid == 0 && pass > 0) issue_pass(t0);
    if constexpr (kTc) {
      int have = -1;  // chunk this warp has waited for
      for (int m = warp; m * 16 < rows; m += kSelWarps) {
        const int ch = (m * 16) / kSelChunkRows;
        if (ch != have) {
          ok = mbar_wait(bar0 + 8 * ch, parity) && ok;
          have = ch;
        }
        // hi, mid and lo products accumulate separately (three independent MMA chains)
        float acc[3][NT / 8][4];
#pragma unroll
        for (int j = 0; j < 3; ++j)
#pragma unroll
          for (int nt = 0; nt < NT / 8; ++nt) acc[j][nt][0] = acc[j][nt][1] = acc[j][nt][2] = acc[j][nt][3] = 0.f;
        const int r0 = m * 16 + gq, r1 = r0 + 8;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int c0 = ks * 16 + 2 * tq;
          const float2 x00 = lds_f32x2(tile + sel_tile_off<D>(r0, c0));
          const float2 x10 = lds_f32x2(tile + sel_tile_off<D>(r1, c0));
          const float2 x01 = lds_f32x2(tile + sel_tile_off<D>(r0, c0 + 8));
          const float2 x11 = lds_f32x2(tile + sel_tile_off<D>(r1, c0 + 8));
          uint32_t ah[4], am[4], al[4];
          split3_bf16(x00.x, x00.y, ah[0], am[0], al[0]);
          split3_bf16(x10.x, x10.y, ah[1], am[1], al[1]);
          split3_bf16(x01.x, x01.y, ah[2], am[2], al[2]);
          split3_bf16(x11.x, x11.y, ah[3], am[3], al[3]);
#pragma unroll
          for (int nt = 0; nt < NT / 8; ++nt) {
            sel_mma_bf16(acc[0][nt], ah, bq[nt][ks][0], bq[nt][ks][1]);
            sel_mma_bf16(acc[1][nt], am, bq[nt][ks][0], bq[nt][ks][1]);
            sel_mma_bf16(acc[2][nt], al, bq[nt][ks][0], bq[nt][ks][1]);
          }
        }
        // row max over the group's R query rows (accumulator columns n < R)
        float s0 = -INFINITY, s1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT / 8; ++nt) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (nt * 8 + 2 * tq + j < R) {
              s0 = fmaxf(s0, scale * (acc[0][nt][j] + (acc[1][nt][j] + acc[2][nt][j])));
              s1 = fmaxf(s1, scale * (acc[0][nt][2 + j] + (acc[1][nt][2 + j] + acc[2][nt][2 + j])));
            }
          }
        }
        s0 = fmaxf(s0, __shfl_xor_sync(0xFFFFFFFFu, s0, 1));
        s0 = fmaxf(s0, __shfl_xor_sync(0xFFFFFFFFu, s0, 2));
        s1 = fmaxf(s1, __shfl_xor_sync(0xFFFFFFFFu, s1, 1));
        s1 = fmaxf(s1, __shfl_xor_sync(0xFFFFFFFFu, s1, 2));
        if (tq == 0) {
          if (r0 < rows) {
            if (scores_out) scores_out[static_cast<size_t>(g) * nb + t0 + r0] = s0;
            st_cluster_f32(all0 + 4u * static_cast<uint32_t>(t0 + r0), s0);
          }
          if (r1 < rows) {
            if (scores_out) scores_out[static_cast<size_t>(g) * nb + t0 + r1] = s1;
            st_cluster_f32(all0 + 4u * static_cast<uint32_t>(t0 + r1), s1);
          }
        }
      }
      // chunks this warp never waited for: their copies have still landed before
      // the buffer is reused (the barrier below orders every warp after them)
      if (tid == 0) {
        for (int c = 0; c < nch; ++c) ok = mbar_wait(bar0 + 8 * c, parity) && ok;
      }
    } else {
      const int r = tid;
      if (r < rows) {
        ok = mbar_wait(bar0 + 8 * (r / kSelChunkRows), parity) && ok;
        float acc[RMAX];
#pragma unroll
        for (int i = 0; i < RMAX; ++i) acc[i] = 0.f;
#pragma unroll 4
        for (int c = 0; c < D / 4; ++c) {
          const float4 kv = lds_f32x4(tile + sel_tile_off<D>(r, c * 4));
#pragma unroll
          for (int i = 0; i < RMAX; ++i) {
            const float4 qv = lds_f32x4(q_sh + 4u * (i * D + c * 4));
            acc[i] = fmaf(qv.x, kv.x, acc[i]);
            acc[i] = fmaf(qv.y, kv.y, acc[i]);
            acc[i] = fmaf(qv.z, kv.z, acc[i]);
            acc[i] = fmaf(qv.w, kv.w, acc[i]);
          }
        }
        float s = -INFINITY;
#pragma unroll
        for (int i = 0; i < RMAX; ++i)
          if (i < R) s = fmaxf(s, acc[i]);
        if (scores_out) scores_out[static_cast<size_t>(g) * nb + t0 + r] = s;
        st_cluster_f32(all0 + 4u * static_cast<uint32_t>(t0 + r), s);
      }
      if (tid == 0) {
        for (int c = 0; c < nch; ++c) ok = mbar_wait(bar0 + 8 * c, parity) && ok;
      }
    }
    if (__syncthreads_or(!ok)) break;  // the staged chunks are refilled next pass
  }
  cluster_sync();  // all scores have landed in rank 0
  if (rank != 0) return;
  int budget = k;
  if (topdelta) {
    // top-delta ("Faster Than Flash" Sec. 2): the candidates scoring at least the
    // pseudo-maximum (over the sink and local blocks) minus delta, at most k of them
    const float thr = fmaxf(lds_f32(all), lds_f32(all + 4u * (nb - 1))) - delta;
    int c = 0;
    for (int base = 0; base < nb; base += kSelThreads) {
      const int bb = base + tid;
      c += __syncthreads_count(bb >= 1 && bb < nb - 1 && lds_f32(all + 4u * bb) >= thr);
    }
    budget = min(c, k);
  }
  block_topk_fast(all, nb, budget, kmax, idx + static_cast<size_t>(g) * kmax, cnt + g, topk_s);
}

// --------------------------------------------------------------------------
// Selection from a given score array (mass mode, decode or prefill).
// grid (nq, groups).  Scores: [groups, nq, nb]; unit (g, i) considers its
// causal blocks 0..c_i-1 (c_i from the host-side rule), forced {0, c_i - 1}.
__global__ void __launch_bounds__(kSelThreads) select_given_kernel(const float* __restrict__ scores, int nb,
                                                                   int prefill, int L, int qtile, int Bk, int k,
                                                                   int frac_num, int frac_den,
                                                                   int32_t* __restrict__ idx,
                                                                   int32_t* __restrict__ cnt, int kmax) {
  extern __shared__ __align__(1024) uint8_t smem_sel_given[];
  const uint32_t topk_s = smem_u32(smem_sel_given);
  const uint32_t sc = topk_s + static_cast<uint32_t>(((sizeof(TopkShared) + 15) / 16) * 16);
  const int i = blockIdx.x, g = blockIdx.y, nq = gridDim.x;
  int nvalid = nb, budget = k;
  if (prefill) {
    const int last = min((i + 1) * qtile, L) - 1;
    nvalid = last / Bk + 1;
    if (frac_num > 0) budget = k + (frac_num * nvalid + frac_den - 1) / frac_den;
  }
  const size_t u = static_cast<size_t>(g) * nq + i;
  for (int b0 = threadIdx.x; b0 < nvalid; b0 += 8 * kSelThreads) {  // eight loads in flight per thread
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int bb = b0 + j * kSelThreads;
      v[j] = bb < nvalid ? __ldg(scores + u * nb + bb) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int bb = b0 + j * kSelThreads;
      if (bb < nvalid) sts_f32(sc + 4u * bb, v[j]);
    }
  }
  __syncthreads();
  block_topk_fast(sc, nvalid, budget, kmax, idx + u * kmax, cnt + u, topk_s);
}

// Selection from a given score array too large for shared memory (one-token
// blocks over a long context): the same selection, with every score read from
// global memory (L2) in each pass.  grid (nq, groups), kSelThreads.
__global__ void __launch_bounds__(kSelThreads, 1) select_given_global_kernel(const float* __restrict__ scores, int nb,
                                                                          int k, int32_t* __restrict__ idx,
                                                                          int32_t* __restrict__ cnt, int kmax) {
  extern __shared__ __align__(16) uint8_t smem_sel_global[];
  const size_t u = static_cast<size_t>(blockIdx.y) * gridDim.x + blockIdx.x;
  const float* sc = scores + u * nb;
  block_topk_impl([&](int b) { return __ldg(sc + b); }, nb, k, kmax, idx + u * kmax, cnt + u,
                  smem_u32(smem_sel_global));
}

// --------------------------------------------------------------------------
// Selection from a long given score array (one-token blocks over a long
// context) by a cluster of CS CTAs per unit: CTA rank r holds the scores
// [r*per, r*per + per) in shared memory.  The radix passes build a histogram
// per CTA, add it into CTA rank 0's through distributed shared memory, and
// after one cluster barrier every CTA reads the cluster total and derives the
// same digit; the output pass adds the CTAs' counts the same way, so each CTA
// writes its own selections at their ascending positions.  Same selection
// as block_topk.  grid (CS, units), cluster (CS, 1, 1), kSelThreads.
constexpr int kSelClusterPer = 16384;  // scores per CTA

struct SelClusterShared {
  uint32_t lhist[4][256];  // this CTA's digit counts per pass
  uint32_t ghist[4][256];  // rank 0: the cluster's
  uint32_t cdef[16], ceq[16];  // rank 0: per-CTA output counts
  uint32_t wdef[kSelWarps], weq[kSelWarps];
};

__device__ __forceinline__ void red_add_cluster(uint32_t a, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_cluster_u32x4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

__global__ void __launch_bounds__(kSelThreads, 1) select_given_cluster_kernel(const float* __restrict__ scores, int nb,
                                                                           int per, int k, int32_t* __restrict__ idx,
                                                                           int32_t* __restrict__ cnt, int kmax) {
  extern __shared__ __align__(16) uint8_t smem_sel_cl[];
  const uint32_t S = smem_u32(smem_sel_cl);
  const uint32_t lhist = S + static_cast<uint32_t>(offsetof(SelClusterShared, lhist));
  const uint32_t ghist = S + static_cast<uint32_t>(offsetof(SelClusterShared, ghist));
  const uint32_t wdef = S + static_cast<uint32_t>(offsetof(SelClusterShared, wdef));
  const uint32_t weq = S + static_cast<uint32_t>(offsetof(SelClusterShared, weq));
  const uint32_t sc = S + static_cast<uint32_t>(((sizeof(SelClusterShared) + 15) / 16) * 16);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int CS = gridDim.x;
  const size_t u = blockIdx.y;
  const int b0 = static_cast<int>(rank) * per, b1 = min(nb, b0 + per), m = max(0, b1 - b0);
  const uint32_t ghist0 = map_cluster(ghist, 0);
  const uint32_t cdef0 = map_cluster(S + static_cast<uint32_t>(offsetof(SelClusterShared, cdef)), 0);
  const uint32_t ceq0 = map_cluster(S + static_cast<uint32_t>(offsetof(SelClusterShared, ceq)), 0);

  const float* src = scores + u * nb + b0;
  for (int i0 = tid; i0 < m; i0 += 16 * kSelThreads) {  // sixteen loads in flight per thread
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int i = i0 + j * kSelThreads;
      v[j] = i < m ? __ldg(src + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int i = i0 + j * kSelThreads;
      if (i < m) sts_f32(sc + 4u * i, v[j]);
    }
  }
  for (int i = tid; i < 2 * 4 * 256 / 4; i += kSelThreads)  // lhist and ghist are adjacent
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(lhist + 16u * i), "r"(0u) : "memory");
  cluster_sync();  // every slice staged and every histogram zeroed before any remote add

  const int n = nb, last = n - 1;
  const int ncand = n > 2 ? n - 2 : 0;
  const int take = k <= 0 ? 0 : (k < ncand ? k : ncand);
  const bool by_key = take > 0 && take < ncand;
  uint32_t thr = 0u, need_eq = 0u;
  if (by_key) {
    uint32_t prefix = 0u, mask = 0u, remaining = static_cast<uint32_t>(take);
    for (int p = 0; p < 4; ++p) {
      const int shift = 24 - 8 * p;
      const uint32_t lp = lhist + 1024u * p;
      for (int i = tid; i < m; i += kSelThreads) {
        const int gi = b0 + i;
        const uint32_t key = float_key(lds_f32(sc + 4u * i));
        if (gi >= 1 && gi < last && (key & mask) == prefix) red_add_shared(lp + 4u * ((key >> shift) & 255u), 1u);
      }
      __syncthreads();
      {
        const uint32_t v = lds_u32(lp + 4u * tid);
        if (v) red_add_cluster(ghist0 + 1024u * p + 4u * tid, v);
      }
      cluster_sync();  // the cluster's counts for this pass are complete in rank 0
      const uint32_t gp = ghist0 + 1024u * p;
      const uint4 lo4 = ld_cluster_u32x4(gp + 4u * (248 - 8 * lane)), hi4 = ld_cluster_u32x4(gp + 4u * (252 - 8 * lane));
      const uint32_t c[8] = {hi4.w, hi4.z, hi4.y, hi4.x, lo4.w, lo4.z, lo4.y, lo4.x};
      uint32_t sum = 0u;
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += c[e];
      uint32_t inc = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
      }
      uint32_t run = inc - sum, hit = 0u, dsel = 0u, rem = 0u;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (hit == 0u && run < remaining && remaining <= run + c[e]) {
          hit = 1u;
          dsel = 255u - 8u * static_cast<uint32_t>(lane) - static_cast<uint32_t>(e);
          rem = remaining - run;
        }
        run += c[e];
      }
      const int srcl = (__ffs(__ballot_sync(0xFFFFFFFFu, hit != 0u)) - 1) & 31;
      dsel = __shfl_sync(0xFFFFFFFFu, dsel, srcl);
      rem = __shfl_sync(0xFFFFFFFFu, rem, srcl);
      prefix |= dsel << shift;
      mask |= 255u << shift;
      remaining = rem;
    }
    thr = prefix;
    need_eq = remaining;
  }
  auto classify = [&](int i, bool& def, bool& eq) {  // local index i, global index b0 + i
    def = false;
    eq = false;
    if (i >= m) return;
    const int gi = b0 + i;
    if (gi == 0 || gi == last) {
      def = true;
    } else if (take > 0) {
      if (!by_key) {
        def = true;
      } else {
        const uint32_t key = float_key(lds_f32(sc + 4u * i));
        def = key > thr;
        eq = key == thr;
      }
    }
  };
  const int span = ((m + kSelThreads - 1) / kSelThreads) * 32;
  const int w0 = warp * span;
  uint32_t ndef = 0u, neq = 0u;
  for (int base = w0; base < w0 + span; base += 32) {
    bool d, e;
    classify(base + lane, d, e);
    ndef += __popc(__ballot_sync(0xFFFFFFFFu, d));
    neq += __popc(__ballot_sync(0xFFFFFFFFu, e));
  }
  if (lane == 0) {
    sts_u32(wdef + 4u * warp, ndef);
    sts_u32(weq + 4u * warp, neq);
  }
  __syncthreads();
  uint32_t def_before = 0u, eq_before = 0u, cta_def = 0u, cta_eq = 0u;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    const uint32_t a = lds_u32(wdef + 4u * w), e = lds_u32(weq + 4u * w);
    def_before += w < warp ? a : 0u;
    eq_before += w < warp ? e : 0u;
    cta_def += a;
    cta_eq += e;
  }
  if (tid == 0) {
    st_cluster_u32(cdef0 + 4u * rank, cta_def);
    st_cluster_u32(ceq0 + 4u * rank, cta_eq);
  }
  cluster_sync();  // every CTA's counts are in rank 0
  uint32_t def_all = 0u, eq_all = 0u;
  for (int r = 0; r < CS; ++r) {
    const uint32_t a = ld_cluster_u32(cdef0 + 4u * r), e = ld_cluster_u32(ceq0 + 4u * r);
    def_before += r < static_cast<int>(rank) ? a : 0u;
    eq_before += r < static_cast<int>(rank) ? e : 0u;
    def_all += a;
    eq_all += e;
  }
  const uint32_t total = def_all + min(eq_all, need_eq);
  uint32_t pos = def_before + min(eq_before, need_eq);
  uint32_t eq_seen = eq_before;
  const uint32_t lt = (1u << lane) - 1u;
  int32_t* out = idx + u * kmax;
  for (int base = w0; base < w0 + span; base += 32) {
    bool d, e;
    classify(base + lane, d, e);
    const uint32_t eb = __ballot_sync(0xFFFFFFFFu, e);
    const bool sel = d || (e && eq_seen + static_cast<uint32_t>(__popc(eb & lt)) < need_eq);
    const uint32_t sb = __ballot_sync(0xFFFFFFFFu, sel);
    if (sel) {
      const uint32_t at = pos + static_cast<uint32_t>(__popc(sb & lt));
      if (at < static_cast<uint32_t>(kmax)) out[at] = b0 + base + lane;
    }
    pos += static_cast<uint32_t>(__popc(sb));
    eq_seen += static_cast<uint32_t>(__popc(eb));
  }
  if (rank == 0) {
    for (int i = static_cast<int>(total) + tid; i < kmax; i += kSelThreads) out[i] = -1;
    if (tid == 0) cnt[u] = static_cast<int32_t>(total);
  }
  cluster_sync();  // rank 0's shared memory stays until every CTA has read it
}

}  // namespace sa
