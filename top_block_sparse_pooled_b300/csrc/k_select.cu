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
// the float32 scores (four 8-bit digit passes over a 256-bin shared-memory
// histogram), followed by an index-ordered scan that resolves ties at the
// threshold key and compacts the selection in ascending order.
#pragma once

#include "sa_ptx.cuh"

namespace sa {

constexpr int kSelThreads = 256;

constexpr int kTopkMaxN = 16384;  // candidates per selection (blocks per sequence)

struct TopkShared {
  uint32_t hist[kSelThreads / 32][256];  // per-warp digit histograms
  uint32_t tot[256];
  uint32_t warp_tot[kSelThreads / 32];
  uint32_t dsel, rem_next, cnt_dsel;
  uint32_t bits[kTopkMaxN / 32];    // selection bitmap, index order
  uint32_t eqbits[kTopkMaxN / 32];  // candidates tied with the threshold key
};

// Exclusive block-wide prefix sum of v (all kSelThreads threads); *total gets the sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, TopkShared& S, uint32_t* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) S.warp_tot[w] = inc;
  __syncthreads();
  uint32_t before = 0, all = 0;
#pragma unroll
  for (int i = 0; i < kSelThreads / 32; ++i) {
    const uint32_t x = S.warp_tot[i];
    before += (i < w) ? x : 0u;
    all += x;
  }
  __syncthreads();
  *total = all;
  return before + inc - v;
}

// Select from scores sc[0:n) (shared memory, n <= kTopkMaxN): the forced blocks
// are the first and the last (0 and n-1, one block when n == 1); the candidates
// are 1..n-2; keep min(budget, n-2) of them with the highest scores, ties to the
// lower index.  Writes idx_out[0:kmax] (ascending, -1 padded) and *cnt_out.
// All kSelThreads threads call.
//
// Exact radix select of the threshold key (4 x 8-bit digits, per-warp
// histograms), then a selection bitmap built with warp ballots (keys above the
// threshold, plus the lowest-index ties at it), compacted in index order.
__device__ void block_topk(const float* sc, int n, int budget, int kmax, int32_t* __restrict__ idx_out,
                           int32_t* __restrict__ cnt_out, TopkShared& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int last = n - 1;                      // forced local / diagonal block
  const int ncand = n > 2 ? n - 2 : 0;         // candidates 1 .. n-2
  const int take = budget <= 0 ? 0 : (budget < ncand ? budget : ncand);
  const int take_all = take == ncand ? 1 : 0;
  uint32_t thr = 0xFFFFFFFFu, need_eq = 0, cnt_eq = 0;
  if (take_all == 0 && take > 0) {
    uint32_t prefix = 0, mask = 0, remaining = static_cast<uint32_t>(take);
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < (kSelThreads / 32) * 256; i += kSelThreads) (&S.hist[0][0])[i] = 0;
      __syncthreads();
      for (int b = 1 + tid; b < last; b += kSelThreads) {
        const uint32_t key = float_key(sc[b]);
        if ((key & mask) == prefix) atomicAdd(&S.hist[warp][(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      {
        uint32_t t = 0;
#pragma unroll
        for (int w = 0; w < kSelThreads / 32; ++w) t += S.hist[w][tid];
        S.tot[tid] = t;
      }
      __syncthreads();
      if (warp == 0) {
        // lane l holds digits 255-8l .. 248-8l (descending); find the digit at
        // which the count of keys above it, plus its own, reaches `remaining`
        uint32_t c[8], s = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          c[e] = S.tot[255 - 8 * lane - e];
          s += c[e];
        }
        uint32_t inc = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
          if (lane >= o) inc += y;
        }
        uint32_t run = inc - s;  // keys in higher digits than this lane's first
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (run < remaining && remaining <= run + c[e]) {  // exactly one (lane, e) matches
            S.dsel = 255u - 8u * static_cast<uint32_t>(lane) - static_cast<uint32_t>(e);
            S.rem_next = remaining - run;
            S.cnt_dsel = c[e];
          }
          run += c[e];
        }
      }
      __syncthreads();
      prefix |= S.dsel << shift;
      mask |= 255u << shift;
      remaining = S.rem_next;
      cnt_eq = S.cnt_dsel;
      __syncthreads();  // S.dsel is rewritten by the next pass
    }
    thr = prefix;
    need_eq = remaining;  // ties at the threshold still to take (lowest indices first)
  }
  const int surplus = (cnt_eq > need_eq) ? 1 : 0;  // more ties than places: resolve by index
  const int nwords = (n + 31) >> 5;
  for (int base = 0; base < n; base += kSelThreads) {
    const int b = base + tid;
    bool sel = false, eq = false;
    if (b < n) {
      if (b == 0 || b == last || take_all != 0) {
        sel = true;
      } else if (take > 0) {
        const uint32_t key = float_key(sc[b]);
        sel = key > thr || (key == thr && surplus == 0);
        eq = surplus != 0 && key == thr;
      }
    }
    const uint32_t bs = __ballot_sync(0xFFFFFFFFu, sel);
    const uint32_t be = __ballot_sync(0xFFFFFFFFu, eq);
    const int word = (base >> 5) + warp;
    if (lane == 0 && word < nwords) {
      S.bits[word] = bs;
      S.eqbits[word] = be;
    }
  }
  __syncthreads();
  if (surplus != 0 && tid == 0) {
    uint32_t need = need_eq;
    for (int w = 0; w < nwords && need > 0; ++w) {
      uint32_t e = S.eqbits[w];
      while (e && need > 0) {
        const uint32_t lo = e & (~e + 1u);
        S.bits[w] |= lo;
        e ^= lo;
        --need;
      }
    }
  }
  __syncthreads();
  uint32_t running = 0;
  for (int wb = 0; wb < nwords; wb += kSelThreads) {
    const int w = wb + tid;
    uint32_t word = w < nwords ? S.bits[w] : 0u;
    uint32_t total;
    uint32_t pos = running + block_excl_scan(static_cast<uint32_t>(__popc(word)), S, &total);
    while (word) {
      const int bit = __ffs(word) - 1;
      if (pos < static_cast<uint32_t>(kmax)) idx_out[pos] = w * 32 + bit;
      ++pos;
      word &= word - 1u;
    }
    running += total;
  }
  for (int i = static_cast<int>(running) + tid; i < kmax; i += kSelThreads) idx_out[i] = -1;
  if (tid == 0) *cnt_out = static_cast<int32_t>(running);
}

// --------------------------------------------------------------------------
// Decode selection.  grid (CS, groups), cluster (CS, 1, 1), kSelThreads.
// Each CTA of a group's cluster scores blocks [rank*per, rank*per + per) from
// a TMA-staged, 128B-swizzled sketch tile (thread per block, q broadcast from
// shared memory); CTA rank 0 then gathers the group's scores through
// distributed shared memory and runs the top-k.
constexpr int kSelTileRows = 256;

// Shared layout (runtime): staged sketch tile | q rows | gathered scores (rank 0) | top-k scratch | mbarrier
struct SelDecodeLayout {
  int tile_bytes, q_bytes, nb;
  __host__ __device__ int q_off() const { return tile_bytes; }
  __host__ __device__ int all_off() const { return tile_bytes + q_bytes; }
  __host__ __device__ int topk_off() const { return all_off() + ((nb * 4 + 15) / 16) * 16; }
  __host__ __device__ int bar_off() const { return topk_off() + static_cast<int>(((sizeof(TopkShared) + 15) / 16) * 16); }
  __host__ __device__ int bytes() const { return bar_off() + 16 + 1024; }
};

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// grid (CS, groups), cluster (CS, 1, 1), kSelThreads threads.  CTA rank r of
// group g's cluster scores blocks [r*per, r*per + per): its sketch rows come in
// by TMA (128B-swizzled tiles of tile_rows rows), one thread per block, q rows
// broadcast from shared memory.  Each score is stored straight into CTA rank
// 0's gather array (distributed shared memory); after one cluster barrier rank
// 0 holds all nb scores and runs the top-k.
template <typename TE, int D, int RMAX>
__global__ void __launch_bounds__(kSelThreads) select_decode_kernel(
    const __grid_constant__ CUtensorMap sk_map, const TE* __restrict__ q, int T, int Hq, int Hkv, int nb,
    int nb_cap, float scale, int per, int tile_rows, int k, float* __restrict__ scores_out,
    int32_t* __restrict__ idx, int32_t* __restrict__ cnt, int kmax, int topdelta, float delta) {
  constexpr int kBoxes = D * 4 / 128;
  extern __shared__ __align__(1024) uint8_t smem_sel_dec[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_sel_dec) + 1023) & ~uintptr_t(1023));
  const SelDecodeLayout lay{kBoxes * tile_rows * 128, RMAX * D * 4, nb};
  float* q_s = reinterpret_cast<float*>(smem + lay.q_off());
  float* all = reinterpret_cast<float*>(smem + lay.all_off());
  TopkShared& S = *reinterpret_cast<TopkShared*>(smem + lay.topk_off());
  const uint32_t bar = smem_u32(smem + lay.bar_off());

  cluster_arrive_relaxed();  // paired with the wait before the first remote store
  const int tid = threadIdx.x;
  const int g = blockIdx.y;
  const uint32_t rank = cluster_ctarank();
  const int G = Hq / Hkv, R = G * T;
  const int b = g / Hkv, kvh = g % Hkv;
  const int b0 = static_cast<int>(rank) * per;
  const int b1 = min(nb, b0 + per);

  auto issue_tile = [&](int t0) {  // thread 0: the sketch rows t0 .. t0 + tile_rows - 1 of this group
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(lay.tile_bytes));
#pragma unroll
    for (int bx = 0; bx < kBoxes; ++bx)
      tma_g2s_2d(smem_u32(smem + bx * tile_rows * 128), &sk_map, bx * 32, g * nb_cap + t0, bar);
  };
  pdl_launch_dependents();
  if (tid == 0) {
    prefetch_tmap(&sk_map);
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  pdl_wait();  // the sketch and q may come from the previous kernel
  if (tid == 0 && b0 < b1) issue_tile(b0);  // the first tile's copy overlaps the q staging below
  for (int i = tid; i < RMAX * D; i += kSelThreads) {
    const int r = i / D, c = i % D;
    float v = 0.f;
    if (r < R) {
      const int t = r / G, hh = r % G;
      v = static_cast<float>(q[((static_cast<size_t>(b) * T + t) * Hq + kvh * G + hh) * D + c]) * scale;
    }
    q_s[i] = v;
  }
  __syncthreads();
  const uint32_t all0 = map_cluster(smem_u32(all), 0);  // rank 0's gather array
  bool waited = false;

  bool ok = true;
  uint32_t phase = 0;
  for (int t0 = b0; t0 < b1; t0 += tile_rows) {
    if (tid == 0 && t0 != b0) issue_tile(t0);
    ok = mbar_wait(bar, phase);
    phase ^= 1;
    if (__syncthreads_or(!ok)) break;
    const int row = t0 + tid;
    float s = -INFINITY;
    if (tid < tile_rows && row < b1) {
      float acc[RMAX];
#pragma unroll
      for (int r = 0; r < RMAX; ++r) acc[r] = 0.f;
#pragma unroll 4
      for (int c = 0; c < D / 4; ++c) {
        const int bx = c >> 3, cc = c & 7;
        const float4 kv =
            *reinterpret_cast<const float4*>(smem + bx * tile_rows * 128 + tid * 128 + ((cc ^ (tid & 7)) << 4));
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          const float4 qv = *reinterpret_cast<const float4*>(q_s + r * D + c * 4);
          acc[r] = fmaf(qv.x, kv.x, acc[r]);
          acc[r] = fmaf(qv.y, kv.y, acc[r]);
          acc[r] = fmaf(qv.z, kv.z, acc[r]);
          acc[r] = fmaf(qv.w, kv.w, acc[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
        if (r < R) s = fmaxf(s, acc[r]);
      if (scores_out) scores_out[static_cast<size_t>(g) * nb + row] = s;
    }
    if (!waited) {
      cluster_wait();  // every CTA of the cluster is running: remote stores are safe
      waited = true;
    }
    if (tid < tile_rows && row < b1) st_cluster_f32(all0 + 4u * static_cast<uint32_t>(row), s);
    __syncthreads();  // the tile buffer is refilled next iteration
  }
  if (!waited) cluster_wait();
  cluster_sync();  // all scores have landed in rank 0
  if (rank != 0) return;
  int budget = k;
  if (topdelta) {
    // top-delta ("Faster Than Flash" Sec. 2): the candidates scoring at least the
    // pseudo-maximum (over the sink and local blocks) minus delta, at most k of them
    const float thr = fmaxf(all[0], all[nb - 1]) - delta;
    int c = 0;
    for (int base = 0; base < nb; base += kSelThreads) {
      const int b = base + tid;
      c += __syncthreads_count(b >= 1 && b < nb - 1 && all[b] >= thr);
    }
    budget = min(c, k);
  }
  block_topk(all, nb, budget, kmax, idx + static_cast<size_t>(g) * kmax, cnt + g, S);
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
  uint8_t* smem_raw = smem_sel_given;
  TopkShared& S = *reinterpret_cast<TopkShared*>(smem_raw);
  float* sc = reinterpret_cast<float*>(smem_raw + ((sizeof(TopkShared) + 15) / 16) * 16);
  const int i = blockIdx.x, g = blockIdx.y, nq = gridDim.x;
  int nvalid = nb, budget = k;
  if (prefill) {
    const int last = min((i + 1) * qtile, L) - 1;
    nvalid = last / Bk + 1;
    if (frac_num > 0) budget = k + (frac_num * nvalid + frac_den - 1) / frac_den;
  }
  const size_t u = static_cast<size_t>(g) * nq + i;
  for (int bb = threadIdx.x; bb < nvalid; bb += kSelThreads) sc[bb] = scores[u * nb + bb];
  __syncthreads();
  block_topk(sc, nvalid, budget, kmax, idx + u * kmax, cnt + u, S);
}

}  // namespace sa
