// k_decode_mma.cu -- bf16 sparse decode over the selected blocks, tensor-core
// tile math, HBM-streaming design.
//
// "How Much Dense Attention is Necessary?" Sec. 2.1: exact attention with the
// original q, k, v on the selected support only.  "Faster Than Flash" Sec. 3:
// only the selected blocks are read from HBM.  "Pulsar Attention" Phase 2:
// partial softmaxes over disjoint key sets merge exactly (online softmax).
//
// Work split: the (group, selected-block) units of all groups are laid end to
// end and cut into equal contiguous ranges, one per CTA (one CTA per SM, a
// four-stage K/V ring), so every SM streams the same number of blocks whatever
// the group count.  (Measured on the B300: one SM sustains only ~45 GB/s of
// these copies, so all SMs must stream; a smaller first burst of requests
// evens out how soon the CTAs are served.)  A CTA whose range spans several groups emits one partial per group;
// the partial of (CTA c, group g) is stored at slot c + g (the pieces of two
// interleaved partitions of a line, counted in order).  The CTA that brings a
// group's arrival counter to its CTA count merges that group's partials and
// writes the output, so the whole decode is one launch.
//
// Per CTA: warp 4 is the TMA producer (K and V tiles of a block, 64 rows each,
// 128B-swizzled, into a ring of stages guarded by full/empty mbarriers);
// warps 0-3 each own 16 of the block's 64 keys and keep their own online
// softmax state for the group's G*T (<= 16) query rows, so consumers never
// synchronize per block.  QK^T and PV use mma.m16n8k16 (bf16 in, fp32
// accumulate) with ldmatrix straight from the swizzled tiles; P stays in
// registers (the QK accumulator fragment is the PV A fragment).  At the end of
// a group's range the four warp states merge through shared memory.
//
// Token mode (kTok): the support is a list of single tokens per batch row,
// shared by every kv head of that row ("How Much Dense Attention is
// Necessary?" Sec. 2.2: one head-collapsed distribution selects the tokens
// for all heads).  A unit is (group, chunk of 64 selected tokens); the
// producer warp gathers the chunk's K and V rows 16 bytes per lane and
// instruction (cp.async, completion counted on the stage's mbarrier) into rows
// padded to 2*D + 16 bytes (ldmatrix stays conflict-free) and records each
// row's key position for the causal mask; rows past the count repeat the sink
// token with a position that no query sees.
#pragma once

#include "sa_ptx.cuh"

#ifndef SA_DM_RAMP
#define SA_DM_RAMP 0
#endif

namespace sa {

constexpr int kDmConsumers = 4;
constexpr int kDmThreads = (kDmConsumers + 1) * 32;  // block mode: one producer warp
constexpr int kDmTokProducers = 4;                   // token mode: four gathering warps
constexpr int kDmThreadsTok = (kDmConsumers + kDmTokProducers) * 32;
constexpr int kDmBk = 64;
constexpr int kDmMaxList = 1024;
constexpr int kDmMaxParts = 64;  // partials per group (CTAs touching one group)

template <int D>
struct DmCfg {
  static constexpr int ROWB = D * 2;
  static constexpr int TILEB = kDmBk * ROWB;
  static constexpr int STAGEB = 2 * TILEB;
  static constexpr int KSTEPS = D / 16;
  static constexpr int NT = D / 8;
};

// Shared-memory layout (runtime, from a 1024-aligned base).  Block mode: each
// stage is a K and a V tile of 64 swizzled 2*D-byte rows.  Token mode: rows
// padded to 2*D + 16 bytes, then one int key position per row and stage.
struct DmLayout {
  int nstages, R, D, per, tok;
  __host__ __device__ int rowb() const { return tok ? D * 2 + 16 : D * 2; }
  __host__ __device__ int stage_bytes() const { return 2 * kDmBk * rowb(); }
  __host__ __device__ int stage_off(int s) const { return s * stage_bytes(); }
  __host__ __device__ int pos_off() const { return nstages * stage_bytes(); }
  __host__ __device__ int merge_off() const { return pos_off() + (tok ? nstages * kDmBk * 4 : 0); }
  __host__ __device__ int merge_bytes() const {
    const int warps = kDmConsumers * R * (D + 2) * 4;  // per-warp states
    const int parts = (8 + 2 * kDmMaxParts) * R * 4;  // mw, lw, then staged partial maxima / denominators
    return warps > parts ? warps : parts;
  }
  __host__ __device__ int list_off() const { return merge_off() + merge_bytes(); }
  __host__ __device__ int bar_off() const { return list_off() + ((per * 8 + 15) / 16) * 16; }
  __host__ __device__ int bytes() const { return bar_off() + 2 * nstages * 8 + 1024; }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// c += a * b, m16n8k16, bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// address of 16-byte chunk `chunk` of row `row` in a 64-row, 128B-swizzled tile
__device__ __forceinline__ uint32_t swz_chunk(uint32_t tile, int row, int chunk) {
  return tile + (chunk >> 3) * (kDmBk * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

struct DmParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;  // token mode: the caches, gathered row by row
  const __nv_bfloat16* vc;
  const int32_t* idx;
  const int32_t* cnt;
  int kmax, upg, T, Hq, Hkv, L, Ls, R;  // upg: units per group (kmax blocks, or chunks of 64 tokens)
  int qpb;  // token mode, per-query prefill: selection rows per batch row (row b' = b * qpb + t), else 0
  float qscale;
  int per, U;
  float* part_o;   // [slots][R][D] (unnormalized numerators)
  float* part_ml;  // [slots][R][2] (max in base-2 units, denominator)
  int* ctr;        // [groups] arrival counters: zero on entry, left zero on exit
  int nctas;
  __nv_bfloat16* out;
  DmLayout lay;
};

// 16-byte asynchronous copy global -> shared (L2 only), and the arrive-on that
// fires on the mbarrier when all of this thread's earlier cp.async copies have
// landed (.noinc: it is one of the barrier's expected arrivals).
__device__ __forceinline__ void dm_cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void dm_cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void dm_sts_s32(uint32_t a, int v) {
  asm volatile("st.shared.s32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ int dm_lds_s32(uint32_t a) {
  int v;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

template <int D, bool kTok>
__global__ void __launch_bounds__(kTok ? kDmThreadsTok : kDmThreads, SA_DM_CTAS_PER_SM) decode_mma_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                   const __grid_constant__ CUtensorMap vmap,
                                                                   const DmParams p) {
  using C = DmCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_dm[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dm) + 1023) & ~uintptr_t(1023));
  const DmLayout& lay = p.lay;
  const int NS = lay.nstages;
  int2* list = reinterpret_cast<int2*>(smem + lay.list_off());
  float* mw = reinterpret_cast<float*>(smem + lay.merge_off());  // [4][R]
  float* lw = mw + kDmConsumers * p.R;                            // [4][R]
  float* ow = lw + kDmConsumers * p.R;                            // [4][R][D]
  const uint32_t full0 = smem_u32(smem + lay.bar_off());
  const uint32_t empty0 = full0 + 8 * NS;
  const uint32_t sbase = smem_u32(smem);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x;
  const int u0 = c * p.per;
  const int nu = min(p.per, p.U - u0);
  const int G = p.Hq / p.Hkv;

  pdl_launch_dependents();
  if (tid == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    for (int s = 0; s < NS; ++s) {
      // token mode: per gathering warp 32 copy arrivals + its own
      mbar_init(full0 + 8 * s, kTok ? kDmTokProducers * 33 : 1);
      mbar_init(empty0 + 8 * s, kDmConsumers);
    }
    fence_mbar_init();
  }
  pdl_wait();  // idx / cnt come from the selection kernel
  // unit list: (group, block id -- token mode: chunk -- or -1 when the unit is
  // past the count); the count and the id are loaded together (the id slot is
  // always in bounds)
  for (int i = tid; i < nu; i += (kTok ? kDmThreadsTok : kDmThreads)) {
    const int u = u0 + i;
    const int g = u / p.upg, s = u % p.upg;
    if constexpr (kTok) {
      const int n = min(p.cnt[g / p.Hkv], p.kmax);
      list[i] = make_int2(g, s * kDmBk < n ? s : -1);
    } else {
      const int n = p.cnt[g];
      int blk = p.idx[static_cast<size_t>(g) * p.kmax + s];
      if (s >= min(n, p.kmax) || blk < 0 || blk * kDmBk >= p.L) blk = -1;
      list[i] = make_int2(g, blk);
    }
  }
  __syncthreads();

  if (kTok && warp >= kDmConsumers) {
    // ---------------------------------- producers, token gather: warp pw takes rows 16pw .. 16pw+15
    const int pw = warp - kDmConsumers;
    int vi = 0;
    bool ok = true;
    for (int i = 0; i < nu && ok; ++i) {
      const int2 e = list[i];
      if (e.y < 0) continue;
      const int st = vi % NS;
      if (vi >= NS) {
        bool w = true;
        if (lane == 0) w = mbar_wait(empty0 + 8 * st, ((vi / NS) - 1) & 1);
        ok = __shfl_sync(0xFFFFFFFFu, w ? 1 : 0, 0) != 0;
      }
      if (!ok) break;
      const uint32_t full = full0 + 8 * st;
      const int b = e.x / p.Hkv;
      const int n = min(p.cnt[b], p.kmax);
      const int32_t* sel = p.idx + static_cast<size_t>(b) * p.kmax;
      const uint32_t kt = sbase + lay.stage_off(st), vt = kt + kDmBk * lay.rowb();
      const uint32_t pos = sbase + lay.pos_off() + st * kDmBk * 4;
      // the group's cache: per-query prefill rows b' = b * qpb + t read batch row b's
      const size_t kvg = p.qpb ? static_cast<size_t>(b / p.qpb) * p.Hkv + e.x % p.Hkv : static_cast<size_t>(e.x);
      const __nv_bfloat16* kg = p.kc + kvg * p.Ls * D;
      const __nv_bfloat16* vg = p.vc + kvg * p.Ls * D;
      int tk = 0;
      if (lane < 16) {
        const int row = 16 * pw + lane, s = e.y * kDmBk + row;
        const int t = s < n ? sel[s] : -1;
        const bool valid = t >= 0 && t < p.L;
        dm_sts_s32(pos + 4 * row, valid ? t : 0x7FFFFFFF);
        tk = valid ? t : 0;  // filler rows repeat token 0 (finite values, never visible)
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(full);  // releases the key positions written above
      // 16-byte pieces: D/8 per row, this warp's 16 K rows then its 16 V rows; lane-strided
      constexpr int kPpr = D / 8;
#pragma unroll 4
      for (int pc = lane; pc < 32 * kPpr; pc += 32) {
        const int rr = pc / kPpr, col = pc % kPpr, r16 = rr & 15;
        const int t = __shfl_sync(0xFFFFFFFFu, tk, r16);  // row r16's token is held by lane r16
        const __nv_bfloat16* src = (rr < 16 ? kg : vg) + static_cast<size_t>(t) * D + col * 8;
        dm_cp_async16((rr < 16 ? kt : vt) + (16 * pw + r16) * lay.rowb() + col * 16, src);
      }
      dm_cp_async_arrive(full);
      ++vi;
    }
    if (lane == 0)
      for (int k = max(0, vi - NS); k < vi; ++k) mbar_wait_drain(full0 + 8 * (k % NS), (k / NS) & 1);
    return;
  }
  if (!kTok && warp == kDmConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int vi = 0;
      bool ok = true;
      for (int i = 0; i < nu && ok; ++i) {
        const int2 e = list[i];
        if (e.y < 0) continue;
        const int st = vi % NS;
        if (vi >= NS) ok = mbar_wait(empty0 + 8 * st, ((vi / NS) - 1) & 1);
        if (!ok) break;
        const uint32_t full = full0 + 8 * st;
        mbar_arrive_expect_tx(full, C::STAGEB);
        const uint32_t kt = sbase + lay.stage_off(st);
        const int row = e.x * p.Ls + e.y * kDmBk;
#pragma unroll
        for (int bx = 0; bx < C::ROWB / 128; ++bx) {
          tma_g2s_2d(kt + bx * kDmBk * 128, &kmap, bx * 64, row, full);
          tma_g2s_2d(kt + C::TILEB + bx * kDmBk * 128, &vmap, bx * 64, row, full);
        }
        ++vi;
#if SA_DM_RAMP
        // ramp: request the rest of the ring once the first tile has landed, so the
        // grid's first burst of requests is one tile per CTA
        if (vi == 1 && ok) ok = mbar_wait(full0, 0);
#endif
      }
      // never leave with copies in flight: wait for the last fill of every used stage
      for (int k = max(0, vi - NS); k < vi; ++k) mbar_wait_drain(full0 + 8 * (k % NS), (k / NS) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates
  const int kb = warp * 16;                  // this warp's keys within the block
  uint32_t qa[C::KSTEPS][4];
  float o[C::NT][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  int lim0 = -1, lim1 = -1;  // last visible key position of rows gq and gq + 8 (-1: no row)
  bool dead = false;

  auto start_group = [&](int g) {
    const int b = g / p.Hkv, kvh = g % p.Hkv;
    const int r0 = gq, r1 = gq + 8;
    const __nv_bfloat16* q0 = nullptr;
    const __nv_bfloat16* q1 = nullptr;
    lim0 = lim1 = -1;
    if (r0 < p.R) {
      q0 = p.q + ((static_cast<size_t>(b) * p.T + r0 / G) * p.Hq + kvh * G + r0 % G) * D;
      lim0 = p.qpb ? b % p.qpb : p.L - p.T + r0 / G;  // per-query prefill: query t = b' % qpb sees keys <= t
    }
    if (r1 < p.R) {
      q1 = p.q + ((static_cast<size_t>(b) * p.T + r1 / G) * p.Hq + kvh * G + r1 % G) * D;
      lim1 = p.qpb ? b % p.qpb : p.L - p.T + r1 / G;
    }
#pragma unroll
    for (int kk = 0; kk < C::KSTEPS; ++kk) {
      const int col = kk * 16 + 2 * tq;
      qa[kk][0] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + col) : 0u;
      qa[kk][1] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + col) : 0u;
      qa[kk][2] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + col + 8) : 0u;
      qa[kk][3] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + col + 8) : 0u;
    }
#pragma unroll
    for (int j = 0; j < C::NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  };

  auto finish_group = [&](int g) {
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
    const int r0 = gq, r1 = gq + 8;
    if (tq == 0) {
      if (r0 < p.R) {
        mw[warp * p.R + r0] = m0;
        lw[warp * p.R + r0] = l0;
      }
      if (r1 < p.R) {
        mw[warp * p.R + r1] = m1;
        lw[warp * p.R + r1] = l1;
      }
    }
#pragma unroll
    for (int j = 0; j < C::NT; ++j) {
      const int col = j * 8 + 2 * tq;
      if (r0 < p.R) *reinterpret_cast<float2*>(ow + (warp * p.R + r0) * D + col) = make_float2(o[j][0], o[j][1]);
      if (r1 < p.R) *reinterpret_cast<float2*>(ow + (warp * p.R + r1) * D + col) = make_float2(o[j][2], o[j][3]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDmConsumers * 32) : "memory");
    const size_t slot = static_cast<size_t>(c) + g;
    if (tid < p.R) {  // row tid: the four warps' weights (into mw), the partial's max and sum
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDmConsumers; ++w) M = fmaxf(M, mw[w * p.R + tid]);
      const float mu = (M == -INFINITY) ? 0.f : M;
      float den = 0.f;
#pragma unroll
      for (int w = 0; w < kDmConsumers; ++w) {
        const float wt = exp2f(mw[w * p.R + tid] - mu);
        den = fmaf(lw[w * p.R + tid], wt, den);
        mw[w * p.R + tid] = wt;
      }
      p.part_ml[(slot * p.R + tid) * 2] = M;
      p.part_ml[(slot * p.R + tid) * 2 + 1] = den;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDmConsumers * 32) : "memory");
    for (int i = tid; i < p.R * D / 4; i += kDmConsumers * 32) {
      const int r = i / (D / 4), d4 = i % (D / 4);
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kDmConsumers; ++w) {
        const float wt = mw[w * p.R + r];
        const float4 x = reinterpret_cast<const float4*>(ow + (w * p.R + r) * D)[d4];
        num.x = fmaf(x.x, wt, num.x);
        num.y = fmaf(x.y, wt, num.y);
        num.z = fmaf(x.z, wt, num.z);
        num.w = fmaf(x.w, wt, num.w);
      }
      reinterpret_cast<float4*>(p.part_o + (slot * p.R + r) * D)[d4] = num;
    }
    // The CTA that completes group g merges its partials (no waiting: the
    // others just leave).  Writers: stores, fence, count.  Last: count, fence,
    // loads from L2.
    __threadfence();
    asm volatile("bar.sync 1, %0;" ::"n"(kDmConsumers * 32) : "memory");
    const int cf = (g * p.upg) / p.per;
    const int cl = min(p.nctas - 1, ((g + 1) * p.upg - 1) / p.per);
    const int np = cl - cf + 1;
    if (tid == 0) {
      const int old = atomicAdd(p.ctr + g, 1);
      lw[0] = (old == np - 1) ? 1.f : 0.f;  // merge buffer is free here; reuse one word as the flag
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDmConsumers * 32) : "memory");
    const bool last = lw[0] != 0.f;
    asm volatile("bar.sync 1, %0;" ::"n"(kDmConsumers * 32) : "memory");
    if (last) {
      __threadfence();
      // every partial's weight per row (into pm [np][R]) and the row's 1 / denominator: eight
      // lanes per row (row tid / 8; R <= 16), lane j taking partials j, j + 8, ... (np <=
      // kDmMaxParts = 64), their (max, denominator) pairs read from L2 all at once, the row max
      // and the denominator combined across the eight lanes
      static_assert(kDmConsumers * 32 == 8 * 16 && kDmMaxParts <= 64, "eight lanes per row, eight partials each");
      float* pm = ow;
      {
        const int r = tid >> 3, j = tid & 7;
        float mk[8], lk[8];
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int k = j + 8 * q;
          mk[q] = -INFINITY;
          lk[q] = 0.f;
          if (r < p.R && k < np) {
            const float2 ml =
                __ldcg(reinterpret_cast<const float2*>(p.part_ml) + (static_cast<size_t>(cf + k) + g) * p.R + r);
            mk[q] = ml.x;
            lk[q] = ml.y;
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) M = fmaxf(M, mk[q]);
        M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, 1));
        M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, 2));
        M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, 4));
        const float mu = (M == -INFINITY) ? 0.f : M;
        float den = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int k = j + 8 * q;
          if (r < p.R && k < np) {
            const float w = exp2f(mk[q] - mu);
            pm[k * p.R + r] = w;
            den = fmaf(lk[q], w, den);
          }
        }
        den += __shfl_xor_sync(0xFFFFFFFFu, den, 1);
        den += __shfl_xor_sync(0xFFFFFFFFu, den, 2);
        den += __shfl_xor_sync(0xFFFFFFFFu, den, 4);
        if (j == 0 && r < p.R) lw[r] = den > 0.f ? 1.f / den : 0.f;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kDmConsumers * 32) : "memory");
      // out[r, d:d+4] = sum_k w[k, r] * part_o[k, r, d:d+4] / den[r]; up to 4 float4 slots per thread,
      // all of a partial's loads issued together
      const int b = g / p.Hkv, kvh = g % p.Hkv;
      const int nq4 = p.R * D / 4;
      for (int j0 = tid; j0 < nq4; j0 += 4 * kDmConsumers * 32) {
        float4 acc[4];
        int rr[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          rr[j] = (j0 + j * kDmConsumers * 32) * 4 / D;
        }
#pragma unroll 4
        for (int k = 0; k < np; ++k) {
          const size_t sl0 = (static_cast<size_t>(cf + k) + g) * p.R;
          float4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int q4 = j0 + j * kDmConsumers * 32;
            v[j] = q4 < nq4 ? __ldcg(reinterpret_cast<const float4*>(p.part_o + sl0 * D) + q4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int q4 = j0 + j * kDmConsumers * 32;
            const float w = q4 < nq4 ? pm[k * p.R + rr[j]] : 0.f;
            acc[j].x = fmaf(v[j].x, w, acc[j].x);
            acc[j].y = fmaf(v[j].y, w, acc[j].y);
            acc[j].z = fmaf(v[j].z, w, acc[j].z);
            acc[j].w = fmaf(v[j].w, w, acc[j].w);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int q4 = j0 + j * kDmConsumers * 32;
          if (q4 < nq4) {
            const int r = rr[j], dd = (q4 * 4) % D;
            const float inv = lw[r];
            const int t = r / G, h = kvh * G + r % G;
            uint2 pk;
            pk.x = pack_bf16(acc[j].x * inv, acc[j].y * inv);
            pk.y = pack_bf16(acc[j].z * inv, acc[j].w * inv);
            *reinterpret_cast<uint2*>(p.out + ((static_cast<size_t>(b) * p.T + t) * p.Hq + h) * D + dd) = pk;
          }
        }
      }
      if (tid == 0) p.ctr[g] = 0;  // ready for the next call on this workspace
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDmConsumers * 32) : "memory");
  };

  int vi = 0, cur = -1;
  for (int i = 0; i < nu; ++i) {
    const int2 e = list[i];
    if (e.x != cur) {
      if (cur >= 0) finish_group(cur);
      start_group(e.x);
      cur = e.x;
    }
    if (e.y < 0) continue;
    const int st = vi % NS;
    const uint32_t full = full0 + 8 * st;
    if (!dead) dead = !mbar_wait(full, (vi / NS) & 1);
    ++vi;
    if (dead) continue;
    const uint32_t kt = sbase + lay.stage_off(st);
    const uint32_t vt = kt + kDmBk * lay.rowb();
    // 16-byte chunk `chunk` of row `row` of a staged K or V tile
    auto chunk_addr = [&](uint32_t tile, int row, int chunk) -> uint32_t {
      if constexpr (kTok) return tile + row * (D * 2 + 16) + chunk * 16;
      else return swz_chunk(tile, row, chunk);
    };

    // S = Q K^T for this warp's 16 keys (two n-tiles of 8)
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3, ri = lane & 7;
      const int key = kb + (mi >> 1) * 8 + ri;
#pragma unroll
      for (int kk = 0; kk < C::KSTEPS; ++kk) {
        uint32_t b00, b01, b10, b11;
        ldsm_x4(chunk_addr(kt, key, 2 * kk + (mi & 1)), b00, b01, b10, b11);
        mma_bf16(s[0], qa[kk], b00, b01);
        mma_bf16(s[1], qa[kk], b10, b11);
      }
    }
    __syncwarp();
    // scale, causal / validity mask, online softmax (base 2)
    const int base = e.y * kDmBk + kb + 2 * tq;
    const uint32_t posw = sbase + lay.pos_off() + (st * kDmBk + kb + 2 * tq) * 4;  // token mode
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        int key;
        if constexpr (kTok) key = dm_lds_s32(posw + (nt * 8 + (x & 1)) * 4);
        else key = base + nt * 8 + (x & 1);
        const int lim = (x < 2) ? lim0 : lim1;
        s[nt][x] = (key <= lim) ? s[nt][x] * p.qscale : -INFINITY;
      }
    float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
    const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
    const float c0 = exp2f(m0 - mu0), c1 = exp2f(m1 - mu1);
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - mu0);
      s[nt][1] = exp2f(s[nt][1] - mu0);
      s[nt][2] = exp2f(s[nt][2] - mu1);
      s[nt][3] = exp2f(s[nt][3] - mu1);
    }
    l0 = l0 * c0 + (s[0][0] + s[0][1]) + (s[1][0] + s[1][1]);
    l1 = l1 * c1 + (s[0][2] + s[0][3]) + (s[1][2] + s[1][3]);
    uint32_t pa[4];
    pa[0] = pack_bf16(s[0][0], s[0][1]);
    pa[1] = pack_bf16(s[0][2], s[0][3]);
    pa[2] = pack_bf16(s[1][0], s[1][1]);
    pa[3] = pack_bf16(s[1][2], s[1][3]);
#pragma unroll
    for (int j = 0; j < C::NT; ++j) {
      o[j][0] *= c0;
      o[j][1] *= c0;
      o[j][2] *= c1;
      o[j][3] *= c1;
    }
    // O += P V for this warp's 16 keys
    {
      const int mi = lane >> 3, ri = lane & 7;
      const int key = kb + (mi & 1) * 8 + ri;
#pragma unroll
      for (int jj = 0; jj < C::NT / 2; ++jj) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(chunk_addr(vt, key, 2 * jj + (mi >> 1)), v0, v1, v2, v3);
        mma_bf16(o[2 * jj], pa, v0, v1);
        mma_bf16(o[2 * jj + 1], pa, v2, v3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
  }
  if (cur >= 0) finish_group(cur);
}

}  // namespace sa
