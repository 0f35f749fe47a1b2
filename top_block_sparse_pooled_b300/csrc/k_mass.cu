// k_mass.cu -- exact per-block attention mass (the selection oracle) on the
// fifth-generation tensor cores.
//
// "How Much Dense Attention is Necessary?" Sec. 2.1: the oracle computes each
// query's full dense attention distribution and aggregates it over the query
// heads; the support is then the top-k of that distribution.  Here, for group
// g = (b, kv-head), query tile i and key block j:
//   mass[g, i, j] = sum over the group's heads h and the tile's rows t of
//                   sum_{key k in block j, k <= t} softmax_h,t(k),
// each softmax taken over the row's whole causal range (dense, not sparse).
//
// Work unit: (group, query tile i), tiles in descending order (tile i has i+1
// causal blocks), dealt in alternating directions (snake_unit) over a
// persistent grid of one CTA per SM.  A
// unit walks the group's heads two at a time (two 128-row M tiles sharing each
// K tile) and makes two passes over its causal blocks:
//   pass 1: row log-sum-exp (online max and sum, base 2);
//   pass 2: P = exp2(S - lse) summed over the block's keys, then over the
//           warp's 32 rows (shuffle tree), then added into a per-(M tile,
//           warp, block) slot in shared memory.
// The slots are summed in a fixed order at the end of the unit, so the result
// is deterministic.
//
// Roles (384 threads): warp 0 TMA producer (Q tiles of the head pair, K tiles
// into a 3-stage ring); warp 1 TMEM allocator and MMA issuer
// (S_t = Q_t K^T into a double-buffered TMEM slot per M tile); warps 4-7 and
// 8-11 softmax warpgroups, thread r = row r of M tile t = TMEM lane r.
// TMEM: S_t[buf] at columns (2t + buf) * 128.
#pragma once

#include "sa_f32x2.cuh"
#include "sa_tc.cuh"

namespace sa {

// sum over e of 2^(s[e] * qscale - sub), keys taken in pairs
__device__ __forceinline__ float ms_exp2_sum(const float (&s)[128], float qscale, float sub) {
  const uint64_t qs2 = f2_pack(qscale, qscale), ns2 = f2_pack(-sub, -sub);
  uint64_t a2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
  for (int e = 0; e < 128; e += 2) {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(s[e], s[e + 1]), qs2, ns2), x0, x1);
    a2[(e >> 1) & 1] = f2_add(a2[(e >> 1) & 1], f2_pack(ex2_approx(x0), ex2_approx(x1)));
  }
  float c0, c1, c2, c3;
  f2_unpack(a2[0], c0, c1);
  f2_unpack(a2[1], c2, c3);
  return (c0 + c1) + (c2 + c3);
}

constexpr int kMsStages = 3;
constexpr int kMsThreads = 384;
constexpr int kMsMaxBlocks = 2048;

struct MsSmem {
  static constexpr int kQ = 0;                        // [2] M tiles, 32 KB each
  static constexpr int kK = kQ + 2 * kPfTile;         // [kMsStages]
  static constexpr int kBar = kK + kMsStages * kPfTile;
  static constexpr int Q_FULL = 0, Q_EMPTY = 1, K_FULL = 2, K_EMPTY = 2 + kMsStages, S_FULL = 2 + 2 * kMsStages,
                       S_FREE = S_FULL + 4, DONE = S_FREE + 4, NBARS = DONE + 1;
  static constexpr int kSlot = kBar + NBARS * 8;
  static constexpr int kAcc = ((kSlot + 16 + 15) / 16) * 16;  // float [2][4][nb]
  __host__ __device__ static int bytes(int nb) { return kAcc + 2 * 4 * nb * 4 + 1024; }
};

struct MsParams {
  int L, Hq, Hkv, G, groups, nq, nb, npairs, units;
  float qscale;  // softmax scale * log2(e)
  float* mass;   // [groups, nq, nb]
};

__global__ void __launch_bounds__(kMsThreads, 1) mass_kernel(const __grid_constant__ CUtensorMap qmap,
                                                             const __grid_constant__ CUtensorMap kmap,
                                                             const MsParams p) {
  extern __shared__ __align__(1024) uint8_t smem_ms[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_ms) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + MsSmem::kBar;
  auto bar = [&](int slot) { return bar0 + 8u * slot; };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + MsSmem::kSlot);
  float* acc = reinterpret_cast<float*>(smem + MsSmem::kAcc);  // [t][warp][nb]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    mbar_init(bar(MsSmem::Q_FULL), 1);
    mbar_init(bar(MsSmem::Q_EMPTY), 1);
    for (int s = 0; s < kMsStages; ++s) {
      mbar_init(bar(MsSmem::K_FULL + s), 1);
      mbar_init(bar(MsSmem::K_EMPTY + s), 1);
    }
    for (int x = 0; x < 4; ++x) {
      mbar_init(bar(MsSmem::S_FULL + x), 1);
      mbar_init(bar(MsSmem::S_FREE + x), kPfRows);
    }
    mbar_init(bar(MsSmem::DONE), 1);
    fence_mbar_init();
  }
  for (int x = tid; x < 8 * p.nb; x += kMsThreads) acc[x] = 0.f;
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tslot), 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const int per_i = p.groups;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kit = 0, qn = 0;
      bool ok = true;
      for (int rnd = 0, u = snake_unit(0); u < p.units; u = snake_unit(++rnd)) {
        const int i = p.nq - 1 - u / per_i, g = u % per_i;
        const int b = g / p.Hkv, kvh = g % p.Hkv;
        const int nc = (min((i + 1) * kPfRows, p.L) - 1) / kPfKeys + 1;  // causal blocks
        for (int pair = 0; pair < p.npairs; ++pair, ++qn) {
          const int nt = min(2, p.G - 2 * pair);
          if (qn > 0 && ok) ok = mbar_wait(bar(MsSmem::Q_EMPTY), (qn - 1) & 1);
          mbar_arrive_expect_tx(bar(MsSmem::Q_FULL), nt * kPfTile);
          for (int t = 0; t < nt; ++t)
            for (int bx = 0; bx < 2; ++bx)
              tma_g2s_3d(sbase + MsSmem::kQ + t * kPfTile + bx * kPfBox, &qmap, bx * 64, kvh * p.G + 2 * pair + t,
                         b * p.L + i * kPfRows, bar(MsSmem::Q_FULL));
          for (int pass = 0; pass < 2; ++pass)
            for (int j = 0; j < nc; ++j, ++kit) {
              const int s = kit % kMsStages;
              if (kit >= kMsStages && ok) ok = mbar_wait(bar(MsSmem::K_EMPTY + s), ((kit / kMsStages) - 1) & 1);
              mbar_arrive_expect_tx(bar(MsSmem::K_FULL + s), kPfTile);
              for (int bx = 0; bx < 2; ++bx)
                tma_g2s_2d(sbase + MsSmem::kK + s * kPfTile + bx * kPfBox, &kmap, bx * 64, g * p.L + j * kPfKeys,
                           bar(MsSmem::K_FULL + s));
            }
        }
      }
      for (uint32_t k = kit > kMsStages ? kit - kMsStages : 0; k < kit; ++k)
        mbar_wait_drain(bar(MsSmem::K_FULL + k % kMsStages), (k / kMsStages) & 1);
      if (qn > 0) mbar_wait_drain(bar(MsSmem::Q_FULL), (qn - 1) & 1);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdQK = tc::idesc_bf16(128, 128, false, false);
      uint32_t kit = 0, qn = 0;
      uint32_t sit[2] = {0, 0};
      bool ok = true;
      for (int rnd = 0, u = snake_unit(0); u < p.units; u = snake_unit(++rnd)) {
        const int i = p.nq - 1 - u / per_i;
        const int nc = (min((i + 1) * kPfRows, p.L) - 1) / kPfKeys + 1;
        for (int pair = 0; pair < p.npairs; ++pair, ++qn) {
          const int nt = min(2, p.G - 2 * pair);
          if (ok) ok = mbar_wait(bar(MsSmem::Q_FULL), qn & 1);
          tc::fence_after_sync();
          for (int pass = 0; pass < 2; ++pass)
            for (int j = 0; j < nc; ++j, ++kit) {
              const int s = kit % kMsStages;
              if (ok) ok = mbar_wait(bar(MsSmem::K_FULL + s), (kit / kMsStages) & 1);
              tc::fence_after_sync();
              const uint32_t kst = sbase + MsSmem::kK + s * kPfTile;
              for (int t = 0; t < nt; ++t) {
                const uint32_t buf = sit[t] & 1;
                if (sit[t] >= 2 && ok) ok = mbar_wait(bar(MsSmem::S_FREE + 2 * t + buf), ((sit[t] >> 1) - 1) & 1);
                tc::fence_after_sync();
                const uint32_t qt = sbase + MsSmem::kQ + t * kPfTile;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const uint32_t off = (k >> 2) * kPfBox + (k & 3) * 32;
                  tc::mma_ss(tmem + (2 * t + buf) * 128, tc::desc_kmajor(qt + off), tc::desc_kmajor(kst + off),
                             kIdQK, k > 0);
                }
                tc::mma_commit(bar(MsSmem::S_FULL + 2 * t + buf));
                ++sit[t];
              }
              tc::mma_commit(bar(MsSmem::K_EMPTY + s));
            }
          tc::mma_commit(bar(MsSmem::Q_EMPTY));
        }
      }
      tc::mma_commit(bar(MsSmem::DONE));
      mbar_wait_drain(bar(MsSmem::DONE), 0);
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;  // warp within the warpgroup = TMEM lane quarter
    const int r = (wq << 5) | lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    uint32_t sit = 0;
    bool ok = true;
    float* my_acc = acc + (t * 4 + wq) * p.nb;
    for (int rnd = 0, u = snake_unit(0); u < p.units; u = snake_unit(++rnd)) {
      const int i = p.nq - 1 - u / per_i, g = u % per_i;
      const int qpos = i * kPfRows + r;
      const bool live = qpos < p.L;
      const int nc = (min((i + 1) * kPfRows, p.L) - 1) / kPfKeys + 1;
      for (int pair = 0; pair < p.npairs; ++pair) {
        if (t >= min(2, p.G - 2 * pair)) continue;
        float m = -INFINITY, l = 0.f;  // base-2 running max and sum of the row
        float lse2 = 0.f;
        for (int pass = 0; pass < 2; ++pass) {
          if (pass == 1) lse2 = (l > 0.f) ? m + log2f(l) : INFINITY;  // INFINITY: row contributes nothing
          for (int j = 0; j < nc; ++j, ++sit) {
            const uint32_t buf = sit & 1;
            if (ok) ok = mbar_wait(bar(MsSmem::S_FULL + 2 * t + buf), (sit >> 1) & 1);
            ok = __all_sync(0xFFFFFFFFu, ok);
            tc::fence_after_sync();
            const uint32_t s_addr = lane_base + (2 * t + buf) * 128;
            const int lim = live ? qpos - j * kPfKeys : -1;  // last visible key column
            const bool full = lim >= kPfKeys - 1;            // every key of the block visible
            // the whole row of S in registers (two loads per wait), then S_t[buf] is free
            float s[128];
#pragma unroll
            for (int c = 0; c < 4; c += 2) {
              tc::tmem_ld32(s_addr + 32 * c, s + 32 * c);
              tc::tmem_ld32(s_addr + 32 * c + 32, s + 32 * c + 32);
            }
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            mbar_arrive(bar(MsSmem::S_FREE + 2 * t + buf));
            if (!full) {
#pragma unroll
              for (int e = 0; e < 128; ++e) s[e] = (e <= lim) ? s[e] : -INFINITY;
            }
            float rs = 0.f;
            if (pass == 0) {
              // online log-sum-exp (base 2): block max first, then one exp per key
              float m4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) m4[e] = -INFINITY;
#pragma unroll
              for (int e = 0; e < 128; e += 2) m4[(e >> 1) & 3] = f2_max3(m4[(e >> 1) & 3], s[e], s[e + 1]);
              float bm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
              bm = (bm == -INFINITY) ? -INFINITY : bm * p.qscale;
              const float mn = fmaxf(m, bm);
              if (mn != -INFINITY) {
                l = l * ex2_approx(m - mn) + ms_exp2_sum(s, p.qscale, mn);
                m = mn;
              }
            } else {
              rs = ms_exp2_sum(s, p.qscale, lse2);
            }
            if (pass == 1) {
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xFFFFFFFFu, rs, o);
              if (lane == 0) my_acc[j] += rs;
            }
          }
        }
      }
      // ---- end of unit: fixed-order sum of the 8 slots, write, reset
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const int st = tid - 128;
      float* dst = p.mass + (static_cast<size_t>(g) * p.nq + i) * p.nb;
      for (int jb = st; jb < p.nb; jb += 256) {
        float v = 0.f;
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          v += acc[x * p.nb + jb];
          acc[x * p.nb + jb] = 0.f;
        }
        dst[jb] = v;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace sa
