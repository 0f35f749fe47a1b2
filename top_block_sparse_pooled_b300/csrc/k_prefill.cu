// k_prefill.cu -- causal sparse prefill over the selected KV blocks on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// "How Much Dense Attention is Necessary?" Sec. 2.1: attention is recomputed
// exactly, with the original q, k, v, on the selected support only, the
// support being shared by a run of consecutive queries (here a 128-row query
// tile).  "The Sparse Frontier" RQ2: block-by-block selection for prefill.
//
// Work unit: (group g = (b, kv-head), query tile i, head pair).  The two heads
// of a pair share every K/V tile the CTA loads (GQA), each head being one
// 128-row M tile.  Units are ordered longest first (tile i descending: tile i
// has up to i + 1 causal blocks) and dealt to a persistent grid of one CTA per
// SM in alternating directions (snake_unit), which evens out the CTAs'
// totals.
//
// Roles (384 threads, kPfThreads; three warpgroups):
//   warp 0    TMA producer: the unit's Q tiles (3-D map: d, head, row), then
//             the K and V tiles of each selected block into 2-stage rings.
//   warp 1    TMEM allocator and MMA issuer (one thread):
//               S_t = Q_t K^T  (M=128, N=128 keys, K=d; both K-major in smem)
//               O_t += P_t V   (A = P_t from TMEM, B = V MN-major in smem)
//   warps 2-3 idle.  Warpgroup 0 (warps 0-3) hands registers to the other two:
//             launched at 168 per thread (three warps per SM sub-partition), it
//             drops to 96 and the softmax warpgroups rise to 200 (128 x 96 +
//             256 x 200 = 63,488 <= 384 x 168), so that a softmax thread holds its
//             whole S row without spilling.
//   warps 4-7, 8-11  softmax warpgroup t = 0, 1: thread r owns query row r of
//             M tile t (= TMEM lane r).  It reads its S row from TMEM, masks
//             (causal on the diagonal block, keys past L), keeps the running
//             max m and sum l (base 2), writes P = exp2(S - m) as bf16 pairs
//             over the first 64 columns of S in TMEM, and rescales its O row
//             only when the running max grows by more than 8 (so P <= 2^8; the
//             result is the same exact softmax, normalised once at the end).
//             At the end of a unit it normalises O, stores it and the lse.
// TMEM: S_0 cols 0-127, S_1 128-255, O_0 256-383, O_1 384-511.
//
// Every mbarrier wait is bounded (sa_ptx.cuh); after a give-up all later
// waits return at once, every role runs out its loops, the producer and the
// MMA issuer drain what they issued, and TMEM is freed before exit.
#pragma once

#include "sa_f32x2.cuh"
#include "sa_tc.cuh"

namespace sa {

constexpr int kPfRows = 128;            // query rows per M tile (= qtile)
constexpr int kPfKeys = 128;            // keys per KV block
constexpr int kPfTile = 128 * 128 * 2;  // bytes of one 128 x 128 bf16 operand (two 64-column boxes)
constexpr int kPfBox = 128 * 128;       // bytes of one 64-column box of 128 rows
#ifndef SA_PF_KSTAGES
#define SA_PF_KSTAGES 2
#endif
constexpr int kPfKStages = SA_PF_KSTAGES;  // K ring (K is consumed first, so it runs ahead)
constexpr int kPfVStages = 2;              // V ring
constexpr int kPfThreads = 384;  // warp 0 producer, warp 1 MMA, warps 4-11 two softmax warpgroups
constexpr int kPfRegsLow = 96;    // registers per thread of warpgroup 0 after the split
constexpr int kPfRegsHigh = 200;  // ... of the softmax warpgroups
static_assert(128 * kPfRegsLow + 256 * kPfRegsHigh <= kPfThreads * 168,
              "the register split must fit the registers the block is launched with (168 per thread)");
constexpr float kPfRescale = 8.0f;  // log2 growth of the running max that forces an O rescale

// Per-warpgroup register budget change (all four warps of the warpgroup execute it).  An
// increase waits until the registers are free, so the increases and decreases of a block must
// balance within the registers it was launched with.
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg: 24..256 in steps of 8");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg: 24..256 in steps of 8");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

struct PfSmem {
  static constexpr int kQ = 0;                         // [2] M tiles
  static constexpr int kK = kQ + 2 * kPfTile;           // [kPfKStages]
  static constexpr int kV = kK + kPfKStages * kPfTile;  // [kPfVStages]
  static constexpr int kBar = kV + kPfVStages * kPfTile;
  // mbarrier slots (8 bytes each)
  static constexpr int Q_FULL = 0, Q_EMPTY = 1, K_FULL = 2, K_EMPTY = K_FULL + kPfKStages,
                       V_FULL = K_EMPTY + kPfKStages, V_EMPTY = V_FULL + kPfVStages, S_FULL = V_EMPTY + kPfVStages,
                       P_FULL = S_FULL + 2, O_BAR = P_FULL + 2, O_FREE = O_BAR + 2, DONE = O_FREE + 2,
                       NBARS = DONE + 1;
  static constexpr int kSlot = kBar + NBARS * 8;
  static constexpr int kBytes = kSlot + 16 + 1024;  // + slack for 1024-byte alignment
};

struct PfParams {
  const int32_t* idx;  // [groups, nq, kmax] ([B, nq, kmax] in token mode)
  const int32_t* cnt;  // [groups, nq]       ([B, nq])
  int kmax;
  // Optional per-query token mask [B, L, wpr] (wpr = 4 * nb words; bit j of row (b, t): key j is
  // in query t's support): keys whose bit is clear get no weight.  The per-query token prefill
  // runs here with, per tile, the blocks that hold any of its queries' tokens.
  const uint32_t* tokmask;
  int wpr;
  int L, Hq, Hkv, G, groups, nq, nb, npairs, units;
  float qscale;  // softmax scale * log2(e)
  __nv_bfloat16* out;
  float* lse;  // optional [B, Hq, L]
};

struct PfUnit {
  int g, i, nt, b, kvh, h0, n;
  const int32_t* ids;
};

// Unit u -> (tile, group, head pair), tiles in descending order.  kTok: the block lists are per
// batch row (shared by its kv heads).
template <bool kTok>
__device__ __forceinline__ PfUnit pf_unit(const PfParams& p, int u) {
  PfUnit w;
  const int per_i = p.groups * p.npairs;
  w.i = p.nq - 1 - u / per_i;
  const int r = u % per_i;
  w.g = r / p.npairs;
  const int pair = r % p.npairs;
  w.nt = min(2, p.G - 2 * pair);
  w.b = w.g / p.Hkv;
  w.kvh = w.g % p.Hkv;
  w.h0 = w.kvh * p.G + 2 * pair;
  const size_t sel = static_cast<size_t>(kTok ? w.b : w.g) * p.nq + w.i;
  w.n = min(p.cnt[sel], p.kmax);
  w.ids = p.idx + sel * p.kmax;
  return w;
}

__device__ __forceinline__ bool pf_valid(int blk, int nb) { return blk >= 0 && blk < nb; }

// kTok: the per-query token mode (p.tokmask set), a separate instantiation so that the
// block mode keeps its registers.
template <bool kTok>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                                                                 const __grid_constant__ CUtensorMap kmap,
                                                                 const __grid_constant__ CUtensorMap vmap,
                                                                 const PfParams p) {
  extern __shared__ __align__(1024) uint8_t smem_pf[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_pf) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + PfSmem::kBar;
  auto bar = [&](int slot) { return bar0 + 8u * slot; };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + PfSmem::kSlot);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    mbar_init(bar(PfSmem::Q_FULL), 1);
    mbar_init(bar(PfSmem::Q_EMPTY), 1);
    for (int s = 0; s < kPfKStages; ++s) {
      mbar_init(bar(PfSmem::K_FULL + s), 1);
      mbar_init(bar(PfSmem::K_EMPTY + s), 1);
    }
    for (int s = 0; s < kPfVStages; ++s) {
      mbar_init(bar(PfSmem::V_FULL + s), 1);
      mbar_init(bar(PfSmem::V_EMPTY + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(PfSmem::S_FULL + t), 1);
      mbar_init(bar(PfSmem::P_FULL + t), kPfRows);
      mbar_init(bar(PfSmem::O_BAR + t), 1);
      mbar_init(bar(PfSmem::O_FREE + t), kPfRows);
    }
    mbar_init(bar(PfSmem::DONE), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tslot), 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    setmaxnreg_dec<kPfRegsLow>();
    if (lane == 0) {
      uint32_t it = 0;  // K/V ring iteration (valid blocks, across units)
      int nu = 0;       // units processed
      bool ok = true;
      for (int rnd = 0, u = snake_unit(0); u < p.units; u = snake_unit(++rnd), ++nu) {
        const PfUnit w = pf_unit<kTok>(p, u);
        if (nu > 0 && ok) ok = mbar_wait(bar(PfSmem::Q_EMPTY), (nu - 1) & 1);
        mbar_arrive_expect_tx(bar(PfSmem::Q_FULL), w.nt * kPfTile);
        for (int t = 0; t < w.nt; ++t)
          for (int bx = 0; bx < 2; ++bx)
            tma_g2s_3d(sbase + PfSmem::kQ + t * kPfTile + bx * kPfBox, &qmap, bx * 64, w.h0 + t,
                       w.b * p.L + w.i * kPfRows, bar(PfSmem::Q_FULL));
        for (int j = 0; j < w.n; ++j) {
          const int blk = w.ids[j];
          if (!pf_valid(blk, p.nb)) continue;
          const int sk = it % kPfKStages, sv = it % kPfVStages;
          const int row = w.g * p.L + blk * kPfKeys;
          if (it >= kPfKStages && ok) ok = mbar_wait(bar(PfSmem::K_EMPTY + sk), ((it / kPfKStages) - 1) & 1);
          mbar_arrive_expect_tx(bar(PfSmem::K_FULL + sk), kPfTile);
          for (int bx = 0; bx < 2; ++bx)
            tma_g2s_2d(sbase + PfSmem::kK + sk * kPfTile + bx * kPfBox, &kmap, bx * 64, row,
                       bar(PfSmem::K_FULL + sk));
          if (it >= kPfVStages && ok) ok = mbar_wait(bar(PfSmem::V_EMPTY + sv), ((it / kPfVStages) - 1) & 1);
          mbar_arrive_expect_tx(bar(PfSmem::V_FULL + sv), kPfTile);
          for (int bx = 0; bx < 2; ++bx)
            tma_g2s_2d(sbase + PfSmem::kV + sv * kPfTile + bx * kPfBox, &vmap, bx * 64, row,
                       bar(PfSmem::V_FULL + sv));
          ++it;
        }
      }
      // never exit with copies in flight: wait for the last fill of each stage and of Q
      for (uint32_t k = it > kPfKStages ? it - kPfKStages : 0; k < it; ++k)
        mbar_wait_drain(bar(PfSmem::K_FULL + k % kPfKStages), (k / kPfKStages) & 1);
      for (uint32_t k = it > kPfVStages ? it - kPfVStages : 0; k < it; ++k)
        mbar_wait_drain(bar(PfSmem::V_FULL + k % kPfVStages), (k / kPfVStages) & 1);
      if (nu > 0) mbar_wait_drain(bar(PfSmem::Q_FULL), (nu - 1) & 1);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    setmaxnreg_dec<kPfRegsLow>();
    if (lane == 0) {
      constexpr uint32_t kIdQK = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdPV = tc::idesc_bf16(128, 128, false, true);
      uint32_t it = 0;
      int nu = 0;
      uint32_t o_commits[2] = {0, 0};  // commits to O_BAR[t]
      uint32_t p_waits[2] = {0, 0};    // completed P_FULL[t] phases consumed
      uint32_t units_t[2] = {0, 0};    // earlier units in which M tile t was active
      bool pv_pending[2] = {false, false};
      bool ok = true;
      for (int rnd = 0, u = snake_unit(0); u < p.units; u = snake_unit(++rnd), ++nu) {
        const PfUnit w = pf_unit<kTok>(p, u);
        if (ok) ok = mbar_wait(bar(PfSmem::Q_FULL), nu & 1);
        tc::fence_after_sync();
        int last_valid = w.n - 1;  // Q is released right after the S MMAs of the unit's last block
        while (last_valid >= 0 && !pf_valid(w.ids[last_valid], p.nb)) --last_valid;
        if (last_valid < 0) tc::mma_commit(bar(PfSmem::Q_EMPTY));
        int jj = 0;
        for (int j = 0; j < w.n; ++j) {
          const int blk = w.ids[j];
          if (!pf_valid(blk, p.nb)) continue;
          const int sk = it % kPfKStages, sv = it % kPfVStages;
          if (ok) ok = mbar_wait(bar(PfSmem::K_FULL + sk), (it / kPfKStages) & 1);
          tc::fence_after_sync();
          const uint32_t kst = sbase + PfSmem::kK + sk * kPfTile;
          for (int t = 0; t < w.nt; ++t) {
            if (pv_pending[t]) {  // P_t (aliasing S_t) must be consumed before S_t is rewritten
              if (ok) ok = mbar_wait(bar(PfSmem::O_BAR + t), (o_commits[t] - 1) & 1);
              tc::fence_after_sync();
              pv_pending[t] = false;
            }
            const uint32_t qt = sbase + PfSmem::kQ + t * kPfTile;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t off = (k >> 2) * kPfBox + (k & 3) * 32;
              tc::mma_ss(tmem + t * 128, tc::desc_kmajor(qt + off), tc::desc_kmajor(kst + off), kIdQK, k > 0);
            }
            tc::mma_commit(bar(PfSmem::S_FULL + t));
          }
          tc::mma_commit(bar(PfSmem::K_EMPTY + sk));
          if (j == last_valid) tc::mma_commit(bar(PfSmem::Q_EMPTY));
          if (ok) ok = mbar_wait(bar(PfSmem::V_FULL + sv), (it / kPfVStages) & 1);
          tc::fence_after_sync();
          const uint32_t vst = sbase + PfSmem::kV + sv * kPfTile;
          for (int t = 0; t < w.nt; ++t) {
            if (ok) ok = mbar_wait(bar(PfSmem::P_FULL + t), p_waits[t] & 1);
            ++p_waits[t];
            if (jj == 0 && units_t[t] > 0) {  // O_t of the previous unit has been read out
              if (ok) ok = mbar_wait(bar(PfSmem::O_FREE + t), (units_t[t] - 1) & 1);
            }
            tc::fence_after_sync();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tc::mma_ts(tmem + 256 + t * 128, tmem + t * 128 + 8 * k,
                         tc::desc_mnmajor(vst + k * 2048, kPfBox), kIdPV, (jj > 0 || k > 0) ? 1u : 0u);
            tc::mma_commit(bar(PfSmem::O_BAR + t));
            ++o_commits[t];
            pv_pending[t] = true;
          }
          tc::mma_commit(bar(PfSmem::V_EMPTY + sv));
          ++it;
          ++jj;
        }
        for (int t = 0; t < w.nt; ++t) ++units_t[t];
      }
      // drain: every MMA issued has completed before TMEM is freed
      tc::mma_commit(bar(PfSmem::DONE));
      mbar_wait_drain(bar(PfSmem::DONE), 0);
    }
  } else if (warp < 4) {
    setmaxnreg_dec<kPfRegsLow>();  // idle: its registers go to the softmax warpgroups
  } else {
    // -------------------------------------------------------------- softmax
    setmaxnreg_inc<kPfRegsHigh>();
    const int t = (warp - 4) >> 2;           // M tile of this warpgroup
    const int r = ((warp & 3) << 5) | lane;  // row within the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_addr = lane_base + t * 128;
    const uint32_t o_addr = lane_base + 256 + t * 128;
    uint32_t s_waits = 0, o_waits = 0;
    bool ok = true;
    for (int rnd = 0, u = snake_unit(0); u < p.units; u = snake_unit(++rnd)) {
      const PfUnit w = pf_unit<kTok>(p, u);
      if (t >= w.nt) continue;
      const int qpos = w.i * kPfRows + r;  // query position of this row
      float m_run = -INFINITY, l_run = 0.f;
      int jj = 0;
      for (int j = 0; j < w.n; ++j) {
        const int blk = w.ids[j];
        if (!pf_valid(blk, p.nb)) continue;
        if (ok) ok = mbar_wait(bar(PfSmem::S_FULL + t), s_waits & 1);
        ok = __all_sync(0xFFFFFFFFu, ok);  // keep the warp converged for its TMEM accesses
        ++s_waits;
        tc::fence_after_sync();
        // the whole S row in registers (one TMEM round trip), then the row max
        // over the visible keys (raw dot products; qscale > 0), four chains of
        // three-input max
        const int kbase = blk * kPfKeys;
        const bool full = kbase + kPfKeys - 1 <= qpos && kbase + kPfKeys <= p.L;
        const int lim = full ? kPfKeys - 1 : min(qpos, p.L - 1) - kbase;  // last visible key column
        uint4 tm = make_uint4(0u, 0u, 0u, 0u);  // token mask words of this row and block
        if (kTok && qpos < p.L)
          tm = __ldg(reinterpret_cast<const uint4*>(p.tokmask + (static_cast<size_t>(w.b) * p.L + qpos) * p.wpr) + blk);
        float sr[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_ld32(s_addr + 32 * c, sr + 32 * c);
        tc::tmem_wait_ld();
        if (!full) {
#pragma unroll
          for (int e = 0; e < 128; ++e) sr[e] = (e <= lim) ? sr[e] : -INFINITY;
        }
        if (kTok) {
          const uint32_t tw[4] = {tm.x, tm.y, tm.z, tm.w};
#pragma unroll
          for (int e = 0; e < 128; ++e) sr[e] = ((tw[e >> 5] >> (e & 31)) & 1u) ? sr[e] : -INFINITY;
        }
        float mx;
        {
          float m4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) m4[e] = fmaxf(sr[2 * e], sr[2 * e + 1]);
#pragma unroll
          for (int e = 8; e < 128; e += 2) m4[(e >> 1) & 3] = f2_max3(m4[(e >> 1) & 3], sr[e], sr[e + 1]);
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        mx = (mx == -INFINITY) ? -INFINITY : mx * p.qscale;
        // lazy rescale: the running max moves only when it grows by more than
        // 2^kPfRescale; P is then taken against the new max and O, l are scaled
        const bool need = mx > m_run + kPfRescale;
        const float m_new = need ? mx : m_run;
        const float corr = (need && m_run != -INFINITY) ? ex2_approx(m_run - m_new) : 1.f;
        // P = exp2(S * qscale - m) as bf16 pairs into columns 0-63 of S_t (the S
        // values are all in registers already; masked keys are -inf, giving 0)
        const float mu = (m_new == -INFINITY) ? 0.f : m_new;
        const uint64_t qs2 = f2_pack(p.qscale, p.qscale), nm2 = f2_pack(-mu, -mu);
        uint64_t ls2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(sr[32 * c + 2 * e], sr[32 * c + 2 * e + 1]), qs2, nm2), x0, x1);
            const float a0 = ex2_approx(x0), a1 = ex2_approx(x1);
            ls2[e & 1] = f2_add(ls2[e & 1], f2_pack(a0, a1));
            pk[e] = pack_bf16x2(a0, a1);
          }
          tc::tmem_st16(s_addr + 16 * c, pk);
        }
        float ls4[4];
        f2_unpack(ls2[0], ls4[0], ls4[1]);
        f2_unpack(ls2[1], ls4[2], ls4[3]);
        if (jj > 0) {  // PV_t of the previous block has completed: O_t is stable
          if (ok) ok = mbar_wait(bar(PfSmem::O_BAR + t), o_waits & 1);
          ok = __all_sync(0xFFFFFFFFu, ok);
          ++o_waits;
          tc::fence_after_sync();
          // TMEM accesses are warp-wide: a warp rescales when any of its rows needs it
          if (__any_sync(0xFFFFFFFFu, need)) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float o[32];
              tc::tmem_ld32(o_addr + 32 * c, o);
              tc::tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= corr;
              tc::tmem_st32(o_addr + 32 * c, o);
            }
          }
        }
        m_run = m_new;
        l_run = l_run * corr + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
        tc::tmem_wait_st();
        tc::fence_before_sync();
        mbar_arrive(bar(PfSmem::P_FULL + t));
        ++jj;
      }
      // ---- epilogue: O / l, lse
      if (jj > 0) {
        if (ok) ok = mbar_wait(bar(PfSmem::O_BAR + t), o_waits & 1);
        ok = __all_sync(0xFFFFFFFFu, ok);
        ++o_waits;
        tc::fence_after_sync();
      }
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const int h = w.h0 + t;
      __nv_bfloat16* dst = p.out + ((static_cast<size_t>(w.b) * p.L + qpos) * p.Hq + h) * kPfRows;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        if (jj > 0) {
          tc::tmem_ld32(o_addr + 32 * c, o);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          __nv_bfloat162 hh = __floats2bfloat162_rn(o[2 * e] * inv, o[2 * e + 1] * inv);
          pk[e] = *reinterpret_cast<uint32_t*>(&hh);
        }
        if (qpos < p.L) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            reinterpret_cast<uint4*>(dst)[4 * c + e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
      tc::fence_before_sync();
      mbar_arrive(bar(PfSmem::O_FREE + t));
      if (p.lse && qpos < p.L)
        p.lse[(static_cast<size_t>(w.b) * p.Hq + h) * p.L + qpos] =
            l_run > 0.f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
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

// Per-query token supports to the prefill kernel's form.  grid (nq, B), 256 threads; dynamic
// shared memory 8 * wpr + ceil(nb / 32) words.  For query tile i of batch row b: each query t's
// token list idx[b, t, 0:cnt[b, t]] becomes its mask row tokmask[b, t, :] (distinct tokens
// 0 <= j <= t; others ignored), and the tile's block list blist[b, i, :] (bcnt[b, i] entries,
// ascending) holds every 128-key block with a token of one of its queries.
__global__ void __launch_bounds__(256) tokprefill_prep_kernel(const int32_t* __restrict__ idx,
                                                              const int32_t* __restrict__ cnt, int kmax, int L, int nq,
                                                              int nb, int wpr, uint32_t* __restrict__ tokmask,
                                                              int32_t* __restrict__ blist, int32_t* __restrict__ bcnt) {
  extern __shared__ uint32_t tp_sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x, b = blockIdx.y;
  uint32_t* rowbm = tp_sm + warp * wpr;  // one query row per warp at a time
  uint32_t* tilebm = tp_sm + 8 * wpr;    // blocks touched by the tile
  for (int x = threadIdx.x; x < (nb + 31) / 32; x += 256) tilebm[x] = 0u;
  __syncthreads();
  for (int rl = warp; rl < kPfRows; rl += 8) {
    const int t = i * kPfRows + rl;
    if (t >= L) break;  // uniform in the warp
    for (int x = lane; x < wpr; x += 32) rowbm[x] = 0u;
    __syncwarp();
    const int n = min(cnt[static_cast<size_t>(b) * L + t], kmax);
    const int32_t* row = idx + (static_cast<size_t>(b) * L + t) * kmax;
    for (int e = lane; e < n; e += 32) {
      const int tok = row[e];
      if (tok >= 0 && tok <= t) atomicOr(rowbm + (tok >> 5), 1u << (tok & 31));
    }
    __syncwarp();
    uint32_t* dst = tokmask + (static_cast<size_t>(b) * L + t) * wpr;
    for (int x = lane; x < wpr; x += 32) {
      const uint32_t wv = rowbm[x];
      dst[x] = wv;
      if (wv) atomicOr(tilebm + ((x >> 2) >> 5), 1u << ((x >> 2) & 31));  // 4 words per block
    }
    __syncwarp();
  }
  __syncthreads();
  if (warp == 0) {
    int base = 0;
    int32_t* out = blist + (static_cast<size_t>(b) * nq + i) * nb;
    for (int j0 = 0; j0 < nb; j0 += 32) {
      const int j = j0 + lane;
      const bool in = j < nb && ((tilebm[j >> 5] >> (j & 31)) & 1u);
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, in);
      if (in) out[base + __popc(bal & ((1u << lane) - 1u))] = j;
      base += __popc(bal);
    }
    if (lane == 0) bcnt[static_cast<size_t>(b) * nq + i] = base;
  }
}

}  // namespace sa
