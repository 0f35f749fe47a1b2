// k_seldec.cu -- sparse decode by clusters of CTAs, one (batch, kv-head) group
// per cluster, optionally with the block selection fused in front of it.
//
// "How Much Dense Attention is Necessary?" Sec. 2.1-2.2: score the blocks, keep
// the top-k, recompute exact attention with the original q, k, v on the kept
// blocks.  "Faster Than Flash" Sec. 1-3: the scan of the small block summaries
// and the reads of the selected blocks run in one pass over memory.  "Pulsar
// Attention" Phase 2: partial softmaxes over disjoint key sets merge exactly.
//
// Work split: cluster c handles groups c, c + clusters, ...; its CS CTAs split
// each group's work.  Per group:
//   S (with selection)  CTA rank r scores sketch rows [r*per, r*per + per) in
//                       64-row chunks (tensor-core product of the fp32 sketch,
//                       split into three bf16 parts, with the group's bf16 query
//                       rows; float32-level scores) and stores them into CTA
//                       rank 0's shared memory (distributed shared memory).
//   K                   rank 0 selects the top-k blocks (forced sink and local
//                       block, ties to the lower index) into its shared memory
//                       and writes idx / cnt; every CTA then reads its share of
//                       the list, the selected blocks at positions r, r + CS, ...
//                       (without selection, the share is read from idx / cnt).
//   A                   the CTA streams its blocks' K and V tiles and keeps an
//                       online softmax per query row and warp; each warp then
//                       parks its unscaled state (max, sum, output rows) in
//                       its own slot over the ring.
//   merge               output row r is merged by CTA r % CS: every CTA
//                       combines its eight warp slots per row (exact
//                       rescaling) while pushing the row into its receiver's
//                       shared memory, then arrives on the receivers'
//                       mbarriers; a receiver combines the CS partials the
//                       same way and writes the row.
//
// Roles (288 threads): warps 0-7 consumers in two quads (quad q takes the ring
// stages of sequence numbers v with v % 2 == q, so the two quads work on
// alternate blocks; the four warps of a quad split a block's 64 keys, or a
// sketch chunk's four 16-row M tiles); warp 8 is the producer: lane 0 issues
// the TMA copies (sketch chunks, then K / V tiles) into a ring of an even
// number of stages guarded by full / empty mbarriers.  The top-k runs on the
// 256 consumer threads of rank 0.
//
// Waits are bounded (sa_ptx.cuh); after a give-up the roles run out their loops
// without waiting, every thread still reaches every barrier, the producer
// drains its copies, and the kernel returns with SA_ERR_TIMEOUT recorded.
#pragma once

#include "sa_ptx.cuh"

namespace sa {

constexpr int kSdQuads = 2;
constexpr int kSdConsumers = 4 * kSdQuads;
constexpr int kSdThreads = (kSdConsumers + 1) * 32;
constexpr int kSdBk = 64;            // keys per block; sketch rows per chunk
constexpr int kSdRmax = 16;          // query rows per group (G * T)
constexpr int kSdRecvRows = 32;      // >= CS * ceil(R / CS) for CS <= 16, R <= 16

// Shared-memory layout (runtime, from a 1024-aligned base).  The ring depth (nstages) must be
// even: stage s then always carries sequence numbers of one parity, i.e. of one quad, which
// waits on its mbarrier phases in order.  A ring stage holds
// one block's K and V tiles (64 rows of 2*D bytes each, 128-byte swizzle) or one
// 64-row chunk of the fp32 sketch (4*D bytes per row, 128-byte swizzle): the
// same number of bytes.
struct SdLayout {
  int nstages, D, nb, kmax, sel;
  // After the attention, each consumer warp parks its partial rows (kSdRmax rows of D floats,
  // padded to a row stride of D + 8 words so that the warp's fragment stores hit distinct banks)
  // over the ring, which is at least that large.
  __host__ __device__ static constexpr int slot_stride(int d) { return d + 8; }
  __host__ __device__ int stage_bytes() const { return 2 * kSdBk * D * 2; }
  __host__ __device__ int ring_bytes() const {
    const int slots = kSdConsumers * kSdRmax * slot_stride(D) * 4;
    const int ring = nstages * stage_bytes();
    return ring > slots ? ring : ((slots + 1023) / 1024) * 1024;
  }
  __host__ __device__ int q_off() const { return ring_bytes(); }
  __host__ __device__ int all_off() const { return q_off() + kSdRmax * D * 2; }
  __host__ __device__ int topk_off() const { return all_off() + (sel ? ((nb * 4 + 15) / 16) * 16 : 0); }
  __host__ __device__ int sel_off() const {
    return topk_off() + (sel ? static_cast<int>(((sizeof(TopkShared) + 15) / 16) * 16) : 0);
  }
  __host__ __device__ int list_off() const { return sel_off() + ((kmax * 4 + 4 + 15) / 16) * 16; }
  __host__ __device__ int mlw_off() const { return list_off() + ((kmax * 4 + 15) / 16) * 16; }
  __host__ __device__ int red_off() const { return mlw_off() + kSdConsumers * kSdRmax * 8; }
  __host__ __device__ int misc_off() const { return red_off() + 128 * 8 * 4; }
  // partial rows pushed here by every CTA of the cluster: slot (sender, row) of D floats, then
  // the row's (max, sum) and two pad words
  __host__ __device__ int recv_off() const { return misc_off() + 16; }
  // with selection: the local block's cached rows, staged for the fused append's sketch row
  __host__ __device__ int astage_off() const { return recv_off() + kSdRecvRows * (D + 4) * 4; }
  __host__ __device__ int bar_off() const { return astage_off() + (sel ? kSdBk * D * 2 : 0); }
  __host__ __device__ int bytes() const { return bar_off() + (2 * nstages + 3) * 8 + 1024; }
};

struct SdParams {
  const __nv_bfloat16* q;  // [B, T, Hq, D]
  int32_t* idx;            // [groups, kmax]: written (with selection) or read
  int32_t* cnt;            // [groups]
  float* scores;           // optional [groups, nb] (with selection)
  __nv_bfloat16* out;      // [B, T, Hq, D]
  int kmax, k, T, Hq, Hkv, G, R, L, Ls, nb, nb_cap, groups;
  int per;      // sketch rows per CTA (a multiple of 64)
  // Cache append fused in (the decode step; with selection only, when the T new rows [pos, L)
  // lie in the local block nb - 1 and no scores are returned): k_new / v_new [B, T, Hkv, D]; one
  // CTA writes the rows into the caches and the block's new sketch row while rank 0 selects.
  // The local block is kept whatever its score, so the selection does not depend on them; the
  // CTA that attends over the block takes the new rows from k_new / v_new into its staged tile.
  const __nv_bfloat16* k_new;  // nullptr: no append
  const __nv_bfloat16* v_new;
  __nv_bfloat16* kc;  // the caches [groups, Ls, D] (written rows)
  __nv_bfloat16* vc;
  float* sketch;      // [groups, nb_cap, D] (the rewritten row)
  int pos;
  // q may be page-locked host memory mapped into the device's address space (the decode step
  // with host I/O): it is then read with plain loads only, never by a bulk copy
  int q_host;
  float scale;  // score scale (the softmax scale)
  float qscale;  // softmax scale * log2(e)
  SdLayout lay;
};

__device__ __forceinline__ void bar_named(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_f32x4(uint32_t a, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32x2(uint32_t a, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this thread's
// earlier writes (and those ordered before them) at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("fence.acq_rel.cluster;\n\tmbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t a) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

// The cache append of one group, by the 256 consumer threads of the appending CTA: the T new
// rows of K and V into the caches, then the local block's sketch row (mean of its rows
// 64*lb .. L-1; the rows before pos come from `stage`, where the producer copied them from the
// cache at the start of the group (abar completes that copy), the new ones from k_new; the same
// thread mapping and summation order as the append kernel's block_mean_rows).  red: 128 * 8
// floats of shared scratch.
template <int D>
__device__ __forceinline__ bool append_rows(const SdParams& p, int g, int b, int kvh, float* red,
                                            const uint8_t* stage, uint32_t abar, uint32_t parity) {
  const int tid = threadIdx.x;
  bool ok = mbar_wait(abar, parity);
  if (!ok) mbar_wait_drain(abar, parity);  // the copy has landed before the buffer is reused
  constexpr int CPR = D / 8;               // 16-byte chunks per row
  for (int i = tid; i < p.T * CPR; i += kSdConsumers * 32) {
    const int t = i / CPR, c = i % CPR;
    const size_t src = ((static_cast<size_t>(b) * p.T + t) * p.Hkv + kvh) * D + c * 8;
    const size_t dst = (static_cast<size_t>(g) * p.Ls + p.pos + t) * D + c * 8;
    *reinterpret_cast<uint4*>(p.kc + dst) = *reinterpret_cast<const uint4*>(p.k_new + src);
    *reinterpret_cast<uint4*>(p.vc + dst) = *reinterpret_cast<const uint4*>(p.v_new + src);
  }
  constexpr int kThr = 128;               // the append kernel's thread count
  constexpr int RSTEP = kThr / CPR;       // rows in flight per iteration
  const int lb = p.pos / kSdBk, j0 = lb * kSdBk, nrows = p.L - j0;
  if (tid < kThr) {
    const int c = tid % CPR, r0 = tid / CPR;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int r = r0; r < nrows; r += RSTEP) {
      const int j = j0 + r;
      const uint4 x = j < p.pos
                          ? *reinterpret_cast<const uint4*>(stage + (static_cast<size_t>(r) * D + c * 8) * 2)
                          : *reinterpret_cast<const uint4*>(
                                p.k_new + ((static_cast<size_t>(b) * p.T + (j - p.pos)) * p.Hkv + kvh) * D + c * 8);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[2 * e] += __uint_as_float(w[e] << 16);
        acc[2 * e + 1] += __uint_as_float(w[e] & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) red[r0 * D + c * 8 + e] = acc[e];
  }
  bar_named(1, kSdConsumers * 32);
  const float inv = 1.0f / static_cast<float>(nrows);
  for (int col = tid; col < D; col += kSdConsumers * 32) {
    float sum = 0.f;
    for (int rr = 0; rr < RSTEP; ++rr) sum += red[rr * D + col];
    p.sketch[(static_cast<size_t>(g) * p.nb_cap + lb) * D + col] = sum * inv;
  }
  fence_proxy_async_smem();          // the stage's reads before a later copy into it
  bar_named(1, kSdConsumers * 32);  // red and the stage are free again
  return ok;
}

// grid (CS, clusters), cluster (CS, 1, 1), kSdThreads threads, one CTA per SM.
template <int D, bool kSel>
__global__ void __launch_bounds__(kSdThreads, 1) seldec_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                const __grid_constant__ CUtensorMap vmap,
                                                                const __grid_constant__ CUtensorMap skmap,
                                                                const SdParams p) {
  using C = DmCfg<D>;
  constexpr int kBoxes = D * 4 / 128;  // 128-byte boxes per fp32 sketch row
  constexpr uint32_t kStageBytes = 2 * kSdBk * D * 2;
  extern __shared__ __align__(1024) uint8_t smem_sd[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_sd) + 1023) & ~uintptr_t(1023));
  const SdLayout& lay = p.lay;
  const int NS = lay.nstages;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_sh = sbase + lay.q_off();
  const uint32_t all = sbase + lay.all_off();
  const uint32_t topk_s = sbase + lay.topk_off();
  const uint32_t sel_sh = sbase + lay.sel_off();  // rank 0: [kmax] selection, then its count
  int32_t* sel_ptr = reinterpret_cast<int32_t*>(smem + lay.sel_off());
  int32_t* list = reinterpret_cast<int32_t*>(smem + lay.list_off());  // this CTA's blocks (-1: skip)
  float* mlw = reinterpret_cast<float*>(smem + lay.mlw_off());        // [warp][row] (max, sum)
  float* red = reinterpret_cast<float*>(smem + lay.red_off());        // the append's sketch scratch
  int* misc = reinterpret_cast<int*>(smem + lay.misc_off());          // [0]: entries in list
  const uint32_t full0 = sbase + lay.bar_off();
  const uint32_t empty0 = full0 + 8 * NS;
  const uint32_t qbar = empty0 + 8 * NS;
  const uint32_t recvbar = qbar + 8;  // CS arrivals per group: every CTA has pushed its rows
  const uint32_t abar = recvbar + 8;  // the fused append's staged rows
  const uint8_t* astage = smem + lay.astage_off();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int CS = gridDim.x;

  cluster_arrive_relaxed();  // paired with the wait below: every CTA runs before any remote access
  pdl_launch_dependents();
  if (tid == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    if (kSel) prefetch_tmap(&skmap);
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 4);  // the four warps of the quad that owns the stage
    }
    mbar_init(qbar, 1);
    mbar_init(recvbar, CS);
    mbar_init(abar, 1);
    fence_mbar_init();
  }
  pdl_wait();  // q, the sketch, the caches and idx / cnt may come from the previous kernel
  __syncthreads();
  cluster_wait();

  const uint32_t all0 = map_cluster(all, 0);
  const uint32_t sel0 = map_cluster(sel_sh, 0);
  uint32_t vi = 0;   // ring sequence number (same count in every role)
  int giter = 0;     // groups done by this CTA
  bool ok = true;    // no wait has given up

  for (int g = blockIdx.y; g < p.groups; g += gridDim.y, ++giter) {
    // a later group's partials may be pushed only once every CTA has merged the previous group's
    // (with selection, the barriers of the selection phase order this)
    if (!kSel && giter > 0) cluster_sync();
    const int b = g / p.Hkv, kvh = g % p.Hkv;
    const int r0s = static_cast<int>(rank) * p.per;                 // this CTA's sketch rows
    const int r1s = kSel ? min(p.nb, r0s + p.per) : 0;
    const int nch = r1s > r0s ? (r1s - r0s + kSdBk - 1) / kSdBk : 0;  // sketch chunks
    // the CTA that appends this group's new rows (while rank 0 selects)
    const bool appender = kSel && p.k_new && static_cast<int>(rank) == (CS > 1 ? 1 : 0);
    // With selection, the forced blocks are known before it: block 0 is list position 0 (rank 0)
    // and the local block nb - 1 is the last position, cnt - 1, where the top-k returns
    // cnt = forced + min(k, nb - 2) entries.  Their K / V loads are issued right after the
    // sketch chunks, so they land while the top-k runs; each owner attends over them first.
    int ne = 0;                   // forced blocks loaded early: 0, 1 or 2
    int early0 = -1, early1 = -1;  // ... in list order
    if (kSel) {
      const int cnt_sel = (p.nb >= 2 ? 2 : 1) + (p.k <= 0 ? 0 : min(p.k, max(p.nb - 2, 0)));
      const bool sink = rank == 0;
      const bool local = p.nb >= 2 && static_cast<int>(rank) == (cnt_sel - 1) % CS;
      early0 = sink ? 0 : (local ? p.nb - 1 : -1);
      early1 = (sink && local) ? p.nb - 1 : -1;
      ne = (sink ? 1 : 0) + (local ? 1 : 0);
    }
    // K and V tiles of block blk into ring stage st (producer lane)
    auto issue_kv = [&](uint32_t st, int blk) {
      const uint32_t full = full0 + 8 * st;
      mbar_arrive_expect_tx(full, kStageBytes);
      const uint32_t kt = sbase + st * kStageBytes;
      const int row = g * p.Ls + blk * kSdBk;
#pragma unroll
      for (int bx = 0; bx < C::ROWB / 128; ++bx) {
        tma_g2s_2d(kt + bx * kSdBk * 128, &kmap, bx * 64, row, full);
        tma_g2s_2d(kt + C::TILEB + bx * kSdBk * 128, &vmap, bx * 64, row, full);
      }
    };
    // ------------------------------------------------------------- phase S
    if (kSel) {
      if (warp == kSdConsumers) {
        if (lane == 0) {
          if (appender) {  // the local block's cached rows, for its new sketch row, land during scoring
            const int j0 = (p.pos / kSdBk) * kSdBk;
            const uint32_t nbytes = static_cast<uint32_t>((p.pos - j0) * D * 2);
            mbar_arrive_expect_tx(abar, nbytes);
            if (nbytes > 0)
              bulk_g2s(smem_u32(astage), p.kc + (static_cast<size_t>(g) * p.Ls + j0) * D, nbytes, abar);
          }
          if (!p.q_host) {
            mbar_arrive_expect_tx(qbar, static_cast<uint32_t>(p.R * D * 2));
            for (int t = 0; t < p.T; ++t)
              bulk_g2s(q_sh + t * p.G * D * 2, p.q + ((static_cast<size_t>(b) * p.T + t) * p.Hq + kvh * p.G) * D,
                       p.G * D * 2, qbar);
          }
          for (int c = 0; c < nch; ++c) {
            const uint32_t v = vi + c, st = v % NS;
            if (v >= static_cast<uint32_t>(NS) && ok) ok = mbar_wait(empty0 + 8 * st, ((v / NS) - 1) & 1);
            if (!ok) break;
            const uint32_t full = full0 + 8 * st;
            mbar_arrive_expect_tx(full, static_cast<uint32_t>(kBoxes * kSdBk * 128));
#pragma unroll
            for (int bx = 0; bx < kBoxes; ++bx)
              tma_g2s_2d(sbase + st * kStageBytes + bx * kSdBk * 128, &skmap, bx * 32, g * p.nb_cap + r0s + c * kSdBk,
                         full);
          }
          for (int e = 0; e < ne && ok; ++e) {  // the forced blocks, sequence numbers after the chunks
            const uint32_t v = vi + nch + e, st = v % NS;
            if (v >= static_cast<uint32_t>(NS)) ok = mbar_wait(empty0 + 8 * st, ((v / NS) - 1) & 1);
            if (ok) issue_kv(st, e == 0 ? early0 : early1);
          }
        }
        __syncwarp();
      } else {
        const int quad = warp >> 2, wq = warp & 3;
        const int gq = lane >> 2, tq = lane & 3;
        if (p.q_host) {  // the group's R query rows (row t * G + head), 16 bytes per thread and load
          for (int i = tid; i < p.R * (D / 8); i += kSdConsumers * 32) {
            const int r = i / (D / 8), c = i % (D / 8);
            const uint4 x = *reinterpret_cast<const uint4*>(
                p.q + ((static_cast<size_t>(b) * p.T + r / p.G) * p.Hq + kvh * p.G + r % p.G) * D + c * 8);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(q_sh + 2u * (r * D + c * 8)), "r"(x.x),
                         "r"(x.y), "r"(x.z), "r"(x.w) : "memory");
          }
          bar_named(1, kSdConsumers * 32);
        } else if (ok) {
          ok = mbar_wait(qbar, giter & 1);
        }
        uint32_t bq[2][D / 16][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t qb = q_sh + 2u * ((nt * 8 + gq) * D + ks * 16 + 2 * tq);
            bq[nt][ks][0] = lds_u32(qb);
            bq[nt][ks][1] = lds_u32(qb + 16u);
          }
        for (int c = 0; c < nch; ++c) {
          const uint32_t v = vi + c;
          if (static_cast<int>(v & 1u) != quad) continue;
          const uint32_t st = v % NS;
          if (ok) ok = mbar_wait(full0 + 8 * st, (v / NS) & 1);
          if (ok) {
            const uint32_t tile = sbase + st * kStageBytes;
            float acc[3][2][4];
#pragma unroll
            for (int j = 0; j < 3; ++j)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) acc[j][nt][0] = acc[j][nt][1] = acc[j][nt][2] = acc[j][nt][3] = 0.f;
            const int rr0 = wq * 16 + gq, rr1 = rr0 + 8;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const int c0 = ks * 16 + 2 * tq;
              const float2 x00 = lds_f32x2(tile + sel_tile_off<D>(rr0, c0));
              const float2 x10 = lds_f32x2(tile + sel_tile_off<D>(rr1, c0));
              const float2 x01 = lds_f32x2(tile + sel_tile_off<D>(rr0, c0 + 8));
              const float2 x11 = lds_f32x2(tile + sel_tile_off<D>(rr1, c0 + 8));
              uint32_t ah[4], am[4], al[4];
              split3_bf16(x00.x, x00.y, ah[0], am[0], al[0]);
              split3_bf16(x10.x, x10.y, ah[1], am[1], al[1]);
              split3_bf16(x01.x, x01.y, ah[2], am[2], al[2]);
              split3_bf16(x11.x, x11.y, ah[3], am[3], al[3]);
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
                if (nt * 8 < p.R) {
                  sel_mma_bf16(acc[0][nt], ah, bq[nt][ks][0], bq[nt][ks][1]);
                  sel_mma_bf16(acc[1][nt], am, bq[nt][ks][0], bq[nt][ks][1]);
                  sel_mma_bf16(acc[2][nt], al, bq[nt][ks][0], bq[nt][ks][1]);
                }
              }
            }
            float s0 = -INFINITY, s1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int j = 0; j < 2; ++j)
                if (nt * 8 + 2 * tq + j < p.R) {
                  s0 = fmaxf(s0, p.scale * (acc[0][nt][j] + (acc[1][nt][j] + acc[2][nt][j])));
                  s1 = fmaxf(s1, p.scale * (acc[0][nt][2 + j] + (acc[1][nt][2 + j] + acc[2][nt][2 + j])));
                }
            s0 = fmaxf(s0, __shfl_xor_sync(0xFFFFFFFFu, s0, 1));
            s0 = fmaxf(s0, __shfl_xor_sync(0xFFFFFFFFu, s0, 2));
            s1 = fmaxf(s1, __shfl_xor_sync(0xFFFFFFFFu, s1, 1));
            s1 = fmaxf(s1, __shfl_xor_sync(0xFFFFFFFFu, s1, 2));
            if (tq == 0) {
              const int blk0 = r0s + c * kSdBk + rr0, blk1 = blk0 + 8;
              if (blk0 < r1s) {
                st_cluster_f32(all0 + 4u * static_cast<uint32_t>(blk0), s0);
                if (p.scores) p.scores[static_cast<size_t>(g) * p.nb + blk0] = s0;
              }
              if (blk1 < r1s) {
                st_cluster_f32(all0 + 4u * static_cast<uint32_t>(blk1), s1);
                if (p.scores) p.scores[static_cast<size_t>(g) * p.nb + blk1] = s1;
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty0 + 8 * st);
        }
      }
      vi += nch;
      cluster_sync();  // every score of the group is in rank 0
      // ----------------------------------------------------------- phase K
      if (rank == 0 && warp < kSdConsumers) {
        int32_t* cnt_sh = sel_ptr + p.kmax;
        block_topk_fast<SyncFirst256>(all, p.nb, p.k, p.kmax, sel_ptr, cnt_sh, topk_s);
        bar_named(1, kSdConsumers * 32);
        for (int i = tid; i < p.kmax; i += kSdConsumers * 32) p.idx[static_cast<size_t>(g) * p.kmax + i] = sel_ptr[i];
        if (tid == 0) p.cnt[g] = *cnt_sh;
      }
      // the fused cache append: no score the top-k reads depends on it, and the attention takes
      // the new rows from the inputs, so it runs here, off the critical path, in rank 1 (rank 0
      // after its top-k when the cluster has one CTA)
      if (appender && warp < kSdConsumers && !append_rows<D>(p, g, b, kvh, red, astage, abar, giter & 1)) ok = false;
      cluster_sync();  // the selection is in rank 0's shared memory
    }
    // --------------------------------------------------- this CTA's block list
    if (warp < kSdConsumers) {
      int n;
      if (kSel) {
        n = ld_cluster_s32(sel0 + 4u * p.kmax);
      } else {
        n = p.cnt[g];
      }
      n = max(0, min(n, p.kmax));
      const int mine = n > static_cast<int>(rank) ? (n - static_cast<int>(rank) + CS - 1) / CS : 0;
      // the forced blocks loaded early lead the list (the sink is position 0 already; the local
      // block, this CTA's last position, moves up behind it)
      const bool local_early = ne > (rank == 0 ? 1 : 0);
      for (int i = tid; i < mine; i += kSdConsumers * 32) {
        const int j = static_cast<int>(rank) + i * CS;
        int blk = kSel ? ld_cluster_s32(sel0 + 4u * j) : p.idx[static_cast<size_t>(g) * p.kmax + j];
        if (blk < 0 || blk * kSdBk >= p.L) blk = -1;
        int at = i;
        if (local_early) at = (i == mine - 1) ? (rank == 0 ? 1 : 0) : ((rank == 0 && i == 0) ? 0 : i + 1);
        list[at] = blk;
      }
      if (tid == 0) misc[0] = mine;
    }
    bar_named(2, kSdThreads);  // list ready for every role
    const int nlist = misc[0];
    // ------------------------------------------------------------- phase A
    if (warp == kSdConsumers) {
      if (lane == 0) {
        uint32_t v = vi + ne;  // the forced blocks (list[0, ne)) were issued during the selection
        for (int i = ne; i < nlist; ++i) {
          const int blk = list[i];
          if (blk < 0) continue;
          const uint32_t st = v % NS;
          if (v >= static_cast<uint32_t>(NS) && ok) ok = mbar_wait(empty0 + 8 * st, ((v / NS) - 1) & 1);
          if (!ok) break;
          issue_kv(st, blk);
          ++v;
        }
        // every copy issued has landed before the ring is reused or the CTA exits
        for (uint32_t u = (v > vi + NS ? v - NS : vi); u < v; ++u) mbar_wait_drain(full0 + 8 * (u % NS), (u / NS) & 1);
      }
      __syncwarp();
      bar_named(3, kSdThreads);  // the consumers' slots (over the ring) are read
    } else {
      const int quad = warp >> 2, wq = warp & 3;
      const int gq = lane >> 2, tq = lane & 3;
      const int kb = wq * 16;  // this warp's keys within a block
      const int r0 = gq, r1 = gq + 8;
      uint32_t qa[C::KSTEPS][4];
      float o[C::NT][4];
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      int lim0 = -1, lim1 = -1;
      {
        const __nv_bfloat16* q0 = nullptr;
        const __nv_bfloat16* q1 = nullptr;
        if (r0 < p.R) {
          q0 = p.q + ((static_cast<size_t>(b) * p.T + r0 / p.G) * p.Hq + kvh * p.G + r0 % p.G) * D;
          lim0 = p.L - p.T + r0 / p.G;
        }
        if (r1 < p.R) {
          q1 = p.q + ((static_cast<size_t>(b) * p.T + r1 / p.G) * p.Hq + kvh * p.G + r1 % p.G) * D;
          lim1 = p.L - p.T + r1 / p.G;
        }
        if (kSel) {  // the rows staged in phase S (same row order), not a second read of q
#pragma unroll
          for (int kk = 0; kk < C::KSTEPS; ++kk) {
            const int col = kk * 16 + 2 * tq;
            qa[kk][0] = q0 ? lds_u32(q_sh + 2u * (r0 * D + col)) : 0u;
            qa[kk][1] = q1 ? lds_u32(q_sh + 2u * (r1 * D + col)) : 0u;
            qa[kk][2] = q0 ? lds_u32(q_sh + 2u * (r0 * D + col + 8)) : 0u;
            qa[kk][3] = q1 ? lds_u32(q_sh + 2u * (r1 * D + col + 8)) : 0u;
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < C::KSTEPS; ++kk) {
            const int col = kk * 16 + 2 * tq;
            qa[kk][0] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + col) : 0u;
            qa[kk][1] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + col) : 0u;
            qa[kk][2] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + col + 8) : 0u;
            qa[kk][3] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + col + 8) : 0u;
          }
        }
#pragma unroll
        for (int j = 0; j < C::NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
      }
      uint32_t v = vi;
      for (int i = 0; i < nlist; ++i) {
        const int blk = list[i];
        if (blk < 0) continue;
        const uint32_t st = v % NS;
        const bool mine_stage = static_cast<int>(v & 1u) == quad;
        const uint32_t par = (v / NS) & 1;
        ++v;
        if (!mine_stage) continue;
        if (ok) ok = mbar_wait(full0 + 8 * st, par);
        if (ok) {
          const uint32_t kt = sbase + st * kStageBytes;
          const uint32_t vt = kt + C::TILEB;
          if (kSel && p.k_new && blk * kSdBk + kSdBk > p.pos) {
            // the block holding the appended rows: this warp's rows among them come from the inputs
            // (the tile was copied from the cache before or while rank 0 wrote them)
            const int r0 = max(kb, p.pos - blk * kSdBk), r1 = min(kb + 16, p.L - blk * kSdBk);
            for (int e = lane; e < (r1 > r0 ? r1 - r0 : 0) * (D / 8); e += 32) {
              const int r = r0 + e / (D / 8), ch = e % (D / 8);
              const size_t src = ((static_cast<size_t>(b) * p.T + (blk * kSdBk + r - p.pos)) * p.Hkv + kvh) * D + ch * 8;
              const uint4 kx = *reinterpret_cast<const uint4*>(p.k_new + src);
              const uint4 vx = *reinterpret_cast<const uint4*>(p.v_new + src);
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(swz_chunk(kt, r, ch)), "r"(kx.x), "r"(kx.y),
                           "r"(kx.z), "r"(kx.w) : "memory");
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(swz_chunk(vt, r, ch)), "r"(vx.x), "r"(vx.y),
                           "r"(vx.z), "r"(vx.w) : "memory");
            }
            __syncwarp();
          }
          float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          {
            const int mi = lane >> 3, ri = lane & 7;
            const int key = kb + (mi >> 1) * 8 + ri;
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; ++kk) {
              uint32_t b00, b01, b10, b11;
              ldsm_x4(swz_chunk(kt, key, 2 * kk + (mi & 1)), b00, b01, b10, b11);
              mma_bf16(s[0], qa[kk], b00, b01);
              mma_bf16(s[1], qa[kk], b10, b11);
            }
          }
          const int base = blk * kSdBk + kb + 2 * tq;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const int key = base + nt * 8 + (x & 1);
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
          {
            const int mi = lane >> 3, ri = lane & 7;
            const int key = kb + (mi & 1) * 8 + ri;
#pragma unroll
            for (int jj = 0; jj < C::NT / 2; ++jj) {
              uint32_t v0, v1, v2, v3;
              ldsm_x4_t(swz_chunk(vt, key, 2 * jj + (mi >> 1)), v0, v1, v2, v3);
              mma_bf16(o[2 * jj], pa, v0, v1);
              mma_bf16(o[2 * jj + 1], pa, v2, v3);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * st);
      }
      // ---- park this warp's unscaled state (o, and the row's max and sum) in its own slot;
      // the slots overlay the ring, which every warp has finished reading after this barrier
      l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
      l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
      l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
      l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
      bar_named(1, kSdConsumers * 32);
      float* slot = reinterpret_cast<float*>(smem) + static_cast<size_t>(warp) * kSdRmax * SdLayout::slot_stride(D);
#pragma unroll
      for (int j = 0; j < C::NT; ++j) {
        const int col = j * 8 + 2 * tq;
        if (r0 < p.R) *reinterpret_cast<float2*>(slot + r0 * SdLayout::slot_stride(D) + col) = make_float2(o[j][0], o[j][1]);
        if (r1 < p.R) *reinterpret_cast<float2*>(slot + r1 * SdLayout::slot_stride(D) + col) = make_float2(o[j][2], o[j][3]);
      }
      if (tq == 0) {
        if (r0 < p.R) {
          mlw[(warp * kSdRmax + r0) * 2] = m0;
          mlw[(warp * kSdRmax + r0) * 2 + 1] = l0;
        }
        if (r1 < p.R) {
          mlw[(warp * kSdRmax + r1) * 2] = m1;
          mlw[(warp * kSdRmax + r1) * 2 + 1] = l1;
        }
      }
      bar_named(1, kSdConsumers * 32);
    }
    vi += 0;  // (sequence numbers advanced below, identically in every role)
    {
      int nv = 0;
      for (int i = 0; i < nlist; ++i) nv += list[i] >= 0 ? 1 : 0;
      vi += static_cast<uint32_t>(nv);
    }
    // ------------------------------------------------ merge across the cluster
    // Row r of the output is merged by CTA r % CS: every CTA pushes its partial rows into their
    // receivers' shared memory and arrives on the receivers' mbarriers; a receiver waits for all
    // CS pushes and combines them (exact rescaling).  Nothing reads this CTA's shared memory
    // from outside after this point, so a CTA that receives nothing may leave at once.
    if (warp < kSdConsumers) {
      const int rpr = (p.R + CS - 1) / CS;  // rows per receiver
      const uint32_t recv_a = sbase + lay.recv_off();
      const float* slots = reinterpret_cast<const float*>(smem);
      constexpr int SS = SdLayout::slot_stride(D);
      // this CTA's partial row r = the eight warp states rescaled to their common max (fixed
      // order), pushed into slot (rank, r / CS) of receiver r % CS
      for (int e = tid; e < p.R * (D / 4); e += kSdConsumers * 32) {
        const int r = e / (D / 4), c4 = e % (D / 4);
        float mw[kSdConsumers];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kSdConsumers; ++w) {
          mw[w] = mlw[(w * kSdRmax + r) * 2];
          M = fmaxf(M, mw[w]);
        }
        const float mu = (M == -INFINITY) ? 0.f : M;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kSdConsumers; ++w) {
          const float wt = exp2f(mw[w] - mu);
          const float4 x = *reinterpret_cast<const float4*>(slots + (w * kSdRmax + r) * SS + c4 * 4);
          acc.x = fmaf(x.x, wt, acc.x);
          acc.y = fmaf(x.y, wt, acc.y);
          acc.z = fmaf(x.z, wt, acc.z);
          acc.w = fmaf(x.w, wt, acc.w);
          lsum = fmaf(mlw[(w * kSdRmax + r) * 2 + 1], wt, lsum);
        }
        const uint32_t rs = static_cast<uint32_t>(static_cast<int>(rank) * rpr + r / CS);
        st_cluster_f32x4(map_cluster(recv_a + (rs * (D + 4) + c4 * 4) * 4u, r % CS), acc);
        if (c4 == 0) st_cluster_f32x2(map_cluster(recv_a + (rs * (D + 4) + D) * 4u, r % CS), M, lsum);
      }
      fence_proxy_async_smem();  // slot writes (generic proxy) before later copies into the ring
      bar_named(3, kSdThreads);  // the slots are read: the producer may refill the ring
      bar_named(1, kSdConsumers * 32);  // every push of this CTA is issued before the arrivals
      const int nrecv = min(CS, p.R);
      if (tid < nrecv) mbar_arrive_remote(map_cluster(recvbar, tid));
      if (static_cast<int>(rank) < nrecv) {
        if (ok) ok = mbar_wait(recvbar, giter & 1);
        const int mine = (p.R - static_cast<int>(rank) + CS - 1) / CS;  // rows rank, rank + CS, ...
        const float* rv = reinterpret_cast<const float*>(smem + lay.recv_off());
        for (int e = tid; e < mine * (D / 4); e += kSdConsumers * 32) {
          const int j = e / (D / 4), dd = (e % (D / 4)) * 4;
          const int r = static_cast<int>(rank) + j * CS;
          float M = -INFINITY;
          for (int k2 = 0; k2 < CS; ++k2) M = fmaxf(M, rv[(k2 * rpr + j) * (D + 4) + D]);
          const float mu = (M == -INFINITY) ? 0.f : M;
          float den = 0.f;
          float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int k2 = 0; k2 < CS; ++k2) {
            const float* row = rv + (k2 * rpr + j) * (D + 4);
            const float w = exp2f(row[D] - mu);
            const float4 ok4 = *reinterpret_cast<const float4*>(row + dd);
            den = fmaf(row[D + 1], w, den);
            num.x = fmaf(ok4.x, w, num.x);
            num.y = fmaf(ok4.y, w, num.y);
            num.z = fmaf(ok4.z, w, num.z);
            num.w = fmaf(ok4.w, w, num.w);
          }
          const float inv = den > 0.f ? 1.f / den : 0.f;
          const int t = r / p.G, h = kvh * p.G + r % p.G;
          uint2 pk;
          pk.x = pack_bf16(num.x * inv, num.y * inv);
          pk.y = pack_bf16(num.z * inv, num.w * inv);
          *reinterpret_cast<uint2*>(p.out + ((static_cast<size_t>(b) * p.T + t) * p.Hq + h) * D + dd) = pk;
        }
      }
    }
  }
}

}  // namespace sa
