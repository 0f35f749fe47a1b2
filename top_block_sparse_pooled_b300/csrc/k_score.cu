// k_score.cu -- prefill tile scoring on the fifth-generation tensor cores.
//
// "How Much Dense Attention is Necessary?" Sec. 2.2 / "The Sparse Frontier"
// RQ2: each query tile scores every causal key block from a cheap summary,
// then keeps the top-k; here the summary is the block's mean key (the sketch)
// and the tile's score of block b is the max over the tile's rows and the
// group's heads of scale * q . sketch_b.
//
// The scores of one (group, tile i) unit form the matrix product
//   D[b, r] = sketch[b, :] . q[r, :]      b < i+1 blocks, r = (head, row)
// followed by a max over r.  It runs transposed (blocks on the MMA's M side,
// 128 per tile = TMEM lanes; query rows on N), so the max over rows is a max
// along one TMEM lane, inside one thread.
//
// Precision: q is bf16 (exact in the MMA); the fp32 sketch is split into three
// bf16 parts hi + mid + lo (each the rounded remainder of the previous), which
// carry its 24-bit significand, and the three products are accumulated in the
// fp32 TMEM accumulator.  This gives float32-level scores from kind::f16 MMAs.
//
// Work unit: (group g, chunk c of 128 query tiles, M tile m <= c of 128 key
// blocks), dealt round-robin over a persistent grid of one CTA per SM.  The
// unit splits its M tile of the sketch once and keeps the three parts in
// shared memory while the query rows of every tile of the chunk stream past:
// per tile, the group's heads are taken in pairs (N = 128 query rows each, 256
// TMEM columns per pair, two pair buffers).  Tile i needs the blocks 0..i, so
// chunk c needs M tiles 0..c; the diagonal unit (m == c) also masks the blocks
// past each tile and writes -inf for the M tiles past the chunk.
// Roles (384 threads):
//   warp 0        TMA producer: one head's 128 query rows per ring slot
//                 (3-D map: d, head, row), in the order the MMA consumes them.
//   warp 1        TMEM allocator and MMA issuer.
//   warps 4-11    convert the unit's fp32 sketch rows into the three bf16
//                 parts (128-byte-swizzled K-major tiles in shared memory);
//                 warps 4-7 also read the accumulators (thread = block lane),
//                 take the max over the tile's rows and heads and write the scores.
#pragma once

#include "sa_tc.cuh"

namespace sa {

constexpr int kScThreads = 384;
constexpr int kScQSlots = 3;
constexpr int kScTile = 128 * 128 * 2;  // one 128 x 128 bf16 operand
constexpr int kScBox = 128 * 128;       // one 64-column box of 128 rows

struct ScSmem {
  static constexpr int kA = 0;                         // [3] sketch parts hi, mid, lo
  static constexpr int kQ = kA + 3 * kScTile;          // [kScQSlots]
  static constexpr int kBar = kQ + kScQSlots * kScTile;
  static constexpr int Q_FULL = 0, Q_EMPTY = kScQSlots, A_FULL = 2 * kScQSlots, A_EMPTY = A_FULL + 1,
                       D_FULL = A_EMPTY + 1, D_FREE = D_FULL + 2, DONE = D_FREE + 2, NBARS = DONE + 1;
  static constexpr int kSlot = kBar + NBARS * 8;
  static constexpr int kBytes = kSlot + 16 + 1024;
};

struct ScParams {
  const float* sketch;  // [groups, nb_cap, 128]
  float* scores;        // [groups, nq, nb]
  int L, Hq, Hkv, G, groups, nq, nb, nb_cap, units;
  int nc;  // chunks of 128 tiles
  float scale;
};

constexpr int kScChunk = 128;  // query tiles per unit (= key blocks per M tile)

struct ScUnit {
  int g, c, m, i0, i1;  // group, chunk, M tile, tiles [i0, i1)
};

// Unit u -> (group, chunk, M tile): groups vary fastest, then the (c, m) pairs
// m <= c in the order (0,0), (1,0), (1,1), (2,0), ...
__device__ __forceinline__ ScUnit sc_unit(const ScParams& p, int u) {
  ScUnit w;
  w.g = u % p.groups;
  int r = u / p.groups, c = 0;
  while (r > c) {
    r -= c + 1;
    ++c;
  }
  w.c = c;
  w.m = r;
  w.i0 = c * kScChunk;
  w.i1 = min(p.nq, w.i0 + kScChunk);
  return w;
}

__device__ __forceinline__ uint32_t bf16_bits(float x) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

__global__ void __launch_bounds__(kScThreads, 1) score_prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                                                                      const ScParams p) {
  extern __shared__ __align__(1024) uint8_t smem_sc[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_sc) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + ScSmem::kBar;
  auto bar = [&](int slot) { return bar0 + 8u * slot; };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + ScSmem::kSlot);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nchunks = (p.G + 1) / 2;

  if (tid == 0) {
    prefetch_tmap(&qmap);
    for (int s = 0; s < kScQSlots; ++s) {
      mbar_init(bar(ScSmem::Q_FULL + s), 1);
      mbar_init(bar(ScSmem::Q_EMPTY + s), 1);
    }
    mbar_init(bar(ScSmem::A_FULL), 256);
    mbar_init(bar(ScSmem::A_EMPTY), 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(ScSmem::D_FULL + x), 1);
      mbar_init(bar(ScSmem::D_FREE + x), 128);
    }
    mbar_init(bar(ScSmem::DONE), 1);
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
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        const ScUnit w = sc_unit(p, u);
        const int b = w.g / p.Hkv, kvh = w.g % p.Hkv;
        for (int i = w.i0; i < w.i1; ++i)
          for (int h = 0; h < p.G; ++h, ++it) {
            const int s = it % kScQSlots;
            if (it >= kScQSlots && ok) ok = mbar_wait(bar(ScSmem::Q_EMPTY + s), ((it / kScQSlots) - 1) & 1);
            mbar_arrive_expect_tx(bar(ScSmem::Q_FULL + s), kScTile);
            for (int bx = 0; bx < 2; ++bx)
              tma_g2s_3d(sbase + ScSmem::kQ + s * kScTile + bx * kScBox, &qmap, bx * 64, kvh * p.G + h,
                         b * p.L + i * 128, bar(ScSmem::Q_FULL + s));
          }
      }
      for (uint32_t k = it > kScQSlots ? it - kScQSlots : 0; k < it; ++k)
        mbar_wait_drain(bar(ScSmem::Q_FULL + k % kScQSlots), (k / kScQSlots) & 1);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kId = tc::idesc_bf16(128, 128, false, false);
      uint32_t it = 0, mt = 0, dc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++mt) {
        const ScUnit w = sc_unit(p, u);
        if (ok) ok = mbar_wait(bar(ScSmem::A_FULL), mt & 1);
        tc::fence_after_sync();
        for (int i = w.i0; i < w.i1; ++i) {
          for (int c = 0; c < nchunks; ++c, ++dc) {
            const uint32_t db = dc & 1;
            if (dc >= 2 && ok) ok = mbar_wait(bar(ScSmem::D_FREE + db), ((dc >> 1) - 1) & 1);
            tc::fence_after_sync();
            for (int hh = 0; hh < 2 && 2 * c + hh < p.G; ++hh, ++it) {
              const int s = it % kScQSlots;
              if (ok) ok = mbar_wait(bar(ScSmem::Q_FULL + s), (it / kScQSlots) & 1);
              tc::fence_after_sync();
              const uint32_t qt = sbase + ScSmem::kQ + s * kScTile;
              const uint32_t d_addr = tmem + db * 256 + hh * 128;
              for (int part = 0; part < 3; ++part) {
                const uint32_t at = sbase + ScSmem::kA + part * kScTile;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const uint32_t off = (k >> 2) * kScBox + (k & 3) * 32;
                  tc::mma_ss(d_addr, tc::desc_kmajor(at + off), tc::desc_kmajor(qt + off), kId,
                             (part > 0 || k > 0) ? 1u : 0u);
                }
              }
              tc::mma_commit(bar(ScSmem::Q_EMPTY + s));
            }
            tc::mma_commit(bar(ScSmem::D_FULL + db));
          }
        }
        tc::mma_commit(bar(ScSmem::A_EMPTY));
      }
      // drain: every MMA issued has completed before TMEM is freed
      tc::mma_commit(bar(ScSmem::DONE));
      mbar_wait_drain(bar(ScSmem::DONE), 0);
    }
  } else if (warp >= 4) {
    // --------------------------------------- sketch conversion + epilogue
    const int ct = tid - 128;                // 0..255 converter thread
    const int wq = warp & 3;                 // TMEM lane quarter
    const int lrow = (wq << 5) | lane;       // block lane of this thread (epilogue warps 4-7)
    const bool epi = warp < 8;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    uint32_t mt = 0, dc = 0;
    bool ok = true;
    // this thread's 16 four-float pieces of the unit's sketch rows (blocks past the sequence read
    // as zero); the next unit's pieces are loaded while the tensor core works on the current one
    float4 cur[16];
    auto load_tile = [&](int uu) {
      const ScUnit w = sc_unit(p, uu);
#pragma unroll
      for (int it = 0; it < 16; ++it) {
        const int item = ct + it * 256;
        const int r = item >> 5, c4 = item & 31;
        const int blk = w.m * 128 + r;
        cur[it] = (blk < p.nb)
                      ? __ldg(reinterpret_cast<const float4*>(p.sketch + (static_cast<size_t>(w.g) * p.nb_cap + blk) * 128) + c4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    if (blockIdx.x < p.units) load_tile(blockIdx.x);
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++mt) {
      const ScUnit w = sc_unit(p, u);
      // ---- convert the unit's sketch rows into the three bf16 parts
      if (mt > 0 && ok) ok = mbar_wait(bar(ScSmem::A_EMPTY), (mt - 1) & 1);
#pragma unroll
      for (int it = 0; it < 16; ++it) {
        const int item = ct + it * 256;
        const int r = item >> 5, c4 = item & 31;  // row, 4-float chunk
        const float4 x = cur[it];
        const float xs[4] = {x.x, x.y, x.z, x.w};
        uint32_t part[3][2];
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          uint32_t hv[2], mv[2], lv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float v = xs[2 * e2 + e];
            const float h = __bfloat162float(__float2bfloat16_rn(v));
            const float r1 = v - h;
            const float mdl = __bfloat162float(__float2bfloat16_rn(r1));
            const float r2 = r1 - mdl;
            hv[e] = bf16_bits(h);
            mv[e] = bf16_bits(mdl);
            lv[e] = bf16_bits(r2);
          }
          part[0][e2] = hv[0] | (hv[1] << 16);
          part[1][e2] = mv[0] | (mv[1] << 16);
          part[2][e2] = lv[0] | (lv[1] << 16);
        }
        const int dcol = c4 * 4;                     // first d column of this chunk
        const int box = dcol >> 6, e64 = dcol & 63;  // 64-column box, column inside it
        const int ch = e64 >> 3;                     // 16-byte chunk in the 128-byte row
        const uint32_t off = box * kScBox + r * 128 + (((ch ^ (r & 7)) << 4) | ((e64 & 7) * 2));
#pragma unroll
        for (int pp = 0; pp < 3; ++pp)
          *reinterpret_cast<uint2*>(smem + ScSmem::kA + pp * kScTile + off) = make_uint2(part[pp][0], part[pp][1]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(ScSmem::A_FULL));
      if (u + static_cast<int>(gridDim.x) < p.units) load_tile(u + gridDim.x);
      if (!epi) continue;
      // ---- epilogue, per tile: max over the tile's rows and heads of this block lane
      const int blk = w.m * 128 + lrow;
      for (int i = w.i0; i < w.i1; ++i) {
        const int rows_valid = min(128, p.L - i * 128);  // query rows of the tile (last tile may be short)
        float mx = -INFINITY;
        for (int c = 0; c < nchunks; ++c, ++dc) {
          const uint32_t db = dc & 1;
          if (ok) ok = mbar_wait(bar(ScSmem::D_FULL + db), (dc >> 1) & 1);
          ok = __all_sync(0xFFFFFFFFu, ok);
          tc::fence_after_sync();
          const int nh = min(2, p.G - 2 * c);
          for (int hh = 0; hh < nh; ++hh)
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              float v[32];
              tc::tmem_ld32(lane_base + db * 256 + hh * 128 + q4 * 32, v);
              tc::tmem_wait_ld();
              if (rows_valid == 128) {
#pragma unroll
                for (int e = 0; e < 32; ++e) mx = fmaxf(mx, v[e]);
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) mx = (q4 * 32 + e < rows_valid) ? fmaxf(mx, v[e]) : mx;
              }
            }
          tc::fence_before_sync();
          mbar_arrive(bar(ScSmem::D_FREE + db));
        }
        float* srow = p.scores + (static_cast<size_t>(w.g) * p.nq + i) * p.nb;
        if (blk < p.nb) srow[blk] = blk <= i ? mx * p.scale : -INFINITY;
        if (w.m == w.c)  // the diagonal unit: the M tiles past the chunk are not causal for any of its tiles
          for (int bb = (w.m + 1) * 128 + lrow; bb < p.nb; bb += 128) srow[bb] = -INFINITY;
      }
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
