// k_decode.cu -- split-KV sparse decode over the selected blocks.
//
// "How Much Dense Attention is Necessary?" Sec. 2.1: exact attention with the
// original q, k, v restricted to the selected support.  "Faster Than Flash"
// Sec. 3: only the selected blocks are fetched from HBM.  "Pulsar Attention"
// Phase 2: partial softmaxes over disjoint key sets are merged exactly with
// the online-softmax rule, which is how the per-CTA partials are combined.
//
// Design (HBM-bound): grid (nsplit, groups); CTA (s, g) walks its chunk of the
// group's selected-block list.  Each block's K and V tiles (Bk = 64 rows) come
// in with TMA 2-D copies into 128-byte-swizzled shared memory, double
// buffered, so one K/V read serves all G*T query rows of the group (GQA heads
// share the tile).  QK^T: one thread per key, q broadcast from shared memory.
// PV: one thread per output column.  Softmax in base 2 with q pre-scaled by
// scale*log2(e).  A second small kernel merges the nsplit partials.
#pragma once

#include "sa_ptx.cuh"

namespace sa {

constexpr int kDecThreads = 128;
constexpr int kDecBk = 64;
constexpr int kDecStages = 2;

template <typename TE, int D, int RMAX>
struct DecodeCfg {
  static constexpr int ESZ = sizeof(TE);
  static constexpr int ROWB = D * ESZ;        // bytes per key row
  static constexpr int NBOX = ROWB / 128;     // 128-byte column boxes per row
  static constexpr int EPB = 128 / ESZ;       // elements per box row
  static constexpr int EPC = 16 / ESZ;        // elements per 16-byte chunk
  static constexpr int NCH = ROWB / 16;       // 16-byte chunks per row
  static constexpr int TILEB = kDecBk * ROWB; // bytes of one K (or V) tile
  static constexpr int STAGEB = 2 * TILEB;
  static constexpr int RPT_QK = RMAX / 2;     // rows per thread in QK (2 threads per key)
  static constexpr int DSPLIT = kDecThreads / D;  // row groups in PV
  static constexpr int RPT_PV = RMAX / DSPLIT;
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int kQOff = kDecStages * STAGEB;
  static constexpr int kLgOff = kQOff + RMAX * D * 4;
  static constexpr int kPOff = kLgOff + RMAX * kDecBk * 4;
  static constexpr int kStatOff = kPOff + RMAX * kDecBk * 4;
  static constexpr int kBarOff = kStatOff + 3 * RMAX * 4;
  static constexpr int kBytes = kBarOff + kDecStages * 8 + 1024;  // + alignment slack
  static_assert(ROWB % 128 == 0, "row must be whole 128-byte boxes");
  static_assert(RMAX % 4 == 0 && RMAX >= 4, "RMAX");
};

template <typename TE>
__device__ __forceinline__ void widen16(const uint8_t* p, float* f);
template <>
__device__ __forceinline__ void widen16<float>(const uint8_t* p, float* f) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
template <>
__device__ __forceinline__ void widen16<__nv_bfloat16>(const uint8_t* p, float* f) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <typename TE>
__device__ __forceinline__ float load_elem(const uint8_t* p);
template <>
__device__ __forceinline__ float load_elem<float>(const uint8_t* p) { return *reinterpret_cast<const float*>(p); }
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const uint8_t* p) {
  return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
}

// byte offset of element (row j, column e) inside a TMA 128B-swizzled tile
template <typename Cfg>
__device__ __forceinline__ int swz_off(int j, int e) {
  const int c = e / Cfg::EPC;                 // 16-byte chunk in the row
  const int bx = c >> 3, cc = c & 7;
  return bx * (kDecBk * 128) + j * 128 + ((cc ^ (j & 7)) << 4) + (e % Cfg::EPC) * Cfg::ESZ;
}

template <typename TE, int D, int RMAX>
__global__ void __launch_bounds__(kDecThreads) decode_split_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap, const TE* __restrict__ q,
    const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt, int kmax, int T, int Hq, int Hkv, int L,
    int Ls, float qscale, int chunk, int nsplit, float* __restrict__ ws_o, float* __restrict__ ws_ml) {
  using C = DecodeCfg<TE, D, RMAX>;
  extern __shared__ __align__(1024) uint8_t smem_dec[];
  uint8_t* smem_raw = smem_dec;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* q_s = reinterpret_cast<float*>(smem + C::kQOff);
  float* lg_s = reinterpret_cast<float*>(smem + C::kLgOff);  // [RMAX][Bk] logits (base-2 units)
  float* p_s = reinterpret_cast<float*>(smem + C::kPOff);    // [Bk][RMAX] probabilities
  float* m_s = reinterpret_cast<float*>(smem + C::kStatOff);
  float* l_s = m_s + RMAX;
  float* corr_s = l_s + RMAX;
  const uint32_t bar0 = smem_u32(smem + C::kBarOff);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, g = blockIdx.y;
  const int G = Hq / Hkv, R = G * T;
  const int b = g / Hkv, kvh = g % Hkv;
  const int n = min(cnt[g], kmax);  // never read past the caller's idx row
  const int s0 = split * chunk;
  const int s1 = min(n, s0 + chunk);
  const int32_t* my_idx = idx + static_cast<size_t>(g) * kmax;

  if (tid == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
#pragma unroll
    for (int s = 0; s < kDecStages; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  for (int i = tid; i < RMAX * D; i += kDecThreads) {
    const int r = i / D, c = i % D;
    float v = 0.f;
    if (r < R) {
      const int t = r / G, hh = r % G;
      v = static_cast<float>(q[((static_cast<size_t>(b) * T + t) * Hq + kvh * G + hh) * D + c]) * qscale;
    }
    q_s[i] = v;
  }
  if (tid < RMAX) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
    corr_s[tid] = 1.f;
  }
  for (int i = tid; i < RMAX * kDecBk; i += kDecThreads) p_s[i] = 0.f;
  __syncthreads();

  auto issue = [&](int s) {  // thread 0: fetch block my_idx[s] into its stage
    const int st = (s - s0) % kDecStages;
    const uint32_t bar = bar0 + 8 * st;
    const int blk = my_idx[s];
    const int row = g * Ls + blk * kDecBk;
    uint8_t* kt = smem + st * C::STAGEB;
    mbar_arrive_expect_tx(bar, C::STAGEB);
#pragma unroll
    for (int bx = 0; bx < C::NBOX; ++bx) {
      tma_g2s_2d(smem_u32(kt + bx * kDecBk * 128), &kmap, bx * C::EPB, row, bar);
      tma_g2s_2d(smem_u32(kt + C::TILEB + bx * kDecBk * 128), &vmap, bx * C::EPB, row, bar);
    }
  };
  if (tid == 0)
    for (int s = s0; s < min(s1, s0 + kDecStages); ++s) issue(s);

  // PV ownership: column dcol, rows rsub + DSPLIT * k
  const int dcol = tid % D, rsub = tid / D;
  float acc[C::RPT_PV];
#pragma unroll
  for (int k = 0; k < C::RPT_PV; ++k) acc[k] = 0.f;

  int consumed = s0;
  bool ok = true;
  for (int s = s0; s < s1; ++s) {
    const int st = (s - s0) % kDecStages;
    const uint32_t parity = ((s - s0) / kDecStages) & 1;
    ok = mbar_wait(bar0 + 8 * st, parity);
    if (__syncthreads_or(!ok)) break;
    consumed = s + 1;
    const uint8_t* kt = smem + st * C::STAGEB;
    const uint8_t* vt = kt + C::TILEB;
    const int blk = my_idx[s];
    const int base = blk * kDecBk;
    // an out-of-range block id contributes nothing (its TMA rows read as fill)
    const int nvalid = (blk < 0 || base >= L) ? 0 : min(kDecBk, L - base);

    // ---- logits: thread (key j, row parity rh)
    {
      const int j = tid % kDecBk, rh = tid / kDecBk;
      float lg[C::RPT_QK];
#pragma unroll
      for (int k = 0; k < C::RPT_QK; ++k) lg[k] = 0.f;
#pragma unroll 4
      for (int c = 0; c < C::NCH; ++c) {
        float kf[C::EPC];
        widen16<TE>(kt + (c >> 3) * (kDecBk * 128) + j * 128 + (((c & 7) ^ (j & 7)) << 4), kf);
#pragma unroll
        for (int k = 0; k < C::RPT_QK; ++k) {
          const float* qr = q_s + (rh + 2 * k) * D + c * C::EPC;
          float a = lg[k];
#pragma unroll
          for (int e = 0; e < C::EPC; e += 4) {
            const float4 qv = *reinterpret_cast<const float4*>(qr + e);
            a = fmaf(qv.x, kf[e], a);
            a = fmaf(qv.y, kf[e + 1], a);
            a = fmaf(qv.z, kf[e + 2], a);
            a = fmaf(qv.w, kf[e + 3], a);
          }
          lg[k] = a;
        }
      }
      const int pos = base + j;
#pragma unroll
      for (int k = 0; k < C::RPT_QK; ++k) {
        const int r = rh + 2 * k;
        if (r < R) {
          const int t = r / G;
          const bool allowed = (j < nvalid) && (pos <= L - T + t);
          lg_s[r * kDecBk + j] = allowed ? lg[k] : -INFINITY;
        }
      }
    }
    __syncthreads();
    // ---- online softmax statistics: warp w owns rows w, w+4, ...
    for (int r = warp; r < R; r += kDecThreads / 32) {
      const float x0 = lg_s[r * kDecBk + lane], x1 = lg_s[r * kDecBk + lane + 32];
      float bm = fmaxf(x0, x1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, o));
      const float m_old = m_s[r];
      const float m_new = fmaxf(m_old, bm);
      const float mu = (m_new == -INFINITY) ? 0.f : m_new;
      const float p0 = exp2f(x0 - mu), p1 = exp2f(x1 - mu);
      p_s[lane * RMAX + r] = p0;
      p_s[(lane + 32) * RMAX + r] = p1;
      float ls = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, o);
      __syncwarp();
      if (lane == 0) {
        const float corr = exp2f(m_old - mu);
        corr_s[r] = corr;
        l_s[r] = l_s[r] * corr + ls;
        m_s[r] = m_new;
      }
    }
    __syncthreads();
    // ---- acc = acc * corr + P V
#pragma unroll
    for (int k = 0; k < C::RPT_PV; ++k) acc[k] *= corr_s[rsub + C::DSPLIT * k];
    for (int j = 0; j < nvalid; ++j) {
      const float v = load_elem<TE>(vt + swz_off<C>(j, dcol));
      if constexpr (C::DSPLIT == 1) {
#pragma unroll
        for (int k = 0; k < C::RPT_PV; k += 4) {
          const float4 p4 = *reinterpret_cast<const float4*>(p_s + j * RMAX + k);
          acc[k] = fmaf(p4.x, v, acc[k]);
          acc[k + 1] = fmaf(p4.y, v, acc[k + 1]);
          acc[k + 2] = fmaf(p4.z, v, acc[k + 2]);
          acc[k + 3] = fmaf(p4.w, v, acc[k + 3]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < C::RPT_PV; ++k) acc[k] = fmaf(p_s[j * RMAX + rsub + C::DSPLIT * k], v, acc[k]);
      }
    }
    __syncthreads();  // stage and p_s free
    if (tid == 0 && s + kDecStages < s1) issue(s + kDecStages);
  }
  if (!ok) {
    // a wait gave up: drain the copies still in flight (bounded) before exiting
    if (tid == 0)
      for (int s = consumed; s < min(s1, consumed + kDecStages); ++s)
        mbar_wait(bar0 + 8 * ((s - s0) % kDecStages), ((s - s0) / kDecStages) & 1);
    __syncthreads();
  }
  // ---- partials
  const size_t part = static_cast<size_t>(g) * nsplit + split;
  if (tid < RMAX) {
    ws_ml[(part * RMAX + tid) * 2 + 0] = m_s[tid];
    ws_ml[(part * RMAX + tid) * 2 + 1] = l_s[tid];
  }
#pragma unroll
  for (int k = 0; k < C::RPT_PV; ++k) ws_o[(part * RMAX + rsub + C::DSPLIT * k) * D + dcol] = acc[k];
}

// Merge the nsplit partials of each group (exact online-softmax combine).
// grid (groups), 128 threads; nsplit <= kmax <= 16384 is staged through
// shared memory in chunks of 64 splits.
template <typename TE, int D, int RMAX>
__global__ void __launch_bounds__(kDecThreads) decode_combine_kernel(const float* __restrict__ ws_o,
                                                                     const float* __restrict__ ws_ml, int nsplit,
                                                                     int T, int Hq, int Hkv, TE* __restrict__ out) {
  constexpr int CH = 64;
  __shared__ float Ms[RMAX], dens[RMAX], wgt[CH * RMAX];
  const int g = blockIdx.x;
  const int G = Hq / Hkv, R = G * T;
  const int b = g / Hkv, kvh = g % Hkv;
  const size_t base = static_cast<size_t>(g) * nsplit;
  if (threadIdx.x < R) {
    const int r = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ws_ml[((base + s) * RMAX + r) * 2]);
    const float mu = (M == -INFINITY) ? 0.f : M;
    float den = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const size_t pr = (base + s) * RMAX + r;
      den = fmaf(ws_ml[pr * 2 + 1], exp2f(ws_ml[pr * 2] - mu), den);
    }
    Ms[r] = mu;
    dens[r] = den > 0.f ? 1.f / den : 0.f;
  }
  __syncthreads();
  constexpr int DSPLIT = kDecThreads / D;
  const int dcol = threadIdx.x % D, rsub = threadIdx.x / D;
  float num[RMAX / DSPLIT];
#pragma unroll
  for (int k = 0; k < RMAX / DSPLIT; ++k) num[k] = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += CH) {
    const int ns = min(CH, nsplit - s0);
    for (int i = threadIdx.x; i < ns * R; i += kDecThreads) {
      const int s = i / R, r = i % R;
      wgt[s * RMAX + r] = exp2f(ws_ml[((base + s0 + s) * RMAX + r) * 2] - Ms[r]);
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < RMAX / DSPLIT; ++k) {
      const int r = rsub + DSPLIT * k;
      if (r < R) {
        float a = num[k];
#pragma unroll 4
        for (int s = 0; s < ns; ++s) a = fmaf(ws_o[((base + s0 + s) * RMAX + r) * D + dcol], wgt[s * RMAX + r], a);
        num[k] = a;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int k = 0; k < RMAX / DSPLIT; ++k) {
    const int r = rsub + DSPLIT * k;
    if (r < R) {
      const int t = r / G, h = kvh * G + r % G;
      out[((static_cast<size_t>(b) * T + t) * Hq + h) * D + dcol] = static_cast<TE>(num[k] * dens[r]);
    }
  }
}

}  // namespace sa
