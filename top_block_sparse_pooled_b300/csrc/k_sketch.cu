// k_sketch.cu -- block sketches (mean key of each KV block) and the fused
// KV-cache append that keeps them current.
//
// "Faster Than Flash" Sec. 1: importance is estimated by scanning a small
// compressed summary of the cache instead of the keys themselves; here the
// summary of a block is the float32 mean of its key rows.  "Sparse Attention
// as a Range Searching Problem" Sec. 2: new keys join the index incrementally
// (the append rewrites only the sketches of the blocks it touches).
//
// Memory-bound: each key row is read once with 16-byte vector loads.
#pragma once

#include "sa_ptx.cuh"

namespace sa {

template <typename TE>
struct Vec16;  // 16 bytes of elements, widened to float
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const float* p, float* f) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* f) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

constexpr int kSketchThreads = 128;

// Mean of `nrows` contiguous rows of D elements starting at `rows`, written to
// out[0:D].  Called by all kSketchThreads threads of the CTA; `red` is
// kSketchThreads * 8 floats of shared scratch.
template <typename TE, int D>
__device__ __forceinline__ void block_mean_rows(const TE* __restrict__ rows, int nrows, float* __restrict__ out,
                                                float* red) {
  using V = Vec16<TE>;
  constexpr int CPR = D / V::N;                 // 16-byte chunks per row
  constexpr int RSTEP = kSketchThreads / CPR;   // rows in flight per iteration
  const int tid = threadIdx.x;
  const int c = tid % CPR, r0 = tid / CPR;
  float acc[V::N];
#pragma unroll
  for (int e = 0; e < V::N; ++e) acc[e] = 0.f;
  for (int r = r0; r < nrows; r += RSTEP) {
    float f[V::N];
    V::load(rows + static_cast<size_t>(r) * D + c * V::N, f);
#pragma unroll
    for (int e = 0; e < V::N; ++e) acc[e] += f[e];
  }
#pragma unroll
  for (int e = 0; e < V::N; ++e) red[r0 * D + c * V::N + e] = acc[e];
  __syncthreads();
  const float inv = 1.0f / static_cast<float>(nrows);
  for (int col = tid; col < D; col += kSketchThreads) {
    float s = 0.f;
    for (int rr = 0; rr < RSTEP; ++rr) s += red[rr * D + col];
    out[col] = s * inv;
  }
  __syncthreads();
}

// grid (nb, groups): one CTA per (group, block).
// The sketch's group stride is nb_cap = ceil(Ls / Bk) blocks (the cache capacity).
template <typename TE, int D>
__global__ void __launch_bounds__(kSketchThreads) build_sketch_kernel(const TE* __restrict__ k, int L, int Ls,
                                                                      int Bk, int nb_cap, float* __restrict__ sketch) {
  __shared__ __align__(16) float red[kSketchThreads * 8];
  const int blk = blockIdx.x, g = blockIdx.y;
  const int j0 = blk * Bk;
  const int j1 = min(j0 + Bk, L);
  block_mean_rows<TE, D>(k + (static_cast<size_t>(g) * Ls + j0) * D, j1 - j0,
                         sketch + (static_cast<size_t>(g) * nb_cap + blk) * D, red);
}

// grid (groups): copy T new rows of K and V into the cache, then rewrite the
// sketch of each block the new rows touch (mean over its rows j < pos + T).
template <typename TE, int D>
__global__ void __launch_bounds__(kSketchThreads) append_kv_kernel(const TE* __restrict__ k_new,
                                                                   const TE* __restrict__ v_new, int T, int Hkv,
                                                                   TE* __restrict__ k_cache, TE* __restrict__ v_cache,
                                                                   int Ls, int pos, int Bk, int nb_cache,
                                                                   float* __restrict__ sketch) {
  __shared__ __align__(16) float red[kSketchThreads * 8];
  using V = Vec16<TE>;
  constexpr int CPR = D / V::N;
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel may still read the cache rows written below
  const int g = blockIdx.x;
  const int b = g / Hkv, kvh = g % Hkv;
  // copy rows: element (t, chunk) per thread
  for (int i = threadIdx.x; i < T * CPR; i += kSketchThreads) {
    const int t = i / CPR, c = i % CPR;
    const size_t src = ((static_cast<size_t>(b) * T + t) * Hkv + kvh) * D + c * V::N;
    const size_t dst = (static_cast<size_t>(g) * Ls + pos + t) * D + c * V::N;
    *reinterpret_cast<uint4*>(k_cache + dst) = *reinterpret_cast<const uint4*>(k_new + src);
    *reinterpret_cast<uint4*>(v_cache + dst) = *reinterpret_cast<const uint4*>(v_new + src);
  }
  __syncthreads();
  const int end = pos + T;
  for (int blk = pos / Bk; blk <= (end - 1) / Bk; ++blk) {
    const int j0 = blk * Bk;
    const int j1 = min(j0 + Bk, end);
    block_mean_rows<TE, D>(k_cache + (static_cast<size_t>(g) * Ls + j0) * D, j1 - j0,
                           sketch + (static_cast<size_t>(g) * nb_cache + blk) * D, red);
  }
}

}  // namespace sa
