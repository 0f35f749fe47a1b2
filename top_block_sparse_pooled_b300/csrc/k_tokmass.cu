// k_tokmass.cu -- head-collapsed token importance for decode.
//
// "How Much Dense Attention is Necessary?" Sec. 2.1-2.2: the dense attention
// distribution of every query head is computed and averaged over the heads
// into one token-importance distribution that selects the support of all
// heads.  For decode the T queries of a batch row share one support, so they
// are averaged too:
//   P[b, j] = 1/(Hq*T) * sum over heads h and queries t of softmax_j(scale * q[b,t,h] . k[b,h/G,j])
// over the causal keys j <= L - T + t (0 elsewhere).
//
// Three launches (HBM-bound: every key row is read once):
//   1. token_logits_kernel: per (group, key range), the R = G*T query rows of
//      the group against each key (mma.sync m16n8k16, bf16 in, fp32
//      accumulate; K rows come straight from global memory into the B
//      fragments, 16 bytes per lane), writes the base-2 logits [group][R][L]
//      and one (max, sum of 2^(s - max)) partial per (row, CTA);
//   2. token_lse_kernel: merges the partials of each row into its base-2
//      log-sum-exp;
//   3. token_mass_kernel: P[b, j] = sum over the rows of all of the row's
//      groups of 2^(s - lse), times 1/(Hq*T).
//
// Per-query prefill (b_sel = 1): the same logits with T = L (query t at
// position t), R = G*L rows tiled 16 at a time over grid.z, and
// token_mass_rows_kernel averaging over the heads only, one distribution per
// query.
//
// The dot product over d is order-free, so d is permuted consistently in the
// A (q) and B (k) fragments: lane (g, t) of a warp holds d = 32p + 8t .. +7 of
// its key row for k-steps 2p and 2p+1, one 16-byte load.
#pragma once

#include "sa_ptx.cuh"

namespace sa {

constexpr int kTmThreads = 256;
constexpr int kTmWarps = kTmThreads / 32;
constexpr int kTmNt = 4;  // n-tiles (8 keys each) per warp iteration

__device__ __forceinline__ void tm_mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// grid (chunks, groups, row tiles), kTmThreads.  CTA x covers keys
// [x * kpc, (x+1) * kpc), split into kTmWarps contiguous warp ranges of kpw keys
// (kpw a multiple of 32); CTA z the rows [16 z, 16 z + 16).  Keys past the
// tile's last query are not computed; they are written as -inf only when
// write_hidden is set (the per-query mass pass never reads them).
// logits: [groups][R][L] base-2 scaled logits (-inf where the key is not
// visible to the row); part: [groups][chunks][R] float2 (max, sum).
template <int D>
__global__ void __launch_bounds__(kTmThreads) token_logits_kernel(const __nv_bfloat16* __restrict__ q,
                                                                  const __nv_bfloat16* __restrict__ kc, int T, int Hq,
                                                                  int Hkv, int L, int Ls, float qscale2, int kpw,
                                                                  int write_hidden, float* __restrict__ logits,
                                                                  float2* __restrict__ part) {
  constexpr int KP = D / 32;  // 16-byte pieces per lane per key row (each covers two k-steps)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  const int g = blockIdx.y, b = g / Hkv, kvh = g % Hkv;
  const int G = Hq / Hkv, R = G * T;
  const int j0 = (blockIdx.x * kTmWarps + warp) * kpw;
  const int rbase = blockIdx.z * 16;
  // q rows gq and gq + 8 (row r = t * G + head), A fragments in the permuted d order
  uint32_t qa[D / 16][4];
  int lim0 = -1, lim1 = -1;  // last visible key of rows gq and gq + 8 (-1: no such row)
  {
    uint4 x0[KP], x1[KP];
    const int r0 = rbase + gq, r1 = rbase + gq + 8;
#pragma unroll
    for (int pc = 0; pc < KP; ++pc) {
      x0[pc] = make_uint4(0u, 0u, 0u, 0u);
      x1[pc] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (r0 < R) {
      const __nv_bfloat16* qr = q + ((static_cast<size_t>(b) * T + r0 / G) * Hq + kvh * G + r0 % G) * D;
#pragma unroll
      for (int pc = 0; pc < KP; ++pc) x0[pc] = *reinterpret_cast<const uint4*>(qr + 32 * pc + 8 * tq);
      lim0 = L - T + r0 / G;
    }
    if (r1 < R) {
      const __nv_bfloat16* qr = q + ((static_cast<size_t>(b) * T + r1 / G) * Hq + kvh * G + r1 % G) * D;
#pragma unroll
      for (int pc = 0; pc < KP; ++pc) x1[pc] = *reinterpret_cast<const uint4*>(qr + 32 * pc + 8 * tq);
      lim1 = L - T + r1 / G;
    }
#pragma unroll
    for (int pc = 0; pc < KP; ++pc) {
      qa[2 * pc][0] = x0[pc].x;
      qa[2 * pc][1] = x1[pc].x;
      qa[2 * pc][2] = x0[pc].y;
      qa[2 * pc][3] = x1[pc].y;
      qa[2 * pc + 1][0] = x0[pc].z;
      qa[2 * pc + 1][1] = x1[pc].z;
      qa[2 * pc + 1][2] = x0[pc].w;
      qa[2 * pc + 1][3] = x1[pc].w;
    }
  }
  const __nv_bfloat16* kg = kc + static_cast<size_t>(g) * Ls * D;
  const bool has0 = rbase + gq < R, has1 = rbase + gq + 8 < R;
  float* lg0 = logits + (static_cast<size_t>(g) * R + rbase + gq) * L;
  float* lg1 = logits + (static_cast<size_t>(g) * R + rbase + gq + 8) * L;
  float m0 = -INFINITY, m1 = -INFINITY, s0 = 0.f, s1 = 0.f;
  const int jend = min(L, j0 + kpw);
  // keys no row of this tile sees: -inf, no loads or math
  const int jvis = min(jend, L - T + min(R - 1, rbase + 15) / G + 1);
  for (int key = max(j0, jvis) + lane; write_hidden && key < jend; key += 32) {
    if (has0) lg0[key] = -INFINITY;
    if (has1) lg1[key] = -INFINITY;
  }
  for (int jb = j0; jb < jvis; jb += 8 * kTmNt) {
    uint4 kv[kTmNt][KP];
#pragma unroll
    for (int nt = 0; nt < kTmNt; ++nt) {
      const int key = jb + nt * 8 + gq;
#pragma unroll
      for (int pc = 0; pc < KP; ++pc)
        kv[nt][pc] = key < L ? __ldg(reinterpret_cast<const uint4*>(kg + static_cast<size_t>(key) * D + 32 * pc + 8 * tq))
                             : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int nt = 0; nt < kTmNt; ++nt) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int pc = 0; pc < KP; ++pc) {
        tm_mma_bf16(c, qa[2 * pc], kv[nt][pc].x, kv[nt][pc].y);
        tm_mma_bf16(c, qa[2 * pc + 1], kv[nt][pc].z, kv[nt][pc].w);
      }
      const int key = jb + nt * 8 + 2 * tq;  // keys key, key + 1 of rows gq (c0, c1) and gq + 8 (c2, c3)
      const float v00 = key <= lim0 ? c[0] * qscale2 : -INFINITY;
      const float v01 = key + 1 <= lim0 ? c[1] * qscale2 : -INFINITY;
      const float v10 = key <= lim1 ? c[2] * qscale2 : -INFINITY;
      const float v11 = key + 1 <= lim1 ? c[3] * qscale2 : -INFINITY;
      if (key + 1 < L && (L & 1) == 0) {  // rows start 8-byte aligned when L is even; key is even
        if (has0) *reinterpret_cast<float2*>(lg0 + key) = make_float2(v00, v01);
        if (has1) *reinterpret_cast<float2*>(lg1 + key) = make_float2(v10, v11);
      } else {
        if (has0) {
          if (key < L) lg0[key] = v00;
          if (key + 1 < L) lg0[key + 1] = v01;
        }
        if (has1) {
          if (key < L) lg1[key] = v10;
          if (key + 1 < L) lg1[key + 1] = v11;
        }
      }
      // running (max, sum of 2^(s - max)) of this lane's entries
      const float n0 = fmaxf(m0, fmaxf(v00, v01)), n1 = fmaxf(m1, fmaxf(v10, v11));
      if (n0 != -INFINITY) {
        s0 = s0 * exp2f(m0 - n0) + exp2f(v00 - n0) + exp2f(v01 - n0);
        m0 = n0;
      }
      if (n1 != -INFINITY) {
        s1 = s1 * exp2f(m1 - n1) + exp2f(v10 - n1) + exp2f(v11 - n1);
        m1 = n1;
      }
    }
  }
  // combine the four lanes of each row
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    const float mo0 = __shfl_xor_sync(0xFFFFFFFFu, m0, o), so0 = __shfl_xor_sync(0xFFFFFFFFu, s0, o);
    const float mo1 = __shfl_xor_sync(0xFFFFFFFFu, m1, o), so1 = __shfl_xor_sync(0xFFFFFFFFu, s1, o);
    const float n0 = fmaxf(m0, mo0), n1 = fmaxf(m1, mo1);
    s0 = (n0 == -INFINITY) ? 0.f : s0 * exp2f(m0 - n0) + so0 * exp2f(mo0 - n0);
    s1 = (n1 == -INFINITY) ? 0.f : s1 * exp2f(m1 - n1) + so1 * exp2f(mo1 - n1);
    m0 = n0;
    m1 = n1;
  }
  // then the CTA's eight warps
  __shared__ float2 wpart[kTmWarps][16];
  if (tq == 0) {
    wpart[warp][gq] = make_float2(m0, s0);
    wpart[warp][gq + 8] = make_float2(m1, s1);
  }
  __syncthreads();
  if (threadIdx.x < 16 && rbase + static_cast<int>(threadIdx.x) < R) {
    const int rl = threadIdx.x, r = rbase + rl;
    float m = -INFINITY, sum = 0.f;
#pragma unroll
    for (int w = 0; w < kTmWarps; ++w) {
      const float2 v = wpart[w][rl];
      const float n = fmaxf(m, v.x);
      if (n != -INFINITY) {
        sum = sum * exp2f(m - n) + v.y * exp2f(v.x - n);
        m = n;
      }
    }
    part[(static_cast<size_t>(g) * gridDim.x + blockIdx.x) * R + r] = make_float2(m, sum);
  }
}

// grid (groups, ceil(R / 16)), 16 warps: row r's base-2 log-sum-exp from its nparts partials.
__global__ void token_lse_kernel(const float2* __restrict__ part, int nparts, int R, float* __restrict__ lse2) {
  const int lane = threadIdx.x & 31, r = blockIdx.y * 16 + (threadIdx.x >> 5), g = blockIdx.x;
  if (r >= R) return;
  float m = -INFINITY, s = 0.f;
  for (int i = lane; i < nparts; i += 32) {
    const float2 v = part[(static_cast<size_t>(g) * nparts + i) * R + r];
    const float n = fmaxf(m, v.x);
    if (n != -INFINITY) {
      s = s * exp2f(m - n) + v.y * exp2f(v.x - n);
      m = n;
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float mo = __shfl_xor_sync(0xFFFFFFFFu, m, o), so = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    const float n = fmaxf(m, mo);
    s = (n == -INFINITY) ? 0.f : s * exp2f(m - n) + so * exp2f(mo - n);
    m = n;
  }
  if (lane == 0) lse2[static_cast<size_t>(g) * R + r] = m + log2f(s);
}

// grid (ceil(L / (4 * kTmThreads)), B): four keys per thread.
__global__ void __launch_bounds__(kTmThreads) token_mass_kernel(const float* __restrict__ logits,
                                                                const float* __restrict__ lse2, int Hkv, int R, int L,
                                                                float inv_rows, float* __restrict__ mass) {
  const int b = blockIdx.y;
  const int j = (blockIdx.x * kTmThreads + threadIdx.x) * 4;
  if (j >= L) return;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  const bool vec = (L % 4 == 0);
  if (vec) {  // rows of eight, loads issued together
    const int nrow = Hkv * R;
    const float* lg = logits + static_cast<size_t>(b) * nrow * L + j;
    const float* ls2 = lse2 + static_cast<size_t>(b) * nrow;
    for (int r0 = 0; r0 < nrow; r0 += 8) {
      float4 v[8];
      float ls[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const bool in = r0 + i < nrow;
        v[i] = in ? __ldcs(reinterpret_cast<const float4*>(lg + static_cast<size_t>(r0 + i) * L))
                  : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        ls[i] = in ? __ldg(ls2 + r0 + i) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        a0 += exp2f(v[i].x - ls[i]);
        a1 += exp2f(v[i].y - ls[i]);
        a2 += exp2f(v[i].z - ls[i]);
        a3 += exp2f(v[i].w - ls[i]);
      }
    }
  }
  for (int kvh = 0; kvh < Hkv && !vec; ++kvh) {
    const int g = b * Hkv + kvh;
    for (int r = 0; r < R; ++r) {
      const float ls = __ldg(lse2 + static_cast<size_t>(g) * R + r);
      const float* row = logits + (static_cast<size_t>(g) * R + r) * L;
      {
        a0 += exp2f(row[j] - ls);
        if (j + 1 < L) a1 += exp2f(row[j + 1] - ls);
        if (j + 2 < L) a2 += exp2f(row[j + 2] - ls);
        if (j + 3 < L) a3 += exp2f(row[j + 3] - ls);
      }
    }
  }
  float* out = mass + static_cast<size_t>(b) * L + j;
  if (vec) {
    *reinterpret_cast<float4*>(out) = make_float4(a0 * inv_rows, a1 * inv_rows, a2 * inv_rows, a3 * inv_rows);
  } else {
    out[0] = a0 * inv_rows;
    if (j + 1 < L) out[1] = a1 * inv_rows;
    if (j + 2 < L) out[2] = a2 * inv_rows;
    if (j + 3 < L) out[3] = a3 * inv_rows;
  }
}

// Per-query prefill: grid (ceil(L / (4 * kTmThreads)), L queries, B).
// P[b, t, j] = 1/Hq * sum over the Hkv groups and their G heads of 2^(s - lse)
// for the rows (t, head); keys past t are 0 (their logits are not read).
__global__ void __launch_bounds__(kTmThreads) token_mass_rows_kernel(const float* __restrict__ logits,
                                                                     const float* __restrict__ lse2, int Hkv, int G,
                                                                     int L, float inv_heads,
                                                                     float* __restrict__ mass) {
  const int t = blockIdx.y, b = blockIdx.z;
  const int j = (blockIdx.x * kTmThreads + threadIdx.x) * 4;
  if (j >= L) return;
  const size_t R = static_cast<size_t>(G) * L;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
  if (j <= t) {
    const int nrow = Hkv * G;  // rows (kvh, head) of query t, eight loads in flight
    const bool vec = (L % 4 == 0);
    for (int i0 = 0; i0 < nrow; i0 += 8) {
      float4 v[8];
      float ls[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int ri = i0 + i;
        const size_t g = static_cast<size_t>(b) * Hkv + (ri < nrow ? ri / G : 0);
        const size_t r = static_cast<size_t>(t) * G + (ri < nrow ? ri % G : 0);
        const float* row = logits + (g * R + r) * L + j;
        ls[i] = ri < nrow ? __ldg(lse2 + g * R + r) : 0.f;
        if (ri >= nrow) {
          v[i] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        } else if (vec) {
          v[i] = __ldcs(reinterpret_cast<const float4*>(row));
        } else {
          v[i].x = __ldcs(row);
          v[i].y = j + 1 < L ? __ldcs(row + 1) : -INFINITY;
          v[i].z = j + 2 < L ? __ldcs(row + 2) : -INFINITY;
          v[i].w = j + 3 < L ? __ldcs(row + 3) : -INFINITY;
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        a[0] += exp2f(v[i].x - ls[i]);
        a[1] += j + 1 <= t ? exp2f(v[i].y - ls[i]) : 0.f;
        a[2] += j + 2 <= t ? exp2f(v[i].z - ls[i]) : 0.f;
        a[3] += j + 3 <= t ? exp2f(v[i].w - ls[i]) : 0.f;
      }
    }
  }
  float* out = mass + (static_cast<size_t>(b) * L + t) * L + j;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (j + e < L) out[e] = a[e] * inv_heads;
}

}  // namespace sa
