/*
 * sparse_attn.h -- C ABI of libsparse_attn: top-k block-sparse GQA attention
 * on one NVIDIA B300 (sm_103a).
 *
 * The method (web summaries of the papers, by title and section):
 *  - "Faster Than Flash: Exploiting Attention Sparsity for Efficient
 *    Long-Context Decoding", Sec. 1 and 3: a small, compressed sketch of the KV
 *    cache is scanned first to estimate which parts matter; only the selected
 *    blocks are then loaded for the exact attention computation.  Sink
 *    (initial) and local tokens dominate the attention distribution (Sec. 2).
 *  - "How Much Dense Attention is Necessary? Oracle-Guided Sparse Prefill ...",
 *    Sec. 2.1: an oracle ranks keys by their exact dense attention mass,
 *    aggregated over the query heads; the top-k under a fixed budget form the
 *    support, optionally shared by a block of consecutive queries; attention
 *    is then recomputed with the original q, k, v on that support only.
 *    Sec. 2.2: the same score -> top-k -> sparse-GQA shape at inference.
 *  - "Pulsar Attention", Phase 1: a fixed attention-sink prefix is always kept;
 *    Phase 2: partial softmaxes over disjoint key sets merge exactly (online
 *    softmax), which is how split-KV partials are combined here.
 *  - "The Sparse Frontier", Sec. 1 and RQ2: block-wise selection for prefill,
 *    page selection with the full cache retained for decode.
 *
 * Notation: B batch, Hq query heads, Hkv kv heads, G = Hq / Hkv, query head h
 * reads kv head h / G; d head dim; L context length (keys); Bk = `block` keys
 * per KV block, nb = ceil(L / Bk); a "group" is one (batch, kv-head) pair,
 * g = b * Hkv + kvh.  scale is the softmax scale (1/sqrt(d) is the usual one).
 *
 * Layouts (all row-major, contiguous, caller-owned DEVICE memory):
 *   K, V cache / prefill K, V : [B, Hkv, L_stride, d]   (rows j < L valid)
 *   decode q, out             : [B, T, Hq, d]           (query t sits at key
 *                                                       position L - T + t)
 *   prefill q, out            : [B, L, Hq, d]           (query t at position t)
 *   k_new, v_new (append)     : [B, T, Hkv, d]
 *   sketch                    : [B, Hkv, ceil(L_stride / Bk), d] float32 (blocks
 *                               past ceil(L / Bk) unused)
 *   scores / mass             : [B, Hkv, nq, nb] float32, nq = 1 for decode,
 *                               ceil(L / qtile) for prefill
 *   idx                       : [B, Hkv, nq, kmax] int32, ascending block ids,
 *                               padded with -1;   cnt : [B, Hkv, nq] int32
 *
 * dtype: SA_F32 or SA_BF16 for q, k, v, k_new, v_new, out (all the same).
 *
 * Conventions.  Every call validates its arguments on the host before any
 * launch and returns SA_ERR_INVALID_ARG / SA_ERR_UNSUPPORTED without touching
 * the device when they are bad; sa_last_error() then gives a message.  Calls
 * are asynchronous: they enqueue work on `stream` (a cudaStream_t; NULL = the
 * legacy default stream) and return.  The library allocates no device memory
 * of its own: scratch space is passed in as `workspace` (sizes from the
 * *_workspace_bytes queries).  Two exceptions, documented at their calls: the
 * fixed scratch array of sa_decode_noalloc and the CUDA graphs that
 * sa_decode_step keeps for repeated argument sets.  Kernels bound every wait
 * (on copies, on other warps); a wait that gives up records SA_ERR_TIMEOUT in
 * a device-side status word that sa_device_status() reads.
 */
#ifndef SPARSE_ATTN_H
#define SPARSE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = 1, /* bad pointer, shape, budget or buffer size */
  SA_ERR_UNSUPPORTED = 2, /* valid but not implemented: dtype, d, block, device */
  SA_ERR_CUDA = 3,        /* a CUDA runtime call failed (message has the name) */
  SA_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up */
} sa_status_t;

typedef enum { SA_F32 = 0, SA_BF16 = 1 } sa_dtype_t;

typedef enum {
  SA_SELECT_SKETCH = 0, /* score blocks by max over the group's rows of scale*q.sketch */
  SA_SELECT_MASS = 1    /* rank blocks by a given score array (e.g. sa_oracle_mass) */
} sa_select_mode_t;

/* Library version (major*10000 + minor*100 + patch). */
int sa_version(void);

/* Message for the last failing call on this host thread ("" if none). */
const char* sa_last_error(void);

/* Name of a status code. */
const char* sa_status_name(int status);

/*
 * Device-side status word.  Synchronizes the current device, then stores in
 * *code the first error code a kernel recorded since the last clear (SA_OK if
 * none) and, if clear != 0, resets it.  Returns SA_ERR_CUDA if the device
 * synchronization itself fails.
 */
sa_status_t sa_device_status(int* code, int clear);

/*
 * a1. Block sketch ("Faster Than Flash" Sec. 1: a compressed summary scanned
 * in place of the keys).  sketch[g, b, :] = mean of the valid key rows
 * j in [b*Bk, min((b+1)*Bk, L)) of k[g], accumulated in float32.
 * k: [B, Hkv, L_stride, d] (dtype); sketch: [B, Hkv, ceil(L_stride/Bk), d]
 * float32, blocks b < nb written.
 * Requires L >= 1, L <= L_stride, d in {64, 128}, block in [1, 1024].
 */
sa_status_t sa_build_sketch(const void* k, int dtype, int B, int Hkv, int L, int L_stride, int d,
                            int block, float* sketch, void* stream);

/*
 * a1 fused with the cache append ("Sparse Attention as a Range Searching
 * Problem" Sec. 2: new keys join the index incrementally, without a rebuild).
 * Writes k_new[b, t, kvh, :] / v_new[...] to cache rows pos + t (t < T) of
 * group (b, kvh), then rewrites the sketch of every block those rows touch as
 * the mean of its valid rows j < pos + T.  Blocks wholly before pos are not
 * read.  k_new, v_new: [B, T, Hkv, d]; caches [B, Hkv, L_stride, d];
 * sketch [B, Hkv, ceil(L_stride/Bk), d] float32.  Requires pos + T <= L_stride.
 */
sa_status_t sa_append_kv(const void* k_new, const void* v_new, int dtype, int B, int Hkv, int T,
                         int d, void* k_cache, void* v_cache, int L_stride, int pos, int block,
                         float* sketch, void* stream);

/*
 * a2 + a3. Block scoring and top-k selection ("How Much Dense Attention is
 * Necessary?" Sec. 2.1-2.2; sink/local kept: "Pulsar Attention" Phase 1,
 * "Faster Than Flash" Sec. 2).
 *
 * prefill == 0 (decode): one selection per group for the T = Tq query tokens
 *   at positions L-T..L-1.  Candidate blocks: 1..nb-2; forced: {0, nb-1}.
 *   Budget: k.
 * prefill != 0: one selection per (group, query tile i of `qtile` rows),
 *   i.e. a support shared by the tile's queries (b_sel = qtile).  The causal
 *   blocks of tile i are 0..c_i-1 with c_i = (last query position of the tile)
 *   / Bk + 1; forced: {0, c_i - 1} (sink and diagonal); candidates: the rest.
 *   Budget of tile i: k + ceil(frac_num * c_i / frac_den) (frac_num = 0: k).
 * Ranking: the budget's worth of highest-scoring candidates, ties to the lower
 *   block index; the output is the union with the forced blocks, ascending.
 *
 * mode SA_SELECT_SKETCH: score s = max over the group's query heads and the
 *   unit's query rows of scale * (q . sketch[g, b]), in float32.  `sketch`
 *   must be given.  Decode: if `scores` is not NULL the scores are written
 *   there ([B, Hkv, 1, nb]).  Prefill: `scores` is required and written
 *   ([B, Hkv, nq, nb]; non-causal entries are -inf); the tile scores are
 *   computed on the tensor cores (q bf16 times the fp32 sketch split into
 *   three bf16 parts, fp32 accumulation), then each tile's top-k is taken.
 * mode SA_SELECT_MASS: `scores` is an input (e.g. from sa_oracle_mass or,
 *   with block == 1 and Hkv == 1, from sa_token_mass_decode); q and sketch
 *   are not read.  Decode score arrays longer than 16384 entries are read
 *   from global memory (one CTA per unit); prefill ones are limited to 16384.
 * idx: [B, Hkv, nq, kmax] int32 written (ascending, -1 padded), cnt:
 *   [B, Hkv, nq] int32 written.  kmax must be >= sa_select_kmax(...).
 * Requires d in {64, 128}; G * Tq <= 32 and (bf16) a 16-byte-aligned q for
 * decode; qtile == Bk == 128, d == 128, bf16 q and scale > 0 for prefill in
 * SKETCH mode.
 */
sa_status_t sa_select_topk(int mode, const void* q, int dtype, const float* sketch, float* scores,
                           int B, int Tq, int Hq, int Hkv, int d, int L, int L_stride, int block,
                           int qtile, int prefill, int k, int frac_num, int frac_den, float scale,
                           int32_t* idx, int32_t* cnt, int kmax, void* stream);

/*
 * Decode top-delta selection ("Faster Than Flash" Sec. 2: a key is kept when
 * its score is at least a pseudo-maximum minus delta; the pseudo-maximum comes
 * from the sink and local-context keys only, so no global reduction is
 * needed).  At block granularity: with the sketch scores s of sa_select_topk
 * (mode SA_SELECT_SKETCH, decode), pm = max(s[0], s[nb-1]); the kept blocks
 * are {0, nb-1} plus every other block with s >= pm - delta, at most `cap` of
 * them (the highest, ties to the lower index).  The count per group varies:
 * cnt[g] in [1, cap + 2]; kmax >= sa_select_kmax(L, block, 0, 0, cap, 0, 1).
 * delta >= 0 in the units of the scores (scaled logits).  Other arguments and
 * requirements as for sa_select_topk in decode mode.
 */
sa_status_t sa_select_topdelta(const void* q, int dtype, const float* sketch, float* scores, int B, int Tq,
                               int Hq, int Hkv, int d, int L, int L_stride, int block, float delta,
                               int cap, float scale, int32_t* idx, int32_t* cnt, int kmax, void* stream);

/*
 * Length-aware block budget ("The Sparse Frontier" RQ3: longer sequences
 * tolerate more sparsity, so the budget should grow sublinearly with the
 * length; "How Much Dense Attention is Necessary?" Sec. 3.1: shared supports
 * need budgets that scale with the length).  Returns
 *   k(L) = ceil(k_ref * (L / L_ref)^exponent),
 * clamped to the candidates available (ceil(L / block) - 2, at least 0):
 * exponent 0 keeps k_ref blocks at every length, 1 keeps a fixed fraction.
 * Host-only; returns -1 for L, block, L_ref < 1, k_ref < 0 or an exponent
 * outside [0, 1].  Pass the result as `k` (decode) to sa_select_topk.
 */
int sa_budget_sublinear(int L, int block, int k_ref, int L_ref, float exponent);

/* Smallest kmax that holds every selection of the given problem (or -1 if invalid). */
int sa_select_kmax(int L, int block, int qtile, int prefill, int k, int frac_num, int frac_den);

/*
 * a4, decode. Exact softmax attention over the selected blocks only ("How
 * Much Dense Attention is Necessary?" Sec. 2.1), split over the selected
 * blocks (flash-decoding) with an exact online-softmax merge of the partials
 * ("Pulsar Attention" Phase 2).  For query row (b, t, h), g = b*Hkv + h/G:
 *   out[b,t,h] = sum_j softmax_j(scale * q[b,t,h] . k[g,j]) v[g,j]
 * over keys j in the blocks idx[g, 0:cnt[g]] with j < L and
 * j <= L - T + t.  workspace: >= sa_decode_workspace_bytes(...) bytes of
 * device memory, 16-byte aligned, ZERO-FILLED before its first use (it holds
 * per-group arrival counters; every call that completes leaves them zero, so
 * a workspace is zeroed once, and again after a call that reported an error).
 * Calls that share a workspace must not overlap on the device.
 * Requires d in {64, 128}; block == 64; G*T <= 32; T <= block;
 * 16-byte-aligned k/v caches.
 */
size_t sa_decode_workspace_bytes(int B, int T, int Hq, int Hkv, int d, int kmax);
sa_status_t sa_decode(const void* q, const void* k_cache, const void* v_cache, int dtype,
                      const int32_t* idx, const int32_t* cnt, int kmax, int B, int T, int Hq,
                      int Hkv, int d, int L, int L_stride, int block, float scale, void* out,
                      void* workspace, size_t ws_bytes, void* stream);

/*
 * a2 + a3 + a4, decode, in one launch: the sketch scoring and top-k selection
 * of sa_select_topk (SKETCH mode, decode) followed by the attention of
 * sa_decode over the blocks just selected ("How Much Dense Attention is
 * Necessary?" Sec. 2.1-2.2: score, keep the top-k, recompute exact attention on
 * them; "Faster Than Flash" Sec. 1-3: one pass that scans the block summaries
 * and then reads only the selected blocks).  One cluster of CTAs per
 * (batch, kv-head) group: the CTAs score slices of the group's sketch, CTA 0
 * of the cluster selects, each CTA attends over a share of the selected blocks,
 * and the partials merge exactly through distributed shared memory.
 *
 * Arguments and layouts are those of sa_select_topk (q [B, T, Hq, d], sketch
 * [B, Hkv, ceil(L_stride/block), d] fp32, idx [B, Hkv, kmax] and cnt [B, Hkv]
 * written, scores [B, Hkv, ceil(L/block)] written when not NULL) and of
 * sa_decode (k/v caches [B, Hkv, L_stride, d], out [B, T, Hq, d]); the
 * selection and the output equal those of the two separate calls.  No
 * workspace.  Requires dtype SA_BF16, d in {64, 128}, block == 64,
 * G*T <= 16, T <= block, at most 16384 blocks; returns SA_ERR_UNSUPPORTED
 * otherwise (use the two separate calls).  Invalid arguments return
 * SA_ERR_INVALID_ARG before any launch.
 */
sa_status_t sa_select_decode(const void* q, int dtype, const float* sketch, const void* k_cache,
                             const void* v_cache, int B, int T, int Hq, int Hkv, int d, int L, int L_stride,
                             int block, int k, float scale, int32_t* idx, int32_t* cnt, int kmax,
                             float* scores, void* out, void* stream);

/*
 * sa_decode without a workspace argument, for callers that cannot allocate
 * device memory: code embedded in a host runtime that owns the whole device
 * memory pool and gives its plugins no allocation hook, or a latency-critical
 * path that must not pay for cudaMalloc (which can synchronize the device).
 * The pages have no counterpart of this call; it is a deployment variant of
 * sa_decode with the same arguments, layouts and results.
 *
 * Scratch: the library keeps one fixed array of 8 MiB (8388608 bytes) in
 * device memory for this call, on every device that loads the library, until
 * the process exits.  A problem whose sa_decode_workspace_bytes(...) exceeds
 * 8 MiB is rejected with SA_ERR_INVALID_ARG before any device work.  No device
 * memory is allocated by this call.
 *
 * The first call made with a given device current looks up the array's device
 * address on that device (cudaGetSymbolAddress); make that first call before
 * any stream capture.  The address is cached with the device's CUDA context;
 * a call made in a new context of the device (after cudaDeviceReset) looks it
 * up again, so that first call in the new context also belongs before any
 * capture.  Each call clears the arrival counters at the head of
 * the array on `stream`, then runs the same kernels as sa_decode.  All calls
 * share the one array: calls that overlap on the device (on different streams,
 * or from several host threads without ordering) race on it and give wrong
 * results; order them on one stream or with events.
 */
sa_status_t sa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, int dtype,
                              const int32_t* idx, const int32_t* cnt, int kmax, int B, int T, int Hq,
                              int Hkv, int d, int L, int L_stride, int block, float scale, void* out,
                              void* stream);

/*
 * a4, prefill. Causal exact attention per query tile over the tile's
 * selected blocks ("How Much Dense Attention is Necessary?" Sec. 2.1,
 * support shared by the tile; "The Sparse Frontier" RQ2, block-sparse
 * prefill).  For query row (b, t, h) in tile i = t / qtile:
 *   out[b,t,h] = sum_j softmax_j(scale * q[b,t,h] . k[g,j]) v[g,j],
 * keys j in blocks idx[g, i, 0:cnt[g,i]] with j <= t.  lse_out (optional,
 * [B, Hq, L] float32): natural-log sum of exp of the row's logits.
 * Tensor cores (tcgen05, TMEM accumulators).  Requires dtype SA_BF16,
 * d == 128, qtile == block == 128.
 */
sa_status_t sa_prefill(const void* q, const void* k, const void* v, int dtype, const int32_t* idx,
                       const int32_t* cnt, int kmax, int B, int L, int Hq, int Hkv, int d,
                       int qtile, int block, float scale, void* out, float* lse_out, void* stream);

/*
 * a5. Exact per-block attention mass ("How Much Dense Attention is
 * Necessary?" Sec. 2.1: the full dense distribution of each query,
 * aggregated over the query heads).  For group g and query tile i:
 *   mass[g, i, b] = sum over the group's heads h and the tile's rows t of
 *                   sum_{j in block b, j <= t} P_{h,t}(j),
 * P_{h,t} the dense causal softmax of row (h, t).  Non-causal entries are 0.
 * workspace: >= sa_oracle_mass_workspace_bytes(...) bytes of device memory.
 * Requires dtype SA_BF16, d == 128, qtile == block == 128.
 */
size_t sa_oracle_mass_workspace_bytes(int B, int L, int Hq, int Hkv, int d, int qtile, int block);
sa_status_t sa_oracle_mass(const void* q, const void* k, int dtype, int B, int L, int Hq, int Hkv,
                           int d, int qtile, int block, float scale, float* mass, void* workspace,
                           size_t ws_bytes, void* stream);

/*
 * Head-collapsed token importance for decode ("How Much Dense Attention is
 * Necessary?" Sec. 2.1: the dense attention distribution of each query,
 * averaged over the query heads; Sec. 2.2: one distribution shared by all
 * heads).  The T decode queries of a batch row share one support, so they
 * are averaged too:
 *   mass[b, j] = 1/(Hq*T) * sum over heads h and queries t of P_{b,t,h}(j),
 * P_{b,t,h} the dense softmax of scale * q[b,t,h] . k[b, h/G, :] over the
 * causal keys j <= L - T + t (0 for the others); each row of mass sums to 1.
 * q: [B, T, Hq, d]; k_cache: [B, Hkv, L_stride, d]; mass: [B, L] float32
 * written.  workspace: >= sa_token_mass_workspace_bytes(...) bytes of device
 * memory (base-2 logits [B*Hkv, G*T, L] float32 and per-row partials).
 * Requires dtype SA_BF16, d in {64, 128}, G*T <= 16, T <= L, 16-byte-aligned
 * q, k_cache, mass and workspace.  Select tokens from it with sa_select_topk
 * (mode SA_SELECT_MASS, Hkv 1, block 1) and attend with sa_decode_tokens.
 */
size_t sa_token_mass_workspace_bytes(int B, int T, int Hq, int Hkv, int L);
sa_status_t sa_token_mass_decode(const void* q, const void* k_cache, int dtype, int B, int T, int Hq,
                                 int Hkv, int d, int L, int L_stride, float scale, float* mass,
                                 void* workspace, size_t ws_bytes, void* stream);

/*
 * a4 at token granularity, shared across the kv heads ("How Much Dense
 * Attention is Necessary?" Sec. 2.1: recompute exactly on the selected
 * support; Sec. 2.2: one head-collapsed support for every head).  For query
 * row (b, t, h):
 *   out[b,t,h] = sum_j softmax_j(scale * q[b,t,h] . k[b,h/G,j]) v[b,h/G,j]
 * over the distinct tokens j in idx[b, 0:cnt[b]] with j < L and
 * j <= L - T + t (entries out of range are ignored; order is free).
 * idx: [B, kmax] int32, cnt: [B] int32 (e.g. from sa_select_topk in MASS
 * mode with block 1).  workspace: >= sa_decode_workspace_bytes(B, T, Hq,
 * Hkv, d, kmax), zero-filled before first use, as for sa_decode.  Requires
 * dtype SA_BF16, d in {64, 128}, G*T <= 16, T <= L, 16-byte-aligned q and
 * caches.
 */
sa_status_t sa_decode_tokens(const void* q, const void* k_cache, const void* v_cache, int dtype,
                             const int32_t* idx, const int32_t* cnt, int kmax, int B, int T, int Hq,
                             int Hkv, int d, int L, int L_stride, float scale, void* out,
                             void* workspace, size_t ws_bytes, void* stream);

/*
 * Per-query (b_sel = 1) head-collapsed token importance for causal prefill
 * ("How Much Dense Attention is Necessary?" Sec. 2.1: each query position
 * selects its own support from its dense attention distribution, averaged
 * over the query heads):
 *   mass[b, t, j] = 1/Hq * sum over heads h of P_{b,t,h}(j),
 * P_{b,t,h} the dense softmax of scale * q[b,t,h] . k[b, h/G, :] over j <= t
 * (0 for j > t); each row sums to 1.  q: [B, L, Hq, d]; k: [B, Hkv, L, d];
 * mass: [B, L, L] float32 written.  workspace: >=
 * sa_token_mass_prefill_workspace_bytes(...) bytes (base-2 logits
 * [B*Hkv, G*L, L] float32: B*Hq*L*L*4 bytes, and per-row partials).  Requires
 * dtype SA_BF16, d in {64, 128}, L <= 65535, 16-byte-aligned pointers.
 * Select with sa_select_topk (mode SA_SELECT_MASS, prefill, Hkv 1,
 * qtile 1, block 1: tokens 0 and t forced per query) and attend with
 * sa_prefill_tokens.
 */
size_t sa_token_mass_prefill_workspace_bytes(int B, int L, int Hq, int Hkv);
sa_status_t sa_token_mass_prefill(const void* q, const void* k, int dtype, int B, int L, int Hq, int Hkv,
                                  int d, float scale, float* mass, void* workspace, size_t ws_bytes,
                                  void* stream);

/*
 * Causal prefill over per-query token supports (b_sel = 1), shared by the
 * kv heads ("How Much Dense Attention is Necessary?" Sec. 2.1; Sec. 2.2 for
 * the head-collapsed support).  For query row (b, t, h):
 *   out[b,t,h] = sum_j softmax_j(scale * q[b,t,h] . k[b,h/G,j]) v[b,h/G,j]
 * over the distinct tokens j in idx[b, t, 0:cnt[b, t]] with j <= t (others
 * ignored; order free).  idx: [B, L, kmax] int32, cnt: [B, L] int32.
 * q, out: [B, L, Hq, d]; k, v: [B, Hkv, L, d].  workspace: >=
 * sa_prefill_tokens_workspace_bytes(...) bytes, zero-filled before first use,
 * as for sa_decode.  Requires dtype SA_BF16, d in {64, 128}, G <= 16,
 * B*L*Hkv <= 2^24, 16-byte-aligned q, k, v, out and workspace.
 * With d == 128 and L <= 16384 the lists become per-query bit masks in the
 * workspace and every 128-query tile is attended on the tensor cores over the
 * 128-key blocks that hold any of its queries' tokens, each query over its own
 * tokens only; otherwise each query's token rows are gathered.
 */
size_t sa_prefill_tokens_workspace_bytes(int B, int L, int Hq, int Hkv, int d, int kmax);
sa_status_t sa_prefill_tokens(const void* q, const void* k, const void* v, int dtype, const int32_t* idx,
                              const int32_t* cnt, int kmax, int B, int L, int Hq, int Hkv, int d,
                              float scale, void* out, void* workspace, size_t ws_bytes, void* stream);

/*
 * Self-test of the failure path every pipeline kernel uses: one CTA waits on
 * an mbarrier phase that nothing completes, gives up after limit_ns
 * nanoseconds (1 ms .. 1 s), records SA_ERR_TIMEOUT in the device status word
 * and returns; read it with sa_device_status.  The context stays usable.  The
 * pages have no counterpart of this call; it exists so that the bounded-wait
 * error reporting can be tested without faulting or hanging a GPU.
 */
sa_status_t sa_selftest_wait_timeout(long long limit_ns, void* stream);

/*
 * Self-test of sa_decode_noalloc's recovery: fills the first `bytes` bytes of
 * the library's decode scratch on the current device (where its arrival
 * counters live) with a non-zero byte pattern, as a call that gave up
 * mid-way could leave them.  The next sa_decode_noalloc must still be exact
 * (it clears the counters on its stream before each launch).  bytes in
 * [1, 8 MiB]; SA_ERR_INVALID_ARG otherwise.  No counterpart in the pages.
 */
sa_status_t sa_selftest_poison_noalloc(int bytes, void* stream);

/*
 * One decode step: a1 append (k_new, v_new at cache rows L-T..L-1, sketch
 * refreshed), a2+a3 sketch selection with budget k, a4 decode.  If
 * host_io != 0, q, k_new, v_new and out are HOST pointers: k_new, v_new and
 * out are read and written in place by the kernels when they are page-locked
 * memory mapped into the device's address space (cudaHostAlloc, or pinned
 * memory under unified addressing), and so is q when the step is one launch
 * (bf16, block 64, G*T <= 16, the new rows inside the last block, no scores);
 * otherwise each is staged by a copy through `workspace` (pageable memory:
 * the copies are then synchronous).  Otherwise they are device pointers.
 * sketch, caches, idx, cnt, scores (optional) are device memory as above.
 * workspace: >= sa_decode_step_workspace_bytes(...) bytes of device memory,
 * zero-filled before first use exactly as for sa_decode (its head is
 * sa_decode's workspace).
 * On a stream other than the legacy default stream, an argument set that
 * repeats (same pointers and sizes) is captured into a CUDA graph on its
 * second call and replayed with one launch afterwards (at most 32 graphs,
 * least recently used evicted); buffer contents may change between calls.
 */
size_t sa_decode_step_workspace_bytes(int B, int T, int Hq, int Hkv, int d, int dtype, int kmax);
sa_status_t sa_decode_step(const void* q, const void* k_new, const void* v_new, int dtype,
                           void* k_cache, void* v_cache, float* sketch, int B, int T, int Hq,
                           int Hkv, int d, int L, int L_stride, int block, int k, float scale,
                           int32_t* idx, int32_t* cnt, int kmax, float* scores, void* out,
                           int host_io, void* workspace, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_ATTN_H */
