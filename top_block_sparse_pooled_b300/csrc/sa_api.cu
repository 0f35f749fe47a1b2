// sa_api.cu -- the C ABI of libsparse_attn (see include/sparse_attn.h):
// argument validation on the host, tensor-map encoding, launch sizing.
// The kernels are compiled into this one translation unit.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <vector>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "sparse_attn.h"

// Resident CTAs per SM of the bf16 decode kernel (each gets an equal share of
// the SM's shared memory for its K/V ring).
#ifndef SA_DM_CTAS_PER_SM
#define SA_DM_CTAS_PER_SM 1
#endif
// Work ranges per resident CTA slot (more, shorter ranges let the block
// scheduler balance SMs that are served later by the memory system).
#ifndef SA_DM_WAVES
#define SA_DM_WAVES 1
#endif
// Upper bound on the K/V ring depth of each decode CTA.
#ifndef SA_DM_MAXSTAGES
#define SA_DM_MAXSTAGES 4
#endif
// Token mode: at least this many 64-token units per CTA, so that the last CTA of a group has
// fewer partials to merge (measured on the 2050-token decode: 1 -> 22.5 us, 3 -> 18.5 us, 4 and
// 6 slower again).
#ifndef SA_DM_TOK_MIN_PER
#define SA_DM_TOK_MIN_PER 3
#endif

#include "k_decode.cu"
#include "k_decode_mma.cu"
#include "k_prefill.cu"
#include "k_mass.cu"
#include "k_select.cu"
#include "k_score.cu"
#include "k_sketch.cu"
#include "k_tokmass.cu"
#include "k_selftest.cu"
#include "k_seldec.cu"

namespace {

thread_local std::string t_err;

sa_status_t fail(sa_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_err = buf;
  return st;
}

#define SA_ARG(cond, ...) \
  do {                    \
    if (!(cond)) return fail(SA_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)
#define SA_SUP(cond, ...) \
  do {                    \
    if (!(cond)) return fail(SA_ERR_UNSUPPORTED, __VA_ARGS__); \
  } while (0)
#define SA_CUDA(call)                                                                 \
  do {                                                                                \
    cudaError_t e_ = (call);                                                          \
    if (e_ != cudaSuccess) return fail(SA_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)
#define SA_TRY(expr)              \
  do {                            \
    sa_status_t s_ = (expr);      \
    if (s_ != SA_OK) return s_;   \
  } while (0)

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }
inline int esize(int dtype) { return dtype == SA_F32 ? 4 : 2; }

// ------------------------------------------------------------------ device info
struct DevInfo {
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
};

sa_status_t dev_info(DevInfo* out) {
  static std::mutex mu;
  static DevInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  SA_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(SA_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (!have[dev]) {
    DevInfo d;
    SA_CUDA(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev));
    SA_CUDA(cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev));
    SA_CUDA(cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev));
    cache[dev] = d;
    have[dev] = true;
  }
  *out = cache[dev];
  if (out->cc_major != 10 || out->cc_minor != 3)
    return fail(SA_ERR_UNSUPPORTED, "built for sm_103a; device is sm_%d%d", out->cc_major, out->cc_minor);
  return SA_OK;
}

// An int derived once per device (occupancy, cluster limits) for one kernel
// instantiation: each call site keeps its own function-local PerDevice.
struct PerDevice {
  std::mutex mu;
  int v[64] = {};
};

template <typename F>
sa_status_t per_device(PerDevice& c, F compute, int* out) {
  int dev = 0;
  SA_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(SA_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(c.mu);
  if (c.v[dev] == 0) {
    int x = 0;
    SA_TRY(compute(&x));
    c.v[dev] = std::max(1, x);
  }
  *out = c.v[dev];
  return SA_OK;
}

// Per-kernel shared-memory opt-in (cached per function).
template <typename K>
sa_status_t set_smem(K kernel, int bytes) {
  SA_CUDA(cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel), cudaFuncAttributeMaxDynamicSharedMemorySize,
                               bytes));
  return SA_OK;
}

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel of the stream finishes (it calls pdl_wait() before
// touching memory that kernel uses).
template <typename... KArgs, typename... Args>
sa_status_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, int smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  SA_CUDA(cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...));
  return SA_OK;
}

// --------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

sa_status_t get_encode(EncodeTiledFn* fn) {
  static std::once_flag once;
  static EncodeTiledFn f = nullptr;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) f = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!f) return fail(SA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  *fn = f;
  return SA_OK;
}

// 2-D tiled map over a row-major [rows, inner] array; box {box_inner, box_rows}.
sa_status_t make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                        uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc;
  SA_TRY(get_encode(&enc));
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(SA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d): inner=%llu rows=%llu stride=%llu box=%ux%u", (int)r,
                (unsigned long long)inner, (unsigned long long)rows, (unsigned long long)row_stride_bytes, box_inner,
                box_rows);
  return SA_OK;
}

// 3-D tiled map: dims {d0 (contiguous), d1, d2}, byte strides of dims 1 and 2.
sa_status_t make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t d1,
                        uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2,
                        CUtensorMapSwizzle sw) {
  EncodeTiledFn enc;
  SA_TRY(get_encode(&enc));
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(SA_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d): dims %llu x %llu x %llu", (int)r,
                (unsigned long long)d0, (unsigned long long)d1, (unsigned long long)d2);
  return SA_OK;
}

inline CUtensorMapDataType map_dtype(int dtype) {
  return dtype == SA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

sa_status_t check_dtype(int dtype) {
  SA_ARG(dtype == SA_F32 || dtype == SA_BF16, "dtype must be SA_F32 (0) or SA_BF16 (1), got %d", dtype);
  return SA_OK;
}

int rmax_for(int R) { return R <= 4 ? 4 : R <= 8 ? 8 : R <= 16 ? 16 : 32; }

// ===================================================================== a1
template <typename TE>
sa_status_t launch_build_sketch(const void* k, int groups, int L, int Ls, int d, int block, float* sketch,
                                cudaStream_t st) {
  const int nb = cdiv(L, block);
  const int nb_cap = cdiv(Ls, block);
  const dim3 grid(nb, groups);
  if (d == 128)
    sa::build_sketch_kernel<TE, 128><<<grid, sa::kSketchThreads, 0, st>>>(static_cast<const TE*>(k), L, Ls, block,
                                                                           nb_cap, sketch);
  else
    sa::build_sketch_kernel<TE, 64><<<grid, sa::kSketchThreads, 0, st>>>(static_cast<const TE*>(k), L, Ls, block,
                                                                          nb_cap, sketch);
  SA_CUDA(cudaGetLastError());
  return SA_OK;
}

template <typename TE>
sa_status_t launch_append(const void* kn, const void* vn, int B, int Hkv, int T, int d, void* kc, void* vc, int Ls,
                          int pos, int block, float* sketch, cudaStream_t st) {
  const int nb_cap = cdiv(Ls, block);
  if (d == 128)
    return launch_pdl(sa::append_kv_kernel<TE, 128>, dim3(B * Hkv), dim3(sa::kSketchThreads), 0, st,
                      static_cast<const TE*>(kn), static_cast<const TE*>(vn), T, Hkv, static_cast<TE*>(kc),
                      static_cast<TE*>(vc), Ls, pos, block, nb_cap, sketch);
  return launch_pdl(sa::append_kv_kernel<TE, 64>, dim3(B * Hkv), dim3(sa::kSketchThreads), 0, st,
                    static_cast<const TE*>(kn), static_cast<const TE*>(vn), T, Hkv, static_cast<TE*>(kc),
                    static_cast<TE*>(vc), Ls, pos, block, nb_cap, sketch);
}

// ================================================================== a2 + a3
struct SelectArgs {
  int mode;
  const void* q;
  int dtype;
  const float* sketch;
  float* scores;
  int B, Tq, Hq, Hkv, d, L, Ls, block, qtile, prefill, k, frac_num, frac_den;
  float scale;
  int32_t* idx;
  int32_t* cnt;
  int kmax;
  int topdelta;  // decode sketch mode: keep candidates >= pseudo-max - delta, at most k
  float delta;
};

int max_cluster_size(const void* fn, int smem, int groups, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(16, groups);
  cfg.blockDim = dim3(sa::kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 16;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int size = 0;
  if (cudaOccupancyMaxPotentialClusterSize(&size, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 8;
  }
  return size;
}

// Co-resident clusters of cs CTAs of `threads` threads and `smem` bytes of a kernel on the
// current device (cached per device, kernel, cluster size and shared-memory size).
sa_status_t active_clusters(const void* kern, int cs, int threads, int smem, int* out) {
  struct Key {
    int dev;
    const void* kern;
    int cs, threads, smem;
  };
  static std::mutex mu;
  static std::vector<std::pair<Key, int>> cache;
  int dev = 0;
  SA_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& e : cache)
    if (e.first.dev == dev && e.first.kern == kern && e.first.cs == cs && e.first.threads == threads &&
        e.first.smem == smem) {
      *out = e.second;
      return SA_OK;
    }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, 64);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = cs;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (cache.size() > 256) cache.clear();
  cache.push_back({Key{dev, kern, cs, threads, smem}, n});
  *out = n;
  return SA_OK;
}

template <typename TE, int D, int RMAX>
sa_status_t launch_select_decode(const SelectArgs& a, const DevInfo& di, cudaStream_t st) {
  const int groups = a.B * a.Hkv;
  const int nb = cdiv(a.L, a.block);
  const int nb_cap = cdiv(a.Ls, a.block);
  auto kern = sa::select_decode_kernel<TE, D, RMAX>;
  constexpr bool kBf16 = std::is_same<TE, __nv_bfloat16>::value;
  static PerDevice max_cs_cache;  // per instantiation and device
  int max_cs = 0;
  SA_TRY(per_device(max_cs_cache, [&](int* v) -> sa_status_t {
    sa::SelDecodeLayout big{sa::sel_tile_bytes(sa::kSelTileRows, D), sa::sel_q_bytes(D, RMAX, kBf16),
                            sa::kTopkMaxN};
    SA_TRY(set_smem(kern, big.bytes()));
    cudaFuncSetAttribute(reinterpret_cast<const void*>(kern), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    *v = std::min(16, max_cluster_size(reinterpret_cast<const void*>(kern), big.bytes(), groups, st));
    return SA_OK;
  }, &max_cs));
  // about one CTA per SM in total, at most 1024 blocks per CTA
  int cs = std::min(max_cs, std::max(1, cdiv(di.sms, groups)));
  cs = std::max(cs, cdiv(nb, 1024));
  SA_SUP(cs <= max_cs, "decode selection over %d blocks needs a cluster of %d CTAs (device allows %d)", nb, cs,
         max_cs);
  cs = std::min(cs, nb);
  // whole 64-row chunks per CTA (only the group's last CTA stages a partial one)
  int per = cdiv(cdiv(nb, cs), sa::kSelChunkRows) * sa::kSelChunkRows;
  cs = cdiv(nb, per);
  int tile_rows = std::min(sa::kSelTileRows, per);
  sa::SelDecodeLayout lay{sa::sel_tile_bytes(tile_rows, D), sa::sel_q_bytes(D, RMAX, kBf16), nb};
  // smaller clusters while the groups' clusters would not all be resident at once (a second
  // wave of clusters doubles the time); never below the 1024-blocks-per-CTA limit
  const int cs_min = cdiv(nb, 1024);
  while (cs > cs_min) {
    int fit = 0;
    SA_TRY(set_smem(kern, lay.bytes()));
    SA_TRY(active_clusters(reinterpret_cast<const void*>(kern), cs, sa::kSelThreads, lay.bytes(), &fit));
    if (fit >= groups || fit == 0) break;
    const int next = std::max(cs_min, cs - 1);
    per = cdiv(cdiv(nb, next), sa::kSelChunkRows) * sa::kSelChunkRows;
    cs = cdiv(nb, per);
    tile_rows = std::min(sa::kSelTileRows, per);
    lay = sa::SelDecodeLayout{sa::sel_tile_bytes(tile_rows, D), sa::sel_q_bytes(D, RMAX, kBf16), nb};
  }
  const int smem = lay.bytes();
  SA_TRY(set_smem(kern, smem));
  CUtensorMap map;
  SA_TRY(make_map_2d(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.sketch, D, static_cast<uint64_t>(groups) * nb_cap,
                     D * 4, 32, sa::kSelChunkRows, CU_TENSOR_MAP_SWIZZLE_128B));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, groups);
  cfg.blockDim = dim3(sa::kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  SA_CUDA(cudaLaunchKernelEx(&cfg, kern, map, static_cast<const TE*>(a.q), a.Tq, a.Hq, a.Hkv, nb, nb_cap, a.scale,
                             per, tile_rows, a.k, a.scores, a.idx, a.cnt, a.kmax, a.topdelta, a.delta));
  return SA_OK;
}

template <typename TE, int D>
sa_status_t dispatch_select_decode_r(const SelectArgs& a, const DevInfo& di, cudaStream_t st) {
  const int R = (a.Hq / a.Hkv) * a.Tq;
  switch (rmax_for(R)) {
    case 4: return launch_select_decode<TE, D, 4>(a, di, st);
    case 8: return launch_select_decode<TE, D, 8>(a, di, st);
    case 16: return launch_select_decode<TE, D, 16>(a, di, st);
    default: return launch_select_decode<TE, D, 32>(a, di, st);
  }
}

sa_status_t run_select(const SelectArgs& a, cudaStream_t st) {
  DevInfo di;
  SA_TRY(dev_info(&di));
  const int groups = a.B * a.Hkv;
  const int nb = cdiv(a.L, a.block);
  if (a.mode == SA_SELECT_MASS) {
    const int nq = a.prefill ? cdiv(a.L, a.qtile) : 1;
    if (nb > sa::kTopkMaxN) {  // decode only (validated)
      // a cluster of CTAs holds the scores in shared memory, 16384 per CTA
      auto ck = sa::select_given_cluster_kernel;
      const int head = static_cast<int>(((sizeof(sa::SelClusterShared) + 15) / 16) * 16);
      static PerDevice max_cs_cl_cache;
      int max_cs_cl = 0;
      SA_TRY(per_device(max_cs_cl_cache, [&](int* v) -> sa_status_t {
        SA_TRY(set_smem(ck, head + sa::kSelClusterPer * 4));
        cudaFuncSetAttribute(reinterpret_cast<const void*>(ck), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        *v = std::min(16, max_cluster_size(reinterpret_cast<const void*>(ck), head + sa::kSelClusterPer * 4, groups,
                                           st));
        return SA_OK;
      }, &max_cs_cl));
      const int cs = cdiv(nb, sa::kSelClusterPer);
      if (cs <= max_cs_cl) {
        const int per = cdiv(nb, cs);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs, groups);
        cfg.blockDim = dim3(sa::kSelThreads);
        cfg.dynamicSmemBytes = head + per * 4;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        SA_CUDA(cudaLaunchKernelEx(&cfg, ck, static_cast<const float*>(a.scores), nb, per, a.k, a.idx, a.cnt,
                                   a.kmax));
        return SA_OK;
      }
      // longer still: one CTA per unit, scores read from global memory in every pass
      const int gsmem = static_cast<int>(sizeof(sa::TopkShared));
      sa::select_given_global_kernel<<<dim3(1, groups), sa::kSelThreads, gsmem, st>>>(a.scores, nb, a.k, a.idx,
                                                                                       a.cnt, a.kmax);
      SA_CUDA(cudaGetLastError());
      return SA_OK;
    }
    const int smem = static_cast<int>(((sizeof(sa::TopkShared) + 15) / 16) * 16) + nb * 4;
    SA_TRY(set_smem(sa::select_given_kernel, smem));
    sa::select_given_kernel<<<dim3(nq, groups), sa::kSelThreads, smem, st>>>(
        a.scores, nb, a.prefill, a.L, a.qtile, a.block, a.k, a.frac_num, a.frac_den, a.idx, a.cnt, a.kmax);
    SA_CUDA(cudaGetLastError());
    return SA_OK;
  }
  if (!a.prefill) {
    if (a.dtype == SA_F32)
      return a.d == 128 ? dispatch_select_decode_r<float, 128>(a, di, st) : dispatch_select_decode_r<float, 64>(a, di, st);
    return a.d == 128 ? dispatch_select_decode_r<__nv_bfloat16, 128>(a, di, st)
                      : dispatch_select_decode_r<__nv_bfloat16, 64>(a, di, st);
  }
  // prefill, sketch mode: tensor-core tile scoring into `scores`, then the top-k of each tile
  const int nq = cdiv(a.L, a.qtile);
  sa::ScParams p;
  p.sketch = a.sketch;
  p.scores = a.scores;
  p.L = a.L;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.groups = groups;
  p.nq = nq;
  p.nb = nb;
  p.nb_cap = cdiv(a.Ls, a.block);
  p.nc = cdiv(nq, sa::kScChunk);
  // units: (group, chunk c, M tile m <= c)
  const long long units = static_cast<long long>(groups) * p.nc * (p.nc + 1) / 2;
  SA_ARG(units < (1LL << 31), "too many tiles");
  p.units = static_cast<int>(units);
  p.scale = a.scale;
  CUtensorMap qm;
  SA_TRY(make_map_3d(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, 128, a.Hq, static_cast<uint64_t>(a.B) * a.L, 256,
                     static_cast<uint64_t>(a.Hq) * 256, 64, 1, 128, CU_TENSOR_MAP_SWIZZLE_128B));
  SA_TRY(set_smem(sa::score_prefill_kernel, sa::ScSmem::kBytes));
  const int grid = static_cast<int>(std::min<long long>(units, di.sms));
  sa::score_prefill_kernel<<<grid, sa::kScThreads, sa::ScSmem::kBytes, st>>>(qm, p);
  SA_CUDA(cudaGetLastError());
  const int smem = static_cast<int>(((sizeof(sa::TopkShared) + 15) / 16) * 16) + nb * 4;
  SA_TRY(set_smem(sa::select_given_kernel, smem));
  sa::select_given_kernel<<<dim3(nq, groups), sa::kSelThreads, smem, st>>>(
      a.scores, nb, 1, a.L, a.qtile, a.block, a.k, a.frac_num, a.frac_den, a.idx, a.cnt, a.kmax);
  SA_CUDA(cudaGetLastError());
  return SA_OK;
}

// ====================================================================== a4
struct DecodeArgs {
  const void* q;
  const void* kc;
  const void* vc;
  int dtype;
  const int32_t* idx;
  const int32_t* cnt;
  int kmax, B, T, Hq, Hkv, d, L, Ls, block;
  float scale;
  void* out;
  void* ws;
  size_t ws_bytes;
  int tok = 0;  // token mode: idx [B, kmax] single tokens shared by the kv heads of a batch row
  int qpb = 0;  // token mode, per-query prefill: B counts (batch row, query) pairs, qpb queries per batch row
};

// token mode: counters, then (CTAs + groups) <= groups * (chunks + 1) partial slots of R rows
size_t tok_ws_bytes(long long groups, int R, int d, int kmax) {
  auto up = [](size_t x) { return ((x + 255) / 256) * 256; };
  const size_t slots = static_cast<size_t>(groups) * (cdiv(kmax, sa::kDmBk) + 1);
  return up(static_cast<size_t>(groups) * 4) + up(slots * R * d * 4) + up(slots * R * 8);
}

size_t decode_ws_bytes(int groups, int R, int d, int kmax) {
  auto up = [](size_t x) { return ((x + 255) / 256) * 256; };
  // CUDA-core path: [groups][nsplit <= kmax][RMAX] partials
  const size_t rm = static_cast<size_t>(rmax_for(R));
  const size_t v1 = up(static_cast<size_t>(groups) * kmax * rm * d * 4) + up(static_cast<size_t>(groups) * kmax * rm * 8);
  // tensor-core path: arrival counters, then (CTAs + groups) <= groups * (kmax + 1)
  // partial slots of R rows
  const size_t slots = static_cast<size_t>(groups) * (kmax + 1);
  const size_t v2 = up(static_cast<size_t>(groups) * 4) + up(slots * R * d * 4) + up(slots * R * 8);
  return v1 > v2 ? v1 : v2;
}

template <int D, bool kTok>
sa_status_t launch_decode_mma(const DecodeArgs& a, const DevInfo& di, cudaStream_t st) {
  const int groups = a.B * a.Hkv;
  const int R = (a.Hq / a.Hkv) * a.T;
  const int upg = kTok ? cdiv(a.kmax, sa::kDmBk) : a.kmax;  // units per group
  const long long U = static_cast<long long>(groups) * upg;
  SA_ARG(U < (1LL << 31), "too many (group, block) units");
  // two CTAs per SM; equal contiguous ranges of units
  const long long target = static_cast<long long>(SA_DM_WAVES) * SA_DM_CTAS_PER_SM * di.sms;
  long long per = (U + target - 1) / target;
  per = std::max<long long>(per, (upg + sa::kDmMaxParts - 2) / (sa::kDmMaxParts - 1));  // <= 64 partials per group
  if (kTok) per = std::max<long long>(per, SA_DM_TOK_MIN_PER);
  per = std::min<long long>(std::max<long long>(per, 1), sa::kDmMaxList);
  const int nctas = static_cast<int>((U + per - 1) / per);
  sa::DmLayout lay{2, R, D, static_cast<int>(per), kTok ? 1 : 0};
  const int budget = (227 * 1024) / SA_DM_CTAS_PER_SM - 1024;  // the CTAs of one SM share its shared memory
  const int per_stage = lay.stage_bytes() + (kTok ? sa::kDmBk * 4 : 0);
  const int fixed = lay.bytes() - 2 * per_stage;
  lay.nstages = std::max(2, std::min(SA_DM_MAXSTAGES, (budget - fixed) / per_stage));
  const int smem = lay.bytes();
  auto kern = sa::decode_mma_kernel<D, kTok>;
  SA_TRY(set_smem(kern, smem));
  const size_t slots = static_cast<size_t>(nctas) + groups;
  auto up = [](size_t x) { return ((x + 255) / 256) * 256; };
  sa::DmParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.kc = static_cast<const __nv_bfloat16*>(a.kc);
  p.vc = static_cast<const __nv_bfloat16*>(a.vc);
  p.idx = a.idx;
  p.cnt = a.cnt;
  p.kmax = a.kmax;
  p.upg = upg;
  p.qpb = a.qpb;
  p.T = a.T;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.L = a.L;
  p.Ls = a.Ls;
  p.R = R;
  p.qscale = a.scale * 1.4426950408889634f;
  p.per = static_cast<int>(per);
  p.U = static_cast<int>(U);
  char* w = static_cast<char*>(a.ws);
  p.ctr = reinterpret_cast<int*>(w);
  p.part_o = reinterpret_cast<float*>(w + up(static_cast<size_t>(groups) * 4));
  p.part_ml = reinterpret_cast<float*>(w + up(static_cast<size_t>(groups) * 4) + up(slots * R * D * 4));
  p.nctas = nctas;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lay = lay;
  CUtensorMap km, vm;
  const uint64_t rows = static_cast<uint64_t>(a.qpb ? a.B / a.qpb * a.Hkv : groups) * a.Ls;  // the caches' rows
  SA_TRY(make_map_2d(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.kc, D, rows, D * 2, 64, sa::kDmBk,
                     CU_TENSOR_MAP_SWIZZLE_128B));
  SA_TRY(make_map_2d(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.vc, D, rows, D * 2, 64, sa::kDmBk,
                     CU_TENSOR_MAP_SWIZZLE_128B));
  return launch_pdl(kern, dim3(nctas), dim3(kTok ? sa::kDmThreadsTok : sa::kDmThreads), smem, st, km, vm, p);
}

// --------------------------------------------------- cluster decode (seldec)
// One cluster of CS CTAs per (batch, kv-head) group; with `sel`, the sketch
// scoring and the top-k run in the same kernel, in front of the attention.
struct SdArgs {
  const void* q;
  const void* kc;
  const void* vc;
  const float* sketch;  // with selection
  int32_t* idx;         // written with selection, read without
  int32_t* cnt;
  float* scores;  // optional, with selection
  void* out;
  int B, T, Hq, Hkv, d, L, Ls, k, kmax;
  float scale;
  bool sel;
  // the decode step's cache append, fused (see SdParams::k_new)
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  float* sketch_w = nullptr;
  int pos = 0;
  bool q_host = false;  // q is mapped host memory: plain loads only (see SdParams::q_host)
};

constexpr int kSdMinSmem = 120 * 1024;  // keeps the kernel at one CTA per SM

// Co-resident clusters of cs CTAs for one seldec instantiation on the current
// device (cudaOccupancyMaxActiveClusters; 0 when cs is not launchable).
template <int D, bool kSel>
sa_status_t sd_max_clusters(int cs, int* out) {
  auto kern = sa::seldec_kernel<D, kSel>;
  static std::mutex mu;
  static int cache[64][17] = {};  // per instantiation: device x cluster size, value + 1
  int dev = 0;
  SA_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64 || cs < 1 || cs > 16) return fail(SA_ERR_UNSUPPORTED, "device %d / cluster size %d", dev, cs);
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev][cs] == 0) {
    SA_TRY(set_smem(kern, 227 * 1024));
    cudaFuncSetAttribute(reinterpret_cast<const void*>(kern), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 64);
    cfg.blockDim = dim3(sa::kSdThreads);
    cfg.dynamicSmemBytes = kSdMinSmem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = cs;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kern), &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cache[dev][cs] = n + 1;
  }
  *out = cache[dev][cs] - 1;
  return SA_OK;
}

// Cluster size and cluster count: the fewest 32 KB loads per CTA (sketch chunks
// and K/V blocks, times the rounds when the groups outnumber the clusters that
// fit at once); ties go to the smaller cluster.
template <int D, bool kSel>
sa_status_t sd_shape(int groups, int nb, int kmax, int* cs_out, int* ncl_out) {
  constexpr bool sel = kSel;
  long long best = -1;
  for (int cs = 1; cs <= 16; ++cs) {
    int fit = 0;
    SA_TRY((sd_max_clusters<D, kSel>(cs, &fit)));
    if (fit < 1) continue;
    const int ncl = std::min(groups, fit);
    const long long rounds = (groups + ncl - 1) / ncl;
    const long long work = rounds * ((sel ? cdiv(cdiv(nb, cs), sa::kSdBk) : 0) + cdiv(kmax, cs));
    if (best < 0 || work < best) {
      best = work;
      *cs_out = cs;
      *ncl_out = ncl;
    }
  }
  if (best < 0) return fail(SA_ERR_UNSUPPORTED, "no launchable cluster shape for the decode kernel");
  return SA_OK;
}

template <int D, bool kSel>
sa_status_t launch_seldec(const SdArgs& a, cudaStream_t st) {
  auto kern = sa::seldec_kernel<D, kSel>;
  const int groups = a.B * a.Hkv;
  const int nb = cdiv(a.L, sa::kSdBk);
  const int nb_cap = cdiv(a.Ls, sa::kSdBk);
  int cs = 1, ncl = 1;
  SA_TRY((sd_shape<D, kSel>(groups, nb, a.kmax, &cs, &ncl)));
  const int per = cdiv(cdiv(nb, cs), sa::kSdBk) * sa::kSdBk;  // sketch rows per CTA, whole chunks
  // The ring depth must be even: each quad then always owns the same stages, so no waiter can
  // be two phases behind a stage's mbarrier (with an odd depth the two quads alternate on a
  // stage and a parity wait can pass on the wrong phase).
  sa::SdLayout lay{4, D, nb, a.kmax, kSel ? 1 : 0};
  if (lay.bytes() > 227 * 1024) lay.nstages = 2;
  static_assert(sa::kSdQuads == 2, "the ring-depth rule below assumes two consumer quads");
  if (lay.nstages % 2 != 0) return fail(SA_ERR_UNSUPPORTED, "decode ring depth %d is odd", lay.nstages);
  SA_SUP(lay.bytes() <= 227 * 1024, "decode over %d blocks needs %d bytes of shared memory", nb, lay.bytes());
  const int smem = std::max(lay.bytes(), kSdMinSmem);
  SA_TRY(set_smem(kern, smem));
  SA_CUDA(cudaFuncSetAttribute(reinterpret_cast<const void*>(kern), cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
  sa::SdParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.idx = a.idx;
  p.cnt = a.cnt;
  p.scores = a.scores;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.kmax = a.kmax;
  p.k = a.k;
  p.T = a.T;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.R = p.G * a.T;
  p.L = a.L;
  p.Ls = a.Ls;
  p.nb = nb;
  p.nb_cap = nb_cap;
  p.groups = groups;
  p.per = per;
  p.k_new = kSel ? static_cast<const __nv_bfloat16*>(a.k_new) : nullptr;
  p.v_new = kSel ? static_cast<const __nv_bfloat16*>(a.v_new) : nullptr;
  p.kc = static_cast<__nv_bfloat16*>(const_cast<void*>(a.kc));
  p.vc = static_cast<__nv_bfloat16*>(const_cast<void*>(a.vc));
  p.sketch = a.sketch_w;
  p.pos = a.pos;
  p.q_host = a.q_host ? 1 : 0;
  p.scale = a.scale;
  p.qscale = a.scale * 1.4426950408889634f;
  p.lay = lay;
  CUtensorMap km, vm, skm;
  const uint64_t rows = static_cast<uint64_t>(groups) * a.Ls;
  SA_TRY(make_map_2d(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.kc, D, rows, D * 2, 64, sa::kSdBk,
                     CU_TENSOR_MAP_SWIZZLE_128B));
  SA_TRY(make_map_2d(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.vc, D, rows, D * 2, 64, sa::kSdBk,
                     CU_TENSOR_MAP_SWIZZLE_128B));
  if (kSel)
    SA_TRY(make_map_2d(&skm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.sketch, D, static_cast<uint64_t>(groups) * nb_cap,
                       D * 4, 32, sa::kSdBk, CU_TENSOR_MAP_SWIZZLE_128B));
  else
    skm = km;  // unused
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, ncl);
  cfg.blockDim = dim3(sa::kSdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  SA_CUDA(cudaLaunchKernelEx(&cfg, kern, km, vm, skm, p));
  return SA_OK;
}

sa_status_t run_seldec(const SdArgs& a, cudaStream_t st) {
  if (a.sel) return a.d == 128 ? launch_seldec<128, true>(a, st) : launch_seldec<64, true>(a, st);
  return a.d == 128 ? launch_seldec<128, false>(a, st) : launch_seldec<64, false>(a, st);
}

// The cluster decode applies to bf16, block 64, G * T <= 16.
bool seldec_fits(int dtype, int block, int G, int T) {
  return dtype == SA_BF16 && block == sa::kSdBk && G * T <= sa::kSdRmax;
}

template <typename TE, int D, int RMAX>
sa_status_t launch_decode(const DecodeArgs& a, const DevInfo& di, cudaStream_t st) {
  using C = sa::DecodeCfg<TE, D, RMAX>;
  auto kern = sa::decode_split_kernel<TE, D, RMAX>;
  SA_TRY(set_smem(kern, C::kBytes));
  static PerDevice occ_cache;  // per instantiation and device
  int occ = 0;
  SA_TRY(per_device(occ_cache, [&](int* v) -> sa_status_t {
    SA_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, kern, sa::kDecThreads, C::kBytes));
    return SA_OK;
  }, &occ));
  const int groups = a.B * a.Hkv;
  const int target = di.sms * occ;
  int nsplit = std::max(1, std::min(a.kmax, target / std::max(groups, 1)));
  const int chunk = cdiv(a.kmax, nsplit);
  nsplit = cdiv(a.kmax, chunk);
  const size_t o_bytes = ((static_cast<size_t>(groups) * a.kmax * RMAX * D * 4 + 255) / 256) * 256;
  float* ws_o = static_cast<float*>(a.ws);
  float* ws_ml = reinterpret_cast<float*>(static_cast<char*>(a.ws) + o_bytes);
  CUtensorMap km, vm;
  const uint64_t rows = static_cast<uint64_t>(groups) * a.Ls;
  SA_TRY(make_map_2d(&km, map_dtype(a.dtype), a.kc, D, rows, D * sizeof(TE), C::EPB, sa::kDecBk,
                     CU_TENSOR_MAP_SWIZZLE_128B));
  SA_TRY(make_map_2d(&vm, map_dtype(a.dtype), a.vc, D, rows, D * sizeof(TE), C::EPB, sa::kDecBk,
                     CU_TENSOR_MAP_SWIZZLE_128B));
  const float qscale = a.scale * 1.4426950408889634f;
  kern<<<dim3(nsplit, groups), sa::kDecThreads, C::kBytes, st>>>(km, vm, static_cast<const TE*>(a.q), a.idx, a.cnt,
                                                                 a.kmax, a.T, a.Hq, a.Hkv, a.L, a.Ls, qscale, chunk,
                                                                 nsplit, ws_o, ws_ml);
  SA_CUDA(cudaGetLastError());
  sa::decode_combine_kernel<TE, D, RMAX><<<groups, sa::kDecThreads, 0, st>>>(ws_o, ws_ml, nsplit, a.T, a.Hq, a.Hkv,
                                                                            static_cast<TE*>(a.out));
  SA_CUDA(cudaGetLastError());
  return SA_OK;
}

template <typename TE, int D>
sa_status_t dispatch_decode_r(const DecodeArgs& a, const DevInfo& di, cudaStream_t st) {
  switch (rmax_for((a.Hq / a.Hkv) * a.T)) {
    case 4: return launch_decode<TE, D, 4>(a, di, st);
    case 8: return launch_decode<TE, D, 8>(a, di, st);
    case 16: return launch_decode<TE, D, 16>(a, di, st);
    default: return launch_decode<TE, D, 32>(a, di, st);
  }
}

sa_status_t run_decode(const DecodeArgs& a, cudaStream_t st) {
  DevInfo di;
  SA_TRY(dev_info(&di));
  if (a.tok) return a.d == 128 ? launch_decode_mma<128, true>(a, di, st) : launch_decode_mma<64, true>(a, di, st);
  // few groups: one cluster per group, merged through distributed shared memory;
  // many groups: equal contiguous ranges of (group, block) units over all SMs
  if (seldec_fits(a.dtype, a.block, a.Hq / a.Hkv, a.T) && 2 * a.B * a.Hkv <= di.sms) {
    const SdArgs sd{a.q, a.kc, a.vc, nullptr, const_cast<int32_t*>(a.idx), const_cast<int32_t*>(a.cnt), nullptr,
                    a.out, a.B, a.T, a.Hq, a.Hkv, a.d, a.L, a.Ls, 0, a.kmax, a.scale, false};
    return run_seldec(sd, st);
  }
  if (a.dtype == SA_BF16 && (a.Hq / a.Hkv) * a.T <= 16)
    return a.d == 128 ? launch_decode_mma<128, false>(a, di, st) : launch_decode_mma<64, false>(a, di, st);
  if (a.dtype == SA_F32)
    return a.d == 128 ? dispatch_decode_r<float, 128>(a, di, st) : dispatch_decode_r<float, 64>(a, di, st);
  return a.d == 128 ? dispatch_decode_r<__nv_bfloat16, 128>(a, di, st) : dispatch_decode_r<__nv_bfloat16, 64>(a, di, st);
}

// ------------------------------------------------------------ validation
sa_status_t check_common(int dtype, int B, int Hq, int Hkv, int d) {
  SA_TRY(check_dtype(dtype));
  SA_ARG(B >= 1 && Hq >= 1 && Hkv >= 1, "B, Hq, Hkv must be >= 1 (got %d, %d, %d)", B, Hq, Hkv);
  SA_ARG(Hq % Hkv == 0, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  SA_ARG(static_cast<long long>(B) * Hkv <= 65535, "B*Hkv must be <= 65535");
  SA_SUP(d == 64 || d == 128, "head dim d must be 64 or 128, got %d", d);
  return SA_OK;
}

sa_status_t validate_decode(const DecodeArgs& a) {
  SA_TRY(check_common(a.dtype, a.qpb ? a.B / a.qpb : a.B, a.Hq, a.Hkv, a.d));
  SA_ARG(a.q && a.kc && a.vc && a.idx && a.cnt && a.out, "null pointer argument");
  SA_ARG(a.T >= 1, "T must be >= 1");
  SA_ARG(a.L >= 1 && a.L <= a.Ls, "need 1 <= L (%d) <= L_stride (%d)", a.L, a.Ls);
  if (a.tok) {
    SA_SUP(a.dtype == SA_BF16, "token decode supports bf16 only");
    SA_SUP((a.Hq / a.Hkv) * a.T <= 16, "token decode: G*T (%d) must be <= 16", (a.Hq / a.Hkv) * a.T);
    SA_ARG(a.T <= a.L, "T (%d) must be <= L", a.T);
  } else {
    SA_SUP(a.block == sa::kDecBk, "decode supports block == %d, got %d", sa::kDecBk, a.block);
    SA_ARG(a.T <= a.block && a.T <= a.L, "T (%d) must be <= block and <= L", a.T);
    SA_SUP((a.Hq / a.Hkv) * a.T <= 32, "G*T (%d) must be <= 32", (a.Hq / a.Hkv) * a.T);
  }
  SA_ARG(a.kmax >= 1, "kmax must be >= 1");
  SA_ARG(aligned16(a.kc) && aligned16(a.vc) && aligned16(a.q), "q and the k/v caches must be 16-byte aligned");
  SA_ARG(static_cast<long long>(a.qpb ? a.B / a.qpb : a.B) * a.Hkv * a.Ls < (1LL << 31), "B*Hkv*L_stride too large");
  SA_ARG(a.ws && aligned16(a.ws), "workspace must be a 16-byte-aligned device pointer");
  const size_t need = a.tok ? tok_ws_bytes(static_cast<long long>(a.B) * a.Hkv, (a.Hq / a.Hkv) * a.T, a.d, a.kmax)
                            : decode_ws_bytes(a.B * a.Hkv, (a.Hq / a.Hkv) * a.T, a.d, a.kmax);
  SA_ARG(a.ws_bytes >= need, "workspace too small: %zu < %zu bytes", a.ws_bytes, need);
  return SA_OK;
}

int select_kmax(int L, int block, int qtile, int prefill, int k, int frac_num, int frac_den) {
  if (L < 1 || block < 1 || k < 0 || (prefill && qtile < 1) || frac_num < 0 || (frac_num > 0 && frac_den < 1))
    return -1;
  const int nb = cdiv(L, block);
  if (!prefill) return (nb >= 2 ? 2 : 1) + std::min(k, std::max(nb - 2, 0));
  const int nq = cdiv(L, qtile);
  int best = 0;
  for (int i = 0; i < nq; ++i) {
    const int last = std::min((i + 1) * qtile, L) - 1;
    const int c = last / block + 1;
    const long long bud = k + (frac_num > 0 ? (static_cast<long long>(frac_num) * c + frac_den - 1) / frac_den : 0);
    const int forced = c >= 2 ? 2 : 1;
    const int take = static_cast<int>(std::min<long long>(bud, c - forced));
    best = std::max(best, forced + take);
  }
  return best;
}

sa_status_t validate_select(const SelectArgs& a) {
  SA_ARG(a.mode == SA_SELECT_SKETCH || a.mode == SA_SELECT_MASS, "mode must be SA_SELECT_SKETCH or SA_SELECT_MASS");
  SA_ARG(a.B >= 1 && a.Hq >= 1 && a.Hkv >= 1 && a.Hq % a.Hkv == 0, "bad head counts");
  SA_ARG(a.idx && a.cnt, "idx and cnt are required");
  SA_ARG(a.L >= 1 && a.L <= a.Ls, "need 1 <= L <= L_stride");
  SA_ARG(a.block >= 1 && a.k >= 0, "block >= 1 and k >= 0 required");
  SA_ARG(a.frac_num >= 0 && (a.frac_num == 0 || a.frac_den >= 1), "bad budget fraction");
  const int need = select_kmax(a.L, a.block, a.qtile, a.prefill, a.k, a.frac_num, a.frac_den);
  SA_ARG(need >= 1, "bad selection parameters");
  SA_ARG(a.kmax >= need, "kmax (%d) too small: the selection needs %d", a.kmax, need);
  const int nb = cdiv(a.L, a.block);
  if (a.mode == SA_SELECT_MASS && !a.prefill)  // given decode scores: any length (long ones are read from L2)
    SA_ARG(static_cast<long long>(a.B) * a.Hkv * nb < (1LL << 40), "score array too large");
  else
    SA_SUP(nb <= sa::kTopkMaxN, "at most %d blocks per sequence (got %d)", sa::kTopkMaxN, nb);
  if (a.prefill) SA_ARG(a.qtile >= 1 && a.Tq == a.L, "prefill: qtile >= 1 and Tq == L required");
  if (a.mode == SA_SELECT_MASS) {
    SA_ARG(a.scores != nullptr, "MASS mode needs the scores array");
    return SA_OK;
  }
  SA_TRY(check_common(a.dtype, a.B, a.Hq, a.Hkv, a.d));
  SA_ARG(a.q && a.sketch, "SKETCH mode needs q and sketch");
  SA_ARG(aligned16(a.sketch), "sketch must be 16-byte aligned");
  if (!a.prefill) {
    SA_ARG(a.Tq >= 1, "Tq must be >= 1");
    SA_ARG(a.dtype != SA_BF16 || aligned16(a.q), "bf16 q must be 16-byte aligned");
    SA_SUP((a.Hq / a.Hkv) * a.Tq <= 32, "G*Tq (%d) must be <= 32 for decode selection", (a.Hq / a.Hkv) * a.Tq);
  } else {
    SA_SUP(a.dtype == SA_BF16 && a.d == 128 && a.qtile == 128 && a.block == 128,
           "prefill sketch selection supports bf16 queries, d == 128, qtile == block == 128");
    SA_ARG(a.scores != nullptr, "prefill sketch selection needs the scores array (it is written)");
    SA_ARG(aligned16(a.q), "q must be 16-byte aligned");
    SA_ARG(a.scale > 0.f && a.scale < 1e30f, "scale must be positive and finite");
    SA_ARG(static_cast<long long>(a.B) * a.L * a.Hq < (1LL << 31), "B*L*Hq must be < 2^31");
  }
  return SA_OK;
}

// ---------------------------------------------------------- prefill / mass
sa_status_t prefill_impl(const void* q, const void* k, const void* v, const int32_t* idx, const int32_t* cnt,
                         int kmax, int B, int L, int Hq, int Hkv, float scale, void* out, float* lse,
                         cudaStream_t st, const uint32_t* tokmask = nullptr, int wpr = 0) {
  DevInfo di;
  SA_TRY(dev_info(&di));
  constexpr int D = 128;
  sa::PfParams p;
  p.idx = idx;
  p.cnt = cnt;
  p.kmax = kmax;
  p.tokmask = tokmask;
  p.wpr = wpr;
  p.L = L;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.groups = B * Hkv;
  p.nq = cdiv(L, sa::kPfRows);
  p.nb = cdiv(L, sa::kPfKeys);
  p.npairs = cdiv(p.G, 2);
  const long long units = static_cast<long long>(p.groups) * p.nq * p.npairs;
  SA_ARG(units < (1LL << 31), "too many prefill work units");
  p.units = static_cast<int>(units);
  p.qscale = scale * 1.4426950408889634f;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  CUtensorMap qm, km, vm;
  SA_TRY(make_map_3d(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, D, Hq, static_cast<uint64_t>(B) * L, D * 2,
                     static_cast<uint64_t>(Hq) * D * 2, 64, 1, sa::kPfRows, CU_TENSOR_MAP_SWIZZLE_128B));
  const uint64_t rows = static_cast<uint64_t>(B) * Hkv * L;
  SA_TRY(make_map_2d(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k, D, rows, D * 2, 64, sa::kPfKeys,
                     CU_TENSOR_MAP_SWIZZLE_128B));
  SA_TRY(make_map_2d(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v, D, rows, D * 2, 64, sa::kPfKeys,
                     CU_TENSOR_MAP_SWIZZLE_128B));
  const int grid = static_cast<int>(std::min<long long>(units, di.sms));
  if (tokmask) {
    SA_TRY(set_smem(sa::prefill_kernel<true>, sa::PfSmem::kBytes));
    sa::prefill_kernel<true><<<grid, sa::kPfThreads, sa::PfSmem::kBytes, st>>>(qm, km, vm, p);
  } else {
    SA_TRY(set_smem(sa::prefill_kernel<false>, sa::PfSmem::kBytes));
    sa::prefill_kernel<false><<<grid, sa::kPfThreads, sa::PfSmem::kBytes, st>>>(qm, km, vm, p);
  }
  SA_CUDA(cudaGetLastError());
  return SA_OK;
}
size_t mass_ws_bytes(int, int, int, int, int, int) { return 0; }

sa_status_t mass_impl(const void* q, const void* k, int B, int L, int Hq, int Hkv, float scale, float* mass,
                      cudaStream_t st) {
  DevInfo di;
  SA_TRY(dev_info(&di));
  constexpr int D = 128;
  sa::MsParams p;
  p.L = L;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.groups = B * Hkv;
  p.nq = cdiv(L, sa::kPfRows);
  p.nb = cdiv(L, sa::kPfKeys);
  p.npairs = cdiv(p.G, 2);
  SA_SUP(p.nb <= sa::kMsMaxBlocks, "oracle mass supports at most %d key blocks (L <= %d)", sa::kMsMaxBlocks,
         sa::kMsMaxBlocks * sa::kPfKeys);
  const long long units = static_cast<long long>(p.groups) * p.nq;
  SA_ARG(units < (1LL << 31), "too many work units");
  p.units = static_cast<int>(units);
  p.qscale = scale * 1.4426950408889634f;
  p.mass = mass;
  CUtensorMap qm, km;
  SA_TRY(make_map_3d(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, D, Hq, static_cast<uint64_t>(B) * L, D * 2,
                     static_cast<uint64_t>(Hq) * D * 2, 64, 1, sa::kPfRows, CU_TENSOR_MAP_SWIZZLE_128B));
  SA_TRY(make_map_2d(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k, D, static_cast<uint64_t>(B) * Hkv * L, D * 2, 64,
                     sa::kPfKeys, CU_TENSOR_MAP_SWIZZLE_128B));
  const int smem = sa::MsSmem::bytes(p.nb);
  SA_TRY(set_smem(sa::mass_kernel, smem));
  const int grid = static_cast<int>(std::min<long long>(units, di.sms));
  sa::mass_kernel<<<grid, sa::kMsThreads, smem, st>>>(qm, km, p);
  SA_CUDA(cudaGetLastError());
  return SA_OK;
}

}  // namespace

// ========================================================================= ABI
// ------------------------------------------------ head-collapsed token mass (decode)
namespace {

struct TokMassWs {
  size_t logits, part, lse, total;
};

// logits [groups][R][L] f32 | partials [groups][nparts][R] float2 | lse [groups][R] f32, with
// nparts = ceil(L / (kTmWarps * kpw)) <= ceil(L / (kTmWarps * 32)) (one per CTA; kpw >= 32)
TokMassWs tokmass_ws(int B, int T, int Hq, int Hkv, int L) {
  auto up = [](size_t x) { return ((x + 255) / 256) * 256; };
  const size_t groups = static_cast<size_t>(B) * Hkv, R = static_cast<size_t>(Hq / Hkv) * T;
  TokMassWs w;
  w.logits = 0;
  w.part = up(groups * R * L * 4);
  const size_t nparts_max = static_cast<size_t>(cdiv(L, sa::kTmWarps * 32));
  w.lse = w.part + up(groups * nparts_max * R * 8);
  w.total = w.lse + up(groups * R * 4);
  return w;
}

template <int D>
sa_status_t launch_token_mass(const void* q, const void* kc, int B, int T, int Hq, int Hkv, int L, int Ls, float scale,
                              float* mass, void* ws, const DevInfo& di, cudaStream_t st, bool per_query) {
  const int groups = B * Hkv, R = (Hq / Hkv) * T;
  const int rtiles = cdiv(R, 16);
  const TokMassWs w = tokmass_ws(B, T, Hq, Hkv, L);
  char* base = static_cast<char*>(ws);
  float* logits = reinterpret_cast<float*>(base + w.logits);
  float2* part = reinterpret_cast<float2*>(base + w.part);
  float* lse2 = reinterpret_cast<float*>(base + w.lse);
  // about four CTAs of kTmThreads per SM over all groups; warp ranges of a multiple of 32 keys
  const long long keys = static_cast<long long>(L) * groups * rtiles;
  const long long want = static_cast<long long>(di.sms) * 4 * sa::kTmWarps;
  int kpw = static_cast<int>(std::max<long long>(32, ((keys + want - 1) / want + 31) / 32 * 32));
  kpw = std::min(kpw, std::max(32, (cdiv(L, sa::kTmWarps) + 31) / 32 * 32));  // every warp of a CTA gets keys
  const int nchunk = cdiv(L, sa::kTmWarps * kpw);  // one partial per CTA and row: fits the workspace (kpw >= 32)
  sa::token_logits_kernel<D><<<dim3(nchunk, groups, rtiles), sa::kTmThreads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(kc), T, Hq, Hkv, L, Ls,
      scale * 1.4426950408889634f, kpw, per_query ? 0 : 1, logits, part);
  SA_CUDA(cudaGetLastError());
  sa::token_lse_kernel<<<dim3(groups, rtiles), 16 * 32, 0, st>>>(part, nchunk, R, lse2);
  SA_CUDA(cudaGetLastError());
  if (per_query)
    sa::token_mass_rows_kernel<<<dim3(cdiv(L, 4 * sa::kTmThreads), L, B), sa::kTmThreads, 0, st>>>(
        logits, lse2, Hkv, Hq / Hkv, L, 1.f / static_cast<float>(Hq), mass);
  else
    sa::token_mass_kernel<<<dim3(cdiv(L, 4 * sa::kTmThreads), B), sa::kTmThreads, 0, st>>>(
        logits, lse2, Hkv, R, L, 1.f / static_cast<float>(Hq * T), mass);
  SA_CUDA(cudaGetLastError());
  return SA_OK;
}

}  // namespace

// ------------------------------------------------ one decode step (a1 + a2 + a3 + a4)
namespace {

struct StepArgs {
  const void* q;
  const void* k_new;
  const void* v_new;
  int dtype;
  void* k_cache;
  void* v_cache;
  float* sketch;
  int B, T, Hq, Hkv, d, L, L_stride, block, k;
  float scale;
  int32_t* idx;
  int32_t* cnt;
  int kmax;
  float* scores;
  void* out;
  int host_io;
  void* workspace;
  size_t ws_bytes;
};

using StepKey = std::array<uint64_t, 26>;

StepKey step_key(const StepArgs& a, int dev) {
  auto P = [](const void* p) { return static_cast<uint64_t>(reinterpret_cast<uintptr_t>(p)); };
  uint32_t sc;
  std::memcpy(&sc, &a.scale, 4);
  return StepKey{P(a.q), P(a.k_new), P(a.v_new), static_cast<uint64_t>(a.dtype), P(a.k_cache), P(a.v_cache),
                 P(a.sketch), static_cast<uint64_t>(a.B), static_cast<uint64_t>(a.T), static_cast<uint64_t>(a.Hq),
                 static_cast<uint64_t>(a.Hkv), static_cast<uint64_t>(a.d), static_cast<uint64_t>(a.L),
                 static_cast<uint64_t>(a.L_stride), static_cast<uint64_t>(a.block), static_cast<uint64_t>(a.k), sc,
                 P(a.idx), P(a.cnt), static_cast<uint64_t>(a.kmax), P(a.scores), P(a.out),
                 static_cast<uint64_t>(a.host_io), P(a.workspace), static_cast<uint64_t>(a.ws_bytes),
                 static_cast<uint64_t>(dev)};
}

struct StepGraph {
  StepKey key;
  cudaGraphExec_t exec;
  uint64_t last_use;
};

constexpr size_t kStepCacheMax = 32;
std::mutex g_step_mu;
std::vector<StepGraph> g_step_cache;
std::vector<StepKey> g_step_seen;  // argument sets seen once (captured the second time)
uint64_t g_step_clock = 0;

}  // namespace

extern "C" {

int sa_version(void) { return 100; }

const char* sa_last_error(void) { return t_err.c_str(); }

const char* sa_status_name(int s) {
  switch (s) {
    case SA_OK: return "SA_OK";
    case SA_ERR_INVALID_ARG: return "SA_ERR_INVALID_ARG";
    case SA_ERR_UNSUPPORTED: return "SA_ERR_UNSUPPORTED";
    case SA_ERR_CUDA: return "SA_ERR_CUDA";
    case SA_ERR_TIMEOUT: return "SA_ERR_TIMEOUT";
    default: return "SA_UNKNOWN_STATUS";
  }
}

sa_status_t sa_selftest_wait_timeout(long long limit_ns, void* stream) {
  t_err.clear();
  SA_ARG(limit_ns >= 1000000 && limit_ns <= 1000000000LL, "limit_ns must be in [1e6, 1e9]");
  sa::selftest_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(static_cast<unsigned long long>(limit_ns));
  SA_CUDA(cudaGetLastError());
  return SA_OK;
}

sa_status_t sa_device_status(int* code, int clear) {
  SA_ARG(code != nullptr, "code must not be NULL");
  SA_CUDA(cudaDeviceSynchronize());
  int v = 0;
  SA_CUDA(cudaMemcpyFromSymbol(&v, sa::g_device_status, sizeof(int)));
  *code = v;
  if (clear) {
    const int zero = 0;
    SA_CUDA(cudaMemcpyToSymbol(sa::g_device_status, &zero, sizeof(int)));
  }
  return SA_OK;
}

sa_status_t sa_build_sketch(const void* k, int dtype, int B, int Hkv, int L, int L_stride, int d, int block,
                            float* sketch, void* stream) {
  t_err.clear();
  SA_TRY(check_common(dtype, B, Hkv, Hkv, d));
  SA_ARG(k && sketch, "null pointer argument");
  SA_ARG(L >= 1 && L <= L_stride, "need 1 <= L (%d) <= L_stride (%d)", L, L_stride);
  SA_ARG(block >= 1 && block <= 1024, "block must be in [1, 1024]");
  SA_ARG(aligned16(k) && aligned16(sketch), "k and sketch must be 16-byte aligned");
  DevInfo di;
  SA_TRY(dev_info(&di));
  if (dtype == SA_F32) return launch_build_sketch<float>(k, B * Hkv, L, L_stride, d, block, sketch, as_stream(stream));
  return launch_build_sketch<__nv_bfloat16>(k, B * Hkv, L, L_stride, d, block, sketch, as_stream(stream));
}

sa_status_t sa_append_kv(const void* k_new, const void* v_new, int dtype, int B, int Hkv, int T, int d,
                         void* k_cache, void* v_cache, int L_stride, int pos, int block, float* sketch,
                         void* stream) {
  t_err.clear();
  SA_TRY(check_common(dtype, B, Hkv, Hkv, d));
  SA_ARG(k_new && v_new && k_cache && v_cache && sketch, "null pointer argument");
  SA_ARG(T >= 1 && pos >= 0 && static_cast<long long>(pos) + T <= L_stride, "need T >= 1, 0 <= pos, pos+T <= L_stride");
  SA_ARG(block >= 1 && block <= 1024, "block must be in [1, 1024]");
  SA_ARG(aligned16(k_new) && aligned16(v_new) && aligned16(k_cache) && aligned16(v_cache) && aligned16(sketch),
         "pointers must be 16-byte aligned");
  DevInfo di;
  SA_TRY(dev_info(&di));
  if (dtype == SA_F32)
    return launch_append<float>(k_new, v_new, B, Hkv, T, d, k_cache, v_cache, L_stride, pos, block, sketch,
                                as_stream(stream));
  return launch_append<__nv_bfloat16>(k_new, v_new, B, Hkv, T, d, k_cache, v_cache, L_stride, pos, block, sketch,
                                      as_stream(stream));
}

int sa_budget_sublinear(int L, int block, int k_ref, int L_ref, float exponent) {
  if (L < 1 || block < 1 || k_ref < 0 || L_ref < 1 || !(exponent >= 0.f && exponent <= 1.f)) return -1;
  const int nb = cdiv(L, block);
  const double k = std::ceil(static_cast<double>(k_ref) * std::pow(static_cast<double>(L) / L_ref, exponent) - 1e-9);
  const double cap = std::max(nb - 2, 0);
  return static_cast<int>(std::min(std::max(k, 0.0), cap));
}

int sa_select_kmax(int L, int block, int qtile, int prefill, int k, int frac_num, int frac_den) {
  return select_kmax(L, block, qtile, prefill, k, frac_num, frac_den);
}

}  // extern "C"

namespace {

// The fused selection + decode, optionally with the decode step's cache append in front (k_new
// and v_new [B, T, Hkv, d], written at rows L - T .. L - 1; the caller checks that the rows lie in
// the local block and that no scores are returned, and the sketch is then writable).
sa_status_t select_decode_impl(const void* q, int dtype, const float* sketch, const void* k_cache,
                               const void* v_cache, int B, int T, int Hq, int Hkv, int d, int L, int L_stride,
                               int block, int k, float scale, int32_t* idx, int32_t* cnt, int kmax, float* scores,
                               void* out, const void* k_new, const void* v_new, cudaStream_t st,
                               bool q_host = false) {
  SelectArgs sel{SA_SELECT_SKETCH, q, dtype, sketch, scores, B, T, Hq, Hkv, d, L, L_stride, block, 0, 0, k,
                 0, 1, scale, idx, cnt, kmax};
  SA_TRY(validate_select(sel));
  SA_SUP(seldec_fits(dtype, block, Hq / Hkv, T),
         "fused selection + decode supports bf16, block == %d and G*T <= %d (got dtype %d, block %d, G*T %d)",
         sa::kSdBk, sa::kSdRmax, dtype, block, (Hq / Hkv) * T);
  SA_ARG(k_cache && v_cache && out, "null pointer argument");
  SA_ARG(aligned16(k_cache) && aligned16(v_cache) && aligned16(out), "k/v caches and out must be 16-byte aligned");
  SA_ARG(T <= block && T <= L, "T (%d) must be <= block and <= L", T);
  SA_ARG(static_cast<long long>(B) * Hkv * L_stride < (1LL << 31), "B*Hkv*L_stride too large");
  SA_ARG(scale > 0.f && scale < 1e30f, "scale must be positive and finite");
  if (k_new) {
    SA_ARG(v_new && aligned16(k_new) && aligned16(v_new), "k_new and v_new must be 16-byte aligned");
    SA_ARG((L - T) / block == (L - 1) / block && scores == nullptr, "fused append needs one local block, no scores");
  }
  DevInfo di;
  SA_TRY(dev_info(&di));
  SdArgs a{q, k_cache, v_cache, sketch, idx, cnt, scores, out, B, T, Hq, Hkv, d, L, L_stride, k, kmax, scale, true};
  a.k_new = k_new;
  a.v_new = v_new;
  a.sketch_w = const_cast<float*>(sketch);
  a.pos = L - T;
  a.q_host = q_host;
  return run_seldec(a, st);
}

}  // namespace

extern "C" {

sa_status_t sa_select_topk(int mode, const void* q, int dtype, const float* sketch, float* scores, int B, int Tq,
                           int Hq, int Hkv, int d, int L, int L_stride, int block, int qtile, int prefill, int k,
                           int frac_num, int frac_den, float scale, int32_t* idx, int32_t* cnt, int kmax,
                           void* stream) {
  t_err.clear();
  SelectArgs a{mode, q, dtype, sketch, scores, B, Tq, Hq, Hkv, d, L, L_stride, block, qtile, prefill ? 1 : 0, k,
               frac_num, frac_den, scale, idx, cnt, kmax};
  SA_TRY(validate_select(a));
  return run_select(a, as_stream(stream));
}

sa_status_t sa_select_topdelta(const void* q, int dtype, const float* sketch, float* scores, int B, int Tq, int Hq,
                               int Hkv, int d, int L, int L_stride, int block, float delta, int cap, float scale,
                               int32_t* idx, int32_t* cnt, int kmax, void* stream) {
  t_err.clear();
  SA_ARG(delta >= 0.f && delta < 1e30f, "delta must be >= 0 and finite");
  SA_ARG(cap >= 0, "cap must be >= 0");
  SelectArgs a{SA_SELECT_SKETCH, q, dtype, sketch, scores, B, Tq, Hq, Hkv, d, L, L_stride, block, 0, 0, cap,
               0, 1, scale, idx, cnt, kmax, 1, delta};
  SA_TRY(validate_select(a));
  return run_select(a, as_stream(stream));
}

size_t sa_decode_workspace_bytes(int B, int T, int Hq, int Hkv, int d, int kmax) {
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || kmax < 1 || d < 1) return 0;
  return decode_ws_bytes(B * Hkv, (Hq / Hkv) * T, d, kmax);
}

sa_status_t sa_decode(const void* q, const void* k_cache, const void* v_cache, int dtype, const int32_t* idx,
                      const int32_t* cnt, int kmax, int B, int T, int Hq, int Hkv, int d, int L, int L_stride,
                      int block, float scale, void* out, void* workspace, size_t ws_bytes, void* stream) {
  t_err.clear();
  DecodeArgs a{q, k_cache, v_cache, dtype, idx, cnt, kmax, B, T, Hq, Hkv, d, L, L_stride, block, scale, out,
               workspace, ws_bytes};
  SA_TRY(validate_decode(a));
  return run_decode(a, as_stream(stream));
}

sa_status_t sa_select_decode(const void* q, int dtype, const float* sketch, const void* k_cache, const void* v_cache,
                             int B, int T, int Hq, int Hkv, int d, int L, int L_stride, int block, int k, float scale,
                             int32_t* idx, int32_t* cnt, int kmax, float* scores, void* out, void* stream) {
  t_err.clear();
  return select_decode_impl(q, dtype, sketch, k_cache, v_cache, B, T, Hq, Hkv, d, L, L_stride, block, k, scale, idx,
                            cnt, kmax, scores, out, nullptr, nullptr, as_stream(stream));
}

sa_status_t sa_decode_tokens(const void* q, const void* k_cache, const void* v_cache, int dtype, const int32_t* idx,
                             const int32_t* cnt, int kmax, int B, int T, int Hq, int Hkv, int d, int L, int L_stride,
                             float scale, void* out, void* workspace, size_t ws_bytes, void* stream) {
  t_err.clear();
  DecodeArgs a{q, k_cache, v_cache, dtype, idx, cnt, kmax, B, T, Hq, Hkv, d, L, L_stride, 1, scale, out,
               workspace, ws_bytes, 1};
  SA_TRY(validate_decode(a));
  return run_decode(a, as_stream(stream));
}

sa_status_t sa_prefill(const void* q, const void* k, const void* v, int dtype, const int32_t* idx, const int32_t* cnt,
                       int kmax, int B, int L, int Hq, int Hkv, int d, int qtile, int block, float scale, void* out,
                       float* lse_out, void* stream) {
  t_err.clear();
  SA_TRY(check_common(dtype, B, Hq, Hkv, d));
  SA_ARG(q && k && v && idx && cnt && out, "null pointer argument");
  SA_ARG(L >= 1 && kmax >= 1, "L >= 1 and kmax >= 1 required");
  SA_SUP(dtype == SA_BF16 && d == 128 && qtile == 128 && block == 128,
         "prefill supports bf16, d == 128, qtile == block == 128");
  SA_ARG(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out), "q, k, v, out must be 16-byte aligned");
  SA_ARG(scale > 0.f && scale < 1e30f, "scale must be positive and finite");
  SA_ARG(static_cast<long long>(B) * L * Hq < (1LL << 31) && static_cast<long long>(B) * Hkv * L < (1LL << 31),
         "B*L*Hq and B*Hkv*L must be < 2^31");
  return prefill_impl(q, k, v, idx, cnt, kmax, B, L, Hq, Hkv, scale, out, lse_out, as_stream(stream));
}


size_t sa_token_mass_workspace_bytes(int B, int T, int Hq, int Hkv, int L) {
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || L < 1) return 0;
  return tokmass_ws(B, T, Hq, Hkv, L).total;
}

sa_status_t sa_token_mass_decode(const void* q, const void* k_cache, int dtype, int B, int T, int Hq, int Hkv, int d,
                                 int L, int L_stride, float scale, float* mass, void* workspace, size_t ws_bytes,
                                 void* stream) {
  t_err.clear();
  SA_TRY(check_common(dtype, B, Hq, Hkv, d));
  SA_SUP(dtype == SA_BF16, "token mass supports bf16 only");
  SA_ARG(q && k_cache && mass && workspace, "null pointer argument");
  SA_ARG(T >= 1 && L >= T && L <= L_stride, "need 1 <= T <= L <= L_stride");
  SA_SUP((Hq / Hkv) * T <= 16, "token mass: G*T (%d) must be <= 16", (Hq / Hkv) * T);
  SA_ARG(aligned16(q) && aligned16(k_cache) && aligned16(mass) && aligned16(workspace),
         "q, k_cache, mass and workspace must be 16-byte aligned");
  SA_ARG(static_cast<long long>(B) * Hkv * L_stride < (1LL << 31), "B*Hkv*L_stride too large");
  SA_ARG(ws_bytes >= tokmass_ws(B, T, Hq, Hkv, L).total, "workspace too small: %zu < %zu bytes", ws_bytes,
         tokmass_ws(B, T, Hq, Hkv, L).total);
  DevInfo di;
  SA_TRY(dev_info(&di));
  cudaStream_t st = as_stream(stream);
  return d == 128 ? launch_token_mass<128>(q, k_cache, B, T, Hq, Hkv, L, L_stride, scale, mass, workspace, di, st, false)
                  : launch_token_mass<64>(q, k_cache, B, T, Hq, Hkv, L, L_stride, scale, mass, workspace, di, st, false);
}

size_t sa_token_mass_prefill_workspace_bytes(int B, int L, int Hq, int Hkv) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || L < 1) return 0;
  return tokmass_ws(B, L, Hq, Hkv, L).total;
}

sa_status_t sa_token_mass_prefill(const void* q, const void* k, int dtype, int B, int L, int Hq, int Hkv, int d,
                                  float scale, float* mass, void* workspace, size_t ws_bytes, void* stream) {
  t_err.clear();
  SA_TRY(check_common(dtype, B, Hq, Hkv, d));
  SA_SUP(dtype == SA_BF16, "token mass supports bf16 only");
  SA_ARG(q && k && mass && workspace, "null pointer argument");
  SA_ARG(L >= 1 && L <= 65535, "need 1 <= L <= 65535");
  SA_ARG(aligned16(q) && aligned16(k) && aligned16(mass) && aligned16(workspace),
         "q, k, mass and workspace must be 16-byte aligned");
  SA_ARG(static_cast<long long>(B) * Hkv * L < (1LL << 31), "B*Hkv*L too large");
  SA_ARG(ws_bytes >= tokmass_ws(B, L, Hq, Hkv, L).total, "workspace too small: %zu < %zu bytes", ws_bytes,
         tokmass_ws(B, L, Hq, Hkv, L).total);
  DevInfo di;
  SA_TRY(dev_info(&di));
  cudaStream_t st = as_stream(stream);
  return d == 128 ? launch_token_mass<128>(q, k, B, L, Hq, Hkv, L, L, scale, mass, workspace, di, st, true)
                  : launch_token_mass<64>(q, k, B, L, Hq, Hkv, L, L, scale, mass, workspace, di, st, true);
}

}  // extern "C"

namespace {

// The per-query token prefill runs on the tensor-core prefill kernel when its shape allows
// (bf16, d = 128, L <= kTokPfMaxL): every query's support becomes a bit mask row, and each
// 128-query tile attends over the 128-key blocks holding any of its queries' tokens, each query
// over its own tokens only.  Other shapes take the token-gather decode kernel.
constexpr int kTokPfMaxL = 16384;

bool tokpf_fits(int dtype, int d, int L) { return dtype == SA_BF16 && d == 128 && L <= kTokPfMaxL; }

struct TokPfWs {
  size_t mask, list, count, total;
  int nq, nb, wpr;
};
TokPfWs tokpf_ws(int B, int L) {
  auto up = [](size_t x) { return ((x + 255) / 256) * 256; };
  TokPfWs w;
  w.nq = cdiv(L, sa::kPfRows);
  w.nb = cdiv(L, sa::kPfKeys);
  w.wpr = 4 * w.nb;
  w.mask = 0;
  w.list = up(static_cast<size_t>(B) * L * w.wpr * 4);
  w.count = w.list + up(static_cast<size_t>(B) * w.nq * w.nb * 4);
  w.total = w.count + up(static_cast<size_t>(B) * w.nq * 4);
  return w;
}

}  // namespace

extern "C" {

size_t sa_prefill_tokens_workspace_bytes(int B, int L, int Hq, int Hkv, int d, int kmax) {
  if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || d < 1 || kmax < 1) return 0;
  const size_t gather = tok_ws_bytes(static_cast<long long>(B) * L * Hkv, Hq / Hkv, d, kmax);
  const size_t tc = L <= kTokPfMaxL ? tokpf_ws(B, L).total : 0;
  return std::max(gather, tc);
}

sa_status_t sa_prefill_tokens(const void* q, const void* k, const void* v, int dtype, const int32_t* idx,
                              const int32_t* cnt, int kmax, int B, int L, int Hq, int Hkv, int d, float scale,
                              void* out, void* workspace, size_t ws_bytes, void* stream) {
  t_err.clear();
  SA_ARG(B >= 1 && L >= 1 && static_cast<long long>(B) * L * Hkv <= (1LL << 24), "B*L*Hkv must be in [1, 2^24]");
  // each (batch row, query) pair is one selection row with a single query at position t
  DecodeArgs a{q, k, v, dtype, idx, cnt, kmax, B * L, 1, Hq, Hkv, d, L, L, 1, scale, out, workspace, ws_bytes, 1, L};
  SA_TRY(validate_decode(a));
  if (tokpf_fits(dtype, d, L)) {
    const TokPfWs w = tokpf_ws(B, L);
    SA_ARG(ws_bytes >= w.total, "workspace too small: %zu < %zu bytes", ws_bytes, w.total);
    SA_ARG(aligned16(workspace) && aligned16(out), "workspace and out must be 16-byte aligned");
    cudaStream_t st = as_stream(stream);
    char* ws = static_cast<char*>(workspace);
    uint32_t* mask = reinterpret_cast<uint32_t*>(ws + w.mask);
    int32_t* blist = reinterpret_cast<int32_t*>(ws + w.list);
    int32_t* bcnt = reinterpret_cast<int32_t*>(ws + w.count);
    const int smem = (8 * w.wpr + (w.nb + 31) / 32) * 4;
    SA_TRY(set_smem(sa::tokprefill_prep_kernel, smem));
    sa::tokprefill_prep_kernel<<<dim3(w.nq, B), 256, smem, st>>>(idx, cnt, kmax, L, w.nq, w.nb, w.wpr, mask, blist,
                                                                 bcnt);
    SA_CUDA(cudaGetLastError());
    return prefill_impl(q, k, v, blist, bcnt, w.nb, B, L, Hq, Hkv, scale, out, nullptr, st, mask, w.wpr);
  }
  return run_decode(a, as_stream(stream));
}

size_t sa_oracle_mass_workspace_bytes(int B, int L, int Hq, int Hkv, int d, int qtile, int block) {
  if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || d < 1 || qtile < 1 || block < 1) return 0;
  return mass_ws_bytes(B, L, Hq, Hkv, qtile, block);
}

sa_status_t sa_oracle_mass(const void* q, const void* k, int dtype, int B, int L, int Hq, int Hkv, int d, int qtile,
                           int block, float scale, float* mass, void* workspace, size_t ws_bytes, void* stream) {
  t_err.clear();
  (void)workspace;
  (void)ws_bytes;
  SA_TRY(check_common(dtype, B, Hq, Hkv, d));
  SA_ARG(q && k && mass, "null pointer argument");
  SA_ARG(L >= 1, "L >= 1 required");
  SA_SUP(dtype == SA_BF16 && d == 128 && qtile == 128 && block == 128,
         "oracle mass supports bf16, d == 128, qtile == block == 128");
  SA_ARG(aligned16(q) && aligned16(k), "q and k must be 16-byte aligned");
  SA_ARG(scale > 0.f && scale < 1e30f, "scale must be positive and finite");
  SA_ARG(static_cast<long long>(B) * L * Hq < (1LL << 31) && static_cast<long long>(B) * Hkv * L < (1LL << 31),
         "B*L*Hq and B*Hkv*L must be < 2^31");
  return mass_impl(q, k, B, L, Hq, Hkv, scale, mass, as_stream(stream));
}

size_t sa_decode_step_workspace_bytes(int B, int T, int Hq, int Hkv, int d, int dtype, int kmax) {
  const size_t dec = sa_decode_workspace_bytes(B, T, Hq, Hkv, d, kmax);
  if (!dec || (dtype != SA_F32 && dtype != SA_BF16)) return 0;
  const size_t es = static_cast<size_t>(esize(dtype));
  const size_t qb = static_cast<size_t>(B) * T * Hq * d * es;
  const size_t kb = static_cast<size_t>(B) * T * Hkv * d * es;
  auto up = [](size_t x) { return ((x + 255) / 256) * 256; };
  return up(dec) + 2 * up(qb) + 2 * up(kb);
}

}  // extern "C"

namespace {

// Device address of page-locked host memory mapped into the current device's address space
// (cudaHostAlloc / cudaHostRegister with mapping, which unified addressing gives by default),
// else nullptr (pageable memory, or memory the device cannot reach).
const void* mapped_host(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
  return at.devicePointer;
}

// The step's copies and launches, in stream order (the body of sa_decode_step).
sa_status_t step_enqueue(const StepArgs& a, cudaStream_t st) {
  auto up = [](size_t x) { return ((x + 255) / 256) * 256; };
  const size_t es = static_cast<size_t>(esize(a.dtype));
  const size_t dec = up(sa_decode_workspace_bytes(a.B, a.T, a.Hq, a.Hkv, a.d, a.kmax));
  const size_t qb = static_cast<size_t>(a.B) * a.T * a.Hq * a.d * es;
  const size_t kb = static_cast<size_t>(a.B) * a.T * a.Hkv * a.d * es;
  char* w = static_cast<char*>(a.workspace);
  const void* qd = a.q;
  const void* knd = a.k_new;
  const void* vnd = a.v_new;
  void* outd = a.out;
  bool out_mapped = false;
  const bool fused = seldec_fits(a.dtype, a.block, a.Hq / a.Hkv, a.T);
  // the append runs inside the fused launch when its rows lie in the local block (kept whatever
  // its score) and no scores are returned; otherwise it is a launch of its own
  const bool fused_append = fused && a.L >= a.T && a.T >= 1 && (a.L - a.T) / a.block == (a.L - 1) / a.block &&
                            a.scores == nullptr;
  bool q_host = false;
  if (a.host_io) {
    // q, k_new, v_new and out are used in place when they are page-locked host memory mapped
    // into the device's address space (the fused launch reads q and the new rows with plain
    // loads and writes out the same way; the other launches read q with bulk copies, so there it
    // is staged), and staged by copies otherwise.
    void* q_dev = w + dec;
    void* out_dev = w + dec + up(qb);
    void* kn_dev = w + dec + 2 * up(qb);
    void* vn_dev = w + dec + 2 * up(qb) + up(kb);
    // Every CTA of a group's cluster reads the group's q rows, so in place the host link carries
    // q once per CTA: worth it for clusters of up to two CTAs (batch 8, 8 kv heads, 32K context:
    // 47.6 -> 40.1 us per step end to end), not for ten (batch 1, 8 kv heads, 256K context: 44.0
    // -> 44.7 us); larger clusters get q by one copy.
    int cs = 0, ncl = 0;
    if (fused_append) {
      const int nb = cdiv(a.L, a.block);
      SA_TRY((a.d == 128 ? sd_shape<128, true>(a.B * a.Hkv, nb, a.kmax, &cs, &ncl)
                         : sd_shape<64, true>(a.B * a.Hkv, nb, a.kmax, &cs, &ncl)));
    }
    const void* q_map = (fused_append && cs <= 2) ? mapped_host(a.q) : nullptr;
    if (q_map) {
      qd = q_map;
      q_host = true;
    } else {
      SA_CUDA(cudaMemcpyAsync(q_dev, a.q, qb, cudaMemcpyHostToDevice, st));
      qd = q_dev;
    }
    const void* kn_map = mapped_host(a.k_new);
    const void* vn_map = mapped_host(a.v_new);
    void* out_map = const_cast<void*>(mapped_host(a.out));
    if (kn_map) {
      knd = kn_map;
    } else {
      SA_CUDA(cudaMemcpyAsync(kn_dev, a.k_new, kb, cudaMemcpyHostToDevice, st));
      knd = kn_dev;
    }
    if (vn_map) {
      vnd = vn_map;
    } else {
      SA_CUDA(cudaMemcpyAsync(vn_dev, a.v_new, kb, cudaMemcpyHostToDevice, st));
      vnd = vn_dev;
    }
    out_mapped = out_map != nullptr;
    outd = out_mapped ? out_map : out_dev;
  }
  void* sp = static_cast<void*>(st);
  if (fused_append) {
    SA_ARG(a.k_cache && a.v_cache && a.sketch, "null pointer argument");
    SA_TRY(select_decode_impl(qd, a.dtype, a.sketch, a.k_cache, a.v_cache, a.B, a.T, a.Hq, a.Hkv, a.d, a.L,
                              a.L_stride, a.block, a.k, a.scale, a.idx, a.cnt, a.kmax, a.scores, outd, knd, vnd, st,
                              q_host));
  } else if (fused) {
    SA_TRY(sa_append_kv(knd, vnd, a.dtype, a.B, a.Hkv, a.T, a.d, a.k_cache, a.v_cache, a.L_stride, a.L - a.T,
                        a.block, a.sketch, sp));
    // selection and attention in one launch (one cluster per group)
    SA_TRY(sa_select_decode(qd, a.dtype, a.sketch, a.k_cache, a.v_cache, a.B, a.T, a.Hq, a.Hkv, a.d, a.L,
                            a.L_stride, a.block, a.k, a.scale, a.idx, a.cnt, a.kmax, a.scores, outd, sp));
  } else {
    SA_TRY(sa_append_kv(knd, vnd, a.dtype, a.B, a.Hkv, a.T, a.d, a.k_cache, a.v_cache, a.L_stride, a.L - a.T,
                        a.block, a.sketch, sp));
    SA_TRY(sa_select_topk(SA_SELECT_SKETCH, qd, a.dtype, a.sketch, a.scores, a.B, a.T, a.Hq, a.Hkv, a.d, a.L,
                          a.L_stride, a.block, 0, 0, a.k, 0, 1, a.scale, a.idx, a.cnt, a.kmax, sp));
    SA_TRY(sa_decode(qd, a.k_cache, a.v_cache, a.dtype, a.idx, a.cnt, a.kmax, a.B, a.T, a.Hq, a.Hkv, a.d, a.L,
                     a.L_stride, a.block, a.scale, outd, w, dec, sp));
  }
  if (a.host_io && !out_mapped) SA_CUDA(cudaMemcpyAsync(a.out, outd, qb, cudaMemcpyDeviceToHost, st));
  return SA_OK;
}

}  // namespace

extern "C" {

sa_status_t sa_decode_step(const void* q, const void* k_new, const void* v_new, int dtype, void* k_cache,
                           void* v_cache, float* sketch, int B, int T, int Hq, int Hkv, int d, int L, int L_stride,
                           int block, int k, float scale, int32_t* idx, int32_t* cnt, int kmax, float* scores,
                           void* out, int host_io, void* workspace, size_t ws_bytes, void* stream) {
  t_err.clear();
  SA_TRY(check_common(dtype, B, Hq, Hkv, d));
  SA_ARG(q && k_new && v_new && out && workspace, "null pointer argument");
  SA_ARG(L >= T && T >= 1, "need 1 <= T <= L");
  const size_t need = sa_decode_step_workspace_bytes(B, T, Hq, Hkv, d, dtype, kmax);
  SA_ARG(need && ws_bytes >= need, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  const StepArgs a{q, k_new, v_new, dtype, k_cache, v_cache, sketch, B, T, Hq, Hkv, d, L, L_stride, block, k,
                   scale, idx, cnt, kmax, scores, out, host_io, workspace, ws_bytes};
  cudaStream_t st = as_stream(stream);
  // Replay one CUDA graph per repeated argument set (copies and the three kernels in one launch);
  // the first call with a set, the legacy default stream and a stream that is already being
  // captured take the direct path.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (st == nullptr || cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return step_enqueue(a, st);
  }
  int dev = 0;
  SA_CUDA(cudaGetDevice(&dev));
  const StepKey key = step_key(a, dev);
  {
    std::lock_guard<std::mutex> lk(g_step_mu);
    for (auto& e : g_step_cache)
      if (e.key == key) {
        e.last_use = ++g_step_clock;
        SA_CUDA(cudaGraphLaunch(e.exec, st));
        return SA_OK;
      }
    // capture only argument sets that repeat: a loop whose context grows every token never
    // pays for a capture
    auto it = std::find(g_step_seen.begin(), g_step_seen.end(), key);
    if (it == g_step_seen.end()) {
      if (g_step_seen.size() >= 4 * kStepCacheMax) g_step_seen.erase(g_step_seen.begin());
      g_step_seen.push_back(key);
      return step_enqueue(a, st);
    }
    g_step_seen.erase(it);
  }
  SA_CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
  const sa_status_t rc = step_enqueue(a, st);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(st, &graph);
  if (rc != SA_OK) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return rc;
  }
  cudaGraphExec_t exec = nullptr;
  if (ec != cudaSuccess || graph == nullptr || cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
    // not capturable (e.g. pageable host buffers): run the step directly
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return step_enqueue(a, st);
  }
  cudaGraphDestroy(graph);
  {
    std::lock_guard<std::mutex> lk(g_step_mu);
    if (g_step_cache.size() >= kStepCacheMax) {
      auto old = std::min_element(g_step_cache.begin(), g_step_cache.end(),
                                  [](const StepGraph& x, const StepGraph& y) { return x.last_use < y.last_use; });
      cudaGraphExecDestroy(old->exec);
      g_step_cache.erase(old);
    }
    g_step_cache.push_back(StepGraph{key, exec, ++g_step_clock});
  }
  SA_CUDA(cudaGraphLaunch(exec, st));
  return SA_OK;
}

}  // extern "C"

// The allocation-free decode entry point (needs the helpers above).
#include "sa_noalloc.cu"
