// sa_noalloc.cu -- sa_decode_noalloc: the split-KV decode with its scratch
// space held by the library itself, for callers that cannot allocate device
// memory (see include/sparse_attn.h).  Included into sa_api.cu's translation
// unit after the decode launch helpers it reuses.
//
// The scratch is one file-scope __device__ array of a fixed size.  Its device
// address is looked up once per device (and context), with that device current,
// through cudaGetSymbolAddress (the name of the array in host code is only a host-side
// stand-in and must never be handed to a kernel).  Every call shares the
// array; the arrival counters at its head are cleared on the caller's stream
// before each launch, and the rest is fully rewritten by the kernels.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of g_noalloc_scratch on the current device.  It is looked up
// with cudaGetSymbolAddress on the first call made with that device current and
// cached for the device's current CUDA context; a call made in another context
// of the same device (after cudaDeviceReset, or a primary-context teardown and
// re-creation) looks it up again, because the array then lives in the new
// context's copy of the module.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

sa_status_t current_context(CUcontext* out) {
  static std::once_flag once;
  static CtxGetCurrentFn f = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  if (!f) return fail(SA_ERR_CUDA, "cuCtxGetCurrent unavailable");
  if (f(out) != CUDA_SUCCESS) return fail(SA_ERR_CUDA, "cuCtxGetCurrent failed");
  return SA_OK;
}

sa_status_t noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  static CUcontext ctx[64] = {};
  int dev = 0;
  SA_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(SA_ERR_UNSUPPORTED, "device ordinal %d", dev);
  CUcontext cur = nullptr;  // null until the runtime has made the device's context current
  SA_TRY(current_context(&cur));
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr || cur == nullptr || ctx[dev] != cur) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(SA_ERR_CUDA, "cudaGetSymbolAddress(decode scratch) on device %d: %s", dev, cudaGetErrorString(e));
    SA_TRY(current_context(&cur));  // the lookup made the context current
    addr[dev] = p;
    ctx[dev] = cur;
  }
  *out = addr[dev];
  return SA_OK;
}

}  // namespace

extern "C" sa_status_t sa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, int dtype,
                                         const int32_t* idx, const int32_t* cnt, int kmax, int B, int T, int Hq,
                                         int Hkv, int d, int L, int L_stride, int block, float scale, void* out,
                                         void* stream) {
  t_err.clear();
  SA_TRY(check_common(dtype, B, Hq, Hkv, d));
  SA_ARG(T >= 1 && kmax >= 1, "T >= 1 and kmax >= 1 required");
  const int groups = B * Hkv;
  const size_t need = decode_ws_bytes(groups, (Hq / Hkv) * T, d, kmax);
  SA_ARG(need <= kNoAllocScratchBytes,
         "sa_decode_noalloc: this problem needs %zu bytes of scratch, more than the library's fixed %zu bytes; "
         "use sa_decode with a caller-provided workspace",
         need, kNoAllocScratchBytes);
  void* ws = nullptr;
  SA_TRY(noalloc_scratch(&ws));
  DecodeArgs a{q, k_cache, v_cache, dtype, idx, cnt, kmax, B, T, Hq, Hkv, d, L, L_stride, block, scale, out,
               ws, kNoAllocScratchBytes};
  SA_TRY(validate_decode(a));
  // the per-group arrival counters at the head of the scratch must start at zero
  const size_t ctr_bytes = ((static_cast<size_t>(groups) * 4 + 255) / 256) * 256;
  SA_CUDA(cudaMemsetAsync(ws, 0, ctr_bytes, as_stream(stream)));
  return run_decode(a, as_stream(stream));
}

// Test-only: overwrite the head of the scratch (where the arrival counters live) with a
// non-zero byte pattern, as a call that gave up mid-way would leave it.
extern "C" sa_status_t sa_selftest_poison_noalloc(int bytes, void* stream) {
  t_err.clear();
  SA_ARG(bytes >= 1 && static_cast<size_t>(bytes) <= kNoAllocScratchBytes, "bytes must be in [1, %zu]",
         kNoAllocScratchBytes);
  void* s = nullptr;
  SA_TRY(noalloc_scratch(&s));
  SA_CUDA(cudaMemsetAsync(s, 0x5A, static_cast<size_t>(bytes), as_stream(stream)));
  return SA_OK;
}
