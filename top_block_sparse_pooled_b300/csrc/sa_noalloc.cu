// sa_noalloc.cu -- sa_decode_noalloc: the split-KV decode with its scratch
// space held by the library itself, for callers that cannot allocate device
// memory (see include/sparse_attn.h).  Included into sa_api.cu's translation
// unit after the decode launch helpers it reuses.
//
// The scratch is one file-scope __device__ array of a fixed size.  Its device
// address is looked up once per device, with that device current, through
// cudaGetSymbolAddress (the name of the array in host code is only a host-side
// stand-in and must never be handed to a kernel).  Every call shares the
// array; the arrival counters at its head are cleared on the caller's stream
// before each launch, and the rest is fully rewritten by the kernels.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of g_noalloc_scratch on the current device (looked up on the
// first call made with that device current, then cached).
sa_status_t noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  SA_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(SA_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(SA_ERR_CUDA, "cudaGetSymbolAddress(decode scratch) on device %d: %s", dev, cudaGetErrorString(e));
    addr[dev] = p;
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
