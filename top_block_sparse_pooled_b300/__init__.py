"""Top-k block-sparse GQA attention on NVIDIA B300 (sm_103a).

A thin ctypes binding over ``libsparse_attn.so`` (C ABI in
``include/sparse_attn.h``).  Every function here has the name of the C entry
point it calls and only marshals arguments: torch tensors supply device memory
and the current CUDA stream, and all computation runs in the library's CUDA
kernels.  There is no CPU fallback: importing this package without the built
library raises, and every call checks the returned status.

Build the library with ``python -m top_block_sparse_pooled_b300._build``.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsparse_attn.so")

SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_CUDA, SA_ERR_TIMEOUT = range(5)
SA_F32, SA_BF16 = 0, 1
SA_SELECT_SKETCH, SA_SELECT_MASS = 0, 1


class SparseAttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s: %s" % (_STATUS_NAMES.get(status, status), msg))
        self.status = status


_STATUS_NAMES = {0: "SA_OK", 1: "SA_ERR_INVALID_ARG", 2: "SA_ERR_UNSUPPORTED", 3: "SA_ERR_CUDA",
                 4: "SA_ERR_TIMEOUT"}

if not os.path.exists(LIB_PATH):
    raise ImportError("libsparse_attn.so is not built (expected at %s); run "
                      "`python -m top_block_sparse_pooled_b300._build`" % LIB_PATH)

lib = ctypes.CDLL(LIB_PATH)

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

# C signatures (argument order as in include/sparse_attn.h)
SIGNATURES = {
    "sa_version": ([], _i),
    "sa_last_error": ([], ctypes.c_char_p),
    "sa_status_name": ([_i], ctypes.c_char_p),
    "sa_device_status": ([ctypes.POINTER(_i), _i], _i),
    "sa_build_sketch": ([_vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp], _i),
    "sa_append_kv": ([_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _i, _i, _i, _vp, _vp], _i),
    "sa_select_topk": ([_i, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f,
                        _vp, _vp, _i, _vp], _i),
    "sa_select_topdelta": ([_vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _f, _vp, _vp, _i, _vp], _i),
    "sa_select_kmax": ([_i, _i, _i, _i, _i, _i, _i], _i),
    "sa_budget_sublinear": ([_i, _i, _i, _i, _f], _i),
    "sa_decode_workspace_bytes": ([_i, _i, _i, _i, _i, _i], _sz),
    "sa_decode": ([_vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp], _i),
    "sa_select_decode": ([_vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _i, _vp, _vp,
                          _vp], _i),
    "sa_decode_noalloc": ([_vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp], _i),
    "sa_prefill": ([_vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp], _i),
    "sa_oracle_mass_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i], _sz),
    "sa_oracle_mass": ([_vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp], _i),
    "sa_token_mass_workspace_bytes": ([_i, _i, _i, _i, _i], _sz),
    "sa_token_mass_decode": ([_vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp], _i),
    "sa_decode_tokens": ([_vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp],
                         _i),
    "sa_token_mass_prefill_workspace_bytes": ([_i, _i, _i, _i], _sz),
    "sa_token_mass_prefill": ([_vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp], _i),
    "sa_prefill_tokens_workspace_bytes": ([_i, _i, _i, _i, _i, _i], _sz),
    "sa_prefill_tokens": ([_vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp], _i),
    "sa_selftest_wait_timeout": ([ctypes.c_longlong, _vp], _i),
    "sa_selftest_poison_noalloc": ([_i, _vp], _i),
    "sa_decode_step_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i], _sz),
    "sa_decode_step": ([_vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _i,
                        _vp, _vp, _i, _vp, _sz, _vp], _i),
}
for _name, (_args, _res) in SIGNATURES.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


def _check(status: int) -> None:
    if status != SA_OK:
        raise SparseAttnError(status, lib.sa_last_error().decode())


def _ptr(t):
    """Device (or host) address of a tensor, None for None; raw ints pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _dtype(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return SA_F32
    if t.dtype == torch.bfloat16:
        return SA_BF16
    raise TypeError("q/k/v must be float32 or bfloat16, got %s" % t.dtype)


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def sa_version() -> int:
    return lib.sa_version()


def sa_device_status(clear: bool = True) -> int:
    code = _i(0)
    _check(lib.sa_device_status(ctypes.byref(code), 1 if clear else 0))
    return code.value


def sa_build_sketch(k, L, block, sketch, stream=None):
    """k: [B, Hkv, L_stride, d]; sketch: [B, Hkv, ceil(L_stride/block), d] float32 (written)."""
    B, Hkv, Ls, d = k.shape
    _check(lib.sa_build_sketch(_ptr(k), _dtype(k), B, Hkv, L, Ls, d, block, _ptr(sketch), _stream(stream)))


def sa_append_kv(k_new, v_new, k_cache, v_cache, pos, block, sketch, stream=None):
    """k_new, v_new: [B, T, Hkv, d]; caches [B, Hkv, L_stride, d]; rows pos..pos+T-1 written."""
    B, T, Hkv, d = k_new.shape
    Ls = k_cache.shape[2]
    _check(lib.sa_append_kv(_ptr(k_new), _ptr(v_new), _dtype(k_new), B, Hkv, T, d, _ptr(k_cache), _ptr(v_cache),
                            Ls, pos, block, _ptr(sketch), _stream(stream)))


def sa_budget_sublinear(L, block, k_ref, L_ref, exponent) -> int:
    """Length-aware block budget k(L) = ceil(k_ref * (L / L_ref)^exponent), clamped to the candidates."""
    return lib.sa_budget_sublinear(L, block, k_ref, L_ref, float(exponent))


def sa_select_kmax(L, block, qtile, prefill, k, frac_num=0, frac_den=1) -> int:
    return lib.sa_select_kmax(L, block, qtile, 1 if prefill else 0, k, frac_num, frac_den)


def sa_select_topk(mode, q, sketch, scores, Hkv, L, L_stride, block, qtile, prefill, k, frac_num, frac_den, scale,
                   idx, cnt, stream=None, d=None, dtype=None, B=None, Tq=None, Hq=None):
    """Scores + top-k.  q: decode [B, T, Hq, d] / prefill [B, L, Hq, d] (may be None in MASS mode,
    then pass B, Tq, Hq, d).  idx: [B, Hkv, nq, kmax] int32, cnt: [B, Hkv, nq] int32 (written)."""
    if q is not None:
        B, Tq, Hq, d = q.shape
        dtype = _dtype(q)
    kmax = idx.shape[-1]
    _check(lib.sa_select_topk(mode, _ptr(q), SA_BF16 if dtype is None else dtype, _ptr(sketch), _ptr(scores), B, Tq,
                              Hq, Hkv, d, L, L_stride, block, qtile, 1 if prefill else 0, k, frac_num, frac_den,
                              float(scale), _ptr(idx), _ptr(cnt), kmax, _stream(stream)))


def sa_select_topdelta(q, sketch, scores, Hkv, L, L_stride, block, delta, cap, scale, idx, cnt, stream=None):
    """Decode top-delta selection: q [B, T, Hq, d]; idx [B, Hkv, 1, kmax], cnt [B, Hkv, 1] (written)."""
    B, Tq, Hq, d = q.shape
    kmax = idx.shape[-1]
    _check(lib.sa_select_topdelta(_ptr(q), _dtype(q), _ptr(sketch), _ptr(scores), B, Tq, Hq, Hkv, d, L, L_stride,
                                  block, float(delta), cap, float(scale), _ptr(idx), _ptr(cnt), kmax,
                                  _stream(stream)))


def sa_decode_workspace_bytes(B, T, Hq, Hkv, d, kmax) -> int:
    return lib.sa_decode_workspace_bytes(B, T, Hq, Hkv, d, kmax)


def sa_decode(q, k_cache, v_cache, idx, cnt, L, block, scale, out, workspace, stream=None):
    """q, out: [B, T, Hq, d]; caches [B, Hkv, L_stride, d]; idx [B, Hkv, 1, kmax]; workspace uint8 device tensor."""
    B, T, Hq, d = q.shape
    Hkv, Ls = k_cache.shape[1], k_cache.shape[2]
    kmax = idx.shape[-1]
    _check(lib.sa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _dtype(q), _ptr(idx), _ptr(cnt), kmax, B, T, Hq, Hkv,
                         d, L, Ls, block, float(scale), _ptr(out), _ptr(workspace), workspace.numel(),
                         _stream(stream)))


def sa_select_decode(q, sketch, k_cache, v_cache, L, block, k, scale, idx, cnt, out, scores=None, stream=None):
    """Sketch selection + sparse decode in one launch.  q, out: [B, T, Hq, d] bf16; sketch
    [B, Hkv, nb_cap, d] float32; caches [B, Hkv, L_stride, d]; idx [B, Hkv, 1, kmax] and cnt [B, Hkv, 1]
    int32 (written); scores [B, Hkv, 1, nb] float32 or None (written)."""
    B, T, Hq, d = q.shape
    Hkv, Ls = k_cache.shape[1], k_cache.shape[2]
    kmax = idx.shape[-1]
    _check(lib.sa_select_decode(_ptr(q), _dtype(q), _ptr(sketch), _ptr(k_cache), _ptr(v_cache), B, T, Hq, Hkv, d, L,
                                Ls, block, k, float(scale), _ptr(idx), _ptr(cnt), kmax, _ptr(scores), _ptr(out),
                                _stream(stream)))


def sa_decode_noalloc(q, k_cache, v_cache, idx, cnt, L, block, scale, out, stream=None):
    """sa_decode with the library's fixed scratch instead of a workspace (for callers that cannot allocate)."""
    B, T, Hq, d = q.shape
    Hkv, Ls = k_cache.shape[1], k_cache.shape[2]
    kmax = idx.shape[-1]
    _check(lib.sa_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _dtype(q), _ptr(idx), _ptr(cnt), kmax, B, T,
                                 Hq, Hkv, d, L, Ls, block, float(scale), _ptr(out), _stream(stream)))


def sa_prefill(q, k, v, idx, cnt, qtile, block, scale, out, lse=None, stream=None):
    """q, out: [B, L, Hq, d]; k, v: [B, Hkv, L, d]; idx [B, Hkv, nq, kmax]; lse [B, Hq, L] float32 or None."""
    B, L, Hq, d = q.shape
    Hkv = k.shape[1]
    kmax = idx.shape[-1]
    _check(lib.sa_prefill(_ptr(q), _ptr(k), _ptr(v), _dtype(q), _ptr(idx), _ptr(cnt), kmax, B, L, Hq, Hkv, d, qtile,
                          block, float(scale), _ptr(out), _ptr(lse), _stream(stream)))


def sa_oracle_mass_workspace_bytes(B, L, Hq, Hkv, d, qtile, block) -> int:
    return lib.sa_oracle_mass_workspace_bytes(B, L, Hq, Hkv, d, qtile, block)


def sa_oracle_mass(q, k, qtile, block, scale, mass, workspace, stream=None):
    """q: [B, L, Hq, d]; k: [B, Hkv, L, d]; mass: [B, Hkv, nq, nb] float32 (written)."""
    B, L, Hq, d = q.shape
    Hkv = k.shape[1]
    ws = _ptr(workspace)
    nbytes = workspace.numel() if workspace is not None else 0
    _check(lib.sa_oracle_mass(_ptr(q), _ptr(k), _dtype(q), B, L, Hq, Hkv, d, qtile, block, float(scale), _ptr(mass),
                              ws, nbytes, _stream(stream)))


def sa_token_mass_workspace_bytes(B, T, Hq, Hkv, L) -> int:
    return lib.sa_token_mass_workspace_bytes(B, T, Hq, Hkv, L)


def sa_token_mass_decode(q, k_cache, L, scale, mass, workspace, stream=None):
    """q: [B, T, Hq, d]; k_cache: [B, Hkv, L_stride, d]; mass: [B, L] float32 (written)."""
    B, T, Hq, d = q.shape
    Hkv, Ls = k_cache.shape[1], k_cache.shape[2]
    _check(lib.sa_token_mass_decode(_ptr(q), _ptr(k_cache), _dtype(q), B, T, Hq, Hkv, d, L, Ls, float(scale),
                                    _ptr(mass), _ptr(workspace), workspace.numel(), _stream(stream)))


def sa_decode_tokens(q, k_cache, v_cache, idx, cnt, L, scale, out, workspace, stream=None):
    """q, out: [B, T, Hq, d]; caches [B, Hkv, L_stride, d]; idx [B, kmax] tokens shared by the kv heads; cnt [B]."""
    B, T, Hq, d = q.shape
    Hkv, Ls = k_cache.shape[1], k_cache.shape[2]
    kmax = idx.shape[-1]
    _check(lib.sa_decode_tokens(_ptr(q), _ptr(k_cache), _ptr(v_cache), _dtype(q), _ptr(idx), _ptr(cnt), kmax, B, T,
                                Hq, Hkv, d, L, Ls, float(scale), _ptr(out), _ptr(workspace), workspace.numel(),
                                _stream(stream)))


def sa_token_mass_prefill_workspace_bytes(B, L, Hq, Hkv) -> int:
    return lib.sa_token_mass_prefill_workspace_bytes(B, L, Hq, Hkv)


def sa_token_mass_prefill(q, k, scale, mass, workspace, stream=None):
    """q: [B, L, Hq, d]; k: [B, Hkv, L, d]; mass: [B, L, L] float32 (written)."""
    B, L, Hq, d = q.shape
    Hkv = k.shape[1]
    _check(lib.sa_token_mass_prefill(_ptr(q), _ptr(k), _dtype(q), B, L, Hq, Hkv, d, float(scale), _ptr(mass),
                                     _ptr(workspace), workspace.numel(), _stream(stream)))


def sa_prefill_tokens_workspace_bytes(B, L, Hq, Hkv, d, kmax) -> int:
    return lib.sa_prefill_tokens_workspace_bytes(B, L, Hq, Hkv, d, kmax)


def sa_prefill_tokens(q, k, v, idx, cnt, scale, out, workspace, stream=None):
    """q, out: [B, L, Hq, d]; k, v: [B, Hkv, L, d]; idx [B, L, kmax] per-query tokens; cnt [B, L]."""
    B, L, Hq, d = q.shape
    Hkv = k.shape[1]
    kmax = idx.shape[-1]
    _check(lib.sa_prefill_tokens(_ptr(q), _ptr(k), _ptr(v), _dtype(q), _ptr(idx), _ptr(cnt), kmax, B, L, Hq, Hkv,
                                 d, float(scale), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)))


def sa_selftest_wait_timeout(limit_ns, stream=None):
    """Launch the bounded-wait self-test (a wait that nothing completes, given up after limit_ns)."""
    _check(lib.sa_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def sa_selftest_poison_noalloc(nbytes, stream=None):
    """Fill the head of sa_decode_noalloc's scratch with a non-zero pattern (recovery test)."""
    _check(lib.sa_selftest_poison_noalloc(int(nbytes), _stream(stream)))


def sa_decode_step_workspace_bytes(B, T, Hq, Hkv, d, dtype, kmax) -> int:
    return lib.sa_decode_step_workspace_bytes(B, T, Hq, Hkv, d, dtype, kmax)


def _decode_step_args(q, k_new, v_new, k_cache, v_cache, sketch, L, block, k, scale, idx, cnt, out, workspace,
                      scores, host_io, stream):
    B, T, Hq, d = q.shape
    Hkv, Ls = k_cache.shape[1], k_cache.shape[2]
    kmax = idx.shape[-1]
    return (_ptr(q), _ptr(k_new), _ptr(v_new), _dtype(q), _ptr(k_cache), _ptr(v_cache), _ptr(sketch), B, T, Hq, Hkv,
            d, L, Ls, block, k, float(scale), _ptr(idx), _ptr(cnt), kmax, _ptr(scores), _ptr(out),
            1 if host_io else 0, _ptr(workspace), workspace.numel(), _stream(stream))


def sa_decode_step(q, k_new, v_new, k_cache, v_cache, sketch, L, block, k, scale, idx, cnt, out, workspace,
                   scores=None, host_io=False, stream=None):
    """Append + select + decode.  With host_io, q/k_new/v_new/out are pinned host tensors."""
    _check(lib.sa_decode_step(*_decode_step_args(q, k_new, v_new, k_cache, v_cache, sketch, L, block, k, scale, idx,
                                                 cnt, out, workspace, scores, host_io, stream)))


class DecodeStep:
    """sa_decode_step with its arguments marshalled once, for a serving loop that calls the same
    buffers every token: step() issues the call with the stored pointers and sizes, step(L) with a new
    context length.  The tensors must stay alive, keep their shapes and stay where they are; their
    contents may change between calls.  The stream is fixed here (default: the current stream)."""

    def __init__(self, q, k_new, v_new, k_cache, v_cache, sketch, L, block, k, scale, idx, cnt, out, workspace,
                 scores=None, host_io=False, stream=None):
        self._keep = (q, k_new, v_new, k_cache, v_cache, sketch, idx, cnt, out, workspace, scores)
        self._args = _decode_step_args(q, k_new, v_new, k_cache, v_cache, sketch, L, block, k, scale, idx, cnt,
                                       out, workspace, scores, host_io, stream)
        self._fn = lib.sa_decode_step

    def __call__(self, L=None):
        if L is not None and L != self._args[12]:
            self._args = self._args[:12] + (int(L),) + self._args[13:]
        status = self._fn(*self._args)
        if status != SA_OK:
            _check(status)
