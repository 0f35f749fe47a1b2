"""fp64 CPU oracle for top-k block-sparse GQA attention (ctypes binding).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg, never by the product package.  The
arithmetic lives in ``oracle.c`` (plain loops in double precision); this module
only marshals numpy arrays and composes the steps in the order the pages give
them: sketch -> score -> select -> exact attention on the selected support
("How Much Dense Attention is Necessary?" Sec. 2.1; "Faster Than Flash" Sec. 1-3).

Inputs are numpy arrays: ``uint16`` = bf16 bit patterns, ``float32``, or
``float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False, src: str = _SRC, out: str = _LIB, defines=()) -> str:
    """Compile oracle.c (gcc, -O2, OpenMP) into a shared library beside it."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11"]
        cmd += ["-D%s" % x for x in defines]
        cmd += ["-o", tmp, src, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, out)
    return out


def load(path: str = None):
    """Load (building if needed) the oracle library and declare its signatures."""
    path = path or build()
    lib = ctypes.CDLL(path)
    vp, i, l, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_double
    lib.orc_block_means.argtypes = [vp, i, l, l, l, l, l, vp]
    lib.orc_decode_scores.argtypes = [vp, i, vp, l, l, l, l, l, l, d, vp]
    lib.orc_prefill_scores.argtypes = [vp, i, vp, l, l, l, l, l, l, l, l, d, vp, l, vp]
    lib.orc_select.argtypes = [vp, l, l, vp, vp, vp, l, vp, vp]
    lib.orc_select.restype = i
    lib.orc_select_delta.argtypes = [vp, l, l, vp, vp, d, vp, l, vp, vp]
    lib.orc_select_delta.restype = i
    lib.orc_attend.argtypes = [vp, vp, vp, i, l, l, l, l, l, l, l, l, l, d, vp, vp, l, l, l, vp, l, vp, vp]
    lib.orc_mass.argtypes = [vp, vp, i, l, l, l, l, l, l, l, l, l, l, d, vp, l, vp]
    lib.orc_causal_blocks.argtypes = [l, l, l, l, l]
    lib.orc_causal_blocks.restype = l
    lib.orc_num_threads.restype = i
    lib.orc_set_threads.argtypes = [i]
    return lib


_lib = None


def _L():
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def use(lib) -> None:
    """Swap the loaded library (the tests use this to run planted-mistake builds)."""
    global _lib
    _lib = lib


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float64:
        return 2
    raise TypeError("unsupported oracle input dtype %s" % a.dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype=None):
    a = np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))
    return a


def threads() -> int:
    return int(_L().orc_num_threads())


def set_threads(n: int) -> None:
    _L().orc_set_threads(int(n))


# --------------------------------------------------------------------------- steps

def block_means(k: np.ndarray, L: int, Bk: int) -> np.ndarray:
    """Sketch: mean of each block's valid key rows.  k: [B, Hkv, Ls, d] -> [B*Hkv, nb, d]."""
    k = _c(k)
    B, Hkv, Ls, d = k.shape
    nb = (L + Bk - 1) // Bk
    out = np.empty((B * Hkv, nb, d), dtype=np.float64)
    _L().orc_block_means(_p(k), _dt(k), B * Hkv, L, Ls, d, Bk, _p(out))
    return out


def decode_scores(q: np.ndarray, sketch: np.ndarray, Hkv: int, scale: float) -> np.ndarray:
    """s[g, b] = max over the group's (head, token) rows of scale * q . sketch[g, b]."""
    q = _c(q)
    B, T, Hq, d = q.shape
    sketch = _c(sketch, np.float64)
    nb = sketch.shape[1]
    out = np.empty((B * Hkv, nb), dtype=np.float64)
    _L().orc_decode_scores(_p(q), _dt(q), _p(sketch), B, T, Hq, Hkv, d, nb, scale, _p(out))
    return out


def prefill_scores(q, sketch, Hkv, Qt, Bk, scale, units) -> np.ndarray:
    """Per (group, tile) unit: max over the tile's rows of scale * q . sketch; -inf if not causal."""
    q = _c(q)
    B, Lq, Hq, d = q.shape
    sketch = _c(sketch, np.float64)
    nb = sketch.shape[1]
    units = _c(np.asarray(units, dtype=np.int64).reshape(-1, 2))
    out = np.empty((len(units), nb), dtype=np.float64)
    _L().orc_prefill_scores(_p(q), _dt(q), _p(sketch), B, Lq, Hq, Hkv, d, Qt, Bk, nb, scale,
                            _p(units), len(units), _p(out))
    return out


def causal_blocks(i: int, Qt: int, Bk: int, Lq: int, pos0: int = 0) -> int:
    return int(_L().orc_causal_blocks(i, Qt, Bk, Lq, pos0))


def select(scores, nvalid, forced_hi, budget, kmax):
    """Top-k of the non-forced valid blocks (ties -> lower index) plus the forced ones, ascending."""
    scores = _c(scores, np.float64)
    n, nb = scores.shape
    nvalid = _c(np.broadcast_to(np.asarray(nvalid, dtype=np.int64), (n,)))
    forced_hi = _c(np.broadcast_to(np.asarray(forced_hi, dtype=np.int64), (n,)))
    budget = _c(np.broadcast_to(np.asarray(budget, dtype=np.int64), (n,)))
    idx = np.empty((n, kmax), dtype=np.int32)
    cnt = np.empty((n,), dtype=np.int32)
    rc = _L().orc_select(_p(scores), n, nb, _p(nvalid), _p(forced_hi), _p(budget), kmax, _p(idx), _p(cnt))
    if rc != 0:
        raise ValueError("kmax too small for the selection")
    return idx, cnt


def select_delta(scores, nvalid, forced_hi, delta, cap, kmax):
    """Top-delta: non-forced blocks scoring >= max(forced scores) - delta, at most cap of them
    (highest first, ties -> lower index), plus the forced ones, ascending."""
    scores = _c(scores, np.float64)
    n, nb = scores.shape
    nvalid = _c(np.broadcast_to(np.asarray(nvalid, dtype=np.int64), (n,)))
    forced_hi = _c(np.broadcast_to(np.asarray(forced_hi, dtype=np.int64), (n,)))
    cap = _c(np.broadcast_to(np.asarray(cap, dtype=np.int64), (n,)))
    idx = np.empty((n, kmax), dtype=np.int32)
    cnt = np.empty((n,), dtype=np.int32)
    rc = _L().orc_select_delta(_p(scores), n, nb, _p(nvalid), _p(forced_hi), float(delta), _p(cap), kmax, _p(idx),
                               _p(cnt))
    if rc != 0:
        raise ValueError("kmax too small for the selection")
    return idx, cnt


def attend(q, k, v, Hkv, L, pos0, Bk, scale, rows, idx=None, cnt=None, nsel=1, rows_per_sel=1 << 40):
    """Exact softmax attention of the given (b, t, h) rows over the selected blocks (all if idx is None)."""
    q, k, v = _c(q), _c(k), _c(v)
    assert q.dtype == k.dtype == v.dtype
    B, Tq, Hq, d = q.shape
    Ls = k.shape[2]
    rows = _c(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    kmax = 0
    if idx is not None:
        idx = _c(idx, np.int32)
        cnt = _c(cnt, np.int32)
        kmax = idx.shape[-1]
    out = np.empty((len(rows), d), dtype=np.float64)
    lse = np.empty((len(rows),), dtype=np.float64)
    _L().orc_attend(_p(q), _p(k), _p(v), _dt(q), B, Tq, Hq, Hkv, d, L, Ls, pos0, Bk, scale,
                    _p(idx), _p(cnt), kmax, nsel, min(rows_per_sel, 1 << 40), _p(rows), len(rows),
                    _p(out), _p(lse))
    return out, lse


def mass(q, k, Hkv, L, pos0, Qt, Bk, scale, units) -> np.ndarray:
    """Exact dense-softmax mass per block, summed over the group's heads and the tile's rows."""
    q, k = _c(q), _c(k)
    assert q.dtype == k.dtype
    B, Lq, Hq, d = q.shape
    Ls = k.shape[2]
    nb = (L + Bk - 1) // Bk
    units = _c(np.asarray(units, dtype=np.int64).reshape(-1, 2))
    out = np.empty((len(units), nb), dtype=np.float64)
    _L().orc_mass(_p(q), _p(k), _dt(q), B, Lq, Hq, Hkv, d, L, Ls, pos0, Qt, Bk, scale,
                  _p(units), len(units), _p(out))
    return out


# ------------------------------------------------------------------ composed paths

def prefill_budget(i: int, k: int, frac_num: int, frac_den: int, Qt: int, Bk: int, Lq: int) -> int:
    """Non-forced blocks kept for tile i: k + ceil(frac_num * n_causal / frac_den)."""
    n = causal_blocks(i, Qt, Bk, Lq)
    return k + (frac_num * n + frac_den - 1) // frac_den if frac_num else k


def decode_select(q, k, wl, kmax=None, sketch=None):
    """Decode selection: sketch -> scores -> top-k + {0, nb-1}.  Returns (idx, cnt, scores, sketch)."""
    if sketch is None:
        sketch = block_means(k, wl.L, wl.Bk)
    s = decode_scores(q, sketch, wl.Hkv, wl.scale)
    nb = wl.nb
    kmax = kmax or (wl.k + 2)
    idx, cnt = select(s, nb, nb - 1, wl.k, kmax)
    return idx, cnt, s, sketch


def decode_select_delta(q, k, wl, delta, cap, kmax=None, sketch=None):
    """Decode top-delta selection on sketch scores: pseudo-max from the sink and local blocks."""
    if sketch is None:
        sketch = block_means(k, wl.L, wl.Bk)
    s = decode_scores(q, sketch, wl.Hkv, wl.scale)
    nb = wl.nb
    kmax = kmax or (cap + 2)
    idx, cnt = select_delta(s, nb, nb - 1, delta, cap, kmax)
    return idx, cnt, s, sketch


def prefill_select(q, k, wl, units, kmax=None, sketch=None, scores=None):
    """Prefill selection for (g, i) units, from sketch scores (mode sketch) or given scores (mode mass)."""
    units = np.asarray(units, dtype=np.int64).reshape(-1, 2)
    if scores is None:
        if sketch is None:
            sketch = block_means(k, wl.L, wl.Bk)
        scores = prefill_scores(q, sketch, wl.Hkv, wl.Qt, wl.Bk, wl.scale, units)
    nvalid = np.array([causal_blocks(int(i), wl.Qt, wl.Bk, wl.L) for _, i in units], dtype=np.int64)
    budget = np.array([prefill_budget(int(i), wl.k, wl.frac_num, wl.frac_den, wl.Qt, wl.Bk, wl.L)
                       for _, i in units], dtype=np.int64)
    kmax = kmax or int(budget.max() + 2)
    idx, cnt = select(scores, nvalid, nvalid - 1, budget, kmax)
    return idx, cnt, scores, sketch


# ------------------------------------------------ head-collapsed token-level support

def token_mass_decode(q, k, Hkv, L, scale):
    """Head-collapsed token importance for decode ("How Much Dense Attention is Necessary?" Sec. 2.1
    and 2.2: the dense attention distribution of each query, averaged over the query heads into one
    distribution shared by every head; the T decode queries share one support, so they are averaged
    too).  P[b, j] = mean over all Hq heads and the T queries of the dense causal softmax probability
    of key j (query t sits at key position L - T + t).  Composed from `mass` at one-token blocks."""
    B, T, Hq, _ = q.shape
    units = [(g, 0) for g in range(B * Hkv)]
    m = mass(q, k, Hkv, L, L - T, T, 1, scale, units)  # [B*Hkv, L]: summed over each group's heads and rows
    return m.reshape(B, Hkv, L).sum(axis=1) / (Hq * T)


def token_select(P, k, kmax=None):
    """Token-level top-k on the shared distribution P [B, L]: the sink token 0 and the newest token
    L - 1 are forced, plus the k highest of the others (ties -> lower index), ascending."""
    B, L = P.shape
    kmax = kmax or (k + 2)
    return select(P, L, L - 1, k, kmax)


def token_attend(q, k, v, Hkv, L, scale, idx, cnt, rows):
    """Exact attention of (b, t, h) rows over the selected tokens idx [B, kmax] (shared by every kv
    head of batch row b); query t sits at key position L - T + t and is causal."""
    T = q.shape[1]
    idx_g = np.repeat(np.asarray(idx, dtype=np.int32), Hkv, axis=0)
    cnt_g = np.repeat(np.asarray(cnt, dtype=np.int32), Hkv)
    return attend(q, k, v, Hkv, L, L - T, 1, scale, rows, idx_g, cnt_g)


def token_mass_prefill(q, k, Hkv, L, scale):
    """Per-query head-collapsed token importance for causal prefill ("How Much Dense Attention is
    Necessary?" Sec. 2.1, per-query support b_sel = 1): P[b, t, j] = mean over all Hq heads of the dense
    causal softmax probability of key j for query t (zero for j > t).  Composed from `mass` at one-token
    blocks and one-query tiles."""
    B, Lq, Hq, _ = q.shape
    units = [(g, t) for g in range(B * Hkv) for t in range(Lq)]
    m = mass(q, k, Hkv, L, 0, 1, 1, scale, units)  # [B*Hkv*Lq, L]: summed over each group's heads
    return m.reshape(B, Hkv, Lq, L).sum(axis=1) / Hq


def token_select_prefill(P, k, kmax=None):
    """Per-query token top-k: for query t, tokens 0 and t forced plus the k highest of 1..t-1 (ties ->
    lower index), ascending.  P: [B, L, L].  Returns idx [B, L, kmax], cnt [B, L]."""
    B, Lq, L = P.shape
    kmax = kmax or (k + 2)
    t = np.arange(Lq, dtype=np.int64)
    nvalid = np.tile(t + 1, B)
    idx, cnt = select(P.reshape(B * Lq, L), nvalid, nvalid - 1, k, kmax)
    return idx.reshape(B, Lq, kmax), cnt.reshape(B, Lq)


def token_attend_prefill(q, k, v, Hkv, L, scale, idx, cnt, rows):
    """Exact causal attention of (b, t, h) rows over each query's own tokens idx [B, L, kmax] (shared
    by every kv head of batch row b)."""
    B, Lq = q.shape[0], q.shape[1]
    kmax = idx.shape[-1]
    idx_g = np.repeat(np.asarray(idx, dtype=np.int32), Hkv, axis=0).reshape(B * Hkv * Lq, kmax)
    cnt_g = np.repeat(np.asarray(cnt, dtype=np.int32), Hkv, axis=0).reshape(B * Hkv * Lq)
    return attend(q, k, v, Hkv, L, 0, 1, scale, rows, idx_g, cnt_g, nsel=Lq, rows_per_sel=1)
