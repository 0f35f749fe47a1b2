"""Seeded synthetic workloads for top-k block-sparse GQA attention.

This package builds inputs only.  It holds the workload table (shapes, budget
parameters, seeds and plant recipes) and a counter-based generator written in C
(``synth.c``), and it contains none of the attention method's arithmetic.  The
CUDA path and the CPU oracle both consume the exact bits produced here: bf16
tensors are returned as ``numpy.uint16`` bit patterns, fp32 tensors as
``numpy.float32``.

Workloads follow the shapes the pages evaluate (long contexts of 4K-256K, a
few percent of blocks kept; "How Much Dense Attention is Necessary?" Sec. 3.1,
"Faster Than Flash" Results, "The Sparse Frontier" RQ3) and stand in for the
benchmark suites named there (RULER, LongBench), which are not available.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")

# stream ids of the counter generator
_S_Q, _S_K, _S_V, _S_BASIS, _S_NEEDLE = 1, 3, 5, 7, 11
_NEEDLE_SEED_XOR = 0x5EED


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so beside it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i, l, u64, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_uint64, ctypes.c_double
        lib.sy_fill_normal.argtypes = [vp, i, ctypes.c_size_t, u64, u64]
        lib.sy_make_queries.argtypes = [vp, i, l, l, l, l, l, u64, u64, vp, l, d]
        lib.sy_make_keys.argtypes = [vp, i, l, l, l, l, l, u64, u64, vp, vp, d, vp, l, d]
        lib.sy_needle_direction.argtypes = [vp, i, l, l, l, l, l, vp]
        lib.sy_needle_blocks.argtypes = [vp, l, l, l, l, l, u64, u64]
        lib.sy_orthonormal_basis.argtypes = [vp, l, l, l, u64, u64]
        lib.sy_normal_at.argtypes = [u64, u64]
        lib.sy_normal_at.restype = d
        lib.sy_stream_key.argtypes = [u64, u64]
        lib.sy_stream_key.restype = u64
        lib.sy_num_threads.restype = i
        _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload.

    kind: "decode" (T query tokens at positions L-T..L-1 against an L-token
    cache) or "prefill" (L causal queries in tiles of Qt).  Budget: decode keeps
    ``k`` non-forced blocks; prefill tile i keeps k + ceil(frac_num*(i+1)/frac_den)
    non-forced blocks (i+1 = its causal blocks when Qt == Bk).  Forced blocks
    (always kept): the sink block 0 and the local block (decode: last block;
    prefill: the diagonal block).
    """
    name: str
    kind: str
    B: int
    Hq: int
    Hkv: int
    d: int
    L: int
    Bk: int
    dtype: str  # "f32" or "bf16"
    T: int = 1
    Qt: int = 128
    k: int = 0
    frac_num: int = 0
    frac_den: int = 1
    mode: str = "sketch"  # "sketch" or "mass"
    needles: int = 0
    alpha: float = 0.0
    plant_rank: int = 0
    gamma: float = 0.0
    seed: int = 1000

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def nb(self) -> int:
        return (self.L + self.Bk - 1) // self.Bk

    @property
    def Tq(self) -> int:
        return self.T if self.kind == "decode" else self.L

    @property
    def nq(self) -> int:
        return 1 if self.kind == "decode" else (self.L + self.Qt - 1) // self.Qt

    @property
    def esize(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads (decode c1-c3, prefill c4-c5).
WORKLOADS = {
    "c1": Workload("c1", "decode", B=1, Hq=4, Hkv=1, d=64, L=4096, Bk=64, dtype="f32", T=1,
                   k=8, needles=2, alpha=3.0, seed=1001),
    "c2": Workload("c2", "decode", B=8, Hq=32, Hkv=8, d=128, L=32768, Bk=64, dtype="bf16", T=1,
                   k=32, needles=5, alpha=2.0, seed=1002),
    "c3": Workload("c3", "decode", B=1, Hq=32, Hkv=8, d=128, L=262144, Bk=64, dtype="bf16", T=4,
                   k=80, needles=20, alpha=2.0, seed=1003),
    "c4": Workload("c4", "prefill", B=1, Hq=16, Hkv=2, d=128, L=32768, Bk=128, Qt=128, dtype="bf16",
                   frac_num=2, frac_den=100, mode="mass", plant_rank=4, gamma=4.0, seed=1004),
    "c5": Workload("c5", "prefill", B=2, Hq=32, Hkv=8, d=128, L=131072, Bk=128, Qt=128, dtype="bf16",
                   frac_num=2, frac_den=100, needles=10, alpha=2.0, seed=1005),
}


@dataclasses.dataclass
class Inputs:
    wl: Workload
    q: np.ndarray        # [B, Tq, Hq, d]
    k: np.ndarray        # [B, Hkv, L, d]
    v: np.ndarray        # [B, Hkv, L, d]
    needle_mask: np.ndarray  # [B*Hkv, nb] uint8
    is_bf16: bool


def _empty(shape, is_bf16):
    return np.empty(shape, dtype=np.uint16 if is_bf16 else np.float32)


def make_inputs(wl: Workload) -> Inputs:
    """Generate q, k, v for a workload (deterministic in wl.seed)."""
    lib = _L()
    bf = wl.dtype == "bf16"
    ib = 1 if bf else 0
    ng = wl.B * wl.Hkv
    U = None
    if wl.plant_rank:
        U = np.empty((ng, wl.d, wl.plant_rank), dtype=np.float64)
        lib.sy_orthonormal_basis(_p(U), ng, wl.d, wl.plant_rank, wl.seed, _S_BASIS)
    q = _empty((wl.B, wl.Tq, wl.Hq, wl.d), bf)
    lib.sy_make_queries(_p(q), ib, wl.B, wl.Tq, wl.Hq, wl.Hkv, wl.d, wl.seed, _S_Q,
                        _p(U), wl.plant_rank, float(wl.gamma))
    mask = np.zeros((ng, wl.nb), dtype=np.uint8)
    qhat = None
    if wl.needles and wl.nb > 2:
        qhat = np.empty((ng, wl.d), dtype=np.float64)
        lib.sy_needle_direction(_p(q), ib, wl.B, wl.Tq, wl.Hq, wl.Hkv, wl.d, _p(qhat))
        lib.sy_needle_blocks(_p(mask), ng, wl.nb, 1, wl.nb - 2, wl.needles,
                             wl.seed ^ _NEEDLE_SEED_XOR, _S_NEEDLE)
    k = _empty((wl.B, wl.Hkv, wl.L, wl.d), bf)
    lib.sy_make_keys(_p(k), ib, wl.B, wl.Hkv, wl.L, wl.d, wl.Bk, wl.seed, _S_K,
                     _p(mask) if qhat is not None else None, _p(qhat), float(wl.alpha),
                     _p(U), wl.plant_rank, float(wl.gamma))
    v = _empty((wl.B, wl.Hkv, wl.L, wl.d), bf)
    lib.sy_fill_normal(_p(v), ib, v.size, wl.seed, _S_V)
    return Inputs(wl, q, k, v, mask, bf)


def normal(n: int, seed: int, stream: int, bf16: bool) -> np.ndarray:
    """A flat N(0,1) tensor of n elements (bf16 bits or float32)."""
    out = _empty((n,), bf16)
    _L().sy_fill_normal(_p(out), 1 if bf16 else 0, n, seed, stream)
    return out


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(a: np.ndarray) -> np.ndarray:
    return bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def threads() -> int:
    return int(_L().sy_num_threads())
