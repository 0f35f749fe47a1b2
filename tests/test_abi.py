"""The C-ABI library: loads, exports every declared symbol, validates on the host.

No GPU is needed: every call below is rejected by host-side validation before
any CUDA call, or is a pure size query.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sa():
    import __graft_entry__
    __graft_entry__._load_builder().build()
    import top_block_sparse_pooled_b300 as m
    return m


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(sa_[a-z0-9_]+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(sa):
    declared = _declared_symbols()
    assert len(declared) >= 14
    for name in declared:
        assert hasattr(sa.lib, name), name
    # the binding covers every entry point under the same name
    assert declared <= set(sa.SIGNATURES)


def test_version_and_status_names(sa):
    assert sa.lib.sa_version() >= 100
    assert sa.lib.sa_status_name(0) == b"SA_OK"
    assert sa.lib.sa_status_name(4) == b"SA_ERR_TIMEOUT"


def test_kmax_queries(sa):
    # decode: forced {0, nb-1} + k candidates
    assert sa.sa_select_kmax(32768, 64, 0, False, 32) == 34
    assert sa.sa_select_kmax(64, 64, 0, False, 8) == 1      # one block: sink == local
    assert sa.sa_select_kmax(128, 64, 0, False, 8) == 2     # two blocks, no candidates
    assert sa.sa_select_kmax(4096, 64, 0, False, 8) == 10
    # prefill: k_i = ceil(2 * c_i / 100) over c_i = 1..nq, + 2 forced (capped by the candidates)
    assert sa.sa_select_kmax(131072, 128, 128, True, 0, 2, 100) == 23
    assert sa.sa_select_kmax(32768, 128, 128, True, 0, 2, 100) == 8
    assert sa.sa_select_kmax(128, 128, 128, True, 0, 2, 100) == 1
    assert sa.sa_select_kmax(0, 64, 0, False, 8) == -1


def test_budget_sublinear(sa):
    """k(L) = ceil(k_ref * (L/L_ref)^e), clamped to the candidate blocks (closed forms)."""
    f = sa.sa_budget_sublinear
    assert f(262144, 64, 80, 262144, 0.5) == 80            # the reference point
    assert f(65536, 64, 80, 262144, 0.5) == 40             # a quarter of the length: half the budget
    assert f(65536, 64, 80, 262144, 1.0) == 20             # exponent 1: a fixed fraction
    assert f(65536, 64, 80, 262144, 0.0) == 80             # exponent 0: a fixed budget
    assert f(32768, 64, 80, 262144, 0.5) == 29             # ceil(80 / sqrt(8)) = ceil(28.28)
    assert f(1024, 64, 80, 262144, 0.0) == 14              # clamped to nb - 2 candidates
    assert f(64, 64, 5, 64, 0.5) == 0                      # one block: no candidates
    ks = [f(L, 64, 80, 262144, 0.5) for L in (4096, 8192, 16384, 32768, 65536, 131072, 262144)]
    assert ks == sorted(ks)                                 # monotone in L
    for L in (8192, 32768):                                 # doubling L scales by 2^e (up to the ceiling)
        assert abs(f(2 * L, 64, 80, 262144, 0.5) - f(L, 64, 80, 262144, 0.5) * 2 ** 0.5) <= 2
    assert f(0, 64, 80, 262144, 0.5) == -1 and f(4096, 64, 80, 262144, 1.5) == -1


def test_workspace_queries(sa):
    assert sa.sa_decode_workspace_bytes(8, 1, 32, 8, 128, 34) >= 8 * 8 * 34 * 4 * 130 * 4
    assert sa.sa_decode_workspace_bytes(1, 1, 3, 2, 128, 10) == 0  # Hq not a multiple of Hkv
    assert sa.sa_decode_step_workspace_bytes(8, 1, 32, 8, 128, sa.SA_BF16, 34) > \
        sa.sa_decode_workspace_bytes(8, 1, 32, 8, 128, 34)


def _expect(sa, status_code, call):
    with pytest.raises(sa.SparseAttnError) as e:
        call()
    assert e.value.status == status_code, str(e.value)
    return str(e.value)


def test_invalid_arguments_rejected_on_host(sa):
    L = sa.lib
    # null pointers / bad shapes return without a launch
    st = L.sa_build_sketch(None, sa.SA_BF16, 1, 1, 64, 64, 128, 64, None, None)
    assert st == sa.SA_ERR_INVALID_ARG and b"null" in L.sa_last_error()
    st = L.sa_build_sketch(16, sa.SA_BF16, 1, 1, 128, 64, 128, 64, 16, None)  # L > L_stride
    assert st == sa.SA_ERR_INVALID_ARG
    st = L.sa_build_sketch(16, 7, 1, 1, 64, 64, 128, 64, 16, None)  # bad dtype
    assert st == sa.SA_ERR_INVALID_ARG and b"dtype" in L.sa_last_error()
    st = L.sa_build_sketch(16, sa.SA_BF16, 1, 1, 64, 64, 96, 64, 16, None)  # d unsupported
    assert st == sa.SA_ERR_UNSUPPORTED
    # decode: kmax too small for the workspace, block size unsupported, G*T too big
    args = [16, 16, 16, sa.SA_BF16, 16, 16, 34, 8, 1, 32, 8, 128, 32768, 32768, 64, 0.088, 16, 16, 0, None]
    st = L.sa_decode(*args)
    assert st == sa.SA_ERR_INVALID_ARG and b"workspace" in L.sa_last_error()
    bad = list(args)
    bad[14] = 128
    assert L.sa_decode(*bad) == sa.SA_ERR_UNSUPPORTED
    bad = list(args)
    bad[8], bad[9] = 16, 64  # T = 16, Hq = 64 -> G*T = 128
    assert L.sa_decode(*bad) == sa.SA_ERR_UNSUPPORTED
    bad = list(args)
    bad[1] = 17  # misaligned cache
    bad[17] = 1 << 30
    assert L.sa_decode(*bad) == sa.SA_ERR_INVALID_ARG
    # select: kmax smaller than the selection needs
    st = L.sa_select_topk(sa.SA_SELECT_SKETCH, 16, sa.SA_BF16, 16, None, 8, 1, 32, 8, 128, 32768, 32768, 64, 0, 0,
                          32, 0, 1, 0.088, 16, 16, 33, None)
    assert st == sa.SA_ERR_INVALID_ARG and b"kmax" in L.sa_last_error()
    # select: MASS mode without scores
    st = L.sa_select_topk(sa.SA_SELECT_MASS, None, sa.SA_BF16, None, None, 1, 32768, 16, 2, 128, 32768, 32768, 128,
                          128, 1, 0, 2, 100, 0.088, 16, 16, 8, None)
    assert st == sa.SA_ERR_INVALID_ARG
    # prefill: unsupported dtype / tile shape
    st = L.sa_prefill(16, 16, 16, sa.SA_F32, 16, 16, 8, 1, 4096, 16, 2, 128, 128, 128, 0.088, 16, None, None)
    assert st == sa.SA_ERR_UNSUPPORTED
    st = L.sa_prefill(16, 16, 16, sa.SA_BF16, 16, 16, 8, 1, 4096, 16, 2, 128, 64, 128, 0.088, 16, None, None)
    assert st == sa.SA_ERR_UNSUPPORTED
    # append past the cache
    st = L.sa_append_kv(16, 16, sa.SA_BF16, 1, 1, 4, 128, 16, 16, 64, 62, 64, 16, None)
    assert st == sa.SA_ERR_INVALID_ARG
    # top-delta: negative delta or cap rejected on the host
    st = L.sa_select_topdelta(16, sa.SA_BF16, 16, None, 8, 1, 32, 8, 128, 32768, 32768, 64, -1.0, 32, 0.088, 16, 16,
                              34, None)
    assert st == sa.SA_ERR_INVALID_ARG and b"delta" in L.sa_last_error()
    st = L.sa_select_topdelta(16, sa.SA_BF16, 16, None, 8, 1, 32, 8, 128, 32768, 32768, 64, 0.5, -2, 0.088, 16, 16,
                              34, None)
    assert st == sa.SA_ERR_INVALID_ARG
    # token mass: fp32 unsupported, G*T > 16 unsupported, a short workspace rejected
    st = L.sa_token_mass_decode(16, 16, sa.SA_F32, 1, 1, 8, 2, 128, 64, 64, 0.1, 16, 16, 1 << 30, None)
    assert st == sa.SA_ERR_UNSUPPORTED
    st = L.sa_token_mass_decode(16, 16, sa.SA_BF16, 1, 4, 32, 4, 128, 64, 64, 0.1, 16, 16, 1 << 30, None)
    assert st == sa.SA_ERR_UNSUPPORTED and b"G*T" in L.sa_last_error()
    st = L.sa_token_mass_decode(16, 16, sa.SA_BF16, 1, 1, 8, 2, 128, 64, 64, 0.1, 16, 16, 64, None)
    assert st == sa.SA_ERR_INVALID_ARG and b"workspace" in L.sa_last_error()
    st = L.sa_token_mass_decode(16, 16, sa.SA_BF16, 1, 8, 8, 8, 128, 4, 64, 0.1, 16, 16, 1 << 30, None)
    assert st == sa.SA_ERR_INVALID_ARG  # T > L
    # token decode: bf16 only, null pointers rejected
    st = L.sa_decode_tokens(16, 16, 16, sa.SA_F32, 16, 16, 8, 1, 1, 8, 2, 128, 64, 64, 0.1, 16, 16, 1 << 30, None)
    assert st == sa.SA_ERR_UNSUPPORTED
    st = L.sa_decode_tokens(16, None, 16, sa.SA_BF16, 16, 16, 8, 1, 1, 8, 2, 128, 64, 64, 0.1, 16, 16, 1 << 30, None)
    assert st == sa.SA_ERR_INVALID_ARG
    # given decode scores may be longer than the shared-memory limit; given prefill scores may not
    st = L.sa_select_topk(sa.SA_SELECT_MASS, None, sa.SA_BF16, None, None, 1, 1, 1, 1, 128, 262144, 262144, 1, 0, 0,
                          2048, 0, 1, 1.0, 16, 16, 2050, None)
    assert st == sa.SA_ERR_INVALID_ARG and b"scores" in L.sa_last_error()  # only the missing array is wrong
    st = L.sa_select_topk(sa.SA_SELECT_MASS, None, sa.SA_BF16, None, 16, 1, 262144, 1, 1, 128, 262144, 262144, 1, 128,
                          1, 8, 0, 1, 1.0, 16, 16, 2050, None)
    assert st == sa.SA_ERR_UNSUPPORTED
    # per-query prefill: L past the grid limit, fp32, a short workspace, G > 16 for the token prefill
    st = L.sa_token_mass_prefill(16, 16, sa.SA_BF16, 1, 70000, 8, 2, 128, 0.1, 16, 16, 1 << 40, None)
    assert st == sa.SA_ERR_INVALID_ARG
    st = L.sa_token_mass_prefill(16, 16, sa.SA_F32, 1, 64, 8, 2, 128, 0.1, 16, 16, 1 << 30, None)
    assert st == sa.SA_ERR_UNSUPPORTED
    st = L.sa_token_mass_prefill(16, 16, sa.SA_BF16, 1, 64, 8, 2, 128, 0.1, 16, 16, 64, None)
    assert st == sa.SA_ERR_INVALID_ARG and b"workspace" in L.sa_last_error()
    st = L.sa_prefill_tokens(16, 16, 16, sa.SA_BF16, 16, 16, 8, 1, 64, 64, 2, 128, 0.1, 16, 16, 1 << 30, None)
    assert st == sa.SA_ERR_UNSUPPORTED  # G = 32 > 16
    st = L.sa_prefill_tokens(16, 16, 16, sa.SA_BF16, 16, 16, 8, 1, 64, 8, 2, 128, 0.1, 16, 16, 64, None)
    assert st == sa.SA_ERR_INVALID_ARG and b"workspace" in L.sa_last_error()
    st = L.sa_prefill_tokens(16, 16, 16, sa.SA_BF16, 16, 16, 8, 1 << 20, 1 << 20, 8, 2, 128, 0.1, 16, 16, 1 << 30,
                             None)
    assert st == sa.SA_ERR_INVALID_ARG  # B*L*Hkv past 2^24
    # workspace queries of the token paths grow with their inputs and reject bad shapes
    assert sa.sa_token_mass_prefill_workspace_bytes(1, 4096, 32, 8) > sa.sa_token_mass_prefill_workspace_bytes(1, 2048,
                                                                                                               32, 8)
    assert sa.sa_token_mass_prefill_workspace_bytes(1, 4096, 32, 7) == 0
    assert sa.sa_prefill_tokens_workspace_bytes(1, 4096, 32, 8, 128, 258) > 0
    assert sa.sa_token_mass_workspace_bytes(1, 4, 32, 8, 262144) >= 8 * 16 * 262144 * 4
    # the decode step rejects null buffers and a short workspace before any launch
    st = L.sa_decode_step(None, 16, 16, sa.SA_BF16, 16, 16, 16, 8, 1, 32, 8, 128, 32768, 32768, 64, 32, 0.08, 16, 16,
                          34, None, 16, 0, 16, 1 << 30, None)
    assert st == sa.SA_ERR_INVALID_ARG
    st = L.sa_decode_step(16, 16, 16, sa.SA_BF16, 16, 16, 16, 8, 1, 32, 8, 128, 32768, 32768, 64, 32, 0.08, 16, 16,
                          34, None, 16, 0, 16, 64, None)
    assert st == sa.SA_ERR_INVALID_ARG and b"workspace" in L.sa_last_error()
    # fused selection + decode: shapes outside the cluster kernel, a short kmax, null caches
    sd = [16, sa.SA_BF16, 16, 16, 16, 8, 1, 32, 8, 128, 32768, 32768, 64, 32, 0.088, 16, 16, 34, None, 16, None]
    bad = list(sd)
    bad[1] = sa.SA_F32
    assert L.sa_select_decode(*bad) == sa.SA_ERR_UNSUPPORTED
    bad = list(sd)
    bad[6] = 8  # T = 8: G*T = 32
    bad[17] = 34
    assert L.sa_select_decode(*bad) == sa.SA_ERR_UNSUPPORTED and b"G*T" in L.sa_last_error()
    bad = list(sd)
    bad[12] = 128  # block 128
    bad[17] = 34
    assert L.sa_select_decode(*bad) == sa.SA_ERR_UNSUPPORTED
    bad = list(sd)
    bad[17] = 33  # kmax below the selection's 34
    assert L.sa_select_decode(*bad) == sa.SA_ERR_INVALID_ARG and b"kmax" in L.sa_last_error()
    bad = list(sd)
    bad[3] = None  # no key cache
    assert L.sa_select_decode(*bad) == sa.SA_ERR_INVALID_ARG and b"null" in L.sa_last_error()
    # the bounded-wait self-test rejects a limit outside [1 ms, 1 s] before any launch
    assert L.sa_selftest_wait_timeout(5, None) == sa.SA_ERR_INVALID_ARG
    assert L.sa_selftest_wait_timeout(5_000_000_000, None) == sa.SA_ERR_INVALID_ARG
    # the scratch poisoning self-test takes 1 .. 8 MiB
    assert L.sa_selftest_poison_noalloc(0, None) == sa.SA_ERR_INVALID_ARG
    assert L.sa_selftest_poison_noalloc(9 << 20, None) == sa.SA_ERR_INVALID_ARG
    # device status needs an output pointer
    assert L.sa_device_status(None, 0) == sa.SA_ERR_INVALID_ARG


def test_binding_raises_with_message(sa):
    msg = _expect(sa, sa.SA_ERR_INVALID_ARG,
                  lambda: sa._check(sa.lib.sa_build_sketch(None, 1, 1, 1, 64, 64, 128, 64, None, None)))
    assert "null" in msg


def test_package_has_no_cpu_fallback():
    """The product package never imports the oracle or the generator."""
    pkg = os.path.join(ROOT, "top_block_sparse_pooled_b300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "oracle.c" not in text and "liboracle" not in text, fn
