"""GPU parity of the head-collapsed token-level decode path against the CPU oracle:
token mass (dense distribution averaged over all heads and decode queries), token
top-k (given-score selection, including arrays longer than shared memory holds) and
attention over the selected tokens shared by every kv head."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, assert_selection, dev, host

pytestmark = pytest.mark.gpu

# mass: |gpu - oracle| <= MASS_RTOL * oracle + MASS_ATOL.  The GPU logits carry
# fp32 rounding (about 1e-6 of |logit|, logits up to ~20 in base 2), which exp2
# turns into a relative error of about 2e-5 of the probability.
MASS_RTOL = 1e-4
MASS_ATOL = 1e-9


@pytest.fixture(scope="module")
def sa():
    import top_block_sparse_pooled_b300 as m
    return m


def _check_status(sa):
    assert sa.sa_device_status(clear=True) == 0


TOKEN_CASES = {
    # GQA decode with four queries (G*T = 16), odd L (scalar logit stores)
    "g4t4_odd": synth.WORKLOADS["c3"].replace(L=8192 + 5, k=256, needles=6, seed=91),
    # d = 64, two batch rows, one query
    "d64_b2": synth.WORKLOADS["c2"].replace(B=2, Hq=8, Hkv=4, d=64, L=3000, k=100, needles=3, seed=92),
    # longer than the shared-memory top-k (scores read from L2), G*T = 16 with G = 8
    "long_g8": synth.WORKLOADS["c3"].replace(T=2, Hq=16, Hkv=2, L=20000, k=512, needles=8, seed=93),
}


def _token_mass(sa, wl, x):
    q, k = dev(x.q), dev(x.k)
    ws = torch.empty(sa.sa_token_mass_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.L), dtype=torch.uint8,
                     device="cuda")
    mass = torch.empty((wl.B, wl.L), dtype=torch.float32, device="cuda")
    sa.sa_token_mass_decode(q, k, wl.L, wl.scale, mass, ws)
    torch.cuda.synchronize()
    _check_status(sa)
    return mass


def _token_select(sa, wl, mass, k):
    kmax = sa.sa_select_kmax(wl.L, 1, 0, False, k)
    idx = torch.full((wl.B, 1, 1, kmax), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((wl.B, 1, 1), dtype=torch.int32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, mass.reshape(wl.B, 1, 1, wl.L), 1, wl.L, wl.L, 1, 0, False, k,
                      0, 1, 1.0, idx, cnt, d=wl.d, dtype=sa.SA_F32, B=wl.B, Tq=1, Hq=1)
    torch.cuda.synchronize()
    _check_status(sa)
    return idx.reshape(wl.B, kmax), cnt.reshape(wl.B)


def _token_decode(sa, wl, x, idx, cnt):
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    kmax = idx.shape[-1]
    ws = torch.zeros(sa.sa_decode_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, kmax), dtype=torch.uint8,
                     device="cuda")
    out = torch.full_like(q, float("nan"))
    sa.sa_decode_tokens(q, k, v, idx, cnt, wl.L, wl.scale, out, ws)
    torch.cuda.synchronize()
    _check_status(sa)
    return out


def _rows(wl):
    return [(b, t, h) for b in range(wl.B) for t in range(wl.T) for h in range(wl.Hq)]


@pytest.mark.parametrize("name", sorted(TOKEN_CASES))
def test_token_mass_matches_oracle(sa, name):
    wl = TOKEN_CASES[name]
    x = synth.make_inputs(wl)
    got = host(_token_mass(sa, wl, x))
    ref = oracle.token_mass_decode(x.q, x.k, wl.Hkv, wl.L, wl.scale)
    assert_close(got, ref, atol=MASS_ATOL, rtol=MASS_RTOL, what="token mass")
    assert np.all(np.abs(got.sum(axis=1) - 1.0) < 1e-4)


@pytest.mark.parametrize("name", sorted(TOKEN_CASES))
def test_token_select_matches_oracle(sa, name):
    wl = TOKEN_CASES[name]
    x = synth.make_inputs(wl)
    mass = _token_mass(sa, wl, x)
    idx, cnt = _token_select(sa, wl, mass, wl.k)
    P = oracle.token_mass_decode(x.q, x.k, wl.Hkv, wl.L, wl.scale)
    o_idx, o_cnt = oracle.token_select(P, wl.k, kmax=idx.shape[-1])
    assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, P, what=name)


@pytest.mark.parametrize("n", [3, 16384, 16385, 40000, 262144, 300000])
def test_long_given_selection_exact(sa, n):
    """Given float32 scores with many exact ties: the GPU selection equals the oracle's, bit for bit."""
    r = np.random.default_rng(n)
    B = 3
    s = (r.integers(-40, 41, size=(B, n)) * 0.25).astype(np.float32)
    s[2] = 1.5  # all equal: the lowest indices win
    for k in (0, 1, 37, 2048, n):
        kmax = max(1, min(k, max(n - 2, 0)) + 2)
        idx = torch.full((B, 1, 1, kmax), -7, dtype=torch.int32, device="cuda")
        cnt = torch.zeros((B, 1, 1), dtype=torch.int32, device="cuda")
        sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, torch.from_numpy(s).cuda().reshape(B, 1, 1, n), 1, n, n, 1,
                          0, False, k, 0, 1, 1.0, idx, cnt, d=128, dtype=sa.SA_F32, B=B, Tq=1, Hq=1)
        torch.cuda.synchronize()
        _check_status(sa)
        o_idx, o_cnt = oracle.select(s.astype(np.float64), n, n - 1, k, kmax)
        g_idx, g_cnt = idx.cpu().numpy().reshape(B, kmax), cnt.cpu().numpy().reshape(B)
        assert np.array_equal(g_cnt, o_cnt), (k, g_cnt, o_cnt)
        assert np.array_equal(g_idx, o_idx), k


@pytest.mark.parametrize("name", sorted(TOKEN_CASES))
def test_token_decode_matches_oracle(sa, name):
    wl = TOKEN_CASES[name]
    x = synth.make_inputs(wl)
    P = oracle.token_mass_decode(x.q, x.k, wl.Hkv, wl.L, wl.scale)
    o_idx, o_cnt = oracle.token_select(P, wl.k)
    out = _token_decode(sa, wl, x, torch.from_numpy(o_idx).cuda(), torch.from_numpy(o_cnt).cuda())
    rows = _rows(wl)
    ref, _ = oracle.token_attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.scale, o_idx, o_cnt, rows)
    got = host(out).reshape(-1, wl.d)
    assert_close(got, ref, what="token decode " + name)


def test_token_decode_short_and_out_of_range_lists(sa):
    """Counts below kmax, a partial last chunk, entries at or past L, and a single token."""
    wl = TOKEN_CASES["d64_b2"]
    x = synth.make_inputs(wl)
    r = np.random.default_rng(5)
    kmax = 150
    idx = np.full((wl.B, kmax), -1, dtype=np.int32)
    cnt = np.array([1, 97], dtype=np.int32)
    idx[0, 0] = wl.L - 1
    sel = np.sort(r.choice(wl.L, size=96, replace=False)).astype(np.int32)
    idx[1, :96] = sel
    idx[1, 96] = wl.L + 5  # past the cache: ignored
    out = _token_decode(sa, wl, x, torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda())
    o_idx = idx.copy()
    o_cnt = cnt.copy()
    o_cnt[1] = 96  # the oracle is given only the in-range entries
    ref, _ = oracle.token_attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.scale, o_idx, o_cnt, _rows(wl))
    assert_close(host(out).reshape(-1, wl.d), ref, what="short token lists")


def test_token_pipeline_full_size(sa):
    """One sequence of 256K tokens, 32 query heads on 8 kv heads, four decode queries, 2048 selected
    tokens: token mass everywhere, the selection (near-tie rule) and the outputs over the GPU's own
    selection."""
    wl = synth.WORKLOADS["c3"].replace(k=2048)
    x = synth.make_inputs(wl)
    mass = _token_mass(sa, wl, x)
    idx, cnt = _token_select(sa, wl, mass, wl.k)
    P = oracle.token_mass_decode(x.q, x.k, wl.Hkv, wl.L, wl.scale)
    assert_close(host(mass), P, atol=MASS_ATOL, rtol=MASS_RTOL, what="token mass (full size)")
    o_idx, o_cnt = oracle.token_select(P, wl.k, kmax=idx.shape[-1])
    g_idx, g_cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    assert_selection(g_idx, g_cnt, o_idx, o_cnt, P, what="full size")
    out = _token_decode(sa, wl, x, idx, cnt)
    ref, _ = oracle.token_attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.scale, g_idx, g_cnt, _rows(wl))
    assert_close(host(out).reshape(-1, wl.d), ref, what="token decode (full size)")


# ---------------------------------------------------------------- per-query prefill (b_sel = 1)

PREFILL_CASES = {
    # odd length, G = 4
    "g4_odd": synth.WORKLOADS["c5"].replace(B=1, Hq=8, Hkv=2, L=300, k=16, needles=3, seed=101),
    # d = 64, G = 1, two batch rows
    "d64_g1_b2": synth.WORKLOADS["c5"].replace(B=2, Hq=4, Hkv=4, d=64, L=257, k=32, needles=2, seed=102),
    # G = 16 (one M tile per query), budget past most rows' candidates
    "g16": synth.WORKLOADS["c5"].replace(B=1, Hq=32, Hkv=2, L=200, k=150, needles=2, seed=103),
    # two batch rows, several 128-query tiles and a ragged last one (the tensor-core path: d = 128)
    "g4_b2_tiles": synth.WORKLOADS["c5"].replace(B=2, Hq=8, Hkv=2, L=128 * 3 + 40, k=40, needles=3, seed=105),
}


def _prefill_mass(sa, wl, x):
    q, k = dev(x.q), dev(x.k)
    ws = torch.empty(sa.sa_token_mass_prefill_workspace_bytes(wl.B, wl.L, wl.Hq, wl.Hkv), dtype=torch.uint8,
                     device="cuda")
    mass = torch.empty((wl.B, wl.L, wl.L), dtype=torch.float32, device="cuda")
    sa.sa_token_mass_prefill(q, k, wl.scale, mass, ws)
    torch.cuda.synchronize()
    _check_status(sa)
    return mass


def _prefill_select(sa, wl, mass, k):
    kmax = sa.sa_select_kmax(wl.L, 1, 1, True, k)
    idx = torch.full((wl.B, 1, wl.L, kmax), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((wl.B, 1, wl.L), dtype=torch.int32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, mass.reshape(wl.B, 1, wl.L, wl.L), 1, wl.L, wl.L, 1, 1, True,
                      k, 0, 1, 1.0, idx, cnt, d=wl.d, dtype=sa.SA_F32, B=wl.B, Tq=wl.L, Hq=1)
    torch.cuda.synchronize()
    _check_status(sa)
    return idx.reshape(wl.B, wl.L, kmax), cnt.reshape(wl.B, wl.L)


def _prefill_tokens(sa, wl, x, idx, cnt):
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    kmax = idx.shape[-1]
    ws = torch.zeros(sa.sa_prefill_tokens_workspace_bytes(wl.B, wl.L, wl.Hq, wl.Hkv, wl.d, kmax), dtype=torch.uint8,
                     device="cuda")
    out = torch.full_like(q, float("nan"))
    sa.sa_prefill_tokens(q, k, v, idx, cnt, wl.scale, out, ws)
    torch.cuda.synchronize()
    _check_status(sa)
    return out


def _prefill_rows(wl):
    return [(b, t, h) for b in range(wl.B) for t in range(wl.L) for h in range(wl.Hq)]


@pytest.mark.parametrize("name", sorted(PREFILL_CASES))
def test_token_mass_prefill_matches_oracle(sa, name):
    wl = PREFILL_CASES[name]
    x = synth.make_inputs(wl)
    got = host(_prefill_mass(sa, wl, x))
    ref = oracle.token_mass_prefill(x.q, x.k, wl.Hkv, wl.L, wl.scale)
    assert_close(got, ref, atol=MASS_ATOL, rtol=MASS_RTOL, what="per-query token mass")
    assert np.all(np.abs(got.sum(axis=2) - 1.0) < 1e-4)
    assert np.all(np.triu(got, 1) == 0.0)  # no mass on future keys


@pytest.mark.parametrize("name", sorted(PREFILL_CASES))
def test_token_select_prefill_matches_oracle(sa, name):
    wl = PREFILL_CASES[name]
    x = synth.make_inputs(wl)
    idx, cnt = _prefill_select(sa, wl, _prefill_mass(sa, wl, x), wl.k)
    P = oracle.token_mass_prefill(x.q, x.k, wl.Hkv, wl.L, wl.scale)
    o_idx, o_cnt = oracle.token_select_prefill(P, wl.k, kmax=idx.shape[-1])
    kmax = idx.shape[-1]
    assert_selection(idx.cpu().numpy().reshape(-1, kmax), cnt.cpu().numpy().reshape(-1),
                     o_idx.reshape(-1, kmax), o_cnt.reshape(-1), P.reshape(-1, wl.L), what=name)


@pytest.mark.parametrize("name", sorted(PREFILL_CASES))
def test_prefill_tokens_matches_oracle(sa, name):
    wl = PREFILL_CASES[name]
    x = synth.make_inputs(wl)
    P = oracle.token_mass_prefill(x.q, x.k, wl.Hkv, wl.L, wl.scale)
    o_idx, o_cnt = oracle.token_select_prefill(P, wl.k)
    out = _prefill_tokens(sa, wl, x, torch.from_numpy(o_idx).cuda(), torch.from_numpy(o_cnt).cuda())
    ref, _ = oracle.token_attend_prefill(x.q, x.k, x.v, wl.Hkv, wl.L, wl.scale, o_idx, o_cnt, _prefill_rows(wl))
    assert_close(host(out).reshape(-1, wl.d), ref, what="per-query prefill " + name)


def test_prefill_tokens_pipeline_1k(sa):
    """1024 queries, 32 heads on 8 kv heads, 64 tokens per query: the GPU's mass, its selection (near-tie
    rule against the oracle) and the outputs over the GPU's own selection on every row."""
    wl = synth.WORKLOADS["c5"].replace(B=1, L=1024, k=64, needles=4, seed=104)
    x = synth.make_inputs(wl)
    mass = _prefill_mass(sa, wl, x)
    idx, cnt = _prefill_select(sa, wl, mass, wl.k)
    P = oracle.token_mass_prefill(x.q, x.k, wl.Hkv, wl.L, wl.scale)
    assert_close(host(mass), P, atol=MASS_ATOL, rtol=MASS_RTOL, what="per-query token mass (1k)")
    kmax = idx.shape[-1]
    o_idx, o_cnt = oracle.token_select_prefill(P, wl.k, kmax=kmax)
    g_idx, g_cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    assert_selection(g_idx.reshape(-1, kmax), g_cnt.reshape(-1), o_idx.reshape(-1, kmax), o_cnt.reshape(-1),
                     P.reshape(-1, wl.L), what="1k")
    out = _prefill_tokens(sa, wl, x, idx, cnt)
    ref, _ = oracle.token_attend_prefill(x.q, x.k, x.v, wl.Hkv, wl.L, wl.scale, g_idx, g_cnt, _prefill_rows(wl))
    assert_close(host(out).reshape(-1, wl.d), ref, what="per-query prefill (1k)")


def test_prefill_tokens_ignores_invalid_entries(sa):
    """Lists with entries that are not tokens of the query's support (negative, future, past L) and
    counts below the list length: only the valid entries j <= t before the count are attended."""
    wl = synth.WORKLOADS["c5"].replace(B=1, Hq=8, Hkv=2, L=300, k=24, needles=2, seed=106)
    x = synth.make_inputs(wl)
    rng = np.random.default_rng(7)
    kmax = 32
    idx = np.full((wl.B, wl.L, kmax), -1, dtype=np.int32)
    cnt = np.zeros((wl.B, wl.L), dtype=np.int32)
    clean = np.full_like(idx, -1)
    ccnt = np.zeros_like(cnt)
    for b in range(wl.B):
        for t in range(wl.L):
            own = rng.choice(t + 1, size=min(t + 1, 20), replace=False)
            bad = np.array([-1, -5, t + 1 + rng.integers(0, 50), wl.L + 3], dtype=np.int64)
            row = np.concatenate([own, bad])
            rng.shuffle(row)
            n = min(len(row), kmax - 2)
            idx[b, t, :n] = row[:n]
            idx[b, t, n:n + 2] = [0, t]  # past the count: must be ignored
            cnt[b, t] = n
            keep = np.sort([j for j in row[:n] if 0 <= j <= t])
            clean[b, t, :len(keep)] = keep
            ccnt[b, t] = len(keep)
    out = _prefill_tokens(sa, wl, x, torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda())
    ref, _ = oracle.token_attend_prefill(x.q, x.k, x.v, wl.Hkv, wl.L, wl.scale, clean, ccnt, _prefill_rows(wl))
    assert_close(host(out).reshape(-1, wl.d), ref, what="per-query prefill, invalid entries")
