"""GPU top-k selection against the oracle's brute-force-pinned selection, over
many sizes, budgets and tie patterns (mass mode: scores given), and the decode
sketch selection at small block counts."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_selection, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    import top_block_sparse_pooled_b300 as m
    return m


@pytest.mark.parametrize("n", [3, 4, 5, 7, 31, 32, 33, 64, 100, 257, 1000, 4096, 16384])
def test_select_given_scores_brute_force(sa, n):
    """One selection per group over n blocks (block = 1 key), forced {0, n-1}."""
    rng = np.random.default_rng(n)
    groups = 6
    budgets = [0, 1, 2, max(0, n // 3), max(0, n - 3), n]
    for trial, k in enumerate(budgets):
        # coarse values make many exact ties; the last group has all-equal scores
        s = rng.integers(-4, 5, size=(groups, n)).astype(np.float32) * 0.25
        s[-1] = 1.0
        kmax = sa.sa_select_kmax(n, 1, 0, False, k)
        scores = torch.from_numpy(s.reshape(1, groups, 1, n)).cuda()
        idx = torch.full((1, groups, 1, kmax), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((1, groups, 1), -7, dtype=torch.int32, device="cuda")
        sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, scores, groups, n, n, 1, 0, False, k, 0, 1, 1.0,
                          idx, cnt, d=128, dtype=sa.SA_BF16, B=1, Tq=1, Hq=groups)
        torch.cuda.synchronize()
        assert sa.sa_device_status(clear=True) == 0
        o_idx, o_cnt = oracle.select(s.astype(np.float64), n, n - 1, k, kmax)
        # exact ties must resolve to the lower index: bit-exact, no swaps
        g_idx = idx.cpu().numpy().reshape(groups, kmax)
        g_cnt = cnt.cpu().numpy().reshape(groups)
        for g in range(groups):
            assert g_cnt[g] == o_cnt[g] and np.array_equal(g_idx[g], o_idx[g]), (
                "n=%d k=%d group %d: gpu %s (cnt %d), oracle %s (cnt %d)" % (
                    n, k, g, g_idx[g][:12].tolist(), g_cnt[g], o_idx[g][:12].tolist(), o_cnt[g]))


@pytest.mark.parametrize("nb", [3, 4, 5, 9, 33])
def test_decode_select_small_block_counts(sa, nb):
    wl = synth.WORKLOADS["c2"].replace(B=2, L=64 * nb - 5, k=2, needles=1, seed=400 + nb)
    x = synth.make_inputs(wl)
    q, k = dev(x.q), dev(x.k)
    sk = torch.empty((wl.B, wl.Hkv, wl.nb, wl.d), dtype=torch.float32, device="cuda")
    sa.sa_build_sketch(k, wl.L, wl.Bk, sk)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    idx = torch.empty((wl.B, wl.Hkv, 1, kmax), dtype=torch.int32, device="cuda")
    cnt = torch.empty((wl.B, wl.Hkv, 1), dtype=torch.int32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_SKETCH, q, sk, None, wl.Hkv, wl.L, wl.L, wl.Bk, 0, False, wl.k, 0, 1, wl.scale,
                      idx, cnt)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    o_idx, o_cnt, o_s, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, o_s, what="nb=%d" % nb)


def _check_topdelta(g_idx, g_cnt, o_idx, o_cnt, s, delta, cap, rel=1e-5, what=""):
    """Exact match, except blocks whose oracle score sits within rel of the threshold
    (fp32 vs fp64 comparison) or of the cap's cut-off score (near-ties)."""
    g_idx = np.asarray(g_idx).reshape(len(o_cnt), -1)
    g_cnt = np.asarray(g_cnt).reshape(-1)
    for u in range(len(o_cnt)):
        su = np.asarray(s[u], dtype=np.float64)
        nb = len(su)
        row = g_idx[u, : g_cnt[u]].tolist()
        assert row == sorted(set(row)) and np.all(g_idx[u, g_cnt[u]:] == -1), (what, u, row)
        assert row[0] == 0 and row[-1] == nb - 1 and len(row) <= cap + 2, (what, u, row)
        gs, os_ = set(row), set(o_idx[u, : o_cnt[u]].tolist())
        if gs == os_:
            continue
        scale = np.abs(su).max()
        thr = max(su[0], su[nb - 1]) - delta
        cands = sorted([b for b in range(1, nb - 1) if su[b] >= thr], key=lambda b: (-su[b], b))
        cut = su[cands[cap - 1]] if 0 < cap <= len(cands) else None
        for b in gs ^ os_:
            near_thr = abs(su[b] - thr) <= rel * scale
            near_cut = cut is not None and abs(su[b] - cut) <= rel * scale
            assert near_thr or near_cut, "%s unit %d: block %d (score %.9g, thr %.9g, cut %s) differs" % (
                what, u, b, su[b], thr, cut)


@pytest.mark.parametrize("name", ["c2", "c3"])
def test_decode_topdelta_matches_oracle(sa, name):
    wl = synth.WORKLOADS[name]
    if name == "c3":
        wl = wl.replace(L=65536, needles=10)
    x = synth.make_inputs(wl)
    q, k = dev(x.q), dev(x.k)
    sk = torch.empty((wl.B, wl.Hkv, wl.nb, wl.d), dtype=torch.float32, device="cuda")
    sa.sa_build_sketch(k, wl.L, wl.Bk, sk)
    sketch = oracle.block_means(x.k, wl.L, wl.Bk)
    for delta, cap in ((0.0, wl.k), (0.1, wl.k), (0.3, 2 * wl.k), (1.0, wl.k), (1e6, wl.k), (0.2, 0)):
        kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, cap)
        idx = torch.full((wl.B, wl.Hkv, 1, kmax), -7, dtype=torch.int32, device="cuda")
        cnt = torch.zeros((wl.B, wl.Hkv, 1), dtype=torch.int32, device="cuda")
        sa.sa_select_topdelta(q, sk, None, wl.Hkv, wl.L, wl.L, wl.Bk, delta, cap, wl.scale, idx, cnt)
        torch.cuda.synchronize()
        assert sa.sa_device_status(clear=True) == 0
        o_idx, o_cnt, o_s, _ = oracle.decode_select_delta(x.q, x.k, wl, delta, cap, kmax=kmax, sketch=sketch)
        _check_topdelta(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, o_s, delta, cap,
                        what="%s delta=%g cap=%d" % (name, delta, cap))
        if delta >= 1e6:  # no threshold: the top-k selection
            t_idx, t_cnt, _, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax, sketch=sketch)
            assert np.array_equal(o_idx, t_idx) and np.array_equal(o_cnt, t_cnt)


@pytest.mark.parametrize("n", [258, 259, 300, 512, 514, 1000, 4096, 16384])
def test_select_small_budgets_patterns(sa, n):
    """Budgets from one to a third of the candidates, on score patterns that stress a
    value-histogram threshold search: exact ties everywhere, all equal, sorted ascending and
    descending, a few large outliers, random, and values spread over 60 octaves (most of
    them in one bin, so the search refines over several rounds); bit-exact against the oracle."""
    rng = np.random.default_rng(1000 + n)
    pats = [
        rng.integers(-4, 5, size=n).astype(np.float32) * 0.25,   # heavy ties
        np.ones(n, dtype=np.float32),                             # all equal
        np.arange(n, dtype=np.float32),                           # ascending: the top is at the end
        -np.arange(n, dtype=np.float32),                          # descending: the top is at the start
        np.where(rng.random(n) < 0.01, 10.0, rng.standard_normal(n)).astype(np.float32),  # needles
        rng.standard_normal(n).astype(np.float32),
        (2.0 ** rng.integers(0, 60, size=n)).astype(np.float32),  # values over 60 octaves: several rounds
    ]
    s = np.stack(pats)
    groups = s.shape[0]
    for k in (1, 7, 32, 80, 128, 200, n // 3):
        kmax = sa.sa_select_kmax(n, 1, 0, False, k)
        scores = torch.from_numpy(np.ascontiguousarray(s.reshape(1, groups, 1, n))).cuda()
        idx = torch.full((1, groups, 1, kmax), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((1, groups, 1), -7, dtype=torch.int32, device="cuda")
        sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, scores, groups, n, n, 1, 0, False, k, 0, 1, 1.0,
                          idx, cnt, d=128, dtype=sa.SA_BF16, B=1, Tq=1, Hq=groups)
        torch.cuda.synchronize()
        assert sa.sa_device_status(clear=True) == 0
        o_idx, o_cnt = oracle.select(s.astype(np.float64), n, n - 1, k, kmax)
        g_idx = idx.cpu().numpy().reshape(groups, kmax)
        g_cnt = cnt.cpu().numpy().reshape(groups)
        for g in range(groups):
            assert g_cnt[g] == o_cnt[g] and np.array_equal(g_idx[g], o_idx[g]), (
                "n=%d k=%d pattern %d: gpu %s (cnt %d), oracle %s (cnt %d)" % (
                    n, k, g, g_idx[g][:12].tolist(), g_cnt[g], o_idx[g][:12].tolist(), o_cnt[g]))


@pytest.mark.parametrize("n", [300, 512, 700, 3000, 4096])
def test_select_fallback_patterns(sa, n):
    """Scores for which the register-resident value-histogram search gives up and the general
    search takes over: infinite scores (no finite key range), a range too wide for a float
    (values near +-3e38), and a crowded threshold bin (most candidates share one value just
    below a few larger ones); plus a tiny range of a few ulps.  Bit-exact against the oracle."""
    rng = np.random.default_rng(2000 + n)
    base = rng.standard_normal(n)
    crowded = np.full(n, 0.5)
    crowded[rng.choice(n, size=8, replace=False)] = 10.0 + rng.random(8)
    pats = [
        np.where(rng.random(n) < 0.05, -np.inf, base),               # -inf entries
        np.where(rng.random(n) < 0.02, np.inf, base),                # +inf entries
        np.where(rng.random(n) < 0.5, 3.0e38, -3.0e38) * rng.random(n),  # width beyond float range
        crowded,                                                     # the threshold bin holds most keys
        1.0 + rng.integers(0, 3, size=n) * 2.0 ** -23,               # three adjacent floats
    ]
    s = np.stack(pats).astype(np.float32)
    groups = s.shape[0]
    for k in (1, 5, 32, 80, n // 3, n - 3):
        kmax = sa.sa_select_kmax(n, 1, 0, False, k)
        scores = torch.from_numpy(np.ascontiguousarray(s.reshape(1, groups, 1, n))).cuda()
        idx = torch.full((1, groups, 1, kmax), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((1, groups, 1), -7, dtype=torch.int32, device="cuda")
        sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, scores, groups, n, n, 1, 0, False, k, 0, 1, 1.0,
                          idx, cnt, d=128, dtype=sa.SA_BF16, B=1, Tq=1, Hq=groups)
        torch.cuda.synchronize()
        assert sa.sa_device_status(clear=True) == 0
        o_idx, o_cnt = oracle.select(s.astype(np.float64), n, n - 1, k, kmax)
        g_idx = idx.cpu().numpy().reshape(groups, kmax)
        g_cnt = cnt.cpu().numpy().reshape(groups)
        for g in range(groups):
            assert g_cnt[g] == o_cnt[g] and np.array_equal(g_idx[g], o_idx[g]), (
                "n=%d k=%d pattern %d: gpu %s (cnt %d), oracle %s (cnt %d)" % (
                    n, k, g, g_idx[g][:12].tolist(), g_cnt[g], o_idx[g][:12].tolist(), o_cnt[g]))
