"""Full-size prefill workloads, in the launch configuration bench.py times:
the whole GPU step runs at full size, and sampled (group, tile) units and rows
are checked against the CPU oracle, which computes them one by one.

  sketch-selected prefill: B=2, Hq=32, Hkv=8, d=128, L=131072, 2% of causal blocks
  oracle-mass prefill:     B=1, Hq=16, Hkv=2, d=128, L=32768, 2% of causal blocks
(The full-size decode workloads are checked element by element in test_gpu_decode.py.)
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, assert_selection, dev, host

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def sa():
    import top_block_sparse_pooled_b300 as m
    return m


def _sample_units(wl, rng, n):
    groups = wl.B * wl.Hkv
    fixed = [(0, 0), (groups - 1, wl.nq - 1), (groups // 2, 1), (1, wl.nq // 2)]
    extra = [(int(rng.integers(groups)), int(rng.integers(wl.nq))) for _ in range(n - len(fixed))]
    return fixed + extra


def _sample_rows(wl, units, rng, per_unit):
    rows = []
    for g, i in units:
        b, kvh = divmod(g, wl.Hkv)
        t0, t1 = i * wl.Qt, min((i + 1) * wl.Qt, wl.L)
        for t in sorted({t0, t1 - 1} | set(rng.integers(t0, t1, size=per_unit - 2).tolist())):
            for h in (kvh * wl.G, kvh * wl.G + wl.G - 1):
                rows.append((b, t, h))
    return np.array(rows, dtype=np.int64)


def _run_gpu_step(sa, wl, x):
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, wl.Qt, True, wl.k, wl.frac_num, wl.frac_den)
    idx = torch.empty((wl.B, wl.Hkv, wl.nq, kmax), dtype=torch.int32, device="cuda")
    cnt = torch.empty((wl.B, wl.Hkv, wl.nq), dtype=torch.int32, device="cuda")
    scores = torch.empty((wl.B, wl.Hkv, wl.nq, wl.nb), dtype=torch.float32, device="cuda")
    if wl.mode == "mass":
        sa.sa_oracle_mass(q, k, wl.Qt, wl.Bk, wl.scale, scores, None)
        sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, scores, wl.Hkv, wl.L, wl.L, wl.Bk, wl.Qt, True, wl.k,
                          wl.frac_num, wl.frac_den, wl.scale, idx, cnt, d=wl.d, dtype=sa.SA_BF16, B=wl.B, Tq=wl.L,
                          Hq=wl.Hq)
    else:
        sk = torch.empty((wl.B, wl.Hkv, wl.nb, wl.d), dtype=torch.float32, device="cuda")
        sa.sa_build_sketch(k, wl.L, wl.Bk, sk)
        sa.sa_select_topk(sa.SA_SELECT_SKETCH, q, sk, scores, wl.Hkv, wl.L, wl.L, wl.Bk, wl.Qt, True, wl.k,
                          wl.frac_num, wl.frac_den, wl.scale, idx, cnt)
    out = torch.empty_like(q)
    sa.sa_prefill(q, k, v, idx, cnt, wl.Qt, wl.Bk, wl.scale, out)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    groups = wl.B * wl.Hkv
    return (idx.cpu().numpy().reshape(groups * wl.nq, kmax), cnt.cpu().numpy().reshape(-1),
            scores.cpu().numpy().reshape(groups * wl.nq, wl.nb).astype(np.float64), out, kmax)


@pytest.mark.parametrize("name", ["c5", "c4"])
def test_full_size_prefill_step_sampled(sa, name):
    wl = synth.WORKLOADS[name]
    x = synth.make_inputs(wl)
    g_idx, g_cnt, g_scores, out, kmax = _run_gpu_step(sa, wl, x)
    rng = np.random.default_rng(11)
    units = _sample_units(wl, rng, 8 if name == "c5" else 6)
    uid = np.array([g * wl.nq + i for g, i in units])
    # scores of the sampled units
    if wl.mode == "mass":
        o_scores = oracle.mass(x.q, x.k, wl.Hkv, wl.L, 0, wl.Qt, wl.Bk, wl.scale, units)
        tot = o_scores.sum(axis=1, keepdims=True)
        assert np.all(np.abs(g_scores[uid] - o_scores) <= 2e-6 * tot + 1e-4 * np.abs(o_scores))
        o_idx, o_cnt, _, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax, scores=o_scores)
    else:
        o_idx, o_cnt, o_scores, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax)
        fin = np.isfinite(o_scores)
        scale = np.abs(np.where(fin, o_scores, 0)).max(axis=1, keepdims=True)
        assert np.all(np.abs(np.where(fin, g_scores[uid] - o_scores, 0)) <= 2e-6 * scale)
    assert_selection(g_idx[uid], g_cnt[uid], o_idx, o_cnt, o_scores, what=name)
    # every unit: ascending, unique, forced blocks present, count as the budget rule says
    for u in range(len(g_cnt)):
        i = u % wl.nq
        row = g_idx[u, : g_cnt[u]]
        assert row[0] == 0 and row[-1] == i and np.all(np.diff(row) > 0)
        budget = wl.k + (wl.frac_num * (i + 1) + wl.frac_den - 1) // wl.frac_den
        assert g_cnt[u] == min(i + 1, 2 + budget) if i > 0 else g_cnt[u] == 1
    # sampled output rows against the oracle on the GPU's (checked) selection
    rows = _sample_rows(wl, units, rng, 6)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, 0, wl.Bk, wl.scale, rows, g_idx, g_cnt, nsel=wl.nq,
                           rows_per_sel=wl.Qt)
    got = out[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(host(got), ref, what=name + " sampled rows")
