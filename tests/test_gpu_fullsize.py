"""Full-size prefill workloads, in the launch configuration bench.py times:
the whole GPU step runs at full size, and sampled (group, tile) units and rows
are checked against the CPU oracle, which computes them one by one.

  sketch-selected prefill: B=2, Hq=32, Hkv=8, d=128, L=131072, 2% of causal blocks
  oracle-mass prefill:     B=1, Hq=16, Hkv=2, d=128, L=32768, 2% of causal blocks

Every unit's selection is checked for shape (ascending, forced blocks, count);
the sampled units' scores and selections against the oracle; and the sampled
rows' outputs against the oracle's exact attention on the ORACLE's selection: the
sampled units of the GPU's index array are overwritten with the oracle's lists
and the full-size prefill is run again.
(The full-size decode workloads are checked element by element in test_gpu_decode.py;
the persistent multi-unit path is checked on every row in test_gpu_persistent.py.)
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


def _sample_units(wl, rng, n_all, n_short=0, short_tiles=64):
    """Every group's last tile and first tile, then random units over all tiles and
    (cheap for the dense-mass oracle) over the first `short_tiles` tiles."""
    groups = wl.B * wl.Hkv
    chosen = []
    for g in range(groups):
        chosen += [(g, wl.nq - 1), (g, 0)]
    seen = set(chosen)
    for n, hi in ((n_all, wl.nq), (n_short, min(short_tiles, wl.nq))):
        added = 0
        while added < n:
            u = (int(rng.integers(groups)), int(rng.integers(hi)))
            if u not in seen:
                seen.add(u)
                chosen.append(u)
                added += 1
    return chosen


def _sample_rows(wl, units, rng, per_unit):
    rows = []
    for g, i in units:
        b, kvh = divmod(g, wl.Hkv)
        t0, t1 = i * wl.Qt, min((i + 1) * wl.Qt, wl.L)
        ts = {t0, t1 - 1} | set(rng.integers(t0, t1, size=per_unit - 2).tolist())
        for t in sorted(ts):
            for h in range(kvh * wl.G, (kvh + 1) * wl.G):
                rows.append((b, t, h))
    return np.array(rows, dtype=np.int64)


def _run_gpu_step(sa, wl, q, k, v):
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
            scores.cpu().numpy().reshape(groups * wl.nq, wl.nb).astype(np.float64), kmax)


@pytest.mark.parametrize("name", ["c5", "c4"])
def test_full_size_prefill_step_sampled(sa, name):
    wl = synth.WORKLOADS[name]
    x = synth.make_inputs(wl)
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    g_idx, g_cnt, g_scores, kmax = _run_gpu_step(sa, wl, q, k, v)
    rng = np.random.default_rng(11)
    # c5: 256 units (all 16 groups' first and last tiles + 224 random).  c4: the dense-mass oracle
    # costs O(i) per unit, so 4 fixed + 60 random units over all tiles + 64 over the first 64 tiles
    # (the persistent grid runs its longest tiles first, so short tiles are the CTAs' later units).
    units = _sample_units(wl, rng, 224) if name == "c5" else _sample_units(wl, rng, 60, 64)
    uid = np.array([g * wl.nq + i for g, i in units])
    if wl.mode == "mass":
        o_scores = oracle.mass(x.q, x.k, wl.Hkv, wl.L, 0, wl.Qt, wl.Bk, wl.scale, units)
        tot = o_scores.sum(axis=1, keepdims=True)
        assert np.all(np.abs(g_scores[uid] - o_scores) <= 2e-6 * tot + 1e-4 * np.abs(o_scores))
        o_idx, o_cnt, _, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax, scores=o_scores)
        rel = 1e-6  # the GPU ranks float32-rounded masses
    else:
        o_idx, o_cnt, o_scores, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax)
        fin = np.isfinite(o_scores)
        scale = np.abs(np.where(fin, o_scores, 0)).max(axis=1, keepdims=True)
        diff = np.subtract(g_scores[uid], o_scores, out=np.zeros_like(o_scores), where=fin)  # finite entries only
        assert np.all(np.abs(diff) <= 2e-6 * scale)
        rel = 1e-5
    assert_selection(g_idx[uid], g_cnt[uid], o_idx, o_cnt, o_scores, rel=rel, what=name)
    # every unit: ascending, unique, forced blocks present, count as the budget rule says
    for u in range(len(g_cnt)):
        i = u % wl.nq
        row = g_idx[u, : g_cnt[u]]
        assert row[0] == 0 and row[-1] == i and np.all(np.diff(row) > 0)
        budget = wl.k + (wl.frac_num * (i + 1) + wl.frac_den - 1) // wl.frac_den
        assert g_cnt[u] == min(i + 1, 2 + budget) if i > 0 else g_cnt[u] == 1
    # outputs: the oracle's selection fed to the full-size prefill, sampled rows of every sampled unit
    fed_idx, fed_cnt = g_idx.copy(), g_cnt.copy()
    fed_idx[uid] = o_idx
    fed_cnt[uid] = o_cnt
    idx_t = torch.from_numpy(fed_idx.reshape(wl.B, wl.Hkv, wl.nq, kmax)).cuda()
    cnt_t = torch.from_numpy(fed_cnt.reshape(wl.B, wl.Hkv, wl.nq)).cuda()
    out = torch.full_like(q, float("nan"))
    sa.sa_prefill(q, k, v, idx_t, cnt_t, wl.Qt, wl.Bk, wl.scale, out)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    rows = _sample_rows(wl, units, rng, 16)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, 0, wl.Bk, wl.scale, rows, fed_idx, fed_cnt, nsel=wl.nq,
                           rows_per_sel=wl.Qt)
    got = out[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(host(got), ref, what="%s sampled rows (%d units, %d rows)" % (name, len(units), len(rows)))
