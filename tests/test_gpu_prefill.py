"""GPU parity of the prefill path: tile selection (sketch and mass modes) and the
tcgen05 sparse prefill kernel, against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, assert_selection, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    import top_block_sparse_pooled_b300 as m
    return m


def _check_status(sa):
    assert sa.sa_device_status(clear=True) == 0


def _units(wl):
    return [(g, i) for g in range(wl.B * wl.Hkv) for i in range(wl.nq)]


# small prefill workloads: several tiles, a ragged tail, GQA group sizes 1, 2, 3, 4, 8
PF_CASES = {
    "g2_ragged": synth.WORKLOADS["c5"].replace(B=1, Hq=4, Hkv=2, L=128 * 11 + 37, frac_num=20, needles=2, seed=201),
    "g4_b2": synth.WORKLOADS["c5"].replace(B=2, Hq=8, Hkv=2, L=128 * 9, frac_num=25, needles=1, seed=202),
    "g1": synth.WORKLOADS["c5"].replace(B=1, Hq=2, Hkv=2, L=128 * 7 + 1, k=1, frac_num=0, needles=1, seed=203),
    "g3_odd": synth.WORKLOADS["c5"].replace(B=1, Hq=6, Hkv=2, L=128 * 6 + 100, k=2, frac_num=0, needles=1, seed=204),
    "g8_mass": synth.WORKLOADS["c4"].replace(L=128 * 8, Hq=16, Hkv=2, frac_num=30, seed=205),
}


def _all_rows(wl):
    return np.array([(b, t, h) for b in range(wl.B) for t in range(wl.L) for h in range(wl.Hq)], dtype=np.int64)


def _prefill_gpu(sa, wl, x, idx_np, cnt_np, kmax, want_lse=False):
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    idx = torch.from_numpy(np.ascontiguousarray(idx_np.reshape(wl.B, wl.Hkv, wl.nq, kmax))).cuda()
    cnt = torch.from_numpy(np.ascontiguousarray(cnt_np.reshape(wl.B, wl.Hkv, wl.nq))).cuda()
    out = torch.full_like(q, float("nan"))
    lse = torch.full((wl.B, wl.Hq, wl.L), float("nan"), dtype=torch.float32, device="cuda") if want_lse else None
    sa.sa_prefill(q, k, v, idx, cnt, wl.Qt, wl.Bk, wl.scale, out, lse)
    torch.cuda.synchronize()
    _check_status(sa)
    return host(out), (host(lse) if want_lse else None)


@pytest.mark.parametrize("name", sorted(PF_CASES))
def test_prefill_matches_oracle_on_oracle_selection(sa, name):
    wl = PF_CASES[name]
    x = synth.make_inputs(wl)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, wl.Qt, True, wl.k, wl.frac_num, wl.frac_den)
    units = _units(wl)
    if wl.mode == "mass":
        m = oracle.mass(x.q, x.k, wl.Hkv, wl.L, 0, wl.Qt, wl.Bk, wl.scale, units)
        o_idx, o_cnt, _, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax, scores=m)
    else:
        o_idx, o_cnt, _, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax)
    got, lse = _prefill_gpu(sa, wl, x, o_idx, o_cnt, kmax, want_lse=True)
    rows = _all_rows(wl)
    ref, ref_lse = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, 0, wl.Bk, wl.scale, rows, o_idx, o_cnt,
                                 nsel=wl.nq, rows_per_sel=wl.Qt)
    err = assert_close(got.reshape(ref.shape), ref, what=name)
    # lse [B, Hq, L] vs oracle rows (b, t, h)
    g_lse = lse[rows[:, 0], rows[:, 2], rows[:, 1]]
    assert_close(g_lse, ref_lse, atol=1e-3, rtol=1e-4, what=name + " lse")
    print("%s max abs err %.3g" % (name, err))


def test_prefill_full_budget_equals_dense(sa):
    """Every causal block selected: block-sparse prefill is dense causal attention."""
    wl = PF_CASES["g2_ragged"]
    x = synth.make_inputs(wl)
    kmax = wl.nb
    idx = -np.ones((wl.B * wl.Hkv * wl.nq, kmax), dtype=np.int32)
    cnt = np.zeros((wl.B * wl.Hkv * wl.nq,), dtype=np.int32)
    for u, (g, i) in enumerate(_units(wl)):
        idx[u, : i + 1] = np.arange(i + 1)
        cnt[u] = i + 1
    got, _ = _prefill_gpu(sa, wl, x, idx, cnt, kmax)
    rows = _all_rows(wl)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, 0, wl.Bk, wl.scale, rows)
    assert_close(got.reshape(ref.shape), ref, what="dense")


def test_prefill_empty_and_skipped_blocks(sa):
    """cnt = 0 gives zeros; out-of-range block ids inside cnt are skipped."""
    wl = PF_CASES["g2_ragged"]
    x = synth.make_inputs(wl)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, wl.Qt, True, wl.k, wl.frac_num, wl.frac_den)
    units = _units(wl)
    o_idx, o_cnt, _, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax)
    # padded selection: an invalid id (-1 and nb) in front of the real ones
    pad_idx = -np.ones((len(units), kmax + 2), dtype=np.int32)
    pad_cnt = o_cnt + 2
    for u in range(len(units)):
        pad_idx[u, 0] = -1
        pad_idx[u, 1] = wl.nb + 5
        pad_idx[u, 2: 2 + o_cnt[u]] = o_idx[u, : o_cnt[u]]
    empty_u = 3
    pad_cnt[empty_u] = 0
    got, lse = _prefill_gpu(sa, wl, x, pad_idx, pad_cnt, kmax + 2, want_lse=True)
    rows = _all_rows(wl)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, 0, wl.Bk, wl.scale, rows, o_idx, o_cnt,
                           nsel=wl.nq, rows_per_sel=wl.Qt)
    ref = ref.reshape(wl.B, wl.L, wl.Hq, wl.d)
    g, i = units[empty_u]
    b, kvh = divmod(g, wl.Hkv)
    hs = slice(kvh * wl.G, (kvh + 1) * wl.G)
    ts = slice(i * wl.Qt, min((i + 1) * wl.Qt, wl.L))
    ref[b, ts, hs] = 0.0
    assert_close(got.reshape(ref.shape), ref, what="padded")
    assert np.all(np.isneginf(lse[b, hs, ts]))


@pytest.mark.parametrize("name", ["g2_ragged", "g4_b2", "g3_odd"])
def test_prefill_select_sketch_matches_oracle(sa, name):
    wl = PF_CASES[name]
    x = synth.make_inputs(wl)
    q, k = dev(x.q), dev(x.k)
    sk = torch.empty((wl.B, wl.Hkv, wl.nb, wl.d), dtype=torch.float32, device="cuda")
    sa.sa_build_sketch(k, wl.L, wl.Bk, sk)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, wl.Qt, True, wl.k, wl.frac_num, wl.frac_den)
    idx = torch.full((wl.B, wl.Hkv, wl.nq, kmax), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((wl.B, wl.Hkv, wl.nq), dtype=torch.int32, device="cuda")
    scores = torch.empty((wl.B, wl.Hkv, wl.nq, wl.nb), dtype=torch.float32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_SKETCH, q, sk, scores, wl.Hkv, wl.L, wl.L, wl.Bk, wl.Qt, True, wl.k,
                      wl.frac_num, wl.frac_den, wl.scale, idx, cnt)
    torch.cuda.synchronize()
    _check_status(sa)
    units = _units(wl)
    o_idx, o_cnt, o_s, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax)
    g_s = host(scores).reshape(o_s.shape)
    fin = np.isfinite(o_s)
    assert np.array_equal(fin, np.isfinite(g_s))
    scale = np.abs(np.where(fin, o_s, 0)).max(axis=1, keepdims=True)
    diff = np.subtract(g_s, o_s, out=np.zeros_like(o_s), where=fin)  # finite entries only
    assert np.all(np.abs(diff) <= 2e-6 * scale), "tile scores differ beyond fp32 rounding"
    assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, o_s, what=name)


def test_select_mass_mode_matches_oracle(sa):
    """Mass-mode selection from given scores (prefill tiles and decode)."""
    wl = PF_CASES["g8_mass"]
    x = synth.make_inputs(wl)
    units = _units(wl)
    m = oracle.mass(x.q, x.k, wl.Hkv, wl.L, 0, wl.Qt, wl.Bk, wl.scale, units)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, wl.Qt, True, wl.k, wl.frac_num, wl.frac_den)
    o_idx, o_cnt, _, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax, scores=m)
    scores = torch.from_numpy(m.astype(np.float32).reshape(wl.B, wl.Hkv, wl.nq, wl.nb)).cuda()
    idx = torch.full((wl.B, wl.Hkv, wl.nq, kmax), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((wl.B, wl.Hkv, wl.nq), dtype=torch.int32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, scores, wl.Hkv, wl.L, wl.L, wl.Bk, wl.Qt, True, wl.k,
                      wl.frac_num, wl.frac_den, wl.scale, idx, cnt, d=wl.d, dtype=sa.SA_BF16, B=wl.B, Tq=wl.L,
                      Hq=wl.Hq)
    torch.cuda.synchronize()
    _check_status(sa)
    # the GPU ranks the float32-rounded masses: ties after rounding may swap
    assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, m, rel=1e-6, what="mass")


MASS_CASES = {
    "g8": synth.WORKLOADS["c4"].replace(L=128 * 6 + 50, Hq=16, Hkv=2, seed=301),
    "g3_odd_b2": synth.WORKLOADS["c4"].replace(B=2, L=128 * 5, Hq=6, Hkv=2, seed=302),
    "g1": synth.WORKLOADS["c4"].replace(L=128 * 4 + 1, Hq=1, Hkv=1, seed=303),
}


def _mass_gpu(sa, wl, x):
    q, k = dev(x.q), dev(x.k)
    mass = torch.full((wl.B, wl.Hkv, wl.nq, wl.nb), float("nan"), dtype=torch.float32, device="cuda")
    sa.sa_oracle_mass(q, k, wl.Qt, wl.Bk, wl.scale, mass, None)
    torch.cuda.synchronize()
    _check_status(sa)
    return host(mass).reshape(wl.B * wl.Hkv * wl.nq, wl.nb)


@pytest.mark.parametrize("name", sorted(MASS_CASES))
def test_oracle_mass_matches_oracle(sa, name):
    wl = MASS_CASES[name]
    x = synth.make_inputs(wl)
    got = _mass_gpu(sa, wl, x)
    ref = oracle.mass(x.q, x.k, wl.Hkv, wl.L, 0, wl.Qt, wl.Bk, wl.scale, _units(wl))
    # each unit sums rows * G probabilities: compare against that total
    tot = ref.sum(axis=1, keepdims=True)
    err = np.abs(got - ref)
    assert np.all(err <= 2e-6 * tot + 1e-4 * np.abs(ref)), "mass differs: worst %.3g of total" % (err / tot).max()
    # invariants: per unit the masses sum to rows * G; non-causal blocks are zero
    for u, (g, i) in enumerate(_units(wl)):
        rows = min((i + 1) * wl.Qt, wl.L) - i * wl.Qt
        assert abs(got[u].sum() - rows * wl.G) <= 1e-4 * rows * wl.G
        assert np.all(got[u, i + 1:] == 0.0)


def test_oracle_mass_then_select_then_prefill(sa):
    """The oracle-mode path on the GPU: mass -> select (mass mode) -> prefill, against the oracle."""
    wl = MASS_CASES["g8"].replace(frac_num=30)
    x = synth.make_inputs(wl)
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    mass = torch.empty((wl.B, wl.Hkv, wl.nq, wl.nb), dtype=torch.float32, device="cuda")
    sa.sa_oracle_mass(q, k, wl.Qt, wl.Bk, wl.scale, mass, None)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, wl.Qt, True, wl.k, wl.frac_num, wl.frac_den)
    idx = torch.empty((wl.B, wl.Hkv, wl.nq, kmax), dtype=torch.int32, device="cuda")
    cnt = torch.empty((wl.B, wl.Hkv, wl.nq), dtype=torch.int32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, mass, wl.Hkv, wl.L, wl.L, wl.Bk, wl.Qt, True, wl.k,
                      wl.frac_num, wl.frac_den, wl.scale, idx, cnt, d=wl.d, dtype=sa.SA_BF16, B=wl.B, Tq=wl.L,
                      Hq=wl.Hq)
    out = torch.empty_like(q)
    sa.sa_prefill(q, k, v, idx, cnt, wl.Qt, wl.Bk, wl.scale, out)
    torch.cuda.synchronize()
    _check_status(sa)
    units = _units(wl)
    m = oracle.mass(x.q, x.k, wl.Hkv, wl.L, 0, wl.Qt, wl.Bk, wl.scale, units)
    o_idx, o_cnt, _, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax, scores=m)
    assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, m, what="mass select")
    # outputs against the oracle on the GPU's own (validated) selection
    g_idx = idx.cpu().numpy().reshape(len(units), kmax)
    g_cnt = cnt.cpu().numpy().reshape(-1)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, 0, wl.Bk, wl.scale, _all_rows(wl), g_idx, g_cnt,
                           nsel=wl.nq, rows_per_sel=wl.Qt)
    assert_close(host(out).reshape(ref.shape), ref, what="oracle-mode prefill")
