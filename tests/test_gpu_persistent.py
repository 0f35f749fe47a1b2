"""The persistent prefill and mass kernels on workloads with many more work units
than SMs, checked element by element against the CPU oracle.

Both kernels run one CTA per SM and deal their units round-robin, so every CTA
here runs several units in a row: the mbarrier phases, the TMEM accumulators and
the Q ring carry over from one unit to the next.  Every output row of every head
(and its log-sum-exp) is compared with the oracle's exact attention on the
ORACLE's selection, and every mass unit with the oracle's dense mass
("How Much Dense Attention is Necessary?" Sec. 2.1: exact attention on the
selected support; the oracle mode's support is the block mass of the dense
distribution).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, assert_selection, dev, host

pytestmark = pytest.mark.gpu

# Work units per kernel: prefill (group, tile, head pair), mass (group, tile).
# All cases have at least twice as many units as the B300 has SMs (148).
PF_MULTI = {
    # sketch-selected prefill, c5's heads at L = 16K: 8 groups x 128 tiles x 2 head pairs = 2048 units
    "c5_heads_16k": synth.WORKLOADS["c5"].replace(B=1, L=16384, needles=2, seed=401),
    # odd group size (head pairs with one head), ragged last tile: 16 groups x 11 tiles x 2 pairs = 352
    "g3_ragged": synth.WORKLOADS["c5"].replace(B=4, Hq=12, Hkv=4, L=128 * 10 + 50, k=1, frac_num=20, needles=1,
                                               seed=402),
}
MASS_MULTI = {
    # c4's heads (G = 8, four head pairs per unit), ragged: 12 groups x 26 tiles = 312 units
    "c4_heads_b6": synth.WORKLOADS["c4"].replace(B=6, L=128 * 25 + 77, seed=403),
    # G = 2, one head pair per unit: 64 groups x 9 tiles = 576 units
    "g2_b8": synth.WORKLOADS["c4"].replace(B=8, Hq=16, Hkv=8, L=128 * 8 + 37, seed=404),
}


@pytest.fixture(scope="module")
def sa():
    import top_block_sparse_pooled_b300 as m
    return m


def _units(wl):
    return [(g, i) for g in range(wl.B * wl.Hkv) for i in range(wl.nq)]


def _all_rows(wl):
    b, t, h = np.meshgrid(np.arange(wl.B), np.arange(wl.L), np.arange(wl.Hq), indexing="ij")
    return np.stack([b.ravel(), t.ravel(), h.ravel()], axis=1).astype(np.int64)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("name", sorted(PF_MULTI))
def test_prefill_many_units_per_cta(sa, name):
    wl = PF_MULTI[name]
    pairs = (wl.G + 1) // 2
    assert wl.B * wl.Hkv * wl.nq * pairs >= 2 * _sms(), "case must give every CTA several units"
    x = synth.make_inputs(wl)
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, wl.Qt, True, wl.k, wl.frac_num, wl.frac_den)
    units = _units(wl)
    o_idx, o_cnt, o_s, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax)
    # the GPU's own selection on the same inputs (sketch build + tile scoring + top-k)
    sk = torch.empty((wl.B, wl.Hkv, wl.nb, wl.d), dtype=torch.float32, device="cuda")
    sa.sa_build_sketch(k, wl.L, wl.Bk, sk)
    g_idx = torch.full((wl.B, wl.Hkv, wl.nq, kmax), -7, dtype=torch.int32, device="cuda")
    g_cnt = torch.zeros((wl.B, wl.Hkv, wl.nq), dtype=torch.int32, device="cuda")
    scores = torch.empty((wl.B, wl.Hkv, wl.nq, wl.nb), dtype=torch.float32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_SKETCH, q, sk, scores, wl.Hkv, wl.L, wl.L, wl.Bk, wl.Qt, True, wl.k,
                      wl.frac_num, wl.frac_den, wl.scale, g_idx, g_cnt)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    assert_selection(g_idx.cpu().numpy(), g_cnt.cpu().numpy(), o_idx, o_cnt, o_s, what=name + " select")
    # the prefill kernel fed the oracle's selection
    idx = torch.from_numpy(np.ascontiguousarray(o_idx.reshape(wl.B, wl.Hkv, wl.nq, kmax))).cuda()
    cnt = torch.from_numpy(np.ascontiguousarray(o_cnt.reshape(wl.B, wl.Hkv, wl.nq))).cuda()
    out = torch.full_like(q, float("nan"))
    lse = torch.full((wl.B, wl.Hq, wl.L), float("nan"), dtype=torch.float32, device="cuda")
    sa.sa_prefill(q, k, v, idx, cnt, wl.Qt, wl.Bk, wl.scale, out, lse)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    rows = _all_rows(wl)
    ref, ref_lse = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, 0, wl.Bk, wl.scale, rows, o_idx, o_cnt,
                                 nsel=wl.nq, rows_per_sel=wl.Qt)
    err = assert_close(host(out).reshape(ref.shape), ref, what=name)
    g_lse = host(lse)[rows[:, 0], rows[:, 2], rows[:, 1]]
    assert_close(g_lse, ref_lse, atol=1e-3, rtol=1e-4, what=name + " lse")
    # a second call on the same buffers gives the same bits (no state left from the first)
    out2 = torch.full_like(q, float("nan"))
    sa.sa_prefill(q, k, v, idx, cnt, wl.Qt, wl.Bk, wl.scale, out2)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    print("%s: %d rows, max abs err %.3g" % (name, len(rows), err))


@pytest.mark.parametrize("name", sorted(MASS_MULTI))
def test_mass_many_units_per_cta(sa, name):
    wl = MASS_MULTI[name]
    units = _units(wl)
    assert len(units) >= 2 * _sms(), "case must give every CTA several units"
    x = synth.make_inputs(wl)
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    mass = torch.full((wl.B, wl.Hkv, wl.nq, wl.nb), float("nan"), dtype=torch.float32, device="cuda")
    sa.sa_oracle_mass(q, k, wl.Qt, wl.Bk, wl.scale, mass, None)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    got = host(mass).reshape(len(units), wl.nb)
    ref = oracle.mass(x.q, x.k, wl.Hkv, wl.L, 0, wl.Qt, wl.Bk, wl.scale, units)
    tot = ref.sum(axis=1, keepdims=True)
    err = np.abs(got - ref)
    assert np.all(err <= 2e-6 * tot + 1e-4 * np.abs(ref)), "mass differs: worst %.3g of the unit total" % (
        err / tot).max()
    for u, (g, i) in enumerate(units):
        nrows = min((i + 1) * wl.Qt, wl.L) - i * wl.Qt
        assert abs(got[u].sum() - nrows * wl.G) <= 1e-4 * nrows * wl.G
        assert np.all(got[u, i + 1:] == 0.0)
    # oracle mode end to end: the oracle's mass selection fed to the prefill kernel, every row
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, wl.Qt, True, wl.k, wl.frac_num, wl.frac_den)
    o_idx, o_cnt, _, _ = oracle.prefill_select(x.q, x.k, wl, units, kmax=kmax, scores=ref)
    g_idx = torch.empty((wl.B, wl.Hkv, wl.nq, kmax), dtype=torch.int32, device="cuda")
    g_cnt = torch.empty((wl.B, wl.Hkv, wl.nq), dtype=torch.int32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, mass, wl.Hkv, wl.L, wl.L, wl.Bk, wl.Qt, True, wl.k,
                      wl.frac_num, wl.frac_den, wl.scale, g_idx, g_cnt, d=wl.d, dtype=sa.SA_BF16, B=wl.B, Tq=wl.L,
                      Hq=wl.Hq)
    torch.cuda.synchronize()
    # the GPU ranks float32-rounded masses: a swap is allowed only between near-equal masses
    assert_selection(g_idx.cpu().numpy(), g_cnt.cpu().numpy(), o_idx, o_cnt, ref, rel=1e-6, what=name + " select")
    idx = torch.from_numpy(np.ascontiguousarray(o_idx.reshape(wl.B, wl.Hkv, wl.nq, kmax))).cuda()
    cnt = torch.from_numpy(np.ascontiguousarray(o_cnt.reshape(wl.B, wl.Hkv, wl.nq))).cuda()
    out = torch.full_like(q, float("nan"))
    sa.sa_prefill(q, k, v, idx, cnt, wl.Qt, wl.Bk, wl.scale, out)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    rows = _all_rows(wl)
    o_ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, 0, wl.Bk, wl.scale, rows, o_idx, o_cnt, nsel=wl.nq,
                             rows_per_sel=wl.Qt)
    assert_close(host(out).reshape(o_ref.shape), o_ref, what=name + " prefill")
