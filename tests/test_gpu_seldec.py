"""GPU parity of the cluster decode kernel: sa_select_decode (sketch scoring,
top-k and sparse attention in one launch) and sa_decode's cluster path.

The fused call must select exactly what sa_select_topk selects (same scores, bit
for bit) and produce sa_decode's output on that selection (up to the order of
the fp32 sums); sa_decode
itself is checked against the oracle on the oracle's selection here and in
test_gpu_decode.py.  Shapes cover one and many clusters per group round (more
groups than fit at once), cluster sizes from 1 to 16, T > 1 causal rows, ragged
last blocks, d = 64, and contexts of one or two blocks.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, assert_selection, dev, host

pytestmark = pytest.mark.gpu

CASES = {
    "c2": synth.WORKLOADS["c2"],
    "c3": synth.WORKLOADS["c3"],
    # 5 groups, T = 3 causal rows, ragged last block
    "ragged_t3": synth.WORKLOADS["c2"].replace(B=1, Hq=20, Hkv=5, L=4096 + 37, T=3, k=12, needles=3, seed=501),
    # d = 64, G * T = 16
    "d64": synth.WORKLOADS["c2"].replace(B=2, Hq=8, Hkv=2, d=64, L=3000, T=4, k=9, needles=2, seed=502),
    # 320 groups: more than the clusters that fit at once (several rounds per cluster)
    "many_groups": synth.WORKLOADS["c2"].replace(B=40, L=2048 + 64, k=6, needles=1, seed=503),
    # G = 1, 16 K/V heads
    "g1": synth.WORKLOADS["c2"].replace(B=1, Hq=16, Hkv=16, L=8192, k=20, needles=2, seed=504),
}


@pytest.fixture(scope="module")
def sa():
    import top_block_sparse_pooled_b300 as m
    return m


def _all_rows(wl):
    return np.array([(b, t, h) for b in range(wl.B) for t in range(wl.T) for h in range(wl.Hq)], dtype=np.int64)


def _run_pair(sa, wl, x):
    """The fused call and the two separate calls on the same inputs."""
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    sk = torch.empty((wl.B, wl.Hkv, wl.nb, wl.d), dtype=torch.float32, device="cuda")
    sa.sa_build_sketch(k, wl.L, wl.Bk, sk)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    shp = (wl.B, wl.Hkv, 1, kmax)
    f_idx = torch.full(shp, -7, dtype=torch.int32, device="cuda")
    f_cnt = torch.full((wl.B, wl.Hkv, 1), -7, dtype=torch.int32, device="cuda")
    f_sc = torch.full((wl.B, wl.Hkv, 1, wl.nb), float("nan"), dtype=torch.float32, device="cuda")
    f_out = torch.full_like(q, float("nan"))
    sa.sa_select_decode(q, sk, k, v, wl.L, wl.Bk, wl.k, wl.scale, f_idx, f_cnt, f_out, scores=f_sc)
    s_idx = torch.full(shp, -7, dtype=torch.int32, device="cuda")
    s_cnt = torch.full((wl.B, wl.Hkv, 1), -7, dtype=torch.int32, device="cuda")
    s_sc = torch.full((wl.B, wl.Hkv, 1, wl.nb), float("nan"), dtype=torch.float32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_SKETCH, q, sk, s_sc, wl.Hkv, wl.L, wl.L, wl.Bk, 0, False, wl.k, 0, 1, wl.scale,
                      s_idx, s_cnt)
    s_out = torch.full_like(q, float("nan"))
    ws = torch.zeros(sa.sa_decode_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, kmax), dtype=torch.uint8,
                     device="cuda")
    sa.sa_decode(q, k, v, s_idx, s_cnt, wl.L, wl.Bk, wl.scale, s_out, ws)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    return (f_idx, f_cnt, f_sc, f_out), (s_idx, s_cnt, s_sc, s_out), kmax


@pytest.mark.parametrize("name", sorted(CASES))
def test_select_decode_equals_separate_calls_and_oracle(sa, name):
    wl = CASES[name]
    x = synth.make_inputs(wl)
    (f_idx, f_cnt, f_sc, f_out), (s_idx, s_cnt, s_sc, s_out), kmax = _run_pair(sa, wl, x)
    # the same scores and the same selection, bit for bit
    assert torch.equal(f_sc.view(torch.int32), s_sc.view(torch.int32)), "scores differ from sa_select_topk"
    assert torch.equal(f_idx, s_idx) and torch.equal(f_cnt, s_cnt), "selection differs from sa_select_topk"
    # the same output as sa_decode on that selection, up to the order of the fp32 sums (the two calls
    # may split a group's blocks over different numbers of CTAs): one bf16 rounding step at most
    assert_close(host(f_out), host(s_out), atol=1e-3, rtol=2.0 ** -7, what=name + " fused vs separate")
    # the selection against the oracle (near-tie swaps only), the output against the oracle's
    # exact attention on the kernel's (checked) selection
    o_idx, o_cnt, o_s, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    g_idx = f_idx.cpu().numpy().reshape(wl.B * wl.Hkv, kmax)
    g_cnt = f_cnt.cpu().numpy().reshape(-1)
    assert_selection(g_idx, g_cnt, o_idx, o_cnt, o_s, what=name)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, _all_rows(wl), g_idx, g_cnt)
    assert_close(host(f_out).reshape(ref.shape), ref, what=name)


@pytest.mark.parametrize("name", ["c3", "ragged_t3", "g1"])
def test_cluster_decode_on_oracle_selection(sa, name):
    """sa_decode (cluster path for these group counts) fed the oracle's selection, every row."""
    wl = CASES[name]
    x = synth.make_inputs(wl)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    o_idx, o_cnt, _, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    idx = torch.from_numpy(np.ascontiguousarray(o_idx.reshape(wl.B, wl.Hkv, 1, kmax))).cuda()
    cnt = torch.from_numpy(np.ascontiguousarray(o_cnt.reshape(wl.B, wl.Hkv, 1))).cuda()
    out = torch.full_like(q, float("nan"))
    ws = torch.zeros(sa.sa_decode_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, kmax), dtype=torch.uint8,
                     device="cuda")
    sa.sa_decode(q, k, v, idx, cnt, wl.L, wl.Bk, wl.scale, out, ws)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, _all_rows(wl), o_idx, o_cnt)
    assert_close(host(out).reshape(ref.shape), ref, what=name)


@pytest.mark.parametrize("L", [1, 40, 64, 65, 128, 200])
def test_select_decode_tiny_contexts(sa, L):
    """One to four blocks: the sink and local blocks coincide or cover everything."""
    T = min(2, L)
    wl = synth.WORKLOADS["c2"].replace(B=1, Hq=8, Hkv=2, L=L, T=T, k=1, needles=0, seed=520 + L)
    x = synth.make_inputs(wl)
    (f_idx, f_cnt, _, f_out), (s_idx, s_cnt, _, s_out), kmax = _run_pair(sa, wl, x)
    assert torch.equal(f_idx, s_idx) and torch.equal(f_cnt, s_cnt)
    assert_close(host(f_out), host(s_out), atol=1e-3, rtol=2.0 ** -7, what="L=%d fused vs separate" % L)
    g_idx = f_idx.cpu().numpy().reshape(wl.B * wl.Hkv, kmax)
    g_cnt = f_cnt.cpu().numpy().reshape(-1)
    o_idx, o_cnt, o_s, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    assert_selection(g_idx, g_cnt, o_idx, o_cnt, o_s, what="L=%d" % L)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, _all_rows(wl), g_idx, g_cnt)
    assert_close(host(f_out).reshape(ref.shape), ref, what="L=%d" % L)


def test_cluster_decode_skips_invalid_entries(sa):
    """Entries past cnt, negative ids and ids past the context are skipped; cnt = 0 gives zeros."""
    wl = CASES["ragged_t3"]
    x = synth.make_inputs(wl)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    o_idx, o_cnt, _, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    groups = wl.B * wl.Hkv
    pad = -np.ones((groups, kmax + 3), dtype=np.int32)
    pcnt = o_cnt + 2
    for g in range(groups):
        pad[g, 0] = -1
        pad[g, 1] = wl.nb + 9
        pad[g, 2: 2 + o_cnt[g]] = o_idx[g, : o_cnt[g]]
        pad[g, 2 + o_cnt[g]] = 3  # past cnt: never read
    pcnt[1] = 0
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    idx = torch.from_numpy(pad.reshape(wl.B, wl.Hkv, 1, kmax + 3)).cuda()
    cnt = torch.from_numpy(pcnt.reshape(wl.B, wl.Hkv, 1).astype(np.int32)).cuda()
    out = torch.full_like(q, float("nan"))
    ws = torch.zeros(sa.sa_decode_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, kmax + 3), dtype=torch.uint8,
                     device="cuda")
    sa.sa_decode(q, k, v, idx, cnt, wl.L, wl.Bk, wl.scale, out, ws)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, _all_rows(wl), o_idx, o_cnt)
    ref = ref.reshape(wl.B, wl.T, wl.Hq, wl.d)
    ref[0, :, wl.G: 2 * wl.G] = 0.0  # group 1 has cnt 0
    assert_close(host(out).reshape(ref.shape), ref, what="padded")


def test_select_decode_repeated_calls_are_identical(sa):
    """Back-to-back fused calls on the same buffers give the same bits (no state carried over)."""
    wl = CASES["c3"]
    x = synth.make_inputs(wl)
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    sk = torch.empty((wl.B, wl.Hkv, wl.nb, wl.d), dtype=torch.float32, device="cuda")
    sa.sa_build_sketch(k, wl.L, wl.Bk, sk)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    outs = []
    for _ in range(3):
        idx = torch.empty((wl.B, wl.Hkv, 1, kmax), dtype=torch.int32, device="cuda")
        cnt = torch.empty((wl.B, wl.Hkv, 1), dtype=torch.int32, device="cuda")
        out = torch.empty_like(q)
        sa.sa_select_decode(q, sk, k, v, wl.L, wl.Bk, wl.k, wl.scale, idx, cnt, out)
        outs.append((idx, cnt, out))
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    for idx, cnt, out in outs[1:]:
        assert torch.equal(idx, outs[0][0]) and torch.equal(cnt, outs[0][1])
        assert torch.equal(out.view(torch.int16), outs[0][2].view(torch.int16))
