"""GPU parity of the decode path (a1 sketch/append, a2+a3 select, a4 decode) against the CPU oracle."""
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


def _sketch_buf(wl, Ls=None):
    Ls = Ls or wl.L
    return torch.empty((wl.B, wl.Hkv, (Ls + wl.Bk - 1) // wl.Bk, wl.d), dtype=torch.float32, device="cuda")


def _check_status(sa):
    assert sa.sa_device_status(clear=True) == 0


DECODE_CASES = {
    "c1": synth.WORKLOADS["c1"],
    "c2": synth.WORKLOADS["c2"],
    "c3": synth.WORKLOADS["c3"],
    # ragged tail (partial last block), T=3 causal rows, G*T = 12, 5 groups
    "ragged": synth.WORKLOADS["c2"].replace(B=1, Hq=20, Hkv=5, L=4096 + 37, T=3, k=12, needles=3, seed=77),
    # fp32, d=128, odd budget
    "f32_d128": synth.WORKLOADS["c1"].replace(d=128, Hq=8, Hkv=2, L=2048 + 5, k=7, seed=78),
    # bf16, d=64, G*T = 32
    "bf16_d64": synth.WORKLOADS["c2"].replace(B=2, Hq=16, Hkv=2, d=64, L=3000, T=4, k=9, seed=79),
    # many groups (80: more than half the SMs), so the decode is the split-KV launch over all SMs
    # with the last CTA of each group merging its partials (G*T = 8, ragged tail)
    "many_groups": synth.WORKLOADS["c2"].replace(B=20, Hq=16, Hkv=4, L=2048 + 13, T=2, k=10, needles=2, seed=80),
}


@pytest.mark.parametrize("name", sorted(DECODE_CASES))
def test_sketch_matches_oracle(sa, name):
    wl = DECODE_CASES[name]
    x = synth.make_inputs(wl)
    k = dev(x.k)
    sk = _sketch_buf(wl)
    sa.sa_build_sketch(k, wl.L, wl.Bk, sk)
    torch.cuda.synchronize()
    _check_status(sa)
    ref = oracle.block_means(x.k, wl.L, wl.Bk)
    got = host(sk).reshape(ref.shape)
    assert_close(got, ref, atol=1e-6, rtol=1e-5, what="sketch")


@pytest.mark.parametrize("name", sorted(DECODE_CASES))
def test_select_matches_oracle(sa, name):
    wl = DECODE_CASES[name]
    x = synth.make_inputs(wl)
    q, k = dev(x.q), dev(x.k)
    sk = _sketch_buf(wl)
    sa.sa_build_sketch(k, wl.L, wl.Bk, sk)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    idx = torch.full((wl.B, wl.Hkv, 1, kmax), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((wl.B, wl.Hkv, 1), dtype=torch.int32, device="cuda")
    scores = torch.empty((wl.B, wl.Hkv, 1, wl.nb), dtype=torch.float32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_SKETCH, q, sk, scores, wl.Hkv, wl.L, wl.L, wl.Bk, 0, False, wl.k, 0, 1, wl.scale,
                      idx, cnt)
    torch.cuda.synchronize()
    _check_status(sa)
    o_idx, o_cnt, o_s, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    g_s = host(scores).reshape(o_s.shape)
    scale = np.abs(o_s).max(axis=1, keepdims=True)
    assert np.all(np.abs(g_s - o_s) <= 2e-6 * scale), "scores differ beyond fp32 rounding"
    assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, o_s, what=name)
    # needle blocks are selected by the kernel too
    g_idx = idx.cpu().numpy().reshape(wl.B * wl.Hkv, -1)
    for g in range(wl.B * wl.Hkv):
        needles = set(np.nonzero(x.needle_mask[g])[0].tolist())
        assert needles <= set(g_idx[g].tolist())


def _decode_gpu(sa, wl, x, idx_np, cnt_np, kmax):
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    idx = torch.from_numpy(np.ascontiguousarray(idx_np.reshape(wl.B, wl.Hkv, 1, kmax))).cuda()
    cnt = torch.from_numpy(np.ascontiguousarray(cnt_np.reshape(wl.B, wl.Hkv, 1))).cuda()
    out = torch.empty_like(q)
    ws = torch.zeros(sa.sa_decode_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, kmax), dtype=torch.uint8,
                     device="cuda")
    sa.sa_decode(q, k, v, idx, cnt, wl.L, wl.Bk, wl.scale, out, ws)
    torch.cuda.synchronize()
    _check_status(sa)
    return host(out)


def _all_rows(wl):
    return np.array([(b, t, h) for b in range(wl.B) for t in range(wl.T) for h in range(wl.Hq)], dtype=np.int64)


@pytest.mark.parametrize("name", sorted(DECODE_CASES))
def test_decode_matches_oracle_on_oracle_selection(sa, name):
    wl = DECODE_CASES[name]
    x = synth.make_inputs(wl)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    o_idx, o_cnt, _, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    got = _decode_gpu(sa, wl, x, o_idx, o_cnt, kmax)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, _all_rows(wl), o_idx, o_cnt)
    tol = 1e-4 if wl.dtype == "f32" else 1e-2
    err = assert_close(got.reshape(ref.shape), ref, atol=tol, rtol=tol, what=name)
    print("%s max abs err %.3g" % (name, err))


def test_full_budget_equals_dense(sa):
    """k >= #candidates: the kernel's sparse attention is dense attention."""
    wl = DECODE_CASES["ragged"].replace(k=1000)
    x = synth.make_inputs(wl)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    assert kmax == wl.nb
    idx = np.tile(np.arange(wl.nb, dtype=np.int32), (wl.B * wl.Hkv, 1))
    cnt = np.full((wl.B * wl.Hkv,), wl.nb, dtype=np.int32)
    got = _decode_gpu(sa, wl, x, idx, cnt, kmax)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, _all_rows(wl))
    assert_close(got.reshape(ref.shape), ref, what="dense")


@pytest.mark.parametrize("L", [1, 40, 64, 65, 128])
def test_tiny_contexts(sa, L):
    """One or two blocks (sink == local), partial blocks, T up to L."""
    T = min(2, L)
    wl = synth.WORKLOADS["c1"].replace(L=L, T=T, k=4, needles=0, seed=90 + L)
    x = synth.make_inputs(wl)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    q, k = dev(x.q), dev(x.k)
    sk = _sketch_buf(wl)
    sa.sa_build_sketch(k, wl.L, wl.Bk, sk)
    idx = torch.empty((1, 1, 1, kmax), dtype=torch.int32, device="cuda")
    cnt = torch.empty((1, 1, 1), dtype=torch.int32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_SKETCH, q, sk, None, wl.Hkv, wl.L, wl.L, wl.Bk, 0, False, wl.k, 0, 1, wl.scale,
                      idx, cnt)
    o_idx, o_cnt, o_s, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, o_s)
    got = _decode_gpu(sa, wl, x, o_idx, o_cnt, kmax)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, _all_rows(wl), o_idx, o_cnt)
    assert_close(got.reshape(ref.shape), ref, atol=1e-4, rtol=1e-4)


def test_split_invariance(sa):
    """Padding the block list (more, shorter splits) leaves the merged output unchanged."""
    wl = DECODE_CASES["c2"].replace(B=2, L=8192)
    x = synth.make_inputs(wl)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    o_idx, o_cnt, _, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    a = _decode_gpu(sa, wl, x, o_idx, o_cnt, kmax)
    big = 4 * kmax
    pad = -np.ones((o_idx.shape[0], big), dtype=np.int32)
    pad[:, :kmax] = o_idx
    b = _decode_gpu(sa, wl, x, pad, o_cnt, big)
    assert_close(a, b, atol=2e-3, rtol=2e-3, what="split invariance")


def test_append_kv_updates_cache_and_sketch(sa):
    wl = DECODE_CASES["ragged"]
    x = synth.make_inputs(wl)
    Ls = wl.L + 50
    pos = wl.L - wl.T
    kc = torch.zeros((wl.B, wl.Hkv, Ls, wl.d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kfull, vfull = dev(x.k), dev(x.v)
    kc[:, :, :pos] = kfull[:, :, :pos]
    vc[:, :, :pos] = vfull[:, :, :pos]
    sk = _sketch_buf(wl, Ls)
    sa.sa_build_sketch(kc, pos, wl.Bk, sk)
    k_new = kfull[:, :, pos:wl.L].permute(0, 2, 1, 3).contiguous()
    v_new = vfull[:, :, pos:wl.L].permute(0, 2, 1, 3).contiguous()
    sa.sa_append_kv(k_new, v_new, kc, vc, pos, wl.Bk, sk)
    torch.cuda.synchronize()
    _check_status(sa)
    assert torch.equal(kc[:, :, :wl.L], kfull) and torch.equal(vc[:, :, :wl.L], vfull)
    assert torch.count_nonzero(kc[:, :, wl.L:]) == 0
    ref = oracle.block_means(x.k, wl.L, wl.Bk)
    got = host(sk)[:, :, : wl.nb].reshape(ref.shape)
    assert_close(got, ref, atol=1e-6, rtol=1e-5, what="sketch after append")


@pytest.mark.parametrize("host_io", [False, True, "pageable"])
def test_decode_step_matches_oracle(sa, host_io):
    """append + select + decode in one call: device I/O, pinned host I/O (new rows and the output
    used in place), pageable host I/O (staged by copies)."""
    wl = DECODE_CASES["c2"].replace(B=2, L=8192)
    x = synth.make_inputs(wl)
    pos = wl.L - wl.T
    kfull, vfull = dev(x.k), dev(x.v)
    kc, vc = kfull.clone(), vfull.clone()
    kc[:, :, pos:] = 0
    vc[:, :, pos:] = 0
    sk = _sketch_buf(wl)
    sa.sa_build_sketch(kc, pos, wl.Bk, sk)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    idx = torch.empty((wl.B, wl.Hkv, 1, kmax), dtype=torch.int32, device="cuda")
    cnt = torch.empty((wl.B, wl.Hkv, 1), dtype=torch.int32, device="cuda")
    ws = torch.zeros(sa.sa_decode_step_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, sa.SA_BF16, kmax),
                     dtype=torch.uint8, device="cuda")
    q = dev(x.q)
    k_new = kfull[:, :, pos:].permute(0, 2, 1, 3).contiguous()
    v_new = vfull[:, :, pos:].permute(0, 2, 1, 3).contiguous()
    out = torch.empty_like(q)
    if host_io == "pageable":
        q, k_new, v_new = (t.cpu() for t in (q, k_new, v_new))
        out = torch.empty(q.shape, dtype=q.dtype)
    elif host_io:
        q, k_new, v_new = (t.cpu().pin_memory() for t in (q, k_new, v_new))
        out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    sa.sa_decode_step(q, k_new, v_new, kc, vc, sk, wl.L, wl.Bk, wl.k, wl.scale, idx, cnt, out, ws,
                      host_io=bool(host_io))
    torch.cuda.synchronize()
    _check_status(sa)
    o_idx, o_cnt, o_s, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, o_s)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, pos, wl.Bk, wl.scale, _all_rows(wl), o_idx, o_cnt)
    assert_close(host(out).reshape(ref.shape), ref, what="decode step")
    _check_appended_state(wl, x, kc, vc, sk)


def _check_appended_state(wl, x, kc, vc, sk):
    """After a step: the caches hold the new rows bit for bit and the sketch equals the oracle's."""
    assert torch.equal(kc.view(torch.int16), dev(x.k).view(torch.int16)), "key cache after the step"
    assert torch.equal(vc.view(torch.int16), dev(x.v).view(torch.int16)), "value cache after the step"
    ref = oracle.block_means(x.k, wl.L, wl.Bk)
    assert_close(host(sk)[:, :, : wl.nb].reshape(ref.shape), ref, atol=1e-6, rtol=1e-5, what="sketch after the step")


@pytest.mark.parametrize("T,L", [(4, 8192), (3, 8193), (2, 65)])
def test_decode_step_multi_token(sa, T, L):
    """T new rows per step: within one block (the append runs inside the selection + decode launch)
    and across a block boundary (a launch of its own), with the cache and sketch checked after."""
    wl = DECODE_CASES["c2"].replace(B=2, L=L, T=T, k=8, needles=2, seed=700 + T)
    x = synth.make_inputs(wl)
    pos = wl.L - wl.T
    kc, vc = dev(x.k).clone(), dev(x.v).clone()
    kc[:, :, pos:] = 0
    vc[:, :, pos:] = 0
    sk = _sketch_buf(wl)
    sa.sa_build_sketch(kc, pos, wl.Bk, sk)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    idx = torch.empty((wl.B, wl.Hkv, 1, kmax), dtype=torch.int32, device="cuda")
    cnt = torch.empty((wl.B, wl.Hkv, 1), dtype=torch.int32, device="cuda")
    ws = torch.zeros(sa.sa_decode_step_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, sa.SA_BF16, kmax),
                     dtype=torch.uint8, device="cuda")
    q = dev(x.q)
    k_new = dev(x.k)[:, :, pos:].permute(0, 2, 1, 3).contiguous()
    v_new = dev(x.v)[:, :, pos:].permute(0, 2, 1, 3).contiguous()
    out = torch.empty_like(q)
    sa.sa_decode_step(q, k_new, v_new, kc, vc, sk, wl.L, wl.Bk, wl.k, wl.scale, idx, cnt, out, ws)
    torch.cuda.synchronize()
    _check_status(sa)
    o_idx, o_cnt, o_s, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, o_s)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, pos, wl.Bk, wl.scale, _all_rows(wl), o_idx, o_cnt)
    assert_close(host(out).reshape(ref.shape), ref, what="decode step T=%d" % T)
    _check_appended_state(wl, x, kc, vc, sk)


@pytest.mark.parametrize("base,B,T,L", [("c3", 1, 4, 8192), ("c3", 1, 1, 4096 + 37), ("c2", 8, 2, 4096 + 37)])
def test_decode_step_host_io_multi_token(sa, base, B, T, L):
    """Pinned host I/O in the one-launch step with T query rows per sequence: the new rows are read
    and out is written in place in mapped host memory; q is read in place too when each group's
    cluster has at most two CTAs (many groups), else staged by one copy (few groups)."""
    wl = DECODE_CASES[base].replace(B=B, L=L, T=T, k=12, needles=2, seed=720 + T)
    x = synth.make_inputs(wl)
    pos = wl.L - wl.T
    kc, vc = dev(x.k).clone(), dev(x.v).clone()
    kc[:, :, pos:] = 0
    vc[:, :, pos:] = 0
    sk = _sketch_buf(wl)
    sa.sa_build_sketch(kc, pos, wl.Bk, sk)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    idx = torch.empty((wl.B, wl.Hkv, 1, kmax), dtype=torch.int32, device="cuda")
    cnt = torch.empty((wl.B, wl.Hkv, 1), dtype=torch.int32, device="cuda")
    ws = torch.zeros(sa.sa_decode_step_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, sa.SA_BF16, kmax),
                     dtype=torch.uint8, device="cuda")
    q = dev(x.q).cpu().pin_memory()
    k_new = dev(x.k)[:, :, pos:].permute(0, 2, 1, 3).contiguous().cpu().pin_memory()
    v_new = dev(x.v)[:, :, pos:].permute(0, 2, 1, 3).contiguous().cpu().pin_memory()
    out = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
    sa.sa_decode_step(q, k_new, v_new, kc, vc, sk, wl.L, wl.Bk, wl.k, wl.scale, idx, cnt, out, ws, host_io=True)
    torch.cuda.synchronize()
    _check_status(sa)
    o_idx, o_cnt, o_s, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, o_s, what="host I/O T=%d" % T)
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, pos, wl.Bk, wl.scale, _all_rows(wl), o_idx, o_cnt)
    assert_close(host(out).reshape(ref.shape), ref, what="host I/O decode step T=%d" % T)
    _check_appended_state(wl, x, kc, vc, sk)


def test_decode_step_many_groups(sa):
    """The one-launch step with more groups than co-resident clusters: clusters take several
    groups in turn (append, selection and attention of each), and sa_decode on the same selection
    takes the split-KV launch over all SMs; both agree with the oracle."""
    wl = DECODE_CASES["many_groups"].replace(B=40, seed=81)  # 160 groups
    x = synth.make_inputs(wl)
    pos = wl.L - wl.T
    kc, vc = dev(x.k).clone(), dev(x.v).clone()
    kc[:, :, pos:] = 0
    vc[:, :, pos:] = 0
    sk = _sketch_buf(wl)
    sa.sa_build_sketch(kc, pos, wl.Bk, sk)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    idx = torch.empty((wl.B, wl.Hkv, 1, kmax), dtype=torch.int32, device="cuda")
    cnt = torch.empty((wl.B, wl.Hkv, 1), dtype=torch.int32, device="cuda")
    ws = torch.zeros(sa.sa_decode_step_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, sa.SA_BF16, kmax),
                     dtype=torch.uint8, device="cuda")
    q = dev(x.q)
    k_new = dev(x.k)[:, :, pos:].permute(0, 2, 1, 3).contiguous()
    v_new = dev(x.v)[:, :, pos:].permute(0, 2, 1, 3).contiguous()
    out = torch.empty_like(q)
    sa.sa_decode_step(q, k_new, v_new, kc, vc, sk, wl.L, wl.Bk, wl.k, wl.scale, idx, cnt, out, ws)
    torch.cuda.synchronize()
    _check_status(sa)
    o_idx, o_cnt, o_s, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, o_s, what="many groups")
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, pos, wl.Bk, wl.scale, _all_rows(wl), o_idx, o_cnt)
    assert_close(host(out).reshape(ref.shape), ref, what="many-group decode step")
    _check_appended_state(wl, x, kc, vc, sk)
    # the attention alone on the oracle's selection (split-KV launch, last-CTA merge)
    got = _decode_gpu(sa, wl, x, o_idx, o_cnt, kmax)
    assert_close(got.reshape(ref.shape), ref, what="many-group decode")


def test_decode_step_graph_replay_reads_new_inputs(sa):
    """On a non-default stream the step is captured once and replayed: a second call with the same
    buffers but new query contents gives the new query's exact result."""
    wl = DECODE_CASES["c2"].replace(B=2, L=8192)
    x = synth.make_inputs(wl)
    pos = wl.L - wl.T
    kfull, vfull = dev(x.k), dev(x.v)
    kc, vc = kfull.clone(), vfull.clone()
    kc[:, :, pos:] = 0
    vc[:, :, pos:] = 0
    sk = _sketch_buf(wl)
    sa.sa_build_sketch(kc, pos, wl.Bk, sk)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    idx = torch.empty((wl.B, wl.Hkv, 1, kmax), dtype=torch.int32, device="cuda")
    cnt = torch.empty((wl.B, wl.Hkv, 1), dtype=torch.int32, device="cuda")
    ws = torch.zeros(sa.sa_decode_step_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, sa.SA_BF16, kmax),
                     dtype=torch.uint8, device="cuda")
    q = dev(x.q).cpu().pin_memory()
    k_new = kfull[:, :, pos:].permute(0, 2, 1, 3).contiguous().cpu().pin_memory()
    v_new = vfull[:, :, pos:].permute(0, 2, 1, 3).contiguous().cpu().pin_memory()
    out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    st = torch.cuda.Stream()
    qs = [x.q, np.ascontiguousarray(x.q[:, :, ::-1, :])]  # second call: the heads in reverse order
    step = sa.DecodeStep(q, k_new, v_new, kc, vc, sk, wl.L, wl.Bk, wl.k, wl.scale, idx, cnt, out, ws,
                         host_io=True, stream=st)
    for call, qn in enumerate(qs):
        q.copy_(torch.from_numpy(qn.view(np.int16)).view(torch.bfloat16))
        if call == 0:  # the plain call, then the prepared one on the same buffers
            with torch.cuda.stream(st):
                sa.sa_decode_step(q, k_new, v_new, kc, vc, sk, wl.L, wl.Bk, wl.k, wl.scale, idx, cnt, out, ws,
                                  host_io=True)
        else:
            step()
        st.synchronize()
        _check_status(sa)
        o_idx, o_cnt, o_s, _ = oracle.decode_select(qn, x.k, wl, kmax=kmax)
        assert_selection(idx.cpu().numpy(), cnt.cpu().numpy(), o_idx, o_cnt, o_s, what="call %d" % call)
        ref, _ = oracle.attend(qn, x.k, x.v, wl.Hkv, wl.L, pos, wl.Bk, wl.scale, _all_rows(wl), o_idx, o_cnt)
        assert_close(host(out).reshape(ref.shape), ref, what="decode step, call %d" % call)


def test_workspace_reuse_keeps_counters_clean(sa):
    """Back-to-back calls on one workspace (different selections) are each exact."""
    wl = DECODE_CASES["c3"].replace(L=16384, k=20, needles=5)
    x = synth.make_inputs(wl)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    ws = torch.zeros(sa.sa_decode_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, kmax), dtype=torch.uint8,
                     device="cuda")
    o_idx, o_cnt, _, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    rng = np.random.default_rng(5)
    alt = o_idx.copy()
    for g in range(alt.shape[0]):  # a different valid selection: shuffle the non-forced blocks
        alt[g, 1:-1] = np.sort(rng.choice(np.arange(1, wl.nb - 1), size=kmax - 2, replace=False))
    rows = _all_rows(wl)
    for sel in (o_idx, alt, o_idx):
        idx = torch.from_numpy(np.ascontiguousarray(sel.reshape(wl.B, wl.Hkv, 1, kmax))).cuda()
        cnt = torch.from_numpy(np.ascontiguousarray(o_cnt.reshape(wl.B, wl.Hkv, 1))).cuda()
        out = torch.empty_like(q)
        sa.sa_decode(q, k, v, idx, cnt, wl.L, wl.Bk, wl.scale, out, ws)
        torch.cuda.synchronize()
        _check_status(sa)
        ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, rows, sel, o_cnt)
        assert_close(host(out).reshape(ref.shape), ref, what="reuse")
    # the arrival counters at the head of the workspace are back to zero
    assert int(ws[: 4 * wl.B * wl.Hkv].view(torch.int32).abs().sum()) == 0
