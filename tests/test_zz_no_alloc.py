"""sa_decode_noalloc: decode through the library's fixed scratch, for callers
that cannot allocate device memory (a host runtime that owns the device memory
pool, or a latency path that must not call cudaMalloc).

It must give the same results as sa_decode with a caller-provided workspace,
on back-to-back calls (the scratch keeps the previous call's contents), and
reject problems whose scratch need exceeds its fixed size before any device
work.  This file is collected last so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    import top_block_sparse_pooled_b300 as m
    return m


def _selection(sa, wl, x, alt_seed=None):
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    o_idx, o_cnt, _, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    if alt_seed is not None:  # a different valid selection of the same size
        rng = np.random.default_rng(alt_seed)
        o_idx = o_idx.copy()
        for g in range(o_idx.shape[0]):
            o_idx[g, 1:-1] = np.sort(rng.choice(np.arange(1, wl.nb - 1), size=kmax - 2, replace=False))
    idx = torch.from_numpy(np.ascontiguousarray(o_idx.reshape(wl.B, wl.Hkv, 1, kmax))).cuda()
    cnt = torch.from_numpy(np.ascontiguousarray(o_cnt.reshape(wl.B, wl.Hkv, 1))).cuda()
    return idx, cnt, kmax


@pytest.mark.parametrize("name", ["bf16_gqa", "f32_split"])
def test_noalloc_matches_workspace_decode_twice(sa, name):
    wl = {"bf16_gqa": synth.WORKLOADS["c2"].replace(B=2, L=8192 + 17, T=2, k=24, seed=601),
          "f32_split": synth.WORKLOADS["c1"].replace(Hq=8, Hkv=2, d=128, L=3000, k=6, seed=602)}[name]
    x = synth.make_inputs(wl)
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    for call, alt in enumerate((None, 7)):
        idx, cnt, kmax = _selection(sa, wl, x, alt)
        ws = torch.zeros(sa.sa_decode_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, kmax), dtype=torch.uint8,
                         device="cuda")
        ref = torch.empty_like(q)
        sa.sa_decode(q, k, v, idx, cnt, wl.L, wl.Bk, wl.scale, ref, ws)
        got = torch.full_like(q, float("nan"))
        sa.sa_decode_noalloc(q, k, v, idx, cnt, wl.L, wl.Bk, wl.scale, got)
        torch.cuda.synchronize()
        assert sa.sa_device_status(clear=True) == 0
        assert_close(host(got), host(ref), what="%s call %d" % (name, call))


def test_noalloc_rejects_oversized_problem(sa):
    """A problem needing more scratch than the fixed array is refused on the host."""
    B, T, Hq, Hkv, d, kmax = 64, 1, 32, 8, 128, 512
    assert sa.sa_decode_workspace_bytes(B, T, Hq, Hkv, d, kmax) > (8 << 20)
    # the shapes the binding passes are the oversized problem's; the memory behind them is a few
    # bytes (broadcast views), since the call is refused before it reads any of it
    q = torch.zeros((1, 1, 1, d), dtype=torch.bfloat16, device="cuda").expand(B, T, Hq, d)
    kc = torch.zeros((1, 1, 1, d), dtype=torch.bfloat16, device="cuda").expand(B, Hkv, 64 * 512, d)
    idx = torch.zeros((1, 1, 1, 1), dtype=torch.int32, device="cuda").expand(B, Hkv, 1, kmax)
    cnt = torch.zeros((1, 1, 1), dtype=torch.int32, device="cuda").expand(B, Hkv, 1)
    out = torch.zeros((1, 1, 1, d), dtype=torch.bfloat16, device="cuda").expand(B, T, Hq, d)
    with pytest.raises(sa.SparseAttnError) as e:
        sa.sa_decode_noalloc(q, kc, kc, idx, cnt, 64 * 512, 64, 0.088, out)
    assert e.value.status == sa.SA_ERR_INVALID_ARG and "scratch" in str(e.value)


@pytest.mark.parametrize("name", ["bf16_gqa", "f32_split"])
def test_noalloc_recovers_from_left_over_counters(sa, name):
    """Arrival counters left non-zero in the scratch (as by a call that gave up) do not change the
    next call's result: it clears them on its stream before the launch."""
    wl = {"bf16_gqa": synth.WORKLOADS["c2"].replace(B=2, L=4096 + 9, T=1, k=16, seed=603),
          "f32_split": synth.WORKLOADS["c1"].replace(Hq=8, Hkv=2, d=128, L=2000, k=5, seed=604)}[name]
    x = synth.make_inputs(wl)
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    idx, cnt, kmax = _selection(sa, wl, x, None)
    ws = torch.zeros(sa.sa_decode_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, kmax), dtype=torch.uint8,
                     device="cuda")
    ref = torch.empty_like(q)
    sa.sa_decode(q, k, v, idx, cnt, wl.L, wl.Bk, wl.scale, ref, ws)
    sa.sa_selftest_poison_noalloc(4096)
    got = torch.full_like(q, float("nan"))
    sa.sa_decode_noalloc(q, k, v, idx, cnt, wl.L, wl.Bk, wl.scale, got)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    assert_close(host(got), host(ref), what="%s after poisoned counters" % name)
