"""Failure detection without a GPU fault: a bounded wait that nothing completes gives up, records
SA_ERR_TIMEOUT in the device status word, and the context stays usable for exact work."""
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


def test_bounded_wait_reports_timeout_and_context_survives(sa):
    assert sa.sa_device_status(clear=True) == 0
    sa.sa_selftest_wait_timeout(20_000_000)  # 20 ms
    assert sa.sa_device_status(clear=True) == sa.SA_ERR_TIMEOUT
    assert sa.sa_device_status(clear=True) == 0  # cleared
    # the same context then runs a decode step exactly
    wl = synth.WORKLOADS["c1"]
    x = synth.make_inputs(wl)
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    sk = torch.empty((wl.B, wl.Hkv, wl.nb, wl.d), dtype=torch.float32, device="cuda")
    sa.sa_build_sketch(k, wl.L, wl.Bk, sk)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    idx = torch.empty((wl.B, wl.Hkv, 1, kmax), dtype=torch.int32, device="cuda")
    cnt = torch.empty((wl.B, wl.Hkv, 1), dtype=torch.int32, device="cuda")
    sa.sa_select_topk(sa.SA_SELECT_SKETCH, q, sk, None, wl.Hkv, wl.L, wl.L, wl.Bk, 0, False, wl.k, 0, 1, wl.scale,
                      idx, cnt)
    ws = torch.zeros(sa.sa_decode_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, kmax), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(q)
    sa.sa_decode(q, k, v, idx, cnt, wl.L, wl.Bk, wl.scale, out, ws)
    torch.cuda.synchronize()
    assert sa.sa_device_status(clear=True) == 0
    o_idx, o_cnt, _, _ = oracle.decode_select(x.q, x.k, wl, kmax=kmax)
    assert np.array_equal(idx.cpu().numpy().reshape(o_idx.shape), o_idx)
    rows = [(b, t, h) for b in range(wl.B) for t in range(wl.T) for h in range(wl.Hq)]
    ref, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, rows, o_idx, o_cnt)
    assert_close(host(out).reshape(ref.shape), ref, atol=1e-4, rtol=1e-4, what="decode after the self-test")
