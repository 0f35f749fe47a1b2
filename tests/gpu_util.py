"""Helpers shared by the GPU parity tests (device upload, comparison rules)."""
from __future__ import annotations

import numpy as np
import torch

# Output tolerance for attention outputs (bf16 inputs, fp32 accumulation):
# |gpu - oracle| <= ATOL + RTOL * |oracle|, per element.
ATOL = 1e-2
RTOL = 1e-2
# Selections must match exactly except swaps whose oracle scores differ by less
# than SEL_REL times the unit's largest |score|.
SEL_REL = 1e-5


def dev(a: np.ndarray, shape=None) -> torch.Tensor:
    """numpy (uint16 bf16 bits or float32) -> CUDA tensor (bfloat16 / float32)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    elif a.dtype == np.float32:
        t = torch.from_numpy(a)
    else:
        raise TypeError(a.dtype)
    if shape is not None:
        t = t.reshape(shape)
    return t.cuda()


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy().astype(np.float64)
    return t.numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, atol=ATOL, rtol=RTOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))), err.shape)
        raise AssertionError("%s: %d/%d elements out of tolerance; worst at %s: got %r ref %r" %
                             (what, int(bad.sum()), bad.size, i, got[i], ref[i]))
    return float(err.max())


def assert_selection(g_idx, g_cnt, o_idx, o_cnt, o_scores, rel=SEL_REL, what=""):
    """Exact match, except swaps between blocks whose oracle scores are near-ties."""
    g_idx = np.asarray(g_idx).reshape(len(o_cnt), -1)
    g_cnt = np.asarray(g_cnt).reshape(-1)
    swaps = 0
    for u in range(len(o_cnt)):
        n = int(g_cnt[u])
        assert n == int(o_cnt[u]), "%s unit %d: count %d vs oracle %d (gpu %s, oracle %s, scores %s)" % (
            what, u, n, o_cnt[u], g_idx[u, :n].tolist(), o_idx[u, : o_cnt[u]].tolist(),
            np.asarray(o_scores[u])[:16].tolist())
        row = g_idx[u, :n].tolist()
        assert row == sorted(set(row)), "%s unit %d: not ascending/unique: %s" % (what, u, row)
        assert np.all(g_idx[u, n:] == -1), "%s unit %d: padding" % (what, u)
        gs, os_ = set(row), set(o_idx[u, : o_cnt[u]].tolist())
        if gs == os_:
            continue
        s = np.asarray(o_scores[u], dtype=np.float64)
        scale = np.max(np.abs(s[np.isfinite(s)]))
        for a in gs - os_:
            for b in os_ - gs:
                gap = abs(s[a] - s[b])
                assert gap <= rel * scale, "%s unit %d: gpu kept %d (%.9g), oracle kept %d (%.9g); gap %.3g" % (
                    what, u, a, s[a], b, s[b], gap / scale)
        swaps += len(gs - os_)
    return swaps
