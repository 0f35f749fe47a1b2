"""The oracle reproduces the stored expected values in tests/golden/."""
import os

import numpy as np

import oracle
import synth

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "c1_decode.txt")
GOLD_TOK = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "c1_token_decode.txt")


def _read(path=GOLD):
    d = {}
    for line in open(path):
        if line.startswith("#"):
            continue
        parts = line.split()
        key = parts[0]
        if key in ("lse", "out"):
            d.setdefault(key, {})[int(parts[1])] = np.array([float(v) for v in parts[2:]])
        else:
            d[key] = np.array([float(v) for v in parts[1:]])
    return d


def test_c1_decode_golden():
    g = _read()
    wl = synth.WORKLOADS["c1"]
    x = synth.make_inputs(wl)
    assert np.nonzero(x.needle_mask[0])[0].tolist() == g["needles"].astype(int).tolist()
    idx, cnt, s, _ = oracle.decode_select(x.q, x.k, wl)
    assert idx[0, : cnt[0]].tolist() == g["selected"].astype(int).tolist()
    # the two needle blocks are among the selected ones
    assert set(g["needles"].astype(int)) <= set(g["selected"].astype(int))
    np.testing.assert_allclose(s[0], g["scores"], rtol=1e-14, atol=1e-15)
    rows = [(0, 0, h) for h in range(wl.Hq)]
    out, lse = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, rows, idx, cnt)
    for h in range(wl.Hq):
        np.testing.assert_allclose(out[h], g["out"][h], rtol=1e-13, atol=1e-14)
        assert abs(lse[h] - g["lse"][h][0]) < 1e-12


def test_c1_token_decode_golden():
    g = _read(GOLD_TOK)
    wl = synth.WORKLOADS["c1"].replace(L=512, k=32)
    x = synth.make_inputs(wl)
    P = oracle.token_mass_decode(x.q, x.k, wl.Hkv, wl.L, wl.scale)
    idx, cnt = oracle.token_select(P, wl.k)
    sel = idx[0, : cnt[0]]
    assert sel.tolist() == g["selected"].astype(int).tolist()
    np.testing.assert_allclose(P[0, sel], g["mass"], rtol=1e-13, atol=1e-17)
    assert abs(P[0].sum() - g["masssum"][0]) < 1e-13
    rows = [(0, 0, h) for h in range(wl.Hq)]
    out, lse = oracle.token_attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.scale, idx, cnt, rows)
    for h in range(wl.Hq):
        np.testing.assert_allclose(out[h], g["out"][h], rtol=1e-13, atol=1e-14)
        assert abs(lse[h] - g["lse"][h][0]) < 1e-12
