"""Pins for the fp64 oracle: each checks it against something other than itself.

Every pin raises AssertionError when the oracle is wrong.  They are collected as
tests in ``test_oracle_pins.py`` and re-run against deliberately broken builds
of the oracle in ``test_oracle_mutants.py`` (each broken build must fail at
least one pin).

Independent references used here:
  * torch's scaled_dot_product_attention (a library routine, CPU, float64),
    with a boolean mask that encodes causality and the selected blocks;
  * torch.softmax + reshape/sum for the per-block attention mass;
  * Python's sorted() for top-k, and hand-built ties / forced-block cases;
  * closed forms (constant-key blocks, arithmetic-progression keys);
  * invariants (mass rows sum to one, mass of non-causal blocks is zero,
    a block's sketch score is the mean of its dense logits).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import synth


def _rng(seed):
    return np.random.default_rng(seed)


def _sdpa(q, k, v, Hkv, allowed, scale):
    """Library attention. q [B,Tq,Hq,d], k/v [B,Hkv,L,d] float64; allowed [B,Hq,Tq,L] bool."""
    B, Tq, Hq, d = q.shape
    G = Hq // Hkv
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)  # B,Hq,Tq,d
    kt = torch.from_numpy(k).repeat_interleave(G, dim=1)
    vt = torch.from_numpy(v).repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(allowed),
                                                         scale=scale)
    return o.permute(0, 2, 1, 3).numpy()  # B,Tq,Hq,d


def _causal_allowed(B, Hq, Tq, L, pos0):
    t = np.arange(Tq)[:, None] + pos0
    j = np.arange(L)[None, :]
    a = j <= t
    return np.broadcast_to(a, (B, Hq, Tq, L)).copy()


def _all_rows(B, Tq, Hq):
    return np.array([(b, t, h) for b in range(B) for t in range(Tq) for h in range(Hq)], dtype=np.int64)


# ----------------------------------------------------------------------------- pins

def pin_dense_prefill_matches_library():
    """idx=None attention == SDPA with a causal mask (ragged L, GQA, several tiles)."""
    r = _rng(1)
    B, Hq, Hkv, d, L, Bk = 2, 6, 2, 16, 77, 8
    q = r.standard_normal((B, L, Hq, d))
    k = r.standard_normal((B, Hkv, L, d))
    v = r.standard_normal((B, Hkv, L, d))
    scale = 1 / math.sqrt(d)
    rows = _all_rows(B, L, Hq)
    out, _ = oracle.attend(q, k, v, Hkv, L, 0, Bk, scale, rows)
    ref = _sdpa(q, k, v, Hkv, _causal_allowed(B, Hq, L, L, 0), scale)
    got = out.reshape(B, L, Hq, d)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def pin_dense_decode_matches_library():
    """Decode rows at positions L-T..L-1 == SDPA with the matching causal mask."""
    r = _rng(2)
    B, T, Hq, Hkv, d, L, Bk = 2, 3, 4, 1, 8, 50, 4
    q = r.standard_normal((B, T, Hq, d))
    k = r.standard_normal((B, Hkv, L, d))
    v = r.standard_normal((B, Hkv, L, d))
    scale = 1 / math.sqrt(d)
    out, lse = oracle.attend(q, k, v, Hkv, L, L - T, Bk, scale, _all_rows(B, T, Hq))
    ref = _sdpa(q, k, v, Hkv, _causal_allowed(B, Hq, T, L, L - T), scale)
    np.testing.assert_allclose(out.reshape(B, T, Hq, d), ref, rtol=1e-12, atol=1e-12)
    # log-sum-exp of the row against a library logsumexp
    G = Hq // Hkv
    for n, (b, t, h) in enumerate(_all_rows(B, T, Hq)):
        logits = scale * (k[b, h // G, : L - T + t + 1] @ q[b, t, h])
        assert abs(lse[n] - torch.logsumexp(torch.from_numpy(logits), 0).item()) < 1e-12


def _block_mask_from_selection(idx, cnt, B, Hkv, G, Tq, L, Bk, pos0, Qt):
    """allowed[b, h, t, j] = block(j) selected for (g, t // Qt) and j <= pos0 + t."""
    Hq = Hkv * G
    nsel = idx.shape[0] // (B * Hkv)
    allowed = np.zeros((B, Hq, Tq, L), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            g = b * Hkv + h // G
            for t in range(Tq):
                u = g * nsel + min(t // Qt, nsel - 1)
                for blk in idx[u, : cnt[u]]:
                    allowed[b, h, t, blk * Bk: min((blk + 1) * Bk, L)] = True
                allowed[b, h, t, pos0 + t + 1:] = False
    return allowed


def pin_sparse_prefill_matches_masked_library():
    """Sparse attention over random tile selections == SDPA with the equivalent mask."""
    r = _rng(3)
    B, Hq, Hkv, d, L, Bk, Qt = 1, 4, 2, 8, 70, 8, 16
    G = Hq // Hkv
    q = r.standard_normal((B, L, Hq, d))
    k = r.standard_normal((B, Hkv, L, d))
    v = r.standard_normal((B, Hkv, L, d))
    scale = 1 / math.sqrt(d)
    nq = (L + Qt - 1) // Qt
    nb = (L + Bk - 1) // Bk
    kmax = nb
    idx = -np.ones((B * Hkv * nq, kmax), dtype=np.int32)
    cnt = np.zeros((B * Hkv * nq,), dtype=np.int32)
    for u in range(B * Hkv * nq):
        i = u % nq
        ncausal = min((i + 1) * Qt, L) - 1
        ncausal = ncausal // Bk + 1
        sel = sorted(set([0, ncausal - 1]) | set(r.choice(ncausal, size=min(2, ncausal), replace=False).tolist()))
        idx[u, : len(sel)] = sel
        cnt[u] = len(sel)
    out, _ = oracle.attend(q, k, v, Hkv, L, 0, Bk, scale, _all_rows(B, L, Hq), idx, cnt, nsel=nq,
                           rows_per_sel=Qt)
    allowed = _block_mask_from_selection(idx, cnt, B, Hkv, G, L, L, Bk, 0, Qt)
    ref = _sdpa(q, k, v, Hkv, allowed, scale)
    np.testing.assert_allclose(out.reshape(B, L, Hq, d), ref, rtol=1e-12, atol=1e-12)


def pin_sparse_decode_matches_masked_library():
    r = _rng(4)
    B, T, Hq, Hkv, d, L, Bk = 2, 2, 6, 3, 8, 61, 8
    G = Hq // Hkv
    q = r.standard_normal((B, T, Hq, d))
    k = r.standard_normal((B, Hkv, L, d))
    v = r.standard_normal((B, Hkv, L, d))
    scale = 1 / math.sqrt(d)
    nb = (L + Bk - 1) // Bk
    idx = -np.ones((B * Hkv, nb), dtype=np.int32)
    cnt = np.zeros((B * Hkv,), dtype=np.int32)
    for u in range(B * Hkv):
        sel = sorted({0, nb - 1, int(r.integers(1, nb - 1)), int(r.integers(1, nb - 1))})
        idx[u, : len(sel)] = sel
        cnt[u] = len(sel)
    out, _ = oracle.attend(q, k, v, Hkv, L, L - T, Bk, scale, _all_rows(B, T, Hq), idx, cnt)
    allowed = _block_mask_from_selection(idx, cnt, B, Hkv, G, T, L, Bk, L - T, 1 << 30)
    ref = _sdpa(q, k, v, Hkv, allowed, scale)
    np.testing.assert_allclose(out.reshape(B, T, Hq, d), ref, rtol=1e-12, atol=1e-12)


def pin_full_budget_equals_dense():
    """With a budget covering every candidate, the selected attention is dense attention."""
    wl = synth.WORKLOADS["c1"].replace(L=700, Bk=64, k=100)  # 11 blocks, ragged tail
    x = synth.make_inputs(wl)
    idx, cnt, _, _ = oracle.decode_select(x.q, x.k, wl, kmax=wl.nb)
    assert (cnt == wl.nb).all()
    rows = _all_rows(wl.B, wl.T, wl.Hq)
    o_sp, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, rows, idx, cnt)
    o_de, _ = oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, wl.L - wl.T, wl.Bk, wl.scale, rows)
    np.testing.assert_allclose(o_sp, o_de, rtol=0, atol=1e-13)


def pin_block_means_closed_form():
    """Constant rows per block give that constant; rows k[j] = j give the block's mid-index."""
    B, Hkv, L, Ls, d, Bk = 1, 2, 45, 48, 4, 8
    nb = (L + Bk - 1) // Bk
    k = np.zeros((B, Hkv, Ls, d))
    c = np.arange(B * Hkv * nb * d, dtype=np.float64).reshape(B * Hkv, nb, d) * 0.25 - 3
    for g in range(B * Hkv):
        for j in range(L):
            k[0, g, j] = c[g, j // Bk]
        k[0, g, L:] = 1e9  # rows past L must not be read
    np.testing.assert_array_equal(oracle.block_means(k, L, Bk), c)
    k2 = np.broadcast_to(np.arange(Ls, dtype=np.float64)[None, None, :, None], (B, Hkv, Ls, d)).copy()
    got = oracle.block_means(k2, L, Bk)
    for blk in range(nb):
        j0, j1 = blk * Bk, min((blk + 1) * Bk, L)
        assert np.all(got[:, blk] == (j0 + j1 - 1) / 2.0)


def pin_score_is_mean_of_block_logits():
    """Linearity: scale*q.mean(k_block) == mean_j(scale*q.k_j); then max over the group's rows."""
    r = _rng(5)
    B, T, Hq, Hkv, d, L, Bk = 2, 2, 6, 2, 16, 100, 16
    G = Hq // Hkv
    q = r.standard_normal((B, T, Hq, d))
    k = r.standard_normal((B, Hkv, L, d))
    scale = 0.3
    s = oracle.decode_scores(q, oracle.block_means(k, L, Bk), Hkv, scale)
    nb = (L + Bk - 1) // Bk
    for b in range(B):
        for kvh in range(Hkv):
            logits = np.stack([scale * (k[b, kvh] @ q[b, t, h]) for t in range(T)
                               for h in range(kvh * G, kvh * G + G)])  # rows x L
            ref = np.array([logits[:, blk * Bk: (blk + 1) * Bk].mean(axis=1).max() for blk in range(nb)])
            np.testing.assert_allclose(s[b * Hkv + kvh], ref, rtol=1e-12, atol=1e-12)
    # prefill scores: rows of tile i only, -inf beyond the causal range
    Lq, Qt = L, 32
    qp = r.standard_normal((B, Lq, Hq, d))
    units = [(g, i) for g in range(B * Hkv) for i in range((Lq + Qt - 1) // Qt)]
    sp = oracle.prefill_scores(qp, oracle.block_means(k, L, Bk), Hkv, Qt, Bk, scale, units)
    for n, (g, i) in enumerate(units):
        b, kvh = divmod(g, Hkv)
        t0, t1 = i * Qt, min((i + 1) * Qt, Lq)
        ncausal = (t1 - 1) // Bk + 1
        logits = np.stack([scale * (k[b, kvh] @ qp[b, t, h]) for t in range(t0, t1)
                           for h in range(kvh * G, kvh * G + G)])
        ref = np.array([logits[:, blk * Bk: (blk + 1) * Bk].mean(axis=1).max() for blk in range(ncausal)])
        np.testing.assert_allclose(sp[n, :ncausal], ref, rtol=1e-12, atol=1e-12)
        assert np.all(np.isneginf(sp[n, ncausal:]))


def _brute_select(scores, nvalid, forced_hi, budget):
    forced = {0, forced_hi} & set(range(nvalid))
    cands = [b for b in range(nvalid) if b not in forced]
    ranked = sorted(cands, key=lambda b: (-scores[b], b))
    return sorted(forced | set(ranked[: max(0, min(budget, len(cands)))]))


def pin_select_brute_force():
    r = _rng(6)
    for trial in range(300):
        nb = int(r.integers(1, 40))
        nvalid = int(r.integers(1, nb + 1))
        # coarse values to create many exact ties
        scores = r.integers(-3, 4, size=nb).astype(np.float64) * 0.5
        budget = int(r.integers(0, nb + 2))
        forced_hi = nvalid - 1
        idx, cnt = oracle.select(scores[None, :], nvalid, forced_hi, budget, nb + 2)
        ref = _brute_select(scores, nvalid, forced_hi, budget)
        assert cnt[0] == len(ref), (trial, cnt[0], ref)
        assert idx[0, : cnt[0]].tolist() == ref
        assert np.all(idx[0, cnt[0]:] == -1)


def pin_select_hand_cases():
    # ties: equal scores -> lower index wins
    s = np.array([0.0, 5.0, 5.0, 5.0, 1.0, 0.0])
    idx, cnt = oracle.select(s[None], 6, 5, 2, 8)
    assert idx[0, : cnt[0]].tolist() == [0, 1, 2, 5]
    # forced blocks are kept even with the lowest scores, and are not counted in the budget
    s = np.array([-9.0, 1.0, 2.0, 3.0, -9.0])
    idx, cnt = oracle.select(s[None], 5, 4, 1, 8)
    assert idx[0, : cnt[0]].tolist() == [0, 3, 4]
    # a single block: sink == local, kept once
    idx, cnt = oracle.select(np.array([[7.0]]), 1, 0, 3, 4)
    assert cnt[0] == 1 and idx[0].tolist() == [0, -1, -1, -1]
    # two blocks: both forced, no candidates
    idx, cnt = oracle.select(np.array([[1.0, 2.0]]), 2, 1, 5, 4)
    assert idx[0, : cnt[0]].tolist() == [0, 1]
    # budget 0: forced only
    idx, cnt = oracle.select(np.array([[1.0, 9.0, 9.0, 1.0]]), 4, 3, 0, 4)
    assert idx[0, : cnt[0]].tolist() == [0, 3]
    # blocks beyond nvalid are never chosen (non-causal)
    idx, cnt = oracle.select(np.array([[0.0, 1.0, 2.0, 99.0, 99.0]]), 3, 2, 5, 5)
    assert idx[0, : cnt[0]].tolist() == [0, 1, 2]


def pin_mass_matches_library_softmax():
    """Per-block mass == sum over rows of torch.softmax of causal logits, binned by block."""
    r = _rng(7)
    B, Hq, Hkv, d, L, Bk, Qt = 1, 4, 2, 8, 53, 8, 16
    G = Hq // Hkv
    q = r.standard_normal((B, L, Hq, d))
    k = r.standard_normal((B, Hkv, L, d))
    scale = 0.4
    nq, nb = (L + Qt - 1) // Qt, (L + Bk - 1) // Bk
    units = [(g, i) for g in range(B * Hkv) for i in range(nq)]
    m = oracle.mass(q, k, Hkv, L, 0, Qt, Bk, scale, units)
    pad = nb * Bk - L
    for n, (g, i) in enumerate(units):
        b, kvh = divmod(g, Hkv)
        ref = np.zeros(nb)
        t0, t1 = i * Qt, min((i + 1) * Qt, L)
        for t in range(t0, t1):
            for h in range(kvh * G, kvh * G + G):
                logits = torch.from_numpy(scale * (k[b, kvh] @ q[b, t, h]))
                logits[t + 1:] = -float("inf")
                p = torch.softmax(logits, 0).numpy()
                ref += np.concatenate([p, np.zeros(pad)]).reshape(nb, Bk).sum(axis=1)
        np.testing.assert_allclose(m[n], ref, rtol=1e-12, atol=1e-12)
        # invariants: total = rows * heads, zero past the causal range
        assert abs(m[n].sum() - (t1 - t0) * G) < 1e-9
        ncausal = (t1 - 1) // Bk + 1
        assert np.all(m[n, ncausal:] == 0.0)


def pin_decode_needles_selected(name="c1", **overrides):
    """Needle blocks (keys shifted along the group's query direction) are all selected."""
    wl = synth.WORKLOADS[name].replace(**overrides)
    x = synth.make_inputs(wl)
    idx, cnt, s, _ = oracle.decode_select(x.q, x.k, wl)
    for g in range(wl.B * wl.Hkv):
        needles = set(np.nonzero(x.needle_mask[g])[0].tolist())
        assert len(needles) == min(wl.needles, wl.nb - 2)
        sel = set(idx[g, : cnt[g]].tolist())
        assert needles <= sel, (g, sorted(needles - sel))
        assert cnt[g] == min(wl.k, wl.nb - 2) + 2


def pin_mass_topk_captures_plant():
    """Top-k by mass captures at least as much mass as any other set of the same size."""
    wl = synth.WORKLOADS["c4"].replace(L=2048, Hq=4, Hkv=1)
    x = synth.make_inputs(wl)
    units = [(0, i) for i in (3, 9, 15)]
    m = oracle.mass(x.q, x.k, wl.Hkv, wl.L, 0, wl.Qt, wl.Bk, wl.scale, units)
    idx, cnt, _, _ = oracle.prefill_select(x.q, x.k, wl.replace(frac_num=20), units, scores=m)
    r = _rng(8)
    captured_frac = []
    for n, (_, i) in enumerate(units):
        sel = idx[n, : cnt[n]]
        total = m[n].sum()
        captured = m[n, sel].sum() / total
        forced = {0, i}
        cands = [b for b in range(i + 1) if b not in forced]
        kk = cnt[n] - len(forced & set(range(i + 1)))
        for _ in range(200):
            alt = list(forced) + list(r.choice(cands, size=kk, replace=False))
            assert m[n, alt].sum() / total <= captured + 1e-12
        captured_frac.append(captured)
    # the planted shared component concentrates the mass: the same budget
    # captures more of it than on the same workload without the plant
    wl0 = wl.replace(plant_rank=0)
    x0 = synth.make_inputs(wl0)
    m0 = oracle.mass(x0.q, x0.k, wl0.Hkv, wl0.L, 0, wl0.Qt, wl0.Bk, wl0.scale, units)
    idx0, cnt0, _, _ = oracle.prefill_select(x0.q, x0.k, wl0.replace(frac_num=20), units, scores=m0)
    for n in range(len(units)):
        base = m0[n, idx0[n, : cnt0[n]]].sum() / m0[n].sum()
        assert captured_frac[n] > base, (units[n], captured_frac[n], base)


ALL_PINS = [
    pin_dense_prefill_matches_library,
    pin_dense_decode_matches_library,
    pin_sparse_prefill_matches_masked_library,
    pin_sparse_decode_matches_masked_library,
    pin_full_budget_equals_dense,
    pin_block_means_closed_form,
    pin_score_is_mean_of_block_logits,
    pin_select_brute_force,
    pin_select_hand_cases,
    pin_mass_matches_library_softmax,
    pin_decode_needles_selected,
    pin_mass_topk_captures_plant,
]


def _brute_select_delta(scores, nvalid, forced_hi, delta, cap):
    forced = {0, forced_hi} & set(range(nvalid))
    pmax = max(scores[b] for b in forced) if forced else -math.inf
    cands = [b for b in range(nvalid) if b not in forced and scores[b] >= pmax - delta]
    ranked = sorted(cands, key=lambda b: (-scores[b], b))
    return sorted(forced | set(ranked[: max(0, min(cap, len(cands)))]))


def pin_select_delta_brute_force():
    """Top-delta selection against a direct filter-then-sort on random small cases with ties."""
    r = _rng(9)
    for trial in range(300):
        nb = int(r.integers(1, 40))
        nvalid = int(r.integers(1, nb + 1))
        scores = r.integers(-4, 5, size=nb).astype(np.float64) * 0.5
        delta = float(r.choice([0.0, 0.5, 1.0, 2.5, 100.0]))
        cap = int(r.integers(0, nb + 2))
        idx, cnt = oracle.select_delta(scores[None, :], nvalid, nvalid - 1, delta, cap, nb + 2)
        ref = _brute_select_delta(scores, nvalid, nvalid - 1, delta, cap)
        assert idx[0, : cnt[0]].tolist() == ref, (trial, idx[0, : cnt[0]].tolist(), ref)
        assert np.all(idx[0, cnt[0]:] == -1)


def pin_select_delta_special_cases():
    s = np.array([2.0, 5.0, 1.9, 1.0, 3.0, 0.0])  # forced 0 and 5: pseudo-max 2.0
    # delta 0: only candidates at or above the pseudo-max
    idx, cnt = oracle.select_delta(s[None], 6, 5, 0.0, 10, 8)
    assert idx[0, : cnt[0]].tolist() == [0, 1, 4, 5]
    # delta 0.1 admits the 1.9 block; a cap of 2 keeps the two highest of the three
    idx, cnt = oracle.select_delta(s[None], 6, 5, 0.1, 10, 8)
    assert idx[0, : cnt[0]].tolist() == [0, 1, 2, 4, 5]
    idx, cnt = oracle.select_delta(s[None], 6, 5, 0.1, 2, 8)
    assert idx[0, : cnt[0]].tolist() == [0, 1, 4, 5]
    # a huge delta with cap k is the top-k selection
    r = _rng(10)
    sc = r.standard_normal((5, 30))
    for k in (0, 3, 10, 28, 40):
        a, ca = oracle.select_delta(sc, 30, 29, 1e9, k, 32)
        b, cb = oracle.select(sc, 30, 29, k, 32)
        assert np.array_equal(a, b) and np.array_equal(ca, cb)
    # the pseudo-max is the larger of the two forced scores (here the local block)
    s2 = np.array([0.0, 0.5, 0.9, 1.0])
    idx, cnt = oracle.select_delta(s2[None], 4, 3, 0.2, 10, 6)
    assert idx[0, : cnt[0]].tolist() == [0, 2, 3]

ALL_PINS += [pin_select_delta_brute_force, pin_select_delta_special_cases]


# ------------------------------------------------ head-collapsed token-level support

def pin_token_mass_matches_library_softmax():
    """Token mass == mean over all heads and decode rows of torch.softmax of the causal logits."""
    r = _rng(11)
    B, T, Hq, Hkv, d, L = 2, 3, 4, 2, 8, 37
    G = Hq // Hkv
    q = r.standard_normal((B, T, Hq, d))
    k = r.standard_normal((B, Hkv, L, d))
    scale = 0.45
    P = oracle.token_mass_decode(q, k, Hkv, L, scale)
    assert P.shape == (B, L)
    for b in range(B):
        ref = np.zeros(L)
        for t in range(T):
            for h in range(Hq):
                logits = torch.from_numpy(scale * (k[b, h // G] @ q[b, t, h]))
                logits[L - T + t + 1:] = -float("inf")
                ref += torch.softmax(logits, 0).numpy()
        np.testing.assert_allclose(P[b], ref / (Hq * T), rtol=1e-12, atol=1e-15)
        assert abs(P[b].sum() - 1.0) < 1e-12 and np.all(P[b] >= 0.0)


def pin_token_mass_uniform_closed_form():
    """Identical keys: each row is uniform over its causal keys, so P[b, j] = mean_t [j <= L-T+t] / (L-T+t+1)."""
    B, T, Hq, Hkv, d, L = 1, 4, 2, 1, 4, 19
    r = _rng(12)
    q = r.standard_normal((B, T, Hq, d))
    k = np.tile(r.standard_normal(d), (B, Hkv, L, 1))
    P = oracle.token_mass_decode(q, k, Hkv, L, 0.7)
    ref = np.zeros(L)
    for t in range(T):
        n = L - T + t + 1
        ref[:n] += 1.0 / n
    np.testing.assert_allclose(P[0], ref / T, rtol=1e-12, atol=1e-15)


def pin_token_select_and_attend_match_library():
    """Shared token support: the selected tokens are the top-k of P (brute force) plus tokens 0 and L-1,
    and attention over them equals SDPA with that token mask applied to every head."""
    r = _rng(13)
    B, T, Hq, Hkv, d, L, k = 2, 2, 4, 2, 8, 41, 7
    G = Hq // Hkv
    q = r.standard_normal((B, T, Hq, d))
    kk = r.standard_normal((B, Hkv, L, d))
    v = r.standard_normal((B, Hkv, L, d))
    scale = 0.5
    P = oracle.token_mass_decode(q, kk, Hkv, L, scale)
    idx, cnt = oracle.token_select(P, k)
    allowed = np.zeros((B, Hq, T, L), dtype=bool)
    for b in range(B):
        cands = sorted(range(1, L - 1), key=lambda j: (-P[b, j], j))[:k]
        ref = sorted({0, L - 1} | set(cands))
        assert idx[b, : cnt[b]].tolist() == ref
        for t in range(T):
            for j in ref:
                if j <= L - T + t:
                    allowed[b, :, t, j] = True
    rows = [(b, t, h) for b in range(B) for t in range(T) for h in range(Hq)]
    out, _ = oracle.token_attend(q, kk, v, Hkv, L, scale, idx, cnt, rows)
    ref_o = _sdpa(q, kk, v, Hkv, allowed, scale)
    for n, (b, t, h) in enumerate(rows):
        np.testing.assert_allclose(out[n], ref_o[b, t, h], rtol=1e-10, atol=1e-12)


ALL_PINS += [pin_token_mass_matches_library_softmax, pin_token_mass_uniform_closed_form,
             pin_token_select_and_attend_match_library]


def pin_token_prefill_matches_library():
    """Per-query support (b_sel = 1): P[b, t] = mean over heads of torch.softmax of the causal logits; the
    selection is the brute-force top-k of 1..t-1 plus tokens 0 and t; attention equals SDPA with each
    query's own token mask applied to every head."""
    r = _rng(14)
    B, Hq, Hkv, d, L, k = 2, 4, 2, 8, 23, 5
    G = Hq // Hkv
    q = r.standard_normal((B, L, Hq, d))
    kk = r.standard_normal((B, Hkv, L, d))
    v = r.standard_normal((B, Hkv, L, d))
    scale = 0.6
    P = oracle.token_mass_prefill(q, kk, Hkv, L, scale)
    assert P.shape == (B, L, L)
    allowed = np.zeros((B, Hq, L, L), dtype=bool)
    idx, cnt = oracle.token_select_prefill(P, k)
    for b in range(B):
        for t in range(L):
            ref = np.zeros(L)
            for h in range(Hq):
                logits = torch.from_numpy(scale * (kk[b, h // G] @ q[b, t, h]))
                logits[t + 1:] = -float("inf")
                ref += torch.softmax(logits, 0).numpy()
            np.testing.assert_allclose(P[b, t], ref / Hq, rtol=1e-12, atol=1e-15)
            assert abs(P[b, t].sum() - 1.0) < 1e-12 and np.all(P[b, t, t + 1:] == 0.0)
            cands = sorted(range(1, t), key=lambda j: (-P[b, t, j], j))[:k]
            want = sorted({0, t} | set(cands))
            assert idx[b, t, : cnt[b, t]].tolist() == want, (b, t)
            allowed[b, :, t, want] = True
    rows = [(b, t, h) for b in range(B) for t in range(L) for h in range(Hq)]
    out, _ = oracle.token_attend_prefill(q, kk, v, Hkv, L, scale, idx, cnt, rows)
    ref_o = _sdpa(q, kk, v, Hkv, allowed, scale)
    for n, (b, t, h) in enumerate(rows):
        np.testing.assert_allclose(out[n], ref_o[b, t, h], rtol=1e-10, atol=1e-12)


ALL_PINS += [pin_token_prefill_matches_library]
