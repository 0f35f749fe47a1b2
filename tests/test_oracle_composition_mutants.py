"""Planted mistakes in the oracle's Python compositions (the head-collapsed token-level
support for decode and for per-query prefill) must be caught by the pins.

Each case replaces one composed function of ``oracle`` with a copy that makes one plausible
mistake (a wrong normaliser, an off-by-one query position or forced token, a selection not
repeated over the kv heads) and re-runs the token-level pins; at least one has to fail.
"""
import numpy as np
import pytest

import oracle
import oracle_pins as P

TOKEN_PINS = [P.pin_token_mass_matches_library_softmax, P.pin_token_mass_uniform_closed_form,
              P.pin_token_select_and_attend_match_library, P.pin_token_prefill_matches_library]

_orig = {name: getattr(oracle, name) for name in
         ("token_mass_decode", "token_select", "token_attend", "token_mass_prefill", "token_select_prefill",
          "token_attend_prefill")}


def _mass_decode_sum_not_mean(q, k, Hkv, L, scale):
    return _orig["token_mass_decode"](q, k, Hkv, L, scale) * q.shape[1]  # divided by Hq only


def _mass_decode_query_shifted(q, k, Hkv, L, scale):
    B, T, Hq, _ = q.shape
    units = [(g, 0) for g in range(B * Hkv)]
    m = oracle.mass(q, k, Hkv, L, L - T - 1, T, 1, scale, units)  # queries one position early
    return m.reshape(B, Hkv, L).sum(axis=1) / (Hq * T)


def _mass_decode_one_group(q, k, Hkv, L, scale):
    B, T, Hq, _ = q.shape
    m = oracle.mass(q, k, Hkv, L, L - T, T, 1, scale, [(g, 0) for g in range(B * Hkv)])
    return m.reshape(B, Hkv, L)[:, 0] / (Hq * T / Hkv)  # only kv head 0's query heads


def _select_newest_not_forced(P_, k, kmax=None):
    B, L = P_.shape
    return oracle.select(P_, L, 0, k, kmax or (k + 2))  # forced_hi = 0: only the sink is forced


def _attend_group0_selection(q, k, v, Hkv, L, scale, idx, cnt, rows):
    T = q.shape[1]
    idx_g = np.repeat(np.asarray(idx, dtype=np.int32)[:1], q.shape[0] * Hkv, axis=0)
    cnt_g = np.repeat(np.asarray(cnt, dtype=np.int32)[:1], q.shape[0] * Hkv)
    return oracle.attend(q, k, v, Hkv, L, L - T, 1, scale, rows, idx_g, cnt_g)


def _mass_prefill_by_group_heads(q, k, Hkv, L, scale):
    return _orig["token_mass_prefill"](q, k, Hkv, L, scale) * Hkv  # divided by G, not Hq


def _select_prefill_forced_previous(P_, k, kmax=None):
    B, Lq, L = P_.shape
    kmax = kmax or (k + 2)
    t = np.arange(Lq, dtype=np.int64)
    nvalid = np.tile(t + 1, B)
    idx, cnt = oracle.select(P_.reshape(B * Lq, L), nvalid, np.maximum(nvalid - 2, 0), k, kmax)
    return idx.reshape(B, Lq, kmax), cnt.reshape(B, Lq)


def _attend_prefill_shared_selection(q, k, v, Hkv, L, scale, idx, cnt, rows):
    B, Lq = q.shape[0], q.shape[1]
    kmax = idx.shape[-1]
    idx_g = np.repeat(np.asarray(idx, dtype=np.int32)[:, -1:], Lq, axis=1)  # every query uses the last one's
    cnt_g = np.repeat(np.asarray(cnt, dtype=np.int32)[:, -1:], Lq, axis=1)
    idx_g = np.repeat(idx_g, Hkv, axis=0).reshape(B * Hkv * Lq, kmax)
    cnt_g = np.repeat(cnt_g, Hkv, axis=0).reshape(B * Hkv * Lq)
    return oracle.attend(q, k, v, Hkv, L, 0, 1, scale, rows, idx_g, cnt_g, nsel=Lq, rows_per_sel=1)


MUTANTS = {
    "token_mass_sums_over_queries": ("token_mass_decode", _mass_decode_sum_not_mean),
    "token_mass_query_position_off_by_one": ("token_mass_decode", _mass_decode_query_shifted),
    "token_mass_one_kv_head": ("token_mass_decode", _mass_decode_one_group),
    "token_select_newest_not_forced": ("token_select", _select_newest_not_forced),
    "token_attend_selection_of_group_0": ("token_attend", _attend_group0_selection),
    "prefill_mass_over_group_heads": ("token_mass_prefill", _mass_prefill_by_group_heads),
    "prefill_select_forces_previous_token": ("token_select_prefill", _select_prefill_forced_previous),
    "prefill_attend_one_selection_for_all_queries": ("token_attend_prefill", _attend_prefill_shared_selection),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_composition_mutant_is_caught(name, monkeypatch):
    fn_name, bad = MUTANTS[name]
    monkeypatch.setattr(oracle, fn_name, bad)
    caught = []
    for pin in TOKEN_PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "planted mistake %r passed every token-level pin" % name


def test_token_pins_pass_on_the_oracle():
    for pin in TOKEN_PINS:
        pin()
