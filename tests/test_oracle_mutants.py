"""Planted mistakes in the oracle must be caught by the pins.

Each case copies oracle.c, applies one plausible mistake (a dropped term, a
wrong sign, index or operand), builds it on the CPU and re-runs the pins
against it; at least one pin has to fail.  This shows the pins constrain every
step of the oracle, not only its happy path.
"""
import os

import pytest

import oracle
import oracle_pins as P

MUTANTS = {
    "sketch_divides_by_block_not_valid_rows": ("o[c] /= (double)(j1 - j0);", "o[c] /= (double)Bk;"),
    "score_drops_scale": ("return scale * acc;", "return acc;"),
    "decode_score_min_not_max": ("        if (s > best) best = s;\n      }\n    out[u] = best;",
                                 "        if (s < best || best == -INFINITY) best = s;\n      }\n    out[u] = best;"),
    "decode_score_wrong_head": ("row_dot(Q, dt, T, Hq, d, b, t, kvh * G + hh,", "row_dot(Q, dt, T, Hq, d, b, t, hh,"),
    "prefill_score_rows_from_zero": ("for (long t = i * Qt; t < tile_end(i, Qt, Lq); ++t)",
                                     "for (long t = 0; t < tile_end(i, Qt, Lq); ++t)"),
    "causal_blocks_drop_diagonal": ("return last / Bk + 1;", "return last / Bk;"),
    "tie_to_higher_index": ("return (a->b < c->b) ? -1 : (a->b > c->b);", "return (a->b > c->b) ? -1 : (a->b < c->b);"),
    "select_ascending_scores": ("if (a->s > c->s) return -1;\n  if (a->s < c->s) return 1;",
                                "if (a->s < c->s) return -1;\n  if (a->s > c->s) return 1;"),
    "local_block_not_forced": ("if (f1 > 0 && f1 < nv) sel[ns++] = f1;", ""),
    "forced_counted_in_budget": ("long take = budget[u] < nc ? budget[u] : nc;",
                                 "long take = budget[u] - 1 < nc ? budget[u] - 1 : nc; if (take < 0) take = 0;"),
    "forced_also_candidate": ("if (b == 0 || b == f1) continue;", "if (b == 0) continue;"),
    "attend_not_causal": ("if (j <= qpos) keys[nk++] = j;", "keys[nk++] = j;"),
    "attend_causal_off_by_one": ("if (j <= qpos) keys[nk++] = j;", "if (j < qpos) keys[nk++] = j;"),
    "attend_logits_use_v": ("acc += widen(Q, dt, qbase + c) * widen(K, dt, kb + c);",
                            "acc += widen(Q, dt, qbase + c) * widen(V, dt, kb + c);"),
    "attend_no_normalisation": ("o[c] = nk ? o[c] / den : 0.0;", "o[c] = nk ? o[c] : 0.0;"),
    "attend_wrong_group": ("long g = b * Hkv + h / G;\n    long unit", "long g = b * Hkv + h % Hkv;\n    long unit"),
    "mass_not_normalised": ("ar[j / Bk] += exp(logit[j] - m) / den;", "ar[j / Bk] += exp(logit[j] - m);"),
    "mass_not_causal": ("long nk = qpos + 1 < L ? qpos + 1 : L;", "long nk = L;"),
    "mass_drops_scale": ("logit[j] = scale * a;", "logit[j] = a;"),
    "delta_strict_threshold": ("if (scores[u * nb + b] >= thr) {", "if (scores[u * nb + b] > thr) {"),
    "delta_pseudo_max_sink_only": ("if (f1 > 0 && f1 < nv && scores[u * nb + f1] > pmax) pmax = scores[u * nb + f1];", ""),
    "delta_cap_ignored": ("long take = cap[u] < nc ? cap[u] : nc;", "long take = nc;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) >= 1, "mutation anchor not found: %s" % name
    mut = src.replace(old, new, 1)
    p_src = tmp_path / "oracle_mut.c"
    p_src.write_text(mut)
    lib_path = oracle.build(force=True, src=str(p_src), out=str(tmp_path / "liboracle_mut.so"))
    original = oracle._L()
    oracle.use(oracle.load(lib_path))
    caught = []
    try:
        for pin in P.ALL_PINS:
            try:
                pin()
            except (AssertionError, ValueError):
                caught.append(pin.__name__)
    finally:
        oracle.use(original)
    assert caught, "planted mistake %s passed every pin" % name
