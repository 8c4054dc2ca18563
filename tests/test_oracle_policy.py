"""Pins of the oracle's adaptive window ("Speculative Decoding, Beyond Text",
runtime policies: size the draft window from measured acceptance by offset,
turn speculation off when acceptance collapses; "CodePredictor Speculative
Decoding", "Options": acceptance flattens past a few drafts).

Reading: each stream picks the window of its next frame from the drafts the
left-to-right test reached and accepted at each offset earlier in the call.
Offsets are kept while each has too few samples or an acceptance of at least
pct percent; window 1 runs rounds without drafts.

- The rule on hand-counted cases.
- pct = 0 reproduces the fixed-window decode exactly.
- Greedy decoding with the policy equals the greedy AR loop.
- Drafts that never match collapse the window to 1 after the first frame:
  later frames take G - 1 passes with no drafts.
- Drafts that always match keep the full window.
(The chi-square law test of test_oracle_model also runs with the policy on.)
"""
import dataclasses

import numpy as np
import pytest

from speculative_decoding_rvq_gb300 import synth as S


def _counts(pairs):
    reach, acc = np.zeros(9, np.int64), np.zeros(9, np.int64)
    for t, (r, a) in enumerate(pairs, start=1):
        reach[t], acc[t] = r, a
    return reach, acc


@pytest.mark.parametrize("N,pct,mn,pairs,want", [
    (4, 0, 8, [(100, 0), (50, 0), (10, 0)], 4),      # policy off
    (4, 30, 8, [(20, 10), (10, 2), (2, 2)], 2),      # offset 2 at 20 % < 30 %: window 2
    (4, 30, 8, [(20, 6), (10, 2), (2, 2)], 2),       # offset 1 at exactly 30 % is kept, offset 2 (10 samples, 20 %) is not
    (8, 50, 8, [(9, 4), (5, 0), (0, 0)], 1),         # offset 1 at 44 % with 9 samples: no drafts
    (8, 50, 8, [(7, 0), (0, 0)], 8),                 # too few samples anywhere: full window
    (3, 50, 4, [(4, 2), (2, 0)], 3),                 # offset 2 under-sampled: kept
    (6, 25, 4, [(40, 30), (30, 20), (20, 5), (5, 1)], 4),  # offsets 1-3 kept (75, 67, 25 %), offset 4 at 20 %
])
def test_policy_window_rule(orc, N, pct, mn, pairs, want):
    reach, acc = _counts(pairs)
    assert orc.Model.policy_window(N, pct, mn, reach, acc) == want


def _spec(G=8):
    return dataclasses.replace(S.TINY_FP32, n_layers=1, num_code_groups=G)


def test_policy_off_is_the_fixed_window(orc):
    spec = _spec()
    w = S.gen_weights(spec, seed=0)
    m = orc.Model(spec, w)
    x, c0 = S.gen_frames(spec, 2, 4, seed=1)
    a, sa, la = m.decode_frames(4, 50, 0.9, 1, x, c0, log_cap=500)
    b, sb, lb = m.decode_frames(4, 50, 0.9, 1, x, c0, log_cap=500, adapt_pct=0)
    assert np.array_equal(a, b) and sa == sb and np.array_equal(la, lb)


def test_greedy_with_policy_equals_greedy_ar(orc):
    spec = _spec()
    w = {**S.gen_weights(spec, seed=0), "draft_offset": S.gen_draft_offsets(spec, 3, seed=2, std=1.0)}
    m = orc.Model(spec, w)
    x, c0 = S.gen_frames(spec, 2, 6, seed=1)
    ar, _, _ = m.decode_frames(0, 50, 0.0, 1, x, c0)
    for N in (2, 4, 8):
        for pct in (30, 90):
            sp, st, _ = m.decode_frames(N, 50, 0.0, 1, x, c0, adapt_pct=pct, adapt_min=4)
            assert np.array_equal(sp, ar), (N, pct)
            assert st["committed"] == 12 * (spec.num_code_groups - 1)


def test_collapsed_acceptance_turns_drafting_off(orc):
    # huge offsets make every draft distribution a spike on an arbitrary code,
    # so greedy drafts almost never match the target's choice
    spec = _spec()
    G = spec.num_code_groups
    w = {**S.gen_weights(spec, seed=0), "draft_offset": S.gen_draft_offsets(spec, 7, seed=5, std=300.0)}
    m = orc.Model(spec, w)
    F = 6
    x, c0 = S.gen_frames(spec, 1, F, seed=3)
    codes, st, log = m.decode_frames(4, 50, 0.0, 1, x, c0, log_cap=1000, adapt_pct=50, adapt_min=4)
    first = log[log["frame"] == 0]
    assert np.all(first["n_d"][1:] > 0)  # frame 0: full window (no samples yet)
    assert np.sum(first["n_acc"]) < np.sum(first["n_d"]) // 2
    later = log[log["frame"] >= 1]
    assert np.all(later["n_d"] == 0)
    assert st["passes"] == len(first) + (F - 1) * (G - 1)  # one pass per code after frame 0


def test_full_acceptance_keeps_the_window(orc):
    # zero lm_heads: every target and draft law is the same top-k uniform, so
    # every draft is accepted (p / q = 1 > u)
    spec = _spec()
    w = S.gen_weights(spec, seed=0)
    w = {**w, "lm_head": np.zeros_like(w["lm_head"])}
    m = orc.Model(spec, w)
    x, c0 = S.gen_frames(spec, 1, 5, seed=3)
    _, st, log = m.decode_frames(4, 20, 0.9, 1, x, c0, log_cap=1000, adapt_pct=90, adapt_min=2)
    rounds = log[log["s"] >= 1]
    R = spec.num_code_groups - 1 - rounds["s"]
    assert np.array_equal(rounds["n_d"], np.minimum(3, R))
    assert st["accepted_by_offset"] == st["drafted_by_offset"]
