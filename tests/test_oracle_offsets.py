"""Pins of the oracle's position-aware draft offsets ("RVQ Position Aware
Speculative Decoding for On Device TTS", section 2.2 and Figure 3).

The draft of lookahead t reads head_{s+t} on h_s + b_t, where h_s is the
hidden state the heads read at depth s and b_1..b_K are shared by every depth.
The verifier heads never see an offset, so the committed law stays the
autoregressive one whatever b is (section 3.2).

- An offset that moves h_j exactly onto h_{j+t} turns the lookahead-t draft
  at position j into the target logits of position j+t.  This fixes the head
  index, the offset index, the sign, and that b is added after the final
  norm (a wrong choice of any of them breaks the equality).
- Teacher-forced draft logits equal a float64 torch restatement built on the
  library forward of test_oracle_model.
- Greedy speculation with offsets equals greedy AR exactly, while the drafts
  themselves do change (so the equality is not vacuous).
- The drafts of every decode round are the argmax of the teacher-forced draft
  logits with offsets (decode and teacher paths agree).
"""
import dataclasses

import numpy as np

from speculative_decoding_rvq_gb300 import synth as S
from test_oracle_model import _rows, _tiny, _torch_forward


def test_offset_onto_later_hidden_turns_draft_into_target(orc):
    spec = _tiny(G=8)
    w = S.gen_weights(spec, seed=9, std=0.3)
    x, _ = S.gen_frames(spec, 1, 1, seed=10)
    codes = [3, 1, 4, 1, 5, 2, 0]
    P = 8
    hn = _torch_forward(spec, w, _rows(orc.Model(spec, w), x[0, 0], codes, P), np.arange(P))
    j, K = 2, 3
    b = np.stack([hn[j + t] - hn[j] for t in range(1, K + 1)]).astype(np.float32)
    m = orc.Model(spec, {**w, "draft_offset": b})
    assert m.K == K
    lg, dl = m.teacher_logits(x[0, 0], codes, P, n_draft=5)
    for t in range(1, K + 1):
        np.testing.assert_allclose(dl[j - 1, t - 1], lg[j + t - 1], rtol=1e-5, atol=1e-5)
    # lookahead beyond K has no offset: head_{j+t} on h_j itself
    heads = w["lm_head"].astype(np.float64)
    for t in (4, 5):
        np.testing.assert_allclose(dl[j - 1, t - 1], (heads[j + t - 1] @ hn[j]).astype(np.float32),
                                   rtol=1e-6, atol=1e-6)
    # the target logits never see an offset
    np.testing.assert_allclose(lg, orc.Model(spec, w).teacher_logits(x[0, 0], codes, P)[0], rtol=0, atol=0)


def test_teacher_draft_logits_with_offsets_match_torch(orc):
    spec = _tiny(G=6)
    w = S.gen_weights(spec, seed=11, std=0.3)
    b = S.gen_draft_offsets(spec, 2, seed=4, std=0.5)
    m = orc.Model(spec, {**w, "draft_offset": b})
    x, _ = S.gen_frames(spec, 1, 1, seed=12)
    codes = [2, 5, 0, 3, 1]
    lg, dl = m.teacher_logits(x[0, 0], codes, 6, n_draft=3)
    hn = _torch_forward(spec, w, _rows(m, x[0, 0], codes, 6), np.arange(6))
    heads = w["lm_head"].astype(np.float64)
    for j in range(1, 6):
        for t in range(1, 4):
            h = hn[j] + (b[t - 1].astype(np.float64) if t <= 2 else 0.0)
            ref = heads[j + t - 1] @ h if j + t <= 5 else np.zeros(spec.vocab)
            np.testing.assert_allclose(dl[j - 1, t - 1], ref.astype(np.float32), rtol=1e-6, atol=1e-6)
        np.testing.assert_allclose(m.draft_logits(min(j + 1, 5), 1, hn[j]),
                                   (heads[min(j + 1, 5) - 1] @ (hn[j] + b[0])).astype(np.float32),
                                   rtol=1e-6, atol=1e-6)


def test_greedy_speculation_with_offsets_equals_greedy_ar(orc):
    for G in (4, 8):
        spec = dataclasses.replace(S.TINY_FP32, num_code_groups=G, n_layers=1)
        w = S.gen_weights(spec, seed=0)
        x, c0 = S.gen_frames(spec, 2, 3, seed=1)
        ar, _, _ = orc.Model(spec, w).decode_frames(0, 50, 0.0, 1, x, c0)
        for K in (3, 7):
            m = orc.Model(spec, {**w, "draft_offset": S.gen_draft_offsets(spec, K, seed=2, std=1.0)})
            plain = orc.Model(spec, w)
            changed = 0
            for N in range(2, 9):
                sp, st, log = m.decode_frames(N, 50, 0.0, 1, x, c0, log_cap=1000)
                assert np.array_equal(ar, sp), (G, K, N)
                assert st["committed"] == 6 * (G - 1)
                _, _, log0 = plain.decode_frames(N, 50, 0.0, 1, x, c0, log_cap=1000)
                r, r0 = log[log["n_d"] > 0], log0[log0["n_d"] > 0]
                n = min(len(r), len(r0))
                changed += int(np.sum(r["drafts"][:n] != r0["drafts"][:n]))
            assert changed > 0, (G, K)


def test_decode_drafts_are_argmax_of_offset_draft_logits(orc):
    spec = dataclasses.replace(S.TINY_FP32, n_layers=1)
    w = {**S.gen_weights(spec, seed=0), "draft_offset": S.gen_draft_offsets(spec, 2, seed=3, std=1.0)}
    m = orc.Model(spec, w)
    x, c0 = S.gen_frames(spec, 1, 3, seed=1)
    G = spec.num_code_groups
    for N in (3, 5):
        codes, _, log = m.decode_frames(N, 50, 0.0, 1, x, c0, log_cap=500)
        checked = 0
        for rec in log[log["n_d"] > 0]:
            f = int(rec["frame"])
            _, dl = m.teacher_logits(x[f, 0], codes[f, 0, : G - 1], G, n_draft=N - 1)
            s = int(rec["s"])
            for t in range(1, int(rec["n_d"]) + 1):
                assert int(rec["drafts"][t - 1]) == int(np.argmax(dl[s - 1, t - 1])), (N, s, t)
                checked += 1
        assert checked > 0
