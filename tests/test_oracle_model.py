"""Pins of the oracle's decoder forward and frame loops.

- The forward is checked against a float64 torch restatement built from
  library routines (``F.rms_norm``, ``F.scaled_dot_product_attention`` with a
  causal mask, ``F.silu``) and a complex-multiplication form of the rotary
  embedding, so a dropped term, a sign or a transposed operand fails.
- Cached block passes equal no-cache full-prefix recomputation ("Speculative
  Decoding, Beyond Text", section 13, ladder steps 2-3).
- Greedy speculative decoding equals the greedy autoregressive loop exactly
  (section 02 "Exact greedy decoding"; section 08 step 4), for every window
  2..8 and odd/even code-group counts.
- The speculative output law equals the autoregressive law ("CodePredictor
  Speculative Decoding", "How a round works": committed codes are distributed
  exactly as the autoregressive loop) by a chi-square test on a tiny vocab.
"""
import dataclasses
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

from speculative_decoding_rvq_gb300 import synth as S


def _tiny(G=5, V=6, H=32, L=2, nq=4, nkv=2, d=8, F=48):
    return S.ModelSpec(hidden=H, n_layers=L, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, ffn=F,
                       vocab=V, num_code_groups=G, dtype=S.DTYPE_F32)


def _torch_forward(spec, w, rows: np.ndarray, positions: np.ndarray) -> np.ndarray:
    """Full causal pass over ``rows`` at consecutive positions 0..n-1, float64, library ops."""
    H, d, nq, nkv = spec.hidden, spec.head_dim, spec.n_q_heads, spec.n_kv_heads
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    h = t(rows).clone()
    n = h.shape[0]
    pos = torch.from_numpy(positions.astype(np.float64))
    inv = 1.0 / (spec.rope_theta ** (torch.arange(0, d, 2, dtype=torch.float64) / d))
    ang = pos[:, None] * inv[None, :]                        # [n, d/2]
    rot = torch.polar(torch.ones_like(ang), ang)             # e^{i ang}

    def rope(x):  # x [n, heads, d]; rotate-half pairs (i, i + d/2) as one complex number
        c = torch.complex(x[..., : d // 2], x[..., d // 2:]) * rot[:, None, :]
        return torch.cat([c.real, c.imag], dim=-1)

    for lw in w["layers"]:
        a = Fn.rms_norm(h, (H,), weight=t(lw["attn_norm"]), eps=spec.rms_eps)
        q = (a @ t(lw["wq"]).T).view(n, nq, d)
        k = (a @ t(lw["wk"]).T).view(n, nkv, d)
        v = (a @ t(lw["wv"]).T).view(n, nkv, d)
        q, k = rope(q), rope(k)
        k = k.repeat_interleave(nq // nkv, dim=1)
        v = v.repeat_interleave(nq // nkv, dim=1)
        o = Fn.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
                                            is_causal=True)
        h = h + o.transpose(0, 1).reshape(n, nq * d) @ t(lw["wo"]).T
        b = Fn.rms_norm(h, (H,), weight=t(lw["ffn_norm"]), eps=spec.rms_eps)
        h = h + (Fn.silu(b @ t(lw["w_gate"]).T) * (b @ t(lw["w_up"]).T)) @ t(lw["w_down"]).T
    return Fn.rms_norm(h, (H,), weight=t(w["final_norm"]), eps=spec.rms_eps).numpy()


def _rows(model, x, codes, P):
    return np.stack([model.input_row(x, j, codes[j - 1] if j > 0 else 0) for j in range(P)])


@pytest.mark.parametrize("spec", [_tiny(), _tiny(nq=4, nkv=4), dataclasses.replace(S.TINY_FP32, n_layers=1)])
def test_forward_matches_torch_float64(orc, spec):
    w = S.gen_weights(spec, seed=3, std=0.3 if spec.hidden < 64 else 0.02)
    m = orc.Model(spec, w)
    x, c0 = S.gen_frames(spec, 1, 1, seed=4)
    rng = np.random.default_rng(0)
    P = spec.num_code_groups
    codes = rng.integers(0, spec.vocab, P)
    rows = _rows(m, x[0, 0], codes, P)
    ref = _torch_forward(spec, w, rows, np.arange(P))
    out = m.forward(m.new_kv(), rows, np.arange(P))
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-10)


def test_cached_blocks_equal_nocache_recompute(orc):
    spec = _tiny(G=8)
    w = S.gen_weights(spec, seed=5, std=0.3)
    m = orc.Model(spec, w)
    x, _ = S.gen_frames(spec, 1, 1, seed=6)
    codes = np.random.default_rng(1).integers(0, spec.vocab, 8)
    rows = _rows(m, x[0, 0], codes, 8)
    # no-cache: every position recomputed from scratch with its full prefix
    full = np.stack([m.forward(m.new_kv(), rows[: p + 1], np.arange(p + 1))[-1] for p in range(8)])
    for chunks in ([2, 3, 3], [2, 1, 1, 1, 1, 1, 1], [4, 4], [8]):
        kv = m.new_kv()
        outs, p0 = [], 0
        for c in chunks:
            outs.append(m.forward(kv, rows[p0:p0 + c], np.arange(p0, p0 + c)))
            p0 += c
        np.testing.assert_allclose(np.concatenate(outs), full, rtol=1e-12, atol=1e-12)


def test_stale_kv_entries_are_never_read(orc):
    """A rejected suffix left in the cache must not change later rows (KV transaction, section 07)."""
    spec = _tiny(G=6)
    w = S.gen_weights(spec, seed=7, std=0.3)
    m = orc.Model(spec, w)
    x, _ = S.gen_frames(spec, 1, 1, seed=8)
    codes = [1, 2, 3, 4, 5]
    rows = _rows(m, x[0, 0], codes, 6)
    kv = m.new_kv()
    m.forward(kv, rows[:2], [0, 1])
    junk = rows[2:5] * 7.0 + 1.0
    m.forward(kv, junk, [2, 3, 4])         # speculative rows later rejected
    a = m.forward(kv, rows[2:4], [2, 3])   # overwrite from the committed length
    b = m.forward(m.new_kv(), rows[:4], [0, 1, 2, 3])[2:]
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_teacher_logits_are_head_j_at_position_j(orc):
    spec = _tiny(G=6)
    w = S.gen_weights(spec, seed=9, std=0.3)
    m = orc.Model(spec, w)
    x, _ = S.gen_frames(spec, 1, 1, seed=10)
    codes = [3, 1, 4, 1, 5]
    lg, dl = m.teacher_logits(x[0, 0], codes, 6, n_draft=3)
    hn = _torch_forward(spec, w, _rows(m, x[0, 0], codes, 6), np.arange(6))
    heads = w["lm_head"].astype(np.float64)
    for j in range(1, 6):
        np.testing.assert_allclose(lg[j - 1], (heads[j - 1] @ hn[j]).astype(np.float32), rtol=1e-6, atol=1e-7)
        for t in range(1, 4):
            ref = heads[j + t - 1] @ hn[j] if j + t <= 5 else np.zeros(spec.vocab)
            np.testing.assert_allclose(dl[j - 1, t - 1], ref.astype(np.float32), rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("G", [2, 3, 4, 7, 8])
def test_greedy_speculative_equals_greedy_ar(orc, G):
    spec = dataclasses.replace(S.TINY_FP32, num_code_groups=G, n_layers=1)
    w = S.gen_weights(spec, seed=0)
    m = orc.Model(spec, w)
    x, c0 = S.gen_frames(spec, 2, 3, seed=1)
    ar, st_ar, _ = m.decode_frames(0, 50, 0.0, 1, x, c0)
    assert st_ar["passes"] == 6 * (G - 1)
    for N in range(2, 9):
        sp, st, log = m.decode_frames(N, 50, 0.0, 1, x, c0, log_cap=1000)
        assert np.array_equal(ar, sp), N
        assert st["committed"] == 6 * (G - 1)
        # every round commits between 1 and N codes, and the KV length is s' + 1
        rounds = log[log["n_d"] > 0]
        ne = rounds["s_new"] - rounds["s"]
        assert np.all((ne >= 1) & (ne <= N))
        assert np.all(rounds["n_acc"] <= rounds["n_d"])


@pytest.mark.parametrize("K,adapt", [(0, 0), (2, 0), (2, 60)])
def test_speculative_law_equals_autoregressive_law(orc, K, adapt):
    """Exact law of (c_1, c_2, c_3) under AR by enumeration vs speculative frequencies (chi-square).

    K = 2 adds position-aware draft offsets: they change only the drafts, so
    the law is the same ("RVQ Position Aware Speculative Decoding for On
    Device TTS", section 3.2).  adapt = 60 lets each frame's window follow the
    acceptance of the frames before it, which leaves every frame's law exact."""
    spec = S.ModelSpec(hidden=16, n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=8, ffn=32, vocab=4,
                       num_code_groups=4, dtype=S.DTYPE_F32)
    w = S.gen_weights(spec, seed=21, std=0.5)
    if K:
        w = {**w, "draft_offset": S.gen_draft_offsets(spec, K, seed=5, std=1.0)}
    m = orc.Model(spec, w)
    x, c0 = S.gen_frames(spec, 1, 1, seed=22)
    k, T = 3, 0.9
    law = {}
    for tup in itertools.product(range(4), repeat=3):
        codes = [int(c0[0, 0]), *tup[:2]]
        lg, _ = m.teacher_logits(x[0, 0], codes, 4)
        pr = 1.0
        for j in range(3):
            pj, _ = orc.process(lg[j], k, T)
            pr *= float(pj[tup[j]])
        law[tup] = pr
    assert abs(sum(law.values()) - 1.0) < 1e-5
    F = 40000
    xs = np.broadcast_to(x, (F, 1, spec.hidden)).copy()
    cs = np.broadcast_to(c0, (F, 1)).copy()
    for N in (0, 2, 3, 4):
        codes, st, _ = m.decode_frames(N, k, T, 77, xs, cs, adapt_pct=adapt, adapt_min=8)
        cnt = {}
        for row in codes[:, 0, 1:]:
            cnt[tuple(int(v) for v in row)] = cnt.get(tuple(int(v) for v in row), 0) + 1
        chi2, df = 0.0, -1
        for tup, pr in law.items():
            o = cnt.get(tup, 0)
            if pr == 0.0:
                assert o == 0, (N, tup)  # outside top-k support: never emitted
                continue
            e = pr * F
            chi2 += (o - e) ** 2 / e
            df += 1
        # chi-square upper tail p < 1e-4 bound via Wilson-Hilferty
        z = ((chi2 / df) ** (1 / 3) - (1 - 2 / (9 * df))) / math.sqrt(2 / (9 * df))
        assert z < 3.7, (N, chi2, df)


def test_sampled_speculative_differs_from_ar_but_commits_all_codes(orc):
    spec = dataclasses.replace(S.TINY_FP32, n_layers=1)
    w = S.gen_weights(spec, seed=0)
    m = orc.Model(spec, w)
    x, c0 = S.gen_frames(spec, 1, 6, seed=1)
    ar, _, _ = m.decode_frames(0, 50, 0.9, 1, x, c0)
    sp, st, log = m.decode_frames(3, 50, 0.9, 1, x, c0, log_cap=500)
    assert np.all((sp >= 0) & (sp < spec.vocab))
    assert st["committed"] == 6 * (spec.num_code_groups - 1)
    assert st["passes"] == 6 + st["rounds"]
    assert not np.array_equal(ar, sp)  # different random draws, same law (previous test)


def test_drafts_come_from_later_heads_on_current_hidden(orc):
    """Greedy drafts of each round = argmax head_{s+t}(h_s) with h_s from teacher forcing on the
    committed codes ("CodePredictor Speculative Decoding", "Why the draft is free")."""
    spec = dataclasses.replace(S.TINY_FP32, n_layers=1)
    w = S.gen_weights(spec, seed=0)
    m = orc.Model(spec, w)
    x, c0 = S.gen_frames(spec, 1, 4, seed=1)
    G = spec.num_code_groups
    for N in (2, 4, 8):
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
