"""Pins of the oracle's RNG, logit processing, categorical draw and acceptance.

Each test checks the oracle against something other than itself: published
known-answer vectors, brute-force sorting, inverse-CDF counting on a uniform
grid, the page's greedy verifier behaviour, and closed forms of the
acceptance law (the sum-min identity of "Speculative Decoding, Beyond Text",
section 02, and the geometric expected-length formula of section 06).
"""
import json
import math
import os

import numpy as np
import pytest

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- Philox
def test_philox_known_answer_vectors(orc):
    kat = json.load(open(os.path.join(GOLD, "philox4x32_10_kat.json")))
    for v in kat["vectors"]:
        ctr = [int(h, 16) for h in v["ctr"]]
        key = [int(h, 16) for h in v["key"]]
        out = orc.philox4x32_10(ctr, key)
        assert [f"{int(w):08x}" for w in out] == v["out"]


def test_uniform_is_top24_bits_of_word0(orc):
    seed = 0x123456789ABCDEF0
    for (s, f, d, p) in [(0, 0, 0, 0), (3, 7, 11, 2), (65535, 999, 31, 1)]:
        w = orc.philox4x32_10([s, f, d, p], [seed & 0xFFFFFFFF, seed >> 32])
        u = orc.uniform(seed, s, f, d, p)
        assert u == (int(w[0]) >> 8) / 16777216.0
        assert 0.0 <= u < 1.0


def test_uniform_moments(orc):
    n = 200000
    ctr = np.zeros((n, 4), np.uint32)
    ctr[:, 0] = np.arange(n)
    ctr[:, 2] = 5
    ctr[:, 3] = 1
    u = orc.uniforms(7, ctr).astype(np.float64)
    assert abs(u.mean() - 0.5) < 5 * math.sqrt(1 / 12 / n)
    assert abs(u.var() - 1 / 12) < 0.002
    # purposes give different streams
    ctr2 = ctr.copy()
    ctr2[:, 3] = 2
    assert np.mean(orc.uniforms(7, ctr2) == u.astype(np.float32)) < 0.01


# ----------------------------------------------------- logit processing
def _brute_topk(z32, k):
    idx = np.lexsort((np.arange(z32.size), -z32.astype(np.float64)))  # by (z desc, index asc)
    return set(int(i) for i in idx[:k])


@pytest.mark.parametrize("V,k,T", [(256, 50, 0.9), (2048, 50, 0.9), (64, 64, 1.0), (100, 1, 0.5),
                                   (300, 299, 2.0), (4096, 50, 0.8)])
def test_process_topk_matches_brute_force(orc, V, k, T):
    rng = np.random.default_rng(V * 7 + k)
    for trial in range(5):
        logits = (rng.standard_normal(V) * 3).astype(np.float32)
        if trial == 1:  # heavy ties
            logits = np.round(logits).astype(np.float32)
        p, _ = orc.process(logits, k, T)
        z = (logits / np.float32(T)).astype(np.float32)
        keep = _brute_topk(z, min(k, V))
        assert set(np.flatnonzero(p > 0).tolist()) == keep
        # closed form: p_i / p_j = exp(z_i - z_j) on the kept set, sum = 1.  The
        # softmax is float64 with one rounding to float32 per probability, so
        # each p_i is within one float32 half-ulp (2^-24 relative) of the
        # exact value, plus float64 rounding far below that
        kept = sorted(keep)
        ref = np.exp(z[kept].astype(np.float64) - z[kept].max())
        ref /= ref.sum()
        np.testing.assert_allclose(p[kept].astype(np.float64), ref, rtol=2e-7, atol=1e-30)
        assert abs(float(p.astype(np.float64).sum()) - 1.0) < 1e-5


@pytest.mark.parametrize("k", [1, 2, 3, 7, 50, 63])
def test_process_uniform_closed_form(orc, k):
    """Equal logits: the first k indices are kept (ties by lowest index) and
    each gets exactly 1/k rounded once to float32 -- a dropped or doubled
    term of the normaliser, or a second rounding, shows here."""
    logits = np.full(64, 0.75, np.float32)
    p, mg = orc.process(logits, k, 0.9)
    assert np.flatnonzero(p > 0).tolist() == list(range(k))
    assert np.all(p[:k] == np.float32(1.0 / k))
    assert mg == 0.0 or k == 64


def test_process_ties_keep_lowest_index(orc):
    logits = np.array([1, 3, 3, 2, 3, 0], np.float32)
    p, _ = orc.process(logits, 2, 1.0)
    assert np.flatnonzero(p > 0).tolist() == [1, 2]
    assert p[1] == p[2]


def test_greedy_is_argmax_lowest_index(orc):
    logits = np.array([0.5, 2.0, -1.0, 2.0, 1.9], np.float32)
    p, mg = orc.process(logits, 3, 0.0)
    assert p.tolist() == [0, 1, 0, 0, 0]
    assert mg == 0.0  # exact tie -> zero decision margin


# ------------------------------------------------------ categorical draw
def test_sample_inverse_cdf_on_grid(orc):
    """Midpoint grid of u: counts per index equal w_i / S * n up to one grid cell per boundary."""
    w = np.array([0.0, 0.1, 0.0, 0.25, 0.05, 0.6], np.float32)
    n = 4096
    counts = np.zeros(w.size, int)
    for i in range(n):
        c, _ = orc.sample(w, (i + 0.5) / n)
        counts[c] += 1
    expected = w / w.sum() * n
    assert np.all(np.abs(counts - expected) <= 1.0)
    assert counts[0] == 0 and counts[2] == 0


def test_sample_edges(orc):
    w = np.array([0.0, 0.3, 0.7], np.float32)
    assert orc.sample(w, 0.0)[0] == 1
    assert orc.sample(w, np.float32(1.0 - 2 ** -24))[0] == 2
    assert orc.sample(np.zeros(4, np.float32), 0.3)[0] == -1
    one = np.array([0, 0, 1, 0], np.float32)
    assert all(orc.sample(one, u)[0] == 2 for u in (0.0, 0.5, 0.999))


# ----------------------------------------------------------- acceptance
def _onehot(ix, V):
    a = np.zeros((len(ix), V), np.float32)
    for r, i in enumerate(ix):
        a[r, i] = 1.0
    return a


def test_verify_greedy_scripted_cases(orc):
    g = json.load(open(os.path.join(GOLD, "verify_greedy_cases.json")))
    V = g["vocab"]
    for case in g["cases"]:
        d, t = case["draft"], case["target_argmax"]
        q = _onehot(d, V) if d else np.zeros((0, V), np.float32)
        p = _onehot(t, V)
        for u in (0.0, 0.37, 0.999):  # greedy decisions never depend on the uniforms
            na, em, _ = orc.accept_chain(q, d, p, [u] * max(len(d), 1), [u] * (len(d) + 1))
            assert em == case["emitted"]
            assert em[:na] == case["accepted"]
            rej = None if (na == len(d)) else na
            assert rej == case["rejected_at"]
    for case in g["errors"]:
        d, t = case["draft"], case["target_argmax"]
        with pytest.raises(ValueError):
            orc.accept_chain(_onehot(d, V), d, _onehot(t, V), [0.5] * len(d), [0.5] * (len(d) + 1))


def test_accept_probability_is_min_one_ratio(orc):
    """P(accept draft y) = min(1, p(y)/q(y)): count accepts over a midpoint grid of u."""
    V = 5
    q = np.array([[0.1, 0.4, 0.2, 0.3, 0.0]], np.float32)
    p = np.array([[0.3, 0.1, 0.2, 0.15, 0.25], [0.2, 0.2, 0.2, 0.2, 0.2]], np.float32)
    n = 2000
    for y in range(4):
        acc = 0
        for i in range(n):
            na, em, _ = orc.accept_chain(q, [y], p, [(i + 0.5) / n], [0.5, 0.5])
            acc += na
        ratio = min(1.0, float(p[0, y]) / float(q[0, y]))
        assert abs(acc / n - ratio) <= 1.0 / n + 1e-9


def test_residual_law_on_rejection(orc):
    """On rejection the emitted token follows norm(max(0, p - q)) (grid over the resample uniform)."""
    q = np.array([[0.5, 0.3, 0.2, 0.0]], np.float32)
    p = np.array([[0.1, 0.3, 0.2, 0.4]], np.float32)
    res = np.maximum(p[0] - q[0], 0)
    n = 4000
    counts = np.zeros(4, int)
    for i in range(n):
        na, em, _ = orc.accept_chain(q, [0], p, [0.9], [(i + 0.5) / n])  # 0.9 >= p/q = 0.2: reject
        assert na == 0 and len(em) == 1
        counts[em[0]] += 1
    assert np.all(np.abs(counts - res / res.sum() * n) <= 1.0)
    assert counts[0] == 0  # p <= q there


def test_sum_min_identity_and_single_position_law(orc):
    """Mean acceptance = sum_x min(p, q) = 1 - TV(p, q); emitted law = p (losslessness)."""
    rng = np.random.default_rng(3)
    V, R = 6, 60000
    for trial in range(3):
        pz = rng.standard_normal(V) * 1.5
        qz = rng.standard_normal(V) * 1.5
        p = (np.exp(pz) / np.exp(pz).sum()).astype(np.float32)
        q = (np.exp(qz) / np.exp(qz).sum()).astype(np.float32)
        tgt = np.broadcast_to(np.stack([p, p]), (R, 2, V)).copy()
        drf = np.broadcast_to(q[None, None], (R, 1, V)).copy()
        tok, na, dr, _ = orc.accept_batch(tgt, drf, V, 1.0, seed=11 + trial, mode=1)
        alpha = float(np.minimum(p.astype(np.float64), q).sum())
        tv = 0.5 * float(np.abs(p.astype(np.float64) - q).sum())
        assert abs(alpha - (1 - tv)) < 1e-6
        sig = math.sqrt(alpha * (1 - alpha) / R)
        assert abs(na.mean() - alpha) < 5 * sig
        # drafts follow q, and the first emitted token follows p exactly in law
        for law, sample in ((q, dr[:, 0]), (p, tok[:, 0])):
            cnt = np.bincount(sample, minlength=V)
            exp = law.astype(np.float64) * R
            chi2 = float(((cnt - exp) ** 2 / exp).sum())
            assert chi2 < 30.0, chi2  # df = 5; p(chi2 > 30) ~ 1.5e-5


def test_expected_tokens_per_round_closed_form(orc):
    """Constant per-position overlap alpha: E[emitted] = (1 - alpha^(g+1)) / (1 - alpha)."""
    V, R, N = 4, 50000, 5
    p = np.array([0.4, 0.3, 0.2, 0.1], np.float32)
    q = np.array([0.1, 0.2, 0.3, 0.4], np.float32)
    alpha = float(np.minimum(p, q).astype(np.float64).sum())
    tgt = np.broadcast_to(p, (R, N, V)).copy()
    drf = np.broadcast_to(q, (R, N - 1, V)).copy()
    tok, na, _, _ = orc.accept_batch(tgt, drf, V, 1.0, seed=5, mode=1)
    emitted = (tok >= 0).sum(1)
    assert np.all(emitted == na + 1)
    g = N - 1
    ev = (1 - alpha ** (g + 1)) / (1 - alpha)
    var = float(np.var(emitted))
    assert abs(emitted.mean() - ev) < 5 * math.sqrt(var / R)
    # P(n_acc >= j) = alpha^j
    for j in range(1, N):
        assert abs(np.mean(na >= j) - alpha ** j) < 5 * math.sqrt(alpha ** j * (1 - alpha ** j) / R) + 1e-9


def test_accept_batch_logits_mode_matches_explicit_processing(orc):
    rng = np.random.default_rng(9)
    R, N, V, k, T = 64, 4, 128, 10, 0.9
    tgt = (rng.standard_normal((R, N, V)) * 3).astype(np.float32)
    drf = (0.7 * tgt[:, :-1] + 0.71 * rng.standard_normal((R, N - 1, V)) * 3).astype(np.float32)
    tok, na, dr, _ = orc.accept_batch(tgt, drf, k, T, seed=1, mode=0)
    pt = np.stack([[orc.process(tgt[r, t], k, T)[0] for t in range(N)] for r in range(R)])
    qd = np.stack([[orc.process(drf[r, t], k, T)[0] for t in range(N - 1)] for r in range(R)])
    tok2, na2, dr2, _ = orc.accept_batch(pt, qd, k, T, seed=1, mode=1)
    assert np.array_equal(tok, tok2) and np.array_equal(na, na2) and np.array_equal(dr, dr2)
    assert np.all(qd[np.arange(R)[:, None], np.arange(N - 1)[None], dr] > 0)
