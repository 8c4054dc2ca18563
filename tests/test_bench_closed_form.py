"""The benchmark's closed-form acceptance (analysis of its acceptance
microbenchmark inputs) against the oracle: the processed laws p and q come
from the oracle's proc, and sum_j prod_{t<=j} sum_v min(p_t, q_t) is then
taken per round; the empirical mean of the oracle's own acceptance over many
rounds falls within a few standard errors of it."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def test_closed_form_matches_oracle_laws(orc):
    import bench
    from speculative_decoding_rvq_gb300 import synth as S
    R, N, V, k, T = 64, 4, 64, 10, 0.9
    tgt, drf = S.gen_accept_inputs(R, N, V, 0.7, seed=3, block_rounds=64)
    got = bench.expected_accepted(torch.from_numpy(tgt), torch.from_numpy(drf), k, T)
    want = 0.0
    for r in range(R):
        prod = 1.0
        for t in range(N - 1):
            p, _ = orc.process(tgt[r, t], k, T)
            q, _ = orc.process(drf[r, t], k, T)
            prod *= float(np.minimum(p, q).astype(np.float64).sum())
            want += prod
    want /= R
    assert abs(got - want) < 1e-4, (got, want)


def test_closed_form_predicts_the_oracle_acceptance(orc):
    import bench
    from speculative_decoding_rvq_gb300 import synth as S
    R, N, V, k, T = 4096, 4, 64, 10, 0.9
    tgt, drf = S.gen_accept_inputs(R, N, V, 0.7, seed=5, block_rounds=1024)
    cf = bench.expected_accepted(torch.from_numpy(tgt), torch.from_numpy(drf), k, T)
    _, n_acc, _, _ = orc.accept_batch(tgt, drf, k, T, 9)
    emp = float(np.mean(n_acc))
    se = float(np.std(n_acc)) / np.sqrt(R)
    assert abs(emp - cf) < 4 * se + 1e-3, (emp, cf, se)


def test_acceptance_histogram_and_rows_touched(orc):
    """The benchmark's per-line histogram of accepted drafts, on the oracle's own
    acceptance: within sampling error of the closed form P(n = j) (sampling), equal
    to it (greedy, where acceptance is decided by argmaxes alone); the tail sums to
    the closed-form mean; rows touched are (N + n) rows of V floats per round."""
    import bench
    from speculative_decoding_rvq_gb300 import synth as S
    R, N, V, k = 4096, 4, 64, 10
    tgt, drf = S.gen_accept_inputs(R, N, V, 0.7, seed=5, block_rounds=1024)
    tt, dt = torch.from_numpy(tgt), torch.from_numpy(drf)
    for T in (0.9, 0.0):
        tail = bench.accepted_tail(tt, dt, k, T)
        assert len(tail) == N - 1 and all(1.0 >= a >= b >= 0.0 for a, b in zip(tail, tail[1:]))
        mean = bench.expected_accepted(tt, dt, k, T) if T > 0 else bench.expected_accepted_greedy(tt, dt)
        assert abs(sum(tail) - mean) < 1e-6  # the mean's products are float32, the tail's float64
        _, n_acc, _, _ = orc.accept_batch(tgt, drf, k, T, 9)
        n_acc = np.asarray(n_acc)
        ex = bench.accept_extras(torch.from_numpy(n_acc), N, V, 2.0, tail, 500.0)
        got, cf = np.array(ex["accept_hist"]), np.array(ex["closed_form_hist"])
        assert got.shape == cf.shape == (N,) and abs(got.sum() - 1) < 1e-3 and abs(cf.sum() - 1) < 1e-3
        if T > 0:
            se = np.sqrt(np.maximum(cf * (1 - cf), 1e-6) / R)
            assert np.all(np.abs(got - cf) < 4 * se + 1e-3), (got, cf)
        else:
            assert np.array_equal(got, cf), (got, cf)
        want = float(np.sum(N + n_acc.astype(np.int64))) * V * 4 / 2e-3 / 1e9
        assert abs(ex["rows_touched_GB_s"] - round(want, 1)) < 1e-9
        assert abs(ex["rows_touched_hbm_frac"] - round(want / 500.0, 4)) < 1e-9
