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
