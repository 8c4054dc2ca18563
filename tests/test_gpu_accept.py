"""GPU acceptance kernels vs the CPU oracle (acceptance-microbenchmark workload:
target logits N(0, 3^2), draft = rho * target + sqrt(1 - rho^2) * N(0, 3^2),
top-k 50, temperature 0.9, Philox uniforms)."""
import numpy as np
import pytest

from gpu_common import require_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def softmax_tol(k, V):
    """Decision margin below which a code may differ between the kernels and
    the oracle in logit mode.  The kernels form each kept probability in
    float32 (an exponential within 2 ulp, a sequential float32 sum of the kk
    kept terms, one division): at most (kk + 4) * 2^-23 relative from the
    oracle's correctly rounded float64 softmax.  An acceptance ratio p/q
    carries two such errors and one rounding, a prefix sum of a draw at most
    one; three times the bound covers both."""
    kk = min(k, V)
    return 3.0 * (kk + 4) * 2.0 ** -23


def draw_margin(tgt_r, drf_r, k, T, seed, r):
    """Smallest margin of round r's float32 draws and acceptance tests (not
    of its top-k sets, which both sides form from the same float32 z): the
    oracle's steps replayed one by one through its public functions."""
    from oracle import oracle as O
    N = tgt_r.shape[0]
    q = np.stack([O.process(drf_r[t], k, T)[0] for t in range(N - 1)])
    p = np.stack([O.process(tgt_r[t], k, T)[0] for t in range(N)])
    mg = np.inf
    dr = []
    for t in range(N - 1):
        c, m = O.sample(q[t], O.uniform(seed, int(r), 0, t + 1, O.ORC_DRAFT))
        dr.append(c)
        mg = min(mg, m)
    ua = [O.uniform(seed, int(r), 0, t + 1, O.ORC_ACCEPT) for t in range(N - 1)]
    ut = [O.uniform(seed, int(r), 0, t + 1, O.ORC_TARGET) for t in range(N)]
    _, _, m = O.accept_chain(q, dr, p, ua, ut)
    return min(mg, m)


def _run_gpu(tgt, drf, k, T, seed, mode):
    from speculative_decoding_rvq_gb300 import binding
    t = torch.from_numpy(tgt).cuda()
    d = torch.from_numpy(drf).cuda()
    tok, na, dr = binding.accept_batch(t, d, k, T, seed, mode)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), na.cpu().numpy(), dr.cpu().numpy()


@pytest.mark.parametrize("N", [2, 4, 8])
@pytest.mark.parametrize("rho", [0.3, 0.95])
def test_probability_mode_bit_exact(orc, N, rho):
    """Identical fp32 probabilities and Philox streams -> identical codes, accept counts, drafts."""
    from speculative_decoding_rvq_gb300 import synth as S
    R, V = 512, 2048
    tgt, drf = S.gen_accept_inputs(R, N, V, rho, seed=3)
    pt = np.stack([[orc.process(tgt[r, t], 50, 0.9)[0] for t in range(N)] for r in range(R)])
    qd = np.stack([[orc.process(drf[r, t], 50, 0.9)[0] for t in range(N - 1)] for r in range(R)])
    o_tok, o_na, o_dr, _ = orc.accept_batch(pt, qd, 50, 0.9, seed=7, mode=1)
    g_tok, g_na, g_dr = _run_gpu(pt, qd, 50, 0.9, 7, 1)
    assert np.array_equal(g_dr, o_dr)
    assert np.array_equal(g_na, o_na)
    assert np.array_equal(g_tok, o_tok)


@pytest.mark.parametrize("N,k,T", [(4, 50, 0.9), (8, 50, 0.9), (2, 2048, 1.3), (4, 1, 0.9), (4, 7, 0.05),
                                   (3, 50, 0.0)])
def test_logit_mode_matches_oracle(orc, N, k, T):
    from speculative_decoding_rvq_gb300 import synth as S
    R, V = 512, 2048
    tgt, drf = S.gen_accept_inputs(R, N, V, 0.7, seed=11)
    o_tok, o_na, o_dr, o_mg = orc.accept_batch(tgt, drf, k, T, seed=5, mode=0)
    g_tok, g_na, g_dr = _run_gpu(tgt, drf, k, T, 5, 0)
    bad = np.flatnonzero((g_tok != o_tok).any(1) | (g_na != o_na) | (g_dr != o_dr).any(1))
    # the kernels' float32 softmax differs from the oracle's float64 one by a
    # few ulp: only a decision closer than that bound may flip, and rarely
    if T > 0:
        tol = softmax_tol(k, V)
        margins = [draw_margin(tgt[r], drf[r], k, T, 5, r) for r in bad]
        assert all(m < tol for m in margins), [(int(r), float(m)) for r, m in zip(bad[:5], margins[:5])]
    assert len(bad) <= 2


def test_ragged_vocab_and_ties(orc):
    """V not a multiple of 32, heavy ties at the top-k boundary."""
    R, N, V = 256, 4, 250
    rng = np.random.default_rng(2)
    tgt = np.round(rng.standard_normal((R, N, V)) * 2).astype(np.float32)
    drf = np.round(rng.standard_normal((R, N - 1, V)) * 2).astype(np.float32)
    o = orc.accept_batch(tgt, drf, 17, 1.0, seed=9, mode=0)
    g = _run_gpu(tgt, drf, 17, 1.0, 9, 0)
    # top-k sets are exact (ties by lowest index); probabilities may differ by
    # the float32 softmax bound, so only a near-tied draw may flip
    bad = np.flatnonzero((g[0] != o[0]).any(1) | (g[1] != o[1]) | (g[2] != o[2]).any(1))
    tol = softmax_tol(17, V)
    assert all(draw_margin(tgt[r], drf[r], 17, 1.0, 9, r) < tol for r in bad), bad
    assert len(bad) <= 1


def test_full_size_invariants_and_sampled_parity(orc):
    """65536 rounds, V 2048, N 4: invariants on every round, oracle on a sample of rounds."""
    from speculative_decoding_rvq_gb300 import synth as S
    R, N, V = 65536, 4, 2048
    tgt, drf = S.gen_accept_inputs(R, N, V, 0.95, seed=1)
    g_tok, g_na, g_dr = _run_gpu(tgt, drf, 50, 0.9, 1, 0)
    assert np.all((g_na >= 0) & (g_na <= N - 1))
    emitted = (g_tok >= 0).sum(1)
    assert np.array_equal(emitted, g_na + 1)
    assert np.all(g_tok[g_tok >= 0] < V)
    for r in np.flatnonzero(g_na > 0)[:200]:
        assert np.array_equal(g_tok[r, : g_na[r]], g_dr[r, : g_na[r]])
    idx = np.random.default_rng(0).choice(R, 300, replace=False)
    # Philox counters use the round index, so each sampled round is replayed with
    # explicit uniforms drawn for its own index
    from oracle import oracle as O
    for r in idx:
        q = np.stack([O.process(drf[r, t], 50, 0.9)[0] for t in range(N - 1)])
        p = np.stack([O.process(tgt[r, t], 50, 0.9)[0] for t in range(N)])
        dr = [O.sample(q[t], O.uniform(1, int(r), 0, t + 1, O.ORC_DRAFT))[0] for t in range(N - 1)]
        ua = [O.uniform(1, int(r), 0, t + 1, O.ORC_ACCEPT) for t in range(N - 1)]
        ut = [O.uniform(1, int(r), 0, t + 1, O.ORC_TARGET) for t in range(N)]
        na, em, _ = O.accept_chain(q, dr, p, ua, ut)
        if draw_margin(tgt[r], drf[r], 50, 0.9, 1, r) < softmax_tol(50, V):
            continue
        assert g_dr[r].tolist() == dr
        assert int(g_na[r]) == na
        assert g_tok[r, : len(em)].tolist() == em
