"""The adaptive verify window on the GPU against the CPU oracle ("Speculative
Decoding, Beyond Text", runtime policies).

Each stream picks the window of its next frame from its acceptance by offset
earlier in the call, with the same integer rule on both sides, so the codes,
the pass counts and the acceptance counters match the oracle (codes with the
near-tie allowance of the other decode tests).  When drafts never match, the
window collapses to 1 after the first frame and later frames take one pass
per code; greedy decoding still equals the greedy AR loop."""
import dataclasses

import numpy as np
import pytest

from gpu_common import compare_codes_with_margins, require_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _pair(orc, spec, K=0, std=1.0):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    w = S.gen_weights(spec, 0)
    if K:
        w["draft_offset"] = S.gen_draft_offsets(spec, K, seed=5, std=std)
    return orc.Model(spec, w), binding.weights_to_device(spec, w)


@pytest.mark.parametrize("N,T,pct", [(4, 0.9, 60), (8, 0.9, 50), (3, 0.0, 70)])
def test_policy_decode_matches_oracle(orc, N, T, pct):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = S.TINY_FP32
    m, dw = _pair(orc, spec)
    B, F = 2, 8
    cp = binding.CpSpec(spec, dw, N, 50, T, 1, max_streams=B, adapt_pct=pct, adapt_min=4)
    x, c0 = S.gen_frames(spec, B, F, seed=3)
    g = cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
    cp.status()
    o, ost, log = m.decode_frames(N, 50, T, 1, x, c0, log_cap=10000, adapt_pct=pct, adapt_min=4)
    tolerated = compare_codes_with_margins(g, o, log, 1e-4)
    st = cp.stats()
    assert st["committed"] == B * F * (spec.num_code_groups - 1)
    if tolerated == 0:  # the same windows and decisions: the same per-stream counters
        assert st["rounds"] == ost["rounds"]
        assert st["accepted_by_offset"] == ost["accepted_by_offset"]
        r = log[(log["s"] >= 1)]
        reached = [0] + [int(np.sum((r["n_d"] >= t) & (r["n_acc"] >= t - 1))) for t in range(1, 9)]
        assert st["drafted_by_offset"] == reached


def test_policy_collapse_turns_drafting_off(orc):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = dataclasses.replace(S.TINY_FP32, n_layers=1)
    m, dw = _pair(orc, spec, K=7, std=300.0)
    G, F = spec.num_code_groups, 6
    x, c0 = S.gen_frames(spec, 1, F, seed=3)
    cp = binding.CpSpec(spec, dw, 4, 50, 0.0, 1, max_streams=1, adapt_pct=50, adapt_min=4)
    g = cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
    cp.status()
    ar, _, _ = m.decode_frames(0, 50, 0.0, 1, x, c0)
    o, ost, log = m.decode_frames(4, 50, 0.0, 1, x, c0, log_cap=1000, adapt_pct=50, adapt_min=4)
    assert np.array_equal(g, ar) and np.array_equal(o, ar)
    first = int(np.sum(log["frame"] == 0))
    st = cp.stats()  # one stream: the library's pass count is the stream's
    assert st["passes"] == ost["passes"] == first + (F - 1) * (G - 1)


def test_policy_greedy_bf16_equals_greedy_ar(orc):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = S.TTS06B_BF16
    _, dw = _pair(orc, spec, K=3, std=1.0)
    x, c0 = S.gen_frames(spec, 1, 4, seed=2)
    xd, cd = torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()
    ar = binding.CpSpec(spec, dw, 0, 50, 0.0, 1).decode_frames(xd, cd).cpu().numpy()
    for N, pct in ((4, 60), (8, 90)):
        cp = binding.CpSpec(spec, dw, N, 50, 0.0, 1, adapt_pct=pct, adapt_min=4)
        c = cp.decode_frames(xd, cd).cpu().numpy()
        cp.status()
        assert np.array_equal(c, ar), (N, pct)
