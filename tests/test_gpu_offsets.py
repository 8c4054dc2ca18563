"""Position-aware draft offsets on the GPU against the CPU oracle ("RVQ
Position Aware Speculative Decoding for On Device TTS", section 2.2).

The library forms head_j . b_t once per context and adds it to the
lookahead-t draft logits; the oracle applies head_j to h + b_t directly.  The
two agree within the logit tolerances of the other decode tests (1e-4 fp32,
2e-2 bf16).  The offsets change only the drafts, so greedy speculation with
offsets still equals greedy AR exactly, while the acceptance counters do
move (the offsets are really applied)."""
import numpy as np
import pytest

from gpu_common import compare_codes_with_margins, require_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


_cache = {}


def _model(orc, spec, K):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    key = (spec, K)
    if key not in _cache:
        w = S.gen_weights(spec, 0)
        if K:
            w["draft_offset"] = S.gen_draft_offsets(spec, K, seed=1, std=1.0)
        _cache[key] = (orc.Model(spec, w), binding.weights_to_device(spec, w))
    return _cache[key]


def _ctx(orc, spec, N, K, T=0.9, B=1):
    from speculative_decoding_rvq_gb300 import binding
    m, dw = _model(orc, spec, K)
    return binding.CpSpec(spec, dw, N, 50, T, 1, max_streams=B), m


@pytest.mark.parametrize("N,K", [(3, 2), (8, 3), (4, 7)])
def test_teacher_draft_logits_with_offsets_fp32(orc, N, K):
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TINY_FP32
    G = spec.num_code_groups
    cp, m = _ctx(orc, spec, N, K, B=2)
    x, _ = S.gen_frames(spec, 2, 1, seed=5)
    codes = np.random.default_rng(0).integers(0, spec.vocab, (2, G - 1)).astype(np.int32)
    lg, dl = cp.teacher_logits(torch.from_numpy(x[0]).cuda(), torch.from_numpy(codes).cuda(), G, draft=True)
    torch.cuda.synchronize()
    cp.status()
    for b in range(2):
        o_lg, o_dl = m.teacher_logits(x[0, b], codes[b], G, n_draft=N - 1)
        np.testing.assert_allclose(lg[b].cpu().numpy(), o_lg, atol=1e-4, rtol=0)
        np.testing.assert_allclose(dl[b].cpu().numpy(), o_dl, atol=1e-4, rtol=0)


@pytest.mark.parametrize("maxs", [1, 16])  # 16 streams x 4 row slots: the tensor-core GEMV path
def test_teacher_draft_logits_with_offsets_bf16(orc, maxs):
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TTS06B_BF16
    G = spec.num_code_groups
    cp, m = _ctx(orc, spec, 4, 3, B=maxs)
    x, _ = S.gen_frames(spec, 1, 1, seed=6)
    codes = np.random.default_rng(1).integers(0, spec.vocab, (1, G - 1)).astype(np.int32)
    lg, dl = cp.teacher_logits(torch.from_numpy(x[0]).cuda(), torch.from_numpy(codes).cuda(), G, draft=True)
    torch.cuda.synchronize()
    cp.status()
    o_lg, o_dl = m.teacher_logits(x[0, 0], codes[0], G, n_draft=3)
    err = np.abs(lg[0].cpu().numpy() - o_lg).max()
    derr = np.abs(dl[0].cpu().numpy() - o_dl).max()
    assert err < 2e-2 and derr < 2e-2, (err, derr)


def test_greedy_spec_with_offsets_equals_greedy_ar(orc):
    from speculative_decoding_rvq_gb300 import synth as S
    for spec, F in ((S.TINY_FP32, 8), (S.TTS06B_BF16, 4)):
        x, c0 = S.gen_frames(spec, 1, F, seed=2)
        xd, cd = torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()
        cp, _ = _ctx(orc, spec, 0, 0, T=0.0)
        ref = cp.decode_frames(xd, cd).cpu().numpy()
        moved = 0
        for N in (2, 4, 8):
            cp, _ = _ctx(orc, spec, N, 3, T=0.0)
            c = cp.decode_frames(xd, cd).cpu().numpy()
            cp.status()
            assert np.array_equal(c, ref), (spec.hidden, N)
            plain, _ = _ctx(orc, spec, N, 0, T=0.0)
            plain.decode_frames(xd, cd)
            moved += int(cp.stats()["accepted_by_offset"] != plain.stats()["accepted_by_offset"])
        assert moved > 0, spec.hidden


@pytest.mark.parametrize("which", ["fp32_N4", "fp32_N8_greedy", "bf16_N4"])
def test_decode_with_offsets_matches_oracle(orc, which):
    from speculative_decoding_rvq_gb300 import synth as S
    if which == "bf16_N4":
        spec, B, F, N, T = S.TTS06B_BF16, 1, 2, 4, 0.9
    else:
        spec, B, F = S.TINY_FP32, 2, 6
        N, T = (4, 0.9) if which == "fp32_N4" else (8, 0.0)
    cp, m = _ctx(orc, spec, N, 3, T=T, B=B)
    x, c0 = S.gen_frames(spec, B, F, seed=3)
    g = cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
    cp.status()
    o, ost, log = m.decode_frames(N, 50, T, 1, x, c0, log_cap=10000)
    tolerated = compare_codes_with_margins(g, o, log, 1e-4, max_frac=0.5 if spec.dtype else 0.05)
    st = cp.stats()
    assert st["committed"] == B * F * (spec.num_code_groups - 1)
    if which != "bf16_N4" and tolerated == 0:  # same drafts and decisions: the same acceptance counters
        assert st["accepted_by_offset"] == ost["accepted_by_offset"]
        # the library counts the drafts the left-to-right test reached (up to the first rejection)
        r = log[: min(len(log), 10000)]
        r = r[r["n_d"] > 0]
        reached = [0] + [int(np.sum((r["n_d"] >= t) & (r["n_acc"] >= t - 1))) for t in range(1, 9)]
        assert st["drafted_by_offset"] == reached
