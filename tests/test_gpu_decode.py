"""GPU decoder passes and frame decoding vs the CPU oracle.

Tolerances: logits within 1e-4 (fp32 weights) / 2e-2 (bf16 weights) of the
float64 oracle.  Codes: identical, except a frame whose first difference was
decided by a near-tie (oracle decision margin below 1e-4) -- the float32 vs
float64 accumulation order may flip such a decision, after which the frame's
conditioning differs."""
import dataclasses

import numpy as np
import pytest

from gpu_common import compare_codes_with_margins, require_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


_cache = {}


def _model(orc, spec, seed=0):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    key = (spec, seed)
    if key not in _cache:
        w = S.gen_weights(spec, seed)
        _cache[key] = (w, orc.Model(spec, w), binding.weights_to_device(spec, w))
    return _cache[key]


def _ctx(orc, spec, N, k=50, T=0.9, seed=1, B=1):
    from speculative_decoding_rvq_gb300 import binding
    w, m, dw = _model(orc, spec)
    return binding.CpSpec(spec, dw, N, k, T, seed, max_streams=B), m


@pytest.mark.parametrize("N", [0, 3, 8])
def test_teacher_logits_fp32(orc, N):
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TINY_FP32
    cp, m = _ctx(orc, spec, N, B=2)
    G = spec.num_code_groups
    x, c0 = S.gen_frames(spec, 2, 1, seed=5)
    codes = np.random.default_rng(0).integers(0, spec.vocab, (2, G - 1)).astype(np.int32)
    lg, dl = cp.teacher_logits(torch.from_numpy(x[0]).cuda(), torch.from_numpy(codes).cuda(), G, draft=N >= 2)
    torch.cuda.synchronize()
    cp.status()
    for b in range(2):
        o_lg, o_dl = m.teacher_logits(x[0, b], codes[b], G, n_draft=max(N - 1, 0))
        np.testing.assert_allclose(lg[b].cpu().numpy(), o_lg, atol=1e-4, rtol=0)
        if N >= 2:
            np.testing.assert_allclose(dl[b].cpu().numpy(), o_dl, atol=1e-4, rtol=0)


def test_teacher_logits_bf16(orc):
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TTS06B_BF16
    cp, m = _ctx(orc, spec, 4)
    G = spec.num_code_groups
    x, _ = S.gen_frames(spec, 1, 1, seed=6)
    codes = np.random.default_rng(1).integers(0, spec.vocab, (1, G - 1)).astype(np.int32)
    lg, dl = cp.teacher_logits(torch.from_numpy(x[0]).cuda(), torch.from_numpy(codes).cuda(), G, draft=True)
    torch.cuda.synchronize()
    cp.status()
    o_lg, o_dl = m.teacher_logits(x[0, 0], codes[0], G, n_draft=3)
    err = np.abs(lg[0].cpu().numpy() - o_lg).max()
    derr = np.abs(dl[0].cpu().numpy() - o_dl).max()
    assert err < 2e-2 and derr < 2e-2, (err, derr)


@pytest.mark.parametrize("N,T", [(0, 0.9), (2, 0.9), (3, 0.9), (4, 0.0), (8, 0.9), (5, 1.5)])
def test_decode_fp32_matches_oracle(orc, N, T):
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TINY_FP32
    B, F = 2, 6
    cp, m = _ctx(orc, spec, N, T=T, B=B)
    x, c0 = S.gen_frames(spec, B, F, seed=1)
    codes = cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda())
    torch.cuda.synchronize()
    cp.status()
    g = codes.cpu().numpy()
    o, ost, log = m.decode_frames(N, 50, T, 1, x, c0, log_cap=10000)
    compare_codes_with_margins(g, o, log, 1e-4)
    st = cp.stats()
    assert st["committed"] == F * B * (spec.num_code_groups - 1)
    assert st["frames"] == F * B


def test_greedy_spec_equals_greedy_ar_on_gpu(orc):
    """Row results do not depend on which rows share a pass: greedy speculative == greedy AR exactly."""
    from speculative_decoding_rvq_gb300 import synth as S
    for spec, F in ((S.TINY_FP32, 8), (S.TTS06B_BF16, 4)):
        x, c0 = S.gen_frames(spec, 1, F, seed=2)
        xd, cd = torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()
        ref = None
        for N in (0, 2, 4, 8):
            cp, _ = _ctx(orc, spec, N, T=0.0)
            c = cp.decode_frames(xd, cd).cpu().numpy()
            cp.status()
            if ref is None:
                ref = c
            assert np.array_equal(c, ref), (spec.hidden, N)


def test_decode_bf16_matches_oracle(orc):
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TTS06B_BF16
    F = 2
    for N in (0, 4):
        cp, m = _ctx(orc, spec, N)
        x, c0 = S.gen_frames(spec, 1, F, seed=3)
        g = cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
        cp.status()
        o, _, log = m.decode_frames(N, 50, 0.9, 1, x, c0, log_cap=1000)
        compare_codes_with_margins(g, o, log, 1e-4, max_frac=0.5)


def test_round_api_equals_decode_frames(orc):
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TINY_FP32
    B = 3
    x, c0 = S.gen_frames(spec, B, 1, seed=4)
    xd, cd = torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()
    cp, _ = _ctx(orc, spec, 4, B=B)
    ref = cp.decode_frames(xd, cd, first_frame=7).cpu().numpy()[0]
    cp2, _ = _ctx(orc, spec, 4, B=B)
    codes = torch.zeros((B, spec.num_code_groups), dtype=torch.int32, device="cuda")
    committed = torch.zeros((B,), dtype=torch.int32, device="cuda")
    cp2.begin_frame(xd[0], cd[0], 7)
    rounds = 0
    while True:
        cp2.round(codes, committed)
        rounds += 1
        if int(committed.min().item()) == spec.num_code_groups or rounds > 64:
            break
    cp2.status()
    assert np.array_equal(codes.cpu().numpy(), ref)
    assert rounds <= spec.num_code_groups - 1


def test_batched_streams_are_independent(orc):
    """Stream b decoded in a batch equals stream b decoded with fewer streams (same Philox stream id)."""
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TINY_FP32
    x, c0 = S.gen_frames(spec, 5, 3, seed=8)
    cp5, _ = _ctx(orc, spec, 3, B=5)
    c5 = cp5.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
    cp2, _ = _ctx(orc, spec, 3, B=2)
    c2 = cp2.decode_frames(torch.from_numpy(x[:, :2].copy()).cuda(), torch.from_numpy(c0[:, :2].copy()).cuda()).cpu().numpy()
    assert np.array_equal(c5[:, :2], c2)


def test_mixed_greedy_and_sampling_streams(orc):
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TINY_FP32
    B, F = 4, 4
    cp, m = _ctx(orc, spec, 4, B=B)
    tk = np.array([50, 50, 50, 20], np.int32)
    tp = np.array([0.0, 0.9, 0.0, 1.2], np.float32)
    cp.set_stream_sampling(tk, tp)
    x, c0 = S.gen_frames(spec, B, F, seed=9)
    g = cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
    cp.status()
    o, _, log = m.decode_frames(4, tk, tp, 1, x, c0, log_cap=10000)
    compare_codes_with_margins(g, o, log, 1e-4)


def test_code_groups_edge_cases(orc):
    """G = 2 (speculation falls back to AR with a warning) and G = 3 (one draft slot)."""
    from speculative_decoding_rvq_gb300 import binding, synth as S
    for G in (2, 3):
        spec = dataclasses.replace(S.TINY_FP32, num_code_groups=G)
        w = S.gen_weights(spec, 0)
        m = orc.Model(spec, w)
        cp = binding.CpSpec(spec, binding.weights_to_device(spec, w), 4, 50, 0.9, 1, 1)
        assert cp.ar_fallback == (G == 2)
        x, c0 = S.gen_frames(spec, 1, 4, seed=1)
        g = cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
        cp.status()
        o, _, log = m.decode_frames(0 if G == 2 else 4, 50, 0.9, 1, x, c0, log_cap=100)
        compare_codes_with_margins(g, o, log, 1e-4)
