"""The tensor-core GEMV path (bf16 contexts whose max_streams x row slots reach
32) against the CPU oracle.

The path splits every fp32 input into bf16 hi + lo parts, so its logits stay
within the bf16 tolerance of the float64 oracle (2e-2 absolute).  Its
reductions, like the CUDA-core path's, do not depend on the other rows of a
pass, so greedy speculation equals greedy AR exactly within contexts of the
same max_streams.  Codes are compared with the same near-tie allowance as
the other decode tests."""
import numpy as np
import pytest

from gpu_common import compare_codes_with_margins, require_gpu, torch

pytestmark = pytest.mark.gpu

MAXS = 16  # 16 streams x 2..8 row slots >= 32 rows: the tensor path


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


_cache = {}


def _model(orc, spec):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    if spec not in _cache:
        w = S.gen_weights(spec, 0)
        _cache[spec] = (orc.Model(spec, w), binding.weights_to_device(spec, w))
    return _cache[spec]


def _ctx(orc, N, T=0.9, maxs=MAXS):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    m, dw = _model(orc, S.TTS06B_BF16)
    return binding.CpSpec(S.TTS06B_BF16, dw, N, 50, T, 1, max_streams=maxs), m


def test_teacher_logits_tensor_path(orc):
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TTS06B_BF16
    G = spec.num_code_groups
    B = 3
    cp, m = _ctx(orc, 4)
    x, _ = S.gen_frames(spec, B, 1, seed=16)
    codes = np.random.default_rng(11).integers(0, spec.vocab, (B, G - 1)).astype(np.int32)
    lg, dl = cp.teacher_logits(torch.from_numpy(x[0]).cuda(), torch.from_numpy(codes).cuda(), G, draft=True)
    torch.cuda.synchronize()
    cp.status()
    for b in range(B):
        o_lg, o_dl = m.teacher_logits(x[0, b], codes[b], G, n_draft=3)
        err = np.abs(lg[b].cpu().numpy() - o_lg).max()
        derr = np.abs(dl[b].cpu().numpy() - o_dl).max()
        assert err < 2e-2 and derr < 2e-2, (b, err, derr)


def test_tensor_path_greedy_spec_equals_greedy_ar(orc):
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TTS06B_BF16
    B, F = 5, 2
    x, c0 = S.gen_frames(spec, B, F, seed=17)
    xd, cd = torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()
    ref = None
    for N in (0, 4, 8):
        cp, _ = _ctx(orc, N, T=0.0)
        c = cp.decode_frames(xd, cd).cpu().numpy()
        cp.status()
        if ref is None:
            ref = c
        assert np.array_equal(c, ref), N


def test_tensor_path_decode_matches_oracle(orc):
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TTS06B_BF16
    B, F = 3, 2
    cp, m = _ctx(orc, 4)
    x, c0 = S.gen_frames(spec, B, F, seed=18)
    g = cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
    cp.status()
    o, _, log = m.decode_frames(4, 50, 0.9, 1, x, c0, log_cap=4000)
    compare_codes_with_margins(g, o, log, 1e-4, max_frac=0.5)
    st = cp.stats()
    assert st["committed"] == B * F * (spec.num_code_groups - 1)


def test_tensor_path_row_split_is_batch_invariant(orc):
    """64 streams x 4 row slots: the O and down GEMVs split each pass's 16-row blocks
    over 2-3 CTAs per weight tile.  An output element is still one warp's MMA chain over K,
    so the first 16 streams decode exactly as in a 16-stream context."""
    from speculative_decoding_rvq_gb300 import synth as S
    spec = S.TTS06B_BF16
    B, F = 64, 1
    x, c0 = S.gen_frames(spec, B, F, seed=19)
    cp64, _ = _ctx(orc, 4, maxs=64)
    c64 = cp64.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
    cp64.status()
    cp16, _ = _ctx(orc, 4, maxs=16)
    c16 = cp16.decode_frames(torch.from_numpy(x[:, :16].copy()).cuda(),
                             torch.from_numpy(c0[:, :16].copy()).cuda()).cpu().numpy()
    cp16.status()
    assert np.array_equal(c64[:, :16], c16)
