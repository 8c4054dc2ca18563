"""The large model shapes on the GPU: H 2048, 32 q / 8 kv heads x 64, FFN 6144
(GEMV inputs of 12 KB rows, three 16-byte chunks per thread), V 4096, G 32
(31 lm_heads, 32 positions per frame).  Two layers keep the oracle's float64
forward short; every per-layer kernel shape of the 8-layer model runs.

- Teacher-forced target and draft logits within the bf16 tolerance (2e-2)
  of the oracle, on both GEMV paths (1 stream: CUDA cores; 16 streams:
  tensor cores).
- Greedy speculation equals the greedy AR loop exactly over whole frames."""
import dataclasses

import numpy as np
import pytest

from gpu_common import require_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.fixture(scope="module")
def large(orc):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = dataclasses.replace(S.LARGE_BF16, n_layers=2)
    w = S.gen_weights(spec, 0)
    return spec, orc.Model(spec, w), binding.weights_to_device(spec, w)


@pytest.mark.parametrize("maxs", [1, 16])
def test_large_teacher_logits(large, maxs):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec, m, dw = large
    P = 7
    cp = binding.CpSpec(spec, dw, 4, 50, 0.8, 1, max_streams=maxs)
    x, _ = S.gen_frames(spec, 1, 1, seed=20)
    codes = np.random.default_rng(21).integers(0, spec.vocab, (1, P - 1)).astype(np.int32)
    lg, dl = cp.teacher_logits(torch.from_numpy(x[0]).cuda(), torch.from_numpy(codes).cuda(), P, draft=True)
    torch.cuda.synchronize()
    cp.status()
    o_lg, o_dl = m.teacher_logits(x[0, 0], codes[0], P, n_draft=3)
    err = np.abs(lg[0].cpu().numpy() - o_lg).max()
    derr = np.abs(dl[0].cpu().numpy() - o_dl).max()
    assert err < 2e-2 and derr < 2e-2, (err, derr)


def test_large_greedy_spec_equals_greedy_ar(large):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec, _, dw = large
    x, c0 = S.gen_frames(spec, 1, 2, seed=22)
    xd, cd = torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()
    ref = None
    for N in (0, 4, 8):
        cp = binding.CpSpec(spec, dw, N, 50, 0.0, 1, max_streams=1)
        c = cp.decode_frames(xd, cd).cpu().numpy()
        cp.status()
        assert cp.stats()["committed"] == 2 * (spec.num_code_groups - 1)
        if ref is None:
            ref = c
        assert np.array_equal(c, ref), N
