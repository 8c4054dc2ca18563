"""GPU decode against the CPU oracle on the shapes the benchmark runs, beyond
the small cases of the other decode tests.

- The batched configuration: 64 streams x 4 row slots (the many-row tensor
  path, whose O and down GEMVs split each pass's row blocks over 2-3 CTAs),
  N = 4, even streams greedy and odd streams top-k 50 / T 0.9.  The oracle
  decodes the first 16 streams (streams are independent and their Philox
  counters carry the stream id, so its codes for those streams do not depend
  on the other 48); two layers keep its float64 forward short, and every
  per-layer kernel shape of the 5-layer model still runs.
- The 0.6B-class model with sampling at N = 2 and N = 8 (the small-batch
  tensor path at 2 and 8 rows per pass).
- The large model (two layers) with sampling at N = 4 on both GEMV paths.

Codes must match frame by frame, except where the frame's first difference
was decided within the oracle's near-tie margin (float64 forward against the
kernels' float32 accumulation, float32 softmax against float64), in at most
10 % of the frames."""
import dataclasses

import numpy as np
import pytest

from gpu_common import compare_codes_with_margins, require_gpu, torch

pytestmark = pytest.mark.gpu

MARGIN = 1e-3  # logit-unit / relative decision margin a bf16-weight pass may flip


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _pair(orc, spec):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    w = S.gen_weights(spec, 0)
    return orc.Model(spec, w), binding.weights_to_device(spec, w)


def test_batched_64_streams_half_greedy(orc):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = dataclasses.replace(S.TTS06B_BF16, n_layers=2)
    m, dw = _pair(orc, spec)
    B, F, Bo = 64, 1, 16
    tk = np.full(B, 50, np.int32)
    tp = np.where(np.arange(B) % 2 == 0, 0.0, 0.9).astype(np.float32)
    cp = binding.CpSpec(spec, dw, 4, 50, 0.9, 1, max_streams=B)
    cp.set_stream_sampling(tk, tp)
    x, c0 = S.gen_frames(spec, B, F, seed=41)
    g = cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
    cp.status()
    o, _, log = m.decode_frames(4, tk[:Bo], tp[:Bo], 1, x[:, :Bo].copy(), c0[:, :Bo].copy(), log_cap=4000)
    compare_codes_with_margins(g[:, :Bo], o, log, MARGIN, max_frac=0.1)
    assert ((g >= 0) & (g < spec.vocab)).all()


@pytest.mark.parametrize("N", [2, 8])
def test_bf16_sampled_decode_small_batch_path(orc, N):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = S.TTS06B_BF16
    m, dw = _pair(orc, spec)
    cp = binding.CpSpec(spec, dw, N, 50, 0.9, 1, max_streams=1)
    x, c0 = S.gen_frames(spec, 1, 2, seed=42 + N)
    g = cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
    cp.status()
    o, _, log = m.decode_frames(N, 50, 0.9, 1, x, c0, log_cap=1000)
    compare_codes_with_margins(g, o, log, MARGIN, max_frac=0.1)


def test_large_model_sampled_decode_both_paths(orc):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = dataclasses.replace(S.LARGE_BF16, n_layers=2)
    m, dw = _pair(orc, spec)
    x, c0 = S.gen_frames(spec, 1, 1, seed=44)
    o, _, log = m.decode_frames(4, 50, 0.8, 1, x, c0, log_cap=1000)
    for maxs in (1, 16):  # the small-batch path; the many-row tensor path
        cp = binding.CpSpec(spec, dw, 4, 50, 0.8, 1, max_streams=maxs)
        g = cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()).cpu().numpy()
        cp.status()
        compare_codes_with_margins(g, o, log, MARGIN, max_frac=0.1)
