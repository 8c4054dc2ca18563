"""The KV rule of the round ("Speculative Decoding, Beyond Text", section 07:
the logical length and the valid-position mask; "CodePredictor Speculative
Decoding", "How a round works" step 4): after each decision, the slots past
the committed depth hold nothing a later pass may read before rewriting it.

With the test hook on, the accept kernel writes NaN into every such slot of
every stream (positions past the committed depth, the tree nodes' slots, the
whole cache at a frame's end).  A pass that read one would carry NaN into its
logits, so the codes, the counters and the status must equal those of the
same decode without the hook, on each GEMV path (small-batch, CUDA-core fp32,
tcgen05 tiles) and for tree rounds.  The step-wise run also checks the
logical length after each round: committed = s + 1, growing by at least one
code per round."""
import dataclasses

import numpy as np
import pytest

from gpu_common import require_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


_cache = {}


def _dw(spec):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    if spec not in _cache:
        _cache[spec] = binding.weights_to_device(spec, S.gen_weights(spec, 0))
    return _cache[spec]


def _run(spec, B, F, poison, N=4, T=0.9, tree=None):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    G = spec.num_code_groups
    x, c0 = S.gen_frames(spec, B, F, seed=5)
    cp = binding.CpSpec(spec, _dw(spec), N, 50, T, 1, max_streams=B, tree=tree)
    if poison:
        cp.test_hooks(poison_kv=True)
    codes = torch.empty((F, B, G), dtype=torch.int32, device="cuda")
    cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda(), codes)
    torch.cuda.synchronize()
    assert cp.status_code() == 0
    st = cp.stats()
    cp.close()
    return codes.cpu().numpy(), st


CASES = {
    "bf16_small_batch": (lambda S: dataclasses.replace(S.TTS06B_BF16, n_layers=2), 2, 2, None),
    "fp32_cuda_cores": (lambda S: S.TINY_FP32, 3, 4, None),
    "bf16_tcgen05_tiles": (lambda S: dataclasses.replace(S.TTS06B_BF16, n_layers=2), 8, 2, None),
    "fp32_tree": (lambda S: S.TINY_FP32, 2, 4, ([-1, -1, 0, 0, 1, 2, 3], [0, 1, 0, 1, 0, 0, 0])),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_stale_kv_slots_are_never_read(case):
    from speculative_decoding_rvq_gb300 import synth as S
    mk, B, F, tree = CASES[case]
    spec = mk(S)
    clean, st0 = _run(spec, B, F, False, tree=tree)
    poisoned, st1 = _run(spec, B, F, True, tree=tree)
    assert np.array_equal(poisoned, clean)
    for k in ("committed", "rounds", "passes", "rejections", "bonus"):
        assert st1[k] == st0[k], k
    assert st1["accepted_by_offset"] == st0["accepted_by_offset"]


def test_logical_length_per_round_with_poison():
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = S.TINY_FP32
    G, B = spec.num_code_groups, 2
    x, c0 = S.gen_frames(spec, B, 2, seed=5)  # the frames _run decodes
    ref, _ = _run(spec, B, 2, False)
    cp = binding.CpSpec(spec, _dw(spec), 4, 50, 0.9, 1, max_streams=B)
    cp.test_hooks(poison_kv=True)
    codes = torch.zeros((B, G), dtype=torch.int32, device="cuda")
    committed = torch.zeros((B,), dtype=torch.int32, device="cuda")
    for f in range(2):
        cp.begin_frame(torch.from_numpy(x[f]).cuda().clone(), torch.from_numpy(c0[f]).cuda().clone(), f)
        prev = np.ones(B, np.int64)  # c_0 is known at the frame start
        for _ in range(G):
            cp.round(codes, committed)
            torch.cuda.synchronize()
            now = committed.cpu().numpy()
            assert np.all(now <= G) and np.all((now > prev) | (prev == G)), (prev, now)
            prev = now
            if np.all(now == G):
                break
        assert np.all(prev == G)
        assert np.array_equal(codes.cpu().numpy(), ref[f])
    assert cp.status_code() == 0
    cp.close()
