"""Sparse-tree rounds on the GPU vs the CPU oracle's tree decode
("RVQ Position Aware Speculative Decoding for On Device TTS", section 2.2,
tree attention and sparse tree attention, Figure 2).

- fp32 tiny model, three trees, greedy and sampled: codes equal the oracle's
  tree decode frame by frame, except frames whose first difference follows an
  oracle decision with margin below 1e-4 (float32 vs float64 order).
- bf16 0.6B-class model (2 layers), sampled: the same comparison.
- The one-rank chain tree under temperature 0 reproduces the GPU chain path
  (N = 4) exactly: codes, rounds, passes and acceptance by depth.
- Greedy tree decoding equals greedy autoregressive decoding of the oracle."""
import dataclasses

import numpy as np
import pytest

from gpu_common import compare_codes_with_margins, require_gpu, torch

pytestmark = pytest.mark.gpu

TREES = {
    "chain3": ([-1, 0, 1], [0, 0, 0]),
    "wide": ([-1, -1, -1, 0, 1], [0, 1, 2, 0, 0]),
    "sparse": ([-1, -1, 0, 0, 1, 2, 3], [0, 1, 0, 1, 0, 0, 0]),
}


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


def _decode(cp, x, c0, G):
    F, B, _ = x.shape
    codes = torch.empty((F, B, G), dtype=torch.int32, device="cuda")
    cp.decode_frames(torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda(), codes)
    torch.cuda.synchronize()
    cp.status()
    return codes.cpu().numpy()


@pytest.mark.parametrize("name", sorted(TREES))
@pytest.mark.parametrize("T", [0.0, 0.9])
def test_tree_decode_matches_oracle_fp32(orc, name, T):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = S.TINY_FP32
    w, m, dw = _model(orc, spec)
    G = spec.num_code_groups
    x, c0 = S.gen_frames(spec, 2, 4, seed=7)
    par, rk = TREES[name]
    cp = binding.CpSpec(spec, dw, 4, 50, T, 1, max_streams=2, tree=(par, rk))
    g = _decode(cp, x, c0, G)
    st = cp.stats()
    o, ost, log = m.decode_frames_tree(par, rk, 50, T, 1, x, c0, log_cap=10000)
    compare_codes_with_margins(g, o, log, 1e-4)
    assert st["committed"] == 8 * (G - 1)
    if np.array_equal(g, o):  # the same decisions: the same rounds and acceptance by depth
        assert st["rounds"] == ost["rounds"]  # (passes: the library counts passes of all streams at once)
        assert st["accepted_by_offset"] == ost["accepted_by_offset"]
    cp.close()


def test_tree_decode_matches_oracle_bf16_sampled(orc):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = dataclasses.replace(S.TTS06B_BF16, n_layers=2)
    w, m, dw = _model(orc, spec)
    G = spec.num_code_groups
    x, c0 = S.gen_frames(spec, 2, 2, seed=3)
    par, rk = TREES["sparse"]
    cp = binding.CpSpec(spec, dw, 4, 50, 0.9, 1, max_streams=2, tree=(par, rk))
    g = _decode(cp, x, c0, G)
    o, _, log = m.decode_frames_tree(par, rk, 50, 0.9, 1, x, c0, log_cap=10000)
    compare_codes_with_margins(g, o, log, 1e-3, max_frac=0.5)
    cp.close()


def test_chain_tree_reproduces_the_greedy_chain(orc):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = S.TINY_FP32
    w, m, dw = _model(orc, spec)
    G = spec.num_code_groups
    x, c0 = S.gen_frames(spec, 2, 6, seed=2)
    ch = binding.CpSpec(spec, dw, 4, 50, 0.0, 1, max_streams=2)
    gc = _decode(ch, x, c0, G)
    sc = ch.stats()
    tr = binding.CpSpec(spec, dw, 4, 50, 0.0, 1, max_streams=2, tree=([-1, 0, 1], [0, 0, 0]))
    gt = _decode(tr, x, c0, G)
    st = tr.stats()
    assert np.array_equal(gt, gc)
    assert (st["rounds"], st["passes"]) == (sc["rounds"], sc["passes"])
    assert st["accepted_by_offset"] == sc["accepted_by_offset"]
    assert sum(sc["accepted_by_offset"]) > 0
    ch.close()
    tr.close()


@pytest.mark.parametrize("name", ["wide", "sparse"])
def test_greedy_tree_equals_greedy_autoregressive(orc, name):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = S.TINY_FP32
    w, m, dw = _model(orc, spec)
    G = spec.num_code_groups
    x, c0 = S.gen_frames(spec, 2, 4, seed=11)
    par, rk = TREES[name]
    cp = binding.CpSpec(spec, dw, 4, 50, 0.0, 1, max_streams=2, tree=(par, rk))
    g = _decode(cp, x, c0, G)
    o, _, log = m.decode_frames(0, 50, 0.0, 1, x, c0, log_cap=10000)
    compare_codes_with_margins(g, o, log, 1e-4)
    cp.close()


@pytest.mark.parametrize("par, rk", [([0], [0]), ([-1, -1], [1, 0]), ([-1, -1], [0, 0]), ([-1, 0, 1, 2, 3, 4, 5, 6], [0] * 8)])
def test_malformed_trees_are_rejected(orc, par, rk):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = S.TINY_FP32
    w, m, dw = _model(orc, spec)
    with pytest.raises(binding.CpSpecError):
        binding.CpSpec(spec, dw, 4, 50, 0.9, 1, tree=(par, rk))


def test_tree_rounds_on_the_tcgen05_tiles(orc):
    """8 streams x 8 row slots = 64 rows per pass: the GEMVs run as tcgen05 tiles, whose
    epilogue appends each tree node's K/V to its own slot.  Greedy: the rank-0 chain tree
    equals the chain path on the same tiles, and the sparse tree equals the oracle's tree
    decode (which equals greedy AR)."""
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec = dataclasses.replace(S.TTS06B_BF16, n_layers=2)
    w, m, dw = _model(orc, spec)
    G = spec.num_code_groups
    B = 8
    x, c0 = S.gen_frames(spec, B, 1, seed=13)
    ch = binding.CpSpec(spec, dw, 4, 50, 0.0, 1, max_streams=B)
    gc = _decode(ch, x, c0, G)
    tr = binding.CpSpec(spec, dw, 4, 50, 0.0, 1, max_streams=B, tree=([-1, 0, 1], [0, 0, 0]))
    gt = _decode(tr, x, c0, G)
    assert np.array_equal(gt, gc)
    par, rk = TREES["sparse"]
    sp = binding.CpSpec(spec, dw, 4, 50, 0.0, 1, max_streams=B, tree=(par, rk))
    gs = _decode(sp, x, c0, G)
    o, _, log = m.decode_frames_tree(par, rk, 50, 0.0, 1, x[:, :2], c0[:, :2], log_cap=10000)  # 2 streams: oracle time
    compare_codes_with_margins(gs[:, :2], o, log, 1e-3, max_frac=0.5)
    for cp in (ch, tr, sp):
        cp.close()
