"""The C-ABI library loads on a machine without a GPU, exports every symbol
include/cp_spec.h declares, and rejects bad arguments on the host (no device
work is enqueued for an argument error)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_rvq_gb300 import build, binding
    build.build()
    return binding.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(cp_spec_\w+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol(lib):
    from speculative_decoding_rvq_gb300 import binding
    declared = _declared()
    assert declared == set(binding.EXPORTS)
    for n in declared:
        assert hasattr(lib, n), n


def _cfg(b, **kw):
    d = dict(verify_window=4, top_k=50, temperature=0.9, seed=1, max_streams=1)
    d.update(kw)
    return b.Config(**d)


def test_workspace_bytes_validates(lib):
    from speculative_decoding_rvq_gb300 import binding as b, synth as S
    m = b.model_struct(S.TTS06B_BF16)
    assert lib.cp_spec_workspace_bytes(C.byref(m), C.byref(_cfg(b))) > 0
    for bad in (dict(verify_window=1), dict(verify_window=9), dict(verify_window=-1), dict(top_k=0),
                dict(top_k=5000), dict(temperature=-1.0), dict(temperature=1e-6), dict(max_streams=0)):
        assert lib.cp_spec_workspace_bytes(C.byref(m), C.byref(_cfg(b, **bad))) == 0, bad
    big = b.model_struct(S.ModelSpec(1024, 2, 8, 8, 128, 3072, 16384, 16, 1))
    assert lib.cp_spec_workspace_bytes(C.byref(big), C.byref(_cfg(b))) == 0
    # workspace grows with the number of streams
    one = lib.cp_spec_workspace_bytes(C.byref(m), C.byref(_cfg(b)))
    many = lib.cp_spec_workspace_bytes(C.byref(m), C.byref(_cfg(b, max_streams=64)))
    assert many > 32 * one // 2


def test_draft_offsets_validate_and_size_the_workspace(lib):
    """K position-aware offsets: 0..7 accepted; the head . b table is sized by
    min(K, N - 1) lookaheads, and nothing is reserved without drafts.  The
    adaptive-window fields are validated on the host and need no workspace."""
    from speculative_decoding_rvq_gb300 import binding as b, synth as S
    spec = S.TTS06B_BF16
    m = b.model_struct(spec)
    ws = lambda **kw: lib.cp_spec_workspace_bytes(C.byref(m), C.byref(_cfg(b, **kw)))
    for bad in (-1, 8):
        assert ws(draft_offsets=bad) == 0, bad
    # the adaptive window: a percentage in [0, 100], and a sample floor >= 1 when on
    for bad in (dict(adapt_accept_pct=-1), dict(adapt_accept_pct=101), dict(adapt_accept_pct=50, adapt_min_reached=0)):
        assert ws(**bad) == 0, bad
    assert ws(adapt_accept_pct=50, adapt_min_reached=4) == ws()
    table = (spec.num_code_groups - 1) * spec.vocab * 4
    base = ws(verify_window=4)
    for K, used in ((1, 1), (3, 3), (7, 3)):
        grown = ws(verify_window=4, draft_offsets=K) - base
        assert used * table <= grown < used * table + 512, (K, grown)
    assert ws(verify_window=0, draft_offsets=3) == ws(verify_window=0)
    # K > 0 with a null offset pointer is rejected before any device call
    w = b.weights_struct(b.weights_to_device(S.TINY_FP32, S.gen_weights(S.TINY_FP32, 0), device="cpu"))
    mt = b.model_struct(S.TINY_FP32)
    ctx = C.c_void_p()
    rc = lib.cp_spec_init(C.byref(mt), C.byref(w), C.byref(_cfg(b, draft_offsets=2)), C.c_void_p(16), 1 << 30,
                          C.byref(ctx))
    assert rc == b.E_INVALID and b"draft_offset" in lib.cp_spec_last_error(None)


def test_init_rejects_on_host(lib):
    from speculative_decoding_rvq_gb300 import binding as b, synth as S
    m = b.model_struct(S.TINY_FP32)
    w = b.Weights()
    ctx = C.c_void_p()
    assert lib.cp_spec_init(C.byref(m), C.byref(w), C.byref(_cfg(b)), None, 0, None) == b.E_INVALID
    assert lib.cp_spec_init(C.byref(m), C.byref(w), C.byref(_cfg(b, verify_window=1)), None, 0, C.byref(ctx)) == b.E_INVALID
    # null weight pointers are caught before any device call
    assert lib.cp_spec_init(C.byref(m), C.byref(w), C.byref(_cfg(b)), C.c_void_p(16), 1 << 30, C.byref(ctx)) == b.E_INVALID
    assert b"aligned" in lib.cp_spec_last_error(None) or b"null" in lib.cp_spec_last_error(None)


def test_context_free_calls_reject_bad_arguments(lib):
    from speculative_decoding_rvq_gb300 import binding as b
    assert lib.cp_spec_accept_batch(4, 1, 256, 50, 0.9, 1, 0, None, None, None, None, None, None) == b.E_INVALID
    assert lib.cp_spec_accept_batch(4, 9, 256, 50, 0.9, 1, 0, None, None, None, None, None, None) == b.E_INVALID
    assert lib.cp_spec_accept_batch(4, 4, 9000, 50, 0.9, 1, 0, None, None, None, None, None, None) == b.E_UNSUPPORTED
    assert lib.cp_spec_accept_batch(4, 4, 256, 0, 0.9, 1, 0, None, None, None, None, None, None) == b.E_INVALID
    assert lib.cp_spec_accept_batch(4, 4, 256, 50, 0.9, 1, 2, None, None, None, None, None, None) == b.E_INVALID
    assert lib.cp_spec_accept_batch(4, 4, 256, 50, 0.9, 1, 0, None, None, None, None, None, None) == b.E_INVALID
    assert lib.cp_spec_accept_batch(0, 4, 256, 50, 0.9, 1, 0, None, None, None, None, None, None) == b.OK
    for fn, args in (("cp_spec_decode_frames", (1, 1, 0, None, None, None, None)),
                     ("cp_spec_round", (None, None, None)),
                     ("cp_spec_begin_frame", (1, None, None, 0, None)),
                     ("cp_spec_status_word", (None,)),
                     ("cp_spec_reset_stats", (None,))):
        assert getattr(lib, fn)(None, *args) == b.E_INVALID, fn
    assert lib.cp_spec_launch_count(None) >= 0
    lib.cp_spec_destroy(None)


def _tree(b, par, rk):
    import numpy as np
    p = np.ascontiguousarray(par, dtype=np.int32)
    r = np.ascontiguousarray(rk, dtype=np.int32)
    return b.Tree(len(p), p.ctypes.data, r.ctypes.data), (p, r)


def test_tree_workspace_validates_the_tree(lib):
    """cp_spec_workspace_bytes_tree (host only): a well-formed tree ("RVQ Position Aware
    Speculative Decoding for On Device TTS", section 2.2) is sized with one row slot per
    node plus the root and one KV slot per node past the G positions; malformed trees
    (parent not earlier, siblings out of rank order or repeated, depth above 7, rank at or
    above the list capacity, more than 62 nodes) are rejected with 0."""
    from speculative_decoding_rvq_gb300 import binding as b, synth as S
    m = b.model_struct(S.TINY_FP32)
    cfg = _cfg(b, top_k=8)
    ok, keep = _tree(b, [-1, -1, 0, 0, 1, 2, 3], [0, 1, 0, 1, 0, 0, 0])
    small, keep2 = _tree(b, [-1, 0, 1], [0, 0, 0])
    n_ok = lib.cp_spec_workspace_bytes_tree(C.byref(m), C.byref(cfg), C.byref(ok))
    n_small = lib.cp_spec_workspace_bytes_tree(C.byref(m), C.byref(cfg), C.byref(small))
    assert n_ok > n_small > 0
    bad = [
        ([0], [0]),                                   # parent not earlier
        ([-1, -1], [1, 0]),                           # siblings out of rank order
        ([-1, -1], [0, 0]),                           # repeated rank
        ([-1, 0, 1, 2, 3, 4, 5, 6], [0] * 8),         # depth 8
        ([-1], [8]),                                  # rank at the list capacity (top-k 8)
        ([-1] * 63, list(range(63))),                 # 63 nodes
    ]
    for par, rk in bad:
        t, keep3 = _tree(b, par, rk)
        assert lib.cp_spec_workspace_bytes_tree(C.byref(m), C.byref(_cfg(b, top_k=256)) if len(par) == 63
                                                else C.byref(cfg), C.byref(t)) == 0, (par, rk)
    empty, keep4 = _tree(b, [], [])
    assert lib.cp_spec_workspace_bytes_tree(C.byref(m), C.byref(cfg), C.byref(empty)) == 0
