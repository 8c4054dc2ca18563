"""Shared helpers of the GPU parity tests (test infrastructure)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_rvq_gb300 import build
    build.build()


def compare_codes_with_margins(gpu_codes, orc_codes, orc_log, margin_tol, max_frac=0.05):
    """Frame-by-frame code equality.  A frame whose first differing code was decided
    in an oracle round with a decision margin below ``margin_tol`` (a near-tie that the
    float64 vs float32 accumulation order may flip) is tolerated; any other difference
    fails.  Returns the number of tolerated frames."""
    F, B, G = orc_codes.shape
    tolerated = 0
    for f in range(F):
        for b in range(B):
            g, o = gpu_codes[f, b], orc_codes[f, b]
            if np.array_equal(g, o):
                continue
            j = int(np.flatnonzero(g != o)[0])
            recs = orc_log[(orc_log["frame"] == f) & (orc_log["stream"] == b)]
            hit = recs[(recs["s"] < j) & (recs["s_new"] >= j)]
            assert len(hit) == 1, (f, b, j)
            assert hit["min_margin"][0] < margin_tol, (f, b, j, g.tolist(), o.tolist(), float(hit["min_margin"][0]))
            tolerated += 1
    assert tolerated <= max(1, int(max_frac * F * B)), tolerated
    return tolerated
