"""cp_spec_decode_frames_static (decode in the library's static scratch, no
context, no caller workspace) against cp_spec_decode_frames on a fresh
context.

Both run the same frame kernel with the same parameters and starting state,
so the codes must be identical (exact integer equality), on each of two calls
in a row with different inputs.  The size check runs on the host and needs no
GPU.  This file is named to be collected last: the static path must also work
after other tests have loaded the library and used the device."""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _lib():
    from speculative_decoding_rvq_gb300 import binding, build
    build.build()
    return binding.load()


def test_static_rejects_scratch_above_maximum():
    from speculative_decoding_rvq_gb300 import binding as b, synth as S
    lib = _lib()
    spec = S.TTS06B_BF16
    m = b.model_struct(spec)
    w = b.Weights()
    w.embed = w.lm_head = w.final_norm = 4096
    for l in range(spec.n_layers):
        for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down"):
            getattr(w, n)[l] = 4096
    big = b.Config(4, 50, 0.9, 1, 64)
    need = lib.cp_spec_workspace_bytes(C.byref(m), C.byref(big))
    assert need > (8 << 20)
    rc = lib.cp_spec_decode_frames_static(C.byref(m), C.byref(w), C.byref(big), 1, 1, 0, 16, 16, 16, None, None)
    assert rc == b.E_WORKSPACE
    assert b"static maximum" in lib.cp_spec_last_error(None)
    # one stream of the same model fits
    assert lib.cp_spec_workspace_bytes(C.byref(m), C.byref(b.Config(4, 50, 0.9, 1, 1))) <= (8 << 20)
    # the boundary: 9 streams fit, 10 do not (the size is checked before any device work, so
    # zero frames return at once)
    nine, ten = b.Config(4, 50, 0.9, 1, 9), b.Config(4, 50, 0.9, 1, 10)
    assert (lib.cp_spec_workspace_bytes(C.byref(m), C.byref(nine)) <= (8 << 20)
            < lib.cp_spec_workspace_bytes(C.byref(m), C.byref(ten)))
    assert lib.cp_spec_decode_frames_static(C.byref(m), C.byref(w), C.byref(nine), 9, 0, 0, 16, 16, 16, None,
                                            None) == b.OK
    assert lib.cp_spec_decode_frames_static(C.byref(m), C.byref(w), C.byref(ten), 10, 0, 0, 16, 16, 16, None,
                                            None) == b.E_WORKSPACE


def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib()


@pytest.mark.gpu
@pytest.mark.parametrize("which", ["tiny_fp32_3streams", "bf16_0p6b_1stream", "tiny_fp32_offsets"])
def test_static_matches_context_decode_twice(which):
    _gpu()
    from speculative_decoding_rvq_gb300 import binding, synth as S
    if which == "bf16_0p6b_1stream":
        spec, B, F, N, k, T = S.TTS06B_BF16, 1, 4, 4, 50, 0.9
    else:
        spec, B, F, N, k, T = S.TINY_FP32, 3, 6, 3, 20, 0.9
    w = S.gen_weights(spec, 0)
    if which == "tiny_fp32_offsets":  # position-aware draft offsets: the static call forms head . b itself
        w["draft_offset"] = S.gen_draft_offsets(spec, 3, seed=1, std=1.0)
    dw = binding.weights_to_device(spec, w)
    status = torch.full((4,), 123, dtype=torch.int32, device="cuda")
    for call, (seed, first) in enumerate(((11, 0), (12, F))):
        x, c0 = S.gen_frames(spec, B, F, seed=seed)
        xd, cd = torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()
        cp = binding.CpSpec(spec, dw, N, k, T, 7, max_streams=B)
        want = cp.decode_frames(xd, cd, first_frame=first)
        torch.cuda.synchronize()
        cp.status()
        cp.close()
        got, rc = binding.decode_frames_static(spec, dw, N, k, T, 7, xd, cd, first_frame=first, status=status)
        torch.cuda.synchronize()
        assert rc == binding.OK
        assert int(status[0].item()) == binding.OK, call
        g, w = got.cpu().numpy(), want.cpu().numpy()
        np.testing.assert_array_equal(g, w, err_msg=f"call {call}")
        assert (g[:, :, 0] == c0).all()
        assert ((g >= 0) & (g < spec.vocab)).all()
