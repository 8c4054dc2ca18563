"""Failure paths on the GPU, made on purpose without faulting anything.

- A bounded device wait that runs out: the test hook makes one wait of the
  first decoder kernel of a pass expect 16 bytes that no copy delivers (a
  barrier that nothing completes) and lowers the wait limit to 200 us.  The
  kernel records CP_SPEC_E_DEVICE_TIMEOUT, drains its own copies with the same
  bound and returns; the pass loop stops.  cp_spec_status_word reports the
  timeout and clears it, and the next call on the same context, with the hook
  off, decodes exactly like a fresh context.  Both GEMV paths: CUDA cores
  (fp32 weights) and the small-batch tensor path (bf16, one stream).
- The shared-memory limits the library sets on its kernels only ever grow:
  a context built for more streams keeps working (same codes) after an
  allocation-free call configured for fewer streams.
- The allocation-free entry point accepts a status slot at a 4-byte offset."""
import dataclasses

import numpy as np
import pytest

from gpu_common import require_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _setup(which):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    if which == "fp32":
        spec = S.TINY_FP32
    else:
        spec = dataclasses.replace(S.TTS06B_BF16, n_layers=2)
    w = S.gen_weights(spec, 0)
    return spec, binding.weights_to_device(spec, w)


@pytest.mark.parametrize("which", ["fp32", "bf16"])
def test_device_wait_timeout_is_reported_and_recoverable(which):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec, dw = _setup(which)
    x, c0 = S.gen_frames(spec, 1, 2, seed=31)
    xd, cd = torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()
    ref_cp = binding.CpSpec(spec, dw, 4, 50, 0.9, 5, max_streams=1)
    ref = ref_cp.decode_frames(xd, cd).cpu().numpy()
    ref_cp.status()
    cp = binding.CpSpec(spec, dw, 4, 50, 0.9, 5, max_streams=1)
    cp.test_hooks(wait_limit_ns=200_000, stall_first_wait=True)
    cp.decode_frames(xd, cd)
    torch.cuda.synchronize()
    assert cp.status_code() == binding.E_DEVICE_TIMEOUT
    assert cp.status_code() == binding.OK  # the read cleared the word
    cp.test_hooks(wait_limit_ns=2_000_000_000, stall_first_wait=False)
    got = cp.decode_frames(xd, cd).cpu().numpy()
    cp.status()
    assert np.array_equal(got, ref)


def test_test_hook_rejects_bad_arguments():
    from speculative_decoding_rvq_gb300 import binding
    spec, dw = _setup("fp32")
    cp = binding.CpSpec(spec, dw, 4, 50, 0.9, 5, max_streams=1)
    for ns, st in ((100, 0), (2_000_000_000, 4), (2_000_000_000, -1)):
        assert cp.lib.cp_spec_test_hooks(cp.ctx, ns, st) == binding.E_INVALID


@pytest.mark.parametrize("which", ["fp32", "bf16"])
def test_context_survives_smaller_allocation_free_call(which):
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec, dw = _setup(which)
    B = 8 if which == "fp32" else 2
    x, c0 = S.gen_frames(spec, B, 2, seed=32)
    xd, cd = torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()
    cp = binding.CpSpec(spec, dw, 4, 50, 0.9, 9, max_streams=B)
    first = cp.decode_frames(xd, cd).cpu().numpy()
    cp.status()
    # an allocation-free call configured for one stream (smaller kernel shared memory)
    xs, cs = xd[:, :1].contiguous(), cd[:, :1].contiguous()
    _, rc = binding.decode_frames_static(spec, dw, 4, 50, 0.9, 9, xs, cs, max_streams=1)
    torch.cuda.synchronize()
    assert rc == binding.OK
    again = cp.decode_frames(xd, cd).cpu().numpy()
    cp.status()
    assert np.array_equal(again, first)


def test_static_status_slot_at_four_byte_offset():
    from speculative_decoding_rvq_gb300 import binding, synth as S
    spec, dw = _setup("fp32")
    x, c0 = S.gen_frames(spec, 1, 1, seed=33)
    xd, cd = torch.from_numpy(x).cuda(), torch.from_numpy(c0).cuda()
    status = torch.full((4,), 77, dtype=torch.int32, device="cuda")
    _, rc = binding.decode_frames_static(spec, dw, 4, 50, 0.9, 3, xd, cd, max_streams=1, status=status[1:])
    torch.cuda.synchronize()
    assert rc == binding.OK
    assert status.cpu().tolist() == [77, binding.OK, 77, 77]
