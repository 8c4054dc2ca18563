"""Seeded synthetic inputs for the CodePredictor speculative round.

This module only draws numbers: model weights, per-frame talker hiddens and
seed codes, and the logit tensors of the acceptance microbenchmark.  It holds
none of the method's arithmetic (no forward pass, no sampling, no acceptance)
and is shared, unchanged, by the CPU oracle tests and the CUDA path.

Every tensor is drawn from its own numpy ``PCG64`` stream keyed by
``SeedSequence([seed, tensor_id])`` so that any tensor (or any block of
microbenchmark rounds) can be regenerated on its own, in any order.

Shapes follow the CodePredictor structure of the pages: one input embedding
table and one lm_head per RVQ depth ("RVQ Position Aware Speculative Decoding
for On Device TTS", section 2.1), a dense pre-norm decoder with GQA attention,
RoPE and a SwiGLU FFN (the 5-layer MTP module of "Awesome-ML-SYS-Tutorial",
Qwen3-Omni section).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

DTYPE_F32 = 0
DTYPE_BF16 = 1


@dataclasses.dataclass(frozen=True)
class ModelSpec:
    """Decoder shape.  G = num_code_groups (codes c_0..c_{G-1})."""

    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    num_code_groups: int
    dtype: int  # DTYPE_F32 or DTYPE_BF16
    rope_theta: float = 10000.0
    rms_eps: float = 1e-6

    @property
    def n_heads_lm(self) -> int:
        """Number of lm_heads (head_1..head_{G-1}) = number of embedding tables."""
        return self.num_code_groups - 1

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == DTYPE_F32 else 2

    def layer_param_count(self) -> int:
        H, d = self.hidden, self.head_dim
        q = self.n_q_heads * d
        kv = self.n_kv_heads * d
        return q * H + 2 * kv * H + H * q + 3 * self.ffn * H

    def layer_weight_bytes(self) -> int:
        """Matrix bytes of one layer (norm gains excluded; they are fp32 vectors)."""
        return self.layer_param_count() * self.elem_bytes

    def head_bytes(self) -> int:
        return self.vocab * self.hidden * self.elem_bytes


# The workloads named by the benchmark description, by what they are.
TINY_FP32 = ModelSpec(hidden=256, n_layers=2, n_q_heads=4, n_kv_heads=4, head_dim=64,
                      ffn=768, vocab=256, num_code_groups=8, dtype=DTYPE_F32)
TTS06B_BF16 = ModelSpec(hidden=1024, n_layers=5, n_q_heads=16, n_kv_heads=8, head_dim=128,
                        ffn=3072, vocab=2048, num_code_groups=16, dtype=DTYPE_BF16)
LARGE_BF16 = ModelSpec(hidden=2048, n_layers=8, n_q_heads=32, n_kv_heads=8, head_dim=64,
                       ffn=6144, vocab=4096, num_code_groups=32, dtype=DTYPE_BF16)

WEIGHT_STD = 0.02


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); returns uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).ravel()
    out = np.empty(u.shape, np.uint16)
    step = 1 << 22
    for i in range(0, u.size, step):  # uint32 arithmetic cannot overflow for finite inputs
        c = u[i:i + step]
        r = (c >> np.uint32(16)) & np.uint32(1)
        r += c
        r += np.uint32(0x7FFF)
        r >>= np.uint32(16)
        out[i:i + step] = r
    return out.reshape(a.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id])))


def _normal(seed: int, tensor_id: int, shape, std: float) -> np.ndarray:
    g = _rng(seed, tensor_id)
    out = g.standard_normal(int(np.prod(shape)), dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out.reshape(shape)


# tensor ids: 0 embed, 1 lm_head, 2 final_norm, 3 draft offsets, then 16 + 16*layer + j
_T_EMBED, _T_HEAD = 0, 1


def _layer_tid(layer: int, j: int) -> int:
    return 16 + 16 * layer + j


def gen_weights(spec: ModelSpec, seed: int = 0, std: float = WEIGHT_STD) -> dict:
    """Weights N(0, 0.02) for every matrix; RMSNorm gains = 1.

    Returns a dict of numpy arrays in storage form: float32 for DTYPE_F32,
    uint16 bf16 bits for DTYPE_BF16.  Norm gains are always float32.
    Layouts (row-major): embed [G-1, V, H]; lm_head [G-1, V, H] (index d-1 is
    head_d); wq [nq*d, H]; wk, wv [nkv*d, H]; wo [H, nq*d]; w_gate, w_up [F, H];
    w_down [H, F].
    """
    H, V, Gm1 = spec.hidden, spec.vocab, spec.n_heads_lm
    qd, kvd, F = spec.n_q_heads * spec.head_dim, spec.n_kv_heads * spec.head_dim, spec.ffn

    def mat(tid, shape):
        a = _normal(seed, tid, shape, std)
        return a if spec.dtype == DTYPE_F32 else f32_to_bf16_bits(a)

    w = {
        "embed": mat(_T_EMBED, (Gm1, V, H)),
        "lm_head": mat(_T_HEAD, (Gm1, V, H)),
        "final_norm": np.ones(H, np.float32),
        "layers": [],
    }
    for l in range(spec.n_layers):
        w["layers"].append({
            "attn_norm": np.ones(H, np.float32),
            "wq": mat(_layer_tid(l, 0), (qd, H)),
            "wk": mat(_layer_tid(l, 1), (kvd, H)),
            "wv": mat(_layer_tid(l, 2), (kvd, H)),
            "wo": mat(_layer_tid(l, 3), (H, qd)),
            "ffn_norm": np.ones(H, np.float32),
            "w_gate": mat(_layer_tid(l, 4), (F, H)),
            "w_up": mat(_layer_tid(l, 5), (F, H)),
            "w_down": mat(_layer_tid(l, 6), (H, F)),
        })
    return w


_T_OFFSET = 3


def gen_draft_offsets(spec: ModelSpec, K: int, seed: int = 0, std: float = 0.25) -> np.ndarray:
    """K position-aware draft offset vectors b_1..b_K ~ N(0, std^2), [K, H] float32.

    The pages train these on speech data; synthetic runs draw them at random,
    which exercises the arithmetic without the acceptance gain."""
    return _normal(seed, _T_OFFSET, (K, spec.hidden), std)


def gen_frames(spec: ModelSpec, n_streams: int, n_frames: int, seed: int = 1,
               first_frame: int = 0):
    """Per-frame talker hidden x ~ N(0,1) [F, B, H] float32 and seed code c0 ~ U[0, V) [F, B] int32.

    Frame f of stream b is drawn from its own stream keyed by (seed, frame, b),
    so any subset of frames can be regenerated independently.
    """
    H, V = spec.hidden, spec.vocab
    x = np.empty((n_frames, n_streams, H), np.float32)
    c0 = np.empty((n_frames, n_streams), np.int32)
    for f in range(n_frames):
        for b in range(n_streams):
            g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1 << 20, first_frame + f, b])))
            x[f, b] = g.standard_normal(H, dtype=np.float32)
            c0[f, b] = int(g.integers(0, V))
    return x, c0


def gen_accept_block(R: int, N: int, V: int, rho: float, seed: int, block: int,
                     sigma: float = 3.0):
    """One block of acceptance-microbenchmark rounds.

    target logits ~ N(0, sigma^2) [R, N, V]; draft logits for position t
    (t = 1..N-1) = rho * target[t-1] + sqrt(1 - rho^2) * N(0, sigma^2), shape
    [R, N-1, V].  Row t-1 of the target scores the draft at position t.
    """
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 2 << 20, block, N, V])))
    tgt = g.standard_normal(R * N * V, dtype=np.float32).reshape(R, N, V)
    tgt *= np.float32(sigma)
    noise = g.standard_normal(R * (N - 1) * V, dtype=np.float32).reshape(R, N - 1, V)
    noise *= np.float32(sigma)
    drf = np.float32(rho) * tgt[:, : N - 1, :] + np.float32(math.sqrt(1.0 - rho * rho)) * noise
    return np.ascontiguousarray(tgt), np.ascontiguousarray(drf.astype(np.float32))


def gen_accept_inputs(R: int, N: int, V: int, rho: float, seed: int = 1, block_rounds: int = 1024,
                      sigma: float = 3.0):
    """Whole acceptance-microbenchmark input, as blocks of ``block_rounds`` rounds."""
    tgt = np.empty((R, N, V), np.float32)
    drf = np.empty((R, max(N - 1, 0), V), np.float32)
    for b0 in range(0, R, block_rounds):
        n = min(block_rounds, R - b0)
        t, d = gen_accept_block(block_rounds, N, V, rho, seed, b0 // block_rounds, sigma)
        tgt[b0:b0 + n] = t[:n]
        drf[b0:b0 + n] = d[:n]
    return tgt, drf
