"""ctypes wrapper of the CPU oracle (cp_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``.  The CUDA library never loads
or calls anything here.  Arrays in, arrays out; every computation happens in
the C file, which is compiled with gcc on first use.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libcp_oracle.so")
_lock = threading.Lock()
_lib = None

ORC_DRAFT, ORC_ACCEPT, ORC_TARGET, ORC_INPUT = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile cp_oracle.c into a shared library (plain gcc, no fast-math, no FMA contraction)."""
    src = os.path.join(_HERE, "cp_oracle.c")
    hdr = os.path.join(_HERE, "cp_oracle.h")
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(src), os.path.getmtime(hdr))
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-Wall", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


class OrcModel(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("H", "L", "nq", "nkv", "d", "F", "V", "G")] + [
        ("theta", C.c_double), ("eps", C.c_double)] + [
        (n, C.c_void_p) for n in ("embed", "head", "final_norm", "attn_norm", "wq", "wk", "wv", "wo",
                                  "ffn_norm", "w_gate", "w_up", "w_down")] + [
        ("K", C.c_int), ("draft_offset", C.c_void_p)]


class OrcTree(C.Structure):
    _fields_ = [("n", C.c_int), ("parent", C.c_void_p), ("rank", C.c_void_p)]


class OrcStats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("frames", "passes", "rounds", "committed", "bonus", "rejections")] + [
        ("drafted_by_offset", C.c_int64 * 9), ("accepted_by_offset", C.c_int64 * 9)]

    def as_dict(self) -> dict:
        d = {n: int(getattr(self, n)) for n in ("frames", "passes", "rounds", "committed", "bonus", "rejections")}
        d["drafted_by_offset"] = [int(v) for v in self.drafted_by_offset]
        d["accepted_by_offset"] = [int(v) for v in self.accepted_by_offset]
        return d


ROUND_DTYPE = np.dtype([("frame", "<i4"), ("stream", "<i4"), ("s", "<i4"), ("n_d", "<i4"), ("m", "<i4"),
                        ("n_acc", "<i4"), ("s_new", "<i4"), ("pad", "<i4"), ("drafts", "<i4", (8,)),
                        ("min_margin", "<f8")])


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            vp, i32, f32, u64 = C.c_void_p, C.c_int, C.c_float, C.c_uint64
            L.orc_philox4x32_10.argtypes = [vp, vp, vp]
            L.orc_uniform.argtypes = [u64, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint32]
            L.orc_uniform.restype = f32
            L.orc_uniform_fill.argtypes = [u64, i32, vp, vp]
            L.orc_process.argtypes = [vp, i32, i32, f32, vp, vp]
            L.orc_sample.argtypes = [vp, i32, f32, vp]
            L.orc_sample.restype = i32
            L.orc_accept_chain.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
            L.orc_accept_chain.restype = i32
            L.orc_accept_batch.argtypes = [i32, i32, i32, i32, f32, u64, i32, vp, vp, vp, vp, vp, vp]
            L.orc_kv_doubles.argtypes = [vp]
            L.orc_kv_doubles.restype = C.c_size_t
            L.orc_forward.argtypes = [vp, vp, i32, vp, vp, vp]
            L.orc_head_logits.argtypes = [vp, i32, vp, vp, vp]
            L.orc_draft_logits.argtypes = [vp, i32, i32, vp, vp]
            L.orc_teacher_logits.argtypes = [vp, vp, vp, i32, i32, vp, vp]
            L.orc_decode_frames.argtypes = [vp, i32, vp, vp, u64, i32, i32, i32, vp, vp, vp, vp, vp, i32, vp]
            L.orc_decode_frames.restype = i32
            L.orc_decode_frames_policy.argtypes = [vp, i32, vp, vp, u64, i32, i32, i32, vp, vp, vp, vp, vp, i32, vp,
                                                   i32, i32]
            L.orc_decode_frames_policy.restype = i32
            L.orc_decode_frames_tree.argtypes = [vp, vp, vp, vp, u64, i32, i32, i32, vp, vp, vp, vp, vp, i32, vp]
            L.orc_decode_frames_tree.restype = i32
            L.orc_policy_window.argtypes = [i32, i32, i32, vp, vp]
            L.orc_policy_window.restype = i32
            _lib = L
    return _lib


# ------------------------------------------------------------------ RNG
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def uniform(seed: int, stream: int, frame: int, depth: int, purpose: int) -> float:
    return float(lib().orc_uniform(seed, stream, frame, depth, purpose))


def uniforms(seed: int, ctr4: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(ctr4, dtype=np.uint32).reshape(-1, 4)
    out = np.empty(len(c), np.float32)
    lib().orc_uniform_fill(seed, len(c), _p(c), _p(out))
    return out


# ------------------------------------------------------------ sampling
def process(logits, top_k: int, temperature: float):
    z = np.ascontiguousarray(logits, dtype=np.float32)
    out = np.empty_like(z)
    mg = C.c_double(0.0)
    lib().orc_process(_p(z), z.size, int(top_k), float(temperature), _p(out), C.byref(mg))
    return out, mg.value


def sample(w, u: float):
    a = np.ascontiguousarray(w, dtype=np.float32)
    mg = C.c_double(0.0)
    r = lib().orc_sample(_p(a), a.size, float(u), C.byref(mg))
    return int(r), mg.value


def accept_chain(q, drafts, p, u_acc, u_tgt):
    """q [n_d, V], p [m, V], drafts [n_d], u_acc [n_d], u_tgt [n_d + 1] -> (n_acc, emitted list, margin)."""
    q = np.ascontiguousarray(q, dtype=np.float32).reshape(-1, np.shape(p)[-1])
    p = np.ascontiguousarray(p, dtype=np.float32)
    V = p.shape[-1]
    n_d = len(drafts)
    q = q[:n_d]
    m = p.shape[0]
    if not (m == n_d or m == n_d + 1):
        raise ValueError("target rows must score every draft position (plus at most one bonus row)")
    dr = np.ascontiguousarray(drafts, dtype=np.int32)
    ua = np.ascontiguousarray(u_acc, dtype=np.float32)
    ut = np.ascontiguousarray(u_tgt, dtype=np.float32)
    if ua.size < max(n_d, 1):
        ua = np.resize(ua, max(n_d, 1))
    if ut.size < n_d + 1:
        ut = np.resize(ut, n_d + 1)
    em = np.full(n_d + 1, -1, np.int32)
    ne = C.c_int(0)
    mg = C.c_double(0.0)
    na = lib().orc_accept_chain(V, n_d, m, _p(q), _p(dr), _p(p), _p(ua), _p(ut), _p(em), C.byref(ne), C.byref(mg))
    return int(na), [int(v) for v in em[: ne.value]], mg.value


def accept_batch(target, draft, top_k: int, temperature: float, seed: int, mode: int = 0):
    """Acceptance microbenchmark rounds.  Returns tokens [R, N] (-1 padded), n_acc [R], drafts [R, N-1], margins [R]."""
    t = np.ascontiguousarray(target, dtype=np.float32)
    R, N, V = t.shape
    d = np.ascontiguousarray(draft, dtype=np.float32).reshape(R, N - 1, V)
    tok = np.empty((R, N), np.int32)
    na = np.empty(R, np.int32)
    dr = np.empty((R, max(N - 1, 1)), np.int32)
    mg = np.empty(R, np.float64)
    lib().orc_accept_batch(R, N, V, int(top_k), float(temperature), int(seed), int(mode), _p(t), _p(d),
                           _p(tok), _p(na), _p(dr), _p(mg))
    return tok, na, dr[:, : N - 1], mg


# --------------------------------------------------------------- model
class Model:
    """Holds float32 copies of the weights and the C model struct."""

    def __init__(self, spec, weights: dict):
        from speculative_decoding_rvq_gb300.synth import bf16_bits_to_f32

        def f32(a):
            a = np.asarray(a)
            if a.dtype == np.uint16:
                return np.ascontiguousarray(bf16_bits_to_f32(a))
            return np.ascontiguousarray(a, dtype=np.float32)

        self.spec = spec
        L = weights["layers"]
        self._arrs = {
            "embed": f32(weights["embed"]),
            "head": f32(weights["lm_head"]),
            "final_norm": f32(weights["final_norm"]),
            "attn_norm": np.ascontiguousarray(np.stack([f32(l["attn_norm"]) for l in L])),
            "wq": np.ascontiguousarray(np.stack([f32(l["wq"]) for l in L])),
            "wk": np.ascontiguousarray(np.stack([f32(l["wk"]) for l in L])),
            "wv": np.ascontiguousarray(np.stack([f32(l["wv"]) for l in L])),
            "wo": np.ascontiguousarray(np.stack([f32(l["wo"]) for l in L])),
            "ffn_norm": np.ascontiguousarray(np.stack([f32(l["ffn_norm"]) for l in L])),
            "w_gate": np.ascontiguousarray(np.stack([f32(l["w_gate"]) for l in L])),
            "w_up": np.ascontiguousarray(np.stack([f32(l["w_up"]) for l in L])),
            "w_down": np.ascontiguousarray(np.stack([f32(l["w_down"]) for l in L])),
        }
        # optional position-aware draft offsets b_1..b_K [K, H] float32
        off = weights.get("draft_offset")
        K = 0
        if off is not None and np.asarray(off).shape[0] > 0:
            self._arrs["draft_offset"] = np.ascontiguousarray(off, dtype=np.float32).reshape(-1, spec.hidden)
            K = self._arrs["draft_offset"].shape[0]
        s = spec
        self.K = K
        self.c = OrcModel(H=s.hidden, L=s.n_layers, nq=s.n_q_heads, nkv=s.n_kv_heads, d=s.head_dim,
                          F=s.ffn, V=s.vocab, G=s.num_code_groups, theta=s.rope_theta, eps=s.rms_eps, K=K,
                          **{k: v.ctypes.data for k, v in self._arrs.items()})

    @property
    def ptr(self):
        return C.byref(self.c)

    def arrays(self) -> dict:
        return self._arrs

    def new_kv(self) -> np.ndarray:
        return np.zeros(lib().orc_kv_doubles(self.ptr), np.float64)

    def forward(self, kv: np.ndarray, rows: np.ndarray, positions) -> np.ndarray:
        rows = np.ascontiguousarray(rows, dtype=np.float64).reshape(-1, self.spec.hidden)
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        out = np.empty_like(rows)
        lib().orc_forward(self.ptr, _p(kv), rows.shape[0], _p(rows), _p(pos), _p(out))
        return out

    def head_logits(self, j: int, hn: np.ndarray):
        hn = np.ascontiguousarray(hn, dtype=np.float64)
        o64 = np.empty(self.spec.vocab, np.float64)
        o32 = np.empty(self.spec.vocab, np.float32)
        lib().orc_head_logits(self.ptr, int(j), _p(hn), _p(o64), _p(o32))
        return o64, o32

    def decode_frames_tree(self, parent, rank, top_k, temperature, seed: int, x: np.ndarray, c0: np.ndarray,
                           first_frame: int = 0, log_cap: int = 0):
        """Tree rounds (orc_decode_frames_tree): parent / rank per node, parents first."""
        F, B, H = x.shape
        par = np.ascontiguousarray(parent, dtype=np.int32)
        rk = np.ascontiguousarray(rank, dtype=np.int32)
        tree = OrcTree(int(par.size), par.ctypes.data, rk.ctypes.data)
        tk = np.ascontiguousarray(np.broadcast_to(np.asarray(top_k, np.int32), (B,)))
        tp = np.ascontiguousarray(np.broadcast_to(np.asarray(temperature, np.float32), (B,)))
        xx = np.ascontiguousarray(x, dtype=np.float32)
        cc = np.ascontiguousarray(c0, dtype=np.int32)
        codes = np.zeros((F, B, self.spec.num_code_groups), np.int32)
        st = OrcStats()
        log = np.zeros(max(log_cap, 1), ROUND_DTYPE)
        nlog = C.c_int(0)
        rc = lib().orc_decode_frames_tree(self.ptr, C.byref(tree), _p(tk), _p(tp), int(seed), B, F,
                                          int(first_frame), _p(xx), _p(cc), _p(codes), C.byref(st), _p(log),
                                          int(log_cap), C.byref(nlog))
        if rc != 0:
            raise ValueError("oracle rejected the tree decode arguments")
        return codes, st.as_dict(), log[: min(nlog.value, log_cap)]

    @staticmethod
    def policy_window(N: int, pct: int, min_reached: int, reach, acc) -> int:
        r = np.ascontiguousarray(reach, dtype=np.int64)
        a = np.ascontiguousarray(acc, dtype=np.int64)
        assert r.shape == (9,) and a.shape == (9,)
        return int(lib().orc_policy_window(int(N), int(pct), int(min_reached), _p(r), _p(a)))

    def draft_logits(self, j: int, t: int, hn: np.ndarray) -> np.ndarray:
        """float32 draft logits of lookahead t read by head_j from the normed hidden hn."""
        hn = np.ascontiguousarray(hn, dtype=np.float64)
        o32 = np.empty(self.spec.vocab, np.float32)
        lib().orc_draft_logits(self.ptr, int(j), int(t), _p(hn), _p(o32))
        return o32

    def input_row(self, x, pos: int, code: int) -> np.ndarray:
        if pos == 0:
            return np.asarray(x, np.float64)
        return self._arrs["embed"][pos - 1, code].astype(np.float64)

    def teacher_logits(self, x, codes, P: int, n_draft: int = 0):
        V = self.spec.vocab
        xx = np.ascontiguousarray(x, dtype=np.float32)
        cc = np.ascontiguousarray(codes, dtype=np.int32)
        lg = np.empty((P - 1, V), np.float32)
        dr = np.empty((P - 1, max(n_draft, 1), V), np.float32)
        lib().orc_teacher_logits(self.ptr, _p(xx), _p(cc), int(P), int(n_draft), _p(lg),
                                 _p(dr) if n_draft > 0 else None)
        return lg, (dr if n_draft > 0 else None)

    def decode_frames(self, N: int, top_k, temperature, seed: int, x: np.ndarray, c0: np.ndarray,
                      first_frame: int = 0, log_cap: int = 0, adapt_pct: int = 0, adapt_min: int = 16):
        """x [F, B, H], c0 [F, B] -> codes [F, B, G], stats dict, round log (structured array).

        adapt_pct > 0 turns on the per-stream adaptive window (orc_policy_window)."""
        F, B, H = x.shape
        tk = np.ascontiguousarray(np.broadcast_to(np.asarray(top_k, np.int32), (B,)))
        tp = np.ascontiguousarray(np.broadcast_to(np.asarray(temperature, np.float32), (B,)))
        xx = np.ascontiguousarray(x, dtype=np.float32)
        cc = np.ascontiguousarray(c0, dtype=np.int32)
        codes = np.zeros((F, B, self.spec.num_code_groups), np.int32)
        st = OrcStats()
        log = np.zeros(max(log_cap, 1), ROUND_DTYPE)
        nlog = C.c_int(0)
        rc = lib().orc_decode_frames_policy(self.ptr, int(N), _p(tk), _p(tp), int(seed), B, F, int(first_frame),
                                            _p(xx), _p(cc), _p(codes), C.byref(st), _p(log), int(log_cap),
                                            C.byref(nlog), int(adapt_pct), int(adapt_min))
        if rc != 0:
            raise ValueError("oracle rejected the decode arguments")
        return codes, st.as_dict(), log[: min(nlog.value, log_cap)]
