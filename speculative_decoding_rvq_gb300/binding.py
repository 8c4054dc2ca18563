"""Thin ctypes binding of the C ABI in include/cp_spec.h.

Argument marshalling only: every step of the decode runs in the CUDA
library.  PyTorch provides device memory and the current CUDA stream.  If the
library is missing or cannot be loaded this module raises; there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcpspec.so")
MAX_LAYERS = 64

OK, W_AR_FALLBACK = 0, 1
E_INVALID, E_UNSUPPORTED, E_CUDA, E_WORKSPACE, E_DEVICE_TIMEOUT, E_STATE, E_DEVICE = -1, -2, -3, -4, -5, -6, -7

# Every symbol include/cp_spec.h declares.
EXPORTS = ("cp_spec_workspace_bytes", "cp_spec_init", "cp_spec_set_stream_sampling", "cp_spec_decode_frames",
           "cp_spec_begin_frame", "cp_spec_round", "cp_spec_teacher_logits", "cp_spec_accept_batch",
           "cp_spec_status_word", "cp_spec_read_stats", "cp_spec_reset_stats", "cp_spec_launch_count",
           "cp_spec_last_error", "cp_spec_destroy", "cp_spec_decode_frames_static", "cp_spec_test_hooks",
           "cp_spec_workspace_bytes_tree", "cp_spec_init_tree")


class CpSpecError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"cp_spec status {code}: {msg}")
        self.code = code


class Model(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
                                         "num_code_groups", "dtype")] + [("rope_theta", C.c_float),
                                                                          ("rms_eps", C.c_float)]


class Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p)] + [
        (n, C.c_void_p * MAX_LAYERS) for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up",
                                               "w_down")] + [("draft_offset", C.c_void_p)]


class Config(C.Structure):
    _fields_ = [("verify_window", C.c_int32), ("top_k", C.c_int32), ("temperature", C.c_float),
                ("seed", C.c_uint64), ("max_streams", C.c_int32), ("draft_offsets", C.c_int32),
                ("adapt_accept_pct", C.c_int32), ("adapt_min_reached", C.c_int32)]


class Tree(C.Structure):
    _fields_ = [("n", C.c_int32), ("parent", C.c_void_p), ("rank", C.c_void_p)]


class Stats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("frames", "passes", "rounds", "committed", "bonus", "rejections")] + [
        ("drafted_by_offset", C.c_int64 * 9), ("accepted_by_offset", C.c_int64 * 9)] + [
        (n, C.c_int64) for n in ("weight_bytes", "kv_bytes", "heads_applied", "kernel_launches")] + [("reserved", C.c_int64 * 7)]

    def as_dict(self) -> dict:
        d = {n: int(getattr(self, n)) for n, _ in self._fields_ if not n.endswith("_offset") and n != "reserved"}
        d["drafted_by_offset"] = [int(v) for v in self.drafted_by_offset]
        d["accepted_by_offset"] = [int(v) for v in self.accepted_by_offset]
        return d


_lib = None


def load():
    """Load libcpspec.so (raises if it is missing: the path has no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} (run __graft_entry__.build())")
    L = C.CDLL(LIB_PATH)
    vp, i32, f32, u64, sz = C.c_void_p, C.c_int32, C.c_float, C.c_uint64, C.c_size_t
    L.cp_spec_workspace_bytes.argtypes = [vp, vp]
    L.cp_spec_workspace_bytes.restype = sz
    L.cp_spec_init.argtypes = [vp, vp, vp, vp, sz, C.POINTER(vp)]
    L.cp_spec_workspace_bytes_tree.argtypes = [vp, vp, vp]
    L.cp_spec_workspace_bytes_tree.restype = sz
    L.cp_spec_init_tree.argtypes = [vp, vp, vp, vp, vp, sz, C.POINTER(vp)]
    L.cp_spec_set_stream_sampling.argtypes = [vp, i32, vp, vp]
    L.cp_spec_decode_frames.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
    L.cp_spec_begin_frame.argtypes = [vp, i32, vp, vp, i32, vp]
    L.cp_spec_round.argtypes = [vp, vp, vp, vp]
    L.cp_spec_teacher_logits.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp]
    L.cp_spec_accept_batch.argtypes = [i32, i32, i32, i32, f32, u64, i32, vp, vp, vp, vp, vp, vp]
    L.cp_spec_decode_frames_static.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp]
    L.cp_spec_status_word.argtypes = [vp, vp]
    L.cp_spec_test_hooks.argtypes = [vp, u64, i32]
    L.cp_spec_read_stats.argtypes = [vp, vp, vp]
    L.cp_spec_reset_stats.argtypes = [vp, vp]
    L.cp_spec_launch_count.argtypes = [vp]
    L.cp_spec_launch_count.restype = C.c_int64
    L.cp_spec_last_error.argtypes = [vp]
    L.cp_spec_last_error.restype = C.c_char_p
    L.cp_spec_destroy.argtypes = [vp]
    L.cp_spec_destroy.restype = None
    for name in ("cp_spec_init", "cp_spec_init_tree", "cp_spec_set_stream_sampling", "cp_spec_decode_frames", "cp_spec_begin_frame",
                 "cp_spec_round", "cp_spec_teacher_logits", "cp_spec_accept_batch", "cp_spec_status_word",
                 "cp_spec_read_stats", "cp_spec_reset_stats", "cp_spec_decode_frames_static", "cp_spec_test_hooks"):
        getattr(L, name).restype = C.c_int
    _lib = L
    return L


def _check(rc: int, ctx=None, allow=(OK,)):
    if rc in allow:
        return rc
    msg = load().cp_spec_last_error(ctx).decode(errors="replace")
    raise CpSpecError(rc, msg)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream():
    import torch
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def model_struct(spec: synth.ModelSpec) -> Model:
    return Model(spec.hidden, spec.n_layers, spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.ffn, spec.vocab,
                 spec.num_code_groups, spec.dtype, spec.rope_theta, spec.rms_eps)


def weights_to_device(spec: synth.ModelSpec, w: dict, device="cuda") -> dict:
    """Copy numpy weights (float32, or uint16 bf16 bits) to device tensors of the storage dtype."""
    import torch

    def dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(a).to(device)

    out = {k: dev(w[k]) for k in ("embed", "lm_head", "final_norm")}
    out["layers"] = [{k: dev(v) for k, v in lw.items()} for lw in w["layers"]]
    if w.get("draft_offset") is not None and len(w["draft_offset"]) > 0:
        out["draft_offset"] = dev(np.asarray(w["draft_offset"], np.float32).reshape(-1, spec.hidden))
    return out


def n_draft_offsets(dw: dict) -> int:
    """K of the position-aware draft offsets held in device weights (0 if none)."""
    off = dw.get("draft_offset")
    return 0 if off is None else int(off.shape[0])


def weights_struct(dw: dict) -> Weights:
    ws = Weights()
    ws.embed, ws.lm_head, ws.final_norm = _ptr(dw["embed"]), _ptr(dw["lm_head"]), _ptr(dw["final_norm"])
    for l, lw in enumerate(dw["layers"]):
        for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down"):
            getattr(ws, n)[l] = _ptr(lw[n])
    ws.draft_offset = _ptr(dw.get("draft_offset"))
    return ws


class CpSpec:
    """One context of the CUDA library over device-resident weights."""

    def __init__(self, spec: synth.ModelSpec, device_weights: dict, verify_window: int, top_k: int,
                 temperature: float, seed: int, max_streams: int = 1, adapt_pct: int = 0, adapt_min: int = 16,
                 tree=None):
        """tree: None (chain rounds of verify_window), or (parent, rank) sequences of a sparse
        draft tree (cp_spec_init_tree; verify_window and the adaptive window are then ignored)."""
        import numpy as np
        import torch
        self.lib = load()
        self.spec = spec
        self.dw = device_weights
        self.model = model_struct(spec)
        self.weights = weights_struct(device_weights)
        self.config = Config(verify_window, top_k, temperature, seed, max_streams, n_draft_offsets(device_weights),
                             adapt_pct, adapt_min)
        self.tree = None
        if tree is not None:
            par = np.ascontiguousarray(tree[0], dtype=np.int32)
            rk = np.ascontiguousarray(tree[1], dtype=np.int32)
            self._tree_arrays = (par, rk)  # kept alive for the call
            self.tree = Tree(len(par), par.ctypes.data, rk.ctypes.data)
            nbytes = self.lib.cp_spec_workspace_bytes_tree(C.byref(self.model), C.byref(self.config),
                                                           C.byref(self.tree))
        else:
            nbytes = self.lib.cp_spec_workspace_bytes(C.byref(self.model), C.byref(self.config))
        if nbytes == 0:
            _check(E_INVALID)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        ctx = C.c_void_p()
        if self.tree is not None:
            rc = self.lib.cp_spec_init_tree(C.byref(self.model), C.byref(self.weights), C.byref(self.config),
                                            C.byref(self.tree), C.c_void_p(_ptr(self.workspace)), nbytes,
                                            C.byref(ctx))
        else:
            rc = self.lib.cp_spec_init(C.byref(self.model), C.byref(self.weights), C.byref(self.config),
                                       C.c_void_p(_ptr(self.workspace)), nbytes, C.byref(ctx))
        _check(rc, None, allow=(OK, W_AR_FALLBACK))
        self.ar_fallback = rc == W_AR_FALLBACK
        self.ctx = ctx

    def close(self):
        if getattr(self, "ctx", None):
            self.lib.cp_spec_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_stream_sampling(self, top_k, temperature):
        tk = np.ascontiguousarray(top_k, dtype=np.int32)
        tp = np.ascontiguousarray(temperature, dtype=np.float32)
        _check(self.lib.cp_spec_set_stream_sampling(self.ctx, tk.size, tk.ctypes.data_as(C.c_void_p),
                                                    tp.ctypes.data_as(C.c_void_p)), self.ctx)

    def decode_frames(self, x, c0, codes=None, first_frame: int = 0):
        """x [F, B, H] float32 cuda, c0 [F, B] int32 cuda -> codes [F, B, G] int32 (asynchronous)."""
        import torch
        F, B, _ = x.shape
        if codes is None:
            codes = torch.empty((F, B, self.spec.num_code_groups), dtype=torch.int32, device=x.device)
        _check(self.lib.cp_spec_decode_frames(self.ctx, B, F, first_frame, _ptr(x), _ptr(c0), _ptr(codes), _stream()),
               self.ctx)
        return codes

    def begin_frame(self, x, c0, frame_idx: int):
        _check(self.lib.cp_spec_begin_frame(self.ctx, x.shape[0], _ptr(x), _ptr(c0), frame_idx, _stream()), self.ctx)

    def round(self, codes, committed=None):
        _check(self.lib.cp_spec_round(self.ctx, _ptr(codes), _ptr(committed), _stream()), self.ctx)

    def teacher_logits(self, x, codes, P: int, draft: bool = False):
        import torch
        B = x.shape[0]
        V = self.spec.vocab
        lg = torch.empty((B, P - 1, V), dtype=torch.float32, device=x.device)
        nd = self.config.verify_window - 1
        dl = torch.empty((B, P - 1, nd, V), dtype=torch.float32, device=x.device) if draft else None
        _check(self.lib.cp_spec_teacher_logits(self.ctx, B, P, _ptr(x), _ptr(codes), _ptr(lg), _ptr(dl), _stream()),
               self.ctx)
        return lg, dl

    def status(self):
        _check(self.lib.cp_spec_status_word(self.ctx, _stream()), self.ctx)

    def status_code(self) -> int:
        """cp_spec_status_word as a code (clears the word)."""
        return int(self.lib.cp_spec_status_word(self.ctx, _stream()))

    def test_hooks(self, wait_limit_ns: int = 2_000_000_000, stall_first_wait: bool = False, poison_kv: bool = False):
        flags = (1 if stall_first_wait else 0) | (2 if poison_kv else 0)
        _check(self.lib.cp_spec_test_hooks(self.ctx, int(wait_limit_ns), flags), self.ctx)

    def stats(self) -> dict:
        st = Stats()
        _check(self.lib.cp_spec_read_stats(self.ctx, C.byref(st), _stream()), self.ctx)
        return st.as_dict()

    def reset_stats(self):
        _check(self.lib.cp_spec_reset_stats(self.ctx, _stream()), self.ctx)

    def launch_count(self) -> int:
        return int(self.lib.cp_spec_launch_count(self.ctx))


def accept_batch(target, draft, top_k: int, temperature: float, seed: int, mode: int = 0, want_drafts=True):
    """Acceptance kernels alone.  target [R, N, V], draft [R, N-1, V] float32 cuda tensors."""
    import torch
    lib = load()
    R, N, V = target.shape
    tok = torch.empty((R, N), dtype=torch.int32, device=target.device)
    na = torch.empty((R,), dtype=torch.int32, device=target.device)
    dr = torch.empty((R, N - 1), dtype=torch.int32, device=target.device) if want_drafts else None
    _check(lib.cp_spec_accept_batch(R, N, V, top_k, temperature, seed, mode, _ptr(target), _ptr(draft), _ptr(tok),
                                    _ptr(na), _ptr(dr), _stream()))
    return tok, na, dr


def decode_frames_static(spec: synth.ModelSpec, device_weights: dict, verify_window: int, top_k: int,
                         temperature: float, seed: int, x, c0, codes=None, first_frame: int = 0, max_streams=None,
                         status=None):
    """cp_spec_decode_frames_static: one decode in the library's static scratch, no context.

    x [F, B, H] float32 cuda, c0 [F, B] int32 cuda -> codes [F, B, G] int32 (asynchronous).
    status (optional) is a 1-element int32 cuda tensor that receives the device status word.
    Returns (codes, rc) with rc OK or W_AR_FALLBACK."""
    import torch
    lib = load()
    F, B, _ = x.shape
    if codes is None:
        codes = torch.empty((F, B, spec.num_code_groups), dtype=torch.int32, device=x.device)
    model = model_struct(spec)
    weights = weights_struct(device_weights)
    config = Config(verify_window, top_k, temperature, seed, B if max_streams is None else max_streams,
                    n_draft_offsets(device_weights))
    rc = lib.cp_spec_decode_frames_static(C.byref(model), C.byref(weights), C.byref(config), B, F, first_frame,
                                          _ptr(x), _ptr(c0), _ptr(codes), _ptr(status), _stream())
    _check(rc, None, allow=(OK, W_AR_FALLBACK))
    return codes, rc
