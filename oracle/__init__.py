"""CPU oracle of layer-major batched int8 prefill -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline
leg may import this package. It wraps ``oracle.c`` (plain C, built here
into ``liborc.so`` with gcc) through ctypes. It shares no code with the
CUDA library and never loads it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liborc.so")
_lock = threading.Lock()
_lib = None

ORC_OK, ORC_ERR_ARG, ORC_ERR_CAPACITY, ORC_ERR_OOM = 0, -1, -2, -3


def build(force: bool = False) -> str:
    """Compile liborc.so: portable C11, IEEE f32 (no contraction, no fast-math)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c11", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class OrcForce(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p * 4), ("scales", ctypes.c_void_p * 4), ("kmax", ctypes.c_int),
                ("mismatches", ctypes.c_int64 * 4), ("scale_mismatches", ctypes.c_int64 * 4),
                ("max_margin", ctypes.c_float * 4), ("max_code_diff", ctypes.c_int * 4),
                ("max_scale_rel", ctypes.c_float * 4)]


class OrcConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("dim", "n_layers", "n_heads", "n_kv_heads", "head_dim", "ffn",
                                               "vocab", "max_seq")] + [("rms_eps", ctypes.c_float),
                                                                        ("rope_theta", ctypes.c_float)]


class OrcWeights(ctypes.Structure):
    _fields_ = [("tok_emb", ctypes.c_void_p), ("w", ctypes.POINTER(ctypes.c_void_p)),
                ("w_scale", ctypes.POINTER(ctypes.c_void_p)), ("attn_norm", ctypes.POINTER(ctypes.c_void_p)),
                ("ffn_norm", ctypes.POINTER(ctypes.c_void_p)), ("final_norm", ctypes.c_void_p),
                ("w_out", ctypes.c_void_p), ("w_out_scale", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp, i32 = ctypes.c_void_p, ctypes.c_int
            sig = {
                "orc_create": ([vp, vp, i32, ctypes.POINTER(vp)], i32),
                "orc_destroy": ([vp], None),
                "orc_prefill": ([vp, vp, i32, i32, i32, vp, vp], i32),
                "orc_forward_one": ([vp, ctypes.c_int32, i32, vp], i32),
                "orc_kv": ([vp, i32, i32], vp),
                "orc_kv_reset": ([vp], None),
                "orc_quantize_row": ([vp, i32, vp, vp], None),
                "orc_quantize_rows": ([vp, i32, i32, vp, vp], None),
                "orc_dot_i8": ([vp, vp, i32], ctypes.c_int32),
                "orc_gemm_i8": ([vp, vp, i32, i32, i32, vp, i32], None),
                "orc_dequant": ([ctypes.c_int32, ctypes.c_float, ctypes.c_float], ctypes.c_float),
                "orc_rmsnorm_row": ([vp, vp, i32, ctypes.c_float, vp], None),
                "orc_rmsnorm_rows": ([vp, vp, i32, i32, ctypes.c_float, vp], None),
                "orc_rope_head": ([vp, i32, i32, ctypes.c_float], None),
                "orc_rope_rows": ([vp, i32, i32, i32, i32, ctypes.c_float], None),
                "orc_silu_mul": ([ctypes.c_float, ctypes.c_float], ctypes.c_float),
                "orc_attention": ([vp, vp, vp, i32, i32, i32, i32, i32, vp, i32], None),
                "orc_layer": ([vp, i32, vp, i32, i32], i32),
                "orc_final_logits": ([vp, vp, vp], i32),
                "orc_layer_forced": ([vp, i32, vp, i32, i32, vp], i32),
            }
            for name, (args, res) in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def n_threads_default() -> int:
    return max(1, os.cpu_count() or 1)


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- steps
def quantize_rows(y: np.ndarray):
    y = np.ascontiguousarray(y, dtype=np.float32)
    rows, k = y.shape
    q = np.empty((rows, k), np.int8)
    s = np.empty((rows,), np.float32)
    lib().orc_quantize_rows(_p(y), rows, k, _p(q), _p(s))
    return q, s


def gemm_i8(a: np.ndarray, w: np.ndarray, n_threads: int | None = None) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    m, k = a.shape
    n, k2 = w.shape
    assert k == k2
    acc = np.empty((m, n), np.int32)
    lib().orc_gemm_i8(_p(a), _p(w), m, n, k, _p(acc), n_threads or n_threads_default())
    return acc


def dot_i8(a: np.ndarray, w: np.ndarray) -> int:
    a = np.ascontiguousarray(a, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    return int(lib().orc_dot_i8(_p(a), _p(w), a.size))


def dequant(acc: int, w_scale: float, a_scale: float) -> np.float32:
    return np.float32(lib().orc_dequant(int(acc), float(w_scale), float(a_scale)))


def dequant_block(acc: np.ndarray, w_scale: np.ndarray, a_scale: np.ndarray) -> np.ndarray:
    out = np.empty(acc.shape, np.float32)
    f = lib().orc_dequant
    for t in range(acc.shape[0]):
        for r in range(acc.shape[1]):
            out[t, r] = f(int(acc[t, r]), float(w_scale[r]), float(a_scale[t]))
    return out


def rmsnorm_rows(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    g = np.ascontiguousarray(g, dtype=np.float32)
    rows, d = x.shape
    y = np.empty_like(x)
    lib().orc_rmsnorm_rows(_p(x), _p(g), rows, d, eps, _p(y))
    return y


def rope_rows(x: np.ndarray, start_pos: int, theta: float) -> np.ndarray:
    """x: [rows, n_heads, hd] f32; returns the rotated copy."""
    y = np.array(x, dtype=np.float32, order="C", copy=True)
    rows, nh, hd = y.shape
    lib().orc_rope_rows(_p(y), rows, nh, hd, start_pos, theta)
    return y


def silu_mul(g: float, u: float) -> np.float32:
    return np.float32(lib().orc_silu_mul(float(g), float(u)))


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, start_pos: int, n_threads: int | None = None):
    """q: [rows, H, hd]; K, V: [>= start_pos+rows, Hkv, hd]; returns o [rows, H, hd]."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    rows, H, hd = q.shape
    Hkv = K.shape[1]
    assert K.shape[0] >= start_pos + rows and V.shape == K.shape and K.shape[2] == hd
    o = np.empty_like(q)
    lib().orc_attention(_p(q), _p(K), _p(V), rows, start_pos, H, Hkv, hd, _p(o), n_threads or n_threads_default())
    return o


# ---------------------------------------------------------------- model
class OracleModel:
    """The oracle model over a synthetic checkpoint (``synth.Model``)."""

    def __init__(self, model, max_seq: int | None = None, n_threads: int | None = None):
        c = model.cfg
        self.model = model
        self.cfg = OrcConfig(c.dim, c.n_layers, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn, c.vocab,
                             max_seq or c.max_seq, c.rms_eps, c.rope_theta)
        P = ctypes.c_void_p
        self._w = (P * len(model.w))(*[_p(a) for a in model.w])
        self._ws = (P * len(model.w_scale))(*[_p(a) for a in model.w_scale])
        self._an = (P * len(model.attn_norm))(*[_p(a) for a in model.attn_norm])
        self._fn = (P * len(model.ffn_norm))(*[_p(a) for a in model.ffn_norm])
        self.weights = OrcWeights(_p(model.tok_emb), self._w, self._ws, self._an, self._fn, _p(model.final_norm),
                                  _p(model.w_out), _p(model.w_out_scale))
        self.n_threads = n_threads or n_threads_default()
        h = ctypes.c_void_p()
        rc = lib().orc_create(ctypes.byref(self.cfg), ctypes.byref(self.weights), self.n_threads, ctypes.byref(h))
        if rc != ORC_OK:
            raise RuntimeError(f"orc_create failed: {rc}")
        self.h = h

    def close(self):
        if self.h:
            lib().orc_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, tokens, start_pos: int = 0, chunk: int = 1, want_hidden: bool = False):
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        logits = np.empty((self.model.cfg.vocab,), np.float32)
        hidden = np.empty((self.model.cfg.dim,), np.float32) if want_hidden else None
        rc = lib().orc_prefill(self.h, _p(t), t.size, start_pos, chunk, _p(logits),
                               _p(hidden) if hidden is not None else None)
        if rc != ORC_OK:
            raise RuntimeError(f"orc_prefill failed: {rc}")
        return (logits, hidden) if want_hidden else logits

    def prefill_rc(self, tokens, start_pos: int = 0, chunk: int = 1) -> int:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        logits = np.empty((self.model.cfg.vocab,), np.float32)
        return int(lib().orc_prefill(self.h, _p(t) if t.size else None, t.size, start_pos, chunk, _p(logits), None))

    def forward_one(self, token: int, pos: int):
        logits = np.empty((self.model.cfg.vocab,), np.float32)
        rc = lib().orc_forward_one(self.h, int(token), pos, _p(logits))
        if rc != ORC_OK:
            raise RuntimeError(f"orc_forward_one failed: {rc}")
        return logits

    def layer(self, layer: int, x, start_pos: int = 0) -> np.ndarray:
        """Layer `layer` alone over rows x [n, dim] (one chunk at start_pos); returns the output rows."""
        y = np.array(x, dtype=np.float32, order="C", copy=True)
        rc = lib().orc_layer(self.h, layer, _p(y), y.shape[0], start_pos)
        if rc != ORC_OK:
            raise RuntimeError(f"orc_layer failed: {rc}")
        return y

    def layer_forced(self, layer: int, x, codes, scales, start_pos: int = 0):
        """Layer `layer` over rows x [n, dim] taking the given codes [4, n, kmax]
        int8 and scales [4, n] at its quantisation points; returns the output
        rows and, per point, where the oracle's own decisions differed."""
        y = np.array(x, dtype=np.float32, order="C", copy=True)
        codes = np.ascontiguousarray(codes, dtype=np.int8)
        scales = np.ascontiguousarray(scales, dtype=np.float32)
        f = OrcForce()
        for i in range(4):
            f.codes[i] = codes[i].ctypes.data
            f.scales[i] = scales[i].ctypes.data
        f.kmax = codes.shape[2]
        rc = lib().orc_layer_forced(self.h, layer, _p(y), y.shape[0], start_pos, ctypes.byref(f))
        if rc != ORC_OK:
            raise RuntimeError(f"orc_layer_forced failed: {rc}")
        stats = {"mismatches": list(f.mismatches), "scale_mismatches": list(f.scale_mismatches),
                 "max_margin": list(f.max_margin), "max_code_diff": list(f.max_code_diff),
                 "max_scale_rel": list(f.max_scale_rel)}
        return y, stats

    def final_logits(self, x_row) -> np.ndarray:
        x = np.ascontiguousarray(x_row, dtype=np.float32)
        logits = np.empty((self.model.cfg.vocab,), np.float32)
        rc = lib().orc_final_logits(self.h, _p(x), _p(logits))
        if rc != ORC_OK:
            raise RuntimeError(f"orc_final_logits failed: {rc}")
        return logits

    def kv(self, layer: int, which: int) -> np.ndarray:
        """Copy of the K (0) or V (1) cache of one layer: [max_seq, Hkv, hd]."""
        c = self.cfg
        ptr = lib().orc_kv(self.h, layer, which)
        n = c.max_seq * c.n_kv_heads * c.head_dim
        arr = np.ctypeslib.as_array(ctypes.cast(ptr, ctypes.POINTER(ctypes.c_float)), shape=(n,))
        return arr.copy().reshape(c.max_seq, c.n_kv_heads, c.head_dim)

    def kv_reset(self):
        lib().orc_kv_reset(self.h)
