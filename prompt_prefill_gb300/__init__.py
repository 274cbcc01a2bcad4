"""Python binding of libpp.so, the GB300 layer-major batched int8 prefill library.

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels. Function names mirror the C entry points of
``include/pp.h``. Device buffers are passed as torch CUDA tensors (or raw
integer addresses); torch is used for device memory and streams only.

The library must have been built (``python -m prompt_prefill_gb300._build``
or ``__graft_entry__.build()``); importing the binding without it raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpp.so")

PP_OK, PP_ERR_ARG, PP_ERR_CAPACITY, PP_ERR_OOM, PP_ERR_CUDA, PP_ERR_DEVICE_TIMEOUT, PP_ERR_UNSUPPORTED = (
    0, -1, -2, -3, -4, -5, -6)
PP_MODE_RESIDENT, PP_MODE_STREAMED = 0, 1
PP_LOOP_CHUNK_OUTER, PP_LOOP_LAYER_OUTER = 0, 1
PP_GEMM_AUTO, PP_GEMM_MMA, PP_GEMM_TC = 0, 1, 2
(PP_KERNEL_NONE, PP_KERNEL_GEMM, PP_KERNEL_ATTENTION, PP_KERNEL_NORM_QUANT, PP_KERNEL_ROPE_KV, PP_KERNEL_LM_HEAD,
 PP_KERNEL_EMBED) = (-1, 0, 1, 2, 3, 4, 5)
PP_KERNEL_COUNT = 6
KERNEL_NAMES = {0: "gemm", 1: "attention", 2: "norm_quant", 3: "rope_kv", 4: "lm_head", 5: "embed"}
PP_EPI_STORE, PP_EPI_RESID, PP_EPI_SWIGLU = 0, 1, 2
# epilogue indices of pp_stats.gemm_launches (3: raw int32, 4: QKV with RoPE + K/V write)
GEMM_EPI_NAMES = {0: "store", 1: "residual", 2: "swiglu", 3: "int32", 4: "rope"}
# tiles of pp_stats.gemm_launches: (tokens, weight rows) per CTA pair
GEMM_TILES = ((256, 256), (256, 192), (256, 128), (128, 256), (64, 256), (32, 256))
PP_NOALLOC_PART_BYTES, PP_NOALLOC_COUNTERS = 32 * 1024 * 1024, 4096


class PPError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} ({status}): {last_error()}")


class pp_config(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_int32) for n in ("dim", "n_layers", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab")]
                + [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)]
                + [(n, ctypes.c_int32) for n in ("max_seq", "max_chunk", "mode", "ring_slots", "gemm_engine",
                                                  "loop_order", "profile_kernel", "kv_grow")])


class pp_weights(ctypes.Structure):
    _fields_ = [("tok_emb", ctypes.c_void_p), ("w", ctypes.POINTER(ctypes.c_void_p)),
                ("w_scale", ctypes.POINTER(ctypes.c_void_p)), ("attn_norm", ctypes.POINTER(ctypes.c_void_p)),
                ("ffn_norm", ctypes.POINTER(ctypes.c_void_p)), ("final_norm", ctypes.c_void_p),
                ("w_out", ctypes.c_void_p), ("w_out_scale", ctypes.c_void_p)]


class pp_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("calls", "chunks", "tokens", "weight_bytes_read", "h2d_bytes",
                                               "prefetch_hits", "prefetch_misses", "kernel_launches",
                                               "prof_launches")] + [("prof_ms", ctypes.c_double),
                                                                    ("kv_bytes", ctypes.c_int64),
                                                                    ("gemm_launches", (ctypes.c_int64 * 6) * 5)]

    def as_dict(self) -> dict:
        d = {n: getattr(self, n) for n, _ in self._fields_}
        d["gemm_launches"] = {(e, GEMM_TILES[b]): int(self.gemm_launches[e][b])
                              for e in range(5) for b in range(6) if self.gemm_launches[e][b]}
        return d


class pp_layer_profile(ctypes.Structure):
    _fields_ = [("compute_ms", ctypes.c_double), ("io_ms", ctypes.c_double), ("wait_ms", ctypes.c_double),
                ("visits", ctypes.c_int64)]


# Exported symbols and their ctypes signatures (same names as include/pp.h).
_vp, _i32, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
SIGNATURES = {
    "pp_model_load": ([_vp, _vp, ctypes.POINTER(_vp)], ctypes.c_int),
    "pp_model_free": ([_vp], None),
    "pp_prefill": ([_vp, _vp, _i32, _i32, _i32, _vp], ctypes.c_int),
    "pp_prefill_device": ([_vp, _vp, _i32, _i32, _i32, _vp, _vp], ctypes.c_int),
    "pp_forward_one": ([_vp, _i32, _i32, _vp], ctypes.c_int),
    "pp_device_status": ([_vp], ctypes.c_int),
    "pp_kv_reset": ([_vp], ctypes.c_int),
    "pp_kv_read": ([_vp, _i32, _i32, _i32, _i32, _vp], ctypes.c_int),
    "pp_get_stats": ([_vp, ctypes.POINTER(pp_stats)], ctypes.c_int),
    "pp_reset_stats": ([_vp], ctypes.c_int),
    "pp_model_gemm_engine": ([_vp], ctypes.c_int),
    "pp_set_profile_kernel": ([_vp, _i32], ctypes.c_int),
    "pp_set_layer_profile": ([_vp, _i32], ctypes.c_int),
    "pp_set_chunk_overlap": ([_vp, _i32], ctypes.c_int),
    "pp_set_graphs": ([_vp, _i32], ctypes.c_int),
    "pp_get_layer_profile": ([_vp, ctypes.POINTER(pp_layer_profile), _i32], ctypes.c_int),
    "pp_set_trace": ([_vp, _vp, _vp, _vp, _i32], ctypes.c_int),
    "pp_status_str": ([ctypes.c_int], ctypes.c_char_p),
    "pp_last_error": ([], ctypes.c_char_p),
    "pp_op_quantize": ([_vp, _i32, _i32, _vp, _vp, _vp, _vp], ctypes.c_int),
    "pp_op_rmsnorm_quantize": ([_vp, _vp, _i32, _i32, _f32, _vp, _vp, _vp, _vp, _vp], ctypes.c_int),
    "pp_op_gemm_acc": ([_i32, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp], ctypes.c_int),
    "pp_op_gemm": ([_i32, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _i32, _vp], ctypes.c_int),
    "pp_set_exact_segment": ([_i32], ctypes.c_int),
    "pp_op_gemm_noalloc": ([_i32, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _i32, _vp], ctypes.c_int),
    "pp_op_rope_kv": ([_vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp], ctypes.c_int),
    "pp_op_rope_table": ([_i32, _i32, _f32, _vp, _vp], ctypes.c_int),
    "pp_op_attention": ([_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp], ctypes.c_int),
    "pp_op_lm_head": ([_vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp], ctypes.c_int),
    "pp_debug_gemm_stall": ([_i32, _vp, _vp, _i32, _i32, _i32, _vp], ctypes.c_int),
    "pp_debug_loader_fault": ([_vp, _i32], ctypes.c_int),
    "pp_debug_alloc_cap": ([ctypes.c_int64], ctypes.c_int),
    "pp_op_status": ([_vp], ctypes.c_int),
    "pp_debug_op_stall": ([_i32], ctypes.c_int),
    "pp_debug_quantize": ([_vp, _i32, _i32, _vp, _vp], ctypes.c_int),
    "pp_debug_gemm_i8": ([_vp, _vp, _i32, _i32, _i32, _vp], ctypes.c_int),
    "pp_debug_gemm_epilogue": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp], ctypes.c_int),
    "pp_op_gemm_noalloc_need": ([_i32, _i32, _i32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)],
                                ctypes.c_int),
    "pp_debug_noalloc_poison": ([_i32], ctypes.c_int),
}

_lock = threading.Lock()
_lib = None


def lib():
    """Load libpp.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with `python -m prompt_prefill_gb300._build`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def status_str(s: int) -> str:
    return lib().pp_status_str(s).decode()


def last_error() -> str:
    return lib().pp_last_error().decode()


def _check(rc: int, what: str):
    if rc != PP_OK:
        raise PPError(rc, what)


def _ptr(x) -> int | None:
    """Address of a torch tensor, numpy array or integer (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"]
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        assert x.is_contiguous()
        return x.data_ptr()
    raise TypeError(type(x))


def _stream(stream) -> int | None:
    if stream is None:
        try:
            import torch

            return torch.cuda.current_stream().cuda_stream
        except Exception:
            return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- model API
def make_config(dim, n_layers, n_heads, n_kv_heads, head_dim, ffn, vocab, rms_eps=1e-5, rope_theta=10000.0,
                max_seq=4096, max_chunk=512, mode=PP_MODE_RESIDENT, ring_slots=2, gemm_engine=PP_GEMM_AUTO,
                loop_order=PP_LOOP_CHUNK_OUTER, profile_kernel=PP_KERNEL_NONE, kv_grow=0) -> pp_config:
    return pp_config(dim, n_layers, n_heads, n_kv_heads, head_dim, ffn, vocab, rms_eps, rope_theta, max_seq,
                     max_chunk, mode, ring_slots, gemm_engine, loop_order, profile_kernel, kv_grow)


def make_weights(tok_emb, w, w_scale, attn_norm, ffn_norm, final_norm, w_out, w_out_scale):
    """pp_weights over host numpy arrays; returns (struct, keepalive)."""
    P = ctypes.c_void_p
    arrs = [np.ascontiguousarray(a) for a in w]
    scs = [np.ascontiguousarray(a, dtype=np.float32) for a in w_scale]
    an = [np.ascontiguousarray(a, dtype=np.float32) for a in attn_norm]
    fn = [np.ascontiguousarray(a, dtype=np.float32) for a in ffn_norm]
    pw = (P * len(arrs))(*[_ptr(a) for a in arrs])
    ps = (P * len(scs))(*[_ptr(a) for a in scs])
    pa = (P * len(an))(*[_ptr(a) for a in an])
    pf = (P * len(fn))(*[_ptr(a) for a in fn])
    keep = [tok_emb, final_norm, w_out, w_out_scale, arrs, scs, an, fn, pw, ps, pa, pf]
    s = pp_weights(_ptr(tok_emb), pw, ps, pa, pf, _ptr(final_norm), _ptr(w_out), _ptr(w_out_scale))
    return s, keep


def pp_model_load(cfg: pp_config, weights: pp_weights) -> int:
    h = ctypes.c_void_p()
    _check(lib().pp_model_load(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(h)), "pp_model_load")
    return h.value


def pp_model_free(h: int):
    lib().pp_model_free(h)


def pp_prefill(h: int, tokens, start_pos: int, chunk: int, vocab: int, out: np.ndarray | None = None) -> np.ndarray:
    """Host-buffer prefill; `out` (f32 [vocab], contiguous, e.g. in pinned memory) receives the logits."""
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    if out is None:
        out = np.empty((vocab,), np.float32)
    assert out.dtype == np.float32 and out.shape == (vocab,) and out.flags["C_CONTIGUOUS"]
    _check(lib().pp_prefill(h, _ptr(t), t.size, start_pos, chunk, _ptr(out)), "pp_prefill")
    return out


def pp_prefill_rc(h: int, tokens, start_pos: int, chunk: int, vocab: int) -> int:
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    logits = np.empty((vocab,), np.float32)
    return int(lib().pp_prefill(h, _ptr(t) if t.size else None, t.size, start_pos, chunk, _ptr(logits)))


def pp_prefill_device(h: int, d_tokens, n: int, start_pos: int, chunk: int, d_logits, stream=None):
    _check(lib().pp_prefill_device(h, _ptr(d_tokens), n, start_pos, chunk, _ptr(d_logits), _stream(stream)),
           "pp_prefill_device")


def pp_forward_one(h: int, token: int, pos: int, vocab: int) -> np.ndarray:
    logits = np.empty((vocab,), np.float32)
    _check(lib().pp_forward_one(h, int(token), pos, _ptr(logits)), "pp_forward_one")
    return logits


def pp_device_status(h: int) -> int:
    return int(lib().pp_device_status(h))


def pp_kv_reset(h: int):
    _check(lib().pp_kv_reset(h), "pp_kv_reset")


def pp_kv_read(h: int, layer: int, which: int, pos0: int, n_pos: int, n_kv_heads: int, head_dim: int) -> np.ndarray:
    out = np.empty((n_pos, n_kv_heads, head_dim), np.float32)
    _check(lib().pp_kv_read(h, layer, which, pos0, n_pos, _ptr(out)), "pp_kv_read")
    return out


def pp_get_stats(h: int) -> dict:
    s = pp_stats()
    _check(lib().pp_get_stats(h, ctypes.byref(s)), "pp_get_stats")
    return s.as_dict()


def pp_reset_stats(h: int):
    _check(lib().pp_reset_stats(h), "pp_reset_stats")


def pp_set_profile_kernel(h: int, kernel_class: int):
    _check(lib().pp_set_profile_kernel(h, kernel_class), "pp_set_profile_kernel")


def pp_set_layer_profile(h: int, enable: bool):
    _check(lib().pp_set_layer_profile(h, 1 if enable else 0), "pp_set_layer_profile")


def pp_set_chunk_overlap(h: int, enable: bool):
    _check(lib().pp_set_chunk_overlap(h, 1 if enable else 0), "pp_set_chunk_overlap")


def pp_set_graphs(h: int, enable: bool):
    _check(lib().pp_set_graphs(h, 1 if enable else 0), "pp_set_graphs")


def pp_get_layer_profile(h: int, n_layers: int) -> list:
    arr = (pp_layer_profile * n_layers)()
    _check(lib().pp_get_layer_profile(h, arr, n_layers), "pp_get_layer_profile")
    return [{n: getattr(x, n) for n, _ in pp_layer_profile._fields_} for x in arr]


def pp_debug_gemm_stall(wait_us: int, a16, w, m: int, n: int, k: int, acc) -> int:
    """Status of a tcgen05 GEMM run with its MMA issuer held back (test hook)."""
    return int(lib().pp_debug_gemm_stall(wait_us, _ptr(a16), _ptr(w), m, n, k, _ptr(acc)))


def pp_debug_loader_fault(h: int, fault: int):
    _check(lib().pp_debug_loader_fault(h, fault), "pp_debug_loader_fault")


def pp_debug_alloc_cap(nbytes: int):
    _check(lib().pp_debug_alloc_cap(nbytes), "pp_debug_alloc_cap")


def pp_set_trace(h: int, d_x, d_codes, d_scales, max_pos: int):
    _check(lib().pp_set_trace(h, _ptr(d_x), _ptr(d_codes), _ptr(d_scales), max_pos), "pp_set_trace")


def pp_model_gemm_engine(h: int) -> int:
    return int(lib().pp_model_gemm_engine(h))


# ---------------------------------------------------------------- single steps
def pp_op_quantize(x, rows, k, q8, q16, a_scale, stream=None):
    _check(lib().pp_op_quantize(_ptr(x), rows, k, _ptr(q8), _ptr(q16), _ptr(a_scale), _stream(stream)),
           "pp_op_quantize")


def pp_op_rmsnorm_quantize(x, g, rows, k, eps, y_out, q8, q16, a_scale, stream=None):
    _check(lib().pp_op_rmsnorm_quantize(_ptr(x), _ptr(g), rows, k, eps, _ptr(y_out), _ptr(q8), _ptr(q16),
                                        _ptr(a_scale), _stream(stream)), "pp_op_rmsnorm_quantize")


def pp_op_gemm_acc(engine, a8, a16, w, m, n, k, acc, stream=None):
    _check(lib().pp_op_gemm_acc(engine, _ptr(a8), _ptr(a16), _ptr(w), m, n, k, _ptr(acc), _stream(stream)),
           "pp_op_gemm_acc")


def pp_op_gemm(engine, epilogue, a8, a16, w, w_scale, a_scale, m, n, k, out, ldo, stream=None):
    _check(lib().pp_op_gemm(engine, epilogue, _ptr(a8), _ptr(a16), _ptr(w), _ptr(w_scale), _ptr(a_scale), m, n, k,
                            _ptr(out), ldo, _stream(stream)), "pp_op_gemm")


def pp_op_gemm_noalloc(epilogue, a16, w, w_scale, a_scale, m, n, k, out, ldo, stream=None):
    """pp_op_gemm on the tcgen05 engine with no device allocation (fixed scratch
    inside the library; see include/pp.h for the size limit and sharing rules)."""
    _check(lib().pp_op_gemm_noalloc(epilogue, _ptr(a16), _ptr(w), _ptr(w_scale), _ptr(a_scale), m, n, k, _ptr(out),
                                    ldo, _stream(stream)), "pp_op_gemm_noalloc")


def pp_op_status(stream=None) -> int:
    """Status of the single-step tcgen05 GEMM calls since the last query (waits for the stream)."""
    return int(lib().pp_op_status(_stream(stream)))


def pp_debug_op_stall(wait_us: int):
    _check(lib().pp_debug_op_stall(wait_us), "pp_debug_op_stall")


def pp_debug_quantize(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """The quantiser on host rows (x [rows][k] f32): (int8 codes, f32 row scales)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, k = x.shape
    q = np.empty((rows, k), np.int8)
    s = np.empty((rows,), np.float32)
    _check(lib().pp_debug_quantize(_ptr(x), rows, k, _ptr(q), _ptr(s)), "pp_debug_quantize")
    return q, s


def pp_debug_gemm_i8(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """acc[t][r] = sum_i a[t][i] w[r][i] (int32) from host int8 a [m][k], w [n][k]."""
    a = np.ascontiguousarray(a, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    (m, k), n = a.shape, w.shape[0]
    assert w.shape[1] == k
    acc = np.empty((m, n), np.int32)
    _check(lib().pp_debug_gemm_i8(_ptr(a), _ptr(w), m, n, k, _ptr(acc)), "pp_debug_gemm_i8")
    return acc


def pp_debug_gemm_epilogue(a: np.ndarray, w: np.ndarray, w_scale: np.ndarray, a_scale: np.ndarray,
                           resid: np.ndarray | None = None) -> np.ndarray:
    """(float(acc) * w_scale[r]) * a_scale[t] (+ resid[t][r]) from host buffers, f32 [m][n]."""
    a = np.ascontiguousarray(a, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    ws = np.ascontiguousarray(w_scale, dtype=np.float32)
    as_ = np.ascontiguousarray(a_scale, dtype=np.float32)
    (m, k), n = a.shape, w.shape[0]
    assert w.shape[1] == k and ws.shape == (n,) and as_.shape == (m,)
    r = None if resid is None else np.ascontiguousarray(resid, dtype=np.float32)
    assert r is None or r.shape == (m, n)
    out = np.empty((m, n), np.float32)
    _check(lib().pp_debug_gemm_epilogue(_ptr(a), _ptr(w), _ptr(ws), _ptr(as_), _ptr(r), m, n, k, _ptr(out)),
           "pp_debug_gemm_epilogue")
    return out


def pp_op_gemm_noalloc_need(m: int, n: int, k: int) -> tuple[int, int]:
    """(partial-tile bytes, counters) the tcgen05 GEMM plans for this shape on the current device."""
    pb, cc = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().pp_op_gemm_noalloc_need(m, n, k, ctypes.byref(pb), ctypes.byref(cc)), "pp_op_gemm_noalloc_need")
    return pb.value, cc.value


def pp_debug_noalloc_poison(value: int):
    _check(lib().pp_debug_noalloc_poison(value), "pp_debug_noalloc_poison")


def pp_set_exact_segment(seg_k: int):
    _check(lib().pp_set_exact_segment(seg_k), "pp_set_exact_segment")


def pp_op_rope_table(max_pos, head_dim, theta, table, stream=None):
    _check(lib().pp_op_rope_table(max_pos, head_dim, theta, _ptr(table), _stream(stream)), "pp_op_rope_table")


def pp_op_rope_kv(qkv, rows, start_pos, n_heads, n_kv_heads, head_dim, table, q_out, k_cache, v_cache, stream=None):
    _check(lib().pp_op_rope_kv(_ptr(qkv), rows, start_pos, n_heads, n_kv_heads, head_dim, _ptr(table), _ptr(q_out),
                               _ptr(k_cache), _ptr(v_cache), _stream(stream)), "pp_op_rope_kv")


def pp_op_attention(q, k_cache, v_cache, rows, start_pos, n_heads, n_kv_heads, head_dim, o, stream=None):
    _check(lib().pp_op_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), rows, start_pos, n_heads, n_kv_heads,
                                 head_dim, _ptr(o), _stream(stream)), "pp_op_attention")


def pp_op_lm_head(q8, a_scale, w_out, w_scale, vocab, dim, logits, stream=None):
    _check(lib().pp_op_lm_head(_ptr(q8), _ptr(a_scale), _ptr(w_out), _ptr(w_scale), vocab, dim, _ptr(logits),
                               _stream(stream)), "pp_op_lm_head")


# ---------------------------------------------------------------- convenience
@dataclass
class ModelShape:
    dim: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0


class PrefillModel:
    """A loaded model: owns the pp_model handle (freed on close)."""

    def __init__(self, shape, weights, max_seq=4096, max_chunk=512, mode=PP_MODE_RESIDENT, ring_slots=2,
                 gemm_engine=PP_GEMM_AUTO, loop_order=PP_LOOP_CHUNK_OUTER, profile_kernel=PP_KERNEL_NONE, kv_grow=0):
        """shape: any object with the ModelShape fields; weights: any object with
        tok_emb, w, w_scale, attn_norm, ffn_norm, final_norm, w_out, w_out_scale (host arrays)."""
        self.cfg = make_config(shape.dim, shape.n_layers, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn,
                               shape.vocab, shape.rms_eps, shape.rope_theta, max_seq, max_chunk, mode, ring_slots,
                               gemm_engine, loop_order, profile_kernel, kv_grow)
        ws, keep = make_weights(weights.tok_emb, weights.w, weights.w_scale, weights.attn_norm, weights.ffn_norm,
                                weights.final_norm, weights.w_out, weights.w_out_scale)
        self.h = pp_model_load(self.cfg, ws)
        del keep  # the library copied or pinned everything it needs
        self.vocab = shape.vocab

    def close(self):
        if getattr(self, "h", None):
            pp_model_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, tokens, start_pos=0, chunk=None, out=None):
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        return pp_prefill(self.h, t, start_pos, chunk or self.cfg.max_chunk, self.vocab, out)

    def prefill_device(self, d_tokens, n, start_pos, chunk, d_logits, stream=None):
        pp_prefill_device(self.h, d_tokens, n, start_pos, chunk, d_logits, stream)

    def forward_one(self, token, pos):
        return pp_forward_one(self.h, token, pos, self.vocab)

    def kv_reset(self):
        pp_kv_reset(self.h)

    def kv(self, layer, which, pos0, n_pos):
        return pp_kv_read(self.h, layer, which, pos0, n_pos, self.cfg.n_kv_heads, self.cfg.head_dim)

    def stats(self):
        return pp_get_stats(self.h)

    def reset_stats(self):
        pp_reset_stats(self.h)

    def set_profile_kernel(self, kernel_class):
        pp_set_profile_kernel(self.h, kernel_class)

    def set_layer_profile(self, enable=True):
        pp_set_layer_profile(self.h, enable)

    def set_chunk_overlap(self, enable=True):
        pp_set_chunk_overlap(self.h, enable)

    def set_graphs(self, enable=True):
        pp_set_graphs(self.h, enable)

    def layer_profile(self):
        return pp_get_layer_profile(self.h, self.cfg.n_layers)

    def set_trace(self, d_x, d_codes, d_scales, max_pos):
        pp_set_trace(self.h, d_x, d_codes, d_scales, max_pos)

    def device_status(self):
        return pp_device_status(self.h)

    @property
    def gemm_engine(self):
        return pp_model_gemm_engine(self.h)
