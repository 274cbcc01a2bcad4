"""Seeded synthetic inputs shared by the tests, the bench and the oracle runs.

Holds no prefill arithmetic: it draws the int8 checkpoint, the f32
embeddings and norm gains, and the prompt token ids, as plain numpy
arrays. The drawing itself is in ``synth.c`` (counter-based SplitMix64 +
Box-Muller), compiled on first use into ``libsynth.so`` next to it.

Model workloads (``CONFIGS``) follow the five model configurations the
prefill method is measured on: a tiny decoder, a 350M-class decoder, a
1B-class decoder and a Llama-3-8B-shaped decoder (resident and streamed).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# Weight kinds in each layer, in the order both libraries take them.
LAYER_KINDS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def build(force: bool = False) -> str:
    """Compile libsynth.so (portable C, no target-specific flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c11", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            u64, i64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
            L.synth_normal_f32.argtypes = [u64, u64, vp, i64, dbl, dbl, ctypes.c_int]
            L.synth_int8_rows.argtypes = [u64, u64, i64, i64, dbl, vp, vp, ctypes.c_int]
            L.synth_tokens.argtypes = [u64, u64, vp, i64, i32]
            L.synth_uniform_f32.argtypes = [u64, u64, vp, i64, dbl, dbl]
            L.synth_uniform_i8.argtypes = [u64, u64, vp, i64, ctypes.c_int, ctypes.c_int]
            for f in (L.synth_normal_f32, L.synth_int8_rows, L.synth_tokens, L.synth_uniform_f32, L.synth_uniform_i8):
                f.restype = None
            _lib = L
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_f32(seed: int, stream: int, shape, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    lib().synth_normal_f32(seed, stream, out.ctypes.data, out.size, mean, std, _threads())
    return out


def int8_rows(seed: int, stream: int, rows: int, cols: int, std=0.02):
    q = np.empty((rows, cols), dtype=np.int8)
    s = np.empty((rows,), dtype=np.float32)
    lib().synth_int8_rows(seed, stream, rows, cols, std, q.ctypes.data, s.ctypes.data, _threads())
    return q, s


def tokens(seed: int, n: int, vocab: int, stream: int = 7) -> np.ndarray:
    out = np.empty((n,), dtype=np.int32)
    lib().synth_tokens(seed, stream, out.ctypes.data, n, vocab)
    return out


def uniform_f32(seed: int, stream: int, shape, lo=-1.0, hi=1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    lib().synth_uniform_f32(seed, stream, out.ctypes.data, out.size, lo, hi)
    return out


def uniform_i8(seed: int, stream: int, shape, lo=-127, hi=127) -> np.ndarray:
    out = np.empty(shape, dtype=np.int8)
    lib().synth_uniform_i8(seed, stream, out.ctypes.data, out.size, lo, hi)
    return out


@dataclass
class ModelConfig:
    name: str
    dim: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    max_seq: int = 4096
    seed: int = 1234
    # workload
    prompt_len: int = 32
    chunk: int = 8
    extra: dict = field(default_factory=dict)

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    def layer_shapes(self):
        """(rows, cols) of each int8 matrix of one layer, in LAYER_KINDS order."""
        D, F, hd = self.dim, self.ffn, self.head_dim
        return [
            (self.n_heads * hd, D),
            (self.n_kv_heads * hd, D),
            (self.n_kv_heads * hd, D),
            (D, self.n_heads * hd),
            (F, D),
            (F, D),
            (D, F),
        ]

    def layer_bytes(self) -> int:
        return sum(r * c for r, c in self.layer_shapes())

    def gemm_ops_per_token(self) -> int:
        """2 x int8 MACs of the four projection groups per token (LM head excluded)."""
        return 2 * self.layer_bytes() * self.n_layers


# The five measured configurations. Seeds are 1234 + index.
CONFIGS = {
    "tiny": ModelConfig("tiny", 256, 4, 4, 4, 64, 768, 1024, max_seq=64, seed=1234, prompt_len=32, chunk=8),
    "350m": ModelConfig("350m", 1024, 24, 16, 8, 64, 4096, 65536, max_seq=1024, seed=1235, prompt_len=747, chunk=32),
    "1b": ModelConfig("1b", 2048, 16, 32, 8, 64, 8192, 128256, max_seq=4096, seed=1236, prompt_len=2048, chunk=512,
                      extra={"chunks": (32, 128, 512, 2048)}),
    "8b": ModelConfig("8b", 4096, 32, 32, 8, 128, 14336, 128256, rope_theta=500000.0, max_seq=4096, seed=1237,
                      prompt_len=4096, chunk=512),
    "8b-streamed": ModelConfig("8b-streamed", 4096, 32, 32, 8, 128, 14336, 128256, rope_theta=500000.0,
                               max_seq=2048, seed=1238, prompt_len=2048, chunk=512,
                               extra={"prompt_lens": (122, 512, 2048)}),
}


def stream_id(layer: int, kind: int) -> int:
    return 1000 + 16 * layer + kind


@dataclass
class Model:
    cfg: ModelConfig
    tok_emb: np.ndarray          # [vocab, dim] f32
    w: list                      # n_layers*7 int8 [rows, cols]
    w_scale: list                # n_layers*7 f32 [rows]
    attn_norm: list              # n_layers f32 [dim]
    ffn_norm: list               # n_layers f32 [dim]
    final_norm: np.ndarray       # [dim] f32
    w_out: np.ndarray            # [vocab, dim] int8
    w_out_scale: np.ndarray      # [vocab] f32


def make_model(cfg: ModelConfig, seed: int | None = None, weight_std: float = 0.02) -> Model:
    """Draw the synthetic checkpoint of ``cfg``.

    Embeddings ~ N(0, 0.02) f32; projection and LM-head weights ~ N(0, 0.02)
    quantised per output row to int8 with an f32 scale; RMSNorm gains
    ~ 1 + N(0, 0.02) so that the gain multiply is exercised.
    """
    s = cfg.seed if seed is None else seed
    D, V = cfg.dim, cfg.vocab
    tok_emb = normal_f32(s, 1, (V, D), 0.0, 0.02)
    w, ws, an, fn = [], [], [], []
    for L in range(cfg.n_layers):
        for k, (r, c) in enumerate(cfg.layer_shapes()):
            q, sc = int8_rows(s, stream_id(L, k), r, c, weight_std)
            w.append(q)
            ws.append(sc)
        an.append(normal_f32(s, stream_id(L, 7), (D,), 1.0, 0.02))
        fn.append(normal_f32(s, stream_id(L, 8), (D,), 1.0, 0.02))
    final_norm = normal_f32(s, 2, (D,), 1.0, 0.02)
    w_out, w_out_scale = int8_rows(s, 3, V, D, weight_std)
    return Model(cfg, tok_emb, w, ws, an, fn, final_norm, w_out, w_out_scale)


def prompt(cfg: ModelConfig, n: int | None = None, seed: int | None = None) -> np.ndarray:
    n = cfg.prompt_len if n is None else n
    return tokens(cfg.seed if seed is None else seed, n, cfg.vocab)
