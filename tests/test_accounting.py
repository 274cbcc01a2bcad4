"""The bench's weight-byte and throughput accounting against the figures the
pages print (tests/golden/pages_arithmetic.txt), and the JSON contract helpers."""
import os

import pytest

import bench
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_arithmetic.txt")


def golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


class _Shape:
    """A model whose layer bytes are the pages' 287 MB, in one layer, no head."""

    def __init__(self, layer_bytes):
        self.n_layers, self.vocab, self.dim = 1, 0, 0
        self.qkv_rows = self.ffn = 0
        self._lb = layer_bytes

    def layer_bytes(self):
        return self._lb


def test_naive_bytes_match_the_pages():
    g = golden()
    c = _Shape(int(g["model_bytes_mb"] * 1e6))
    naive = bench.weight_bytes_read(c, int(g["prompt_tokens"]), 1)  # chunk 1 = the per-token loop
    assert round(naive / 1e9) == g["naive_bytes_gb"]


def test_work_per_weight_byte_is_the_chunk():
    g = golden()
    assert bench.macs_per_weight_byte(1, 1) == g["macs_per_byte_gemv"]
    assert bench.macs_per_weight_byte(32 * 24, int(g["chunk"])) == g["macs_per_byte_gemm32"]
    # ragged last chunk: 747 tokens in chunks of 32 read the weights 24 times
    assert bench.weight_bytes_read(_Shape(100), 747, 32) == 24 * 100


def test_throughput_matches_the_pages():
    g = golden()
    assert round(bench.tok_per_s(int(g["prompt_tokens"]), g["seconds_before"])) == g["tok_per_s_before"]
    assert round(bench.tok_per_s(int(g["prompt_tokens"]), g["seconds_after"])) == g["tok_per_s_after"]


def test_8b_algorithmic_work():
    c = synth.CONFIGS["8b"]
    w = bench.algorithmic_work(c, 4096, 512)
    assert abs(w["gemm"]["work"] / 1e12 - 57.1746) < 1e-3
    assert abs(w["attention"]["work"] / 1e12 - 4.3991) < 1e-3  # 4 hd H * P(P+1)/2 * L
    assert bench.weight_bytes_read(c, 4096, 512) == 8 * 32 * bench.layer_weight_bytes(c) + c.vocab * c.dim + 4 * c.vocab


def test_peaks_and_alu_peak():
    peaks = {"hbm_gbs": 6790.7, "bf16_tflops": 1909.9, "bf16_tflops_sustained": 1715.2, "sm_max_mhz": 2070.0,
             "source": "measured"}
    assert bench.peak_for("tensor", peaks)[0] == 1715.2
    assert bench.peak_for("hbm", peaks)[0] == 6790.7
    assert abs(bench.peak_for("alu", peaks, sms=152)[0] - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9


def test_clock_sampler_without_nvidia_smi(monkeypatch):
    import subprocess

    def boom(*a, **k):
        raise FileNotFoundError

    monkeypatch.setattr(subprocess, "Popen", boom)
    s = bench.ClockSampler(0).start()
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]
