"""The host-buffer entry points (pp_debug_quantize, pp_debug_gemm_i8,
pp_debug_gemm_epilogue): the library's own kernels on caller-owned host memory,
bit for bit against the oracle ("Batched Prefill", section "Correctness": the
batched GEMM equals per-token dot products exactly)."""
import numpy as np
import pytest

import oracle
import prompt_prefill_gb300 as pp
import synth
from tests.gpu_util import bits, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    torch_cuda()


@pytest.mark.parametrize("rows,k", [(1, 4), (9, 4096), (3, 14336)])
def test_host_quantize_bit_exact(rows, k):
    x = synth.normal_f32(41, k, (rows, k), 0.0, 2.0)
    x[0, :8] = [127.0, 2.5, 3.5, -2.5, 0.5, -126.5, 1.5, -0.5][: min(8, k)]  # ties at amax = 127
    if rows > 2:
        x[1] = 0.0
    q, s = pp.pp_debug_quantize(x)
    rq, rs = oracle.quantize_rows(x)
    assert np.array_equal(q, rq)
    assert np.array_equal(bits(s), bits(rs))


# n % 128 == 0 runs the tcgen05 engine, the others the mma.sync engine
@pytest.mark.parametrize("m,n,k", [(1, 128, 64), (37, 256, 768), (200, 1024, 1024), (8, 96, 256), (33, 160, 320)])
def test_host_gemm_i8_bit_exact(m, n, k):
    a = synth.uniform_i8(42, m + k, (m, k))
    w = synth.uniform_i8(43, n + k, (n, k))
    assert np.array_equal(pp.pp_debug_gemm_i8(a, w), oracle.gemm_i8(a, w))


def test_host_gemm_i8_extremes():
    # all +-127 at K = 14336: |acc| = 127^2 * 14336, the largest the projections reach
    m, n, k = 4, 128, 14336
    a = np.full((m, k), 127, np.int8)
    a[1] = -127
    w = np.full((n, k), 127, np.int8)
    w[::2] = -127
    acc = pp.pp_debug_gemm_i8(a, w)
    assert np.array_equal(acc, oracle.gemm_i8(a, w))
    assert acc[0, 1] == 127 * 127 * k and acc[0, 0] == -127 * 127 * k


@pytest.mark.parametrize("m,n,k,resid", [(5, 128, 128, False), (19, 256, 512, True), (7, 64, 128, True)])
def test_host_gemm_epilogue_bit_exact(m, n, k, resid):
    a = synth.uniform_i8(44, m + k, (m, k))
    w = synth.uniform_i8(45, n + k, (n, k))
    ws = synth.uniform_f32(46, n, (n,), 1e-4, 2e-2)
    as_ = synth.uniform_f32(47, m, (m,), 1e-3, 5e-2)
    r = synth.normal_f32(48, m, (m, n), 0.0, 1.0) if resid else None
    out = pp.pp_debug_gemm_epilogue(a, w, ws, as_, r)
    ref = oracle.dequant_block(oracle.gemm_i8(a, w), ws, as_)
    if resid:
        ref = (r + ref).astype(np.float32)  # f32 round-to-nearest add, residual first
    assert np.array_equal(bits(out), bits(ref))
