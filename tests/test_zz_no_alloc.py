"""The GEMM entry point that allocates no device memory (pp_op_gemm_noalloc).

It exists for callers that may not allocate device memory while they run --
an application whose device memory is all held by its own pool allocator, or
a latency-critical loop where cudaMalloc/cudaFree would block or synchronise
the device. It runs the same tcgen05 GEMM as pp_op_gemm, with the stream-K
scratch in a fixed array inside the library instead of a buffer allocated on
demand. Its results must equal pp_op_gemm's bit for bit (the integer sums are
exact), on two calls in a row (the array keeps the previous call's contents).

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.
"""
import numpy as np
import pytest

import prompt_prefill_gb300 as pp
import synth
from tests.gpu_util import bits, dev, empty, host, torch_cuda

pytestmark = pytest.mark.gpu

# (m, n, k): the long-K down projection at 512 and 256 rows (planned with
# stream-K partial tiles on a GB300, i.e. they use the scratch), and a
# QKV-shaped GEMM that runs whole tiles. Whether a shape uses the scratch
# depends on the device's SM count; the tests read the plan from the library.
SHAPES = [(512, 4096, 14336), (256, 8192, 14336), (512, 6144, 4096)]


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    pp.pp_set_exact_segment(1024)
    return t


def _inputs(m, n, k, seed):
    a = synth.uniform_i8(seed, 1, (m, k))
    w = synth.uniform_i8(seed, 2, (n, k))
    ws = synth.uniform_f32(seed, 3, (n,), 1e-4, 2e-3)
    as_ = synth.uniform_f32(seed, 4, (m,), 1e-3, 5e-2)
    x0 = synth.normal_f32(seed, 5, (m, n), 0.0, 2.0)
    return a, w, ws, as_, x0


@pytest.mark.parametrize("m,n,k", SHAPES)
@pytest.mark.parametrize("epi", [pp.PP_EPI_STORE, pp.PP_EPI_RESID, pp.PP_EPI_SWIGLU])
def test_noalloc_equals_allocating_gemm_twice(torch, m, n, k, epi):
    a, w, ws, as_, x0 = _inputs(m, n, k, 90 + epi)
    da, da16, dw, dws, das = dev(a), dev(a.astype(np.float16)), dev(w), dev(ws), dev(as_)
    cols = n // 2 if epi == pp.PP_EPI_SWIGLU else n
    x0 = x0[:, :cols].copy()

    def fresh_out():
        return dev(x0) if epi == pp.PP_EPI_RESID else empty((m, cols), torch.float32)

    ref = fresh_out()
    pp.pp_op_gemm(pp.PP_GEMM_TC, epi, da, da16, dw, dws, das, m, n, k, ref, cols)
    ref = host(ref)
    for _ in range(2):  # the second call starts from the first call's scratch contents
        out = fresh_out()
        pp.pp_op_gemm_noalloc(epi, da16, dw, dws, das, m, n, k, out, cols)
        assert np.array_equal(bits(host(out)), bits(ref))


def test_noalloc_clears_counters_left_behind(torch):
    # Arrival counters that a call which gave up part of the way would leave in the fixed scratch
    # (set here from the host): the next call clears what it uses and still equals pp_op_gemm.
    m, n, k = SHAPES[0]
    part, cnt = pp.pp_op_gemm_noalloc_need(m, n, k)
    if cnt == 0:
        pytest.skip("this device plans the shape without stream-K scratch")
    a, w, ws, as_, _ = _inputs(m, n, k, 97)
    da, da16, dw, dws, das = dev(a), dev(a.astype(np.float16)), dev(w), dev(ws), dev(as_)
    ref = empty((m, n), torch.float32)
    pp.pp_op_gemm(pp.PP_GEMM_TC, pp.PP_EPI_STORE, da, da16, dw, dws, das, m, n, k, ref, n)
    ref = host(ref)
    for value in (1, 7):
        pp.pp_debug_noalloc_poison(value)
        out = empty((m, n), torch.float32)
        pp.pp_op_gemm_noalloc(pp.PP_EPI_STORE, da16, dw, dws, das, m, n, k, out, n)
        assert np.array_equal(bits(host(out)), bits(ref))
    assert pp.pp_op_status() == pp.PP_OK


def test_noalloc_accepts_exactly_the_shapes_its_scratch_holds(torch):
    # the library's own plan decides: a shape whose partial tiles or counters exceed the fixed
    # capacity is rejected with PP_ERR_ARG, every other shape runs
    for m, n, k in [(1024, 4096, 14336), (768, 4096, 14336)] + SHAPES:
        part, cnt = pp.pp_op_gemm_noalloc_need(m, n, k)
        fits = part <= pp.PP_NOALLOC_PART_BYTES and cnt <= pp.PP_NOALLOC_COUNTERS
        a16 = empty((m, k), torch.float16)
        w = empty((n, k), torch.int8)
        ws = empty((n,), torch.float32)
        as_ = empty((m,), torch.float32)
        out = empty((m, n), torch.float32)
        if fits:
            a16.zero_()
            w.zero_()
            pp.pp_op_gemm_noalloc(pp.PP_EPI_STORE, a16, w, ws, as_, m, n, k, out, n)
            continue
        with pytest.raises(pp.PPError) as e:
            pp.pp_op_gemm_noalloc(pp.PP_EPI_STORE, a16, w, ws, as_, m, n, k, out, n)
        assert e.value.status == pp.PP_ERR_ARG
        assert "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert pp.pp_op_status() == pp.PP_OK


def test_noalloc_rejects_shapes_beyond_its_scratch(torch):
    m, n, k = 1024, 4096, 14336  # on a GB300 the stream-K plan needs more than the fixed 32 MiB
    part, cnt = pp.pp_op_gemm_noalloc_need(m, n, k)
    if part <= pp.PP_NOALLOC_PART_BYTES and cnt <= pp.PP_NOALLOC_COUNTERS:
        pytest.skip("on this device the shape fits the fixed scratch")
    a16 = empty((m, k), torch.float16)
    w = empty((n, k), torch.int8)
    ws = empty((n,), torch.float32)
    as_ = empty((m,), torch.float32)
    out = empty((m, n), torch.float32)
    with pytest.raises(pp.PPError) as e:
        pp.pp_op_gemm_noalloc(pp.PP_EPI_STORE, a16, w, ws, as_, m, n, k, out, n)
    assert e.value.status == pp.PP_ERR_ARG
    assert "scratch" in str(e.value)
