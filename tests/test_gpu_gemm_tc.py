"""The tcgen05 exact-integer GEMM engine against the oracle, through the C ABI.

tcgen05 MMAs accumulate fp16 products of int8 codes in f32. The engine drains
each K segment of at most 1024 products (|partial sums| <= 127^2 * 1024 <
2^24, exact in f32) into int32, so every accumulator must equal the oracle's
int32 dot product bit for bit -- including all-+-127 inputs that put partial
sums at the top of that range.
"""
import numpy as np
import pytest

import oracle
import prompt_prefill_gb300 as pp
import synth
from tests.gpu_util import bits, dev, empty, host, swiglu_close, torch_cuda

pytestmark = pytest.mark.gpu
TC = pp.PP_GEMM_TC


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    pp.pp_set_exact_segment(1024)
    return t


def _acc(torch, engine, a, w):
    m, k = a.shape
    n = w.shape[0]
    acc = empty((m, n), torch.int32)
    a16 = dev(a.astype(np.float16))
    pp.pp_op_gemm_acc(engine, dev(a), a16, dev(w), m, n, k, acc)
    return host(acc)


TC_SHAPES = [(1, 256, 64), (8, 768, 256), (37, 256, 768), (130, 512, 320), (200, 2048, 1024), (300, 512, 4096),
             (512, 1024, 14336), (600, 768, 2048), (33, 384, 704)]

# Both tcgen05 kernels and every tile: chunks of at most 128 rows run 256
# weight rows x 32 / 64 / 128 tokens (weights in tensor memory), longer chunks
# 256 tokens x 256 / 192 / 128 weight rows; with whole tiles and with stream-K
# partial tiles (fewer tiles than CTA pairs and long k; a GB300 holds 76 pairs
# of the full forms and 152 of the lean short-chunk form): the 350M down
# projection at a 32-row chunk, a 64-row chunk over k = 8192, the 8B down
# projection at 512 rows, a ragged 300-row chunk with k not a multiple of the
# 1024-k segment, a 100-row chunk split 32 k-blocks per pair, and a 24-row
# chunk over 96 weight tiles whose K is split into runs of 29 k-blocks (not a
# whole number of segments) across ~150 lean pairs.
WIDTH_SHAPES = [(16, 19456, 128), (40, 14592, 192), (290, 512, 1024), (32, 1024, 4096), (64, 2048, 8192),
                (512, 4096, 14336), (512, 28672, 4096), (300, 4096, 2880), (100, 4096, 4096), (24, 24576, 2880)]


@pytest.mark.parametrize("m,n,k", TC_SHAPES)
def test_tc_acc_bit_exact(torch, m, n, k):
    a = synth.uniform_i8(81, m * 3 + k, (m, k))
    w = synth.uniform_i8(82, n * 5 + k, (n, k))
    assert np.array_equal(_acc(torch, TC, a, w), oracle.gemm_i8(a, w))


def test_tc_adversarial_extremes(torch):
    m, n, k = 256, 512, 14336
    a = np.full((m, k), 127, np.int8)
    a[1::2] = -127
    w = np.full((n, k), 127, np.int8)
    w[1::3] = -127
    w[2::3, ::2] = -127
    got = _acc(torch, TC, a, w)
    assert got[0, 0] == 127 * 127 * k and got[1, 0] == -127 * 127 * k and got[0, 1] == -127 * 127 * k
    assert np.array_equal(got, oracle.gemm_i8(a, w))


@pytest.mark.parametrize("seg", [64, 256, 1024])
def test_tc_segment_length_is_invisible(torch, seg):
    m, n, k = 96, 512, 4096
    a = synth.uniform_i8(83, 1, (m, k))
    w = synth.uniform_i8(83, 2, (n, k))
    try:
        pp.pp_set_exact_segment(seg)
        got = _acc(torch, TC, a, w)
    finally:
        pp.pp_set_exact_segment(1024)
    assert np.array_equal(got, oracle.gemm_i8(a, w))


def test_tc_and_mma_engines_agree_at_8b_shapes(torch):
    # the bench's launch shapes: QKV, O, gate/up, down at 512 tokens
    for (n, k) in ((6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336)):
        m = 512
        a = synth.uniform_i8(84, n, (m, k))
        w = synth.uniform_i8(85, n + k, (n, k))
        tc = _acc(torch, TC, a, w)
        mma = _acc(torch, pp.PP_GEMM_MMA, a, w)
        assert np.array_equal(tc, mma), (n, k)
        rng = np.random.default_rng(n)
        for t, r in zip(rng.integers(0, m, 64), rng.integers(0, n, 64)):
            assert tc[t, r] == oracle.dot_i8(a[t], w[r])


def test_short_chunk_shapes_plan_stream_k(torch):
    # the stream-K cases above are stream-K on this device (the plan depends on its SM count)
    for m, n, k in ((32, 1024, 4096), (64, 2048, 8192), (100, 4096, 4096), (24, 24576, 2880)):
        part, counters = pp.pp_op_gemm_noalloc_need(m, n, k)
        assert part > 0 and counters > 0, (m, n, k)


@pytest.mark.parametrize("m,n,k", WIDTH_SHAPES)
def test_tc_acc_bit_exact_every_token_tile(torch, m, n, k):
    a = synth.uniform_i8(88, m + k, (m, k))
    w = synth.uniform_i8(88, n + k, (n, k))
    assert np.array_equal(_acc(torch, TC, a, w), oracle.gemm_i8(a, w))


@pytest.mark.parametrize("m,n,k", WIDTH_SHAPES)
@pytest.mark.parametrize("epi", [pp.PP_EPI_STORE, pp.PP_EPI_RESID])
def test_tc_epilogue_bit_exact(torch, epi, m, n, k):
    a = synth.uniform_i8(86, 1, (m, k))
    w = synth.uniform_i8(86, 2, (n, k))
    ws = synth.uniform_f32(86, 3, (n,), 1e-4, 2e-3)
    as_ = synth.uniform_f32(86, 4, (m,), 1e-3, 5e-2)
    x0 = synth.normal_f32(86, 5, (m, n), 0.0, 2.0)
    out = dev(x0) if epi == pp.PP_EPI_RESID else empty((m, n), torch.float32)
    pp.pp_op_gemm(TC, epi, dev(a), dev(a.astype(np.float16)), dev(w), dev(ws), dev(as_), m, n, k, out, n)
    ref = oracle.dequant_block(oracle.gemm_i8(a, w), ws, as_)
    if epi == pp.PP_EPI_RESID:
        ref = (x0 + ref).astype(np.float32)
    assert np.array_equal(bits(host(out)), bits(ref))


@pytest.mark.parametrize("m,F,k", [(70, 256, 512), (16, 9728, 128), (40, 7296, 192)])
def test_tc_swiglu(torch, m, F, k):
    a = synth.uniform_i8(87, 1, (m, k))
    wg = synth.uniform_i8(87, 2, (F, k))
    wu = synth.uniform_i8(87, 3, (F, k))
    sg = synth.uniform_f32(87, 4, (F,), 1e-4, 1e-3)
    su = synth.uniform_f32(87, 5, (F,), 1e-4, 1e-3)
    as_ = synth.uniform_f32(87, 6, (m,), 1e-2, 5e-2)
    B = 16
    wgu = np.concatenate([np.concatenate([wg[b * B:(b + 1) * B], wu[b * B:(b + 1) * B]]) for b in range(F // B)])
    sgu = np.concatenate([np.concatenate([sg[b * B:(b + 1) * B], su[b * B:(b + 1) * B]]) for b in range(F // B)])
    out_tc = empty((m, F), torch.float32)
    out_mma = empty((m, F), torch.float32)
    for eng, out in ((TC, out_tc), (pp.PP_GEMM_MMA, out_mma)):
        pp.pp_op_gemm(eng, pp.PP_EPI_SWIGLU, dev(a), dev(a.astype(np.float16)), dev(wgu), dev(sgu), dev(as_), m,
                      2 * F, k, out, F)
    got = host(out_tc)
    g = oracle.dequant_block(oracle.gemm_i8(a, wg), sg, as_)
    u = oracle.dequant_block(oracle.gemm_i8(a, wu), su, as_)
    ref = np.vectorize(lambda x, y: float(oracle.silu_mul(x, y)), otypes=[np.float32])(g, u)
    # full-accuracy expf (<= 2 ulp) and IEEE add, division and multiply: within a few ulp of each value
    assert swiglu_close(got, ref)
    assert np.array_equal(bits(got), bits(host(out_mma)))  # same epilogue code, same integers


# gate values at and around the edges of the f32 exponential: exp(-g) overflows for g < -88.72, the
# quotient g / (1 + exp(-g)) is subnormal or near the smallest normal for g in about [-103, -87],
# and 1 + exp(-g) rounds to 1 for g > 16.6
EDGE_G = (-100.0, -88.0, -87.5, 0.0, 30.0, 88.0, -30.0, -5.0, 1.0, 16.0, 17.0, -16.5)


@pytest.mark.parametrize("eng", [TC, pp.PP_GEMM_MMA])
def test_swiglu_gate_edges(torch, eng):
    # Every token row is the one-hot code 1 at k = t, every gate row holds the code 127 at each k and a
    # row scale that puts g = (float(127) * s_g) * 1 at one of EDGE_G; up rows are random. Both engines
    # compute the same exact integers, so the epilogue sees the same g and u as the oracle.
    m, k, F = 64, 64, 192
    a = np.zeros((m, k), np.int8)
    a[np.arange(m), np.arange(m)] = 1
    wg = np.full((F, k), 127, np.int8)
    wu = synth.uniform_i8(85, 3, (F, k))
    sg = np.array([EDGE_G[r % len(EDGE_G)] / 127.0 for r in range(F)], np.float32)
    su = synth.uniform_f32(85, 5, (F,), 1e-3, 5e-2)
    as_ = np.ones((m,), np.float32)
    B = 16
    wgu = np.concatenate([np.concatenate([wg[b * B:(b + 1) * B], wu[b * B:(b + 1) * B]]) for b in range(F // B)])
    sgu = np.concatenate([np.concatenate([sg[b * B:(b + 1) * B], su[b * B:(b + 1) * B]]) for b in range(F // B)])
    out = empty((m, F), torch.float32)
    pp.pp_op_gemm(eng, pp.PP_EPI_SWIGLU, dev(a), dev(a.astype(np.float16)), dev(wgu), dev(sgu), dev(as_), m, 2 * F,
                  k, out, F)
    got = host(out)
    g = oracle.dequant_block(oracle.gemm_i8(a, wg), sg, as_)
    u = oracle.dequant_block(oracle.gemm_i8(a, wu), su, as_)
    assert np.allclose(g[0, :len(EDGE_G)], EDGE_G, rtol=1e-6, atol=0)  # the gate values reach the edges
    ref = np.vectorize(lambda x, y: float(oracle.silu_mul(x, y)), otypes=[np.float32])(g, u)
    assert np.all(np.isfinite(got))
    assert swiglu_close(got, ref)
    # the far negative gates give (signed) zero or a value within the subnormal floor
    far = np.array([EDGE_G[r % len(EDGE_G)] <= -87.5 for r in range(F)])
    assert np.abs(got[:, far]).max() <= 1e-35


def test_tc_shape_errors(torch):
    t8 = empty((1024,), torch.int8)
    t16 = empty((1024,), torch.float16)
    acc = empty((1024,), torch.int32)
    with pytest.raises(pp.PPError) as e:
        pp.pp_op_gemm_acc(TC, t8, t16, t8, 4, 96, 64, acc)  # n % 128 != 0
    assert e.value.status == pp.PP_ERR_ARG
    with pytest.raises(pp.PPError):
        pp.pp_set_exact_segment(2048)  # would overflow the exact f32 range
    with pytest.raises(pp.PPError):
        pp.pp_set_exact_segment(100)
