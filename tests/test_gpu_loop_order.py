"""Layer-outer prefill over the whole prompt ("Single-pass prefill": each
layer is streamed once for the whole prompt) against the default chunk-outer
loop ("Batched Prefill", "The Solution"). Every position's computation is the
same in both orders -- the same kernels on the same rows, attention over the
same K/V rows in the same order -- so logits and the K/V cache must be equal
bit for bit; only the streamed-mode copy count changes (once per layer per
call instead of once per layer per chunk)."""
import numpy as np
import pytest

import prompt_prefill_gb300 as pp
import synth
from tests.gpu_util import bits, load, torch_cuda

pytestmark = pytest.mark.gpu


def _layer_block_bytes(c):
    def up(x):
        return (x + 255) // 256 * 256
    D, F, QD, QKV = c.dim, c.ffn, c.n_heads * c.head_dim, c.qkv_rows
    return (up(QKV * D) + up(D * QD) + up(2 * F * D) + up(D * F) + up(4 * QKV) + up(4 * D) + up(8 * F) + up(4 * D)
            + up(4 * D) + up(4 * D))


@pytest.fixture(scope="module")
def m350():
    torch_cuda()
    return synth.make_model(synth.CONFIGS["350m"])


@pytest.fixture(scope="module")
def m1b():
    torch_cuda()
    return synth.make_model(synth.CONFIGS["1b"])


def test_layer_outer_equals_chunk_outer_resident(m350):
    c = m350.cfg
    toks = synth.prompt(c)  # 747 tokens: 23 chunks of 32 and one of 11
    ref_g = load(m350, max_seq=1024, max_chunk=32)
    ref = ref_g.prefill(toks, 0, 32)
    ref_kv = [ref_g.kv(l, w, 0, len(toks)) for l in (0, c.n_layers - 1) for w in (0, 1)]
    ref_g.close()
    g = load(m350, max_seq=1024, max_chunk=32, loop_order=pp.PP_LOOP_LAYER_OUTER)
    got = g.prefill(toks, 0, 32)
    got_kv = [g.kv(l, w, 0, len(toks)) for l in (0, c.n_layers - 1) for w in (0, 1)]
    g.close()
    assert np.array_equal(bits(got), bits(ref))
    for a, b in zip(got_kv, ref_kv):
        assert np.array_equal(bits(a), bits(b))


def test_layer_outer_chunk_invariance_and_continuation(m350):
    toks = synth.prompt(m350.cfg)
    g = load(m350, max_seq=1024, max_chunk=64, loop_order=pp.PP_LOOP_LAYER_OUTER)
    whole = g.prefill(toks, 0, 64)
    g.kv_reset()
    g.prefill(toks[:300], 0, 17)
    cont = g.prefill(toks[300:], 300, 64)
    g.close()
    assert np.array_equal(bits(whole), bits(cont))


@pytest.mark.parametrize("slots", [2, 1])
def test_layer_outer_streamed_copies_each_layer_once(m1b, slots):
    c = m1b.cfg
    P, chunk = 700, 128
    toks = synth.prompt(c, P)
    res = load(m1b, max_seq=1024, max_chunk=chunk)
    ref = res.prefill(toks, 0, chunk)
    res.close()
    g = load(m1b, max_seq=1024, max_chunk=chunk, mode=pp.PP_MODE_STREAMED, ring_slots=slots,
             loop_order=pp.PP_LOOP_LAYER_OUTER)
    g.reset_stats()
    got = g.prefill(toks, 0, chunk)
    s = g.stats()
    g.close()
    assert np.array_equal(bits(got), bits(ref))
    assert s["h2d_bytes"] == c.n_layers * _layer_block_bytes(c) + 4 * P  # once per layer, not per chunk
    assert s["prefetch_hits"] + s["prefetch_misses"] == c.n_layers
    n_chunks = -(-P // chunk)
    layer_w = c.layer_bytes() + 4 * (c.qkv_rows + c.dim + 2 * c.ffn + c.dim)
    # the GEMMs still read every layer's weights once per chunk (from the ring slot)
    assert s["weight_bytes_read"] == n_chunks * c.n_layers * layer_w + c.vocab * c.dim + 4 * c.vocab


def test_layer_profile_resident(m350):
    """The per-layer profile: one visit per layer per chunk, compute time for
    every layer, no copy or wait in resident mode; profiling changes no bits."""
    c = m350.cfg
    toks = synth.prompt(c)[:200]
    g = load(m350, max_seq=1024, max_chunk=64)
    ref = g.prefill(toks, 0, 64)
    g.kv_reset()
    g.set_layer_profile(True)
    g.reset_stats()
    got = g.prefill(toks, 0, 64)
    prof = g.layer_profile()
    g.close()
    assert np.array_equal(bits(got), bits(ref))
    assert len(prof) == c.n_layers
    for p in prof:
        assert p["visits"] == 4  # 200 tokens in chunks of 64
        assert p["compute_ms"] > 0 and p["io_ms"] == 0 and p["wait_ms"] == 0


@pytest.mark.parametrize("slots,order", [(2, pp.PP_LOOP_CHUNK_OUTER), (1, pp.PP_LOOP_CHUNK_OUTER),
                                         (2, pp.PP_LOOP_LAYER_OUTER)])
def test_layer_profile_streamed(m1b, slots, order):
    """Streamed: every visit has a copy; with one slot the copy of a layer can
    only start once the previous layer's compute has freed the slot, so every
    layer after the first waits for its copy."""
    c = m1b.cfg
    P, chunk = 384, 128
    toks = synth.prompt(c, P)
    g = load(m1b, max_seq=1024, max_chunk=chunk, mode=pp.PP_MODE_STREAMED, ring_slots=slots, loop_order=order)
    ref = g.prefill(toks, 0, chunk)
    g.set_layer_profile(True)
    g.reset_stats()
    g.kv_reset()
    got = g.prefill(toks, 0, chunk)
    prof = g.layer_profile()
    s = g.stats()
    g.close()
    assert np.array_equal(bits(got), bits(ref))
    visits = 1 if order == pp.PP_LOOP_LAYER_OUTER else -(-P // chunk)
    assert all(p["visits"] == visits for p in prof)
    assert all(p["compute_ms"] > 0 and p["io_ms"] > 0 for p in prof)
    if slots == 1:
        assert all(p["wait_ms"] > 0 for p in prof[1:])
    assert s["prefetch_hits"] + s["prefetch_misses"] == visits * c.n_layers


def test_layer_outer_chunk_overlap_resident(m350):
    # the chunks of each layer rotating over the overlap streams: same bits as the serial chunk-outer order
    c = m350.cfg
    toks = synth.prompt(c)  # 747 tokens: 23 chunks of 32 and one of 11
    ref_g = load(m350, max_seq=1024, max_chunk=32)
    ref = ref_g.prefill(toks, 0, 32)
    ref_kv = [ref_g.kv(l, w, 0, len(toks)) for l in (0, c.n_layers - 1) for w in (0, 1)]
    ref_g.close()
    g = load(m350, max_seq=1024, max_chunk=32, loop_order=pp.PP_LOOP_LAYER_OUTER)
    try:
        g.set_chunk_overlap(True)
        got = g.prefill(toks, 0, 32)
        got_kv = [g.kv(l, w, 0, len(toks)) for l in (0, c.n_layers - 1) for w in (0, 1)]
        g.kv_reset()
        g.prefill(toks[:300], 0, 17)
        cont = g.prefill(toks[300:], 300, 32)
    finally:
        g.close()
    assert np.array_equal(bits(got), bits(ref))
    assert np.array_equal(bits(cont), bits(ref))
    for a, b in zip(got_kv, ref_kv):
        assert np.array_equal(bits(a), bits(b))


@pytest.mark.parametrize("slots", [2, 1])
def test_layer_outer_streamed_chunk_overlap(m1b, slots):
    # streamed weights, each layer's chunks rotating over the overlap streams (11 chunks: more than
    # streams): every stream waits for the layer's copy and the slot is released after all of them; same
    # bits and the same copies as without overlap
    c = m1b.cfg
    P, chunk = 700, 64
    toks = synth.prompt(c, P)
    res = load(m1b, max_seq=1024, max_chunk=chunk)
    ref = res.prefill(toks, 0, chunk)
    res.close()
    g = load(m1b, max_seq=1024, max_chunk=chunk, mode=pp.PP_MODE_STREAMED, ring_slots=slots,
             loop_order=pp.PP_LOOP_LAYER_OUTER)
    try:
        g.set_chunk_overlap(True)
        g.reset_stats()
        got = g.prefill(toks, 0, chunk)
        s = g.stats()
    finally:
        g.close()
    assert np.array_equal(bits(got), bits(ref))
    assert s["h2d_bytes"] == c.n_layers * _layer_block_bytes(c) + 4 * P
    assert s["prefetch_hits"] + s["prefetch_misses"] == c.n_layers
