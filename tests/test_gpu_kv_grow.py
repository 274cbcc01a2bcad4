"""Grow-on-demand K/V cache ("Single-pass prefill", "What it unlocked": prefill
pairs with grow-on-demand KV so memory stays bounded). With kv_grow the cache
is a reserved address range whose device memory is mapped only as far as the
positions written, and released by pp_kv_reset. Results must not change: the
kernels see the same addresses and the same rows."""
import numpy as np
import pytest

import prompt_prefill_gb300 as pp
import synth
from tests.gpu_util import bits, load, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m350():
    torch_cuda()
    return synth.make_model(synth.CONFIGS["350m"])


def _row_bytes(c):
    return c.n_kv_heads * c.head_dim * 4


def test_grow_equals_reserved(m350):
    c = m350.cfg
    toks = synth.prompt(c)  # 747 tokens
    ref_g = load(m350, max_seq=2048, max_chunk=32)
    ref = ref_g.prefill(toks, 0, 32)
    ref_kv = [ref_g.kv(l, w, 0, len(toks)) for l in (0, c.n_layers - 1) for w in (0, 1)]
    full = ref_g.stats()["kv_bytes"]
    ref_g.close()
    assert full == 2 * c.n_layers * 2048 * _row_bytes(c)  # reserved: the whole cache, always
    g = load(m350, max_seq=2048, max_chunk=32, kv_grow=1)
    assert g.stats()["kv_bytes"] == 0  # nothing mapped before the first call
    got = g.prefill(toks, 0, 32)
    got_kv = [g.kv(l, w, 0, len(toks)) for l in (0, c.n_layers - 1) for w in (0, 1)]
    grown = g.stats()["kv_bytes"]
    g.close()
    assert np.array_equal(bits(got), bits(ref))
    for a, b in zip(got_kv, ref_kv):
        assert np.array_equal(bits(a), bits(b))
    assert 2 * c.n_layers * len(toks) * _row_bytes(c) <= grown < full


def test_grow_continuation_reset_and_errors(m350):
    c = m350.cfg
    toks = synth.prompt(c)
    g = load(m350, max_seq=4096, max_chunk=64, kv_grow=1)
    whole = g.prefill(toks, 0, 64)
    b_whole = g.stats()["kv_bytes"]
    g.kv_reset()
    assert g.stats()["kv_bytes"] == 0  # released
    with pytest.raises(pp.PPError) as e:
        g.kv(0, 0, 0, 1)  # nothing written since the reset
    assert e.value.status == pp.PP_ERR_ARG
    g.prefill(toks[:100], 0, 64)
    b_100 = g.stats()["kv_bytes"]
    cont = g.prefill(toks[100:], 100, 37)
    b_cont = g.stats()["kv_bytes"]
    assert np.array_equal(bits(whole), bits(cont))
    assert 0 < b_100 <= b_cont == b_whole
    assert b_100 % (2 * c.n_layers) == 0
    assert pp.pp_prefill_rc(g.h, np.ones(8, np.int32), 4090, 8, c.vocab) == pp.PP_ERR_CAPACITY
    g.close()


def test_grow_with_chunk_overlap(m350):
    # memory mapped at the start of each call, chunks on the overlap streams: same bits as the reserved cache
    c = m350.cfg
    toks = synth.prompt(c)
    ref_g = load(m350, max_seq=2048, max_chunk=64)
    ref = ref_g.prefill(toks, 0, 64)
    ref_g.close()
    g = load(m350, max_seq=2048, max_chunk=64, kv_grow=1)
    try:
        g.set_chunk_overlap(True)
        g.prefill(toks[:200], 0, 64)
        got = g.prefill(toks[200:], 200, 64)  # grows the mapping, then continues the cache
    finally:
        g.close()
    assert np.array_equal(bits(got), bits(ref))
