"""Streamed weights ("Predictive prefetch", section "The fix: an async
double-buffer ring"): layers live in pinned host memory and are copied into a
device ring on a side stream, layer L+1 while layer L computes. The backend
never changes results ("Three backends, one truth"): streamed with one or two
slots must equal resident bit for bit; only the counters differ."""
import numpy as np
import pytest

import prompt_prefill_gb300 as pp
import synth
from tests.gpu_util import bits, load, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def model_1b():
    torch_cuda()
    return synth.make_model(synth.CONFIGS["1b"])


def _layer_block_bytes(c):
    # size of one packed layer block (256-byte aligned sections), as copied per layer visit
    def up(x):
        return (x + 255) // 256 * 256
    D, F, QD, QKV = c.dim, c.ffn, c.n_heads * c.head_dim, c.qkv_rows
    return (up(QKV * D) + up(D * QD) + up(2 * F * D) + up(D * F) + up(4 * QKV) + up(4 * D) + up(8 * F) + up(4 * D)
            + up(4 * D) + up(4 * D))


@pytest.mark.parametrize("prompt,chunk", [(300, 128), (512, 512)])
def test_streamed_equals_resident(model_1b, prompt, chunk):
    m = model_1b
    c = m.cfg
    toks = synth.prompt(c, prompt)
    res = load(m, max_seq=1024, max_chunk=chunk)
    ref = res.prefill(toks, 0, chunk)
    res.close()
    n_chunks = -(-prompt // chunk)
    for slots in (2, 1):
        g = load(m, max_seq=1024, max_chunk=chunk, mode=pp.PP_MODE_STREAMED, ring_slots=slots)
        g.reset_stats()
        got = g.prefill(toks, 0, chunk)
        s = g.stats()
        g.close()
        assert np.array_equal(bits(got), bits(ref)), slots
        visits = n_chunks * c.n_layers
        assert s["h2d_bytes"] == visits * _layer_block_bytes(c) + 4 * prompt
        assert s["prefetch_hits"] + s["prefetch_misses"] == visits
        if slots == 1:
            assert s["prefetch_hits"] == 0  # one slot: every load waits for the previous layer's compute
        # weights read by the GEMMs are the same in both modes
        layer_w = c.layer_bytes() + 4 * (c.qkv_rows + c.dim + 2 * c.ffn + c.dim)
        assert s["weight_bytes_read"] == n_chunks * c.n_layers * layer_w + c.vocab * c.dim + 4 * c.vocab


def test_streamed_continuation_and_chunk_invariance(model_1b):
    m = model_1b
    toks = synth.prompt(m.cfg, 384)
    g = load(m, max_seq=1024, max_chunk=256, mode=pp.PP_MODE_STREAMED, ring_slots=2)
    whole = g.prefill(toks, 0, 256)
    g.kv_reset()
    g.prefill(toks[:100], 0, 64)
    cont = g.prefill(toks[100:], 100, 128)
    g.close()
    assert np.array_equal(bits(whole), bits(cont))


@pytest.mark.parametrize("side_stream", [False, True])
def test_streamed_device_call_is_ordered_on_the_callers_stream(model_1b, side_stream):
    """pp_prefill_device in streamed mode: the copies and the compute run on
    the model's own streams, joined to the caller's stream at both ends. Work
    enqueued on the caller's stream after the call (CUDA events, a copy of the
    logits) must see the whole call: the events bracket at least the time the
    layer copies need at 1 TB/s (well above any host link), and the logits
    read on that stream alone equal the host path's."""
    torch = torch_cuda()
    m = model_1b
    c = m.cfg
    toks = synth.prompt(c, 256)
    g = load(m, max_seq=1024, max_chunk=256, mode=pp.PP_MODE_STREAMED, ring_slots=2)
    ref = g.prefill(toks, 0, 256)
    d_tok = torch.from_numpy(toks).cuda()
    d_logits = torch.zeros(c.vocab, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream() if side_stream else torch.cuda.current_stream()
    g.reset_stats()
    with torch.cuda.stream(s):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        g.prefill_device(d_tok, len(toks), 0, 256, d_logits, s)
        e1.record(s)
        out = d_logits.clone()
    s.synchronize()
    got = out.cpu().numpy()
    ms = e0.elapsed_time(e1)
    h2d = g.stats()["h2d_bytes"]
    g.close()
    assert np.array_equal(bits(got), bits(ref))
    assert ms >= h2d / 1e12 * 1e3, f"{ms:.3f} ms for {h2d} bytes of layer copies"
