"""CUDA-graph replay of prefill calls (pp_set_graphs).

A call captured into a graph and replayed must compute exactly what the same
call launched kernel by kernel computes ("Batched Prefill", section
"Correctness": the batched path is checked against the per-token path, here
bit for bit): logits, K/V rows and statistics, for chunk-outer and
layer-outer order, with and without chunk overlap, for continuation calls,
through the host and the device entry points, and past the cache's size.
"""
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


def _counts(s):
    return {k: s[k] for k in ("calls", "chunks", "tokens", "weight_bytes_read", "kernel_launches", "gemm_launches")}


@pytest.mark.parametrize("loop,overlap", [(pp.PP_LOOP_CHUNK_OUTER, False), (pp.PP_LOOP_CHUNK_OUTER, True),
                                          (pp.PP_LOOP_LAYER_OUTER, True)])
def test_graph_replay_equals_launch_by_launch(model_1b, loop, overlap):
    torch = torch_cuda()
    m = model_1b
    c = m.cfg
    toks = synth.prompt(c, 1200)
    g = load(m, max_seq=2048, max_chunk=256, loop_order=loop)
    try:
        g.set_chunk_overlap(overlap)
        # launch by launch: a first call, a continuation, their logits, K/V rows and counters
        g.reset_stats()
        ref1 = g.prefill(toks[:700], 0, 256)
        ref2 = g.prefill(toks[700:], 700, 128)
        ref_stats = _counts(g.stats())
        ref_kv = [g.kv(L, w, 0, 1200) for L in (0, c.n_layers - 1) for w in (0, 1)]
        g.set_graphs(True)
        for rep in range(3):  # capture, then two replays
            g.kv_reset()
            g.reset_stats()
            got1 = g.prefill(toks[:700], 0, 256)
            got2 = g.prefill(toks[700:], 700, 128)
            assert np.array_equal(bits(got1), bits(ref1)), rep
            assert np.array_equal(bits(got2), bits(ref2)), rep
            assert _counts(g.stats()) == ref_stats, rep
            kv = [g.kv(L, w, 0, 1200) for L in (0, c.n_layers - 1) for w in (0, 1)]
            for a, b in zip(kv, ref_kv):
                assert np.array_equal(bits(a), bits(b)), rep
        # the device entry point on the caller's stream, replayed on another stream
        d_tok = torch.from_numpy(toks[:700]).cuda()
        d_logits = torch.empty(c.vocab, dtype=torch.float32, device="cuda")
        side = torch.cuda.Stream()
        for st in (torch.cuda.current_stream(), side, torch.cuda.current_stream()):
            g.kv_reset()
            g.prefill_device(d_tok, 700, 0, 256, d_logits, st)
            st.synchronize()
            assert np.array_equal(bits(d_logits.cpu().numpy()), bits(ref1))
        assert g.device_status() == pp.PP_OK
    finally:
        g.close()


def test_graph_cache_evicts_and_stays_exact(model_1b):
    # more distinct calls than the cache holds (8), each checked against the launch-by-launch result
    m = model_1b
    toks = synth.prompt(m.cfg, 600)
    g = load(m, max_seq=1024, max_chunk=128)
    try:
        refs = {}
        shapes = [(n, ch) for n in (100, 250, 600) for ch in (32, 64, 128)]  # 9 shapes
        for n, ch in shapes:
            g.kv_reset()
            refs[(n, ch)] = g.prefill(toks[:n], 0, ch)
        g.set_graphs(True)
        for _ in range(2):
            for n, ch in shapes:
                g.kv_reset()
                assert np.array_equal(bits(g.prefill(toks[:n], 0, ch)), bits(refs[(n, ch)])), (n, ch)
        g.set_graphs(False)
        g.kv_reset()
        assert np.array_equal(bits(g.prefill(toks[:100], 0, 32)), bits(refs[(100, 32)]))
    finally:
        g.close()


def test_graphs_step_aside_while_profiling(model_1b):
    # a profiled kernel class needs its per-launch events: those calls run launch by launch and still
    # count their launches
    m = model_1b
    toks = synth.prompt(m.cfg, 300)
    g = load(m, max_seq=512, max_chunk=128)
    try:
        ref = g.prefill(toks, 0, 128)
        g.set_graphs(True)
        g.set_profile_kernel(pp.PP_KERNEL_ATTENTION)
        g.reset_stats()
        g.kv_reset()
        got = g.prefill(toks, 0, 128)
        s = g.stats()
        assert np.array_equal(bits(got), bits(ref))
        assert s["prof_launches"] == 3 * m.cfg.n_layers and s["prof_ms"] > 0
    finally:
        g.close()
