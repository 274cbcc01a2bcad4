"""End-to-end parity of the GPU prefill with the oracle, and the invariants
the pages state, through the C ABI.

Criteria: final-position logits within 1e-2 x std(oracle logits) and the
same top-1 token; the GPU's chunked path bit-identical to its own chunk = 1
path ("Batched Prefill", "Correctness": byte-identical output); continuation
and causality bit-identical ("Single-pass prefill": per-position results do
not change).
"""
import numpy as np
import pytest

import oracle
import prompt_prefill_gb300 as pp
import synth
from tests.gpu_util import bits, layerwise_forced, load, logits_close, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    torch_cuda()
    m = synth.make_model(synth.CONFIGS["tiny"])
    g = load(m, max_seq=64, max_chunk=64)
    yield m, g
    g.close()


def _assert_e2e(gpu, ref, label=""):
    ok, rel, top_ok, gap = logits_close(gpu, ref)
    assert ok, f"{label}: max|d| = {rel:.3g} x std"
    if gap > 1e-2:  # top-1 is well conditioned
        assert top_ok, f"{label}: top-1 differs (oracle top-2 gap {gap:.3g} x std)"


def test_tiny_matches_oracle(tiny):
    m, g = tiny
    toks = synth.prompt(m.cfg)
    g.kv_reset()
    got = g.prefill(toks, 0, 8)
    ref = oracle.OracleModel(m).prefill(toks, 0, 8)
    _assert_e2e(got, ref, "tiny")


def test_tiny_kv_cache_matches_oracle(tiny):
    m, g = tiny
    toks = synth.prompt(m.cfg)
    g.kv_reset()
    g.prefill(toks, 0, 8)
    om = oracle.OracleModel(m)
    om.prefill(toks, 0, 8)
    for L in range(m.cfg.n_layers):
        for which in (0, 1):
            a = g.kv(L, which, 0, 32)
            b = om.kv(L, which)[:32]
            assert np.abs(a - b).max() <= 1e-2 * b.std(), (L, which)


@pytest.mark.parametrize("chunk", [3, 8, 32, 64])
def test_tiny_chunked_equals_per_token(tiny, chunk):
    m, g = tiny
    toks = synth.prompt(m.cfg)
    g.kv_reset()
    ref = g.prefill(toks, 0, 1)
    kref = g.kv(3, 0, 0, 32)
    g.kv_reset()
    got = g.prefill(toks, 0, chunk)
    assert np.array_equal(bits(got), bits(ref))
    assert np.array_equal(bits(g.kv(3, 0, 0, 32)), bits(kref))


def test_tiny_forward_one_loop(tiny):
    m, g = tiny
    toks = synth.prompt(m.cfg, 12)
    g.kv_reset()
    for i, t in enumerate(toks):
        last = g.forward_one(int(t), i)
    g.kv_reset()
    assert np.array_equal(bits(last), bits(g.prefill(toks, 0, 5)))


def test_tiny_continuation_and_causality(tiny):
    m, g = tiny
    toks = synth.prompt(m.cfg, 40)
    g.kv_reset()
    whole = g.prefill(toks, 0, 8)
    k_whole = g.kv(2, 1, 0, 40)
    g.kv_reset()
    first = g.prefill(toks[:23], 0, 8)
    k_first = g.kv(2, 1, 0, 23)
    cont = g.prefill(toks[23:], 23, 8)
    assert np.array_equal(bits(whole), bits(cont))
    assert np.array_equal(bits(k_whole[:23]), bits(k_first))  # later tokens never touch earlier rows
    g.kv_reset()
    assert np.array_equal(bits(g.prefill(toks[:23], 0, 6)), bits(first))


def test_tiny_max_capacity_and_ragged(tiny):
    m, g = tiny
    toks = synth.tokens(77, 64, m.cfg.vocab)
    g.kv_reset()
    got = g.prefill(toks, 0, 9)  # 64 = 7 x 9 + 1: ragged last chunk, exactly max_seq
    ref = oracle.OracleModel(m).prefill(toks, 0, 9)
    _assert_e2e(got, ref, "tiny max_seq")


def test_stats_weight_bytes_once_per_chunk(tiny):
    m, g = tiny
    c = m.cfg
    g.kv_reset()
    g.reset_stats()
    g.prefill(synth.prompt(c), 0, 8)  # 32 tokens -> 4 chunks
    s = g.stats()
    layer_w = c.layer_bytes() + 4 * (c.qkv_rows + c.dim + 2 * c.ffn + c.dim)
    head = c.vocab * c.dim + 4 * c.vocab
    assert s["chunks"] == 4 and s["tokens"] == 32 and s["calls"] == 1
    assert s["weight_bytes_read"] == 4 * c.n_layers * layer_w + head
    assert s["h2d_bytes"] == 32 * 4
    g.reset_stats()
    g.prefill(synth.prompt(c), 0, 1)  # per-token path reads the model once per token
    assert g.stats()["weight_bytes_read"] == 32 * c.n_layers * layer_w + head


def test_argument_errors(tiny):
    m, g = tiny
    V = m.cfg.vocab
    assert pp.pp_prefill_rc(g.h, np.zeros(0, np.int32), 0, 8, V) == pp.PP_ERR_ARG
    assert pp.pp_prefill_rc(g.h, np.ones(4, np.int32), 0, 0, V) == pp.PP_ERR_ARG
    assert pp.pp_prefill_rc(g.h, np.ones(4, np.int32), 0, 65, V) == pp.PP_ERR_ARG  # chunk > max_chunk
    assert pp.pp_prefill_rc(g.h, np.ones(4, np.int32), -1, 8, V) == pp.PP_ERR_ARG
    assert pp.pp_prefill_rc(g.h, np.array([1, V], np.int32), 0, 8, V) == pp.PP_ERR_ARG
    assert pp.pp_prefill_rc(g.h, np.ones(65, np.int32), 0, 8, V) == pp.PP_ERR_CAPACITY
    assert pp.pp_prefill_rc(g.h, np.ones(2, np.int32), 63, 8, V) == pp.PP_ERR_CAPACITY


def test_device_path_flags_bad_token(tiny):
    torch = torch_cuda()
    m, g = tiny
    d_tok = torch.tensor([1, 2, m.cfg.vocab + 5], dtype=torch.int32, device="cuda")
    d_logits = torch.empty(m.cfg.vocab, dtype=torch.float32, device="cuda")
    g.kv_reset()
    g.prefill_device(d_tok, 3, 0, 8, d_logits)
    assert g.device_status() == pp.PP_ERR_ARG
    assert g.device_status() == pp.PP_OK  # cleared after being read


def test_device_path_equals_host_path(tiny):
    torch = torch_cuda()
    m, g = tiny
    toks = synth.prompt(m.cfg)
    g.kv_reset()
    ref = g.prefill(toks, 0, 8)
    g.kv_reset()
    d_logits = torch.empty(m.cfg.vocab, dtype=torch.float32, device="cuda")
    g.prefill_device(torch.from_numpy(toks).cuda(), len(toks), 0, 8, d_logits)
    torch.cuda.synchronize()
    assert np.array_equal(bits(d_logits.cpu().numpy()), bits(ref))


def test_device_path_on_a_side_stream(tiny):
    """The call is enqueued on the stream it is given: a copy of the logits
    enqueued on that stream afterwards, waited for on that stream alone, sees
    the result."""
    torch = torch_cuda()
    m, g = tiny
    toks = synth.prompt(m.cfg)
    g.kv_reset()
    ref = g.prefill(toks, 0, 8)
    g.kv_reset()
    d_tok = torch.from_numpy(toks).cuda()
    d_logits = torch.zeros(m.cfg.vocab, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.prefill_device(d_tok, len(toks), 0, 8, d_logits, s)
        out = d_logits.clone()
    s.synchronize()
    assert np.array_equal(bits(out.cpu().numpy()), bits(ref))


# ------------------------------------------------------------------ 350M class
def _summary(report):
    return [(sum(st["mismatches"]), max(st["max_margin"])) for st in report]


def test_350m_layer_by_layer_and_logits():
    torch_cuda()
    c = synth.CONFIGS["350m"]
    m = synth.make_model(c)
    toks = synth.prompt(c)  # 747 tokens, chunk 32 -> 23 full chunks + 1 of 11
    g = load(m, max_seq=c.max_seq, max_chunk=32)
    try:
        g.reset_stats()
        got, ref, report = layerwise_forced(m, g, toks, 32)
        s = g.stats()
    finally:
        g.close()
    print("350m per-layer (tie decisions, max margin):", _summary(report))
    _assert_e2e(got, ref, "350m final")
    layer_w = c.layer_bytes() + 4 * (c.qkv_rows + c.dim + 2 * c.ffn + c.dim)
    assert s["weight_bytes_read"] == 24 * c.n_layers * layer_w + c.vocab * c.dim + 4 * c.vocab


# ------------------------------------------------------------------ 1B class
@pytest.fixture(scope="module")
def one_b():
    torch_cuda()
    c = synth.CONFIGS["1b"]
    m = synth.make_model(c)
    g = load(m, max_seq=4096, max_chunk=2048)
    yield m, g
    g.close()


def test_1b_chunk_sweep_bit_identical(one_b):
    m, g = one_b
    toks = synth.prompt(m.cfg, 2048)
    outs = {}
    for chunk in (32, 128, 512, 2048):
        g.kv_reset()
        outs[chunk] = g.prefill(toks, 0, chunk)
    for chunk in (128, 512, 2048):
        assert np.array_equal(bits(outs[chunk]), bits(outs[32])), chunk


def test_1b_second_call_continues_cache(one_b):
    m, g = one_b
    toks = synth.prompt(m.cfg, 4096)
    g.kv_reset()
    g.prefill(toks[:2048], 0, 512)
    second = g.prefill(toks[2048:], 2048, 512)
    g.kv_reset()
    whole = g.prefill(toks, 0, 512)
    assert np.array_equal(bits(second), bits(whole))


def test_1b_layer_by_layer_and_logits(one_b):
    m, g = one_b
    toks = synth.prompt(m.cfg, 256)
    got, ref, report = layerwise_forced(m, g, toks, 128)
    print("1b per-layer (tie decisions, max margin):", _summary(report))
    _assert_e2e(got, ref, "1b final")


def test_chunk_overlap_both_engines():
    # tiny model, 32 tokens in chunks of 8 (fewer chunks than streams) and of 3 (11 chunks, more than
    # streams, so scratch sets are reused; a ragged last chunk): the serial bits with either GEMM engine
    # (the mma.sync path also keeps its RoPE kernel)
    torch_cuda()
    m = synth.make_model(synth.CONFIGS["tiny"])
    toks = synth.prompt(m.cfg)
    out = []
    for eng in (pp.PP_GEMM_MMA, pp.PP_GEMM_TC):
        for overlap in (False, True):
            g = load(m, max_seq=64, max_chunk=32, gemm_engine=eng)
            try:
                g.set_chunk_overlap(overlap)
                for chunk in (8, 3):
                    g.kv_reset()
                    out.append(g.prefill(toks, 0, chunk))
            finally:
                g.close()
    for o in out[1:]:
        assert np.array_equal(bits(o), bits(out[0]))


def test_engines_give_identical_logits():
    # the two GEMM engines compute the same integers, so whole prefills agree bit for bit
    torch_cuda()
    m = synth.make_model(synth.CONFIGS["tiny"])
    toks = synth.prompt(m.cfg)
    out = {}
    for eng in (pp.PP_GEMM_MMA, pp.PP_GEMM_TC):
        g = load(m, max_seq=64, max_chunk=32, gemm_engine=eng)
        assert g.gemm_engine == eng
        out[eng] = g.prefill(toks, 0, 8)
        g.close()
    assert np.array_equal(bits(out[pp.PP_GEMM_MMA]), bits(out[pp.PP_GEMM_TC]))


def test_head_dim_128_fused_rope_engines_and_oracle():
    # The 8B head layout (head_dim 128, 4 query heads per KV head, theta 5e5) on a 2-layer model. The
    # tcgen05 path applies RoPE and writes K/V in its QKV GEMM epilogue; the mma.sync path runs the RoPE
    # kernel on the same pair-ordered columns: logits and K/V rows agree bit for bit, the chunked prefill
    # equals the per-token one, and layer by layer (codes forced at tie decisions) the tcgen05 path matches
    # the oracle, as for the 350M and 1B classes.
    torch_cuda()
    cfg = synth.ModelConfig("hd128", 1024, 2, 8, 2, 128, 2048, 2048, rope_theta=500000.0, max_seq=256,
                            seed=4321, prompt_len=200, chunk=64)
    m = synth.make_model(cfg)
    toks = synth.prompt(cfg)
    out, kv = {}, {}
    for eng in (pp.PP_GEMM_MMA, pp.PP_GEMM_TC):
        g = load(m, max_seq=256, max_chunk=64, gemm_engine=eng)
        try:
            out[eng] = g.prefill(toks, 0, 64)
            kv[eng] = [g.kv(L, which, 0, len(toks)) for L in range(cfg.n_layers) for which in (0, 1)]
            if eng == pp.PP_GEMM_TC:
                g.kv_reset()
                assert np.array_equal(bits(g.prefill(toks, 0, 1)), bits(out[eng]))
                got, ref, report = layerwise_forced(m, g, toks, 64)
                assert np.array_equal(bits(got), bits(out[eng]))
        finally:
            g.close()
    assert np.array_equal(bits(out[pp.PP_GEMM_MMA]), bits(out[pp.PP_GEMM_TC]))
    for a, b in zip(kv[pp.PP_GEMM_MMA], kv[pp.PP_GEMM_TC]):
        assert np.array_equal(bits(a), bits(b))
    print("hd128 per-layer (tie decisions, max margin):", _summary(report))
    _assert_e2e(got, ref, "hd128 final")


def test_1b_chunk_overlap_bit_identical(one_b):
    # Chunks rotating over the overlap streams (each waits only for the previous chunk's K/V rows of a
    # layer) give the serial path's bits: logits, K/V rows, ragged chunks (21 chunks of 100), more chunks
    # than streams (64 chunks of 32 on 32 streams: chunk k + 32 reuses chunk k's stream and scratch set),
    # launch by launch and replayed from a graph, and a continuation call.
    m, g = one_b
    toks = synth.prompt(m.cfg)  # 2048 tokens
    g.kv_reset()
    ref = g.prefill(toks, 0, 256)
    kv_ref = [g.kv(L, which, 0, len(toks)) for L in (0, m.cfg.n_layers - 1) for which in (0, 1)]
    g.set_chunk_overlap(True)
    try:
        for chunk in (256, 512, 100, 32):
            g.kv_reset()
            assert np.array_equal(bits(g.prefill(toks, 0, chunk)), bits(ref)), chunk
            kv = [g.kv(L, which, 0, len(toks)) for L in (0, m.cfg.n_layers - 1) for which in (0, 1)]
            for a, b in zip(kv, kv_ref):
                assert np.array_equal(bits(a), bits(b)), chunk
        g.set_graphs(True)
        for _ in range(2):  # capture, then replay
            g.kv_reset()
            assert np.array_equal(bits(g.prefill(toks, 0, 32)), bits(ref))
        g.set_graphs(False)
        g.kv_reset()
        g.prefill(toks[:1000], 0, 256)
        assert np.array_equal(bits(g.prefill(toks[1000:], 1000, 256)), bits(ref))
    finally:
        g.set_graphs(False)
        g.set_chunk_overlap(False)
