"""Oracle parity at the 8B-shaped decoder's own dimensions, in the launch
configuration the benchmark times.

A 2-layer decoder with the Llama-3-8B shapes (dim 4096, FFN 14336, 32 query
heads over 8 KV heads of 128, RoPE theta 5e5; a smaller vocabulary) runs
1024 tokens in chunks of 512 with chunk overlap on and the tcgen05 engine (the
benchmark's policy: the chunks on their own streams, no stream-K), then a
continuation call of 512 tokens at position 1024, whose attention merges two
key ranges and whose single chunk takes the serial rule (the stream-K down
projection among them).

Checked ("Batched Prefill", section "Correctness": the batched path computes
what the per-token path computes):
  - which GEMM instantiations ran (pp_stats.gemm_launches), so the test
    provably covers the QKV/RoPE, SwiGLU and residual kernels with the
    256 x 256 tiles that the benchmark launches;
  - layer by layer against the oracle with codes forced at tie decisions
    (bit-exact residual rows, K/V rows within f32 rounding), on both calls;
  - the final logits from the GPU's last row within 1e-2 x std of the oracle's,
    with the same top-1 token;
  - tracing changes no bits.
"""
import numpy as np
import pytest

import prompt_prefill_gb300 as pp
import synth
from tests.gpu_util import bits, layerwise_forced, load, logits_close, torch_cuda

pytestmark = pytest.mark.gpu

CFG = synth.ModelConfig("8b-shape-2-layer", 4096, 2, 32, 8, 128, 14336, 16384, rope_theta=500000.0, max_seq=1536,
                        seed=4322, prompt_len=1536, chunk=512)
CALLS = [(0, 1024, 512), (1024, 512, 512)]


def test_8b_dims_chunk_overlap_matches_oracle():
    torch_cuda()
    m = synth.make_model(CFG)
    toks = synth.prompt(CFG)
    g = load(m, max_seq=CFG.max_seq, max_chunk=512, gemm_engine=pp.PP_GEMM_TC)
    try:
        assert g.gemm_engine == pp.PP_GEMM_TC
        g.set_chunk_overlap(True)
        # untraced pass: which kernels each call launches
        launches = []
        for start, n, ch in CALLS:
            g.reset_stats()
            ref_logits = g.prefill(toks[start:start + n], start, ch)
            launches.append(g.stats()["gemm_launches"])
        kv_ref = [g.kv(L, which, 0, CFG.prompt_len) for L in range(CFG.n_layers) for which in (0, 1)]
        L2 = CFG.n_layers * 2  # layers x chunks of the first call
        # 512-row chunks with chunk overlap: 256-token x 256-weight-row tiles for every projection
        T = (256, 256)
        assert launches[0] == {(4, T): L2, (2, T): L2, (1, T): 2 * L2}, launches[0]
        # the continuation's single chunk: serial tile rule, one launch per projection and layer
        by_epi = {}
        for (e, _), v in launches[1].items():
            by_epi[e] = by_epi.get(e, 0) + v
        assert by_epi == {4: CFG.n_layers, 2: CFG.n_layers, 1: 2 * CFG.n_layers}, launches[1]
        # traced pass (same policy): layer by layer against the oracle
        got, ref, report = layerwise_forced(m, g, toks, 512, calls=CALLS)
        assert np.array_equal(bits(got), bits(ref_logits)), "tracing changed the logits"
        kv = [g.kv(L, which, 0, CFG.prompt_len) for L in range(CFG.n_layers) for which in (0, 1)]
        for a, b in zip(kv, kv_ref):
            assert np.array_equal(bits(a), bits(b)), "tracing changed the K/V rows"
    finally:
        g.close()
    ok, rel, top_ok, gap = logits_close(got, ref)
    forced = [sum(st["mismatches"]) for st in report]
    print(f"8B dims: codes forced per layer and call {forced}, final logits max|d| = {rel:.3g} x std, "
          f"top-2 gap {gap:.3g} x std")
    assert ok, f"final logits max|d| = {rel:.3g} x std"
    if gap > 1e-2:
        assert top_ok
