"""Failure paths, made on purpose without faulting the GPU.

* A bounded device wait that runs out: the tcgen05 GEMM with its MMA issuer
  held back (nothing ever completes an accumulator), every wait bounded to a
  few milliseconds. Each role must record the timeout, let its copies land,
  free its tensor memory and exit; the host reads PP_ERR_DEVICE_TIMEOUT and the
  device stays usable (a normal GEMM right after is exact).
* A loader that never prefetches ("Predictive prefetch": a miss blocks until
  the copy is ready): results unchanged, every layer visit a miss.
* An allocation cap: a load or a K/V growth past it fails with PP_ERR_OOM,
  leaks nothing, and the K/V rows written before stay intact.
"""
import numpy as np
import pytest

import oracle
import prompt_prefill_gb300 as pp
import synth
from tests.gpu_util import bits, dev, empty, host, load, torch_cuda

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_the_device_stays_usable():
    torch = torch_cuda()
    m, n, k = 256, 512, 1024
    a = synth.uniform_i8(91, 1, (m, k))
    w = synth.uniform_i8(91, 2, (n, k))
    a16, dw = dev(a.astype(np.float16)), dev(w)
    acc = empty((m, n), torch.int32)
    assert pp.pp_debug_gemm_stall(20000, a16, dw, m, n, k, acc) == pp.PP_ERR_DEVICE_TIMEOUT
    assert "bounded device wait" in pp.last_error()
    pp.pp_op_gemm_acc(pp.PP_GEMM_TC, dev(a), a16, dw, m, n, k, acc)
    torch.cuda.synchronize()
    assert np.array_equal(host(acc), oracle.gemm_i8(a, w))


@pytest.mark.parametrize("call", ["gemm", "gemm_acc", "noalloc"])
def test_single_step_gemm_reports_a_bounded_wait_that_runs_out(call):
    # The single-step GEMM calls share a device status word: with their MMA issuer held back and every
    # wait bounded to 20 ms (pp_debug_op_stall) each call's kernel gives up and records the timeout,
    # which pp_op_status reports once; normal calls afterwards are exact and report PP_OK.
    torch = torch_cuda()
    m, n, k = 512, 4096, 14336  # the down projection at 512 rows: stream-K partial tiles on a GB300
    a = synth.uniform_i8(92, 1, (m, k))
    w = synth.uniform_i8(92, 2, (n, k))
    ws = synth.uniform_f32(92, 3, (n,), 1e-4, 2e-3)
    as_ = synth.uniform_f32(92, 4, (m,), 1e-3, 5e-2)
    da, a16, dw, dws, das = dev(a), dev(a.astype(np.float16)), dev(w), dev(ws), dev(as_)
    out = empty((m, n), torch.float32)
    acc = empty((m, n), torch.int32)

    def run():
        if call == "gemm":
            pp.pp_op_gemm(pp.PP_GEMM_TC, pp.PP_EPI_STORE, da, a16, dw, dws, das, m, n, k, out, n)
        elif call == "gemm_acc":
            pp.pp_op_gemm_acc(pp.PP_GEMM_TC, da, a16, dw, m, n, k, acc)
        else:
            pp.pp_op_gemm_noalloc(pp.PP_EPI_STORE, a16, dw, dws, das, m, n, k, out, n)

    assert pp.pp_op_status() == pp.PP_OK
    pp.pp_debug_op_stall(20000)
    try:
        run()
    finally:
        pp.pp_debug_op_stall(0)
    assert pp.pp_op_status() == pp.PP_ERR_DEVICE_TIMEOUT
    assert "bounded device wait" in pp.last_error()
    assert pp.pp_op_status() == pp.PP_OK  # reported once, then cleared
    run()
    assert pp.pp_op_status() == pp.PP_OK
    ref = oracle.gemm_i8(a, w)
    if call == "gemm_acc":
        assert np.array_equal(host(acc), ref)
    else:
        assert np.array_equal(bits(host(out)), bits(oracle.dequant_block(ref, ws, as_)))


def test_loader_without_prefetch_changes_nothing():
    torch_cuda()
    mod = synth.make_model(synth.CONFIGS["1b"])
    c = mod.cfg
    toks = synth.prompt(c, 300)
    g = load(mod, max_seq=1024, max_chunk=128, mode=pp.PP_MODE_STREAMED, ring_slots=2)
    ref = g.prefill(toks, 0, 128)
    pp.pp_debug_loader_fault(g.h, 1)
    g.kv_reset()
    g.reset_stats()
    got = g.prefill(toks, 0, 128)
    s = g.stats()
    pp.pp_debug_loader_fault(g.h, 0)
    g.close()
    assert np.array_equal(bits(got), bits(ref))
    assert s["prefetch_hits"] == 0 and s["prefetch_misses"] == 3 * c.n_layers


def test_allocation_cap_gives_oom_without_damage():
    torch_cuda()
    mod = synth.make_model(synth.CONFIGS["350m"])
    c = mod.cfg
    row = c.n_kv_heads * c.head_dim * 4
    try:
        pp.pp_debug_alloc_cap(1 << 20)  # far below the 350M model's weights
        with pytest.raises(pp.PPError) as e:
            load(mod, max_seq=1024, max_chunk=32)
        assert e.value.status == pp.PP_ERR_OOM
        pp.pp_debug_alloc_cap(0)
        g = load(mod, max_seq=8192, max_chunk=32, kv_grow=1)
        g.prefill(synth.prompt(c, 1), 0, 32)
        per_step = g.stats()["kv_bytes"] // (2 * c.n_layers) // row  # positions one growth step maps
        g.kv_reset()
        if per_step + 40 > 8192:
            pytest.skip(f"allocation granularity of {per_step} positions leaves no second step to refuse")
        n1 = per_step - 10  # the second call crosses into the next step
        toks = synth.prompt(c, n1 + 40)
        ref_g = load(mod, max_seq=8192, max_chunk=32)
        ref_g.prefill(toks[:n1], 0, 32)
        ref = ref_g.prefill(toks[n1:], n1, 32)
        ref_g.close()
        g.prefill(toks[:n1], 0, 32)
        kv_before = g.kv(3, 0, 0, n1)
        pp.pp_debug_alloc_cap(1)  # any further growth is over the cap
        assert pp.pp_prefill_rc(g.h, toks[n1:], n1, 32, c.vocab) == pp.PP_ERR_OOM
        assert np.array_equal(bits(g.kv(3, 0, 0, n1)), bits(kv_before))  # earlier rows intact
        pp.pp_debug_alloc_cap(0)
        got = g.prefill(toks[n1:], n1, 32)
        g.close()
        assert np.array_equal(bits(got), bits(ref))
    finally:
        pp.pp_debug_alloc_cap(0)


def test_chunk_overlap_sets_are_made_on_demand_and_resume_after_oom():
    # pp_set_chunk_overlap allocates nothing; a call of several chunks makes the scratch sets it needs first
    # (here over the cap: PP_ERR_OOM before anything is launched), and a later call resumes from there
    torch_cuda()
    mod = synth.make_model(synth.CONFIGS["350m"])
    c = mod.cfg
    toks = synth.prompt(c, 200)  # 7 chunks of 32
    ref_g = load(mod, max_seq=1024, max_chunk=32)
    ref = ref_g.prefill(toks, 0, 32)
    ref_kv = ref_g.kv(5, 1, 0, 200)
    ref_g.kv_reset()
    ref_one = ref_g.prefill(toks[:32], 0, 32)
    ref_g.close()
    g = load(mod, max_seq=1024, max_chunk=32)
    try:
        pp.pp_debug_alloc_cap(1)  # any further device allocation is over the cap
        g.set_chunk_overlap(True)
        one = g.prefill(toks[:32], 0, 32)  # a single chunk needs no second set
        assert np.array_equal(bits(one), bits(ref_one))
        g.kv_reset()
        assert pp.pp_prefill_rc(g.h, toks, 0, 32, c.vocab) == pp.PP_ERR_OOM
        pp.pp_debug_alloc_cap(0)
        g.kv_reset()
        got = g.prefill(toks, 0, 32)
        assert np.array_equal(bits(got), bits(ref))
        assert np.array_equal(bits(g.kv(5, 1, 0, 200)), bits(ref_kv))
    finally:
        pp.pp_debug_alloc_cap(0)
        g.close()

