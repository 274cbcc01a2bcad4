"""The C ABI library: builds, loads without a GPU, exports every symbol that
include/pp.h declares, and fails loudly (no CPU fallback) without a device."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pp.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pp_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libpp():
    from prompt_prefill_gb300 import _build

    _build.build()
    import prompt_prefill_gb300 as pp

    return pp.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pp_model_load", "pp_prefill", "pp_forward_one", "pp_prefill_device", "pp_kv_reset",
                     "pp_get_stats", "pp_model_free", "pp_op_gemm", "pp_op_attention", "pp_op_quantize"):
        assert required in names


def test_every_declared_symbol_is_exported(libpp):
    missing = [n for n in declared_functions() if not hasattr(libpp, n)]
    assert not missing, missing


def test_binding_covers_every_symbol():
    import prompt_prefill_gb300 as pp

    assert sorted(pp.SIGNATURES) == declared_functions()


def test_struct_layouts_match_header():
    import prompt_prefill_gb300 as pp

    text = open(HEADER).read()
    body = re.search(r"typedef struct pp_config \{(.*?)\} pp_config;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\b(int32_t|float)\s+(\w+);", body)
    assert [n for _, n in fields] == [n for n, _ in pp.pp_config._fields_]
    assert ctypes.sizeof(pp.pp_config) == 4 * len(fields)
    sbody = re.search(r"typedef struct pp_stats \{(.*?)\} pp_stats;", text, re.S).group(1)
    sbody = re.sub(r"/\*.*?\*/", "", sbody, flags=re.S)
    sfields = re.findall(r"\b(int64_t|double)\s+(\w+)((?:\[\d+\])*);", sbody)
    assert [n for _, n, _ in sfields] == [n for n, _ in pp.pp_stats._fields_]
    n_words = sum(int(np.prod([int(d) for d in re.findall(r"\d+", dims)] or [1])) for _, _, dims in sfields)
    assert ctypes.sizeof(pp.pp_stats) == 8 * n_words
    lbody = re.search(r"typedef struct pp_layer_profile \{(.*?)\} pp_layer_profile;", text, re.S).group(1)
    lbody = re.sub(r"/\*.*?\*/", "", lbody, flags=re.S)
    lfields = re.findall(r"\b(int64_t|double)\s+(\w+);", lbody)
    assert [n for _, n in lfields] == [n for n, _ in pp.pp_layer_profile._fields_]
    assert ctypes.sizeof(pp.pp_layer_profile) == 8 * len(lfields)


def test_status_strings(libpp):
    import prompt_prefill_gb300 as pp

    assert pp.status_str(pp.PP_OK) == "ok"
    assert pp.status_str(pp.PP_ERR_CAPACITY) == "KV capacity exceeded"
    assert pp.status_str(-99) == "unknown status"


def test_host_side_validation_needs_no_device(libpp):
    import prompt_prefill_gb300 as pp

    # null model / bad sizes are rejected on the host before any CUDA call
    assert libpp.pp_prefill(None, None, 4, 0, 8, None) == pp.PP_ERR_ARG
    assert libpp.pp_op_quantize(None, 1, 4, None, None, None, None) == pp.PP_ERR_ARG
    assert libpp.pp_op_gemm_acc(pp.PP_GEMM_MMA, None, None, None, 4, 32, 60, None, None) == pp.PP_ERR_ARG
    # the host-buffer checks validate before allocating or copying anything
    x = np.zeros((2, 6), np.float32)
    q, s = np.zeros((2, 6), np.int8), np.zeros(2, np.float32)
    assert libpp.pp_debug_quantize(x.ctypes.data, 2, 6, q.ctypes.data, s.ctypes.data) == pp.PP_ERR_ARG  # k % 4
    a, w, acc = np.zeros((4, 64), np.int8), np.zeros((48, 64), np.int8), np.zeros((4, 48), np.int32)
    assert libpp.pp_debug_gemm_i8(a.ctypes.data, w.ctypes.data, 4, 48, 64, acc.ctypes.data) == pp.PP_ERR_ARG  # n % 32
    assert libpp.pp_debug_gemm_i8(a.ctypes.data, w.ctypes.data, 4, 32, 60, acc.ctypes.data) == pp.PP_ERR_ARG  # k % 64
    assert libpp.pp_debug_gemm_i8(a.ctypes.data, w.ctypes.data, 4, 32, 64, None) == pp.PP_ERR_ARG
    out = np.zeros((4, 32), np.float32)
    assert libpp.pp_debug_gemm_epilogue(a.ctypes.data, w.ctypes.data, None, None, None, 4, 32, 64,
                                        out.ctypes.data) == pp.PP_ERR_ARG  # scales missing
    bad = pp.make_config(100, 1, 4, 4, 64, 256, 10)  # dim % 64 != 0
    h = ctypes.c_void_p()
    assert libpp.pp_model_load(ctypes.byref(bad), None, ctypes.byref(h)) == pp.PP_ERR_ARG
    bad = pp.make_config(128, 1, 4, 4, 64, 256, 10, loop_order=2)  # no such loop order
    assert libpp.pp_model_load(ctypes.byref(bad), None, ctypes.byref(h)) == pp.PP_ERR_ARG


def test_header_constants_match_binding():
    import prompt_prefill_gb300 as pp

    text = open(HEADER).read()
    defs = {k: int(v) for k, v in re.findall(r"#define\s+(PP_[A-Z0-9_]+)\s+(-?\d+)", text)}
    assert defs, "no constants found"
    for name, value in defs.items():
        assert getattr(pp, name) == value, name


def test_no_cpu_fallback_without_a_device(libpp):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    import prompt_prefill_gb300 as pp
    import synth

    m = synth.make_model(synth.CONFIGS["tiny"])
    with pytest.raises(pp.PPError) as e:
        pp.PrefillModel(m.cfg, m, max_seq=64, max_chunk=8)
    assert e.value.status == pp.PP_ERR_CUDA
