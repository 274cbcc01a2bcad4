"""Helpers for the GPU tests: device buffers through torch, the CUDA library
through its C ABI, the oracle on the CPU. Nothing here computes the method."""
import numpy as np

import prompt_prefill_gb300 as pp


def torch_cuda():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch


def dev(a: np.ndarray):
    """Host numpy array -> device torch tensor (same dtype, contiguous)."""
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def empty(shape, dtype):
    torch = torch_cuda()
    return torch.empty(shape, dtype=dtype, device="cuda")


def host(t) -> np.ndarray:
    torch = torch_cuda()
    torch.cuda.synchronize()
    return t.cpu().numpy()


def bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a).view(np.uint32)


def swiglu_close(got: np.ndarray, ref: np.ndarray, rel: float = 1e-6, floor: float = 1e-36) -> bool:
    """Each SwiGLU output within `rel` of the oracle's value (a few ulp of f32), with an
    absolute floor for results in the subnormal range (exp(-g) overflows for g < -88.7)."""
    d = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    return bool(np.all(d <= rel * np.abs(ref.astype(np.float64)) + floor))


def max_rel(a, b, scale) -> float:
    return float(np.abs(a.astype(np.float64) - b.astype(np.float64)).max() / scale)


def load(model, **kw) -> pp.PrefillModel:
    c = model.cfg
    kw.setdefault("max_seq", c.max_seq)
    kw.setdefault("max_chunk", max(c.chunk, 1))
    return pp.PrefillModel(c, model, **kw)


def logits_close(gpu: np.ndarray, ref: np.ndarray, tol: float = 1e-2):
    """End-to-end criterion: max|d| <= tol * std(ref) and the same top-1 token."""
    std = float(ref.astype(np.float64).std())
    err = float(np.abs(gpu.astype(np.float64) - ref.astype(np.float64)).max())
    top_ref = int(np.argmax(ref))
    s = np.sort(ref.astype(np.float64))
    gap = float(s[-1] - s[-2])
    return err <= tol * std, err / std, int(np.argmax(gpu)) == top_ref, gap / std


def layerwise_forced(model, g, toks, chunk, margin_tol=4e-3, calls=None, layers=None):
    """Verify a GPU prefill layer by layer against the oracle.

    calls: the prefill calls that cover toks, as (start_pos, n, chunk) in
    position order (default: one call of every token from position 0); later
    calls continue the K/V cache of earlier ones, on both sides.
    layers: the layers the oracle checks (default: all). Each checked layer
    runs on the GPU's own input rows, so any subset is a valid check of those
    layers while the GPU runs the whole model.

    The GPU runs with its trace on (residual stream at every layer boundary,
    int8 codes and scales at every quantisation point). For each layer the
    oracle runs the same layer on the GPU's input rows and takes, at each
    quantisation point, the GPU's codes in place of its own after recording
    where its own decision differs. Then:
      - the layer's output rows must equal the GPU's bit for bit (the integer
        GEMMs and the fixed-order f32 epilogue are exact given equal codes);
      - every code the two sides decided differently must differ by one and
        lie within `margin_tol` of a half-integer tie, i.e. be a rounding
        decision that the f32 (GPU) and double (oracle) evaluation of RMSNorm,
        attention or SiLU may legitimately take differently;
      - the K/V rows agree within f32 rounding of the RoPE evaluation.
    Deep random int8 models amplify any such tie decision through the layers,
    so whole-model comparison of two correct implementations is not a test;
    this check is. Returns (gpu logits, oracle logits of the GPU's final row,
    per-layer mismatch report).
    """
    import oracle

    torch = torch_cuda()
    c = model.cfg
    P = len(toks)
    kmax = max(c.dim, c.n_heads * c.head_dim, c.ffn)
    tx = torch.empty(((c.n_layers + 1) * P * c.dim,), dtype=torch.float32, device="cuda")
    tc = torch.zeros((c.n_layers * 4 * P * kmax,), dtype=torch.int8, device="cuda")
    ts = torch.empty((c.n_layers * 4 * P,), dtype=torch.float32, device="cuda")
    calls = calls or [(0, P, chunk)]
    assert calls[0][0] == 0 and all(a[0] + a[1] == b[0] for a, b in zip(calls, calls[1:]))
    assert calls[-1][0] + calls[-1][1] == P
    g.kv_reset()
    g.set_trace(tx, tc, ts, P)
    try:
        for start, n, ch in calls:
            logits = g.prefill(toks[start:start + n], start, ch)
    finally:
        g.set_trace(None, None, None, 0)
    X = host(tx).reshape(c.n_layers + 1, P, c.dim)
    codes = host(tc).reshape(c.n_layers, 4, P, kmax)
    scales = host(ts).reshape(c.n_layers, 4, P)
    assert np.array_equal(X[0], model.tok_emb[toks]), "layer-0 input is not the embedding gather"
    om = oracle.OracleModel(model, max_seq=P)
    widths = (c.dim, c.n_heads * c.head_dim, c.dim, c.ffn)
    report = []
    checked = list(range(c.n_layers)) if layers is None else sorted(layers)
    for start, n, _ in calls:
        rows = slice(start, start + n)
        for L in checked:
            y, st = om.layer_forced(L, X[L][rows], codes[L][:, rows], scales[L][:, rows], start)
            assert np.array_equal(bits(y), bits(X[L + 1][rows])), \
                f"layer {L}, positions {start}..: residual rows differ with equal codes"
            for pt in range(4):
                if st["mismatches"][pt]:
                    assert st["max_code_diff"][pt] == 1, (L, pt, st)
                    assert st["max_margin"][pt] <= margin_tol, (L, pt, st)
                    assert st["mismatches"][pt] <= 1e-3 * n * widths[pt], (L, pt, st)
                if st["scale_mismatches"][pt]:
                    assert st["max_scale_rel"][pt] <= 1e-5, (L, pt, st)
            report.append(st)
    for L in checked:
        for which in (0, 1):
            ref = om.kv(L, which)[:P]
            got = g.kv(L, which, 0, P)
            assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max(), (L, which)
    ref_logits = om.final_logits(X[c.n_layers][P - 1])
    om.close()
    return logits, ref_logits, report
