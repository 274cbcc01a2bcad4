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
