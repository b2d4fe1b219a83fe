"""Shared helpers for the GPU parity tests (inputs, oracle references, errors)."""
import numpy as np
import torch

from mixture_experts_layer_19_gb300.workload import LayerShape, make_inputs, to_f64

BF16_TOL = 2e-2     # max |gpu - oracle| / max |oracle| for bf16 GEMM outputs and gradients


def rel_err(gpu, ref):
    gpu = to_f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = np.abs(ref).max()
    if denom == 0:
        return float(np.abs(gpu).max())
    return float(np.abs(gpu - ref).max() / denom)


def rel_err_norm(gpu, ref):
    """Normwise relative error ||gpu - oracle||_2 / ||oracle||_2: the aggregate
    drift of a whole tensor, insensitive to a single element whose quantised
    code flips at a rounding boundary."""
    gpu = to_f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = np.linalg.norm(ref.ravel())
    diff = np.linalg.norm((gpu - ref).ravel())
    return float(diff if denom == 0 else diff / denom)


def cpu_and_gpu_inputs(T, d, F, E, k, seed=0, alpha=0.0, logits_fn=None):
    inp = make_inputs(LayerShape(T, d, F, E, k), seed=seed, alpha=alpha, device="cpu")
    if logits_fn is not None:
        inp.logits = logits_fn(inp.logits).contiguous()
    dev = torch.device("cuda", 0)
    g = {n: getattr(inp, n).to(dev) for n in ("X", "logits", "Wg", "Wu", "Wd", "dY")}
    h = {n: to_f64(getattr(inp, n)) for n in ("X", "logits", "Wg", "Wu", "Wd", "dY")}
    return g, h
