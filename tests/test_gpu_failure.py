"""Failure detection on the GPU without a fault: every device-side wait is
bounded.  MOE_DEBUG_STALL_TEST keeps the forward's up-GEMM producer from
issuing any load, so the MMA and epilogue waits on it can never complete;
they must give up after the plan's wait_timeout_ns, record MOE_ERR_TIMEOUT in
the status word, free what they hold and exit, leaving the CUDA context usable
for the next plan."""
import time

import pytest
import torch

from mixture_experts_layer_19_gb300 import moe
from oracle import moe_ref
from tests.util import BF16_TOL, cpu_and_gpu_inputs, rel_err

pytestmark = pytest.mark.gpu


def test_stalled_producer_times_out_and_context_survives():
    flags = 0
    T, d, F, E, k = 256, 512, 512, 8, 2
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=3)
    timeout_ns = 50_000_000
    stalled = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, wait_timeout_ns=timeout_ns,
                                  debug_flags=moe.MOE_DEBUG_STALL_TEST | moe.MOE_DEBUG_SEPARATE_KERNELS | flags))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    stalled.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert stalled.device_status() == moe.MOE_ERR_TIMEOUT
    assert elapsed < 2.0, elapsed                  # the bound, not a hang (50 ms per wait chain)
    assert stalled.device_status() == 0            # reading the status cleared it
    # the context still runs correct work, on a fresh plan and on the same stream
    ok = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, debug_flags=flags))
    Y, saved = ok.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    assert ok.device_status() == 0
    Yr, _ = moe_ref.forward(h["X"], h["logits"], h["Wg"], h["Wu"], h["Wd"], k)
    assert rel_err(Y, Yr) <= BF16_TOL


def test_stalled_token_pass_times_out_and_context_survives():
    """The block-scaled weight gradients' token pass (a producer / quantiser
    ring in shared memory): with the producers stalled, the quantising warps'
    waits on the ring expire, the backward records MOE_ERR_TIMEOUT, and the
    next plan's backward runs cleanly and repeats bit for bit."""
    T, d, F, E, k = 256, 512, 512, 8, 2
    g, h = cpu_and_gpu_inputs(T, d, F, E, k, seed=5)
    dY = g["dY"]
    stalled = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=moe.MOE_MXFP8, wait_timeout_ns=50_000_000,
                                  debug_flags=moe.MOE_DEBUG_STALL_TEST))
    stalled.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    Y, saved = stalled.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    assert stalled.device_status() == 0            # the forward has no stall hook in block-scaled plans
    t0 = time.perf_counter()
    stalled.backward(dY, g["X"], g["Wg"], g["Wu"], g["Wd"], saved)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert stalled.device_status() == moe.MOE_ERR_TIMEOUT
    assert elapsed < 2.0, elapsed
    ok = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=moe.MOE_MXFP8))
    ok.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    _, saved2 = ok.forward(g["X"], g["logits"], g["Wg"], g["Wu"], g["Wd"])
    g1 = ok.backward(dY, g["X"], g["Wg"], g["Wu"], g["Wd"], saved2)
    g2 = ok.backward(dY, g["X"], g["Wg"], g["Wu"], g["Wd"], saved2)
    torch.cuda.synchronize()
    assert ok.device_status() == 0
    for name in ("dWg", "dWu", "dWd", "dX"):
        assert torch.isfinite(g1[name].float()).all()
        assert torch.equal(g1[name], g2[name]), name
