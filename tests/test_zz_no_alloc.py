"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (code inside a host framework whose allocator already owns the
device memory, or latency-critical paths that cannot afford an allocation)
cannot create a plan, because moe_plan allocates.  This entry point keeps its
scratch in a fixed array inside the library instead.  The test calls it
through the C ABI twice in a row, with different shapes so the second call
runs over the first call's leftovers, and checks both results against the
CPU oracle's routing and layout (bit-exact ids, counts, offsets, permutation
and destinations; weights within 1e-6) and against the routing moe_forward
stores (read back with moe_get_routing).  Collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_19_gb300 import moe
from oracle import moe_ref
from tests.util import cpu_and_gpu_inputs

pytestmark = pytest.mark.gpu


def _noalloc_routing(T, E, k, logits):
    dev = logits.device
    out = {
        "idx": torch.full((T, k), -7, dtype=torch.int32, device=dev),
        "w": torch.full((T, k), -7.0, dtype=torch.float32, device=dev),
        "counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
        "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        "perm_src": torch.full((T * k,), -7, dtype=torch.int32, device=dev),
        "dest": torch.full((T, k), -7, dtype=torch.int32, device=dev),
    }
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = moe.lib().moe_route_noalloc(T, E, k, p(logits), p(out["idx"]), p(out["w"]), p(out["counts"]),
                                     p(out["offsets"]), p(out["perm_src"]), p(out["dest"]),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, moe.lib().moe_last_error()
    return out


def _plan_routing(T, d, E, k, X, logits):
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=256, E=E, k=k, debug_flags=moe.MOE_DEBUG_IDENTITY_EXPERTS))
    _, saved = plan.forward(X, logits, None, None, None)
    return plan.routing(saved, T)


def test_noalloc_routing_matches_plan_routing_two_calls():
    for (T, d, E, k, alpha) in [(1000, 256, 32, 4, 1.1), (300, 256, 16, 2, 0.0)]:
        g, h = cpu_and_gpu_inputs(T, d, 256, E, k, seed=T, alpha=alpha)
        got = _noalloc_routing(T, E, k, g["logits"])
        ref = _plan_routing(T, d, E, k, g["X"], g["logits"])
        torch.cuda.synchronize()
        idx_o, w_o = moe_ref.route(h["logits"], k)
        lay = moe_ref.layout(idx_o, E)
        oracle = {"idx": idx_o, "counts": lay["counts"], "offsets": lay["offsets"],
                  "perm_src": lay["perm_src"], "dest": lay["dest"]}
        for key in ("idx", "counts", "offsets", "perm_src", "dest"):
            assert np.array_equal(got[key].cpu().numpy(), oracle[key]), key
            assert torch.equal(got[key], ref[key]), key
        assert np.abs(got["w"].cpu().numpy() - w_o).max() <= 1e-6
        assert (got["w"] - ref["w"]).abs().max().item() <= 1e-6


def test_noalloc_rejects_sizes_beyond_its_array():
    dev = torch.device("cuda", 0)
    dummy = torch.zeros(16, dtype=torch.int32, device=dev)
    p = ctypes.c_void_p(dummy.data_ptr())
    T, E, k = 200_000, 256, 8
    st = moe.lib().moe_route_noalloc(T, E, k, p, p, p, p, p, p, p, ctypes.c_void_p(0))
    assert st == 2  # MOE_ERR_UNSUPPORTED, nothing enqueued
    assert b"scratch" in moe.lib().moe_last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(dummy).item() == 0
