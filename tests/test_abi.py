"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every entry point include/moe.h declares, the pure-host minibatch floor
reproduces the figure the pages print, and argument errors come back
synchronously as status codes."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")
GOLDEN_FLOOR = os.path.join(ROOT, "tests", "golden", "minibatch_floor.txt")


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_19_gb300 import build as b
    b.build()
    from mixture_experts_layer_19_gb300 import moe
    return moe.load_library()


def _declared_symbols():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    from mixture_experts_layer_19_gb300 import moe
    declared = _declared_symbols()
    assert declared, "no declarations parsed"
    assert set(declared) == set(moe.EXPORTED), (declared, moe.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_minibatch_floor_matches_pages(lib):
    with open(GOLDEN_FLOOR, encoding="utf-8") as fh:
        golden_lines = fh.read().splitlines(keepends=True)
    for line in golden_lines:
        if line.startswith("#") or not line.strip():
            continue
        hidden, ffn, waves, sms, tm, tn, expect = map(int, line.split())
        out = ctypes.c_int64()
        assert lib.moe_minibatch_floor(sms, tm, tn, ffn, waves, ctypes.byref(out)) == 0
        assert out.value == expect
    out = ctypes.c_int64()
    assert lib.moe_minibatch_floor(0, 128, 128, 2048, 2, ctypes.byref(out)) == 1


def test_status_strings(lib):
    for s in range(7):
        assert lib.moe_status_string(s)
    assert lib.moe_status_string(5).decode() == "device-side wait timed out"


def test_plan_rejects_bad_configs_without_touching_a_gpu(lib):
    from mixture_experts_layer_19_gb300 import moe
    h = ctypes.c_void_p()
    assert lib.moe_plan(None, ctypes.byref(h)) == 1
    bad = [
        dict(T_max=0, d=256, F=256, E=8, k=2),          # T_max out of range
        dict(T_max=16, d=200, F=256, E=8, k=2),         # d not a multiple of 256
        dict(T_max=16, d=256, F=384, E=8, k=2),         # F not a multiple of 256
        dict(T_max=16, d=256, F=256, E=2, k=4),         # k > E
        dict(T_max=16, d=256, F=256, E=2048, k=4),      # E > 1024
        dict(T_max=16, d=256, F=256, E=8, k=33),        # k > 32
        dict(T_max=16, d=256, F=256, E=8, k=2, prec=7),  # unknown precision
    ]
    for kw in bad:
        c = moe.Config(**kw).to_c()
        st = lib.moe_plan(ctypes.byref(c), ctypes.byref(h))
        assert st in (1, 2), (kw, st)
        assert lib.moe_last_error()
    # null-plan calls are argument errors, not crashes
    assert lib.moe_forward(None, 4, None, None, None, None, None, None, None, None) == 1
    n = ctypes.c_size_t()
    assert lib.moe_saved_bytes(None, 4, ctypes.byref(n)) == 1
    assert lib.moe_plan_destroy(None) == 0


def test_product_path_has_no_cpu_fallback():
    """The binding refuses to run without the compiled library."""
    from mixture_experts_layer_19_gb300 import moe
    with pytest.raises(ImportError):
        moe.load_library("/nonexistent/libmoe.so")
    src = open(os.path.join(ROOT, "mixture_experts_layer_19_gb300", "moe.py"), encoding="utf-8").read()
    assert "oracle" not in src.replace("no fallback", "")


class _FakeLib:
    """Stands in for libmoe.so: records which plan handles were destroyed."""

    def __init__(self):
        self.destroyed = []

    def moe_plan_destroy(self, handle):
        self.destroyed.append(handle)
        return 0


def test_plan_destroyed_during_a_capture_is_deferred(monkeypatch):
    """Host logic of the binding: a plan closed (or collected) while the
    current stream is being captured is queued, not destroyed -- destroying
    synchronises the device and would invalidate the capture -- and the queue
    is emptied by the next close made outside a capture, oldest or newest
    alike, each handle exactly once."""
    from mixture_experts_layer_19_gb300 import moe
    fake = _FakeLib()
    monkeypatch.setattr(moe, "lib", lambda: fake)
    monkeypatch.setattr(moe, "_deferred_destroy", [])
    capturing = {"on": True}
    monkeypatch.setattr(moe, "_capturing", lambda: capturing["on"])

    def plan_with(handle):
        p = object.__new__(moe.Plan)     # no device: only the handle matters here
        p.handle = handle
        return p

    a, b, c = plan_with(11), plan_with(12), plan_with(13)
    a.close()
    b.__del__()                          # what the garbage collector calls
    assert fake.destroyed == [] and sorted(moe._deferred_destroy) == [11, 12]
    assert a.handle is None and b.handle is None
    a.close()                            # closing twice queues nothing more
    assert sorted(moe._deferred_destroy) == [11, 12]
    capturing["on"] = False
    c.close()
    assert sorted(fake.destroyed) == [11, 12, 13] and moe._deferred_destroy == []
    c.close()
    assert sorted(fake.destroyed) == [11, 12, 13]
    with plan_with(14) as d:             # a plan used as a context manager is closed on exit
        assert d.handle == 14
    assert d.handle is None and sorted(fake.destroyed) == [11, 12, 13, 14]


def test_binding_rejects_wrong_dtypes_and_shapes_before_the_abi(monkeypatch):
    """The C ABI takes untyped pointers, so the binding checks each tensor's
    dtype and shape against the plan's config and raises ValueError before
    any library call (CPU tensors suffice: the checks come first)."""
    import torch
    from mixture_experts_layer_19_gb300 import moe

    class NoCalls:
        def __getattr__(self, name):
            raise AssertionError(f"library called: {name}")

    monkeypatch.setattr(moe, "lib", lambda: NoCalls())
    plan = object.__new__(moe.Plan)
    plan.cfg = moe.Config(T_max=8, d=256, F=512, E=4, k=2)
    plan.handle = None
    plan.device = torch.device("cpu")
    T, d, F, E = 8, 256, 512, 4
    X = torch.zeros((T, d), dtype=torch.bfloat16)
    L = torch.zeros((T, E), dtype=torch.float32)
    W = torch.zeros((E, F, d), dtype=torch.bfloat16)
    Wd = torch.zeros((E, d, F), dtype=torch.bfloat16)
    cases = [
        lambda: plan.forward(X.float(), L, W, W, Wd),                 # X must be bf16
        lambda: plan.forward(X, L.to(torch.bfloat16), W, W, Wd),      # logits must be fp32
        lambda: plan.forward(X, L[:, :3], W, W, Wd),                  # logits [T, E]
        lambda: plan.forward(X, L, Wd, W, Wd),                        # Wg is [E, F, d], not [E, d, F]
        lambda: plan.forward(X, L, W, W, W[:, :, :128]),              # Wd [E, d, F]
        lambda: plan.forward(X, L, None, W, Wd),                      # weights required
        lambda: plan.backward(X[:4], X, W, W, Wd, None),              # dY rows = X rows
        lambda: plan.backward(X, X, W, W, Wd, None),                  # the saved context is required
        lambda: plan.backward(X, X, W, W, Wd, torch.zeros(16)),       # saved is bytes (new_saved)
        lambda: plan.router_forward(X, torch.zeros((E + 1, d), dtype=torch.bfloat16)),
        lambda: plan.router_backward(X, torch.zeros((E, d), dtype=torch.bfloat16), L, X.float()),
        lambda: plan.quantize_weights(W, W.float(), Wd),
    ]
    for call in cases:
        with pytest.raises(ValueError):
            call()
