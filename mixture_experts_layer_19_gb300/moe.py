"""Thin Python binding of the C ABI in include/moe.h (ctypes).

Argument marshalling only: every step of the layer runs in the CUDA kernels
of libmoe.so.  The library must be built (``__graft_entry__.build()`` or
``python -m mixture_experts_layer_19_gb300.build``); importing this module
without it raises ImportError -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_OK = 0
MOE_BF16 = 0
MOE_MXFP8 = 1
MOE_NVFP4 = 2
MOE_DEBUG_IDENTITY_EXPERTS = 0x1
MOE_DEBUG_TIMING = 0x2
MOE_DEBUG_SEPARATE_KERNELS = 0x4
MOE_DEBUG_RING_MEGAKERNEL = 0x8
MOE_DEBUG_MULTI_LAUNCH = 0x20
MOE_DEBUG_DUMP_QUANT = 0x40
MOE_DEBUG_STALL_TEST = 0x80
MOE_ERR_INVALID_ARG = 1
MOE_ERR_TIMEOUT = 5

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_OOM",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_INTERNAL"}

# Every symbol include/moe.h declares (the test suite checks the library exports them).
EXPORTED = ("moe_plan", "moe_plan_destroy", "moe_saved_bytes", "moe_forward", "moe_backward",
            "moe_get_routing", "moe_device_status", "moe_kernel_times", "moe_minibatch_floor",
            "moe_status_string", "moe_last_error", "moe_route_noalloc", "moe_quantize_weights",
            "moe_mx_quantize", "moe_router_forward", "moe_router_backward", "moe_mx_quantize_transposed",
            "moe_plan_info", "moe_nv_tensor_scale", "moe_nv_quantize", "moe_nv_quantize_transposed",
            "moe_nv_weight_scales", "moe_debug_quant_dump", "moe_plan_padded_rows")


class moe_config_t(ctypes.Structure):
    _fields_ = [("T_max", ctypes.c_int64), ("d", ctypes.c_int32), ("F", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("prec", ctypes.c_int32),
                ("minibatch_rows", ctypes.c_int32), ("ring_slots", ctypes.c_int32),
                ("mover_ctas", ctypes.c_int32), ("wait_timeout_ns", ctypes.c_int64),
                ("debug_flags", ctypes.c_uint32), ("device", ctypes.c_int32), ("ep_ranks", ctypes.c_int32)]


def load_library(path: str = _LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libmoe.so not built ({path}); run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    P, I64, I32, VP, FP = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p
    sig = {
        "moe_plan": [ctypes.POINTER(moe_config_t), ctypes.POINTER(P)],
        "moe_plan_destroy": [P],
        "moe_saved_bytes": [P, I64, ctypes.POINTER(ctypes.c_size_t)],
        "moe_forward": [P, I64, VP, FP, VP, VP, VP, VP, VP, P],
        "moe_backward": [P, I64, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, FP, FP, P],
        "moe_get_routing": [P, I64, VP, VP, VP, VP, VP, VP, VP, P],
        "moe_device_status": [P, P, ctypes.POINTER(I32)],
        "moe_kernel_times": [P, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                             ctypes.POINTER(I64), I32, ctypes.POINTER(I32)],
        "moe_minibatch_floor": [I32, I32, I32, I32, I32, ctypes.POINTER(I64)],
        "moe_status_string": [I32],
        "moe_last_error": [],
        "moe_route_noalloc": [I64, I32, I32, FP, VP, VP, VP, VP, VP, VP, P],
        "moe_quantize_weights": [P, VP, VP, VP, P],
        "moe_mx_quantize": [VP, I64, I64, VP, VP, P],
        "moe_mx_quantize_transposed": [VP, I64, I64, I64, VP, VP, P],
        "moe_plan_info": [P, ctypes.POINTER(I32), ctypes.POINTER(I32)],
        "moe_router_forward": [P, I64, VP, VP, FP, P],
        "moe_router_backward": [P, I64, VP, VP, FP, VP, VP, P],
        "moe_nv_tensor_scale": [VP, I64, VP, I64, FP, P],
        "moe_nv_quantize": [VP, I64, I64, FP, VP, VP, P],
        "moe_nv_quantize_transposed": [VP, I64, I64, I64, FP, VP, VP, P],
        "moe_nv_weight_scales": [P, FP, P],
        "moe_debug_quant_dump": [P, I32, FP, VP, VP, P],
        "moe_plan_padded_rows": [P, ctypes.POINTER(I64)],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name in ("moe_status_string", "moe_last_error") else ctypes.c_int
    return lib


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library()
    return _lib


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        detail = lib().moe_last_error().decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({detail})")
        self.status = status


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoEError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError("tensors must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _expect(t: Optional[torch.Tensor], name: str, shape, dtype, optional: bool = False) -> None:
    """The C ABI takes untyped pointers, so the binding checks what the header
    fixes for each tensor (dtype, shape) before passing it on."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _stream(stream: Optional[torch.cuda.Stream] = None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def minibatch_floor(num_sms: int, tile_m: int, tile_n: int, n_out: int, waves: int = 2) -> int:
    out = ctypes.c_int64()
    _check(lib().moe_minibatch_floor(num_sms, tile_m, tile_n, n_out, waves, ctypes.byref(out)),
           "moe_minibatch_floor")
    return out.value


def mx_quantize(src: torch.Tensor, stream=None):
    """MXFP8 of a bf16 [rows, K] CUDA tensor along K: (E4M3 bytes [rows, K] uint8,
    scale atoms uint8 [ceil(rows/128) * K/128 * 512]) -- layout in include/moe.h."""
    rows, K = src.shape
    q = torch.empty((rows, K), dtype=torch.uint8, device=src.device)
    sf = torch.empty(((rows + 127) // 128) * (K // 128) * 512, dtype=torch.uint8, device=src.device)
    _check(lib().moe_mx_quantize(_ptr(src), rows, K, _ptr(q), _ptr(sf), _stream(stream)), "moe_mx_quantize")
    return q, sf


def mx_quantize_transposed(src: torch.Tensor, stream=None):
    """MXFP8 of the transposes of a bf16 [E, A, B] CUDA tensor along A: (E4M3 bytes
    [E, B, A] uint8, scale atoms of the E*B rows with K = A)."""
    E, A, B = src.shape
    q = torch.empty((E, B, A), dtype=torch.uint8, device=src.device)
    sf = torch.empty(((E * B + 127) // 128) * (A // 128) * 512, dtype=torch.uint8, device=src.device)
    _check(lib().moe_mx_quantize_transposed(_ptr(src), E, A, B, _ptr(q), _ptr(sf), _stream(stream)),
           "moe_mx_quantize_transposed")
    return q, sf


def nv_tensor_scale(x0: torch.Tensor, x1: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """NVFP4 tensor scale amax / 2688 over one or two bf16 CUDA tensors, as a
    one-element fp32 CUDA tensor (1 for all-zero input)."""
    g = torch.empty((1,), dtype=torch.float32, device=x0.device)
    n1 = x1.numel() if x1 is not None else 0
    _check(lib().moe_nv_tensor_scale(_ptr(x0), x0.numel(), _ptr(x1), n1, _ptr(g), _stream(stream)),
           "moe_nv_tensor_scale")
    return g


def nv_quantize(src: torch.Tensor, g: Optional[torch.Tensor] = None, stream=None):
    """NVFP4 of a bf16 [rows, K] CUDA tensor along K with tensor scale g (a
    one-element fp32 CUDA tensor, None = 1): (packed E2M1 bytes [rows, K/2]
    uint8, E4M3 scale atoms uint8 [ceil(rows/128) * K/64 * 512])."""
    rows, K = src.shape
    q = torch.empty((rows, K // 2), dtype=torch.uint8, device=src.device)
    sf = torch.empty(((rows + 127) // 128) * (K // 64) * 512, dtype=torch.uint8, device=src.device)
    _check(lib().moe_nv_quantize(_ptr(src), rows, K, _ptr(g), _ptr(q), _ptr(sf), _stream(stream)),
           "moe_nv_quantize")
    return q, sf


def nv_quantize_transposed(src: torch.Tensor, g: Optional[torch.Tensor] = None, stream=None):
    """NVFP4 of the transposes of a bf16 [E, A, B] CUDA tensor along A: (packed
    bytes [E, B, A/2] uint8, scale atoms of the E*B rows with K = A)."""
    E, A, B = src.shape
    q = torch.empty((E, B, A // 2), dtype=torch.uint8, device=src.device)
    sf = torch.empty(((E * B + 127) // 128) * (A // 64) * 512, dtype=torch.uint8, device=src.device)
    _check(lib().moe_nv_quantize_transposed(_ptr(src), E, A, B, _ptr(g), _ptr(q), _ptr(sf), _stream(stream)),
           "moe_nv_quantize_transposed")
    return q, sf


def sf_atom_index(rows: int, K: int):
    """Host copy of the scale-atom layout: flat offsets [rows, K/32] into the sf buffer."""
    import numpy as np
    r = np.arange(rows)[:, None]
    b = np.arange(K // 32)[None, :]
    atom = (r >> 7) * (K // 128) + (b >> 2)
    return atom * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3)


@dataclass
class Config:
    T_max: int
    d: int
    F: int
    E: int
    k: int
    prec: int = MOE_BF16
    minibatch_rows: int = 0
    ring_slots: int = 0
    mover_ctas: int = 0
    wait_timeout_ns: int = 0
    debug_flags: int = 0
    device: int = 0
    ep_ranks: int = 0

    def to_c(self) -> moe_config_t:
        return moe_config_t(self.T_max, self.d, self.F, self.E, self.k, self.prec, self.minibatch_rows,
                            self.ring_slots, self.mover_ctas, self.wait_timeout_ns, self.debug_flags,
                            self.device, self.ep_ranks)


# Plans whose destruction came while the current stream was being captured
# into a CUDA graph (typically the garbage collector reaching an unreferenced
# plan inside a capture).  moe_plan_destroy synchronises the device and frees
# memory, which would invalidate the capture, so these handles are destroyed
# at the next Plan creation or close made outside a capture.
_deferred_destroy: list = []


def _capturing() -> bool:
    try:
        return torch.cuda.is_current_stream_capturing()
    except Exception:
        return False


def _destroy_deferred() -> None:
    while _deferred_destroy and not _capturing():
        lib().moe_plan_destroy(_deferred_destroy.pop())


class Plan:
    """One moe_plan_t: owns the device workspace for tokens T <= T_max."""

    def __init__(self, cfg: Config):
        _destroy_deferred()
        self.cfg = cfg
        self._c = cfg.to_c()
        h = ctypes.c_void_p()
        _check(lib().moe_plan(ctypes.byref(self._c), ctypes.byref(h)), "moe_plan")
        self.handle = h
        self.device = torch.device("cuda", cfg.device)

    def close(self):
        h = getattr(self, "handle", None)
        self.handle = None
        if h:
            if _capturing():
                _deferred_destroy.append(h)
            else:
                lib().moe_plan_destroy(h)
        _destroy_deferred()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def saved_bytes(self, T: int) -> int:
        n = ctypes.c_size_t()
        _check(lib().moe_saved_bytes(self.handle, T, ctypes.byref(n)), "moe_saved_bytes")
        return n.value

    def new_saved(self, T: int) -> torch.Tensor:
        return torch.empty(self.saved_bytes(T), dtype=torch.uint8, device=self.device)

    def _expect_weights(self, Wg, Wu, Wd):
        c = self.cfg
        optional = bool(c.debug_flags & MOE_DEBUG_IDENTITY_EXPERTS)
        _expect(Wg, "Wg", (c.E, c.F, c.d), torch.bfloat16, optional)
        _expect(Wu, "Wu", (c.E, c.F, c.d), torch.bfloat16, optional)
        _expect(Wd, "Wd", (c.E, c.d, c.F), torch.bfloat16, optional)

    def _expect_saved(self, saved, T: int):
        """The saved context is written (forward) and read (backward) through an
        untyped pointer: it must hold moe_saved_bytes(T) bytes."""
        if saved is None:
            raise ValueError("saved is required")
        if saved.dtype != torch.uint8:
            raise ValueError(f"saved: dtype {saved.dtype}, expected torch.uint8 (from new_saved)")
        need = self.saved_bytes(T)
        if saved.numel() < need:
            raise ValueError(f"saved: {saved.numel()} bytes, the context of T={T} needs {need}")

    def forward(self, X, logits, Wg, Wu, Wd, Y=None, saved=None, stream=None):
        T, c = X.shape[0], self.cfg
        _expect(X, "X", (T, c.d), torch.bfloat16)
        _expect(logits, "logits", (T, c.E), torch.float32)
        self._expect_weights(Wg, Wu, Wd)
        _expect(Y, "Y", (T, c.d), torch.bfloat16, optional=True)
        if Y is None:
            Y = torch.empty((T, self.cfg.d), dtype=torch.bfloat16, device=self.device)
        if saved is None:
            saved = self.new_saved(T)
        else:
            self._expect_saved(saved, T)
        _check(lib().moe_forward(self.handle, T, _ptr(X), _ptr(logits), _ptr(Wg), _ptr(Wu), _ptr(Wd),
                                 _ptr(Y), _ptr(saved), _stream(stream)), "moe_forward")
        return Y, saved

    def backward(self, dY, X, Wg, Wu, Wd, saved, out=None, want_dlogits=True, stream=None):
        T, c = X.shape[0], self.cfg
        dev = self.device
        _expect(X, "X", (T, c.d), torch.bfloat16)
        _expect(dY, "dY", (T, c.d), torch.bfloat16)
        self._expect_weights(Wg, Wu, Wd)
        if out is not None:
            for name, shape, dtype in (("dX", (T, c.d), torch.bfloat16), ("dWg", (c.E, c.F, c.d), torch.bfloat16),
                                       ("dWu", (c.E, c.F, c.d), torch.bfloat16),
                                       ("dWd", (c.E, c.d, c.F), torch.bfloat16), ("dg", (T, c.k), torch.float32)):
                _expect(out.get(name), f"out[{name!r}]", shape, dtype)
            _expect(out.get("dlogits"), "out['dlogits']", (T, c.E), torch.float32, optional=True)
        self._expect_saved(saved, T)
        if out is None:
            out = {
                "dX": torch.empty((T, c.d), dtype=torch.bfloat16, device=dev),
                "dWg": torch.empty((c.E, c.F, c.d), dtype=torch.bfloat16, device=dev),
                "dWu": torch.empty((c.E, c.F, c.d), dtype=torch.bfloat16, device=dev),
                "dWd": torch.empty((c.E, c.d, c.F), dtype=torch.bfloat16, device=dev),
                "dg": torch.empty((T, c.k), dtype=torch.float32, device=dev),
                "dlogits": torch.empty((T, c.E), dtype=torch.float32, device=dev) if want_dlogits else None,
            }
        _check(lib().moe_backward(self.handle, T, _ptr(dY), _ptr(X), _ptr(Wg), _ptr(Wu), _ptr(Wd),
                                  _ptr(saved), _ptr(out["dX"]), _ptr(out["dWg"]), _ptr(out["dWu"]),
                                  _ptr(out["dWd"]), _ptr(out["dg"]), _ptr(out.get("dlogits")),
                                  _stream(stream)), "moe_backward")
        return out

    def routing(self, saved, T, stream=None):
        c, dev = self.cfg, self.device
        self._expect_saved(saved, T)
        R = T * c.k
        out = {
            "idx": torch.empty((T, c.k), dtype=torch.int32, device=dev),
            "w": torch.empty((T, c.k), dtype=torch.float32, device=dev),
            "counts": torch.empty((c.E,), dtype=torch.int32, device=dev),
            "offsets": torch.empty((c.E + 1,), dtype=torch.int32, device=dev),
            "perm_src": torch.empty((R,), dtype=torch.int32, device=dev),
            "dest": torch.empty((T, c.k), dtype=torch.int32, device=dev),
        }
        _check(lib().moe_get_routing(self.handle, T, _ptr(saved), _ptr(out["idx"]), _ptr(out["w"]),
                                     _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm_src"]),
                                     _ptr(out["dest"]), _stream(stream)), "moe_get_routing")
        return out

    def quantize_weights(self, Wg, Wu, Wd, stream=None):
        """MXFP8 / NVFP4 plans: fill the plan's quantised weight copies (once per weight update)."""
        self._expect_weights(Wg, Wu, Wd)
        _check(lib().moe_quantize_weights(self.handle, _ptr(Wg), _ptr(Wu), _ptr(Wd), _stream(stream)),
               "moe_quantize_weights")

    def padded_rows(self) -> int:
        """Padded sorted-row capacity of the plan (T = T_max)."""
        n = ctypes.c_int64()
        _check(lib().moe_plan_padded_rows(self.handle, ctypes.byref(n)), "moe_plan_padded_rows")
        return n.value

    def debug_quant_dump(self, which: int, stream=None):
        """MOE_DEBUG_DUMP_QUANT plans: (fp32 values or None, quantised bytes,
        scale atoms) of one quantised operand over the padded row capacity P.
        which 0: h of the last forward, 1: dA|dB of the last backward (both
        [P, C] quantised along C); 2: dY^T, 3: X^T, 4: [dA|dB]^T, 5: (w h)^T of
        the last backward ([C, P] quantised along P; values [P, C] for 4 and 5,
        None for 2 and 3); 6: the dispatch's quantised sorted rows of the last
        call (X after forward, dY after backward; [P, d] quantised along d,
        values None)."""
        c = self.cfg
        P = self.padded_rows()
        C = {0: c.F, 1: 2 * c.F, 2: c.d, 3: c.d, 4: 2 * c.F, 5: c.F, 6: c.d}.get(which, c.F)
        nv = c.prec == MOE_NVFP4
        vals = None if which in (2, 3, 6) else torch.empty((P, C), dtype=torch.float32, device=self.device)
        shape = (P, C) if which in (0, 1, 6) else (C, P)
        q = torch.empty((shape[0], shape[1] // 2 if nv else shape[1]), dtype=torch.uint8, device=self.device)
        sf = torch.empty((P * C // (16 if nv else 32),), dtype=torch.uint8, device=self.device)
        _check(lib().moe_debug_quant_dump(self.handle, which, _ptr(vals), _ptr(q), _ptr(sf), _stream(stream)),
               "moe_debug_quant_dump")
        return vals, q, sf

    def nv_weight_scales(self, stream=None) -> torch.Tensor:
        """NVFP4 plans: the weights' tensor scales [g(Wg, Wu), g(Wd)] as a 2-element fp32 CUDA tensor."""
        out = torch.empty((2,), dtype=torch.float32, device=self.device)
        _check(lib().moe_nv_weight_scales(self.handle, _ptr(out), _stream(stream)), "moe_nv_weight_scales")
        return out

    def device_status(self, stream=None) -> int:
        st = ctypes.c_int32()
        _check(lib().moe_device_status(self.handle, _stream(stream), ctypes.byref(st)), "moe_device_status")
        return st.value

    def info(self):
        """Launch geometry: {"num_sms": n, "movers": .., "ring_slots": .., "minibatch_tiles": ..,
        "slot_tiles": ..} (the ring pipeline's shape, in 128-row tiles)."""
        n = ctypes.c_int32()
        ring = (ctypes.c_int32 * 4)()
        _check(lib().moe_plan_info(self.handle, ctypes.byref(n), ring), "moe_plan_info")
        return {"num_sms": n.value, "movers": ring[0], "ring_slots": ring[1], "minibatch_tiles": ring[2],
                "slot_tiles": ring[3]}

    def router_forward(self, X, Wr, logits=None, stream=None):
        """logits = X Wr^T (fp32) on the tensor cores."""
        T, c = X.shape[0], self.cfg
        _expect(X, "X", (T, c.d), torch.bfloat16)
        _expect(Wr, "Wr", (c.E, c.d), torch.bfloat16)
        _expect(logits, "logits", (T, c.E), torch.float32, optional=True)
        if logits is None:
            logits = torch.empty((T, self.cfg.E), dtype=torch.float32, device=self.device)
        _check(lib().moe_router_forward(self.handle, T, _ptr(X), _ptr(Wr), _ptr(logits), _stream(stream)),
               "moe_router_forward")
        return logits

    def router_backward(self, X, Wr, dlogits, dX, dWr=None, stream=None):
        """dX += dlogits Wr (in place); returns dWr = dlogits^T X."""
        T, c = X.shape[0], self.cfg
        _expect(X, "X", (T, c.d), torch.bfloat16)
        _expect(Wr, "Wr", (c.E, c.d), torch.bfloat16)
        _expect(dlogits, "dlogits", (T, c.E), torch.float32)
        _expect(dX, "dX", (T, c.d), torch.bfloat16)
        _expect(dWr, "dWr", (c.E, c.d), torch.bfloat16, optional=True)
        if dWr is None:
            dWr = torch.empty((self.cfg.E, self.cfg.d), dtype=torch.bfloat16, device=self.device)
        _check(lib().moe_router_backward(self.handle, X.shape[0], _ptr(X), _ptr(Wr), _ptr(dlogits), _ptr(dX),
                                         _ptr(dWr), _stream(stream)), "moe_router_backward")
        return dWr

    def kernel_times(self):
        cap = 64
        names = (ctypes.c_char_p * cap)()
        ms = (ctypes.c_double * cap)()
        cnt = (ctypes.c_int64 * cap)()
        n = ctypes.c_int32()
        _check(lib().moe_kernel_times(self.handle, names, ms, cnt, cap, ctypes.byref(n)), "moe_kernel_times")
        return {names[i].decode(): (ms[i], cnt[i]) for i in range(min(n.value, cap))}


class _MoEFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, plan: Plan, X, logits, Wg, Wu, Wd):
        X = X.contiguous()
        Y, saved = plan.forward(X, logits.contiguous(), Wg, Wu, Wd)
        ctx.plan = plan
        ctx.save_for_backward(X, Wg, Wu, Wd, saved)
        return Y

    @staticmethod
    def backward(ctx, dY):
        X, Wg, Wu, Wd, saved = ctx.saved_tensors
        want_dlogits = ctx.needs_input_grad[2]   # no dlogits kernel work when logits need no gradient
        g = ctx.plan.backward(dY.contiguous(), X, Wg, Wu, Wd, saved, want_dlogits=want_dlogits)
        return None, g["dX"], g["dlogits"], g["dWg"], g["dWu"], g["dWd"]


class _RoutedMoEFunction(torch.autograd.Function):
    """Router GEMM + MoE layer: logits = X Wr^T, then the layer; the backward
    adds the router's share of dX to the experts' share."""

    @staticmethod
    def forward(ctx, plan: Plan, X, Wr, Wg, Wu, Wd):
        X = X.contiguous()
        logits = plan.router_forward(X, Wr)
        Y, saved = plan.forward(X, logits, Wg, Wu, Wd)
        ctx.plan = plan
        ctx.save_for_backward(X, Wr, Wg, Wu, Wd, saved)
        return Y

    @staticmethod
    def backward(ctx, dY):
        X, Wr, Wg, Wu, Wd, saved = ctx.saved_tensors
        g = ctx.plan.backward(dY.contiguous(), X, Wg, Wu, Wd, saved, want_dlogits=True)
        dWr = ctx.plan.router_backward(X, Wr, g["dlogits"], g["dX"])
        return None, g["dX"], dWr, g["dWg"], g["dWu"], g["dWd"]


class MoELayer(torch.nn.Module):
    """Fused MoE layer over bf16 expert weights; router logits are an input.

    prec = MOE_BF16, MOE_MXFP8 or MOE_NVFP4.  A block-scaled layer quantises
    its weights again whenever they changed since the last quantisation (an
    optimiser step, a copy_ or a load_state_dict bumps the parameters'
    version counters), before the forward that first sees the change."""

    def __init__(self, d: int, F: int, E: int, k: int, T_max: int, device=0, debug_flags: int = 0,
                 prec: int = MOE_BF16):
        super().__init__()
        dev = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        self.plan = Plan(Config(T_max=T_max, d=d, F=F, E=E, k=k, prec=prec, device=dev.index or 0,
                                debug_flags=debug_flags))
        self.Wg = torch.nn.Parameter(torch.empty((E, F, d), dtype=torch.bfloat16, device=dev))
        self.Wu = torch.nn.Parameter(torch.empty((E, F, d), dtype=torch.bfloat16, device=dev))
        self.Wd = torch.nn.Parameter(torch.empty((E, d, F), dtype=torch.bfloat16, device=dev))
        self._quantized_key = None
        self.reset_parameters()

    def reset_parameters(self):
        """Each weight ~ N(0, 1/fan_in): fan_in = d for Wg, Wu (and Wr), F for Wd."""
        c = self.plan.cfg
        with torch.no_grad():
            self.Wg.normal_(0.0, c.d ** -0.5)
            self.Wu.normal_(0.0, c.d ** -0.5)
            self.Wd.normal_(0.0, c.F ** -0.5)
            if hasattr(self, "Wr"):
                self.Wr.normal_(0.0, c.d ** -0.5)

    def _sync_quantized_weights(self):
        if self.plan.cfg.prec == MOE_BF16:
            return
        key = tuple((w.data_ptr(), w._version) for w in (self.Wg, self.Wu, self.Wd))
        if key != self._quantized_key:
            self.plan.quantize_weights(self.Wg.detach(), self.Wu.detach(), self.Wd.detach())
            self._quantized_key = key

    def forward(self, X, logits):
        self._sync_quantized_weights()
        return _MoEFunction.apply(self.plan, X, logits, self.Wg, self.Wu, self.Wd)


class RoutedMoELayer(MoELayer):
    """Fused MoE layer with its router: logits = X Wr^T (bf16 Wr [E, d])."""

    def __init__(self, d: int, F: int, E: int, k: int, T_max: int, device=0, debug_flags: int = 0,
                 prec: int = MOE_BF16):
        super().__init__(d, F, E, k, T_max, device=device, debug_flags=debug_flags, prec=prec)
        self.Wr = torch.nn.Parameter(torch.empty((E, d), dtype=torch.bfloat16, device=self.Wg.device))
        self.reset_parameters()

    def forward(self, X):
        self._sync_quantized_weights()
        return _RoutedMoEFunction.apply(self.plan, X, self.Wr, self.Wg, self.Wu, self.Wd)
