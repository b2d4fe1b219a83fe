"""NVFP4 codec for the oracle (TEST INFRASTRUCTURE ONLY).

The fluidifia page "Cursor ouvre MoK, un mégakernel qui accélère
l'entraînement MoE" (section "Quand la communication devient le vrai
problème") names NVFP4 kernels among the team's earlier work and says nothing
more about the format.  The format itself follows public definitions:

* OCP Microscaling Formats (MX) v1.0, FP4 element E2M1: one sign bit, two
  exponent bits (bias 1), one mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3,
  4, 6; no infinities or NaN;
* NVIDIA's NVFP4: 16 consecutive elements share one E4M3 scale, and one
  fp32 scale multiplies the whole tensor.

Readings where the definitions leave a choice.  Every step that decides a
code is IEEE fp32 arithmetic (round to nearest even), emulated here with
numpy float32, because the device takes the same decisions in fp32:

* tensor scale g = fl32(amax / 2688) (2688 = 6 * 448: largest E2M1 times
  largest E4M3), and g = 1 for an all-zero tensor;
* rc = fl32(1 / fl32(6 g)) once per tensor; block scale
  s = E4M3(fl32(amax_block * rc)), round to nearest even, saturating at 448;
* element code = E2M1(fl32(v * fl32(1 / fl32(s g)))), round to nearest even,
  saturating at +-6, the sign kept (a negative value that rounds to zero is
  -0, code 8); a block whose scale rounds to zero gets codes 0;
* inputs are rounded to fp32 first (exact for bf16 and for fp32 values);
* packing: element 2i in the low nibble of byte i, element 2i+1 in the high.

The dequantised value is e2m1(code) * s * g (exact in fp64).
"""
from __future__ import annotations

import numpy as np

from .mxfp8 import e4m3_decode, e4m3_encode

NV_BLOCK = 16                      # elements sharing one E4M3 scale
E2M1_MAX = 6.0
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
SCALE_DENOM = 6.0 * 448.0          # E2M1 max times E4M3 max


def e2m1_decode(code):
    """Value of 4-bit E2M1 code(s): bit 3 is the sign, bits 0-2 the magnitude index."""
    c = np.asarray(code, dtype=np.int64)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where(c & 8, -mag, mag)


def e2m1_round(v):
    """Round fp64 values to E2M1 (nearest, ties to even mantissa), saturating at +-6.

    Binade quanta: 0.5 below 2 (the subnormal 0.5 included), 1 in [2, 4),
    2 in [4, 8); rint on the quotient is ties-to-even, and an even quotient is
    an even mantissa in each binade.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                        # a = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, 0)                  # binade exponent; below 1 shares 1's quantum
    quantum = np.ldexp(1.0, e - 1)             # one mantissa bit
    q = np.minimum(np.rint(a / quantum) * quantum, E2M1_MAX)
    return np.copysign(q, v)


def e2m1_encode(v):
    """4-bit E2M1 code of each fp64 value (round to nearest even, saturating, sign kept)."""
    q = e2m1_round(v)
    a = np.abs(q)
    idx = np.searchsorted(E2M1_MAGNITUDES, a)  # exact members of the magnitude table
    sign = np.signbit(q).astype(np.int64) << 3
    return (sign | idx).astype(np.uint8)


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def tensor_scale(amax):
    """fp32 tensor scale g = fl32(amax / 2688); 1 when amax is 0."""
    a = np.float32(amax)
    if a == 0:
        return np.float32(1.0)
    return np.float32(a / np.float32(SCALE_DENOM))


def weight_scales(Wg, Wu, Wd):
    """(g_gu, g_d): one scale for Wg and Wu together (the dx GEMM contracts over
    both), one for Wd.  Accepts arrays or per-expert indexables."""
    def amax(W):
        if isinstance(W, np.ndarray):
            return float(np.abs(W).max()) if W.size else 0.0
        return max(float(np.abs(np.asarray(W[e], dtype=np.float64)).max()) for e in range(len(W)))
    return tensor_scale(max(amax(Wg), amax(Wu))), tensor_scale(amax(Wd))


def nv_quantize(v, axis=-1, g=1.0):
    """Quantise ``v`` to NVFP4 along ``axis`` (length a multiple of 16) with tensor scale ``g``.

    Returns (codes uint8 with v's shape, one unpacked 4-bit code per element;
    scale bytes uint8 (E4M3) with that axis divided by 16).
    """
    g = np.float32(g)
    vm = np.moveaxis(_f32(v), axis, -1)
    n = vm.shape[-1]
    if n % NV_BLOCK:
        raise ValueError("quantised axis must be a multiple of 16")
    blocks = vm.reshape(vm.shape[:-1] + (n // NV_BLOCK, NV_BLOCK))
    rc = np.float32(1.0) / (np.float32(6.0) * g)
    amax = np.abs(blocks).max(axis=-1)                       # exact in fp32
    s_code = e4m3_encode((amax * rc).astype(np.float64))     # fl32 product, then E4M3
    s_val = e4m3_decode(s_code)
    live = s_val > 0
    d = _f32(s_val) * g                                      # fl32(s g)
    r = np.where(live, np.float32(1.0) / np.where(live, d, np.float32(1.0)), np.float32(0.0))
    scaled = blocks * r[..., None]                           # fl32(v r)
    codes = np.where(live[..., None], e2m1_encode(scaled.astype(np.float64)), 0).astype(np.uint8)
    codes = np.moveaxis(codes.reshape(vm.shape), -1, axis)
    scales = np.moveaxis(s_code.astype(np.uint8), -1, axis)
    return codes, scales


def nv_dequantize(codes, scales, axis=-1, g=1.0):
    """Inverse of :func:`nv_quantize`: e2m1(code) * e4m3(scale) * g, in fp64."""
    cm = np.moveaxis(np.asarray(codes), axis, -1)
    sm = np.moveaxis(np.asarray(scales), axis, -1)
    vals = e2m1_decode(cm).reshape(cm.shape[:-1] + (sm.shape[-1], NV_BLOCK))
    out = vals * (e4m3_decode(sm) * float(np.float32(g)))[..., None]
    return np.moveaxis(out.reshape(cm.shape), -1, axis)


def nv_fake_quant(v, axis=-1, g=1.0):
    """Dequantised NVFP4 image of ``v`` along ``axis`` (pads the axis to 16 with zeros)."""
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[axis]
    pad = (-n) % NV_BLOCK
    if pad:
        widths = [(0, 0)] * v.ndim
        widths[axis % v.ndim] = (0, pad)
        v = np.pad(v, widths)
    out = nv_dequantize(*nv_quantize(v, axis, g), axis=axis, g=g)
    if pad:
        out = np.take(out, np.arange(n), axis=axis)
    return out


def nv_pack(codes):
    """Pack 4-bit codes along the last axis: element 2i -> low nibble of byte i."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def nv_unpack(packed):
    """Inverse of :func:`nv_pack`."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out
