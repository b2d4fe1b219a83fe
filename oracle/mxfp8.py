"""MXFP8 codec for the oracle (TEST INFRASTRUCTURE ONLY).

The Mixture-of-Kittens pages only say that MXFP8 activation quantisation is
fused into dispatch, grouped GEMM and SwiGLU (kucoin page "Cursor's MoK
réalise une amélioration des performances de 2,37x sur NVIDIA GB300 NVL72",
section 02).  The format itself follows two public specifications:

* OCP Microscaling Formats (MX) v1.0, section 5 (MXFP8: 32-element blocks
  sharing one E8M0 scale) and section 6.3 (scale = floor(log2(amax)) minus the
  element type's largest exponent);
* OCP 8-bit Floating Point (OFP8) v1.0, E4M3 (bias 7, no infinities, 0x7F and
  0xFF are NaN, largest finite 448).

Readings where the specs leave a choice:
* an all-zero block takes the smallest scale exponent, -127 (byte 0x00);
* elements are rounded to nearest, ties to even, and clamp to +-448
  ("saturating" conversion);
* the scale exponent is clamped to [-127, 127].

Everything is exact fp64 arithmetic (frexp / ldexp / rint), no log2().
"""
from __future__ import annotations

import numpy as np

E4M3_EMAX = 8          # exponent of the largest finite E4M3 value (448 = 1.75 * 2^8)
E4M3_MAX = 448.0
E4M3_EMIN = -6         # smallest normal exponent (bias 7)
MX_BLOCK = 32          # elements sharing one scale (OCP MX v1.0, MXFP8)


def e4m3_decode(code):
    """Value of E4M3 byte(s) per OFP8 v1.0 (NaN for 0x7F / 0xFF)."""
    c = np.asarray(code, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    mt = c & 0x7
    val = np.where(ex == 0, mt / 8.0 * 2.0 ** E4M3_EMIN,
                   (1.0 + mt / 8.0) * np.ldexp(1.0, ex - 7))
    val = np.where((ex == 15) & (mt == 7), np.nan, val)
    return s * val


def e4m3_round(v):
    """Round fp64 values to the nearest E4M3 value (ties to even), saturating at +-448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                       # a = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, E4M3_EMIN)         # binade exponent; subnormals share 2^-6's quantum
    quantum = np.ldexp(1.0, e - 3)            # 3 mantissa bits
    q = np.rint(a / quantum) * quantum        # exact: division by a power of two
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, v)


def e4m3_encode(v):
    """E4M3 byte of each fp64 value (round to nearest even, saturating)."""
    q = e4m3_round(v)
    a = np.abs(q)
    sign = np.signbit(q).astype(np.int64) << 7
    m, ex = np.frexp(a)
    e = ex - 1
    normal = (a != 0) & (e >= E4M3_EMIN)
    safe_e = np.where(normal, e, 0)
    mant_n = np.rint((a / np.ldexp(1.0, safe_e) - 1.0) * 8.0).astype(np.int64)
    code_n = ((safe_e + 7) << 3) | mant_n
    code_s = np.rint(a / np.ldexp(1.0, E4M3_EMIN - 3)).astype(np.int64)   # multiples of 2^-9
    code = np.where(normal, code_n, code_s)
    return (sign | code).astype(np.uint8)


def e8m0_exponent(amax):
    """Shared block exponent X = floor(log2(amax)) - 8, clamped to [-127, 127]; 0 -> -127."""
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)
    x = np.where(amax > 0, ex - 1 - E4M3_EMAX, -127)
    return np.clip(x, -127, 127).astype(np.int64)


def mx_quantize(v, axis=-1):
    """Quantise ``v`` to MXFP8 along ``axis`` (length a multiple of 32).

    Returns (codes uint8 with v's shape, scale bytes uint8 with that axis
    divided by 32).  Scale byte = X + 127; element = E4M3(v / 2^X).
    """
    v = np.asarray(v, dtype=np.float64)
    vm = np.moveaxis(v, axis, -1)
    n = vm.shape[-1]
    if n % MX_BLOCK:
        raise ValueError("quantised axis must be a multiple of 32")
    blocks = vm.reshape(vm.shape[:-1] + (n // MX_BLOCK, MX_BLOCK))
    x = e8m0_exponent(np.abs(blocks).max(axis=-1))
    codes = e4m3_encode(blocks / np.ldexp(1.0, x)[..., None])
    codes = np.moveaxis(codes.reshape(vm.shape), -1, axis)
    scales = np.moveaxis((x + 127).astype(np.uint8), -1, axis)
    return codes, scales


def mx_dequantize(codes, scales, axis=-1):
    """Inverse of :func:`mx_quantize`: element value times 2^(scale - 127)."""
    cm = np.moveaxis(np.asarray(codes), axis, -1)
    sm = np.moveaxis(np.asarray(scales, dtype=np.int64), axis, -1)
    vals = e4m3_decode(cm).reshape(cm.shape[:-1] + (sm.shape[-1], MX_BLOCK))
    out = vals * np.ldexp(1.0, sm - 127)[..., None]
    return np.moveaxis(out.reshape(cm.shape), -1, axis)


def mx_fake_quant(v, axis=-1):
    """Dequantised MXFP8 image of ``v`` along ``axis`` (pads the axis to 32 with zeros)."""
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[axis]
    pad = (-n) % MX_BLOCK
    if pad:
        widths = [(0, 0)] * v.ndim
        widths[axis % v.ndim] = (0, pad)
        v = np.pad(v, widths)
    out = mx_dequantize(*mx_quantize(v, axis), axis=axis)
    if pad:
        out = np.take(out, np.arange(n), axis=axis)
    return out
