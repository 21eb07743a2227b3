"""Independent numpy restatement of the MX element formats, used only to pin the oracle.

Nothing here is shared with the oracle (which encodes by codebook search) or
with the CUDA library.  Rounding here is arithmetic: split the magnitude into
binade and quantum with frexp, round the quotient with numpy's
round-half-to-even, saturate.  E4M3 decoding goes through torch's
``float8_e4m3fn`` dtype, a library routine.
"""
from __future__ import annotations

import numpy as np
import torch

E4M3, E2M1 = 0, 1
MBITS = {E4M3: 3, E2M1: 1}
EMIN = {E4M3: -6, E2M1: 0}  # unbiased exponent of the smallest normal
EMAX = {E4M3: 8, E2M1: 2}  # unbiased exponent of the largest normal
MAXV = {E4M3: 448.0, E2M1: 6.0}
E2M1_TABLE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                       -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def rne_value(y, fmt):
    """Round already-scaled values to the format's grid (RNE, satfinite); keeps the sign."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex - 1, EMIN[fmt])
    q = np.ldexp(1.0, e - MBITS[fmt])
    v = np.rint(a / q) * q
    v = np.minimum(v, MAXV[fmt])
    return np.copysign(v, y)


def e4m3_decode_all():
    """Values of all 256 E4M3 codes through torch's float8_e4m3fn (NaN for 0x7F, 0xFF)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


E4M3_TABLE = e4m3_decode_all()


def decode(codes, fmt):
    codes = np.asarray(codes).astype(np.int64)
    return E4M3_TABLE[codes & 255] if fmt == E4M3 else E2M1_TABLE[codes & 15]


def scale_exponent(amax, fmt):
    """Unbiased exponent of the shared scale: floor(log2 amax) - emax, clamped to E8M0's range."""
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(np.where(amax > 0, amax, 1.0))
    p = ex - 1 - EMAX[fmt]
    p = np.clip(p, -127, 127)
    tiny = amax < 2.0 ** -126  # zero or fp32-subnormal block
    return np.where(tiny, -127, p), tiny


def quantize_values(v, fmt):
    """fp32 rows [..., K] -> dequantised values of their MX quantisation (fp64), and scale bytes."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    shp = v.shape
    blocks = v.reshape(-1, 32)
    amax = np.abs(blocks).max(axis=1)
    p, tiny = scale_exponent(amax, fmt)
    X = np.ldexp(1.0, p)[:, None]
    vals = rne_value(blocks / X, fmt) * X
    vals = np.where(tiny[:, None], np.copysign(0.0, blocks), vals)
    return vals.reshape(shp), (p + 127).astype(np.uint8).reshape(shp[:-1] + (shp[-1] // 32,))


def unpack_fp4(packed):
    """uint8 [..., K/2] -> codes [..., K], element 2i from the low nibble."""
    packed = np.asarray(packed, dtype=np.uint8)
    lo = packed & 15
    hi = packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(packed.shape[:-1] + (packed.shape[-1] * 2,))


def dequant_weights(packed, scales):
    """MXFP4 weights -> fp64 values."""
    codes = unpack_fp4(packed)
    vals = E2M1_TABLE[codes]
    sc = np.ldexp(1.0, scales.astype(np.int64) - 127)
    return vals * np.repeat(sc, 32, axis=-1)


def bf16_rne(d):
    """float64 -> bf16 values (fp64), round to nearest even, computed from the double directly."""
    d = np.asarray(d, dtype=np.float64)
    a = np.abs(d)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex - 1, -126)
    q = np.ldexp(1.0, e - 7)
    return np.copysign(np.rint(a / q) * q, d)


def bf16_bits_to_f64(bits):
    with np.errstate(invalid="ignore"):
        return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
