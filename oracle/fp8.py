"""FP8 E4M3 storage for the KV-cache oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

E4M3 as defined by the OCP 8-bit floating point specification (the format
GB300's fp8 conversions implement): 1 sign bit, 4 exponent bits with bias 7,
3 mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6; the code with
exponent 1111 and mantissa 111 is NaN and there is no infinity, so the largest
finite magnitude is 1.110b * 2^8 = 448.

Quantisation (the KV pages give no format; see the design notes): a value x
of KV head h is stored as code = E4M3(x / scale[h]), with x / scale[h]
computed in fp32 (IEEE division), rounded to the nearest representable value
with ties to an even mantissa, and finite values beyond 448 clamped to 448
(saturation).  Dequantised value = decode(code) * scale[h].
"""
from __future__ import annotations

import numpy as np


def decode_table() -> np.ndarray:
    """float64 value of every code 0..255 (NaN for the two NaN codes)."""
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            out[code] = np.nan
        elif e == 0:
            out[code] = s * (m / 8.0) * 2.0 ** -6
        else:
            out[code] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_TABLE = decode_table()
_POS_VALUES = _TABLE[:127]          # codes 0..126, non-negative finite, increasing


def decode(codes) -> np.ndarray:
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(y) -> np.ndarray:
    """Round-to-nearest-even onto E4M3 with saturation at +-448 (y already
    divided by the scale).  Returns uint8 codes."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    neg = np.signbit(y)
    a_sat = np.minimum(a, 448.0)
    hi = np.clip(np.searchsorted(_POS_VALUES, a_sat, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_hi = np.abs(_POS_VALUES[hi] - a_sat)
    d_lo = np.abs(a_sat - _POS_VALUES[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.uint8)
    code = np.where(np.isnan(y), 0x7F, code).astype(np.uint8)
    return (code | np.where(neg, 0x80, 0x00).astype(np.uint8)).astype(np.uint8)


def quantize_rows(x_bf16_as_f32: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """x [..., Hkv, D] (float32 values of the bf16 inputs), scales [Hkv] float32
    -> uint8 codes of the same shape; the division is done in fp32."""
    x = np.asarray(x_bf16_as_f32, dtype=np.float32)
    s = np.asarray(scales, dtype=np.float32)[:, None]
    return encode((x / s).astype(np.float32).astype(np.float64))


def kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, k_scale, v_scale, block_size=16):
    """Quantise and scatter (numpy arrays; pools uint8 [NB, Hkv, bs, D])."""
    kq = quantize_rows(k_new, k_scale)
    vq = quantize_rows(v_new, v_scale)
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        k_cache[slot // block_size, :, slot % block_size, :] = kq[t]
        v_cache[slot // block_size, :, slot % block_size, :] = vq[t]


def dequantize_pool(pool_u8, scales) -> np.ndarray:
    """uint8 pool [NB, Hkv, bs, D] -> float64 values decode(code) * scale[h]."""
    vals = decode(pool_u8)
    return vals * np.asarray(scales, dtype=np.float64)[None, :, None, None]
