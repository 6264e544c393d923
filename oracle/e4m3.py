"""Per-row e4m3 rounding of decoder weights (the 1-byte weight format of the
decode GEMVs), written from the format definition.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests and the
CPU-baseline leg of ``bench.py`` use it to give the oracle the weights the
library computes with when it is created with the e4m3 weight format.  The
pages' decoder streams bf16 or f32 weights; this format is an extension of
their weight-streaming decode step, so no page fixes it, and the rules below
follow the OCP 8-bit floating point specification's E4M3 encoding:

* a byte is sign (bit 7) | exponent (bits 6..3, bias 7) | mantissa (bits 2..0);
* exponent field 0 encodes subnormals m/8 * 2^-6, so the spacing below 2^-6 is
  2^-9; other fields encode (1 + m/8) * 2^(e - 7);
* exponent 15 with mantissa 7 is NaN; there are no infinities, so the largest
  finite magnitude is (1 + 6/8) * 2^8 = 448;
* rounding is to the nearest value, ties to the even mantissa, saturating at
  +-448 (the conversion the library uses, "satfinite").

A weight row w gets the scale 2^e, e the smallest integer with
max|w| <= 448 * 2^e (1 for an all-zero row), and each weight becomes
round_e4m3(w / 2^e) * 2^e.  Scaling by a power of two is exact, so every step
is exact in float64 except the one rounding to e4m3.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Values (float64) of e4m3 bytes; NaN for the NaN patterns."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    return np.where((e == 15) & (m == 7), np.nan, sign * mag)


def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value of each element (ties to even, saturating at
    +-448), as float64."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                 # a in [2^(ex-1), 2^ex)
    e = np.maximum(ex - 1, -6)          # subnormals share the spacing of 2^-6's binade
    step = np.ldexp(1.0, e - 3)         # three mantissa bits
    # a / step is exact; numpy rounds halves to even, and within a binade the
    # multiple's parity is the mantissa's (a carry lands on the next binade's
    # even mantissa 0)
    q = np.minimum(np.round(a / step) * step, E4M3_MAX)
    return np.copysign(q, x)


def row_scales(w) -> np.ndarray:
    """Power-of-two scale of each row of w (float32 [rows, cols]): the
    smallest 2^e with max|w| <= 448 * 2^e, computed as the library does
    (float32 division by 448, then the exponent of the quotient)."""
    w = np.asarray(w, np.float32)
    amax = np.max(np.abs(w), axis=1).astype(np.float32)
    r = amax / np.float32(E4M3_MAX)
    f, x = np.frexp(r)
    e = np.where(f == np.float32(0.5), x - 1, x)
    e = np.where(amax > 0, e, 0)
    return np.ldexp(np.float32(1.0), e.astype(np.int32)).astype(np.float32)


def quantize_rows(w):
    """(rounded weights float32 [rows, cols], scales float32 [rows], e4m3
    values float64 [rows, cols]) of the rows of w."""
    w = np.asarray(w, np.float32)
    s = row_scales(w)
    q = e4m3_round(w.astype(np.float64) / s[:, None].astype(np.float64))
    return (q * s[:, None]).astype(np.float32), s, q


E4M3_TENSORS = ("q", "k", "v", "o", "gate", "up", "down")


def e4m3_weights(weights: dict) -> dict:
    """The model the library computes with for the e4m3 weight format: every
    projection matrix and the tied embedding rounded row by row; norm weights
    unchanged."""
    out = {k: v for k, v in weights.items() if k != "layers"}
    out["embed"] = quantize_rows(weights["embed"])[0]
    out["layers"] = []
    for L in weights["layers"]:
        d = dict(L)
        for n in E4M3_TENSORS:
            d[n] = quantize_rows(L[n])[0]
        out["layers"].append(d)
    return out
