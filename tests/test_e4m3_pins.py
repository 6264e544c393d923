"""Pins of the oracle's e4m3 weight rounding against the format definition
(OCP 8-bit floating point, E4M3: sign | 4 exponent bits, bias 7 | 3 mantissa
bits; subnormals m/8 * 2^-6; exponent 15 with mantissa 7 is NaN; no
infinities; largest finite 448) and the row-scale rule (the smallest power
of two 2^e with max|w| <= 448 * 2^e)."""
import numpy as np
import pytest

import oracle as O


def finite_positive_values():
    v = O.e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8))      # 0x7F is NaN
    return np.unique(v[v > 0])


def test_decode_landmarks():
    d = O.e4m3_decode
    assert d(0x00) == 0.0 and np.signbit(d(0x80)) and d(0x80) == 0.0
    assert d(0x01) == 2.0 ** -9                   # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9                # largest subnormal
    assert d(0x08) == 2.0 ** -6                    # smallest normal
    assert d(0x38) == 1.0                          # exponent field 7 = bias
    assert d(0x3C) == 1.5
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0  # largest finite
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x78) == 256.0                        # exponent 15, mantissa 0: finite (no infinity)


def test_code_values_are_distinct_and_complete():
    v = finite_positive_values()
    # 15 binades of 8 normals + 7 subnormals
    assert len(v) == 15 * 8 - 1 + 7
    assert v.max() == 448.0 and v.min() == 2.0 ** -9


def test_rounding_is_identity_on_the_grid():
    v = finite_positive_values()
    assert np.array_equal(O.e4m3_round(v), v)
    assert np.array_equal(O.e4m3_round(-v), -v)


def test_midpoints_round_to_even_mantissa():
    v = np.concatenate([[0.0], finite_positive_values()])
    mid = (v[:-1] + v[1:]) / 2
    got = O.e4m3_round(mid)
    codes = np.arange(0x00, 0x7F, dtype=np.uint8)
    val = O.e4m3_decode(codes)
    mant = {float(x): int(c) & 7 for x, c in zip(val, codes) if x >= 0}
    for m, g, lo, hi in zip(mid, got, v[:-1], v[1:]):
        assert g in (lo, hi)
        assert mant[float(g)] % 2 == 0, (m, g)
    # just off a midpoint goes to the nearer neighbour
    eps = 1e-12
    assert np.array_equal(O.e4m3_round(mid - eps * mid), v[:-1])
    assert np.array_equal(O.e4m3_round(mid + eps * mid), v[1:])


@pytest.mark.parametrize("x,want", [(0.1, 13 / 128), (17.0, 16.0), (19.0, 20.0), (2.0 ** -10, 0.0),
                                    (3 * 2.0 ** -10, 2 * 2.0 ** -9), (-0.3, -0.3125), (1.9375, 2.0),
                                    (460.0, 448.0), (1e6, 448.0), (-1e6, -448.0), (0.0, 0.0)])
def test_worked_values(x, want):
    assert O.e4m3_round(x) == want


def test_row_scales_rule():
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((64, 96)) * np.exp(rng.uniform(-20, 8, (64, 1)))).astype(np.float32)
    w[3] = 0.0
    w[5, :] = 0.0
    w[5, 7] = 448.0 * 2.0 ** -3                       # exactly on a power-of-two boundary
    w[6, :] = 0.0
    w[6, 2] = np.float32(448.0 * 2.0 ** -3) * np.float32(1 + 2 ** -7)   # just above it
    s = O.row_scales(w)
    assert s[3] == 1.0
    assert s[5] == 2.0 ** -3 and s[6] == 2.0 ** -2
    amax = np.max(np.abs(w), axis=1).astype(np.float64)
    e = np.log2(s.astype(np.float64))
    assert np.all(e == np.round(e))                     # powers of two
    nz = amax > 0
    assert np.all(amax[nz] <= 448.0 * s[nz])            # the row fits
    assert np.all(amax[nz] > 448.0 * s[nz] / 2)         # and no smaller power of two does


def test_quantize_rows_is_scale_times_grid_value():
    rng = np.random.default_rng(8)
    w = (rng.standard_normal((32, 256)) * 0.02).astype(np.float32)
    r, s, q = O.quantize_rows(w)
    grid = np.concatenate([-finite_positive_values()[::-1], [0.0], finite_positive_values()])
    assert np.all(np.isin(q, grid))
    assert np.array_equal(r.astype(np.float64), q * s[:, None])
    # the largest magnitude of each row lies in (224, 448] before rounding, so
    # its code is in the top binade or on its lower edge
    assert np.all(np.max(np.abs(q), axis=1) >= 224.0)
    # rounded weights are exact in bf16 (at most 4 significant bits)
    bits = r.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)
    # relative rounding error of e4m3 (3 mantissa bits): at most 2^-4 of the
    # value for normals, plus half the subnormal spacing
    err = np.abs(r.astype(np.float64) - w)
    assert np.all(err <= np.abs(w) * 2.0 ** -4 + s[:, None] * 2.0 ** -10)


def test_e4m3_weights_rounds_projections_only():
    rng = np.random.default_rng(9)
    mk = lambda *sh: (rng.standard_normal(sh) * 0.02).astype(np.float32)
    L = {n: mk(8, 16) for n in ("q", "k", "v", "o", "gate", "up", "down")}
    L.update(attn_norm=mk(16) + 1, ffn_norm=mk(16) + 1, q_norm=mk(4) + 1, k_norm=mk(4) + 1)
    w = {"embed": mk(10, 16), "final_norm": mk(16) + 1, "layers": [L]}
    r = O.e4m3_weights(w)
    assert np.array_equal(r["final_norm"], w["final_norm"])
    for n in ("attn_norm", "ffn_norm", "q_norm", "k_norm"):
        assert np.array_equal(r["layers"][0][n], L[n])
    for n in ("q", "k", "v", "o", "gate", "up", "down"):
        assert np.array_equal(r["layers"][0][n], O.quantize_rows(L[n])[0])
        assert not np.array_equal(r["layers"][0][n], L[n])
    assert np.array_equal(r["embed"], O.quantize_rows(w["embed"])[0])
