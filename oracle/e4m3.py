"""FP8 e4m3fn codec, written from the format's definition.  Test infrastructure.

The pages say K and V are quantised to FP8 once, when a chunk enters the cache
([ai.info] § "La gestione della cache spostata al momento della scrittura";
[neurocartel] § "Кэш: 240 attention calls и работа на запись"), and that the
attention reads them with per-head scales ([ai.info] § "Latenza dei turni e
altre configurazioni GPU").  They do not name the FP8 variant; e4m3 is the
reading used throughout.

e4m3fn layout: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
  exponent field 0       -> subnormal, value = m * 2**-9
  exponent field 1..15   -> normal,    value = (1 + m/8) * 2**(e-7)
  e = 15 and m = 7       -> NaN (0x7F / 0xFF); there is no infinity
Largest finite value 448 (0x7E), smallest normal 2**-6, smallest subnormal 2**-9.

Encoding is round-to-nearest-even with saturation to +-448 ("satfinite"):
anything whose magnitude exceeds 448, infinities included, becomes +-448;
NaN becomes 0x7F.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def decode_table() -> np.ndarray:
    """float64 value of each of the 256 codes (NaN for 0x7F and 0xFF)."""
    codes = np.arange(256)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e = (codes >> 3) & 0xF
    m = codes & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = sign * mag
    val[(e == 15) & (m == 7)] = np.nan
    return val


_TABLE = decode_table()


def decode(codes: np.ndarray) -> np.ndarray:
    """uint8 codes -> float64 values (exact)."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(x: np.ndarray) -> np.ndarray:
    """float32 (or float64 holding float32 values) -> uint8 e4m3fn codes.

    Round to nearest, ties to even, saturating at +-448.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint8)
    nan = np.isnan(x)
    neg = np.signbit(x)
    a = np.abs(np.where(nan, 0.0, x))
    a = np.minimum(a, 1e300)  # keep inf out of frexp; it saturates below
    # binade of a: a in [2**e, 2**(e+1)); frexp gives a = f * 2**E, f in [0.5, 1)
    _, E = np.frexp(a)
    e = E.astype(np.int64) - 1
    e_eff = np.maximum(e, -6)               # below 2**-6 the spacing stays 2**-9
    quantum = np.ldexp(1.0, (e_eff - 3))    # 3 mantissa bits
    n = np.rint(a / quantum)                # exact division by a power of two; rint = RNE
    v = n * quantum                         # rounded magnitude, possibly one binade up
    v = np.minimum(v, E4M3_MAX)             # satfinite
    # encode the rounded magnitude v (0 or a representable value <= 448)
    _, Ev = np.frexp(np.where(v > 0, v, 1.0))
    ev = Ev.astype(np.int64) - 1
    is_sub = v < 2.0 ** -6
    field_e = np.where(is_sub, 0, ev + 7)
    mant = np.where(is_sub, np.rint(v / 2.0 ** -9), np.rint((v / np.ldexp(1.0, ev) - 1.0) * 8.0))
    code = (field_e.astype(np.int64) << 3) | mant.astype(np.int64)
    code = np.where(v == 0, 0, code)
    code = code | np.where(neg, 0x80, 0)
    out[...] = code.astype(np.uint8)
    out[nan] = 0x7F
    return out


def ulp_at(mag: np.ndarray) -> np.ndarray:
    """Spacing of the e4m3 grid at magnitude ``mag`` (float64).

    For |x| in [2**e, 2**(e+1)) with e >= -6 the spacing is 2**(e-3); below
    2**-6 it is 2**-9; at and above 256 it is 32.
    """
    mag = np.abs(np.asarray(mag, dtype=np.float64))
    _, E = np.frexp(np.where(mag > 0, mag, 1.0))
    e = np.where(mag > 0, E.astype(np.int64) - 1, -6)
    e = np.clip(e, -6, 8)
    return np.ldexp(1.0, e - 3)
