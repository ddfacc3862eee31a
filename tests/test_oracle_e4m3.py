"""Pins for the oracle's e4m3 codec: format definition, library casts, saturation."""
import os

import numpy as np
import pytest
import torch

from oracle import e4m3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_spec.txt")


def _torch_cast(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_spec_code_points():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) >= 10
    for code_s, val_s in rows:
        code = int(code_s, 16)
        got = e4m3.decode(np.array([code], np.uint8))[0]
        if val_s == "nan":
            assert np.isnan(got)
        else:
            want = float(val_s)
            assert got == want and np.signbit(got) == np.signbit(want), (code_s, got, want)
            if code not in (0x80,):
                assert e4m3.encode(np.array([want]))[0] == code


def test_decode_matches_library_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3.decode(np.arange(256, dtype=np.uint8))
    both_nan = np.isnan(lib) & np.isnan(ours)
    assert np.all(both_nan | (lib == ours))


@pytest.mark.parametrize("scale", [1.0, 448.0 / 3.7, 0.013, 1.0 / 64, 1024.0, 448.0 / 81.25])
def test_encode_matches_library_cast_all_bf16(scale):
    bits = np.arange(65536, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        x = (x * np.float32(scale)).astype(np.float32)
    keep = np.isfinite(x) & (np.abs(x) <= 448.0)
    x = x[keep]
    assert np.array_equal(e4m3.encode(x), _torch_cast(x))


def test_encode_at_rounding_midpoints():
    vals = e4m3.decode(np.arange(0, 0x7E, dtype=np.uint8))   # 0 .. 416 (positive finite, below max)
    nxt = e4m3.decode(np.arange(1, 0x7F, dtype=np.uint8))
    mid = ((vals + nxt) / 2).astype(np.float32)              # exact midpoints (representable in fp32)
    probe = np.concatenate([mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9)),
                            -mid, -np.nextafter(mid, np.float32(1e9))]).astype(np.float32)
    assert np.array_equal(e4m3.encode(probe), _torch_cast(probe))
    # ties go to the even code
    codes = e4m3.encode(mid)
    assert np.all(codes % 2 == 0)


def test_encode_random_float32_matches_library():
    rng = np.random.default_rng(1234)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 6, 200000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    assert np.array_equal(e4m3.encode(x), _torch_cast(x))


def test_satfinite():
    big = np.array([448.0, 449.0, 463.99, 464.0, 464.01, 480.0, 1e10, np.inf], np.float64)
    assert np.all(e4m3.encode(big) == 0x7E)
    assert np.all(e4m3.encode(-big) == 0xFE)
    assert e4m3.encode(np.array([np.nan]))[0] == 0x7F


def test_round_trip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    again = e4m3.encode(e4m3.decode(codes))
    zero = codes == 0x80  # -0 keeps its sign
    assert np.array_equal(again[~zero], codes[~zero]) and again[zero][0] == 0x80


def test_ulp_closed_form():
    assert e4m3.ulp_at(np.array([1.0]))[0] == 0.125
    assert e4m3.ulp_at(np.array([1.99]))[0] == 0.125
    assert e4m3.ulp_at(np.array([2.0]))[0] == 0.25
    assert e4m3.ulp_at(np.array([300.0]))[0] == 32.0
    assert e4m3.ulp_at(np.array([0.001]))[0] == 2.0 ** -9
    # spacing equals the gap between neighbouring codes
    vals = e4m3.decode(np.arange(0x08, 0x7E, dtype=np.uint8))
    gaps = np.diff(e4m3.decode(np.arange(0x08, 0x7F, dtype=np.uint8)))
    assert np.array_equal(e4m3.ulp_at(vals), gaps)
