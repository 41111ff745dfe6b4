"""Pins for the oracle's FP8 codec: the printed format limits, a library
routine (torch's float8 types) on every code and on in-range values, and a
brute-force nearest-code search on dense grids that include every tie."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "fp8_format_points.json")
FMTS = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2}
TORCH_T = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def _gold():
    with open(GOLD) as f:
        return json.load(f)


def test_decode_printed_points():
    for e in _gold()["decode"]:
        assert oracle.fp8_decode(np.array([e["code"]]), FMTS[e["fmt"]])[0] == e["value"], e


def test_encode_printed_points_and_ties():
    for e in _gold()["encode"]:
        got = int(oracle.fp8_encode(np.array([e["x"]], np.float32), FMTS[e["fmt"]])[0])
        assert got == e["code"], e


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_decode_table_matches_torch(fmt):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.fp8_decode(codes, fmt)
    ref = torch.from_numpy(codes).view(TORCH_T[fmt]).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


def test_decode_special_codes():
    d4 = oracle.fp8_decode(np.arange(256, dtype=np.uint8), oracle.E4M3)
    d5 = oracle.fp8_decode(np.arange(256, dtype=np.uint8), oracle.E5M2)
    # E4M3 ("fn"): only S.1111.111 is NaN, no infinity; E5M2: exponent 31.
    assert [c for c in range(256) if np.isnan(d4[c])] == [0x7F, 0xFF]
    assert not np.isinf(d4).any()
    assert d5[0x7C] == np.inf and d5[0xFC] == -np.inf
    assert [c for c in range(256) if np.isnan(d5[c])] == [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]
    assert d4[0x08] == 2.0 ** -6 and d5[0x01] == 2.0 ** -16 and d5[0x04] == 2.0 ** -14


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_decode_roundtrip_and_monotone(fmt):
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.fp8_decode(codes, fmt)
    fin = np.isfinite(vals)
    back = oracle.fp8_encode(vals[fin].astype(np.float32), fmt)
    assert np.array_equal(back, codes[fin])
    x = np.linspace(-2 * oracle_max(fmt), 2 * oracle_max(fmt), 200001).astype(np.float32)
    dec = oracle.fp8_decode(oracle.fp8_encode(x, fmt), fmt)
    assert np.all(np.diff(dec) >= 0)


def oracle_max(fmt):
    return 448.0 if fmt == oracle.E4M3 else 57344.0


def _tie_grid(fmt):
    """Every finite code value, every midpoint between neighbours, and points
    just either side of each midpoint, with both signs."""
    vals = np.unique(oracle.fp8_decode(np.arange(128, dtype=np.uint8), fmt))
    vals = vals[np.isfinite(vals)]
    mids = (vals[:-1] + vals[1:]) / 2
    pts = np.concatenate([vals, mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf),
                          [oracle_max(fmt) * 1.03, oracle_max(fmt) * 1.07, 1e30, 1e-30]])
    pts = pts.astype(np.float32)
    return np.concatenate([pts, -pts, np.array([0.0, -0.0], np.float32)])


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_matches_bruteforce_on_ties(fmt):
    x = _tie_grid(fmt)
    assert np.array_equal(oracle.fp8_encode(x, fmt), oracle.fp8_encode_bruteforce(x, fmt))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_matches_bruteforce_random(fmt):
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-20, 18, 200000))).astype(np.float32)
    assert np.array_equal(oracle.fp8_encode(x, fmt), oracle.fp8_encode_bruteforce(x, fmt))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_matches_torch_in_range(fmt):
    # torch's fp32 -> float8 cast rounds to nearest-even but does not
    # saturate, so compare inside +-max only.
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(500000) * np.exp2(rng.integers(-24, 16, 500000))).astype(np.float32)
    x = np.concatenate([x, _tie_grid(fmt)])
    x = x[np.abs(x) <= oracle_max(fmt)]
    ref = torch.from_numpy(x).to(TORCH_T[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(oracle.fp8_encode(x, fmt), ref)


def test_encode_nan_and_inf():
    x = np.array([np.nan, np.inf, -np.inf], np.float32)
    assert list(oracle.fp8_encode(x, oracle.E4M3)) == [0x7F, 0x7E, 0xFE]
    assert list(oracle.fp8_encode(x, oracle.E5M2)) == [0x7F, 0x7B, 0xFB]


def test_int8_decode_is_the_excess_128_integer():
    codes = np.arange(256, dtype=np.uint8)
    want = codes.astype(np.float64) - 128.0
    assert np.array_equal(oracle.fp8_decode(codes, oracle.INT8), want)


def test_int8_encode_matches_numpy_rint_and_bruteforce():
    """Symmetric INT8 codes: nearest integer, ties to even (numpy's rint),
    clamped to [-127, 127], stored + 128; every half-integer tie in range and
    random values, against numpy and against the oracle's own scan of all
    codes."""
    rng = np.random.default_rng(11)
    ties = np.arange(-130, 130).astype(np.float32) + np.float32(0.5)
    rand = rng.uniform(-300.0, 300.0, 20000).astype(np.float32)
    edges = np.array([0.0, -0.0, 126.5, -126.5, 127.0, -127.0, 127.49, -127.5, 1e30, -1e30,
                      np.inf, -np.inf], np.float32)
    x = np.concatenate([ties, rand, edges])
    want = (np.clip(np.rint(x.astype(np.float64)), -127, 127) + 128).astype(np.uint8)
    assert np.array_equal(oracle.fp8_encode(x, oracle.INT8), want)
    fin = np.isfinite(x)
    assert np.array_equal(oracle.fp8_encode_bruteforce(x[fin], oracle.INT8), want[fin])
