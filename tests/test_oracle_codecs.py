"""Pins of the oracle's number-format codecs (CPU only).

Each codec is checked against things other than itself: the format
specifications' special values (tests/golden/, with their sources),
exhaustive comparison with independent library implementations (PyTorch's
and ml_dtypes' dtype casts), and tie / boundary cases whose rounding is
fixed by IEEE 754 roundTiesToEven.
"""

from pathlib import Path

import numpy as np
import pytest
import torch

import oracle

GOLDEN = Path(__file__).parent / "golden"


def _rows(name):
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            yield line.split()


def _same(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(
        np.where(np.isnan(a), 0, a), np.where(np.isnan(b), 0, b)) and np.array_equal(
        np.signbit(np.where(np.isnan(a), 0, a)), np.signbit(np.where(np.isnan(b), 0, b)))


# --------------------------------------------------------------------------- BF16

def test_bf16_decode_exhaustive_vs_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert _same(oracle.bf16_to_f64(codes), ref)


def test_bf16_decode_exhaustive_vs_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(ml.bfloat16).astype(np.float64)
    assert _same(oracle.bf16_to_f64(codes), ref)


def test_bf16_rne_golden_cases():
    for x, bits, *_ in _rows("bf16_rounding_cases.txt"):
        got = int(oracle.f64_to_bf16_rne(np.array([float.fromhex(x)]))[0])
        assert got == int(bits, 16), (x, hex(got), bits)


def test_bf16_rne_matches_torch_on_float32_inputs():
    # For binary32 inputs one rounding step to BF16 is what torch's cast does.
    rng = np.random.Generator(np.random.PCG64(7))
    bits = rng.integers(0, 2**32, size=100_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    edges = np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 3.4e38, 1e-45, 1.1754944e-38],
                     dtype=np.float32)
    x = np.concatenate([x, edges])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16_rne(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_rne_ties_from_float64():
    # Exact midpoints between adjacent BF16 values at many scales go to the
    # even code; a nudge of one float64 ulp either way decides the direction.
    rng = np.random.Generator(np.random.PCG64(8))
    lo_bits = rng.integers(0x0080, 0x7F7F, size=20_000).astype(np.uint16) & np.uint16(0xFFFE)
    for parity in (0, 1):
        b = (lo_bits | np.uint16(parity)).astype(np.uint16)
        lo = oracle.bf16_to_f64(b)
        hi = oracle.bf16_to_f64(b + np.uint16(1))
        mid = (lo + hi) / 2
        even = b if parity == 0 else b + np.uint16(1)
        np.testing.assert_array_equal(oracle.f64_to_bf16_rne(mid), even)
        np.testing.assert_array_equal(oracle.f64_to_bf16_rne(np.nextafter(mid, np.inf)), b + np.uint16(1))
        np.testing.assert_array_equal(oracle.f64_to_bf16_rne(np.nextafter(mid, -np.inf)), b)


# --------------------------------------------------------------------------- E4M3

def test_e4m3_golden_values():
    for code, val, *_ in _rows("e4m3_special_values.txt"):
        got = oracle.e4m3_to_f64(np.array([int(code, 16)], dtype=np.uint8))[0]
        exp = float(val)
        if np.isnan(exp):
            assert np.isnan(got), code
        else:
            assert got == exp and np.signbit(got) == np.signbit(exp), (code, got, exp)


def test_e4m3_decode_exhaustive_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert _same(oracle.e4m3_to_f64(codes), ref)


def test_e4m3_decode_exhaustive_vs_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    codes = np.arange(256, dtype=np.uint8)
    ref = codes.view(ml.float8_e4m3fn).astype(np.float64)
    assert _same(oracle.e4m3_to_f64(codes), ref)


def test_e4m3_encode_golden_cases():
    for x, code, *_ in _rows("e4m3_rounding_cases.txt"):
        got = int(oracle.f32_to_e4m3_satfinite(np.array([float(x)], dtype=np.float32))[0])
        assert got == int(code, 16), (x, hex(got), code)


def _e4m3_boundary_inputs():
    mags = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = (mags[:-1] + mags[1:]) / 2  # exact in float32
    pts = np.concatenate([mags, mids]).astype(np.float32)
    pts = np.concatenate([pts, np.nextafter(pts, np.float32(np.inf)), np.nextafter(pts, np.float32(-np.inf))])
    pts = np.concatenate([pts, -pts])
    rng = np.random.Generator(np.random.PCG64(9))
    rnd = (rng.standard_normal(200_000) * np.exp(rng.uniform(-12, 7, 200_000))).astype(np.float32)
    return np.concatenate([pts, rnd])


def test_e4m3_encode_vs_torch_after_clamp():
    # torch's cast is round-to-nearest-even but overflows to NaN; clamping to
    # +-448 first gives the saturating behaviour being checked.
    x = _e4m3_boundary_inputs()
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.f32_to_e4m3_satfinite(x), ref)


def test_e4m3_encode_vs_ml_dtypes_after_clamp():
    ml = pytest.importorskip("ml_dtypes")
    x = _e4m3_boundary_inputs()
    ref = np.clip(x, -448, 448).astype(ml.float8_e4m3fn).view(np.uint8)
    np.testing.assert_array_equal(oracle.f32_to_e4m3_satfinite(x), ref)


def test_e4m3_encode_saturates_and_nan():
    x = np.array([449, 479.9, 480, 1e38, np.inf, -np.inf, -1e38, np.nan], dtype=np.float32)
    got = oracle.f32_to_e4m3_satfinite(x)
    np.testing.assert_array_equal(got[:5], 0x7E)
    np.testing.assert_array_equal(got[5:7], 0xFE)
    assert got[7] & 0x7F == 0x7F


def test_e4m3_ordinal_counts_ulps():
    codes = np.arange(0x7F, dtype=np.uint8)
    o = oracle.e4m3_ordinal(codes)
    np.testing.assert_array_equal(np.diff(o), 1)
    assert oracle.e4m3_ordinal(np.array([0x80], dtype=np.uint8))[0] == 0
    assert oracle.e4m3_ordinal(np.array([0x81], dtype=np.uint8))[0] == -1


# --------------------------------------------------------------------------- E8M0

def test_e8m0_golden_values():
    for code, val, *_ in _rows("e8m0_special_values.txt"):
        got = oracle.e8m0_to_f64(np.array([int(code, 16)], dtype=np.uint8))[0]
        exp = float(val)
        assert (np.isnan(got) and np.isnan(exp)) or got == exp, (code, got, exp)


def test_e8m0_exhaustive_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert _same(oracle.e8m0_to_f64(codes), ref)


def test_e8m0_exhaustive_vs_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    codes = np.arange(256, dtype=np.uint8)
    ref = codes.view(ml.float8_e8m0fnu).astype(np.float64)
    assert _same(oracle.e8m0_to_f64(codes), ref)
