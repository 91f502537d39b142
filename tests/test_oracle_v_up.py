"""Pins of the oracle's V up-projection (CPU only).

What pins it, other than itself:
  * brute force: a pure-Python triple loop with correctly rounded sums
    (math.fsum) over operands decoded by PyTorch's dtype casts;
  * closed forms: identity and one-hot weights, small-integer data;
  * the MXFP8 scale axis: raising one scale byte doubles exactly the 32
    output columns of its block and nothing else;
  * a library routine: numpy.einsum in float64 on the decoded operands.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from mla_decode_query_gb300 import inputs

C, V = 512, 128


def _lib_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def _lib_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _lib_weight(d, fmt):
    if fmt == "bf16":
        return _lib_bf16(d["weight"])
    return _lib_e4m3(d["weight"]) * np.power(2.0, d["weight_scale"].astype(np.int64) - 127).repeat(32, axis=-1)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
def test_brute_force_triple_loop(fmt):
    H, M = 2, 3
    d = inputs.make_v_layer(41, H, fmt, m_max=M)
    out, acc = oracle.mla_v_up(d["x"], d["weight"], d["weight_scale"], fmt)
    x = _lib_bf16(d["x"])
    w = _lib_weight(d, fmt)
    for m in range(M):
        for h in range(H):
            for v in list(range(0, V, 13)) + [V - 1]:
                terms = [x[m, h, c] * w[h, c, v] for c in range(C)]
                exact = math.fsum(terms)
                assert abs(acc[m, h, v] - exact) <= 1e-13 * math.fsum(abs(t) for t in terms) + 1e-300
                _assert_nearest_bf16(int(out[m, h, v]), exact)


def _assert_nearest_bf16(b, exact):
    """BF16 code b is a nearest BF16 value to `exact`, ties to the even code
    (checked against both neighbouring codes of the same sign)."""
    val = _lib_bf16(np.array([b], dtype=np.uint16))[0]
    err = abs(val - exact)
    mag = b & 0x7FFF
    for nb in (mag - 1, mag + 1):
        if 0 <= nb < 0x7F80:
            nval = abs(_lib_bf16(np.array([nb], dtype=np.uint16))[0])
            nerr = abs(nval - abs(exact))
            assert err < nerr or (err == nerr and mag % 2 == 0), (b, exact)
    assert (b >> 15) == (1 if exact < 0 else 0) or val == 0


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
def test_einsum_cross_check(fmt):
    d = inputs.make_v_layer(42, 11, fmt, m_max=5)
    _, acc = oracle.mla_v_up(d["x"], d["weight"], d["weight_scale"], fmt)
    ref = np.einsum("mhc,hcv->mhv", _lib_bf16(d["x"]), _lib_weight(d, fmt))
    np.testing.assert_allclose(acc, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
def test_identity_weights_copy_x(fmt):
    H, M = 3, 4
    x = inputs.make_v_layer(43, H, fmt, m_max=M)["x"]
    eye = np.zeros((H, C, V), dtype=np.float32)
    for v in range(V):
        eye[:, v, v] = 1.0
    if fmt == "bf16":
        w, s = _bf16_bits(eye), None
    else:
        w = np.where(eye == 1.0, 0x38, 0x00).astype(np.uint8)
        s = np.full((H, C, V // 32), 127, dtype=np.uint8)
    out, _ = oracle.mla_v_up(x, w, s, fmt)
    np.testing.assert_array_equal(out, x[..., :V])


def test_one_hot_weight():
    H, M = 2, 5
    x = inputs.make_v_layer(44, H, "bf16", m_max=M)["x"]
    for (h0, c0, v0, c) in [(0, 0, 0, 1.5), (1, 511, 127, -0.375), (1, 300, 64, 3.0)]:
        w = np.zeros((H, C, V), dtype=np.float32)
        w[h0, c0, v0] = c
        out, _ = oracle.mla_v_up(x, _bf16_bits(w), None, "bf16")
        np.testing.assert_array_equal(out[:, h0, v0], _bf16_bits(_lib_bf16(x[:, h0, c0]) * c))
        mask = np.ones((M, H, V), dtype=bool)
        mask[:, h0, v0] = False
        assert not out[mask].any()


def test_mxfp8_scale_block_is_along_the_output_axis():
    H, M = 2, 3
    d = inputs.make_v_layer(45, H, "mxfp8", m_max=M)
    _, acc = oracle.mla_v_up(d["x"], d["weight"], d["weight_scale"], "mxfp8")
    x = _lib_bf16(d["x"])
    w = _lib_weight(d, "mxfp8")
    for (h0, c0, j) in [(0, 7, 0), (1, 400, 3), (1, 0, 2)]:
        s2 = d["weight_scale"].copy()
        s2[h0, c0, j] += 1
        _, acc2 = oracle.mla_v_up(d["x"], d["weight"], s2, "mxfp8")
        delta = acc2 - acc
        expect = np.zeros_like(acc)
        expect[:, h0, 32 * j:32 * j + 32] = x[:, h0, c0, None] * w[h0, c0, 32 * j:32 * j + 32]
        np.testing.assert_allclose(delta, expect, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
def test_small_integer_sums_are_exact(fmt):
    d = inputs.small_integer_v_layer(46, 8, 9, fmt)
    out, acc = oracle.mla_v_up(d["x"], d["weight"], d["weight_scale"], fmt)
    assert np.all(acc == np.round(acc)) and np.abs(acc).max() <= 1024
    np.testing.assert_array_equal(_lib_bf16(out), _lib_bf16(_bf16_bits(acc.astype(np.float32))))


def test_shape_is_checked():
    d = inputs.make_v_layer(47, 2, "bf16", m_max=2)
    with pytest.raises(ValueError):
        oracle.mla_v_up(d["x"][..., :128], d["weight"][:, :128, :], None, "bf16")


def test_algorithmic_bytes_closed_form():
    # W_UV + scales + x + out, H = 16
    assert oracle.v_up_algorithmic_bytes(1, 16, "bf16") == 16 * 512 * 128 * 2 + 2 * 16 * 512 + 2 * 16 * 128
    assert oracle.v_up_algorithmic_bytes(32, 16, "mxfp8") == (16 * 512 * 128 + 16 * 512 * 4 + 2 * 32 * 16 * 512
                                                             + 2 * 32 * 16 * 128)
