"""Pins of the oracle's projection and assembly (CPU only).

What pins it, other than itself:
  * brute force: a pure-Python triple loop with correctly rounded sums
    (math.fsum) whose operands are decoded by the libraries' dtype casts;
  * closed forms: identity and one-hot weights, small-integer data;
  * invariants: power-of-two scaling, the q_pe bit copy;
  * a library routine: numpy.einsum in float64 on the decoded operands;
  * the E4M3 output of identity weights against PyTorch's E4M3 cast.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from mla_decode_query_gb300 import inputs

K, N, R = 128, 512, 64


def _lib_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def _lib_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _layer(seed, H, M, fmt):
    d = inputs.make_layer(seed, H, fmt, m_max=M)
    return d["q_nope"], d["q_pe"], d["weight"], d["weight_scale"]


@pytest.mark.parametrize("fmt,K", [("bf16", 128), ("mxfp8", 128), ("bf16", 192), ("mxfp8", 192)])
def test_brute_force_triple_loop(fmt, K):
    H, M = 2, 3
    d = inputs.make_layer(11, H, fmt, m_max=M, nope=K)
    qn, qp, w, s = d["q_nope"], d["q_pe"], d["weight"], d["weight_scale"]
    _, acc = oracle.mla_query(qn, qp, w, s, fmt, "bf16")
    q = _lib_bf16(qn)
    if fmt == "bf16":
        wv = _lib_bf16(w)
    else:
        wv = _lib_e4m3(w) * np.power(2.0, s.astype(np.int64) - 127).repeat(32, axis=-1)
    cols = list(range(0, N, 37)) + [N - 1]
    for m in range(M):
        for h in range(H):
            for n in cols:
                terms = [q[m, h, k] * wv[h, k, n] for k in range(K)]
                exact = math.fsum(terms)
                scale = math.fsum(abs(x) for x in terms)
                assert abs(acc[m, h, n] - exact) <= 1e-13 * scale + 1e-300, (m, h, n)


def test_einsum_cross_check():
    qn, qp, w, s = _layer(12, 11, 5, "mxfp8")
    _, acc = oracle.mla_query(qn, qp, w, s, "mxfp8", "bf16")
    wv = _lib_e4m3(w) * np.power(2.0, s.astype(np.int64) - 127).repeat(32, axis=-1)
    ref = np.einsum("mhk,hkn->mhn", _lib_bf16(qn), wv)
    np.testing.assert_allclose(acc, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
def test_identity_weights_copy_q_nope(fmt):
    H, M = 3, 4
    qn, qp, _, _ = _layer(13, H, M, fmt)
    eye = np.zeros((H, K, N), dtype=np.float32)
    for k in range(K):
        eye[:, k, k] = 1.0
    if fmt == "bf16":
        w, s = _bf16_bits(eye), None
    else:
        w = np.where(eye == 1.0, 0x38, 0x00).astype(np.uint8)
        s = np.full((H, K, N // 32), 127, dtype=np.uint8)
    out, _ = oracle.mla_query(qn, qp, w, s, fmt, "bf16")
    np.testing.assert_array_equal(out[..., :K], qn)
    assert not out[..., K:N].any()
    np.testing.assert_array_equal(out[..., N:], qp)


def test_one_hot_weight():
    H, M = 2, 5
    qn, qp, _, _ = _layer(14, H, M, "bf16")
    for (h0, k0, n0, c) in [(0, 0, 0, 1.5), (1, 127, 511, -0.375), (1, 64, 300, 3.0)]:
        w = np.zeros((H, K, N), dtype=np.float32)
        w[h0, k0, n0] = c
        out, _ = oracle.mla_query(qn, qp, _bf16_bits(w), None, "bf16", "bf16")
        expect = _bf16_bits(_lib_bf16(qn[:, h0, k0]) * c)  # exact product, exact cast
        np.testing.assert_array_equal(out[:, h0, n0], expect)
        mask = np.ones((M, H, N), dtype=bool)
        mask[:, h0, n0] = False
        assert not out[..., :N][mask].any()


def test_scale_of_two_invariance_mxfp8():
    H, M = 2, 6
    qn, qp, w, s = _layer(15, H, M, "mxfp8")
    _, acc = oracle.mla_query(qn, qp, w, s, "mxfp8", "bf16")
    out1, _ = oracle.mla_query(qn, qp, w, s, "mxfp8", "bf16")
    out2, acc2 = oracle.mla_query(qn, qp, w, (s + 1).astype(np.uint8), "mxfp8", "bf16")
    np.testing.assert_array_equal(acc2, 2 * acc)
    v1 = _lib_bf16(out1[..., :N])
    v2 = _lib_bf16(out2[..., :N])
    normal = np.abs(v1) >= 2.0 ** -125
    np.testing.assert_array_equal(v2[normal], 2 * v1[normal])


def test_scale_of_two_invariance_q_and_weights_bf16():
    H, M = 2, 6
    qn, qp, w, _ = _layer(16, H, M, "bf16")
    out1, acc1 = oracle.mla_query(qn, qp, w, None, "bf16", "bf16")
    q2 = _bf16_bits(_lib_bf16(qn) * 2)
    w2 = _bf16_bits(_lib_bf16(w) * 2)
    _, acc_q = oracle.mla_query(q2, qp, w, None, "bf16", "bf16")
    _, acc_w = oracle.mla_query(qn, qp, w2, None, "bf16", "bf16")
    np.testing.assert_array_equal(acc_q, 2 * acc1)
    np.testing.assert_array_equal(acc_w, 2 * acc1)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
def test_q_pe_bit_copy(fmt):
    qn, qp, w, s = _layer(17, 16, 7, fmt)
    out, _ = oracle.mla_query(qn, qp, w, s, fmt, "bf16")
    np.testing.assert_array_equal(out[..., N:], qp)
    assert out.dtype == np.uint16 and out.shape == (7, 16, N + R)


def test_small_integer_sums_are_exact():
    d = inputs.small_integer_layer(18, 8, 9, "mxfp8")
    out, acc = oracle.mla_query(d["q_nope"], d["q_pe"], d["weight"], d["weight_scale"], "mxfp8", "bf16")
    assert np.all(acc == np.round(acc)) and np.abs(acc).max() <= 256
    np.testing.assert_array_equal(_lib_bf16(out[..., :N]), acc)


def test_e4m3_output_of_identity_weights_matches_torch_cast():
    H, M = 2, 8
    qn, qp, _, _ = _layer(19, H, M, "bf16")
    eye = np.zeros((H, K, N), dtype=np.float32)
    for k in range(K):
        eye[:, k, k] = 1.0
    q_scale = np.float32(0.5)  # division by 0.5 is exact: x * 2
    out, _ = oracle.mla_query(qn, qp, _bf16_bits(eye), None, "bf16", "e4m3", q_scale)
    assert out.dtype == np.uint8

    def lib_e4m3(x):
        x = np.clip(np.asarray(x, dtype=np.float32), -448, 448)
        return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    np.testing.assert_array_equal(out[..., :K], lib_e4m3(_lib_bf16(qn) * 2))
    np.testing.assert_array_equal(out[..., N:], lib_e4m3(_lib_bf16(qp) * 2))
    assert not (out[..., K:N] & 0x7F).any()


def test_e4m3_small_scale_saturates():
    qn, qp, w, s = _layer(20, 2, 4, "mxfp8")
    out, acc = oracle.mla_query(qn, qp, w, s, "mxfp8", "e4m3", np.float32(1e-3))
    big = np.abs(acc) > 0.5
    assert big.any()
    np.testing.assert_array_equal(out[..., :N][big] & 0x7F, 0x7E)


def test_scale_arguments_are_validated():
    qn, qp, w, s = _layer(21, 2, 2, "mxfp8")
    with pytest.raises(ValueError):
        oracle.mla_query(qn, qp, w, s, "mxfp8", "e4m3", None)
    with pytest.raises(ValueError):
        oracle.mla_query(qn, qp, w, s, "mxfp8", "bf16", np.float32(1.0))
    with pytest.raises(ValueError):
        oracle.decode_weight(w, s, "bf16")


def test_workspace_write_leaves_other_rows():
    H, M, stride = 2, 3, 2 * 576 + 64
    out = np.arange(M * H * 576, dtype=np.uint16).reshape(M, H, 576)
    ws = np.full(5 * stride, 0xABCD, dtype=np.uint16)
    got = oracle.write_workspace(ws, out, stride)
    for m in range(5):
        row = got[m * stride:(m + 1) * stride]
        if m < M:
            np.testing.assert_array_equal(row[:H * 576], out[m].reshape(-1))
            assert (row[H * 576:] == 0xABCD).all()
        else:
            assert (row == 0xABCD).all()


def test_algorithmic_bytes_closed_form():
    # weights + scales + q_nope + q_pe + output, per layer call, H = 16
    assert oracle.algorithmic_bytes(1, 16, "bf16", "bf16") == 2_121_728
    assert oracle.algorithmic_bytes(32, 16, "bf16", "bf16") == 2_883_584
    assert oracle.algorithmic_bytes(1, 16, "mxfp8", "e4m3") == 1_096_704
    assert oracle.algorithmic_bytes(32, 16, "mxfp8", "e4m3") == 1_572_864
