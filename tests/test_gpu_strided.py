"""GPU parity of the general entry point mlaqp_run_strided: nope dim 192
(the GLM shape of SparkInfer PR #75, section What) and strided q_nope /
q_pe views -- the upstream [M, H, K+64] projection output and a head-major
[H, M, K] q_nope -- against the CPU oracle."""

import numpy as np
import pytest
import torch

import mla_decode_query_gb300 as mq
import oracle
from helpers import check_output, to_device, to_host_bits
from mla_decode_query_gb300 import inputs

pytestmark = pytest.mark.gpu
D = 576


def _run_strided(qn, qn_ts, qn_hs, qp, qp_ts, qp_hs, d, M, H, K, fmt, od, qs=None, pdl=False, out=None,
                 stride=None):
    stride = stride or D * H
    w = to_device(d["weight"])
    sc = None if d["weight_scale"] is None else to_device(d["weight_scale"])
    if out is None:
        out = torch.zeros((M * stride,), dtype=torch.int16 if od == "bf16" else torch.uint8, device="cuda")
    q_scale = None if qs is None else torch.tensor([qs], dtype=torch.float32, device="cuda")
    st = mq.mlaqp_run_strided(qn, qn_ts, qn_hs, qp, qp_ts, qp_hs, w, sc, out, stride, q_scale, M, H, K, fmt, od,
                              pdl=pdl)
    assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
    torch.cuda.synchronize()
    bits = to_host_bits(out, np.uint16 if od == "bf16" else np.uint8)
    return np.stack([bits[m * stride: m * stride + H * D].reshape(H, D) for m in range(M)])


@pytest.mark.parametrize("fmt,od", [("bf16", "bf16"), ("bf16", "e4m3"), ("mxfp8", "bf16"), ("mxfp8", "e4m3")])
@pytest.mark.parametrize("H", [8, 11, 16])
def test_nope192_contiguous(cuda_device, fmt, od, H):
    K = 192
    d = inputs.make_layer(inputs.layer_seed(20, H), H, fmt, nope=K)
    qs = inputs.make_q_scale(20) if od == "e4m3" else None
    qn, qp = to_device(d["q_nope"]), to_device(d["q_pe"])
    for M in (1, 5, 8, 9, 17, 24, 32):
        got = _run_strided(qn, H * K, K, qp, H * 64, 64, d, M, H, K, fmt, od, qs, pdl=(M % 2 == 0))
        ref, acc = oracle.mla_query(d["q_nope"][:M], d["q_pe"][:M], d["weight"], d["weight_scale"], fmt, od, qs)
        check_output(got, ref, acc, od, f"K192 {fmt}->{od} H{H} M{M}")


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
@pytest.mark.parametrize("K", [128, 192])
def test_small_integers_bit_exact(cuda_device, fmt, K):
    for H, M in ((16, 32), (11, 9), (8, 1)):
        d = inputs.small_integer_layer(200 + M, H, M, fmt, nope=K)
        got = _run_strided(to_device(d["q_nope"]), H * K, K, to_device(d["q_pe"]), H * 64, 64, d, M, H, K, fmt,
                           "bf16")
        ref, _ = oracle.mla_query(d["q_nope"], d["q_pe"], d["weight"], d["weight_scale"], fmt, "bf16")
        np.testing.assert_array_equal(got, ref, err_msg=f"K{K} {fmt} H{H} M{M}")


@pytest.mark.parametrize("K", [128, 192])
@pytest.mark.parametrize("fmt,od", [("bf16", "bf16"), ("mxfp8", "e4m3")])
def test_views_of_upstream_projection(cuda_device, K, fmt, od):
    # q = [M, H, K+64] per head, nope first: q_nope and q_pe are strided
    # views into the same buffer (token stride H*(K+64), head stride K+64).
    H = 16
    d = inputs.make_layer(inputs.layer_seed(21, K), H, fmt, nope=K)
    qs = inputs.make_q_scale(21) if od == "e4m3" else None
    q = np.concatenate([d["q_nope"], d["q_pe"]], axis=-1)  # [32, H, K+64]
    qd = to_device(np.ascontiguousarray(q).reshape(-1))
    for M in (1, 8, 13, 32):
        got = _run_strided(qd, H * (K + 64), K + 64, qd[K:], H * (K + 64), K + 64, d, M, H, K, fmt, od, qs,
                           pdl=True)
        ref, acc = oracle.mla_query(d["q_nope"][:M], d["q_pe"][:M], d["weight"], d["weight_scale"], fmt, od, qs)
        check_output(got, ref, acc, od, f"views K{K} {fmt}->{od} M{M}")


def test_head_major_q_nope(cuda_device):
    # The BMM layout [H, M, K]: token stride K, head stride M_alloc*K.
    H, K, Ma = 11, 128, 32
    d = inputs.make_layer(inputs.layer_seed(22, 0), H, "bf16")
    hm = np.ascontiguousarray(np.transpose(d["q_nope"], (1, 0, 2)))  # [H, 32, K]
    qn = to_device(hm.reshape(-1))
    qp = to_device(d["q_pe"])
    for M in (1, 16, 32):
        got = _run_strided(qn, K, Ma * K, qp, H * 64, 64, d, M, H, K, "bf16", "bf16")
        ref, acc = oracle.mla_query(d["q_nope"][:M], d["q_pe"][:M], d["weight"], d["weight_scale"], "bf16", "bf16")
        check_output(got, ref, acc, "bf16", f"head-major M{M}")


def test_run_strided_matches_run(cuda_device):
    # With K=128 and contiguous strides the general entry point is the same
    # launch as mlaqp_run: identical bits.
    H, K = 16, 128
    d = inputs.make_layer(inputs.layer_seed(23, 0), H, "mxfp8")
    qs = np.float32(0.05)
    qn, qp = to_device(d["q_nope"]), to_device(d["q_pe"])
    w, sc = to_device(d["weight"]), to_device(d["weight_scale"])
    q_scale = torch.tensor([qs], device="cuda")
    for M in (3, 32):
        a = torch.zeros(M * D * H, dtype=torch.uint8, device="cuda")
        b = torch.zeros_like(a)
        assert mq.mlaqp_run(qn, qp, w, sc, a, D * H, q_scale, M, H, "mxfp8", "e4m3") == mq.MLAQP_OK
        assert mq.mlaqp_run_strided(qn, H * K, K, qp, H * 64, 64, w, sc, b, D * H, q_scale, M, H, K, "mxfp8",
                                    "e4m3") == mq.MLAQP_OK
        torch.cuda.synchronize()
        assert torch.equal(a, b)


def test_can_implement_nope192(cuda_device):
    assert mq.mlaqp_can_implement(16, 32, nope_dim=192, weight_format="mxfp8", out_dtype="e4m3") == 1
    assert mq.mlaqp_can_implement(16, 32, nope_dim=256) == 0
