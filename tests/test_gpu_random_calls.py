"""Seeded random calls across the whole supported domain, against the CPU oracle.

Each query call draws M (spread over 1..256, so that every kernel form and
its boundaries are crossed: the CTA-tile and warp-tile decode kernels, the
chunked CTA-tile kernel at two, three and four CTAs per SM, the tcgen05
kernel), H, the nope dim, the format pair, the q_nope / q_pe layout (contiguous,
views of the upstream [M,H,K+64] projection, head-major q_nope), a pitched
output with canaries in the padding and the pdl mode, and compares the
result with the oracle: q_pe bit-exact, the BF16 projection within its
tolerance, E4M3 within one ulp.  Each V call draws M, H, the weight format,
the x layout (contiguous, a padded view, head-major), a pitched output and
the pdl mode.  Inputs are the library's seeded synthetic layers.
"""

import numpy as np
import pytest
import torch

import mla_decode_query_gb300 as mq
import oracle
from helpers import check_bf16_region, check_output, to_device, to_host_bits
from mla_decode_query_gb300 import inputs

pytestmark = pytest.mark.gpu

D = 576
V = 128
C = 512
CANARY = 0x5A


def _draw_m(rng):
    lo, hi = [(1, 33), (33, 97), (97, 257), (1, 17)][int(rng.integers(0, 4))]
    return int(rng.integers(lo, hi))


def _query_call(rng, i):
    M = _draw_m(rng)
    H = int(rng.choice([8, 11, 16]))
    K = int(rng.choice([128, 192]))
    fmt = str(rng.choice(["bf16", "mxfp8"]))
    od = str(rng.choice(["bf16", "e4m3"]))
    layout = str(rng.choice(["contiguous", "views", "head_major"]))
    pad = int(rng.choice([0, 16, 48]))  # output row padding, elements (rows stay 16-byte multiples)
    pdl = int(rng.integers(0, 3))
    d = inputs.make_layer(inputs.layer_seed(70, i), H, fmt, m_max=M, nope=K)
    qs = inputs.make_q_scale(70 + i) if od == "e4m3" else None
    if layout == "contiguous":
        qn, qn_ts, qn_hs = to_device(d["q_nope"]), H * K, K
        qp, qp_ts, qp_hs = to_device(d["q_pe"]), H * 64, 64
    elif layout == "views":
        q = to_device(np.ascontiguousarray(np.concatenate([d["q_nope"], d["q_pe"]], axis=-1)).reshape(-1))
        qn, qn_ts, qn_hs = q, H * (K + 64), K + 64
        qp, qp_ts, qp_hs = q[K:], H * (K + 64), K + 64
    else:
        qn = to_device(np.ascontiguousarray(np.transpose(d["q_nope"], (1, 0, 2))).reshape(-1))
        qn_ts, qn_hs = K, M * K
        qp, qp_ts, qp_hs = to_device(d["q_pe"]), H * 64, 64
    stride = D * H + pad
    elem = torch.int16 if od == "bf16" else torch.uint8
    fill = (CANARY << 8 | CANARY) if od == "bf16" else CANARY
    out = torch.full((M * stride + 64,), fill, dtype=elem, device="cuda")
    w = to_device(d["weight"])
    sc = None if d["weight_scale"] is None else to_device(d["weight_scale"])
    q_scale = None if qs is None else torch.tensor([qs], dtype=torch.float32, device="cuda")
    st = mq.mlaqp_run_strided(qn, qn_ts, qn_hs, qp, qp_ts, qp_hs, w, sc, out, stride, q_scale, M, H, K, fmt, od,
                              pdl=pdl)
    where = f"call {i}: M{M} H{H} K{K} {fmt}->{od} {layout} pad{pad} pdl{pdl}"
    assert st == mq.MLAQP_OK, f"{where}: {mq.mlaqp_last_error()}"
    torch.cuda.synchronize()
    bits = to_host_bits(out, np.uint16 if od == "bf16" else np.uint8)
    rows = np.stack([bits[m * stride: m * stride + D * H].reshape(H, D) for m in range(M)])
    mask = np.zeros(bits.shape, dtype=bool)
    for m in range(M):
        mask[m * stride: m * stride + D * H] = True
    assert (bits[~mask] == fill).all(), f"{where}: bytes outside the output rows changed"
    ref, acc = oracle.mla_query(d["q_nope"], d["q_pe"], d["weight"], d["weight_scale"], fmt, od, qs)
    check_output(rows, ref, acc, od, where)


def test_random_query_calls(cuda_device):
    rng = np.random.default_rng(20261203)
    for i in range(40):
        _query_call(rng, i)


def _v_call(rng, i):
    M = _draw_m(rng)
    H = int(rng.choice([8, 11, 16]))
    fmt = str(rng.choice(["bf16", "mxfp8"]))
    layout = str(rng.choice(["contiguous", "padded", "head_major"]))
    pad = int(rng.choice([0, 8, 40]))
    pdl = int(rng.integers(0, 3))
    d = inputs.make_v_layer(inputs.layer_seed(71, i), H, fmt, m_max=M)
    if layout == "contiguous":
        x, x_ts, x_hs = to_device(d["x"]), H * C, C
    elif layout == "padded":  # x as the first 512 columns of a [M, H, 576] buffer
        padded = np.zeros((M, H, D), dtype=np.uint16)
        padded[..., :C] = d["x"]
        x, x_ts, x_hs = to_device(padded), H * D, D
    else:
        x = to_device(np.ascontiguousarray(np.transpose(d["x"], (1, 0, 2))))
        x_ts, x_hs = C, M * C
    stride = V * H + pad
    out = torch.full((M * stride + 64,), CANARY << 8 | CANARY, dtype=torch.int16, device="cuda")
    w = to_device(d["weight"])
    sc = None if d["weight_scale"] is None else to_device(d["weight_scale"])
    st = mq.mlaqp_v_up_run(x, x_ts, x_hs, w, sc, out, stride, M, H, fmt, pdl=pdl)
    where = f"v call {i}: M{M} H{H} {fmt} {layout} pad{pad} pdl{pdl}"
    assert st == mq.MLAQP_OK, f"{where}: {mq.mlaqp_last_error()}"
    torch.cuda.synchronize()
    bits = to_host_bits(out, np.uint16)
    rows = np.stack([bits[m * stride: m * stride + V * H].reshape(H, V) for m in range(M)])
    mask = np.zeros(bits.shape, dtype=bool)
    for m in range(M):
        mask[m * stride: m * stride + V * H] = True
    assert (bits[~mask] == (CANARY << 8 | CANARY)).all(), f"{where}: bytes outside the output rows changed"
    _, acc = oracle.mla_v_up(d["x"], d["weight"], d["weight_scale"], fmt)
    check_bf16_region(rows, acc, where)


def test_random_v_up_calls(cuda_device):
    rng = np.random.default_rng(20261204)
    for i in range(30):
        _v_call(rng, i)
