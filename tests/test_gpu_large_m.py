"""GPU parity of the larger token counts, 33 <= M <= 256 (multi-token
prediction and prefill-sized steps; up to M = 64 the CTA-tile kernel in
32-token chunks, above that the tcgen05 / TMEM kernel), against the CPU
oracle through the C ABI.

Tokens are independent rows of the operation, so one oracle evaluation at
M = 256 serves every smaller M of the same layer (its first M rows).
Tolerances as in helpers: q_pe bit-exact, BF16 within 1e-2*|ref| + 1e-3,
E4M3 within one ulp, exact-arithmetic inputs bit-exact.
"""

import numpy as np
import pytest
import torch

import mla_decode_query_gb300 as mq
import oracle
from helpers import check_output, to_device, to_host_bits
from mla_decode_query_gb300 import inputs

pytestmark = pytest.mark.gpu

D = 576
M_MAX = 256
# chunk edges of the 32-, 64- and 128-token CTA tiles, ragged tails, 16-token MMA edges
M_POINTS = (33, 40, 47, 48, 63, 64, 65, 80, 100, 127, 128, 129, 191, 200, 255, 256)
PAIRS = [("bf16", "bf16"), ("bf16", "e4m3"), ("mxfp8", "bf16"), ("mxfp8", "e4m3")]


def _dev(d):
    return dict(q_nope=to_device(d["q_nope"]), q_pe=to_device(d["q_pe"]), weight=to_device(d["weight"]),
                weight_scale=None if d["weight_scale"] is None else to_device(d["weight_scale"]))


def _run(t, M, H, fmt, od, qs=None, out=None, stride=None, pdl=False, K=128, stream=None):
    stride = stride or D * H
    if out is None:
        out = torch.zeros((M * stride,), dtype=torch.int16 if od == "bf16" else torch.uint8, device="cuda")
    q_scale = None if qs is None else torch.tensor([qs], dtype=torch.float32, device="cuda")
    st = mq.mlaqp_run_strided(t["q_nope"], H * K, K, t["q_pe"], H * 64, 64, t["weight"], t["weight_scale"], out,
                              stride, q_scale, M, H, K, fmt, od, pdl=pdl, stream=stream)
    assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
    return out


def _rows(out, M, H, stride, od):
    bits = to_host_bits(out, np.uint16 if od == "bf16" else np.uint8)
    return np.stack([bits[m * stride: m * stride + H * D].reshape(H, D) for m in range(M)])


def _oracle(d, fmt, od, qs):
    return oracle.mla_query(d["q_nope"], d["q_pe"], d["weight"], d["weight_scale"], fmt, od, qs)


def test_domain_and_launch_shape(cuda_device):
    for fmt, od in PAIRS:
        for h in (8, 11, 16):
            assert mq.mlaqp_can_implement(h, M_MAX, weight_format=fmt, out_dtype=od) == 1, mq.mlaqp_last_error()
            assert mq.mlaqp_prewarm(h, M_MAX, fmt, od) == mq.MLAQP_OK, mq.mlaqp_last_error()
    assert mq.mlaqp_can_implement(16, M_MAX + 1) == 0
    # Above M = 32 the CTA-tile kernel in 32-token chunks (256 threads): up to
    # M = 64 always, beyond while its 8*H*chunks CTAs fit at four per SM;
    # otherwise the tcgen05 kernel, 4 CTAs per head and token chunk (32 tokens
    # up to M = 64, 64 up to 128, then 128), 512 threads from 64-token chunks.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for fmt, od in PAIRS:
        for h in (8, 11, 16):
            for m in (33, 40, 64, 65, 96, 97, 128, 129, 200, 256):
                st, grid, threads = mq.mlaqp_launch_shape(m, h, fmt, od)
                assert st == mq.MLAQP_OK
                chunks = -(-m // 32)
                if m <= 64 or 8 * h * chunks <= 4 * sms:
                    assert grid == 8 * h * chunks and threads == 256, (fmt, od, h, m)
                else:
                    tt = 32 if m <= 64 else (64 if m <= 128 else 128)
                    assert grid == 4 * h * -(-m // tt) and threads == (256 if tt == 32 else 512), (fmt, od, h, m)


@pytest.mark.parametrize("fmt,od", PAIRS)
def test_token_counts_h16(cuda_device, fmt, od):
    H = 16
    d = inputs.make_layer(inputs.layer_seed(30, H), H, fmt, m_max=M_MAX)
    qs = inputs.make_q_scale(30) if od == "e4m3" else None
    ref, acc = _oracle(d, fmt, od, qs)
    t = _dev(d)
    for M in M_POINTS:
        got = _rows(_run(t, M, H, fmt, od, qs, pdl=(M % 2 == 1)), M, H, D * H, od)
        check_output(got, ref[:M], acc[:M], od, f"{fmt}->{od} H{H} M{M}")


@pytest.mark.parametrize("fmt,od", PAIRS)
@pytest.mark.parametrize("H", [8, 11])
def test_token_counts_h8_h11(cuda_device, fmt, od, H):
    d = inputs.make_layer(inputs.layer_seed(31, H), H, fmt, m_max=M_MAX)
    qs = inputs.make_q_scale(31) if od == "e4m3" else None
    ref, acc = _oracle(d, fmt, od, qs)
    t = _dev(d)
    for M in (33, 64, 100, 129, 256):
        got = _rows(_run(t, M, H, fmt, od, qs), M, H, D * H, od)
        check_output(got, ref[:M], acc[:M], od, f"{fmt}->{od} H{H} M{M}")


@pytest.mark.parametrize("fmt,od", PAIRS)
def test_nope192(cuda_device, fmt, od):
    H, K = 16, 192
    d = inputs.make_layer(inputs.layer_seed(32, H), H, fmt, m_max=M_MAX, nope=K)
    qs = inputs.make_q_scale(32) if od == "e4m3" else None
    ref, acc = _oracle(d, fmt, od, qs)
    t = _dev(d)
    for M in (33, 64, 65, 150, 256):
        got = _rows(_run(t, M, H, fmt, od, qs, K=K), M, H, D * H, od)
        check_output(got, ref[:M], acc[:M], od, f"K192 {fmt}->{od} M{M}")


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
@pytest.mark.parametrize("K", [128, 192])
def test_small_integers_bit_exact(cuda_device, fmt, K):
    # Every partial sum is an integer of magnitude <= 2K: exact in FP32 in any
    # order, so the tensor-core result must equal the oracle bit for bit.
    for H, M in ((16, 256), (11, 97), (8, 33), (8, 100)):
        d = inputs.small_integer_layer(300 + M, H, M, fmt, nope=K)
        for od, qs in (("bf16", None), ("e4m3", np.float32(0.25))):
            got = _rows(_run(_dev(d), M, H, fmt, od, qs, K=K), M, H, D * H, od)
            ref, _ = _oracle(d, fmt, od, qs)
            np.testing.assert_array_equal(got, ref, err_msg=f"K{K} {fmt}->{od} H{H} M{M}")


def test_one_hot_rows_select_weight_rows(cuda_device):
    # Token m has q_nope = e_{k(m)}: out[m,h,:512] is exactly weight row k(m)
    # of head h (BF16 weights pass through unchanged), for every k.
    H, M = 16, 256
    rng = np.random.Generator(np.random.PCG64(33))
    d = inputs.make_layer(33, H, "bf16", m_max=M)
    k_of_m = rng.permutation(np.arange(M) % 128)
    q = np.zeros((M, H, 128), dtype=np.float32)
    q[np.arange(M), :, k_of_m] = 1.0
    qb = torch.from_numpy(q).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    dd = dict(d, q_nope=qb)
    got = _rows(_run(_dev(dd), M, H, "bf16", "bf16"), M, H, D * H, "bf16")
    expect = np.transpose(d["weight"][:, k_of_m, :], (1, 0, 2))
    np.testing.assert_array_equal(got[..., :512], expect)
    np.testing.assert_array_equal(got[..., 512:], d["q_pe"])


def test_pitched_workspace_canaries(cuda_device):
    for fmt, od in (("bf16", "bf16"), ("mxfp8", "e4m3")):
        H = 11
        stride = D * H + 64
        d = inputs.make_layer(inputs.layer_seed(34, H), H, fmt, m_max=M_MAX)
        qs = inputs.make_q_scale(34) if od == "e4m3" else None
        ref, acc = _oracle(d, fmt, od, qs)
        t = _dev(d)
        dt = torch.int16 if od == "bf16" else torch.uint8
        canary = 0x5A5A if od == "bf16" else 0xA5
        for M in (33, 130, 256):
            ws = torch.full((M_MAX * stride + 64,), canary, dtype=dt, device="cuda")
            _run(t, M, H, fmt, od, qs, out=ws, stride=stride)
            bits = to_host_bits(ws, np.uint16 if od == "bf16" else np.uint8)
            mask = np.zeros(bits.shape, dtype=bool)
            for m in range(M):
                mask[m * stride: m * stride + H * D] = True
            assert (bits[~mask] == canary).all(), f"{fmt} M{M}: bytes outside the rows changed"
            check_output(_rows(ws, M, H, stride, od), ref[:M], acc[:M], od, f"{fmt}->{od} M{M} pitched")


def test_graph_chain_mixed_token_counts(cuda_device):
    # A captured chain of PDL launches alternating decode (M <= 32) and
    # large-M calls on distinct layers; every output checked.
    H = 16
    Ms = (64, 8, 256, 33, 32, 129, 1, 100)
    layers = []
    for i, M in enumerate(Ms):
        fmt, od = PAIRS[i % 4]
        d = inputs.make_layer(inputs.layer_seed(35, i), H, fmt, m_max=M)
        qs = inputs.make_q_scale(35 + i) if od == "e4m3" else None
        layers.append((d, fmt, od, qs, M, _dev(d)))
    outs = [torch.zeros((M * D * H,), dtype=torch.int16 if od == "bf16" else torch.uint8, device="cuda")
            for (_, _, od, _, M, _) in layers]
    scales = [None if qs is None else torch.tensor([qs], dtype=torch.float32, device="cuda")
              for (_, _, _, qs, _, _) in layers]
    for i, (d, fmt, od, qs, M, t) in enumerate(layers):
        assert mq.mlaqp_prewarm(H, M, fmt, od) == mq.MLAQP_OK
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i, (d, fmt, od, qs, M, t) in enumerate(layers):
            st = mq.mlaqp_run_strided(t["q_nope"], H * 128, 128, t["q_pe"], H * 64, 64, t["weight"],
                                      t["weight_scale"], outs[i], D * H, scales[i], M, H, 128, fmt, od, pdl=True,
                                      stream=stream)
            assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
    for _ in range(3):
        for o in outs:
            o.zero_()
        graph.replay()
        torch.cuda.synchronize()
    for i, (d, fmt, od, qs, M, t) in enumerate(layers):
        ref, acc = _oracle(d, fmt, od, qs)
        check_output(_rows(outs[i], M, H, D * H, od), ref, acc, od, f"graph layer {i} {fmt}->{od} M{M}")


@pytest.mark.parametrize("H,M", [(8, 64), (8, 100), (16, 160)])
def test_bounded_wait_reports_timeout_and_frees_tmem(cuda_device, H, M):
    # Every CTA's weight wait runs out (2 ms): the kernel records the timeout,
    # writes nothing, and (H = 16, M = 160: the tcgen05 kernel) releases its
    # tensor memory; later runs (which allocate tensor memory again on the
    # same SMs) still work.  H = 8 runs the CTA-tile kernel in two and four
    # token chunks.
    st, _ = mq.mlaqp_device_status(reset=True)
    assert st == mq.MLAQP_OK
    for fmt in ("bf16", "mxfp8"):
        d = inputs.make_layer(36, H, fmt, m_max=M)
        t = _dev(d)
        out = torch.full((M * D * H,), 0x7777, dtype=torch.int16, device="cuda")
        st = mq.mlaqp_debug_run_bounded_wait(t["q_nope"], t["q_pe"], t["weight"], t["weight_scale"], out, D * H,
                                             None, M, H, fmt, "bf16", 2_000_000, 16)
        assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
        torch.cuda.synchronize()
        assert (out == 0x7777).all()
        st, word = mq.mlaqp_device_status(reset=True)
        assert st == mq.MLAQP_OK and word & mq.MLAQP_DEVSTATUS_WAIT_TIMEOUT
        ref, acc = _oracle(d, fmt, "bf16", None)
        for _ in range(3):
            got = _rows(_run(t, M, H, fmt, "bf16"), M, H, D * H, "bf16")
            check_output(got, ref, acc, "bf16", f"after timeout {fmt}")
        st, word = mq.mlaqp_device_status(reset=False)
        assert word == 0


@pytest.mark.parametrize("M", [96, 160])
@pytest.mark.parametrize("qs", [1e-3, 2.0 ** -110, 2.0 ** 110])
def test_e4m3_saturation_and_plain_division(cuda_device, qs, M):
    # Saturation to 448, and q_scale outside the table range (plain division),
    # in the chunked CTA-tile kernel (M = 96, three chunks) and the tcgen05
    # kernel (M = 160).
    H = 16
    d = inputs.make_layer(inputs.layer_seed(37, 0), H, "mxfp8", m_max=M)
    qs = np.float32(qs)
    got = _rows(_run(_dev(d), M, H, "mxfp8", "e4m3", qs), M, H, D * H, "e4m3")
    ref, acc = _oracle(d, "mxfp8", "e4m3", qs)
    check_output(got, ref, acc, "e4m3", f"qs={qs}")


@pytest.mark.parametrize("K", [128, 192])
def test_strided_and_head_major_inputs(cuda_device, K):
    # The kernels above 32 tokens (H = 16: the chunked CTA-tile kernel at
    # M = 33 and 100, the tcgen05 kernel at 256) read q_nope / q_pe through
    # token and head strides: views into the upstream [M, H, K+64]
    # projection, and a head-major [H, M, K] q_nope with a head-major
    # [H, M, 64] q_pe.
    H = 16
    for fmt, od in (("bf16", "bf16"), ("mxfp8", "e4m3")):
        d = inputs.make_layer(inputs.layer_seed(38, K), H, fmt, m_max=M_MAX, nope=K)
        qs = inputs.make_q_scale(38) if od == "e4m3" else None
        ref, acc = _oracle(d, fmt, od, qs)
        w = to_device(d["weight"])
        sc = None if d["weight_scale"] is None else to_device(d["weight_scale"])
        q_scale = None if qs is None else torch.tensor([qs], dtype=torch.float32, device="cuda")
        up = np.concatenate([d["q_nope"], d["q_pe"]], axis=-1)  # [M, H, K+64]
        upd = to_device(up)
        qn_hm = to_device(np.ascontiguousarray(np.transpose(d["q_nope"], (1, 0, 2))))
        qp_hm = to_device(np.ascontiguousarray(np.transpose(d["q_pe"], (1, 0, 2))))
        for M in (33, 100, 256):
            for name, args in (
                ("upstream view", (upd, H * (K + 64), K + 64, upd[..., K:], H * (K + 64), K + 64)),
                ("head-major", (qn_hm, K, M_MAX * K, qp_hm, 64, M_MAX * 64)),
            ):
                out = torch.zeros((M * D * H,), dtype=torch.int16 if od == "bf16" else torch.uint8, device="cuda")
                st = mq.mlaqp_run_strided(args[0], args[1], args[2], args[3], args[4], args[5], w, sc, out, D * H,
                                          q_scale, M, H, K, fmt, od, pdl=(M == 100))
                assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
                torch.cuda.synchronize()
                check_output(_rows(out, M, H, D * H, od), ref[:M], acc[:M], od, f"K{K} {fmt}->{od} M{M} {name}")
