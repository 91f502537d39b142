"""GPU parity of every kernel form the library can run a decode call on,
forced through mlaqp_debug_run_arm, against the CPU oracle: the warp-tile
kernel with the tensor-core (mma.sync) and the CUDA-core (FP32 FMA +
warp-shuffle) contraction, the CTA-tile mma.sync kernel and the tcgen05
kernel.  Same tolerances as every parity test (see helpers); exact-arithmetic
inputs bit-exact; the forms agree with each other bit for bit on q_pe and
within one E4M3 ulp on E4M3 codes.  Also: a PDL graph chain that alternates
the forms, and the warp-tile kernel's launch shape (one CTA per SM).
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
PAIRS = [("bf16", "bf16"), ("bf16", "e4m3"), ("mxfp8", "bf16"), ("mxfp8", "e4m3")]


def _dev(d):
    return dict(q_nope=to_device(d["q_nope"]), q_pe=to_device(d["q_pe"]), weight=to_device(d["weight"]),
                weight_scale=None if d["weight_scale"] is None else to_device(d["weight_scale"]))


def _run_arm(t, M, H, K, fmt, od, arm, q_scale=None, stride=None, out=None, pdl=False, stream=None):
    stride = stride or D * H
    if out is None:
        out = torch.zeros((M * stride,), dtype=torch.int16 if od == "bf16" else torch.uint8, device="cuda")
    qs = None if q_scale is None else torch.tensor([q_scale], dtype=torch.float32, device="cuda")
    st = mq.mlaqp_debug_run_arm(t["q_nope"], H * K, K, t["q_pe"], H * 64, 64, t["weight"], t["weight_scale"], out,
                                stride, qs, M, H, K, fmt, od, pdl=pdl, arm=arm, stream=stream)
    assert st == mq.MLAQP_OK, (arm, M, H, K, mq.mlaqp_last_error())
    return out, qs


def _rows(out, M, H, stride, od):
    bits = to_host_bits(out, np.uint16 if od == "bf16" else np.uint8)
    return np.stack([bits[m * stride: m * stride + H * D].reshape(H, D) for m in range(M)])


def _arms_for(M, K):
    arms = ["warp_mma", "cta_mma", "tcgen05"]
    if M <= 8 and K == 128:
        arms.append("warp_fma")
    return arms


@pytest.mark.parametrize("fmt,od", PAIRS)
@pytest.mark.parametrize("H", [8, 11, 16])
@pytest.mark.parametrize("K", [128, 192])
def test_every_arm_matches_the_oracle(cuda_device, fmt, od, H, K):
    d = inputs.make_layer(inputs.layer_seed(21, H), H, fmt, nope=K)
    qs = inputs.make_q_scale(5) if od == "e4m3" else None
    t = _dev(d)
    for M in (1, 2, 5, 8, 9, 16, 17, 31, 32):
        ref, acc = oracle.mla_query(d["q_nope"][:M], d["q_pe"][:M], d["weight"], d["weight_scale"], fmt, od, qs)
        outs = {}
        for arm in _arms_for(M, K):
            out, _ = _run_arm(t, M, H, K, fmt, od, arm, qs)
            torch.cuda.synchronize()
            got = _rows(out, M, H, D * H, od)
            check_output(got, ref, acc, od, f"{arm} {fmt}->{od} H{H} K{K} M{M}")
            outs[arm] = got
        base = outs["warp_mma"]
        for arm, got in outs.items():
            np.testing.assert_array_equal(got[..., 512:], base[..., 512:], err_msg=f"{arm}: q_pe region")


@pytest.mark.parametrize("fmt,od", PAIRS)
def test_every_arm_small_integers_bit_exact(cuda_device, fmt, od):
    # Every partial sum is an integer small enough to be exact in binary32,
    # so every summation order gives the oracle's value exactly.
    H = 11
    for M in (1, 4, 8, 13, 32):
        d = inputs.small_integer_layer(31 + M, H, M, fmt)
        qs = np.float32(0.25) if od == "e4m3" else None
        ref, _ = oracle.mla_query(d["q_nope"], d["q_pe"], d["weight"], d["weight_scale"], fmt, od, qs)
        t = _dev(d)
        for arm in _arms_for(M, 128):
            out, _ = _run_arm(t, M, H, 128, fmt, od, arm, qs)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(_rows(out, M, H, D * H, od), ref, err_msg=f"{arm} {fmt}->{od} M{M}")


@pytest.mark.parametrize("arm", ["warp_mma", "warp_fma", "cta_mma", "tcgen05"])
def test_every_arm_pitched_workspace_canaries(cuda_device, arm):
    # Rows >= M and the pitch padding keep their bytes.
    H, fmt, od = 16, "mxfp8", "e4m3"
    M = 5
    stride = D * H + 64
    d = inputs.make_layer(inputs.layer_seed(22, 0), H, fmt)
    qs = inputs.make_q_scale(6)
    out = torch.full((32 * stride,), 0x5A, dtype=torch.uint8, device="cuda")
    _run_arm(_dev(d), M, H, 128, fmt, od, arm, qs, stride=stride, out=out)
    torch.cuda.synchronize()
    bits = to_host_bits(out, np.uint8)
    ref, acc = oracle.mla_query(d["q_nope"][:M], d["q_pe"][:M], d["weight"], d["weight_scale"], fmt, od, qs)
    check_output(_rows(out, M, H, stride, od), ref, acc, od, arm)
    for m in range(32):
        row = bits[m * stride:(m + 1) * stride]
        if m < M:
            assert (row[D * H:] == 0x5A).all(), f"{arm}: padding of row {m} written"
        else:
            assert (row == 0x5A).all(), f"{arm}: row {m} >= M written"


def test_arms_reject_calls_they_do_not_cover(cuda_device):
    d = inputs.make_layer(1, 8, "bf16", m_max=136, nope=192)
    t = _dev(d)
    out = torch.zeros((136 * D * 8,), dtype=torch.int16, device="cuda")
    for M, K, arm in ((9, 128, "warp_fma"), (4, 192, "warp_fma"), (33, 192, "warp_mma"), (257, 192, "cta_mma")):
        st = mq.mlaqp_debug_run_arm(t["q_nope"], 8 * K, K, t["q_pe"], 8 * 64, 64, t["weight"], None, out, D * 8,
                                    None, M, 8, K, "bf16", "bf16", arm=arm)
        assert st == mq.MLAQP_ERR_UNSUPPORTED, (M, K, arm)


def _crossover(fmt, od, h):
    # the library's measured choice: warp-tile kernel from this token count on
    if h > 8:
        return 17
    return {("bf16", "bf16"): 15, ("bf16", "e4m3"): 13, ("mxfp8", "bf16"): 13, ("mxfp8", "e4m3"): 16}[(fmt, od)]


def test_launch_shape_follows_the_policy(cuda_device):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for fmt, od in PAIRS:
        for h in (8, 11, 16):
            g = min(max(sms, 8 * h), 32 * h)  # warp-tile kernel: one CTA per SM, 8..32 per head
            tpc = -(-32 // (g // h))          # tiles of the head with the fewest CTAs
            for m in (1, 8, 9, 12, 13, 14, 15, 16, 17, 32):
                st, grid, threads = mq.mlaqp_launch_shape(m, h, fmt, od)
                assert st == mq.MLAQP_OK
                # two chunks of the CTA-tile kernel (8 tokens up to M = 16, 16 tokens
                # for MXFP8 weights above) where their 16*H CTAs fit one per SM
                if m > 8 and 16 * h <= sms and (m <= 16 or fmt == "mxfp8"):
                    assert grid == 16 * h and threads == (128 if m <= 16 else 256), (fmt, od, h, m)
                elif m >= _crossover(fmt, od, h):
                    assert grid == g and threads == 32 * tpc * (1 if m <= 8 else 2), (fmt, od, h, m)
                else:
                    assert grid == 8 * h and threads == (128 if m <= 8 else 256), (fmt, od, h, m)


@pytest.mark.parametrize("fmt,od", [("bf16", "bf16"), ("mxfp8", "e4m3")])
def test_pdl_chain_alternating_arms(cuda_device, fmt, od):
    # A CUDA graph of programmatic-dependent launches that alternates the
    # kernel forms (trigger points and TMEM use differ between them); every
    # layer has its own inputs and output, and every output must be right.
    H, K, L = 16, 128, 12
    arms = ["warp_mma", "warp_fma", "cta_mma", "tcgen05"]
    Ms = [1, 4, 8, 3]
    qs_val = inputs.make_q_scale(7) if od == "e4m3" else None
    layers = [inputs.make_layer(inputs.layer_seed(23, l), H, fmt) for l in range(L)]
    dev = [_dev(d) for d in layers]
    outs = [torch.zeros((32 * D * H,), dtype=torch.int16 if od == "bf16" else torch.uint8, device="cuda")
            for _ in range(L)]
    qs = None if qs_val is None else torch.tensor([qs_val], dtype=torch.float32, device="cuda")

    def launch_all(stream=None):
        for l in range(L):
            arm, M = arms[l % 4], Ms[l % 4]
            st = mq.mlaqp_debug_run_arm(dev[l]["q_nope"], H * K, K, dev[l]["q_pe"], H * 64, 64, dev[l]["weight"],
                                        dev[l]["weight_scale"], outs[l], D * H, qs, M, H, K, fmt, od, pdl=True,
                                        arm=arm, stream=stream)
            assert st == mq.MLAQP_OK, mq.mlaqp_last_error()

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        launch_all(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch_all()
    for o in outs:
        o.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for l in range(L):
        M = Ms[l % 4]
        d = layers[l]
        ref, acc = oracle.mla_query(d["q_nope"][:M], d["q_pe"][:M], d["weight"], d["weight_scale"], fmt, od, qs_val)
        check_output(_rows(outs[l], M, H, D * H, od), ref, acc, od, f"layer {l} ({arms[l % 4]})")


@pytest.mark.parametrize("fmt,od", [("bf16", "bf16"), ("mxfp8", "e4m3")])
def test_prefetch_weights_then_run(cuda_device, fmt, od):
    # The L2 warm-up on a parallel graph branch, then the layer call: same
    # results, in a graph replayed twice and eagerly.
    H, M = 16, 5
    d = inputs.make_layer(inputs.layer_seed(24, 0), H, fmt)
    t = _dev(d)
    qs_val = inputs.make_q_scale(8) if od == "e4m3" else None
    qs = None if qs_val is None else torch.tensor([qs_val], dtype=torch.float32, device="cuda")
    out = torch.zeros((M * D * H,), dtype=torch.int16 if od == "bf16" else torch.uint8, device="cuda")
    side = torch.cuda.Stream()

    def step():
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        with torch.cuda.stream(side):
            for pdl in (False, True):
                assert mq.mlaqp_prefetch_weights(t["weight"], t["weight_scale"], H, 128, fmt, pdl=pdl,
                                                 stream=side) == mq.MLAQP_OK, mq.mlaqp_last_error()
        assert mq.mlaqp_run_pdl(t["q_nope"], t["q_pe"], t["weight"], t["weight_scale"], out, D * H, qs, M, H,
                                fmt, od) == mq.MLAQP_OK, mq.mlaqp_last_error()
        main.wait_stream(side)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    ref, acc = oracle.mla_query(d["q_nope"][:M], d["q_pe"][:M], d["weight"], d["weight_scale"], fmt, od, qs_val)
    check_output(_rows(out, M, H, D * H, od), ref, acc, od, f"prefetch {fmt}->{od}")


@pytest.mark.parametrize("with_prefetch", [False, True])
def test_dependent_chain_reads_previous_output(cuda_device, with_prefetch):
    # Layer l+1's q_nope / q_pe are views of layer l's output (columns 0..127
    # and 512..575 of its [M,H,576] rows), so every op depends on the one
    # before it.  All launches are programmatic-dependent; the op triggers
    # its successor at entry, and a weight prefetch launched in between must
    # not break the chain (it exits only after its predecessor).  Small
    # integers keep every layer exact: |q| <= 2 and weights in {-1, 0, 1}
    # give |out_0| <= 256, |out_1| <= 2^15 and partial sums of layer 2 below
    # 2^22, so the oracle's own chain must match the GPU's bit for bit.
    H, M, L = 16, 8, 3
    row = 576 * H
    fmts = ["bf16", "mxfp8", "bf16"]
    layers = [inputs.small_integer_layer(26 + l, H, M, fmts[l]) for l in range(L)]
    dev = [_dev(d) for d in layers]
    outs = [torch.zeros((M * row,), dtype=torch.int16, device="cuda") for _ in range(L)]

    def launch_all(stream=None):
        for l in range(L):
            if l == 0:
                qn, qn_ts, qn_hs, qp, qp_ts, qp_hs = dev[0]["q_nope"], H * 128, 128, dev[0]["q_pe"], H * 64, 64
            else:
                qn, qn_ts, qn_hs = outs[l - 1], row, 576
                qp, qp_ts, qp_hs = outs[l - 1].data_ptr() + 2 * 512, row, 576
            if with_prefetch:
                assert mq.mlaqp_prefetch_weights(dev[l]["weight"], dev[l]["weight_scale"], H, 128, fmts[l], pdl=True,
                                                 stream=stream) == mq.MLAQP_OK, mq.mlaqp_last_error()
            st = mq.mlaqp_run_strided(qn, qn_ts, qn_hs, qp, qp_ts, qp_hs, dev[l]["weight"], dev[l]["weight_scale"],
                                      outs[l], row, None, M, H, 128, fmts[l], "bf16", pdl=1, stream=stream)
            assert st == mq.MLAQP_OK, mq.mlaqp_last_error()

    # The oracle's chain, from the original inputs only.
    refs = []
    qn, qp = layers[0]["q_nope"], layers[0]["q_pe"]
    for l in range(L):
        ref, acc = oracle.mla_query(qn, qp, layers[l]["weight"], layers[l]["weight_scale"], fmts[l], "bf16")
        assert np.all(acc == np.round(acc)) and np.abs(acc).max() < 2 ** 22
        refs.append(ref)
        qn, qp = ref[..., :128].copy(), ref[..., 512:].copy()

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        launch_all(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch_all()
    for rep in range(3):
        for o in outs:
            o.fill_(0x7FC0)  # BF16 NaN: a read of a not-yet-written output would show
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for l in range(L):
            np.testing.assert_array_equal(_rows(outs[l], M, H, row, "bf16"), refs[l], err_msg=f"replay {rep} layer {l}")


def test_plan_matches_launch_shape_on_this_device(cuda_device):
    # The host-side plan (tests/test_plan_host.py pins its rules) at this
    # device's SM count is the launch the library reports and makes.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for fmt, od in PAIRS:
        for h in (8, 11, 16):
            for m in (1, 8, 9, 16, 17, 24, 32, 33, 64, 65, 96, 128, 129, 160, 192, 224, 256):
                st, grid, threads = mq.mlaqp_launch_shape(m, h, fmt, od)
                assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
                st, p = mq.mlaqp_debug_plan(m, h, fmt, od, sm_count=sms)
                assert st == mq.MLAQP_OK
                assert (p["grid_ctas"], p["threads_per_cta"]) == (grid, threads), (fmt, od, h, m, p)
