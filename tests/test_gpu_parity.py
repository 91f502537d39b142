"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Tolerances (see helpers): q_pe columns bit-exact; BF16 projection within
1e-2*|ref| + 1e-3 of the float64 projection; E4M3 projection within one
E4M3 ulp of the oracle's code; exact-arithmetic cases bit-exact.
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


def _dev_layer(d, dev):
    return dict(q_nope=to_device(d["q_nope"], dev), q_pe=to_device(d["q_pe"], dev),
                weight=to_device(d["weight"], dev),
                weight_scale=None if d["weight_scale"] is None else to_device(d["weight_scale"], dev))


def _run(t, M, H, fmt, od, q_scale=None, out=None, stride=None, pdl=False, dev="cuda", arm="auto"):
    stride = stride or D * H
    if out is None:
        out = torch.zeros((M * stride,), dtype=torch.int16 if od == "bf16" else torch.uint8, device=dev)
    qs = None if q_scale is None else torch.tensor([q_scale], dtype=torch.float32, device=dev)
    if arm != "auto":
        st = mq.mlaqp_debug_run_arm(t["q_nope"], H * 128, 128, t["q_pe"], H * 64, 64, t["weight"], t["weight_scale"],
                                    out, stride, qs, M, H, 128, fmt, od, pdl=pdl, arm=arm)
        assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
        torch.cuda.synchronize()
        return out
    fn = mq.mlaqp_run_pdl if pdl else mq.mlaqp_run
    st = fn(t["q_nope"], t["q_pe"], t["weight"], t["weight_scale"], out, stride, qs, M, H, fmt, od)
    assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
    torch.cuda.synchronize()
    return out


def _rows(out, M, H, stride, od):
    bits = to_host_bits(out, np.uint16 if od == "bf16" else np.uint8)
    return np.stack([bits[m * stride: m * stride + H * D].reshape(H, D) for m in range(M)])


def _check(d, M, H, fmt, od, q_scale=None, pdl=False, dev="cuda", where=""):
    t = _dev_layer(d, dev)
    out = _run(t, M, H, fmt, od, q_scale, pdl=pdl, dev=dev)
    got = _rows(out, M, H, D * H, od)
    ref, acc = oracle.mla_query(d["q_nope"][:M], d["q_pe"][:M], d["weight"], d["weight_scale"], fmt, od,
                                q_scale)
    return check_output(got, ref, acc, od, where)


def test_can_implement_and_prewarm(cuda_device):
    for fmt in ("bf16", "mxfp8"):
        for od in ("bf16", "e4m3"):
            for h in (8, 11, 16):
                assert mq.mlaqp_can_implement(h, 32, weight_format=fmt, out_dtype=od) == 1, mq.mlaqp_last_error()
                assert mq.mlaqp_prewarm(h, 32, fmt, od) == mq.MLAQP_OK, mq.mlaqp_last_error()
    assert mq.mlaqp_can_implement(16, 257) == 0


def test_single_layer_bf16_h16_m1(cuda_device):
    # BF16 weights, H=16, M=1, one layer, seed 0, contiguous [1,16,576] output.
    d = inputs.make_layer(inputs.layer_seed(0, 0), 16, "bf16", m_max=1)
    _check(d, 1, 16, "bf16", "bf16", where="bf16 H16 M1")


@pytest.mark.parametrize("fmt,od", [("bf16", "bf16"), ("bf16", "e4m3"), ("mxfp8", "bf16"), ("mxfp8", "e4m3")])
@pytest.mark.parametrize("H", [8, 11, 16])
def test_every_token_count(cuda_device, fmt, od, H):
    d = inputs.make_layer(inputs.layer_seed(7, H), H, fmt)
    qs = inputs.make_q_scale(3) if od == "e4m3" else None
    for M in range(1, 33):
        _check(d, M, H, fmt, od, qs, where=f"{fmt}->{od} H{H} M{M}")


@pytest.mark.parametrize("fmt,od", [("bf16", "bf16"), ("bf16", "e4m3"), ("mxfp8", "bf16"), ("mxfp8", "e4m3")])
def test_small_integers_bit_exact(cuda_device, fmt, od):
    # Every partial sum is an integer <= 256 in magnitude: any FP32 summation
    # order is exact, so the GPU must reproduce the oracle bit for bit.
    for H, M in ((16, 32), (11, 9), (8, 1)):
        d = inputs.small_integer_layer(100 + M, H, M, fmt)
        qs = np.float32(0.25) if od == "e4m3" else None
        t = _dev_layer(d, "cuda")
        got = _rows(_run(t, M, H, fmt, od, qs), M, H, D * H, od)
        ref, _ = oracle.mla_query(d["q_nope"], d["q_pe"], d["weight"], d["weight_scale"], fmt, od, qs)
        np.testing.assert_array_equal(got, ref, err_msg=f"{fmt}->{od} H{H} M{M}")


def test_mxfp8_dequant_every_code_bit_exact(cuda_device):
    # One-hot q_nope picks a single weight row per token, so out[m,h,:512] is
    # bf16(e4m3(code) * 2^(scale-127)) exactly: every finite E4M3 code under
    # scale bytes 90..160 must come out bit-exact.
    H, M = 16, 32
    rng = np.random.Generator(np.random.PCG64(5))
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]
    w = rng.choice(codes, size=(H, 128, 512)).astype(np.uint8)
    w[:, :, :254] = codes[None, None, :]  # every finite code in every row
    s = rng.integers(90, 161, size=(H, 128, 16)).astype(np.uint8)
    k_of_m = np.arange(M) * 4 + 1
    q = np.zeros((M, H, 128), dtype=np.float32)
    q[np.arange(M), :, k_of_m] = 1.0
    qb = torch.from_numpy(q).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    pe = inputs.make_layer(1, H, "bf16", m_max=M)["q_pe"]
    d = {"q_nope": qb, "q_pe": pe, "weight": w, "weight_scale": s}
    got = _rows(_run(_dev_layer(d, "cuda"), M, H, "mxfp8", "bf16"), M, H, D * H, "bf16")
    ref, _ = oracle.mla_query(qb, pe, w, s, "mxfp8", "bf16")
    np.testing.assert_array_equal(got, ref)


def test_pitched_workspace_canaries(cuda_device):
    # Rows >= M and the padding between 576*H and the row stride keep their
    # bytes; rows < M match the oracle.
    for fmt, od in (("bf16", "bf16"), ("mxfp8", "e4m3")):
        for H in (8, 11, 16):
            stride = D * H + 64
            d = inputs.make_layer(inputs.layer_seed(4, H), H, fmt)
            qs = inputs.make_q_scale(4) if od == "e4m3" else None
            t = _dev_layer(d, "cuda")
            for M in (1, 7, 17, 32):
                dt = torch.int16 if od == "bf16" else torch.uint8
                canary = 0x5A5A if od == "bf16" else 0xA5
                ws = torch.full((32 * stride + 64,), canary, dtype=dt, device="cuda")
                _run(t, M, H, fmt, od, qs, out=ws, stride=stride)
                bits = to_host_bits(ws, np.uint16 if od == "bf16" else np.uint8)
                ref, acc = oracle.mla_query(d["q_nope"][:M], d["q_pe"][:M], d["weight"], d["weight_scale"],
                                            fmt, od, qs)
                mask = np.zeros(bits.shape, dtype=bool)
                for m in range(M):
                    mask[m * stride: m * stride + H * D] = True
                assert (bits[~mask] == canary).all(), f"{fmt} H{H} M{M}: bytes outside the rows changed"
                check_output(_rows(ws, M, H, stride, od), ref, acc, od, f"{fmt}->{od} H{H} M{M} pitched")


def test_pdl_launch_matches(cuda_device):
    for fmt, od in (("bf16", "bf16"), ("mxfp8", "e4m3")):
        d = inputs.make_layer(inputs.layer_seed(5, 0), 16, fmt)
        qs = inputs.make_q_scale(5) if od == "e4m3" else None
        for M in (1, 13, 32):
            _check(d, M, 16, fmt, od, qs, pdl=True, where=f"pdl {fmt} M{M}")


def test_e4m3_saturation(cuda_device):
    d = inputs.make_layer(inputs.layer_seed(6, 0), 16, "mxfp8")
    for qs in (np.float32(1e-3), np.float32(0.01)):
        t = _dev_layer(d, "cuda")
        got = _rows(_run(t, 32, 16, "mxfp8", "e4m3", qs), 32, 16, D * 16, "e4m3")
        ref, acc = oracle.mla_query(d["q_nope"], d["q_pe"], d["weight"], d["weight_scale"], "mxfp8", "e4m3", qs)
        check_output(got, ref, acc, "e4m3", f"saturation qs={qs}")
        assert ((got[..., :512] & 0x7F) == 0x7E).sum() > 100


def test_zero_tokens_writes_nothing(cuda_device):
    d = inputs.make_layer(1, 16, "bf16", m_max=1)
    t = _dev_layer(d, "cuda")
    out = torch.full((D * 16,), 0x1234, dtype=torch.int16, device="cuda")
    assert mq.mlaqp_run(t["q_nope"], t["q_pe"], t["weight"], None, out, D * 16, None, 0, 16, "bf16",
                        "bf16") == mq.MLAQP_OK
    torch.cuda.synchronize()
    assert (out == 0x1234).all()


def test_bounded_wait_reports_timeout_and_writes_nothing(cuda_device):
    # The copy barrier is told to expect 16 bytes more than the copies
    # deliver, so every CTA's bounded wait runs out (2 ms): the kernel must
    # record the timeout, write nothing, and leave the context usable.
    st, _ = mq.mlaqp_device_status(reset=True)
    assert st == mq.MLAQP_OK
    for fmt in ("bf16", "mxfp8"):
        d = inputs.make_layer(2, 8, fmt, m_max=4)
        t = _dev_layer(d, "cuda")
        out = torch.full((4 * D * 8,), 0x7777, dtype=torch.int16, device="cuda")
        st = mq.mlaqp_debug_run_bounded_wait(t["q_nope"], t["q_pe"], t["weight"], t["weight_scale"], out, D * 8,
                                             None, 4, 8, fmt, "bf16", 2_000_000, 16)
        assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
        torch.cuda.synchronize()
        assert (out == 0x7777).all()
        st, word = mq.mlaqp_device_status(reset=True)
        assert st == mq.MLAQP_OK and word & mq.MLAQP_DEVSTATUS_WAIT_TIMEOUT
        _check(d, 4, 8, fmt, "bf16", where="after timeout")  # context still works
        st, word = mq.mlaqp_device_status(reset=False)
        assert word == 0


@pytest.mark.parametrize("M,arm", [(8, "auto"), (32, "auto"), (64, "auto"), (8, "cta_mma"), (32, "cta_mma"),
                                   (4, "warp_fma"), (64, "tcgen05")])
@pytest.mark.parametrize("qs", [0.01, 0.0371, 0.1, 3.0, 1e-20, 1e20, 2.0 ** -110, 2.0 ** 110,
                                0.012109374627470970, 0.02734375])
def test_e4m3_division_every_bf16_value(cuda_device, qs, M, arm):
    # The q_pe columns of an E4M3 output are e4m3_satfinite(q_pe / q_scale):
    # feed every non-NaN BF16 bit pattern through them and require the codes
    # bit for bit.  The scales cover every exact conversion form: the
    # warp-tile kernels' one-multiply form (M = 8, 32, 4: allowed by the
    # per-CTA check for most scales) and their table fallback (the last two
    # scales, for which the check refuses: one multiply by RN(1/q_scale)
    # would get 32 and 60 BF16 values' codes wrong); the CTA-tile kernel's
    # table (M = 8) and checked-multiply (M = 32) forms; its 32-token chunked
    # form, which builds the table before its weight wait (M = 64); the
    # tcgen05 kernel (M = 64, forced); results that overflow or underflow
    # binary32; and q_scale outside 2^-100..2^100 (plain division).
    H = 16
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # drop inf / NaN patterns
    per_call = M * H * 64
    qs = np.float32(qs)
    d = inputs.make_layer(3, H, "bf16", m_max=M)
    for start in range(0, bits.size, per_call):
        chunk = bits[start:start + per_call]
        pe = np.zeros(per_call, dtype=np.uint16)
        pe[:chunk.size] = chunk
        pe = pe.reshape(M, H, 64)
        dd = dict(d, q_pe=pe)
        got = _rows(_run(_dev_layer(dd, "cuda"), M, H, "bf16", "e4m3", qs, arm=arm), M, H, D * H, "e4m3")
        with np.errstate(all="ignore"):
            ref = oracle.f32_to_e4m3_satfinite(oracle.bf16_to_f32(pe) / qs)
        np.testing.assert_array_equal(got[..., 512:], ref, err_msg=f"q_scale={qs} chunk {start}")
