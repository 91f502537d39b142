"""GPU parity of the V up-projection (mlaqp_v_up_run) against the CPU oracle.

Tolerance as for the query projection's BF16 region (helpers): within
1e-2*|ref| + 1e-3 of the float64 sum; exact-arithmetic inputs bit-exact.
Tokens are independent rows, so one oracle evaluation at M = 32 serves every
smaller M of the same layer.
"""

import numpy as np
import pytest
import torch

import mla_decode_query_gb300 as mq
import oracle
from helpers import check_bf16_region, to_device, to_host_bits
from mla_decode_query_gb300 import inputs

pytestmark = pytest.mark.gpu

V = 128
C = 512


def _dev(d):
    return dict(x=to_device(d["x"]), weight=to_device(d["weight"]),
                weight_scale=None if d["weight_scale"] is None else to_device(d["weight_scale"]))


def _run(t, M, H, fmt, x=None, x_ts=None, x_hs=C, out=None, stride=None, pdl=False, stream=None):
    stride = stride or V * H
    x = t["x"] if x is None else x
    x_ts = H * C if x_ts is None else x_ts
    if out is None:
        out = torch.zeros((M * stride,), dtype=torch.int16, device="cuda")
    st = mq.mlaqp_v_up_run(x, x_ts, x_hs, t["weight"], t["weight_scale"], out, stride, M, H, fmt, pdl=pdl,
                           stream=stream)
    assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
    return out


def _rows(out, M, H, stride):
    bits = to_host_bits(out, np.uint16)
    return np.stack([bits[m * stride: m * stride + H * V].reshape(H, V) for m in range(M)])


def _oracle(d, fmt):
    return oracle.mla_v_up(d["x"], d["weight"], d["weight_scale"], fmt)


def test_domain_and_prewarm(cuda_device):
    for fmt in ("bf16", "mxfp8"):
        for h in (8, 11, 16):
            assert mq.mlaqp_v_up_can_implement(h, 32, fmt) == 1, mq.mlaqp_last_error()
            assert mq.mlaqp_v_up_prewarm(h, 32, fmt) == mq.MLAQP_OK, mq.mlaqp_last_error()
    assert mq.mlaqp_v_up_can_implement(16, 256) == 1
    assert mq.mlaqp_v_up_can_implement(16, 257) == 0


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
@pytest.mark.parametrize("H", [8, 11, 16])
def test_every_token_count(cuda_device, fmt, H):
    d = inputs.make_v_layer(inputs.layer_seed(50, H), H, fmt)
    _, acc = _oracle(d, fmt)
    t = _dev(d)
    for M in range(1, 33):
        got = _rows(_run(t, M, H, fmt, pdl=(M % 3 == 0)), M, H, V * H)
        check_bf16_region(got, acc[:M], f"v_up {fmt} H{H} M{M}")


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
def test_small_integers_bit_exact(cuda_device, fmt):
    # Every partial sum is an integer of magnitude <= 1024: exact in FP32 in
    # any order, so the BF16 result must equal the oracle's bit for bit.
    for H, M in ((16, 32), (11, 9), (8, 1)):
        d = inputs.small_integer_v_layer(500 + M, H, M, fmt)
        got = _rows(_run(_dev(d), M, H, fmt), M, H, V * H)
        ref, _ = _oracle(d, fmt)
        np.testing.assert_array_equal(got, ref, err_msg=f"{fmt} H{H} M{M}")


def test_one_hot_rows_select_weight_rows(cuda_device):
    # x[m,h,:] = e_{c(m)}: out[m,h,:] is exactly row c(m) of W_UV[h] (BF16
    # weights pass unchanged; MXFP8 rows are e4m3 * 2^(s-127), exact in BF16
    # for these scale bytes), for every contraction index c.
    H, M = 16, 32
    rng = np.random.Generator(np.random.PCG64(51))
    for fmt in ("bf16", "mxfp8"):
        d = inputs.make_v_layer(51, H, fmt, m_max=M)
        t = _dev(d)
        perm = rng.permutation(C)
        for rep in range(C // M):
            c_of_m = perm[rep * M:(rep + 1) * M]
            xs = np.zeros((M, H, C), dtype=np.float32)
            xs[np.arange(M), :, c_of_m] = 1.0
            xb = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            got = _rows(_run(t, M, H, fmt, x=to_device(xb)), M, H, V * H)
            ref, _ = oracle.mla_v_up(xb, d["weight"], d["weight_scale"], fmt)
            np.testing.assert_array_equal(got, ref, err_msg=f"{fmt} rep {rep}")
            if fmt == "bf16":  # as values: a -0.0 weight sums with the +0 products to +0
                np.testing.assert_array_equal(oracle.bf16_to_f64(got),
                                              oracle.bf16_to_f64(np.transpose(d["weight"][:, c_of_m, :], (1, 0, 2))))


def test_pitched_workspace_canaries(cuda_device):
    for fmt in ("bf16", "mxfp8"):
        H = 11
        stride = V * H + 24
        d = inputs.make_v_layer(inputs.layer_seed(52, H), H, fmt)
        _, acc = _oracle(d, fmt)
        t = _dev(d)
        for M in (1, 7, 17, 32):
            ws = torch.full((32 * stride + 64,), 0x5A5A, dtype=torch.int16, device="cuda")
            _run(t, M, H, fmt, out=ws, stride=stride)
            bits = to_host_bits(ws, np.uint16)
            mask = np.zeros(bits.shape, dtype=bool)
            for m in range(M):
                mask[m * stride: m * stride + H * V] = True
            assert (bits[~mask] == 0x5A5A).all(), f"{fmt} M{M}: bytes outside the rows changed"
            check_bf16_region(_rows(ws, M, H, stride), acc[:M], f"{fmt} M{M} pitched")


def test_strided_inputs(cuda_device):
    # x head-major [H, M, 512], and x as a view with a 576-wide padded row.
    H, M = 16, 24
    for fmt in ("bf16", "mxfp8"):
        d = inputs.make_v_layer(inputs.layer_seed(53, 0), H, fmt, m_max=M)
        _, acc = _oracle(d, fmt)
        t = _dev(d)
        hm = to_device(np.ascontiguousarray(np.transpose(d["x"], (1, 0, 2))))
        got = _rows(_run(t, M, H, fmt, x=hm, x_ts=C, x_hs=M * C), M, H, V * H)
        check_bf16_region(got, acc, f"{fmt} head-major")
        padded = np.zeros((M, H, 576), dtype=np.uint16)
        padded[..., :C] = d["x"]
        pv = to_device(padded)
        got = _rows(_run(t, M, H, fmt, x=pv, x_ts=H * 576, x_hs=576, pdl=True), M, H, V * H)
        check_bf16_region(got, acc, f"{fmt} padded view")


@pytest.mark.parametrize("pdl", [1, 2])
def test_graph_chain_with_query_projection(cuda_device, pdl):
    # A captured PDL chain alternating the query projection and the V
    # up-projection on distinct layers, replayed three times.  pdl = 2 lets
    # the tcgen05 kernels (query and V above 64 tokens) trigger the
    # next launch at their entry: every kernel here allocates tensor memory
    # only after its dependency wait, which is the contract that needs.
    H = 16
    Ms = (1, 8, 9, 32, 5, 16, 40, 100, 256, 3)
    steps = []
    for i, M in enumerate(Ms):
        fmt = "bf16" if i % 2 == 0 else "mxfp8"
        dq = inputs.make_layer(inputs.layer_seed(54, i), H, fmt, m_max=M)
        dv = inputs.make_v_layer(inputs.layer_seed(55, i), H, fmt, m_max=M)
        steps.append((M, fmt, dq, dv, _dev(dv),
                      dict(q_nope=to_device(dq["q_nope"]), q_pe=to_device(dq["q_pe"]), weight=to_device(dq["weight"]),
                           weight_scale=None if dq["weight_scale"] is None else to_device(dq["weight_scale"]))))
        assert mq.mlaqp_prewarm(H, M, fmt, "bf16") == mq.MLAQP_OK
        assert mq.mlaqp_v_up_prewarm(H, M, fmt) == mq.MLAQP_OK
    q_outs = [torch.zeros((M * 576 * H,), dtype=torch.int16, device="cuda") for M in Ms]
    v_outs = [torch.zeros((M * V * H,), dtype=torch.int16, device="cuda") for M in Ms]
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i, (M, fmt, dq, dv, tv, tq) in enumerate(steps):
            st = mq.mlaqp_run_strided(tq["q_nope"], H * 128, 128, tq["q_pe"], H * 64, 64, tq["weight"],
                                      tq["weight_scale"], q_outs[i], 576 * H, None, M, H, 128, fmt, "bf16", pdl=pdl,
                                      stream=stream)
            assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
            st = mq.mlaqp_v_up_run(tv["x"], H * C, C, tv["weight"], tv["weight_scale"], v_outs[i], V * H, M, H,
                                   fmt, pdl=pdl, stream=stream)
            assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
    for _ in range(3):
        for o in q_outs + v_outs:
            o.zero_()
        graph.replay()
        torch.cuda.synchronize()
    for i, (M, fmt, dq, dv, tv, tq) in enumerate(steps):
        _, acc = _oracle(dv, fmt)
        check_bf16_region(_rows(v_outs[i], M, H, V * H), acc, f"graph v_up {i}")
        _, qacc = oracle.mla_query(dq["q_nope"], dq["q_pe"], dq["weight"], dq["weight_scale"], fmt, "bf16")
        qbits = to_host_bits(q_outs[i], np.uint16).reshape(M, H, 576)
        check_bf16_region(qbits[..., :512], qacc, f"graph query {i}")
        np.testing.assert_array_equal(qbits[..., 512:], dq["q_pe"])


@pytest.mark.parametrize("H,M", [(8, 4), (8, 20), (8, 40), (8, 100), (16, 100)])
def test_bounded_wait_reports_timeout_and_writes_nothing(cuda_device, H, M):
    # H = 8, M = 20 / 40 / 100 run the x-multicast kernel (1, 2 and 4 token
    # chunks): every CTA gives up on its weight copy but still sends its x
    # box and waits for the others'.  H = 16, M = 100 runs the tcgen05
    # cluster kernel: every CTA gives up on its weight copy but still passes
    # both cluster barriers, and no cluster writes.
    st, _ = mq.mlaqp_device_status(reset=True)
    assert st == mq.MLAQP_OK
    for fmt in ("bf16", "mxfp8"):
        d = inputs.make_v_layer(56, H, fmt, m_max=M)
        t = _dev(d)
        out = torch.full((M * V * H,), 0x7777, dtype=torch.int16, device="cuda")
        st = mq.mlaqp_debug_v_up_bounded_wait(t["x"], H * C, C, t["weight"], t["weight_scale"], out, V * H, M, H,
                                              fmt, 2_000_000, 16)
        assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
        torch.cuda.synchronize()
        assert (out == 0x7777).all()
        st, word = mq.mlaqp_device_status(reset=True)
        assert st == mq.MLAQP_OK and word & mq.MLAQP_DEVSTATUS_WAIT_TIMEOUT
        _, acc = _oracle(d, fmt)
        check_bf16_region(_rows(_run(t, M, H, fmt), M, H, V * H), acc, f"after timeout {fmt}")
        st, word = mq.mlaqp_device_status(reset=False)
        assert word == 0


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
@pytest.mark.parametrize("H", [8, 11, 16])
def test_larger_token_counts(cuda_device, fmt, H):
    # Above M = 32: the chunked kernels (H = 8 to M = 128, H = 11 to 96,
    # H = 16 to 64) and the tcgen05 cluster kernel beyond, with token tiles
    # of 64 / 128 and their edges, ragged tails (16-token MMA padding, chunks
    # of 1 token), strided x and a pitched workspace.
    MM = 256
    d = inputs.make_v_layer(inputs.layer_seed(57, H), H, fmt, m_max=MM)
    _, acc = _oracle(d, fmt)
    t = _dev(d)
    for M in (33, 47, 63, 64, 65, 100, 128, 129, 200, 255, 256):
        got = _rows(_run(t, M, H, fmt, pdl=(M % 2 == 1)), M, H, V * H)
        check_bf16_region(got, acc[:M], f"v_up {fmt} H{H} M{M}")
    stride = V * H + 40
    ws = torch.full((MM * stride + 64,), 0x5A5A, dtype=torch.int16, device="cuda")
    hm = to_device(np.ascontiguousarray(np.transpose(d["x"], (1, 0, 2))))
    _run(t, 200, H, fmt, x=hm, x_ts=C, x_hs=MM * C, out=ws, stride=stride)
    bits = to_host_bits(ws, np.uint16)
    mask = np.zeros(bits.shape, dtype=bool)
    for m in range(200):
        mask[m * stride: m * stride + H * V] = True
    assert (bits[~mask] == 0x5A5A).all(), "bytes outside the rows changed"
    check_bf16_region(_rows(ws, 200, H, stride), acc[:200], f"v_up {fmt} M200 head-major pitched")


def test_larger_token_counts_bit_exact(cuda_device):
    # Small-integer data is exact in any summation order, so the cluster
    # kernel's split contraction must match bit for bit (64- and 128-token
    # tiles) as the chunked kernel does (M = 64).
    for fmt in ("bf16", "mxfp8"):
        d = inputs.small_integer_v_layer(58, 16, 256, fmt)
        ref, _ = _oracle(d, fmt)
        t = _dev(d)
        for M in (64, 100, 256):
            got = _rows(_run(t, M, 16, fmt), M, 16, V * 16)
            np.testing.assert_array_equal(got, ref[:M], err_msg=f"{fmt} M{M}")
        # H = 8: four 32-token chunks of the x-multicast kernel at M = 128
        d8 = inputs.small_integer_v_layer(59, 8, 128, fmt)
        ref8, _ = _oracle(d8, fmt)
        got = _rows(_run(_dev(d8), 128, 8, fmt), 128, 8, V * 8)
        np.testing.assert_array_equal(got, ref8, err_msg=f"{fmt} H8 M128")


@pytest.mark.parametrize("M,qfmt,vfmt", [(20, "bf16", "mxfp8"), (40, "mxfp8", "bf16"), (5, "bf16", "bf16")])
def test_reads_x_written_by_the_previous_kernel(cuda_device, M, qfmt, vfmt):
    # A PDL chain in which the V up-projection's x is the query op's output
    # (columns 0..511 of its [M,H,576] rows, head stride 576), so the V
    # kernel reads data the kernel just before it wrote: at M = 20 and 40
    # through the x multicast (a TMA copy after the dependency wait), at
    # M = 5 through plain loads.  Small integers keep both steps exact
    # (|projection| <= 256, V partial sums <= 2^17), so the oracle's own
    # chain must match bit for bit.  Outputs start as BF16 NaN each replay.
    H = 16
    row = 576 * H
    dq = inputs.small_integer_layer(60 + M, H, M, qfmt)
    dv = inputs.small_integer_v_layer(61 + M, H, M, vfmt)
    tq = dict(q_nope=to_device(dq["q_nope"]), q_pe=to_device(dq["q_pe"]), weight=to_device(dq["weight"]),
              weight_scale=None if dq["weight_scale"] is None else to_device(dq["weight_scale"]))
    tv = _dev(dv)
    q_out = torch.zeros((M * row,), dtype=torch.int16, device="cuda")
    v_out = torch.zeros((M * V * H,), dtype=torch.int16, device="cuda")

    def launch(stream=None):
        st = mq.mlaqp_run_strided(tq["q_nope"], H * 128, 128, tq["q_pe"], H * 64, 64, tq["weight"], tq["weight_scale"],
                                  q_out, row, None, M, H, 128, qfmt, "bf16", pdl=1, stream=stream)
        assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
        st = mq.mlaqp_v_up_run(q_out, row, 576, tv["weight"], tv["weight_scale"], v_out, V * H, M, H, vfmt, pdl=1,
                               stream=stream)
        assert st == mq.MLAQP_OK, mq.mlaqp_last_error()

    qref, qacc = oracle.mla_query(dq["q_nope"], dq["q_pe"], dq["weight"], dq["weight_scale"], qfmt, "bf16")
    assert np.all(qacc == np.round(qacc)) and np.abs(qacc).max() <= 256
    vref, vacc = oracle.mla_v_up(np.ascontiguousarray(qref[..., :C]), dv["weight"], dv["weight_scale"], vfmt)
    assert np.all(vacc == np.round(vacc)) and np.abs(vacc).max() <= 2 ** 17

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        launch(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch()
    for rep in range(3):
        q_out.fill_(0x7FC0)
        v_out.fill_(0x7FC0)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_host_bits(q_out, np.uint16).reshape(M, H, 576), qref, err_msg=f"query {rep}")
        np.testing.assert_array_equal(_rows(v_out, M, H, V * H), vref, err_msg=f"v_up {rep}")
