"""Parity at full size, in the launch configuration the benchmark times:
CUDA graphs of one programmatic-dependent launch per layer over 128 (or
256) distinct layers, each layer with its own weights, inputs and output.
Sampled layers {first, middle, last} are compared with the oracle in full
for every token count."""

import numpy as np
import pytest
import torch

import bench
import oracle
from helpers import check_output, to_host_bits

pytestmark = pytest.mark.gpu


def _check_set(ls, layers, where):
    for M in ls.m_points:
        out = to_host_bits(ls.out[M], np.uint16 if ls.out_dtype == "bf16" else np.uint8)
        for l in layers:
            d = ls.host[l]
            ref, acc = oracle.mla_query(d["q_nope"][:M], d["q_pe"][:M], d["weight"], d["weight_scale"],
                                        ls.weight_format, ls.out_dtype, ls.q_scale_value)
            check_output(out[l], ref, acc, ls.out_dtype, f"{where} M{M} layer{l}")


@pytest.mark.parametrize("fmt,od,H,L,m_points,cfg", [
    ("bf16", "bf16", 11, 128, (1, 2, 4, 8, 16, 32), 1),      # BF16 weights, H=11
    ("mxfp8", "bf16", 8, 128, tuple(range(1, 33)), 2),        # MXFP8 weights, H=8, every M
    ("mxfp8", "e4m3", 16, 128, tuple(range(1, 33)), 3),       # MXFP8 -> E4M3, H=16, every M
    ("bf16", "bf16", 16, 128, (1, 2, 4, 8, 16, 32), 1),       # the benchmark's BF16 set
    ("mxfp8", "e4m3", 16, 256, (1, 8, 32), 3),                # the benchmark's MXFP8 set size
])
def test_graph_replay_full_size(cuda_device, fmt, od, H, L, m_points, cfg):
    ls = bench.LayerSet(fmt, od, L, h=H, m_points=m_points, config_index=cfg)
    for M in m_points:
        g = ls.capture(M, pdl=True)
        ls.out[M].zero_()
        g.replay()
        g.replay()  # a second replay over already-written outputs must not change them
    torch.cuda.synchronize()
    _check_set(ls, (0, L // 2 - 1, L - 1), f"{fmt}->{od} H{H}")


def test_graph_replay_with_mutated_inputs(cuda_device):
    # Capture once, then overwrite q_nope, q_pe and q_scale in place between
    # replays: the replay must use the new values (q_scale is read on device).
    ls = bench.LayerSet("mxfp8", "e4m3", 4, h=16, m_points=(5, 32), config_index=3)
    graphs = {M: ls.capture(M, pdl=True) for M in ls.m_points}
    from mla_decode_query_gb300 import inputs
    for it in range(3):
        fresh = [inputs.make_layer(inputs.layer_seed(50 + it, l), 16, "mxfp8") for l in range(ls.L)]
        qs = np.float32(0.02 + 0.03 * it)
        ls.q_scale.fill_(float(qs))
        ls.q_scale_value = qs
        for M in ls.m_points:
            qn = np.stack([f["q_nope"][:M] for f in fresh]).view(np.int16)
            qp = np.stack([f["q_pe"][:M] for f in fresh]).view(np.int16)
            ls.q_nope[M].copy_(torch.from_numpy(qn))
            ls.q_pe[M].copy_(torch.from_numpy(qp))
            graphs[M].replay()
        torch.cuda.synchronize()
        for l in range(ls.L):
            ls.host[l] = dict(ls.host[l], q_nope=fresh[l]["q_nope"], q_pe=fresh[l]["q_pe"])
        _check_set(ls, range(ls.L), f"mutated it{it}")
