"""Shared test helpers: device transfer and oracle comparisons.

The tolerances are the acceptance bounds of this operation: the q_pe
columns bit-exact, the BF16 projection within |gpu - ref| <= 1e-2*|ref| +
1e-3 of the float64 projection, E4M3 output within one E4M3 ulp of the
oracle's code.
"""

import numpy as np

import oracle

BF16_RTOL = 1e-2
BF16_ATOL = 1e-3
E4M3_MAX_ULP = 1


def to_device(bits, device="cuda"):
    import torch
    a = np.ascontiguousarray(bits)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    elif a.dtype == np.uint8:
        t = torch.from_numpy(a)
    else:
        raise TypeError(a.dtype)
    return t.to(device)


def to_host_bits(t, dtype):
    a = t.detach().cpu().contiguous().numpy()
    return a.view(dtype)


def check_bf16_region(gpu_bits, acc, where=""):
    g = oracle.bf16_to_f64(gpu_bits)
    err = np.abs(g - acc)
    bound = BF16_RTOL * np.abs(acc) + BF16_ATOL
    bad = ~(err <= bound)
    assert not bad.any(), (
        f"{where}: {int(bad.sum())} BF16 values out of tolerance; worst at "
        f"{np.unravel_index(np.argmax(err - bound), err.shape)}: gpu={g.flat[np.argmax(err - bound)]} "
        f"ref={acc.flat[np.argmax(err - bound)]}")
    return float(err.max()) if err.size else 0.0


def check_e4m3_region(gpu_codes, ref_codes, where=""):
    d = np.abs(oracle.e4m3_ordinal(gpu_codes) - oracle.e4m3_ordinal(ref_codes))
    assert (d <= E4M3_MAX_ULP).all(), (
        f"{where}: {int((d > E4M3_MAX_ULP).sum())} E4M3 codes more than {E4M3_MAX_ULP} ulp apart; "
        f"max {int(d.max())}")
    return int(d.max()) if d.size else 0


def check_output(gpu_out, ref_out, acc, out_dtype, where=""):
    """gpu_out/ref_out: [M,H,576] bits; acc: float64 [M,H,512]."""
    assert gpu_out.shape == ref_out.shape, (gpu_out.shape, ref_out.shape)
    np.testing.assert_array_equal(gpu_out[..., 512:], ref_out[..., 512:], err_msg=f"{where}: q_pe region")
    if out_dtype == "bf16":
        return check_bf16_region(gpu_out[..., :512], acc, where)
    return check_e4m3_region(gpu_out[..., :512], ref_out[..., :512], where)
