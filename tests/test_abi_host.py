"""The C-ABI library builds, loads and exports what include/mlaqp.h declares;
host-side argument validation returns the documented status codes before
any CUDA call (no GPU needed)."""

import subprocess

import pytest

import mla_decode_query_gb300 as mq
from mla_decode_query_gb300 import build

A = 1 << 20  # a 16-byte aligned fake device address, never dereferenced
H, M = 16, 4
STRIDE = 576 * H


def test_every_declared_symbol_is_exported(built_library):
    declared = mq.header_functions()
    assert {"mlaqp_can_implement", "mlaqp_prewarm", "mlaqp_run", "mlaqp_last_error"} <= set(declared)
    for name in declared:
        assert hasattr(built_library, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", str(build.LIB_PATH)], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = {line.split()[-1] for line in nm.stdout.splitlines() if line.strip()}
        assert set(declared) <= exported, set(declared) - exported


def test_library_is_built_for_sm103a(built_library):
    assert "compute_103a,code=sm_103a" in " ".join(build.ARCH_FLAGS)
    assert mq.mlaqp_version() == 100


def _args(**kw):
    a = dict(q_nope=A, q_pe=2 * A, weight=4 * A, weight_scale=None, out=16 * A, out_row_stride=STRIDE,
             q_scale=None, M=M, H=H, weight_format="bf16", out_dtype="bf16", stream=0)
    a.update(kw)
    return a


def _run(**kw):
    return mq.mlaqp_run(**_args(**kw))


@pytest.mark.parametrize("kw,code", [
    (dict(weight_format=7), mq.MLAQP_ERR_INVALID_ARG),
    (dict(out_dtype=-1), mq.MLAQP_ERR_INVALID_ARG),
    (dict(M=-1), mq.MLAQP_ERR_INVALID_ARG),
    (dict(H=12), mq.MLAQP_ERR_UNSUPPORTED),
    (dict(H=32), mq.MLAQP_ERR_UNSUPPORTED),
    (dict(M=257), mq.MLAQP_ERR_UNSUPPORTED),
    (dict(q_nope=None), mq.MLAQP_ERR_INVALID_ARG),
    (dict(q_pe=None), mq.MLAQP_ERR_INVALID_ARG),
    (dict(weight=None), mq.MLAQP_ERR_INVALID_ARG),
    (dict(out=None), mq.MLAQP_ERR_INVALID_ARG),
    (dict(weight_scale=8 * A), mq.MLAQP_ERR_INVALID_ARG),              # BF16 takes no scale
    (dict(weight_format="mxfp8"), mq.MLAQP_ERR_INVALID_ARG),           # MXFP8 needs a scale
    (dict(q_scale=32 * A), mq.MLAQP_ERR_INVALID_ARG),                  # BF16 output takes none
    (dict(out_dtype="e4m3"), mq.MLAQP_ERR_INVALID_ARG),                # E4M3 output needs one
    (dict(q_nope=A + 8), mq.MLAQP_ERR_INVALID_ARG),                    # misaligned
    (dict(out=16 * A + 4), mq.MLAQP_ERR_INVALID_ARG),
    (dict(out_dtype="e4m3", q_scale=32 * A + 2), mq.MLAQP_ERR_INVALID_ARG),
    (dict(out_row_stride=STRIDE - 8), mq.MLAQP_ERR_INVALID_ARG),       # < 576*H
    (dict(out_row_stride=STRIDE + 4), mq.MLAQP_ERR_INVALID_ARG),       # 8 bytes, not 16
    (dict(out=A + 4096), mq.MLAQP_ERR_INVALID_ARG),                    # overlaps q_nope
    (dict(out=4 * A), mq.MLAQP_ERR_INVALID_ARG),                       # overlaps the weights
])
def test_validation_status_codes(built_library, kw, code):
    assert _run(**kw) == code
    assert mq.mlaqp_last_error() != ""


def test_e4m3_stride_must_be_16_byte_multiple(built_library):
    # 576*11 E4M3 bytes = 6336 = 16*396 is fine; +8 elements is not.
    a = dict(H=11, out_row_stride=576 * 11 + 8, out_dtype="e4m3", q_scale=32 * A)
    assert _run(**a) == mq.MLAQP_ERR_INVALID_ARG


def test_zero_tokens_is_a_no_op(built_library):
    assert _run(M=0, q_nope=None, out=None) == mq.MLAQP_OK


def test_valid_arguments_reach_the_device_check(built_library):
    import torch
    st = _run()
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    assert st == mq.MLAQP_ERR_CUDA
    assert mq.mlaqp_can_implement(16, 32) == 0


def test_can_implement_domain(built_library):
    # Shape gating is decided before the device is queried.
    for bad in [dict(num_heads=12), dict(max_m=0), dict(max_m=257), dict(nope_dim=256),
                dict(latent_dim=256), dict(rope_dim=32), dict(weight_format=5)]:
        a = dict(num_heads=16, max_m=32)
        a.update(bad)
        assert mq.mlaqp_can_implement(**a) == 0, bad


def test_launch_shape(built_library):
    # Up to M = 8 the CTA-tile kernel: 8 CTAs of 64 latent columns per head,
    # one 4-warp token group.  From the crossover (M = 9..17) the warp-tile
    # kernel, whose grid follows the device's SM count: checked on the GPU.
    for h in (8, 11, 16):
        for m in (1, 5, 8):
            st, grid, threads = mq.mlaqp_launch_shape(m, h, "mxfp8", "e4m3")
            assert st == mq.MLAQP_OK and grid == 8 * h and threads == 128
    # M = 33..64: the CTA-tile kernel in two 32-token chunks (grid.z), two
    # token groups.  Above M = 64 the choice depends on the device's SM count
    # (checked on the GPU).
    for m in (33, 64):
        st, grid, threads = mq.mlaqp_launch_shape(m, 11, "bf16", "bf16")
        assert st == mq.MLAQP_OK and grid == 8 * 11 * 2 and threads == 256
    assert mq.mlaqp_launch_shape(0, 16)[0] == mq.MLAQP_ERR_UNSUPPORTED
    assert mq.mlaqp_launch_shape(257, 16)[0] == mq.MLAQP_ERR_UNSUPPORTED
    assert mq.mlaqp_launch_shape(4, 12)[0] == mq.MLAQP_ERR_UNSUPPORTED


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from mla_decode_query_gb300 import mlaqp
    monkeypatch.setattr(mlaqp, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        mlaqp.load_library(tmp_path / "libmlaqp.so")


def _strided(**kw):
    a = dict(q_nope=A, q_nope_token_stride=H * 128, q_nope_head_stride=128, q_pe=2 * A,
             q_pe_token_stride=H * 64, q_pe_head_stride=64, weight=4 * A, weight_scale=None, out=16 * A,
             out_row_stride=STRIDE, q_scale=None, M=M, H=H, nope_dim=128, weight_format="bf16", out_dtype="bf16",
             pdl=False, stream=0)
    a.update(kw)
    return mq.mlaqp_run_strided(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(nope_dim=256), mq.MLAQP_ERR_UNSUPPORTED),
    (dict(nope_dim=64), mq.MLAQP_ERR_UNSUPPORTED),
    (dict(q_nope_token_stride=H * 128 + 4), mq.MLAQP_ERR_INVALID_ARG),   # not a 16-byte row
    (dict(q_nope_head_stride=130), mq.MLAQP_ERR_INVALID_ARG),
    (dict(q_pe_head_stride=65), mq.MLAQP_ERR_INVALID_ARG),               # odd: 4-byte pairs
    (dict(q_pe_token_stride=-64), mq.MLAQP_ERR_INVALID_ARG),
    (dict(q_pe=2 * A + 2), mq.MLAQP_ERR_INVALID_ARG),                    # q_pe needs 4-byte alignment
    (dict(q_nope=A + 8), mq.MLAQP_ERR_INVALID_ARG),
    (dict(out=A + 4096), mq.MLAQP_ERR_INVALID_ARG),                      # overlaps the q_nope span
])
def test_strided_validation(built_library, kw, code):
    assert _strided(**kw) == code
    assert mq.mlaqp_last_error() != ""


def test_strided_accepts_views_and_nope192_shapes(built_library):
    # Shapes and strides of the upstream [M, H, 192+64] projection pass every
    # host check; without a GPU the call then stops at the device query.
    import torch
    st = _strided(nope_dim=192, q_nope_token_stride=H * 256, q_nope_head_stride=256, q_pe=A + 384,
                  q_pe_token_stride=H * 256, q_pe_head_stride=256)
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    assert st == mq.MLAQP_ERR_CUDA


def _v_up(**kw):
    a = dict(x=A, x_token_stride=H * 512, x_head_stride=512, weight=4 * A, weight_scale=None, out=16 * A,
             out_row_stride=128 * H, M=M, H=H, weight_format="bf16", pdl=False, stream=0)
    a.update(kw)
    return mq.mlaqp_v_up_run(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(weight_format=3), mq.MLAQP_ERR_INVALID_ARG),
    (dict(M=-1), mq.MLAQP_ERR_INVALID_ARG),
    (dict(H=12), mq.MLAQP_ERR_UNSUPPORTED),
    (dict(M=257), mq.MLAQP_ERR_UNSUPPORTED),                             # M <= 256
    (dict(x=None), mq.MLAQP_ERR_INVALID_ARG),
    (dict(weight=None), mq.MLAQP_ERR_INVALID_ARG),
    (dict(out=None), mq.MLAQP_ERR_INVALID_ARG),
    (dict(weight_scale=8 * A), mq.MLAQP_ERR_INVALID_ARG),                # BF16 takes no scale
    (dict(weight_format="mxfp8"), mq.MLAQP_ERR_INVALID_ARG),             # MXFP8 needs one
    (dict(x=A + 8), mq.MLAQP_ERR_INVALID_ARG),                           # misaligned
    (dict(out=16 * A + 4), mq.MLAQP_ERR_INVALID_ARG),
    (dict(x_head_stride=516), mq.MLAQP_ERR_INVALID_ARG),                 # not a 16-byte row
    (dict(x_token_stride=-512), mq.MLAQP_ERR_INVALID_ARG),
    (dict(out_row_stride=128 * H - 8), mq.MLAQP_ERR_INVALID_ARG),        # < 128*H
    (dict(out_row_stride=128 * H + 4), mq.MLAQP_ERR_INVALID_ARG),        # 8 bytes, not 16
    (dict(out=A + 4096), mq.MLAQP_ERR_INVALID_ARG),                      # overlaps x
    (dict(out=4 * A + 1024), mq.MLAQP_ERR_INVALID_ARG),                  # overlaps the weights
])
def test_v_up_validation(built_library, kw, code):
    assert _v_up(**kw) == code
    assert mq.mlaqp_last_error() != ""


def test_v_up_zero_tokens_and_domain(built_library):
    assert _v_up(M=0, x=None, out=None) == mq.MLAQP_OK
    for bad in [dict(num_heads=12), dict(max_m=0), dict(max_m=257), dict(weight_format=4)]:
        a = dict(num_heads=16, max_m=32, weight_format="bf16")
        a.update(bad)
        assert mq.mlaqp_v_up_can_implement(**a) == 0, bad


@pytest.mark.parametrize("kw,code", [
    (dict(weight_format=7), mq.MLAQP_ERR_INVALID_ARG),
    (dict(H=12), mq.MLAQP_ERR_UNSUPPORTED),
    (dict(nope_dim=64), mq.MLAQP_ERR_UNSUPPORTED),
    (dict(weight=None), mq.MLAQP_ERR_INVALID_ARG),
    (dict(weight=0x1008), mq.MLAQP_ERR_INVALID_ARG),              # not 16-byte aligned
    (dict(weight_scale=0x2000), mq.MLAQP_ERR_INVALID_ARG),        # BF16 weights take no scales
    (dict(weight_format="mxfp8", weight_scale=None), mq.MLAQP_ERR_INVALID_ARG),
])
def test_prefetch_validation(built_library, kw, code):
    # Every argument check runs before the device is touched.
    a = dict(weight=0x1000, weight_scale=None, H=16, nope_dim=128, weight_format="bf16", stream=0)
    a.update(kw)
    assert mq.mlaqp_prefetch_weights(**a) == code, mq.mlaqp_last_error()


def test_pdl_mode_is_validated(built_library):
    # pdl must be 0, 1 or 2 (2: the opt-in early trigger of the tcgen05 kernels)
    for pdl in (-1, 3):
        st = mq.mlaqp_run_strided(0x1000, 16 * 128, 128, 0x2000, 16 * 64, 64, 0x3000, None, 0x100000, 576 * 16,
                                  None, 4, 16, 128, "bf16", "bf16", pdl=pdl, stream=0)
        assert st == mq.MLAQP_ERR_INVALID_ARG, (pdl, mq.mlaqp_last_error())
        st = mq.mlaqp_v_up_run(0x1000, 16 * 512, 512, 0x3000, None, 0x100000, 128 * 16, 4, 16, "bf16", pdl=pdl,
                               stream=0)
        assert st == mq.MLAQP_ERR_INVALID_ARG, (pdl, mq.mlaqp_last_error())
