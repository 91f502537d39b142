"""The library's launch decisions, checked on the host (no GPU).

mlaqp_debug_plan / mlaqp_debug_v_plan run the same planning code as the
launch path, for a given SM count.  The expectations are the decision rules
the library documents (kernel crossovers, token chunks, CTA caps, the fit
tiers), written out as explicit cases at the GB300's 152 SMs and at other
SM counts, so that a change to any rule shows up here before a GPU run.
"""

import pytest

import mla_decode_query_gb300 as mq

SMS = 152


def plan(M, H, fmt="bf16", od="bf16", **kw):
    st, p = mq.mlaqp_debug_plan(M, H, fmt, od, sm_count=kw.pop("sm", SMS), **kw)
    assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
    return p


def v_plan(M, H, fmt="bf16", **kw):
    st, p = mq.mlaqp_debug_v_plan(M, H, fmt, sm_count=kw.pop("sm", SMS), **kw)
    assert st == mq.MLAQP_OK, mq.mlaqp_last_error()
    return p


@pytest.mark.parametrize("M,H,fmt,od,arm,chunk,cap,grid,threads", [
    # M <= 8: the CTA-tile kernel, 8 CTAs per head, one token group
    (1, 16, "mxfp8", "e4m3", "cta_mma", 0, 2, 128, 128),
    (8, 8, "bf16", "bf16", "cta_mma", 0, 2, 64, 128),
    # H = 16 / 11: CTA-tile below M = 17, warp-tile (one CTA per SM) from it
    (16, 16, "bf16", "bf16", "cta_mma", 0, 2, 128, 256),
    (17, 16, "bf16", "bf16", "warp_mma", 0, 2, 152, 256),
    (32, 16, "mxfp8", "e4m3", "warp_mma", 0, 2, 152, 256),
    (16, 11, "mxfp8", "bf16", "cta_mma", 0, 2, 88, 256),
    (17, 11, "mxfp8", "bf16", "warp_mma", 0, 2, 152, 192),  # 13 CTAs for some heads: 3 tiles each
    # H = 8: two 8-token chunks up to M = 16, two 16-token chunks for MXFP8 above
    (9, 8, "bf16", "bf16", "cta_mma", 8, 2, 128, 128),
    (16, 8, "bf16", "e4m3", "cta_mma", 8, 2, 128, 128),
    (17, 8, "mxfp8", "e4m3", "cta_mma", 16, 2, 128, 256),
    (32, 8, "mxfp8", "bf16", "cta_mma", 16, 2, 128, 256),
    (24, 8, "bf16", "bf16", "warp_mma", 0, 2, 152, 128),
    # above 32: 32-token chunks at two, three, four CTAs per SM, then tcgen05
    (33, 16, "bf16", "bf16", "cta_mma", 32, 2, 256, 256),
    (64, 16, "mxfp8", "e4m3", "cta_mma", 32, 2, 256, 256),
    (96, 16, "bf16", "bf16", "cta_mma", 32, 3, 384, 256),
    (128, 16, "bf16", "e4m3", "cta_mma", 32, 4, 512, 256),
    (129, 16, "bf16", "bf16", "tcgen05", 0, 0, 4 * 16 * 2, 512),
    (192, 11, "mxfp8", "e4m3", "cta_mma", 32, 4, 528, 256),
    (193, 11, "mxfp8", "e4m3", "tcgen05", 0, 0, 4 * 11 * 2, 512),
    (256, 8, "bf16", "bf16", "cta_mma", 32, 4, 512, 256),
])
def test_query_plan_at_152_sms(M, H, fmt, od, arm, chunk, cap, grid, threads):
    p = plan(M, H, fmt, od)
    assert (p["arm"], p["chunk_tokens"], p["cta_cap"], p["grid_ctas"], p["threads_per_cta"]) == \
        (arm, chunk, cap, grid, threads), p


def test_query_trigger_points():
    assert plan(1, 16)["trig"] == 0                      # entry
    assert plan(24, 16, "bf16", "e4m3", arm="cta_mma")["trig"] == 1  # BF16->E4M3, 17..32: after the wait
    assert plan(40, 16, "bf16", "e4m3")["trig"] == 0     # chunked above 32: entry again
    tc = plan(200, 16)
    assert tc["arm"] == "tcgen05" and tc["trig"] == 1    # after its tensor-memory allocation
    assert plan(200, 16, pdl=2)["trig"] == 0             # the opt-in entry trigger
    assert plan(1, 16, pdl=0)["cta_cap"] == 0            # no padding without PDL


def test_query_plan_follows_the_sm_count():
    # Fewer SMs: the small-M chunks at H = 8 need 128 free SMs.
    assert plan(12, 8, sm=152)["chunk_tokens"] == 8
    assert plan(12, 8, sm=120)["chunk_tokens"] == 0
    # The fit tiers shrink with the SM count: at 132 SMs, four chunks of
    # H = 16 (512 CTAs) still fit at four per SM, at 120 (480 slots) not.
    assert plan(128, 16, sm=132)["arm"] == "cta_mma"
    assert plan(128, 16, sm=120)["arm"] == "tcgen05"
    # The warp-tile grid is the SM count, clamped to 8..32 CTAs per head.
    assert plan(20, 16, sm=132)["grid_ctas"] == 132
    assert plan(20, 16, sm=600)["grid_ctas"] == 32 * 16
    assert plan(20, 8, sm=40)["grid_ctas"] == 8 * 8


def test_nope192_stays_in_one_launch_below_33_and_has_no_four_per_sm_tier():
    assert plan(12, 8, nope_dim=192)["chunk_tokens"] == 0
    assert plan(96, 16, nope_dim=192)["cta_cap"] == 3
    assert plan(128, 16, nope_dim=192)["arm"] == "tcgen05"   # 80 registers: four 256-thread CTAs do not fit


def test_forced_arms_and_invalid_arguments():
    assert mq.mlaqp_debug_plan(9, 16, arm="warp_fma")[0] == mq.MLAQP_ERR_UNSUPPORTED
    assert mq.mlaqp_debug_plan(33, 16, arm="warp_mma")[0] == mq.MLAQP_ERR_UNSUPPORTED
    assert mq.mlaqp_debug_plan(4, 16, arm="tcgen05")[1]["arm"] == "tcgen05"
    assert mq.mlaqp_debug_plan(4, 16, arm="warp_fma")[1]["arm"] == "warp_fma"
    assert mq.mlaqp_debug_plan(0, 16)[0] == mq.MLAQP_ERR_UNSUPPORTED
    assert mq.mlaqp_debug_plan(4, 12)[0] == mq.MLAQP_ERR_UNSUPPORTED
    assert mq.mlaqp_debug_plan(4, 16, nope_dim=256)[0] == mq.MLAQP_ERR_UNSUPPORTED
    assert mq.mlaqp_debug_plan(4, 16, pdl=3)[0] == mq.MLAQP_ERR_INVALID_ARG
    assert mq.mlaqp_debug_plan(4, 16, sm_count=0)[0] == mq.MLAQP_ERR_INVALID_ARG


@pytest.mark.parametrize("M,H,fmt,form,chunk,cap,grid,cluster", [
    (4, 16, "bf16", "plain", 32, 2, 128, 1),
    (8, 8, "mxfp8", "plain", 32, 2, 64, 1),
    (9, 16, "bf16", "multicast", 32, 2, 128, 8),
    (11, 16, "mxfp8", "plain", 32, 2, 128, 1),
    (12, 16, "mxfp8", "multicast", 32, 2, 128, 8),
    # H = 8: two 8-token chunks with plain loads, two 16-token chunks (MXFP8)
    (12, 8, "mxfp8", "plain", 8, 2, 128, 1),
    (16, 8, "bf16", "plain", 8, 2, 128, 1),
    (20, 8, "mxfp8", "multicast", 16, 2, 128, 8),
    (20, 8, "bf16", "multicast", 32, 0, 64, 8),
    # above 64: chunks while they fit (two per SM, else up to 2.6), then the cluster kernel
    (96, 16, "bf16", "multicast", 32, 3, 384, 8),
    (97, 16, "bf16", "cluster", 64, 0, 4 * 16 * 2, 4),
    (192, 8, "bf16", "multicast", 32, 3, 384, 8),
    (224, 8, "bf16", "cluster", 128, 0, 4 * 8 * 2, 4),
])
def test_v_plan_at_152_sms(M, H, fmt, form, chunk, cap, grid, cluster):
    p = v_plan(M, H, fmt)
    assert (p["form"], p["chunk_tokens"], p["cta_cap"], p["grid_ctas"], p["cluster"]) == \
        (form, chunk, cap, grid, cluster), p
