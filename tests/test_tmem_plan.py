"""The TMEM plan of double-buffered block-scaled accumulators, pinned to the worked values
printed by the Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix
Multiplication" (tests/golden/tmem_overlap_plan.txt).  Host only: no GPU is used."""
import os

import pytest

import block_scaled_fp8_persistent_gb300 as bsfp8
from block_scaled_fp8_persistent_gb300 import build as libbuild

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tmem_overlap_plan.txt")
KEYS = ("left_offset", "left_cols", "right_offset", "right_cols", "a_scale_offset",
        "a_scale_cols", "b_scale_offset", "b_scale_cols", "early_release_subtile")


def _cases():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        lhs, rhs = line.split("|")
        out.append((tuple(int(x) for x in lhs.split()), rhs.split()))
    return out


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()


@pytest.mark.parametrize("args,expect", _cases())
def test_plan_matches_page_worked_values(args, expect):
    plan = bsfp8.bsmxfp8_tmem_plan(*args)
    for key, val in zip(KEYS, expect):
        if val != "-":
            assert plan[key] == int(val), (key, plan)


def test_compiled_pair_kernel_plan():
    # the CTA-pair MXFP8 kernel uses BLOCK_K 128, 32-column subtiles, UE8M0 per 32
    assert bsfp8.bsmxfp8_tmem_plan(0, 0, 0, 0) == bsfp8.bsmxfp8_tmem_plan(128, 32, 32, True)


def test_plan_invariants():
    for bk, vec in ((128, 32), (256, 16), (256, 32), (128, 16)):
        p = bsfp8.bsmxfp8_tmem_plan(bk, 32, vec, True)
        # the two accumulators overlap exactly by the scale columns, which end at column 512
        assert p["left_offset"] + p["left_cols"] - p["right_offset"] == p["a_scale_cols"] + p["b_scale_cols"]
        assert p["right_offset"] + p["right_cols"] == p["a_scale_offset"]
        assert p["b_scale_offset"] + p["b_scale_cols"] == 512


def test_plan_rejects_bad_shapes():
    with pytest.raises(bsfp8.BsFp8Error):
        bsfp8.bsmxfp8_tmem_plan(100, 32, 32, True)


@pytest.mark.parametrize("slots,vec,right,a_off,b_off", [(3, 32, 184, 440, 464), (2, 16, 160, 416, 448)])
def test_fp4_pair_slot_plans(slots, vec, right, a_off, b_off):
    # the fp4 x fp4 CTA-pair forms keep `slots` K blocks of 256 worth of scales in TMEM (mxfp4
    # three, nvfp4 two): the plan of one K block that long, whose shared columns must lie in
    # the column half an epilogue warp drains first (release before its fifth 32-column
    # subtile); the same planner for one K block gives the page's worked values
    p = bsfp8.bsmxfp8_tmem_plan(slots * 256, 32, vec, True)
    assert (p["right_offset"], p["a_scale_offset"], p["b_scale_offset"]) == (right, a_off, b_off)
    assert p["a_scale_cols"] == slots * (256 // vec) and p["b_scale_cols"] == 2 * p["a_scale_cols"]
    assert p["early_release_subtile"] < 4
    assert p["a_scale_offset"] % 4 == 0 and p["b_scale_offset"] % 4 == 0
    # a third nvfp4 slot would reach past that half
    assert bsfp8.bsmxfp8_tmem_plan(3 * 256, 32, 16, True)["early_release_subtile"] >= 4
