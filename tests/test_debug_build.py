"""The bounds-checking debug build (build(debug=True), -DBSFP8_DEBUG=1): its kernels check
every tile's coordinates against the problem and would record BSFP8_ERR_DEVICE_BOUNDS
instead of going out of range.  On correct inputs it must report nothing and compute what
the release build computes (every blockwise and MX tile form, and the fp4 MMA kinds with
256-K and 128-K stages).  Runs in a child process that loads only the debug library."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, os.path.join({root!r}, "tests"))
import numpy as np
import gen, oracle
from gpu_util import DeviceProblem
from helpers import parity_report
import block_scaled_fp8_persistent_gb300 as bsfp8
assert bsfp8.LIB_PATH.endswith("libbsfp8_debug.so"), bsfp8.LIB_PATH
cases = [("blockwise", "cta1_96", [130, 0, 77, 1], 384, 640),
         ("blockwise", "pair_224", [500, 3, 0, 230], 256, 384),
         ("blockwise", "split", [500, 3, 0, 447, 448, 900], 256, 256),
         ("mx", "swap", [3, 17, 0, 32, 1, 9], 256, 512),
         ("mx", "pair", [700, 0, 513], 256, 640),
         ("mx", "split", [300, 7, 0, 45, 260, 129], 256, 512),
         ("fp4", "mxfp8:mxfp4", [3, 17, 0, 32, 1, 9], 256, 1024),
         ("fp4", "mxfp4:mxfp4", [40, 0, 7, 64], 384, 1024),
         ("fp4", "nvfp4:nvfp4", [3, 17, 0, 32, 1, 9], 256, 768),
         ("fp4", "mxfp4:mxfp4", [40, 0, 7], 256, 640),
         ("fp4pair", "mxfp8:mxfp4", [300, 0, 270], 256, 1024),
         ("fp4pair", "mxfp4:mxfp4", [300, 0, 270], 256, 1024),
         ("fp4pair", "nvfp4:nvfp4", [300, 0, 270], 256, 768)]
for mode, form, counts, N, K in cases:
    if mode == "blockwise":
        os.environ["BSFP8_BLOCKWISE_TILE"] = form
        p = gen.blockwise_problem(counts, N, K, seed=77)
    elif mode in ("fp4", "fp4pair"):
        a_fmt, b_fmt = form.split(":")
        if mode == "fp4pair":
            os.environ["BSFP8_MX_KERNEL"] = "pair"
        p = gen.fmt_problem(counts, N, K, seed=79, a_fmt=a_fmt, b_fmt=b_fmt)
    else:
        os.environ["BSFP8_MX_KERNEL"] = form
        p = gen.mx_problem(counts, N, K, seed=78)
    d = DeviceProblem(p, c_rows_extra=2)
    d.run()
    assert bsfp8.bsfp8_get_device_error() == 0, (mode, form)
    ref, T = oracle.problem_reference(p)
    bad, ratio, exact = parity_report(d.c_bits(), ref, T)
    assert bad == 0, (mode, form, bad, ratio)
    assert np.all(d.guard_bits() == d.sentinel), (mode, form)
print("debug build ok")
"""


def test_debug_build_reports_nothing_and_matches_the_oracle():
    from block_scaled_fp8_persistent_gb300 import build as libbuild
    path = libbuild.build(debug=True)
    env = dict(os.environ, BSFP8_LIBRARY=path)
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug build ok" in r.stdout
