"""GPU parity at the workloads' full sizes, every output element against the CPU oracle.

The oracle's result for a workload is computed once (seconds to tens of seconds on the host
cores) and compared with the GPU output of every kernel form that runs it: the seven tile
configurations of the blockwise kernel for the three blockwise workloads, the swap-AB
kernel (row-major and pre-packed weight scales) for the decode-shaped MXFP8 workload, the
CTA-pair kernel for the dense MXFP8 one, and the three fp4 format pairs on the decode
workload's routing and shape (the both-fp4 pairs on the fp4 MMA kinds and on the converting
kernels).  Acceptance per element as everywhere:
|gpu - oracle| <= 2 ulp_bf16(oracle) + 1e-6 * sum|scaled terms|.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import parity_report_chunked

pytestmark = pytest.mark.gpu

TILES = ["cta1_256", "pair_256", "pair_160", "pair_128", "cta1_128", "cta1_96", "pair_192",
         "cta1_96x192", "pair_192x192", "cta1_128x192", "pair_224"]
FP4_PAIRS = [("mxfp8", "mxfp4"), ("mxfp4", "mxfp4"), ("nvfp4", "nvfp4")]

_REFS = {}


def _reference(key, make):
    """(problem, oracle bf16 bits, T) for a workload, computed once per test session."""
    if key not in _REFS:
        p = make()
        ref, T = oracle.problem_reference(p)
        _REFS[key] = (p, ref, T)
    return _REFS[key]


def _run_and_compare(p, ref, T):
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    d = DeviceProblem(p, c_rows_extra=2)
    d.run()
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    bad, ratio, exact = parity_report_chunked(got, ref, T)
    assert bad == 0, f"{bad} of {got.size} elements outside tolerance (max err/tol {ratio:.3g})"
    assert np.all(d.guard_bits() == d.sentinel)
    del d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_blockwise_workload_every_element(cfg, tile, monkeypatch):
    monkeypatch.setenv("BSFP8_BLOCKWISE_TILE", tile)
    p, ref, T = _reference(("config", cfg), lambda: gen.config_problem(cfg))
    _run_and_compare(p, ref, T)


def test_blockwise_workload_default_plan_every_element():
    # the tile configuration the library picks by itself, on the headline workload
    p, ref, T = _reference(("config", 1), lambda: gen.config_problem(1))
    _run_and_compare(p, ref, T)


@pytest.mark.parametrize("tn", ["plan", "32", "64", "128"])
def test_decode_mxfp8_every_element(tn, monkeypatch):
    if tn != "plan":
        monkeypatch.setenv("BSFP8_MX_TN", tn)
    p, ref, T = _reference(("config", 4), lambda: gen.config_problem(4))
    _run_and_compare(p, ref, T)


def test_decode_mxfp8_prepacked_every_element():
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    p, ref, T = _reference(("config", 4), lambda: gen.config_problem(4))
    d = DeviceProblem(p, c_rows_extra=2)
    packed = torch.empty_like(d.sb)
    bsfp8.bsmxfp8_pack_b_scales(d.sb, packed, p.E, p.N, p.K)
    bsfp8.bsmxfp8_grouped_gemm_prepacked(d.A, d.B, d.sa, packed, d.off, d.C, p.M_total, p.N,
                                         p.K, p.E)
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    bad, ratio, _ = parity_report_chunked(got, ref, T)
    assert bad == 0, f"{bad} elements outside tolerance (max err/tol {ratio:.3g})"
    assert np.all(d.guard_bits() == d.sentinel)


@pytest.mark.parametrize("kernel", ["pair", "swap"])
def test_dense_mxfp8_every_element(kernel, monkeypatch):
    monkeypatch.setenv("BSFP8_MX_KERNEL", kernel)
    p, ref, T = _reference(("config", 5), lambda: gen.config_problem(5))
    _run_and_compare(p, ref, T)


@pytest.mark.parametrize("a_fmt,b_fmt,path", [("mxfp8", "mxfp4", "mma"),
                                                ("mxfp8", "mxfp4", "convert"),
                                                ("mxfp4", "mxfp4", "mma"),
                                                ("mxfp4", "mxfp4", "convert"),
                                                ("nvfp4", "nvfp4", "mma"),
                                                ("nvfp4", "nvfp4", "convert")])
def test_fp4_decode_shape_every_element(a_fmt, b_fmt, path, monkeypatch):
    # the decode workload's routing and shape with fp4 operands, as the bench times it (the
    # both-fp4 pairs on the fp4 MMA kinds, and on the converting kernels)
    monkeypatch.setenv("BSFP8_FP4_MMA", path)
    p, ref, T = _reference(("fp4", a_fmt, b_fmt), lambda: gen.fmt_problem(
        gen.config_counts(4), 4096, 7168, seed=4, a_fmt=a_fmt, b_fmt=b_fmt,
        a_recipe="quantized"))
    _run_and_compare(p, ref, T)


@pytest.mark.parametrize("kernel", ["pair", "swap"])
@pytest.mark.parametrize("a_fmt,b_fmt", FP4_PAIRS)
def test_fp4_dense_prefill_every_element(a_fmt, b_fmt, kernel, monkeypatch):
    # a dense prefill-sized fp4 problem (one expert, 4096 x 4096 x 7168): the CTA-pair kernel
    # the plan picks, and the 128-token swap-AB tiles of the fp4 kinds
    monkeypatch.setenv("BSFP8_MX_KERNEL", kernel)
    p, ref, T = _reference(("fp4 dense", a_fmt, b_fmt), lambda: gen.fmt_problem(
        [4096], 4096, 7168, seed=6, a_fmt=a_fmt, b_fmt=b_fmt))
    _run_and_compare(p, ref, T)
