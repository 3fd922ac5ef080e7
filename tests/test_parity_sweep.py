"""Seeded randomized sweep against the oracle: expert sizes around every tile height the
kernels use (96, 128, 192, 256 rows; 32 / 64 / 128 token rows in MX swap-AB tiles), random
N and K, every tile form; both modes, and the fp4 format pairs (32 / 64 token rows)."""
import numpy as np
import pytest

import gen
import oracle
from helpers import parity_report

pytestmark = pytest.mark.gpu

SIZES = [0, 1, 7, 31, 32, 33, 63, 64, 65, 95, 96, 97, 127, 128, 129, 191, 192, 193, 223, 224,
         225, 255, 256, 257]
BLOCKWISE_TILES = ["cta1_96", "pair_192", "cta1_256", "pair_256", "pair_160", "pair_128",
                   "cta1_128", "cta1_96x192", "pair_192x192", "cta1_128x192", "pair_224",
                   "split"]
MX_FORMS = [("swap", "32"), ("swap", "64"), ("swap", "128"), ("pair", None), ("split", None)]


def _case(rng):
    E = int(rng.integers(1, 6))
    counts = [int(c) for c in rng.choice(SIZES, size=E)]
    if sum(counts) == 0:
        counts[0] = 1
    N = int(rng.choice([128, 256, 384, 640]))
    K = int(rng.choice([128, 256, 384, 640, 1024]))
    return counts, N, K


def _check(p):
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    d = DeviceProblem(p, c_rows_extra=2)
    d.run()
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    ref, T = oracle.problem_reference(p)
    bad, ratio, _ = parity_report(got, ref, T)
    assert bad == 0, f"{bad} elements outside tolerance (max err/tol {ratio:.3g})"
    assert np.all(d.guard_bits() == d.sentinel)


@pytest.mark.parametrize("seed", range(2 * len(BLOCKWISE_TILES)))
def test_blockwise_sweep(seed, monkeypatch):
    rng = np.random.default_rng(1000 + seed)
    counts, N, K = _case(rng)
    monkeypatch.setenv("BSFP8_BLOCKWISE_TILE", BLOCKWISE_TILES[seed % len(BLOCKWISE_TILES)])
    _check(gen.blockwise_problem(counts, N, K, seed=1000 + seed, exact=bool(seed % 2)))


@pytest.mark.parametrize("seed", range(2 * len(MX_FORMS)))
def test_mx_sweep(seed, monkeypatch):
    rng = np.random.default_rng(2000 + seed)
    counts, N, K = _case(rng)
    kernel, tn = MX_FORMS[seed % len(MX_FORMS)]
    monkeypatch.setenv("BSFP8_MX_KERNEL", kernel)
    if tn:
        monkeypatch.setenv("BSFP8_MX_TN", tn)
    _check(gen.mx_problem(counts, N, K, seed=2000 + seed, exact=bool(seed % 2)))


# (a format, b format, token tile, path): every pair on its fp4 MMA kind and on the converting
# kernels
FP4_FORMS = [(a, b, tn, path)
             for (a, b, path) in (("mxfp8", "mxfp4", "mma"), ("mxfp8", "mxfp4", "convert"),
                                  ("mxfp4", "mxfp4", "mma"),
                                  ("mxfp4", "mxfp4", "convert"), ("nvfp4", "nvfp4", "mma"),
                                  ("nvfp4", "nvfp4", "convert"))
             for tn in ("32", "64")]


@pytest.mark.parametrize("seed", range(2 * len(FP4_FORMS)))
def test_fp4_sweep(seed, monkeypatch):
    rng = np.random.default_rng(3000 + seed)
    counts, N, K = _case(rng)
    a_fmt, b_fmt, tn, path = FP4_FORMS[seed % len(FP4_FORMS)]
    monkeypatch.setenv("BSFP8_MX_TN", tn)
    monkeypatch.setenv("BSFP8_FP4_MMA", path)
    _check(gen.fmt_problem(counts, N, K, seed=3000 + seed, a_fmt=a_fmt, b_fmt=b_fmt,
                           a_recipe="quantized" if seed % 2 else "grid"))


@pytest.mark.parametrize("seed", range(12))
def test_fp4_pair_sweep(seed, monkeypatch):
    # the fp4 pairs with BSFP8_MX_KERNEL=pair: CTA-pair tiles where the form allows, the
    # swap-AB tiles otherwise
    rng = np.random.default_rng(4000 + seed)
    counts, N, K = _case(rng)
    a_fmt, b_fmt = (("mxfp8", "mxfp4"), ("mxfp4", "mxfp4"), ("nvfp4", "nvfp4"))[seed % 3]
    monkeypatch.setenv("BSFP8_MX_KERNEL", "pair")
    _check(gen.fmt_problem(counts, N, K, seed=4000 + seed, a_fmt=a_fmt, b_fmt=b_fmt,
                           a_recipe="quantized" if seed % 2 else "grid"))
