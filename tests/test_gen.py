"""The input generator: determinism, the quantizer rules, and the workload recipes."""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import decode_e4m3_torch


def test_normals_deterministic_and_standard():
    a = gen.normals(123, 1, 0, 200000)
    b = gen.normals(123, 1, 0, 200000)
    assert np.array_equal(a, b)
    # any window equals the same slice of a longer draw (counter based)
    assert np.array_equal(gen.normals(123, 1, 777, 1001), a[777:1778])
    assert abs(float(a.mean())) < 0.01 and abs(float(a.std()) - 1.0) < 0.01
    assert not np.array_equal(gen.normals(124, 1, 0, 1000), a[:1000])
    assert not np.array_equal(gen.normals(123, 2, 0, 1000), a[:1000])


def test_own_log_exp():
    for x in [1e-300, 1e-20, 0.001, 0.3, 0.5, 0.7071, 1.0, 1.5, 2.0, 123.456, 1e200]:
        assert abs(gen.gen_log(x) - math.log(x)) <= 4e-16 * max(1.0, abs(math.log(x)))
    for x in [-50.0, -1.3, 0.0, 0.2, 1.0, 7.7, 40.0]:
        assert abs(gen.gen_exp(x) - math.exp(x)) <= 4e-15 * math.exp(x)


def test_e4m3_encode_round_trip_every_finite_code():
    vals = decode_e4m3_torch(np.arange(256, dtype=np.uint8)).numpy()
    for c in range(256):
        if math.isnan(vals[c]):
            continue
        assert gen.e4m3_encode(float(vals[c])) == c, c


def test_e4m3_encode_matches_torch_below_saturation():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(size=20000) * s for s in (0.001, 0.1, 1.0, 30.0, 200.0)])
    x = x[np.abs(x) < 464].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([gen.e4m3_encode(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_ties_and_saturation():
    # halfway between 1.0 (M=0) and 1.125 (M=1) -> even (1.0); between 1.125 and 1.25 -> 1.25
    assert gen.e4m3_encode(1.0625) == 0x38
    assert gen.e4m3_encode(1.1875) == 0x3A
    assert gen.e4m3_encode(464.0) == 0x7E and gen.e4m3_encode(500.0) == 0x7E
    assert gen.e4m3_encode(1e30) == 0x7E and gen.e4m3_encode(-1e30) == 0xFE
    assert gen.e4m3_encode(float("inf")) == 0x7E
    assert gen.e4m3_encode(2.0 ** -10) == 0x00        # tie between 0 and 2^-9 -> 0
    assert gen.e4m3_encode(3 * 2.0 ** -10) == 0x02    # tie between 2^-9 and 2^-8 -> even


def test_ceil_log2():
    for r in [1.0, 0.5, 0.75, 3.0, 4.0, 4.0001, 2.0 ** -126, 1e-3]:
        expect = math.ceil(math.log2(float(np.float32(r))))
        if float(np.float32(r)) == 2.0 ** round(math.log2(float(np.float32(r)))):
            expect = round(math.log2(float(np.float32(r))))
        assert gen.ceil_log2(r) == expect, r


def test_blockwise_quantizer_rules():
    p = gen.blockwise_problem([7, 0, 9], 256, 384, seed=3)
    dA = decode_e4m3_torch(p.A).numpy()
    src = gen.normals(3, gen.STREAM_A, 0, p.M_total * p.K).reshape(p.M_total, p.K)
    for m in range(p.M_total):
        for kb in range(p.K // 128):
            x = src[m, kb * 128:(kb + 1) * 128]
            s = np.float32(np.max(np.abs(x))) / np.float32(448.0)
            assert p.a_scales[kb, m] == s
            q = dA[m, kb * 128:(kb + 1) * 128]
            assert np.max(np.abs(q)) == 448.0
            # each code is the e4m3 RNE of x/s: within half an e4m3 step of x/s
            np.testing.assert_allclose(q, (x / s).astype(np.float64), rtol=2 ** -4, atol=2 ** -10)
    dB = decode_e4m3_torch(p.B).numpy()
    for e in range(3):
        for nb in range(2):
            for kb in range(3):
                blk = dB[e, nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
                assert np.max(np.abs(blk)) == 448.0
                assert p.b_scales[e, nb, kb] > 0


def test_mx_quantizer_rules():
    p = gen.mx_problem([5, 3], 64, 256, seed=4)
    src = gen.normals(4, gen.STREAM_A, 0, p.M_total * p.K).reshape(p.M_total, p.K)
    for m in range(p.M_total):
        for sb in range(p.K // 32):
            amax = np.float32(np.max(np.abs(src[m, sb * 32:(sb + 1) * 32])))
            r = float(amax / np.float32(448.0))
            e = int(p.a_scales[m, sb]) - 127
            assert 2.0 ** e >= r and 2.0 ** (e - 1) < r


def test_exact_inputs_are_on_the_grid():
    p = gen.blockwise_problem([10, 20], 128, 256, seed=5, exact=True)
    vals = set(np.unique(np.abs(decode_e4m3_torch(p.A).numpy())).tolist())
    assert vals <= {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}
    assert set(np.unique(p.a_scales).tolist()) <= {0.5, 1.0, 2.0}
    q = gen.mx_problem([10, 20], 128, 256, seed=5, exact=True)
    assert set(np.unique(q.b_scales).tolist()) <= {126, 127, 128}


def test_thread_count_does_not_change_bytes():
    a = gen.blockwise_problem([33, 40], 256, 512, seed=21, nthreads=1)
    b = gen.blockwise_problem([33, 40], 256, 512, seed=21, nthreads=5)
    for f in ("A", "B", "a_scales", "b_scales"):
        assert np.array_equal(getattr(a, f), getattr(b, f))


def test_config_routing_recipes():
    c1 = gen.config_counts(1)
    assert c1.sum() == 4096 and len(c1) == 8 and c1.min() > 300
    c2 = gen.config_counts(2)
    assert c2.sum() == 16384 and len(c2) == 64
    assert (c2 == 0).sum() >= 2 and c2.max() > 2000
    c4 = gen.config_counts(4)
    assert len(c4) == 128 and c4.min() >= 1 and c4.max() <= 32
    assert 1800 <= c4.sum() <= 2400
    m = gen.outlier_mask(2, 16384, 164)
    assert m.sum() == 164


def test_config0_problem_shapes():
    p = gen.config_problem(0)
    assert p.A.shape == (256, 512) and p.B.shape == (1, 256, 512)
    assert p.a_scales.shape == (4, 256) and p.b_scales.shape == (1, 2, 4)
    assert p.flops() == 2 * 256 * 256 * 512


@pytest.mark.parametrize("a_fmt,b_fmt", [("mxfp8", "mxfp4"), ("mxfp4", "mxfp4"),
                                         ("nvfp4", "nvfp4")])
def test_fmt_problem_layouts_and_ranges(a_fmt, b_fmt):
    p = gen.fmt_problem([3, 0, 9], 256, 384, seed=4, a_fmt=a_fmt, b_fmt=b_fmt)
    q = gen.fmt_problem([3, 0, 9], 256, 384, seed=4, a_fmt=a_fmt, b_fmt=b_fmt)
    assert np.array_equal(p.A, q.A) and np.array_equal(p.B, q.B)
    a_cols = 384 if a_fmt == "mxfp8" else 192
    assert p.A.shape == (12, a_cols) and p.B.shape == (3, 256, 192)
    vec = 16 if b_fmt == "nvfp4" else 32
    assert p.a_scales.shape == (12, 384 // vec) and p.b_scales.shape == (3, 256, 384 // vec)
    if b_fmt == "nvfp4":
        # powers of two 2^-7 .. 2 as e4m3 codes: 0x04 (subnormal 2^-7), then (j + 7) << 3
        assert set(np.unique(p.b_scales)) <= {0x04} | {(j + 7) << 3 for j in range(-6, 2)}
    else:
        assert p.b_scales.min() >= 120 and p.b_scales.max() <= 128
    # every nibble value occurs (uniform codes)
    nib = np.concatenate([(p.B & 0xF).ravel(), (p.B >> 4).ravel()])
    assert set(np.unique(nib)) == set(range(16))
    assert p.bytes() == p.A.nbytes + p.a_scales.nbytes + 2 * (p.B.nbytes // 3) + \
        2 * (p.b_scales.nbytes // 3) + 12 * 256 * 2


def test_fmt_problem_general_nvfp4_scales():
    p = gen.fmt_problem([5], 128, 256, seed=6, a_fmt="nvfp4", b_fmt="nvfp4", scales="e4m3")
    assert p.a_scales.min() >= 0x20 and p.a_scales.max() <= 0x47
    assert len(np.unique(p.a_scales)) > 20
