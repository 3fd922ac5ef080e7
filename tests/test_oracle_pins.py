"""Pins for the CPU oracle: it is checked against facts that do not come from itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped K block, a wrong
sign or index, a transposed operand or scale, a wrong expert lookup, double rounding)
fails at least one of them:

  * every e4m3 / UE8M0 code against torch's own float8 decode and the OCP special values;
  * bf16 rounding against torch's fp32->bf16 and against exact rational rounding,
    including a case where rounding through fp32 first would give another answer;
  * unit scales: brute force (torch decode + float64 matmul; every sum is exact here);
  * non-unit scales: dequantize-then-matmul (the construction of make_problem in the
    Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix Multiplication");
    bitwise on exact-arithmetic inputs, within 0.5 ulp + 1e-12*T on N(0,1) inputs;
  * doubling one row's A scales doubles that row of C exactly;
  * the grouped result equals per-expert GEMMs concatenated, empty experts own no rows;
  * MX with every scale code 127 equals blockwise with every scale 1.0;
  * T equals |A_deq| @ |B_deq|^T;
  * expert ids (group -> expert, the expert_ids argument of promote_accumulators): the
    result equals the brute force run on the groups' gathered experts, identity ids give the
    plain grouped result, ids outside [0, num_experts) are rejected;
  * the packed scale layout: every byte at the position the closed form of the page's
    reshape/permute gives (written out as loops), including padded shapes, and the inverse
    view restores the input;
  * the fp4 formats (mxfp4, nvfp4; the format pairs of the Gluon example): all 16 e2m1
    codes against the literal FP4 value table, a hand-worked two-element case fixing the
    nibble order, dequantize-then-matmul bitwise for every format pair (general e4m3
    nvfp4 scales included), an mxfp4 operand re-encoded as e4m3 giving the mxfp8 result
    bit for bit, and the nvfp4 scale block being 16 wide (mxfp4: 32).
"""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import (E2M1_TABLE, bf16_bits_to_f64, bf16_exact_round, brute_force,
                     decode_e4m3_torch, decode_ue8m0_torch, f32_bits, ulp_bf16, unpack_fp4)


# ---------------------------------------------------------------------------
# encodings
# ---------------------------------------------------------------------------
def test_e4m3_all_256_codes_match_torch_decode():
    ref = decode_e4m3_torch(np.arange(256, dtype=np.uint8)).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), c


def test_e4m3_special_values():
    # OCP 8-bit FP spec, E4M3: max normal 448 = S.1111.110, min subnormal 2^-9,
    # min normal 2^-6, 1.0 = 0.0111.000, NaN = S.1111.111, no infinity.
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x3F) == 1.875
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    assert oracle.e4m3_decode(0x00) == 0.0
    assert math.copysign(1.0, oracle.e4m3_decode(0x80)) == -1.0
    finite = [oracle.e4m3_decode(c) for c in range(256) if not math.isnan(oracle.e4m3_decode(c))]
    assert len(finite) == 254 and max(finite) == 448.0


def test_ue8m0_all_256_codes():
    ref = decode_ue8m0_torch(np.arange(256, dtype=np.uint8)).numpy()
    for c in range(256):
        got = oracle.ue8m0_decode(c)
        if c == 255:
            assert math.isnan(got) and math.isnan(ref[c])
        else:
            assert got == ref[c] == 2.0 ** (c - 127), c


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------
def test_bf16_rne_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rne_hand_cases():
    one = 0x3F80
    assert oracle.bf16_rne(1.0) == one
    assert oracle.bf16_rne(1 + 2 ** -8) == one                    # tie -> even (down)
    assert oracle.bf16_rne(1 + 3 * 2 ** -8) == 0x3F82              # tie -> even (up)
    # direct rounding: just above the tie rounds up; via fp32 it would tie and go down
    x = 1 + 2 ** -8 + 2 ** -40
    assert oracle.bf16_rne(x) == 0x3F81
    assert float(np.float32(x)) == 1 + 2 ** -8                    # fp32 first would lose 2^-40
    assert oracle.bf16_rne(-2.5) == 0xC020
    assert oracle.bf16_rne(0.0) == 0x0000
    assert oracle.bf16_rne(-0.0) == 0x8000
    assert oracle.bf16_rne(2.0 ** -133) == 0x0001                  # min subnormal
    assert oracle.bf16_rne(2.0 ** -134) == 0x0000                  # tie to even (zero)
    assert oracle.bf16_rne(3 * 2.0 ** -134) == 0x0002              # tie to even (up)
    assert oracle.bf16_rne(2.0 ** 128) == 0x7F80
    assert oracle.bf16_rne((2 - 2 ** -8) * 2.0 ** 127) == 0x7F80   # rounds past max
    assert oracle.bf16_rne((2 - 2 ** -7) * 2.0 ** 127) == 0x7F7F   # max finite
    assert oracle.bf16_rne(float("inf")) == 0x7F80
    assert (oracle.bf16_rne(float("nan")) & 0x7F80) == 0x7F80


def test_bf16_rne_matches_exact_rational_rounding():
    rng = np.random.default_rng(1)
    for _ in range(3000):
        # doubles with many significant bits, across normal and subnormal bf16 ranges
        e = int(rng.integers(-140, 128))
        m = float(rng.random()) + 1.0
        x = math.ldexp(m, e) * (1 if rng.random() < 0.5 else -1)
        assert oracle.bf16_rne(x) == bf16_exact_round(x), x


# ---------------------------------------------------------------------------
# GEMM definition
# ---------------------------------------------------------------------------
def _oracle_vs_bruteforce(p, exact_bits: bool):
    C, T = oracle.problem_reference(p)
    Cb, Tb = brute_force(p)
    if exact_bits:
        ref = np.array([[bf16_exact_round(v) for v in row] for row in Cb], np.uint16)
        assert np.array_equal(C, ref)
    else:
        got = bf16_bits_to_f64(C)
        # exact value lies within 0.5 ulp of the oracle's bf16; the brute force differs
        # from the exact value by double rounding only
        assert np.all(np.abs(got - Cb) <= 0.5 * ulp_bf16(got) * (1 + 1e-9) + 1e-12 * Tb)
    np.testing.assert_allclose(T, Tb, rtol=1e-12, atol=0)
    return C, T


def test_unit_scales_equal_plain_gemm():
    # unit scales: the plain triple loop, every sum exact in double
    for (M, K) in [(1, 128), (5, 128), (8, 256)]:
        p = gen.blockwise_problem([M], 128, K, seed=11 + M)
        p.a_scales[:] = 1.0
        p.b_scales[:] = 1.0
        C, _ = oracle.problem_reference(p)
        dA = decode_e4m3_torch(p.A)
        dB = decode_e4m3_torch(p.B[0])
        ref = np.zeros((M, 128))
        for m in range(M):
            for n in range(128):
                ref[m, n] = float(sum(float(dA[m, k]) * float(dB[n, k]) for k in range(K)))
        assert np.array_equal(C, np.array([[bf16_exact_round(v) for v in r] for r in ref], np.uint16))


def test_blockwise_scales_exact_inputs_bitwise():
    # 3 experts (one empty), N/128 = 3 != K/128 = 5, so a transposed scale index cannot
    # line up; exact-arithmetic inputs make the result unique
    p = gen.blockwise_problem([37, 0, 130], 384, 640, seed=5, exact=True)
    _oracle_vs_bruteforce(p, exact_bits=True)


def test_blockwise_scales_random_inputs():
    p = gen.blockwise_problem([70, 0, 1, 58], 256, 384, seed=6)
    _oracle_vs_bruteforce(p, exact_bits=False)


def test_mx_scales_exact_inputs_bitwise():
    p = gen.mx_problem([3, 40, 0, 17], 64, 256, seed=7, exact=True)
    _oracle_vs_bruteforce(p, exact_bits=True)


def test_mx_scales_random_inputs():
    p = gen.mx_problem([9, 0, 33], 128, 384, seed=8)
    _oracle_vs_bruteforce(p, exact_bits=False)


def test_power_of_two_linearity_blockwise():
    p = gen.blockwise_problem([19, 45], 256, 512, seed=9)
    C0, T0 = oracle.problem_reference(p)
    m = 23
    p.a_scales[:, m] *= 2.0
    C1, T1 = oracle.problem_reference(p)
    v0, v1 = bf16_bits_to_f64(C0), bf16_bits_to_f64(C1)
    assert np.array_equal(v1[m], 2.0 * v0[m])
    assert np.array_equal(np.delete(C1, m, 0), np.delete(C0, m, 0))
    assert np.array_equal(T1[m], 2.0 * T0[m])


def test_power_of_two_linearity_mx():
    p = gen.mx_problem([12, 20], 128, 256, seed=10)
    C0, _ = oracle.problem_reference(p)
    m = 13
    p.a_scales[m, :] += 1
    C1, _ = oracle.problem_reference(p)
    assert np.array_equal(bf16_bits_to_f64(C1)[m], 2.0 * bf16_bits_to_f64(C0)[m])
    assert np.array_equal(np.delete(C1, m, 0), np.delete(C0, m, 0))


def test_grouped_equals_concatenated_per_expert():
    counts = [33, 0, 70, 0, 0, 5]
    p = gen.blockwise_problem(counts, 256, 384, seed=12)
    C, T = oracle.problem_reference(p)
    assert C.shape[0] == sum(counts)
    off = p.offsets
    for e in range(len(counts)):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        q = gen.Problem("blockwise", p.A[r0:r1].copy(), p.B[e:e + 1].copy(),
                        np.ascontiguousarray(p.a_scales[:, r0:r1]), p.b_scales[e:e + 1].copy(),
                        np.array([0, r1 - r0], np.int32), p.N, p.K)
        Ce, Te = oracle.problem_reference(q)
        assert np.array_equal(Ce, C[r0:r1])
        assert np.array_equal(Te, T[r0:r1])
    # an expert's B only reaches its own rows: perturb expert 2's weights
    p.B[2] ^= 0x01
    C2, _ = oracle.problem_reference(p)
    assert np.array_equal(C2[: off[2]], C[: off[2]]) and np.array_equal(C2[off[5]:], C[off[5]:])
    assert not np.array_equal(C2[off[2]:off[3]], C[off[2]:off[3]])


def test_cross_mode_unit_scales():
    p = gen.blockwise_problem([21, 0, 40], 256, 384, seed=13)
    p.a_scales[:] = 1.0
    p.b_scales[:] = 1.0
    Cb, Tb = oracle.problem_reference(p)
    q = gen.Problem("mx", p.A, p.B, np.full((p.M_total, p.K // 32), 127, np.uint8),
                    np.full((p.E, p.N, p.K // 32), 127, np.uint8), p.offsets, p.N, p.K)
    Cm, Tm = oracle.problem_reference(q)
    assert np.array_equal(Cb, Cm) and np.array_equal(Tb, Tm)


def test_points_match_full_output():
    p = gen.blockwise_problem([50, 0, 77], 256, 256, seed=14)
    C, T = oracle.problem_reference(p)
    rng = np.random.default_rng(3)
    rows = rng.integers(0, p.M_total, 300)
    cols = rng.integers(0, p.N, 300)
    Cp, Tp = oracle.problem_points(p, rows, cols)
    assert np.array_equal(Cp, C[rows, cols]) and np.array_equal(Tp, T[rows, cols])


def test_bad_offsets_rejected():
    p = gen.blockwise_problem([4, 4], 128, 128, seed=15)
    bad = np.array([0, 6, 5], np.int32)  # non-monotone, offsets[E] = 5
    with pytest.raises(oracle.OracleError):
        oracle.grouped_gemm("blockwise", p.A[:5], p.B, p.a_scales[:, :5].copy(), p.b_scales,
                            bad, p.N, p.K)
    bad2 = np.array([1, 4, 8], np.int32)  # offsets[0] != 0
    with pytest.raises(oracle.OracleError):
        oracle.grouped_gemm("blockwise", p.A, p.B, p.a_scales, p.b_scales, bad2, p.N, p.K)


def test_empty_problem():
    p = gen.blockwise_problem([0, 0], 128, 128, seed=16)
    C, T = oracle.problem_reference(p)
    assert C.shape == (0, 128)


# ---------------------------------------------------------------------------
# expert ids: group g multiplies expert expert_ids[g]
# ---------------------------------------------------------------------------
def test_expert_ids_blockwise_exact_bitwise():
    # 5 groups over 6 experts: expert 2 used twice, experts 4 and 5 never, one empty group
    p = gen.routed_problem([37, 0, 20, 130, 5], [2, 0, 2, 1, 3], 6, 384, 640, seed=21,
                           exact=True)
    C, _ = _oracle_vs_bruteforce(p, exact_bits=True)
    # ignoring the ids (group g -> expert g) gives a different result
    q = gen.Problem(p.mode, p.A, p.B[:5], p.a_scales, p.b_scales[:5], p.offsets, p.N, p.K)
    assert not np.array_equal(C, oracle.problem_reference(q)[0])


def test_expert_ids_blockwise_random_inputs():
    p = gen.routed_problem([64, 3, 0, 90], [3, 3, 0, 1], 4, 256, 512, seed=22)
    _oracle_vs_bruteforce(p, exact_bits=False)


def test_expert_ids_mx_exact_bitwise():
    p = gen.routed_problem([9, 40, 0, 17], [1, 0, 1, 2], 3, 64, 256, seed=23, mode="mx",
                           exact=True)
    _oracle_vs_bruteforce(p, exact_bits=True)


def test_expert_ids_identity_equals_plain_grouped():
    p = gen.blockwise_problem([30, 0, 70], 256, 384, seed=24)
    C0, T0 = oracle.problem_reference(p)
    C1, T1 = oracle.grouped_gemm_ids(p.mode, p.A, p.B, p.a_scales, p.b_scales, p.offsets,
                                     np.arange(3, dtype=np.int32), p.N, p.K)
    assert np.array_equal(C0, C1) and np.array_equal(T0, T1)


@pytest.mark.parametrize("bad", [-1, 4])
def test_expert_ids_out_of_range_rejected(bad):
    p = gen.routed_problem([8, 8], [0, 1], 4, 128, 128, seed=25)
    with pytest.raises(oracle.OracleError, match="code 8"):
        oracle.grouped_gemm_ids(p.mode, p.A, p.B, p.a_scales, p.b_scales, p.offsets,
                                np.array([0, bad], np.int32), p.N, p.K)


# ---------------------------------------------------------------------------
# packed scale-factor layout (swizzle_scales_packed_block of the Gluon example)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("R,SK", [(128, 4), (256, 12), (300, 7), (5, 1)])
def test_pack_mx_scales_element_formula(R, SK):
    rng = np.random.default_rng(R * 100 + SK)
    S = rng.integers(0, 256, size=(R, SK), dtype=np.uint8)
    P = oracle.pack_mx_scales(S)
    rep_mn, rep_k = -(-R // 128), -(-SK // 4)
    assert P.size == rep_mn * 128 * rep_k * 4
    for mb in range(rep_mn):
        for kq in range(rep_k):
            base = (mb * rep_k + kq) * 512
            for r in range(128):
                for j in range(4):
                    row, col = mb * 128 + r, kq * 4 + j
                    want = S[row, col] if (row < R and col < SK) else 0
                    assert P[base + (r % 32) * 16 + (r // 32) * 4 + j] == want


def test_pack_mx_scales_inverse_view():
    rng = np.random.default_rng(3)
    S = rng.integers(0, 256, size=(384, 8), dtype=np.uint8)
    P = oracle.pack_mx_scales(S)
    back = P.reshape(3, 2, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(384, 8)
    assert np.array_equal(back, S)


# ---------------------------------------------------------------------------
# fp4 formats (mxfp4, nvfp4)
# ---------------------------------------------------------------------------
def test_e2m1_all_16_codes():
    for c in range(16):
        v = oracle.e2m1_decode(c)
        assert v == E2M1_TABLE[c] and math.copysign(1.0, v) == math.copysign(1.0, E2M1_TABLE[c])


def test_fp4_nibble_order_hand_case():
    # A row 0: byte 0 = 0x21 -> element 0 = code 1 (0.5), element 1 = code 2 (1.0).
    # B row 0: byte 0 = 0x02 -> (1.0, 0); row 1: byte 0 = 0x20 -> (0, 1.0).  Unit scales.
    # So C[0,0] = 0.5 (bf16 0x3F00) and C[0,1] = 1.0 (0x3F80); every other element is 0.
    K, N = 128, 128
    A = np.zeros((1, K // 2), np.uint8)
    A[0, 0] = 0x21
    B = np.zeros((1, N, K // 2), np.uint8)
    B[0, 0, 0] = 0x02
    B[0, 1, 0] = 0x20
    sa = np.full((1, K // 32), 127, np.uint8)
    sb = np.full((1, N, K // 32), 127, np.uint8)
    off = np.array([0, 1], np.int32)
    C, _ = oracle.grouped_gemm_fmt("mxfp4", "mxfp4", A, B, sa, sb, off, N, K)
    assert C[0, 0] == 0x3F00 and C[0, 1] == 0x3F80
    assert not C[0, 2:].any()
    # the same through an nvfp4 view: unit e4m3 scales (code 0x38) per 16
    sa16 = np.full((1, K // 16), 0x38, np.uint8)
    sb16 = np.full((1, N, K // 16), 0x38, np.uint8)
    C2, _ = oracle.grouped_gemm_fmt("nvfp4", "nvfp4", A, B, sa16, sb16, off, N, K)
    assert np.array_equal(C, C2)


@pytest.mark.parametrize("a_fmt,b_fmt,scales", [("mxfp8", "mxfp4", "pow2"),
                                                ("mxfp4", "mxfp4", "pow2"),
                                                ("nvfp4", "nvfp4", "pow2"),
                                                ("nvfp4", "nvfp4", "e4m3"),
                                                ("mxfp8", "mxfp8", "pow2")])
def test_fmt_exact_inputs_bitwise(a_fmt, b_fmt, scales):
    # fp4-grid values with power-of-two or e4m3 scales: every product and sum is exact in
    # float64, so the brute force rounds to the one correct bf16 value
    p = gen.fmt_problem([5, 0, 21, 3], 256, 384, seed=31, a_fmt=a_fmt, b_fmt=b_fmt,
                        scales=scales)
    _oracle_vs_bruteforce(p, exact_bits=True)


def test_fmt_expert_ids_exact_bitwise():
    p = gen.fmt_problem([4, 9, 0, 2], 128, 256, seed=32, a_fmt="mxfp8", b_fmt="mxfp4",
                        expert_ids=[2, 0, 1, 2], num_experts=3)
    _oracle_vs_bruteforce(p, exact_bits=True)


def test_mxfp4_equals_mxfp8_reencoded():
    # every e2m1 value is an e4m3 value: re-encode the fp4 codes as e4m3 (the generator's
    # encoder, pinned on its own) and the mxfp8 path must give the same bits
    p = gen.fmt_problem([7, 30], 256, 512, seed=33, a_fmt="mxfp4", b_fmt="mxfp4")
    enc = np.array([gen.e4m3_encode(float(v)) for v in E2M1_TABLE], np.uint8)
    A8 = enc[unpack_fp4(p.A)]
    B8 = enc[unpack_fp4(p.B)]
    C4, T4 = oracle.problem_reference(p)
    C8, T8 = oracle.grouped_gemm("mx", A8, B8, p.a_scales, p.b_scales, p.offsets, p.N, p.K)
    assert np.array_equal(C4, C8)
    assert np.array_equal(T4, T8)
    C48, _ = oracle.grouped_gemm_fmt("mxfp8", "mxfp4", A8, p.B, p.a_scales, p.b_scales,
                                     p.offsets, p.N, p.K)
    assert np.array_equal(C4, C48)


@pytest.mark.parametrize("fmt,vec", [("nvfp4", 16), ("mxfp4", 32)])
def test_fp4_scale_block_width(fmt, vec):
    # only elements k in [16, 32) are non-zero in B: scale block 1 of nvfp4 covers them, block
    # 0 of mxfp4 does.  Doubling the scale of the block that covers them doubles C exactly;
    # changing any other block of that row leaves C unchanged.
    p = gen.fmt_problem([6], 128, 256, seed=34, a_fmt=fmt, b_fmt=fmt)
    p.B[:] = 0
    src = gen.fmt_problem([6], 128, 256, seed=35, a_fmt=fmt, b_fmt=fmt)
    p.B[..., 8:16] = src.B[..., 8:16]          # bytes 8..15 hold elements 16..31
    step = 8 if fmt == "nvfp4" else 1          # e4m3 code + 8 doubles a normal value
    blk = 16 // vec                            # the block holding element 16
    p.b_scales[:, :, blk] = 0x38 if fmt == "nvfp4" else 127   # 1.0 (normal)
    C0, _ = oracle.problem_reference(p)
    other = 3
    p.b_scales[:, :, other] += step
    C1, _ = oracle.problem_reference(p)
    assert np.array_equal(C1, C0)
    p.b_scales[:, :, blk] += step
    C2, _ = oracle.problem_reference(p)
    assert np.array_equal(bf16_bits_to_f64(C2), 2.0 * bf16_bits_to_f64(C0))
    assert np.any(C0 != 0)


def test_nvfp4_signed_and_subnormal_scales():
    # e4m3 scale codes of both signs over the whole finite range (subnormals included): the
    # oracle against dequantize-then-matmul (torch's float8 decode of the scales)
    rng = np.random.default_rng(36)
    p = gen.fmt_problem([6, 0, 11], 128, 256, seed=36, a_fmt="nvfp4", b_fmt="nvfp4")
    for sc in (p.a_scales, p.b_scales):
        sc[:] = (rng.integers(1, 0x7F, sc.shape) | (rng.integers(0, 2, sc.shape) << 7)).astype(np.uint8)
    _oracle_vs_bruteforce(p, exact_bits=False)
