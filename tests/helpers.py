"""Test-side helpers: torch float64 brute force, exact bf16 rounding and the tolerance.

The brute force here is deliberately written differently from the oracle: operands are
decoded by torch's own float8 types, dequantized (value x scale, scales expanded over
their blocks) and multiplied with torch.matmul in float64 -- the reference construction
of make_problem in the Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix
Multiplication".  The acceptance bound is the workload's stated one:
|gpu - ref| <= 2 ulp_bf16(ref) + 1e-6 * sum|scaled terms|.
"""
from __future__ import annotations

import struct
from fractions import Fraction

import numpy as np
import torch


def decode_e4m3_torch(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)


def decode_ue8m0_torch(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e8m0fnu).to(torch.float64)


# The FP4 (E2M1) values of the OCP Microscaling formats, codes 0..7; codes 8..15 are the
# same values negated.  A literal table, not the oracle's bit-field formula.
E2M1_TABLE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                       -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], np.float64)


def unpack_fp4(Q: np.ndarray) -> np.ndarray:
    """e2m1 codes [..., 2*bytes] from packed bytes [..., bytes]: element 2i is the low
    nibble of byte i, element 2i+1 the high nibble."""
    Q = np.asarray(Q, np.uint8)
    out = np.empty(Q.shape[:-1] + (2 * Q.shape[-1],), np.uint8)
    out[..., 0::2] = Q & 0xF
    out[..., 1::2] = Q >> 4
    return out


def decode_operand(Q: np.ndarray, fmt: str) -> torch.Tensor:
    if fmt == "mxfp8":
        return decode_e4m3_torch(Q)
    return torch.from_numpy(E2M1_TABLE[unpack_fp4(Q)])


def decode_scales(S: np.ndarray, fmt: str) -> torch.Tensor:
    """Scales expanded over their K blocks (32 for mxfp8 / mxfp4, 16 for nvfp4)."""
    if fmt == "nvfp4":
        return decode_e4m3_torch(S).repeat_interleave(16, dim=-1)
    return decode_ue8m0_torch(S).repeat_interleave(32, dim=-1)


def dequantize(p):
    """(A_deq [M,K], B_deq [E,N,K]) in float64 for a gen.Problem."""
    a_fmt, b_fmt = getattr(p, "a_fmt", "mxfp8"), getattr(p, "b_fmt", "mxfp8")
    if p.mode == "mx" and (a_fmt, b_fmt) != ("mxfp8", "mxfp8"):
        A = decode_operand(p.A, a_fmt) * decode_scales(p.a_scales, a_fmt)
        B = decode_operand(p.B, b_fmt) * decode_scales(p.b_scales, b_fmt)
        return A, B
    A = decode_e4m3_torch(p.A)
    B = decode_e4m3_torch(p.B)
    if p.mode == "blockwise":
        sa = torch.from_numpy(p.a_scales).to(torch.float64)            # [K/128, M]
        A = A * sa.t().repeat_interleave(128, dim=1)
        sb = torch.from_numpy(p.b_scales).to(torch.float64)            # [E, N/128, K/128]
        B = B * sb.repeat_interleave(128, dim=1).repeat_interleave(128, dim=2)
    else:
        A = A * decode_ue8m0_torch(p.a_scales).repeat_interleave(32, dim=1)   # [M, K/32]
        B = B * decode_ue8m0_torch(p.b_scales).repeat_interleave(32, dim=2)   # [E, N, K/32]
    return A, B


def brute_force(p):
    """(C float64 [M,N], T float64 [M,N]) by dequantized matmul per group (group e uses
    expert expert_ids[e] when the problem has expert ids, else expert e)."""
    A, B = dequantize(p)
    M, N = p.M_total, p.N
    C = torch.zeros(M, N, dtype=torch.float64)
    T = torch.zeros(M, N, dtype=torch.float64)
    off = p.offsets
    ids = getattr(p, "expert_ids", None)
    for e in range(p.E):
        r0, r1 = int(off[e]), int(off[e + 1])
        x = int(ids[e]) if ids is not None else e
        if r1 > r0:
            C[r0:r1] = A[r0:r1] @ B[x].t()
            T[r0:r1] = A[r0:r1].abs() @ B[x].abs().t()
    return C.numpy(), T.numpy()


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def bf16_exact_round(v) -> int:
    """Round an exact rational (or float) to bf16 bits, RNE, with exact arithmetic."""
    v = Fraction(v)
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    E = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** E > a:
        E -= 1
    if Fraction(2) ** (E + 1) <= a:
        E += 1
    E = max(E, -126)
    q = Fraction(2) ** (E - 7)
    r = a / q
    fl = r.numerator // r.denominator
    rem = r - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = fl * q
    if val >= Fraction(2) ** 128:
        return sign | 0x7F80
    return sign | (f32_bits(float(val)) >> 16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    bits = np.asarray(bits, np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_bf16(ref_vals: np.ndarray) -> np.ndarray:
    """2^(max(floor(log2|x|), -126) - 7); 2^-133 at zero."""
    a = np.abs(np.asarray(ref_vals, np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -126), -126)
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def tolerance(ref_bits: np.ndarray, T: np.ndarray) -> np.ndarray:
    return 2.0 * ulp_bf16(bf16_bits_to_f64(ref_bits)) + 1e-6 * np.asarray(T, np.float64)


def parity_report(got_bits: np.ndarray, ref_bits: np.ndarray, T: np.ndarray):
    """(n_bad, max_err/tol, n_exact) for bf16 outputs against the oracle."""
    got = bf16_bits_to_f64(got_bits)
    ref = bf16_bits_to_f64(ref_bits)
    tol = tolerance(ref_bits, T)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    ratio = float(np.max(err / tol)) if err.size else 0.0
    return int(bad.sum()), ratio, int((np.asarray(got_bits) == np.asarray(ref_bits)).sum())


def parity_report_chunked(got_bits: np.ndarray, ref_bits: np.ndarray, T: np.ndarray,
                          rows_per_chunk: int = 2048):
    """parity_report over row chunks (the full-size outputs hold up to 67 M elements):
    (n_bad, max_err/tol, n_exact)."""
    bad, ratio, exact = 0, 0.0, 0
    for r0 in range(0, got_bits.shape[0], rows_per_chunk):
        b, q, x = parity_report(got_bits[r0:r0 + rows_per_chunk], ref_bits[r0:r0 + rows_per_chunk],
                                T[r0:r0 + rows_per_chunk])
        bad, ratio, exact = bad + b, max(ratio, q), exact + x
    return bad, ratio, exact
