"""CPU oracle for the blockwise-scaled FP8 grouped GEMM -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its Python
binding) never does, and this package never imports the product.  It shares no code
with the CUDA kernels.

The arithmetic lives in ``bsfp8_oracle.cpp`` (plain C++, fp64); see its header for the
definition it writes out and the page passages it follows:

  * promote_accumulators (MAX kernels, linalg/grouped_matmul_sm100_blockwise_fp8):
    per-K-block partials times (A scale x B scale), accumulated in fp32 tiles;
    b_scales [num_experts, N // BN, K // BK].
  * Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix Multiplication",
    make_problem / random_quantized_tensor: the block-scaled result is the matmul of the
    dequantized operands (UE8M0 scales repeated over 32 K elements).

Parity pins (tests/test_oracle_pins.py) tie it to the e4m3 closed form, torch's own
float8 decode, brute force, exact power-of-two linearity, per-expert concatenation and
the exact-arithmetic inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsfp8_oracle.cpp")
_LIB = os.path.join(_HERE, "libbsfp8_oracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/libbsfp8_oracle.so (skipped when up to date)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-ffp-contract=off", "-std=c++17", "-shared",
                               "-fPIC", "-pthread", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.bsfp8_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.bsfp8_oracle_e4m3_decode.restype = ctypes.c_double
        lib.bsfp8_oracle_ue8m0_decode.argtypes = [ctypes.c_uint8]
        lib.bsfp8_oracle_ue8m0_decode.restype = ctypes.c_double
        lib.bsfp8_oracle_bf16_rne.argtypes = [ctypes.c_double]
        lib.bsfp8_oracle_bf16_rne.restype = ctypes.c_uint16
        for name in ("bsfp8_oracle_blockwise", "bsfp8_oracle_mx"):
            f = getattr(lib, name)
            f.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, p, i32]
            f.restype = i32
        for name in ("bsfp8_oracle_blockwise_points", "bsfp8_oracle_mx_points"):
            f = getattr(lib, name)
            f.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, p, i64, p, p, i32]
            f.restype = i32
        lib.bsfp8_oracle_ids.argtypes = [i32, p, p, p, p, p, p, i64, i64, i64, i64, i64, p, p, i32]
        lib.bsfp8_oracle_ids.restype = i32
        lib.bsfp8_oracle_fmt.argtypes = [i32, i32, p, p, p, p, p, p, i64, i64, i64, i64, i64,
                                         p, p, i32]
        lib.bsfp8_oracle_fmt.restype = i32
        lib.bsfp8_oracle_fmt_points.argtypes = [i32, i32, p, p, p, p, p, p, i64, i64, i64, i64,
                                                i64, p, p, i64, p, p, i32]
        lib.bsfp8_oracle_fmt_points.restype = i32
        lib.bsfp8_oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.bsfp8_oracle_e2m1_decode.restype = ctypes.c_double
        lib.bsfp8_oracle_threads.argtypes = [i32]
        lib.bsfp8_oracle_threads.restype = i32
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def e4m3_decode(code: int) -> float:
    return float(_L().bsfp8_oracle_e4m3_decode(code))


def ue8m0_decode(code: int) -> float:
    return float(_L().bsfp8_oracle_ue8m0_decode(code))


def e2m1_decode(nibble: int) -> float:
    return float(_L().bsfp8_oracle_e2m1_decode(nibble))


def bf16_rne(x: float) -> int:
    return int(_L().bsfp8_oracle_bf16_rne(float(x)))


def threads(n: int = 0) -> int:
    return int(_L().bsfp8_oracle_threads(n))


def _args(mode, A, B, a_scales, b_scales, offsets):
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    if mode == "blockwise":
        a_scales = _c(a_scales, np.float32)
        b_scales = _c(b_scales, np.float32)
    elif mode == "mx":
        a_scales = _c(a_scales, np.uint8)
        b_scales = _c(b_scales, np.uint8)
    else:
        raise ValueError(mode)
    offsets = _c(offsets, np.int32)
    return A, B, a_scales, b_scales, offsets


def grouped_gemm(mode: str, A, B, a_scales, b_scales, offsets, N: int, K: int,
                 nthreads: int = 0, want_t: bool = True):
    """Full output.  Returns (C as bf16 bit patterns uint16 [M_total, N], T float64 or None)."""
    A, B, a_scales, b_scales, offsets = _args(mode, A, B, a_scales, b_scales, offsets)
    E = offsets.shape[0] - 1
    M = int(offsets[-1])
    C = np.empty((M, N), np.uint16)
    T = np.empty((M, N), np.float64) if want_t else None
    f = _L().bsfp8_oracle_blockwise if mode == "blockwise" else _L().bsfp8_oracle_mx
    rc = f(A.ctypes.data, B.ctypes.data, a_scales.ctypes.data, b_scales.ctypes.data,
           offsets.ctypes.data, M, N, K, E, C.ctypes.data,
           T.ctypes.data if T is not None else None, nthreads)
    if rc:
        raise OracleError(f"oracle rejected the problem (code {rc})")
    return C, T


def grouped_gemm_ids(mode: str, A, B, a_scales, b_scales, offsets, expert_ids, N: int, K: int,
                     nthreads: int = 0, want_t: bool = True):
    """Full output with an expert indirection: group g (rows offsets[g]..offsets[g+1]-1)
    uses expert expert_ids[g] of B [num_experts, N, K].  Returns (C bits, T or None)."""
    A, B, a_scales, b_scales, offsets = _args(mode, A, B, a_scales, b_scales, offsets)
    ids = _c(expert_ids, np.int32)
    G = offsets.shape[0] - 1
    assert ids.shape == (G,)
    M = int(offsets[-1])
    C = np.empty((M, N), np.uint16)
    T = np.empty((M, N), np.float64) if want_t else None
    rc = _L().bsfp8_oracle_ids(0 if mode == "blockwise" else 1, A.ctypes.data, B.ctypes.data,
                               a_scales.ctypes.data, b_scales.ctypes.data, offsets.ctypes.data,
                               ids.ctypes.data, M, N, K, G, B.shape[0], C.ctypes.data,
                               T.ctypes.data if T is not None else None, nthreads)
    if rc:
        raise OracleError(f"oracle rejected the problem (code {rc})")
    return C, T


def grouped_gemm_points(mode: str, A, B, a_scales, b_scales, offsets, N: int, K: int,
                        rows, cols, nthreads: int = 0):
    """Sampled output elements (rows[i], cols[i]).  Returns (C bits uint16 [n], T float64 [n])."""
    A, B, a_scales, b_scales, offsets = _args(mode, A, B, a_scales, b_scales, offsets)
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    assert rows.shape == cols.shape
    E = offsets.shape[0] - 1
    M = int(offsets[-1])
    C = np.empty(rows.shape, np.uint16)
    T = np.empty(rows.shape, np.float64)
    f = _L().bsfp8_oracle_blockwise_points if mode == "blockwise" else _L().bsfp8_oracle_mx_points
    rc = f(A.ctypes.data, B.ctypes.data, a_scales.ctypes.data, b_scales.ctypes.data,
           offsets.ctypes.data, M, N, K, E, rows.ctypes.data, cols.ctypes.data, rows.size,
           C.ctypes.data, T.ctypes.data, nthreads)
    if rc:
        raise OracleError(f"oracle rejected the problem (code {rc})")
    return C, T


FORMATS = {"mxfp8": 0, "mxfp4": 1, "nvfp4": 2}


def _fmt_args(a_fmt, b_fmt, A, B, a_scales, b_scales, offsets, expert_ids):
    A, B = _c(A, np.uint8), _c(B, np.uint8)
    a_scales, b_scales = _c(a_scales, np.uint8), _c(b_scales, np.uint8)
    offsets = _c(offsets, np.int32)
    ids = None if expert_ids is None else _c(expert_ids, np.int32)
    G = offsets.shape[0] - 1
    assert ids is None or ids.shape == (G,)
    return FORMATS[a_fmt], FORMATS[b_fmt], A, B, a_scales, b_scales, offsets, ids, G


def grouped_gemm_fmt(a_fmt: str, b_fmt: str, A, B, a_scales, b_scales, offsets, N: int, K: int,
                     expert_ids=None, nthreads: int = 0, want_t: bool = True):
    """Block-scaled grouped GEMM with a format per operand ("mxfp8", "mxfp4", "nvfp4").
    fp4 operands are packed two elements per byte along K (A [M_total, K/2], B [E, N, K/2]);
    scales are [rows, K/32] UE8M0 (mx formats) or [rows, K/16] e4m3 codes (nvfp4).  Group g
    uses expert expert_ids[g] of B, or expert g when expert_ids is None.
    Returns (C bits uint16 [M_total, N], T float64 or None)."""
    fa, fb, A, B, a_scales, b_scales, offsets, ids, G = _fmt_args(
        a_fmt, b_fmt, A, B, a_scales, b_scales, offsets, expert_ids)
    M = int(offsets[-1])
    C = np.empty((M, N), np.uint16)
    T = np.empty((M, N), np.float64) if want_t else None
    rc = _L().bsfp8_oracle_fmt(fa, fb, A.ctypes.data, B.ctypes.data, a_scales.ctypes.data,
                               b_scales.ctypes.data, offsets.ctypes.data,
                               ids.ctypes.data if ids is not None else None, M, N, K, G,
                               B.shape[0], C.ctypes.data,
                               T.ctypes.data if T is not None else None, nthreads)
    if rc:
        raise OracleError(f"oracle rejected the problem (code {rc})")
    return C, T


def grouped_gemm_fmt_points(a_fmt: str, b_fmt: str, A, B, a_scales, b_scales, offsets, N: int,
                            K: int, rows, cols, expert_ids=None, nthreads: int = 0):
    """Sampled elements of grouped_gemm_fmt.  Returns (C bits [n], T float64 [n])."""
    fa, fb, A, B, a_scales, b_scales, offsets, ids, G = _fmt_args(
        a_fmt, b_fmt, A, B, a_scales, b_scales, offsets, expert_ids)
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    assert rows.shape == cols.shape
    M = int(offsets[-1])
    C = np.empty(rows.shape, np.uint16)
    T = np.empty(rows.shape, np.float64)
    rc = _L().bsfp8_oracle_fmt_points(fa, fb, A.ctypes.data, B.ctypes.data, a_scales.ctypes.data,
                                      b_scales.ctypes.data, offsets.ctypes.data,
                                      ids.ctypes.data if ids is not None else None, M, N, K, G,
                                      B.shape[0], rows.ctypes.data, cols.ctypes.data, rows.size,
                                      C.ctypes.data, T.ctypes.data, nthreads)
    if rc:
        raise OracleError(f"oracle rejected the problem (code {rc})")
    return C, T


def _formats(p):
    return getattr(p, "a_fmt", "mxfp8"), getattr(p, "b_fmt", "mxfp8")


def problem_reference(p, nthreads: int = 0, want_t: bool = True):
    """Full oracle output for a gen.Problem-like object (mode, A, B, scales, offsets, N, K,
    and expert_ids / operand formats when it has them)."""
    if p.mode == "mx" and _formats(p) != ("mxfp8", "mxfp8"):
        return grouped_gemm_fmt(*_formats(p), p.A, p.B, p.a_scales, p.b_scales, p.offsets, p.N,
                                p.K, expert_ids=getattr(p, "expert_ids", None),
                                nthreads=nthreads, want_t=want_t)
    if getattr(p, "expert_ids", None) is not None:
        return grouped_gemm_ids(p.mode, p.A, p.B, p.a_scales, p.b_scales, p.offsets,
                                p.expert_ids, p.N, p.K, nthreads=nthreads, want_t=want_t)
    return grouped_gemm(p.mode, p.A, p.B, p.a_scales, p.b_scales, p.offsets, p.N, p.K,
                        nthreads=nthreads, want_t=want_t)


def problem_points(p, rows, cols, nthreads: int = 0):
    if p.mode == "mx" and (_formats(p) != ("mxfp8", "mxfp8") or
                           getattr(p, "expert_ids", None) is not None):
        return grouped_gemm_fmt_points(*_formats(p), p.A, p.B, p.a_scales, p.b_scales,
                                       p.offsets, p.N, p.K, rows, cols,
                                       expert_ids=getattr(p, "expert_ids", None),
                                       nthreads=nthreads)
    return grouped_gemm_points(p.mode, p.A, p.B, p.a_scales, p.b_scales, p.offsets, p.N, p.K,
                               rows, cols, nthreads=nthreads)


def timed_rows(p, row_count: int, nthreads: int = 0, keep: bool = False):
    """Time the oracle on row_count rows spread evenly over the workload, every column (a
    bounded sample).  Returns (seconds, flops_done, threads_used); with keep, a fourth item
    (row indices, bf16 bits [rows, N], the bound T [rows, N]) holds the sample's results."""
    M = p.M_total
    rows_sel = np.linspace(0, M - 1, num=min(row_count, M)).astype(np.int64)
    rows = np.repeat(rows_sel, p.N)
    cols = np.tile(np.arange(p.N, dtype=np.int64), rows_sel.size)
    t0 = time.perf_counter()
    ref, T = problem_points(p, rows, cols, nthreads=nthreads)
    dt = time.perf_counter() - t0
    out = (dt, 2.0 * rows.size * p.K, threads(nthreads))
    if keep:
        n = rows_sel.size
        return out + ((rows_sel, np.asarray(ref).reshape(n, p.N), np.asarray(T).reshape(n, p.N)),)
    return out


def pack_mx_scales(S) -> np.ndarray:
    """UE8M0 scales [rows, cols] in the tensor core's 128-row packed block layout, as
    swizzle_scales_packed_block of the Triton Gluon example "Overlapping Accumulator
    Block-Scaled Matrix Multiplication" builds it: zero-pad rows to a multiple of 128 and
    columns to a multiple of 4, view as (rows/128, 4, 32, cols/4, 4), swap axes 1 and 3
    (permute (0, 3, 2, 1, 4)), flatten.  For weight scales [E, N, K/32] pass them reshaped
    to [E*N, K/32]: the result is [E][N/128][K/128] blocks of 512 bytes."""
    S = np.asarray(S, np.uint8)
    R, SK = S.shape
    Rp, SKp = -(-R // 128) * 128, -(-SK // 4) * 4
    P = np.zeros((Rp, SKp), np.uint8)
    P[:R, :SK] = S
    return np.ascontiguousarray(
        P.reshape(Rp // 128, 4, 32, SKp // 4, 4).transpose(0, 3, 2, 1, 4)).reshape(-1)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    bits = np.asarray(bits, np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
