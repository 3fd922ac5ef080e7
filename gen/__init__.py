"""Seeded synthetic inputs for the blockwise-scaled FP8 grouped GEMM.

This package only makes inputs (quantized e4m3 operands, their scales and the
per-expert row offsets).  It holds none of the GEMM's arithmetic.  The oracle and
the CUDA library both consume what it returns; it imports neither of them.

The five standard workloads (``config_problem``) are:

  0  one expert, M=256, N=256, K=512, blockwise, seed 0
  1  8 experts, 4096 rows by uniform multinomial routing, N=4096, K=7168, blockwise
  2  64 experts, 16384 rows by Zipf(1.2) routing (4 lowest-weight experts emptied into
     the top one), 1% of rows scaled x50 before quantization, N=2048, K=7168, blockwise
  3  one expert, M=N=K=8192, blockwise (the 256x256 CTA-pair tile workload)
  4  128 experts with U{1..32} rows each, N=4096, K=7168, MXFP8 (UE8M0 per 32 K)

Config k uses seed k.  The quantization rules (amax/448 fp32 scales per 1x128 A block
and 128x128 B block; 2^ceil(log2(amax/448)) UE8M0 scales per 1x32 block) are those of
the workload descriptions; the exact-arithmetic variant follows the fp4-grid idea of
``random_quantized_tensor`` in the Triton Gluon example "Overlapping Accumulator
Block-Scaled Matrix Multiplication".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsfp8_gen.cpp")
_LIB = os.path.join(_HERE, "libbsfp8_gen.so")

STREAM_A, STREAM_B, STREAM_ROUTE, STREAM_OUTLIER = 1, 2, 3, 4
STREAM_A_EXACT, STREAM_B_EXACT, STREAM_SA_EXACT, STREAM_SB_EXACT = 5, 6, 7, 8


def build(force: bool = False) -> str:
    """Compile the generator into gen/libbsfp8_gen.so (skipped when up to date)."""
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
        u64, i64, i32, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.bsfp8_gen_normals.argtypes = [u64, u64, u64, u64, p]
        lib.bsfp8_gen_e4m3_encode.argtypes = [ctypes.c_float]
        lib.bsfp8_gen_e4m3_encode.restype = ctypes.c_uint8
        lib.bsfp8_gen_ceil_log2.argtypes = [ctypes.c_float]
        lib.bsfp8_gen_ceil_log2.restype = ctypes.c_int
        lib.bsfp8_gen_log.argtypes = [ctypes.c_double]
        lib.bsfp8_gen_log.restype = ctypes.c_double
        lib.bsfp8_gen_exp.argtypes = [ctypes.c_double]
        lib.bsfp8_gen_exp.restype = ctypes.c_double
        lib.bsfp8_gen_blockwise_rows.argtypes = [u64, u64, i64, i64, i64, p, p, p, i64, i32]
        lib.bsfp8_gen_blockwise_b.argtypes = [u64, u64, i64, i64, i64, p, p, i32]
        lib.bsfp8_gen_mx_rows.argtypes = [u64, u64, i64, i64, i64, p, p, p, i32]
        lib.bsfp8_gen_exact_codes.argtypes = [u64, u64, i64, p, i32]
        lib.bsfp8_gen_exact_scales_f32.argtypes = [u64, u64, i64, p]
        lib.bsfp8_gen_exact_scales_ue8m0.argtypes = [u64, u64, i64, p]
        lib.bsfp8_gen_fp4_bytes.argtypes = [u64, u64, i64, p, i32]
        lib.bsfp8_gen_pow2_scales.argtypes = [u64, u64, i64, i32, p, i32]
        lib.bsfp8_gen_e4m3_scale_codes.argtypes = [u64, u64, i64, i32, i32, p, i32]
        lib.bsfp8_gen_route_uniform.argtypes = [u64, i64, i64, p]
        lib.bsfp8_gen_route_zipf.argtypes = [u64, i64, i64, ctypes.c_double, i64, p]
        lib.bsfp8_gen_route_counts.argtypes = [u64, i64, i64, i64, p]
        lib.bsfp8_gen_outlier_rows.argtypes = [u64, i64, i64, p]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------------------
# primitives (exposed for the generator's own tests)
# ---------------------------------------------------------------------------
def normals(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, np.float32)
    _L().bsfp8_gen_normals(seed, stream, start, count, _ptr(out))
    return out


def e4m3_encode(x: float) -> int:
    return int(_L().bsfp8_gen_e4m3_encode(float(x)))


def ceil_log2(r: float) -> int:
    return int(_L().bsfp8_gen_ceil_log2(float(r)))


def gen_log(x: float) -> float:
    return float(_L().bsfp8_gen_log(x))


def gen_exp(x: float) -> float:
    return float(_L().bsfp8_gen_exp(x))


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------
def route_uniform(seed: int, M_total: int, E: int) -> np.ndarray:
    c = np.empty(E, np.int32)
    _L().bsfp8_gen_route_uniform(seed, M_total, E, _ptr(c))
    return c


def route_zipf(seed: int, M_total: int, E: int, s: float = 1.2, zero_lowest: int = 4) -> np.ndarray:
    c = np.empty(E, np.int32)
    _L().bsfp8_gen_route_zipf(seed, M_total, E, s, zero_lowest, _ptr(c))
    return c


def route_counts(seed: int, E: int, lo: int, hi: int) -> np.ndarray:
    c = np.empty(E, np.int32)
    _L().bsfp8_gen_route_counts(seed, E, lo, hi, _ptr(c))
    return c


def outlier_mask(seed: int, M_total: int, n_out: int) -> np.ndarray:
    m = np.empty(M_total, np.uint8)
    _L().bsfp8_gen_outlier_rows(seed, M_total, n_out, _ptr(m))
    return m


def counts_to_offsets(counts) -> np.ndarray:
    counts = np.asarray(counts, np.int64)
    off = np.zeros(len(counts) + 1, np.int32)
    off[1:] = np.cumsum(counts)
    return off


# ---------------------------------------------------------------------------
# problems
# ---------------------------------------------------------------------------
@dataclass
class Problem:
    """One grouped-GEMM input set, in the library's boundary layouts.

    blockwise: A u8 [M_total, K], B u8 [E, N, K], a_scales f32 [K/128, M_total],
               b_scales f32 [E, N/128, K/128]
    mx:        A, B as above, a_scales u8 [M_total, K/32], b_scales u8 [E, N, K/32]
               with operand formats a_fmt / b_fmt other than "mxfp8": an "mxfp4" or
               "nvfp4" operand holds e2m1 codes two per byte along K ([rows, K/2]); nvfp4
               scales are e4m3 codes per 16 K ([rows, K/16])
    offsets:   i32 [E+1], offsets[0] = 0, offsets[E] = M_total
    expert_ids: None (group e uses expert e; B has E experts), or i32 [E]: group e uses
               expert expert_ids[e] of the B.shape[0] experts in B
    """
    mode: str
    A: np.ndarray
    B: np.ndarray
    a_scales: np.ndarray
    b_scales: np.ndarray
    offsets: np.ndarray
    N: int
    K: int
    name: str = ""
    meta: dict = field(default_factory=dict)
    expert_ids: np.ndarray | None = None
    a_fmt: str = "mxfp8"
    b_fmt: str = "mxfp8"

    @property
    def num_experts(self) -> int:
        return int(self.B.shape[0])

    @property
    def E(self) -> int:
        return int(self.offsets.shape[0] - 1)

    @property
    def M_total(self) -> int:
        return int(self.offsets[-1])

    @property
    def counts(self) -> np.ndarray:
        return np.diff(self.offsets.astype(np.int64))

    def flops(self) -> float:
        """Algorithmic FLOPs: 2 * sum_e M_e * N * K (real rows only)."""
        return 2.0 * self.M_total * self.N * self.K

    def bytes(self) -> int:
        """Algorithmic bytes: A + B of experts with rows + scales + C, each once."""
        if self.expert_ids is None:
            active = int((self.counts > 0).sum())
        else:
            active = int(np.unique(self.expert_ids[self.counts > 0]).size)
        b = self.A.nbytes + active * (self.B.nbytes // self.num_experts) + self.a_scales.nbytes
        per_expert_sb = self.b_scales.nbytes // self.num_experts
        b += active * per_expert_sb + self.M_total * self.N * 2
        return int(b)


def blockwise_problem(counts, N: int, K: int, seed: int, outlier_rows: int = 0,
                      outlier_mult: float = 50.0, exact: bool = False, nthreads: int = 0,
                      name: str = "") -> Problem:
    counts = np.asarray(counts, np.int32)
    E = len(counts)
    off = counts_to_offsets(counts)
    M = int(off[-1])
    assert N % 128 == 0 and K % 128 == 0
    A = np.empty((M, K), np.uint8)
    B = np.empty((E, N, K), np.uint8)
    sa = np.empty((K // 128, M), np.float32)
    sb = np.empty((E, N // 128, K // 128), np.float32)
    L = _L()
    if exact:
        L.bsfp8_gen_exact_codes(seed, STREAM_A_EXACT, A.size, _ptr(A), nthreads)
        L.bsfp8_gen_exact_codes(seed, STREAM_B_EXACT, B.size, _ptr(B), nthreads)
        L.bsfp8_gen_exact_scales_f32(seed, STREAM_SA_EXACT, sa.size, _ptr(sa))
        L.bsfp8_gen_exact_scales_f32(seed, STREAM_SB_EXACT, sb.size, _ptr(sb))
    else:
        mult = None
        if outlier_rows:
            mask = outlier_mask(seed, M, outlier_rows)
            mult = np.where(mask == 1, np.float32(outlier_mult), np.float32(1.0)).astype(np.float32)
        if M:
            L.bsfp8_gen_blockwise_rows(seed, STREAM_A, 0, M, K, _ptr(mult), _ptr(A), _ptr(sa), M,
                                       nthreads)
        L.bsfp8_gen_blockwise_b(seed, STREAM_B, E, N, K, _ptr(B), _ptr(sb), nthreads)
    return Problem("blockwise", A, B, sa, sb, off, N, K, name=name,
                   meta={"seed": seed, "exact": exact, "outlier_rows": outlier_rows})


def mx_problem(counts, N: int, K: int, seed: int, exact: bool = False, nthreads: int = 0,
               name: str = "") -> Problem:
    counts = np.asarray(counts, np.int32)
    E = len(counts)
    off = counts_to_offsets(counts)
    M = int(off[-1])
    assert K % 32 == 0
    A = np.empty((M, K), np.uint8)
    B = np.empty((E, N, K), np.uint8)
    sa = np.empty((M, K // 32), np.uint8)
    sb = np.empty((E, N, K // 32), np.uint8)
    L = _L()
    if exact:
        L.bsfp8_gen_exact_codes(seed, STREAM_A_EXACT, A.size, _ptr(A), nthreads)
        L.bsfp8_gen_exact_codes(seed, STREAM_B_EXACT, B.size, _ptr(B), nthreads)
        L.bsfp8_gen_exact_scales_ue8m0(seed, STREAM_SA_EXACT, sa.size, _ptr(sa))
        L.bsfp8_gen_exact_scales_ue8m0(seed, STREAM_SB_EXACT, sb.size, _ptr(sb))
    else:
        if M:
            L.bsfp8_gen_mx_rows(seed, STREAM_A, 0, M, K, None, _ptr(A), _ptr(sa), nthreads)
        L.bsfp8_gen_mx_rows(seed, STREAM_B, 0, E * N, K, None, _ptr(B), _ptr(sb), nthreads)
    return Problem("mx", A, B, sa, sb, off, N, K, name=name,
                   meta={"seed": seed, "exact": exact})


STREAM_A_FP4, STREAM_B_FP4, STREAM_SA_FMT, STREAM_SB_FMT = 10, 11, 12, 13
FP4_FORMATS = ("mxfp8", "mxfp4", "nvfp4")


def _fmt_operand(fmt: str, rows: int, K: int, seed: int, s_elem: int, s_scale: int,
                 scales: str, exact_stream: int, nthreads: int):
    """One operand [rows, K] in format fmt, drawn as random_quantized_tensor draws it:
    fp4-grid values (random e2m1 codes; for mxfp8 the same grid stored as e4m3) and
    power-of-two scales in [1/128, 2] (scales="pow2"), or for nvfp4 general positive e4m3
    scale codes 0x20..0x47 (0.125 .. 3.75, scales="e4m3")."""
    L = _L()
    vec = 16 if fmt == "nvfp4" else 32
    if fmt == "mxfp8":
        Q = np.empty((rows, K), np.uint8)
        L.bsfp8_gen_exact_codes(seed, exact_stream, Q.size, _ptr(Q), nthreads)
    else:
        Q = np.empty((rows, K // 2), np.uint8)
        L.bsfp8_gen_fp4_bytes(seed, s_elem, Q.size, _ptr(Q), nthreads)
    S = np.empty((rows, K // vec), np.uint8)
    if fmt == "nvfp4" and scales == "e4m3":
        L.bsfp8_gen_e4m3_scale_codes(seed, s_scale, S.size, 0x20, 0x47, _ptr(S), nthreads)
    else:
        L.bsfp8_gen_pow2_scales(seed, s_scale, S.size, 1 if fmt == "nvfp4" else 0, _ptr(S),
                                nthreads)
    return Q, S


def fmt_problem(counts, N: int, K: int, seed: int, a_fmt: str, b_fmt: str,
                a_recipe: str = "grid", scales: str = "pow2", expert_ids=None,
                num_experts: int | None = None, nthreads: int = 0, name: str = "") -> Problem:
    """Block-scaled MX problem with a format per operand (the format pairs of the Gluon
    example: mxfp8 x mxfp8, mxfp8 x mxfp4, mxfp4 x mxfp4, nvfp4 x nvfp4).  Operands follow
    random_quantized_tensor (see _fmt_operand); a_recipe="quantized" instead draws an mxfp8 A
    as the decode workload does (N(0,1) rows, 2^ceil(log2(amax/448)) UE8M0 scales per 32).
    With expert_ids, group g uses expert expert_ids[g] of num_experts."""
    assert a_fmt in FP4_FORMATS and b_fmt in FP4_FORMATS
    counts = np.asarray(counts, np.int32)
    off = counts_to_offsets(counts)
    M = int(off[-1])
    E = len(counts) if expert_ids is None else int(num_experts)
    assert N % 128 == 0 and K % 128 == 0
    if a_fmt == "mxfp8" and a_recipe == "quantized":
        A = np.empty((M, K), np.uint8)
        sa = np.empty((M, K // 32), np.uint8)
        if M:
            _L().bsfp8_gen_mx_rows(seed, STREAM_A, 0, M, K, None, _ptr(A), _ptr(sa), nthreads)
    else:
        A, sa = _fmt_operand(a_fmt, M, K, seed, STREAM_A_FP4, STREAM_SA_FMT, scales,
                             STREAM_A_EXACT, nthreads)
    B, sb = _fmt_operand(b_fmt, E * N, K, seed, STREAM_B_FP4, STREAM_SB_FMT, scales,
                         STREAM_B_EXACT, nthreads)
    B = B.reshape(E, N, -1)
    sb = sb.reshape(E, N, -1)
    ids = None if expert_ids is None else np.asarray(expert_ids, np.int32)
    return Problem("mx", A, B, sa, sb, off, N, K, name=name,
                   meta={"seed": seed, "a_recipe": a_recipe, "scales": scales},
                   expert_ids=ids, a_fmt=a_fmt, b_fmt=b_fmt)


def routed_problem(counts, expert_ids, num_experts: int, N: int, K: int, seed: int,
                   mode: str = "blockwise", exact: bool = False, nthreads: int = 0,
                   name: str = "") -> Problem:
    """Rows in len(counts) groups, group g multiplying expert expert_ids[g] of num_experts:
    the rows (A and its scales) come from a problem with these group counts, the experts (B
    and its scales) from one with num_experts empty groups and another seed."""
    make = blockwise_problem if mode == "blockwise" else mx_problem
    ids = np.asarray(expert_ids, np.int32)
    assert ids.shape == (len(counts),)
    rows = make(counts, N, K, seed=seed, exact=exact, nthreads=nthreads)
    experts = make([0] * num_experts, N, K, seed=seed + 7919, exact=exact, nthreads=nthreads)
    return Problem(mode, rows.A, experts.B, rows.a_scales, experts.b_scales, rows.offsets, N, K,
                   name=name, meta={"seed": seed, "exact": exact}, expert_ids=ids)


CONFIG_NAMES = {
    0: "single-expert blockwise FP8, M=256 N=256 K=512",
    1: "grouped MoE blockwise FP8, E=8 M_total=4096 (uniform) N=4096 K=7168",
    2: "grouped MoE blockwise FP8 skewed, E=64 M_total=16384 (Zipf 1.2, 1% x50 outlier rows) N=2048 K=7168",
    3: "dense blockwise FP8, M=N=K=8192 (256x256 CTA-pair tiles)",
    4: "decode MXFP8 grouped, E=128 x U{1..32} rows, N=4096 K=7168, swap-AB",
    5: "extra workload (not one of the five above): dense MXFP8, M=N=K=8192",
}


def config_counts(idx: int) -> np.ndarray:
    if idx == 0:
        return np.array([256], np.int32)
    if idx == 1:
        return route_uniform(1, 4096, 8)
    if idx == 2:
        return route_zipf(2, 16384, 64, 1.2, 4)
    if idx == 3:
        return np.array([8192], np.int32)
    if idx == 4:
        return route_counts(4, 128, 1, 32)
    if idx == 5:
        return np.array([8192], np.int32)
    raise ValueError(idx)


CONFIG_SHAPES = {0: (256, 512), 1: (4096, 7168), 2: (2048, 7168), 3: (8192, 8192), 4: (4096, 7168),
                 5: (8192, 8192)}


def config_problem(idx: int, nthreads: int = 0) -> Problem:
    counts = config_counts(idx)
    N, K = CONFIG_SHAPES[idx]
    if idx in (4, 5):
        return mx_problem(counts, N, K, seed=idx, nthreads=nthreads, name=CONFIG_NAMES[idx])
    outliers = int(round(0.01 * int(counts.sum()))) if idx == 2 else 0
    return blockwise_problem(counts, N, K, seed=idx, outlier_rows=outliers, nthreads=nthreads,
                             name=CONFIG_NAMES[idx])
