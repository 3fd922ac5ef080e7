"""Python binding of the bsfp8 C ABI (include/bsfp8.h).

Argument marshalling only: every step of the GEMM runs in the CUDA library
``lib/libbsfp8.so``.  There is no fallback: if the library is missing or the device is
not a GB300 (compute capability 10.3) the calls raise.

    import block_scaled_fp8_persistent_gb300 as bsfp8
    bsfp8.bsfp8_grouped_gemm(A, B, a_scales, b_scales, expert_offsets, C,
                             M_total, N, K, num_experts, stream=None)
    bsfp8.bsmxfp8_grouped_gemm(...)   # MXFP8: UE8M0 scales per 32 K
    bsfp8.bsmx_grouped_gemm("mxfp8", "mxfp4", ...)   # a format per operand

Tensors are torch CUDA tensors (or raw device addresses as ints) in the layouts of
include/bsfp8.h; ``stream`` is a torch.cuda.Stream, a raw cudaStream_t int, or None for
torch's current stream.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
# The library: lib/libbsfp8.so, or the build named by BSFP8_LIBRARY (for example the
# bounds-checking lib/libbsfp8_debug.so that build.build(debug=True) makes).
LIB_PATH = os.environ.get("BSFP8_LIBRARY") or os.path.join(_PKG, "lib", "libbsfp8.so")

BSFP8_OK = 0
STATUS_NAMES = {
    0: "BSFP8_OK", 1: "BSFP8_ERR_NULL", 2: "BSFP8_ERR_SHAPE", 3: "BSFP8_ERR_ALIGN",
    4: "BSFP8_ERR_UNSUPPORTED_DEVICE", 5: "BSFP8_ERR_CUDA", 6: "BSFP8_ERR_DEVICE_OFFSETS",
    7: "BSFP8_ERR_DEVICE_TIMEOUT", 8: "BSFP8_ERR_DEVICE_EXPERT_IDS", 9: "BSFP8_ERR_FORMAT",
    10: "BSFP8_ERR_DEVICE_BOUNDS",
}

# bsmx_format values of include/bsfp8.h
FORMATS = {"mxfp8": 0, "mxfp4": 1, "nvfp4": 2}

# Every symbol include/bsfp8.h declares (the CPU test checks the library exports them).
EXPORTED = ("bsfp8_grouped_gemm", "bsmxfp8_grouped_gemm", "bsfp8_grouped_gemm_ids",
            "bsmxfp8_grouped_gemm_ids", "bsmxfp8_pack_b_scales", "bsmxfp8_grouped_gemm_prepacked",
            "bsmxfp8_tmem_plan", "bsfp8_blockwise_plan", "bsmxfp8_plan", "bsmx_plan",
            "bsmx_grouped_gemm", "bsfp8_get_device_error", "bsfp8_check_wait_timeout",
            "bsfp8_status_string")


class BsFp8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


_lib = None


def load_library() -> ctypes.CDLL:
    """Load lib/libbsfp8.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m block_scaled_fp8_persistent_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.bsfp8_grouped_gemm.argtypes = [p, p, p, p, p, p, i64, i32, i32, i32, p]
        lib.bsfp8_grouped_gemm.restype = i32
        lib.bsmxfp8_grouped_gemm.argtypes = [p, p, p, p, p, p, i64, i32, i32, i32, p]
        lib.bsmxfp8_grouped_gemm.restype = i32
        lib.bsfp8_grouped_gemm_ids.argtypes = [p, p, p, p, p, p, p, i64, i32, i32, i32, i32, p]
        lib.bsfp8_grouped_gemm_ids.restype = i32
        lib.bsmxfp8_grouped_gemm_ids.argtypes = [p, p, p, p, p, p, p, i64, i32, i32, i32, i32, p]
        lib.bsmxfp8_grouped_gemm_ids.restype = i32
        lib.bsmx_grouped_gemm.argtypes = [i32, i32, p, p, p, p, i32, p, p, p, i64, i32, i32,
                                          i32, i32, p]
        lib.bsmx_grouped_gemm.restype = i32
        lib.bsmxfp8_pack_b_scales.argtypes = [p, p, i32, i32, i32, p]
        lib.bsmxfp8_pack_b_scales.restype = i32
        lib.bsmxfp8_grouped_gemm_prepacked.argtypes = [p, p, p, p, p, p, i64, i32, i32, i32, p]
        lib.bsmxfp8_grouped_gemm_prepacked.restype = i32
        lib.bsmxfp8_tmem_plan.argtypes = [i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int32)]
        lib.bsmxfp8_tmem_plan.restype = i32
        lib.bsfp8_blockwise_plan.argtypes = [ctypes.c_int64, i32, i32, i32,
                                             ctypes.POINTER(ctypes.c_int32)]
        lib.bsfp8_blockwise_plan.restype = i32
        lib.bsmxfp8_plan.argtypes = [ctypes.c_int64, i32, ctypes.POINTER(ctypes.c_int32)]
        lib.bsmxfp8_plan.restype = i32
        lib.bsmx_plan.argtypes = [ctypes.c_int64, i32, ctypes.POINTER(ctypes.c_int32)]
        lib.bsmx_plan.restype = i32
        lib.bsfp8_get_device_error.argtypes = [p, ctypes.POINTER(ctypes.c_int)]
        lib.bsfp8_get_device_error.restype = i32
        lib.bsfp8_check_wait_timeout.argtypes = [ctypes.c_int64, p]
        lib.bsfp8_check_wait_timeout.restype = i32
        lib.bsfp8_status_string.argtypes = [i32]
        lib.bsfp8_status_string.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().bsfp8_status_string(int(status)).decode()


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("tensors must be CUDA tensors (device memory)")
    if not x.is_contiguous():
        raise ValueError("tensors must be contiguous (row-major)")
    return x.data_ptr() or None


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def bsfp8_grouped_gemm(A, B, a_scales, b_scales, expert_offsets, C, M_total: int, N: int,
                       K: int, num_experts: int, stream=None) -> None:
    """Blockwise FP8 grouped GEMM; see include/bsfp8.h for layouts.  Raises BsFp8Error."""
    st = load_library().bsfp8_grouped_gemm(_addr(A), _addr(B), _addr(a_scales), _addr(b_scales),
                                           _addr(expert_offsets), _addr(C), int(M_total), int(N),
                                           int(K), int(num_experts), _stream(stream))
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsfp8_grouped_gemm")


def bsmxfp8_grouped_gemm(A, B, a_scales, b_scales, expert_offsets, C, M_total: int, N: int,
                         K: int, num_experts: int, stream=None) -> None:
    """MXFP8 grouped GEMM (UE8M0 scales per 32 K); see include/bsfp8.h.  Raises BsFp8Error."""
    st = load_library().bsmxfp8_grouped_gemm(_addr(A), _addr(B), _addr(a_scales), _addr(b_scales),
                                             _addr(expert_offsets), _addr(C), int(M_total), int(N),
                                             int(K), int(num_experts), _stream(stream))
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsmxfp8_grouped_gemm")


def bsfp8_grouped_gemm_ids(A, B, a_scales, b_scales, group_offsets, expert_ids, C, M_total: int,
                           N: int, K: int, num_groups: int, num_experts: int, stream=None) -> None:
    """Blockwise FP8 grouped GEMM where group g uses expert expert_ids[g]'s weights; see
    include/bsfp8.h.  Raises BsFp8Error."""
    st = load_library().bsfp8_grouped_gemm_ids(
        _addr(A), _addr(B), _addr(a_scales), _addr(b_scales), _addr(group_offsets),
        _addr(expert_ids), _addr(C), int(M_total), int(N), int(K), int(num_groups),
        int(num_experts), _stream(stream))
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsfp8_grouped_gemm_ids")


def bsmxfp8_grouped_gemm_ids(A, B, a_scales, b_scales, group_offsets, expert_ids, C,
                             M_total: int, N: int, K: int, num_groups: int, num_experts: int,
                             stream=None) -> None:
    """MXFP8 grouped GEMM where group g uses expert expert_ids[g]'s weights; see
    include/bsfp8.h.  Raises BsFp8Error."""
    st = load_library().bsmxfp8_grouped_gemm_ids(
        _addr(A), _addr(B), _addr(a_scales), _addr(b_scales), _addr(group_offsets),
        _addr(expert_ids), _addr(C), int(M_total), int(N), int(K), int(num_groups),
        int(num_experts), _stream(stream))
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsmxfp8_grouped_gemm_ids")


def bsmx_grouped_gemm(a_format: str, b_format: str, A, B, a_scales, b_scales, group_offsets,
                      C, M_total: int, N: int, K: int, num_groups: int, num_experts: int,
                      expert_ids=None, b_scales_packed: bool = False, stream=None) -> None:
    """Block-scaled grouped GEMM with a format per operand ("mxfp8", "mxfp4", "nvfp4");
    see include/bsfp8.h.  expert_ids None: group g uses expert g.  Raises BsFp8Error."""
    st = load_library().bsmx_grouped_gemm(
        FORMATS[a_format], FORMATS[b_format], _addr(A), _addr(B), _addr(a_scales),
        _addr(b_scales), 1 if b_scales_packed else 0, _addr(group_offsets), _addr(expert_ids),
        _addr(C), int(M_total), int(N), int(K), int(num_groups), int(num_experts),
        _stream(stream))
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsmx_grouped_gemm")


def bsmxfp8_pack_b_scales(b_scales, b_scales_packed, num_experts: int, N: int, K: int,
                          stream=None) -> None:
    """Rearrange UE8M0 weight scales [E, N, K/32] into the packed 512-byte block layout
    (include/bsfp8.h).  Raises BsFp8Error."""
    st = load_library().bsmxfp8_pack_b_scales(_addr(b_scales), _addr(b_scales_packed),
                                              int(num_experts), int(N), int(K), _stream(stream))
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsmxfp8_pack_b_scales")


def bsmxfp8_grouped_gemm_prepacked(A, B, a_scales, b_scales_packed, expert_offsets, C,
                                   M_total: int, N: int, K: int, num_experts: int,
                                   stream=None) -> None:
    """MXFP8 grouped GEMM with pre-packed weight scales; see include/bsfp8.h."""
    st = load_library().bsmxfp8_grouped_gemm_prepacked(
        _addr(A), _addr(B), _addr(a_scales), _addr(b_scales_packed), _addr(expert_offsets),
        _addr(C), int(M_total), int(N), int(K), int(num_experts), _stream(stream))
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsmxfp8_grouped_gemm_prepacked")


def bsmxfp8_tmem_plan(block_k: int, epilogue_n: int, vec: int, overlap: bool) -> dict:
    """TMEM plan of double-buffered block-scaled accumulators (host only).  block_k=0 gives
    the plan the CTA-pair MXFP8 kernel is compiled with."""
    out = (ctypes.c_int32 * 9)()
    st = load_library().bsmxfp8_tmem_plan(int(block_k), int(epilogue_n), int(vec), int(bool(overlap)),
                                          out)
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsmxfp8_tmem_plan")
    keys = ("left_offset", "left_cols", "right_offset", "right_cols", "a_scale_offset",
            "a_scale_cols", "b_scale_offset", "b_scale_cols", "early_release_subtile")
    return dict(zip(keys, list(out)))


def bsfp8_blockwise_plan(M_total: int, N: int, num_experts: int, num_sms: int) -> dict:
    """Tile plan of the blockwise GEMM for this problem size on num_sms SMs (host only)."""
    out = (ctypes.c_int32 * 3)()
    st = load_library().bsfp8_blockwise_plan(int(M_total), int(N), int(num_experts),
                                             int(num_sms), out)
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsfp8_blockwise_plan")
    return {"tile_rows": out[0], "tile_cols": out[1], "ctas_per_tile": out[2]}


def bsmxfp8_plan(M_total: int, num_experts: int) -> dict:
    """Kernel plan of the MXFP8 GEMM for M_total token rows over num_experts groups (host
    only): which kernel(s) run, the swap-AB tile height and the split's row threshold."""
    out = (ctypes.c_int32 * 3)()
    st = load_library().bsmxfp8_plan(int(M_total), int(num_experts), out)
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsmxfp8_plan")
    return {"kernel": ("swap", "pair", "split")[out[0]], "token_rows": out[1],
            "split_rows": out[2]}


def bsmx_plan(M_total: int, num_groups: int) -> dict:
    """Tile form of the fp4-format GEMM for M_total token rows over num_groups groups (host
    only): CTA-pair or swap-AB tiles and the swap-AB tile height."""
    out = (ctypes.c_int32 * 2)()
    st = load_library().bsmx_plan(int(M_total), int(num_groups), out)
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsmx_plan")
    return {"kernel": ("swap", "pair")[out[0]], "token_rows": out[1]}


def bsfp8_check_wait_timeout(limit_ns: int, stream=None) -> None:
    """Launch the failure-detection check: a bounded wait that nothing completes gives up
    after limit_ns and records BSFP8_ERR_DEVICE_TIMEOUT in the device error word."""
    st = load_library().bsfp8_check_wait_timeout(int(limit_ns), _stream(stream))
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsfp8_check_wait_timeout")


def bsfp8_get_device_error(stream=None) -> int:
    """Read and clear the device error word (synchronises the stream)."""
    code = ctypes.c_int(0)
    st = load_library().bsfp8_get_device_error(_stream(stream), ctypes.byref(code))
    if st != BSFP8_OK:
        raise BsFp8Error(st, "bsfp8_get_device_error")
    return code.value
