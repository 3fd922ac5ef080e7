"""The C-ABI library on the host: it loads, exports every declared symbol, and rejects bad
arguments with the documented status codes before touching any GPU."""
import ctypes
import os
import re

import pytest

import block_scaled_fp8_persistent_gb300 as bsfp8
from block_scaled_fp8_persistent_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return bsfp8.load_library()


def _declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(bs[a-z0-9_]+)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert "bsfp8_grouped_gemm" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(bsfp8.EXPORTED)


def test_status_strings(lib):
    for code in range(10):
        assert len(bsfp8.status_string(code)) > 0
    assert bsfp8.status_string(8) == "device: expert id out of range"
    assert bsfp8.status_string(9) == "unsupported operand format pair"
    assert bsfp8.status_string(99) == "unknown status"


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced on these paths


def _call(lib, **kw):
    a = dict(A=FAKE, B=FAKE, sa=FAKE, sb=FAKE, off=FAKE, C=FAKE, M=256, N=256, K=512, E=1)
    a.update(kw)
    return lib.bsfp8_grouped_gemm(a["A"], a["B"], a["sa"], a["sb"], a["off"], a["C"], a["M"],
                                  a["N"], a["K"], a["E"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=None), 1), (dict(sb=None), 1), (dict(off=None), 1), (dict(A=None), 1),
    (dict(C=None), 1), (dict(sa=None), 1),
    (dict(N=192), 2), (dict(N=0), 2), (dict(K=100), 2), (dict(K=0), 2), (dict(E=0), 2),
    (dict(M=-1), 2), (dict(M=1 << 31), 2), (dict(E=1 << 20, N=4096), 2),
    (dict(A=FAKE + 8), 3), (dict(B=FAKE + 4), 3), (dict(C=FAKE + 2), 3), (dict(sa=FAKE + 2), 3),
    (dict(off=FAKE + 1), 3),
])
def test_host_validation(lib, kw, status):
    assert _call(lib, **kw) == status


def test_empty_problem_needs_no_row_buffers(lib):
    # M_total == 0: A, a_scales and C may be NULL; shape errors still reported first
    assert _call(lib, M=0, A=None, sa=None, C=None, N=100) == 2


def test_binding_raises_on_bad_shape():
    with pytest.raises(bsfp8.BsFp8Error) as ei:
        bsfp8.bsfp8_grouped_gemm(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256, 200, 512, 1, stream=0)
    assert ei.value.status == 2


def _call_ids(lib, mx=False, **kw):
    a = dict(A=FAKE, B=FAKE, sa=FAKE, sb=FAKE, off=FAKE, ids=FAKE, C=FAKE, M=256, N=256, K=512,
             G=3, E=2)
    a.update(kw)
    f = lib.bsmxfp8_grouped_gemm_ids if mx else lib.bsfp8_grouped_gemm_ids
    return f(a["A"], a["B"], a["sa"], a["sb"], a["off"], a["ids"], a["C"], a["M"], a["N"],
             a["K"], a["G"], a["E"], None)


@pytest.mark.parametrize("mx", [False, True])
@pytest.mark.parametrize("kw,status", [
    (dict(ids=None), 1), (dict(off=None), 1), (dict(B=None), 1),
    (dict(G=0), 2), (dict(E=0), 2), (dict(E=1 << 20, N=4096), 2), (dict(N=192), 2),
    (dict(ids=FAKE + 2), 3), (dict(off=FAKE + 1), 3),
])
def test_host_validation_expert_ids(lib, mx, kw, status):
    assert _call_ids(lib, mx=mx, **kw) == status


def test_binding_ids_raises_on_null_ids():
    with pytest.raises(bsfp8.BsFp8Error) as ei:
        bsfp8.bsfp8_grouped_gemm_ids(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 256, 256, 512, 2, 2,
                                     stream=0)
    assert ei.value.status == 1


@pytest.mark.parametrize("kw,status", [
    (dict(src=None), 1), (dict(dst=None), 1), (dict(E=0), 2), (dict(N=192), 2), (dict(K=100), 2),
    (dict(E=1 << 20, N=4096), 2), (dict(src=FAKE + 2), 3), (dict(dst=FAKE + 4), 3),
])
def test_host_validation_pack_b_scales(lib, kw, status):
    a = dict(src=FAKE, dst=FAKE, E=2, N=256, K=512)
    a.update(kw)
    assert lib.bsmxfp8_pack_b_scales(a["src"], a["dst"], a["E"], a["N"], a["K"], None) == status


def test_host_validation_prepacked_gemm(lib):
    f = lib.bsmxfp8_grouped_gemm_prepacked
    # packed scales must be 16-byte aligned (they are copied as 512-byte blocks)
    assert f(FAKE, FAKE, FAKE, FAKE + 4, FAKE, FAKE, 256, 256, 512, 1, None) == 3
    assert f(FAKE, FAKE, FAKE, None, FAKE, FAKE, 256, 256, 512, 1, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256, 200, 512, 1, None) == 2


@pytest.mark.parametrize("limit", [0, -5, 2_000_000_000])
def test_host_validation_wait_timeout_check(lib, limit):
    assert lib.bsfp8_check_wait_timeout(limit, None) == 2


def _call_fmt(lib, af, bf, **kw):
    a = dict(A=FAKE, B=FAKE, sa=FAKE, sb=FAKE, packed=0, off=FAKE, ids=None, C=FAKE, M=256,
             N=256, K=512, G=2, E=2)
    a.update(kw)
    return lib.bsmx_grouped_gemm(af, bf, a["A"], a["B"], a["sa"], a["sb"], a["packed"], a["off"],
                                 a["ids"], a["C"], a["M"], a["N"], a["K"], a["G"], a["E"], None)


@pytest.mark.parametrize("af,bf", [(1, 0), (2, 0), (0, 2), (2, 1), (1, 2), (3, 1), (-1, 1),
                                   (0, 3)])
def test_fmt_unsupported_pairs(lib, af, bf):
    # rejected before any other check or GPU use
    assert _call_fmt(lib, af, bf) == 9
    assert _call_fmt(lib, af, bf, B=None) == 9


@pytest.mark.parametrize("af,bf", [(0, 1), (1, 1)])
@pytest.mark.parametrize("kw,status", [
    (dict(B=None), 1), (dict(off=None), 1), (dict(sb=None), 1),
    (dict(N=192), 2), (dict(K=96), 2), (dict(G=3), 2), (dict(M=-1), 2),
    (dict(A=FAKE + 8), 3), (dict(B=FAKE + 8), 3), (dict(sb=FAKE + 2), 3),
    (dict(packed=1, sb=FAKE + 4), 3),
])
def test_fmt_host_validation(lib, af, bf, kw, status):
    assert _call_fmt(lib, af, bf, **kw) == status


def test_fmt_binding_raises_on_unsupported_pair():
    with pytest.raises(bsfp8.BsFp8Error) as ei:
        bsfp8.bsmx_grouped_gemm("mxfp4", "mxfp8", FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256, 256,
                                512, 1, 1, stream=0)
    assert ei.value.status == 9


def test_nvfp4_host_rules(lib):
    # nvfp4 x nvfp4 is supported; the packed UE8M0 scale layout is not (format error), and
    # its e4m3 scales must be 8-byte aligned
    assert _call_fmt(lib, 2, 2, packed=1) == 9
    assert _call_fmt(lib, 2, 2, sa=FAKE + 4) == 3
    assert _call_fmt(lib, 2, 2, sb=FAKE + 4) == 3
    assert _call_fmt(lib, 2, 2, N=192) == 2
    assert _call_fmt(lib, 2, 2, B=None) == 1
