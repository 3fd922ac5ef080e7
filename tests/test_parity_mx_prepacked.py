"""GPU parity of the pre-packed MXFP8 weight scales: the pack kernel against the oracle's
statement of the packed block layout (swizzle_scales_packed_block, Triton Gluon example
"Overlapping Accumulator Block-Scaled Matrix Multiplication"), bit for bit, and the GEMM on
pre-packed scales, on the swap-AB and the CTA-pair kernels, against the oracle and against
the GEMM on row-major scales."""
import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import parity_report

pytestmark = pytest.mark.gpu


def _pack_on_device(sb: torch.Tensor, E: int, N: int, K: int) -> torch.Tensor:
    import block_scaled_fp8_persistent_gb300 as bsfp8
    packed = torch.full((E * N * (K // 32),), 0xAB, dtype=torch.uint8, device=sb.device)
    bsfp8.bsmxfp8_pack_b_scales(sb, packed, E, N, K)
    torch.cuda.synchronize()
    return packed


@pytest.mark.parametrize("E,N,K", [(1, 128, 128), (3, 256, 512), (5, 384, 640), (2, 128, 7168)])
def test_pack_kernel_matches_oracle(E, N, K):
    rng = np.random.default_rng(E * 1000 + N + K)
    sb = rng.integers(0, 256, size=(E, N, K // 32), dtype=np.uint8)
    got = _pack_on_device(torch.from_numpy(sb).cuda(), E, N, K).cpu().numpy()
    assert np.array_equal(got, oracle.pack_mx_scales(sb.reshape(E * N, K // 32)))


@pytest.fixture(params=["swap32", "swap64", "swap128", "pair", "split"])
def form(request, monkeypatch):
    """Kernel form: swap-AB tiles of 32 / 64 / 128 token rows, CTA-pair 256 x 256 tiles, or
    both with the groups split by size (all read pre-packed weight scales); the row-major
    comparison runs the same form."""
    if request.param in ("pair", "split"):
        monkeypatch.setenv("BSFP8_MX_KERNEL", request.param)
    else:
        monkeypatch.setenv("BSFP8_MX_KERNEL", "swap")
        monkeypatch.setenv("BSFP8_MX_TN", request.param[4:])
    return request.param


def _run_both(p):
    """(prepacked result, row-major-scale result) as bf16 bits, on the same kernel form."""
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    d = DeviceProblem(p, c_rows_extra=2)
    packed = _pack_on_device(d.sb, p.E, p.N, p.K)
    bsfp8.bsmxfp8_grouped_gemm_prepacked(d.A, d.B, d.sa, packed, d.off, d.C, p.M_total, p.N,
                                         p.K, p.E)
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    assert np.all(d.guard_bits() == d.sentinel)
    ref = DeviceProblem(p)
    ref.run()
    assert bsfp8.bsfp8_get_device_error() == 0
    return got, ref.c_bits()


CASES = [("decode_like", [3, 17, 0, 32, 1, 9], 256, 512),
         ("ragged", [40, 0, 7, 130], 384, 640),
         ("many_tiles", [700, 0, 513], 640, 512),
         ("sizes_both_sides", [300, 7, 0, 45, 260, 129], 256, 1024)]


@pytest.mark.parametrize("name,counts,N,K", CASES, ids=[c[0] for c in CASES])
def test_prepacked_gemm(name, counts, N, K, form):
    p = gen.mx_problem(counts, N, K, seed=400 + len(name))
    got, plain = _run_both(p)
    assert np.array_equal(got, plain)
    ref, T = oracle.problem_reference(p)
    bad, ratio, _ = parity_report(got, ref, T)
    assert bad == 0, f"{bad} elements outside tolerance (max err/tol {ratio:.3g})"


def test_prepacked_gemm_exact_bitwise(form):
    p = gen.mx_problem([5, 30, 0, 12], 256, 1024, seed=410, exact=True)
    got, _ = _run_both(p)
    ref, _ = oracle.problem_reference(p, want_t=False)
    assert np.array_equal(got, ref)


def test_full_size_decode_prepacked_equals_row_major(monkeypatch):
    """The decode workload at its full size (128 experts, N=4096, K=7168): the pack kernel
    matches the oracle's layout and the GEMM on packed scales equals, bit for bit, the GEMM
    on row-major scales."""
    monkeypatch.setenv("BSFP8_MX_KERNEL", "swap")
    p = gen.config_problem(4)
    got, plain = _run_both(p)
    assert np.array_equal(got, plain)
    from gpu_util import DeviceProblem
    d = DeviceProblem(p)
    packed = _pack_on_device(d.sb, p.E, p.N, p.K).cpu().numpy()
    assert np.array_equal(packed, oracle.pack_mx_scales(p.b_scales.reshape(p.E * p.N, -1)))


def test_full_size_dense_prepacked_pair_equals_row_major(monkeypatch):
    """The dense 8192^3 MXFP8 workload on the CTA-pair kernel: pre-packed weight scales give
    the same bits as row-major ones."""
    monkeypatch.setenv("BSFP8_MX_KERNEL", "pair")
    got, plain = _run_both(gen.config_problem(5))
    assert np.array_equal(got, plain)
