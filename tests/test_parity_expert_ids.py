"""GPU parity of the grouped GEMMs with an expert indirection (group g multiplies the
weights of expert expert_ids[g]: the expert_ids argument of promote_accumulators, MAX
kernels grouped_matmul_sm100_blockwise_fp8) against the CPU oracle, through the C ABI
entry points bsfp8_grouped_gemm_ids / bsmxfp8_grouped_gemm_ids."""
import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import parity_report

pytestmark = pytest.mark.gpu

BLOCKWISE_TILES = ["cta1_96", "pair_192", "cta1_256", "pair_256", "cta1_96x192", "pair_192x192",
                   "pair_224"]
MX_FORMS = ["swap32", "swap128", "pair", "split"]


def _set_form(monkeypatch, mode, form):
    if mode == "blockwise":
        monkeypatch.setenv("BSFP8_BLOCKWISE_TILE", form)
    elif form in ("pair", "split"):
        monkeypatch.setenv("BSFP8_MX_KERNEL", form)
    else:
        monkeypatch.setenv("BSFP8_MX_KERNEL", "swap")
        monkeypatch.setenv("BSFP8_MX_TN", form[4:])


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
    return got, ref


# groups, expert ids, experts: repeats, unused experts, empty groups, ragged tails
CASES = [
    ("repeats", [37, 0, 20, 130, 5], [2, 0, 2, 1, 3], 6, 384, 640),
    ("reversed", [64, 64, 64, 64], [3, 2, 1, 0], 4, 256, 512),
    ("one_expert_for_all", [100, 29, 1], [1, 1, 1], 2, 256, 256),
    ("sparse_experts", [33, 0, 77], [7, 3, 0], 8, 128, 384),
]


@pytest.mark.parametrize("tile", BLOCKWISE_TILES)
@pytest.mark.parametrize("name,counts,ids,E,N,K", CASES, ids=[c[0] for c in CASES])
def test_blockwise_expert_ids(name, counts, ids, E, N, K, tile, monkeypatch):
    _set_form(monkeypatch, "blockwise", tile)
    _check(gen.routed_problem(counts, ids, E, N, K, seed=300 + len(name)))


@pytest.mark.parametrize("tile", BLOCKWISE_TILES)
def test_blockwise_expert_ids_exact_bitwise(tile, monkeypatch):
    _set_form(monkeypatch, "blockwise", tile)
    p = gen.routed_problem([200, 0, 57, 9], [1, 0, 1, 2], 3, 256, 1024, seed=310, exact=True)
    got, ref = _check(p)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("form", MX_FORMS)
@pytest.mark.parametrize("name,counts,ids,E,N,K", CASES, ids=[c[0] for c in CASES])
def test_mx_expert_ids(name, counts, ids, E, N, K, form, monkeypatch):
    _set_form(monkeypatch, "mx", form)
    _check(gen.routed_problem(counts, ids, E, N, K, seed=320 + len(name), mode="mx"))


@pytest.mark.parametrize("form", MX_FORMS)
def test_mx_expert_ids_exact_bitwise(form, monkeypatch):
    _set_form(monkeypatch, "mx", form)
    p = gen.routed_problem([5, 30, 0, 12], [2, 2, 0, 1], 3, 256, 1024, seed=330, mode="mx",
                           exact=True)
    got, ref = _check(p)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("mode", ["blockwise", "mx"])
@pytest.mark.parametrize("bad", [-1, 3])
def test_expert_id_out_of_range_reported_on_device(mode, bad):
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    p = gen.routed_problem([64, 40], [0, 1], 3, 256, 256, seed=340, mode=mode)
    d = DeviceProblem(p)
    d.ids.copy_(torch.tensor([0, bad], dtype=torch.int32))
    d.run()
    assert bsfp8.bsfp8_get_device_error() == 8
    assert np.all(d.c_bits() == d.sentinel)          # C untouched
    assert bsfp8.bsfp8_get_device_error() == 0       # read clears


@pytest.mark.parametrize("cfg", [1, 4])
def test_full_size_ids_equal_gathered_experts(cfg):
    """At the full workload size: routing a config through a permutation of its experts
    gives, bit for bit, the plain grouped GEMM run on the experts gathered in group order."""
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    p = gen.config_problem(cfg)
    perm = np.random.default_rng(cfg).permutation(p.E).astype(np.int32)
    routed = gen.Problem(p.mode, p.A, p.B, p.a_scales, p.b_scales, p.offsets, p.N, p.K,
                         expert_ids=perm)
    d = DeviceProblem(routed)
    d.run()
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    idx = torch.from_numpy(perm.astype(np.int64)).cuda()
    plain = DeviceProblem(p)
    plain.B = d.B.index_select(0, idx).contiguous()
    plain.sb = d.sb.index_select(0, idx).contiguous()
    plain.run()
    assert bsfp8.bsfp8_get_device_error() == 0
    assert np.array_equal(got, plain.c_bits())
