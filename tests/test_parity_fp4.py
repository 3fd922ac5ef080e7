"""GPU parity of the fp4 block-scaled formats (the format pairs mxfp8 x mxfp4, mxfp4 x mxfp4
and nvfp4 x nvfp4 of the Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix
Multiplication") against the CPU oracle, through bsmx_grouped_gemm.  Same acceptance bound
as MXFP8; inputs whose fp32 sums are exact (fp4-grid values, scales 0.5 / 1 / 2) must match
bit for bit."""
import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import parity_report

pytestmark = pytest.mark.gpu

PAIRS = [("mxfp8", "mxfp4"), ("mxfp4", "mxfp4"), ("nvfp4", "nvfp4")]
MX_PAIRS = PAIRS[:2]
# (a format, b format, path): every pair runs an fp4 MMA kind by default ("mma") and the
# converting kernels on request ("convert")
FORMS = [("mxfp8", "mxfp4", "mma"), ("mxfp8", "mxfp4", "convert"), ("mxfp4", "mxfp4", "mma"),
         ("mxfp4", "mxfp4", "convert"), ("nvfp4", "nvfp4", "mma"), ("nvfp4", "nvfp4", "convert")]
MX_FORMS = [f for f in FORMS if f[0] != "nvfp4"]
NV_PATHS = ["mma", "convert"]


@pytest.fixture
def path_env(monkeypatch):
    def use(path):
        monkeypatch.setenv("BSFP8_FP4_MMA", path)
    return use


@pytest.fixture(params=["32", "64", "128"])
def tn(request, monkeypatch):
    """Token rows per swap-AB tile (the converting forms hold at most 64: a request for 128
    runs 64 there)."""
    monkeypatch.setenv("BSFP8_MX_TN", request.param)
    return int(request.param)


def _check_full(p, **kw):
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    d = DeviceProblem(p, c_rows_extra=2, **kw)
    d.run()
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    ref, T = oracle.problem_reference(p)
    bad, ratio, exact = parity_report(got, ref, T)
    assert bad == 0, f"{bad} elements outside tolerance (max err/tol {ratio:.3g})"
    assert np.all(d.guard_bits() == d.sentinel)
    return got, ref


CASES = [
    ("decode_like", [3, 17, 0, 32, 1, 9], 256, 512),
    ("many_tiles", [700, 0, 513], 640, 512),
    ("ragged_k", [40, 0, 7], 384, 640),
    ("mixed", [0, 129, 64, 65, 2, 0, 31], 256, 384),
]


@pytest.mark.parametrize("a_fmt,b_fmt,path", FORMS)
@pytest.mark.parametrize("name,counts,N,K", CASES, ids=[c[0] for c in CASES])
def test_small_cases(name, counts, N, K, a_fmt, b_fmt, tn, path, path_env):
    path_env(path)
    _check_full(gen.fmt_problem(counts, N, K, seed=300 + len(name), a_fmt=a_fmt, b_fmt=b_fmt))


@pytest.mark.parametrize("a_fmt,b_fmt", [pr for pr in PAIRS if pr[0] == "mxfp8"])
def test_quantized_tokens(a_fmt, b_fmt, tn):
    # mxfp8 tokens drawn as the decode workload draws them (N(0,1) rows, UE8M0 per 32); the
    # recipe exists for mxfp8 tokens only
    _check_full(gen.fmt_problem([5, 30, 0, 12, 64], 512, 1024, seed=41, a_fmt=a_fmt,
                                b_fmt=b_fmt, a_recipe="quantized"))


@pytest.mark.parametrize("a_fmt,b_fmt,path", FORMS)
def test_exact_inputs_bitwise(a_fmt, b_fmt, tn, path, path_env):
    path_env(path)
    p = gen.fmt_problem([5, 30, 0, 12], 256, 1024, seed=42, a_fmt=a_fmt, b_fmt=b_fmt)
    # scales 0.5 / 1 / 2 (UE8M0 codes 126..128, e4m3 codes 0x30 / 0x38 / 0x40): every
    # partial sum is exact in fp32, so the result is unique
    if a_fmt == "nvfp4":
        p.a_scales[:] = 0x30 + 8 * (p.a_scales % 3)
        p.b_scales[:] = 0x30 + 8 * (p.b_scales % 3)
    else:
        p.a_scales[:] = 126 + p.a_scales % 3
        p.b_scales[:] = 126 + p.b_scales % 3
    got, ref = _check_full(p)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("a_fmt,b_fmt,path", FORMS)
def test_expert_ids(a_fmt, b_fmt, tn, path, path_env):
    path_env(path)
    p = gen.fmt_problem([9, 0, 33, 4, 17], 256, 512, seed=43, a_fmt=a_fmt, b_fmt=b_fmt,
                        expert_ids=[3, 1, 3, 0, 2], num_experts=4)
    _check_full(p)


@pytest.mark.parametrize("path", NV_PATHS)
@pytest.mark.parametrize("counts,N,K", [([3, 17, 0, 32, 1, 9], 256, 512), ([40, 0, 77], 384, 1024)])
def test_nvfp4_general_e4m3_scales(counts, N, K, tn, path, path_env):
    path_env(path)
    # non-power-of-two e4m3 scales (0.125 .. 3.75), as nvfp4 quantization produces them
    _check_full(gen.fmt_problem(counts, N, K, seed=49, a_fmt="nvfp4", b_fmt="nvfp4",
                                scales="e4m3"))


@pytest.mark.parametrize("a_fmt,b_fmt,path", MX_FORMS)
def test_prepacked_weight_scales(a_fmt, b_fmt, path, path_env):
    path_env(path)
    import block_scaled_fp8_persistent_gb300 as bsfp8
    from gpu_util import DeviceProblem
    p = gen.fmt_problem([12, 0, 40], 384, 1024, seed=44, a_fmt=a_fmt, b_fmt=b_fmt)
    d = DeviceProblem(p)
    E, N, K = p.num_experts, p.N, p.K
    packed = torch.empty(E * N * K // 32, dtype=torch.uint8, device="cuda")
    bsfp8.bsmxfp8_pack_b_scales(d.sb, packed, E, N, K)
    bsfp8.bsmx_grouped_gemm(a_fmt, b_fmt, d.A, d.B, d.sa, packed, d.off, d.C, p.M_total, N, K,
                            p.E, E, b_scales_packed=True)
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    ref, T = oracle.problem_reference(p)
    bad, ratio, _ = parity_report(got, ref, T)
    assert bad == 0, f"{bad} elements outside tolerance (max err/tol {ratio:.3g})"


def test_mxfp8_pair_through_format_entry():
    # (mxfp8, mxfp8) through bsmx_grouped_gemm is the MXFP8 GEMM
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    p = gen.fmt_problem([7, 0, 50], 256, 512, seed=45, a_fmt="mxfp8", b_fmt="mxfp8")
    d = DeviceProblem(p)
    bsfp8.bsmx_grouped_gemm("mxfp8", "mxfp8", d.A, d.B, d.sa, d.sb, d.off, d.C, p.M_total, p.N,
                            p.K, p.E, p.num_experts)
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    ref, T = oracle.problem_reference(p)
    assert parity_report(got, ref, T)[0] == 0


@pytest.mark.parametrize("a_fmt,b_fmt,path", FORMS)
def test_empty_and_degenerate(a_fmt, b_fmt, path, path_env):
    path_env(path)
    # no rows at all; one expert with one row; all rows in the last expert
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    p = gen.fmt_problem([0, 0, 0], 128, 128, seed=46, a_fmt=a_fmt, b_fmt=b_fmt)
    d = DeviceProblem(p, c_rows_extra=1)
    d.run()
    torch.cuda.synchronize()
    assert bsfp8.bsfp8_get_device_error() == 0
    assert np.all(d.guard_bits() == d.sentinel)
    _check_full(gen.fmt_problem([1], 128, 128, seed=47, a_fmt=a_fmt, b_fmt=b_fmt))
    _check_full(gen.fmt_problem([0, 0, 77], 128, 256, seed=48, a_fmt=a_fmt, b_fmt=b_fmt))


@pytest.mark.parametrize("a_fmt,b_fmt,path", FORMS)
def test_invalid_offsets_reported_on_device(a_fmt, b_fmt, path, path_env):
    path_env(path)
    # offsets that are not a partition of [0, M_total): device error 6, C untouched
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    p = gen.fmt_problem([10, 10], 128, 256, seed=50, a_fmt=a_fmt, b_fmt=b_fmt)
    d = DeviceProblem(p)
    d.off.copy_(torch.tensor([0, 15, 12], dtype=torch.int32))
    d.run()
    assert bsfp8.bsfp8_get_device_error() == 6
    assert np.all(d.c_bits() == d.sentinel)


@pytest.mark.parametrize("a_fmt,b_fmt,path", FORMS)
@pytest.mark.parametrize("bad", [-1, 3])
def test_expert_id_out_of_range_reported_on_device(a_fmt, b_fmt, bad, path, path_env):
    path_env(path)
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    p = gen.fmt_problem([64, 40], 256, 256, seed=51, a_fmt=a_fmt, b_fmt=b_fmt,
                        expert_ids=[0, 1], num_experts=3)
    d = DeviceProblem(p)
    d.ids.copy_(torch.tensor([0, bad], dtype=torch.int32))
    d.run()
    assert bsfp8.bsfp8_get_device_error() == 8
    assert np.all(d.c_bits() == d.sentinel)
    assert bsfp8.bsfp8_get_device_error() == 0


@pytest.mark.parametrize("a_fmt,b_fmt,path", FORMS)
def test_cuda_graph_capture_and_replay(a_fmt, b_fmt, path, path_env):
    path_env(path)
    # the fp4 launch records into a CUDA graph and replays with the inputs changed in place
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    p = gen.fmt_problem([100, 0, 29], 256, 512, seed=52, a_fmt=a_fmt, b_fmt=b_fmt)
    q = gen.fmt_problem([100, 0, 29], 256, 512, seed=53, a_fmt=a_fmt, b_fmt=b_fmt)
    d = DeviceProblem(p)
    d.run()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            d.run(stream=s)
    for src in (q, p):
        d.A.copy_(torch.from_numpy(src.A)); d.B.copy_(torch.from_numpy(src.B))
        d.sa.copy_(torch.from_numpy(src.a_scales)); d.sb.copy_(torch.from_numpy(src.b_scales))
        g.replay()
        torch.cuda.synchronize()
        assert bsfp8.bsfp8_get_device_error() == 0
        ref, T = oracle.problem_reference(src)
        bad, ratio, _ = parity_report(d.c_bits(), ref, T)
        assert bad == 0


@pytest.mark.parametrize("path", NV_PATHS)
def test_nvfp4_scale_codes_and_subnormals(tn, path, path_env):
    # nvfp4 scale codes over the whole finite unsigned e4m3 (UE4M3) range, 0x00 .. 0x7E,
    # subnormals (0x01 .. 0x07) and zero included: the Gluon example draws its nvfp4 scales
    # positive (1/128 .. 2, converted to float8_e4m3fn), and the tensor core's scale type is
    # unsigned, so codes with bit 7 set are outside the format
    path_env(path)
    rng = np.random.default_rng(54)
    p = gen.fmt_problem([3, 17, 0, 32, 9], 256, 512, seed=54, a_fmt="nvfp4", b_fmt="nvfp4")
    for s in (p.a_scales, p.b_scales):
        s[:] = rng.integers(0, 0x7F, s.shape).astype(np.uint8)
    _check_full(p)


@pytest.mark.parametrize("path", NV_PATHS)
def test_nvfp4_subnormal_scales(tn, path, path_env):
    # every scale code subnormal or zero (0x00 .. 0x07: 0 .. 7 * 2^-9), the low end of the
    # Gluon example's range (its 1/128 is the subnormal 0x04)
    path_env(path)
    rng = np.random.default_rng(56)
    p = gen.fmt_problem([3, 17, 0, 32, 9], 256, 512, seed=56, a_fmt="nvfp4", b_fmt="nvfp4")
    for s in (p.a_scales, p.b_scales):
        s[:] = rng.integers(0, 8, s.shape).astype(np.uint8)
    _check_full(p)


@pytest.mark.parametrize("a_fmt,b_fmt,path", MX_FORMS)
def test_mx_fp4_wide_scale_range(a_fmt, b_fmt, tn, path, path_env):
    path_env(path)
    # UE8M0 codes 100..160 (2^-27 .. 2^33): the 2^-6 re-encoding and its 2^6 undo in the
    # epilogue stay exact across a wide exponent range
    rng = np.random.default_rng(55)
    p = gen.fmt_problem([5, 30, 0, 12], 256, 512, seed=55, a_fmt=a_fmt, b_fmt=b_fmt)
    p.a_scales[:] = rng.integers(100, 161, p.a_scales.shape).astype(np.uint8)
    p.b_scales[:] = rng.integers(100, 161, p.b_scales.shape).astype(np.uint8)
    _check_full(p)


def _unit_magnitudes(p, a_fmt, rng):
    """Set every operand element to +-1 or +-1.5 (one octave of products), keeping the
    layout: packed e2m1 nibbles (codes 2 / 3, sign bit 8) or e4m3 bytes (0x38 / 0x3C)."""
    def fp4(shape):
        lo = (rng.integers(2, 4, shape) | (rng.integers(0, 2, shape) << 3)).astype(np.uint8)
        hi = (rng.integers(2, 4, shape) | (rng.integers(0, 2, shape) << 3)).astype(np.uint8)
        return lo | (hi << 4)
    p.B[:] = fp4(p.B.shape)
    if a_fmt == "mxfp4":
        p.A[:] = fp4(p.A.shape)
    else:
        p.A[:] = (np.where(rng.integers(0, 2, p.A.shape) == 1, 0x3C, 0x38) |
                  (rng.integers(0, 2, p.A.shape) << 7)).astype(np.uint8)


@pytest.mark.parametrize("a_fmt,b_fmt,path", MX_FORMS)
def test_low_scales(a_fmt, b_fmt, tn, path, path_env):
    path_env(path)
    # scale codes 72 and 72: every product is 2^-110 times 1 .. 2.25, inside the documented
    # range (the tensor core sums them 2^-6 per fp4 operand lower, 2^-116 / 2^-122, still
    # fp32-normal), and the sums are far below 1 but in bf16's normal range
    p = gen.fmt_problem([5, 30, 0, 12], 256, 1024, seed=46, a_fmt=a_fmt, b_fmt=b_fmt)
    _unit_magnitudes(p, a_fmt, np.random.default_rng(46))
    p.a_scales[:] = 72
    p.b_scales[:] = 72
    _check_full(p)


@pytest.mark.parametrize("a_fmt,b_fmt,path", MX_FORMS)
def test_high_scales(a_fmt, b_fmt, tn, path, path_env):
    path_env(path)
    # token scale codes up to 254 (2^127) with weight codes low enough that the products stay
    # finite: the 2^6 per fp4 operand is applied after the sums, in fp32
    p = gen.fmt_problem([5, 30, 0, 12], 256, 1024, seed=47, a_fmt=a_fmt, b_fmt=b_fmt)
    rng = np.random.default_rng(47)
    _unit_magnitudes(p, a_fmt, rng)
    p.a_scales[:] = rng.integers(246, 255, p.a_scales.shape).astype(np.uint8)
    p.b_scales[:] = rng.integers(20, 30, p.b_scales.shape).astype(np.uint8)
    _check_full(p)


def _shifted(t, offset_bytes):
    """A copy of device tensor t whose data starts offset_bytes into a fresh allocation."""
    flat = torch.empty(t.numel() * t.element_size() + offset_bytes, dtype=torch.uint8,
                       device=t.device)
    view = flat[offset_bytes:offset_bytes + t.numel() * t.element_size()].view(t.dtype)
    view.copy_(t.reshape(-1))
    return view.view(t.shape)


@pytest.mark.parametrize("a_fmt,b_fmt", PAIRS)
def test_stage_k_128_forced(a_fmt, b_fmt, tn, monkeypatch):
    # K % 512 == 0 and aligned scales pick 256-K stages; BSFP8_FP4_STAGE_K=128 keeps the
    # 128-K form (64-byte rows, or one padded box per stage) on the same inputs
    monkeypatch.setenv("BSFP8_FP4_STAGE_K", "128")
    _check_full(gen.fmt_problem([9, 0, 33, 64, 1], 384, 1024, seed=57, a_fmt=a_fmt, b_fmt=b_fmt))


def test_mixed_weights_only_16_byte_aligned():
    # the padded e2m1 load needs a 32-byte aligned B: a B 16 bytes past such a boundary runs
    # the converting form, with the same results
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    p = gen.fmt_problem([12, 0, 40, 7], 384, 1024, seed=58, a_fmt="mxfp8", b_fmt="mxfp4")
    d = DeviceProblem(p, c_rows_extra=2)
    B16 = _shifted(d.B, 16)
    assert B16.data_ptr() % 32 == 16
    bsfp8.bsmx_grouped_gemm("mxfp8", "mxfp4", d.A, B16, d.sa, d.sb, d.off, d.C, p.M_total, p.N,
                            p.K, p.E, p.num_experts)
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    ref, T = oracle.problem_reference(p)
    bad, ratio, _ = parity_report(got, ref, T)
    assert bad == 0, f"{bad} elements outside tolerance (max err/tol {ratio:.3g})"
    assert np.all(d.guard_bits() == d.sentinel)


@pytest.mark.parametrize("a_fmt,b_fmt", PAIRS)
def test_scales_not_16_byte_aligned(a_fmt, b_fmt, tn):
    # scale arrays 8 bytes past a 16-byte boundary: the scale writers cannot fetch 16-byte
    # chunks, so the loader warps pack each stage and the writers relay (128-K stages)
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    p = gen.fmt_problem([5, 30, 0, 12, 64], 256, 1024, seed=59, a_fmt=a_fmt, b_fmt=b_fmt)
    d = DeviceProblem(p, c_rows_extra=2)
    sa8, sb8 = _shifted(d.sa, 8), _shifted(d.sb, 8)
    assert sa8.data_ptr() % 16 == 8 and sb8.data_ptr() % 16 == 8
    bsfp8.bsmx_grouped_gemm(a_fmt, b_fmt, d.A, d.B, sa8, sb8, d.off, d.C, p.M_total, p.N, p.K,
                            p.E, p.num_experts)
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    ref, T = oracle.problem_reference(p)
    bad, ratio, _ = parity_report(got, ref, T)
    assert bad == 0, f"{bad} elements outside tolerance (max err/tol {ratio:.3g})"
    assert np.all(d.guard_bits() == d.sentinel)


PAIR_CASES = [
    ("one_pair_tile", [256], 256, 1024),
    ("ragged", [700, 0, 513, 1], 640, 1024),
    ("many_experts", [300, 7, 0, 45, 260, 129, 511], 384, 2048),
    ("k_256", [300, 40], 256, 256),       # one K block of 256 (nvfp4), swap for mxfp4
    ("k_not_chunkable", [300, 40], 256, 640),  # the fp4 x fp4 pairs fall back to swap tiles
]


@pytest.mark.parametrize("a_fmt,b_fmt", PAIRS)
@pytest.mark.parametrize("name,counts,N,K", PAIR_CASES, ids=[c[0] for c in PAIR_CASES])
def test_cta_pair_tiles(name, counts, N, K, a_fmt, b_fmt, monkeypatch):
    # BSFP8_MX_KERNEL=pair: the CTA-pair 256 x 256 kernel on the fp4 kinds (mxfp8 x mxfp4 on
    # padded e2m1 weights; the fp4 x fp4 pairs in K blocks of 256 where the scale rows are
    # chunkable, else the swap-AB tiles)
    monkeypatch.setenv("BSFP8_MX_KERNEL", "pair")
    _check_full(gen.fmt_problem(counts, N, K, seed=60 + len(name), a_fmt=a_fmt, b_fmt=b_fmt))


@pytest.mark.parametrize("a_fmt,b_fmt", PAIRS)
def test_cta_pair_tiles_exact_and_ids(a_fmt, b_fmt, monkeypatch):
    monkeypatch.setenv("BSFP8_MX_KERNEL", "pair")
    p = gen.fmt_problem([300, 0, 260, 41], 256, 1024, seed=61, a_fmt=a_fmt, b_fmt=b_fmt)
    if a_fmt == "nvfp4":
        p.a_scales[:] = 0x30 + 8 * (p.a_scales % 3)
        p.b_scales[:] = 0x30 + 8 * (p.b_scales % 3)
    else:
        p.a_scales[:] = 126 + p.a_scales % 3
        p.b_scales[:] = 126 + p.b_scales % 3
    got, ref = _check_full(p)
    assert np.array_equal(got, ref)
    q = gen.fmt_problem([300, 0, 260, 41], 256, 1024, seed=62, a_fmt=a_fmt, b_fmt=b_fmt,
                        expert_ids=[2, 0, 2, 1], num_experts=3)
    _check_full(q)


@pytest.mark.parametrize("a_fmt,b_fmt", PAIRS)
def test_cta_pair_c_only_16_byte_aligned(a_fmt, b_fmt, monkeypatch):
    # C 16-byte aligned but not 32-byte aligned: the epilogue's 16-byte stores
    monkeypatch.setenv("BSFP8_MX_KERNEL", "pair")
    p = gen.fmt_problem([300, 0, 261], 384, 1024, seed=64, a_fmt=a_fmt, b_fmt=b_fmt)
    _check_full(p, c_offset=8)


def test_cta_pair_mixed_prepacked_weight_scales(monkeypatch):
    import block_scaled_fp8_persistent_gb300 as bsfp8
    from gpu_util import DeviceProblem
    monkeypatch.setenv("BSFP8_MX_KERNEL", "pair")
    p = gen.fmt_problem([300, 0, 270], 384, 1024, seed=63, a_fmt="mxfp8", b_fmt="mxfp4")
    d = DeviceProblem(p)
    E, N, K = p.num_experts, p.N, p.K
    packed = torch.empty(E * N * K // 32, dtype=torch.uint8, device="cuda")
    bsfp8.bsmxfp8_pack_b_scales(d.sb, packed, E, N, K)
    bsfp8.bsmx_grouped_gemm("mxfp8", "mxfp4", d.A, d.B, d.sa, packed, d.off, d.C, p.M_total, N,
                            K, p.E, E, b_scales_packed=True)
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    ref, T = oracle.problem_reference(p)
    bad, ratio, _ = parity_report(got, ref, T)
    assert bad == 0, f"{bad} elements outside tolerance (max err/tol {ratio:.3g})"
