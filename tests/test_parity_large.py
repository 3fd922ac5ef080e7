"""GPU parity at sizes that stress the index arithmetic (long K loops, many experts in B, a
million token rows), checked on sampled outputs that the oracle recomputes one by one, and
the GEMMs captured in a CUDA graph and replayed."""
import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import parity_report

pytestmark = pytest.mark.gpu


def _sampled(p, n_points=3000, seed=0):
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    d = DeviceProblem(p)
    d.run()
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    rng = np.random.default_rng(seed)
    off = p.offsets.astype(np.int64)
    edges = sorted({int(r) for e in range(p.E) if off[e + 1] > off[e]
                    for r in (off[e], off[e + 1] - 1)})[:8]
    rows = np.concatenate([np.repeat(edges, min(p.N, 256)), rng.integers(0, p.M_total, n_points)])
    cols = np.concatenate([np.tile(np.arange(min(p.N, 256)), len(edges)),
                           rng.integers(0, p.N, n_points)])
    ref, T = oracle.problem_points(p, rows, cols)
    bad, ratio, _ = parity_report(got[rows, cols], ref, T)
    assert bad == 0, f"{bad} sampled elements outside tolerance (max err/tol {ratio:.3g})"


@pytest.mark.parametrize("mode", ["blockwise", "mx"])
def test_long_k(mode):
    # K = 131072: 1024 K blocks of 128 (4096 UE8M0 codes per row in MX mode)
    make = gen.blockwise_problem if mode == "blockwise" else gen.mx_problem
    _sampled(make([40, 0, 9], 256, 131072, seed=60))


@pytest.mark.parametrize("mode", ["blockwise", "mx"])
def test_many_experts_in_b(mode):
    # 512 experts x N = 2048: B row indices up to 2^20, most experts with a handful of rows
    counts = np.random.default_rng(61).integers(0, 5, size=512)
    make = gen.blockwise_problem if mode == "blockwise" else gen.mx_problem
    _sampled(make(counts, 2048, 128, seed=61))


def test_million_rows():
    # 2^20 + 77 token rows in ragged groups (A 134 MB, C 268 MB)
    counts = [300_000, 0, 448_576, 300_000 + 77]
    _sampled(gen.blockwise_problem(counts, 128, 128, seed=62), n_points=6000)


@pytest.mark.parametrize("mode", ["blockwise", "mx"])
def test_cuda_graph_capture_and_replay(mode):
    """The GEMM launch records into a CUDA graph (host-side set-up happens at capture) and
    replays with the inputs changed in place."""
    from gpu_util import DeviceProblem
    import block_scaled_fp8_persistent_gb300 as bsfp8
    make = gen.blockwise_problem if mode == "blockwise" else gen.mx_problem
    p = make([100, 0, 29], 256, 512, seed=63)
    q = make([100, 0, 29], 256, 512, seed=64)
    d = DeviceProblem(p)
    d.run()                      # first call on this device outside the capture
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


@pytest.mark.parametrize("path", ["mma", "convert"])
def test_fp4_long_k(path, monkeypatch):
    # K = 65536 (512 K blocks of packed e2m1, 2048 nvfp4 scale codes per row)
    monkeypatch.setenv("BSFP8_FP4_MMA", path)
    for a_fmt, b_fmt in (("mxfp8", "mxfp4"), ("mxfp4", "mxfp4"), ("nvfp4", "nvfp4")):
        _sampled(gen.fmt_problem([40, 0, 9], 256, 65536, seed=66, a_fmt=a_fmt, b_fmt=b_fmt))
