"""Host logic of the blockwise tile choice (no GPU): bsfp8_blockwise_plan reports the tile
the GEMM would launch, the environment override is honoured, and the default picks the
configuration with the smaller estimated makespan."""
import math

import pytest

import block_scaled_fp8_persistent_gb300 as bsfp8
from block_scaled_fp8_persistent_gb300 import build as libbuild

SMS = 152


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()


@pytest.fixture(autouse=True)
def _no_override(monkeypatch):
    monkeypatch.delenv("BSFP8_BLOCKWISE_TILE", raising=False)


def plan(M, N, E, sms=SMS):
    return bsfp8.bsfp8_blockwise_plan(M, N, E, sms)


def test_named_workloads():
    # grouped MoE (E=8, 4096 rows, N=4096): 47 x 16 single-CTA tiles fill 5 waves, pair
    # tiles would need 6
    assert plan(4096, 4096, 8) == {"tile_rows": 96, "tile_cols": 256, "ctas_per_tile": 1}
    # dense 8192^3: both need 19 rounds, the pair tile is faster per round
    assert plan(8192, 8192, 1) == {"tile_rows": 192, "tile_cols": 256, "ctas_per_tile": 2}
    # 64 Zipf-sized experts, N=2048
    assert plan(16384, 2048, 64) == {"tile_rows": 96, "tile_cols": 256, "ctas_per_tile": 1}


def _model(M, N, E, rows, units):
    row_tiles = math.ceil(M / rows) + (0.5 * E if E > 1 else 0.0)
    return math.ceil(row_tiles * math.ceil(N / 256) / units)


@pytest.mark.parametrize("M", [1, 95, 97, 1000, 4096, 8192, 30000])
@pytest.mark.parametrize("N", [128, 256, 2048, 7168])
@pytest.mark.parametrize("E", [1, 2, 8, 64])
def test_default_is_smaller_estimated_makespan(M, N, E):
    single = _model(M, N, E, 96, SMS)
    pair = _model(M, N, E, 192, SMS // 2) * 0.97
    want = 192 if pair < single else 96
    got = plan(M, N, E)
    assert got["tile_rows"] == want and got["tile_cols"] == 256
    assert got["ctas_per_tile"] == (2 if want == 192 else 1)


@pytest.mark.parametrize("name,rows,cols,ctas", [
    ("cta1_256", 128, 256, 1), ("pair_256", 256, 256, 2), ("pair_160", 256, 160, 2),
    ("pair_128", 256, 128, 2), ("cta1_128", 128, 128, 1), ("cta1_96", 96, 256, 1),
    ("pair_192", 192, 256, 2), ("cta1_96x192", 96, 192, 1), ("pair_192x192", 192, 192, 2),
    ("cta1_128x192", 128, 192, 1)])
def test_environment_override(monkeypatch, name, rows, cols, ctas):
    monkeypatch.setenv("BSFP8_BLOCKWISE_TILE", name)
    assert plan(4096, 4096, 8) == {"tile_rows": rows, "tile_cols": cols, "ctas_per_tile": ctas}


@pytest.mark.parametrize("args", [(-1, 256, 1), (10, 100, 1), (10, 256, 0)])
def test_bad_input(args):
    with pytest.raises(bsfp8.BsFp8Error):
        plan(*args)


def test_null_out_pointer():
    lib = bsfp8.load_library()
    assert lib.bsfp8_blockwise_plan(10, 256, 1, SMS, None) == 1  # BSFP8_ERR_NULL
