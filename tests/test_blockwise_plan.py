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
    # grouped MoE (E=8, 4096 rows, N=4096): single-CTA 96-row tiles fill 5 waves; 3 pair tiles
    # per ~512-row expert need 6
    assert plan(4096, 4096, 8) == {"tile_rows": 96, "tile_cols": 256, "ctas_per_tile": 1}
    # dense 8192^3: 16 waves of 224-row pair tiles against 19 of the others
    assert plan(8192, 8192, 1) == {"tile_rows": 224, "tile_cols": 256, "ctas_per_tile": 2}
    # 64 Zipf-sized experts, N=2048
    assert plan(16384, 2048, 64) == {"tile_rows": 96, "tile_cols": 256, "ctas_per_tile": 1}


def _model(M, N, E, rows, units):
    row_tiles = E * math.ceil(M / (E * rows))
    return math.ceil(row_tiles * math.ceil(N / 256) / units)


@pytest.mark.parametrize("M", [1, 95, 97, 1000, 4096, 8192, 30000])
@pytest.mark.parametrize("N", [128, 256, 2048, 7168])
@pytest.mark.parametrize("E", [1, 2, 8, 64])
def test_default_follows_the_makespan_model(M, N, E):
    single = _model(M, N, E, 96, SMS)
    p192 = _model(M, N, E, 192, SMS // 2) * 0.95
    p224 = _model(M, N, E, 224, SMS // 2) * 0.97
    if min(p192, p224) >= 0.92 * single:
        want = (96, 1)
    else:
        want = (224, 2) if p224 <= p192 else (192, 2)
    got = plan(M, N, E)
    assert (got["tile_rows"], got["ctas_per_tile"]) == want and got["tile_cols"] == 256


@pytest.mark.parametrize("name,rows,cols,ctas", [
    ("cta1_256", 128, 256, 1), ("pair_256", 256, 256, 2), ("pair_160", 256, 160, 2),
    ("pair_128", 256, 128, 2), ("cta1_128", 128, 128, 1), ("cta1_96", 96, 256, 1),
    ("pair_192", 192, 256, 2), ("cta1_96x192", 96, 192, 1), ("pair_192x192", 192, 192, 2),
    ("cta1_128x192", 128, 192, 1), ("pair_224", 224, 256, 2)])
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
