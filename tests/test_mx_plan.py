"""Host logic of the MXFP8 kernel choice (no GPU): bsmxfp8_plan reports which kernel(s)
bsmxfp8_grouped_gemm enqueues for a batch, from the average token rows per expert (swap-AB
tiles up to 24, both kernels split by expert size up to 56, CTA-pair tiles above), and the
environment overrides."""
import pytest

import block_scaled_fp8_persistent_gb300 as bsfp8


@pytest.fixture(autouse=True)
def _no_overrides(monkeypatch):
    monkeypatch.delenv("BSFP8_MX_KERNEL", raising=False)
    monkeypatch.delenv("BSFP8_MX_TN", raising=False)


@pytest.mark.parametrize("M,E,kernel,rows,split", [
    (2091, 128, "swap", 32, 0),      # the decode workload: 1..32 tokens per expert
    (0, 128, "swap", 32, 0),         # nothing routed
    (3072, 128, "swap", 32, 0),      # 24 per expert: still swap-AB
    (3073, 128, "split", 64, 256),   # just above 24 per expert
    (3200, 64, "split", 64, 256),    # 50 per expert
    (4096, 64, "pair", 0, 0),        # 64 per expert
])
def test_plan_bands(M, E, kernel, rows, split):
    assert bsfp8.bsmxfp8_plan(M, E) == {"kernel": kernel, "token_rows": rows, "split_rows": split}


def test_plan_named_workloads():
    # dense 8192^3 (one group) and 8 experts x 512 rows: CTA-pair tiles only
    assert bsfp8.bsmxfp8_plan(8192, 1) == {"kernel": "pair", "token_rows": 0, "split_rows": 0}
    assert bsfp8.bsmxfp8_plan(4096, 8)["kernel"] == "pair"
    # Zipf routing of 16384 rows over 64 experts (256 per expert on average): CTA pair
    assert bsfp8.bsmxfp8_plan(16384, 64)["kernel"] == "pair"
    # 56 rows per expert is the split's upper end, 57 the pair kernel's lower end
    assert bsfp8.bsmxfp8_plan(56 * 64, 64)["kernel"] == "split"
    assert bsfp8.bsmxfp8_plan(56 * 64 + 1, 64)["kernel"] == "pair"
    # one group never splits: its size is known on the host
    assert bsfp8.bsmxfp8_plan(20, 1)["kernel"] == "swap"
    assert bsfp8.bsmxfp8_plan(30, 1)["kernel"] == "pair"


def test_swap_tile_height_follows_the_average():
    assert bsfp8.bsmxfp8_plan(32 * 100, 200)["token_rows"] == 32   # 16 per expert
    assert bsfp8.bsmxfp8_plan(24 * 10, 10)["token_rows"] == 32


def test_environment_overrides(monkeypatch):
    monkeypatch.setenv("BSFP8_MX_KERNEL", "swap")
    monkeypatch.setenv("BSFP8_MX_TN", "128")
    assert bsfp8.bsmxfp8_plan(8192, 1) == {"kernel": "swap", "token_rows": 128, "split_rows": 0}
    monkeypatch.setenv("BSFP8_MX_KERNEL", "split")
    assert bsfp8.bsmxfp8_plan(8192, 1) == {"kernel": "split", "token_rows": 128,
                                           "split_rows": 256}
    monkeypatch.delenv("BSFP8_MX_TN")
    assert bsfp8.bsmxfp8_plan(8192, 1)["token_rows"] == 64
    monkeypatch.setenv("BSFP8_MX_KERNEL", "pair")
    assert bsfp8.bsmxfp8_plan(100, 100)["kernel"] == "pair"


def test_bad_input():
    lib = bsfp8.load_library()
    assert lib.bsmxfp8_plan(10, 1, None) == 1  # BSFP8_ERR_NULL
    with pytest.raises(bsfp8.BsFp8Error):
        bsfp8.bsmxfp8_plan(10, 0)
    with pytest.raises(bsfp8.BsFp8Error):
        bsfp8.bsmxfp8_plan(-1, 4)


@pytest.mark.parametrize("M,G,kernel,rows", [
    (2091, 128, "swap", 32),     # decode: 1..32 tokens per expert
    (8 * 64, 8, "swap", 64),
    (8 * 128, 8, "swap", 128),   # 128 per group: one 128-token swap-AB tile still holds it
    (8 * 128 + 1, 8, "pair", 0),
    (8192, 1, "pair", 0),        # dense prefill
    (0, 4, "swap", 32),
])
def test_fp4_plan_bands(M, G, kernel, rows, monkeypatch):
    # the fp4 formats' own threshold: CTA-pair tiles above 128 rows per group on average
    monkeypatch.delenv("BSFP8_FP4_MMA", raising=False)
    assert bsfp8.bsmx_plan(M, G) == {"kernel": kernel, "token_rows": rows}
    # the MXFP8 plan keeps its own bands (CTA pair above 56 rows per expert)
    if M == 8 * 64:
        assert bsfp8.bsmxfp8_plan(M, G)["kernel"] == "pair"


def test_fp4_plan_overrides(monkeypatch):
    monkeypatch.delenv("BSFP8_FP4_MMA", raising=False)
    monkeypatch.setenv("BSFP8_MX_KERNEL", "pair")
    assert bsfp8.bsmx_plan(100, 8)["kernel"] == "pair"
    monkeypatch.setenv("BSFP8_MX_KERNEL", "split")  # no split for the fp4 forms: swap-AB
    assert bsfp8.bsmx_plan(8192, 1) == {"kernel": "swap", "token_rows": 128}
    monkeypatch.delenv("BSFP8_MX_KERNEL")
    monkeypatch.setenv("BSFP8_MX_TN", "32")
    assert bsfp8.bsmx_plan(8 * 100, 8) == {"kernel": "swap", "token_rows": 32}
    monkeypatch.delenv("BSFP8_MX_TN")
    # the converting forms: swap-AB tiles only, at most 64 token rows
    monkeypatch.setenv("BSFP8_FP4_MMA", "convert")
    assert bsfp8.bsmx_plan(8192, 1) == {"kernel": "swap", "token_rows": 64}
    assert bsfp8.bsmx_plan(8 * 16, 8) == {"kernel": "swap", "token_rows": 32}


def test_fp4_plan_rejects_bad_input():
    with pytest.raises(bsfp8.BsFp8Error):
        bsfp8.bsmx_plan(-1, 8)
    with pytest.raises(bsfp8.BsFp8Error):
        bsfp8.bsmx_plan(100, 0)
