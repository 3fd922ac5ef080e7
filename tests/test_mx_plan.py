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
