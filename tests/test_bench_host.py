"""Host-side logic of bench.py: the reference arm's JSON line (CPU oracle) and the
max-over-ranks aggregation of replicas, run as two gloo ranks on the CPU."""
import json
import os
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "0", "--steps", "2", "--warmup", "3", "--ref-budget", "2"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["steps"] == 2 and line["warmup"] == 3 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.dist_init(world, "gloo")
    ms, flops = bench.aggregate(dist, 1.0 + rank, 10.0 * (rank + 1))
    bench.barrier(dist)
    q.put((rank, ms, flops))
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    # max of the step times, sum of the work, identical on every rank
    assert out == [(0, 2.0, 30.0), (1, 2.0, 30.0)]


def test_kernel_hash_ignores_comments_only():
    sys.path.insert(0, ROOT)
    import bench
    src = 'int a = 1; // one\n/* block\n comment */ const char* s = "x // y";\n\n'
    assert bench.strip_comments(src) == 'int a = 1;\n const char* s = "x // y";'
    names = bench.KERNEL_SOURCES[bench.WORKLOAD_KERNEL["config4"]]
    base = {n: f"int f_{i}() {{ return {i}; }}\n" for i, n in enumerate(names)}
    commented = {n: "// header\n/* a block\n   comment */\n" + t.replace("\n", "  // why\n")
                 for n, t in base.items()}
    changed = dict(base)
    changed[names[-1]] = base[names[-1]].replace("return", "return 1 +")
    h = bench.kernel_hash("config4", base)
    assert bench.kernel_hash("config4", commented) == h
    assert bench.kernel_hash("config4", changed) != h


def test_traffic_read_from_the_workloads_own_section(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    h = bench.kernel_hash("fp4:nvfp4xnvfp4")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "two.txt").write_text(
        f"kernel_sources_sha256_12: {h}\n"
        "workload_key: fp4:mxfp8xmxfp4\ndram_bytes_per_launch: 111\n"
        "workload_key: fp4:nvfp4xnvfp4\ndram_bytes_per_launch: 222\n")
    (tmp_path / "profiles" / "stale.txt").write_text(
        "kernel_sources_sha256_12: 000000000000\nworkload_key: config5\n"
        "dram_bytes_per_launch: 333\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_hash", lambda key, sources=None: h)
    assert bench.traffic_from_profiles("fp4:mxfp8xmxfp4") == (111.0, "two.txt")
    assert bench.traffic_from_profiles("fp4:nvfp4xnvfp4") == (222.0, "two.txt")
    assert bench.traffic_from_profiles("config5") == (None, None)   # recorded hash differs


def test_sample_parity_matches_the_tests_bound():
    # the bench's check of the CPU baseline's rows uses the parity tests' acceptance bound:
    # a planted one-element error (in a copy of the oracle's result) is found by both
    import numpy as np
    import bench
    import gen
    import oracle
    from helpers import parity_report
    p = gen.config_problem(0)
    _, _, _, (rows, ref, T) = oracle.timed_rows(p, 24, keep=True)
    assert rows.size == 24 and ref.shape == (24, p.N) == T.shape
    ok = bench.sample_parity(ref, ref, T)
    assert ok["outside_bound"] == 0 and ok["bit_identical"] == ref.size
    bad = ref.copy()
    bad[3, 17] ^= 0x20
    bad[20, 200] ^= 0x01
    got = bench.sample_parity(bad, ref, T)
    n_bad, ratio, exact = parity_report(bad, ref, T)
    assert got["outside_bound"] == n_bad >= 1
    assert got["bit_identical"] == exact == ref.size - 2
    assert abs(got["max_err_over_bound"] - ratio) < 1e-12
