"""Host-side helpers of the benchmark (CPU only): the oracle baseline's start
barrier, all-cores aggregate and row sampling, and the rule that recorded DRAM
traffic is reported only for the kernel source it was captured on."""
import os
import types

import bench


def test_barrier_releases_once_all_workers_are_ready(tmp_path):
    (tmp_path / "ready_other").write_text("")
    assert bench._barrier(str(tmp_path), 2, limit_s=5.0)


def test_barrier_gives_up_after_its_limit(tmp_path):
    assert not bench._barrier(str(tmp_path), 2, limit_s=0.05)


def test_concurrent_workers_start_together_and_aggregate():
    args = types.SimpleNamespace(workload="decode_stress", seed=0)
    # a per-worker size that lets half the free memory hold two workers
    res = bench.cpu_all_cores(args, worker_bytes=int(bench._mem_available() * 0.5 / 2.5),
                              steps=1, warmup=1)
    assert res["value"] and res["value"] > 0, res
    assert res["cores"] == min(2, len(os.sched_getaffinity(0)))
    assert res["synced"]


def test_offset_moves_the_first_output_pair():
    import workloads
    scn = workloads.SCENARIOS["tiny"](0)
    a = bench.OracleRunner(scn, 0, offset=0)
    b = bench.OracleRunner(scn, 0, offset=7)
    assert (a.cursor, b.cursor) == (0, 7)
    a.step(5)
    b.step(5)
    assert (a.cursor, b.cursor) == (5, 12)


def test_traffic_is_reported_only_for_the_captured_source(monkeypatch):
    import hashlib
    path = os.path.join(bench.ROOT, "ragged_blocked_kv_gb300", "csrc", "rbkv_decode.cu")
    with open(path, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:12]
    monkeypatch.setattr(bench, "TRAFFIC_BYTES", {
        ("w", "decode"): ("rbkv_decode.cu", sha, 123),
        ("w", "stale"): ("rbkv_decode.cu", "000000000000", 456),
        ("w", "missing"): ("no_such_file.cu", sha, 789),
    })
    assert bench.traffic_bytes("w", "decode") == 123
    assert bench.traffic_bytes("w", "stale") is None
    assert bench.traffic_bytes("w", "missing") is None
    assert bench.traffic_bytes("other", "decode") is None


def test_cpu_model_is_named():
    assert bench.cpu_model()


def test_sampled_rows_are_a_permutation_spread_over_the_pass():
    """The oracle sample walks a pass's rows in a stride permutation: every
    row exactly once per T rows, and the first few rows already spread over
    the pass (its first and last quarters both reached)."""
    for T in (1, 2, 7, 64, 512, 2048, 2111, 12288):
        rows = [bench.sample_row(i, T) for i in range(T)]
        assert sorted(rows) == list(range(T)), T
        if T >= 64:
            head = rows[:8]
            assert min(head) < T // 4 and max(head) >= 3 * T // 4, (T, head)
