"""Host-side timing of the oracle baseline: the start barrier of the
concurrent workers and the all-cores aggregate (CPU only)."""
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
