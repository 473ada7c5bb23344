"""Serving metrics of a trace (TTFT, pace, effective throughput), CPU only.

Timelines small enough to work out by hand: each expected value below is
derived in the comments from the SplitFuse rules (generation first, then
prompt chunks, list order) and the recorded pass end times."""
import pytest

import oracle
import workloads
from ragged_blocked_kv_gb300.serving import TraceRecorder, serving_metrics


def _run(reqs, clients, budget, max_chunk):
    comp = oracle.Composer(16, workloads.trace_block_pool(reqs, clients, 16))
    rec = TraceRecorder()
    n = workloads.run_trace(reqs, clients, budget, max_chunk, comp.compose, comp.release,
                            on_pass=rec.on_pass)
    return rec, n


def test_one_client_two_requests():
    # A (prompt 5, output 3) then B (prompt 2, output 1), budget 4:
    # pass 0: A prompt 0..3; pass 1: A prompt 4 -> token 1; passes 2, 3: tokens
    # 2, 3 (A done, B arrives at the end of pass 3); pass 4: B prompt -> token 1.
    reqs = [workloads.Request(1, 0, 5, 3), workloads.Request(2, 0, 2, 1)]
    rec, n = _run(reqs, 1, 4, 4)
    assert n == 5
    assert rec.first_seen == {1: 0, 2: 4}
    assert rec.token_passes == {1: [1, 2, 3], 2: [4]}
    end = [10.0, 25.0, 30.0, 42.0, 50.0]
    # A: TTFT 25, gaps 5 and 12 -> pace 8.5; B: TTFT 50 - 42 = 8, pace 0
    m = serving_metrics(rec, end, ttft_sla_ms=20.0, pace_sla_ms=10.0)
    assert m["requests"] == 2 and m["sla"]["met"] == 1           # A misses TTFT
    assert m["makespan_s"] == pytest.approx(0.05)
    assert m["effective_rps"] == pytest.approx(20.0) and m["rps"] == pytest.approx(40.0)
    assert m["ttft_ms"]["mean"] == pytest.approx((25 + 8) / 2)
    assert m["pace_ms"]["mean"] == pytest.approx(8.5 / 2)
    assert m["token_interval_ms"]["max"] == 12.0
    assert serving_metrics(rec, end, 30.0, 8.0)["sla"]["met"] == 1   # A misses pace
    assert serving_metrics(rec, end, 30.0, 9.0)["sla"]["met"] == 2


def test_waiting_request_keeps_its_arrival():
    # two clients, budget 1, A and B both (prompt 1, output 2):
    # pass 0: A prompt -> token 1 (B waits); pass 1: A decodes first -> token 2,
    # done; pass 2: B prompt -> token 1; pass 3: B token 2.
    reqs = [workloads.Request(1, 0, 1, 2), workloads.Request(2, 1, 1, 2)]
    rec, n = _run(reqs, 2, 1, 0)
    assert n == 4
    assert rec.first_seen == {1: 0, 2: 0}
    assert rec.token_passes == {1: [0, 1], 2: [2, 3]}
    m = serving_metrics(rec, [1.0, 2.0, 3.0, 4.0], 2.0, 1.0)
    # A: TTFT 1, pace 1; B: arrived at 0, TTFT 3 -> misses
    assert m["ttft_ms"]["p50"] == 1.0 and m["ttft_ms"]["p99"] == 3.0
    assert m["sla"]["met"] == 1


def test_trace_conservation():
    """Every request of the standard trace yields output_len tokens, one per
    pass, the first in the pass that completes its prompt."""
    reqs = workloads.trace_requests(seed=3, num_requests=64, num_clients=8)
    want = {r.seq_id: r.output_len for r in reqs}
    rec, n = _run(reqs, 8, 512, 512)
    assert {k: len(v) for k, v in rec.token_passes.items()} == want
    for v in rec.token_passes.values():
        assert all(b > a for a, b in zip(v, v[1:]))
    m = serving_metrics(rec, [float(i + 1) for i in range(n)], 1e9, 1e9)
    assert m["sla"]["met"] == 64
    # at one ms per pass, a request's pace is at least one pass per token
    assert m["pace_ms"]["p50"] >= 1.0 and m["token_interval_ms"]["p50"] >= 1.0


def test_missing_pass_times_rejected():
    reqs = [workloads.Request(1, 0, 5, 3)]
    rec, n = _run(reqs, 1, 4, 4)
    with pytest.raises(ValueError):
        serving_metrics(rec, [1.0] * (n - 1), 1.0, 1.0)
