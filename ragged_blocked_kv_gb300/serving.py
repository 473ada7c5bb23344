"""User-facing serving metrics of a closed-loop trace of SplitFuse passes.

Source: DeepSpeed-FastGen paper summary page, Key points and idea I4 - rate a
chat service by an "effective throughput" tied to time to first token (TTFT)
and how regularly the following tokens arrive, and report token-level tail
latency; the FastGen guide's benchmark table reports TTFT P90, per-token P99
latency and requests per second served within a per-token latency bound.

Readings (the pages define no formula):

* A request arrives when its client's previous request finishes, i.e. at the
  end of the pass in which that one produced its last token (closed loop, no
  think time); the first requests arrive at time 0.  In pass terms, a request
  first listed in pass k arrived at the end of pass k-1 (0 for k = 0).
* Output token 1 appears at the end of the pass that completes the prompt;
  each later pass that schedules the request appears one more token.
* TTFT = time of token 1 - arrival.  The pace of a request is the mean interval
  between its successive tokens (0 for a one-token answer).
* A request meets the service level when TTFT <= ttft_sla_ms and its pace <=
  pace_sla_ms; effective throughput = such requests / the trace's makespan.

This module is bookkeeping on pass indices and pass end times only.
"""
from __future__ import annotations

from typing import Dict, List, Sequence


class TraceRecorder:
    """Record, per request, when it arrived and in which passes it produced
    output tokens.  Pass ``on_pass`` as the per-pass hook of the trace loop: it
    must see the pass's schedule before the request states advance."""

    def __init__(self):
        self.first_seen: Dict[int, int] = {}
        self.token_passes: Dict[int, List[int]] = {}
        self.passes = 0

    def on_pass(self, npass: int, meta, active) -> None:
        sched = dict(zip([int(s) for s in meta.seq_ids], [int(n) for n in meta.n_new]))
        for r in active:
            self.first_seen.setdefault(r.seq_id, npass)
            n = sched.get(r.seq_id, 0)
            if n == 0:
                continue
            if r.seen < r.prompt_len:
                if r.seen + n >= r.prompt_len:
                    self.token_passes.setdefault(r.seq_id, []).append(npass)
            else:
                self.token_passes.setdefault(r.seq_id, []).append(npass)
        self.passes = max(self.passes, npass + 1)


def _pct(sorted_x: Sequence[float], q: float) -> float:
    if not sorted_x:
        return 0.0
    return float(sorted_x[min(len(sorted_x) - 1, int(round(q / 100.0 * (len(sorted_x) - 1))))])


def serving_metrics(rec: TraceRecorder, pass_end_ms: Sequence[float], ttft_sla_ms: float,
                    pace_sla_ms: float) -> dict:
    """TTFT, token intervals and effective throughput from ``rec`` and the end
    time of every pass (ms from the start of the trace, non-decreasing)."""
    if len(pass_end_ms) < rec.passes:
        raise ValueError("need an end time for every recorded pass")
    ttft, pace, gaps = [], [], []
    met = 0
    for sid, first in rec.first_seen.items():
        toks = rec.token_passes.get(sid, [])
        if not toks:
            continue                        # still prefilling when the trace stopped
        arrival = 0.0 if first == 0 else float(pass_end_ms[first - 1])
        t = [float(pass_end_ms[k]) for k in toks]
        tt = t[0] - arrival
        g = [b - a for a, b in zip(t, t[1:])]
        pc = sum(g) / len(g) if g else 0.0
        ttft.append(tt)
        pace.append(pc)
        gaps.extend(g)
        if tt <= ttft_sla_ms and pc <= pace_sla_ms:
            met += 1
    span_s = float(pass_end_ms[rec.passes - 1]) / 1e3 if rec.passes else 0.0
    ttft.sort()
    pace.sort()
    gaps.sort()
    return {
        "requests": len(ttft),
        "ttft_ms": {"p50": _pct(ttft, 50), "p90": _pct(ttft, 90), "p99": _pct(ttft, 99),
                    "mean": sum(ttft) / len(ttft) if ttft else 0.0},
        "pace_ms": {"p50": _pct(pace, 50), "p90": _pct(pace, 90), "p99": _pct(pace, 99),
                    "mean": sum(pace) / len(pace) if pace else 0.0},
        "token_interval_ms": {"p50": _pct(gaps, 50), "p95": _pct(gaps, 95),
                              "p99": _pct(gaps, 99), "max": gaps[-1] if gaps else 0.0},
        "sla": {"ttft_ms": ttft_sla_ms, "pace_ms": pace_sla_ms, "met": met},
        "effective_rps": met / span_s if span_s > 0 else 0.0,
        "rps": len(ttft) / span_s if span_s > 0 else 0.0,
        "makespan_s": span_s,
    }
