"""Serving over several independent replicas behind a router.

InfoQ release note on DeepSpeed-FastGen: throughput grows with the number of
replicas behind a load balancer (16 replicas, 23.7 queries/s).  A replica here
is a whole serving instance: its own GPU, composer, block pool and KV caches.
Replicas share nothing on the data path; the router (the library's
``rbkv_router``: the replica with the fewest outstanding tokens takes the next
request) only decides where a request goes.

``serve`` runs a closed-loop trace over N replicas as a discrete-event
simulation on the host: each replica composes its own SplitFuse passes with
the library's composer, and a pass of T tokens takes the time a measured
latency profile predicts for T tokens (the library's piecewise-linear
predictor).  The replica whose clock is earliest composes next; a request
arrives when its client's previous request ends; the router is told the tokens
each pass consumed (the pass completing a prompt also yields output token 1)
and each request's end.  ``serve_distributed`` runs the same loop with the
router on rank 0 and replica r on rank r + 1 of a ``torch.distributed`` group:
only control messages (requests in, pass reports out) cross processes, in the
same order, so both give the same results.

Run ``python -m ragged_blocked_kv_gb300.replicas`` for the scaling of the trace
with the number of replicas (32 clients per replica).
"""
from __future__ import annotations

import argparse
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence, Tuple

# Pass latency (ms) against pass tokens of 32 Llama-2-7B decoder layers
# (random weights; this library's append and attention, cuBLAS projections),
# one CUDA-graph replay per pass, measured with this library on one GB300
# (bench.py --workload profile --layer full).
PROFILE_TOKENS = [16, 64, 256, 512, 768, 1024, 1536, 2048, 3072, 4096]
PROFILE_MS = [3.27, 3.38, 4.20, 5.91, 7.93, 9.80, 14.36, 19.01, 28.42, 39.71]


@dataclass
class Request:
    seq_id: int
    client: int
    prompt_len: int
    output_len: int
    arrival: float = 0.0
    seen: int = 0
    generated: int = 0
    first_token: Optional[float] = None
    finish: Optional[float] = None
    replica: int = -1


class Replica:
    """One serving instance: a composer over the requests routed to it, in
    arrival order, and a clock advanced by the predicted latency of each pass."""

    def __init__(self, rbkv, config, budget: int, max_chunk: int,
                 latency: Callable[[int], float]):
        self.rbkv = rbkv
        self.comp = rbkv.Composer(config)
        self.budget, self.max_chunk = budget, max_chunk
        self.latency = latency
        self.active: List[Request] = []
        self.clock = 0.0
        self.passes = 0
        self.tokens = 0

    def add(self, req: Request) -> None:
        if not self.active:
            self.clock = max(self.clock, req.arrival)
        self.active.append(req)

    def has_work(self) -> bool:
        return bool(self.active)

    def step(self) -> dict:
        """Compose and run one pass; returns what the router must learn: the
        tokens each request consumed and the requests that ended (with the
        pass's end time)."""
        states = [(r.seq_id, r.prompt_len, r.seen) for r in self.active]
        p = self.comp.compose(self.budget, self.max_chunk, states)
        meta = p.meta
        T = p.num_tokens
        p.destroy()
        self.clock += self.latency(T)
        self.passes += 1
        self.tokens += T
        sched = dict(zip([int(s) for s in meta.seq_ids], [int(n) for n in meta.n_new]))
        progress, finished = [], []
        for r in self.active:
            n = sched.get(r.seq_id, 0)
            if n == 0:
                continue
            prefill = r.seen < r.prompt_len
            r.seen += n
            if prefill:
                used = n
                if r.seen >= r.prompt_len:
                    r.generated = 1
                    r.first_token = self.clock
                    used += 1
            else:
                r.generated += 1
                used = 1
            progress.append((r.seq_id, used))
            if r.generated >= r.output_len:
                r.finish = self.clock
                finished.append(r)
        for r in finished:
            self.active.remove(r)
            self.comp.release(r.seq_id)
        return {"tokens": T, "clock": self.clock, "progress": progress,
                "finished": [(r.seq_id, r.first_token, r.finish) for r in finished]}


def profile_latency(rbkv, tokens: Sequence[int] = PROFILE_TOKENS,
                    ms: Sequence[float] = PROFILE_MS) -> Callable[[int], float]:
    """Pass latency (ms) predicted from a (tokens, ms) profile by the library;
    passes below the profile's first point take its latency."""
    import ctypes as C
    n = len(tokens)
    t = (C.c_int32 * n)(*[int(x) for x in tokens])
    l = (C.c_double * n)(*[float(x) for x in ms])
    lo, hi = int(tokens[0]), int(tokens[-1])

    def latency(T: int) -> float:
        if T <= 0:
            return 0.0
        x = min(max(int(T), lo), hi)
        v = float(rbkv.lib().rbkv_latency_at(t, l, n, x))
        return v * (T / hi) if T > hi else v
    return latency


def _clients(reqs: Sequence[Request], num_clients: int) -> Dict[int, List[Request]]:
    return {c: [r for r in reqs if r.client == c] for c in range(num_clients)}


class _Loop:
    """The event loop shared by both drivers.  ``run(k, new)`` hands the
    requests `new` to replica k, runs one pass there and returns its report."""

    def __init__(self, rbkv, reqs: Sequence[Request], num_clients: int, num_replicas: int):
        self.router = rbkv.Router(num_replicas)
        self.queues = _clients(reqs, num_clients)
        self.by_id = {r.seq_id: r for r in reqs}
        self.pending: List[List[Request]] = [[] for _ in range(num_replicas)]
        self.clock = [0.0] * num_replicas
        self.work = [0] * num_replicas      # requests held by each replica
        self.n = num_replicas
        self.assignments: List[Tuple[int, int]] = []
        for c in range(num_clients):
            if self.queues[c]:
                self._arrive(self.queues[c].pop(0), 0.0)

    def _arrive(self, req: Request, t: float) -> None:
        req.arrival = t
        k = self.router.assign(req.seq_id, req.prompt_len, req.output_len)
        req.replica = k
        self.assignments.append((req.seq_id, k))
        if self.work[k] == 0:
            self.clock[k] = max(self.clock[k], t)
        self.work[k] += 1
        self.pending[k].append(req)

    def drive(self, run: Callable[[int, List[Request]], dict]) -> None:
        while True:
            ks = [k for k in range(self.n) if self.work[k] > 0]
            if not ks:
                break
            k = min(ks, key=lambda i: (self.clock[i], i))
            new, self.pending[k] = self.pending[k], []
            rep = run(k, new)
            self.clock[k] = rep["clock"]
            for sid, used in rep["progress"]:
                self.router.progress(sid, used)
            for sid, first, fin in sorted(rep["finished"], key=lambda x: self.by_id[x[0]].client):
                req = self.by_id[sid]
                req.first_token, req.finish = first, fin
                self.router.finish(sid)
                self.work[k] -= 1
                if self.queues[req.client]:
                    self._arrive(self.queues[req.client].pop(0), fin)


def serve(rbkv, reqs: Sequence[Request], num_clients: int, num_replicas: int, config,
          budget: int = 512, max_chunk: int = 512,
          latency: Optional[Callable[[int], float]] = None) -> dict:
    """Serve ``reqs`` (closed loop, ``num_clients`` clients) on ``num_replicas``
    replicas in this process.  Returns the summary of ``summarize``."""
    latency = latency or profile_latency(rbkv)
    replicas = [Replica(rbkv, config, budget, max_chunk, latency) for _ in range(num_replicas)]
    loop = _Loop(rbkv, reqs, num_clients, num_replicas)

    def run(k, new):
        for r in new:
            replicas[k].add(r)
        return replicas[k].step()
    loop.drive(run)
    return summarize(reqs, loop, [(r.passes, r.tokens) for r in replicas])


def serve_distributed(rbkv, reqs: Sequence[Request], num_clients: int, config,
                      budget: int = 512, max_chunk: int = 512,
                      latency: Optional[Callable[[int], float]] = None) -> Optional[dict]:
    """``serve`` over a ``torch.distributed`` group: rank 0 runs the router and
    the clients, rank r + 1 runs replica r.  Returns the summary on rank 0,
    None elsewhere."""
    import torch.distributed as dist
    rank, world = dist.get_rank(), dist.get_world_size()
    n = world - 1
    if n < 1:
        raise ValueError("needs at least one replica rank besides rank 0")
    latency = latency or profile_latency(rbkv)
    if rank > 0:
        rep = Replica(rbkv, config, budget, max_chunk, latency)
        while True:
            msg = [None]
            dist.recv_object_list(msg, src=0)
            kind, payload = msg[0]
            if kind == "stop":
                dist.send_object_list([(rep.passes, rep.tokens)], dst=0)
                return None
            for r in payload:
                rep.add(Request(**r))
            dist.send_object_list([rep.step()], dst=0)
    loop = _Loop(rbkv, reqs, num_clients, n)

    def run(k, new):
        payload = [dict(seq_id=r.seq_id, client=r.client, prompt_len=r.prompt_len,
                        output_len=r.output_len, arrival=r.arrival) for r in new]
        dist.send_object_list([("step", payload)], dst=k + 1)
        out = [None]
        dist.recv_object_list(out, src=k + 1)
        return out[0]
    loop.drive(run)
    stats = []
    for k in range(n):
        dist.send_object_list([("stop", None)], dst=k + 1)
        out = [None]
        dist.recv_object_list(out, src=k + 1)
        stats.append(out[0])
    return summarize(reqs, loop, stats)


def summarize(reqs: Sequence[Request], loop: _Loop, replica_stats) -> dict:
    done = [r for r in reqs if r.finish is not None]
    makespan = max(r.finish for r in done) if done else 0.0
    ttft = sorted(r.first_token - r.arrival for r in done)
    tokens = [t for _, t in replica_stats]
    mean_t = sum(tokens) / len(tokens)
    return {
        "requests": len(done),
        "makespan_ms": makespan,
        "requests_per_s": len(done) / (makespan / 1e3) if makespan else 0.0,
        "ttft_p50_ms": ttft[len(ttft) // 2] if ttft else 0.0,
        "ttft_p99_ms": ttft[min(len(ttft) - 1, int(0.99 * (len(ttft) - 1)))] if ttft else 0.0,
        "passes": [p for p, _ in replica_stats],
        "tokens": tokens,
        "token_imbalance": max(tokens) / mean_t if mean_t else 1.0,
        "assignments": list(loop.assignments),
    }


def trace(seed: int, num_clients: int, per_client: int = 16) -> List[Request]:
    """The trace workload's request lengths (512 requests, 32 clients at the
    default scale), ``per_client`` requests for each of ``num_clients``."""
    import workloads
    base = workloads.trace_requests(seed=seed, num_requests=num_clients * per_client,
                                    num_clients=num_clients)
    return [Request(r.seq_id, r.client, r.prompt_len, r.output_len) for r in base]


def main() -> None:
    import os
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import ragged_blocked_kv_gb300 as rbkv
    import workloads
    ap = argparse.ArgumentParser()
    ap.add_argument("--replicas", type=int, nargs="+", default=[1, 2, 4, 8, 16])
    ap.add_argument("--clients-per-replica", type=int, default=32)
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args()
    for n in args.replicas:
        clients = n * args.clients_per_replica
        reqs = trace(args.seed, clients)
        nb = workloads.trace_block_pool(reqs, clients, 64)
        cfg = rbkv.Config(32, 32, 128, 64, "bf16", nb)
        s = serve(rbkv, reqs, clients, n, cfg)
        print(f"replicas {n:3d}  clients {clients:4d}  requests {s['requests']:5d}  "
              f"{s['requests_per_s']:7.2f} req/s  TTFT p50 {s['ttft_p50_ms']:7.1f} ms  "
              f"p99 {s['ttft_p99_ms']:7.1f} ms  token imbalance {s['token_imbalance']:.3f}")


if __name__ == "__main__":
    main()
