"""Routing requests over independent replicas (oracle).

Source: InfoQ release note on DeepSpeed-FastGen - throughput scales with the
number of replicas placed behind a load balancer (16 replicas reached 23.7
queries/s).  The note names no policy.  Reading taken here: each replica is a
whole serving instance (one GPU, its own composer and KV cache), and a new
request goes to the replica with the least outstanding work, counted in
tokens: for every request it holds, the prompt tokens not yet prefilled plus
the output tokens not yet generated.  Ties go to the replica holding fewer
requests, then to the lowest index.

Written as the plain definition: loads are recomputed from the held requests
at every decision, with no running totals.
"""
from __future__ import annotations

from typing import Dict, List


class Router:
    def __init__(self, num_replicas: int):
        if num_replicas < 1:
            raise ValueError("num_replicas must be >= 1")
        self.num_replicas = int(num_replicas)
        # request id -> [replica, outstanding tokens]
        self.held: Dict[int, List[int]] = {}

    def load(self, replica: int) -> int:
        return sum(t for r, t in self.held.values() if r == replica)

    def active(self, replica: int) -> int:
        return sum(1 for r, _ in self.held.values() if r == replica)

    def assign(self, request_id: int, prompt_len: int, output_len: int) -> int:
        if prompt_len < 1 or output_len < 1:
            raise ValueError("prompt_len and output_len must be >= 1")
        if request_id in self.held:
            raise ValueError("request id already routed")
        keys = [(self.load(i), self.active(i), i) for i in range(self.num_replicas)]
        best = min(keys)[2]
        self.held[request_id] = [best, prompt_len + output_len]
        return best

    def progress(self, request_id: int, tokens: int) -> None:
        entry = self.held[request_id]
        if tokens < 0 or tokens > entry[1]:
            raise ValueError("tokens must be in [0, outstanding]")
        entry[1] -= tokens

    def finish(self, request_id: int) -> None:
        del self.held[request_id]
