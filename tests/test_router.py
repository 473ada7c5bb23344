"""Routing over replicas: the library's router against the oracle's, the
oracle pinned by hand-derived decisions and the greedy balance bound, and the
multi-replica serving loop - in one process and over gloo ranks (rank 0 the
router, ranks 1..N the replicas) - conserving every request and token."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle.router as orouter
import workloads


# ---- the oracle against what the policy fixes by hand ------------------------

def test_oracle_hand_derived_decisions():
    r = orouter.Router(3)
    # empty replicas tie on load and held requests: the lowest index
    assert r.assign(1, 100, 10) == 0          # loads 110, 0, 0
    assert r.assign(2, 50, 5) == 1            # 110, 55, 0
    assert r.assign(3, 20, 2) == 2            # 110, 55, 22
    assert r.assign(4, 10, 1) == 2            # 110, 55, 33
    assert r.assign(5, 30, 1) == 2            # 110, 55, 64
    assert [r.load(i) for i in range(3)] == [110, 55, 64]
    r.progress(1, 100)                         # replica 0 prefilled: 10 left
    assert r.assign(6, 1, 1) == 0              # 12, 55, 64
    r.finish(2)                                # replica 1 empty: 0 tokens, 0 held
    assert r.assign(7, 12, 0 + 1) == 1         # 12, 13, 64
    # equal loads: fewer requests held wins (replica 1 holds one, replica 0 two)
    r.progress(7, 1)                           # 12, 12, 64
    assert r.assign(8, 5, 5) == 1
    with pytest.raises(ValueError):
        r.assign(8, 1, 1)                      # already routed
    with pytest.raises(ValueError):
        r.progress(1, 11)                      # more than outstanding


def test_oracle_greedy_balance_bound():
    """With no progress reported, least-loaded assignment keeps every load
    within the largest request of the least one (list scheduling)."""
    rng = np.random.default_rng(1)
    for n in (2, 3, 5, 8):
        r = orouter.Router(n)
        biggest = 0
        for i in range(300):
            p, g = int(rng.integers(1, 4000)), int(rng.integers(1, 200))
            r.assign(i, p, g)
            biggest = max(biggest, p + g)
            loads = [r.load(k) for k in range(n)]
            assert max(loads) - min(loads) <= biggest


# ---- the library's router against the oracle ---------------------------------

def test_library_router_matches_oracle(rbkv):
    rng = np.random.default_rng(7)
    for n in (1, 2, 4, 7):
        lib = rbkv.Router(n)
        orc = orouter.Router(n)
        live = {}
        nid = 0
        for _ in range(2000):
            op = rng.integers(0, 3)
            if op == 0 or not live:
                p, g = int(rng.integers(1, 3000)), int(rng.integers(1, 120))
                assert lib.assign(nid, p, g) == orc.assign(nid, p, g)
                live[nid] = p + g
                nid += 1
            elif op == 1:
                sid = int(rng.choice(list(live)))
                t = int(rng.integers(0, live[sid] + 1))
                lib.progress(sid, t)
                orc.progress(sid, t)
                live[sid] -= t
            else:
                sid = int(rng.choice(list(live)))
                lib.finish(sid)
                orc.finish(sid)
                del live[sid]
            for k in range(n):
                assert lib.load(k) == orc.load(k) and lib.active(k) == orc.active(k)
        with pytest.raises(rbkv.RbkvError):
            lib.finish(10 ** 9)


# ---- serving over replicas --------------------------------------------------

def _config(rbkv, reqs, clients):
    nb = workloads.trace_block_pool(reqs, clients, 64)
    return rbkv.Config(32, 32, 128, 64, "bf16", nb)


def _check_summary(reqs, s, n):
    assert s["requests"] == len(reqs)
    assert all(r.finish is not None and r.first_token is not None for r in reqs)
    assert sorted(sid for sid, _ in s["assignments"]) == sorted(r.seq_id for r in reqs)
    # every replica's pass tokens are exactly its requests' P + G - 1
    per = [0] * n
    for r in reqs:
        per[r.replica] += r.prompt_len + r.output_len - 1
    assert per == s["tokens"]
    # closed loop: a client's requests run one after another
    for c in {r.client for r in reqs}:
        mine = [r for r in reqs if r.client == c]
        for a, b in zip(mine, mine[1:]):
            assert b.arrival == a.finish and a.first_token <= a.finish


@pytest.mark.parametrize("n", [1, 3, 4])
def test_serve_in_process(rbkv, n):
    from ragged_blocked_kv_gb300 import replicas
    clients = 8 * n
    reqs = replicas.trace(3, clients, per_client=4)
    s = replicas.serve(rbkv, reqs, clients, n, _config(rbkv, reqs, clients))
    _check_summary(reqs, s, n)
    if n > 1:
        assert s["token_imbalance"] < 1.25, s["token_imbalance"]
    again = replicas.trace(3, clients, per_client=4)
    s2 = replicas.serve(rbkv, again, clients, n, _config(rbkv, again, clients))
    assert s2["assignments"] == s["assignments"] and s2["makespan_ms"] == s["makespan_ms"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _dist_worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    import ragged_blocked_kv_gb300 as rbkv
    from ragged_blocked_kv_gb300 import replicas
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    clients = 8 * (world - 1)
    reqs = replicas.trace(5, clients, per_client=4)
    nb = workloads.trace_block_pool(reqs, clients, 64)
    cfg = rbkv.Config(32, 32, 128, 64, "bf16", nb)
    s = replicas.serve_distributed(rbkv, reqs, clients, cfg)
    if rank == 0:
        out[0] = (s, [(r.seq_id, r.replica, r.arrival, r.first_token, r.finish) for r in reqs])
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_serve_over_gloo_ranks_matches_one_process(rbkv, world):
    from ragged_blocked_kv_gb300 import replicas
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_dist_worker, args=(world, port, out), nprocs=world, join=True)
        s_dist, rows = out[0]
    n = world - 1
    clients = 8 * n
    reqs = replicas.trace(5, clients, per_client=4)
    s = replicas.serve(rbkv, reqs, clients, n, _config(rbkv, reqs, clients))
    assert s_dist["assignments"] == s["assignments"]
    assert s_dist["tokens"] == s["tokens"] and s_dist["passes"] == s["passes"]
    assert rows == [(r.seq_id, r.replica, r.arrival, r.first_token, r.finish) for r in reqs]
