"""Pins for the oracle's Dynamic SplitFuse composer (CPU only).

What the pages fix: every pass holds exactly the token budget when there is
enough demand (paper summary page, Summary: passes are topped up to the whole
budget); long
prompts are spread over passes in chunks; generation tokens ride along in every
pass (FastGen guide, "Prompt-Decode Decoupling").  The tiny workload statement
fixes its pass's token counts (40 + 3 + 21).
"""
import json
import os

import numpy as np
import pytest

import workloads
from oracle import Composer, InvalidRequest, NoBlocks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_pass.json")


def _as_dict(meta):
    return {k: list(getattr(meta, k)) for k in
            ("seq_ids", "q_start", "n_new", "seen", "ctx", "block_start", "block_ids")}


def test_tiny_worked_pass():
    g = json.load(open(GOLDEN))
    c = Composer(16, 64)
    r = g["registration"]
    c.compose(r["budget"], r["max_chunk"], [tuple(s) for s in r["states"]])
    p = g["pass"]
    meta = c.compose(p["budget"], p["max_chunk"], [tuple(s) for s in p["states"]])
    assert _as_dict(meta) == g["expected"]
    assert meta.num_tokens == 64
    # slot = block * B + offset for every token, in pass order
    B = 16
    t = 0
    for s in range(meta.num_seqs):
        for j in range(meta.n_new[s]):
            pos = meta.seen[s] + j
            assert meta.slot[t] == meta.blocks_of(s)[pos // B] * B + pos % B
            t += 1


def test_tiny_scenario_matches_golden():
    scn = workloads.tiny()
    g = json.load(open(GOLDEN))
    b, st = scn.registration()
    assert b == g["registration"]["budget"]
    assert [list(s) for s in st] == g["registration"]["states"]
    assert [list(s) for s in scn.requests] == g["pass"]["states"]


def _random_states(rng, comp, n):
    """Register some decoding histories, return a mixed list of states."""
    states = []
    sid = 1
    hist = []
    for _ in range(n):
        if rng.random() < 0.5:
            L = int(rng.integers(1, 200))
            hist.append((sid, L, 0))
            states.append([sid, L, L])          # decoding after registration
        else:
            states.append([sid, int(rng.integers(1, 300)), 0])
        sid += 1
    if hist:
        comp.compose(sum(h[1] for h in hist), 0, hist)
    rng.shuffle(states)
    return [tuple(s) for s in states]


@pytest.mark.parametrize("seed", range(40))
def test_budget_filled_exactly_when_demand_allows(seed):
    rng = np.random.default_rng(seed)
    comp = Composer(int(rng.choice([1, 16, 64])), 100000)
    states = _random_states(rng, comp, int(rng.integers(0, 12)))
    budget = int(rng.integers(0, 400))
    M = int(rng.choice([0, 1, 7, 64, 512]))
    meta = comp.compose(budget, M, states)
    decodes = sum(1 for _, p, s in states if s >= p)
    demand = decodes + sum(min(p - s, M if M > 0 else p) for _, p, s in states if s < p)
    assert meta.num_tokens == min(budget, demand)
    # decodes before prompts: while a decode waits, no prompt token is scheduled
    sched = dict(zip(meta.seq_ids, meta.n_new))
    waiting = [sid for sid, p, s in states if s >= p and sid not in sched]
    if waiting:
        assert all(s >= p for sid, p, s in states if sid in sched)
    for sid, p, s in states:
        n = sched.get(sid, 0)
        if s >= p:
            assert n in (0, 1)
        else:
            assert n <= p - s and (M <= 0 or n <= M)
    # layout keeps list order
    order = [sid for sid, _, _ in states if sid in sched]
    assert meta.seq_ids == order
    assert all(n > 0 for n in meta.n_new)


def test_decodes_beyond_budget_take_list_order():
    comp = Composer(16, 1000)
    comp.compose(50, 0, [(i, 10, 0) for i in range(1, 6)])
    states = [(9, 30, 0)] + [(i, 10, 10) for i in range(1, 6)]
    meta = comp.compose(3, 0, states)
    assert meta.seq_ids == [1, 2, 3] and meta.n_new == [1, 1, 1]


def test_prompt_positions_scheduled_once_in_order_and_blocks_cover():
    rng = np.random.default_rng(7)
    B = 16
    comp = Composer(B, 5000)
    prompts = {i: int(rng.integers(1, 400)) for i in range(1, 9)}
    seen = {i: 0 for i in prompts}
    positions = {i: [] for i in prompts}
    owner = {}
    for _ in range(200):
        states = [(i, prompts[i], seen[i]) for i in prompts]
        meta = comp.compose(97, 41, states)
        if meta.num_tokens == 0:
            break
        t = 0
        for s in range(meta.num_seqs):
            sid = meta.seq_ids[s]
            table = meta.blocks_of(s)
            assert len(table) == -(-meta.ctx[s] // B)
            for b in table:
                assert owner.setdefault(b, sid) == sid   # blocks never shared
            for j in range(meta.n_new[s]):
                positions[sid].append(meta.seen[s] + j)
                assert meta.slot[t] // B == table[(meta.seen[s] + j) // B]
                t += 1
            seen[sid] += meta.n_new[s]
    for i in prompts:
        # positions 0..P-1 (the prompt) then one per generated token, in order
        assert positions[i][:prompts[i]] == list(range(prompts[i]))
        assert positions[i] == list(range(len(positions[i])))


def test_fresh_pool_allocates_lowest_ids_in_layout_order_and_reuses():
    comp = Composer(4, 20)
    meta = comp.compose(100, 0, [(7, 9, 0), (3, 5, 0)])
    assert meta.block_ids == [0, 1, 2, 3, 4]
    comp.release(7)
    assert comp.free_blocks() == 18
    meta = comp.compose(100, 0, [(8, 6, 0)])
    assert meta.block_ids == [0, 1]
    # the decode of seq 3 (5 tokens -> 6) stays in its second block
    meta = comp.compose(1, 0, [(3, 5, 5)])
    assert meta.block_ids == [3, 4] and meta.slot == [4 * 4 + 1]


def test_pool_shortfall_changes_nothing():
    comp = Composer(8, 4)
    comp.compose(16, 0, [(1, 16, 0)])
    before = (comp.free_blocks(), comp.tokens_of(1), comp.held_blocks(1))
    with pytest.raises(NoBlocks):
        comp.compose(40, 0, [(1, 16, 16), (2, 30, 0)])
    assert (comp.free_blocks(), comp.tokens_of(1), comp.held_blocks(1)) == before
    meta = comp.compose(10, 0, [(1, 16, 16), (2, 8, 0)])
    assert meta.n_new == [1, 8] and meta.block_ids == [0, 1, 2, 3]
    assert comp.free_blocks() == 0


def test_invalid_calls():
    comp = Composer(16, 10)
    with pytest.raises(InvalidRequest):
        comp.compose(-1, 0, [])
    with pytest.raises(InvalidRequest):
        comp.compose(10, 0, [(1, 5, 0), (1, 5, 0)])
    with pytest.raises(InvalidRequest):
        comp.compose(10, 0, [(1, 0, 0)])
    with pytest.raises(InvalidRequest):
        comp.compose(10, 0, [(1, 5, 3)])      # nothing cached for seq 1
    with pytest.raises(InvalidRequest):
        comp.release(42)


def test_empty_pass():
    comp = Composer(16, 10)
    meta = comp.compose(0, 0, [(1, 5, 0)])
    assert meta.num_tokens == 0 and meta.num_seqs == 0 and meta.block_ids == []
    meta = comp.compose(10, 0, [])
    assert meta.num_tokens == 0


def test_trace_conserves_tokens():
    reqs = workloads.trace_requests(seed=3, num_requests=48, num_clients=6,
                                    prompt_mean=300.0, output_mean=12.0)
    comp = Composer(64, workloads.trace_block_pool(reqs, 6, 64))
    totals = []

    def on_pass(i, meta, active):
        totals.append(meta.num_tokens)
        demand = sum(1 if r.seen >= r.prompt_len else min(r.prompt_len - r.seen, 128)
                     for r in active)
        assert meta.num_tokens == min(128, demand)

    npass = workloads.run_trace(reqs, 6, 128, 128, comp.compose, comp.release, on_pass)
    assert npass == len(totals)
    assert sum(totals) == sum(r.prompt_len + r.output_len - 1 for r in reqs)
    assert comp.free_blocks() == workloads.trace_block_pool(reqs, 6, 64)


def test_rollback_is_the_inverse_of_compose():
    comp = Composer(8, 64)
    comp.compose(20, 0, [(1, 20, 0)])
    base = (comp.free_blocks(), comp.tokens_of(1), comp.held_blocks(1))
    m1 = comp.compose(30, 0, [(1, 20, 20), (2, 25, 0)])
    m2 = comp.compose(30, 10, [(1, 20, 21), (2, 25, 25), (3, 9, 0)])
    comp.rollback(m2)
    comp.rollback(m1)
    assert (comp.free_blocks(), comp.tokens_of(1), comp.held_blocks(1)) == base
    assert comp.tokens_of(2) == 0 and comp.held_blocks(2) == []
    again = comp.compose(30, 0, [(1, 20, 20), (2, 25, 0)])
    assert again == m1
