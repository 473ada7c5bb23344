"""The library's C++ composer matches the oracle's bit for bit (CPU only).

Both sides compose the same call sequences independently; every metadata array
(sequence ids, row offsets, token counts, contexts, block tables, slots) must be
identical, errors must fall in the same class, and the pool must agree.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_pass.json")
FIELDS = ("seq_ids", "q_start", "n_new", "seen", "ctx", "block_start", "block_ids", "slot")


def _same(lib_pass, ometa):
    m = lib_pass.meta
    for f in FIELDS:
        a = np.asarray(getattr(m, f), dtype=np.int64)
        b = np.asarray(getattr(ometa, f), dtype=np.int64)
        assert a.shape == b.shape and np.array_equal(a, b), f
    return True


class Both:
    """Drive the library composer and the oracle composer in lockstep."""

    def __init__(self, rbkv, B, num_blocks, shape=(8, 2, 64, "f32")):
        hq, hkv, d, dt = shape
        self.lib = rbkv.Composer(rbkv.Config(hq, hkv, d, B, dt, num_blocks))
        self.orc = oracle.Composer(B, num_blocks)
        self.rbkv = rbkv

    def compose(self, budget, max_chunk, states):
        err_l = err_o = None
        p = m = None
        try:
            p = self.lib.compose(budget, max_chunk, states)
        except self.rbkv.NoBlocksError:
            err_l = "noblocks"
        except self.rbkv.RbkvError:
            err_l = "invalid"
        try:
            m = self.orc.compose(budget, max_chunk, states)
        except oracle.NoBlocks:
            err_o = "noblocks"
        except oracle.InvalidRequest:
            err_o = "invalid"
        assert err_l == err_o
        if p is not None:
            _same(p, m)
        assert self.lib.free_blocks() == self.orc.free_blocks()
        return m

    def release(self, sid):
        err_l = err_o = None
        try:
            self.lib.release(sid)
        except self.rbkv.RbkvError:
            err_l = "invalid"
        try:
            self.orc.release(sid)
        except oracle.InvalidRequest:
            err_o = "invalid"
        assert err_l == err_o
        assert self.lib.free_blocks() == self.orc.free_blocks()


def test_tiny_worked_pass_bit_exact(rbkv):
    g = json.load(open(GOLDEN))
    both = Both(rbkv, 16, 64)
    r = g["registration"]
    both.compose(r["budget"], r["max_chunk"], [tuple(s) for s in r["states"]])
    p = g["pass"]
    m = both.compose(p["budget"], p["max_chunk"], [tuple(s) for s in p["states"]])
    assert list(m.block_ids) == g["expected"]["block_ids"]


@pytest.mark.parametrize("seed", range(25))
def test_random_call_sequences(rbkv, seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.choice([1, 4, 16, 64]))
    both = Both(rbkv, B, int(rng.integers(0, 300)))
    known = {}      # seq_id -> (prompt_len, seen)
    next_id = 1
    for _ in range(60):
        r = rng.random()
        if r < 0.1 and known:
            sid = int(rng.choice(list(known)))
            both.release(sid)
            known.pop(sid)
            continue
        if r < 0.13:
            both.release(10_000 + next_id)       # unknown id: both reject
            continue
        states = []
        for sid, (pl, seen) in known.items():
            if rng.random() < 0.8:
                states.append((sid, pl, seen))
        for _ in range(int(rng.integers(0, 3))):
            states.append((next_id, int(rng.integers(1, 200)), 0))
            next_id += 1
        if rng.random() < 0.05 and states:
            states.append(states[0])                 # duplicate: both reject
        if rng.random() < 0.05 and states:
            sid, pl, seen = states[-1]
            states[-1] = (sid, pl, seen + 1)         # wrong seen: both reject
        order = rng.permutation(len(states))
        states = [states[i] for i in order]
        budget = int(rng.integers(-1, 300))
        M = int(rng.choice([-5, 0, 1, 16, 100]))
        m = both.compose(budget, M, states)
        if m is not None:
            for s in range(m.num_seqs):
                sid = m.seq_ids[s]
                pl = dict((x[0], x[1]) for x in states)[sid]
                known[sid] = (pl, m.ctx[s])
            for sid, pl, seen in states:
                if sid not in known and seen == 0:
                    pass


@pytest.mark.parametrize("name", ["tiny", "llama2_7b", "decode_stress", "mistral_7b"])
def test_scenarios_bit_exact(rbkv, name):
    scn = workloads.SCENARIOS[name](0)
    sh = scn.shape
    both = Both(rbkv, sh.block_size, scn.num_blocks,
                (sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.dtype))
    b, st = scn.registration()
    both.compose(b, 0, st)
    states = list(scn.requests)
    for _ in range(12):
        m = both.compose(scn.budget, scn.max_chunk, states)
        n = dict(zip(m.seq_ids, m.n_new))
        states = [(sid, pl, seen + n.get(sid, 0)) for sid, pl, seen in states]
        if m.num_tokens == 0:
            break


def test_llama2_7b_chunks_are_497(rbkv):
    scn = workloads.llama2_7b(0)
    sh = scn.shape
    both = Both(rbkv, sh.block_size, scn.num_blocks,
                (sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.dtype))
    b, st = scn.registration()
    both.compose(b, 0, st)
    states = list(scn.requests)
    chunks = []
    while True:
        m = both.compose(scn.budget, scn.max_chunk, states)
        n = dict(zip(m.seq_ids, m.n_new))
        if states[0][2] >= states[0][1]:
            break
        chunks.append(n[1])
        states = [(sid, pl, seen + n.get(sid, 0)) for sid, pl, seen in states]
    assert chunks == [497] * 8 + [120]


def test_full_trace_bit_exact(rbkv):
    """512 requests, 32 closed-loop clients, budget 512: every pass identical."""
    reqs_l = workloads.trace_requests(seed=0)
    reqs_o = workloads.trace_requests(seed=0)
    nb = workloads.trace_block_pool(reqs_l, 32, 64)
    lib_c = rbkv.Composer(rbkv.Config(32, 32, 128, 64, "bf16", nb))
    orc_c = oracle.Composer(64, nb)
    lib_metas = []

    def lib_compose(b, M, st):
        p = lib_c.compose(b, M, st)
        lib_metas.append(p.meta)
        return p.meta

    n_l = workloads.run_trace(reqs_l, 32, 512, 512, lib_compose, lib_c.release)
    i = [0]

    def orc_compose(b, M, st):
        m = orc_c.compose(b, M, st)
        lm = lib_metas[i[0]]
        for f in FIELDS:
            assert np.array_equal(np.asarray(getattr(lm, f), np.int64),
                                  np.asarray(getattr(m, f), np.int64)), (i[0], f)
        i[0] += 1
        return m

    n_o = workloads.run_trace(reqs_o, 32, 512, 512, orc_compose, orc_c.release)
    assert n_l == n_o == len(lib_metas)
    assert 2000 < n_l < 3500
    assert lib_c.free_blocks() == orc_c.free_blocks() == nb


def test_plan_covers_every_row_and_head(rbkv):
    scn = workloads.decode_stress(0)
    sh = scn.shape
    comp = rbkv.Composer(rbkv.Config(sh.num_heads_q, sh.num_heads_kv, sh.head_dim,
                                     sh.block_size, sh.dtype, scn.num_blocks))
    b, st = scn.registration()
    comp.compose(b, 0, st)
    p = comp.compose(scn.budget, scn.max_chunk, scn.requests)
    info = p.plan_for_sms(152)
    assert info["decode_rows"] == 64
    items = info["decode_items"] + info["generic_items"]
    assert items >= 64 * sh.num_heads_kv
    # splits exist for the long contexts and partials match the split rows
    assert info["max_splits"] > 1 and info["partials"] > 0
    keys = info["split_keys"]
    ctx = p.meta.ctx
    expect_max = max(-(-int(c) // keys) for c in ctx)
    assert info["max_splits"] == expect_max
    # forcing the split length changes only the plan
    p2 = comp.compose(0, 0, [])
    assert p2.plan_for_sms(152)["decode_items"] + p2.plan_for_sms(152)["generic_items"] == 0


def test_rollback_restores_state_bit_exact(rbkv):
    """Rolling passes back (newest first) restores the pool and contexts on both
    sides; composing the same states again gives identical metadata."""
    scn = workloads.scaled(workloads.llama2_7b(2), 4)
    sh = scn.shape
    lib_c = rbkv.Composer(rbkv.Config(sh.num_heads_q, sh.num_heads_kv, sh.head_dim,
                                      sh.block_size, sh.dtype, scn.num_blocks))
    orc_c = oracle.Composer(sh.block_size, scn.num_blocks)
    b, st = scn.registration()
    lib_c.compose(b, 0, st)
    orc_c.compose(b, 0, st)
    free0 = lib_c.free_blocks()
    for cycle in range(3):
        states = list(scn.requests)
        passes = []
        metas = []
        for _ in range(6):
            p = lib_c.compose(scn.budget, scn.max_chunk, states)
            m = orc_c.compose(scn.budget, scn.max_chunk, states)
            _same(p, m)
            if cycle == 0:
                metas.append(p.meta)
            passes.append((p, m))
            n = dict(zip(m.seq_ids, m.n_new))
            states = [(sid, pl, seen + n.get(sid, 0)) for sid, pl, seen in states]
        # the oldest pass cannot go first
        with pytest.raises(rbkv.RbkvError):
            lib_c.rollback(passes[0][0])
        with pytest.raises(oracle.InvalidRequest):
            orc_c.rollback(passes[0][1])
        for p, m in reversed(passes):
            lib_c.rollback(p)
            orc_c.rollback(m)
            assert lib_c.free_blocks() == orc_c.free_blocks()
        assert lib_c.free_blocks() == free0


# -- chunk policy "equal" and the latency-bounded budget --------------------


class BothPolicy(Both):
    def __init__(self, rbkv, B, num_blocks, policy, shape=(8, 2, 64, "f32")):
        super().__init__(rbkv, B, num_blocks, shape)
        self.policy = policy

    def compose(self, budget, max_chunk, states):
        p = self.lib.compose(budget, max_chunk, states, policy=self.policy)
        m = self.orc.compose(budget, max_chunk, states, policy=self.policy)
        _same(p, m)
        assert self.lib.free_blocks() == self.orc.free_blocks()
        return m


def _prefill_passes(both, budget, max_chunk, states):
    """Compose until every prompt is consumed; return [{seq_id: n_new}]."""
    out = []
    for _ in range(10_000):
        m = both.compose(budget, max_chunk, states)
        if all(seen >= pl for _, pl, seen in states):
            break
        n = dict(zip(m.seq_ids, m.n_new))
        out.append(n)
        assert sum(n.values()) <= budget
        states = [(sid, pl, seen + n.get(sid, 0)) for sid, pl, seen in states]
    return out


def test_equal_chunks_llama2_7b(rbkv):
    """4096-token prompt behind 15 decodes, budget 512, cap 512: the greedy
    policy cuts 8 x 497 + 120; the equal policy keeps the same 9 passes with
    chunks that differ by at most one token (4096 = 456 + 8 x 455)."""
    scn = workloads.llama2_7b(0)
    sh = scn.shape
    both = BothPolicy(rbkv, sh.block_size, scn.num_blocks, "equal",
                      (sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.dtype))
    b, st = scn.registration()
    both.compose(b, 0, st)
    passes = _prefill_passes(both, scn.budget, scn.max_chunk, list(scn.requests))
    chunks = [p[1] for p in passes]
    assert len(chunks) == 9 and sum(chunks) == 4096
    assert max(chunks) - min(chunks) <= 1
    assert chunks == [456] + [455] * 8


@pytest.mark.parametrize("seed", range(12))
def test_equal_policy_random_bit_exact(rbkv, seed):
    rng = np.random.default_rng(700 + seed)
    B = int(rng.choice([1, 16, 64]))
    both = BothPolicy(rbkv, B, 100_000, "equal")
    states = [(i + 1, int(rng.integers(1, 3000)), 0) for i in range(int(rng.integers(1, 8)))]
    budget = int(rng.integers(1, 700))
    M = int(rng.choice([0, 64, 256, 512]))
    passes = _prefill_passes(both, budget, M, states)
    # with one prompt the equal policy needs no more passes than greedy
    if len(states) == 1:
        g = BothPolicy(rbkv, B, 100_000, "greedy")
        assert len(_prefill_passes(g, budget, M, states)) == len(passes)
        ch = [p[1] for p in passes]
        assert max(ch) - min(ch) <= 1


def test_unknown_policy_rejected(rbkv):
    c = rbkv.Composer(rbkv.Config(8, 2, 64, 16, "f32", 10))
    with pytest.raises(rbkv.RbkvError):
        c.compose(10, 0, [(1, 5, 0)], policy="bogus")
    with pytest.raises(oracle.InvalidRequest):
        oracle.Composer(16, 10).compose(10, 0, [(1, 5, 0)], policy="bogus")


def test_budget_for_latency_pins(rbkv):
    """Closed forms: a linear profile l(t) = a + b t gives floor((L - a) / b);
    below the first point gives 0; above the last gives the last token count;
    a flat segment at the bound keeps its far end."""
    tok, lat = [0, 1000], [2.0, 12.0]          # 2 ms + 0.01 ms per token
    for L, want in [(7.0, 500), (2.0, 0), (1.0, 0), (12.0, 1000), (50.0, 1000), (7.005, 500)]:
        assert oracle.budget_for_latency(tok, lat, L) == want
        assert rbkv.budget_for_latency(tok, lat, L) == want
    tok, lat = [64, 128, 512, 2048], [3.0, 3.0, 5.0, 14.0]
    assert oracle.budget_for_latency(tok, lat, 3.0) == 128
    assert oracle.budget_for_latency(tok, lat, 2.0) == 0
    assert oracle.budget_for_latency(tok, lat, 5.0) == 512
    assert oracle.budget_for_latency(tok, [5.0, 3.0, 9.0, 1.0], 4.0) == 2048  # not monotone
    assert oracle.budget_for_latency([5, 5], [1.0, 2.0], 3.0) == -1
    with pytest.raises(rbkv.RbkvError):
        rbkv.budget_for_latency([5, 5], [1.0, 2.0], 3.0)


@pytest.mark.parametrize("seed", range(20))
def test_budget_for_latency_random_bit_exact(rbkv, seed):
    rng = np.random.default_rng(900 + seed)
    n = int(rng.integers(2, 9))
    tok = np.sort(rng.choice(5000, size=n, replace=False)).tolist()
    lat = np.cumsum(rng.random(n) * 3).tolist()
    for L in rng.random(6) * (lat[-1] + 1):
        a = oracle.budget_for_latency(tok, lat, float(L))
        assert rbkv.budget_for_latency(tok, lat, float(L)) == a
        if a > 0:
            assert oracle.latency_at(tok, lat, a) <= L
            if a < tok[-1]:
                assert oracle.latency_at(tok, lat, a + 1) > L


def test_planner_packs_short_prompt_chunks(rbkv):
    """Prompt chunks of at most 16 rows whose keys fit one decode split become
    decode units holding 8 / g consecutive rows each; longer chunks, or short
    ones behind a long prefix, stay tensor-core tiles (CPU-side plan only)."""
    for hq, hkv in [(8, 8), (16, 4), (16, 2), (32, 2)]:
        g = hq // hkv
        pack = 8 // g if g <= 8 else 1
        c = rbkv.Composer(rbkv.Config(hq, hkv, 128, 64, "bf16", 4096))
        c.compose(20000, 0, [(1, 12000, 0)])                  # a long cached prefix
        states = [(1, 12010, 12000)]                           # 10 rows behind 12000 keys
        states += [(10 + i, n, 0) for i, n in enumerate([2, 5, 16, 17, 300])]
        p = c.compose(100000, 0, states)
        info = p.plan_for_sms(152)
        packed_rows = [2, 5, 16]
        want_items = sum(-(-n // pack) for n in packed_rows) * hkv
        assert info["decode_items"] == want_items, (hq, hkv, info)
        # tiles: the 10-row chunk behind the prefix, 17 rows, 300 rows (3 tiles)
        assert info["chunk_tiles"] >= 1 + 1 + 3
        assert info["decode_rows"] == 0
