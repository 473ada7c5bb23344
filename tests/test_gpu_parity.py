"""GPU parity: the CUDA library against the fp64 oracle, element by element.

Bars: composer metadata and KV-cache contents bit-exact; attention outputs
within max-abs 1e-2 and mean-abs 1e-3 of the oracle (bf16 or fp32 inputs,
fp32 accumulation).  Every call goes through the C ABI.
"""
import numpy as np
import pytest
import torch

import workloads
from harness import MAX_ABS_TOL, MEAN_ABS_TOL, Pair, run_scenario

pytestmark = pytest.mark.gpu


def _ok(r, tight=False):
    assert r["meta_equal"]
    assert r["finite"]
    tol = (1e-5, 1e-6) if tight else (MAX_ABS_TOL, MEAN_ABS_TOL)
    assert r["max_abs"] <= tol[0], r["max_abs"]
    assert r["mean_abs"] <= tol[1], r["mean_abs"]


# forced split lengths: one key block (the most splits), two splits of the
# longest context, and one split of every context (1 << 20 keys)
@pytest.mark.parametrize("split", [None, 16, 32, 64, 1 << 20])
def test_tiny_fp32_all_outputs(rbkv, split):
    (r,) = run_scenario(rbkv, workloads.tiny(), split_keys=split)
    assert r["tokens"] == 64
    _ok(r, tight=True)     # fp32 CUDA-core arithmetic: far inside the bar
    assert r["pair"].cache_equal()
    if split is not None:
        assert r["plan"]["max_splits"] == -(-101 // split)


@pytest.mark.parametrize("name,factor", [("llama2_7b", 8), ("decode_stress", 16),
                                         ("mistral_7b", 8)])
@pytest.mark.parametrize("split", [None, 64, 256, 1 << 20])
def test_scaled_scenarios_all_outputs(rbkv, name, factor, split):
    scn = workloads.scaled(workloads.SCENARIOS[name](0), factor)
    (r,) = run_scenario(rbkv, scn, split_keys=split)
    _ok(r)
    assert r["pair"].cache_equal()
    plan = r["plan"]
    assert plan["decode_items"] > 0
    if split == 1 << 20:
        assert plan["max_splits"] == 1, plan   # every decode row in one piece
    if name != "decode_stress":
        # the scaled pass keeps its prompt chunks, on the tensor-core kernel
        assert plan["chunk_rows"] > 0 and plan["chunk_tiles"] > 0, plan


@pytest.mark.parametrize("mode", ["pairs", "single"])
@pytest.mark.parametrize("name,factor", [("mistral_7b", 8), ("llama2_7b", 2), ("llama2_7b", 4)])
@pytest.mark.parametrize("split", [None, 128])
def test_chunk_work_item_modes(rbkv, mode, name, factor, split):
    """Both tensor-core chunk kernels on the same passes: items that pair two
    query tiles reading the same K/V tiles (two heads of a KV group for
    Mistral-7B's groups of four; two consecutive row tiles for Llama-2-7B's
    groups of one, 248- and 124-row chunks: a pair and a lone tile) and items
    of one tile; with a forced split every tile's keys come in 128-key pieces
    merged by the combine.  Every output against the oracle."""
    scn = workloads.scaled(workloads.SCENARIOS[name](0), factor)
    (r,) = run_scenario(rbkv, scn, split_keys=split, chunk_items=mode)
    plan = r["plan"]
    assert plan["chunk_tiles"] > 0 and plan["chunk_single"] == (mode == "single"), plan
    if mode == "pairs" and (name == "mistral_7b" or factor == 2):
        assert plan["chunk_items"] < plan["chunk_tiles"] * scn.shape.num_heads_q, plan
    _ok(r)
    assert r["pair"].cache_equal()


@pytest.mark.parametrize("split", [None, 64, 192])
def test_chunked_prompt_over_passes(rbkv, split):
    """Every pass of a prompt chunked over several passes, with decodes; with a
    forced split the prompt-chunk tiles' key ranges are cut too (rows whose
    keys all lie before a split's start get an empty piece)."""
    scn = workloads.scaled(workloads.llama2_7b(1), 8)
    res = run_scenario(rbkv, scn, passes=9, split_keys=split)
    for r in res:
        _ok(r)
    assert res[-1]["pair"].cache_equal()


def test_equal_chunk_policy_over_passes(rbkv):
    """The equal-chunk policy's passes (near-equal chunks, passes under the
    budget) through the kernels, every pass against the oracle."""
    scn = workloads.scaled(workloads.llama2_7b(1), 4)
    res = run_scenario(rbkv, scn, passes=9, policy="equal")
    chunks = [max(r["meta"].n_new) for r in res if max(r["meta"].n_new) > 1]
    assert chunks and max(chunks) - min(chunks) <= 1
    for r in res:
        _ok(r)
    assert res[-1]["pair"].cache_equal()


@pytest.mark.parametrize("hq,hkv", [(16, 4), (8, 8)])
def test_many_prompt_chunks_persistent_grid(rbkv, hq, hkv):
    """Hundreds of prompt chunks of mixed length (fresh prompts and chunks behind
    cached prefixes) next to decodes: many more (tile, head) items than SMs, so
    every chunk CTA walks several items in snake order, with items as short as
    one key tile.  Every output against the oracle."""
    rng = np.random.default_rng(hq * 7 + hkv)
    shape = workloads.Shape(hq, hkv, 128, 64, "bf16", 1.0 / np.sqrt(128.0))
    hist = [(1000 + i, int(rng.integers(1, 700))) for i in range(40)]
    reqs = [(1000 + i, c + int(rng.integers(1, 90)), c) for i, (_, c) in enumerate(hist[:30])]
    reqs += [(1000 + i, c, c) for i, (_, c) in enumerate(hist[30:], start=30)]      # decodes
    reqs += [(5000 + i, int(rng.integers(1, 160)), 0) for i in range(160)]            # fresh prompts
    budget = sum(p - s if p > s else 1 for _, p, s in reqs)
    nb = sum(-(-(c + 300) // 64) for _, c in hist) + sum(-(-p // 64) for sid, p, s in reqs
                                                           if sid >= 5000) + 64
    scn = workloads.Scenario("many", shape, budget, 0, hist, reqs, nb)
    (r,) = run_scenario(rbkv, scn)
    # chunks of up to 16 rows with short contexts run as packed decode units,
    # the rest as tensor-core tiles: both paths carry many items
    assert r["plan"]["chunk_tiles"] * hq > 152 and r["plan"]["decode_items"] > 152
    _ok(r)
    assert r["pair"].cache_equal()


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (16, 2), (32, 2)])
def test_short_prompts_packed_decode_units(rbkv, hq, hkv):
    """Prompt chunks of 2..16 rows with short contexts run on the decode kernel,
    several causal rows per unit (8 / g of them): fresh prompts, chunks behind a
    short cached prefix, next to plain decodes.  Every output against the oracle."""
    scn = workloads.short_prompts(hq, hkv, seed=hq + 100 * hkv)
    (r,) = run_scenario(rbkv, scn)
    assert r["plan"]["chunk_tiles"] == 0            # every chunk took the decode kernel
    assert r["plan"]["chunk_rows"] > 0 and r["plan"]["decode_items"] > 0
    _ok(r)
    assert r["pair"].cache_equal()


@pytest.mark.parametrize("split", [None, 64])
@pytest.mark.parametrize("mode", ["pairs", "single"])
def test_garbage_in_unwritten_slots_does_not_leak(rbkv, split, mode):
    """Slots past a sequence's context hold whatever the caller left there
    (here NaN); outputs must not see them.  The pass has decode units and
    tensor-core chunk tiles whose key ranges end inside a 128-key tile (96 and
    288 keys), so the decode kernel and both chunk kernels meet NaN rows in
    their last K/V tile."""
    scn = workloads.scaled(workloads.mistral_7b(0), 8)
    (r,) = run_scenario(rbkv, scn, cache_fill=float("nan"), split_keys=split, chunk_items=mode)
    _ok(r)
    plan = r["plan"]
    assert plan["chunk_tiles"] > 0 and plan["decode_items"] > 0, plan
    m = r["meta"]
    assert any(n > 1 and c % 128 for n, c in zip(m.n_new, m.ctx))


def test_empty_pass_and_repeat_determinism(rbkv):
    scn = workloads.scaled(workloads.decode_stress(3), 16)
    shape = scn.shape
    pair = Pair(rbkv, shape, scn.num_blocks)
    b, st = scn.registration()
    pair.step(b, 0, st, attend=False)
    r0 = pair.step(0, 0, list(scn.requests))
    assert r0["tokens"] == 0
    r1 = pair.step(scn.budget, scn.max_chunk, list(scn.requests))
    _ok(r1)
    p = r1["pass"]
    q = workloads.make_qkv(shape, p.num_tokens, 0, 1, which="q")[0].cuda()
    torch.cuda.synchronize()
    o1 = rbkv.ragged_attention(p, q, pair.kc, pair.vc)
    o2 = rbkv.ragged_attention(p, q, pair.kc, pair.vc)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


@pytest.mark.parametrize("hq,hkv,B,D,dt", [
    (16, 16, 64, 128, "bf16"), (32, 8, 64, 128, "bf16"), (64, 8, 64, 128, "bf16"),
    (16, 1, 64, 128, "bf16"),                     # g = 16: the largest group on the MMA decode path
    (64, 2, 64, 128, "bf16"),                     # g = 32: decode on the CUDA-core path
    (8, 2, 16, 128, "bf16"), (8, 2, 32, 128, "bf16"), (8, 4, 128, 128, "bf16"),
    (8, 2, 256, 128, "bf16"),                     # blocks larger than a key tile
    (8, 2, 64, 64, "bf16"),                       # head_dim 64: CUDA-core path
    (16, 4, 64, 128, "f32"),                      # fp32 with grouped heads
])
def test_shapes_and_block_sizes(rbkv, hq, hkv, B, D, dt):
    shape = workloads.Shape(hq, hkv, D, B, dt, 1.0 / np.sqrt(D))
    rng = np.random.default_rng(hq * 131 + hkv * 7 + B)
    # contexts at and around block/tile boundaries, a 1-token prompt, a chunk
    hist = [(10 + i, c) for i, c in enumerate([1, 63, 64, 65, 127, 128, 129, 300,
                                               int(rng.integers(500, 1500))])]
    nb = sum(-(-(c + 200) // B) for _, c in hist) + 64
    scn = workloads.Scenario("edges", shape, 200, 150, hist,
                             [(1, 1, 0), (2, 150, 0)] + [(s, c, c) for s, c in hist], nb)
    (r,) = run_scenario(rbkv, scn)
    _ok(r)
    assert r["pair"].cache_equal()


def test_long_context_decode_and_chunk(rbkv):
    """A 40k-token decode context and a 200-row chunk behind a 30k prefix."""
    shape = workloads.Shape(16, 4, 128, 64, "bf16", 1.0 / np.sqrt(128.0))
    hist = [(10, 40000), (11, 30000), (12, 777)]
    nb = sum(-(-(c + 800) // 64) for _, c in hist) + 16
    scn = workloads.Scenario("long", shape, 202, 200, hist,
                             [(10, 40000, 40000), (11, 30200, 30000), (12, 777, 777)], nb)
    (r,) = run_scenario(rbkv, scn, only_seqs={10, 11, 12}, input_device="cuda")
    assert r["meta_equal"] and r["finite"]
    assert r["max_abs"] <= MAX_ABS_TOL and r["mean_abs"] <= MEAN_ABS_TOL
    assert r["plan"]["max_splits"] >= 1


@pytest.mark.parametrize("name", ["decode_stress", "mistral_7b", "llama2_7b"])
def test_full_size_sampled(rbkv, name):
    """Full-size passes, in the launch configuration the benchmark times; the
    oracle checks every output row of a sample of sequences."""
    scn = workloads.SCENARIOS[name](0)
    ids = [s for s, _, _ in scn.requests]
    rng = np.random.default_rng(5)
    sample = set(ids[:2]) | set(int(x) for x in rng.choice(ids, size=min(6, len(ids)), replace=False))
    if name == "mistral_7b":
        # both prompt chunks are sampled on a few rows only (the oracle is slow)
        sample |= {1, 2}
    res = run_scenario(rbkv, scn, only_seqs=sample, input_device="cuda")
    r = res[0]
    assert r["meta_equal"]
    assert r["finite"]
    assert r["max_abs"] <= MAX_ABS_TOL and r["mean_abs"] <= MEAN_ABS_TOL
    pair = r["pair"]
    blocks = []
    m = r["meta"]
    for s in range(m.num_seqs):
        if m.seq_ids[s] in sample:
            blocks.extend(m.blocks_of(s))
    assert pair.cache_equal(blocks)


@pytest.mark.parametrize("name,factor", [("decode_stress", 16), ("llama2_7b", 8)])
def test_q_written_by_a_kernel_just_before_attention(rbkv, name, factor):
    """The attention kernels start early (programmatic dependent launch); a Q
    written by the caller's own kernel right before the call must still be
    read only after that kernel has finished."""
    scn = workloads.scaled(workloads.SCENARIOS[name](0), factor)
    (r,) = run_scenario(rbkv, scn)
    _ok(r)
    p, pair = r["pass"], r["pair"]
    q = workloads.make_qkv(scn.shape, p.num_tokens, 0, 1, which="q")[0].cuda()
    torch.cuda.synchronize()
    for _ in range(3):
        q2 = torch.full_like(q, float("nan"))
        torch.mul(q * 2, 0.5, out=q2)           # exact; runs just before the call
        o2 = rbkv.ragged_attention(p, q2, pair.kc, pair.vc)
        torch.cuda.synchronize()
        assert torch.equal(o2.view(torch.int16), r["o"].view(torch.int16))


def test_closed_loop_trace_every_pass(rbkv):
    """A small closed-loop trace (requests finish, are released, and clients
    send their next ones): every pass's metadata, cache and outputs against
    the oracle, the pool back to full at the end."""
    reqs = workloads.trace_requests(seed=4, num_requests=12, num_clients=4,
                                    prompt_mean=160.0, output_mean=6.0)
    shape = workloads.Shape(32, 32, 128, 64, "bf16", 1.0 / np.sqrt(128.0))
    nb = workloads.trace_block_pool(reqs, 4, 64)
    pair = Pair(rbkv, shape, nb)
    results = []

    def compose(budget, max_chunk, states):
        r = pair.step(budget, max_chunk, states)
        results.append(r)
        return r["meta"]

    n = workloads.run_trace(reqs, 4, 64, 64, compose, pair.release)
    assert n == len(results) and n > 10
    for r in results:
        if r["tokens"]:
            _ok(r)
    assert pair.cache_equal()
    assert pair.lib.free_blocks() == nb


@pytest.mark.parametrize("seed", range(6))
def test_random_mixed_passes(rbkv, seed):
    """Seeded random passes: a random group shape and block size, decodes with
    log-uniform contexts (1 … 4000 keys), fresh prompts and prompts behind a
    cached prefix, a random budget and chunk cap; three passes with states
    advanced between them, every output against the oracle and the whole
    cache bit-exact at the end."""
    rng = np.random.default_rng(1000 + seed)
    hq, hkv, B = [(8, 2, 64), (16, 2, 64), (8, 8, 16), (32, 4, 64), (16, 1, 64),
                  (8, 2, 32)][seed]
    shape = workloads.Shape(hq, hkv, 128, B, "bf16", 1.0 / np.sqrt(128.0))
    hist, reqs = [], []
    sid = 100
    for _ in range(int(rng.integers(1, 24))):           # decodes
        c = int(np.exp(rng.uniform(0.0, np.log(4000.0))))
        hist.append((sid, c))
        reqs.append((sid, c, c))
        sid += 1
    for _ in range(int(rng.integers(0, 4))):            # prompts behind a cached prefix
        s0 = int(rng.integers(1, 2000))
        hist.append((sid, s0))
        reqs.append((sid, s0 + int(rng.integers(1, 600)), s0))
        sid += 1
    for _ in range(int(rng.integers(0, 5))):            # fresh prompts
        reqs.append((sid, int(rng.integers(1, 700)), 0))
        sid += 1
    order = rng.permutation(len(reqs))
    reqs = [reqs[i] for i in order]
    budget = int(rng.integers(32, 1025))
    cap = int(rng.choice([0, 16, 100, 512]))
    nb = sum(-(-(pl + 3) // B) for _, pl, _ in reqs) + 8
    scn = workloads.Scenario("random", shape, budget, cap, hist, reqs, nb)
    res = run_scenario(rbkv, scn, passes=3)
    for r in res:
        if r["tokens"]:
            _ok(r)
        else:
            assert r["meta_equal"]
    assert res[-1]["pair"].cache_equal()
