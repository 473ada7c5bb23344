"""Frames (fixed-address passes for CUDA graphs) against the plain entry points.

A frame runs the same kernels on the same plan as rbkv_kv_append +
rbkv_ragged_attention, so its outputs and cache contents must match the plain
path bit for bit - directly, and when its launches are captured once as a CUDA
graph and replayed for every later pass.  The plain path's parity with the
oracle is covered by the other GPU tests; one case here also checks the
replayed outputs against the oracle directly.
"""
import numpy as np
import pytest
import torch

import workloads
from harness import MAX_ABS_TOL, MEAN_ABS_TOL, Pair

pytestmark = pytest.mark.gpu

BIG_CAPS = dict(max_decode_items=1 << 15, max_chunk_tiles=512, max_combine_rows=1 << 15,
                max_parts=1 << 19)


def _drive(rbkv, scn, passes, use_graph, split_keys=None, caps=None, seed=0):
    sh = scn.shape
    cfg = rbkv.Config(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size, sh.dtype,
                      scn.num_blocks)
    comp = rbkv.Composer(cfg)
    dt = cfg.torch_dtype
    caches = [torch.zeros(cfg.cache_shape(), dtype=dt, device="cuda") for _ in range(4)]
    kc_a, vc_a, kc_b, vc_b = caches
    b, st = scn.registration()
    if b > 0:
        p = comp.compose(b, 0, st)
        k, v = workloads.make_qkv(sh, p.num_tokens, seed, 10_000, device="cuda", which="kv")
        rbkv.kv_append(p, k, v, kc_a, vc_a)
        rbkv.kv_append(p, k, v, kc_b, vc_b)
    tmax = scn.budget
    frame = rbkv.Frame(cfg, tmax, **(caps or {}))
    ws = torch.empty(frame.workspace_bytes(), dtype=torch.uint8, device="cuda")
    qb = torch.zeros(tmax, sh.num_heads_q, sh.head_dim, dtype=dt, device="cuda")
    kb = torch.zeros(tmax, sh.num_heads_kv, sh.head_dim, dtype=dt, device="cuda")
    vb = torch.zeros_like(kb)
    ob = torch.zeros_like(qb)
    graph = None
    states = list(scn.requests)
    for i in range(passes):
        p = comp.compose(scn.budget, scn.max_chunk, states)
        if split_keys:
            p.set_split_keys(split_keys)
        p.set_chunk_items(frame.chunk_items)   # the plain path plans the pass first
        T = p.num_tokens
        q, k, v = workloads.make_qkv(sh, T, seed, i, device="cuda")
        rbkv.kv_append(p, k, v, kc_a, vc_a)
        oa = rbkv.ragged_attention(p, q, kc_a, vc_a)
        frame.load(p)
        qb[:T], kb[:T], vb[:T] = q, k, v
        if graph is None:
            frame.kv_append(kb, vb, kc_b, vc_b)
            frame.attention(qb, kc_b, vc_b, ob, ws)
            if use_graph:
                torch.cuda.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    frame.kv_append(kb, vb, kc_b, vc_b)
                    frame.attention(qb, kc_b, vc_b, ob, ws)
        else:
            graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(ob[:T], oa), f"pass {i}"
        n = dict(zip(p.meta.seq_ids, p.meta.n_new))
        states = [(sid, pl, seen + n.get(sid, 0)) for sid, pl, seen in states]
    frame.device_status()
    assert torch.equal(kc_a, kc_b) and torch.equal(vc_a, vc_b)
    return frame


@pytest.mark.parametrize("use_graph", [False, True])
@pytest.mark.parametrize("name,passes", [("llama2_7b", 9), ("mistral_7b", 2),
                                         ("decode_stress", 3)])
def test_frame_matches_plain_path(rbkv, name, passes, use_graph):
    _drive(rbkv, workloads.SCENARIOS[name](0), passes, use_graph)


@pytest.mark.parametrize("split", [64, 256])
def test_frame_with_forced_splits(rbkv, split):
    """Many partial outputs and combine rows: still bit-exact, replayed."""
    _drive(rbkv, workloads.scaled(workloads.llama2_7b(0), 2), 5, True, split_keys=split,
           caps=BIG_CAPS)


def test_replayed_graph_against_oracle(rbkv):
    """Passes of a chunked prompt with decodes, replayed from one graph, checked
    element by element against the fp64 oracle."""
    scn = workloads.scaled(workloads.llama2_7b(1), 8)
    sh = scn.shape
    pair = Pair(rbkv, sh, scn.num_blocks)
    b, st = scn.registration()
    pair.step(b, 0, st, attend=False)
    # the prompt's last chunk (16 rows) runs as packed decode units
    frame = rbkv.Frame(pair.cfg, scn.budget, packed_units=1)
    dt = pair.cfg.torch_dtype
    ws = torch.empty(frame.workspace_bytes(), dtype=torch.uint8, device="cuda")
    kc, vc = pair.kc.clone(), pair.vc.clone()
    qb = torch.zeros(scn.budget, sh.num_heads_q, sh.head_dim, dtype=dt, device="cuda")
    kb = torch.zeros(scn.budget, sh.num_heads_kv, sh.head_dim, dtype=dt, device="cuda")
    vb, ob = torch.zeros_like(kb), torch.zeros_like(qb)
    graph = None
    states = list(scn.requests)
    for i in range(9):
        r = pair.step(scn.budget, scn.max_chunk, states)       # plain path + oracle
        assert r["meta_equal"] and r["max_abs"] <= MAX_ABS_TOL
        p = r["pass"]
        T = p.num_tokens
        q, k, v = (t.cuda() for t in workloads.make_qkv(sh, T, pair.seed, pair.npass - 1,
                                                         device=pair.input_device))
        frame.load(p)
        qb[:T], kb[:T], vb[:T] = q, k, v
        if graph is None:
            frame.kv_append(kb, vb, kc, vc)
            frame.attention(qb, kc, vc, ob, ws)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                frame.kv_append(kb, vb, kc, vc)
                frame.attention(qb, kc, vc, ob, ws)
        else:
            graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(ob[:T], r["o"])
        n = dict(zip(r["meta"].seq_ids, r["meta"].n_new))
        states = [(sid, pl, seen + n.get(sid, 0)) for sid, pl, seen in states]
    assert pair.cache_equal()
    assert torch.equal(kc, pair.kc) and torch.equal(vc, pair.vc)


def test_empty_pass_changes_nothing(rbkv):
    scn = workloads.llama2_7b(0)
    sh = scn.shape
    cfg = rbkv.Config(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size, sh.dtype,
                      scn.num_blocks)
    comp = rbkv.Composer(cfg)
    frame = rbkv.Frame(cfg, 64)
    dt = cfg.torch_dtype
    kc = torch.zeros(cfg.cache_shape(), dtype=dt, device="cuda")
    vc = torch.zeros_like(kc)
    ws = torch.empty(frame.workspace_bytes(), dtype=torch.uint8, device="cuda")
    qb = torch.randn(64, 32, 128, device="cuda").to(dt)
    kb = torch.randn(64, 32, 128, device="cuda").to(dt)
    ob = torch.full_like(qb, 7.0)
    frame.load(comp.compose(0, 0, []))
    frame.kv_append(kb, kb, kc, vc)
    frame.attention(qb, kc, vc, ob, ws)
    torch.cuda.synchronize()
    frame.device_status()
    assert int(kc.count_nonzero()) == 0 and int(vc.count_nonzero()) == 0
    assert bool((ob == 7.0).all())


def test_capacity_refusals(rbkv):
    scn = workloads.llama2_7b(0)
    sh = scn.shape
    cfg = rbkv.Config(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size, sh.dtype,
                      scn.num_blocks)
    comp = rbkv.Composer(cfg)
    p = comp.compose(100, 0, [(1, 100, 0)])
    with pytest.raises(rbkv.RbkvError) as e:
        rbkv.Frame(cfg, 64).load(p)
    assert e.value.status == -6
    with pytest.raises(rbkv.RbkvError) as e:
        rbkv.Frame(cfg, 128, max_chunk_tiles=0, max_seqs=1).load(
            comp.compose(8, 0, [(2, 4, 0), (3, 4, 0)]))
    assert e.value.status == -6
    f32 = rbkv.Config(8, 2, 64, 16, "f32", 16)
    with pytest.raises(rbkv.RbkvError) as e:
        rbkv.Frame(f32, 64)
    assert e.value.status == -5
    with pytest.raises(rbkv.RbkvError):
        rbkv.Frame(cfg, 0)


def test_frame_with_packed_short_prompts(rbkv):
    """Short prompt chunks run as packed decode units: a frame refuses such a
    pass unless created with packed_units=1, and then matches the plain path."""
    shape = workloads.Shape(16, 4, 128, 64, "bf16", 1.0 / np.sqrt(128.0))
    cfg = rbkv.Config(16, 4, 128, 64, "bf16", 256)
    comp = rbkv.Composer(cfg)
    hist = [(1, 300), (2, 40)]
    comp.compose(340, 0, [(s, n, 0) for s, n in hist])
    states = [(1, 300, 300), (2, 52, 40)] + [(10 + i, 3 + i, 0) for i in range(12)]
    p = comp.compose(512, 0, states)
    assert p.plan()["chunk_tiles"] == 0
    T = p.num_tokens
    dt = cfg.torch_dtype
    kc = torch.zeros(cfg.cache_shape(), dtype=dt, device="cuda")
    vc = torch.zeros_like(kc)
    q, k, v = workloads.make_qkv(shape, T, 0, 3, device="cuda")
    with pytest.raises(rbkv.RbkvError) as e:
        rbkv.Frame(cfg, 256).load(p)
    assert e.value.status == -5
    frame = rbkv.Frame(cfg, 256, packed_units=1)
    frame.load(p)
    kb = torch.zeros(256, 4, 128, dtype=dt, device="cuda")
    vb, qb = torch.zeros_like(kb), torch.zeros(256, 16, 128, dtype=dt, device="cuda")
    ob = torch.zeros_like(qb)
    qb[:T], kb[:T], vb[:T] = q, k, v
    ws = torch.empty(frame.workspace_bytes(), dtype=torch.uint8, device="cuda")
    kc2, vc2 = kc.clone(), vc.clone()
    frame.kv_append(kb, vb, kc2, vc2)
    frame.attention(qb, kc2, vc2, ob, ws)
    rbkv.kv_append(p, k, v, kc, vc)
    oa = rbkv.ragged_attention(p, q, kc, vc)
    torch.cuda.synchronize()
    assert torch.equal(ob[:T], oa)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
