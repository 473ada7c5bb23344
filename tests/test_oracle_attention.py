"""Pins for the oracle's blocked cache and attention (CPU only).

Each pin checks the oracle against something other than itself:

* brute force on tiny inputs, pure-Python loops over per-sequence key lists
  that the test collects itself (no block tables);
* PyTorch's scaled-dot-product attention in fp64, a library routine, for the
  special case of one sequence (causal mask with a cached prefix, grouped heads
  expanded);
* closed forms: a single key gives its value exactly; identical keys give the
  mean of the visible values;
* split invariance: the FastGen guide's verification harness (Step 4: dense
  attention vs 8 splits over 4096 keys, 8 heads, head_dim 128) redone in fp64;
* chunk invariance: a prompt processed in chunks over several passes gives the
  same outputs as one-shot causal attention over the whole sequence (paper
  summary page: SplitFuse changes how tokens are batched, not what they
  compute).

A last group plants plausible mistakes in the oracle (on the CPU) and checks
that one of these pins catches each.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.attention as oatt
from oracle import BlockedCache, Composer, kv_append, widen


def _run_passes(rng, H_q, H_kv, D, B, storage, plan):
    """Compose and append a sequence of passes; collect per-seq rows and O.

    ``plan`` = list of (budget, max_chunk, states).  Returns the composer, the
    caches, a list of (meta, q) per pass, and per-seq dense K/V row lists in
    position order (collected by the test, not through the cache)."""
    comp = Composer(B, 4096)
    kc = BlockedCache(H_kv, B, D, storage)
    vc = BlockedCache(H_kv, B, D, storage)
    rows_k, rows_v = {}, {}
    passes = []
    for budget, M, states in plan:
        meta = comp.compose(budget, M, states)
        T = meta.num_tokens
        q = rng.standard_normal((T, H_q, D)).astype(storage)
        k = rng.standard_normal((T, H_kv, D)).astype(storage)
        v = rng.standard_normal((T, H_kv, D)).astype(storage)
        kv_append(meta, k, v, kc, vc)
        for s in range(meta.num_seqs):
            sid = meta.seq_ids[s]
            for j in range(meta.n_new[s]):
                rows_k.setdefault(sid, []).append(k[meta.q_start[s] + j])
                rows_v.setdefault(sid, []).append(v[meta.q_start[s] + j])
        passes.append((meta, q))
    return comp, kc, vc, passes, rows_k, rows_v


# --------------------------------------------------------------------------
# cache
# --------------------------------------------------------------------------

def test_append_then_gather_reproduces_rows_and_leaves_rest_zero():
    rng = np.random.default_rng(1)
    H_kv, D, B = 2, 8, 4
    plan = [(30, 0, [(1, 11, 0), (2, 7, 0)]),
            (9, 5, [(1, 11, 11), (2, 7, 7), (3, 13, 0)]),
            (9, 5, [(1, 11, 12), (2, 7, 8), (3, 13, 5)])]
    comp, kc, vc, passes, rk, rv = _run_passes(rng, 4, H_kv, D, B, np.float32, plan)
    last = passes[-1][0]
    for s in range(last.num_seqs):
        sid = last.seq_ids[s]
        for h in range(H_kv):
            got = kc.gather(last.blocks_of(s), last.ctx[s], h)
            want = np.stack([r[h] for r in rk[sid]])
            assert got.tobytes() == want.tobytes()
            got = vc.gather(last.blocks_of(s), last.ctx[s], h)
            want = np.stack([r[h] for r in rv[sid]])
            assert got.tobytes() == want.tobytes()
    # slots past each sequence's context in its last block were never written
    dense = kc.dense(16)
    written = set()
    for s in range(last.num_seqs):
        for p in range(last.ctx[s]):
            b = last.blocks_of(s)[p // B]
            written.add((b, p % B))
    for b in range(16):
        for off in range(B):
            if (b, off) not in written:
                assert not dense[b, :, off].any()


def test_bf16_bit_patterns_widen_exactly():
    x = torch.randn(1000, dtype=torch.float32).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(widen(bits), x.to(torch.float64).numpy())


# --------------------------------------------------------------------------
# attention: brute force, library special case, closed forms
# --------------------------------------------------------------------------

def _brute(q_row, keys, vals, scale):
    """Pure-Python softmax attention of one query over lists of key/value rows."""
    scores = [scale * sum(a * b for a, b in zip(q_row, k)) for k in keys]
    m = max(scores)
    w = [math.exp(s - m) for s in scores]
    z = sum(w)
    return [sum(wi * v[d] for wi, v in zip(w, vals)) / z for d in range(len(vals[0]))]


def _check_brute_force(rng):
    H_q, H_kv, D, B = 4, 2, 6, 4
    plan = [(20, 0, [(1, 9, 0), (2, 5, 0)]),
            (12, 4, [(3, 10, 0), (1, 9, 9), (2, 5, 5), (4, 3, 0)])]
    _, kc, vc, passes, rk, rv = _run_passes(rng, H_q, H_kv, D, B, np.float64, plan)
    meta, q = passes[-1]
    got = oracle.blocked_attention(meta, q, kc, vc, H_q)
    scale = 1.0 / math.sqrt(D)
    err = 0.0
    for s in range(meta.num_seqs):
        sid = meta.seq_ids[s]
        for j in range(meta.n_new[s]):
            t = meta.q_start[s] + j
            p = meta.seen[s] + j
            for h in range(H_q):
                kvh = h // (H_q // H_kv)
                keys = [r[kvh].tolist() for r in rk[sid][: p + 1]]
                vals = [r[kvh].tolist() for r in rv[sid][: p + 1]]
                want = _brute(q[t, h].tolist(), keys, vals, scale)
                err = max(err, float(np.max(np.abs(got[(t, h)] - np.array(want)))))
    return err


def test_brute_force_tiny():
    assert _check_brute_force(np.random.default_rng(2)) < 1e-12


def _check_sdpa(rng, prefix=37, n=23, H_q=6, H_kv=2, D=16, B=8):
    """One sequence: prefix cached by a first pass, then an n-token chunk."""
    plan = [(prefix, 0, [(1, prefix + n, 0)]), (n, 0, [(1, prefix + n, prefix)])]
    _, kc, vc, passes, rk, rv = _run_passes(rng, H_q, H_kv, D, B, np.float64, plan)
    meta, q = passes[-1]
    got = oracle.blocked_attention_array(meta, q, kc, vc, H_q)
    L = prefix + n
    K = torch.from_numpy(np.stack(rk[1])).permute(1, 0, 2)      # [H_kv, L, D]
    V = torch.from_numpy(np.stack(rv[1])).permute(1, 0, 2)
    g = H_q // H_kv
    K = K.repeat_interleave(g, dim=0)
    V = V.repeat_interleave(g, dim=0)
    Q = torch.from_numpy(q).permute(1, 0, 2)                       # [H_q, n, D]
    mask = torch.arange(L)[None, :] <= (prefix + torch.arange(n))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask)
    return float(np.max(np.abs(got - ref.permute(1, 0, 2).numpy())))


def test_library_special_case_sdpa():
    assert _check_sdpa(np.random.default_rng(3)) < 1e-12
    assert _check_sdpa(np.random.default_rng(4), prefix=0, n=17, H_q=4, H_kv=4) < 1e-12


def _check_context_one(rng):
    H_q, H_kv, D, B = 4, 2, 8, 4
    plan = [(1, 0, [(1, 1, 0)])]
    _, kc, vc, passes, rk, rv = _run_passes(rng, H_q, H_kv, D, B, np.float32, plan)
    meta, q = passes[0]
    got = oracle.blocked_attention_array(meta, q, kc, vc, H_q)
    v = widen(rv[1][0])
    return all(np.array_equal(got[0, h], v[h // 2]) for h in range(H_q))


def test_single_key_returns_its_value_exactly():
    assert _check_context_one(np.random.default_rng(5))


def _check_constant_keys(rng):
    H_q, H_kv, D, B = 2, 1, 8, 4
    comp = Composer(B, 64)
    kc = BlockedCache(H_kv, B, D, np.float64)
    vc = BlockedCache(H_kv, B, D, np.float64)
    meta = comp.compose(19, 0, [(1, 19, 0)])
    kk = np.tile(rng.standard_normal(D), (19, H_kv, 1))
    vv = rng.standard_normal((19, H_kv, D))
    kv_append(meta, kk, vv, kc, vc)
    q = rng.standard_normal((19, H_q, D))
    got = oracle.blocked_attention_array(meta, q, kc, vc, H_q)
    err = 0.0
    for t in range(19):
        err = max(err, float(np.max(np.abs(got[t, 0] - vv[: t + 1, 0].mean(axis=0)))))
    return err


def test_identical_keys_give_mean_of_visible_values():
    assert _check_constant_keys(np.random.default_rng(6)) < 1e-12


# --------------------------------------------------------------------------
# split invariance (FastGen guide, Step 4) and the combine
# --------------------------------------------------------------------------

def _check_split_invariance(rng):
    seq, heads, D = 4096, 8, 128
    scale = 1.0 / math.sqrt(D)
    err = 0.0
    for h in range(heads):
        q = rng.standard_normal(D)
        K = rng.standard_normal((seq, D))
        V = rng.standard_normal((seq, D))
        dense = oracle.dense_causal_attention(q[None, None, :], K[:, None, :],
                                              V[:, None, :], offset=seq - 1)[0, 0]
        c = -(-seq // 8)
        bounds = [min(i * c, seq) for i in range(9)]
        err = max(err, float(np.max(np.abs(oracle.split_attention(q, K, V, bounds, scale) - dense))))
        # ragged cuts, including an empty split
        bounds = [0, 1, 1, 700, 2049, 4000, seq]
        err = max(err, float(np.max(np.abs(oracle.split_attention(q, K, V, bounds, scale) - dense))))
    return err


def test_split_invariance_fp64():
    assert _check_split_invariance(np.random.default_rng(8)) < 1e-12


# --------------------------------------------------------------------------
# chunk invariance
# --------------------------------------------------------------------------

def test_chunked_prompt_equals_one_shot_causal():
    rng = np.random.default_rng(9)
    H_q, H_kv, D, B = 4, 2, 16, 8
    P = 101
    comp = Composer(B, 256)
    kc = BlockedCache(H_kv, B, D, np.float64)
    vc = BlockedCache(H_kv, B, D, np.float64)
    comp.compose(30, 0, [(2, 30, 0)])          # a decoding neighbour
    q_all = rng.standard_normal((P, H_q, D))
    k_all = rng.standard_normal((P, H_kv, D))
    v_all = rng.standard_normal((P, H_kv, D))
    out = np.zeros((P, H_q, D))
    seen, other = 0, 30
    while seen < P:
        meta = comp.compose(13, 7, [(2, 30, other), (1, P, seen)])
        T = meta.num_tokens
        q = np.zeros((T, H_q, D))
        k = rng.standard_normal((T, H_kv, D))
        v = rng.standard_normal((T, H_kv, D))
        s1 = meta.seq_ids.index(1)
        a, n = meta.q_start[s1], meta.n_new[s1]
        q[a:a + n], k[a:a + n], v[a:a + n] = (q_all[seen:seen + n], k_all[seen:seen + n],
                                              v_all[seen:seen + n])
        kv_append(meta, k, v, kc, vc)
        res = oracle.blocked_attention(meta, q, kc, vc, H_q, tokens=range(a, a + n))
        for j in range(n):
            for h in range(H_q):
                out[seen + j, h] = res[(a + j, h)]
        seen += n
        other += 1
    ref = oracle.dense_causal_attention(q_all, k_all, v_all, offset=0)
    assert np.max(np.abs(out - ref)) < 1e-12


# --------------------------------------------------------------------------
# planted mistakes: each must trip at least one pin
# --------------------------------------------------------------------------

def _pins_fail():
    rng = np.random.default_rng(11)
    try:
        checks = [
            _check_brute_force(rng) < 1e-12,
            _check_sdpa(rng) < 1e-12,
            _check_context_one(rng),
            _check_constant_keys(rng) < 1e-12,
        ]
    except Exception:
        return True
    return not all(checks)


def test_pins_hold_for_the_oracle_as_written():
    assert not _pins_fail()


def test_pins_catch_dropped_scale(monkeypatch):
    orig = oatt._softmax_attend
    monkeypatch.setattr(oatt, "_softmax_attend", lambda q, K, V, s: orig(q, K, V, 1.0))
    assert _pins_fail()


def test_pins_catch_off_by_one_causal_range(monkeypatch):
    orig = oatt._softmax_attend
    monkeypatch.setattr(oatt, "_softmax_attend",
                        lambda q, K, V, s: orig(q, K[:-1], V[:-1], s) if len(K) > 1 else orig(q, K, V, s))
    assert _pins_fail()


def test_pins_catch_wrong_group_mapping(monkeypatch):
    monkeypatch.setattr(oatt, "kv_head_of", lambda h, g: h % 2)
    assert _pins_fail()


def test_pins_catch_transposed_weights(monkeypatch):
    def bad(q, K, V, scale):
        s = (K @ q) * scale
        w = np.exp(s - s.max())
        return (w[::-1] @ V) / w.sum()          # weights applied to the wrong rows
    monkeypatch.setattr(oatt, "_softmax_attend", bad)
    assert _pins_fail()


def test_split_pin_catches_max_instead_of_lse(monkeypatch):
    """The guide's diagram combines with local maxima m_i; with normalised
    partial outputs that is wrong, and split invariance catches it."""
    def bad_split(q, K, V, bounds, scale):
        parts = []
        for a, b in zip(bounds[:-1], bounds[1:]):
            if b <= a:
                continue
            s = (K[a:b] @ q) * scale
            m = s.max()
            w = np.exp(s - m)
            parts.append(((w @ V[a:b]) / w.sum(), m))
        return oatt.lse_combine(parts)
    monkeypatch.setattr(oracle, "split_attention", bad_split)
    assert _check_split_invariance(np.random.default_rng(12)) > 1e-6
