"""The decoder-layer oracle pinned by what the mathematics fixes: bf16
rounding on exact values, RMSNorm's closed forms and invariances, SiLU's
closed forms, a layer with identity-like weights whose output is known in
closed form, and brute force on a tiny layer written as plain loops."""
import math

import numpy as np
import pytest

import oracle
from oracle import layer as L


def test_round_bf16_exact_cases():
    # representable values stay; ties go to the even neighbour
    assert L.round_bf16(np.array([1.0, -2.0, 0.0]))[0] == 1.0
    # bf16 keeps 7 mantissa bits: ulp(1) = 2^-7, ulp(3) = 2^-6
    one = 1.0
    assert L.round_bf16(np.array([one + 2 ** -8]))[0] == 1.0                 # tie -> even mantissa 0
    assert L.round_bf16(np.array([one + 3 * 2 ** -8]))[0] == one + 2 ** -6   # tie -> even mantissa 2
    assert L.round_bf16(np.array([one + 2 ** -8 + 2 ** -20]))[0] == one + 2 ** -7  # above the tie
    assert L.round_bf16(np.array([one + 2 ** -9]))[0] == 1.0                 # below half an ulp
    assert L.round_bf16(np.array([3.0 + 2 ** -8]))[0] == 3.0                 # a quarter ulp
    assert L.round_bf16(np.array([-(one + 3 * 2 ** -9)]))[0] == -(one + 2 ** -7)
    x = np.random.default_rng(0).normal(size=1000)
    r = L.round_bf16(x)
    assert np.all(np.abs(r - x) <= np.abs(x) * 2 ** -8)
    assert np.array_equal(L.round_bf16(r), r)                             # idempotent


def test_rmsnorm_closed_forms():
    w = np.ones(16)
    # a constant row normalises to its sign
    assert np.allclose(L.rmsnorm(np.full((1, 16), -3.0), w, 0.0), -1.0)
    x = np.random.default_rng(1).normal(size=(5, 16))
    y = L.rmsnorm(x, w, 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0)              # unit RMS
    assert np.allclose(L.rmsnorm(7.5 * x, w, 0.0), y)                     # scale invariant
    g = np.arange(1, 17, dtype=np.float64)
    assert np.allclose(L.rmsnorm(x, g, 0.0), y * g)                       # weight per column
    # eps enters under the root
    assert np.isclose(L.rmsnorm(np.full((1, 4), 2.0), np.ones(4), 5.0)[0, 0], 2.0 / 3.0)


def test_silu_closed_forms():
    x = np.array([0.0, 2.0, -2.0, 40.0, -40.0])
    s = L.silu(x)
    assert s[0] == 0.0
    assert np.isclose(s[1], 2.0 / (1.0 + math.exp(-2.0)))
    assert np.isclose(s[1] - s[2], 2.0)                                   # silu(x) - silu(-x) = x
    assert np.isclose(s[3], 40.0) and abs(s[4]) < 1e-15


def _single_token_pass(hidden, hq, hkv, D):
    comp = oracle.Composer(16, 8)
    m = comp.compose(1, 0, [(1, 1, 0)])
    kc = oracle.BlockedCache(hkv, 16, D, np.float32)
    vc = oracle.BlockedCache(hkv, 16, D, np.float32)
    return m, kc, vc


def test_identity_layer_closed_form():
    """Q, K, V and output projections the identity, zero MLP down weights, unit
    norm weights: one token attends only itself, so attention returns V = the
    normalised input and the layer outputs x + rmsnorm(x)."""
    hidden, hq, hkv, D, ffn = 8, 2, 2, 4, 6
    eye = np.eye(hidden)
    w = {"w_qkv": np.concatenate([eye, eye, eye]), "w_o": eye,
         "w_gate": np.ones((ffn, hidden)), "w_up": np.ones((ffn, hidden)),
         "w_down": np.zeros((hidden, ffn)), "g_attn": np.ones(hidden), "g_mlp": np.ones(hidden)}
    x = np.random.default_rng(2).normal(size=(1, hidden))
    m, kc, vc = _single_token_pass(hidden, hq, hkv, D)
    r = L.decoder_layer(m, x, w, kc, vc, hq, hkv, eps=1e-6)
    assert np.allclose(r["out"], x + L.rmsnorm(x, np.ones(hidden), 1e-6), atol=1e-12)
    # with the MLP: down = identity on the first hidden of ffn outputs
    w["w_down"] = np.eye(hidden, ffn)
    m, kc, vc = _single_token_pass(hidden, hq, hkv, D)
    r = L.decoder_layer(m, x, w, kc, vc, hq, hkv, eps=1e-6)
    h = x + L.rmsnorm(x, np.ones(hidden), 1e-6)
    b = L.rmsnorm(h, np.ones(hidden), 1e-6)
    s = b.sum()
    act = (s / (1 + math.exp(-s))) * s
    # the identity of [hidden][ffn] feeds the first ffn (6) of the 8 outputs
    assert np.allclose(r["out"], h + act * (np.arange(hidden) < ffn), atol=1e-10)


def test_tiny_layer_brute_force():
    """A 3-token prompt through a tiny GQA layer, every step as plain loops."""
    rng = np.random.default_rng(3)
    hidden, hq, hkv, D, ffn, T = 8, 4, 2, 2, 5, 3
    w = {"w_qkv": rng.normal(size=((hq + 2 * hkv) * D, hidden)), "w_o": rng.normal(size=(hidden, hq * D)),
         "w_gate": rng.normal(size=(ffn, hidden)), "w_up": rng.normal(size=(ffn, hidden)),
         "w_down": rng.normal(size=(hidden, ffn)), "g_attn": rng.normal(size=hidden),
         "g_mlp": rng.normal(size=hidden)}
    x = rng.normal(size=(T, hidden))
    comp = oracle.Composer(2, 8)
    m = comp.compose(T, 0, [(1, T, 0)])
    kc = oracle.BlockedCache(hkv, 2, D, np.float32)
    vc = oracle.BlockedCache(hkv, 2, D, np.float32)
    r = L.decoder_layer(m, x, w, kc, vc, hq, hkv, eps=1e-5)

    def norm(row, g):
        ms = sum(v * v for v in row) / len(row)
        return [row[i] / math.sqrt(ms + 1e-5) * g[i] for i in range(len(row))]

    def mv(mat, vec):
        return [sum(mat[o][i] * vec[i] for i in range(len(vec))) for o in range(len(mat))]

    f32 = lambda v: float(np.float32(v))   # the cache stores K and V as fp32
    qs, ks, vs = [], [], []
    for t in range(T):
        a = norm(list(x[t]), w["g_attn"])
        qkv = mv(w["w_qkv"], a)
        qs.append(qkv[: hq * D])
        ks.append([f32(v) for v in qkv[hq * D: (hq + hkv) * D]])
        vs.append([f32(v) for v in qkv[(hq + hkv) * D:]])
    for t in range(T):
        o = []
        for h in range(hq):
            kv = h // (hq // hkv)
            q = qs[t][h * D:(h + 1) * D]
            sc = [sum(q[d] * ks[j][kv * D + d] for d in range(D)) / math.sqrt(D) for j in range(t + 1)]
            mx = max(sc)
            e = [math.exp(s - mx) for s in sc]
            z = sum(e)
            o.extend(sum(e[j] * vs[j][kv * D + d] for j in range(t + 1)) / z for d in range(D))
        h1 = [x[t][i] + mv(w["w_o"], o)[i] for i in range(hidden)]
        b = norm(h1, w["g_mlp"])
        g = mv(w["w_gate"], b)
        u = mv(w["w_up"], b)
        act = [g[i] / (1 + math.exp(-g[i])) * u[i] for i in range(ffn)]
        out = [h1[i] + mv(w["w_down"], act)[i] for i in range(hidden)]
        assert np.allclose(r["out"][t], out, rtol=1e-9, atol=1e-9)


def test_planted_mistakes_trip_the_pins(monkeypatch):
    """Mistakes planted in the oracle - gate and up swapped, SiLU dropped, the
    RMS taken without the square root - each break a closed form above."""
    hidden, hq, hkv, D, ffn = 8, 2, 2, 4, 6
    eye = np.eye(hidden)
    w = {"w_qkv": np.concatenate([eye, eye, eye]), "w_o": eye,
         "w_gate": np.ones((ffn, hidden)), "w_up": 2 * np.ones((ffn, hidden)),
         "w_down": np.eye(hidden, ffn), "g_attn": np.ones(hidden), "g_mlp": np.ones(hidden)}
    x = np.random.default_rng(4).normal(size=(1, hidden))

    def run(weights):
        m, kc, vc = _single_token_pass(hidden, hq, hkv, D)
        return L.decoder_layer(m, x, weights, kc, vc, hq, hkv, eps=1e-6)["out"]
    good = run(w)
    assert not np.allclose(good, run(dict(w, w_gate=w["w_up"], w_up=w["w_gate"])))
    monkeypatch.setattr(L, "silu", lambda v: np.asarray(v, np.float64))
    assert not np.allclose(good, run(w))
    monkeypatch.undo()
    monkeypatch.setattr(L, "rmsnorm", lambda v, g, eps: np.asarray(v) / (np.mean(np.asarray(v) ** 2, axis=-1, keepdims=True) + eps) * g)
    y = L.rmsnorm(np.random.default_rng(5).normal(size=(3, 16)), np.ones(16), 0.0)
    assert not np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0)
