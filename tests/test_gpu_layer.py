"""The decoder layer's dense steps (tensor-core GEMM with fused epilogues,
RMSNorm) and a whole Llama-2-7B-shape layer around the attention pass, all
through the C ABI, against the fp64 oracle.

GEMM bar: the exact product of the bf16 operands (fp64) rounded once to bf16,
up to fp32 accumulation: |C - C_ref| <= 2^-8 |C_ref| + 2^-14 sum_k |A_ik B_jk|
for every element, and at least 98% of elements equal to the bf16 rounding of
the exact value.  Layer bar: see test_decoder_layer_against_oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import to_storage
from oracle import layer as L

pytestmark = pytest.mark.gpu


def _bf16(shape, gen, scale=1.0):
    return (torch.randn(*shape, generator=gen) * scale).to(torch.bfloat16)


def _f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def _check_gemm(got, ref, absdot):
    g = _f64(got)
    err = np.abs(g - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * absdot + 1e-30
    assert np.all(err <= bound), float((err / bound).max())
    exact = np.mean(g == L.round_bf16(ref))
    assert exact >= 0.98, exact


def _workspace(rbkv, m, n, k, split):
    if not split:
        return None
    need = rbkv.gemm_workspace_bytes(m, n, k)
    return torch.empty(max(256, need), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("m,n,k", [(1, 32, 8), (100, 288, 200), (128, 256, 64), (257, 4096, 4096),
                                   (512, 12288, 4096), (300, 4096, 11008), (16, 4096, 11008),
                                   (1, 12288, 4096), (1280, 12288, 2048), (384, 26624, 1024)])
@pytest.mark.parametrize("epilogue", ["plain", "residual"])
@pytest.mark.parametrize("split", [False, True])
def test_gemm_against_fp64(rbkv, m, n, k, epilogue, split):
    """With a workspace, products with fewer 128 x 256 tiles than SMs split K
    over several SMs (16 and 48 tiles), and products whose tiles fill a last
    wave only in part run whole waves whole and split the rest (512 x 12288:
    152 whole tiles and 40 in 3 pieces; 1280 x 12288 x 2048: 450 whole, 30 in 4;
    384 x 26624: 303 whole, 9 in 2); same bar."""
    gen = torch.Generator().manual_seed(m * 7 + n + k)
    a = _bf16((m, k), gen)
    b = _bf16((n, k), gen, 1.0 / math.sqrt(k))
    r = _bf16((m, n), gen) if epilogue == "residual" else None
    if split and (m, n, k) in ((16, 4096, 11008), (1, 12288, 4096), (512, 12288, 4096),
                               (1280, 12288, 2048), (384, 26624, 1024)):
        assert rbkv.gemm_workspace_bytes(m, n, k) > 0
    if (m, n, k) == (512, 12288, 4096):
        # the partials cover only the 40 split tiles' columns: 3 x 512 x 2560 fp32
        assert rbkv.gemm_workspace_bytes(m, n, k) == 3 * 512 * 2560 * 4
    c = rbkv.gemm(a.cuda(), b.cuda(), residual=None if r is None else r.cuda(), epilogue=epilogue,
                  workspace=_workspace(rbkv, m, n, k, split))
    torch.cuda.synchronize()
    a64, b64 = _f64(a), _f64(b)
    ref = a64 @ b64.T + (0.0 if r is None else _f64(r))
    _check_gemm(c, ref, np.abs(a64) @ np.abs(b64).T)


@pytest.mark.parametrize("m,ffn,k", [(77, 256, 512), (200, 11008, 4096), (8, 2048, 4096)])
@pytest.mark.parametrize("split", [False, True])
def test_gemm_swiglu_against_fp64(rbkv, m, ffn, k, split):
    from ragged_blocked_kv_gb300.layer import interleave_gate_up
    gen = torch.Generator().manual_seed(m + ffn)
    a = _bf16((m, k), gen)
    wg = _bf16((ffn, k), gen, 1.0 / math.sqrt(k))
    wu = _bf16((ffn, k), gen, 1.0 / math.sqrt(k))
    c = rbkv.gemm(a.cuda(), interleave_gate_up(wg, wu).cuda(), epilogue="swiglu",
                  workspace=_workspace(rbkv, m, 2 * ffn, k, split))
    torch.cuda.synchronize()
    a64 = _f64(a)
    gate, up = a64 @ _f64(wg).T, a64 @ _f64(wu).T
    ref = L.silu(gate) * up
    # silu(g) * u moves a product's error by at most |d(silu(g) u)| <= (|u| + |g|) x that error
    absdot = (np.abs(a64) @ np.abs(_f64(wg)).T) * (np.abs(up) + np.abs(gate) + 1.0) + \
        (np.abs(a64) @ np.abs(_f64(wu)).T) * np.abs(L.silu(gate))
    _check_gemm(c, ref, absdot)


@pytest.mark.parametrize("hq,hkv,m", [(32, 32, 130), (32, 8, 130), (32, 8, 5), (32, 32, 512)])
def test_gemm_qkv_split_outputs(rbkv, hq, hkv, m):
    k, D = 4096, 128
    gen = torch.Generator().manual_seed(hq + hkv)
    a = _bf16((m, k), gen)
    w = _bf16(((hq + 2 * hkv) * D, k), gen, 1.0 / math.sqrt(k))
    n = (hq + 2 * hkv) * D
    q, kk, vv = rbkv.gemm_qkv(a.cuda(), w.cuda(), hq, hkv, D,
                              workspace=_workspace(rbkv, m, n, k, True))
    torch.cuda.synchronize()
    assert q.shape == (m, hq, D) and kk.shape == (m, hkv, D) and q.is_contiguous()
    full = torch.cat([q.reshape(m, -1), kk.reshape(m, -1), vv.reshape(m, -1)], dim=1)
    a64, w64 = _f64(a), _f64(w)
    _check_gemm(full, a64 @ w64.T, np.abs(a64) @ np.abs(w64).T)


@pytest.mark.parametrize("m,h", [(1, 8), (37, 4096), (512, 4096)])
def test_rmsnorm_against_oracle(rbkv, m, h):
    gen = torch.Generator().manual_seed(m + h)
    x = _bf16((m, h), gen, 3.0)
    g = (1.0 + torch.randn(h, generator=gen) / 10).to(torch.bfloat16)
    y = rbkv.rmsnorm(x.cuda(), g.cuda(), eps=1e-5)
    torch.cuda.synchronize()
    ref = L.rmsnorm(_f64(x), _f64(g), 1e-5)
    err = np.abs(_f64(y) - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-5 * np.abs(ref).max())


def test_decoder_layer_against_oracle(rbkv):
    """A Llama-2-7B decoder layer (hidden 4096, 32 heads, ffn 11008) on a pass
    holding a 100-row chunk behind a 200-token prefix, a fresh 30-token prompt
    and 12 decodes, every step a library kernel, against the oracle layer with
    the same storage rounding (bf16 at every stored tensor).

    Bar: the oracle and the layer may store an intermediate one bf16 ulp apart
    where a rounding decision falls differently (fp32 against fp64 sums); such
    flips carried through the residual stream stay within a few bf16 ulps of
    the output: max-abs <= 4 x 2^-8 x max|out| and mean-abs <= 2^-8 x mean|out|."""
    from ragged_blocked_kv_gb300.layer import DecoderLayer, random_weights
    hidden, hq, hkv, D, ffn = 4096, 32, 32, 128, 11008
    shape = workloads.Shape(hq, hkv, D, 64, "bf16", 1.0)
    w = random_weights(hidden, hq, hkv, D, ffn, seed=11)
    layer = DecoderLayer(rbkv, w, hq, hkv, D)
    rng = np.random.default_rng(12)
    hist = [(1, 200)] + [(10 + i, int(rng.integers(50, 400))) for i in range(12)]
    reqs = [(1, 300, 200), (2, 30, 0)] + [(sid, n, n) for sid, n in hist[1:]]
    nb = sum(-(-(n + 120) // 64) for _, n in hist) + 8
    cfg = rbkv.Config(hq, hkv, D, 64, "bf16", nb)
    comp = rbkv.Composer(cfg)
    orc = oracle.Composer(64, nb)
    kc = torch.zeros(cfg.cache_shape(), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    okc = oracle.BlockedCache(hkv, 64, D, np.uint16)
    ovc = oracle.BlockedCache(hkv, 64, D, np.uint16)
    # the histories' K and V: seeded rows in both caches
    b0 = sum(n for _, n in hist)
    p0 = comp.compose(b0, 0, [(s, n, 0) for s, n in hist])
    m0 = orc.compose(b0, 0, [(s, n, 0) for s, n in hist])
    k0, v0 = workloads.make_qkv(shape, p0.num_tokens, 3, 0, device="cuda", which="kv")
    rbkv.kv_append(p0, k0, v0, kc, vc)
    oracle.kv_append(m0, to_storage(k0), to_storage(v0), okc, ovc)
    # the measured pass through the whole layer
    p = comp.compose(10_000, 0, reqs)
    m = orc.compose(10_000, 0, reqs)
    T = p.num_tokens
    assert T == 100 + 30 + 12
    x = (torch.randn(T, hidden, generator=torch.Generator().manual_seed(5))).to(torch.bfloat16)
    got = layer.forward(p, x.cuda(), kc, vc)
    torch.cuda.synchronize()
    p.device_status()
    ow = {k: _f64(v) for k, v in w.items() if k != "w_gu"}
    want = L.decoder_layer(m, _f64(x), ow, okc, ovc, hq, hkv, eps=1e-5, store=L.round_bf16)
    out_g, out_w = _f64(got["out"]), want["out"]
    err = np.abs(out_g - out_w)
    print(f"layer out: max-abs {err.max():.3e} mean-abs {err.mean():.3e} "
          f"max|out| {np.abs(out_w).max():.3f} mean|out| {np.abs(out_w).mean():.3f}")
    for name in ("a", "q", "o", "h", "b", "act"):
        e = np.abs(_f64(got[name]).reshape(T, -1) - want[name].reshape(T, -1))
        print(f"  {name}: max-abs {e.max():.3e} mean-abs {e.mean():.3e}")
    assert np.isfinite(out_g).all()
    assert err.max() <= 4 * 2.0 ** -8 * np.abs(out_w).max()
    assert err.mean() <= 2.0 ** -8 * np.abs(out_w).mean()
