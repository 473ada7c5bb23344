"""One decoder layer around the attention pass (oracle).

Source: DeepSpeed-FastGen paper summary page, idea I1 - a forward pass's
latency follows its token count; its token-proportional work is the layer's
projections around attention.  The pages give no layer; the reading taken is
a Llama-2-7B decoder layer (the model of the paper summary's benchmark
setup): pre-normalisation with RMSNorm, QKV projection, causal attention over
the blocked cache, output projection with a residual, RMSNorm, a SwiGLU MLP
(silu(x W_gate^T) * (x W_up^T)) W_down^T with a residual.  Rotary position
embeddings are left out (they would only rotate Q and K before the append).

Every product is computed in fp64 from the stored (bf16 or fp32) values.
``store`` rounds a result to the precision the layer stores it in: None keeps
fp64 (the exact layer), ``round_bf16`` rounds as a bf16 layer does (to fp32,
then to bf16, round-to-nearest-even), so that a comparison with such a layer
measures arithmetic error only.
"""
from __future__ import annotations

import math
from typing import Callable, Optional

import numpy as np

from .attention import blocked_attention
from .cache import BlockedCache, kv_append
from .composer import PassMeta


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 -> bf16 (round-to-nearest-even on the 16 dropped bits),
    returned as fp64 values."""
    f = np.asarray(x, np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of values already representable in bf16."""
    return (np.asarray(x, np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def rmsnorm(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """Each row divided by the root of its mean square (plus eps), times weight."""
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(weight, np.float64)


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x)."""
    x = np.asarray(x, np.float64)
    return x / (1.0 + np.exp(-x))


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """x W^T with W stored [out][in]."""
    return np.asarray(x, np.float64) @ np.asarray(w, np.float64).T


def decoder_layer(meta: PassMeta, x: np.ndarray, weights: dict, k_cache: BlockedCache,
                  v_cache: BlockedCache, num_heads_q: int, num_heads_kv: int,
                  eps: float = 1e-5,
                  store: Optional[Callable[[np.ndarray], np.ndarray]] = None) -> dict:
    """The layer for the pass's rows x ([T][hidden], values): returns its
    intermediates and output.  The pass's K and V rows are appended to the
    caches (as bf16 bit patterns when ``store`` is given, else as fp32).
    ``weights``: w_qkv [(H_q + 2 H_kv) D][hidden] (Q rows, then K, then V),
    w_o [hidden][H_q D], w_gate and w_up [ffn][hidden], w_down [hidden][ffn],
    g_attn and g_mlp [hidden]."""
    s = store if store is not None else (lambda a: a)
    T, hidden = x.shape
    D = hidden // num_heads_q
    a = s(rmsnorm(x, weights["g_attn"], eps))
    qkv = s(linear(a, weights["w_qkv"]))
    q = qkv[:, : num_heads_q * D].reshape(T, num_heads_q, D)
    k = qkv[:, num_heads_q * D: (num_heads_q + num_heads_kv) * D].reshape(T, num_heads_kv, D)
    v = qkv[:, (num_heads_q + num_heads_kv) * D:].reshape(T, num_heads_kv, D)
    if store is not None:
        kv_append(meta, to_bf16_bits(k), to_bf16_bits(v), k_cache, v_cache)
        qs = to_bf16_bits(q)
    else:
        kv_append(meta, k.astype(np.float32), v.astype(np.float32), k_cache, v_cache)
        qs = q
    att = blocked_attention(meta, qs, k_cache, v_cache, num_heads_q)
    o = np.zeros((T, num_heads_q, D), np.float64)
    for (t, h), row in att.items():
        o[t, h] = row
    o = s(o).reshape(T, num_heads_q * D)
    h1 = s(x + linear(o, weights["w_o"]))
    b = s(rmsnorm(h1, weights["g_mlp"], eps))
    act = s(silu(linear(b, weights["w_gate"])) * linear(b, weights["w_up"]))
    out = s(h1 + linear(act, weights["w_down"]))
    return {"a": a, "q": q, "k": k, "v": v, "o": o, "h": h1, "b": b, "act": act, "out": out}
