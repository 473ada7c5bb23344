"""Exact blocked-cache causal attention in fp64 (oracle).

Definition (FastGen guide, Step 3's unsplit path and Step 4's ground truth):
scores are the query-key dot products scaled by 1/sqrt(d), a softmax over them
gives the weights, and the output is the weighted sum of the value rows.

For sequence s and its pass token at position p = seen[s] + j, query head h
reads KV head ``h // g`` (g = H_q / H_kv, contiguous groups - the pages use one
KV head per query head; grouped heads are read this way) and attends keys
0..p of its sequence (the cached prefix, the earlier tokens of its own chunk
and itself), read through the block table after this pass's append:

    O[t, h, :] = sum_i softmax_i(q . K_i / sqrt(D)) V_i,   i = 0..p

The method reaches exactly this result with split-KV and a log-sum-exp combine
(FastGen guide, "Two-Phase Softmax Reduction", and Step 3's split path), and
with chunked prefill (paper summary page, Summary).  The oracle computes the
definition directly; ``split_attention`` and ``lse_combine`` restate the split
method so that tests can check it reproduces the definition.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np

from .cache import BlockedCache
from .composer import PassMeta


def widen(x: np.ndarray) -> np.ndarray:
    """Storage values -> fp64.  ``uint16`` arrays are bf16 bit patterns: a bf16
    is the top half of an IEEE binary32, so shifting left 16 bits gives the
    float32 with the same value, which widens exactly to fp64."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def kv_head_of(h: int, group: int) -> int:
    """Query head h reads KV head h // g (contiguous groups of g query heads)."""
    return h // group


def _softmax_attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """One query row against rows of K and V (all fp64)."""
    s = (K @ q) * scale
    m = s.max()
    w = np.exp(s - m)
    return (w @ V) / w.sum()


def blocked_attention(meta: PassMeta, q: np.ndarray, k_cache: BlockedCache,
                      v_cache: BlockedCache, num_heads_q: int,
                      tokens: Optional[Iterable[int]] = None,
                      heads: Optional[Iterable[int]] = None,
                      scale: Optional[float] = None) -> Dict[Tuple[int, int], np.ndarray]:
    """O rows for pass tokens ``tokens`` (default all) and query heads ``heads``
    (default all), as {(t, h): fp64 vector of length D}.

    ``q`` is ``[T][H_q][D]`` in storage type or fp64; the caches hold the pass's
    appended rows already.
    """
    D = k_cache.head_dim
    H_kv = k_cache.num_heads_kv
    g = num_heads_q // H_kv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    q64 = widen(q) if q.dtype != np.float64 else q
    T = meta.num_tokens
    tok_list = list(range(T)) if tokens is None else list(tokens)
    head_list = list(range(num_heads_q)) if heads is None else list(heads)
    seq_of = np.zeros(T, dtype=np.int64)
    for s in range(meta.num_seqs):
        seq_of[meta.q_start[s]:meta.q_start[s + 1]] = s
    out: Dict[Tuple[int, int], np.ndarray] = {}
    gathered: Dict[Tuple[int, int], Tuple[np.ndarray, np.ndarray]] = {}
    for t in tok_list:
        s = int(seq_of[t])
        p = meta.seen[s] + (t - meta.q_start[s])
        for h in head_list:
            kvh = kv_head_of(h, g)
            key = (s, kvh)
            if key not in gathered:
                table = meta.blocks_of(s)
                gathered[key] = (widen(k_cache.gather(table, meta.ctx[s], kvh)),
                                 widen(v_cache.gather(table, meta.ctx[s], kvh)))
            K, V = gathered[key]
            out[(t, h)] = _softmax_attend(q64[t, h], K[: p + 1], V[: p + 1], scale)
    return out


def blocked_attention_array(meta: PassMeta, q: np.ndarray, k_cache: BlockedCache,
                            v_cache: BlockedCache, num_heads_q: int) -> np.ndarray:
    """All of O as an fp64 array ``[T][H_q][D]``."""
    D = k_cache.head_dim
    res = blocked_attention(meta, q, k_cache, v_cache, num_heads_q)
    out = np.zeros((meta.num_tokens, num_heads_q, D), np.float64)
    for (t, h), v in res.items():
        out[t, h] = v
    return out


def dense_causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, offset: int,
                           scale: Optional[float] = None) -> np.ndarray:
    """Independent formulation without blocks: one sequence, whole arrays.

    ``q`` is ``[n][H_q][D]`` for positions offset..offset+n-1, ``k``/``v`` are
    ``[L][H_kv][D]`` for positions 0..L-1 (L >= offset + n).  Query row j sees
    keys 0..offset+j.  fp64 in, fp64 out.
    """
    n, H_q, D = q.shape
    H_kv = k.shape[1]
    g = H_q // H_kv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros((n, H_q, D), np.float64)
    for h in range(H_q):
        Kh = k[:, kv_head_of(h, g), :]
        Vh = v[:, kv_head_of(h, g), :]
        s = (q[:, h, :] @ Kh.T) * scale                      # [n, L]
        pos = offset + np.arange(n)[:, None]
        s = np.where(np.arange(k.shape[0])[None, :] <= pos, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        w = np.exp(s)
        out[:, h, :] = (w @ Vh) / w.sum(axis=1, keepdims=True)
    return out


def lse_combine(parts: Sequence[Tuple[np.ndarray, float]]) -> np.ndarray:
    """Combine normalised partial outputs O_i with their log-sum-exp LSE_i.

    O = sum_i exp(LSE_i - M) O_i / sum_i exp(LSE_i - M), M = max_i LSE_i
    (FastGen guide, Step 3's split path: rescale each split's normalised output
    by exp(lse_i - max lse) and divide by the summed rescale factors).  A split
    with no keys carries LSE = -inf and weight 0.
    """
    lses = np.array([l for _, l in parts], np.float64)
    M = lses.max()
    w = np.exp(lses - M)
    acc = sum(wi * o for wi, (o, _) in zip(w, parts))
    return acc / w.sum()


def split_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray,
                    bounds: Sequence[int], scale: float) -> np.ndarray:
    """Split-KV attention of one query row: keys cut at ``bounds``
    (0 = b_0 <= b_1 <= ... = len(K)); each split yields its softmax-normalised
    partial output and log-sum-exp, then ``lse_combine`` merges them."""
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b <= a:
            parts.append((np.zeros(V.shape[1]), -math.inf))
            continue
        s = (K[a:b] @ q) * scale
        m = s.max()
        w = np.exp(s - m)
        parts.append(((w @ V[a:b]) / w.sum(), m + math.log(w.sum())))
    return lse_combine(parts)
