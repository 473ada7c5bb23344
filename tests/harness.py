"""Side-by-side driver: the CUDA library and the fp64 oracle on the same
seeded inputs (test infrastructure; imports both, neither imports it).

A ``Pair`` holds a library composer with its device caches and an oracle
composer with its host caches.  Every pass is composed by both, appended by
both and, when asked, attended by both; results come back as plain numbers.
Inputs are drawn once by ``workloads.make_qkv`` and handed to each side.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Optional, Sequence, Set, Tuple

import numpy as np
import torch

import oracle
import workloads

FIELDS = ("seq_ids", "q_start", "n_new", "seen", "ctx", "block_start", "block_ids", "slot")

MAX_ABS_TOL = 1e-2
MEAN_ABS_TOL = 1e-3


def to_storage(t: torch.Tensor) -> np.ndarray:
    """Tensor -> numpy in the oracle's storage type (uint16 bits for bf16)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


class Pair:
    def __init__(self, rbkv, shape: workloads.Shape, num_blocks: int, seed: int = 0,
                 only_seqs: Optional[Set[int]] = None, input_device: str = "cpu",
                 cache_fill: Optional[float] = None, policy: str = "greedy"):
        self.rbkv = rbkv
        self.policy = policy
        self.shape = shape
        self.seed = seed
        self.only = only_seqs
        self.input_device = input_device
        self.cfg = rbkv.Config(shape.num_heads_q, shape.num_heads_kv, shape.head_dim,
                               shape.block_size, shape.dtype, num_blocks)
        self.lib = rbkv.Composer(self.cfg)
        self.orc = oracle.Composer(shape.block_size, num_blocks)
        dt = self.cfg.torch_dtype
        if cache_fill is None:
            self.kc = torch.zeros(self.cfg.cache_shape(), dtype=dt, device="cuda")
            self.vc = torch.zeros(self.cfg.cache_shape(), dtype=dt, device="cuda")
        else:
            self.kc = torch.full(self.cfg.cache_shape(), cache_fill, dtype=dt, device="cuda")
            self.vc = torch.full(self.cfg.cache_shape(), cache_fill, dtype=dt, device="cuda")
        storage = np.uint16 if shape.dtype == "bf16" else np.float32
        self.okc = oracle.BlockedCache(shape.num_heads_kv, shape.block_size, shape.head_dim, storage)
        self.ovc = oracle.BlockedCache(shape.num_heads_kv, shape.block_size, shape.head_dim, storage)
        self.npass = 0
        self.stream = torch.cuda.Stream()

    # ------------------------------------------------------------------
    def _rows_of(self, meta, seqs: Optional[Set[int]]) -> np.ndarray:
        rows = []
        for s in range(meta.num_seqs):
            if seqs is None or meta.seq_ids[s] in seqs:
                rows.extend(range(meta.q_start[s], meta.q_start[s + 1]))
        return np.asarray(rows, dtype=np.int64)

    def step(self, budget: int, max_chunk: int, states: Sequence[Tuple[int, int, int]],
             attend: bool = True, split_keys: Optional[int] = None,
             tokens: Optional[Iterable[int]] = None, chunk_items: Optional[str] = None) -> dict:
        """Compose, append and (optionally) attend one pass on both sides."""
        res: dict = {}
        p = self.lib.compose(budget, max_chunk, states, policy=self.policy)
        m = self.orc.compose(budget, max_chunk, states, policy=self.policy)
        res["meta_equal"] = all(
            np.array_equal(np.asarray(getattr(p.meta, f), np.int64), np.asarray(getattr(m, f), np.int64))
            for f in FIELDS)
        res["meta"] = m
        res["tokens"] = m.num_tokens
        T = m.num_tokens
        idx = self.npass
        self.npass += 1
        if T == 0:
            res["plan"] = p.plan()
            return res
        if split_keys is not None:
            p.set_split_keys(split_keys)
        if chunk_items is not None:
            p.set_chunk_items(chunk_items)
        which = "qkv" if attend else "kv"
        ten = workloads.make_qkv(self.shape, T, self.seed, idx, device=self.input_device, which=which)
        if attend:
            q, k, v = ten
        else:
            k, v = ten
        # inputs and caches were made on the default stream: order after them
        self.stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(self.stream):
            kd, vd = k.cuda(), v.cuda()
            self.rbkv.kv_append(p, kd, vd, self.kc, self.vc, stream=self.stream)
        # oracle append (restricted to sampled sequences for big passes)
        if self.only is None:
            ok, ov = to_storage(k), to_storage(v)
        else:
            rows = self._rows_of(m, self.only)
            ok = np.zeros((T,) + tuple(k.shape[1:]), dtype=to_storage(k[:1]).dtype)
            ov = np.zeros_like(ok)
            if len(rows):
                ridx = torch.as_tensor(rows, device=k.device)
                ok[rows] = to_storage(k.index_select(0, ridx))
                ov[rows] = to_storage(v.index_select(0, ridx))
        oracle.kv_append(m, ok, ov, self.okc, self.ovc, only_seqs=self.only)
        res["plan"] = p.plan()
        if attend:
            self.stream.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(self.stream):
                qd = q.cuda()
                o = self.rbkv.ragged_attention(p, qd, self.kc, self.vc, stream=self.stream)
            self.stream.synchronize()
            p.device_status(self.stream)
            if tokens is None:
                tok = list(self._rows_of(m, self.only)) if self.only is not None else list(range(T))
            else:
                tok = list(tokens)
            qs = to_storage(q) if self.only is None else None
            if qs is None:
                ridx = torch.as_tensor(np.asarray(tok, np.int64), device=q.device)
                qsub = to_storage(q.index_select(0, ridx))
                qs = np.zeros((T,) + qsub.shape[1:], qsub.dtype)
                qs[np.asarray(tok, np.int64)] = qsub
            want = oracle.blocked_attention(m, qs, self.okc, self.ovc, self.shape.num_heads_q,
                                            tokens=tok)
            got = to_f64(o)
            diffs = np.stack([np.abs(got[t, h] - w) for (t, h), w in want.items()]) if want else np.zeros(1)
            res["max_abs"] = float(diffs.max())
            res["mean_abs"] = float(diffs.mean())
            res["finite"] = bool(np.isfinite(got[tok]).all()) if tok else True
            res["o"] = o
            res["checked"] = len(want)
        else:
            self.stream.synchronize()
            p.device_status(self.stream)
        res["pass"] = p
        return res

    def cache_equal(self, blocks: Optional[Iterable[int]] = None) -> bool:
        """Bit-exact comparison of the device caches with the oracle's
        (all blocks, or the given ones)."""
        torch.cuda.synchronize()
        nb = self.cfg.num_blocks
        if blocks is None:
            gk, gv = to_storage(self.kc), to_storage(self.vc)
            return (np.array_equal(gk, self.okc.dense(nb)) and np.array_equal(gv, self.ovc.dense(nb)))
        for b in blocks:
            if not np.array_equal(to_storage(self.kc[b]), self.okc.block(b)):
                return False
            if not np.array_equal(to_storage(self.vc[b]), self.ovc.block(b)):
                return False
        return True

    def release(self, sid: int) -> None:
        self.lib.release(sid)
        self.orc.release(sid)


def run_scenario(rbkv, scn: workloads.Scenario, seed: int = 0, split_keys: Optional[int] = None,
                 passes: int = 1, only_seqs: Optional[Set[int]] = None,
                 input_device: str = "cpu", cache_fill: Optional[float] = None,
                 policy: str = "greedy", chunk_items: Optional[str] = None) -> List[dict]:
    """Registration pass, then ``passes`` measured passes with states advanced
    between them.  Returns the measured passes' results."""
    pair = Pair(rbkv, scn.shape, scn.num_blocks, seed, only_seqs, input_device, cache_fill,
                policy)
    b, st = scn.registration()
    if b > 0:
        r = pair.step(b, 0, st, attend=False)
        assert r["meta_equal"]
    states = list(scn.requests)
    out = []
    for _ in range(passes):
        r = pair.step(scn.budget, scn.max_chunk, states, split_keys=split_keys,
                      chunk_items=chunk_items)
        r["pair"] = pair
        out.append(r)
        n = dict(zip(r["meta"].seq_ids, r["meta"].n_new))
        states = [(sid, pl, seen + n.get(sid, 0)) for sid, pl, seen in states]
    return out
