"""Seeded synthetic workloads for the ragged blocked-KV attention pass.

This module is the one piece that both the fp64 oracle (``oracle/``) and the
CUDA library's tests and benchmark share.  It holds no arithmetic of the method
itself: it only draws request lengths and Q/K/V values from seeds, and states
which sequences sit in the cache before a pass and in which order the caller
lists them.  Composition, appending and attention are done by each side on its
own.

Workload shapes follow the pages' settings: Llama-2-7B, Llama-2-70B and
Mistral-7B attention shapes; normally distributed prompt and output lengths
with means 2600 and 60 and 30% standard deviation
("DeepSpeed-FastGen" paper summary page, Key points, benchmark setup); a
512-request closed-loop trace from up to 32 clients (same passage).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np

# --------------------------------------------------------------------------
# Shapes and scenarios
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class Shape:
    """Attention shape of one layer and the storage type of Q/K/V/O."""
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    block_size: int
    dtype: str            # "f32" or "bf16"
    input_scale: float    # Q/K/V values are N(0,1) * input_scale

    @property
    def group(self) -> int:
        return self.num_heads_q // self.num_heads_kv


@dataclass
class Scenario:
    """A pass (or a run of passes) and the cache contents it starts from.

    ``histories``: (seq_id, tokens) already in the cache before the first
    measured pass.  They are put there by ONE registration pass in which every
    history is listed as a prompt ``(seq_id, prompt_len=tokens, seen=0)`` in
    this order, with a budget equal to the total and no chunk cap.
    ``requests``: (seq_id, prompt_len, seen) for the first measured pass, in
    the caller's list order.
    """
    name: str
    shape: Shape
    budget: int
    max_chunk: int
    histories: List[Tuple[int, int]]
    requests: List[Tuple[int, int, int]]
    num_blocks: int
    notes: str = ""

    def registration(self) -> Tuple[int, List[Tuple[int, int, int]]]:
        """(budget, states) of the registration pass that fills the histories."""
        states = [(sid, n, 0) for sid, n in self.histories]
        return sum(n for _, n in self.histories), states


def _blocks_for(lengths: Sequence[int], block_size: int) -> int:
    return sum((int(n) + block_size - 1) // block_size for n in lengths)


def tiny(seed: int = 0) -> Scenario:
    """8 query heads, 2 KV heads, head_dim 64, block 16, budget 64, fp32.

    The pass lists a 90-token prompt (A), three decoding sequences whose caches
    hold 37, 100 and 5 tokens, and a 60-token prompt (B).  With a chunk cap of
    40 the pass holds 40 + 3 + 21 = 64 tokens.
    """
    del seed  # lengths are fixed by the configuration text
    shape = Shape(8, 2, 64, 16, "f32", 1.0)
    hist = [(1, 37), (2, 100), (3, 5)]
    reqs = [(4, 90, 0), (1, 37, 37), (2, 100, 100), (3, 5, 5), (5, 60, 0)]
    return Scenario("tiny", shape, 64, 40, hist, reqs, num_blocks=64)


def llama2_7b(seed: int = 0, prompt_len: int = 4096) -> Scenario:
    """32/32 heads, head_dim 128, bf16, block 64, budget 512, chunk cap 512.

    One 4096-token prompt chunked over successive passes alongside 15 decode
    sequences whose contexts are round(N(2600, 780^2)) clipped to [64, 8192].
    """
    rng = np.random.default_rng(seed)
    ctx = np.clip(np.rint(rng.normal(2600.0, 0.3 * 2600.0, size=15)), 64, 8192)
    ctx = [int(c) for c in ctx]
    shape = Shape(32, 32, 128, 64, "bf16", 1.0 / math.sqrt(128.0))
    hist = [(100 + i, c) for i, c in enumerate(ctx)]
    reqs = [(1, prompt_len, 0)] + [(100 + i, c, c) for i, c in enumerate(ctx)]
    # room for the prompt twice over (a fresh prompt per cycle) plus decode
    # growth of a few thousand passes
    nb = _blocks_for([c + 4096 for c in ctx], 64) + 2 * _blocks_for([prompt_len], 64) + 16
    return Scenario("llama2_7b", shape, 512, 512, hist, reqs, num_blocks=nb)


def decode_stress(seed: int = 0) -> Scenario:
    """64/8 heads (GQA 8), head_dim 128, bf16, block 64; 64 decodes only.

    Contexts are round(exp(U[ln 512, ln 16000])).
    """
    rng = np.random.default_rng(seed)
    ctx = np.rint(np.exp(rng.uniform(math.log(512.0), math.log(16000.0), size=64)))
    ctx = [int(c) for c in ctx]
    shape = Shape(64, 8, 128, 64, "bf16", 1.0 / math.sqrt(128.0))
    hist = [(100 + i, c) for i, c in enumerate(ctx)]
    reqs = [(100 + i, c, c) for i, c in enumerate(ctx)]
    nb = _blocks_for([c + 512 for c in ctx], 64) + 16
    return Scenario("decode_stress", shape, 64, 0, hist, reqs, num_blocks=nb)


def mistral_7b(seed: int = 0) -> Scenario:
    """32/8 heads, head_dim 128, bf16, block 64, budget 2048, chunk cap 768.

    Prompt X (2304 tokens, nothing cached), prompt Y (2304 tokens, 1536
    cached) and 512 decodes with contexts uniform in [128, 8192].
    """
    rng = np.random.default_rng(seed)
    ctx = [int(c) for c in rng.integers(128, 8193, size=512)]
    shape = Shape(32, 8, 128, 64, "bf16", 1.0 / math.sqrt(128.0))
    hist = [(2, 1536)] + [(100 + i, c) for i, c in enumerate(ctx)]
    reqs = [(1, 2304, 0), (2, 2304, 1536)] + [(100 + i, c, c) for i, c in enumerate(ctx)]
    nb = _blocks_for([c + 64 for c in ctx] + [2304, 2304], 64) + 16
    return Scenario("mistral_7b", shape, 2048, 768, hist, reqs, num_blocks=nb)


def prefill_mistral(seed: int = 0, prompts: int = 16) -> Scenario:
    """A chunk-dominated pass at the Mistral-7B attention shape (32/8 heads,
    head_dim 128, bf16, block 64): ``prompts`` prompts of 2304 tokens, each
    with 1536 tokens cached and its last 768-token chunk in the pass (the
    second prompt of the Mistral-7B workload, ``prompts`` times); budget
    768 x prompts, chunk cap 768, no decodes."""
    del seed  # lengths are fixed
    shape = Shape(32, 8, 128, 64, "bf16", 1.0 / math.sqrt(128.0))
    hist = [(10 + i, 1536) for i in range(prompts)]
    reqs = [(10 + i, 2304, 1536) for i in range(prompts)]
    nb = _blocks_for([2304] * prompts, 64) + 16
    return Scenario("prefill_mistral", shape, 768 * prompts, 768, hist, reqs, num_blocks=nb)


def short_prompts(num_heads_q: int, num_heads_kv: int, seed: int = 0) -> Scenario:
    """Short prompt chunks next to decodes, head_dim 128, bf16, block 64.

    12 prompts of 2..16 new tokens behind a cached prefix of 1..299 tokens, 12
    decodes with such contexts, and 40 fresh prompts of 2..16 tokens; the
    budget holds every token (no chunk cap)."""
    rng = np.random.default_rng(seed)
    shape = Shape(num_heads_q, num_heads_kv, 128, 64, "bf16", 1.0 / math.sqrt(128.0))
    hist = [(100 + i, int(rng.integers(1, 300))) for i in range(24)]
    reqs = [(100 + i, c + int(rng.integers(2, 17)), c) for i, (_, c) in enumerate(hist[:12])]
    reqs += [(100 + i, c, c) for i, (_, c) in enumerate(hist[12:], start=12)]
    reqs += [(900 + i, int(rng.integers(2, 17)), 0) for i in range(40)]
    budget = sum(p - s if p > s else 1 for _, p, s in reqs)
    nb = sum(-(-(c + 40) // 64) for _, c in hist) + 40 + 16
    return Scenario("short_prompts", shape, budget, 0, hist, reqs, nb)


SCENARIOS = {
    "tiny": tiny,
    "llama2_7b": llama2_7b,
    "decode_stress": decode_stress,
    "mistral_7b": mistral_7b,
    "prefill_mistral": prefill_mistral,
}


def scaled(scn: Scenario, factor: int) -> Scenario:
    """Same scenario with every cached length and prompt divided by ``factor``
    (at least 1 token each): a cheaper case of the same structure.

    Every decoding request is kept, and so is its one token in the budget;
    only the budget's prompt share (budget minus the decode count) and the
    chunk cap are divided by ``factor``.  The scaled pass therefore holds the
    same kinds of rows as the full one: decodes and prompt chunks."""
    def d(n: int) -> int:
        return max(1, n // factor)
    hist = [(s, d(n)) for s, n in scn.histories]
    hmap = dict(hist)
    reqs = []
    n_decode = 0
    for s, p, seen in scn.requests:
        if s in hmap and seen > 0:
            ns = hmap[s]
            if seen >= p:
                n_decode += 1
            reqs.append((s, ns if seen >= p else max(ns + 1, d(p)), ns))
        else:
            reqs.append((s, d(p), 0))
    prompt_share = max(0, scn.budget - n_decode)
    budget = n_decode + (max(1, prompt_share // factor) if prompt_share else 0)
    return Scenario(scn.name + f"/{factor}", scn.shape, max(1, budget),
                    max(0, scn.max_chunk // factor), hist, reqs, scn.num_blocks, scn.notes)


# --------------------------------------------------------------------------
# Q/K/V values
# --------------------------------------------------------------------------

_TAGS = {"q": 1, "k": 2, "v": 3}


def _stream_seed(seed: int, pass_index: int, tag: str) -> int:
    # distinct, reproducible stream per (seed, pass, tensor)
    return (int(seed) * 1_000_003 + int(pass_index) * 7919 + _TAGS[tag] * 104_729) % (2**63 - 1)


def make_qkv(shape: Shape, num_tokens: int, seed: int, pass_index: int,
             device: str = "cpu", which: str = "qkv"):
    """Q ``[T][H_q][D]`` and new K, V ``[T][H_kv][D]`` for one pass.

    Values are i.i.d. N(0,1) drawn in fp32 from a seeded torch generator on
    ``device``, multiplied by ``shape.input_scale`` and rounded to the storage
    type (round-to-nearest-even for bf16).  The same (seed, pass, device) gives
    the same values.  ``which`` selects the tensors returned (e.g. "kv").
    """
    import torch
    dt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    out = []
    for tag, heads in (("q", shape.num_heads_q), ("k", shape.num_heads_kv), ("v", shape.num_heads_kv)):
        if tag not in which:
            continue
        g = torch.Generator(device=device)
        g.manual_seed(_stream_seed(seed, pass_index, tag))
        x = torch.randn((num_tokens, heads, shape.head_dim), generator=g,
                        dtype=torch.float32, device=device)
        if shape.input_scale != 1.0:
            x = x * shape.input_scale
        out.append(x.to(dt).contiguous())
    return tuple(out)


# --------------------------------------------------------------------------
# Closed-loop request trace (512 requests, 32 clients)
# --------------------------------------------------------------------------


@dataclass
class Request:
    seq_id: int
    client: int
    prompt_len: int
    output_len: int
    seen: int = 0
    generated: int = 0


def trace_requests(seed: int = 0, num_requests: int = 512, num_clients: int = 32,
                   prompt_mean: float = 2600.0, output_mean: float = 60.0) -> List[Request]:
    """Prompt lengths round(N(2600, 780^2)) and output lengths round(N(60, 18^2)),
    both clipped to at least 1.  Client c owns requests c*k .. c*k+k-1 (k =
    num_requests / num_clients) and sends them one after another."""
    rng = np.random.default_rng(seed)
    p = np.maximum(1, np.rint(rng.normal(prompt_mean, 0.3 * prompt_mean, size=num_requests))).astype(int)
    g = np.maximum(1, np.rint(rng.normal(output_mean, 0.3 * output_mean, size=num_requests))).astype(int)
    per = num_requests // num_clients
    reqs = []
    for i in range(num_requests):
        reqs.append(Request(seq_id=1000 + i, client=min(i // per, num_clients - 1),
                            prompt_len=int(p[i]), output_len=int(g[i])))
    return reqs


def trace_block_pool(reqs: Sequence[Request], num_clients: int, block_size: int) -> int:
    """Blocks enough for every client to hold its largest request at once."""
    worst = max(r.prompt_len + r.output_len for r in reqs)
    return num_clients * ((worst + block_size - 1) // block_size) + 16


def run_trace(reqs: Sequence[Request], num_clients: int, budget: int, max_chunk: int,
              compose: Callable[[int, int, List[Tuple[int, int, int]]], object],
              release: Callable[[int], None],
              on_pass: Optional[Callable[[int, object, List[Request]], None]] = None,
              max_passes: Optional[int] = None) -> int:
    """Drive a closed-loop trace through ``compose`` until every request ends.

    Bookkeeping only.  ``compose(budget, max_chunk, states)`` must return an
    object with ``seq_ids`` and ``n_new`` (the tokens it scheduled per listed
    sequence).  A request is prefilling while ``seen < prompt_len``; the pass
    that completes its prompt yields output token 1, and every later pass in
    which it is scheduled yields one more, so its cache ends at
    ``prompt_len + output_len - 1`` tokens.  A finished request is released
    and its client's next request joins the end of the list (list order =
    submission order, ties by client id).  Returns the number of passes.
    """
    queues = {c: [r for r in reqs if r.client == c] for c in range(num_clients)}
    active: List[Request] = []
    for c in range(num_clients):
        if queues[c]:
            active.append(queues[c].pop(0))
    npass = 0
    while active:
        if max_passes is not None and npass >= max_passes:
            break
        states = [(r.seq_id, r.prompt_len, r.seen) for r in active]
        meta = compose(budget, max_chunk, states)
        if on_pass is not None:
            on_pass(npass, meta, active)
        sched = dict(zip([int(s) for s in meta.seq_ids], [int(n) for n in meta.n_new]))
        finished = []
        for r in active:
            n = sched.get(r.seq_id, 0)
            if n == 0:
                continue
            was_prefill = r.seen < r.prompt_len
            r.seen += n
            if was_prefill:
                if r.seen >= r.prompt_len:
                    r.generated = 1
            else:
                r.generated += 1
            if r.generated >= r.output_len:
                finished.append(r)
        for r in sorted(finished, key=lambda x: x.client):
            active.remove(r)
            release(r.seq_id)
        for r in sorted(finished, key=lambda x: x.client):
            if queues[r.client]:
                active.append(queues[r.client].pop(0))
        npass += 1
    return npass
