"""Dynamic SplitFuse pass composition, written out step by step (oracle).

Source: "DeepSpeed-FastGen" paper summary page, Summary and idea I3 - each
pass is held to one token budget: a long prompt is cut into pieces that go
into successive passes, and generation tokens and short prompts take up the
rest of the budget; InfoQ release note - passes of a steady size, made
of pieces of prompts mixed with generation tokens.  The FastGen guide's
"Prompt-Decode Decoupling" adds that chunks are bounded (e.g. 512 tokens) and
interleaved with decode steps so generation never stalls.

The pages fix the goal, not the order of the steps.  Readings taken here:

1. The budget counts every token of the pass, generation tokens included.
2. Generation tokens are admitted first, one per decoding sequence, in the
   caller's list order, while budget remains (generation never waits behind a
   prompt).
3. Then each prefilling sequence, in list order, takes
   ``min(prompt_len - seen, max_chunk, remaining)`` tokens (no cap when
   ``max_chunk <= 0``).  Under the "equal" policy a prompt longer than that
   allowance ``a`` takes ``ceil(r / ceil(r / a))`` of its ``r`` remaining
   tokens instead (same number of passes, near-equal chunks).
4. The pass lays out the scheduled sequences in list order.
5. Each laid-out sequence receives ``ceil(ctx / B) - held`` new blocks, lowest
   free id first, sequences in layout order.  If the pool is short the call
   fails and changes nothing.  Released blocks return to the pool.
6. A sequence whose ``seen`` differs from the number of tokens the composer has
   recorded for it (0 if unknown) is rejected.
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass, field
from typing import Dict, List, Sequence, Tuple


class InvalidRequest(ValueError):
    """A malformed call (bad budget, bad state, unknown or duplicated id)."""


class NoBlocks(RuntimeError):
    """The block pool cannot cover the pass; nothing was changed."""


@dataclass
class PassMeta:
    """Ragged-batch metadata of one pass (all int, list order of the pass)."""
    seq_ids: List[int] = field(default_factory=list)
    q_start: List[int] = field(default_factory=lambda: [0])
    n_new: List[int] = field(default_factory=list)
    seen: List[int] = field(default_factory=list)
    ctx: List[int] = field(default_factory=list)
    block_start: List[int] = field(default_factory=lambda: [0])
    block_ids: List[int] = field(default_factory=list)
    slot: List[int] = field(default_factory=list)

    @property
    def num_seqs(self) -> int:
        return len(self.seq_ids)

    @property
    def num_tokens(self) -> int:
        return self.q_start[-1]

    def blocks_of(self, s: int) -> List[int]:
        return self.block_ids[self.block_start[s]:self.block_start[s + 1]]


class Composer:
    """Token-budgeted pass composer over a pool of ``num_blocks`` KV blocks."""

    def __init__(self, block_size: int, num_blocks: int):
        if block_size < 1 or num_blocks < 0:
            raise InvalidRequest("block_size must be >= 1 and num_blocks >= 0")
        self.block_size = int(block_size)
        self.num_blocks = int(num_blocks)
        self._free: List[int] = list(range(self.num_blocks))  # a min-heap
        heapq.heapify(self._free)
        self._held: Dict[int, List[int]] = {}
        self._tokens: Dict[int, int] = {}

    # -- queries --------------------------------------------------------------
    def free_blocks(self) -> int:
        return len(self._free)

    def held_blocks(self, seq_id: int) -> List[int]:
        return list(self._held.get(seq_id, []))

    def tokens_of(self, seq_id: int) -> int:
        return self._tokens.get(seq_id, 0)

    # -- the pass -------------------------------------------------------------
    def compose(self, budget: int, max_chunk: int,
                states: Sequence[Tuple[int, int, int]], policy: str = "greedy") -> PassMeta:
        """Compose one pass from ``states`` = [(seq_id, prompt_len, seen), ...].

        ``policy`` "greedy": a prefilling request takes min(remaining prompt,
        max_chunk, remaining budget).  "equal" (paper summary page, idea I2:
        throughput is concave in tokens per pass, so a pool of tokens is best
        spread evenly): a prompt longer than what it is allowed this pass
        (a = min(max_chunk, remaining budget)) is cut into the fewest chunks of
        at most a tokens, all of near-equal size."""
        if policy not in ("greedy", "equal"):
            raise InvalidRequest("unknown chunk policy")
        if budget < 0:
            raise InvalidRequest("token budget must be >= 0")
        ids = [int(s[0]) for s in states]
        if len(set(ids)) != len(ids):
            raise InvalidRequest("a sequence is listed twice")
        for sid, plen, seen in states:
            if plen < 1 or seen < 0:
                raise InvalidRequest(f"sequence {sid}: prompt_len must be >= 1 and seen >= 0")
            if seen != self._tokens.get(int(sid), 0):
                raise InvalidRequest(f"sequence {sid}: seen={seen} but the cache holds "
                                     f"{self._tokens.get(int(sid), 0)} tokens")

        remaining = int(budget)
        take = [0] * len(states)
        # step 2: one generation token per decoding sequence, list order
        for i, (_, plen, seen) in enumerate(states):
            if seen >= plen and remaining > 0:
                take[i] = 1
                remaining -= 1
        # step 3: prompt chunks, list order
        for i, (_, plen, seen) in enumerate(states):
            if seen < plen:
                rem = plen - seen
                allow = remaining if max_chunk <= 0 else min(remaining, max_chunk)
                n = min(rem, allow)
                if policy == "equal" and allow > 0 and rem > allow:
                    k = -(-rem // allow)          # fewest chunks of at most `allow`
                    n = -(-rem // k)              # their (near-)equal size
                take[i] = n
                remaining -= n

        # step 4: layout in list order
        order = [i for i in range(len(states)) if take[i] > 0]

        # step 5: blocks (all-or-nothing)
        B = self.block_size
        need = []
        for i in order:
            sid, _, seen = states[i]
            ctx = seen + take[i]
            have = len(self._held.get(int(sid), []))
            need.append(max(0, -(-ctx // B) - have))
        if sum(need) > len(self._free):
            raise NoBlocks(f"pass needs {sum(need)} new blocks, {len(self._free)} free")

        meta = PassMeta()
        for i, k in zip(order, need):
            sid, _, seen = states[i]
            sid = int(sid)
            held = self._held.setdefault(sid, [])
            for _ in range(k):
                held.append(heapq.heappop(self._free))
            n = take[i]
            ctx = seen + n
            self._tokens[sid] = ctx
            meta.seq_ids.append(sid)
            meta.n_new.append(n)
            meta.seen.append(int(seen))
            meta.ctx.append(ctx)
            meta.q_start.append(meta.q_start[-1] + n)
            blocks = held[: -(-ctx // B)]
            meta.block_ids.extend(blocks)
            meta.block_start.append(meta.block_start[-1] + len(blocks))
            for j in range(n):
                p = seen + j
                meta.slot.append(blocks[p // B] * B + p % B)
        return meta

    def rollback(self, meta: PassMeta) -> None:
        """Undo composing ``meta``: each of its sequences returns to ``seen``
        tokens and gives back the blocks the pass allocated (newest last in its
        list); a sequence that started in this pass is forgotten.  Fails, with
        no change, if a later pass moved any of them."""
        for s in range(meta.num_seqs):
            if self._tokens.get(meta.seq_ids[s]) != meta.ctx[s]:
                raise InvalidRequest(f"sequence {meta.seq_ids[s]} changed after this pass")
        B = self.block_size
        for s in reversed(range(meta.num_seqs)):
            sid, seen = meta.seq_ids[s], meta.seen[s]
            held = self._held.get(sid, [])
            while len(held) > -(-seen // B):
                heapq.heappush(self._free, held.pop())
            if seen == 0:
                self._tokens.pop(sid, None)
                self._held.pop(sid, None)
            else:
                self._tokens[sid] = seen

    def release(self, seq_id: int) -> None:
        """Return every block of ``seq_id`` to the pool and forget it."""
        sid = int(seq_id)
        if sid not in self._tokens and sid not in self._held:
            raise InvalidRequest(f"unknown sequence {sid}")
        for b in self._held.pop(sid, []):
            heapq.heappush(self._free, b)
        self._tokens.pop(sid, None)


def latency_at(tokens: Sequence[int], latency: Sequence[float], t: int) -> float:
    """Predicted latency of t tokens: linear interpolation between the two
    profile points around t (paper summary page, idea I1: latency of a pass
    follows its token count)."""
    i = 0
    while i + 2 < len(tokens) and t > tokens[i + 1]:
        i += 1
    f = float(t - tokens[i]) / float(tokens[i + 1] - tokens[i])
    return latency[i] + (latency[i + 1] - latency[i]) * f


def budget_for_latency(tokens: Sequence[int], latency: Sequence[float], bound: float) -> int:
    """Largest token count in the profile's range whose predicted latency is
    within ``bound`` (FastGen guide, "Prompt-Decode Decoupling": keep each
    iteration under a latency bound); 0 if none; -1 for a bad profile."""
    n = len(tokens)
    if n < 2 or any(tokens[i + 1] <= tokens[i] for i in range(n - 1)) or tokens[0] < 0:
        return -1
    for t in range(tokens[-1], tokens[0] - 1, -1):
        if latency_at(tokens, latency, t) <= bound:
            return t
    return 0
