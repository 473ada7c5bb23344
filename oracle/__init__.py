"""fp64 CPU oracle for the Dynamic SplitFuse ragged attention pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
(``ragged_blocked_kv_gb300``) never imports it, and it imports nothing from the
library: the two share only the seeded input generators in ``workloads``.

What it computes, plainly and slowly:

* ``composer``   - Dynamic SplitFuse pass composition: every forward pass holds
  a fixed token budget; long prompts are cut into chunks over several passes;
  generation tokens and short prompts top the pass up ("DeepSpeed-FastGen"
  paper summary page, Summary and idea I3; InfoQ release note, second
  paragraph).  Fixed-size KV blocks are assigned from a free pool.
* ``cache``      - the blocked (paged) KV cache and the append step: each new
  K/V row is copied into slot ``p mod B`` of block ``table[p // B]``
  (FastGen guide, "Paged KV Memory Management"; summary page, Key points).
* ``attention``  - exact causal softmax attention of every pass token over its
  sequence's cached keys, read through the block table, in fp64 (FastGen guide,
  Step 3 dense path and Step 4 ground truth: scores scaled by 1/sqrt(d),
  softmax, weighted sum of values).  The split-KV + log-sum-exp combine that the
  method uses to reach the same numbers faster is written out separately
  (``split_attention`` / ``lse_combine``) so that its equivalence can be
  checked; the oracle's own outputs never go through it.

* ``router``     - routing requests over independent replicas: the replica
  with the fewest outstanding tokens takes the next request (InfoQ release
  note: replicas behind a load balancer; the policy is this repository's
  reading), loads recomputed from the held requests at every decision.

Pins (tests marked ``not gpu``): the tiny configuration's worked pass, budget
and conservation invariants, brute force on tiny inputs, closed forms,
PyTorch's scaled-dot-product attention as an independent library special case,
split invariance and chunk invariance.  Block ids follow a stated rule (lowest
free id first, in layout order) that the pages do not fix: for the choice of
block ids, parity unpinned (only that rule and the pool invariants - distinct
ids, ceil(ctx / B) held per sequence, all-or-nothing - hold them).
"""
from .composer import Composer, PassMeta, InvalidRequest, NoBlocks, budget_for_latency, latency_at  # noqa: F401
from . import router  # noqa: F401
from .cache import BlockedCache, kv_append  # noqa: F401
from .attention import (  # noqa: F401
    widen,
    blocked_attention,
    blocked_attention_array,
    dense_causal_attention,
    split_attention,
    lse_combine,
)
