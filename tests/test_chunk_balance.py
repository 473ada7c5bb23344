"""Placement of tensor-core chunk work items over the persistent chunk grid
(CPU only: the split planner runs on the host).

The plan reports the chunk work in key-tile steps and the most of it that one
CTA walks.  The placement can do no better than the lower bounds
max(ceil(total / CTAs), the largest item) and is checked to come within one
item of the first of them; on passes whose items come in a few sizes (chunks of
equal length behind equal prefixes) it must reach the lower bound within one
step.
"""
import math

import numpy as np
import pytest

import ragged_blocked_kv_gb300 as rbkv


def _pass(hq, hkv, prompts, seed=0):
    """prompts: list of (prefix, chunk rows); the prefixes are cached first."""
    nb = sum(-(-(pre + rows) // 64) for pre, rows in prompts) + 8
    comp = rbkv.Composer(rbkv.Config(hq, hkv, 128, 64, "bf16", nb))
    hist = [(10 + i, pre) for i, (pre, _) in enumerate(prompts) if pre > 0]
    if hist:
        comp.compose(sum(n for _, n in hist), 0, [(s, n, 0) for s, n in hist])
    reqs = [(10 + i, pre + rows, pre) for i, (pre, rows) in enumerate(prompts)]
    return comp.compose(sum(r for _, r in prompts), 0, reqs)


def _item_cost_bound(hq, hkv, prompts):
    """Largest item: both query tiles of a pair over the longest key range."""
    longest = max(pre + rows for pre, rows in prompts)
    return 2 * math.ceil(longest / 128) + 1


@pytest.mark.parametrize("sms", [152, 148, 100, 37])
def test_equal_prompts_reach_the_bound(sms):
    # 16 prompts, each a 768-row chunk behind 1536 cached keys, 32/8 heads
    p = _pass(32, 8, [(1536, 768)] * 16)
    info = p.plan_for_sms(sms)
    assert info["chunk_items"] == 16 * 6 * 16 and info["chunk_single"] == 0
    ctas = min(sms, info["chunk_items"])
    lower = math.ceil(info["chunk_steps_total"] / ctas)
    assert lower <= info["chunk_steps_max"] <= lower + 1


@pytest.mark.parametrize("seed", range(6))
def test_mixed_prompts_within_one_item(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(6, 24))
    prompts = [(int(rng.integers(0, 6000)), int(rng.integers(129, 1600))) for _ in range(n)]
    p = _pass(32, 8, prompts)
    for sms in (152, 64):
        info = p.plan_for_sms(sms)
        if info["chunk_single"]:
            continue
        ctas = min(sms, info["chunk_items"])
        lower = max(math.ceil(info["chunk_steps_total"] / ctas), 1)
        assert info["chunk_steps_max"] >= lower
        assert info["chunk_steps_max"] <= lower + _item_cost_bound(32, 8, prompts)


def test_fewer_items_than_ctas_is_the_largest_item():
    # 2 prompts of 200 rows behind 300 keys, 8 heads of 8: fewer items than SMs
    p = _pass(8, 8, [(300, 200), (300, 200)])
    info = p.plan_for_sms(152)
    assert 0 < info["chunk_items"] < 152
    # an item: one or two query tiles over at most 500 keys (4 key tiles each)
    assert 1 < info["chunk_steps_max"] <= 2 * 4 + 1
