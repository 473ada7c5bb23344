"""Failure detection on the GPU without a fault: bad metadata is reported and
skipped, a bounded wait that gives up is reported, and the context stays
usable (the next pass is checked against the oracle)."""
import numpy as np
import pytest
import torch

import workloads
from harness import MAX_ABS_TOL, MEAN_ABS_TOL, Pair

pytestmark = pytest.mark.gpu

ERR_DEVICE_BOUNDS = -4
ERR_TIMEOUT = -7


def _setup(rbkv):
    scn = workloads.scaled(workloads.llama2_7b(0), 8)
    pair = Pair(rbkv, scn.shape, scn.num_blocks)
    b, st = scn.registration()
    pair.step(b, 0, st, attend=False)
    return scn, pair


def _next_pass_is_correct(pair, scn):
    r = pair.step(scn.budget, scn.max_chunk, list(scn.requests))
    assert r["meta_equal"] and r["finite"]
    assert r["max_abs"] <= MAX_ABS_TOL and r["mean_abs"] <= MEAN_ABS_TOL
    return r


@pytest.mark.parametrize("which", ["block", "slot"])
def test_out_of_range_ids_are_reported(rbkv, which):
    scn, pair = _setup(rbkv)
    sh = scn.shape
    comp = rbkv.Composer(pair.cfg)               # a second composer: the pair's stays intact
    b, st = scn.registration()
    comp.compose(b, 0, st)
    p = comp.compose(scn.budget, scn.max_chunk, list(scn.requests))
    n = len(p.meta.block_ids) if which == "block" else p.num_tokens
    bad = pair.cfg.num_blocks + 5 if which == "block" else pair.cfg.num_blocks * sh.block_size + 5
    p.debug_corrupt(which, n // 2, bad)
    p.debug_corrupt(which, n - 1, -3)
    T = p.num_tokens
    q, k, v = workloads.make_qkv(sh, T, 0, 77, device="cuda")
    kc, vc = torch.zeros_like(pair.kc), torch.zeros_like(pair.vc)
    rbkv.kv_append(p, k, v, kc, vc)
    rbkv.ragged_attention(p, q, kc, vc)
    with pytest.raises(rbkv.RbkvError) as e:
        p.device_status()
    assert e.value.status == ERR_DEVICE_BOUNDS
    p.device_status()                            # reading cleared it
    _next_pass_is_correct(pair, scn)


def test_bounded_wait_reports_timeout(rbkv):
    scn, pair = _setup(rbkv)
    r = _next_pass_is_correct(pair, scn)
    p = r["pass"]
    p.debug_wait_timeout(2_000_000)              # about a millisecond
    with pytest.raises(rbkv.RbkvError) as e:
        p.device_status()
    assert e.value.status == ERR_TIMEOUT
    assert "site 99" in str(e.value)
    p.device_status()
    # the context and the library still work
    n = dict(zip(r["meta"].seq_ids, r["meta"].n_new))
    states = [(sid, pl, seen + n.get(sid, 0)) for sid, pl, seen in scn.requests]
    r2 = pair.step(scn.budget, scn.max_chunk, states)
    assert r2["meta_equal"] and r2["max_abs"] <= MAX_ABS_TOL
    assert pair.cache_equal()


def test_debug_calls_reject_misuse(rbkv):
    scn, pair = _setup(rbkv)
    r = _next_pass_is_correct(pair, scn)
    with pytest.raises(rbkv.RbkvError):
        r["pass"].debug_corrupt("block", 0, 1)       # already on the device
    comp = rbkv.Composer(pair.cfg)
    p = comp.compose(4, 0, [(1, 4, 0)])
    with pytest.raises(rbkv.RbkvError):
        p.debug_wait_timeout(1000)                   # not on the device yet
