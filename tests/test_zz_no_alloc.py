"""The entry point that allocates nothing, against the ordinary one.

rbkv_ragged_attention_noalloc serves callers that cannot allocate device
memory where they run attention; it keeps the split-KV scratch in a static
array inside the library.  Its outputs must match rbkv_ragged_attention's
(same kernels, same tolerance as the other parity tests) on two calls in a
row, and a pass that needs more scratch than the array holds is refused.
This file is collected last so that a failure here stops a run only after
every other test has run.
"""
import pytest
import torch

import workloads
from harness import MAX_ABS_TOL, MEAN_ABS_TOL, Pair

pytestmark = pytest.mark.gpu


def _pass_with_splits(rbkv, scn, split_keys):
    pair = Pair(rbkv, scn.shape, scn.num_blocks)
    b, st = scn.registration()
    pair.step(b, 0, st, attend=False)
    p = pair.lib.compose(scn.budget, scn.max_chunk, list(scn.requests))
    if split_keys:
        p.set_split_keys(split_keys)
    T = p.num_tokens
    q, k, v = workloads.make_qkv(scn.shape, T, 0, 1, device="cuda")
    torch.cuda.synchronize()
    rbkv.kv_append(p, k, v, pair.kc, pair.vc)        # uploads the pass's metadata
    return pair, p, q


def _chunk_only():
    """One 128-row prompt chunk behind a 600-token cached prefix, no decodes:
    the tensor-core kernel runs alone (it waits for the append itself) and its
    key range is cut in 128-key pieces that the combine merges."""
    shape = workloads.llama2_7b(0).shape
    return workloads.Scenario("chunk_only", shape, 128, 128, [(2, 600)], [(2, 900, 600)],
                              num_blocks=32)


@pytest.mark.parametrize("case", ["mixed", "chunk_only"])
def test_noalloc_matches_workspace_entry_twice(rbkv, case):
    if case == "mixed":
        scn = workloads.scaled(workloads.llama2_7b(0), 4)    # a prompt chunk + split decodes
    else:
        scn = _chunk_only()
    pair, p, q = _pass_with_splits(rbkv, scn, 128)
    assert p.workspace_bytes() > 0                        # the scratch is used
    plan = p.plan()
    assert plan["chunk_rows"] > 0 and plan["chunk_tiles"] > 0, plan
    if case == "mixed":
        assert plan["decode_items"] > 0, plan
    else:
        assert plan["decode_items"] == 0, plan
    ref = rbkv.ragged_attention(p, q, pair.kc, pair.vc)
    outs = []
    for _ in range(2):
        o = torch.full_like(ref, float("nan"))
        rbkv.ragged_attention_noalloc(p, q, pair.kc, pair.vc, o)
        outs.append(o)
    torch.cuda.synchronize()
    p.device_status()
    for o in outs:
        d = (o.double() - ref.double()).abs()
        assert torch.isfinite(o).all()
        assert d.max().item() <= MAX_ABS_TOL and d.mean().item() <= MEAN_ABS_TOL


def test_noalloc_rejects_passes_beyond_the_static_scratch(rbkv):
    scn = workloads.scaled(workloads.decode_stress(0), 2)
    pair, p, q = _pass_with_splits(rbkv, scn, 64)
    assert p.workspace_bytes() > (16 << 20)
    o = torch.empty((p.num_tokens, scn.shape.num_heads_q, scn.shape.head_dim),
                    dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rbkv.RbkvError) as ei:
        rbkv.ragged_attention_noalloc(p, q, pair.kc, pair.vc, o)
    assert ei.value.status == rbkv.ERR_WORKSPACE
