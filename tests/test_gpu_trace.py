"""The full closed-loop trace through the library, sampled against the oracle.

The trace workload at full size (paper summary page, Key points: 512 requests
from 32 clients, prompt lengths N(2600, 30%), outputs N(60, 30%)): requests
are prefilled in 512-token passes with decodes, finish, are released, and
their clients send the next ones, over about 2,700 passes.  Each pass appends
K/V into 32 layer caches that share one block table (Llama-2-7B attention
shape), as a serving loop does.

Checked: the metadata of every pass bit-exact against the oracle composer;
every 64 passes - on the first pass from every 64th on that holds a request
of four sampled clients (prefilling or decoding; a prefilling request can get
no tokens in a full pass, and near the end of the trace those clients may be
done) - the attention outputs of those requests and their cached rows, for
layers 0 and 31, against the oracle; at the end, every block back in the pool
and the token count of the trace conserved.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import FIELDS, MAX_ABS_TOL, MEAN_ABS_TOL, to_f64, to_storage

pytestmark = pytest.mark.gpu

LAYERS = 32
CHECKED_LAYERS = (0, 31)
CHECK_EVERY = 64
SAMPLED_CLIENTS = (0, 9, 17, 26)
ROWS_PER_CHUNK = 8        # sampled rows of a prefilling request's chunk (all heads)


def test_full_trace_sampled(rbkv):
    seed = 0
    reqs = workloads.trace_requests(seed=seed)
    clients = 32
    shape = workloads.Shape(32, 32, 128, 64, "bf16", 1.0 / math.sqrt(128.0))
    nb = workloads.trace_block_pool(reqs, clients, 64)
    cfg = rbkv.Config(32, 32, 128, 64, "bf16", nb)
    comp = rbkv.Composer(cfg)
    orc = oracle.Composer(64, nb)
    caches = [(torch.zeros(cfg.cache_shape(), dtype=torch.bfloat16, device="cuda"),
               torch.zeros(cfg.cache_shape(), dtype=torch.bfloat16, device="cuda"))
              for _ in range(LAYERS)]
    ocaches = {l: (oracle.BlockedCache(32, 64, 128, np.uint16),
                   oracle.BlockedCache(32, 64, 128, np.uint16)) for l in CHECKED_LAYERS}
    sampled = {r.seq_id for r in reqs if r.client in SAMPLED_CLIENTS}
    # layers that are not checked append the same seeded rows every pass
    filler = workloads.make_qkv(shape, 512, seed, 99_999, device="cuda", which="kv")
    ws = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(seed)
    stats = {"passes": 0, "checked": 0, "outputs": 0, "max_abs": 0.0, "sum_abs": 0.0,
             "tokens": 0, "next_check": 0}

    def compose(budget, max_chunk, states):
        i = stats["passes"]
        stats["passes"] += 1
        p = comp.compose(budget, max_chunk, states)
        m = orc.compose(budget, max_chunk, states)
        for f in FIELDS:
            assert np.array_equal(np.asarray(getattr(p.meta, f), np.int64),
                                  np.asarray(getattr(m, f), np.int64)), (i, f)
        T = m.num_tokens
        stats["tokens"] += T
        if T == 0:
            return m
        # pass rows of the sampled requests (their whole history is in the
        # oracle's caches), and the rows whose outputs are checked
        rows, out_rows = [], []
        for s in range(m.num_seqs):
            if m.seq_ids[s] not in sampled:
                continue
            r = list(range(m.q_start[s], m.q_start[s + 1]))
            rows.extend(r)
            if len(r) > ROWS_PER_CHUNK:
                pick = {r[0], r[-1]} | set(int(x) for x in rng.choice(r, ROWS_PER_CHUNK - 2,
                                                                        replace=False))
                out_rows.extend(sorted(pick))
            else:
                out_rows.extend(r)
        check = bool(out_rows) and i >= stats["next_check"]
        if check:
            stats["next_check"] = (i // CHECK_EVERY + 1) * CHECK_EVERY
        ridx = torch.as_tensor(rows, dtype=torch.int64, device="cuda")
        for l in range(LAYERS):
            kc, vc = caches[l]
            if l in CHECKED_LAYERS:
                k, v = workloads.make_qkv(shape, T, seed, 2 * i + (l > 0), device="cuda",
                                          which="kv")
            else:
                k, v = filler[0][:T], filler[1][:T]
            rbkv.kv_append(p, k, v, kc, vc)
            if l in CHECKED_LAYERS and rows:
                ok_, ov_ = ocaches[l]
                kk = np.zeros((T, 32, 128), np.uint16)
                vv = np.zeros((T, 32, 128), np.uint16)
                kk[rows] = to_storage(k.index_select(0, ridx))
                vv[rows] = to_storage(v.index_select(0, ridx))
                oracle.kv_append(m, kk, vv, ok_, ov_, only_seqs=sampled)
            if check and l in CHECKED_LAYERS:
                (q,) = workloads.make_qkv(shape, T, seed, 1_000_000 + 2 * i + (l > 0),
                                          device="cuda", which="q")
                o = rbkv.ragged_attention(p, q, kc, vc, workspace=ws)
                torch.cuda.synchronize()
                p.device_status()
                oidx = torch.as_tensor(out_rows, dtype=torch.int64, device="cuda")
                qs = np.zeros((T, 32, 128), np.uint16)
                qs[out_rows] = to_storage(q.index_select(0, oidx))
                ok_, ov_ = ocaches[l]
                want = oracle.blocked_attention(m, qs, ok_, ov_, 32, tokens=out_rows)
                got = to_f64(o)
                d = np.stack([np.abs(got[t, h] - w) for (t, h), w in want.items()])
                assert np.isfinite(got[out_rows]).all()
                stats["max_abs"] = max(stats["max_abs"], float(d.max()))
                stats["sum_abs"] += float(d.sum())
                stats["outputs"] += d.size
                # the sampled sequences' cached rows, bit for bit (a
                # reused block's slots past a sequence's context keep
                # whatever its previous owner left: not compared)
                for s in range(m.num_seqs):
                    if m.seq_ids[s] not in sampled:
                        continue
                    table = m.blocks_of(s)
                    pos = np.arange(m.ctx[s])
                    blk = torch.as_tensor(np.asarray(table)[pos // 64], device="cuda")
                    off = torch.as_tensor(pos % 64, device="cuda")
                    for cache, ocache in ((kc, ok_), (vc, ov_)):
                        rows_dev = to_storage(cache[blk, :, off, :])     # [ctx][H][D]
                        ob = np.stack([ocache.block(b) for b in table])  # [nb][H][B][D]
                        rows_orc = ob[pos // 64, :, pos % 64, :]         # [ctx][H][D]
                        assert np.array_equal(rows_dev, rows_orc), (i, l, s)
                stats["checked"] += 1
        return m

    def release(sid):
        comp.release(sid)
        orc.release(sid)

    n = workloads.run_trace(reqs, clients, 512, 512, compose, release)
    torch.cuda.synchronize()
    assert n == stats["passes"] and n > 2000
    # conservation: every prompt token once, and output_len - 1 decode tokens
    assert stats["tokens"] == sum(r.prompt_len + r.output_len - 1 for r in reqs)
    assert comp.free_blocks() == nb
    windows = -(-n // CHECK_EVERY)
    assert stats["checked"] >= 2 * int(0.9 * windows), stats
    assert stats["max_abs"] <= MAX_ABS_TOL, stats
    assert stats["sum_abs"] / stats["outputs"] <= MEAN_ABS_TOL, stats
