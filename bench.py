#!/usr/bin/env python
"""Benchmark of the ragged SplitFuse attention pass (one pass per step).

Workload (default): the Llama-2-7B attention shape - 32 query heads, 32 KV
heads, head_dim 128, bf16, KV block 64, token budget 512, chunk cap 512.  A
4096-token prompt is carried through 9 passes (8 chunks of 497 tokens and one
of 120) next to 15 decode sequences whose contexts start at round(N(2600,
780^2)) clipped to [64, 8192] and grow by one token per pass; when a prompt
completes it is released and a fresh one starts, so every pass mixes a prompt
chunk with the decodes.  A step is one whole pass of the hot path: host
composition and block allocation, the metadata upload, kv_append and ragged
attention (tensor-core chunk tiles, split-KV decode, log-sum-exp combine).

Output: one JSON line (rank 0).  ``value`` is pass tokens per second with
inputs already resident in HBM; ``e2e`` is the same through the same calls with
Q/K/V copied from pinned host memory and O copied back inside the timed
region.  ``--impl reference`` times the fp64 CPU oracle instead.

Several GPUs (torchrun) run independent replicas of the workload, one per
rank: the path has no exchange step, so there is no collective.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=18)
    ap.add_argument("--warmup", type=int, default=9)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama2_7b",
                    choices=["llama2_7b", "decode_stress", "mistral_7b"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


# ---------------------------------------------------------------------------
# pass stream: the workload's passes, one after another
# ---------------------------------------------------------------------------
class PassStream:
    """Yields the states of successive passes of a scenario.

    llama2_7b: the prompt is re-issued under a new id once it completes.
    decode_stress / mistral_7b: the same pass shape every step (decodes grow
    by one token; prompt chunks restart at their first chunk under new ids).
    """

    def __init__(self, scn):
        self.scn = scn
        self.states = list(scn.requests)
        self.next_id = 10_000_000
        self.initial = {s: (pl, seen) for s, pl, seen in scn.requests}

    def advance(self, seq_ids, n_new, release):
        n = dict(zip([int(x) for x in seq_ids], [int(x) for x in n_new]))
        out = []
        for sid, pl, seen in self.states:
            seen2 = seen + n.get(sid, 0)
            prefilling = seen < pl
            if prefilling and (seen2 >= pl or self.scn.name != "llama2_7b"):
                # prompt done (or, for single-pass shapes, chunk done): a fresh
                # request of the same shape replaces it
                release(sid)
                pl0, seen0 = self.initial.get(sid, (pl, 0))
                if seen0 > 0:
                    # a prompt with a cached prefix: keep the prefix sequence
                    # itself and restart from its prefix is not possible, so a
                    # new id is registered with the prefix by the caller
                    out.append(("reprefix", sid, pl0, seen0))
                else:
                    nid = self.next_id
                    self.next_id += 1
                    self.initial[nid] = (pl0, 0)
                    out.append((nid, pl0, 0))
                continue
            out.append((sid, pl, seen2))
        self.states = out


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    hbm, bf16, bf16_sus, src = HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, BF16_FALLBACK_TFLOPS, "fallback"
    try:
        with open(path) as f:
            d = json.load(f)
        flat = {}

        def walk(x, pre=""):
            if isinstance(x, dict):
                for k, v in x.items():
                    walk(v, pre + k.lower() + ".")
            elif isinstance(x, (int, float)):
                flat[pre[:-1]] = float(x)
        walk(d)
        h = [v for k, v in flat.items() if "hbm" in k and "gbs" in k]
        b = [v for k, v in flat.items() if "bf16" in k and "tflops" in k and "sustained" not in k]
        bs = [v for k, v in flat.items() if "bf16" in k and "tflops" in k and "sustained" in k]
        if h:
            hbm, src = h[0], "measured"
        if b:
            bf16 = b[0]
        if bs:
            bf16_sus = bs[0]
    except Exception:
        pass
    return hbm, bf16, bf16_sus, src


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def step_work(meta, shape):
    """Algorithmic work of one pass from its metadata."""
    e = 2 if shape.dtype == "bf16" else 4
    H_q, H_kv, D = shape.num_heads_q, shape.num_heads_kv, shape.head_dim
    dec_kv = dec_rows = 0
    chunk_flops = 0
    chunk_kv = 0
    all_kv = 0
    for s in range(len(meta.seq_ids)):
        n, c = int(meta.n_new[s]), int(meta.ctx[s])
        all_kv += c * H_kv * D * 2 * e
        if n == 1:
            dec_kv += c * H_kv * D * 2 * e
            dec_rows += 1
        else:
            seen = int(meta.seen[s])
            # row j (position seen + j) attends seen + j + 1 keys
            keys = n * seen + n * (n + 1) // 2
            chunk_flops += keys * H_q * D * 4
            chunk_kv += c * H_kv * D * 2 * e
    T = int(meta.q_start[-1])
    return {
        "tokens": T,
        "kv_read_bytes": all_kv,
        "decode_bytes": dec_kv + dec_rows * H_q * D * e * 2,
        "chunk_flops": chunk_flops,
        "append_bytes": 2 * T * H_kv * D * e * 2,
        "pass_bytes": all_kv + 2 * T * H_q * D * e + 2 * T * H_kv * D * e,
    }


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class GpuRunner:
    def __init__(self, rbkv, scn, seed, device):
        import torch
        import workloads
        self.torch = torch
        self.rbkv = rbkv
        self.scn = scn
        self.shape = scn.shape
        sh = scn.shape
        self.cfg = rbkv.Config(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size,
                               sh.dtype, scn.num_blocks)
        self.comp = rbkv.Composer(self.cfg)
        dt = self.cfg.torch_dtype
        self.kc = torch.zeros(self.cfg.cache_shape(), dtype=dt, device=device)
        self.vc = torch.zeros(self.cfg.cache_shape(), dtype=dt, device=device)
        self.device = device
        self.seed = seed
        self.stream = torch.cuda.current_stream()
        b, st = scn.registration()
        if b:
            p = self.comp.compose(b, 0, st)
            k, v = workloads.make_qkv(sh, p.num_tokens, seed, 0, device=device, which="kv")
            rbkv.kv_append(p, k, v, self.kc, self.vc)
            del k, v
        self.ps = PassStream(scn)
        self.max_T = scn.budget
        self.ws = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        self.o = torch.empty((self.max_T, sh.num_heads_q, sh.head_dim), dtype=dt, device=device)
        torch.cuda.synchronize()

    def make_inputs(self, n, base_index):
        import workloads
        sets = []
        for i in range(n):
            sets.append(workloads.make_qkv(self.shape, self.max_T, self.seed, base_index + i,
                                           device=self.device))
        return sets

    def _resolve_states(self):
        # a prompt with a cached prefix is re-registered under a new id
        states = []
        for st in self.ps.states:
            if st[0] == "reprefix":
                _, old, pl, seen0 = st
                nid = self.ps.next_id
                self.ps.next_id += 1
                p = self.comp.compose(seen0, 0, [(nid, seen0, 0)])
                import workloads
                k, v = workloads.make_qkv(self.shape, seen0, self.seed, 1, device=self.device,
                                          which="kv")
                self.rbkv.kv_append(p, k, v, self.kc, self.vc, stream=self.stream)
                self.ps.initial[nid] = (pl, seen0)
                states.append((nid, pl, seen0))
            else:
                states.append(st)
        self.ps.states = states
        return states

    def step(self, inputs, work_acc=None, host=None):
        """One pass.  ``inputs`` = (q, k, v) device tensors of max_T rows, or
        with ``host`` = (q_h, k_h, v_h, o_h) pinned tensors copied in and out."""
        rbkv = self.rbkv
        states = self._resolve_states()
        p = self.comp.compose(self.scn.budget, self.scn.max_chunk, states)
        T = p.num_tokens
        q, k, v = inputs
        if host is not None:
            q_h, k_h, v_h, o_h = host
            q[:T].copy_(q_h[:T], non_blocking=True)
            k[:T].copy_(k_h[:T], non_blocking=True)
            v[:T].copy_(v_h[:T], non_blocking=True)
        rbkv.kv_append(p, k[:T], v[:T], self.kc, self.vc, stream=self.stream)
        need = p.workspace_bytes()
        if need > self.ws.numel():
            raise RuntimeError(f"workspace {need} > {self.ws.numel()}")
        rbkv.ragged_attention(p, q[:T], self.kc, self.vc, o=self.o[:T], workspace=self.ws,
                              stream=self.stream)
        if host is not None:
            o_h[:T].copy_(self.o[:T], non_blocking=True)
        if work_acc is not None:
            w = step_work(p.meta, self.shape)
            for kk, vv in w.items():
                work_acc[kk] = work_acc.get(kk, 0) + vv
        self.ps.advance(p.meta.seq_ids, p.meta.n_new, self.comp.release)
        return T


def run_ours(args, rank, world, local_rank):
    import torch
    import workloads
    from ragged_blocked_kv_gb300 import build as _build
    if rank == 0:
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    import ragged_blocked_kv_gb300 as rbkv
    rbkv.lib()

    device = f"cuda:{local_rank}"
    torch.cuda.set_device(local_rank)
    scn = workloads.SCENARIOS[args.workload](args.seed)
    run = GpuRunner(rbkv, scn, args.seed, device)
    W, K = args.warmup, args.steps
    inputs = run.make_inputs(W + K, 100)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for i in range(W):
        run.step(inputs[i])
    torch.cuda.synchronize()

    # ---- timed region: K passes, inputs resident in HBM -----------------
    rbkv.profile_reset()
    rbkv.profile_enable(True)
    clocks = ClockSampler(local_rank)
    work = {}
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = rbkv.kernel_launches()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    t_start.record(run.stream)
    tokens = 0
    for i in range(K):
        tokens += run.step(inputs[W + i], work)
    t_end.record(run.stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier()
    launches = rbkv.kernel_launches() - launches0
    clk = clocks.stop()
    rbkv.profile_enable(False)
    prof = rbkv.profile_read()
    ms = t_start.elapsed_time(t_end)

    # ---- e2e: same passes through the same calls, host buffers ----------
    del inputs
    dev_bufs = run.make_inputs(1, 5000)[0]
    host_sets = []
    for i in range(min(K, 6)):
        q, k, v = run.make_inputs(1, 6000 + i)[0]
        host_sets.append((q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory(),
                          torch.empty(run.o.shape, dtype=run.o.dtype).pin_memory()))
    for i in range(2):
        run.step(dev_bufs, host=host_sets[i % len(host_sets)])
    torch.cuda.synchronize()
    e2e_work = {}
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(run.stream)
    e2e_tokens = 0
    for i in range(K):
        e2e_tokens += run.step(dev_bufs, e2e_work, host=host_sets[i % len(host_sets)])
    e1.record(run.stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    sh = scn.shape
    esz = 2 if sh.dtype == "bf16" else 4
    h2d = e2e_work["tokens"] * (sh.num_heads_q + 2 * sh.num_heads_kv) * sh.head_dim * esz / K
    d2h = e2e_work["tokens"] * sh.num_heads_q * sh.head_dim * esz / K

    # ---- max over ranks --------------------------------------------------
    t = torch.tensor([ms, e2e_ms, float(tokens), float(e2e_tokens)], dtype=torch.float64,
                     device=device)
    if world > 1:
        mx = t.clone()
        torch.distributed.all_reduce(mx[:2], op=torch.distributed.ReduceOp.MAX)
        sm = t.clone()
        torch.distributed.all_reduce(sm[2:], op=torch.distributed.ReduceOp.SUM)
        ms, e2e_ms = float(mx[0]), float(mx[1])
        tot_tokens, tot_e2e = float(sm[2]), float(sm[3])
    else:
        tot_tokens, tot_e2e = float(tokens), float(e2e_tokens)
    if rank != 0:
        return

    hbm, bf16, bf16_sus, src = read_peaks()
    # dominant kernel by device time
    kinds = {k: v for k, v in prof.items() if v[1] > 0}
    dom = max(kinds, key=lambda k: kinds[k][0])
    dom_ms, dom_n = kinds[dom]
    avg_s = dom_ms / dom_n / 1e3
    if dom in ("chunk",):
        per_launch = work["chunk_flops"] / dom_n
        achieved = per_launch / avg_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16_sus, "unit": "TFLOP/s"}
    else:
        key = {"decode": "decode_bytes", "generic": "kv_read_bytes",
               "kv_append": "append_bytes", "combine": "decode_bytes"}[dom]
        per_launch = work[key] / dom_n
        achieved = per_launch / avg_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = None
    roof["kernel"] = dom
    roof["peak_source"] = src
    roof["avg_launch_us"] = avg_s * 1e6

    line = {
        "metric": "ragged SplitFuse attention pass tokens/s",
        "value": tot_tokens / (ms / 1e3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": sh.dtype,
        "data": "synthetic",
        "config": {
            "workload": f"{scn.name}: {sh.num_heads_q}q/{sh.num_heads_kv}kv heads, head_dim "
                        f"{sh.head_dim}, block {sh.block_size}, budget {scn.budget}, chunk cap "
                        f"{scn.max_chunk}",
            "tokens_per_step": tot_tokens / K / world,
            "kv_read_gb_per_step": work["kv_read_bytes"] / K / 1e9,
            "kv_read_gbs": work["kv_read_bytes"] / (ms / 1e3) / 1e9,
            "kv_read_frac_of_hbm": work["kv_read_bytes"] / (ms / 1e3) / 1e9 / hbm,
            "l2": "inputs larger than L2 (each pass reads "
                  f"{work['kv_read_bytes'] / K / 1e6:.0f} MB of KV > 129 MB L2); no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "kernel_ms": {k: round(v[0], 4) for k, v in kinds.items()},
            "kernel_launches": {k: v[1] for k, v in kinds.items()},
            "host_wall_ms": wall * 1e3,
        },
        "roofline": roof,
        "e2e": {"value": tot_e2e / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_subprocess(args)
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the oracle on the host cores (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
class OracleRunner:
    """The fp64 oracle driven through the same pass stream.

    A step is one pass: oracle composition and appending of the whole pass,
    and oracle attention for a sample of its rows - every decode row and every
    32nd prompt-chunk row - so that one step costs about a second.  Tokens
    counted are the rows whose outputs were computed."""

    def __init__(self, scn, seed):
        import numpy as np
        import oracle
        import workloads
        self.np = np
        self.oracle = oracle
        self.workloads = workloads
        self.scn = scn
        sh = scn.shape
        self.shape = sh
        self.seed = seed
        self.comp = oracle.Composer(sh.block_size, scn.num_blocks)
        storage = np.uint16 if sh.dtype == "bf16" else np.float32
        self.kc = oracle.BlockedCache(sh.num_heads_kv, sh.block_size, sh.head_dim, storage)
        self.vc = oracle.BlockedCache(sh.num_heads_kv, sh.block_size, sh.head_dim, storage)
        b, st = scn.registration()
        if b:
            m = self.comp.compose(b, 0, st)
            k, v = workloads.make_qkv(sh, m.num_tokens, seed, 0, which="kv")
            oracle.kv_append(m, self._st(k), self._st(v), self.kc, self.vc)
        self.ps = PassStream(scn)
        self.q, self.k, self.v = workloads.make_qkv(sh, scn.budget, seed, 100)

    def _st(self, t):
        import torch
        t = t.contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(self.np.uint16)
        return t.numpy()

    def _resolve(self):
        states = []
        for st in self.ps.states:
            if st[0] == "reprefix":
                _, old, pl, seen0 = st
                nid = self.ps.next_id
                self.ps.next_id += 1
                m = self.comp.compose(seen0, 0, [(nid, seen0, 0)])
                k, v = self.workloads.make_qkv(self.shape, seen0, self.seed, 1, which="kv")
                self.oracle.kv_append(m, self._st(k), self._st(v), self.kc, self.vc)
                self.ps.initial[nid] = (pl, seen0)
                states.append((nid, pl, seen0))
            else:
                states.append(st)
        self.ps.states = states
        return states

    def step(self):
        states = self._resolve()
        m = self.comp.compose(self.scn.budget, self.scn.max_chunk, states)
        T = m.num_tokens
        k, v, q = self._st(self.k[:T]), self._st(self.v[:T]), self._st(self.q[:T])
        self.oracle.kv_append(m, k, v, self.kc, self.vc)
        rows = []
        for s in range(m.num_seqs):
            a, n = m.q_start[s], m.n_new[s]
            rows.extend(range(a, a + n) if n == 1 else range(a, a + n, 32))
        self.oracle.blocked_attention(m, q, self.kc, self.vc, self.shape.num_heads_q, tokens=rows)
        self.ps.advance(m.seq_ids, m.n_new, self.comp.release)
        return len(rows)


def oracle_measure(workload, seed, steps, warmup):
    import workloads
    scn = workloads.SCENARIOS[workload](seed)
    t0 = time.perf_counter()
    r = OracleRunner(scn, seed)
    setup = time.perf_counter() - t0
    for _ in range(warmup):
        r.step()
    t0 = time.perf_counter()
    rows = 0
    for _ in range(steps):
        rows += r.step()
    dt = time.perf_counter() - t0
    return {"value": rows / dt, "rows": rows, "seconds": dt, "setup_seconds": setup}


def cpu_env():
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    return env


def cpu_baseline_subprocess(args, steps=5, warmup=1):
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", "--workload", args.workload,
           "--seed", str(args.seed), "--steps", str(steps), "--warmup", str(warmup)]
    try:
        out = subprocess.run(cmd, capture_output=True, text=True, env=cpu_env(), timeout=600)
        res = json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal
        return {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "sample": f"failed: {e}"}
    return {"value": res["value"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{steps} passes after {warmup} warm-up; per pass the oracle composes and "
                      "appends the whole pass and computes attention for every decode row and "
                      f"every 32nd prompt-chunk row ({res['rows']} rows in {res['seconds']:.1f} s); "
                      "value = rows / s; one thread (BLAS threads = 1)"}


def run_reference(args, rank):
    if rank != 0:
        return
    import workloads
    res = oracle_measure(args.workload, args.seed, args.steps, args.warmup)
    scn = workloads.SCENARIOS[args.workload](args.seed)
    sh = scn.shape
    v = res["value"]
    line = {
        "impl": "reference",
        "metric": "ragged SplitFuse attention pass tokens/s",
        "value": v,
        "unit": "tokens/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": res["seconds"] / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{scn.name}: {sh.num_heads_q}q/{sh.num_heads_kv}kv heads, head_dim "
                               f"{sh.head_dim}, block {sh.block_size}, budget {scn.budget}, chunk "
                               f"cap {scn.max_chunk}"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "per pass: whole-pass composition and append, attention for "
                                   "every decode row and every 32nd prompt-chunk row; value = "
                                   "rows / s; one thread"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.cpu_worker:
        res = oracle_measure(args.workload, args.seed, args.steps, args.warmup)
        print(json.dumps(res), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            # the oracle needs no GPU; run it with BLAS threads pinned to one
            for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
                os.environ.setdefault(v, "1")
            run_reference(args, rank)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
