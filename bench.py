#!/usr/bin/env python
"""Benchmark of the ragged SplitFuse attention pass (one pass per step).

Workload (default, ``--workload mistral_7b``): the Mistral-7B attention
shape - 32 query heads, 8 KV heads, head_dim 128, bf16, KV block 64, token
budget 2048, chunk cap 768.  Each pass holds two 768-token prompt chunks (one
at the start of a 2304-token prompt, one behind a 1536-token cached prefix)
and 512 decode tokens whose contexts are uniform in [128, 8192]: about 9 GB of
KV read per pass, the largest pass of the workloads.  After each pass it is
rolled back on the composer, so every step is the same pass.  A step is one
whole pass of the hot path: host composition and block allocation, the
metadata upload, kv_append and ragged attention (tensor-core chunk tiles,
split-KV decode, log-sum-exp combine).

``--workload llama2_7b``: 32/32 heads, budget 512, chunk cap 512; a 4096-token
prompt is carried through 9 passes (8 chunks of 497 tokens and one of 120)
next to 15 decode sequences (contexts round(N(2600, 780^2)) clipped to [64,
8192], one more token per pass); the 9 passes form a cycle that is rolled back
and repeated.  ``--workload decode_stress``: 64/8 heads, 64 decodes with
contexts log-uniform in [512, 16000].  ``--workload prefill_mistral``: a
chunk-dominated pass, 16 prompts each taking a 768-token chunk behind 1536
cached tokens at the Mistral-7B shape (tensor-core bound).

Output: one JSON line (rank 0).  ``value`` is pass tokens per second with
inputs already resident in HBM; ``e2e`` is the same through the same calls with
Q/K/V copied from pinned host memory and O copied back inside the timed
region (pipelined: the next pass's inputs go in on a copy stream while a pass
computes, its O comes back on another).  ``--impl reference`` times the fp64 CPU oracle instead.

Several GPUs (torchrun) run independent replicas of the workload, one per
rank: the path has no exchange step, so there is no collective.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import resource
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HBM_FALLBACK_GBS = 6800.0
# DRAM bytes (read + write) per launch of a kernel, from the ncu captures
# summarised under profiles/, keyed by (workload, kernel) and valid only for
# the kernel source they were taken on (sha256 prefix of its .cu file)
TRAFFIC_BYTES = {
    ("mistral_7b", "decode"): ("rbkv_decode.cu", "b394238259fb", 9_182_830_000),
    ("llama2_7b", "decode"): ("rbkv_decode.cu", "b394238259fb", 614_143_744),
    ("decode_stress", "decode"): ("rbkv_decode.cu", "b394238259fb", 1_182_816_768),
    ("prefill_mistral", "chunk"): ("rbkv_chunk.cu", "a1a66ed0886e", 770_232_832),
}
BF16_FALLBACK_TFLOPS = 1900.0
BF16_SUSTAINED_FALLBACK_TFLOPS = 1700.0   # the same GEMM held for seconds under the power cap
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3600)
    ap.add_argument("--warmup", type=int, default=90)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mistral_7b",
                    choices=["llama2_7b", "decode_stress", "mistral_7b", "prefill_mistral", "trace",
                             "profile"])
    ap.add_argument("--layers", type=int, default=32,
                    help="layers per pass (trace and profile workloads)")
    ap.add_argument("--layer", choices=["attention", "full"], default="attention",
                    help="per layer: the library's append + attention, or a whole "
                         "random-weight decoder layer (trace and profile workloads)")
    ap.add_argument("--policy", choices=["greedy", "equal"], default="greedy",
                    help="prompt chunk policy (trace workload)")
    ap.add_argument("--budget", type=int, default=512,
                    help="tokens per pass (trace workload); 0 = from the latency profile")
    ap.add_argument("--latency-bound", type=float, default=30.0,
                    help="pass latency bound in ms for --budget 0 and the profile workload")
    ap.add_argument("--eager", dest="graph", action="store_false",
                    help="launch every pass eagerly instead of replaying a CUDA graph "
                         "(trace and profile workloads)")
    ap.add_argument("--ttft-sla", type=float, default=1000.0, help="TTFT bound, ms")
    ap.add_argument("--pace-sla", type=float, default=25.0,
                    help="bound on a request's mean interval between tokens, ms")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-offset", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-core", type=int, default=-1, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-barrier", default="", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-world", type=int, default=1, help=argparse.SUPPRESS)
    return ap.parse_args()


# ---------------------------------------------------------------------------
# the workload's cycle of passes
# ---------------------------------------------------------------------------
def cycle_states(scn, compose, rollback):
    """States of one cycle of passes, found by composing them once and rolling
    them back.  llama2_7b: the passes that carry the prompt from its first to
    its last chunk next to the decodes (9 passes).  Other workloads: one pass.
    Returns ([states per pass], [metadata per pass])."""
    states = list(scn.requests)
    out, metas, made = [], [], []
    while True:
        m = compose(scn.budget, scn.max_chunk, states)
        made.append(m)
        meta = m.meta if hasattr(m, "meta") else m
        out.append(list(states))
        metas.append(meta)
        n = dict(zip([int(x) for x in meta.seq_ids], [int(x) for x in meta.n_new]))
        states = [(sid, pl, seen + n.get(sid, 0)) for sid, pl, seen in states]
        prompts_left = any(seen < pl for _, pl, seen in states)
        if scn.name != "llama2_7b" or not prompts_left:
            break
    for m in reversed(made):
        rollback(m)
    return out, metas


def workload_label(scn, ncyc):
    """The ``config.workload`` string, the same in both arms."""
    sh = scn.shape
    return (f"{scn.name}: {sh.num_heads_q}q/{sh.num_heads_kv}kv heads, head_dim {sh.head_dim}, "
            f"block {sh.block_size}, budget {scn.budget}, chunk cap {scn.max_chunk}; a cycle of "
            f"{ncyc} pass{'es' if ncyc != 1 else ''} repeated (rolled back on the composer after "
            "each cycle)")


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    hbm, bf16, bf16_sus, src = (HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS,
                                BF16_SUSTAINED_FALLBACK_TFLOPS, "fallback")
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
    """SM clocks and throttle reasons sampled while timing (read-only queries).

    A thread reads the GPU's SM clock and its clock-event reasons through NVML
    (libnvidia-ml, the library nvidia-smi uses) every 5 ms, so that even a
    timed region of a few tens of milliseconds has samples inside it; without
    NVML it falls back to ``nvidia-smi -lms 50``.  ``stop(t0, t1)`` reports the
    samples between wall-clock times t0 and t1, or, when none landed there,
    the nearest sample on each side of the region (``"window": "bracketing"``)."""

    # NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, uuid: str = ""):
        self.gpu = gpu_index
        self.uuid = uuid
        self.proc = None
        self.path = None
        self.thread = None
        self.samples = []      # (wall time, sm MHz, max sm MHz, reason bits)
        self.source = None

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.gpu, ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        return lib, h

    def start(self):
        import threading
        try:
            import ctypes
            lib, h = self._nvml()
            self.stop_evt = threading.Event()
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))   # NVML_CLOCK_SM
            reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons

            def run():
                clk = ctypes.c_uint()
                rs = ctypes.c_ulonglong()
                while not self.stop_evt.is_set():
                    t = time.time()
                    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                        bits = rs.value if reasons_fn(h, ctypes.byref(rs)) == 0 else 0
                        self.samples.append((t, float(clk.value), float(mx.value), int(bits)))
                    self.stop_evt.wait(0.005)
            self.thread = threading.Thread(target=run, daemon=True)
            self.thread.start()
            self.source = "nvml, 5 ms"
            return
        except Exception:
            self.thread = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi, 50 ms"
        except Exception:
            self.proc = None

    def _read_smi(self):
        import datetime
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    clk, cmax = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                bits = 0
                for n, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                 "sw_power_cap"), parts[6:10]):
                    if v.lower().startswith("active"):
                        bits |= self.REASON_BITS[n]
                self.samples.append((ts, clk, cmax, bits))
        os.unlink(self.path)

    def stop(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen between wall-clock
        times t0 and t1 (all samples when not given)."""
        if self.thread is not None:
            self.stop_evt.set()
            self.thread.join(timeout=5)
        elif self.proc is not None:
            self._read_smi()
        else:
            return None
        smp = sorted(self.samples)
        if not smp:
            return None
        window = "timed region"
        if t0 is None:
            sel = smp
        else:
            sel = [x for x in smp if t0 <= x[0] <= t1]
            if not sel:
                before = [x for x in smp if x[0] < t0][-1:]
                after = [x for x in smp if x[0] > t1][:1]
                sel = before + after
                window = "bracketing (no sample inside the timed region)"
        if not sel:
            return None
        reasons = sorted(n for n, b in self.REASON_BITS.items() if any(x[3] & b for x in sel))
        return {"sm_mhz": statistics.median(x[1] for x in sel),
                "sm_max_mhz": max(x[2] for x in sel), "samples": len(sel),
                "reasons": reasons, "window": window, "source": self.source}


def over_ranks(times, counts, world, device="cpu"):
    """Replicas: the job's time is the slowest rank's, its work the sum of all
    ranks' (max of ``times``, sum of ``counts``).  One rank: unchanged."""
    if world <= 1:
        return [float(x) for x in times], [float(x) for x in counts]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in times], dtype=torch.float64, device=device)
    c = torch.tensor([float(x) for x in counts], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(c, op=dist.ReduceOp.SUM)
    return [float(x) for x in t.tolist()], [float(x) for x in c.tolist()]


def traffic_bytes(workload, kernel):
    """ncu DRAM traffic per launch recorded for this kernel and workload, or
    None when there is none or the kernel source changed since."""
    import hashlib
    rec = TRAFFIC_BYTES.get((workload, kernel))
    if rec is None:
        return None
    src, sha, nbytes = rec
    path = os.path.join(ROOT, "ragged_blocked_kv_gb300", "csrc", src)
    try:
        with open(path, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:12] != sha:
                return None
    except OSError:
        return None
    return nbytes


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
    """Runs the workload's cycle of passes through the library, again and
    again: after the last pass of a cycle the cycle's passes are rolled back on
    the composer (newest first), so every cycle composes, appends and attends
    exactly the same passes.  Each step is one whole pass."""

    def __init__(self, rbkv, scn, seed, device):
        import torch
        import workloads
        self.torch = torch
        self.rbkv = rbkv
        self.scn = scn
        self.shape = sh = scn.shape
        self.cfg = rbkv.Config(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size,
                               sh.dtype, scn.num_blocks)
        self.comp = rbkv.Composer(self.cfg)
        dt = self.cfg.torch_dtype
        self.kc = torch.zeros(self.cfg.cache_shape(), dtype=dt, device=device)
        self.vc = torch.zeros(self.cfg.cache_shape(), dtype=dt, device=device)
        self.device = device
        self.seed = seed
        self.stream = torch.cuda.current_stream()
        self.h_stream = rbkv._P(self.stream.cuda_stream)
        b, st = scn.registration()
        if b:
            p = self.comp.compose(b, 0, st)
            k, v = workloads.make_qkv(sh, p.num_tokens, seed, 0, device=device, which="kv")
            rbkv.kv_append(p, k, v, self.kc, self.vc)
            torch.cuda.synchronize()
            del k, v, p
        states, metas = cycle_states(scn, self.comp.compose, self.comp.rollback)
        self.cycle = [rbkv.seq_states(st) for st in states]
        self.work = [step_work(m, sh) for m in metas]
        self.T = [int(m.q_start[-1]) for m in metas]
        self.max_T = max(self.T)
        self.pending = []
        self.ws = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        self.o = torch.empty((self.max_T, sh.num_heads_q, sh.head_dim), dtype=dt, device=device)
        # one input set per pass of the cycle, reused every cycle
        self.inputs = []
        for k in range(len(self.cycle)):
            q, kk, vv = workloads.make_qkv(sh, self.T[k], seed, 100 + k, device=device)
            self.inputs.append((q, kk, vv, self.o[:self.T[k]]))
        torch.cuda.synchronize()

    def step(self, i):
        """Pass i of the run (position i % cycle length), inputs in HBM."""
        rbkv = self.rbkv
        kpos = i % len(self.cycle)
        q, k, v, o = self.inputs[kpos]
        p = self.comp.compose(self.scn.budget, self.scn.max_chunk, self.cycle[kpos])
        rbkv.kv_append(p, k, v, self.kc, self.vc, stream=self.h_stream)
        rbkv.ragged_attention(p, q, self.kc, self.vc, o=o, workspace=self.ws,
                              stream=self.h_stream)
        self.pending.append(p)
        if kpos == len(self.cycle) - 1:
            for pp in reversed(self.pending):
                self.comp.rollback(pp)
            self.pending.clear()
        return self.T[kpos]

    def run_e2e(self, first, count):
        """Passes first .. first+count-1 with Q/K/V copied in from pinned host
        memory and O copied back, pipelined the way a serving loop would: the
        next pass's inputs (Q, K and V of a pass in one buffer, one copy) go in
        on one copy stream while this pass computes, and O goes back on another
        once its pass has finished.  Every copy is inside the caller's timed
        region (the last O copy is waited for on the compute stream).  Returns
        the pass tokens."""
        torch, rbkv = self.torch, self.rbkv
        n = len(self.cycle)
        # at least two buffer sets, so that one pass's copies overlap the
        # next pass's compute also when the cycle has a single pass
        nsets = max(2, n)
        if not hasattr(self, "e2e_sets"):
            self.e2e_sets = []
            for j in range(nsets):
                q, k, v, o = self.inputs[j % n]
                parts = (q, k, v)
                flat = torch.empty(sum(t.numel() for t in parts), dtype=q.dtype,
                                   device=q.device)
                views, off = [], 0
                for t in parts:
                    views.append(flat[off:off + t.numel()].view(t.shape))
                    off += t.numel()
                host_flat = torch.cat([t.reshape(-1) for t in parts]).cpu().pin_memory()
                o_dev = torch.empty_like(o)
                o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
                self.e2e_sets.append((flat, views, o_dev, host_flat, o_host))
            self.cs_in, self.cs_out = torch.cuda.Stream(), torch.cuda.Stream()
            self.ev_in = [torch.cuda.Event() for _ in range(nsets)]
            self.ev_done = [torch.cuda.Event() for _ in range(nsets)]
            self.ev_out = [torch.cuda.Event() for _ in range(nsets)]
        comp = self.stream

        def copy_in(i):
            b = i % nsets
            flat, _, _, host_flat, _ = self.e2e_sets[b]
            self.cs_in.wait_event(self.ev_done[b])        # the set's last pass is done
            with torch.cuda.stream(self.cs_in):
                flat.copy_(host_flat, non_blocking=True)
            self.ev_in[b].record(self.cs_in)

        tokens = 0
        copy_in(first)
        for i in range(first, first + count):
            kpos, b = i % n, i % nsets
            if i + 1 < first + count:
                copy_in(i + 1)
            _, (q, k, v), o, _, o_host = self.e2e_sets[b]
            p = self.comp.compose(self.scn.budget, self.scn.max_chunk, self.cycle[kpos])
            comp.wait_event(self.ev_in[b])
            comp.wait_event(self.ev_out[b])                 # O of the set copied out
            rbkv.kv_append(p, k, v, self.kc, self.vc, stream=self.h_stream)
            rbkv.ragged_attention(p, q, self.kc, self.vc, o=o, workspace=self.ws,
                                  stream=self.h_stream)
            self.ev_done[b].record(comp)
            self.cs_out.wait_event(self.ev_done[b])
            with torch.cuda.stream(self.cs_out):
                o_host.copy_(o, non_blocking=True)
            self.ev_out[b].record(self.cs_out)
            self.pending.append(p)
            if kpos == n - 1:
                for pp in reversed(self.pending):
                    self.comp.rollback(pp)
                self.pending.clear()
            tokens += self.T[kpos]
        comp.wait_event(self.ev_out[(first + count - 1) % nsets])
        return tokens

    def work_of(self, first, count):
        acc = {}
        for i in range(first, first + count):
            for kk, vv in self.work[i % len(self.work)].items():
                acc[kk] = acc.get(kk, 0) + vv
        return acc


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
    ncyc = len(run.cycle)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    i = 0
    for _ in range(W):
        run.step(i)
        i += 1
    torch.cuda.synchronize()

    # ---- timed region: K passes, inputs resident in HBM -----------------
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local_rank).uuid)
    except Exception:
        uuid = ""
    clocks = ClockSampler(local_rank, uuid)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.5)                      # the sampler starts before the timed region
    launches0 = rbkv.kernel_launches()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    first = i
    wall_t0 = time.time()
    wall0 = time.perf_counter()
    t_start.record(run.stream)
    tokens = 0
    for _ in range(K):
        tokens += run.step(i)
        i += 1
    t_end.record(run.stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    wall_t1 = time.time()
    barrier()
    launches = rbkv.kernel_launches() - launches0
    clk = clocks.stop(wall_t0, wall_t1)
    ms = t_start.elapsed_time(t_end)
    work = run.work_of(first, K)

    # ---- per-kernel device times: the same passes again with CUDA events
    # around every launch (these events keep kernels from overlapping, so the
    # timed region above runs without them)
    P = min(K, 900 - 900 % ncyc) or ncyc
    rbkv.profile_reset()
    rbkv.profile_enable(True)
    prof_first = i
    for _ in range(P):
        run.step(i)
        i += 1
    torch.cuda.synchronize()
    rbkv.profile_enable(False)
    prof = rbkv.profile_read()
    prof_work = run.work_of(prof_first, P)

    # ---- e2e: the same passes through the same calls, host buffers ------
    run.run_e2e(i, ncyc)
    i += ncyc
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_first = i
    e0.record(run.stream)
    e2e_tokens = run.run_e2e(i, K)
    i += K
    e1.record(run.stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    sh = scn.shape
    esz = 2 if sh.dtype == "bf16" else 4
    e2e_work = run.work_of(e2e_first, K)
    h2d = e2e_work["tokens"] * (sh.num_heads_q + 2 * sh.num_heads_kv) * sh.head_dim * esz / K
    d2h = e2e_work["tokens"] * sh.num_heads_q * sh.head_dim * esz / K

    # ---- max over ranks --------------------------------------------------
    (ms, e2e_ms), (tot_tokens, tot_e2e) = over_ranks([ms, e2e_ms], [tokens, e2e_tokens],
                                                     world, device)
    if rank != 0:
        return

    hbm, bf16, bf16_sus, src = read_peaks()
    kinds = {k: v for k, v in prof.items() if v[1] > 0}
    dom = max(kinds, key=lambda k: kinds[k][0])
    dom_ms, dom_n = kinds[dom]
    avg_s = dom_ms / dom_n / 1e3
    if dom == "chunk":
        # each launch is timed on its own (events around it): the burst peak
        per_launch = prof_work["chunk_flops"] / dom_n
        roof = {"bound": "tensor", "achieved": per_launch / avg_s / 1e12, "peak": bf16,
                "unit": "TFLOP/s"}
    else:
        key = {"decode": "decode_bytes", "generic": "kv_read_bytes",
               "kv_append": "append_bytes", "combine": "decode_bytes"}[dom]
        per_launch = prof_work[key] / dom_n
        roof = {"bound": "hbm", "achieved": per_launch / avg_s / 1e9, "peak": hbm, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = traffic_bytes(args.workload, dom)
    roof["kernel"] = dom
    roof["peak_source"] = src
    roof["avg_launch_us"] = avg_s * 1e6
    roof["algorithmic_per_launch"] = per_launch

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
            "workload": workload_label(scn, ncyc),
            "tokens_per_step": tot_tokens / K / world,
            "kv_read_gb_per_step": work["kv_read_bytes"] / K / 1e9,
            "kv_read_gbs": work["kv_read_bytes"] / (ms / 1e3) / 1e9,
            "kv_read_frac_of_hbm": work["kv_read_bytes"] / (ms / 1e3) / 1e9 / hbm,
            "kv_read_frac_target": 0.70,
            "chunk_tflops": prof_work["chunk_flops"] / (kinds.get("chunk", (1e30, 1))[0] / 1e3) / 1e12,
            # the chunk kernel's causal flops over its own launch time (each launch
            # timed alone, between events), against the measured burst bf16 peak
            "chunk_frac_of_bf16_peak": prof_work["chunk_flops"]
            / (kinds.get("chunk", (1e30, 1))[0] / 1e3) / 1e12 / bf16,
            "l2": "inputs larger than L2 (each pass reads "
                  f"{work['kv_read_bytes'] / K / 1e6:.0f} MB of KV > 129 MB L2); no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "kernel_us_per_launch": {k: round(v[0] * 1e3 / v[1], 2) for k, v in kinds.items()},
            "profiled_passes": P,
            "host_wall_ms": wall * 1e3,
        },
        "roofline": roof,
        "e2e": {"value": tot_e2e / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    try:
        line["layer"] = layer_profile(torch, rbkv, device)
    except Exception as e:  # reported, not fatal: the headline is the attention pass
        line["layer"] = {"error": str(e)[:200]}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_subprocess(args)
        rss = resource.getrusage(resource.RUSAGE_CHILDREN).ru_maxrss * 1024
        line["cpu_baseline"]["all_cores"] = cpu_all_cores(args, rss)
    print(json.dumps(line), flush=True)


def layer_profile(torch, rbkv, device, tokens=(16, 512, 2048), reps=5):
    """One Llama-2-7B decoder layer on the library's kernels (RMSNorm, the QKV,
    output and MLP projections as tensor-core GEMMs with fused epilogues, the
    KV append and ragged attention) on a pass of one fresh prompt of T
    tokens: median device time over `reps` runs (each composed, run and
    rolled back), and the projections' rate (their flops over that time)."""
    from ragged_blocked_kv_gb300.layer import DecoderLayer, random_weights
    hidden, hq, hkv, d, ffn = 4096, 32, 32, 128, 11008
    w = random_weights(hidden, hq, hkv, d, ffn, seed=7, device=device)
    del w["w_gate"], w["w_up"]
    layer = DecoderLayer(rbkv, w, hq, hkv, d)
    tmax = max(tokens)
    buf = layer.buffers(tmax, device)
    cfg = rbkv.Config(hq, hkv, d, 64, "bf16", -(-tmax // 64) + 4)
    comp = rbkv.Composer(cfg)
    kc = torch.zeros(cfg.cache_shape(), dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=device)
    x = torch.randn(tmax, hidden, device=device).to(torch.bfloat16)
    out = torch.empty_like(x)
    gemm_macs = hidden * ((hq + 2 * hkv) * d) + hq * d * hidden + 2 * ffn * hidden + ffn * hidden
    res = {"model": "Llama-2-7B decoder layer (hidden 4096, 32/32 heads, ffn 11008), random bf16 "
                    "weights, every step a library kernel; one fresh prompt of T tokens",
           "tokens": list(tokens), "ms": [], "projection_tflops": []}
    for T in tokens:
        times = []
        for r in range(reps + 2):
            p = comp.compose(T, 0, [(1, T, 0)])

            def attend(q, k, v, o, p=p):
                rbkv.kv_append(p, k, v, kc, vc)
                rbkv.ragged_attention(p, q, kc, vc, o=o, workspace=ws)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            layer.forward_into(x[:T], out[:T], buf, attend, T)
            e1.record()
            torch.cuda.synchronize()
            comp.rollback(p)
            if r >= 2:
                times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        res["ms"].append(round(ms, 4))
        res["projection_tflops"].append(round(2.0 * T * gemm_macs / (ms / 1e3) / 1e12, 1))
    return res


# ---------------------------------------------------------------------------
# trace workload: closed-loop SplitFuse serving of 512 requests
# ---------------------------------------------------------------------------
class DenseStack:
    """Random-weight Llama-2-7B-shaped decoder layers around the library's
    attention, every step a library kernel (ragged_blocked_kv_gb300.layer):
    RMSNorm, the QKV projection as one tensor-core GEMM writing Q, K and V,
    the KV append and ragged attention, the output projection with a fused
    residual, RMSNorm, the gate/up GEMM with a fused SwiGLU, the down
    projection with a fused residual (hidden 4096, intermediate 11008).
    Rotary embeddings are left out (elementwise work that does not change the
    shape of the pass).  It exists to measure pass latency against token
    count (paper summary page, ideas I1/I2)."""

    HIDDEN, INTER = 4096, 11008

    def __init__(self, torch, rbkv, cfg, layers, max_tokens, device, seed):
        from ragged_blocked_kv_gb300.layer import DecoderLayer, random_weights
        hq, hkv, d = cfg.num_heads_q, cfg.num_heads_kv, cfg.head_dim
        self.layers = []
        for l in range(layers):
            w = random_weights(self.HIDDEN, hq, hkv, d, self.INTER, seed * 1000 + l, device)
            del w["w_gate"], w["w_up"]          # the interleaved w_gu is what runs
            self.layers.append(DecoderLayer(rbkv, w, hq, hkv, d))
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        self.x0 = torch.randn(max_tokens, self.HIDDEN, generator=g, device=device,
                              dtype=torch.float32).to(torch.bfloat16)
        self.xs = [torch.empty_like(self.x0), torch.empty_like(self.x0)]
        self.buf = self.layers[0].buffers(max_tokens, device)
        self.torch, self.rbkv, self.cfg = torch, rbkv, cfg

    def weight_bytes(self):
        return sum(t.numel() * t.element_size() for l in self.layers for t in l.w.values())

    def _layers(self, T, attend):
        x = self.x0[:T]
        for l, layer in enumerate(self.layers):
            out = self.xs[l & 1][:T]
            layer.forward_into(x, out, self.buf, lambda q, k, v, o, l=l: attend(l, q, k, v, o), T)
            x = out
        return x

    def forward(self, p, caches, ws, hs):
        rbkv = self.rbkv

        def attend(l, q, k, v, o):
            kc, vc = caches[l]
            rbkv.kv_append(p, k, v, kc, vc, stream=hs)
            rbkv.ragged_attention(p, q, kc, vc, o=o, workspace=ws, stream=hs)
        return self._layers(p.num_tokens, attend)

    def forward_frame(self, frame, caches, ws):
        """The pass loaded in ``frame``, on frame-sized buffers and the current
        stream (capturable)."""
        def attend(l, q, k, v, o):
            kc, vc = caches[l]
            frame.kv_append(k, v, kc, vc)
            frame.attention(q, kc, vc, o, ws)
        return self._layers(frame.max_tokens, attend)


def _trace_setup(args, rank, world, local_rank, max_tokens):
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
    L = args.layers
    reqs = workloads.trace_requests(seed=args.seed)
    nb = workloads.trace_block_pool(reqs, 32, 64)
    cfg = rbkv.Config(32, 32, 128, 64, "bf16", nb)
    caches = [(torch.zeros(cfg.cache_shape(), dtype=torch.bfloat16, device=device),
               torch.zeros(cfg.cache_shape(), dtype=torch.bfloat16, device=device))
              for _ in range(L)]
    ws = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    if args.layer == "full":
        stack = DenseStack(torch, rbkv, cfg, L, max_tokens, device, args.seed)
    else:
        stack = AttentionStack(torch, rbkv, cfg, L, max_tokens, device, args.seed)
    stream = torch.cuda.current_stream()
    hs = rbkv._P(stream.cuda_stream)
    torch.cuda.synchronize()
    return torch, rbkv, workloads, reqs, cfg, caches, ws, stack, stream, hs


class AttentionStack:
    """Per layer only the library's part of the pass: the KV append and ragged
    attention (Llama-2-7B attention shape, one K/V cache per layer, one block
    table shared by all layers), on seeded Q/K/V."""

    def __init__(self, torch, rbkv, cfg, layers, max_tokens, device, seed):
        import workloads
        import math as _m
        shape = workloads.Shape(32, 32, 128, 64, "bf16", 1.0 / _m.sqrt(128.0))
        self.inputs = [workloads.make_qkv(shape, max_tokens, seed, 1000 + l, device=device)
                       for l in range(layers)]
        self.o = torch.empty((max_tokens, 32, 128), dtype=torch.bfloat16, device=device)
        self.rbkv = rbkv

    def weight_bytes(self):
        return 0

    def forward(self, p, caches, ws, hs):
        T = p.num_tokens
        for l, (q, k, v) in enumerate(self.inputs):
            kc, vc = caches[l]
            self.rbkv.kv_append(p, k[:T], v[:T], kc, vc, stream=hs)
            self.rbkv.ragged_attention(p, q[:T], kc, vc, o=self.o[:T], workspace=ws, stream=hs)

    def forward_frame(self, frame, caches, ws):
        T = frame.max_tokens
        for l, (q, k, v) in enumerate(self.inputs):
            kc, vc = caches[l]
            frame.kv_append(k[:T], v[:T], kc, vc)
            frame.attention(q[:T], kc, vc, self.o[:T], ws)


class GraphRunner:
    """Runs passes of a stack through a frame and one CUDA graph: the first
    pass runs eagerly (warming the library's kernels), then the stack's
    launches are captured once; every later pass is a metadata load plus a
    replay.  A pass the frame cannot hold runs eagerly through the plain entry
    points."""

    def __init__(self, torch, rbkv, cfg, stack, caches, ws, hs, max_tokens, **caps):
        self.torch, self.rbkv, self.stack, self.caches, self.ws, self.hs = (
            torch, rbkv, stack, caches, ws, hs)
        self.frame = rbkv.Frame(cfg, max_tokens, **caps)
        self.fws = torch.empty(max(256, self.frame.workspace_bytes()), dtype=torch.uint8,
                               device=ws.device)
        self.graph = None
        self.per_replay = 0
        self.replays = 0
        self.eager = 0

    def run(self, p):
        torch, rbkv = self.torch, self.rbkv
        try:
            self.frame.load(p)
        except rbkv.RbkvError:
            self.eager += 1
            self.stack.forward(p, self.caches, self.ws, self.hs)
            return
        if self.graph is None:
            self.stack.forward_frame(self.frame, self.caches, self.fws)
            torch.cuda.synchronize()
            n0 = rbkv.kernel_launches()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph):
                self.stack.forward_frame(self.frame, self.caches, self.fws)
            self.per_replay = rbkv.kernel_launches() - n0
            return
        self.graph.replay()
        self.replays += 1

    def close(self):
        self.graph = None
        self.frame.close()


PROFILE_TOKENS = (16, 32, 64, 128, 256, 384, 512, 768, 1024, 1536, 2048, 3072, 4096)


def measure_profile(torch, rbkv, cfg, caches, ws, stack, stream, hs, tokens=PROFILE_TOKENS,
                    reps=10, warm=3, graph=True):
    """Pass latency (median of ``reps`` CUDA-event timings) against the pass's
    token count, for two compositions of the same count: one fresh prompt of T
    tokens, and min(T, 32) fresh prompts sharing T tokens.  Each pass is
    composed, run ``warm + reps`` times (replays of one captured graph when
    ``graph``) and rolled back."""
    out = []
    for T in tokens:
        row = {"tokens": int(T)}
        for kind in ("one_prompt", "many_prompts"):
            n = 1 if kind == "one_prompt" else min(T, 32)
            states = [(90_000 + i, T // n + (1 if i < T % n else 0), 0) for i in range(n)]
            comp = rbkv.Composer(cfg)
            p = comp.compose(T, T, states)
            assert p.num_tokens == T
            if graph:
                # room for one tensor-core tile per prompt, whatever the mix
                runner = GraphRunner(torch, rbkv, cfg, stack, caches, ws, hs, T,
                                     max_chunk_tiles=-(-T // 128) + n + 8, packed_units=1)
                run = runner.run
            else:
                def run(p):
                    stack.forward(p, caches, ws, hs)
            for _ in range(warm):
                run(p)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(reps)]
            for a, b in ev:
                a.record(stream)
                run(p)
                b.record(stream)
            torch.cuda.synchronize()
            row[f"latency_ms_{kind}"] = statistics.median(a.elapsed_time(b) for a, b in ev)
            if graph:
                assert runner.eager == 0
                runner.close()
            comp.rollback(p)
        row["tokens_per_s"] = T / (row["latency_ms_one_prompt"] / 1e3)
        out.append(row)
    return out


def run_profile_bench(args, rank, world, local_rank):
    """Pass latency against token count (paper summary page, idea I1: latency
    follows the token count, not the number of sequences; idea I2: throughput
    saturates and is concave), and the largest budget whose interpolated
    latency stays within ``--latency-bound`` (FastGen guide, "Prompt-Decode
    Decoupling")."""
    torch, rbkv, workloads, reqs, cfg, caches, ws, stack, stream, hs = _trace_setup(
        args, rank, world, local_rank, max(PROFILE_TOKENS))
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local_rank).uuid)
    except Exception:
        uuid = ""
    clocks = ClockSampler(local_rank, uuid)
    clocks.start()
    time.sleep(0.3)
    w0 = time.time()
    prof = measure_profile(torch, rbkv, cfg, caches, ws, stack, stream, hs, graph=args.graph)
    w1 = time.time()
    clk = clocks.stop(w0, w1)
    toks = [r["tokens"] for r in prof]
    lat = [r["latency_ms_one_prompt"] for r in prof]
    budget = rbkv.budget_for_latency(toks, lat, args.latency_bound)
    if rank != 0:
        return
    best = max(prof, key=lambda r: r["tokens_per_s"])
    line = {
        "metric": "pass latency vs tokens",
        "value": best["tokens_per_s"],
        "unit": "tokens/s (best over the sweep)",
        "n_gpus": world,
        "higher_is_better": True,
        "dtype": "bf16",
        "data": "synthetic, random weights",
        "config": {
            "workload": f"profile: {args.layers} layers, "
                        + ("Llama-2-7B-shaped decoder layers (library tensor-core "
                           "projections and attention)" if args.layer == "full" else
                           "library KV append + attention only") + ", fresh prompts, "
                        + ("one CUDA graph per pass" if args.graph else "eager launches"),
            "weights_gb": stack.weight_bytes() / 1e9,
            "latency_bound_ms": args.latency_bound,
            "budget_for_bound": budget,
        },
        "profile": prof,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_trace_bench(args, rank, world, local_rank):
    """512 requests from 32 closed-loop clients (prompt lengths round(N(2600,
    780^2)), output lengths round(N(60, 18^2)), at least 1), composed into
    passes of ``--budget`` tokens (chunk cap the same, ``--policy`` greedy or
    equal chunks) until every request has finished.  Each pass runs every
    layer: the library's KV append and attention alone (``--layer attention``),
    or whole random-weight decoder layers (``--layer full``).  ``--budget 0``
    measures the latency profile first and takes the largest budget whose
    interpolated pass latency is within ``--latency-bound``.  Reports pass
    tokens per second over the whole trace, the per-pass latency distribution,
    and the serving metrics of the trace on the GPU timeline (pass end times
    from CUDA events; the host composes ahead of the GPU): TTFT, pace, token
    intervals and effective throughput under ``--ttft-sla``/``--pace-sla``."""
    from ragged_blocked_kv_gb300.serving import TraceRecorder, serving_metrics
    max_tok = max(max(PROFILE_TOKENS), args.budget)
    torch, rbkv, workloads, reqs, cfg, caches, ws, stack, stream, hs = _trace_setup(
        args, rank, world, local_rank, max_tok)
    L = args.layers
    budget = args.budget
    prof = None
    if budget <= 0:
        prof = measure_profile(torch, rbkv, cfg, caches, ws, stack, stream, hs,
                               graph=args.graph)
        budget = rbkv.budget_for_latency([r["tokens"] for r in prof],
                                         [r["latency_ms_one_prompt"] for r in prof],
                                         args.latency_bound)
        if budget <= 0:
            raise SystemExit(f"no budget meets a {args.latency_bound} ms pass latency")

    runner = GraphRunner(torch, rbkv, cfg, stack, caches, ws, hs, budget) if args.graph else None

    def drive(trace_reqs, comp, record, rec=None):
        events, tokens = [], []

        def compose(b, M, states):
            p = comp.compose(b, M, states, policy=args.policy)
            if p.num_tokens:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if runner:
                    runner.run(p)
                else:
                    stack.forward(p, caches, ws, hs)
                e1.record(stream)
                if record:
                    events.append((e0, e1))
                    tokens.append(p.num_tokens)
            elif record:
                events.append(None)
                tokens.append(0)
            return p.meta
        n = workloads.run_trace(trace_reqs, 32, budget, budget, compose, comp.release,
                                on_pass=rec.on_pass if rec else None)
        return n, events, tokens

    # warm-up: a short trace of the same shape on its own composer
    warm = workloads.trace_requests(seed=args.seed + 1, num_requests=64, num_clients=32)
    drive(warm, rbkv.Composer(cfg), False)
    torch.cuda.synchronize()

    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local_rank).uuid)
    except Exception:
        uuid = ""
    clocks = ClockSampler(local_rank, uuid)
    clocks.start()
    time.sleep(0.5)
    comp = rbkv.Composer(cfg)
    rec = TraceRecorder()
    launches0 = rbkv.kernel_launches()
    replays0 = runner.replays if runner else 0
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    wall_t0 = time.time()
    t0.record(stream)
    npass, events, tokens = drive(reqs, comp, True, rec)
    t1.record(stream)
    torch.cuda.synchronize()
    wall_t1 = time.time()
    clk = clocks.stop(wall_t0, wall_t1)
    launches = rbkv.kernel_launches() - launches0
    if runner:
        launches += (runner.replays - replays0) * runner.per_replay
    total_ms = t0.elapsed_time(t1)
    lat = sorted(e[0].elapsed_time(e[1]) for e in events if e is not None)
    ends, last = [], 0.0
    for e in events:
        last = t0.elapsed_time(e[1]) if e is not None else last
        ends.append(last)
    serving = serving_metrics(rec, ends, args.ttft_sla, args.pace_sla)

    def pct(x):
        return lat[min(len(lat) - 1, int(round(x / 100.0 * (len(lat) - 1))))]

    (total_ms,), (ntok,) = over_ranks([total_ms], [sum(tokens)], world, device=f"cuda:{local_rank}")
    if rank != 0:
        return
    what = ("Llama-2-7B-shaped decoder layers (random weights, library tensor-core "
            "projections, KV append and attention)" if args.layer == "full" else
            "library KV append + attention of 32q/32kv heads, head_dim 128, block 64")
    line = {
        "metric": ("SplitFuse forward pass tokens/s" if args.layer == "full"
                   else "ragged SplitFuse attention pass tokens/s"),
        "value": ntok / (total_ms / 1e3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": npass,
        "warmup": 0,
        "ms_per_step": total_ms / max(1, npass),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic" + (", random weights" if args.layer == "full" else ""),
        "config": {
            "workload": f"trace: {len(reqs)} requests, 32 closed-loop clients, budget {budget}, "
                        f"chunk cap {budget}, {args.policy} chunks, {L} layers of {what}",
            "passes": npass,
            "pass_tokens": int(ntok),
            "expected_tokens": sum(r.prompt_len + r.output_len - 1 for r in reqs),
            "latency_ms": {"p50": pct(50), "p90": pct(90), "p99": pct(99), "max": lat[-1],
                           "mean": sum(lat) / len(lat)},
            "kv_cache_gb": 2 * L * caches[0][0].numel() * 2 / 1e9,
            "weights_gb": stack.weight_bytes() / 1e9,
            "l2": "KV of every layer exceeds L2; no flush",
            "warmup": "a separate 64-request trace on its own composer",
            "budget_from": (f"latency profile, bound {args.latency_bound} ms" if prof
                            else "--budget"),
            "launch": ("frame + one CUDA graph replayed per pass "
                       f"({runner.per_replay} library kernels per replay, "
                       f"{runner.eager} passes eager)" if runner else "eager launches"),
        },
        "serving": serving,
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if prof:
        line["profile"] = prof
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the oracle on the host cores (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def sample_row(i, T):
    """The i-th row (0 <= i < T) a sampled oracle pass computes: rows in a
    stride permutation of the pass (the stride is odd, near 0.618 T and prime
    to T), so that a short sample spreads over prompt rows and decode rows
    alike instead of taking the pass's first rows."""
    stride = next(d for d in range(max(1, int(T * 0.618)) | 1, 2 * T + 2, 2)
                  if math.gcd(d, T) == 1)
    return (i * stride) % T


class OracleRunner:
    """The fp64 oracle driven through the same cycle of passes (rolled back on
    the oracle composer after each cycle).

    A step is one pass: oracle composition and appending of the whole pass,
    then oracle attention for ``pairs`` (row, query head) outputs of it, the
    rows taken in a stride permutation of the pass and continuing from step to
    step, so that every row and head of the cycle is covered in turn.  A token counts as 1/H_q per output
    pair computed.  ``step`` returns the tokens credited, the seconds spent
    composing and appending, and the pass's tokens (for charging that per-pass
    cost in proportion to the tokens a sample credits)."""

    def __init__(self, scn, seed, offset=0):
        import numpy as np
        import oracle
        import workloads
        self.np = np
        self.oracle = oracle
        self.scn = scn
        self.shape = sh = scn.shape
        self.comp = oracle.Composer(sh.block_size, scn.num_blocks)
        storage = np.uint16 if sh.dtype == "bf16" else np.float32
        self.kc = oracle.BlockedCache(sh.num_heads_kv, sh.block_size, sh.head_dim, storage)
        self.vc = oracle.BlockedCache(sh.num_heads_kv, sh.block_size, sh.head_dim, storage)
        b, st = scn.registration()
        if b:
            m = self.comp.compose(b, 0, st)
            k, v = workloads.make_qkv(sh, m.num_tokens, seed, 0, which="kv")
            oracle.kv_append(m, self._st(k), self._st(v), self.kc, self.vc)
        self.cycle, metas = cycle_states(scn, self.comp.compose, self.comp.rollback)
        self.inputs = []
        for k in range(len(self.cycle)):
            T = int(metas[k].q_start[-1])
            q, kk, vv = workloads.make_qkv(sh, T, seed, 100 + k)
            self.inputs.append((self._st(q), self._st(kk), self._st(vv)))
        self.pending = []
        self.i = 0
        self.cursor = offset  # next (row * H_q + head) to compute, per pass

    def _st(self, t):
        import torch
        t = t.contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(self.np.uint16)
        return t.numpy()

    def step(self, pairs):
        kpos = self.i % len(self.cycle)
        self.i += 1
        t0 = time.perf_counter()
        m = self.comp.compose(self.scn.budget, self.scn.max_chunk, self.cycle[kpos])
        q, k, v = self.inputs[kpos]
        self.oracle.kv_append(m, k, v, self.kc, self.vc)
        fixed = time.perf_counter() - t0
        H = self.shape.num_heads_q
        T = m.num_tokens
        total = T * H
        done = 0
        while done < pairs and total:
            c = self.cursor % total
            i, h0 = divmod(c, H)
            t = sample_row(i, T)
            n = min(pairs - done, H - h0)
            self.oracle.blocked_attention(m, q, self.kc, self.vc, H, tokens=[t],
                                          heads=range(h0, h0 + n))
            done += n
            self.cursor += n
        self.pending.append(m)
        if kpos == len(self.cycle) - 1:
            for mm in reversed(self.pending):
                self.comp.rollback(mm)
            self.pending.clear()
        return done / H, fixed, m.num_tokens


class OracleTraceRunner:
    """The oracle over the trace workload (one layer): each step is the next
    pass of the closed-loop trace - oracle composition and appending of the
    whole pass, then ``pairs`` (row, query head) outputs of it."""

    def __init__(self, seed):
        import numpy as np
        import oracle
        import workloads
        self.np, self.oracle, self.workloads = np, oracle, workloads
        self.shape = workloads.Shape(32, 32, 128, 64, "bf16", 1.0 / math.sqrt(128.0))
        self.reqs = workloads.trace_requests(seed=seed)
        nb = workloads.trace_block_pool(self.reqs, 32, 64)
        self.comp = oracle.Composer(64, nb)
        self.kc = oracle.BlockedCache(32, 64, 128, np.uint16)
        self.vc = oracle.BlockedCache(32, 64, 128, np.uint16)
        q, k, v = workloads.make_qkv(self.shape, 512, seed, 1000)
        self.inputs = [t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)
                       for t in (q, k, v)]
        self.seed = seed

    def run(self, steps, pairs, on_step):
        q, k, v = self.inputs
        H = self.shape.num_heads_q

        def compose(b, M, states):
            m = self.comp.compose(b, M, states)
            T = m.num_tokens
            self.oracle.kv_append(m, k[:T], v[:T], self.kc, self.vc)
            done = 0
            c = 0
            while done < pairs and T:
                t, h0 = divmod(c % (T * H), H)
                n = min(pairs - done, H - h0)
                self.oracle.blocked_attention(m, q[:T], self.kc, self.vc, H, tokens=[t],
                                              heads=range(h0, h0 + n))
                done += n
                c += n
            on_step(done / H)
            return m
        self.workloads.run_trace(self.reqs, 32, 512, 512, compose, self.comp.release,
                                 max_passes=steps)


def _barrier(path, world, limit_s=300.0):
    """File barrier between ``world`` concurrent oracle workers: announce this
    one, then wait (at most ``limit_s``) until all have.  Returns whether all
    arrived."""
    fd, _ = tempfile.mkstemp(dir=path, prefix="ready")
    os.close(fd)
    end = time.monotonic() + limit_s
    while time.monotonic() < end:
        if sum(1 for f in os.listdir(path) if f.startswith("ready")) >= world:
            return True
        time.sleep(0.01)
    return False


def oracle_measure(workload, seed, steps, warmup, pair_budget=2000, offset=0, barrier="",
                   world=1):
    """Time ``steps`` oracle steps after ``warmup``; each step computes about
    pair_budget // (steps + warmup) output pairs, in whole rows (every query
    head of a token) and at least one row, so the whole run stays within a few
    minutes whatever the step count.  ``offset`` moves the
    first output pair (concurrent workers cover disjoint pairs); with
    ``barrier`` the timed region starts once ``world`` workers are ready."""
    import workloads
    pairs = max(1, pair_budget // max(1, steps + warmup))
    if workload != "trace":
        # whole rows: all query heads of a token in one call, as a whole pass
        # computes them (the oracle gathers a sequence's keys once per call)
        H = workloads.SCENARIOS[workload](seed).shape.num_heads_q
        pairs = H * max(1, round(pairs / H))
    if workload == "trace":
        t0 = time.perf_counter()
        tr = OracleTraceRunner(seed)
        setup = time.perf_counter() - t0
        marks = []

        def on_step(tok):
            marks.append((time.perf_counter(), tok))
        tr.run(steps + warmup, pairs, on_step)
        timed = marks[warmup:]
        t_start = marks[warmup - 1][0] if warmup else (marks[0][0] - 1e-9)
        dt = timed[-1][0] - t_start
        tokens = sum(x[1] for x in timed)
        return {"value": tokens / dt, "tokens": tokens, "pairs_per_step": pairs, "seconds": dt,
                "setup_seconds": setup}
    scn = workloads.SCENARIOS[workload](seed)
    t0 = time.perf_counter()
    r = OracleRunner(scn, seed, offset * pairs * (steps + warmup))
    setup = time.perf_counter() - t0
    for _ in range(warmup):
        r.step(pairs)
    synced = _barrier(barrier, world) if barrier else True
    wall0 = time.time()
    t0 = time.perf_counter()
    tokens = fixed = pass_tokens = 0.0
    for _ in range(steps):
        tok, fx, pt = r.step(pairs)
        tokens += tok
        fixed += fx
        pass_tokens += pt
    dt = time.perf_counter() - t0
    # a whole pass pays its composition and append once for all its tokens:
    # the sample is charged that cost in proportion to the tokens it credits
    # (with many steps and few outputs each, the per-pass cost would swamp it)
    share = tokens / pass_tokens if pass_tokens else 1.0
    charged = dt - fixed + fixed * share
    return {"value": tokens / charged, "tokens": tokens, "pairs_per_step": pairs,
            "seconds": dt, "charged_seconds": charged, "compose_append_seconds": fixed,
            "setup_seconds": setup, "wall_start": wall0, "wall_end": wall0 + dt,
            "synced": synced, "cycle": len(r.cycle)}


def cpu_env():
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    return env


def cpu_model():
    """The host CPU's model name (x86), or its architecture and part number (Arm)."""
    import platform
    part = ""
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key, _, val = ln.partition(":")
                key = key.strip()
                if key == "model name":
                    return val.strip()
                if key == "CPU part" and not part:
                    part = val.strip()
    except OSError:
        pass
    return f"{platform.machine()} (CPU part {part})" if part else platform.machine()


def cpu_baseline_subprocess(args, steps=5, warmup=1):
    core = min(os.sched_getaffinity(0))
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", "--workload", args.workload,
           "--seed", str(args.seed), "--steps", str(steps), "--warmup", str(warmup),
           "--cpu-core", str(core)]
    try:
        out = subprocess.run(cmd, capture_output=True, text=True, env=cpu_env(), timeout=600)
        res = json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal
        return {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "sample": f"failed: {e}"}
    return {"value": res["value"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{steps} passes after {warmup} warm-up; per pass the oracle composes and "
                      f"appends the whole pass and computes {res['pairs_per_step']} (row, head) "
                      f"outputs ({res['tokens']:.1f} tokens in {res['seconds']:.1f} s; a token "
                      "counts 1/H_q per output, and the composition and append time is charged "
                      "in proportion to the tokens credited); one thread (BLAS threads = 1) "
                      "pinned to one core",
            "cpu": cpu_model()}


def _mem_available():
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    return int(ln.split()[1]) * 1024
    except OSError:
        pass
    return 0


def cpu_all_cores(args, worker_bytes, steps=5, warmup=1):
    """The same oracle sample on every host core at once: one single-threaded
    worker per core (as many as half the free memory holds, ``worker_bytes``
    each), each on its own output pairs, all starting their timed steps
    together.  Throughput = all workers' tokens / (last end - first start)."""
    cores = sorted(os.sched_getaffinity(0))
    n = len(cores)
    if worker_bytes > 0:
        n = max(1, min(n, int(_mem_available() * 0.5 // worker_bytes)))
    tmp = tempfile.mkdtemp(prefix="rbkv_oracle_")
    procs = []
    try:
        for w in range(n):
            cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", "--workload",
                   args.workload, "--seed", str(args.seed), "--steps", str(steps), "--warmup",
                   str(warmup), "--cpu-offset", str(w), "--cpu-core", str(cores[w]),
                   "--cpu-barrier", tmp, "--cpu-world", str(n)]
            procs.append(subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                          stderr=subprocess.DEVNULL, text=True, env=cpu_env()))
        res = []
        for p in procs:
            out, _ = p.communicate(timeout=900)
            res.append(json.loads(out.strip().splitlines()[-1]))
    except Exception as e:  # reported, not fatal
        for p in procs:
            if p.poll() is None:
                p.kill()
                p.wait()
        return {"value": None, "cores": n, "sample": f"failed: {e}"}
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    tokens = sum(r["tokens"] for r in res)
    span = max(r["wall_end"] for r in res) - min(r["wall_start"] for r in res)
    # the per-pass composition and append charged as in the 1-core sample
    span *= sum(r["charged_seconds"] / r["seconds"] for r in res) / len(res)
    room = "" if n == len(cores) else f" (the free memory holds {n} of {len(cores)} cores' workers)"
    return {"value": tokens / span, "cores": n,
            "synced": all(r["synced"] for r in res),
            "sample": f"{n} single-threaded oracle worker(s), one per core{room}, each the 1-core "
                      f"sample on its own output pairs ({tokens:.1f} tokens in {span:.1f} s of wall "
                      "time from the first start to the last end)"}


def run_reference(args, rank):
    if rank != 0:
        return
    import workloads
    if args.workload == "profile" or args.layer == "full":
        print(json.dumps({"impl": "reference", "unavailable": "the oracle covers the "
                          "attention pass only, not the dense layers or a latency profile"}),
              flush=True)
        return
    res = oracle_measure(args.workload, args.seed, args.steps, args.warmup)
    if args.workload == "trace":
        scn = workloads.Scenario("trace", workloads.Shape(32, 32, 128, 64, "bf16", 1.0), 512,
                                 512, [], [], 0)
    else:
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
        "config": {"workload": workload_label(scn, res.get("cycle", 1))
                   if args.workload != "trace" else "trace: 512 requests, 32 clients, "
                   "Llama-2-7B attention shape, budget 512, chunk cap 512 (one layer)"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"per pass: whole-pass composition and append, then "
                                   f"{res['pairs_per_step']} (row, head) outputs; a token counts "
                                   "1/H_q per output, and the passes' composition and append "
                                   "time is charged in proportion to the tokens credited; one "
                                   "thread (BLAS threads = 1)",
                         "cpu": cpu_model()},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.cpu_worker:
        if args.cpu_core >= 0:
            os.sched_setaffinity(0, {args.cpu_core})
        res = oracle_measure(args.workload, args.seed, args.steps, args.warmup,
                             offset=args.cpu_offset, barrier=args.cpu_barrier,
                             world=args.cpu_world)
        print(json.dumps(res), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            # the oracle needs no GPU; run it with BLAS threads pinned to one
            for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
                os.environ[v] = "1"
            run_reference(args, rank)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    try:
        if args.workload == "trace":
            run_trace_bench(args, rank, world, local_rank)
        elif args.workload == "profile":
            run_profile_bench(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
