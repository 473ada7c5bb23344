"""Python binding of librbkv (ctypes; argument marshalling only).

Every step of the pass runs in the library: composition, block allocation and
split planning in its host C++ code, appending and attention in its sm_103a
kernels.  This module turns torch tensors into device pointers and streams into
handles, and raises on a non-OK status.  There is no fallback: if the library
is missing, importing the names below raises.

    cfg = Config(num_heads_q=32, num_heads_kv=8, head_dim=128, block_size=64,
                 dtype="bf16", num_blocks=4096)
    comp = Composer(cfg)
    p = comp.compose(budget=2048, max_chunk=768, states=[(seq_id, prompt_len, seen), ...])
    kv_append(p, k_new, v_new, k_cache, v_cache)
    o = ragged_attention(p, q, k_cache, v_cache)
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from pathlib import Path
from typing import List, Optional, Sequence, Tuple

import numpy as np

_LIB_PATH = Path(__file__).resolve().parent / "_lib" / "librbkv.so"

OK, ERR_INVALID, ERR_NO_BLOCKS, ERR_CUDA, ERR_DEVICE_BOUNDS, ERR_UNSUPPORTED, ERR_WORKSPACE, \
    ERR_TIMEOUT = 0, -1, -2, -3, -4, -5, -6, -7
BF16, F32 = 0, 1


class RbkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"rbkv status {status}: {message}")
        self.status = status


class NoBlocksError(RbkvError):
    pass


class _Config(C.Structure):
    _fields_ = [("num_heads_q", C.c_int32), ("num_heads_kv", C.c_int32), ("head_dim", C.c_int32),
                ("block_size", C.c_int32), ("dtype", C.c_int32), ("num_blocks", C.c_int32)]


class _SeqState(C.Structure):
    _fields_ = [("seq_id", C.c_int64), ("prompt_len", C.c_int32), ("seen", C.c_int32)]


class _PassMeta(C.Structure):
    _fields_ = [("num_seqs", C.c_int32), ("num_tokens", C.c_int32), ("num_block_ids", C.c_int32),
                ("block_size", C.c_int32),
                ("seq_ids", C.POINTER(C.c_int64)), ("q_start", C.POINTER(C.c_int32)),
                ("n_new", C.POINTER(C.c_int32)), ("seen", C.POINTER(C.c_int32)),
                ("ctx", C.POINTER(C.c_int32)), ("block_start", C.POINTER(C.c_int32)),
                ("block_ids", C.POINTER(C.c_int32)), ("slot", C.POINTER(C.c_int32))]


class _PlanInfo(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "num_sms", "decode_rows", "decode_items", "max_splits", "split_keys", "partials",
        "chunk_rows", "chunk_tiles", "generic_items", "fast_decode", "fast_chunk",
        "chunk_items", "chunk_single", "chunk_steps_total", "chunk_steps_max",
        "decode_grid", "decode_keys_total", "decode_keys_max")]


class _FrameCaps(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "max_tokens", "max_seqs", "max_blocks", "max_decode_items", "max_chunk_tiles",
        "max_combine_rows", "max_parts", "packed_units", "chunk_items")]


# Every symbol include/rbkv.h declares, with (restype, argtypes).
_P = C.c_void_p
SIGNATURES = {
    "rbkv_abi_version": (C.c_int32, []),
    "rbkv_last_error": (C.c_char_p, []),
    "rbkv_composer_create": (C.c_int, [C.POINTER(_Config), C.POINTER(_P)]),
    "rbkv_composer_destroy": (None, [_P]),
    "rbkv_compose_pass": (C.c_int, [_P, C.c_int32, C.c_int32, C.POINTER(_SeqState), C.c_int32,
                                    C.POINTER(_P)]),
    "rbkv_release_seq": (C.c_int, [_P, C.c_int64]),
    "rbkv_compose_pass_policy": (C.c_int, [_P, C.c_int32, C.c_int32, C.c_int32,
                                           C.POINTER(_SeqState), C.c_int32, C.POINTER(_P)]),
    "rbkv_budget_for_latency": (C.c_int32, [C.POINTER(C.c_int32), C.POINTER(C.c_double),
                                            C.c_int32, C.c_double]),
    "rbkv_latency_at": (C.c_double, [C.POINTER(C.c_int32), C.POINTER(C.c_double), C.c_int32,
                                     C.c_int32]),
    "rbkv_pass_rollback": (C.c_int, [_P, _P]),
    "rbkv_composer_free_blocks": (C.c_int32, [_P]),
    "rbkv_pass_get_meta": (C.c_int, [_P, C.POINTER(_PassMeta)]),
    "rbkv_pass_set_split_keys": (C.c_int, [_P, C.c_int32]),
    "rbkv_pass_set_chunk_items": (C.c_int, [_P, C.c_int32]),
    "rbkv_pass_get_plan": (C.c_int, [_P, C.POINTER(_PlanInfo)]),
    "rbkv_pass_plan_for_sms": (C.c_int, [_P, C.c_int32, C.POINTER(_PlanInfo)]),
    "rbkv_pass_destroy": (None, [_P]),
    "rbkv_kv_append": (C.c_int, [_P, _P, _P, _P, _P, _P]),
    "rbkv_attention_workspace_bytes": (C.c_size_t, [_P]),
    "rbkv_ragged_attention": (C.c_int, [_P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "rbkv_pass_device_status": (C.c_int, [_P, _P]),
    "rbkv_ragged_attention_noalloc": (C.c_int, [_P, _P, _P, _P, _P, _P]),
    "rbkv_frame_create": (C.c_int, [C.POINTER(_Config), C.POINTER(_FrameCaps), C.POINTER(_P),
                                    C.POINTER(_FrameCaps)]),
    "rbkv_frame_destroy": (None, [_P]),
    "rbkv_frame_load": (C.c_int, [_P, _P, _P]),
    "rbkv_frame_kv_append": (C.c_int, [_P, _P, _P, _P, _P, _P]),
    "rbkv_frame_workspace_bytes": (C.c_size_t, [_P]),
    "rbkv_frame_attention": (C.c_int, [_P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "rbkv_frame_device_status": (C.c_int, [_P, _P]),
    "rbkv_debug_corrupt_pass": (C.c_int, [_P, C.c_int32, C.c_int32, C.c_int32]),
    "rbkv_debug_wait_timeout": (C.c_int, [_P, C.c_int64, _P]),
    "rbkv_kernel_launches": (C.c_int64, []),
    "rbkv_profile_enable": (None, [C.c_int32]),
    "rbkv_profile_read": (C.c_int, [C.c_int32, C.POINTER(C.c_double), C.POINTER(C.c_int64)]),
    "rbkv_profile_reset": (None, []),
    "rbkv_gemm_bf16": (C.c_int, [_P, _P, _P, C.c_int64, C.c_int64, C.c_int64, _P, C.c_int32,
                                 _P, C.c_size_t, _P, _P]),
    "rbkv_gemm_workspace_bytes": (C.c_size_t, [C.c_int64, C.c_int64, C.c_int64]),
    "rbkv_rmsnorm_bf16": (C.c_int, [_P, _P, _P, C.c_int64, C.c_int64, C.c_float, _P]),
    "rbkv_gemm_bf16_qkv": (C.c_int, [_P, _P, _P, _P, _P, C.c_int64, C.c_int64, C.c_int64,
                                     C.c_int64, _P, C.c_size_t, _P, _P]),
    "rbkv_router_create": (C.c_int, [C.c_int32, C.POINTER(_P)]),
    "rbkv_router_destroy": (None, [_P]),
    "rbkv_router_assign": (C.c_int, [_P, C.c_int64, C.c_int32, C.c_int32,
                                     C.POINTER(C.c_int32)]),
    "rbkv_router_progress": (C.c_int, [_P, C.c_int64, C.c_int32]),
    "rbkv_router_finish": (C.c_int, [_P, C.c_int64]),
    "rbkv_router_load": (C.c_int64, [_P, C.c_int32]),
    "rbkv_router_active": (C.c_int32, [_P, C.c_int32]),
}

KERNEL_KINDS = {"kv_append": 0, "chunk": 1, "decode": 2, "generic": 3, "combine": 4,
                "upload": 5}

_lib = None


def library_path() -> Path:
    return _LIB_PATH


def lib():
    """The loaded librbkv (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not _LIB_PATH.exists():
            raise ImportError(
                f"{_LIB_PATH} is missing; build it with `python -m ragged_blocked_kv_gb300.build` "
                "(there is no fallback implementation)")
        L = C.CDLL(str(_LIB_PATH))
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int):
    if status != OK:
        msg = lib().rbkv_last_error().decode(errors="replace")
        if status == ERR_NO_BLOCKS:
            raise NoBlocksError(status, msg)
        raise RbkvError(status, msg)


@dataclass(frozen=True)
class Config:
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    block_size: int
    dtype: str          # "bf16" or "f32"
    num_blocks: int

    def _c(self) -> _Config:
        return _Config(self.num_heads_q, self.num_heads_kv, self.head_dim, self.block_size,
                       BF16 if self.dtype == "bf16" else F32, self.num_blocks)

    @property
    def torch_dtype(self):
        import torch
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def cache_shape(self) -> Tuple[int, int, int, int]:
        return (self.num_blocks, self.num_heads_kv, self.block_size, self.head_dim)


@dataclass
class PassMeta:
    seq_ids: np.ndarray
    q_start: np.ndarray
    n_new: np.ndarray
    seen: np.ndarray
    ctx: np.ndarray
    block_start: np.ndarray
    block_ids: np.ndarray
    slot: np.ndarray

    @property
    def num_tokens(self) -> int:
        return int(self.q_start[-1])

    @property
    def num_seqs(self) -> int:
        return len(self.seq_ids)


def _arr(ptr, n, dtype):
    if n == 0:
        return np.zeros(0, dtype)
    return np.ctypeslib.as_array(ptr, shape=(n,)).astype(dtype, copy=True)


class Pass:
    """One composed pass (owns its library handle)."""

    def __init__(self, handle: int, config: Config):
        self._h = _P(handle)
        self.config = config
        self._view = _PassMeta()
        _check(lib().rbkv_pass_get_meta(self._h, C.byref(self._view)))
        self.num_tokens = int(self._view.num_tokens)
        self._meta = None

    @property
    def meta(self) -> PassMeta:
        """Copies of the pass's metadata arrays (made on first access)."""
        if self._meta is None:
            m = self._view
            S, T = m.num_seqs, m.num_tokens
            self._meta = PassMeta(_arr(m.seq_ids, S, np.int64), _arr(m.q_start, S + 1, np.int32),
                                  _arr(m.n_new, S, np.int32), _arr(m.seen, S, np.int32),
                                  _arr(m.ctx, S, np.int32), _arr(m.block_start, S + 1, np.int32),
                                  _arr(m.block_ids, m.num_block_ids, np.int32),
                                  _arr(m.slot, T, np.int32))
        return self._meta

    def set_split_keys(self, keys: int) -> None:
        _check(lib().rbkv_pass_set_split_keys(self._h, int(keys)))

    def set_chunk_items(self, mode: str) -> None:
        """Group prompt-chunk tiles as "auto", "pairs" or "single" work items."""
        m = {"auto": 0, "pairs": 1, "single": 2}[mode]
        _check(lib().rbkv_pass_set_chunk_items(self._h, m))

    def plan(self) -> dict:
        info = _PlanInfo()
        _check(lib().rbkv_pass_get_plan(self._h, C.byref(info)))
        return {n: getattr(info, n) for n, _ in _PlanInfo._fields_}

    def plan_for_sms(self, num_sms: int) -> dict:
        info = _PlanInfo()
        _check(lib().rbkv_pass_plan_for_sms(self._h, int(num_sms), C.byref(info)))
        return {n: getattr(info, n) for n, _ in _PlanInfo._fields_}

    def workspace_bytes(self) -> int:
        return int(lib().rbkv_attention_workspace_bytes(self._h))

    def device_status(self, stream=None) -> None:
        _check(lib().rbkv_pass_device_status(self._h, _stream(stream)))

    def debug_corrupt(self, which: str, index: int, value: int) -> None:
        """Fault injection for tests: overwrite a block-table ("block") or
        slot ("slot") entry before the pass reaches the device."""
        w = {"block": 0, "slot": 1}[which]
        _check(lib().rbkv_debug_corrupt_pass(self._h, w, int(index), int(value)))

    def debug_wait_timeout(self, limit_cycles: int, stream=None) -> None:
        """Run a bounded wait that is bound to give up (reported in the status)."""
        _check(lib().rbkv_debug_wait_timeout(self._h, int(limit_cycles), _stream(stream)))

    def destroy(self) -> None:
        if self._h:
            lib().rbkv_pass_destroy(self._h)
            self._h = _P(None)

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


class SeqStates:
    """A request list in the library's layout (see ``seq_states``)."""

    def __init__(self, arr, n):
        self.arr, self.n = arr, n


def seq_states(states: Sequence[Tuple[int, int, int]]) -> SeqStates:
    arr = (_SeqState * max(1, len(states)))()
    for i, (sid, plen, seen) in enumerate(states):
        arr[i] = _SeqState(int(sid), int(plen), int(seen))
    return SeqStates(arr, len(states))


class Composer:
    """Dynamic SplitFuse composer and block pool of one cache layout."""

    def __init__(self, config: Config):
        self.config = config
        h = _P()
        cfg = config._c()
        _check(lib().rbkv_composer_create(C.byref(cfg), C.byref(h)))
        self._h = h

    def compose(self, budget: int, max_chunk: int, states, policy: str = "greedy") -> Pass:
        """``states``: [(seq_id, prompt_len, seen), ...] in list order, or an
        array made once with ``seq_states`` (cheaper when reused).  ``policy``:
        "greedy" (fill the budget) or "equal" (near-equal prompt chunks)."""
        if not isinstance(states, SeqStates):
            states = seq_states(states)
        out = _P()
        if policy == "greedy":
            _check(lib().rbkv_compose_pass(self._h, int(budget), int(max_chunk), states.arr,
                                           states.n, C.byref(out)))
        else:
            pol = {"equal": 1}.get(policy, -1)
            _check(lib().rbkv_compose_pass_policy(self._h, int(budget), int(max_chunk), pol,
                                                  states.arr, states.n, C.byref(out)))
        return Pass(out.value, self.config)

    def rollback(self, p: Pass) -> None:
        """Undo what composing ``p`` did to the pool and the recorded contexts
        (newest pass first)."""
        _check(lib().rbkv_pass_rollback(self._h, p._h))

    def release(self, seq_id: int) -> None:
        _check(lib().rbkv_release_seq(self._h, int(seq_id)))

    def free_blocks(self) -> int:
        return int(lib().rbkv_composer_free_blocks(self._h))

    def close(self) -> None:
        if self._h:
            lib().rbkv_composer_destroy(self._h)
            self._h = _P(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _stream(stream):
    if isinstance(stream, _P):
        return stream
    if stream is None:
        import torch
        return _P(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return _P(stream)
    return _P(stream.cuda_stream)


def _dev_ptr(t, name, dtype, shape):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return _P(t.data_ptr())


def kv_append(p: Pass, k_new, v_new, k_cache, v_cache, stream=None) -> None:
    """Scatter the pass's new K/V rows into the blocked caches (in place)."""
    c = p.config
    T = p.num_tokens
    dt = c.torch_dtype
    row = (T, c.num_heads_kv, c.head_dim)
    _check(lib().rbkv_kv_append(p._h, _dev_ptr(k_new, "k_new", dt, row),
                                _dev_ptr(v_new, "v_new", dt, row),
                                _dev_ptr(k_cache, "k_cache", dt, c.cache_shape()),
                                _dev_ptr(v_cache, "v_cache", dt, c.cache_shape()),
                                _stream(stream)))


def ragged_attention(p: Pass, q, k_cache, v_cache, o=None, workspace=None, stream=None):
    """Ragged causal attention of every pass row; returns O ``[T][H_q][D]``."""
    import torch
    c = p.config
    T = p.num_tokens
    dt = c.torch_dtype
    qshape = (T, c.num_heads_q, c.head_dim)
    if o is None:
        o = torch.empty(qshape, dtype=dt, device=q.device)
    need = p.workspace_bytes()
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _P(workspace.data_ptr()) if workspace is not None else _P(None)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().rbkv_ragged_attention(p._h, _dev_ptr(q, "q", dt, qshape),
                                       _dev_ptr(k_cache, "k_cache", dt, c.cache_shape()),
                                       _dev_ptr(v_cache, "v_cache", dt, c.cache_shape()),
                                       _dev_ptr(o, "o", dt, qshape), ws_ptr, ws_bytes,
                                       _stream(stream)))
    return o


def ragged_attention_noalloc(p: Pass, q, k_cache, v_cache, o, stream=None):
    """Ragged attention with the library's own static scratch instead of a
    workspace: for callers that must not allocate device memory.  ``o`` must
    be given (this call allocates nothing) and the pass must already have been
    through ``kv_append``.  Calls that overlap on the GPU share the scratch and
    race; keep them ordered on one stream."""
    c = p.config
    T = p.num_tokens
    dt = c.torch_dtype
    qshape = (T, c.num_heads_q, c.head_dim)
    _check(lib().rbkv_ragged_attention_noalloc(p._h, _dev_ptr(q, "q", dt, qshape),
                                               _dev_ptr(k_cache, "k_cache", dt, c.cache_shape()),
                                               _dev_ptr(v_cache, "v_cache", dt, c.cache_shape()),
                                               _dev_ptr(o, "o", dt, qshape), _stream(stream)))
    return o


class Frame:
    """Fixed device home for one pass at a time, so that the append and
    attention launches are identical for every pass (capturable once as a CUDA
    graph and replayed).  ``load(pass)`` before each replay, on the same
    stream.  Q/K/V/O buffers have ``max_tokens`` rows; rows past the loaded
    pass's tokens are ignored."""

    CHUNK_ITEMS = {"auto": 0, "pairs": 1, "single": 2}

    def __init__(self, config: Config, max_tokens: int, **caps):
        if isinstance(caps.get("chunk_items"), str):
            caps["chunk_items"] = self.CHUNK_ITEMS[caps["chunk_items"]]
        want = _FrameCaps(max_tokens=int(max_tokens), **{k: int(v) for k, v in caps.items()})
        got = _FrameCaps()
        h = _P()
        _check(lib().rbkv_frame_create(C.byref(config._c()), C.byref(want), C.byref(h),
                                       C.byref(got)))
        self._h = h
        self.config = config
        self.caps = {n: getattr(got, n) for n, _ in _FrameCaps._fields_}
        self.max_tokens = self.caps["max_tokens"]
        # the grouping of chunk tiles every pass loaded here is planned with
        self.chunk_items = {1: "pairs", 2: "single"}[self.caps["chunk_items"]]

    def workspace_bytes(self) -> int:
        return int(lib().rbkv_frame_workspace_bytes(self._h))

    def load(self, p: "Pass", stream=None) -> None:
        _check(lib().rbkv_frame_load(self._h, p._h, _stream(stream)))

    def kv_append(self, k_new, v_new, k_cache, v_cache, stream=None) -> None:
        c = self.config
        dt = c.torch_dtype
        row = (self.max_tokens, c.num_heads_kv, c.head_dim)
        _check(lib().rbkv_frame_kv_append(self._h, _dev_ptr(k_new, "k_new", dt, row),
                                          _dev_ptr(v_new, "v_new", dt, row),
                                          _dev_ptr(k_cache, "k_cache", dt, c.cache_shape()),
                                          _dev_ptr(v_cache, "v_cache", dt, c.cache_shape()),
                                          _stream(stream)))

    def attention(self, q, k_cache, v_cache, o, workspace, stream=None) -> None:
        c = self.config
        dt = c.torch_dtype
        qshape = (self.max_tokens, c.num_heads_q, c.head_dim)
        _check(lib().rbkv_frame_attention(
            self._h, _dev_ptr(q, "q", dt, qshape),
            _dev_ptr(k_cache, "k_cache", dt, c.cache_shape()),
            _dev_ptr(v_cache, "v_cache", dt, c.cache_shape()), _dev_ptr(o, "o", dt, qshape),
            _P(workspace.data_ptr()), workspace.numel() * workspace.element_size(),
            _stream(stream)))

    def device_status(self, stream=None) -> None:
        _check(lib().rbkv_frame_device_status(self._h, _stream(stream)))

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().rbkv_frame_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def budget_for_latency(tokens, latency, bound: float) -> int:
    """Largest token count whose latency, interpolated from a measured
    (tokens, latency) profile, stays within ``bound`` (0 if none)."""
    n = len(tokens)
    t = (C.c_int32 * n)(*[int(x) for x in tokens])
    l = (C.c_double * n)(*[float(x) for x in latency])
    r = int(lib().rbkv_budget_for_latency(t, l, n, float(bound)))
    if r < 0:
        raise RbkvError(ERR_INVALID, "bad latency profile")
    return r


def kernel_launches() -> int:
    """Kernels launched through the library by this process so far."""
    return int(lib().rbkv_kernel_launches())


def profile_enable(on: bool = True) -> None:
    lib().rbkv_profile_enable(1 if on else 0)


def profile_reset() -> None:
    lib().rbkv_profile_reset()


def profile_read() -> dict:
    """{kernel: (total_ms, launches)} of the launches timed since the last reset."""
    out = {}
    for name, k in KERNEL_KINDS.items():
        ms, n = C.c_double(), C.c_int64()
        _check(lib().rbkv_profile_read(k, C.byref(ms), C.byref(n)))
        out[name] = (ms.value, n.value)
    return out


GEMM_EPILOGUES = {"plain": 0, "residual": 1, "swiglu": 2}


def gemm_workspace_bytes(m: int, n: int, k: int) -> int:
    """Workspace a GEMM of this size can use to split K (0: it does not)."""
    return int(lib().rbkv_gemm_workspace_bytes(int(m), int(n), int(k)))


def _ws(workspace):
    if workspace is None:
        return _P(None), 0
    return _P(workspace.data_ptr()), workspace.numel() * workspace.element_size()


def gemm(a, b, c=None, residual=None, epilogue: str = "plain", workspace=None, status=None,
         stream=None):
    """C = A B^T (bf16, fp32 accumulation) on the tensor cores with a fused
    epilogue: "plain", "residual" (+ residual) or "swiglu" (B's rows in blocks
    of 128 gate rows and the 128 up rows of the same outputs; C = silu(gate) *
    up).  a: [m][k], b: [n][k]; returns c ([m][n], [m][n/2] for SwiGLU)."""
    import torch
    m, k = a.shape
    n = b.shape[0]
    out_n = n // 2 if epilogue == "swiglu" else n
    if c is None:
        c = torch.empty((m, out_n), dtype=torch.bfloat16, device=a.device)
    dt = torch.bfloat16
    r = _P(None)
    if residual is not None:
        r = _dev_ptr(residual, "residual", dt, (m, n))
    st = _P(status.data_ptr()) if status is not None else _P(None)
    wsp, wsb = _ws(workspace)
    _check(lib().rbkv_gemm_bf16(_dev_ptr(a, "a", dt, (m, k)), _dev_ptr(b, "b", dt, (n, k)),
                                _dev_ptr(c, "c", dt, (m, out_n)), int(m), int(n), int(k), r,
                                GEMM_EPILOGUES[epilogue], wsp, wsb, st, _stream(stream)))
    return c


def gemm_qkv(a, w_qkv, num_heads_q: int, num_heads_kv: int, head_dim: int, out=None,
             workspace=None, status=None, stream=None):
    """The QKV projection in one GEMM: returns Q [m][H_q][D], K and V
    [m][H_kv][D] (contiguous, the attention pass's inputs; written into `out`
    = (q, k, v) when given)."""
    import torch
    m, k = a.shape
    n_q, n_kv = num_heads_q * head_dim, num_heads_kv * head_dim
    dt = torch.bfloat16
    if out is None:
        q = torch.empty((m, num_heads_q, head_dim), dtype=dt, device=a.device)
        kk = torch.empty((m, num_heads_kv, head_dim), dtype=dt, device=a.device)
        vv = torch.empty_like(kk)
    else:
        q, kk, vv = out
    st = _P(status.data_ptr()) if status is not None else _P(None)
    wsp, wsb = _ws(workspace)
    _check(lib().rbkv_gemm_bf16_qkv(_dev_ptr(a, "a", dt, (m, k)),
                                    _dev_ptr(w_qkv, "w_qkv", dt, (n_q + 2 * n_kv, k)),
                                    _dev_ptr(q, "q", dt, (m, num_heads_q, head_dim)),
                                    _dev_ptr(kk, "k", dt, (m, num_heads_kv, head_dim)),
                                    _dev_ptr(vv, "v", dt, (m, num_heads_kv, head_dim)),
                                    int(m), int(n_q), int(n_kv), int(k), wsp, wsb, st,
                                    _stream(stream)))
    return q, kk, vv


def rmsnorm(x, weight, y=None, eps: float = 1e-5, stream=None):
    """RMSNorm of the rows of x ([m][hidden] bf16) with a bf16 weight."""
    import torch
    m, h = x.shape
    if y is None:
        y = torch.empty_like(x)
    dt = torch.bfloat16
    _check(lib().rbkv_rmsnorm_bf16(_dev_ptr(x, "x", dt, (m, h)), _dev_ptr(weight, "weight", dt, (h,)),
                                   _dev_ptr(y, "y", dt, (m, h)), int(m), int(h), float(eps),
                                   _stream(stream)))
    return y


class Router:
    """Routing of requests over independent replicas (host only): the replica
    with the fewest outstanding tokens takes the next request (ties: fewer
    requests held, then the lower index)."""

    def __init__(self, num_replicas: int):
        h = _P()
        _check(lib().rbkv_router_create(int(num_replicas), C.byref(h)))
        self._h = h
        self.num_replicas = int(num_replicas)

    def assign(self, request_id: int, prompt_len: int, output_len: int) -> int:
        out = C.c_int32()
        _check(lib().rbkv_router_assign(self._h, int(request_id), int(prompt_len),
                                        int(output_len), C.byref(out)))
        return int(out.value)

    def progress(self, request_id: int, tokens: int) -> None:
        _check(lib().rbkv_router_progress(self._h, int(request_id), int(tokens)))

    def finish(self, request_id: int) -> None:
        _check(lib().rbkv_router_finish(self._h, int(request_id)))

    def load(self, replica: int) -> int:
        return int(lib().rbkv_router_load(self._h, int(replica)))

    def active(self, replica: int) -> int:
        return int(lib().rbkv_router_active(self._h, int(replica)))

    def close(self) -> None:
        if self._h:
            lib().rbkv_router_destroy(self._h)
            self._h = _P(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


__all__ = ["gemm", "gemm_qkv", "gemm_workspace_bytes", "rmsnorm", "Router", "Frame", "budget_for_latency", "seq_states", "SeqStates", "ragged_attention_noalloc", "kernel_launches", "profile_enable", "profile_reset", "profile_read", "Config", "Composer", "Pass", "PassMeta", "kv_append", "ragged_attention",
           "RbkvError", "NoBlocksError", "lib", "library_path", "SIGNATURES"]
