"""GB300-native single-launch decode MegaKernel (sm_103a).

One ``DecodeEngine.step`` runs a whole decode step of a Llama-style decoder
stack plus LM head as a single persistent-kernel launch (the MegaKernel of the
Ada-MK technical summary, gist.science, Problem Statement and Methodology).
This module is the thin Python binding of the C ABI in ``include/amk.h``:
it marshals arguments (torch tensors are used only as device memory and
streams) and calls ``libamk.so``.  Every step of the decode path runs in the
library's CUDA kernel; there is no Python or CPU fallback, and the binding
raises if the library is missing or rejects a call.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Dict, List, Optional, Sequence

from . import _build

__all__ = ["AmkError", "Config", "ScheduleOptions", "DecodeEngine", "UnfusedEngine", "Plan", "lib", "build",
           "chrome_trace",
           "level_times",
           "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_CUDA", "ERR_OOM", "ERR_SCHEDULE",
           "ERR_COOPERATIVE", "ERR_TIMEOUT", "WEIGHT_BF16", "WEIGHT_INT8", "WEIGHT_INT4"]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_SCHEDULE, ERR_COOPERATIVE, ERR_TIMEOUT = range(8)
WEIGHT_BF16, WEIGHT_INT8, WEIGHT_INT4 = 0, 1, 2
OPS = ("QKV", "ATT", "OPR", "GUP", "DWN", "LMH", "MRG", "ARG")

i32, i64, f32, f64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_void_p


class Config(ctypes.Structure):
    _fields_ = [("n_layers", i32), ("hidden", i32), ("n_heads", i32), ("n_kv_heads", i32), ("head_dim", i32),
                ("intermediate", i32), ("vocab", i32), ("rms_eps", f32), ("rope_theta", f32),
                ("max_batch", i32), ("max_seq", i32), ("weight_dtype", i32), ("tied_embeddings", i32),
                ("group_size", i32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, vp) for n in ("attn_norm", "mlp_norm", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down",
                                  "s_q", "s_k", "s_v", "s_o", "s_gate", "s_up", "s_down")]


class Weights(ctypes.Structure):
    _fields_ = [("embed", vp), ("final_norm", vp), ("lm_head", vp), ("s_lm", vp),
                ("layers", ctypes.POINTER(LayerWeights))]


class ScheduleOptions(ctypes.Structure):
    _fields_ = [("n_sm", i32), ("att_chunks", i32), ("slot_bytes", i32), ("n_slots", i32), ("ksplit", i32),
                ("scratch_depth", i32), ("l2_prefetch_kb", i32), ("trace", i32), ("wait_timeout_ns", i64),
                ("l2_evict_first", i32), ("task_order", i32)]


class ErrorInfo(ctypes.Structure):
    _fields_ = [("code", i32), ("sm", i32), ("task", i32), ("counter", i32), ("observed", ctypes.c_uint32),
                ("target", ctypes.c_uint32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, i32) for n in ("n_sm", "n_tasks", "n_counters", "n_levels", "att_chunks", "slot_bytes",
                                   "n_slots", "ksplit", "scratch_depth", "att_tile", "smem_bytes",
                                   "max_tasks_per_sm")] + \
               [("weight_bytes", i64), ("scratch_bytes", i64), ("modeled_us", f64), ("search_ms", f64),
                ("candidates", i32), ("l2_evict_first", i32), ("simulated_us", f64), ("task_order", i32)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


class AmkError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, lib().amk_status_string(status).decode(), status))


_lock = threading.Lock()
_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libamk.so (nvcc, sm_103a) in-tree."""
    return _build.build(force=force, verbose=verbose)


def lib():
    """The loaded C library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError("libamk.so is not built; run persistent_sm_decode_gb300.build() "
                                   "(there is no fallback path)")
            L = ctypes.CDLL(_build.LIB)
            L.amk_status_string.argtypes = [ctypes.c_int]
            L.amk_status_string.restype = ctypes.c_char_p
            L.amk_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights),
                                     ctypes.POINTER(ScheduleOptions), ctypes.POINTER(vp)]
            L.amk_decode_step.argtypes = [vp, i32, vp, vp, vp, vp, vp]
            L.amk_decode_step_greedy.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp]
            L.amk_decode_step_noalloc.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), i32, vp, vp,
                                                  vp, vp, vp]
            L.amk_sync_status.argtypes = [vp]
            L.amk_destroy.argtypes = [vp]
            L.amk_last_error.argtypes = [vp, ctypes.POINTER(ErrorInfo)]
            L.amk_get_plan_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
            L.amk_debug_drop_signal.argtypes = [vp, i32, i32]
            L.amk_debug_read_residuals.argtypes = [vp, vp, vp]
            L.amk_debug_read_trace.argtypes = [vp, vp, ctypes.c_size_t]
            L.amk_plan_build.argtypes = [ctypes.POINTER(Config), i32, i32, i32, ctypes.POINTER(ScheduleOptions),
                                         ctypes.POINTER(vp)]
            L.amk_plan_validate.argtypes = [vp, ctypes.c_char_p, ctypes.c_size_t]
            L.amk_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
            L.amk_plan_num_tasks.argtypes = [vp, i32]
            L.amk_plan_num_tasks.restype = i32
            L.amk_plan_get_task.argtypes = [vp, i32, i32, ctypes.POINTER(i32)]
            L.amk_plan_mutate.argtypes = [vp, i32, ctypes.c_uint64]
            L.amk_plan_last_message.restype = ctypes.c_char_p
            L.amk_plan_simulate.argtypes = [vp, ctypes.POINTER(f64), i32, ctypes.POINTER(f64)]
            L.amk_plan_simulate.restype = ctypes.c_int
            L.amk_plan_destroy.argtypes = [vp]
            L.amk_plan_destroy.restype = None
            L.amk_unfused_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), ctypes.POINTER(vp)]
            L.amk_unfused_decode_step.argtypes = [vp, i32, vp, vp, vp, vp, vp]
            L.amk_unfused_destroy.argtypes = [vp]
            for f in ("amk_create", "amk_decode_step", "amk_decode_step_greedy", "amk_decode_step_noalloc", "amk_sync_status", "amk_destroy", "amk_last_error",
                      "amk_get_plan_info", "amk_debug_drop_signal", "amk_debug_read_residuals", "amk_debug_read_trace", "amk_plan_build", "amk_plan_validate",
                      "amk_plan_get_info", "amk_plan_get_task", "amk_plan_mutate", "amk_unfused_create",
                      "amk_unfused_decode_step", "amk_unfused_destroy"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != OK:
        raise AmkError(status, what)


def _options(opts: Optional[dict]) -> Optional[ScheduleOptions]:
    if not opts:
        return None
    o = ScheduleOptions()
    for k, v in opts.items():
        setattr(o, k, int(v))
    return o


def make_config(n_layers, hidden, n_heads, n_kv_heads, head_dim, intermediate, vocab, max_seq, max_batch=1,
                rms_eps=1e-5, rope_theta=1e4, int8=False, tied=False, int4=False, group_size=0) -> Config:
    wd = WEIGHT_INT4 if int4 else WEIGHT_INT8 if int8 else WEIGHT_BF16
    return Config(n_layers, hidden, n_heads, n_kv_heads, head_dim, intermediate, vocab, rms_eps, rope_theta,
                  max_batch, max_seq, wd, int(bool(tied)), int(group_size))


# --------------------------------------------------------------- planner

class Plan:
    """The offline schedule (DAG, search, solidified per-CTA tables, validator)
    built on the host without a GPU."""

    def __init__(self, cfg: Config, batch: int, n_sm: int, smem_per_cta: int = 232448, options=None):
        self._p = vp()
        o = _options(options)
        st = lib().amk_plan_build(ctypes.byref(cfg), batch, n_sm, smem_per_cta,
                                  ctypes.byref(o) if o else None, ctypes.byref(self._p))
        if st != OK:
            raise AmkError(st, "amk_plan_build: " + lib().amk_plan_last_message().decode())
        self.n_sm = n_sm

    def info(self) -> dict:
        pi = PlanInfo()
        _check(lib().amk_plan_get_info(self._p, ctypes.byref(pi)), "amk_plan_get_info")
        return pi.as_dict()

    def validate(self):
        buf = ctypes.create_string_buffer(512)
        st = lib().amk_plan_validate(self._p, buf, 512)
        return st, buf.value.decode()

    def tasks(self, sm: int) -> List[dict]:
        out = []
        n = lib().amk_plan_num_tasks(self._p, sm)
        arr = (i32 * 16)()
        for i in range(n):
            _check(lib().amk_plan_get_task(self._p, sm, i, arr), "amk_plan_get_task")
            v = list(arr)
            out.append({"op": OPS[v[0]], "layer": v[1], "r0": v[2], "r1": v[3], "b": v[4], "g": v[5],
                        "wait": v[6], "wait_count": v[7], "sig": v[9:9 + v[8]], "mat": v[15]})
        return out

    def simulate(self, consts: Optional[Sequence[float]] = None) -> float:
        """The task-level simulation's step time (µs) under the built-in cost
        constants, or under `consts` (15 values; see amk_plan_simulate)."""
        out = f64()
        arr = None if consts is None else (f64 * len(consts))(*consts)
        _check(lib().amk_plan_simulate(self._p, arr, 0 if consts is None else len(consts), ctypes.byref(out)),
               "amk_plan_simulate")
        return out.value

    def mutate(self, kind: int, seed: int) -> int:
        return lib().amk_plan_mutate(self._p, kind, seed)

    def close(self):
        if self._p:
            lib().amk_plan_destroy(self._p)
            self._p = vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# --------------------------------------------------------------- engine

_LAYER_KEYS = ("attn_norm", "mlp_norm", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")
_SCALE_KEYS = ("s_q", "s_k", "s_v", "s_o", "s_gate", "s_up", "s_down")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("weights and buffers must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("weights and buffers must be contiguous")
    return t.data_ptr()


class DecodeEngine:
    """A created amk handle plus references to the device tensors it reads.

    ``layers`` is a list of dicts with keys attn_norm, mlp_norm, wq, wk, wv, wo,
    w_gate, w_up, w_down (and s_q ... s_down for int8 weights); every matrix is
    [out, in] row-major on the current CUDA device."""

    def __init__(self, cfg: Config, embed, final_norm, layers: Sequence[Dict], lm_head=None, s_lm=None,
                 options: Optional[dict] = None):
        self.cfg = cfg
        self._keep = [embed, final_norm, lm_head, s_lm] + [v for d in layers for v in d.values()]
        arr = (LayerWeights * cfg.n_layers)()
        for l, d in enumerate(layers):
            for k in _LAYER_KEYS + _SCALE_KEYS:
                setattr(arr[l], k, _ptr(d.get(k)))
        self._arr = arr
        w = Weights(_ptr(embed), _ptr(final_norm), _ptr(lm_head), _ptr(s_lm), arr)
        o = _options(options)
        self._h = vp()
        st = lib().amk_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(o) if o else None,
                              ctypes.byref(self._h))
        _check(st, "amk_create")

    @property
    def handle(self) -> int:
        return self._h.value

    def step(self, tokens, positions, kv_cache, logits, stream=None, batch: Optional[int] = None) -> None:
        """Enqueue one decode step (device int32 tokens/positions [B], bf16 KV
        cache [2][L][Bmax][nkv][Smax][d], fp32 logits [B][V])."""
        B = int(tokens.numel()) if batch is None else int(batch)
        s = None if stream is None else (stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
        st = lib().amk_decode_step(self._h, B, _ptr(tokens), _ptr(positions), _ptr(kv_cache), _ptr(logits), s)
        _check(st, "amk_decode_step")

    def step_greedy(self, tokens, positions, kv_cache, logits, next_tokens, next_positions, stream=None,
                    batch: Optional[int] = None) -> None:
        """Enqueue one decode step that also writes each sequence's greedy
        token (argmax of its logits, lowest index on ties) to next_tokens and
        positions + 1 to next_positions (device int32 [B], not aliasing the
        inputs)."""
        B = int(tokens.numel()) if batch is None else int(batch)
        s = None if stream is None else (stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
        st = lib().amk_decode_step_greedy(self._h, B, _ptr(tokens), _ptr(positions), _ptr(kv_cache), _ptr(logits),
                                          _ptr(next_tokens), _ptr(next_positions), s)
        _check(st, "amk_decode_step_greedy")

    def greedy_graph(self, tokens, positions, kv_cache, logits):
        """A CUDA graph of two greedy steps that ping-pong between (tokens,
        positions) and a second pair of device buffers: each replay decodes two
        tokens per sequence with no host involvement.  Returns (graph,
        (tokens_b, positions_b)); after a replay the latest inputs are back in
        (tokens, positions).  The buffers must stay alive with the graph."""
        import torch
        tb, pb = torch.empty_like(tokens), torch.empty_like(positions)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.step_greedy(tokens, positions, kv_cache, logits, tb, pb, stream=s)
            self.step_greedy(tb, pb, kv_cache, logits, tokens, positions, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        return g, (tb, pb)

    def step_raw(self, batch: int, tokens: int, positions: int, kv_cache: int, logits: int, stream: int = 0) -> int:
        """The same call with raw device addresses; returns the status."""
        return lib().amk_decode_step(self._h, batch, tokens, positions, kv_cache, logits, stream or None)

    def sync(self) -> int:
        return lib().amk_sync_status(self._h)

    def last_error(self) -> dict:
        e = ErrorInfo()
        lib().amk_last_error(self._h, ctypes.byref(e))
        return {k: getattr(e, k) for k, _ in ErrorInfo._fields_}

    def plan_info(self) -> dict:
        pi = PlanInfo()
        _check(lib().amk_get_plan_info(self._h, ctypes.byref(pi)), "amk_get_plan_info")
        return pi.as_dict()

    def drop_signal(self, sm: int, task: int) -> None:
        _check(lib().amk_debug_drop_signal(self._h, sm, task), "amk_debug_drop_signal")

    def read_residuals(self):
        """(x_in [L+1][Bmax][H], x_mid [L][Bmax][H]) of the last step as numpy
        float32; needs options={"scratch_depth": n_layers + 1}."""
        import numpy as np
        L, B, H = self.cfg.n_layers, self.cfg.max_batch, self.cfg.hidden
        xi = np.empty((L + 1, B, H), dtype=np.float32)
        xm = np.empty((L, B, H), dtype=np.float32)
        _check(lib().amk_debug_read_residuals(self._h, xi.ctypes.data, xm.ctypes.data), "amk_debug_read_residuals")
        return xi, xm

    def read_trace(self):
        """[n_tasks][16] timestamps and durations (ns) of the last step, tasks
        in CTA order; see amk_debug_read_trace.  Needs a handle created with
        options={"trace": 1} on the library built with AMK_TRACE=1 (the
        default build leaves the timing code out and refuses the option).
        chrome_trace and level_times turn the result into a timeline."""
        import numpy as np
        n = self.plan_info()["n_tasks"]
        out = np.zeros((n, 16), dtype=np.uint64)
        _check(lib().amk_debug_read_trace(self._h, out.ctypes.data, out.size), "amk_debug_read_trace")
        return out

    def close(self) -> None:
        if self._h:
            lib().amk_destroy(self._h)
            self._h = vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def chrome_trace(trace, plan: "Plan") -> dict:
    """Chrome trace-event JSON (chrome://tracing, ui.perfetto.dev) of one
    traced decode step: one track per CTA, one slice per task, with its
    inputs-and-prologue, tiles and epilogue nested inside; times in µs from
    the first task's start.

    ``trace`` is ``DecodeEngine.read_trace()`` of a handle created with
    ``options={"trace": 1}`` on the AMK_TRACE=1 build; ``plan`` is the host
    ``Plan`` of the same configuration, batch (the config's max_batch), CTA
    count and options.  The planner is deterministic, so its task tables are
    the handle's, row for row."""
    rows = iter(trace)
    t0 = min((int(r[0]) for r in trace if int(r[0]) > 0), default=0)
    us = lambda t: (int(t) - t0) / 1e3
    ev = [{"name": "process_name", "ph": "M", "pid": 0, "args": {"name": "amk_decode_kernel"}}]
    for sm in range(plan.n_sm):
        ev.append({"name": "thread_name", "ph": "M", "pid": 0, "tid": sm, "args": {"name": "CTA %d" % sm}})
        for t in plan.tasks(sm):
            r = next(rows)
            start, end = int(r[0]), int(r[3])
            if start == 0 or end < start:
                continue
            name = "%s L%d" % (t["op"], t["layer"]) + (" c%d" % t["r0"] if t["op"] == "ATT" else "")
            ev.append({"name": name, "ph": "X", "pid": 0, "tid": sm, "ts": us(start), "dur": (end - start) / 1e3,
                       "args": {"rows": [t["r0"], t["r1"]], "seq": t["b"], "head": t["g"],
                                "tile_wait_us": int(r[4]) / 1e3, "tile_us": int(r[5]) / 1e3,
                                "loader_wait_us": int(r[9]) / 1e3}})
            pro, last, epi = int(r[6]), int(r[7]), int(r[8])
            for part, a, b in (("inputs + prologue", start, pro), ("tiles", pro, last), ("epilogue", last, epi)):
                if a >= start and b >= a and b <= end and a > 0:
                    ev.append({"name": part, "ph": "X", "pid": 0, "tid": sm, "ts": us(a), "dur": (b - a) / 1e3})
    return {"traceEvents": ev, "displayTimeUnit": "ns"}


def level_times(trace, plan: "Plan") -> List[dict]:
    """Per dependency level of a traced step, in program order: the level's
    last task end, and its time from the previous level's last task end
    (the critical-path share of that level).  Arguments as for chrome_trace."""
    rows = iter(trace)
    ends: Dict[tuple, int] = {}
    starts: Dict[tuple, int] = {}
    for sm in range(plan.n_sm):
        for t in plan.tasks(sm):
            r = next(rows)
            if int(r[0]) == 0:
                continue
            key = (t["layer"], t["op"])
            ends[key] = max(ends.get(key, 0), int(r[3]))
            starts[key] = min(starts.get(key, 1 << 63), int(r[0]))
    order = {op: i for i, op in enumerate(("QKV", "ATT", "MRG", "OPR", "GUP", "DWN", "LMH", "ARG"))}
    keys = sorted(ends, key=lambda k: (k[0] + (1 if k[1] in ("LMH", "ARG") else 0), order[k[1]]))
    out, prev = [], None
    for k in keys:
        base = prev if prev is not None else starts[k]
        out.append({"layer": k[0], "op": k[1], "end_ns": ends[k], "level_us": (ends[k] - base) / 1e3})
        prev = ends[k]
    return out


_PRODUCER = {"ATT": "QKV", "MRG": "ATT", "OPR": "MRG", "GUP": "OPR", "DWN": "GUP"}


def prologue_lag(trace, plan: "Plan", layer: int) -> List[dict]:
    """For every operator of one layer of a traced step, when its tasks got
    their inputs: the end of each task's inputs-and-prologue phase minus
    the end of the last task of the level it reads (the previous layer's
    down projection for QKV, the merge level for the O projection, or the
    attention level where a step has no merge tasks), as min / median / max
    over the operator's tasks, in µs; and the median durations of its
    prologue, tiles and epilogue phases.  A lag near the prologue's own
    duration means the inputs were ready when the task began; a long lag
    after every producer has finished is the prologue's own cost.
    Arguments as for chrome_trace; ``layer`` >= 1."""
    rows = iter(trace)
    ends: Dict[tuple, int] = {}
    tasks: Dict[str, List[tuple]] = {}
    for sm in range(plan.n_sm):
        for t in plan.tasks(sm):
            r = [int(v) for v in next(rows)]
            if r[0] == 0:
                continue
            key = (t["layer"], t["op"])
            ends[key] = max(ends.get(key, 0), r[3])
            if t["layer"] == layer:
                tasks.setdefault(t["op"], []).append(r)

    def med(v: List[float]) -> float:
        v = sorted(v)
        return (v[(len(v) - 1) // 2] + v[len(v) // 2]) / 2 if v else float("nan")

    out = []
    for op in ("QKV", "ATT", "MRG", "OPR", "GUP", "DWN"):
        if op not in tasks:
            continue
        src = (layer - 1, "DWN") if op == "QKV" else (layer, _PRODUCER[op])
        if src not in ends and op == "OPR":
            src = (layer, "ATT")
        if src not in ends:
            continue
        lag = [(r[6] - ends[src]) / 1e3 for r in tasks[op] if r[6] >= r[0] > 0]
        out.append({"op": op, "after": src[1], "tasks": len(tasks[op]),
                    "lag_min_us": min(lag), "lag_median_us": med(lag), "lag_max_us": max(lag),
                    "prologue_us": med([(r[6] - r[0]) / 1e3 for r in tasks[op]]),
                    "tiles_us": med([(r[7] - r[6]) / 1e3 for r in tasks[op]]),
                    "epilogue_us": med([(r[8] - r[7]) / 1e3 for r in tasks[op]])})
    return out


class UnfusedEngine:
    """The same decode step as one kernel launch per operator
    (include/amk_unfused.h), for comparison with DecodeEngine on the same
    device and data.  Arguments as for DecodeEngine; ``step`` as
    DecodeEngine.step."""

    def __init__(self, cfg: Config, embed, final_norm, layers: Sequence[Dict], lm_head=None, s_lm=None):
        self.cfg = cfg
        self._keep = [embed, final_norm, lm_head, s_lm] + [v for d in layers for v in d.values()]
        arr = (LayerWeights * cfg.n_layers)()
        for l, d in enumerate(layers):
            for k in _LAYER_KEYS + _SCALE_KEYS:
                setattr(arr[l], k, _ptr(d.get(k)))
        self._arr = arr
        w = Weights(_ptr(embed), _ptr(final_norm), _ptr(lm_head), _ptr(s_lm), arr)
        self._h = vp()
        _check(lib().amk_unfused_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(self._h)),
               "amk_unfused_create")

    def step(self, tokens, positions, kv_cache, logits, stream=None, batch: Optional[int] = None) -> None:
        B = int(tokens.numel()) if batch is None else int(batch)
        s = None if stream is None else (stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
        _check(lib().amk_unfused_decode_step(self._h, B, _ptr(tokens), _ptr(positions), _ptr(kv_cache),
                                             _ptr(logits), s), "amk_unfused_decode_step")

    def close(self) -> None:
        if self._h:
            lib().amk_unfused_destroy(self._h)
            self._h = vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def decode_step_noalloc(cfg: Config, embed, final_norm, layers: Sequence[Dict], tokens, positions, kv_cache,
                        logits, lm_head=None, s_lm=None, stream=None, batch: Optional[int] = None) -> int:
    """One decode step through amk_decode_step_noalloc, which keeps all of its
    device state in a static array and allocates nothing (for callers that
    cannot allocate device memory).  Arguments as for DecodeEngine and
    DecodeEngine.step; waits for the step and returns the amk status."""
    arr = (LayerWeights * cfg.n_layers)()
    for l, d in enumerate(layers):
        for k in _LAYER_KEYS + _SCALE_KEYS:
            setattr(arr[l], k, _ptr(d.get(k)))
    w = Weights(_ptr(embed), _ptr(final_norm), _ptr(lm_head), _ptr(s_lm), arr)
    B = int(tokens.numel()) if batch is None else int(batch)
    s = None if stream is None else (stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    return lib().amk_decode_step_noalloc(ctypes.byref(cfg), ctypes.byref(w), B, _ptr(tokens), _ptr(positions),
                                         _ptr(kv_cache), _ptr(logits), s)
