"""CPU oracle for one Llama-style decode step (decoder stack + LM head).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product decode
path (``persistent_sm_decode_gb300``) never imports it, and the two share no
code; both read their inputs from ``synth``.

The arithmetic lives in ``oracle.c`` (plain loops, IEEE double, bf16
rounding only where the decode step defines it); this module only
marshals arguments.  Every function of ``oracle.c`` is pinned by
``tests/test_oracle_*.py`` against closed forms, library routines and
brute-force formulations that are independent of it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_SO_F32 = os.path.join(_HERE, "liboracle_f32.so")
_lock = threading.Lock()
_lib = None

c_i32, c_dbl, vp = ctypes.c_int32, ctypes.c_double, ctypes.c_void_p


class OrcConfig(ctypes.Structure):
    _fields_ = [("n_layers", c_i32), ("hidden", c_i32), ("n_heads", c_i32), ("n_kv_heads", c_i32),
                ("head_dim", c_i32), ("intermediate", c_i32), ("vocab", c_i32),
                ("weight_int8", c_i32), ("lm_head_int8", c_i32),
                ("rms_eps", c_dbl), ("rope_theta", c_dbl),
                ("weight_int4", c_i32), ("lm_head_int4", c_i32), ("group_size", c_i32)]


class OrcLayer(ctypes.Structure):
    _fields_ = [(n, vp) for n in ("attn_norm", "mlp_norm", "wq", "wk", "wv", "wo", "wg", "wu", "wd",
                                  "sq", "sk", "sv", "so", "sg", "su", "sd")]


class OrcWeights(ctypes.Structure):
    _fields_ = [("embed", vp), ("final_norm", vp), ("lm_head", vp), ("s_lm", vp),
                ("layers", ctypes.POINTER(OrcLayer))]


def build(force: bool = False, fp32_accumulation: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc -O3, OpenMP, no fast-math).
    fp32_accumulation builds liboracle_f32.so instead (see ORC_ACC_FLOAT in
    oracle.c): a measuring stick for rounding sensitivity, not the oracle."""
    so = _SO_F32 if fp32_accumulation else _SO
    if force or not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(_SRC):
        tmp = so + ".%d.tmp" % os.getpid()
        flags = ["-DORC_ACC_FLOAT"] if fp32_accumulation else []
        subprocess.check_call(["gcc", "-O3", "-fopenmp", "-fPIC", "-shared"] + flags + [_SRC, "-o", tmp, "-lm"])
        os.replace(tmp, so)
    return so


_lib_f32 = None


def lib_fp32_accumulation():
    """The ORC_ACC_FLOAT build (GEMV partial sums rounded to float)."""
    global _lib_f32
    with _lock:
        if _lib_f32 is None:
            _lib_f32 = load(build(fp32_accumulation=True))
    return _lib_f32


def load(path: str):
    """Load an oracle build and declare its signatures."""
    L = ctypes.CDLL(path)
    L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.orc_bf16_to_double.restype = c_dbl
    L.orc_double_to_bf16.argtypes = [c_dbl]
    L.orc_double_to_bf16.restype = ctypes.c_uint16
    L.orc_round_bf16.argtypes = [c_dbl]
    L.orc_round_bf16.restype = c_dbl
    L.orc_rmsnorm.argtypes = [ctypes.c_int, vp, vp, c_dbl, vp]
    L.orc_rmsnorm.restype = None
    L.orc_gemv.argtypes = [ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]
    L.orc_gemv.restype = None
    L.orc_gemv_int4.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]
    L.orc_gemv_int4.restype = None
    L.orc_rope.argtypes = [ctypes.c_int, ctypes.c_int, c_dbl, vp]
    L.orc_rope.restype = None
    L.orc_attention.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp]
    L.orc_attention.restype = None
    L.orc_silu.argtypes = [c_dbl]
    L.orc_silu.restype = c_dbl
    L.orc_argmax.argtypes = [ctypes.c_int, vp]
    L.orc_argmax.restype = ctypes.c_int
    L.orc_num_threads.restype = ctypes.c_int
    L.orc_set_num_threads.argtypes = [ctypes.c_int]
    L.orc_set_num_threads.restype = None
    L.orc_decode_step.argtypes = [ctypes.POINTER(OrcConfig), ctypes.POINTER(OrcWeights),
                                  ctypes.c_int, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp]
    L.orc_decode_step.restype = ctypes.c_int
    L.orc_layer_forward.argtypes = [ctypes.POINTER(OrcConfig), ctypes.POINTER(OrcLayer), ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp]
    L.orc_layer_forward.restype = ctypes.c_int
    L.orc_lm_head.argtypes = [ctypes.POINTER(OrcConfig), ctypes.POINTER(OrcWeights), vp, vp]
    L.orc_lm_head.restype = None
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


def use_library(L) -> None:
    """Point this module at another oracle build (the mutation tests use this to
    check that the pins catch planted mistakes); ``None`` restores the default."""
    global _lib
    with _lock:
        _lib = L


def _p(a: Optional[np.ndarray]) -> Optional[int]:
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


# ------------------------------------------------------------- operators

def bf16_to_double(bits: int) -> float:
    return lib().orc_bf16_to_double(int(bits))


def double_to_bf16(y: float) -> int:
    return int(lib().orc_double_to_bf16(float(y)))


def rmsnorm(x: np.ndarray, gain_bits: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = np.ascontiguousarray(gain_bits, dtype=np.uint16)
    y = np.empty_like(x)
    lib().orc_rmsnorm(x.size, _p(x), _p(g), eps, _p(y))
    return y


def gemv(W: np.ndarray, h_bits: np.ndarray, scales: Optional[np.ndarray] = None) -> np.ndarray:
    W = np.ascontiguousarray(W)
    h = np.ascontiguousarray(h_bits, dtype=np.uint16)
    rows, K = W.shape
    assert h.size == K
    i8 = W.dtype == np.int8
    if i8:
        assert scales is not None and scales.size == rows
        scales = np.ascontiguousarray(scales, dtype=np.float32)
    else:
        assert W.dtype == np.uint16
    y = np.empty(rows, dtype=np.float64)
    lib().orc_gemv(rows, K, _p(W), int(i8), _p(scales), _p(h), _p(y))
    return y


def gemv_int4(W_packed: np.ndarray, h_bits: np.ndarray, scales: np.ndarray, group: int) -> np.ndarray:
    """y = W h for 4-bit codes (two per byte, element 2j in the low nibble of
    byte j; value = scale * (code - 8)) with one scale per `group` weights
    along K (scales [rows][K / group])."""
    W = np.ascontiguousarray(W_packed, dtype=np.uint8)
    h = np.ascontiguousarray(h_bits, dtype=np.uint16)
    rows, K = W.shape[0], 2 * W.shape[1]
    assert h.size == K and K % group == 0
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    assert sc.shape == (rows, K // group)
    y = np.empty(rows, dtype=np.float64)
    lib().orc_gemv_int4(rows, K, group, _p(W), _p(sc), _p(h), _p(y))
    return y


def rope(u: np.ndarray, pos: int, theta: float) -> np.ndarray:
    u = np.array(u, dtype=np.float64, copy=True)
    lib().orc_rope(u.size, pos, theta, _p(u))
    return u


def attention(q: np.ndarray, Kc_bits: np.ndarray, Vc_bits: np.ndarray):
    """Returns (softmax weights [n], output [d]) for one query over n cached rows."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(Kc_bits, dtype=np.uint16)
    Vb = np.ascontiguousarray(Vc_bits, dtype=np.uint16)
    n, d = K.shape
    w = np.empty(max(n, 1), dtype=np.float64)
    o = np.empty(d, dtype=np.float64)
    lib().orc_attention(n, d, _p(q), _p(K), _p(Vb), _p(w), _p(o))
    return w[:n], o


def silu(z: float) -> float:
    return lib().orc_silu(float(z))


def argmax(v: np.ndarray) -> int:
    v = np.ascontiguousarray(v, dtype=np.float64)
    return int(lib().orc_argmax(v.size, _p(v)))


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# ------------------------------------------------------------- whole step

class Oracle:
    """Runs decode steps of a ``synth.HostModel`` on the CPU.

    The oracle owns a private copy of the KV cache (``kc``, ``vc``), so the
    caller's cache is never touched."""

    def __init__(self, model, kc: np.ndarray, vc: np.ndarray, library=None):
        self._L = library
        wl = model.wl
        self.model = model
        self.wl = wl
        self.kc = np.array(kc, copy=True)
        self.vc = np.array(vc, copy=True)
        self.Bmax = self.kc.shape[1]
        self.Smax = self.kc.shape[3]
        i8 = wl.weight_dtype == "int8"
        i4 = wl.weight_dtype == "int4"
        self.cfg = OrcConfig(wl.n_layers, wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim,
                             wl.intermediate, wl.vocab, int(i8), int(i8 and not wl.tied),
                             wl.rms_eps, wl.rope_theta, int(i4), int(i4 and not wl.tied),
                             getattr(wl, "group_size", 128))
        n = wl.n_layers
        self._layers = (OrcLayer * n)()
        for l, hl in enumerate(model.layers):
            s = hl.scales or {}
            self._layers[l] = OrcLayer(_p(hl.attn_norm), _p(hl.mlp_norm), _p(hl.wq), _p(hl.wk), _p(hl.wv),
                                       _p(hl.wo), _p(hl.w_gate), _p(hl.w_up), _p(hl.w_down),
                                       _p(s.get("s_q")), _p(s.get("s_k")), _p(s.get("s_v")), _p(s.get("s_o")),
                                       _p(s.get("s_gate")), _p(s.get("s_up")), _p(s.get("s_down")))
        self.w = OrcWeights(_p(model.embed), _p(model.final_norm), _p(model.lm_head), _p(model.lm_scale),
                            self._layers)

    def step(self, tokens, positions, trace: bool = False):
        """One decode step; returns logits [B, V] (float64), and the residual trace
        [B, L+1, H] if ``trace``."""
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        B = tok.size
        assert pos.size == B
        logits = np.empty((B, self.wl.vocab), dtype=np.float64)
        xt = np.empty((B, self.wl.n_layers + 1, self.wl.hidden), dtype=np.float64) if trace else None
        rc = (self._L or lib()).orc_decode_step(ctypes.byref(self.cfg), ctypes.byref(self.w), B, _p(tok), _p(pos),
                                   _p(self.kc), _p(self.vc), self.Bmax, self.Smax, _p(logits), _p(xt))
        if rc != 0:
            raise ValueError("oracle rejected the step arguments")
        return (logits, xt) if trace else logits


def _layer(self, l: int, b: int, p: int, x: np.ndarray):
    """Layer l of sequence b at position p from residual x (float64 [H]), against
    this oracle's caches (slot p of layer l is written).  Returns (x_mid, x_out)."""
    xo = np.array(x, dtype=np.float64, copy=True)
    xm = np.empty_like(xo)
    rc = (self._L or lib()).orc_layer_forward(ctypes.byref(self.cfg), ctypes.byref(self._layers[l]), l, b, p, _p(xo),
                                 _p(self.kc), _p(self.vc), self.Bmax, self.Smax, _p(xm))
    if rc != 0:
        raise ValueError("oracle rejected the layer arguments")
    return xm, xo


def _lm_head(self, x: np.ndarray) -> np.ndarray:
    """Final norm and LM head from residual x (float64 [H])."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(self.wl.vocab, dtype=np.float64)
    (self._L or lib()).orc_lm_head(ctypes.byref(self.cfg), ctypes.byref(self.w), _p(x), _p(out))
    return out


Oracle.layer = _layer
Oracle.lm_head = _lm_head


def greedy(logits: np.ndarray):
    """Per row: (argmax with lowest index on ties, top-1 minus top-2 margin)."""
    out, margins = [], []
    for row in np.atleast_2d(logits):
        i = argmax(row)
        top2 = np.partition(row, -2)[-2:]
        out.append(i)
        margins.append(float(top2[1] - top2[0]))
    return np.array(out, dtype=np.int32), np.array(margins)
