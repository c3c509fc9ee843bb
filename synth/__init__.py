"""Seeded synthetic inputs for the decode-step workloads.

Both the CUDA decode path and the CPU oracle take their inputs from here, and
this package holds none of the decode step's arithmetic: it draws weights,
the prefilled KV cache and the first tokens, and decodes bf16 bit patterns for
display.  The draws are made by ``synth.c`` (splitmix64 streams keyed by
tensor name, Box-Muller normals); see that file for the definitions.

Workload shapes follow the Llama-family decoders that the AutoMegaKernel
abstract compiles (SmolLM2-135M, TinyLlama-1.1B, W8A16) plus a Llama-2-7B
shape; every model here is random-init, never a trained checkpoint.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, replace
from typing import Dict, List, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libsynth.so next to its source (gcc, OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            u64, i64, c_d, c_i = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_int
            vp, cp = ctypes.c_void_p, ctypes.c_char_p
            L.synth_name_hash.argtypes = [cp]
            L.synth_name_hash.restype = u64
            L.synth_normal_bf16.argtypes = [u64, cp, c_d, c_d, u64, vp, i64]
            L.synth_normal_f32.argtypes = [u64, cp, c_d, c_d, u64, vp, i64]
            L.synth_uniform_i8.argtypes = [u64, cp, u64, vp, i64]
            L.synth_uniform_u4.argtypes = [u64, cp, u64, vp, i64]
            L.synth_scales_f32.argtypes = [u64, cp, c_d, c_d, vp, i64]
            L.synth_raw_u64.argtypes = [u64, cp, u64, vp, i64]
            L.synth_kv_cache.argtypes = [u64, c_i, c_i, c_i, c_i, c_i, c_i, vp, vp]
            L.synth_splitmix64_seq.argtypes = [u64, i64, vp]
            for f in ("synth_normal_bf16", "synth_normal_f32", "synth_uniform_i8", "synth_uniform_u4",
                      "synth_scales_f32", "synth_raw_u64", "synth_kv_cache", "synth_splitmix64_seq"):
                getattr(L, f).restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- raw draws

def normal_bf16(seed: int, name: str, shape, std: float = 1.0, mean: float = 0.0, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    lib().synth_normal_bf16(seed, name.encode(), mean, std, offset, _ptr(out), out.size)
    return out


def normal_f32(seed: int, name: str, shape, std: float = 1.0, mean: float = 0.0, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    lib().synth_normal_f32(seed, name.encode(), mean, std, offset, _ptr(out), out.size)
    return out


def uniform_i8(seed: int, name: str, shape, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.int8)
    lib().synth_uniform_i8(seed, name.encode(), offset, _ptr(out), out.size)
    return out


def uniform_u4(seed: int, name: str, shape, offset: int = 0) -> np.ndarray:
    """4-bit codes uniform in [1, 15], packed two per byte (element 2j in the
    low nibble of byte j); `shape` is the unpacked shape, its last dimension even."""
    shape = tuple(shape)
    assert shape[-1] % 2 == 0
    out = np.empty(shape[:-1] + (shape[-1] // 2,), dtype=np.uint8)
    lib().synth_uniform_u4(seed, name.encode(), offset, _ptr(out), int(np.prod(shape)))
    return out


def scales_f32(seed: int, name: str, n: int, base: float, jitter: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().synth_scales_f32(seed, name.encode(), base, jitter, _ptr(out), n)
    return out


def raw_u64(seed: int, name: str, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    lib().synth_raw_u64(seed, name.encode(), offset, _ptr(out), n)
    return out


def splitmix64_seq(state: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    lib().synth_splitmix64_seq(state, n, _ptr(out))
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


BF16_ONE = 0x3F80  # bit pattern of 1.0 in bf16


# ---------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Workload:
    """Shape and data recipe of one synthetic decode workload."""
    name: str
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    ctx: int            # seeded prior positions per sequence; first decode position
    max_seq: int        # KV-cache capacity (Smax)
    steps: int          # greedy decode steps of the workload
    batch: int = 1
    rms_eps: float = 1e-5
    rope_theta: float = 1e4
    tied: bool = False
    weight_dtype: str = "bf16"   # "bf16", "int8" (W8A16) or "int4" (W4A16: 4-bit codes, group scales)
    group_size: int = 128        # int4 only: weights per scale along K
    weight_std: float = 0.02
    scale_jitter: float = 0.0    # int8 only: per-row scale = 0.02/127 * (1 + jitter*U)
    description: str = ""

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    def matrix_bytes(self, rows: int, k: int) -> int:
        """Bytes of one [rows, k] matrix in the workload's weight format, with its scales."""
        if self.weight_dtype == "int8":
            return rows * k + rows * 4
        if self.weight_dtype == "int4":
            return rows * k // 2 + rows * (k // self.group_size) * 4
        return rows * k * 2

    def weight_bytes(self) -> int:
        """Bytes of every linear weight (plus int8 row or int4 group scales) read by one step."""
        H, I, V, d = self.hidden, self.intermediate, self.vocab, self.head_dim
        per_layer_rows_k = [(self.qkv_rows, H), (H, self.n_heads * d), (2 * I, H), (H, I)]
        tot = sum(self.matrix_bytes(rows, k) for rows, k in per_layer_rows_k) * self.n_layers
        # LM head (tied: the bf16 embedding, read once)
        tot += V * H * 2 if self.tied else self.matrix_bytes(V, H)
        tot += (2 * self.n_layers + 1) * H * 2          # norm gains
        return tot

    def kv_read_bytes(self, position: int) -> int:
        """K and V bytes attention reads at one decode position, per sequence (positions 0..p)."""
        return self.n_layers * self.n_kv_heads * (position + 1) * self.head_dim * 2 * 2


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload(
        "tiny", 2, 256, 4, 2, 64, 688, 1024, ctx=16, max_seq=48, steps=32,
        description="tiny Llama-style decoder: 2 layers, hidden 256, 4q/2kv heads d64, inter 688, "
                    "vocab 1024; 16 seeded prior positions; 32 greedy steps"),
    "smollm2_135m": Workload(
        "smollm2_135m", 30, 576, 9, 3, 64, 1536, 49152, ctx=512, max_seq=640, steps=128, tied=True,
        description="SmolLM2-135M-shaped decoder, random init, tied embeddings; context 512; 128 steps"),
    "tinyllama_1b1": Workload(
        "tinyllama_1b1", 22, 2048, 32, 4, 64, 5632, 32000, ctx=2048, max_seq=2176, steps=128,
        description="TinyLlama-1.1B-shaped decoder, random init, bf16; context 2048; 128 steps"),
    "tinyllama_1b1_w8a16": Workload(
        "tinyllama_1b1_w8a16", 22, 2048, 32, 4, 64, 5632, 32000, ctx=1024, max_seq=1152, steps=128,
        weight_dtype="int8",
        description="TinyLlama-1.1B shape, W8A16: int8 weights U[-127,127], per-row scale 0.02/127; "
                    "context 1024; 128 steps"),
    "llama2_7b": Workload(
        "llama2_7b", 32, 4096, 32, 32, 128, 11008, 32000, ctx=4096, max_seq=4160, steps=64,
        description="Llama-2-7B-shaped decoder, random init, bf16, MHA d128; context 4096; 64 steps"),
    "llama2_7b_b8": Workload(
        "llama2_7b_b8", 32, 4096, 32, 32, 128, 11008, 32000, ctx=4096, max_seq=4160, steps=64, batch=8,
        description="Llama-2-7B shape at batch 8, context 4096, 64 steps"),
    "tinyllama_1b1_w4a16": Workload(
        "tinyllama_1b1_w4a16", 22, 2048, 32, 4, 64, 5632, 32000, ctx=1024, max_seq=1152, steps=128,
        weight_dtype="int4",
        description="TinyLlama-1.1B shape, W4A16: 4-bit codes uniform in [1, 15] around zero point 8, one "
                    "fp32 scale 0.02/7 per 128 weights along K; context 1024; 128 steps"),
    "tinyllama_1b1_short": Workload(
        "tinyllama_1b1_short", 22, 2048, 32, 4, 64, 5632, 32000, ctx=64, max_seq=80, steps=12,
        description="TinyLlama-1.1B shape with a short sequence: 64 prompt positions, 12 decode steps; the "
                    "batch-size sweep (1, 2, 4, 8, 16) runs on it"),
}


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


# ---------------------------------------------------------------- host model

@dataclass
class HostLayer:
    attn_norm: np.ndarray   # [H] bf16 bits
    mlp_norm: np.ndarray    # [H] bf16 bits
    wq: np.ndarray          # [nq*d, H]     bf16 bits (uint16) or int8
    wk: np.ndarray          # [nkv*d, H]
    wv: np.ndarray          # [nkv*d, H]
    wo: np.ndarray          # [H, nq*d]
    w_gate: np.ndarray      # [I, H]
    w_up: np.ndarray        # [I, H]
    w_down: np.ndarray      # [H, I]
    scales: Optional[Dict[str, np.ndarray]] = None   # int8 only: per-output-row fp32


@dataclass
class HostModel:
    wl: Workload
    embed: np.ndarray        # [V, H] bf16 bits
    final_norm: np.ndarray   # [H] bf16 bits
    lm_head: np.ndarray      # [V, H] bf16 bits or int8 (tied: same object as embed)
    lm_scale: Optional[np.ndarray]
    layers: List[HostLayer]


_MATS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")
_SCALE_KEY = {"wq": "s_q", "wk": "s_k", "wv": "s_v", "wo": "s_o",
              "w_gate": "s_gate", "w_up": "s_up", "w_down": "s_down"}


def mat_shapes(wl: Workload) -> Dict[str, tuple]:
    H, I, d = wl.hidden, wl.intermediate, wl.head_dim
    return {"wq": (wl.n_heads * d, H), "wk": (wl.n_kv_heads * d, H), "wv": (wl.n_kv_heads * d, H),
            "wo": (H, wl.n_heads * d), "w_gate": (I, H), "w_up": (I, H), "w_down": (H, I)}


def _matrix(wl: Workload, seed: int, name: str, shape):
    if wl.weight_dtype == "int4":
        assert shape[1] % wl.group_size == 0, "K must be a whole number of scale groups"
        q = uniform_u4(seed, name, shape)
        s = scales_f32(seed, name + ".scale", shape[0] * (shape[1] // wl.group_size), wl.weight_std / 7.0,
                       wl.scale_jitter).reshape(shape[0], shape[1] // wl.group_size)
        return q, s
    if wl.weight_dtype == "int8":
        q = uniform_i8(seed, name, shape)
        s = scales_f32(seed, name + ".scale", shape[0], wl.weight_std / 127.0, wl.scale_jitter)
        return q, s
    return normal_bf16(seed, name, shape, std=wl.weight_std), None


def make_model(wl: Workload, seed: int = 1) -> HostModel:
    """All weights of a random-init model.  Norm gains are 1.0; matrices N(0, 0.02) bf16,
    or int8 uniform in [-127, 127] with per-output-row fp32 scales for W8A16.  The
    embedding is bf16 in every case."""
    H, V = wl.hidden, wl.vocab
    ones = np.full(H, BF16_ONE, dtype=np.uint16)
    layers = []
    shapes = mat_shapes(wl)
    for l in range(wl.n_layers):
        mats, scales = {}, {}
        for m in _MATS:
            q, s = _matrix(wl, seed, "layers.%d.%s" % (l, m), shapes[m])
            mats[m] = q
            if s is not None:
                scales[_SCALE_KEY[m]] = s
        layers.append(HostLayer(attn_norm=ones.copy(), mlp_norm=ones.copy(),
                                scales=scales or None, **mats))
    embed = normal_bf16(seed, "embed", (V, H), std=wl.weight_std)
    if wl.tied:
        lm, lms = embed, None
    else:
        lm, lms = _matrix(wl, seed, "lm_head", (V, H))
    return HostModel(wl, embed, ones.copy(), lm, lms, layers)


def make_kv(wl: Workload, seed: int = 2, batch: Optional[int] = None, ctx: Optional[int] = None):
    """Prefilled K and V caches, each [L][B][nkv][Smax][d] bf16 bits; N(0,1) at positions < ctx."""
    B = wl.batch if batch is None else batch
    c = wl.ctx if ctx is None else ctx
    shape = (wl.n_layers, B, wl.n_kv_heads, wl.max_seq, wl.head_dim)
    kc = np.empty(shape, dtype=np.uint16)
    vc = np.empty(shape, dtype=np.uint16)
    lib().synth_kv_cache(seed, wl.n_layers, B, wl.n_kv_heads, wl.max_seq, wl.head_dim, c,
                         _ptr(kc), _ptr(vc))
    return kc, vc


def initial_tokens(wl: Workload, batch: Optional[int] = None) -> np.ndarray:
    B = wl.batch if batch is None else batch
    return np.array([(1 + 7919 * b) % wl.vocab for b in range(B)], dtype=np.int32)
