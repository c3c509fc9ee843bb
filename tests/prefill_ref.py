"""Brute-force reference for pinning the oracle (test helper, numpy float64).

It runs the decoder over a whole token sequence at once, the way a prefill
does: matrix products over all positions, RoPE as complex multiplication
(the RoFormer paper's own formulation), and a causal mask over the score
matrix.  The oracle instead decodes one token at a time against a KV cache.
The two formulations share no code; they agree only if the oracle's cache
writes, causal range, GQA head mapping, RoPE positions, residual wiring and
bf16 rounding points are right.
"""
from __future__ import annotations

import numpy as np


def rne_bf16(y) -> np.ndarray:
    """Round float64 values to bf16 (8-bit significand), ties to even, as float64."""
    y = np.asarray(y, dtype=np.float64)
    m, e = np.frexp(y)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def bits(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dense(W, scales=None) -> np.ndarray:
    if W.dtype == np.int8:
        return W.astype(np.float64) * np.asarray(scales, dtype=np.float64)[:, None]
    if W.dtype == np.uint8:
        # 4-bit codes two per byte (low nibble first), value scale[row][k // group] * (code - 8)
        codes = np.stack([W & 15, W >> 4], axis=-1).reshape(W.shape[0], 2 * W.shape[1]).astype(np.float64)
        sc = np.asarray(scales, dtype=np.float64)
        group = codes.shape[1] // sc.shape[1]
        return (codes - 8.0) * np.repeat(sc, group, axis=1)
    return bits(W)


def rmsnorm_rows(X, gain, eps):
    ms = np.mean(X * X, axis=-1, keepdims=True)
    return X / np.sqrt(ms + eps) * bits(gain)[None, :]


def rope_complex(U, positions, base):
    """U: [T, d] rows at the given positions; rotate-half pairs as complex numbers."""
    T, d = U.shape
    h = d // 2
    inv = base ** (-2.0 * np.arange(h) / d)
    z = U[:, :h] + 1j * U[:, h:]
    z = z * np.exp(1j * np.outer(np.asarray(positions, dtype=np.float64), inv))
    return np.concatenate([z.real, z.imag], axis=1)


def silu(z):
    return z / (1.0 + np.exp(-z))


def prefill_logits(model, tokens, prior_k=None, prior_v=None):
    """Logits [T, V] for tokens at positions ctx..ctx+T-1, where ctx is the
    number of prior cached positions (prior_k[l]: [nkv, ctx, d] bf16 bits)."""
    wl = model.wl
    H, nq, nkv, d = wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim
    G = nq // nkv
    T = len(tokens)
    ctx = 0 if prior_k is None else prior_k[0].shape[1]
    pos = np.arange(ctx, ctx + T)
    X = bits(model.embed)[np.asarray(tokens)]
    causal = np.triu(np.ones((T, ctx + T), dtype=bool), k=ctx + 1)
    for l, ly in enumerate(model.layers):
        s = ly.scales or {}
        Hn = rne_bf16(rmsnorm_rows(X, ly.attn_norm, wl.rms_eps))
        Q = Hn @ dense(ly.wq, s.get("s_q")).T
        K = Hn @ dense(ly.wk, s.get("s_k")).T
        V = Hn @ dense(ly.wv, s.get("s_v")).T
        O = np.zeros((T, nq * d))
        for g in range(nkv):
            Kg = rne_bf16(rope_complex(K[:, g * d:(g + 1) * d], pos, wl.rope_theta))
            Vg = rne_bf16(V[:, g * d:(g + 1) * d])
            if ctx:
                Kg = np.concatenate([bits(prior_k[l][g]), Kg], axis=0)
                Vg = np.concatenate([bits(prior_v[l][g]), Vg], axis=0)
            for j in range(g * G, (g + 1) * G):
                Qj = rope_complex(Q[:, j * d:(j + 1) * d], pos, wl.rope_theta)
                S = (Qj @ Kg.T) / np.sqrt(d)
                S[causal] = -np.inf
                P = np.exp(S - S.max(axis=1, keepdims=True))
                P /= P.sum(axis=1, keepdims=True)
                O[:, j * d:(j + 1) * d] = P @ Vg
        X = X + rne_bf16(O) @ dense(ly.wo, s.get("s_o")).T
        H2 = rne_bf16(rmsnorm_rows(X, ly.mlp_norm, wl.rms_eps))
        A = rne_bf16(silu(H2 @ dense(ly.w_gate, s.get("s_gate")).T) * (H2 @ dense(ly.w_up, s.get("s_up")).T))
        X = X + A @ dense(ly.w_down, s.get("s_down")).T
    Hf = rne_bf16(rmsnorm_rows(X, model.final_norm, wl.rms_eps))
    return Hf @ dense(model.lm_head, model.lm_scale).T
