"""Copies seeded host inputs to CUDA tensors (torch as device-memory plumbing).

No decode arithmetic happens here: bf16 bit patterns are reinterpreted as
``torch.bfloat16`` without conversion, int8 and fp32 arrays are copied as is.
"""
from __future__ import annotations

import numpy as np


def _t(a: np.ndarray, device):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def model_to_device(model, device="cuda") -> dict:
    """Device tensors of a synth.HostModel, keyed the way DecodeEngine takes them."""
    layers = []
    for hl in model.layers:
        d = {"attn_norm": _t(hl.attn_norm, device), "mlp_norm": _t(hl.mlp_norm, device),
             "wq": _t(hl.wq, device), "wk": _t(hl.wk, device), "wv": _t(hl.wv, device), "wo": _t(hl.wo, device),
             "w_gate": _t(hl.w_gate, device), "w_up": _t(hl.w_up, device), "w_down": _t(hl.w_down, device)}
        if hl.scales:
            for k, v in hl.scales.items():
                d[k] = _t(v, device)
        layers.append(d)
    embed = _t(model.embed, device)
    out = {"embed": embed, "final_norm": _t(model.final_norm, device), "layers": layers,
           "lm_head": None if model.wl.tied else _t(model.lm_head, device),
           "s_lm": None if model.lm_scale is None else _t(model.lm_scale, device)}
    return out


def kv_to_device(kc: np.ndarray, vc: np.ndarray, device="cuda"):
    """One bf16 tensor [2][L][B][nkv][Smax][d]: the K cache followed by the V cache."""
    import torch
    both = np.stack([kc, vc])
    return torch.from_numpy(both.view(np.int16)).view(torch.bfloat16).to(device)


def kv_from_device(kv) -> tuple:
    """Back to two uint16 bit-pattern arrays (K, V)."""
    import torch
    a = kv.view(torch.int16).cpu().numpy().view(np.uint16)
    return a[0], a[1]


def kv_rows_from_device(kv, rows) -> tuple:
    """K and V of the given sequences only, as uint16 arrays [L][len(rows)][nkv][Smax][d]."""
    import torch
    idx = torch.tensor(list(rows), dtype=torch.long, device=kv.device)
    a = kv.index_select(2, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    return np.ascontiguousarray(a[0]), np.ascontiguousarray(a[1])
