"""amk_decode_step_noalloc, the entry point that allocates no device memory,
against amk_decode_step on the same inputs: two decode steps in a row.  Both
run the same kernel on the same default schedule, so the logits of each step
and the KV slots they write must be bit-identical; the parity tolerance
(max |d| <= 1e-2 * max |logit| + 1e-3 per sequence) is reported only to say
how far apart they are when they are not.

The file name makes pytest collect it last, so it also runs after every other
GPU test has used the device; it must pass alone in a fresh process as well.
"""
import numpy as np
import pytest

import synth
from synth.device import kv_from_device, kv_to_device, model_to_device
from tests.gpu_harness import ABS_TOL, REL_TOL, engine_config, make_engine

pytestmark = pytest.mark.gpu


def lib_status(st):
    import persistent_sm_decode_gb300 as amk
    return amk.lib().amk_status_string(st).decode()


def _identical(a, b, what):
    """Bit equality; the message says how far apart the arrays are (against
    the parity tolerance) when they differ."""
    if np.array_equal(a, b):
        return
    x, y = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    d = np.abs(x - y).max()
    bound = REL_TOL * np.abs(x).max() + ABS_TOL
    raise AssertionError("%s differ: max |d| %.3g (%.3g of the parity bound)" % (what, d, d / bound))


def _compare_two_steps(name, batch, ragged):
    import torch
    import persistent_sm_decode_gb300 as amk
    amk.build()
    wl = synth.workload(name)
    model = synth.make_model(wl, seed=1)
    dev = model_to_device(model)
    kc, vc = synth.make_kv(wl, seed=2, batch=batch)
    kv_a = kv_to_device(kc, vc)
    kv_b = kv_a.clone()
    cfg = engine_config(wl, batch)
    eng = make_engine(wl, dev, max_batch=batch)
    tokens = synth.initial_tokens(wl, batch).copy()
    pos = np.array([wl.ctx - (5 * b if ragged else 0) for b in range(batch)], dtype=np.int32)
    pos0 = pos.copy()
    la = torch.empty((batch, wl.vocab), dtype=torch.float32, device="cuda")
    lb = torch.empty_like(la)
    for _ in range(2):
        t = torch.from_numpy(tokens).cuda()
        p = torch.from_numpy(pos).cuda()
        eng.step(t, p, kv_a, la)
        assert eng.sync() == amk.OK
        st = amk.decode_step_noalloc(cfg, dev["embed"], dev["final_norm"], dev["layers"], t, p, kv_b, lb,
                                     dev["lm_head"], dev["s_lm"])
        assert st == amk.OK, lib_status(st)
        a = la.cpu().numpy()
        b = lb.cpu().numpy()
        _identical(a, b, "logits")
        tokens = np.argmax(a, axis=1).astype(np.int32)
        pos = pos + 1
    ka, va = kv_from_device(kv_a)
    kb, vb = kv_from_device(kv_b)
    for name, x, y in (("K", ka, kb), ("V", va, vb)):
        for s in range(batch):
            # the seeded prefix, untouched by both, and the slots the two steps wrote
            assert np.array_equal(x[:, s, :, : pos0[s]], y[:, s, :, : pos0[s]])
            for q in range(int(pos0[s]), int(pos[s])):
                _identical(synth.bf16_bits_to_f32(x[:, s, :, q]), synth.bf16_bits_to_f32(y[:, s, :, q]),
                           "%s slot %d of sequence %d" % (name, q, s))
    eng.close()
    return cfg, dev, kv_b, tokens, pos


def test_no_alloc_matches_handle_tiny_ragged_batch():
    _compare_two_steps("tiny", batch=3, ragged=True)


def test_no_alloc_matches_handle_tinyllama():
    import torch
    import persistent_sm_decode_gb300 as amk
    cfg, dev, kv, tokens, pos = _compare_two_steps("tinyllama_1b1", batch=1, ragged=False)
    # further calls with the same configuration take no device memory
    t = torch.from_numpy(tokens).cuda()
    p = torch.from_numpy(pos).cuda()
    lg = torch.empty((1, cfg.vocab), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        assert amk.decode_step_noalloc(cfg, dev["embed"], dev["final_norm"], dev["layers"], t, p, kv, lg,
                                       dev["lm_head"], dev["s_lm"]) == amk.OK
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_no_alloc_refuses_oversized_state_and_bad_batch():
    import torch
    import persistent_sm_decode_gb300 as amk
    amk.build()
    wl = synth.workload("tiny")
    dev = model_to_device(synth.make_model(wl, seed=1))
    # a 70000-position RoPE table alone needs more than the 16 MiB array; the
    # KV buffer is sized for that capacity all the same
    big = amk.make_config(wl.n_layers, wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.intermediate,
                          wl.vocab, 70000, 1, wl.rms_eps, wl.rope_theta)
    kv = torch.zeros((2, wl.n_layers, 1, wl.n_kv_heads, 70000, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    t = torch.tensor([3], dtype=torch.int32, device="cuda")
    p = torch.tensor([wl.ctx], dtype=torch.int32, device="cuda")
    lg = torch.empty((1, wl.vocab), dtype=torch.float32, device="cuda")
    st = amk.decode_step_noalloc(big, dev["embed"], dev["final_norm"], dev["layers"], t, p, kv, lg,
                                 dev["lm_head"], dev["s_lm"])
    assert st == amk.ERR_UNSUPPORTED
    cfg = engine_config(wl, 1)
    st = amk.decode_step_noalloc(cfg, dev["embed"], dev["final_norm"], dev["layers"], t, p, kv, lg,
                                 dev["lm_head"], dev["s_lm"], batch=2)
    assert st == amk.ERR_INVALID_ARG
    # the refusals leave the entry point usable
    _compare_two_steps("tiny", batch=1, ragged=False)
