"""Pins of the oracle's whole decode step (CPU only): brute-force prefill
agreement, a closed form of the layer wiring, GQA/MHA equivalence, batch
independence and determinism."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from tests.prefill_ref import bits, prefill_logits, rmsnorm_rows, rne_bf16


def with_random_gains(model, seed=7):
    """Norm gains ~ N(1, 0.25) instead of 1.0, so that a gain applied to the
    wrong norm, or not at all, changes the result."""
    H = model.wl.hidden
    layers = [dataclasses.replace(l, attn_norm=synth.normal_bf16(seed, "g1.%d" % i, (H,), std=0.25, mean=1.0),
                                  mlp_norm=synth.normal_bf16(seed, "g2.%d" % i, (H,), std=0.25, mean=1.0))
              for i, l in enumerate(model.layers)]
    return dataclasses.replace(model, layers=layers,
                               final_norm=synth.normal_bf16(seed, "gf", (H,), std=0.25, mean=1.0))


@pytest.fixture(scope="module")
def tiny():
    wl = synth.workload("tiny")
    return wl, with_random_gains(synth.make_model(wl, seed=1))


def _decode_sequence(model, kc, vc, tokens, start, b=0):
    orc = oracle.Oracle(model, kc, vc)
    out = []
    B = kc.shape[1]
    for t, tok in enumerate(tokens):
        toks = np.zeros(B, dtype=np.int32)
        toks[b] = tok
        pos = np.full(B, start + t, dtype=np.int32)
        out.append(orc.step(toks[: b + 1], pos[: b + 1])[b])
    return np.array(out), orc


def test_decode_matches_prefill_brute_force_empty_cache(tiny):
    wl, model = tiny
    kc, vc = synth.make_kv(wl, seed=2, ctx=0)
    tokens = [5, 900, 17, 17, 333, 1023, 0, 64]
    dec, _ = _decode_sequence(model, kc, vc, tokens, start=0)
    ref = prefill_logits(model, tokens)
    scale = np.abs(ref).max()
    np.testing.assert_allclose(dec, ref, rtol=0, atol=1e-10 * scale)


def test_decode_matches_prefill_brute_force_seeded_cache(tiny):
    wl, model = tiny
    kc, vc = synth.make_kv(wl, seed=2)          # 16 seeded prior positions
    tokens = [1, 2, 3, 500, 777]
    dec, orc = _decode_sequence(model, kc, vc, tokens, start=wl.ctx)
    prior_k = [kc[l, 0, :, : wl.ctx] for l in range(wl.n_layers)]
    prior_v = [vc[l, 0, :, : wl.ctx] for l in range(wl.n_layers)]
    ref = prefill_logits(model, tokens, prior_k, prior_v)
    np.testing.assert_allclose(dec, ref, rtol=0, atol=1e-10 * np.abs(ref).max())
    # the seeded prefix is untouched and the decoded slots were written
    np.testing.assert_array_equal(orc.kc[:, :, :, : wl.ctx], kc[:, :, :, : wl.ctx])
    assert np.any(orc.kc[:, :, :, wl.ctx: wl.ctx + len(tokens)] != 0)
    assert np.all(orc.kc[:, :, :, wl.ctx + len(tokens):] == 0)


def test_decode_matches_prefill_int8_weights():
    wl = synth.workload("tiny", weight_dtype="int8", scale_jitter=0.5)
    model = with_random_gains(synth.make_model(wl, seed=3))
    kc, vc = synth.make_kv(wl, seed=4)
    tokens = [11, 12, 1000]
    dec, _ = _decode_sequence(model, kc, vc, tokens, start=wl.ctx)
    prior_k = [kc[l, 0, :, : wl.ctx] for l in range(wl.n_layers)]
    prior_v = [vc[l, 0, :, : wl.ctx] for l in range(wl.n_layers)]
    ref = prefill_logits(model, tokens, prior_k, prior_v)
    np.testing.assert_allclose(dec, ref, rtol=0, atol=1e-10 * np.abs(ref).max())


def test_decode_matches_prefill_int4_weights():
    wl = synth.workload("tiny", weight_dtype="int4", group_size=16, scale_jitter=0.5)  # I = 688 = 43 x 16
    model = with_random_gains(synth.make_model(wl, seed=3))
    kc, vc = synth.make_kv(wl, seed=4)
    tokens = [11, 12, 1000]
    dec, _ = _decode_sequence(model, kc, vc, tokens, start=wl.ctx)
    prior_k = [kc[l, 0, :, : wl.ctx] for l in range(wl.n_layers)]
    prior_v = [vc[l, 0, :, : wl.ctx] for l in range(wl.n_layers)]
    ref = prefill_logits(model, tokens, prior_k, prior_v)
    np.testing.assert_allclose(dec, ref, rtol=0, atol=1e-10 * np.abs(ref).max())


def test_zero_output_projections_make_every_layer_the_identity(tiny):
    # With Wo = Wd = 0 the residual stream never changes, so the logits have the
    # closed form W_lm . bf16(rmsnorm(E[t]) * g_final).
    wl, model = tiny
    layers = [dataclasses.replace(l, wo=np.zeros_like(l.wo), w_down=np.zeros_like(l.w_down)) for l in model.layers]
    m0 = dataclasses.replace(model, layers=layers)
    kc, vc = synth.make_kv(wl, seed=2)
    orc = oracle.Oracle(m0, kc, vc)
    tok = 321
    logits, xt = orc.step([tok], [wl.ctx], trace=True)
    x = bits(model.embed[tok])
    for l in range(wl.n_layers + 1):
        np.testing.assert_array_equal(xt[0, l], x)
    h = rne_bf16(rmsnorm_rows(x[None, :], model.final_norm, wl.rms_eps))[0]
    np.testing.assert_allclose(logits[0], bits(model.lm_head) @ h, rtol=0, atol=1e-14)


def test_gqa_equals_mha_with_repeated_kv_heads(tiny):
    wl, model = tiny
    G, d = wl.group, wl.head_dim
    wl_m = dataclasses.replace(wl, n_kv_heads=wl.n_heads)
    rep = lambda W: np.repeat(W.reshape(wl.n_kv_heads, d, -1), G, axis=0).reshape(wl.n_heads * d, -1)
    layers = [dataclasses.replace(l, wk=np.ascontiguousarray(rep(l.wk)), wv=np.ascontiguousarray(rep(l.wv)))
              for l in model.layers]
    mm = dataclasses.replace(model, wl=wl_m, layers=layers)
    kc, vc = synth.make_kv(wl, seed=2)
    kcm = np.ascontiguousarray(np.repeat(kc, G, axis=2))
    vcm = np.ascontiguousarray(np.repeat(vc, G, axis=2))
    for tok in (3, 99):
        a = oracle.Oracle(model, kc, vc).step([tok], [wl.ctx])
        b = oracle.Oracle(mm, kcm, vcm).step([tok], [wl.ctx])
        np.testing.assert_array_equal(a, b)


def test_batch_rows_are_independent_and_ragged_positions_work(tiny):
    wl, model = tiny
    B = 3
    kc, vc = synth.make_kv(wl, seed=2, batch=B)
    toks = np.array([7, 8, 9], dtype=np.int32)
    pos = np.array([16, 10, 3], dtype=np.int32)
    batched = oracle.Oracle(model, kc, vc).step(toks, pos)
    for b in range(B):
        kb = np.ascontiguousarray(kc[:, b: b + 1])
        vb = np.ascontiguousarray(vc[:, b: b + 1])
        single = oracle.Oracle(model, kb, vb).step(toks[b: b + 1], pos[b: b + 1])
        np.testing.assert_array_equal(batched[b], single[0])


def test_greedy_decode_is_deterministic(tiny):
    wl, model = tiny
    kc, vc = synth.make_kv(wl, seed=2)
    runs = []
    for _ in range(2):
        orc = oracle.Oracle(model, kc, vc)
        tok = synth.initial_tokens(wl)
        seq, all_logits = [], []
        for s in range(6):
            lg = orc.step(tok, [wl.ctx + s])
            tok, _ = oracle.greedy(lg)
            seq.append(int(tok[0]))
            all_logits.append(lg)
        runs.append((seq, np.array(all_logits)))
    assert runs[0][0] == runs[1][0]
    np.testing.assert_array_equal(runs[0][1], runs[1][1])


def test_thread_count_does_not_change_results(tiny):
    wl, model = tiny
    kc, vc = synth.make_kv(wl, seed=2)
    n0 = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        a = oracle.Oracle(model, kc, vc).step([42], [wl.ctx])
        oracle.set_num_threads(max(2, n0))
        b = oracle.Oracle(model, kc, vc).step([42], [wl.ctx])
    finally:
        oracle.set_num_threads(n0)
    np.testing.assert_array_equal(a, b)


def test_bad_arguments_are_rejected(tiny):
    wl, model = tiny
    kc, vc = synth.make_kv(wl, seed=2)
    orc = oracle.Oracle(model, kc, vc)
    with pytest.raises(ValueError):
        orc.step([wl.vocab], [0])
    with pytest.raises(ValueError):
        orc.step([0], [wl.max_seq])
