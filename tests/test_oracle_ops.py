"""Pins of the oracle's operators against closed forms, library routines and
identities that are independent of the oracle's own code (CPU only)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.prefill_ref import bits, rne_bf16

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------- bf16 rounding

def test_bf16_decode_known_patterns():
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x3F00) == 0.5
    assert oracle.bf16_to_double(0x0000) == 0.0
    assert oracle.bf16_to_double(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127


def test_bf16_round_matches_torch_on_float32_inputs():
    # torch's float32 -> bfloat16 conversion is round-to-nearest-even; on
    # float32-representable inputs there is no double rounding to worry about.
    x = RNG.standard_normal(4000).astype(np.float32) * np.float32(3.0)
    # add exact ties: bf16 value + half an ulp
    base = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    ties = (base.view(np.uint32) + np.uint32(0x8000)).view(np.float32)
    allx = np.concatenate([x, ties, np.float32([1e-30, -3e-35, 6e37])])
    ref = torch.from_numpy(allx).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.double_to_bf16(float(v)) for v in allx], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_bf16_round_ties_and_double_rounding():
    assert oracle.double_to_bf16(1 + 2 ** -8) == 0x3F80           # tie -> even (1.0)
    assert oracle.double_to_bf16(1 + 3 * 2 ** -8) == 0x3F82       # tie -> even (1 + 2^-6)
    # just above a tie, below float32 resolution: rounding through float32 first
    # would land on the tie and then on 1.0; the direct rounding goes up.
    assert oracle.double_to_bf16(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert oracle.double_to_bf16(-(1 + 2 ** -8 + 2 ** -40)) == 0xBF81
    assert oracle.double_to_bf16(3.4e38) == 0x7F80                # overflow -> inf


def test_numpy_rne_helper_agrees_with_torch():
    # the brute-force helper used by other pins is itself pinned to torch
    x = RNG.standard_normal(3000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(rne_bf16(x.astype(np.float64)), ref)


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_closed_form_mean_square():
    n, eps = 576, 1e-5
    x = RNG.standard_normal(n) * 0.7
    ones = np.full(n, synth.BF16_ONE, dtype=np.uint16)
    y = oracle.rmsnorm(x, ones, eps)
    m = np.mean(x * x)
    assert abs(np.mean(y * y) - m / (m + eps)) < 1e-13


def test_rmsnorm_constant_vector():
    n, eps, c = 256, 1e-5, 0.37
    y = oracle.rmsnorm(np.full(n, c), np.full(n, synth.BF16_ONE, dtype=np.uint16), eps)
    np.testing.assert_allclose(y, c / math.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_gain_is_elementwise_and_eps_matters():
    n = 300
    x = RNG.standard_normal(n)
    g = synth.normal_bf16(5, "gain", (n,), std=1.0)
    y = oracle.rmsnorm(x, g, 1e-5)
    ratio = y / (x * bits(g))
    np.testing.assert_allclose(ratio, ratio[0], rtol=1e-13)
    np.testing.assert_allclose(ratio[0], 1 / math.sqrt(np.mean(x * x) + 1e-5), rtol=1e-14)
    # tiny input: eps dominates, output ~ x / sqrt(eps)
    t = np.full(n, 1e-6)
    yt = oracle.rmsnorm(t, np.full(n, synth.BF16_ONE, dtype=np.uint16), 1e-5)
    np.testing.assert_allclose(yt, 1e-6 / math.sqrt(1e-12 + 1e-5), rtol=1e-14)


def test_rmsnorm_scale_invariance():
    x = RNG.standard_normal(512)
    ones = np.full(512, synth.BF16_ONE, dtype=np.uint16)
    np.testing.assert_allclose(oracle.rmsnorm(1000 * x, ones, 0.0), oracle.rmsnorm(x, ones, 0.0), rtol=1e-14)


# ----------------------------------------------------------------- GEMV

def _onehot_bf16(K, i):
    h = np.zeros(K, dtype=np.uint16)
    h[i] = synth.BF16_ONE
    return h


def test_gemv_bf16_onehot_returns_column():
    W = synth.normal_bf16(3, "W", (37, 96), std=0.02)
    for i in (0, 1, 50, 95):
        np.testing.assert_array_equal(oracle.gemv(W, _onehot_bf16(96, i)), bits(W[:, i]))


def test_gemv_int8_onehot_returns_scaled_column():
    W = synth.uniform_i8(3, "W8", (41, 64))
    s = synth.scales_f32(3, "W8.scale", 41, 0.02 / 127, 0.5)   # jittered: a wrong row scale shows
    for i in (0, 7, 63):
        np.testing.assert_array_equal(oracle.gemv(W, _onehot_bf16(64, i), s),
                                      s.astype(np.float64) * W[:, i].astype(np.float64))


def test_gemv_brute_force_against_numpy_matmul():
    W = synth.normal_bf16(4, "W", (129, 688), std=0.02)
    h = synth.normal_bf16(4, "h", (688,), std=1.0)
    ref = bits(W) @ bits(h)
    got = oracle.gemv(W, h)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-14)
    W8 = synth.uniform_i8(4, "W8", (65, 256))
    s = synth.scales_f32(4, "W8.scale", 65, 0.02 / 127, 0.5)
    h8 = synth.normal_bf16(4, "h8", (256,), std=1.0)
    # int8 x bf16 products and their sums are exact in double here (|sum| < 2^53 ulps)
    ref8 = s.astype(np.float64) * (W8.astype(np.float64) @ bits(h8))
    np.testing.assert_array_equal(oracle.gemv(W8, h8, s), ref8)


def _unpack_u4(Wp):
    """4-bit codes from bytes, element 2j from the low nibble of byte j (numpy, independent of the oracle)."""
    return np.stack([Wp & 15, Wp >> 4], axis=-1).reshape(Wp.shape[0], 2 * Wp.shape[1]).astype(np.int64)


def test_gemv_int4_onehot_returns_scaled_column():
    # element i is code u = nibble (i % 2) of byte i // 2, value s[row][i // 128] * (u - 8)
    Wp = synth.uniform_u4(5, "W4", (19, 384))
    s = synth.scales_f32(5, "W4.scale", 19 * 3, 0.02 / 7, 0.5).reshape(19, 3)   # jittered per group
    u = _unpack_u4(Wp)
    for i in (0, 1, 127, 128, 255, 383):
        want = s[:, i // 128].astype(np.float64) * (u[:, i] - 8).astype(np.float64)
        np.testing.assert_array_equal(oracle.gemv_int4(Wp, _onehot_bf16(384, i), s, 128), want)


def test_gemv_int4_brute_force_against_numpy_dequantised_matmul():
    Wp = synth.uniform_u4(6, "W4", (33, 512))
    s = synth.scales_f32(6, "W4.scale", 33 * 8, 0.02 / 7, 0.5).reshape(33, 8)
    h = synth.normal_bf16(6, "h4", (512,), std=1.0)
    dq = (_unpack_u4(Wp) - 8).astype(np.float64) * np.repeat(s.astype(np.float64), 64, axis=1)
    got = oracle.gemv_int4(Wp, h, s, 64)
    np.testing.assert_allclose(got, dq @ bits(h), rtol=1e-13, atol=1e-15)
    # the codes cover 1..15 only (values -7..7) and are roughly uniform
    u = _unpack_u4(Wp)
    assert u.min() == 1 and u.max() == 15 and abs(u.mean() - 8.0) < 0.2


# ----------------------------------------------------------------- RoPE

def test_rope_identity_at_position_zero():
    u = RNG.standard_normal(64)
    np.testing.assert_array_equal(oracle.rope(u, 0, 1e4), u)


def test_rope_matches_complex_rotation():
    # RoFormer's own statement: pair (u_i, u_{i+d/2}) as a complex number,
    # multiplied by exp(i * p * base^(-2i/d)).
    for d, p, base in ((64, 7, 1e4), (128, 4095, 1e4), (64, 1, 500.0)):
        u = RNG.standard_normal(d)
        h = d // 2
        z = (u[:h] + 1j * u[h:]) * np.exp(1j * p * base ** (-2.0 * np.arange(h) / d))
        np.testing.assert_allclose(oracle.rope(u, p, base), np.concatenate([z.real, z.imag]),
                                   rtol=0, atol=1e-12)


def test_rope_preserves_pair_norms_and_relative_positions():
    d = 64
    q, k = RNG.standard_normal(d), RNG.standard_normal(d)
    rq = oracle.rope(q, 9, 1e4)
    h = d // 2
    np.testing.assert_allclose(rq[:h] ** 2 + rq[h:] ** 2, q[:h] ** 2 + q[h:] ** 2, rtol=1e-12)
    lhs = oracle.rope(q, 40, 1e4) @ oracle.rope(k, 13, 1e4)
    rhs = oracle.rope(q, 27, 1e4) @ k
    assert abs(lhs - rhs) < 1e-11


# ----------------------------------------------------------------- attention

def test_attention_single_cached_token_returns_v():
    d = 64
    q = RNG.standard_normal(d)
    K = synth.normal_bf16(6, "K", (1, d))
    V = synth.normal_bf16(6, "V", (1, d))
    w, o = oracle.attention(q, K, V)
    assert w[0] == 1.0
    np.testing.assert_array_equal(o, bits(V[0]))


def test_attention_softmax_rows_sum_to_one():
    for n in (1, 2, 17, 300):
        q = RNG.standard_normal(128) * 3
        w, _ = oracle.attention(q, synth.normal_bf16(7, "K%d" % n, (n, 128)), synth.normal_bf16(7, "V", (n, 128)))
        assert abs(w.sum() - 1.0) < 1e-14
        assert np.all(w > 0)


def test_attention_zero_query_gives_mean_of_v():
    n, d = 33, 64
    K = synth.normal_bf16(8, "K", (n, d))
    V = synth.normal_bf16(8, "V", (n, d))
    w, o = oracle.attention(np.zeros(d), K, V)
    np.testing.assert_allclose(w, 1.0 / n, rtol=1e-15)
    np.testing.assert_allclose(o, bits(V).mean(axis=0), rtol=0, atol=1e-14)


def test_attention_two_token_closed_form_pins_scale():
    # scores 0 and ln(3): softmax weights exactly 1/4 and 3/4 iff the scale is 1/sqrt(d)
    d = 64
    q = np.zeros(d)
    q[0] = math.sqrt(d) * math.log(3.0)
    K = np.zeros((2, d), dtype=np.uint16)
    K[1, 0] = synth.BF16_ONE
    V = synth.normal_bf16(9, "V", (2, d))
    w, o = oracle.attention(q, K, V)
    np.testing.assert_allclose(w, [0.25, 0.75], rtol=1e-14)
    np.testing.assert_allclose(o, 0.25 * bits(V[0]) + 0.75 * bits(V[1]), rtol=0, atol=1e-14)


def test_attention_dominant_key_selects_its_value_and_is_permutation_invariant():
    n, d = 20, 64
    K = synth.normal_bf16(10, "K", (n, d))
    V = synth.normal_bf16(10, "V", (n, d))
    q = bits(K[13]) * 40.0
    w, o = oracle.attention(q, K, V)
    assert int(np.argmax(w)) == 13 and w[13] > 1 - 1e-9
    np.testing.assert_allclose(o, bits(V[13]), atol=1e-8)
    perm = RNG.permutation(n)
    w2, o2 = oracle.attention(RNG.standard_normal(d), K, V)
    # same query on permuted rows: same output, permuted weights
    q3 = RNG.standard_normal(d)
    wa, oa = oracle.attention(q3, K, V)
    wb, ob = oracle.attention(q3, K[perm], V[perm])
    np.testing.assert_allclose(wb, wa[perm], rtol=1e-13)
    np.testing.assert_allclose(ob, oa, rtol=0, atol=1e-14)


# ----------------------------------------------------------------- SiLU, argmax

def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(oracle.silu(40.0) - 40.0) < 1e-14
    assert abs(oracle.silu(-40.0)) < 1e-15
    for z in (0.3, 1.7, 5.0):
        # silu(-z) = -z * sigmoid(-z) = silu(z) - z
        assert abs(oracle.silu(-z) - (oracle.silu(z) - z)) < 1e-14


def test_silu_matches_torch():
    z = RNG.standard_normal(200) * 4
    ref = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    np.testing.assert_allclose([oracle.silu(v) for v in z], ref, rtol=1e-14, atol=1e-16)


def test_argmax_lowest_index_on_ties():
    v = np.array([0.1, 3.0, -1.0, 3.0, 2.9])
    assert oracle.argmax(v) == 1 == int(np.argmax(v))
    for _ in range(20):
        r = np.round(RNG.standard_normal(50), 1)
        assert oracle.argmax(r) == int(np.argmax(r))
