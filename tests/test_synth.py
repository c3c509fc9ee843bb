"""The seeded input generator: known answers, distributions, determinism (CPU)."""
import numpy as np

import synth


def test_splitmix64_known_answer():
    # published first outputs of splitmix64 seeded with 0
    got = synth.splitmix64_seq(0, 3)
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_streams_are_deterministic_and_sliceable():
    a = synth.normal_bf16(1, "layers.0.wq", (1000,), std=0.02)
    b = synth.normal_bf16(1, "layers.0.wq", (1000,), std=0.02)
    np.testing.assert_array_equal(a, b)
    tail = synth.normal_bf16(1, "layers.0.wq", (400,), std=0.02, offset=600)
    np.testing.assert_array_equal(a[600:], tail)
    assert not np.array_equal(a, synth.normal_bf16(1, "layers.0.wk", (1000,), std=0.02))
    assert not np.array_equal(a, synth.normal_bf16(2, "layers.0.wq", (1000,), std=0.02))


def test_normal_moments():
    n = 1 << 20
    z = synth.normal_f32(7, "z", (n,))
    assert abs(z.mean()) < 5 / np.sqrt(n)
    assert abs(z.std() - 1.0) < 5 * np.sqrt(2.0 / n)
    # tails of a normal: P(|z| > 3) = 0.0027
    assert abs(np.mean(np.abs(z) > 3) - 0.0027) < 0.0005
    w = synth.bf16_bits_to_f32(synth.normal_bf16(7, "w", (n,), std=0.02))
    assert abs(w.std() - 0.02) < 0.0002


def test_int8_uniform_range():
    q = synth.uniform_i8(3, "q", (255 * 4000,))
    assert q.min() == -127 and q.max() == 127
    counts = np.bincount(q.astype(np.int64) + 127, minlength=255)
    assert counts.size == 255
    assert np.all(np.abs(counts - 4000) < 6 * np.sqrt(4000))


def test_scales():
    s = synth.scales_f32(3, "s", 1000, 0.02 / 127, 0.5)
    assert np.all(s >= np.float32(0.02 / 127)) and np.all(s < np.float32(0.02 / 127 * 1.5))
    s0 = synth.scales_f32(3, "s", 10, 0.02 / 127, 0.0)
    assert np.all(s0 == np.float32(0.02 / 127))


def test_kv_cache_prefix_and_independence_from_ctx():
    wl = synth.workload("tiny")
    kc, vc = synth.make_kv(wl, seed=2)
    assert kc.shape == (wl.n_layers, 1, wl.n_kv_heads, wl.max_seq, wl.head_dim)
    assert np.all(kc[:, :, :, wl.ctx:] == 0) and np.all(vc[:, :, :, wl.ctx:] == 0)
    assert np.count_nonzero(kc[:, :, :, : wl.ctx]) > 0.99 * kc[:, :, :, : wl.ctx].size
    k5, _ = synth.make_kv(wl, seed=2, ctx=5)
    np.testing.assert_array_equal(k5[:, :, :, :5], kc[:, :, :, :5])
    v = synth.bf16_bits_to_f32(vc[:, :, :, : wl.ctx])
    assert abs(v.std() - 1.0) < 0.05


def test_model_recipe():
    wl = synth.workload("tiny")
    m = synth.make_model(wl)
    assert m.embed.shape == (wl.vocab, wl.hidden) and m.embed.dtype == np.uint16
    assert m.layers[0].wq.shape == (wl.n_heads * wl.head_dim, wl.hidden)
    assert m.layers[0].wo.shape == (wl.hidden, wl.n_heads * wl.head_dim)
    assert m.layers[1].w_down.shape == (wl.hidden, wl.intermediate)
    assert np.all(m.layers[0].attn_norm == synth.BF16_ONE)
    w8 = synth.workload("tiny", weight_dtype="int8")
    m8 = synth.make_model(w8)
    assert m8.layers[0].wq.dtype == np.int8 and m8.layers[0].scales["s_q"].shape == (wl.n_heads * wl.head_dim,)
    assert m8.embed.dtype == np.uint16 and m8.lm_head.dtype == np.int8
    tied = synth.make_model(synth.workload("tiny", tied=True))
    assert tied.lm_head is tied.embed
    assert list(synth.initial_tokens(wl, 3)) == [1, 7920 % 1024, 15839 % 1024]
