"""GPU parity: the decode MegaKernel, called through the C ABI, against the CPU
oracle on seeded synthetic workloads (teacher-forced, see gpu_harness)."""
import numpy as np
import pytest

import synth
from tests.gpu_harness import assert_end_to_end, assert_layers_ok, assert_ok, layerwise, teacher_forced

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import persistent_sm_decode_gb300 as amk
    amk.build()


def test_tiny_32_greedy_steps():
    res = teacher_forced(synth.workload("tiny"))
    assert_ok(res)
    assert res.checked_argmax > 20


def test_tiny_w8a16_jittered_scales():
    wl = synth.workload("tiny", weight_dtype="int8", scale_jitter=0.5)
    assert_ok(teacher_forced(wl))


def test_tiny_batch3_ragged_positions():
    wl = synth.workload("tiny", batch=3)
    assert_ok(teacher_forced(wl, steps=8, positions0=[16, 9, 2]))


def test_tiny_empty_cache_position_zero():
    # p = 0 with nothing cached: attention over the single new token returns V
    wl = synth.workload("tiny", ctx=0)
    assert_ok(teacher_forced(wl, steps=6))


def test_tiny_last_cache_slot():
    wl = synth.workload("tiny")
    assert_ok(teacher_forced(wl, steps=3, positions0=[wl.max_seq - 3]))


@pytest.mark.parametrize("opts", [
    {"ksplit": 2}, {"ksplit": 4, "slot_bytes": 8192}, {"att_chunks": 1}, {"att_chunks": 7},
    {"n_slots": 2, "slot_bytes": 8192}, {"scratch_depth": 1}, {"scratch_depth": 3}, {"n_sm": 5},
])
def test_tiny_schedule_variants(opts):
    wl = synth.workload("tiny", batch=2)
    assert_ok(teacher_forced(wl, steps=4, options=opts))


def test_tiny_32_steps_bit_identical_across_runs():
    import torch
    from synth.device import kv_from_device, kv_to_device, model_to_device
    from tests.gpu_harness import make_engine
    wl = synth.workload("tiny")
    model = synth.make_model(wl)
    kc, vc = synth.make_kv(wl)
    eng = make_engine(wl, model_to_device(model))
    runs = []
    for _ in range(2):
        kv = kv_to_device(kc, vc)
        lg = torch.empty((1, wl.vocab), device="cuda")
        tok, seq = 1, []
        for s in range(wl.steps):
            eng.step(torch.tensor([tok], dtype=torch.int32, device="cuda"),
                     torch.tensor([wl.ctx + s], dtype=torch.int32, device="cuda"), kv, lg)
            assert eng.sync() == 0
            seq.append(lg.cpu().numpy().copy())
            tok = int(np.argmax(seq[-1]))
        runs.append((np.array(seq), kv_from_device(kv)))
    np.testing.assert_array_equal(runs[0][0], runs[1][0])
    np.testing.assert_array_equal(runs[0][1][0], runs[1][1][0])
    np.testing.assert_array_equal(runs[0][1][1], runs[1][1][1])
    eng.close()


def test_determinism_bit_identical():
    import torch
    from synth.device import kv_to_device, model_to_device
    from tests.gpu_harness import make_engine
    wl = synth.workload("smollm2_135m")
    model = synth.make_model(wl)
    kc, vc = synth.make_kv(wl)
    dev = model_to_device(model)
    eng = make_engine(wl, dev)
    outs = []
    for _ in range(2):
        kv = kv_to_device(kc, vc)
        lg = torch.empty((1, wl.vocab), device="cuda")
        eng.step(torch.tensor([5], dtype=torch.int32, device="cuda"),
                 torch.tensor([wl.ctx], dtype=torch.int32, device="cuda"), kv, lg)
        assert eng.sync() == 0
        outs.append(lg.cpu().numpy())
    np.testing.assert_array_equal(outs[0], outs[1])
    eng.close()


# ---- per-layer parity from a shared state, full sizes (the gate) ----

def test_smollm2_135m_per_layer():
    assert_layers_ok(layerwise(synth.workload("smollm2_135m"), steps=3))


def test_tinyllama_1b1_per_layer():
    assert_layers_ok(layerwise(synth.workload("tinyllama_1b1"), steps=3))


def test_tinyllama_1b1_w8a16_per_layer():
    assert_layers_ok(layerwise(synth.workload("tinyllama_1b1_w8a16", scale_jitter=0.5), steps=3))


def test_llama2_7b_per_layer():
    assert_layers_ok(layerwise(synth.workload("llama2_7b"), steps=2))


def test_llama2_7b_batch8_per_layer_all_rows():
    assert_layers_ok(layerwise(synth.workload("llama2_7b_b8"), steps=1))


def test_tiny_per_layer_batch4_ragged():
    wl = synth.workload("tiny", batch=4)
    assert_layers_ok(layerwise(wl, steps=4, positions0=[16, 0, 30, 47 - 4]))


# ---- end to end, teacher-forced over the workloads' step counts ----

def test_smollm2_135m_end_to_end_128_steps():
    assert_end_to_end(teacher_forced(synth.workload("smollm2_135m"), floor=True))


def test_tinyllama_1b1_end_to_end_128_steps():
    assert_end_to_end(teacher_forced(synth.workload("tinyllama_1b1"), floor=True))


def test_tinyllama_1b1_w8a16_end_to_end_128_steps():
    assert_end_to_end(teacher_forced(synth.workload("tinyllama_1b1_w8a16"), floor=True))


def test_llama2_7b_end_to_end_64_steps():
    # the workload's full 64 greedy steps
    assert_end_to_end(teacher_forced(synth.workload("llama2_7b"), check_cache=False, floor=True))


def test_llama2_7b_batch8_end_to_end_all_rows():
    # all eight sequences over 16 steps: the oracle decodes every row in full
    # (fp64 and the fp32-accumulation build), so the step count is what bounds
    # the test's CPU time
    wl = synth.workload("llama2_7b_b8")
    assert_end_to_end(teacher_forced(wl, steps=16, check_cache=False, floor=True))


# ---- batches above 1: the tensor-core GEMV (bf16) and the batch-size sweep shape ----

def test_tiny_batch16_ragged_positions():
    # M = 16: both halves of the tensor-core A fragment carry sequences
    wl = synth.workload("tiny", batch=16)
    assert_ok(teacher_forced(wl, steps=5, positions0=[16 - (b % 9) * 2 for b in range(16)]))


def test_tiny_batch9_and_k_split():
    # one sequence in the upper half of the fragment; a K split adds the
    # second slice's sums to the first's
    wl = synth.workload("tiny", batch=9)
    assert_ok(teacher_forced(wl, steps=4))
    assert_ok(teacher_forced(synth.workload("tiny", batch=8), steps=4, options={"ksplit": 2}))


def test_tiny_w8a16_batch5():
    # int8 weights at batch above 1 take the CUDA-core tile
    wl = synth.workload("tiny", batch=5, weight_dtype="int8", scale_jitter=0.5)
    assert_ok(teacher_forced(wl, steps=4))


def test_tinyllama_short_batch16_per_layer_and_end_to_end():
    wl = synth.workload("tinyllama_1b1_short", batch=16)
    assert_layers_ok(layerwise(wl, steps=1, check_rows=[0, 7, 8, 15]))
    assert_end_to_end(teacher_forced(wl, steps=4, check_rows=[0, 9, 15], check_cache=False, floor=True))


# ---- the per-operator comparison path (one launch per operator) ----

def _unfused_teacher_forced(wl, steps):
    import torch
    import oracle
    from tests.gpu_harness import engine_config
    import persistent_sm_decode_gb300 as amk
    from synth.device import kv_to_device, model_to_device
    model = synth.make_model(wl, seed=1)
    kc, vc = synth.make_kv(wl, seed=2)
    dev = model_to_device(model)
    u = amk.UnfusedEngine(engine_config(wl), dev["embed"], dev["final_norm"], dev["layers"], dev["lm_head"],
                          dev["s_lm"])
    kv = kv_to_device(kc, vc)
    orc = oracle.Oracle(model, kc, vc)
    lg = torch.empty((wl.batch, wl.vocab), dtype=torch.float32, device="cuda")
    tok = synth.initial_tokens(wl)
    worst = 0.0
    for s in range(steps):
        pos = np.full(wl.batch, wl.ctx + s, dtype=np.int32)
        u.step(torch.from_numpy(tok).cuda(), torch.from_numpy(pos).cuda(), kv, lg)
        torch.cuda.synchronize()
        ref = orc.step(tok, pos)
        got = lg.cpu().numpy().astype(np.float64)
        worst = max(worst, float(np.abs(got - ref).max() / (1e-2 * np.abs(ref).max() + 1e-3)))
        tok, _ = oracle.greedy(ref)
    u.close()
    return worst


def test_unfused_tiny_matches_oracle():
    assert _unfused_teacher_forced(synth.workload("tiny"), 8) <= 1.0


def test_unfused_tiny_w8a16_matches_oracle():
    assert _unfused_teacher_forced(synth.workload("tiny", weight_dtype="int8", scale_jitter=0.5), 6) <= 1.0


# ---- W4A16: 4-bit weight codes with per-group scales (batch 1) ----

def test_tiny_w4a16_group32():
    # the tiny shape with I = 704 (a whole number of 32-weight chunks) and a
    # scale every 32 weights, jittered so that a wrong group index shows
    wl = synth.workload("tiny", weight_dtype="int4", intermediate=704, group_size=32, scale_jitter=0.5)
    assert_ok(teacher_forced(wl))


def test_tinyllama_1b1_w4a16_per_layer():
    assert_layers_ok(layerwise(synth.workload("tinyllama_1b1_w4a16", scale_jitter=0.5), steps=2))


def test_tinyllama_1b1_w4a16_end_to_end_32_steps():
    assert_end_to_end(teacher_forced(synth.workload("tinyllama_1b1_w4a16"), steps=32, floor=True))
