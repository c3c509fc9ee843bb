"""Failure handling on the GPU without faulting it: a dropped dependency signal
makes the waits that depend on it run into their (short) limit; the kernel
reports the timeout through the error word and the next step runs normally.
Out-of-range inputs are refused by the kernel before any memory access."""
import numpy as np
import pytest

import synth
from synth.device import kv_to_device, model_to_device
from tests.gpu_harness import make_engine

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny_engine():
    import persistent_sm_decode_gb300 as amk
    amk.build()
    wl = synth.workload("tiny")
    model = synth.make_model(wl)
    dev = model_to_device(model)
    eng = make_engine(wl, dev, options={"wait_timeout_ns": 20_000_000, "n_sm": 8})
    kc, vc = synth.make_kv(wl)
    yield wl, eng, dev, kv_to_device(kc, vc)
    eng.close()


def _step(eng, wl, kv, tok=3, pos=None):
    import torch
    lg = torch.zeros((1, wl.vocab), device="cuda")
    eng.step(torch.tensor([tok], dtype=torch.int32, device="cuda"),
             torch.tensor([wl.ctx if pos is None else pos], dtype=torch.int32, device="cuda"), kv, lg)
    return lg


def test_dropped_signal_times_out_and_recovers(tiny_engine):
    import persistent_sm_decode_gb300 as amk
    wl, eng, dev, kv = tiny_engine
    _step(eng, wl, kv)
    assert eng.sync() == amk.OK
    ref = _step(eng, wl, kv).cpu().numpy()
    assert eng.sync() == amk.OK
    eng.drop_signal(0, 0)            # CTA 0's first task (a layer-0 QKV row block) never signals
    _step(eng, wl, kv)
    _step(eng, wl, kv)               # launched after the error: must do nothing
    assert eng.sync() == amk.ERR_TIMEOUT
    info = eng.last_error()
    assert info["code"] == 1 and info["counter"] >= 0 and info["observed"] < info["target"]
    eng.drop_signal(-1, -1)
    again = _step(eng, wl, kv).cpu().numpy()
    assert eng.sync() == amk.OK
    np.testing.assert_array_equal(again, ref)


def test_out_of_range_token_is_refused(tiny_engine):
    import persistent_sm_decode_gb300 as amk
    wl, eng, dev, kv = tiny_engine
    _step(eng, wl, kv, tok=wl.vocab + 5)
    assert eng.sync() == amk.ERR_INVALID_ARG
    _step(eng, wl, kv, pos=wl.max_seq)
    assert eng.sync() == amk.ERR_INVALID_ARG
    _step(eng, wl, kv)
    assert eng.sync() == amk.OK


def test_host_side_argument_checks(tiny_engine):
    import torch
    import persistent_sm_decode_gb300 as amk
    wl, eng, dev, kv = tiny_engine
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    lg = torch.zeros((1, wl.vocab), device="cuda")
    assert eng.step_raw(0, t.data_ptr(), t.data_ptr(), kv.data_ptr(), lg.data_ptr()) == amk.ERR_INVALID_ARG
    assert eng.step_raw(2, t.data_ptr(), t.data_ptr(), kv.data_ptr(), lg.data_ptr()) == amk.ERR_INVALID_ARG
    assert eng.step_raw(1, 0, t.data_ptr(), kv.data_ptr(), lg.data_ptr()) == amk.ERR_INVALID_ARG
    assert eng.step_raw(1, t.data_ptr(), t.data_ptr(), kv.data_ptr() + 2, lg.data_ptr()) == amk.ERR_INVALID_ARG
