"""Host logic of the GPU parity harness that needs no GPU."""
from tests.gpu_harness import Result


def _res(agrees):
    r = Result()
    r.steps = len(agrees)
    r.records = [(s, b, 0.5, a, None) for s, row in enumerate(agrees) for b, a in enumerate(row)]
    return r


def test_free_running_length_ends_at_the_first_disagreement():
    assert _res([[True], [True], [False], [True], [False]]).free_running == 2
    assert _res([[True, True], [True, False], [True, True]]).free_running == 1
    assert _res([[False]]).free_running == 0


def test_free_running_length_is_every_step_when_all_agree():
    r = _res([[True, True]] * 4)
    assert r.free_running == 4
    assert "free-running 4" in repr(r)
