"""The binding's call path without a GPU: a stage call is issued at once, or
recorded while a step is being prepared and issued only when the prepared step
runs; a failing status raises either way.  A fake library stands in for
libbastion.so, so nothing here touches a device."""
import pytest

from tree_speculative_decoding_bastion_gb300 import binding as bn


class _Fake:
    def __init__(self, status=0):
        self.log = []
        self.status = status

        def stage(*args):
            self.log.append(args)
            return self.status
        self.bastion_topk_softmax = stage
        self.bastion_accept = stage
        self.bastion_status_string = lambda s: b"fake status"
        self.bastion_last_error = lambda: b"fake detail"


@pytest.fixture
def fake(monkeypatch):
    f = _Fake()
    monkeypatch.setattr(bn, "_lib", f)
    return f


def test_a_call_outside_prepare_is_issued_at_once(fake):
    bn._call("bastion_topk_softmax", 1, 2, 3)
    assert fake.log == [(1, 2, 3)]


def test_calls_made_while_preparing_are_recorded_then_replayed(fake):
    bn._rec.calls = []
    try:
        bn._call("bastion_topk_softmax", "a")
        bn._call("bastion_accept", "b", 7)
        calls = bn._rec.calls
    finally:
        bn._rec.calls = None
    assert fake.log == []                          # nothing issued while recording
    run = bn.PreparedStep(calls, keep=())
    run()
    run()
    assert fake.log == [("a",), ("b", 7), ("a",), ("b", 7)]   # in order, on every call


def test_a_failing_status_raises_on_replay(fake):
    bn._rec.calls = []
    try:
        bn._call("bastion_accept", 1)
        calls = bn._rec.calls
    finally:
        bn._rec.calls = None
    fake.status = 1
    with pytest.raises(bn.BastionError, match="bastion_accept: fake status"):
        bn.PreparedStep(calls, keep=())()


def test_prepare_does_not_nest(fake):
    class _Step:
        def __call__(self, *a, **k):
            pass
    bn._rec.calls = []
    try:
        with pytest.raises(bn.BastionError, match="does not nest"):
            bn.SpecTreeStep.prepare(_Step(), *([None] * 11))
    finally:
        bn._rec.calls = None
