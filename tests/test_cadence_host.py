"""The re-plan cadence policy (host bookkeeping only, no GPU).

README item 1: the arena is planned again after a prompt's prefill, after
every few hundred generated tokens, and between requests.
"""
import pytest

from resident_expert_routed_gb300.layer import Cadence


def test_every_n_tokens():
    c = Cadence(every_tokens=256, after_prefill=False, between_requests=False)
    due = [c.step(2) for _ in range(300)]
    assert [i for i, d in enumerate(due) if d] == [127, 255]     # 2 tokens a step: every 128 steps
    assert c.tokens_since == 2 * (300 - 256)


def test_after_prefill_resets_the_count():
    c = Cadence(every_tokens=100, after_prefill=True)
    assert not c.step(60)
    assert c.step(8192, prefill=True)                           # a prefill chunk: re-plan now
    assert c.tokens_since == 0
    assert not c.step(99) and c.step(1)


def test_between_requests_only_when_something_was_generated():
    c = Cadence(every_tokens=0, after_prefill=False, between_requests=True)
    assert not c.request_done()
    assert not c.step(5)                                        # the token interval is off
    assert c.request_done() and not c.request_done()


def test_switches_off():
    c = Cadence(every_tokens=0, after_prefill=False, between_requests=False)
    assert not any(c.step(1000, prefill=True) for _ in range(10))
    assert not c.request_done()
    with pytest.raises(ValueError):
        Cadence(every_tokens=-1)
