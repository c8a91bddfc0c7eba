"""Host logic of the autograd wrappers' deferred error check (no GPU): error
words are read in issue order, only once their copy has landed, each one
reported once, and a wait drains them all."""
import pytest
import torch

import linear_cross_entropy_gb300 as cce
from linear_cross_entropy_gb300._lib import DEVERR_TARGET_RANGE, DEVERR_TIMEOUT


class FakeEvent:
    def __init__(self, done):
        self.done = done

    def query(self):
        return self.done

    def synchronize(self):
        self.done = True


def _queue(*entries):
    q = cce._DeferredErrors()
    for word, done, name in entries:
        q._pending.append((torch.tensor([word], dtype=torch.int32), FakeEvent(done), name))
    return q


def test_clean_words_raise_nothing_and_drain():
    q = _queue((0, True, "a"), (0, True, "b"))
    q.poll()
    assert q._pending == []


def test_an_unfinished_call_blocks_later_ones_until_waited_for():
    q = _queue((0, False, "a"), (DEVERR_TARGET_RANGE, True, "b"))
    q.poll()  # "a" has not landed: nothing is read, order is kept
    assert [e[2] for e in q._pending] == ["a", "b"]
    with pytest.raises(cce.CCEError) as ei:
        q.poll(wait=True)
    assert ei.value.status == 8 and "b" in str(ei.value)
    assert q._pending == []
    q.poll(wait=True)  # reported once


def test_watching_a_call_leaves_its_own_word_for_later():
    q = _queue((DEVERR_TARGET_RANGE, True, "a"))
    q.poll(keep_last=True)
    assert [e[2] for e in q._pending] == ["a"]
    q._pending.append((torch.tensor([0], dtype=torch.int32), FakeEvent(True), "b"))
    with pytest.raises(cce.CCEError):
        q.poll(keep_last=True)
    assert [e[2] for e in q._pending] == ["b"]


def test_timeout_word_is_reported_first_and_the_rest_stays_queued():
    q = _queue((DEVERR_TIMEOUT | DEVERR_TARGET_RANGE, True, "a"), (DEVERR_TARGET_RANGE, True, "b"))
    with pytest.raises(cce.CCEError) as ei:
        q.poll()
    assert ei.value.status == 9
    assert [e[2] for e in q._pending] == ["b"]
    with pytest.raises(cce.CCEError) as ei:
        q.poll()
    assert ei.value.status == 8
