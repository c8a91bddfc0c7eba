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


def test_a_full_ring_keeps_the_current_calls_word():
    """Every slot of the ring is pending and the oldest holds an error: the
    next call frees that slot, and the older error is reported, but the new
    call's own word is still recorded and reported after it."""
    q = cce._DeferredErrors()
    n = q.SLOTS
    words = torch.zeros(n, dtype=torch.int32)
    events = [FakeEvent(False) for _ in range(n)]
    q._make_ring = lambda device: [words, events, 0]

    def record(word, evs, slot, dev_err):
        word.copy_(dev_err)
        evs[slot] = FakeEvent(True)
        return evs[slot]

    q._record = record
    dev = torch.zeros(1, dtype=torch.int32)
    ring = q._make_ring(None)
    q._rings[dev.device.index] = ring
    for i in range(n):  # the ring is full; none of the copies has landed yet
        words[i] = DEVERR_TIMEOUT if i == 0 else 0
        q._pending.append((words[i:i + 1], events[i], f"call{i}"))
    bad = torch.tensor([DEVERR_TARGET_RANGE], dtype=torch.int32)
    reported = []
    try:
        q.watch(bad, "new")
    except cce.CCEError as e:
        reported.append((e.status, str(e)))
    assert [e[2] for e in q._pending][-1] == "new"
    while True:
        try:
            q.poll(wait=True)
            break
        except cce.CCEError as e:
            reported.append((e.status, str(e)))
    assert [r[0] for r in reported] == [9, 8]
    assert "call0" in reported[0][1] and "new" in reported[1][1]
    assert q._pending == [] and q._found == []
