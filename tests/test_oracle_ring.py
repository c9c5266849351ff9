"""Pins of the integer ring model: schedules worked out by hand from the flush,
verify and rollback rules (ring slot of logical record j = (head + j) mod L)."""
import pytest

from oracle.ring import RingModel, SeqRing


def test_decode_flushes_every_L_steps():
    """64 decode steps from an empty ring with L = 16 flush on steps 16, 32,
    48 and 64 (four flushes), each folding 16 tokens; head stays 0."""
    r = SeqRing(16)
    flushes = []
    for t in range(1, 65):
        folded = r.decode(t)
        if folded is not None:
            flushes.append(t)
            assert folded == list(range(t - 15, t + 1))
            assert (r.head, r.len) == (0, 0)
        else:
            assert r.len == t % 16
    assert flushes == [16, 32, 48, 64]


def test_mixed_schedule_L4():
    r = SeqRing(4)
    assert r.decode("t1") is None and r.decode("t2") is None
    assert r.slots() == {0: "t1", 1: "t2"}
    # 2 + 2 <= 4: no flush, drafts go to slots 2 and 3
    assert r.verify(["d1", "d2"]) is None
    assert (r.head, r.len) == (0, 4) and r.slots() == {0: "t1", 1: "t2", 2: "d1", 3: "d2"}
    r.rollback(2, 1)
    assert (r.head, r.len) == (0, 3)
    # 3 + 1 >= 4: fold t1 t2 d1 and the current token; head = (0 + 3 + 1) mod 4
    assert r.decode("t3") == ["t1", "t2", "d1", "t3"]
    assert (r.head, r.len) == (0, 0)
    assert r.verify(["e1", "e2", "e3"]) is None
    r.rollback(3, 3)
    assert (r.head, r.len) == (0, 3)
    # 3 + 2 > 4: fold e1..e3 first, head = 3, drafts at slots 3 and 0
    assert r.verify(["f1", "f2"]) == ["e1", "e2", "e3"]
    assert (r.head, r.len) == (3, 2) and r.slots() == {3: "f1", 0: "f2"}
    r.rollback(2, 0)
    assert (r.head, r.len) == (3, 0)
    assert r.decode("t4") is None and r.slots() == {3: "t4"}
    assert r.flush() == ["t4"]
    assert (r.head, r.len) == (0, 0)


def test_decode_after_full_verify_folds_L_plus_one():
    """A verify may leave exactly L records; the next decode folds all of them
    plus the current token and moves head past all L + 1."""
    r = SeqRing(4)
    r.verify(["a", "b", "c", "d"])
    r.rollback(4, 4)
    assert r.decode("e") == ["a", "b", "c", "d", "e"]
    assert (r.head, r.len) == (1, 0)


def test_rollback_bounds():
    r = SeqRing(4)
    r.verify(["a", "b"])
    with pytest.raises(ValueError):
        r.rollback(2, 3)
    with pytest.raises(ValueError):
        r.rollback(3, 0)


def test_batch_masks():
    m = RingModel(3, 4)
    m.decode([1, 2, 3])
    out = m.flush([True, False, True])
    assert out == [[1], None, [3]]
    assert m.lens() == [0, 1, 0] and m.heads() == [1, 0, 1]
