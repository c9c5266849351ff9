"""Integer model of the per-sequence ring of input records -- the oracle.

TEST INFRASTRUCTURE (see the package docstring): never imported by the product.

The method keeps, beside each sequence's checkpoint, a buffer of at most L
per-token input records; normal steps append one record, and every L steps a
flush folds the buffer into the checkpoint ([AT Pulse] §What happened and
§Technical analysis, core idea; [WittyWires] §What happened: the checkpoint is
updated when the buffer fills).  Speculative decoding appends draft records
and discards rejected ones by moving the buffer pointer ([AT Pulse]
§Technical analysis, speculative decoding).

The pages do not give the flush rule in full (one page's text stops where the
buffer fills).  The readings modelled here:

* ring slot of logical record j (0 = oldest) is (head + j) mod L;
* decode: with len records buffered, the current token is record len+1.  If
  len + 1 >= L the step folds all buffered records and the current token into
  the checkpoint, does not store the current token, and leaves the ring empty
  with head advanced past every folded token: head <- (head + len + 1) mod L,
  len <- 0.  Otherwise the record goes to slot (head + len) mod L and
  len <- len + 1.  From an empty ring this flushes on steps L, 2L, ...
  (64 decode steps with L = 16 give 4 flushes);
* verify with T drafts: if len + T > L, first fold the len buffered records
  (head <- (head + len) mod L, len <- 0); then append the T drafts at slots
  (head + len + i) mod L and len <- len + T.  Drafts are never folded by a
  verify, so that rejecting them stays a pointer move;
* rollback after a verify of T drafts with a accepted (0 <= a <= T):
  len <- len - (T - a).  Rejected records stay in memory, unread;
* standalone flush of a sequence: fold its len records, head <- (head + len)
  mod L, len <- 0.

Each buffered record is tracked by an opaque tag (the caller's token id), so
the tests can check the ring's slot contents bit for bit.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass
class SeqRing:
    L: int
    head: int = 0
    tags: list = field(default_factory=list)   # buffered records, oldest first

    @property
    def len(self) -> int:
        return len(self.tags)

    def slot(self, j: int) -> int:
        return (self.head + j) % self.L

    def slots(self) -> dict:
        """physical slot -> tag of every buffered record."""
        return {self.slot(j): t for j, t in enumerate(self.tags)}

    # --- operations; each returns the tags folded into the checkpoint (or None)
    def decode(self, tag):
        if self.len + 1 >= self.L:
            folded = self.tags + [tag]
            self.head = (self.head + self.len + 1) % self.L
            self.tags = []
            return folded
        self.tags.append(tag)
        return None

    def verify(self, draft_tags):
        folded = None
        if self.len + len(draft_tags) > self.L:
            folded = self.tags
            self.head = (self.head + self.len) % self.L
            self.tags = []
        self.tags = self.tags + list(draft_tags)
        return folded

    def rollback(self, T: int, accepted: int) -> None:
        if not (0 <= accepted <= T) or self.len < T - accepted:
            raise ValueError("rollback outside the last verify's drafts")
        keep = self.len - (T - accepted)
        self.tags = self.tags[:keep]

    def flush(self):
        folded = self.tags
        self.head = (self.head + self.len) % self.L
        self.tags = []
        return folded


class RingModel:
    """One SeqRing per sequence of the batch."""

    def __init__(self, batch: int, L: int):
        self.seqs = [SeqRing(L) for _ in range(batch)]

    def heads(self):
        return [s.head for s in self.seqs]

    def lens(self):
        return [s.len for s in self.seqs]

    def decode(self, tags):
        return [s.decode(t) for s, t in zip(self.seqs, tags)]

    def verify(self, draft_tags):
        return [s.verify(d) for s, d in zip(self.seqs, draft_tags)]

    def rollback(self, T, accepted):
        for s, a in zip(self.seqs, accepted):
            s.rollback(T, int(a))

    def flush(self, mask=None):
        return [s.flush() if (mask is None or mask[i]) else None
                for i, s in enumerate(self.seqs)]
