"""Oracle: the SWA prefix-hit rule ([SWA note], "prefix cache: tombstones and
the window hit rule").

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

A cached prefix may hold tokens whose full KV is alive but whose SWA KV was
evicted (tombstones).  Continuing prefill from a match end ``e`` needs the
SWA KV of the ``W`` tokens before ``e`` only, so ``e`` is usable iff those
tokens are live; otherwise the match falls back to the last usable position.
The validator walks from the root keeping a run counter that a tombstone
resets to 0.

Reading where the page is silent: near the root, where fewer than ``W``
tokens precede ``e``, ``e`` is usable iff all of them are live (the run
reaches the root); ``e = 0`` (no reuse) is always usable.
"""
from __future__ import annotations


def usable_positions(tombstone: list[bool], window: int) -> list[bool]:
    """``ok[e]`` for ``e = 0 .. n``: may a match end at ``e``?"""
    n = len(tombstone)
    ok = [True]
    run = 0
    reached_root = True
    for i in range(n):
        if tombstone[i]:
            run = 0
            reached_root = False
        else:
            run += 1
        ok.append(run >= window or reached_root)
    return ok


def match_end(tombstone: list[bool], matched_len: int, window: int) -> int:
    """Longest usable end ``<= matched_len``."""
    ok = usable_positions(tombstone[:matched_len], window)
    for e in range(matched_len, -1, -1):
        if ok[e]:
            return e
    return 0


def usable_brute(tombstone: list[bool], e: int, window: int) -> bool:
    """Direct statement: all of the tokens ``max(0, e - W) .. e - 1`` live."""
    return all(not tombstone[j] for j in range(max(0, e - window), e))
