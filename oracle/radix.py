"""Oracle: the radix prefix cache's SWA component ([SWA note], "prefix cache:
tombstones and the window hit rule").

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What the page states, and how it is taken here:

* a cached node may keep its full KV while its SWA KV was released: a
  *tombstone*.  Continuing a prefill from a match end ``e`` needs live SWA KV
  for the ``W`` tokens before ``e`` only, so a match ends at the last position
  that has ``min(e, W)`` live tokens before it (``oracle.hitrule``), here also
  a page boundary; ``W`` is the SWA layers' lookback.
* two LRU lists: full eviction deletes leaf nodes (full and SWA KV); SWA
  eviction releases a node's SWA KV and turns it into a tombstone.  A leaf may
  not be a tombstone, so SWA eviction of a leaf deletes it, and a tombstone
  left without children is deleted too.
* locks: a request using a prefix full-locks every node up to the root, but
  SWA-locks only the nodes holding the last ``W`` tokens before its match end;
  earlier nodes can still lose their SWA KV.
* insert at request end: ``[0, swa_evicted)`` has no SWA KV and goes in as a
  tombstone prefix (only ahead of live tokens: never as a leaf); where the new
  request has SWA KV over a tombstone node, the node takes the request's slots
  and is live again (its old slots are released).

Readings where the page is silent (the same in the C++ tree):

* keys are token ids; the tree works in whole pages (match and insert use
  ``floor(len / ps) * ps`` tokens; a trailing partial page is the caller's);
* a match that ends inside a node splits it, so the match ends on a node
  boundary; every node on the matched path gets the current time stamp in
  both lists; inserting stamps the nodes it passes or creates;
* where an inserted request duplicates tokens already cached (live, or
  tombstone with the request evicted there too), the request's slots are
  released, unless they are the node's own (the request took its prefix from
  the tree); ties in LRU order go to the older node (creation order).
* releases are reported, not performed: ``released_full`` lists full slots
  whose full and SWA KV (if mapped) go back (``free``), ``released_swa`` full
  slots whose SWA KV only goes back (``free_swa``), each with page counts.
"""
from __future__ import annotations

from . import hitrule


class Node:
    __slots__ = ("key", "full", "tomb", "children", "parent", "full_lock", "swa_lock",
                 "t_full", "t_swa", "id")

    def __init__(self, key, full, tomb, parent, nid, t):
        self.key = list(key)
        self.full = list(full)
        self.tomb = bool(tomb)
        self.children = {}
        self.parent = parent
        self.full_lock = 0
        self.swa_lock = 0
        self.t_full = t
        self.t_swa = t
        self.id = nid


class RadixSWA:
    def __init__(self, page_size: int, window: int):
        self.ps = int(page_size)
        self.W = int(window)
        self.clock = 0
        self.next_id = 1
        self.root = Node([], [], False, None, 0, 0)
        self.nodes = {0: self.root}
        self.released_full: list[int] = []
        self.released_swa: list[int] = []

    # -- helpers -------------------------------------------------------------
    def _tick(self):
        self.clock += 1
        return self.clock

    def _page(self, key, i):
        return tuple(key[i:i + self.ps])

    def _new(self, key, full, tomb, parent):
        n = Node(key, full, tomb, parent, self.next_id, self.clock)
        self.next_id += 1
        self.nodes[n.id] = n
        parent.children[self._page(n.key, 0)] = n
        return n

    def _split(self, node, k):
        """Node keeps key[k:]; a new parent takes key[:k] (k a page multiple)."""
        parent = node.parent
        top = Node(node.key[:k], node.full[:k], node.tomb, parent, self.next_id, node.t_full)
        self.next_id += 1
        top.t_swa = node.t_swa
        top.full_lock = node.full_lock
        top.swa_lock = node.swa_lock
        self.nodes[top.id] = top
        parent.children[self._page(top.key, 0)] = top
        node.key = node.key[k:]
        node.full = node.full[k:]
        node.parent = top
        top.children[self._page(node.key, 0)] = node
        return top

    def _release(self, slots, swa_only=False):
        (self.released_swa if swa_only else self.released_full).extend(int(s) for s in slots)

    def _delete(self, node):
        del node.parent.children[self._page(node.key, 0)]
        del self.nodes[node.id]

    def take_releases(self):
        f, s = self.released_full, self.released_swa
        self.released_full, self.released_swa = [], []
        return f, s

    # -- match -----------------------------------------------------------------
    def match(self, tokens):
        """Returns (e, slots of tokens[0:e], id of the node ending at e)."""
        n = (len(tokens) // self.ps) * self.ps
        key = list(tokens[:n])
        now = self._tick()
        path = []           # (node, tokens of it matched)
        node, pos = self.root, 0
        while pos < n:
            child = node.children.get(self._page(key, pos))
            if child is None:
                break
            c = 0
            while (c < len(child.key) and pos + c < n
                   and child.key[c:c + self.ps] == key[pos + c:pos + c + self.ps]):
                c += self.ps
            path.append((child, c))
            pos += c
            if c < len(child.key):
                break
            node = child
        tomb = []
        for nd, c in path:
            tomb += [nd.tomb] * c
        ok = hitrule.usable_positions(tomb, self.W)
        e = pos
        while e > 0 and not ok[e]:
            e -= self.ps
        # the nodes up to e; split the one e falls inside
        acc, end, slots = 0, self.root, []
        for nd, c in path:
            if acc >= e:
                break
            take = min(len(nd.key), e - acc)
            if take < len(nd.key):
                nd = self._split(nd, take)
            slots += nd.full
            nd.t_full = nd.t_swa = now
            acc += take
            end = nd
        return e, slots, end.id

    # -- locks -----------------------------------------------------------------
    def lock(self, nid):
        """Full-lock the path from node ``nid`` to the root and SWA-lock the
        nodes holding the last W tokens; returns the SWA-locked span (tokens),
        which ``unlock`` needs: a later split can move a node boundary, but it
        copies the counts, so walking the same span finds the same tokens."""
        nd, acc, span = self.nodes[nid], 0, 0
        while nd is not self.root:
            nd.full_lock += 1
            if acc < self.W:
                nd.swa_lock += 1
                span = acc + len(nd.key)
            acc += len(nd.key)
            nd = nd.parent
        return span

    def unlock(self, nid, swa_span):
        nd, acc = self.nodes[nid], 0
        while nd is not self.root:
            nd.full_lock -= 1
            if acc < swa_span:
                nd.swa_lock -= 1
            acc += len(nd.key)
            nd = nd.parent

    # -- insert ----------------------------------------------------------------
    def insert(self, tokens, slots, swa_evicted):
        n = (len(tokens) // self.ps) * self.ps
        key, val = list(tokens[:n]), [int(s) for s in slots[:n]]
        ev = min(int(swa_evicted), n)
        now = self._tick()
        node, pos = self.root, 0
        while pos < n:
            child = node.children.get(self._page(key, pos))
            if child is None:
                break
            c = 0
            while (c < len(child.key) and pos + c < n
                   and child.key[c:c + self.ps] == key[pos + c:pos + c + self.ps]):
                c += self.ps
            if c < len(child.key):
                child = self._split(child, c)
            if child.tomb and pos < ev < pos + c:
                # the request has SWA KV from ev on: treat the two parts apart
                self._split(child, ev - pos)
                continue
            if child.full == val[pos:pos + c]:
                pass                                      # the request's prefix came from here
            elif child.tomb and pos >= ev:
                self._release(child.full)                 # old slots: no SWA KV left
                child.full = val[pos:pos + c]             # the node is live again
                child.tomb = False
            else:
                self._release(val[pos:pos + c])           # duplicate of cached tokens
            child.t_full = child.t_swa = now
            node, pos = child, pos + c
        if pos < n:
            if pos < ev:
                if ev < n:                                # a tombstone only ahead of live tokens
                    node = self._new(key[pos:ev], val[pos:ev], True, node)
                    pos = ev
                else:
                    self._release(val[pos:n])
                    return
            self._new(key[pos:n], val[pos:n], False, node)

    # -- eviction ----------------------------------------------------------------
    def _drop_leaf(self, leaf):
        """Delete a leaf (full + SWA released), then any tombstone it leaves
        childless above it."""
        freed = len(leaf.key)
        self._release(leaf.full)
        parent = leaf.parent
        self._delete(leaf)
        while parent is not self.root and not parent.children and parent.tomb:
            freed += len(parent.key)
            self._release(parent.full)
            up = parent.parent
            self._delete(parent)
            parent = up
        return freed

    def evict_full(self, n_tokens):
        freed = 0
        while freed < n_tokens:
            cand = [nd for nd in self.nodes.values()
                    if nd is not self.root and not nd.children and nd.full_lock == 0]
            if not cand:
                break
            leaf = min(cand, key=lambda x: (x.t_full, x.id))
            freed += self._drop_leaf(leaf)
        return freed

    def evict_swa(self, n_tokens):
        freed = 0
        while freed < n_tokens:
            cand = [nd for nd in self.nodes.values()
                    if nd is not self.root and not nd.tomb and nd.swa_lock == 0
                    and (nd.children or nd.full_lock == 0)]
            if not cand:
                break
            nd = min(cand, key=lambda x: (x.t_swa, x.id))
            freed += len(nd.key)
            if nd.children:
                self._release(nd.full, swa_only=True)
                nd.tomb = True
            else:
                self._drop_leaf(nd)
        return freed

    # -- inspection ----------------------------------------------------------------
    def cached_tokens(self):
        return sum(len(nd.key) for nd in self.nodes.values())

    def live_tokens(self):
        return sum(len(nd.key) for nd in self.nodes.values() if not nd.tomb)

    def check(self):
        """Invariants: no tombstone leaf; keys a page multiple; slots unique."""
        seen = set()
        for nd in self.nodes.values():
            if nd is self.root:
                continue
            assert len(nd.key) % self.ps == 0 and len(nd.key) == len(nd.full) > 0
            assert nd.children or not nd.tomb, "tombstone leaf"
            assert nd.full_lock >= 0 and nd.swa_lock >= 0
            for s in nd.full:
                assert s not in seen
                seen.add(s)
        return seen
