"""Brute-force linked-list LRU simulator of the swap-in step (test pin).

It computes the same swap-in semantics as the oracle by a different mechanism,
so a slip in the oracle's stamp arithmetic, tie-break or pairing shows up as a
mismatch:

  - there is no token->slot table: a token is found by scanning every slot;
  - there are no stamps: recency is a doubly linked list of slots, least
    recently used at the head.  It starts as 0, 1, ..., S-1 (all slots unused,
    lowest index first).  After a step the slots touched by it (hits and
    refilled victims) are unlinked and re-linked at the most-recent end in
    ascending slot order, because they share one last-use time and ties go to
    the lowest slot index;
  - victims are collected by walking from the head and skipping the slots hit
    in this step; they are then used in ascending slot order, paired with the
    misses in top-k row order.
  - with ``fifo=True`` only refilled slots move to the most-recent end: hits
    leave the order alone (first in, first out), but a slot hit in this step
    is still skipped as a victim.
  - with ``sliding=True`` the tail holds the last T tokens written; an append
    copies the leaving token's tail row into ``host_store`` first.
  - with ``alias=True`` a repeated token is not an error: it takes the slot of
    its first occurrence (several draft positions resolved together).

Semantics: HiSparse blog, "Efficient swap-in kernel" (miss detection, LRU
eviction, page-table update + host fetch); vLLM Hybrid HiSparse post, "Mixed
Residency" (tail read in place, hits refresh LRU, one row per miss).
"""


class LinkedLRU:
    def __init__(self, S, T, C, length, host_row, tail_row=None, fifo=False, sliding=False,
                 host_store=None, alias=False):
        self.alias = alias
        self.S, self.T, self.C, self.len = S, T, C, length
        self.fifo = fifo
        self.sliding = sliding
        self.host_store = host_store
        self.host_row = host_row          # token -> bytes
        self.content = [None] * S         # token held by each slot
        self.buf = [None] * (S + T)       # bytes per slot
        self.prev = [i - 1 for i in range(S)]
        self.next = [i + 1 if i + 1 < S else -1 for i in range(S)]
        self.head = 0 if S else -1
        self.tail = S - 1
        self.tail_row = tail_row

    def _unlink(self, s):
        p, n = self.prev[s], self.next[s]
        if p >= 0:
            self.next[p] = n
        else:
            self.head = n
        if n >= 0:
            self.prev[n] = p
        else:
            self.tail = p
        self.prev[s] = self.next[s] = -1

    def _push_back(self, s):
        self.prev[s] = self.tail
        self.next[s] = -1
        if self.tail >= 0:
            self.next[self.tail] = s
        else:
            self.head = s
        self.tail = s

    def order(self):
        out, s = [], self.head
        while s >= 0:
            out.append(s)
            s = self.next[s]
        return out

    def append(self, row):
        t = self.len
        if self.sliding:
            if self.T <= 0 or t >= self.C:
                return 1
            if t >= self.T:
                old = self.buf[self.S + t % self.T]
                if old is not None:
                    self.host_store[t - self.T] = old
            self.buf[self.S + t % self.T] = row
            self.len = t + 1
            return 0
        if self.T <= 0 or t < self.C - self.T or t >= self.C:
            return 1
        self.buf[self.S + t % self.T] = row
        self.len = t + 1
        return 0

    def step(self, topk):
        S, T, C = self.S, self.T, self.C
        tail0 = max(self.len - T, 0) if self.sliding else C - T
        out = [-1] * len(topk)
        err = 0
        hits, misses, inplace = [], [], 0
        repeats = []
        for j, t in enumerate(topk):
            if t == -1:
                continue
            if t < -1 or t >= self.len or t >= C:
                err |= 1
                continue
            earlier = [i for i in range(j) if topk[i] == t]
            if earlier:
                if self.alias:
                    repeats.append((j, earlier[0]))
                else:
                    err |= 2
                continue
            if t >= tail0:
                out[j] = S + t % T
                inplace += 1
                continue
            found = [s for s in range(S) if self.content[s] == t]
            if found:
                out[j] = found[0]
                hits.append(found[0])
            else:
                misses.append((t, j))
        hit_set = set(hits)
        victims = []
        s = self.head
        while s >= 0 and len(victims) < len(misses):
            if s not in hit_set:
                victims.append(s)
            s = self.next[s]
        assert len(victims) == len(misses), "not enough free slots"
        victims.sort()
        for (t, j), v in zip(misses, victims):
            self.content[v] = t
            self.buf[v] = self.host_row(t)
            out[j] = v
        for j, i in repeats:
            out[j] = out[i]
        touched = sorted(set(victims) if self.fifo else hit_set | set(victims))
        for s in touched:
            self._unlink(s)
        for s in touched:
            self._push_back(s)
        return out, (len(hits), len(misses), inplace), err
