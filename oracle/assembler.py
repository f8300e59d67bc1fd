"""Reference assembler of the reuse-time chunk table (TEST INFRASTRUCTURE ONLY: only tests/
may import it).  Plain Python, one dictionary for the registry, following the assembly loop of
"Irminsul论文详解" §5 (exact prefix first, then per CDC segment of the tail: carve-out prefill
below position 32, registry hit -> reuse with delta = p - p_src, else prefill and register)
and the S1 fallback of §6 (a missed CDC chunk is looked up again as fixed 128-token
sub-windows).  It shares no code with the library's C++ registry.

Readings (also listed in the design notes):
  - the registry key is the chunk's xxHash64 fingerprint together with its length;
  - registry rows live in a ring of `pool_rows` rows starting at `pool_base` in the row
    store: a chunk takes the next `len` rows of the ring (skipping to the ring's start when it
    would not fit before the end), and an entry is stale once the ring has moved a full turn
    past its first row;
  - an entry inserted while assembling a request is not a hit for later segments of the same
    request (its rows are only written by that request's own prefill);
  - S1: on a miss, the segment's 128-token sub-windows (aligned to the segment start, the last
    one shorter) are looked up; consecutive missed windows form one prefilled piece.  A segment
    takes ring rows for its whole length; its whole-segment key is registered only when all of
    it was prefilled (rows of reused windows are never written), and with S1 on each prefilled
    window registers its own key.
"""
from __future__ import annotations

import numpy as np

from . import chunk_fingerprint

CARVE_OUT = 32
S1_WINDOW = 128


class Registry:
    def __init__(self, pool_rows: int, pool_base: int = 0):
        self.pool_rows = int(pool_rows)
        self.pool_base = int(pool_base)
        self.cursor = 0          # rows ever allocated (ring position = cursor mod pool_rows)
        self.table = {}          # (hash, len) -> (cursor of first row, base_pos, call)
        self.call = 0

    def _alloc(self, n: int) -> int:
        if n > self.pool_rows:
            raise ValueError("chunk longer than the pool")
        pos = self.cursor % self.pool_rows
        if pos + n > self.pool_rows:            # do not wrap a chunk around the ring's end
            self.cursor += self.pool_rows - pos
        c = self.cursor
        self.cursor += n
        return c

    def _live(self, c: int) -> bool:
        return self.cursor <= c + self.pool_rows

    def _row(self, c: int) -> int:
        return self.pool_base + c % self.pool_rows

    def lookup(self, key):
        e = self.table.get(key)
        if e is None or not self._live(e[0]) or e[2] == self.call:
            return None
        return self._row(e[0]), e[1]

    def insert(self, key, c: int, base_pos: int):
        self.table[key] = (c, base_pos, self.call)

    def assemble(self, tokens, prefix_len: int, prefix_row: int, seg_start, seg_len, seg_hash,
                 s1: bool = False, seed: int = 0):
        """Chunk table of one request.  tokens: the request's token ids; segments: the CDC
        chunks of the tail tokens[prefix_len:], starts relative to the tail.  Returns a list of
        (pool_offset, len, p_src, p_tgt, reused, prefill)."""
        self.call += 1
        out = []
        if prefix_len > 0:
            out.append((prefix_row, prefix_len, 0, 0, 0, 0))
        for st, ln, h in zip(seg_start, seg_len, seg_hash):
            p = prefix_len + int(st)
            ln = int(ln)
            if p < CARVE_OUT:
                c = self._alloc(ln)
                out.append((self._row(c), ln, p, p, 0, 1))
                continue
            hit = self.lookup((int(h), ln))
            if hit is not None:
                row, base = hit
                out.append((row, ln, base, p, 1, 0))
                continue
            pieces = [(0, ln, None)]
            if s1:
                pieces = []
                for w0 in range(0, ln, S1_WINDOW):
                    wl = min(S1_WINDOW, ln - w0)
                    wh = chunk_fingerprint(tokens, p + w0, wl, seed)
                    pieces.append((w0, wl, self.lookup((wh, wl))))
            # emit hits as reused pieces, runs of missed pieces as one prefilled piece
            c = self._alloc(ln)  # rows for the whole segment (its prefill writes all of them)
            i = 0
            while i < len(pieces):
                w0, wl, hit = pieces[i]
                if hit is not None:
                    out.append((hit[0], wl, hit[1], p + w0, 1, 0))
                    i += 1
                    continue
                j = i
                while j < len(pieces) and pieces[j][2] is None:
                    j += 1
                a0 = pieces[i][0]
                a1 = pieces[j - 1][0] + pieces[j - 1][1]
                out.append((self._row(c + a0), a1 - a0, p + a0, p + a0, 0, 1))
                i = j
            if all(hit is None for _, _, hit in pieces):
                self.insert((int(h), ln), c, p)
            if s1:
                for w0 in range(0, ln, S1_WINDOW):
                    wl = min(S1_WINDOW, ln - w0)
                    if pieces[w0 // S1_WINDOW][2] is None:
                        self.insert((chunk_fingerprint(tokens, p + w0, wl, seed), wl), c + w0, p + w0)
        return out
