"""KV-cache reorder by beam_idx: naive gather and paged block table with copy-on-write.

TEST INFRASTRUCTURE.  Imported only by tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference arm; shares no code with the CUDA library.

What it follows: "9.2 贪心搜索与束搜索：确定性与近似搜索" (llm_internals):

* §9.2.2, the KV paragraph: after a step, new beam r reads the cache of its
  parent beam_idx[r]; the naive way gathers every layer's K and V by beam_idx
  (a parent with two children is copied twice); a paged cache instead rewrites
  block-table pointers and copies only when a shared block is written.
* §9.2.4: prompt sharing; with P prompt tokens and t generated, naive storage is
  W(P + t) tokens while sharing needs at most P + W t.

Cache layout (naive): [L, 2, rows, H, T_max, D], K at index 0 and V at 1.
Paged pool: [N_blocks, L, 2, H, block, D]; table[r][i] is the pool block that
holds row r's positions [i*block, (i+1)*block).

Readings
--------
K1 A row with beam_idx = -1 (a finished sentence's pad row) is not written.
K2 Copy-on-write is done eagerly, right after the remap, for the block that the
   next write (position t_valid) lands in; every live row writes there next, so
   this equals copying at write time.  Of the rows sharing that block, the
   lowest row keeps it and every other row copies its filled slots
   (t_valid mod block) into a fresh block.  A row whose next write starts a new
   block gets a fresh block, with nothing to copy.
K3 Blocks are never shared across sentences, so each sentence draws from its own
   sub-pool (a LIFO free stack); which physical block a row gets is not part of
   the contract, only the logical contents and the block counts are.
"""

from __future__ import annotations

import numpy as np


def reorder_naive(src: np.ndarray, dst: np.ndarray, beam_idx, t_valid: int) -> np.ndarray:
    """dst[:, :, r, :, :t_valid] = src[:, :, beam_idx[r], :, :t_valid] for live rows (K1)."""
    out = np.array(dst, copy=True)
    for r, p in enumerate(np.asarray(beam_idx)):
        if p >= 0:
            out[:, :, r, :, :t_valid, :] = src[:, :, int(p), :, :t_valid, :]
    return out


class PagedKV:
    """Reference model of a paged KV cache for B sentences x W rows (K2, K3)."""

    def __init__(self, B: int, W: int, blocks_per_sentence: int, L: int, H: int, D: int,
                 block: int = 16, dtype=np.float32):
        self.B, self.W, self.S, self.block = B, W, blocks_per_sentence, block
        self.pool = np.zeros((B * blocks_per_sentence, L, 2, H, block, D), dtype=dtype)
        self.tables = [[] for _ in range(B * W)]
        self.refcnt = np.zeros(B * blocks_per_sentence, dtype=np.int64)
        self.free = [list(range((b + 1) * blocks_per_sentence - 1, b * blocks_per_sentence - 1, -1))
                     for b in range(B)]
        self.copied_slots = 0      # filled slots copied by copy-on-write, summed

    def _alloc(self, b: int) -> int:
        if not self.free[b]:
            raise MemoryError(f"sentence {b}: sub-pool exhausted")
        blk = self.free[b].pop()
        self.refcnt[blk] = 1
        return blk

    def _release(self, blk: int):
        self.refcnt[blk] -= 1
        assert self.refcnt[blk] >= 0
        if self.refcnt[blk] == 0:
            self.free[blk // self.S].append(blk)

    def prefill(self, P: int):
        """Allocate the prompt's blocks once per sentence and point all W rows at them."""
        nb = -(-P // self.block)
        for b in range(self.B):
            blocks = [self._alloc(b) for _ in range(nb)]
            for blk in blocks:
                self.refcnt[blk] = self.W
            for w in range(self.W):
                self.tables[b * self.W + w] = list(blocks)

    def prepare(self, t_write: int):
        """Give every row exclusive ownership of the block that position t_write lands in (K2)."""
        self._prepare(range(self.B), t_write)

    def reorder(self, beam_idx, t_valid: int):
        """Remap tables by beam_idx (K1), drop the old references, then prepare(t_valid)."""
        beam_idx = np.asarray(beam_idx)
        old = [list(t) for t in self.tables]
        for r, p in enumerate(beam_idx):
            if p >= 0:
                self.tables[r] = list(old[int(p)])
                for blk in self.tables[r]:
                    self.refcnt[blk] += 1
        for r, p in enumerate(beam_idx):
            if p >= 0:
                for blk in old[r]:
                    self._release(blk)
        live = [b for b in range(self.B) if (beam_idx[b * self.W:(b + 1) * self.W] >= 0).any()]
        self._prepare(live, t_valid)

    def _prepare(self, sentences, t_write: int):
        i, fill = divmod(t_write, self.block)
        for b in sentences:
            kept = set()
            for r in range(b * self.W, (b + 1) * self.W):          # ascending: lowest row keeps
                tab = self.tables[r]
                if len(tab) == i:
                    tab.append(self._alloc(b))                     # fresh block, nothing to copy
                    continue
                assert len(tab) == i + 1, "the table must cover [0, t_write) exactly"
                blk = tab[i]
                if self.refcnt[blk] == 1:
                    continue
                if blk not in kept:
                    kept.add(blk)
                    continue
                new = self._alloc(b)
                self.pool[new, :, :, :, :fill, :] = self.pool[blk, :, :, :, :fill, :]
                self.copied_slots += fill
                self.refcnt[blk] -= 1
                tab[i] = new

    def write(self, t_write: int, values: np.ndarray, rows=None):
        """The model's write of one position: values [L, 2, R, H, D] (rows = all by default)."""
        i, s = divmod(t_write, self.block)
        rows = range(len(self.tables)) if rows is None else rows
        for n, r in enumerate(rows):
            self.pool[self.tables[r][i], :, :, :, s, :] = values[:, :, n, :, :]

    def logical(self, t_valid: int) -> np.ndarray:
        """The cache as a naive [L, 2, R, H, t_valid, D] array, read through the tables.

        Positions a row's table does not cover (a finished sentence stops growing) read 0.
        """
        R = len(self.tables)
        _, L, _, H, _, D = self.pool.shape
        out = np.zeros((L, 2, R, H, t_valid, D), dtype=self.pool.dtype)
        for r in range(R):
            for pos in range(min(t_valid, len(self.tables[r]) * self.block)):
                i, s = divmod(pos, self.block)
                out[:, :, r, :, pos, :] = self.pool[self.tables[r][i], :, :, :, s, :]
        return out

    def blocks_in_use(self) -> int:
        return int((self.refcnt > 0).sum())

    def check_refcounts(self):
        """Every block's count equals the number of table entries naming it."""
        cnt = np.zeros_like(self.refcnt)
        for tab in self.tables:
            for blk in tab:
                cnt[blk] += 1
        return bool((cnt == self.refcnt).all())
