"""Host-side KV block manager: the free pool, per-sequence block tables,
reference-counted sharing and copy-on-write.

Sources (pages on PagedAttention and continuous batching):

* "Batching Continuo y PagedAttention" (cruxr.ai), section "PagedAttention:
  Memoria virtual para la KV cache": KV memory is cut into fixed blocks of
  P = 16 tokens; each request keeps a page table from logical block index to
  physical block; a scheduled request receives one block, a new block comes
  from the free pool when the current one is full, and every block returns
  to the pool when the request finishes.  A request of L tokens holds
  ceil(L / P) blocks, and only its last block has unused slots.
* same page, copy-on-write paragraph: requests with a common prefix point
  their tables at the same physical blocks, like Unix ``fork()``.
* iplexlaw.co.kr "pagedattention-vllm-kv-cache", section "Dos respuestas a
  una entrada: ejemplo hipotético": a shared block with free room is copied
  when written while other references exist; full shared blocks stay
  shared; blocks without references are freed.
* "PagedAttention: gestionar la KV cache como memoria de un sistema
  operativo" (josueisai.com), section "Cómo funciona por dentro": append
  asks for a new block only when the last one is full; any free block will
  do.

The manager produces exactly what the device calls consume: int32 block
tables, int32 context lengths, int64 slot numbers (block * 16 + offset) for
the KV append, and int64 (src, dst) pairs for the block copy.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field
from typing import Deque, Dict, List, Optional, Tuple

import numpy as np

BLOCK_SIZE = 16


class NoFreeBlocks(RuntimeError):
    """The pool cannot satisfy an allocation (the scheduler must preempt or wait)."""


def blocks_needed(num_tokens: int, block_size: int = BLOCK_SIZE) -> int:
    """ceil(L / P): the blocks a sequence of L tokens holds."""
    return -(-int(num_tokens) // block_size)


@dataclass
class _Seq:
    table: List[int] = field(default_factory=list)
    length: int = 0


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE, order: Optional[np.ndarray] = None):
        """``order``: optional permutation giving the free pool's hand-out order
        (a shuffled pool); by default blocks are handed out 0, 1, 2, ..."""
        if num_blocks <= 0:
            raise ValueError("num_blocks must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        ids = range(self.num_blocks) if order is None else [int(b) for b in order]
        self._free: Deque[int] = deque(ids)
        if sorted(self._free) != list(range(self.num_blocks)):
            raise ValueError("order must be a permutation of the pool")
        self.refcount = np.zeros(self.num_blocks, dtype=np.int64)
        self._seqs: Dict[int, _Seq] = {}

    # -- pool ---------------------------------------------------------------
    @property
    def num_free(self) -> int:
        return len(self._free)

    def can_allocate(self, n_blocks: int) -> bool:
        return n_blocks <= len(self._free)

    def _alloc(self) -> int:
        if not self._free:
            raise NoFreeBlocks("KV block pool exhausted")
        b = self._free.popleft()
        self.refcount[b] = 1
        return b

    def _decref(self, b: int) -> None:
        self.refcount[b] -= 1
        if self.refcount[b] < 0:
            raise AssertionError(f"block {b} released more often than referenced")
        if self.refcount[b] == 0:
            self._free.append(b)

    # -- sequences ----------------------------------------------------------
    def has_seq(self, seq_id: int) -> bool:
        return seq_id in self._seqs

    def allocate(self, seq_id: int, num_tokens: int = 0) -> List[int]:
        """Admit a sequence whose first ``num_tokens`` (its prompt) are written
        by prefill: ceil(num_tokens / P) blocks, all or nothing."""
        if seq_id in self._seqs:
            raise ValueError(f"sequence {seq_id} already allocated")
        need = blocks_needed(num_tokens, self.block_size)
        if not self.can_allocate(need):
            raise NoFreeBlocks(f"need {need} blocks, {self.num_free} free")
        seq = _Seq([self._alloc() for _ in range(need)], int(num_tokens))
        self._seqs[seq_id] = seq
        return list(seq.table)

    def fork(self, parent_id: int, child_id: int) -> None:
        """The child shares every block of the parent (no copy yet)."""
        if child_id in self._seqs:
            raise ValueError(f"sequence {child_id} already allocated")
        p = self._seqs[parent_id]
        for b in p.table:
            self.refcount[b] += 1
        self._seqs[child_id] = _Seq(list(p.table), p.length)

    def append_slot(self, seq_id: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserve the slot of the sequence's next token.

        Returns ``(slot, cow)``: ``slot = block * P + offset`` for the KV
        append, and ``cow = (src, dst)`` when the last block was shared and
        partly filled, so it had to be copied before this write (otherwise
        None).  A new block is taken only when the last one is full.
        """
        seq = self._seqs[seq_id]
        off = seq.length % self.block_size
        cow = None
        if not seq.table or (off == 0 and seq.length >= len(seq.table) * self.block_size):
            seq.table.append(self._alloc())
        else:
            last = seq.table[-1]
            if self.refcount[last] > 1:
                dst = self._alloc()
                self._decref(last)
                seq.table[-1] = dst
                cow = (last, dst)
        slot = seq.table[-1] * self.block_size + off
        seq.length += 1
        return slot, cow

    def swap_out(self, seq_id: int, host: "BlockManager") -> List[Tuple[int, int]]:
        """Moves a sequence to a host pool (preemption by swapping, "Juntándolo
        todo: Arquitectura de vLLM"): one host block per table entry, all or
        nothing; returns the (device block, host block) pairs to copy, then
        releases the device blocks (freed when no other table refers to
        them). The sequence's length and table now live in ``host``."""
        seq = self._seqs[seq_id]
        if not host.can_allocate(len(seq.table)):
            raise NoFreeBlocks(f"host pool: need {len(seq.table)} blocks, {host.num_free} free")
        host_table = [host._alloc() for _ in seq.table]
        host._seqs[seq_id] = _Seq(host_table, seq.length)
        pairs = list(zip(seq.table, host_table))
        self.free(seq_id)
        return pairs

    def swap_in(self, seq_id: int, host: "BlockManager") -> List[Tuple[int, int]]:
        """Brings a swapped-out sequence back: fresh device blocks, all or
        nothing; returns the (host block, device block) pairs to copy and
        frees the host blocks."""
        hseq = host._seqs[seq_id]
        if seq_id in self._seqs:
            raise ValueError(f"sequence {seq_id} is already resident")
        if not self.can_allocate(len(hseq.table)):
            raise NoFreeBlocks(f"need {len(hseq.table)} blocks, {self.num_free} free")
        table = [self._alloc() for _ in hseq.table]
        self._seqs[seq_id] = _Seq(table, hseq.length)
        pairs = list(zip(hseq.table, table))
        host.free(seq_id)
        return pairs

    def free(self, seq_id: int) -> None:
        """Release all of a finished (or preempted) sequence's blocks."""
        seq = self._seqs.pop(seq_id)
        for b in seq.table:
            self._decref(b)

    def block_table(self, seq_id: int) -> List[int]:
        return list(self._seqs[seq_id].table)

    def context_len(self, seq_id: int) -> int:
        return self._seqs[seq_id].length

    def seq_ids(self) -> List[int]:
        return list(self._seqs)

    def tables_array(self, seq_ids: List[int], fill: int = 0) -> Tuple[np.ndarray, np.ndarray]:
        """int32 block tables [len(seq_ids), maxB] (unused entries = ``fill``)
        and int32 context lengths, as the decode call takes them."""
        maxb = max([len(self._seqs[s].table) for s in seq_ids] + [1])
        tables = np.full((len(seq_ids), maxb), fill, dtype=np.int32)
        lens = np.zeros(len(seq_ids), dtype=np.int32)
        for i, s in enumerate(seq_ids):
            t = self._seqs[s].table
            tables[i, :len(t)] = t
            lens[i] = self._seqs[s].length
        return tables, lens

    def check_invariants(self) -> None:
        """Every referenced block is counted once per referencing table; free
        blocks have no references; each table has ceil(len / P) blocks."""
        counts = np.zeros(self.num_blocks, dtype=np.int64)
        for seq in self._seqs.values():
            if len(seq.table) != blocks_needed(seq.length, self.block_size):
                raise AssertionError("table length differs from ceil(len / P)")
            for b in seq.table:
                counts[b] += 1
        if not np.array_equal(counts, self.refcount):
            raise AssertionError("reference counts differ from table references")
        free = set(self._free)
        if len(free) != len(self._free):
            raise AssertionError("a block is twice in the free pool")
        for b in range(self.num_blocks):
            if (b in free) != (counts[b] == 0):
                raise AssertionError(f"block {b}: free-pool membership disagrees with its references")


# -- byte accounting ("El problema de fragmentación de la KV cache" and
#    "PagedAttention: Memoria virtual para la KV cache", cruxr.ai) ----------

def kv_bytes_per_request(num_layers: int, num_heads: int, head_dim: int, num_tokens: int,
                         elem_bytes: int) -> int:
    """KV cache of one request at position t: 2 (K and V) x L x h x d_h x t x bytes."""
    return 2 * num_layers * num_heads * head_dim * num_tokens * elem_bytes


def padding_waste_fraction(mean_len: float, max_len: float) -> float:
    """Share of slots spent on padding under static batching (or on reserved,
    untouched memory under pre-allocation): 1 - mean / max."""
    return 1.0 - mean_len / max_len


def last_block_waste_bound(num_tokens: int, block_size: int = BLOCK_SIZE) -> float:
    """Upper bound on the per-request waste fraction under paging as the page
    states it: P / L (the true maximum number of unused slots is P - 1)."""
    return block_size / num_tokens


def unused_slots(num_tokens: int, block_size: int = BLOCK_SIZE) -> int:
    """Slots allocated but not filled: ceil(L / P) * P - L (at most P - 1)."""
    return blocks_needed(num_tokens, block_size) * block_size - int(num_tokens)


def cow_savings_bytes(prefix_tokens: int, num_requests: int, bytes_per_token: float) -> float:
    """Memory saved by sharing a prefix of S tokens among N requests: (N - 1) * S * c."""
    return (num_requests - 1) * prefix_tokens * bytes_per_token
