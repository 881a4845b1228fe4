"""Iteration-level (continuous) batching on top of the block manager, and the
static-batching comparison.

Sources:

* "Continuous Batching" (ultralytics.com glossary), section "Cómo funciona la
  planificación a nivel de iteración": after each decode step the scheduler
  returns finished sequences, frees their memory and admits queued requests
  that fit in the KV cache; its worked example schedules eight requests on
  four slots (static batching runs each group of four until its longest
  member finishes; continuous batching starts the next request in the first
  slot that frees up).
* "Batching Continuo y PagedAttention" (cruxr.ai), sections "Batching
  continuo (In-Flight Batching)" and "Juntándolo todo: Arquitectura de
  vLLM": a running batch of at most B requests, a waiting queue, a block at
  admission, a new block when the current one fills, all blocks back to the
  pool at the end, and preemption when the pool runs dry.

``IterationScheduler.step()`` yields the metadata one decode step hands to
the device calls: the copy-on-write pairs, the append slots, and the block
tables and context lengths of the running batch.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field
from typing import Deque, Dict, List, Optional, Sequence, Tuple

import numpy as np

from .block_manager import BlockManager, NoFreeBlocks, blocks_needed


def slot_simulation(output_lengths: Sequence[int], slots: int, continuous: bool) -> List[float]:
    """Runs requests (each needing ``output_lengths[i]`` decode steps, in queue
    order) on ``slots`` slots, one decode step per loop iteration, and returns
    the fraction of busy slots at every step. Static batching admits the next
    ``slots`` requests only once every slot is idle; continuous batching
    refills any idle slot before each step."""
    queue = deque(output_lengths)
    left = [0] * slots                       # decode steps each slot's request still needs
    busy: List[float] = []
    while queue or any(left):
        if continuous or not any(left):
            for i in range(slots):
                if left[i] == 0 and queue:
                    left[i] = queue.popleft()
        if not any(left):                    # only zero-length requests were admitted
            continue
        busy.append(sum(1 for n in left if n > 0) / slots)
        left = [n - 1 if n > 0 else 0 for n in left]
    return busy


def static_batching(output_lengths: Sequence[int], slots: int) -> Tuple[int, float]:
    """Decode steps and mean slot occupancy when each group of ``slots``
    requests runs until its longest member finishes."""
    busy = slot_simulation(output_lengths, slots, continuous=False)
    return len(busy), sum(busy) / max(len(busy), 1)


def continuous_batching(output_lengths: Sequence[int], slots: int) -> Tuple[int, float]:
    """Decode steps and mean slot occupancy when a queued request takes any
    slot that is idle at the start of a step."""
    busy = slot_simulation(output_lengths, slots, continuous=True)
    return len(busy), sum(busy) / max(len(busy), 1)


def utilisation_traces(output_lengths: Sequence[int], slots: int) -> Tuple[List[float], List[float]]:
    """Per-step fraction of busy slots for static and continuous batching
    (queue order), without padding either trace to the other's length."""
    return (slot_simulation(output_lengths, slots, continuous=False),
            slot_simulation(output_lengths, slots, continuous=True))


@dataclass
class Request:
    req_id: int
    prompt_len: int
    output_len: int
    generated: int = 0
    parent: Optional[int] = None     # fork from this request's prompt (parallel sampling)


@dataclass
class StepBatch:
    """Device-call metadata of one decode step. The device runs it in this
    order: swap-in copies (host pool -> device), prefill of newly admitted
    sequences, swap-out copies (device -> host pool), copy-on-write copies,
    the KV append of one token per running sequence, then attention over the
    tables. (A sequence swapped in can be preempted again in the same step,
    and blocks a swap-out releases can be written by the copies and appends
    that follow, so no other order is safe.)"""
    seq_ids: List[int]
    cow_pairs: np.ndarray        # int64 [n, 2]
    slot_mapping: np.ndarray     # int64 [len(seq_ids)], one appended token per running sequence
    block_tables: np.ndarray     # int32 [len(seq_ids), maxB]
    context_lens: np.ndarray     # int32 [len(seq_ids)]
    finished: List[int] = field(default_factory=list)
    preempted: List[int] = field(default_factory=list)
    swap_out_pairs: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), dtype=np.int64))  # (device, host)
    swap_in_pairs: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), dtype=np.int64))   # (host, device)
    prefilled: List[Tuple[int, int, List[int]]] = field(default_factory=list)  # (sequence, tokens, its blocks)


class IterationScheduler:
    """Continuous batching over a paged KV pool.

    Each ``step()``: bring swapped-out sequences back first, then admit queued
    requests while a slot is free and the pool holds their prompt blocks;
    reserve one slot per running sequence (taking a new block only when the
    last is full, copying a shared partly filled block first); if the pool
    runs dry, preempt the most recently admitted sequence -- swap its blocks
    out to the host pool when one is configured and has room, otherwise free
    them and put the request back at the head of the queue to be recomputed;
    then retire the sequences that reached their output length.
    """

    def __init__(self, num_blocks: int, max_batch: int, block_size: int = 16,
                 order: Optional[np.ndarray] = None, host_blocks: int = 0):
        self.bm = BlockManager(num_blocks, block_size, order)
        self.host = BlockManager(host_blocks, block_size) if host_blocks else None
        self.max_batch = int(max_batch)
        self.waiting: Deque[Request] = deque()
        self.swapped: Deque[Request] = deque()
        self.running: List[Request] = []
        self.requests: Dict[int, Request] = {}
        self.steps = 0
        self.busy_slot_steps = 0
        self.preemptions = 0
        self.swaps = 0
        self._swap_out: List[Tuple[int, int]] = []
        self._swap_in: List[Tuple[int, int]] = []
        self._prefilled: List[Tuple[int, int, List[int]]] = []

    def add(self, req: Request) -> None:
        self.requests[req.req_id] = req
        self.waiting.append(req)

    def idle(self) -> bool:
        return not self.waiting and not self.running and not self.swapped

    def _admit(self) -> None:
        while self.swapped and len(self.running) < self.max_batch:
            req = self.swapped[0]
            if not self.bm.can_allocate(len(self.host.block_table(req.req_id))):
                return                      # swapped sequences go back before anything new
            self._swap_in += self.bm.swap_in(req.req_id, self.host)
            self.swapped.popleft()
            self.running.append(req)
        while self.waiting and len(self.running) < self.max_batch:
            req = self.waiting[0]
            parent = self.requests.get(req.parent) if req.parent is not None else None
            if (parent is not None and req.generated == 0 and parent.generated == 0
                    and self.bm.has_seq(req.parent)):
                # a fresh sample shares its parent's just-written prompt
                self.bm.fork(req.parent, req.req_id)
            else:
                # prefill writes the prompt (and anything generated before a preemption)
                need = blocks_needed(req.prompt_len + req.generated, self.bm.block_size)
                if not self.bm.can_allocate(need):
                    break
                self.bm.allocate(req.req_id, req.prompt_len + req.generated)
                self._prefilled.append((req.req_id, req.prompt_len + req.generated,
                                        self.bm.block_table(req.req_id)))
            self.waiting.popleft()
            self.running.append(req)

    def _preempt_one(self) -> Request:
        victim = self.running.pop()
        n = len(self.bm.block_table(victim.req_id))
        if self.host is not None and self.host.can_allocate(n):
            self._swap_out += self.bm.swap_out(victim.req_id, self.host)
            self.swapped.appendleft(victim)
            self.swaps += 1
        else:
            self.bm.free(victim.req_id)
            self.waiting.appendleft(victim)
        self.preemptions += 1
        return victim

    def step(self) -> Optional[StepBatch]:
        self._swap_out, self._swap_in, self._prefilled = [], [], []
        self._admit()
        if not self.running:
            return None
        pairs, slots, ids, preempted = [], [], [], []
        i = 0
        while i < len(self.running):
            req = self.running[i]
            try:
                slot, cow = self.bm.append_slot(req.req_id)
            except NoFreeBlocks:
                if len(self.running) == 1:
                    raise
                victim = self._preempt_one()
                preempted.append(victim.req_id)
                if victim is req:
                    break
                continue
            if cow is not None:
                pairs.append(cow)
            slots.append(slot)
            ids.append(req.req_id)
            i += 1
        # the preempted sequences' slots were released with their blocks
        keep = [k for k, s in enumerate(ids) if self.bm.has_seq(s)]
        ids = [ids[k] for k in keep]
        slots = [slots[k] for k in keep]
        tables, lens = self.bm.tables_array(ids)
        self.steps += 1
        self.busy_slot_steps += len(ids)
        finished = []
        for req in list(self.running):
            req.generated += 1
            if req.generated >= req.output_len:
                finished.append(req.req_id)
        as_pairs = lambda x: np.array(x, dtype=np.int64).reshape(-1, 2)
        return StepBatch(ids, as_pairs(pairs), np.array(slots, dtype=np.int64), tables, lens, finished, preempted,
                         as_pairs(self._swap_out), as_pairs(self._swap_in), list(self._prefilled))

    def retire(self, batch: StepBatch) -> None:
        """Free the blocks of the sequences the step finished."""
        done = set(batch.finished)
        for req in [r for r in self.running if r.req_id in done]:
            self.bm.free(req.req_id)
        self.running = [r for r in self.running if r.req_id not in done]

    def run(self, max_steps: int = 10 ** 7) -> Tuple[int, float]:
        """Drive until every request finished; returns (decode steps, slot occupancy)."""
        while not self.idle() and self.steps < max_steps:
            batch = self.step()
            if batch is None:
                raise RuntimeError("nothing runnable: the pool cannot hold a single waiting request")
            self.retire(batch)
        return self.steps, self.busy_slot_steps / (self.steps * self.max_batch)
