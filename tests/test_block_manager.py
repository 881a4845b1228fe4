"""Host block manager, scheduler simulation and byte accounting, pinned to
the pages' worked numbers (tests/golden/) and to the paging invariants."""
import json
import os
import random

import numpy as np
import pytest

from paged_kv_cache_177_gb300 import block_manager as bmod
from paged_kv_cache_177_gb300 import scheduler as sched
from paged_kv_cache_177_gb300.block_manager import BlockManager, NoFreeBlocks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --- the pages' scheduling example ------------------------------------------------

def test_static_and_continuous_match_the_worked_example():
    g = golden("scheduling_example.json")
    steps, busy = sched.static_batching(g["output_lengths"], g["slots"])
    assert steps == g["static_steps"]
    assert round(100 * busy) == g["static_busy_percent"]
    steps, busy = sched.continuous_batching(g["output_lengths"], g["slots"])
    assert steps == g["continuous_steps"]
    assert round(100 * busy) == g["continuous_busy_percent"]


def test_iteration_scheduler_over_paged_pool_matches_the_example():
    """The block-managed scheduler, with ample memory, schedules the example
    in the same 50 steps at 78% occupancy."""
    g = golden("scheduling_example.json")
    s = sched.IterationScheduler(num_blocks=64, max_batch=g["slots"])
    for i, n in enumerate(g["output_lengths"]):
        s.add(sched.Request(i, prompt_len=0, output_len=n))
    steps, busy = s.run()
    assert steps == g["continuous_steps"]
    assert round(100 * busy) == g["continuous_busy_percent"]
    assert s.bm.num_free == 64 and s.preemptions == 0


def test_scheduler_preempts_under_memory_pressure_and_finishes():
    rng = random.Random(5)
    lengths = [rng.randint(10, 120) for _ in range(24)]
    s = sched.IterationScheduler(num_blocks=20, max_batch=8)
    for i, n in enumerate(lengths):
        s.add(sched.Request(i, prompt_len=rng.randint(1, 40), output_len=n))
    while not s.idle():
        b = s.step()
        assert b is not None
        assert s.bm.num_free >= 0
        # every reserved slot sits inside its sequence's table at position len - 1
        for i, sid in enumerate(b.seq_ids):
            n = int(b.context_lens[i])
            blk = int(b.block_tables[i, (n - 1) // 16])
            assert int(b.slot_mapping[i]) == blk * 16 + (n - 1) % 16
        s.bm.check_invariants()
        s.retire(b)
    assert s.preemptions > 0
    assert s.bm.num_free == 20


def test_utilisation_traces_show_continuous_above_static():
    """The 24-request right-skewed simulation: continuous batching keeps more
    slots busy than static batching (without padding either trace)."""
    rng = random.Random(42)
    lengths = [rng.randint(10, 40) if rng.random() < 0.7 else rng.randint(80, 150) for _ in range(24)]
    st, ct = sched.utilisation_traces(lengths, 8)
    assert sum(st) * 8 == pytest.approx(sum(lengths))
    assert sum(ct) * 8 == pytest.approx(sum(lengths))
    assert len(ct) < len(st)
    assert sum(ct) / len(ct) > sum(st) / len(st)
    steps, _ = sched.static_batching(lengths, 8)
    assert steps == len(st)


# --- block manager --------------------------------------------------------------------

@pytest.mark.parametrize("n", [0, 1, 15, 16, 17, 31, 32, 33, 1000, 4096])
def test_block_count_is_ceil_len_over_16(n):
    bm = BlockManager(300)
    bm.allocate(0, n)
    assert len(bm.block_table(0)) == -(-n // 16)
    bm.check_invariants()
    # growing token by token keeps the invariant and allocates only on a full block
    before = len(bm.block_table(0))
    for k in range(40):
        slot, cow = bm.append_slot(0)
        assert cow is None
        assert len(bm.block_table(0)) == -(-(n + k + 1) // 16)
        if (n + k) % 16 == 0:
            assert len(bm.block_table(0)) == before + 1
        before = len(bm.block_table(0))
        bm.check_invariants()


def test_unused_slots_at_most_p_minus_1():
    for n in range(1, 200):
        assert 0 <= bmod.unused_slots(n) <= 15
    assert max(bmod.unused_slots(n) for n in range(1, 200)) == 15


def test_free_returns_all_blocks_and_any_free_block_serves():
    order = np.random.default_rng(0).permutation(32)
    bm = BlockManager(32, order=order)
    bm.allocate(1, 40)
    bm.allocate(2, 70)
    assert bm.num_free == 32 - 3 - 5
    assert bm.block_table(1) == [int(b) for b in order[:3]]     # taken from anywhere in the pool
    bm.free(1)
    assert bm.num_free == 32 - 5
    bm.free(2)
    assert bm.num_free == 32
    bm.check_invariants()


def test_pool_exhaustion_raises_without_side_effects():
    bm = BlockManager(4)
    bm.allocate(0, 48)
    with pytest.raises(NoFreeBlocks):
        bm.allocate(1, 40)
    assert not bm.has_seq(1) and bm.num_free == 1
    bm.allocate(2, 15)                       # the last free block, one slot left in it
    slot, _ = bm.append_slot(2)              # fits in place
    assert slot == bm.block_table(2)[0] * 16 + 15
    with pytest.raises(NoFreeBlocks):
        bm.append_slot(0)                    # 48 tokens fill three blocks: the 49th needs a fourth
    assert bm.context_len(0) == 48 and len(bm.block_table(0)) == 3
    bm.check_invariants()


def test_copy_on_write_of_a_shared_partly_filled_block():
    """Four samples of one 40-token prompt: the two full blocks stay shared;
    the partly filled third block is copied by each writer while another
    reference exists, and the last writer writes in place."""
    bm = BlockManager(64)
    bm.allocate(0, 40)
    for c in (1, 2, 3):
        bm.fork(0, c)
    shared = bm.block_table(0)
    assert all(bm.refcount[b] == 4 for b in shared)
    pairs = []
    for sid in (0, 1, 2, 3):
        slot, cow = bm.append_slot(sid)
        if cow:
            pairs.append(cow)
        assert slot % 16 == 40 % 16
    assert len(pairs) == 3 and all(p[0] == shared[2] for p in pairs)
    assert len({p[1] for p in pairs}) == 3
    for sid in (0, 1, 2, 3):
        assert bm.block_table(sid)[:2] == shared[:2]           # full blocks still shared
    assert bm.refcount[shared[0]] == 4 and bm.refcount[shared[2]] == 1
    bm.check_invariants()
    for sid in (0, 1, 2, 3):
        bm.free(sid)
    assert bm.num_free == 64


def test_copy_on_write_keeps_sharing_for_samples_that_have_not_written():
    bm = BlockManager(16)
    bm.allocate(0, 20)
    bm.fork(0, 1)
    _, cow = bm.append_slot(0)
    assert cow is not None                                   # 1 still references the block
    assert bm.refcount[cow[0]] == 1 and bm.block_table(1)[1] == cow[0]
    _, cow2 = bm.append_slot(1)
    assert cow2 is None                                      # now the only reference: in place
    bm.check_invariants()


def test_full_shared_block_is_not_copied():
    bm = BlockManager(16)
    bm.allocate(0, 32)
    bm.fork(0, 1)
    _, cow = bm.append_slot(0)
    assert cow is None                                       # block full: a new block, no copy
    assert bm.block_table(0)[:2] == bm.block_table(1)
    bm.check_invariants()


def test_tables_array_layout():
    bm = BlockManager(16)
    bm.allocate(5, 17)
    bm.allocate(9, 3)
    t, l = bm.tables_array([9, 5], fill=-1)
    assert t.dtype == np.int32 and l.dtype == np.int32
    assert list(l) == [3, 17]
    assert t[0, 1] == -1 and t[1, 1] == bm.block_table(5)[1]


# --- byte accounting against the pages' figures ----------------------------------------

def test_kv_bytes_example():
    g = golden("kv_accounting.json")["kv_bytes_per_request"]
    b = bmod.kv_bytes_per_request(g["num_layers"], g["num_heads"], g["head_dim"], g["num_tokens"], g["elem_bytes"])
    assert round(b / 1e9, 1) == g["stated_gb"]
    assert round(32 * b / 2 ** 30) == 64 and abs(32 * b / 1e9 - g["stated_gb_for_32_requests"]) < 2


def test_waste_and_ratio_examples():
    g = golden("kv_accounting.json")
    pw = g["padding_waste"]
    assert round(bmod.padding_waste_fraction(pw["mean_len"], pw["max_len"]), 2) == pw["stated_waste"]
    assert round(pw["max_len"] / pw["mean_len"]) == pw["stated_throughput_ratio"]
    pa = g["prealloc_waste"]
    assert round(100 * bmod.padding_waste_fraction(pa["mean_len"], pa["max_len"])) == pa["stated_waste_percent"]
    fr = g["internal_fragmentation"]
    assert round(100 * bmod.padding_waste_fraction(fr["used"], fr["max_len"])) == fr["stated_untouched_percent"]
    lb = g["last_block_waste"]
    for n, pct in lb["cases"]:
        assert round(100 * bmod.last_block_waste_bound(n, lb["block_size"]), 1) == pct
    cw = g["cow_savings"]
    mb = bmod.cow_savings_bytes(cw["prefix_tokens"], cw["num_requests"], cw["kb_per_token"] * 1024) / 2 ** 20
    assert round(mb, 1) == cw["stated_mb"]
