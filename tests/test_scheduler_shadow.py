"""Replays every step's device metadata on a shadow cache of token ids (on the
CPU) and checks that each running sequence reads back exactly its own
history through its block table: prefill, continuous batching, forks with
copy-on-write, preemption by recompute and by swapping to a host pool."""
import random

import numpy as np
import pytest

from paged_kv_cache_177_gb300 import scheduler as S


def code(seq, pos):
    return seq * 100_000 + pos


def replay(num_blocks, host_blocks, max_batch, requests, seed=0):
    s = S.IterationScheduler(num_blocks, max_batch, host_blocks=host_blocks,
                             order=np.random.default_rng(seed).permutation(num_blocks))
    for r in requests:
        s.add(r)
    root = {r.req_id: (r.parent if r.parent is not None else r.req_id) for r in requests}
    prompt = {r.req_id: r.prompt_len for r in requests}

    def expect(sid, p):
        return code(root[sid], p) if p < prompt[sid] else code(sid, p)

    dev = np.full((num_blocks, 16), -1, dtype=np.int64)
    host = np.full((max(host_blocks, 1), 16), -1, dtype=np.int64)
    steps = 0
    while not s.idle():
        b = s.step()
        assert b is not None
        for h, d in b.swap_in_pairs:
            dev[d] = host[h]
        for sid, n, table in b.prefilled:
            for p in range(n):
                dev[table[p // 16], p % 16] = expect(sid, p)
        for d, h in b.swap_out_pairs:
            host[h] = dev[d]
        for src, dst in b.cow_pairs:
            dev[dst] = dev[src]
        for i, sid in enumerate(b.seq_ids):
            slot = int(b.slot_mapping[i])
            dev[slot // 16, slot % 16] = code(sid, int(b.context_lens[i]) - 1)
        for i, sid in enumerate(b.seq_ids):
            n = int(b.context_lens[i])
            t = b.block_tables[i]
            got = [int(dev[t[p // 16], p % 16]) for p in range(n)]
            assert got == [expect(sid, p) for p in range(n)], f"sequence {sid} reads a wrong history at step {steps}"
        s.bm.check_invariants()
        if s.host is not None:
            s.host.check_invariants()
        s.retire(b)
        steps += 1
    assert s.bm.num_free == num_blocks
    return s


@pytest.mark.parametrize("host_blocks", [0, 64])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_continuous_batching_under_pressure(host_blocks, seed):
    rng = random.Random(seed)
    reqs = [S.Request(i, prompt_len=rng.randint(1, 60), output_len=rng.randint(5, 90)) for i in range(30)]
    s = replay(24, host_blocks, 8, reqs, seed)
    assert s.preemptions > 0
    if host_blocks:
        assert s.swaps > 0


@pytest.mark.parametrize("host_blocks", [0, 96])
def test_parallel_sampling_with_copy_on_write(host_blocks):
    rng = random.Random(7)
    reqs = []
    for p in range(6):
        parent = 10 * p
        plen = rng.randint(17, 50)
        reqs.append(S.Request(parent, prompt_len=plen, output_len=rng.randint(3, 40)))
        for c in range(1, 4):
            reqs.append(S.Request(parent + c, prompt_len=plen, output_len=rng.randint(3, 40), parent=parent))
    s = replay(14, host_blocks, 8, reqs, 5)
    assert s.preemptions > 0


def test_ample_memory_never_preempts():
    reqs = [S.Request(i, prompt_len=10, output_len=20) for i in range(12)]
    s = replay(200, 0, 4, reqs)
    assert s.preemptions == 0
