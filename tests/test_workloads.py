"""Seeded input generators: shapes, pool layout, poison, and the
copy-on-write structure of the parallel-sampling workload."""
import numpy as np
import pytest
import torch

from paged_kv_cache_177_gb300 import workloads as W
from paged_kv_cache_177_gb300.block_manager import BlockManager


@pytest.mark.parametrize("name", W.CONFIG_ORDER)
def test_layout_invariants(name):
    lay = W.make_layout(W.spec(name))
    sp = lay.spec
    assert lay.context_lens.shape == (sp.num_seqs,)
    nblk = -(-lay.context_lens.astype(np.int64) // 16)
    assert lay.block_tables.shape[1] == nblk.max()
    refs = {}
    for s in range(sp.num_seqs):
        ids = lay.block_tables[s, :nblk[s]]
        assert np.all((ids >= 0) & (ids < lay.num_blocks))
        assert len(set(ids.tolist())) == len(ids)
        for b in ids.tolist():
            refs[b] = refs.get(b, 0) + 1
        # unused entries point at a block no table uses
        rest = lay.block_tables[s, nblk[s]:]
        assert np.all(~lay.used_blocks[rest])
    assert set(refs) == set(np.nonzero(lay.used_blocks)[0].tolist())
    if name != "parallel_sampling":
        assert max(refs.values()) == 1          # no sharing
    # every appended slot lies inside its sequence's readable tokens
    slot_blocks = lay.slot_mapping // 16
    assert np.all(lay.used_blocks[slot_blocks])
    assert len(set(lay.slot_mapping.tolist())) == len(lay.slot_mapping)


def test_lengths_follow_the_recipes():
    assert W.make_layout(W.spec("tiny")).context_lens.max() <= 64
    l2 = W.make_layout(W.spec("mha13b")).context_lens
    assert l2.min() >= 16 and l2.max() <= 2048
    l3 = W.make_layout(W.spec("gqa8b")).context_lens
    assert l3.min() >= 32 and l3.max() <= 4096 and 600 < np.median(l3) < 1600
    l5 = W.make_layout(W.spec("long_context")).context_lens
    assert l5.min() >= 32768 and l5.max() <= 131072
    l4 = W.make_layout(W.spec("parallel_sampling")).context_lens
    assert l4.min() >= 1000 and l4.max() <= 1256


def test_parallel_sampling_copy_on_write_matches_block_manager():
    """The generator's copy pairs follow the block manager's rule: per
    prompt, each writer copies the shared partly filled block while another
    reference exists; full prompt blocks stay shared."""
    lay = W.make_layout(W.spec("parallel_sampling"))
    sp = lay.spec
    G = sp.samples_per_prompt
    suffix = lay.context_lens.astype(np.int64) - sp.prompt_len
    expected = 0
    for p in range(sp.num_prompts):
        bm = BlockManager(200)
        bm.allocate(0, sp.prompt_len)
        for c in range(1, G):
            bm.fork(0, c)
        for s in range(G):
            if suffix[p * G + s] > 0:
                _, cow = bm.append_slot(s)
                expected += cow is not None
        # full prompt blocks shared by all samples in the generated tables
        t = lay.block_tables[p * G:(p + 1) * G, :sp.prompt_len // 16]
        assert np.all(t == t[0])
    assert len(lay.cow_pairs) == expected
    assert len(set(lay.cow_pairs[:, 1].tolist())) == len(lay.cow_pairs)
    assert not set(lay.cow_pairs[:, 1].tolist()) & set(lay.cow_pairs[:, 0].tolist())


def test_tiny_workload_tensors_and_poison():
    w = W.make_workload("tiny")
    lay = w.layout
    assert w.q.dtype == torch.float32 and w.k_cache.shape == (lay.num_blocks, 8, 16, 64)
    kc = w.k_cache.numpy()
    assert np.all(np.isnan(kc[~lay.used_blocks]))
    # the appended slots hold NaN before the step
    for slot in lay.slot_mapping.tolist():
        assert np.all(np.isnan(kc[slot // 16, :, slot % 16]))
    # readable tokens other than the appended ones are finite
    for s in range(lay.spec.num_seqs):
        n = int(lay.context_lens[s])
        for t in range(n - 1):
            assert np.all(np.isfinite(kc[lay.block_tables[s, t // 16], :, t % 16]))
    # the same seed gives the same tensors
    w2 = W.make_workload("tiny")
    assert torch.equal(w.q, w2.q) and torch.equal(w.k_cache.nan_to_num(), w2.k_cache.nan_to_num())


def test_bf16_poison_bits_and_numpy_round_trip():
    w = W.make_workload("gqa8b", num_seqs=4)
    kc = W.to_numpy(w.k_cache)
    assert kc.dtype == np.uint16
    unused = ~w.layout.used_blocks
    assert np.all(kc[unused] == 0x7FC0)
    back = W.from_numpy_bits(kc)
    assert back.dtype == torch.bfloat16 and torch.equal(back.view(torch.int16), w.k_cache.view(torch.int16))
