"""GPU parity: the CUDA path (through the C-ABI binding) against the fp64
oracle, element by element on the same seeded inputs.

* KV append and block copy: bit-exact caches.
* Attention: |gpu - ref| <= 2e-3 + 1e-2 |ref| for bf16, 1e-5 + 1e-5 |ref|
  for fp32.
Small cases span several blocks, several partitions and ragged tails; the
full-size workloads run in the launch configuration the benchmark times and
are checked on every sequence and head.
"""
import zlib

import numpy as np
import pytest
import torch

from paged_kv_cache_177_gb300 import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

EDGE_LENGTHS = H.EDGE_LENGTHS


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    b = H.lib()
    b.device_error(clear=True)
    yield
    assert b.device_error(clear=True) == 0, "a kernel raised the device error word"


def _parity(w_cpu, partition_tokens=0, seq_ids=None):
    h = H.host_arrays(w_cpu)
    w = w_cpu.to("cuda")
    out = H.gpu_step(w, partition_tokens)
    torch.cuda.synchronize()
    ref = H.oracle_step(h, w.layout, w.scale, seq_ids)
    H.assert_caches_equal(w, h)
    got = out if seq_ids is None else out[torch.as_tensor(seq_ids, device=out.device)]
    return H.assert_close(got, ref, w.spec.dtype, w.spec.name)


def test_tiny_workload_full_step():
    """fp32, 4 sequences, 8 heads, d=64, 32-block pool, 1-token append per
    sequence and 2 copy pairs."""
    _parity(W.make_workload("tiny"))


CASES = [
    # name, dtype, Hq, Hkv, d
    ("mha_d128", "bf16", 4, 4, 128),
    ("gqa4_d128", "bf16", 16, 4, 128),
    ("gqa8_d128", "bf16", 16, 2, 128),
    ("gqa16_d128", "bf16", 32, 2, 128),
    ("gqa3_d64", "bf16", 6, 2, 64),
    ("mha_d64", "bf16", 3, 3, 64),
    ("gqa12_d64", "bf16", 12, 1, 64),
    ("f32_gqa4_d128", "f32", 8, 2, 128),
    ("f32_gqa16_d64", "f32", 16, 1, 64),
    ("f32_mha_d128", "f32", 4, 4, 128),
    ("f32_gqa8_d128", "f32", 16, 2, 128),
    ("f32_gqa2_d128", "f32", 4, 2, 128),
    ("f32_gqa3_d64", "f32", 6, 2, 64),
    ("f32_gqa6_d128", "f32", 12, 2, 128),
    ("f32_gqa12_d64", "f32", 12, 1, 64),
    ("f32_gqa16_d128", "f32", 32, 2, 128),
]


@pytest.mark.parametrize("partition_tokens", [0, -1, 16, 48, 128])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_small_cases_all_partitions(case, partition_tokens):
    name, dt, hq, hkv, d = case
    w = W.make_workload("gqa8b", lengths_list=EDGE_LENGTHS, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, dtype=dt,
                        seed=zlib.crc32(name.encode()) % 1000)
    _parity(w, partition_tokens)


def test_all_empty_and_single_sequence():
    _parity(W.make_workload("gqa8b", lengths_list=(0, 0, 0)))
    _parity(W.make_workload("gqa8b", lengths_list=(4096,)), partition_tokens=0)


def test_outputs_are_bit_invariant_under_block_permutation():
    """The same K/V placed on two different shuffles of the pool gives
    bit-identical outputs (the kernel sees the same values in the same order)."""
    b = H.lib()
    w1 = W.make_workload("gqa8b", lengths_list=EDGE_LENGTHS, seed=7).to("cuda")
    H.gpu_step(w1, attention=False)
    perm = torch.randperm(w1.layout.num_blocks, generator=torch.Generator().manual_seed(3)).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel(), device=perm.device)
    k2 = torch.empty_like(w1.k_cache)
    v2 = torch.empty_like(w1.v_cache)
    k2[perm] = w1.k_cache                      # block b moves to perm[b]
    v2[perm] = w1.v_cache
    t2 = perm[w1.block_tables.long()].int()
    outs = []
    for kc, vc, bt in ((w1.k_cache, w1.v_cache, w1.block_tables), (k2, v2, t2)):
        out = torch.empty_like(w1.q)
        b.paged_decode_attention(out, w1.q, kc, vc, bt, w1.context_lens, w1.scale,
                                 max_context_len=w1.layout.max_context_len, partition_tokens=64)
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


def test_shared_prefix_blocks_equal_duplicated_copies():
    b = H.lib()
    w = W.make_workload("parallel_sampling", num_prompts=3).to("cuda")
    H.gpu_step(w, attention=False)
    lay = w.layout
    # duplicate every shared block into a fresh pool region and repoint the tables
    bt = w.block_tables.long().clone()
    S, maxb = bt.shape
    nblk = (w.context_lens.long() + 15) // 16
    mask = torch.arange(maxb, device=bt.device)[None, :] < nblk[:, None]
    n_entries = int(mask.sum())
    k2 = torch.cat([w.k_cache, w.k_cache[bt[mask]]])
    v2 = torch.cat([w.v_cache, w.v_cache[bt[mask]]])
    t2 = bt.clone()
    t2[mask] = lay.num_blocks + torch.arange(n_entries, device=bt.device)
    outs = []
    for kc, vc, tb in ((w.k_cache, w.v_cache, w.block_tables), (k2, v2, t2.int())):
        out = torch.empty_like(w.q)
        b.paged_decode_attention(out, w.q, kc, vc, tb, w.context_lens, w.scale, max_context_len=lay.max_context_len)
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


def test_step_on_a_side_stream_and_in_a_cuda_graph():
    """The three calls are stream-ordered on the caller's stream and capture
    into a CUDA graph (no host synchronisation, caller-owned workspace)."""
    b = H.lib()
    wc = W.make_workload("parallel_sampling", num_prompts=2)
    h = H.host_arrays(wc)
    ref = H.oracle_step(h, wc.layout, wc.scale)
    w = wc.to("cuda")
    lay = w.layout
    ws = torch.zeros(max(1, b.workspace_bytes(lay.spec.num_seqs, lay.spec.num_q_heads, lay.spec.num_kv_heads,
                                                lay.spec.head_dim, lay.max_context_len, 64)),
                     dtype=torch.uint8, device="cuda")
    k0, v0 = w.k_cache.clone(), w.v_cache.clone()
    out = torch.empty_like(w.q)
    s = torch.cuda.Stream()

    def step():
        b.copy_blocks(w.k_cache, w.v_cache, w.cow_pairs, check=False, stream=s)
        b.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache, stream=s)
        b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                                 max_context_len=lay.max_context_len, partition_tokens=64, workspace=ws, stream=s)

    b.check_copy_pairs(lay.cow_pairs, lay.num_blocks)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    s.synchronize()
    H.assert_close(out, ref, "bf16", "side stream")
    H.assert_caches_equal(w, h)
    # graph: restore the pre-step caches, capture, replay twice
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(2):
        w.k_cache.copy_(k0)
        w.v_cache.copy_(v0)
        out.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        H.assert_close(out, ref, "bf16", "graph replay")
        H.assert_caches_equal(w, h)


def test_device_error_word_and_validators():
    """Bad device contents never fault: the kernels skip or zero-fill the bad
    element and raise a bit in the device error word; the validators flag
    the metadata without running the step."""
    b = H.lib()
    w = W.make_workload("gqa8b", lengths_list=(40, 3, 70)).to("cuda")
    lay = w.layout
    b.device_error(clear=True)
    err = b.validate(w.block_tables, w.context_lens, lay.num_blocks, lay.max_context_len)
    assert int(err.item()) == 0
    bad_tables = w.block_tables.clone()
    bad_tables[0, 1] = lay.num_blocks + 5
    err = b.validate(bad_tables, w.context_lens, lay.num_blocks, lay.max_context_len)
    assert int(err.item()) == b.DEVERR_BLOCK_ID
    too_long = w.context_lens.clone()
    too_long[1] = lay.max_context_len + 1
    err = b.validate(w.block_tables, too_long, lay.num_blocks, lay.max_context_len)
    assert int(err.item()) == b.DEVERR_LENGTH
    bad_slots = w.slot_mapping.clone()
    bad_slots[0] = lay.num_blocks * 16
    assert int(b.validate_slots(bad_slots, lay.num_blocks).item()) == b.DEVERR_SLOT
    assert int(b.validate_slots(w.slot_mapping, lay.num_blocks).item()) == 0
    assert b.device_error(clear=True) == 0

    out = torch.empty_like(w.q)
    b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, bad_tables, w.context_lens, w.scale,
                             max_context_len=lay.max_context_len)
    torch.cuda.synchronize()
    assert b.device_error(clear=True) == b.DEVERR_BLOCK_ID
    b.kv_append(w.k_new, w.v_new, bad_slots, w.k_cache, w.v_cache)
    torch.cuda.synchronize()
    assert b.device_error(clear=True) == b.DEVERR_SLOT
    bad_pairs = torch.tensor([[0, lay.num_blocks]], dtype=torch.int64, device="cuda")
    b.copy_blocks(w.k_cache, w.v_cache, bad_pairs, check=False)
    torch.cuda.synchronize()
    assert b.device_error(clear=True) == b.DEVERR_PAIR
    with pytest.raises(b.PagedKVError):
        b.copy_blocks(w.k_cache, w.v_cache, bad_pairs)            # host check rejects it
    b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, too_long, w.scale,
                             max_context_len=lay.max_context_len)
    torch.cuda.synchronize()
    assert b.device_error(clear=True) == b.DEVERR_LENGTH


# ---- full-size workloads, in the benchmark's launch configuration ----------------------

FULL = ["mha13b", "gqa8b", "parallel_sampling", "long_context"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    """The benchmarked batches, in the benchmark's launch configuration:
    caches bit-exact after the step's copies and appends, and every output
    element of every sequence and head within the bf16 bound of the oracle."""
    w = W.make_workload(name, device="cuda")
    lay = w.layout
    h = H.host_arrays(w)
    out = H.gpu_step(w, lay.spec.partition_tokens)
    torch.cuda.synchronize()
    ref = H.oracle_step(h, lay, w.scale)
    H.assert_caches_equal(w, h)
    H.assert_close(out, ref, lay.spec.dtype, name)


@pytest.mark.parametrize("name", ["mha13b", "gqa8b", "long_context"])
def test_full_size_fp32(name):
    """The 13B-class, GQA and long-context batches with fp32 caches (the
    CUDA-core path): every sequence and head against the oracle at the fp32
    bound."""
    w = W.make_workload(name, device="cuda", dtype="f32")
    lay = w.layout
    h = H.host_arrays(w)
    out = H.gpu_step(w, lay.spec.partition_tokens)
    torch.cuda.synchronize()
    ref = H.oracle_step(h, lay, w.scale)
    H.assert_close(out, ref, "f32", f"{name} fp32")


def test_persistent_path_leaves_counters_zero_and_repeats_bit_identically():
    """bf16 with automatic partitioning runs the persistent balanced kernel:
    its arrival counters return to zero after every call, and the merge of
    cut sequences does not depend on which warp arrives last."""
    b = H.lib()
    for lens, hq, hkv in ((EDGE_LENGTHS, 16, 4), ((3000, 1, 2, 4000, 17), 64, 8), ((1, 1, 1), 8, 8)):
        wc = W.make_workload("gqa8b", lengths_list=lens, num_q_heads=hq, num_kv_heads=hkv, seed=len(lens))
        h = H.host_arrays(wc)
        w = wc.to("cuda")
        H.gpu_step(w, attention=False)
        lay = w.layout
        assert b.decode_persistent(lay.spec.num_seqs, hkv, -1, torch.bfloat16)
        assert b.decode_launches(lay.spec.num_seqs, hkv, lay.max_context_len, -1, torch.bfloat16) == 1
        need = b.workspace_bytes(lay.spec.num_seqs, hq, hkv, 128, lay.max_context_len, -1)
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        outs = []
        for _ in range(3):
            out = torch.empty_like(w.q)
            b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                                     max_context_len=lay.max_context_len, workspace=ws, partition_tokens=-1)
            torch.cuda.synchronize()
            counters = ws[: b.DECODE_COUNTER_BYTES]
            assert int(counters.count_nonzero()) == 0
            outs.append(out)
        assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
        ref = H.oracle_step(h, lay, w.scale)
        H.assert_close(outs[0], ref, "bf16", f"persistent {lens}")


def test_one_workspace_serves_every_decode_path_in_turn():
    """One workspace, zero-filled once and sized for the largest call, serves
    a split grid call, a persistent call, a fixed-partition call, a
    persistent call on a larger batch and a split fp32 call, in that order (a
    serving loop whose batch crosses the persistent threshold): every output
    matches the oracle on every sequence and head, and the counter header is
    zero after each call."""
    b = H.lib()
    cases = H.path_switching_calls()
    need = max(b.workspace_bytes(wc.spec.num_seqs, wc.spec.num_q_heads, wc.spec.num_kv_heads, wc.spec.head_dim,
                                 wc.layout.max_context_len, pt) for _, wc, pt, _ in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for case in cases + cases[:2]:
        label, wc, pt, persistent = case
        sp, lay = wc.spec, wc.layout
        assert b.decode_persistent(sp.num_seqs, sp.num_kv_heads, pt, H.torch_dtype(sp)) == persistent, label
        assert persistent or b.decode_launches(sp.num_seqs, sp.num_kv_heads, lay.max_context_len, pt) == 2, label
        w, ref = H.prepared(case)
        out = torch.full_like(w.q, float("nan"))
        b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                                 max_context_len=lay.max_context_len, partition_tokens=pt, workspace=ws)
        torch.cuda.synchronize()
        assert int(ws[: b.DECODE_COUNTER_BYTES].count_nonzero()) == 0, label
        H.assert_close(out, ref, sp.dtype, f"reused workspace, {label}")
        del w


LARGE_CASES = [
    # name, Hq, Hkv, sequences, longest context
    ("mha_large", 16, 16, 128, 1200),
    ("gqa8_large", 64, 8, 256, 1200),
    ("gqa4_large", 16, 4, 256, 1200),
]


@pytest.mark.parametrize("case", LARGE_CASES, ids=[c[0] for c in LARGE_CASES])
def test_persistent_large_batches(case):
    """Batches of at least 8 positions per persistent warp: every warp's
    range cuts units at both ends, so nearly every warp writes segment
    states and many merge; the arrival counters are zero after each call, the
    output repeats bit for bit and matches the oracle on every sequence."""
    name, hq, hkv, S, longest = case
    b = H.lib()
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    lens = tuple(int(x) for x in rng.integers(1, longest + 1, S))
    wc = W.make_workload("gqa8b", lengths_list=lens, num_q_heads=hq, num_kv_heads=hkv, seed=S + hq)
    h = H.host_arrays(wc)
    w = wc.to("cuda")
    H.gpu_step(w, attention=False)
    lay = w.layout
    assert hkv * sum((x + 15) // 16 for x in lens) >= 8 * 152 * 12
    assert b.decode_persistent(S, hkv, -1, torch.bfloat16)
    ws = torch.zeros(b.workspace_bytes(S, hq, hkv, 128, lay.max_context_len, -1), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        out = torch.empty_like(w.q)
        b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                                 max_context_len=lay.max_context_len, workspace=ws, partition_tokens=-1)
        torch.cuda.synchronize()
        assert int(ws[: b.DECODE_COUNTER_BYTES].count_nonzero()) == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    ref = H.oracle_step(h, lay, w.scale)
    H.assert_close(outs[0], ref, "bf16", name)


def test_persistent_step_in_a_cuda_graph():
    b = H.lib()
    wc = W.make_workload("gqa8b", lengths_list=EDGE_LENGTHS, seed=21)
    h = H.host_arrays(wc)
    ref = H.oracle_step(h, wc.layout, wc.scale)
    w = wc.to("cuda")
    lay = w.layout
    ws = torch.zeros(b.workspace_bytes(lay.spec.num_seqs, 32, 8, 128, lay.max_context_len, -1), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(w.q)
    s = torch.cuda.Stream()
    H.gpu_step(w, attention=False)
    torch.cuda.synchronize()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):     # first call outside capture
        b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                                 max_context_len=lay.max_context_len, workspace=ws, stream=s, partition_tokens=-1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                                 max_context_len=lay.max_context_len, workspace=ws, stream=s, partition_tokens=-1)
    for _ in range(3):
        out.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        H.assert_close(out, ref, "bf16", "persistent graph replay")


def test_per_step_arguments_in_pinned_host_memory():
    """q, out, tables, lengths, new K/V, slots and copy pairs read and written
    in place in pinned host memory give the same bits as device copies, on
    the persistent and the split grid paths."""
    b = H.lib()
    for name, pt in (("gqa8b", -1), ("parallel_sampling", 128)):
        w = W.make_workload(name, num_seqs=24, num_prompts=6, seed=77) if name == "parallel_sampling" else \
            W.make_workload(name, lengths_list=tuple(range(1, 2000, 83)), seed=77)
        lay = w.layout
        wd = w.to("cuda")
        pin = lambda t: t.contiguous().pin_memory()
        kc2, vc2 = wd.k_cache.clone(), wd.v_cache.clone()
        # device arguments
        b.copy_blocks(wd.k_cache, wd.v_cache, wd.cow_pairs, host_pairs=lay.cow_pairs)
        b.kv_append(wd.k_new, wd.v_new, wd.slot_mapping, wd.k_cache, wd.v_cache)
        out_d = torch.empty_like(wd.q)
        b.paged_decode_attention(out_d, wd.q, wd.k_cache, wd.v_cache, wd.block_tables, wd.context_lens, w.scale,
                                 max_context_len=lay.max_context_len, partition_tokens=pt)
        # the same step with the per-step arguments in pinned host memory
        b.copy_blocks(kc2, vc2, pin(w.cow_pairs), host_pairs=lay.cow_pairs)
        b.kv_append(pin(w.k_new), pin(w.v_new), pin(w.slot_mapping), kc2, vc2)
        out_h = torch.full(tuple(w.q.shape), float("nan"), dtype=w.q.dtype).pin_memory()
        b.paged_decode_attention(out_h, pin(w.q), kc2, vc2, pin(w.block_tables), pin(w.context_lens), w.scale,
                                 max_context_len=lay.max_context_len, partition_tokens=pt)
        torch.cuda.synchronize()
        assert torch.equal(kc2.view(torch.int16), wd.k_cache.view(torch.int16))
        assert torch.equal(vc2.view(torch.int16), wd.v_cache.view(torch.int16))
        assert torch.equal(out_h.view(torch.int16), out_d.cpu().view(torch.int16)), name


@pytest.mark.parametrize("partition_tokens", [-1, 0, 16])
def test_short_contexts_stay_within_tolerance(partition_tokens):
    """Rows that see 2..17 tokens, where rounding the softmax weights to bf16
    alone can move an output past 2e-3 + 1e-2 |ref| when comparable weights
    meet cancelling V rows: 512 sequences x 32 query heads x 128 outputs."""
    lens = tuple(2 + (i % 16) for i in range(512))
    w = W.make_workload("gqa8b", lengths_list=lens, seed=171 + partition_tokens)
    h = H.host_arrays(w)
    ref = H.oracle_step(h, w.layout, w.scale)
    wd = w.to("cuda")
    out = H.gpu_step(wd, partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    H.assert_close(out, ref, "bf16", f"short contexts, partition_tokens={partition_tokens}")


@pytest.mark.parametrize("partition_tokens", [0, -1])
def test_batch_beyond_the_persistent_kernels_limit(partition_tokens):
    """9,000 sequences (more than the persistent kernel's 8,192): the call falls
    back to the grid kernel, balanced request included; lengths 0..47."""
    lens = tuple(i % 48 for i in range(9000))
    w = W.make_workload("gqa8b", lengths_list=lens, num_q_heads=8, num_kv_heads=2, head_dim=64, seed=91)
    h = H.host_arrays(w)
    ref = H.oracle_step(h, w.layout, w.scale)
    out = H.gpu_step(w.to("cuda"), partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    H.assert_close(out, ref, "bf16", f"9000 sequences, partition_tokens={partition_tokens}")
    assert torch.all(out[torch.tensor([i for i, n in enumerate(lens) if n == 0], device="cuda")] == 0)


@pytest.mark.parametrize("name,pt,over", [("gqa8b", -1, dict(lengths_list=tuple(range(1, 3000, 97)))),
                                         ("parallel_sampling", 128, dict(num_prompts=6)),
                                         ("tiny", 0, {})])
def test_decode_step_call_matches_the_three_calls(name, pt, over):
    """paged_decode_step (copies, append, attention launched right after the
    append) gives the same bits as the three separate calls -- persistent,
    split-grid and fp32 paths -- directly, replayed from a CUDA graph, and with
    its per-step arguments in pinned host memory."""
    b = H.lib()
    w = W.make_workload(name, seed=55, **over)
    lay = w.layout
    ref_d = w.to("cuda")
    out_ref = H.gpu_step(ref_d, partition_tokens=pt)
    torch.cuda.synchronize()
    for variant in ("direct", "graph", "pinned"):
        d = w.to("cuda")
        out = torch.full_like(d.q, float("nan"))
        if variant == "pinned":
            pin = lambda t: t.contiguous().pin_memory() if t.numel() else t
            q, kn, vn, sl, bt, cl, pr = (pin(x) for x in (w.q, w.k_new, w.v_new, w.slot_mapping, w.block_tables,
                                                          w.context_lens, w.cow_pairs))
            out = torch.full(tuple(w.q.shape), float("nan"), dtype=w.q.dtype).pin_memory()
        else:
            q, kn, vn, sl, bt, cl, pr = d.q, d.k_new, d.v_new, d.slot_mapping, d.block_tables, d.context_lens, d.cow_pairs
        ws = torch.zeros(max(16, b.workspace_bytes(lay.spec.num_seqs, lay.spec.num_q_heads, lay.spec.num_kv_heads,
                                                   lay.spec.head_dim, lay.max_context_len, pt)),
                         dtype=torch.uint8, device="cuda")

        def step():
            b.paged_decode_step(out, q, d.k_cache, d.v_cache, bt, cl, w.scale, kn, vn, sl, pr,
                                host_pairs=lay.cow_pairs, max_context_len=lay.max_context_len,
                                partition_tokens=pt, workspace=ws)

        if variant == "graph":
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                step()
            g.replay()
        else:
            step()
        torch.cuda.synchronize()
        iv = torch.int16 if w.q.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(out.cpu().view(iv), out_ref.cpu().view(iv)), f"{name} {variant}"
        assert torch.equal(d.k_cache.view(iv), ref_d.k_cache.view(iv)) and torch.equal(d.v_cache.view(iv),
                                                                                        ref_d.v_cache.view(iv))


@pytest.mark.parametrize("where", ["first blocks of other sequences", "last blocks"])
def test_decode_step_with_appends_anywhere_matches_the_three_calls(where):
    """paged_decode_step launches the attention right behind its append and
    waits for the append before reading the caches: slots aimed at the first
    (earliest-read) blocks of other sequences, and the usual last-block slots,
    both give the bits of the three separate calls on the persistent path, and
    the oracle's result."""
    b = H.lib()
    wc = W.make_workload("gqa8b", lengths_list=tuple(range(40, 40 + 97 * 23, 23)), seed=313)
    lay = wc.layout
    S = lay.spec.num_seqs
    slots = lay.slot_mapping.copy()
    if where.startswith("first"):
        # the newest positions (NaN until appended) get this step's rows, as if appended earlier ...
        for t, slot in enumerate(slots.tolist()):
            wc.k_cache[slot // 16, :, slot % 16] = wc.k_new[t]
            wc.v_cache[slot // 16, :, slot % 16] = wc.v_new[t]
        # ... and token t now overwrites slot 3 of sequence t+1's first block (every sequence has 3+ blocks)
        slots = np.array([int(lay.block_tables[(t + 1) % S][0]) * 16 + 3 for t in range(S)], np.int64)
        assert len(set(slots.tolist())) == S
    lay.slot_mapping[:] = slots
    wc.slot_mapping.copy_(torch.from_numpy(slots))
    h = H.host_arrays(wc)
    ref = H.oracle_step(h, lay, wc.scale)
    outs = []
    for one_call in (False, True):
        d = wc.to("cuda")
        ws = torch.zeros(b.workspace_bytes(S, 32, 8, 128, lay.max_context_len, -1), dtype=torch.uint8, device="cuda")
        out = torch.full_like(d.q, float("nan"))
        if one_call:
            b.paged_decode_step(out, d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, wc.scale, d.k_new,
                                d.v_new, d.slot_mapping, None, max_context_len=lay.max_context_len,
                                partition_tokens=-1, workspace=ws)
        else:
            b.kv_append(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache)
            b.paged_decode_attention(out, d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, wc.scale,
                                     max_context_len=lay.max_context_len, partition_tokens=-1, workspace=ws)
        torch.cuda.synchronize()
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16)), where
    H.assert_close(outs[1], ref, "bf16", where)
