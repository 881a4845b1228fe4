"""GPU parity of shared-prefix (cascade) decode: the same results as plain
paged decode -- checked against the oracle -- while each group's shared
blocks are read once."""
import numpy as np
import pytest
import torch

from paged_kv_cache_177_gb300 import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    torch.cuda.set_device(0)
    b = H.lib()
    b.device_error(clear=True)
    yield
    assert b.device_error(clear=True) == 0


def _run(w, groups, shared, partition_tokens=0):
    b = H.lib()
    out = torch.full_like(w.q, float("nan"))
    b.paged_decode_attention_shared_prefix(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                                           torch.from_numpy(groups).cuda(), torch.from_numpy(shared).cuda(),
                                           max_context_len=w.layout.max_context_len,
                                           partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("partition_tokens", [0, 128])
def test_parallel_sampling_matches_the_oracle(partition_tokens):
    wc = W.make_workload("parallel_sampling", num_prompts=6)
    h = H.host_arrays(wc)
    ref = H.oracle_step(h, wc.layout, wc.scale)
    w = wc.to("cuda")
    H.gpu_step(w, attention=False)
    out = _run(w, w.layout.group_members, w.layout.shared_blocks, partition_tokens)
    H.assert_close(out, ref, "bf16", "shared prefix")


def test_matches_plain_decode_with_ragged_groups():
    """Groups with empty slots, members shorter than the declared prefix,
    sequences in no group and an empty context, for GQA group sizes that
    fill 8 and 16 MMA columns."""
    for hq, hkv, d, M in ((8, 4, 128, 4), (16, 4, 64, 4), (4, 4, 128, 3)):
        lens = (300, 300, 305, 290, 17, 0, 400, 64, 33)
        wc = W.make_workload("gqa8b", lengths_list=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             seed=hq * 7 + d)
        lay = wc.layout
        # make sequences 0..3 share their first 18 blocks and 6, 7 their first 4
        kt = lay.block_tables.copy()
        kt[1:4, :18] = kt[0, :18]
        kt[7, :4] = kt[6, :4]
        wc.block_tables = torch.from_numpy(kt)
        lay.block_tables = kt
        b = H.lib()
        # a group of one with a shared count past its length; with M = 3, sequence 3
        # still points at sequence 0's blocks but is attended alone
        groups, shared = b.prefix_groups(len(lens), [[0, 1, 2, 3][:M], [6, 7], [8]], [18, 4, 9])
        h = H.host_arrays(wc)
        ref = H.oracle_step(h, lay, wc.scale)
        w = wc.to("cuda")
        H.gpu_step(w, attention=False)
        out = _run(w, groups, shared)
        H.assert_close(out, ref, "bf16", f"ragged groups hq={hq} hkv={hkv} d={d}")
        assert torch.all(out[5] == 0)         # empty context


def test_full_size_parallel_sampling_against_plain_decode():
    w = W.make_workload("parallel_sampling", device="cuda")
    H.gpu_step(w, attention=False)
    lay = w.layout
    b = H.lib()
    plain = torch.empty_like(w.q)
    b.paged_decode_attention(plain, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                             max_context_len=lay.max_context_len)
    out = _run(w, lay.group_members, lay.shared_blocks)
    # both within the bf16 tolerance of the oracle on every sequence and head
    h = H.host_arrays(w)
    import oracle
    ref = oracle.paged_decode_attention(h["q"], h["k_cache"], h["v_cache"], lay.block_tables, lay.context_lens,
                                        w.scale, lay.spec.num_kv_heads)
    H.assert_close(out, ref, "bf16", "full size shared prefix")
    H.assert_close(plain, ref, "bf16", "full size plain decode of the shared-prefix batch")


def test_one_uncleared_workspace_serves_every_partition_size():
    """One workspace, filled with garbage once and never cleared, serves calls
    with different partition sizes (a union of one partition, and unions cut
    into many): each call matches the oracle and repeats bit for bit."""
    wc = W.make_workload("parallel_sampling", num_prompts=5)
    h = H.host_arrays(wc)
    ref = H.oracle_step(h, wc.layout, wc.scale)
    w = wc.to("cuda")
    H.gpu_step(w, attention=False)
    lay = w.layout
    b = H.lib()
    sp = lay.spec
    groups = torch.from_numpy(lay.group_members).cuda()
    shared = torch.from_numpy(lay.shared_blocks).cuda()
    need = max(b.shared_prefix_workspace_bytes(sp.num_seqs, sp.num_q_heads, sp.head_dim, lay.max_context_len,
                                               groups.shape[1], pt) for pt in (64, 512, 4096))
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    for pt in (64, 4096, 512, 64):
        outs = []
        for _ in range(3):
            out = torch.full_like(w.q, float("nan"))
            b.paged_decode_attention_shared_prefix(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                                   w.scale, groups, shared, max_context_len=lay.max_context_len,
                                                   partition_tokens=pt, workspace=ws)
            torch.cuda.synchronize()
            outs.append(out)
        H.assert_close(outs[0], ref, "bf16", f"shared prefix, partition_tokens={pt}")
        assert all(torch.equal(outs[0], o) for o in outs[1:]), f"partition_tokens={pt}: repeat differs"
