"""paged_decode_attention_static_workspace: decode that allocates nothing.

Some callers cannot allocate device memory where they call this library -- a
plugin or extension hook that is handed raw device pointers and has no
allocator, or a serving loop that owns all device memory from start-up and
forbids later cudaMalloc.  For them the split-context scratch lives in the
library's own device array, shared by every call.  These tests call that
entry point through the C ABI, calls in a row that take the split grid and
the persistent paths in turn (each call runs over whatever the one before
left in the array), and check every output against the oracle and against
paged_decode_attention with a fresh zero-filled workspace of its own.
"""
import ctypes

import pytest
import torch

from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

PKV_ERR_WORKSPACE = -6
STATIC_BYTES = 32 << 20


def _entry():
    lib = H.lib().raw_library()
    fn = lib.paged_decode_attention_static_workspace
    vp = ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [vp] * 6 + [ctypes.c_float] + [ctypes.c_int] * 9 + [vp]
    return fn


def _call_static(fn, out, w, partition_tokens):
    lay, sp = w.layout, w.spec
    return fn(out.data_ptr(), w.q.data_ptr(), w.k_cache.data_ptr(), w.v_cache.data_ptr(), w.block_tables.data_ptr(),
              w.context_lens.data_ptr(), w.scale, sp.num_kv_heads, sp.num_seqs, sp.num_q_heads, sp.head_dim,
              lay.max_blocks_per_seq, lay.num_blocks, lay.max_context_len, 1 if sp.dtype == "bf16" else 0,
              partition_tokens, torch.cuda.current_stream().cuda_stream)


def _with_own_workspace(w, partition_tokens):
    b = H.lib()
    out = torch.full_like(w.q, float("nan"))
    b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                             max_context_len=w.layout.max_context_len, partition_tokens=partition_tokens)
    return out


def _run(fn, case):
    label, wc, pt, persistent = case
    b = H.lib()
    sp = wc.spec
    need = b.workspace_bytes(sp.num_seqs, sp.num_q_heads, sp.num_kv_heads, sp.head_dim, wc.layout.max_context_len, pt)
    assert 0 < need <= STATIC_BYTES, label           # the call really uses the scratch
    assert b.decode_persistent(sp.num_seqs, sp.num_kv_heads, pt, H.torch_dtype(sp)) == persistent, label
    w, ref = H.prepared(case)
    out = torch.full_like(w.q, float("nan"))
    assert _call_static(fn, out, w, pt) == 0, label
    own = _with_own_workspace(w, pt)
    torch.cuda.synchronize()
    H.assert_close(out, ref, sp.dtype, f"static workspace, {label}")
    H.assert_close(out, own.double().cpu().numpy(), sp.dtype, f"static vs own workspace, {label}")


def test_static_workspace_matches_the_oracle_on_calls_that_switch_paths():
    """Split grid, persistent, fixed partitions, persistent on a larger batch,
    split fp32, then split grid and persistent again -- seven calls in a row on
    the one array."""
    torch.cuda.set_device(0)
    fn = _entry()
    cases = H.path_switching_calls()
    for case in cases + cases[:2]:
        _run(fn, case)
    assert H.lib().device_error(clear=True) == 0


def test_static_workspace_two_calls_in_a_row_balanced_request():
    """The balanced split asked for explicitly (PKV_PARTITION_BALANCED) on two
    different batches, one after the other."""
    torch.cuda.set_device(0)
    fn = _entry()
    from paged_kv_cache_177_gb300 import workloads as W
    cases = [
        ("balanced, GQA edge lengths", W.make_workload("gqa8b", lengths_list=H.EDGE_LENGTHS, seed=11), -1, True),
        ("balanced, MHA d=64", W.make_workload("mha13b", lengths_list=(300, 1, 33, 1200, 515), num_q_heads=6,
                                               num_kv_heads=6, head_dim=64, seed=12), -1, True),
    ]
    for case in cases:
        _run(fn, case)
    assert H.lib().device_error(clear=True) == 0


def test_static_workspace_rejects_requests_beyond_its_size():
    torch.cuda.set_device(0)
    fn = _entry()
    # 8 sequences x 64 heads x 256 partitions x (2 + 128) floats = 65 MiB > 32 MiB.
    # The buffers match the arguments and every length is 0, so nothing would be
    # read out of bounds even if the call launched.
    S, Hq, Hkv, D, maxb, nb = 8, 64, 8, 128, 8192, 4
    q = torch.zeros(S, Hq, D, dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(q, 7.0)
    kc = torch.zeros(nb, Hkv, 16, D, dtype=torch.bfloat16, device="cuda")
    tables = torch.zeros(S, maxb, dtype=torch.int32, device="cuda")
    lens = torch.zeros(S, dtype=torch.int32, device="cuda")
    rc = fn(out.data_ptr(), q.data_ptr(), kc.data_ptr(), kc.data_ptr(), tables.data_ptr(), lens.data_ptr(),
            0.088, Hkv, S, Hq, D, maxb, nb, 131072, 1, 512, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == PKV_ERR_WORKSPACE
    assert bool((out == 7.0).all())            # nothing was launched
