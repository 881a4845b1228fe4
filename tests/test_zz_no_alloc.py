"""paged_decode_attention_static_workspace: decode that allocates nothing.

Some callers cannot allocate device memory where they call this library -- a
plugin or extension hook that is handed raw device pointers and has no
allocator, or a serving loop that owns all device memory from start-up and
forbids later cudaMalloc.  For them the split-context scratch lives in the
library's own device array.  These tests call that entry point through the C
ABI and check it against paged_decode_attention (which takes a caller
workspace) on the same inputs, for two calls in a row with different shapes,
so the second call runs over whatever the first left in the shared array.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_177_gb300 import workloads as W
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


def _reference(w, partition_tokens):
    b = H.lib()
    out = torch.empty_like(w.q)
    b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                             max_context_len=w.layout.max_context_len, partition_tokens=partition_tokens)
    return out


def test_static_workspace_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    torch.cuda.set_device(0)
    fn = _entry()
    b = H.lib()
    cases = [
        (W.make_workload("gqa8b", lengths_list=(1, 17, 700, 2000, 0, 1537, 64, 999), seed=11), 64),
        (W.make_workload("mha13b", lengths_list=(300, 1, 33, 1200, 515), num_q_heads=6, num_kv_heads=6,
                         head_dim=64, seed=12), 48),
    ]
    for wc, pt in cases:
        w = wc.to("cuda")
        H.gpu_step(w, attention=False)
        sp = w.spec
        need = b.workspace_bytes(sp.num_seqs, sp.num_q_heads, sp.num_kv_heads, sp.head_dim,
                                 w.layout.max_context_len, pt)
        assert 0 < need <= STATIC_BYTES          # the call really uses the scratch
        ref = _reference(w, pt)
        out = torch.full_like(w.q, float("nan"))
        assert _call_static(fn, out, w, pt) == 0
        torch.cuda.synchronize()
        H.assert_close(out, ref.double().cpu().numpy(), sp.dtype, f"static workspace, {sp.name}")
    assert b.device_error(clear=True) == 0


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
