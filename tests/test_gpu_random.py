"""Seeded random decode calls against the oracle, every output.

Each case draws, from its own seed: the kv heads and the group size (1..16),
head_dim (64 or 128), the cache type (bf16, fp32, or bf16 with fp32 output),
the partitioning (automatic, balanced, or fixed partitions of 16..2048
tokens), and 1..40 sequences whose lengths mix empty contexts, single tokens,
block edges and long tails. One workspace, zero-filled once, serves all the
calls in order, so every path also starts from whatever the previous call
left in it. The result must not depend on any of these choices beyond the
tolerance of the output type.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_177_gb300 import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

N_CASES = 100


def _draw(seed):
    rng = np.random.default_rng(seed)
    g = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 12, 16]))
    hkv = int(rng.integers(1, max(2, 17 // g) + 1))
    d = int(rng.choice([64, 128]))
    kind = str(rng.choice(["bf16", "f32", "bf16_out_f32"]))
    pt = int(rng.choice([0, 0, -1, 16, 48, 128, 512, 2048]))
    if kind == "f32" and pt == -1:
        pt = 0  # the balanced split is a bf16 path
    n = int(rng.integers(1, 41))
    pool = np.concatenate([[0, 1, 15, 16, 17, 31, 32, 33], rng.integers(1, 600, 8), rng.integers(600, 5000, 2)])
    lens = tuple(int(x) for x in rng.choice(pool, n))
    return g, hkv, d, kind, pt, lens


@pytest.fixture(scope="module")
def workspace():
    b = H.lib()
    need = 0
    for i in range(N_CASES):
        g, hkv, d, kind, pt, lens = _draw(1000 + i)
        need = max(need, b.workspace_bytes(len(lens), g * hkv, hkv, d, max(max(lens), 1), pt))
    return torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_decode_call(case, workspace):
    g, hkv, d, kind, pt, lens = _draw(1000 + case)
    label = f"g={g} hkv={hkv} d={d} {kind} partition_tokens={pt} lens={lens}"
    dtype = "f32" if kind == "f32" else "bf16"
    wc = W.make_workload("gqa8b", lengths_list=lens, num_q_heads=g * hkv, num_kv_heads=hkv, head_dim=d, dtype=dtype,
                         seed=2000 + case)
    h = H.host_arrays(wc)
    ref = H.oracle_step(h, wc.layout, wc.scale)
    w = wc.to("cuda")
    H.gpu_step(w, attention=False)
    b = H.lib()
    out_dtype = torch.float32 if kind != "bf16" else torch.bfloat16
    out = torch.full(tuple(w.q.shape), float("nan"), dtype=out_dtype, device="cuda")
    b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                             max_context_len=w.layout.max_context_len, partition_tokens=pt, workspace=workspace)
    torch.cuda.synchronize()
    assert int(workspace[: b.DECODE_COUNTER_BYTES].count_nonzero()) == 0, label
    assert b.device_error(clear=True) == 0, label
    H.assert_caches_equal(w, h)
    if kind == "bf16_out_f32":
        # the accumulator before rounding: 2e-3 absolute alone
        err = np.abs(out.double().cpu().numpy() - ref)
        assert np.all(np.isfinite(err)) and err.max() <= 2e-3, f"{label}: unrounded max abs err {err.max():.3e}"
    else:
        H.assert_close(out, ref, dtype, label)
