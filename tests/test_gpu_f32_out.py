"""bf16 decode with fp32 output (PKV_BF16_OUT_F32): the accumulated O / L
before it is rounded to bf16.

The bf16 bound |gpu - ref| <= 2e-3 + 1e-2 |ref| covers the output rounding
(a bf16 half-ulp alone exceeds 2e-3 for |x| >= 1). This mode measures the
kernels' own error -- bf16 softmax weights on the tensor cores, fp32
accumulation, partition merges -- against 2e-3 absolute alone, and checks
that rounding it to nearest even gives the bf16 output bit for bit (the same
arithmetic, only the store differs).
"""
import zlib

import numpy as np
import pytest
import torch

from paged_kv_cache_177_gb300 import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

ABS = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    b = H.lib()
    b.device_error(clear=True)
    yield
    assert b.device_error(clear=True) == 0, "a kernel raised the device error word"


def _both(w, partition_tokens):
    """bf16 and fp32 outputs of the same attention call (after the step's
    copies and appends)."""
    b = H.lib()
    lay = w.layout
    out16 = H.gpu_step(w, partition_tokens)
    out32 = torch.full(tuple(w.q.shape), float("nan"), dtype=torch.float32, device=w.q.device)
    b.paged_decode_attention(out32, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                             max_context_len=lay.max_context_len, partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    return out16, out32


def _check(out16, out32, ref, what):
    g = out32.double().cpu().numpy()
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= ABS, f"{what}: unrounded max abs err {err.max():.3e} at {worst} (ref {ref[worst]:.6f})"
    assert torch.equal(out32.to(torch.bfloat16).view(torch.int16), out16.view(torch.int16)), \
        f"{what}: the rounded accumulator differs from the bf16 output"
    return float(err.max())


@pytest.mark.parametrize("name", ["mha13b", "gqa8b", "parallel_sampling", "long_context"])
def test_unrounded_error_full_size(name):
    """Every bf16 benchmark batch, in the benchmark's launch configuration,
    every sequence and head."""
    w = W.make_workload(name, device="cuda")
    lay = w.layout
    h = H.host_arrays(w)
    out16, out32 = _both(w, lay.spec.partition_tokens)
    ref = H.oracle_step(h, lay, w.scale)
    _check(out16, out32, ref, f"{name} fp32 out")


CASES = [("mha_d128", 4, 4, 128), ("gqa4_d128", 16, 4, 128), ("gqa8_d128", 16, 2, 128),
         ("gqa16_d128", 32, 2, 128), ("gqa3_d64", 6, 2, 64), ("mha_d64", 3, 3, 64)]


@pytest.mark.parametrize("partition_tokens", [0, -1, 16, 128])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_unrounded_error_edge_lengths(case, partition_tokens):
    """Edge lengths (0, 1, 15, 16, 17, .. 1537) on every decode path: the
    persistent kernel (with and without cut sequences), fixed partitions and
    the log-sum-exp reduce."""
    name, hq, hkv, d = case
    wc = W.make_workload("gqa8b", lengths_list=H.EDGE_LENGTHS, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                         seed=zlib.crc32(name.encode()) % 1000 + 5)
    h = H.host_arrays(wc)
    out16, out32 = _both(wc.to("cuda"), partition_tokens)
    ref = H.oracle_step(h, wc.layout, wc.scale)
    _check(out16, out32, ref, f"{name}, partition_tokens={partition_tokens}")


def test_unrounded_error_short_contexts():
    """Rows of 2..17 tokens, where few comparable weights meet cancelling V
    rows (512 sequences x 32 query heads)."""
    lens = tuple(2 + (i % 16) for i in range(512))
    wc = W.make_workload("gqa8b", lengths_list=lens, seed=404)
    h = H.host_arrays(wc)
    out16, out32 = _both(wc.to("cuda"), 0)
    ref = H.oracle_step(h, wc.layout, wc.scale)
    _check(out16, out32, ref, "short contexts")
