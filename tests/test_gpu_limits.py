"""Decode at the library's size limits, every output against the oracle.

- One sequence of 131,072 tokens cut into 16-token partitions: 8,192
  partitions, the most the log-sum-exp reduce takes; one token more needs
  8,193 and is refused before any launch.
- 65,535 sequences, the most the launch grid addresses: far past the
  persistent kernel's table of 8,192, so the automatic choice is the grid
  kernel; short ragged contexts, and the same batch with fp32 caches.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_177_gb300 import binding as B
from paged_kv_cache_177_gb300 import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    b = H.lib()
    b.device_error(clear=True)
    yield
    assert b.device_error(clear=True) == 0, "a kernel raised the device error word"


def _check(wc, partition_tokens):
    h = H.host_arrays(wc)
    ref = H.oracle_step(h, wc.layout, wc.scale)
    w = wc.to("cuda")
    out = H.gpu_step(w, partition_tokens)
    torch.cuda.synchronize()
    H.assert_caches_equal(w, h)
    return H.assert_close(out, ref, wc.spec.dtype, f"{wc.spec.name}, partition_tokens={partition_tokens}")


def test_most_partitions_the_reduce_takes():
    wc = W.make_workload("gqa8b", lengths_list=(131072, 5), num_q_heads=4, num_kv_heads=1, seed=902)
    b = H.lib()
    assert b.decode_launches(2, 1, wc.layout.max_context_len, 16) == 2
    _check(wc, 16)


def test_one_partition_past_the_limit_is_refused():
    # 131,073 tokens in 16-token partitions: 8,193 partitions. The buffers match the
    # arguments, so even a launch would read nothing out of bounds; none happens.
    S, Hq, Hkv, D, L = 1, 4, 1, 128, 131073
    nb = (L + 15) // 16
    q = torch.zeros(S, Hq, D, dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(q, 7.0)
    kc = torch.zeros(nb, Hkv, 16, D, dtype=torch.bfloat16, device="cuda")
    tables = torch.arange(nb, dtype=torch.int32, device="cuda").reshape(1, nb)
    lens = torch.full((S,), L, dtype=torch.int32, device="cuda")
    ws = torch.zeros(H.lib().workspace_bytes(S, Hq, Hkv, D, L, 16), dtype=torch.uint8, device="cuda")
    with pytest.raises(B.PagedKVError) as e:
        H.lib().paged_decode_attention(out, q, kc, kc, tables, lens, 0.088, max_context_len=L, partition_tokens=16,
                                       workspace=ws)
    torch.cuda.synchronize()
    assert e.value.code == -2    # PKV_ERR_UNSUPPORTED
    assert bool((out == 7.0).all())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_most_sequences_the_grid_addresses(dtype):
    rng = np.random.default_rng(7)
    lens = tuple(int(x) for x in rng.integers(1, 34, 65535))
    wc = W.make_workload("gqa8b", lengths_list=lens, num_q_heads=2, num_kv_heads=1, dtype=dtype, seed=901)
    assert not H.lib().decode_persistent(65535, 1, 0, H.torch_dtype(wc.spec))
    _check(wc, 0)
