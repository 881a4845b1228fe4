"""Seeded random prefill steps against the oracle, every row.

Each case draws, from its own seed, the kv heads and group size (1..16),
head_dim (64 or 128) and 1..10 sequences, each with 0..400 new tokens after
0..700 cached ones (whole prompts, chunks after cached context, empty and
single-token queries mixed). The multi-token append must leave the caches
bit-identical to the oracle's, and every query row of the causal attention
must match the oracle within the bf16 bound. Batches of one kind or the
other take the one-pair kernel or the per-unit kernel and either CTA order.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_177_gb300 import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

N_CASES = 40
N_UNITS = 6  # the last cases: whole prompts in batches with >= 4 (sequence, kv head) units per SM


def _draw(seed):
    rng = np.random.default_rng(seed)
    if seed - 3000 >= N_CASES - N_UNITS:
        g = int(rng.choice([1, 2]))
        hkv = int(rng.integers(8, 17))
        s = int(rng.integers(80, 129))
        new = rng.integers(0, 97, s)
        return g, hkv, 64 if g == 1 else 128, tuple(int(x) for x in new), (0,) * s
    g = int(rng.choice([1, 2, 3, 4, 6, 8, 16]))
    hkv = int(rng.integers(1, max(2, 9 // g) + 1))
    d = int(rng.choice([64, 128]))
    s = int(rng.integers(1, 11))
    new = rng.choice(np.concatenate([[0, 1, 16, 17, 127, 128, 129], rng.integers(1, 401, 6)]), s)
    whole = bool(rng.integers(0, 2))  # whole prompts, or chunks after cached context
    prior = np.zeros(s, dtype=np.int64) if whole else rng.integers(0, 701, s)
    return g, hkv, d, tuple(int(x) for x in new), tuple(int(x) for x in prior)


@pytest.fixture(scope="module", autouse=True)
def _device():
    torch.cuda.set_device(0)
    b = H.lib()
    b.device_error(clear=True)
    yield
    assert b.device_error(clear=True) == 0


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_prefill_step(case):
    g, hkv, d, new, prior = _draw(3000 + case)
    label = f"g={g} hkv={hkv} d={d} new={new} prior={prior}"
    w = W.make_prefill("chunked_gqa", num_seqs=len(new), num_q_heads=g * hkv, num_kv_heads=hkv, head_dim=d,
                       new_lengths="explicit", new_list=new, prior_list=prior, seed=4000 + case)
    h = {k: W.to_numpy(getattr(w, k)) for k in ("q", "k_cache", "v_cache", "k_new", "v_new")}
    hs = w.host
    oracle.kv_append(h["k_new"], h["v_new"], hs["slot_mapping"], h["k_cache"], h["v_cache"])
    ref = oracle.paged_prefill_attention(h["q"], h["k_cache"], h["v_cache"], hs["block_tables"], hs["context_lens"],
                                         hs["query_start"], w.scale, w.spec.num_kv_heads)
    wg = w.to("cuda")
    b = H.lib()
    b.kv_append(wg.k_new, wg.v_new, wg.slot_mapping, wg.k_cache, wg.v_cache)
    out = torch.full_like(wg.q, float("nan"))
    b.paged_prefill_attention(out, wg.q, wg.k_cache, wg.v_cache, wg.block_tables, wg.context_lens, wg.query_start,
                              wg.scale, max_query_len=wg.max_query_len, max_context_len=wg.max_context_len)
    torch.cuda.synchronize()
    assert b.device_error(clear=True) == 0, label
    for name in ("k_cache", "v_cache"):
        assert np.array_equal(W.to_numpy(getattr(wg, name)).view(np.uint8), h[name].view(np.uint8)), \
            f"{label}: {name} after the multi-token append differs from the oracle"
    if out.shape[0]:
        H.assert_close(out, ref, "bf16", label)
