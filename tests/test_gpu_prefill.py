"""GPU parity of a prefill step: the multi-token KV append of every new token
(bit-exact) and causal prefill attention over the paged cache, against the
oracle."""
import numpy as np
import pytest
import torch

import oracle
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


def _host(w):
    return {k: W.to_numpy(getattr(w, k)) for k in ("q", "k_cache", "v_cache", "k_new", "v_new")}


def _oracle(h, w, seqs=None):
    """Oracle append (in place on the host caches) and prefill attention, for
    every sequence or for the listed ones (their query rows, in order)."""
    hs = w.host
    oracle.kv_append(h["k_new"], h["v_new"], hs["slot_mapping"], h["k_cache"], h["v_cache"])
    if seqs is None:
        return oracle.paged_prefill_attention(h["q"], h["k_cache"], h["v_cache"], hs["block_tables"],
                                              hs["context_lens"], hs["query_start"], w.scale,
                                              w.spec.num_kv_heads)
    qs = hs["query_start"]
    rows = np.concatenate([np.arange(qs[s], qs[s + 1]) for s in seqs])
    sub_qs = np.concatenate([[0], np.cumsum([qs[s + 1] - qs[s] for s in seqs])]).astype(np.int32)
    return oracle.paged_prefill_attention(np.ascontiguousarray(h["q"][rows]), h["k_cache"], h["v_cache"],
                                          np.ascontiguousarray(hs["block_tables"][seqs]),
                                          np.ascontiguousarray(hs["context_lens"][seqs]), sub_qs, w.scale,
                                          w.spec.num_kv_heads), rows


def _gpu(w):
    b = H.lib()
    b.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)
    out = torch.full_like(w.q, float("nan"))
    b.paged_prefill_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.query_start,
                              w.scale, max_query_len=w.max_query_len, max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    return out


def _check(w, what):
    h = _host(w)
    ref = _oracle(h, w)
    wg = w.to("cuda")
    out = _gpu(wg)
    for name in ("k_cache", "v_cache"):
        assert np.array_equal(W.to_numpy(getattr(wg, name)).view(np.uint8), h[name].view(np.uint8)), \
            f"{what}: {name} after the multi-token append differs from the oracle"
    if out.shape[0]:
        H.assert_close(out, ref, "bf16", what)
    return out


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 64), (32, 8, 128), (12, 4, 64), (16, 2, 128), (64, 1, 64)])
def test_chunked_prefill_matches_the_oracle(hq, hkv, d):
    """Whole prompts and chunks after cached context, for group sizes 1, 3, 4,
    8 and 64 (a 128-row tile holds 128, 42, 32, 16 and 2 tokens)."""
    w = W.make_prefill("chunked_gqa", num_seqs=6, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, new_hi=150,
                       prior_hi=300, seed=hq * 131 + d)
    _check(w, f"chunked hq={hq} hkv={hkv} d={d}")


def test_edge_cases():
    """No new tokens, one new token (a decode step), a whole prompt that ends
    on a block boundary, one of a single token, a chunk starting mid-block,
    and a long prompt over many tiles with a ragged last tile."""
    new = (0, 1, 32, 1, 17, 333, 5, 64)
    prior = (9, 40, 0, 0, 23, 0, 11, 64)
    w = W.make_prefill("chunked_gqa", new_list=new, prior_list=prior, seed=5)
    _check(w, "edge cases")


def test_single_token_prefill_equals_decode():
    """With one new token per sequence, prefill is the decode step: same
    result as paged_decode_attention on the same cache (both within the
    oracle's tolerance, and close to each other)."""
    w = W.make_prefill("chunked_gqa", new_list=(1,) * 7, prior_list=(0, 15, 16, 100, 257, 31, 1000), seed=9)
    out = _check(w, "one token per sequence")
    wg = w.to("cuda")
    b = H.lib()
    b.kv_append(wg.k_new, wg.v_new, wg.slot_mapping, wg.k_cache, wg.v_cache)
    dec = torch.empty_like(wg.q)
    b.paged_decode_attention(dec, wg.q, wg.k_cache, wg.v_cache, wg.block_tables, wg.context_lens, wg.scale,
                             max_context_len=w.max_context_len, partition_tokens=64)
    torch.cuda.synchronize()
    assert float((out.float() - dec.float()).abs().max()) < 4e-3


def test_over_long_query_is_flagged_and_rows_left_alone():
    """n_s larger than the context: the sequence is skipped and flagged."""
    b = H.lib()
    w = W.make_prefill("chunked_gqa", new_list=(5, 3), prior_list=(10, 4), seed=3).to("cuda")
    b.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)
    lens = w.context_lens.clone()
    lens[1] = 2                                   # 3 new tokens in a context of 2
    out = torch.zeros_like(w.q)
    b.paged_prefill_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.query_start, w.scale,
                              max_query_len=5, max_context_len=14)
    torch.cuda.synchronize()
    assert b.device_error(clear=True) == b.DEVERR_LENGTH
    assert torch.all(out[5:] == 0)
    assert torch.all(torch.isfinite(out[:5].float())) and bool(torch.any(out[:5] != 0))


def test_full_size_prefill13b_sampled():
    """The 13B-class prefill step at full size; attention checked against the
    oracle on the longest, the shortest and two middle prompts, the append
    on every slot."""
    w = W.make_prefill("prefill13b", device="cuda")
    h = _host(w)
    out = _gpu(w)
    n = np.diff(w.host["query_start"])
    order = np.argsort(n)
    seqs = [int(order[-1]), int(order[0]), int(order[len(n) // 2]), int(order[len(n) // 3])]
    ref, rows = _oracle(h, w, seqs)
    for name in ("k_cache", "v_cache"):
        assert np.array_equal(W.to_numpy(getattr(w, name)).view(np.uint8), h[name].view(np.uint8))
    H.assert_close(out[torch.from_numpy(rows).cuda()], ref, "bf16", "prefill13b sample")
    assert bool(torch.all(torch.isfinite(out.float())))


def test_short_prompts_stay_within_tolerance():
    """Prompts of 2..17 tokens (every query sees at most 17 keys), the case the
    first chunk's weight remainder is there for."""
    new = tuple(2 + (i % 16) for i in range(96))
    w = W.make_prefill("chunked_gqa", new_list=new, prior_list=(0,) * len(new), seed=29)
    _check(w, "short prompts")


def test_long_prefix_chunks_sampled():
    """512-token chunks after 16K-32K cached tokens: four query rows at the
    start and four at the end of three sequences' chunks, each checked as the
    last four tokens of a context cut right after them."""
    w = W.make_prefill("long_prefix", device="cuda")
    h = _host(w)
    out = _gpu(w)
    hs = w.host
    oracle.kv_append(h["k_new"], h["v_new"], hs["slot_mapping"], h["k_cache"], h["v_cache"])
    qs, lens = hs["query_start"], hs["context_lens"]
    for s in (0, 3, 7):
        n = int(qs[s + 1] - qs[s])
        for first in (0, n - 4):
            rows = np.arange(qs[s] + first, qs[s] + first + 4)
            cut = np.array([lens[s] - n + first + 4], np.int32)
            ref = oracle.paged_prefill_attention(np.ascontiguousarray(h["q"][rows]), h["k_cache"], h["v_cache"],
                                                 np.ascontiguousarray(hs["block_tables"][s:s + 1]), cut,
                                                 np.array([0, 4], np.int32), w.scale, w.spec.num_kv_heads)
            H.assert_close(out[torch.from_numpy(rows).cuda()], ref, "bf16", f"long prefix seq {s} rows {first}..")


@pytest.mark.parametrize("num_seqs", [24, 130])
def test_cta_order_does_not_change_the_result(num_seqs):
    """The grid is issued pair index slowest when the contexts are not much
    longer than the new tokens, else one sequence at a time in decreasing order
    of context length (ranked inside the kernel for batches of up to 128 sequences,
    in index order beyond). A larger host bound on the context length selects
    the second order for the same inputs: both outputs match the oracle, and
    where the same kernel runs both orders (24 sequences x 8 kv heads, too few
    units for the per-unit kernel) they are bit-identical. With 130 sequences
    the first order runs the per-unit kernel, which splits the first chunk's
    weights only in tiles holding rows that see at most 64 keys, so other
    tiles' first-chunk weights round differently there. Lengths repeat, so the
    ranking meets ties."""
    rng = np.random.default_rng(num_seqs)
    new = tuple(int(x) for x in rng.choice([1, 7, 64, 130, 300] if num_seqs < 100 else [1, 7, 40, 150], num_seqs))
    prior = tuple(int(x) for x in rng.choice([0, 5, 100], num_seqs))
    w = W.make_prefill("chunked_gqa", new_list=new, prior_list=prior, seed=num_seqs)
    h = _host(w)
    ref = _oracle(h, w)
    wg = w.to("cuda")
    b = H.lib()
    b.kv_append(wg.k_new, wg.v_new, wg.slot_mapping, wg.k_cache, wg.v_cache)
    outs = []
    assert w.max_context_len < 2 * w.max_query_len          # the default bound gives the first order
    for bound in (w.max_context_len, max(w.max_context_len, 2 * w.max_query_len)):
        out = torch.full_like(wg.q, float("nan"))
        b.paged_prefill_attention(out, wg.q, wg.k_cache, wg.v_cache, wg.block_tables, wg.context_lens,
                                  wg.query_start, wg.scale, max_query_len=w.max_query_len, max_context_len=bound)
        torch.cuda.synchronize()
        outs.append(out)
    for o, order in zip(outs, ("pair index slowest", "one sequence at a time")):
        H.assert_close(o, ref, "bf16", f"{num_seqs} sequences, {order}")
    if w.spec.num_seqs * w.spec.num_kv_heads < 4 * torch.cuda.get_device_properties(0).multi_processor_count:
        assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
