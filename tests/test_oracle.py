"""Pins for the fp64 oracle, none of which reuse its code.

Each test fixes the oracle against something other than itself: closed forms
of special cases, a dense (never paged) brute force built from scipy's
softmax and numpy products, invariances of the paged layout, the
log-sum-exp merge identity, and explicit expected bytes for the copies.
A dropped scale, a sign error, a wrong softmax normaliser, a swapped
block/slot index, a wrong GQA mapping or a read past a sequence's tokens each
fails at least one of them.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_kv_cache_177_gb300 import workloads as W

P = 16


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (torch's round-to-nearest-even) and return the bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def widen_bits(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def paginate(K, V, num_blocks, rng, nan_fill=True, perm=None):
    """Scatter dense per-sequence K/V ([Hkv, len, d] each) over a pool of
    ``num_blocks`` blocks in a random order.  Returns caches, tables, lens."""
    S = len(K)
    Hkv, _, d = K[0].shape
    need = [-(-k.shape[1] // P) for k in K]
    perm = rng.permutation(num_blocks) if perm is None else perm
    maxb = max(max(need), 1)
    kc = np.full((num_blocks, Hkv, P, d), np.nan if nan_fill else 0.0, dtype=np.float32)
    vc = kc.copy()
    tables = np.zeros((S, maxb), dtype=np.int32)
    pos = 0
    for s in range(S):
        n = K[s].shape[1]
        for j in range(need[s]):
            b = int(perm[pos])
            pos += 1
            tables[s, j] = b
            lo, hi = j * P, min(n, (j + 1) * P)
            kc[b, :, :hi - lo] = K[s][:, lo:hi]
            vc[b, :, :hi - lo] = V[s][:, lo:hi]
        tables[s, need[s]:] = int(perm[-1]) if pos < num_blocks else 0
    lens = np.array([k.shape[1] for k in K], dtype=np.int32)
    return kc, vc, tables, lens


def dense_reference(q, K, V, scale, g):
    """Textbook attention on dense arrays with scipy's softmax."""
    S, Hq, d = q.shape
    out = np.zeros((S, Hq, d))
    for s in range(S):
        for hq in range(Hq):
            Ks = K[s][hq // g].astype(np.float64)
            Vs = V[s][hq // g].astype(np.float64)
            if Ks.shape[0] == 0:
                continue
            w = scipy.special.softmax(scale * (Ks @ q[s, hq].astype(np.float64)))
            out[s, hq] = w @ Vs
    return out


def run_oracle(q, kc, vc, tables, lens, scale, hkv, **kw):
    return oracle.paged_decode_attention(q, kc, vc, tables, lens, scale, hkv, **kw)


# --- closed forms -------------------------------------------------------------

@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_two_token_closed_form(sign):
    """q = +-e0, K0 = (ln 3 / scale) e0, K1 = 0: weights (3/4, 1/4) for +, (1/4, 3/4) for -."""
    d, scale = 64, 1.0 / 8.0
    rng = np.random.default_rng(0)
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = sign
    K = np.zeros((1, 2, d), np.float32)
    K[0, 0, 0] = math.log(3.0) / scale
    V = rng.standard_normal((1, 2, d)).astype(np.float32)
    kc, vc, t, lens = paginate([K], [V], 4, rng)
    out = run_oracle(q, kc, vc, t, lens, scale, 1)[0, 0]
    w0 = 0.75 if sign > 0 else 0.25
    expect = w0 * V[0, 0].astype(np.float64) + (1 - w0) * V[0, 1].astype(np.float64)
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-6)


def test_single_token_returns_value_row():
    rng = np.random.default_rng(1)
    d = 128
    q = rng.standard_normal((1, 2, d)).astype(np.float32)
    K = rng.standard_normal((2, 1, d)).astype(np.float32) * 30
    V = rng.standard_normal((2, 1, d)).astype(np.float32)
    kc, vc, t, lens = paginate([K], [V], 3, rng)
    out = run_oracle(q, kc, vc, t, lens, 0.1, 2)
    assert np.array_equal(out[0, 0], V[0, 0].astype(np.float64))
    assert np.array_equal(out[0, 1], V[1, 0].astype(np.float64))


@pytest.mark.parametrize("n", [2, 15, 16, 17, 100])
def test_equal_keys_and_zero_query_give_mean(n):
    rng = np.random.default_rng(n)
    d = 64
    row = rng.standard_normal(d).astype(np.float32)
    K = np.broadcast_to(row, (1, n, d)).copy()
    V = rng.standard_normal((1, n, d)).astype(np.float32)
    q = rng.standard_normal((2, 1, d)).astype(np.float32)
    q[1] = 0.0
    kc, vc, t, lens = paginate([K, rng.standard_normal((1, n, d)).astype(np.float32)], [V, V], 32, rng)
    out = run_oracle(q, kc, vc, t, lens, 0.125, 1)
    mean = V[0].astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(out[0, 0], mean, rtol=0, atol=1e-12)   # equal keys
    np.testing.assert_allclose(out[1, 0], mean, rtol=0, atol=1e-12)   # zero query


def test_gqa_consecutive_grouping():
    """q head hq reads kv head hq // g: constant V per kv head gives that
    constant; a key that matches only in kv head h picks that head's row."""
    rng = np.random.default_rng(2)
    Hkv, g, d, n = 4, 3, 64, 40
    Hq = Hkv * g
    K = rng.standard_normal((Hkv, n, d)).astype(np.float32) * 0.01
    V = np.empty((Hkv, n, d), np.float32)
    for h in range(Hkv):
        V[h] = 0.5 * (h + 1)
    q = rng.standard_normal((1, Hq, d)).astype(np.float32)
    kc, vc, t, lens = paginate([K], [V], 8, rng)
    out = run_oracle(q, kc, vc, t, lens, 0.125, Hkv)
    for hq in range(Hq):
        np.testing.assert_allclose(out[0, hq], 0.5 * (hq // g + 1), rtol=0, atol=1e-12)
    # keys: kv head h has a dominant match at token 7 + h; values differ per token
    q = np.zeros((1, Hq, d), np.float32)
    q[0, :, 0] = 1.0
    K = np.zeros((Hkv, n, d), np.float32)
    for h in range(Hkv):
        K[h, 7 + h, 0] = 400.0
    V = rng.standard_normal((Hkv, n, d)).astype(np.float32)
    kc, vc, t, lens = paginate([K], [V], 8, rng)
    out = run_oracle(q, kc, vc, t, lens, 0.125, Hkv)
    for hq in range(Hq):
        h = hq // g
        np.testing.assert_allclose(out[0, hq], V[h, 7 + h], rtol=0, atol=1e-12)


def test_empty_context_gives_zeros():
    rng = np.random.default_rng(3)
    d = 64
    K = [np.zeros((2, 0, d), np.float32), rng.standard_normal((2, 5, d)).astype(np.float32)]
    V = [np.zeros((2, 0, d), np.float32), rng.standard_normal((2, 5, d)).astype(np.float32)]
    q = rng.standard_normal((2, 2, d)).astype(np.float32)
    kc, vc, t, lens = paginate(K, V, 4, rng)
    out = run_oracle(q, kc, vc, t, lens, 0.125, 2)
    assert np.array_equal(out[0], np.zeros((2, d)))
    assert np.all(np.isfinite(out[1]))


# --- brute force on dense tensors ----------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_matches_dense_bruteforce(dtype, g):
    rng = np.random.default_rng(10 + g)
    d, Hkv = 64 if g != 8 else 128, 2
    lens = [1, 15, 16, 17, 33, 64, 5, 100]
    K = [rng.standard_normal((Hkv, n, d)).astype(np.float32) for n in lens]
    V = [rng.standard_normal((Hkv, n, d)).astype(np.float32) for n in lens]
    q = rng.standard_normal((len(lens), Hkv * g, d)).astype(np.float32)
    if dtype == "bf16":
        K = [widen_bits(bf16_bits(k)).astype(np.float32) for k in K]
        V = [widen_bits(bf16_bits(v)).astype(np.float32) for v in V]
        q = widen_bits(bf16_bits(q)).astype(np.float32)
    kc, vc, t, ln = paginate(K, V, 64, rng)
    scale = 1.0 / math.sqrt(d)
    if dtype == "bf16":
        got = run_oracle(bf16_bits(q), bf16_bits(kc), bf16_bits(vc), t, ln, scale, Hkv)
    else:
        got = run_oracle(q, kc, vc, t, ln, scale, Hkv)
    ref = dense_reference(q, K, V, scale, g)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


# --- layout invariances ---------------------------------------------------------

def test_permutation_of_physical_blocks_is_bit_invariant():
    rng = np.random.default_rng(4)
    d, Hkv = 64, 2
    lens = [3, 16, 31, 48, 70]
    K = [rng.standard_normal((Hkv, n, d)).astype(np.float32) for n in lens]
    V = [rng.standard_normal((Hkv, n, d)).astype(np.float32) for n in lens]
    q = rng.standard_normal((len(lens), 4, d)).astype(np.float32)
    outs = []
    for seed in range(3):
        kc, vc, t, ln = paginate(K, V, 40, np.random.default_rng(100 + seed))
        outs.append(run_oracle(q, kc, vc, t, ln, 0.125, Hkv))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_shared_prefix_equals_duplicated_blocks():
    rng = np.random.default_rng(5)
    d, Hkv = 64, 2
    prefix = 48  # three full blocks
    Kp = rng.standard_normal((Hkv, prefix, d)).astype(np.float32)
    Vp = rng.standard_normal((Hkv, prefix, d)).astype(np.float32)
    suff = [rng.standard_normal((Hkv, n, d)).astype(np.float32) for n in (0, 5, 16, 21)]
    suffv = [rng.standard_normal((Hkv, n, d)).astype(np.float32) for n in (0, 5, 16, 21)]
    K = [np.concatenate([Kp, s], axis=1) for s in suff]
    V = [np.concatenate([Vp, s], axis=1) for s in suffv]
    q = rng.standard_normal((4, Hkv, d)).astype(np.float32)
    kc, vc, t, ln = paginate(K, V, 40, rng)               # duplicated prefix blocks
    dup = run_oracle(q, kc, vc, t, ln, 0.125, Hkv)
    t_shared = t.copy()
    t_shared[1:, :3] = t[0, :3]                           # every sample points at sample 0's prefix
    shared = run_oracle(q, kc, vc, t_shared, ln, 0.125, Hkv)
    assert np.array_equal(dup, shared)


def test_poisoned_unread_memory_does_not_leak():
    rng = np.random.default_rng(6)
    d, Hkv = 64, 1
    lens = [1, 17, 40]
    K = [rng.standard_normal((Hkv, n, d)).astype(np.float32) for n in lens]
    V = [rng.standard_normal((Hkv, n, d)).astype(np.float32) for n in lens]
    q = rng.standard_normal((3, 1, d)).astype(np.float32)
    perm = rng.permutation(16)
    clean = run_oracle(q, *paginate(K, V, 16, rng, nan_fill=False, perm=perm), 0.125, 1)
    kc, vc, t, ln = paginate(K, V, 16, rng, nan_fill=True, perm=perm)
    poisoned = run_oracle(q, kc, vc, t, ln, 0.125, 1)
    assert np.isnan(kc).any()
    assert np.all(np.isfinite(poisoned)) and np.array_equal(clean, poisoned)


# --- partition identity (what split-context decode relies on) ----------------------

def test_log_sum_exp_merge_of_partitions_equals_whole():
    rng = np.random.default_rng(7)
    d, n, part = 64, 1500, 512
    K = rng.standard_normal((1, n, d)).astype(np.float32)
    V = rng.standard_normal((1, n, d)).astype(np.float32)
    q = rng.standard_normal((1, 1, d)).astype(np.float32) * 3
    kc, vc, t, ln = paginate([K], [V], 100, rng)
    whole = run_oracle(q, kc, vc, t, ln, 0.125, 1)[0, 0]
    ms, ls, os_ = [], [], []
    for lo in range(0, n, part):
        x = 0.125 * (K[0, lo:lo + part].astype(np.float64) @ q[0, 0].astype(np.float64))
        m = x.max()
        e = np.exp(x - m)
        ms.append(m)
        ls.append(e.sum())
        os_.append(e @ V[0, lo:lo + part].astype(np.float64) / e.sum())
    M = max(ms)
    w = np.array([l * math.exp(m - M) for m, l in zip(ms, ls)])
    merged = (w[:, None] * np.array(os_)).sum(0) / w.sum()
    np.testing.assert_allclose(whole, merged, rtol=0, atol=1e-12)


# --- error behaviour ----------------------------------------------------------------

def test_out_of_range_block_and_overlong_context_raise():
    rng = np.random.default_rng(8)
    K = [rng.standard_normal((1, 20, 64)).astype(np.float32)]
    kc, vc, t, ln = paginate(K, K, 4, rng)
    q = np.ones((1, 1, 64), np.float32)
    bad = t.copy()
    bad[0, 1] = 4
    with pytest.raises(ValueError):
        run_oracle(q, kc, vc, bad, ln, 0.1, 1)
    with pytest.raises(ValueError):
        run_oracle(q, kc, vc, t, np.array([t.shape[1] * P + 1], np.int32), 0.1, 1)


def test_seq_subset_matches_full():
    w = W.make_workload("tiny")
    q, kc, vc = (W.to_numpy(x) for x in (w.q, w.k_cache, w.v_cache))
    kn, vn = W.to_numpy(w.k_new), W.to_numpy(w.v_new)
    oracle.kv_append(kn, vn, w.layout.slot_mapping, kc, vc)
    full = oracle.paged_decode_attention(q, kc, vc, w.layout.block_tables, w.layout.context_lens, w.scale, 8)
    sub = oracle.paged_decode_attention(q, kc, vc, w.layout.block_tables, w.layout.context_lens, w.scale, 8,
                                        seq_ids=[2, 0], nthreads=1)
    assert np.array_equal(sub[0], full[2]) and np.array_equal(sub[1], full[0])
    assert np.all(np.isfinite(full))


def test_tiny_workload_against_dense_gather():
    """The oracle on the tiny workload equals scipy attention on K/V gathered
    with numpy fancy indexing (an independent gather)."""
    w = W.make_workload("tiny")
    lay = w.layout
    q, kc, vc = (W.to_numpy(x) for x in (w.q, w.k_cache, w.v_cache))
    oracle.kv_append(W.to_numpy(w.k_new), W.to_numpy(w.v_new), lay.slot_mapping, kc, vc)
    Ks, Vs = [], []
    for s in range(lay.spec.num_seqs):
        n = int(lay.context_lens[s])
        tok = np.arange(n)
        blk = lay.block_tables[s, tok // P]
        Ks.append(kc[blk, :, tok % P, :].transpose(1, 0, 2))
        Vs.append(vc[blk, :, tok % P, :].transpose(1, 0, 2))
    ref = dense_reference(q, Ks, Vs, w.scale, 1)
    got = oracle.paged_decode_attention(q, kc, vc, lay.block_tables, lay.context_lens, w.scale, 8)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


# --- copies -------------------------------------------------------------------------

def test_kv_append_writes_exactly_the_mapped_slots():
    NB, Hkv, d = 3, 2, 8
    kc = np.arange(NB * Hkv * P * d, dtype=np.float32).reshape(NB, Hkv, P, d)
    vc = -kc
    before_k, before_v = kc.copy(), vc.copy()
    k = np.full((3, Hkv, d), 7.0, np.float32)
    v = np.full((3, Hkv, d), -7.0, np.float32)
    k[1] = 9.0
    oracle.kv_append(k, v, np.array([17, -1, 47], np.int64), kc, vc)
    # slot 17 = block 1, offset 1; slot 47 = block 2, offset 15; -1 skipped
    expect_k = before_k.copy()
    expect_v = before_v.copy()
    expect_k[1, :, 1, :] = 7.0
    expect_v[1, :, 1, :] = -7.0
    expect_k[2, :, 15, :] = 7.0
    expect_v[2, :, 15, :] = -7.0
    assert np.array_equal(kc, expect_k) and np.array_equal(vc, expect_v)


def test_copy_blocks_copies_whole_blocks():
    NB, Hkv, d = 5, 3, 4
    kc = np.arange(NB * Hkv * P * d, dtype=np.float32).reshape(NB, Hkv, P, d)
    vc = kc * 2
    ek, ev = kc.copy(), vc.copy()
    oracle.copy_blocks(kc, vc, np.array([[0, 3], [2, 4]], np.int64))
    ek[3], ev[3] = ek[0], ev[0]
    ek[4], ev[4] = ek[2], ev[2]
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)
    with pytest.raises(ValueError):
        oracle.copy_blocks(kc, vc, np.array([[0, 5]], np.int64))


# --- causal prefill ---------------------------------------------------------------------

def dense_causal_reference(q_rows, K, V, scale, g, n_new):
    """scipy softmax over each query's visible prefix of dense K/V."""
    ctx = K.shape[1]
    out = np.zeros(q_rows.shape, dtype=np.float64)
    for i in range(n_new):
        pos = ctx - n_new + i
        for hq in range(q_rows.shape[1]):
            Ks = K[hq // g, :pos + 1].astype(np.float64)
            Vs = V[hq // g, :pos + 1].astype(np.float64)
            w = scipy.special.softmax(scale * (Ks @ q_rows[i, hq].astype(np.float64)))
            out[i, hq] = w @ Vs
    return out


@pytest.mark.parametrize("g", [1, 4])
def test_prefill_matches_dense_causal_bruteforce(g):
    rng = np.random.default_rng(50 + g)
    d, Hkv = 64, 2
    # (context length, new tokens): whole prompts, chunks after earlier context, single tokens
    shapes = [(1, 1), (17, 17), (40, 9), (33, 1), (64, 64), (100, 37)]
    K = [rng.standard_normal((Hkv, c, d)).astype(np.float32) for c, _ in shapes]
    V = [rng.standard_normal((Hkv, c, d)).astype(np.float32) for c, _ in shapes]
    qs = np.concatenate([[0], np.cumsum([n for _, n in shapes])]).astype(np.int32)
    q = rng.standard_normal((int(qs[-1]), Hkv * g, d)).astype(np.float32)
    kc, vc, t, ln = paginate(K, V, 64, rng)
    got = oracle.paged_prefill_attention(q, kc, vc, t, ln, qs, 0.125, Hkv)
    for s, (c, n) in enumerate(shapes):
        ref = dense_causal_reference(q[qs[s]:qs[s + 1]], K[s], V[s], 0.125, g, n)
        np.testing.assert_allclose(got[qs[s]:qs[s + 1]], ref, rtol=1e-12, atol=1e-12)


def test_prefill_first_query_sees_only_itself_and_last_query_is_decode():
    rng = np.random.default_rng(60)
    d, Hkv, n = 128, 1, 30
    K = [rng.standard_normal((Hkv, n, d)).astype(np.float32)]
    V = [rng.standard_normal((Hkv, n, d)).astype(np.float32)]
    kc, vc, t, ln = paginate(K, V, 8, rng)
    q = rng.standard_normal((n, 2, d)).astype(np.float32)
    out = oracle.paged_prefill_attention(q, kc, vc, t, ln, np.array([0, n], np.int32), 0.1, Hkv)
    assert np.array_equal(out[0, 0], V[0][0, 0].astype(np.float64))      # position 0 attends to itself alone
    dec = oracle.paged_decode_attention(q[n - 1:n], kc, vc, t, ln, 0.1, Hkv)
    np.testing.assert_allclose(out[n - 1], dec[0], rtol=0, atol=1e-14)
