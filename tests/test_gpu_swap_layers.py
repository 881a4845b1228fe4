"""GPU parity of the block moves beyond copy-on-write: swapping blocks to a
pinned host pool and back, multi-layer copy and append, and an engine loop
that drives the scheduler through every device call of a decode step."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_177_gb300 import scheduler as S
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


def _bits(t):
    return W.to_numpy(t).view(np.uint8)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_swap_out_and_back_in_is_bit_exact_and_attention_unchanged(dtype):
    b = H.lib()
    w = W.make_workload("gqa8b", lengths_list=(40, 3, 70, 16, 129), dtype="bf16" if dtype == torch.bfloat16 else "f32",
                        seed=31).to("cuda")
    H.gpu_step(w, attention=False)
    lay = w.layout
    out0 = torch.empty_like(w.q)
    b.paged_decode_attention(out0, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                             max_context_len=lay.max_context_len, partition_tokens=64)
    # swap every referenced block out to a pinned host pool ...
    used = np.nonzero(lay.used_blocks)[0]
    host_nb = len(used) + 5
    hk = torch.zeros((host_nb,) + tuple(w.k_cache.shape[1:]), dtype=dtype, pin_memory=True)
    hv = torch.zeros_like(hk).pin_memory()
    host_ids = np.random.default_rng(0).permutation(host_nb)[:len(used)]
    out_pairs = np.stack([used, host_ids], 1).astype(np.int64)
    b.swap_blocks(hk, hv, w.k_cache, w.v_cache, torch.from_numpy(out_pairs).cuda(), host_pairs=out_pairs)
    torch.cuda.synchronize()
    ek, ev = oracle_pool_copy(_np(w.k_cache), _np(hk), out_pairs), oracle_pool_copy(_np(w.v_cache), _np(hv), out_pairs)
    assert np.array_equal(_np(hk).view(np.uint8), ek.view(np.uint8))
    assert np.array_equal(_np(hv).view(np.uint8), ev.view(np.uint8))
    # ... and back in to different device blocks (pairs given as a pinned host tensor)
    dk = torch.full_like(w.k_cache, float("nan"))
    dv = torch.full_like(w.v_cache, float("nan"))
    new_ids = np.random.default_rng(1).permutation(lay.num_blocks)[:len(used)]
    in_pairs = np.stack([host_ids, new_ids], 1).astype(np.int64)
    b.swap_blocks(dk, dv, hk, hv, torch.from_numpy(in_pairs).pin_memory(), host_pairs=in_pairs)
    remap = np.arange(lay.num_blocks)
    remap[used] = new_ids
    tables = torch.from_numpy(remap[lay.block_tables].astype(np.int32)).cuda()
    out1 = torch.empty_like(w.q)
    b.paged_decode_attention(out1, w.q, dk, dv, tables, w.context_lens, w.scale, max_context_len=lay.max_context_len,
                             partition_tokens=64)
    torch.cuda.synchronize()
    for o, n in zip(used, new_ids):
        assert torch.equal(dk[n].view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                           w.k_cache[o].view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    assert torch.equal(out0, out1)


def _np(t):
    return W.to_numpy(t)


def oracle_pool_copy(src, dst, pairs):
    dst = dst.copy()
    for s_, d_ in pairs:
        dst[d_] = src[s_]
    return dst


def test_swap_pair_checks_and_device_flag():
    b = H.lib()
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    hk = torch.zeros(3, 2, 16, 64, dtype=torch.bfloat16, pin_memory=True)
    with pytest.raises(b.PagedKVError):
        b.check_swap_pairs([[0, 3]], 4, 3)           # destination past the host pool
    with pytest.raises(b.PagedKVError):
        b.check_swap_pairs([[0, 1], [2, 1]], 4, 3)   # repeated destination
    b.check_swap_pairs([[0, 1], [0, 2]], 4, 3)       # one source to two places is fine
    bad = torch.tensor([[0, 7]], dtype=torch.int64, device="cuda")
    b.swap_blocks(hk, hk, kc, kc, bad, check=False)
    torch.cuda.synchronize()
    assert b.device_error(clear=True) == b.DEVERR_PAIR


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_multi_layer_append_and_copy_are_bit_exact(dtype):
    b = H.lib()
    L = 3
    w0 = W.make_workload("tiny", dtype=dtype, seed=40, num_kv_heads=4, num_q_heads=4)
    lay = w0.layout
    # one layout for every layer (one slot mapping, one set of pairs), different values per layer
    ks = [w0.k_cache + l for l in range(L)]
    vs = [w0.v_cache - l for l in range(L)]
    kns = [w0.k_new * (l + 1) for l in range(L)]
    vns = [w0.v_new * (l + 2) for l in range(L)]
    kcs = [k.cuda() for k in ks]
    vcs = [v.cuda() for v in vs]
    kn = [k.cuda() for k in kns]
    vn = [v.cuda() for v in vns]
    slots = torch.from_numpy(lay.slot_mapping.copy()).cuda()
    pairs = torch.from_numpy(lay.cow_pairs.copy()).cuda()
    b.copy_blocks_layers(kcs, vcs, pairs, host_pairs=lay.cow_pairs)
    b.kv_append_layers(kn, vn, slots, kcs, vcs)
    torch.cuda.synchronize()
    for l in range(L):
        k, v = _np(ks[l]), _np(vs[l])
        oracle.copy_blocks(k, v, lay.cow_pairs)
        oracle.kv_append(_np(kns[l]), _np(vns[l]), lay.slot_mapping, k, v)
        assert np.array_equal(_np(kcs[l]).view(np.uint8), k.view(np.uint8)), f"layer {l} K"
        assert np.array_equal(_np(vcs[l]).view(np.uint8), v.view(np.uint8)), f"layer {l} V"


def test_multi_layer_null_pointer_is_flagged_not_followed():
    b = H.lib()
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    ptrs = torch.tensor([kc.data_ptr(), 0], dtype=torch.int64, device="cuda")   # layer 1 has no cache
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
    lib = b.raw_library()
    rc = lib.copy_blocks_layers(ptrs.data_ptr(), ptrs.data_ptr(), 2, pairs.data_ptr(), 1, 2, 64, 4, 1,
                                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert b.device_error(clear=True) == b.DEVERR_POINTER


# ---- an engine loop: the scheduler drives every device call of each step, including the
# prefill attention of newly admitted prompts ----------------------------------------------

def test_engine_loop_matches_the_oracle_every_step():
    b = H.lib()
    rng = np.random.default_rng(3)
    Hq, Hkv, D, NB, HNB = 8, 4, 128, 12, 60
    scale = 1.0 / np.sqrt(D)
    reqs = []
    for p in range(4):
        plen = int(rng.integers(10, 40))
        reqs.append(S.Request(10 * p, prompt_len=plen, output_len=int(rng.integers(5, 30))))
        for c in (1, 2):
            reqs.append(S.Request(10 * p + c, prompt_len=plen, output_len=int(rng.integers(5, 30)), parent=10 * p))
    for i in range(6):
        reqs.append(S.Request(100 + i, prompt_len=int(rng.integers(1, 50)), output_len=int(rng.integers(3, 40))))
    sched = S.IterationScheduler(NB, 6, host_blocks=HNB, order=rng.permutation(NB))
    for r in reqs:
        sched.add(r)
    root = {r.req_id: (r.parent if r.parent is not None else r.req_id) for r in reqs}
    prompt = {r.req_id: r.prompt_len for r in reqs}

    def kv_of(sid, pos):
        owner = root[sid] if pos < prompt[sid] else sid
        g = np.random.default_rng(owner * 100_000 + pos)
        return g.standard_normal((2, Hkv, D)).astype(np.float32)

    def bf(x):
        return torch.from_numpy(x).to(torch.bfloat16)

    dk = torch.full((NB, Hkv, 16, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    dv = torch.full_like(dk, float("nan"))
    hk = torch.zeros((HNB, Hkv, 16, D), dtype=torch.bfloat16, pin_memory=True)
    hv = torch.zeros_like(hk).pin_memory()
    sk, sv = _np(dk).copy(), _np(dv).copy()          # host shadows of the device pools
    shk, shv = _np(hk).copy(), _np(hv).copy()
    steps = swaps_seen = prefills_seen = 0
    while not sched.idle():
        st = sched.step()
        assert st is not None
        cuda = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        if len(st.swap_in_pairs):
            swaps_seen += 1
            b.swap_blocks(dk, dv, hk, hv, cuda(st.swap_in_pairs), host_pairs=st.swap_in_pairs)
            for h, d in st.swap_in_pairs:
                sk[d], sv[d] = shk[h], shv[h]
        # prefill: every prompt (and recomputed) token of newly admitted sequences
        pre_slots, pre_kv = [], []
        for sid, n, table in st.prefilled:
            for pos in range(n):
                pre_slots.append(table[pos // 16] * 16 + pos % 16)
                pre_kv.append(kv_of(sid, pos))
        if pre_slots:
            kvs = np.stack(pre_kv)
            kb, vb = bf(kvs[:, 0]), bf(kvs[:, 1])
            b.kv_append(kb.cuda(), vb.cuda(), cuda(np.array(pre_slots, np.int64)), dk, dv)
            oracle.kv_append(_np(kb), _np(vb), np.array(pre_slots, np.int64), sk, sv)
            # prefill attention of the admitted prompts (causal over their own tokens)
            n_pre = [n for _, n, _ in st.prefilled]
            maxb = max(len(tb) for _, _, tb in st.prefilled)
            ptab = np.zeros((len(n_pre), maxb), np.int32)
            for i, (_, _, tb) in enumerate(st.prefilled):
                ptab[i, :len(tb)] = tb
            plens = np.array(n_pre, np.int32)
            pqs = np.concatenate([[0], np.cumsum(n_pre)]).astype(np.int32)
            pq = bf(rng.standard_normal((int(pqs[-1]), Hq, D)).astype(np.float32))
            pout = torch.empty(pq.shape, dtype=torch.bfloat16, device="cuda")
            b.paged_prefill_attention(pout, pq.cuda(), dk, dv, cuda(ptab), cuda(plens), cuda(pqs), scale,
                                      max_query_len=int(plens.max()), max_context_len=int(plens.max()))
            torch.cuda.synchronize()
            pref = oracle.paged_prefill_attention(_np(pq), sk, sv, ptab, plens, pqs, scale, Hkv)
            H.assert_close(pout, pref, "bf16", f"engine step {steps} prefill")
            prefills_seen += 1
        if len(st.swap_out_pairs):
            b.swap_blocks(hk, hv, dk, dv, cuda(st.swap_out_pairs), host_pairs=st.swap_out_pairs)
            for d, h in st.swap_out_pairs:
                shk[h], shv[h] = sk[d], sv[d]
        if len(st.cow_pairs):
            b.copy_blocks(dk, dv, cuda(st.cow_pairs), host_pairs=st.cow_pairs)
            oracle.copy_blocks(sk, sv, st.cow_pairs)
        kvs = np.stack([kv_of(sid, int(st.context_lens[i]) - 1) for i, sid in enumerate(st.seq_ids)])
        kb, vb = bf(kvs[:, 0]), bf(kvs[:, 1])
        b.kv_append(kb.cuda(), vb.cuda(), cuda(st.slot_mapping), dk, dv)
        oracle.kv_append(_np(kb), _np(vb), st.slot_mapping, sk, sv)
        q = bf(rng.standard_normal((len(st.seq_ids), Hq, D)).astype(np.float32))
        out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
        b.paged_decode_attention(out, q.cuda(), dk, dv, cuda(st.block_tables), cuda(st.context_lens), scale,
                                 max_context_len=int(st.context_lens.max()))
        torch.cuda.synchronize()
        ref = oracle.paged_decode_attention(_np(q), sk, sv, st.block_tables, st.context_lens, scale, Hkv)
        H.assert_close(out, ref, "bf16", f"engine step {steps}")
        assert np.array_equal(_np(hk).view(np.uint8), shk.view(np.uint8))
        sched.retire(st)
        steps += 1
    assert sched.preemptions > 0 and sched.swaps > 0 and swaps_seen > 0 and prefills_seen > 0
