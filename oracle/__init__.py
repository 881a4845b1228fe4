"""Plain CPU oracle for PagedAttention decode, KV append and block copy.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and ``--impl reference`` arm) may import
this package.  The product path -- the CUDA library ``libpagedkv.so`` and its
Python binding -- never imports, links or calls anything here, and nothing
here imports the product path.  The two share only the seeded input
generators, which hold none of the method's arithmetic.

Sources followed (pages on PagedAttention and continuous batching):

* "PagedAttention: gestionar la KV cache como memoria de un sistema operativo"
  (josueisai.com), section "Cómo funciona por dentro": append writes into the
  last block of the table, asking for a new block only when it is full;
  attention walks the table in logical order and takes a softmax-weighted sum.
* "Batching Continuo y PagedAttention" (cruxr.ai), section "PagedAttention:
  Memoria virtual para la KV cache": fixed blocks of P = 16 tokens, logical
  block i holds tokens 16i..16i+15.
* iplexlaw.co.kr "pagedattention-vllm-kv-cache", section "Dos respuestas a
  una entrada: ejemplo hipotético": a shared, partly filled block is copied
  when written while other references exist.

``paged_decode_attention`` runs the fp64 C implementation in
``pkv_oracle.c`` (textbook softmax over the gathered, contiguous K/V).
``kv_append`` and ``copy_blocks`` are element copies written with numpy
indexing: the definition of those operations is a copy.

Every function here is pinned by ``tests/test_oracle.py`` against closed
forms, brute force on dense tensors, invariances, and the pages' worked
numbers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

BLOCK_SIZE = 16  # tokens per block ("típicamente P = 16")

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile ``pkv_oracle.c`` into ``libpkv_oracle.so`` beside it (gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            fn = lib.oracle_paged_decode_attention
            fn.restype = ctypes.c_int
            fn.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_double] + [ctypes.c_int] * 6 + \
                [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
            pf = lib.oracle_paged_prefill_attention
            pf.restype = ctypes.c_int
            pf.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_double] + [ctypes.c_int] * 8
            _lib = lib
    return _lib


class use_library:
    """Context manager that points the wrappers at another build of
    ``pkv_oracle.c`` (the mutation tests load deliberately broken copies)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        lib = ctypes.CDLL(self.path)
        for name in ("oracle_paged_decode_attention", "oracle_paged_prefill_attention"):
            getattr(lib, name).restype = ctypes.c_int
            getattr(lib, name).argtypes = getattr(self._saved, name).argtypes
        _lib = lib
        return lib

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 arrays or uint16 bf16 bit patterns, got {a.dtype}")


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                           seq_ids=None, nthreads=None) -> np.ndarray:
    """fp64 paged decode attention.

    q: [S, Hq, d]; k_cache, v_cache: [NB, Hkv, 16, d]; both float32, or both
    uint16 arrays of bf16 bit patterns.  block_tables: int32 [S, maxB];
    context_lens: int32 [S].  Returns float64 [len(seq_ids) or S, Hq, d].
    A context length of 0 gives a zero row.  Raises on an out-of-range block
    id or a length beyond the table.
    """
    q = np.ascontiguousarray(q)
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    code = _dtype_code(q)
    if _dtype_code(k_cache) != code or _dtype_code(v_cache) != code:
        raise TypeError("q, k_cache and v_cache must share one dtype")
    S, Hq, d = q.shape
    NB, Hkv, P, d2 = k_cache.shape
    if P != BLOCK_SIZE or d2 != d or v_cache.shape != k_cache.shape or Hkv != num_kv_heads:
        raise ValueError("cache shape must be [NB, num_kv_heads, 16, head_dim]")
    if bt.ndim != 2 or bt.shape[0] != S or cl.shape != (S,):
        raise ValueError("block_tables must be [S, maxB] and context_lens [S]")
    if seq_ids is None:
        ids = None
        n_out = S
    else:
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        if ids.size and (ids.min() < 0 or ids.max() >= S):
            raise ValueError("seq_ids out of range")
        n_out = ids.size
    out = np.zeros((n_out, Hq, d), dtype=np.float64)
    lib = _load()
    rc = lib.oracle_paged_decode_attention(
        out.ctypes.data, q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
        bt.ctypes.data, cl.ctypes.data, float(scale), int(num_kv_heads), int(Hq), int(d),
        int(bt.shape[1]), int(NB), code, None if ids is None else ids.ctypes.data, int(n_out),
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_paged_decode_attention failed with code {rc}")
    return out


def paged_prefill_attention(q, k_cache, v_cache, block_tables, context_lens, query_start, scale, num_kv_heads,
                            nthreads=None) -> np.ndarray:
    """fp64 causal prefill attention.  q: [total queries, Hq, d] with the
    queries of sequence s in rows query_start[s] .. query_start[s+1]-1; they
    are the last n_s tokens of its context_lens[s] cached tokens and query i
    attends to positions 0 .. context_lens[s] - n_s + i.  Returns float64
    [total queries, Hq, d]."""
    q = np.ascontiguousarray(q)
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    code = _dtype_code(q)
    if _dtype_code(k_cache) != code or _dtype_code(v_cache) != code:
        raise TypeError("q, k_cache and v_cache must share one dtype")
    TQ, Hq, d = q.shape
    NB, Hkv, P, d2 = k_cache.shape
    S = cl.shape[0]
    if P != BLOCK_SIZE or d2 != d or Hkv != num_kv_heads or qs.shape != (S + 1,) or qs[-1] != TQ or qs[0] != 0:
        raise ValueError("bad prefill shapes")
    out = np.zeros((TQ, Hq, d), dtype=np.float64)
    rc = _load().oracle_paged_prefill_attention(
        out.ctypes.data, q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data, bt.ctypes.data, cl.ctypes.data,
        qs.ctypes.data, float(scale), int(num_kv_heads), int(Hq), int(d), int(bt.shape[1]), int(NB), code, int(S),
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_paged_prefill_attention failed with code {rc}")
    return out


def kv_append(k, v, slot_mapping, k_cache, v_cache) -> None:
    """In place: for token t with slot = slot_mapping[t] >= 0, write k[t] and
    v[t] (all kv heads) into cache[slot // 16, :, slot % 16, :].  Negative
    slots are skipped.  Follows the append of the block-table sketch: a token
    goes into the last block at its next free position."""
    slots = np.asarray(slot_mapping, dtype=np.int64)
    NB = k_cache.shape[0]
    for t, slot in enumerate(slots.tolist()):
        if slot < 0:
            continue
        if slot >= NB * BLOCK_SIZE:
            raise ValueError(f"slot {slot} beyond the pool")
        k_cache[slot // BLOCK_SIZE, :, slot % BLOCK_SIZE, :] = k[t]
        v_cache[slot // BLOCK_SIZE, :, slot % BLOCK_SIZE, :] = v[t]


def copy_blocks(k_cache, v_cache, src_dst_pairs) -> None:
    """In place: for each (src, dst) pair copy the whole physical block --
    every kv head, all 16 slots -- of both caches from src to dst (the
    copy-on-write of a shared block)."""
    pairs = np.asarray(src_dst_pairs, dtype=np.int64).reshape(-1, 2)
    NB = k_cache.shape[0]
    for src, dst in pairs.tolist():
        if not (0 <= src < NB and 0 <= dst < NB):
            raise ValueError(f"pair ({src}, {dst}) out of range")
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]
