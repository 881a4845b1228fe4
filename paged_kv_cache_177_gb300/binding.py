"""Python binding of ``libpagedkv.so`` (include/pagedkv.h) over ctypes.

Argument marshalling only: shape/dtype/device checks, device pointers from
torch tensors, the caller's current CUDA stream, and (when the caller passes
none) a workspace tensor from torch's allocator.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.  If the
library is missing the import fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

from .build import LIB

if not os.path.exists(LIB):
    raise ImportError(f"{LIB} is missing: build it with paged_kv_cache_177_gb300.build.build_library() "
                      "(or __graft_entry__.build()); there is no CPU fallback")

_lib = ctypes.CDLL(LIB)

PKV_F32, PKV_BF16, PKV_BF16_OUT_F32 = 0, 1, 2
PARTITION_AUTO, PARTITION_BALANCED = 0, -1
DEVERR_BLOCK_ID, DEVERR_SLOT, DEVERR_PAIR, DEVERR_TIMEOUT, DEVERR_LENGTH = 0x1, 0x2, 0x4, 0x8, 0x10
DEVERR_POINTER = 0x20
BLOCK_SIZE = 16
# the arrival counters at the head of every decode workspace (PKV_DECODE_COUNTER_BYTES)
DECODE_COUNTER_BYTES = 10240

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


def _decl(name, restype, *argtypes):
    fn = getattr(_lib, name)
    fn.restype = restype
    fn.argtypes = list(argtypes)
    return fn


_status_string = _decl("pkv_status_string", ctypes.c_char_p, _i)
_version = _decl("pkv_version", _i)
_partition_tokens = _decl("pkv_decode_partition_tokens", _i, _i, _i, _i, _i)
_workspace_bytes = _decl("pkv_decode_workspace_bytes", _sz, _i, _i, _i, _i, _i, _i)
_decode_launches = _decl("pkv_decode_launches", _i, _i, _i, _i, _i, _i)
_decode_persistent = _decl("pkv_decode_persistent", _i, _i, _i, _i, _i)
_decode = _decl("paged_decode_attention", _i, _vp, _vp, _vp, _vp, _vp, _vp, _f, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                _vp, _sz, _vp)
_shared = _decl("paged_decode_attention_shared_prefix", _i, _vp, _vp, _vp, _vp, _vp, _vp, _f, _i, _i, _i, _i, _i,
                _i, _i, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _vp)
_prefill = _decl("paged_prefill_attention", _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f, _i, _i, _i, _i, _i, _i, _i,
                 _i, _i, _i, _vp)
_step = _decl("paged_decode_step", _i, _vp, _vp, _vp, _vp, _vp, _vp, _f, _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp,
               _sz, _vp, _vp, _vp, _i, _vp, _i, _vp)
_shared_ws = _decl("pkv_shared_prefix_workspace_bytes", _sz, _i, _i, _i, _i, _i, _i)
_append = _decl("kv_append", _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp)
_copy = _decl("copy_blocks", _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp)
_swap = _decl("swap_blocks", _i, _vp, _vp, _i, _vp, _vp, _i, _vp, _i, _i, _i, _i, _vp)
_check_swap = _decl("pkv_check_swap_pairs", _i, _vp, _i, _i, _i)
_copy_layers = _decl("copy_blocks_layers", _i, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _vp)
_append_layers = _decl("kv_append_layers", _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp)
_check_pairs = _decl("pkv_check_copy_pairs", _i, _vp, _i, _i)
_validate = _decl("pkv_validate", _i, _vp, _vp, _i, _i, _i, _i, _vp, _vp)
_validate_slots = _decl("pkv_validate_slots", _i, _vp, _i, _i, _vp, _vp)
_device_error = _decl("pkv_device_error", _i, ctypes.POINTER(ctypes.c_uint32), _i)


class PagedKVError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise PagedKVError(rc, what)


def status_string(code: int) -> str:
    return _status_string(int(code)).decode()


def version() -> int:
    return int(_version())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    if t.dtype == torch.float32:
        return PKV_F32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32")


def _dev(*ts: torch.Tensor) -> torch.device:
    d = ts[0].device
    if d.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    for t in ts:
        if t.device != d:
            raise ValueError("all tensors must be on the same device")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    return d


def _dev_io(device_tensors, io_tensors) -> torch.device:
    """Device of the calls whose per-step arguments may also sit in pinned
    host memory: ``device_tensors`` (the caches, the workspace) must be on one
    CUDA device; each of ``io_tensors`` on that device or pinned on the host,
    where the kernels read or write it in place over the host link."""
    d = _dev(*device_tensors)
    for t in io_tensors:
        if t is None or t.numel() == 0:      # nothing the kernels would touch
            continue
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
        if t.device != d and not (t.device.type == "cpu" and t.is_pinned()):
            raise ValueError("per-step arguments must be on the caches' device or in pinned host memory")
    return d


def _stream_ptr(device: torch.device, stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _p(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def partition_tokens(num_seqs: int, num_kv_heads: int, max_context_len: int, requested: int = 0) -> int:
    return int(_partition_tokens(num_seqs, num_kv_heads, max_context_len, requested))


def workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_context_len: int,
                    partition_tokens: int = 0) -> int:
    return int(_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len, partition_tokens))


def decode_launches(num_seqs: int, num_kv_heads: int, max_context_len: int, partition_tokens: int = 0,
                    dtype: torch.dtype = torch.bfloat16) -> int:
    """Kernel launches of one decode call: 1 (persistent balanced kernel, or
    no split), 2 (partition kernel + reduce), 0 (empty batch)."""
    code = PKV_BF16 if dtype == torch.bfloat16 else PKV_F32
    return int(_decode_launches(num_seqs, num_kv_heads, max_context_len, partition_tokens, code))


def decode_persistent(num_seqs: int, num_kv_heads: int, partition_tokens: int = 0,
                      dtype: torch.dtype = torch.bfloat16) -> bool:
    """Whether a decode call with these arguments runs the persistent
    balanced kernel."""
    code = PKV_BF16 if dtype == torch.bfloat16 else PKV_F32
    return bool(_decode_persistent(num_seqs, num_kv_heads, partition_tokens, code))


def decode_args(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                num_kv_heads: Optional[int] = None, *, max_context_len: Optional[int] = None,
                partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> tuple:
    """Checks and marshals the arguments of one paged_decode_attention call
    (see there) into the C-ABI argument tuple, for ``decode_raw``."""
    dev = _dev_io([k_cache, v_cache], [out, q, block_tables, context_lens])
    dt = _dtype_code(q)
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q and the caches must share one dtype")
    if out.dtype != q.dtype:
        if not (q.dtype == torch.bfloat16 and out.dtype == torch.float32):
            raise TypeError("out must have q's dtype, or be fp32 with bf16 q (the unrounded accumulator)")
        dt = PKV_BF16_OUT_F32
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    S, Hq, D = q.shape
    NB, Hkv, P, D2 = k_cache.shape
    if P != BLOCK_SIZE or D2 != D or v_cache.shape != k_cache.shape or out.shape != q.shape:
        raise ValueError("expected q/out [S, Hq, D] and caches [NB, Hkv, 16, D]")
    if num_kv_heads is not None and num_kv_heads != Hkv:
        raise ValueError("num_kv_heads does not match the cache")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("expected block_tables [S, maxB] and context_lens [S]")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    need = workspace_bytes(S, Hq, Hkv, D, max_context_len, partition_tokens)
    if need and workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)   # must start zero-filled
    if workspace is not None and _dev(workspace) != dev:
        raise ValueError("the workspace must be on the caches' device")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    # the tensors ride along so they outlive the raw pointers
    return ((_p(out), _p(q), _p(k_cache), _p(v_cache), _p(block_tables), _p(context_lens), float(scale), Hkv, S, Hq,
             D, block_tables.shape[1], NB, int(max_context_len), dt, int(partition_tokens), _p(workspace), ws_bytes,
             _stream_ptr(dev, stream)), (out, q, k_cache, v_cache, block_tables, context_lens, workspace))


def decode_raw(args: tuple) -> None:
    """Calls paged_decode_attention with arguments prepared by ``decode_args``."""
    _check(_decode(*args[0]), "paged_decode_attention")


def paged_decode_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           num_kv_heads: Optional[int] = None, *, max_context_len: Optional[int] = None,
                           partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """out[s, hq] = softmax(scale * K_s q[s, hq]) V_s over context_lens[s] tokens
    read through block_tables[s]; see include/pagedkv.h.

    q, out: [S, Hq, D]; k_cache, v_cache: [NB, Hkv, 16, D] (bf16 or fp32,
    all one dtype); block_tables int32 [S, maxB]; context_lens int32 [S].
    With bf16 q and caches, ``out`` may be fp32: it then receives the
    accumulated O / L before rounding to bf16 (PKV_BF16_OUT_F32), the same
    arithmetic otherwise.
    ``max_context_len`` defaults to context_lens.max() (a device sync).
    ``partition_tokens``: 0 automatic, -1 balanced (persistent kernel, bf16),
    > 0 fixed partitions of that many tokens.
    A caller-provided ``workspace`` must have been zero-filled once before
    its first use; its counter header (the first DECODE_COUNTER_BYTES) is
    left zero after each call and no decode path writes anything else there,
    so one workspace sized for the largest call serves every call and path
    without clearing.
    q, out, block_tables and context_lens may be pinned host tensors: the
    kernels then read and write them in place (no separate copy).
    """
    decode_raw(decode_args(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                           max_context_len=max_context_len, partition_tokens=partition_tokens, workspace=workspace,
                           stream=stream))
    return out


def paged_decode_step(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, k_new: torch.Tensor,
                      v_new: torch.Tensor, slot_mapping: torch.Tensor, src_dst_pairs: Optional[torch.Tensor] = None,
                      *, host_pairs=None, check: bool = True, max_context_len: Optional[int] = None,
                      partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """One decode step in one call: ``copy_blocks(src_dst_pairs)``, then
    ``kv_append(k_new, v_new, slot_mapping)``, then ``paged_decode_attention``
    (arguments as for those calls); the attention's set-up overlaps the
    append (see include/pagedkv.h)."""
    args, keep = decode_args(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                             max_context_len=max_context_len, partition_tokens=partition_tokens, workspace=workspace,
                             stream=stream)
    _dev_io([k_cache, v_cache], [k_new, v_new, slot_mapping, src_dst_pairs])
    if not (k_new.dtype == v_new.dtype == k_cache.dtype) or slot_mapping.dtype != torch.int64:
        raise TypeError("k_new, v_new in the cache dtype and slot_mapping int64")
    T = k_new.shape[0]
    NB, Hkv, P, D = k_cache.shape
    if k_new.shape != (T, Hkv, D) or v_new.shape != k_new.shape or slot_mapping.shape != (T,):
        raise ValueError("expected k_new, v_new [T, Hkv, D] and slot_mapping [T]")
    n = 0
    if src_dst_pairs is not None:
        if src_dst_pairs.dtype != torch.int64 or src_dst_pairs.numel() % 2:
            raise TypeError("src_dst_pairs must be int64 [n, 2]")
        n = src_dst_pairs.numel() // 2
        if check and n:
            check_copy_pairs(host_pairs if host_pairs is not None else src_dst_pairs.cpu().numpy(), NB)
    _check(_step(*args[:-1], _p(k_new), _p(v_new), _p(slot_mapping), T, _p(src_dst_pairs) if n else None, n,
                 args[-1]), "paged_decode_step")
    del keep
    return out


def shared_prefix_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int, max_context_len: int,
                                  group_size: int, partition_tokens: int = 0) -> int:
    return int(_shared_ws(num_seqs, num_q_heads, head_dim, max_context_len, group_size, partition_tokens))


def prefix_groups(num_seqs: int, groups, shared_blocks):
    """Completes a partial grouping into the partition the shared-prefix call
    takes: ``groups`` lists the sharing groups (sequence ids per group), every
    sequence not in one becomes a group of one with no shared blocks.
    Returns (group_members int32 [G, M] with -1 padding, shared_blocks int32 [G])."""
    groups = [list(map(int, g)) for g in groups]
    seen = {s for g in groups for s in g}
    if len(seen) != sum(len(g) for g in groups):
        raise ValueError("a sequence is in two groups")
    groups += [[s] for s in range(num_seqs) if s not in seen]
    shared = list(map(int, shared_blocks)) + [0] * (len(groups) - len(shared_blocks))
    width = max([len(g) for g in groups] + [1])
    members = np.full((len(groups), width), -1, dtype=np.int32)
    for i, g in enumerate(groups):
        members[i, :len(g)] = g
    return members, np.array(shared, dtype=np.int32)


def paged_decode_attention_shared_prefix(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                         v_cache: torch.Tensor, block_tables: torch.Tensor,
                                         context_lens: torch.Tensor, scale: float, group_members: torch.Tensor,
                                         shared_blocks: torch.Tensor, *, max_context_len: Optional[int] = None,
                                         partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                                         stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """paged_decode_attention with the leading blocks shared by each group of
    sequences read once per group.  group_members: int32 [G, M] sequence ids
    (-1 = empty slot), listing every sequence exactly once (see
    ``prefix_groups``); shared_blocks: int32 [G] blocks the members share."""
    dev = _dev(out, q, k_cache, v_cache, block_tables, context_lens, group_members, shared_blocks)
    if q.dtype != torch.bfloat16 or not (out.dtype == k_cache.dtype == v_cache.dtype == q.dtype):
        raise TypeError("shared-prefix decode is bf16")
    if group_members.dtype != torch.int32 or shared_blocks.dtype != torch.int32 or group_members.dim() != 2:
        raise TypeError("group_members int32 [G, M] and shared_blocks int32 [G]")
    G, M = group_members.shape
    if shared_blocks.shape != (G,):
        raise ValueError("shared_blocks must be [G]")
    S, Hq, D = q.shape
    NB, Hkv, P, _ = k_cache.shape
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    need = shared_prefix_workspace_bytes(S, Hq, D, max_context_len, max(M, 1), partition_tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_shared(_p(out), _p(q), _p(k_cache), _p(v_cache), _p(block_tables), _p(context_lens), float(scale), Hkv, S,
                   Hq, D, block_tables.shape[1], NB, int(max_context_len), _p(group_members) if G else None,
                   _p(shared_blocks) if G else None, G, max(M, 1), PKV_BF16, int(partition_tokens), _p(workspace),
                   ws_bytes, _stream_ptr(dev, stream)), "paged_decode_attention_shared_prefix")
    return out


def paged_prefill_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor, query_start: torch.Tensor,
                            scale: float, *, max_query_len: Optional[int] = None,
                            max_context_len: Optional[int] = None,
                            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Causal attention of each sequence's last n_s context tokens (a prompt
    or a chunk of one, already appended to the cache); see include/pagedkv.h.

    q, out: bf16 [T, Hq, D], sequence s owning rows query_start[s] ..
    query_start[s+1]-1; query_start int32 [S + 1]; caches, tables and lengths
    as for ``paged_decode_attention``.  ``max_query_len`` and
    ``max_context_len`` default to the maxima of the device arrays (a sync).
    """
    dev = _dev(out, q, k_cache, v_cache, block_tables, context_lens, query_start)
    if q.dtype != torch.bfloat16 or not (out.dtype == k_cache.dtype == v_cache.dtype == q.dtype):
        raise TypeError("prefill attention is bf16")
    if query_start.dtype != torch.int32 or context_lens.dtype != torch.int32 or block_tables.dtype != torch.int32:
        raise TypeError("query_start, context_lens and block_tables are int32")
    if q.dim() != 3 or out.shape != q.shape or not (q.is_contiguous() and out.is_contiguous()):
        raise ValueError("q and out must be contiguous [T, Hq, D]")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous() and block_tables.is_contiguous()):
        raise ValueError("caches and block tables must be contiguous")
    S = context_lens.shape[0]
    if query_start.shape != (S + 1,):
        raise ValueError("query_start must be [S + 1]")
    _, Hq, D = q.shape
    NB, Hkv, P, _ = k_cache.shape
    if P != BLOCK_SIZE or k_cache.shape[3] != D or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [NB, Hkv, 16, D] with q's head_dim")
    if max_query_len is None:
        max_query_len = int((query_start[1:] - query_start[:-1]).max().item()) if S else 0
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if S else 0
    _check(_prefill(_p(out), _p(q), _p(k_cache), _p(v_cache), _p(block_tables), _p(context_lens), _p(query_start),
                    float(scale), Hkv, S, Hq, D, block_tables.shape[1] if S else 1, NB, q.shape[0],
                    int(max_query_len), int(max_context_len), PKV_BF16, _stream_ptr(dev, stream)),
           "paged_prefill_attention")
    return out


def kv_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, *, stream: Optional[torch.cuda.Stream] = None) -> None:
    """cache[slot // 16, :, slot % 16, :] = k[t] (and v) for each slot >= 0.
    k, v and slot_mapping may be pinned host tensors (read in place)."""
    dev = _dev_io([k_cache, v_cache], [k, v, slot_mapping])
    dt = _dtype_code(k)
    if not (k.dtype == v.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("k, v and the caches must share one dtype")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    T, Hkv, D = k.shape
    NB, Hkv2, P, D2 = k_cache.shape
    if v.shape != k.shape or Hkv2 != Hkv or D2 != D or P != BLOCK_SIZE or slot_mapping.shape != (T,) \
            or v_cache.shape != k_cache.shape:
        raise ValueError("expected k, v [T, Hkv, D], slot_mapping [T], caches [NB, Hkv, 16, D]")
    _check(_append(_p(k), _p(v), _p(slot_mapping), _p(k_cache), _p(v_cache), T, Hkv, D, NB, dt,
                   _stream_ptr(dev, stream)), "kv_append")


def check_copy_pairs(pairs, num_blocks: int) -> None:
    """Host-side range/overlap check of (src, dst) pairs; raises PagedKVError."""
    arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    _check(_check_pairs(arr.ctypes.data if arr.size else None, arr.shape[0], int(num_blocks)), "copy_blocks pairs")


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs: torch.Tensor, *,
                host_pairs=None, check: bool = True, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copies whole blocks src -> dst of both caches.  ``src_dst_pairs``:
    int64 [n, 2] on the device.  With ``check`` the pairs are range- and
    overlap-checked on the host first (``host_pairs`` if given, else a copy
    of the device pairs, which synchronises).  The pairs may also be a
    pinned host tensor (read in place)."""
    dev = _dev_io([k_cache, v_cache], [src_dst_pairs])
    dt = _dtype_code(k_cache)
    if src_dst_pairs.dtype != torch.int64:
        raise TypeError("src_dst_pairs must be int64")
    n = src_dst_pairs.numel() // 2
    if src_dst_pairs.numel() != 2 * n:
        raise ValueError("src_dst_pairs must be [n, 2]")
    NB, Hkv, P, D = k_cache.shape
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype or P != BLOCK_SIZE:
        raise ValueError("caches must be [NB, Hkv, 16, D] of one dtype")
    if check:
        check_copy_pairs(host_pairs if host_pairs is not None else src_dst_pairs.cpu().numpy(), NB)
    _check(_copy(_p(k_cache), _p(v_cache), _p(src_dst_pairs) if n else None, n, Hkv, D, NB, dt,
                 _stream_ptr(dev, stream)), "copy_blocks")


def _pool_ok(t: torch.Tensor) -> None:
    if not t.is_contiguous():
        raise ValueError("pools must be contiguous")
    if t.device.type != "cuda" and not t.is_pinned():
        raise ValueError("a pool must be a CUDA tensor or pinned host memory")


def check_swap_pairs(pairs, src_num_blocks: int, dst_num_blocks: int) -> None:
    """Host-side range check of (src, dst) swap pairs and distinct destinations."""
    arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    _check(_check_swap(arr.ctypes.data if arr.size else None, arr.shape[0], int(src_num_blocks), int(dst_num_blocks)),
           "swap_blocks pairs")


def swap_blocks(dst_k: torch.Tensor, dst_v: torch.Tensor, src_k: torch.Tensor, src_v: torch.Tensor,
                src_dst_pairs: torch.Tensor, *, host_pairs=None, check: bool = True,
                stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copies block src of the source pool onto block dst of the destination
    pool (both caches) for each pair.  A pool is a CUDA tensor or a pinned
    host tensor [NB, Hkv, 16, D]; swap-out goes device -> host, swap-in host ->
    device.  ``src_dst_pairs``: int64 [n, 2], on the device or pinned."""
    for t in (dst_k, dst_v, src_k, src_v, src_dst_pairs):
        _pool_ok(t)
    if src_dst_pairs.dtype != torch.int64:
        raise TypeError("src_dst_pairs must be int64")
    if not (dst_k.dtype == dst_v.dtype == src_k.dtype == src_v.dtype):
        raise TypeError("pools must share one dtype")
    dt = _dtype_code(dst_k)
    NBd, Hkv, P, D = dst_k.shape
    NBs = src_k.shape[0]
    if dst_v.shape != dst_k.shape or src_v.shape != src_k.shape or src_k.shape[1:] != dst_k.shape[1:] or P != BLOCK_SIZE:
        raise ValueError("pools must be [NB, Hkv, 16, D] with matching block shapes")
    n = src_dst_pairs.numel() // 2
    if check:
        check_swap_pairs(host_pairs if host_pairs is not None else src_dst_pairs.cpu().numpy(), NBs, NBd)
    dev = next((t.device for t in (dst_k, src_k, src_dst_pairs) if t.device.type == "cuda"), None)
    if dev is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    _check(_swap(_p(dst_k), _p(dst_v), NBd, _p(src_k), _p(src_v), NBs, _p(src_dst_pairs) if n else None, n, Hkv, D,
                 dt, _stream_ptr(dev, stream)), "swap_blocks")


def _ptr_array(ts, dev) -> torch.Tensor:
    return torch.tensor([t.data_ptr() for t in ts], dtype=torch.int64, device=dev)


def layer_pointers(tensors, device=None) -> torch.Tensor:
    """A device array of the tensors' data pointers, for the per-layer calls.
    Build it once and pass it back through ``ptrs=`` to keep the calls free of
    host-to-device copies (for example inside CUDA graph capture); the tensors
    must stay alive and in place while the array is used."""
    dev = device if device is not None else tensors[0].device
    return _ptr_array(tensors, dev)


def copy_blocks_layers(k_caches, v_caches, src_dst_pairs: torch.Tensor, *, host_pairs=None, check: bool = True,
                       stream: Optional[torch.cuda.Stream] = None, ptrs=None) -> None:
    """copy_blocks over every layer's caches (lists of [NB, Hkv, 16, D] CUDA
    tensors, one per layer) in one launch.  ``ptrs``: optional prebuilt
    (k_caches, v_caches) pointer arrays from ``layer_pointers``."""
    if len(k_caches) != len(v_caches):
        raise ValueError("one K and one V cache per layer")
    if not k_caches:
        return
    dev = _dev(*k_caches, *v_caches, src_dst_pairs)
    dt = _dtype_code(k_caches[0])
    shape = k_caches[0].shape
    for t in (*k_caches, *v_caches):
        if t.shape != shape or t.dtype != k_caches[0].dtype:
            raise ValueError("every layer's caches must share shape and dtype")
    NB, Hkv, P, D = shape
    n = src_dst_pairs.numel() // 2
    if check:
        check_copy_pairs(host_pairs if host_pairs is not None else src_dst_pairs.cpu().numpy(), NB)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.stream(st):  # the pointer arrays are copied in on the launch stream
        kp, vp = ptrs if ptrs is not None else (_ptr_array(k_caches, dev), _ptr_array(v_caches, dev))
        _check(_copy_layers(_p(kp), _p(vp), len(k_caches), _p(src_dst_pairs) if n else None, n, Hkv, D, NB, dt,
                            st.cuda_stream), "copy_blocks_layers")


def kv_append_layers(ks, vs, slot_mapping: torch.Tensor, k_caches, v_caches, *,
                     stream: Optional[torch.cuda.Stream] = None, ptrs=None) -> None:
    """kv_append for every layer in one launch: layer l writes ks[l], vs[l]
    ([T, Hkv, D]) into k_caches[l], v_caches[l] at the same slots.  ``ptrs``:
    optional prebuilt (ks, vs, k_caches, v_caches) pointer arrays."""
    L = len(k_caches)
    if not (len(ks) == len(vs) == L == len(v_caches)):
        raise ValueError("one k, v, K cache and V cache per layer")
    if L == 0:
        return
    dev = _dev(*ks, *vs, *k_caches, *v_caches, slot_mapping)
    dt = _dtype_code(k_caches[0])
    T, Hkv, D = ks[0].shape
    NB = k_caches[0].shape[0]
    for t in (*ks, *vs):
        if t.shape != (T, Hkv, D) or t.dtype != k_caches[0].dtype:
            raise ValueError("every layer's k and v must be [T, Hkv, D] of the cache dtype")
    for t in (*k_caches, *v_caches):
        if t.shape != (NB, Hkv, BLOCK_SIZE, D) or t.dtype != k_caches[0].dtype:
            raise ValueError("every layer's caches must be [NB, Hkv, 16, D]")
    if slot_mapping.dtype != torch.int64 or slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be int64 [T]")
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.stream(st):  # the pointer arrays are copied in on the launch stream
        arrs = list(ptrs) if ptrs is not None else [_ptr_array(x, dev) for x in (ks, vs, k_caches, v_caches)]
        _check(_append_layers(*(_p(a) for a in arrs[:2]), _p(slot_mapping), *(_p(a) for a in arrs[2:]), L, T, Hkv, D,
                              NB, dt, st.cuda_stream), "kv_append_layers")


def validate(block_tables: torch.Tensor, context_lens: torch.Tensor, num_blocks: int, max_context_len: int,
             err_word: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Device-side range check of decode metadata; returns the int32 error word tensor."""
    dev = _dev(block_tables, context_lens)
    if err_word is None:
        err_word = torch.empty(1, dtype=torch.int32, device=dev)
    S = context_lens.shape[0]
    _check(_validate(_p(block_tables), _p(context_lens), S, block_tables.shape[1], int(num_blocks),
                     int(max_context_len), _p(err_word), _stream_ptr(dev, stream)), "pkv_validate")
    return err_word


def validate_slots(slot_mapping: torch.Tensor, num_blocks: int, err_word: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    dev = _dev(slot_mapping)
    if err_word is None:
        err_word = torch.empty(1, dtype=torch.int32, device=dev)
    _check(_validate_slots(_p(slot_mapping), slot_mapping.numel(), int(num_blocks), _p(err_word),
                           _stream_ptr(dev, stream)), "pkv_validate_slots")
    return err_word


def device_error(clear: bool = True) -> int:
    """The library's device error word on the current device (synchronous)."""
    v = ctypes.c_uint32(0)
    _check(_device_error(ctypes.byref(v), 1 if clear else 0), "pkv_device_error")
    return int(v.value)


def raw_library() -> ctypes.CDLL:
    """The loaded ctypes library (for callers that pass raw pointers)."""
    return _lib
