"""The C-ABI library loads, exports every function include/pagedkv.h
declares, and rejects bad scalar arguments on the host -- all without a GPU
(no call here reaches a kernel)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from paged_kv_cache_177_gb300.build import INCLUDE, build_library

HEADER = os.path.join(INCLUDE, "pagedkv.h")


@pytest.fixture(scope="module")
def lib():
    path = build_library()
    return ctypes.CDLL(path)


@pytest.fixture(scope="module")
def binding(lib):
    from paged_kv_cache_177_gb300 import binding as b
    return b


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_three_calls_and_helpers():
    names = declared_functions()
    for required in ("paged_decode_attention", "kv_append", "copy_blocks", "pkv_status_string",
                     "pkv_decode_workspace_bytes", "pkv_validate", "pkv_check_copy_pairs"):
        assert required in names
    assert len(names) >= 11


def test_library_exports_every_declared_function(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_status_strings(binding):
    assert binding.status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5, -6, -7):
        assert binding.status_string(code) not in ("ok", "unknown status")
    assert binding.status_string(-99) == "unknown status"
    assert binding.version() >= 100


def test_partition_and_workspace_sizing(binding):
    assert binding.partition_tokens(8, 8, 131072, 0) % 16 == 0
    assert binding.partition_tokens(8, 8, 131072, 512) == 512
    # a context no longer than one partition needs no workspace
    assert binding.workspace_bytes(64, 40, 40, 128, 512, 512) == 0
    # otherwise: the counter header, then S * Hq * ceil(L / P) * (2 + D) floats
    hdr = binding.DECODE_COUNTER_BYTES
    assert binding.workspace_bytes(8, 64, 8, 128, 131072, 512) == hdr + 8 * 64 * 256 * 130 * 4
    assert binding.workspace_bytes(2, 4, 4, 64, 1000, 64) == hdr + 2 * 4 * 16 * 66 * 4
    # the persistent layout does not depend on the batch size: one state per
    # group head for two segments of each of up to 160 x 12 workers
    for S in (1, 64, 8192):
        assert binding.workspace_bytes(S, 32, 8, 128, 64, -1) == hdr + 160 * 12 * 2 * 4 * 130 * 4


def test_counter_header_size_matches_the_header():
    from paged_kv_cache_177_gb300 import binding as b
    m = re.search(r"#define\s+PKV_DECODE_COUNTER_BYTES\s+(\d+)u?", open(HEADER).read())
    assert m and int(m.group(1)) == b.DECODE_COUNTER_BYTES
    assert b.DECODE_COUNTER_BYTES % 256 == 0 and b.DECODE_COUNTER_BYTES >= 160 * 12 * 4


def test_which_decode_kernel_runs(binding):
    """The planning queries agree on the path: the balanced split always
    runs the persistent kernel (one launch), fixed partitions and fp32 never
    do; bad arguments give 0. (Without a GPU the SM count defaults to the
    largest the workspace is sized for.)"""
    bf16, f32 = torch.bfloat16, torch.float32
    assert binding.decode_persistent(64, 40, -1, bf16)
    assert binding.decode_launches(64, 40, 4096, -1, bf16) == 1
    assert not binding.decode_persistent(64, 40, 512, bf16)
    assert binding.decode_launches(64, 40, 4096, 512, bf16) == 2
    assert not binding.decode_persistent(64, 40, -1, f32)
    assert not binding.decode_persistent(0, 40, -1, bf16) and not binding.decode_persistent(64, 40, -2, bf16)
    # automatic: a quarter as many units as persistent warps or more
    assert binding.decode_persistent(8192, 8, 0, bf16)
    assert not binding.decode_persistent(8, 8, 0, bf16)


def _decode(lib, **kw):
    args = dict(out=1 << 12, q=1 << 12, k=1 << 12, v=1 << 12, bt=1 << 12, cl=1 << 12, scale=0.1, hkv=8, S=4, hq=8,
                d=64, maxb=4, nb=32, maxlen=64, dtype=0, pt=0, ws=None, wsb=0, stream=None)
    args.update(kw)
    f = lib.paged_decode_attention
    f.restype = ctypes.c_int
    vp = ctypes.c_void_p
    f.argtypes = [vp] * 6 + [ctypes.c_float] + [ctypes.c_int] * 9 + [vp, ctypes.c_size_t, vp]
    return f(args["out"], args["q"], args["k"], args["v"], args["bt"], args["cl"], args["scale"], args["hkv"],
             args["S"], args["hq"], args["d"], args["maxb"], args["nb"], args["maxlen"], args["dtype"], args["pt"],
             args["ws"], args["wsb"], args["stream"])


def test_decode_rejects_bad_arguments_before_any_cuda_call(lib):
    assert _decode(lib, d=96) == -2                  # unsupported head_dim
    assert _decode(lib, dtype=7) == -2               # unsupported dtype
    assert _decode(lib, hq=12, hkv=8) == -1          # heads not a multiple
    assert _decode(lib, hq=8 * 17, hkv=8) == -2      # group of 17 > 16
    assert _decode(lib, hkv=0) == -1
    assert _decode(lib, S=-1) == -1
    assert _decode(lib, pt=-2) == -1                 # below PKV_PARTITION_BALANCED
    assert _decode(lib, out=None) == -1              # null pointer
    assert _decode(lib, q=(1 << 12) + 4) == -7       # misaligned
    assert _decode(lib, pt=24) == -1                 # partition not a multiple of 16
    assert _decode(lib, maxlen=4096, pt=64) == -6    # split needed, no workspace
    assert _decode(lib, scale=float("nan")) == -1
    assert _decode(lib, S=0) == 0                    # empty batch: nothing to do
    # bf16 inputs with fp32 output: the same checks apply
    assert _decode(lib, dtype=2, d=96) == -2
    assert _decode(lib, dtype=2, maxlen=4096, pt=64) == -6
    assert _decode(lib, dtype=2, S=0) == 0
    assert _decode(lib, dtype=3) == -2


def test_fp32_output_mode_plans_like_bf16(lib):
    for fn, args in (("pkv_decode_persistent", (64, 40, -1)), ("pkv_decode_launches", (64, 40, 4096, -1))):
        f = getattr(lib, fn)
        f.restype = ctypes.c_int
        assert f(*args, 2) == f(*args, 1) != f(*args, 0)


def _prefill(lib, **kw):
    args = dict(out=1 << 12, q=1 << 12, k=1 << 12, v=1 << 12, bt=1 << 12, cl=1 << 12, qs=1 << 12, scale=0.1, hkv=8,
                S=4, hq=8, d=64, maxb=4, nb=32, T=40, maxq=16, maxlen=64, dtype=1, stream=None)
    args.update(kw)
    f = lib.paged_prefill_attention
    f.restype = ctypes.c_int
    vp = ctypes.c_void_p
    f.argtypes = [vp] * 7 + [ctypes.c_float] + [ctypes.c_int] * 10 + [vp]
    return f(args["out"], args["q"], args["k"], args["v"], args["bt"], args["cl"], args["qs"], args["scale"],
             args["hkv"], args["S"], args["hq"], args["d"], args["maxb"], args["nb"], args["T"], args["maxq"],
             args["maxlen"], args["dtype"], args["stream"])


def test_prefill_rejects_bad_arguments_before_any_cuda_call(lib):
    assert _prefill(lib, dtype=0) == -2              # fp32 prefill is not provided
    assert _prefill(lib, dtype=2) == -2              # nor fp32 output
    assert _prefill(lib, d=96) == -2
    assert _prefill(lib, hq=12, hkv=8) == -1
    assert _prefill(lib, hq=8 * 65, hkv=8) == -2     # group of 65 > the largest supported (64)
    assert _prefill(lib, maxq=-1) == -1
    assert _prefill(lib, qs=None) == -1
    assert _prefill(lib, q=(1 << 12) + 2) == -7
    assert _prefill(lib, scale=float("inf")) == -1
    assert _prefill(lib, S=0) == 0
    assert _prefill(lib, maxq=0) == 0                # no new tokens: nothing to do
    assert _prefill(lib, T=-1) == -1
    # more than 65,535 pairs of query tiles (the grid's pair dimension): 64 heads in one group
    # make 2-token tiles, so 2**18 new tokens are 65,536 pairs
    assert _prefill(lib, hq=64, hkv=1, maxq=1 << 18, T=1 << 18) == -2


def test_decode_step_checks_everything_before_launching(lib):
    vp, ci = ctypes.c_void_p, ctypes.c_int
    f = lib.paged_decode_step
    f.restype = ci
    f.argtypes = [vp] * 6 + [ctypes.c_float] + [ci] * 9 + [vp, ctypes.c_size_t, vp, vp, vp, ci, vp, ci, vp]
    a = 1 << 12

    def call(d=64, T=4, dt=1, pairs=0, kn=a):
        return f(a, a, a, a, a, a, 0.1, 8, 4, 8, d, 4, 32, 64, dt, 0, a, 1 << 30, kn, a, a, T, a, pairs, None)
    assert call(d=96) == -2             # attention arguments
    assert call(T=-1) == -1             # append arguments
    assert call(kn=a + 8) == -7         # misaligned new keys
    assert call(dt=7) == -2


def test_append_and_copy_reject_bad_arguments(lib):
    vp, ci = ctypes.c_void_p, ctypes.c_int
    ap = lib.kv_append
    ap.restype = ci
    ap.argtypes = [vp] * 5 + [ci] * 5 + [vp]
    a = 1 << 12
    assert ap(a, a, a, a, a, 4, 8, 96, 32, 0, None) == -2
    assert ap(a, a, a, a, a, -1, 8, 64, 32, 0, None) == -1
    assert ap(a, a + 8, a, a, a, 4, 8, 64, 32, 0, None) == -7
    assert ap(a, a, a, a, a, 0, 8, 64, 32, 0, None) == 0
    cp = lib.copy_blocks
    cp.restype = ci
    cp.argtypes = [vp] * 3 + [ci] * 5 + [vp]
    assert cp(a, a, a, -1, 8, 64, 32, 0, None) == -1
    assert cp(a, a, a, 2, 8, 64, 32, 3, None) == -2
    assert cp(a, a, a, 0, 8, 64, 32, 0, None) == 0


def test_host_pair_check(binding):
    binding.check_copy_pairs(np.array([[0, 3], [1, 4]]), 8)
    binding.check_copy_pairs(np.zeros((0, 2)), 8)
    with pytest.raises(binding.PagedKVError) as e:
        binding.check_copy_pairs(np.array([[0, 3], [1, 3]]), 8)     # repeated destination
    assert e.value.code == -4
    with pytest.raises(binding.PagedKVError) as e:
        binding.check_copy_pairs(np.array([[0, 3], [3, 5]]), 8)     # destination also a source
    assert e.value.code == -4
    with pytest.raises(binding.PagedKVError) as e:
        binding.check_copy_pairs(np.array([[0, 8]]), 8)
    assert e.value.code == -3


def test_binding_refuses_cpu_tensors(binding):
    import torch
    q = torch.zeros(1, 1, 64)
    kc = torch.zeros(2, 1, 16, 64)
    with pytest.raises(ValueError):
        binding.paged_decode_attention(q.clone(), q, kc, kc, torch.zeros(1, 1, dtype=torch.int32),
                                       torch.ones(1, dtype=torch.int32), 0.1, max_context_len=1)
