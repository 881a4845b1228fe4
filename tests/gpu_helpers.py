"""Shared steps of the GPU parity tests: run one decode step (copy-on-write
copies, KV append, attention) through the C-ABI binding, run the same step
on the oracle, and compare."""
import numpy as np
import torch

import oracle
from paged_kv_cache_177_gb300 import workloads as W

# Tolerances: bf16 K/V with fp32 accumulation, |gpu - ref| <= 2e-3 + 1e-2 |ref|
# per element (max-abs 2e-3 and max-rel 1e-2 read as one allclose bound); fp32
# K/V, |gpu - ref| <= 1e-5 + 1e-5 |ref|.
TOL = {"bf16": (2e-3, 1e-2), "f32": (1e-5, 1e-5)}


def lib():
    from paged_kv_cache_177_gb300 import build
    build.build_library()
    from paged_kv_cache_177_gb300 import binding
    return binding


def gpu_step(w, partition_tokens=0, stream=None, attention=True):
    """Runs the step on the GPU copy of ``w`` (modified in place); returns out."""
    b = lib()
    lay = w.layout
    b.copy_blocks(w.k_cache, w.v_cache, w.cow_pairs, host_pairs=lay.cow_pairs, stream=stream)
    b.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache, stream=stream)
    out = torch.empty_like(w.q)
    if attention:
        b.paged_decode_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                                 max_context_len=lay.max_context_len, partition_tokens=partition_tokens,
                                 stream=stream)
    return out


def host_arrays(w):
    return {k: W.to_numpy(getattr(w, k)) for k in ("q", "k_cache", "v_cache", "k_new", "v_new")}


def oracle_step(h, lay, scale, seq_ids=None):
    """Oracle copy + append on the host caches (in place), then attention."""
    oracle.copy_blocks(h["k_cache"], h["v_cache"], lay.cow_pairs)
    oracle.kv_append(h["k_new"], h["v_new"], lay.slot_mapping, h["k_cache"], h["v_cache"])
    return oracle.paged_decode_attention(h["q"], h["k_cache"], h["v_cache"], lay.block_tables, lay.context_lens,
                                         scale, lay.spec.num_kv_heads, seq_ids=seq_ids)


def assert_close(got: torch.Tensor, ref: np.ndarray, dtype: str, what: str = ""):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    atol, rtol = TOL[dtype]
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (f"{what}: max abs err {err.max():.3e} (bound at worst element "
                                  f"{bound[worst]:.3e}, index {worst}, got {g[worst]:.6f}, ref {ref[worst]:.6f})")
    return float(err.max())


def assert_caches_equal(w, h):
    for name in ("k_cache", "v_cache"):
        got = W.to_numpy(getattr(w, name)).view(np.uint8)
        exp = h[name].view(np.uint8)
        assert np.array_equal(got, exp), f"{name} after copy_blocks + kv_append differs from the oracle"


EDGE_LENGTHS = (0, 1, 15, 16, 17, 31, 33, 64, 100, 255, 511, 512, 513, 1000, 1537, 7)


def path_switching_calls():
    """Decode calls that take the decode paths in turn, for one reused
    workspace: (label, host workload, partition_tokens, persistent?).

    1. a few long 13B-class sequences, automatic partitioning: the split grid
       kernel, whose partial states land in the workspace;
    2. a 13B-class batch of 64, automatic: the persistent kernel, whose
       arrival counters must read zero although call 1 wrote partials;
    3. fixed 128-token partitions on a GQA batch with edge lengths;
    4. a larger GQA batch, automatic: the persistent kernel again;
    5. a GQA batch with fp32 caches split into partitions (the staged fp32
       kernel writes its partial states after the counter header too)."""
    return [
        ("grid split", W.make_workload("mha13b", lengths_list=(600, 1500, 2048, 513, 1024, 77, 1800, 900),
                                       seed=301), 0, False),
        ("persistent", W.make_workload("mha13b", seed=302), 0, True),
        ("fixed partitions", W.make_workload("gqa8b", lengths_list=EDGE_LENGTHS, seed=303), 128, False),
        ("persistent, larger batch", W.make_workload("gqa8b", num_seqs=160, len_hi=1500, seed=304), 0, True),
        ("fp32 grid split", W.make_workload("gqa8b", lengths_list=(600, 1500, 2048, 513, 77, 1024), dtype="f32",
                                            seed=305), 0, False),
    ]


def torch_dtype(spec):
    """The cache element type of a workload spec."""
    return torch.bfloat16 if spec.dtype == "bf16" else torch.float32


def prepared(case):
    """GPU copy of a path_switching_calls case after its copies and appends,
    and the oracle's output for it (every sequence, every head)."""
    label, wc, pt, persistent = case
    h = host_arrays(wc)
    ref = oracle_step(h, wc.layout, wc.scale)
    w = wc.to("cuda")
    gpu_step(w, attention=False)
    return w, ref
