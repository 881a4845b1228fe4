"""Benchmark of one paged decode step on GB300.

A step is one pass of the whole hot path over one batch of the workload:
copy-on-write block copies (when the workload has any), the KV append of
this step's tokens, and paged decode attention (split-context partitions and
their log-sum-exp reduce included) for every sequence -- one
paged_decode_step call, captured once as a CUDA graph and replayed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mha13b]
    python bench.py --impl reference ...     # the fp64 CPU oracle on the host cores

Prints one JSON line.  ``value`` is the step's algorithmic bytes (K/V read,
q read, output written, tables, append and copy traffic) divided by the
device time of the step, as GB/s, summed over ranks; inputs are resident in
HBM.  ``e2e`` repeats the measurement with the per-step inputs in pinned host
memory and the output going back there, inside the timed region: through the
copy engine, and in place (the kernels read and write the pinned host
buffers over NVLink-C2C); the faster is reported, both are shown.
``parity`` compares the timed step's output with the oracle on every
sequence and head of the batch, and reports the error of the same call with
fp32 output (the accumulator before bf16 rounding) against 2e-3 alone.
Without ``--workload`` the line headlines mha13b (the 13B-class batch) and
adds a ``configs`` object: every other configuration of the workload set
(tiny, gqa8b, parallel_sampling, long_context) timed the same way (step and
attention call), checked against the oracle on every sequence, and with the
oracle's own rate on the host cores; and ``next_rows``: the shared-prefix
decode call on parallel_sampling (against plain decode, oracle on every
sequence) and a prefill step on each prefill workload (TFLOP/s against the
measured bf16 peak; the two shortest prompts against the oracle, every
prompt's last row against the decode kernels).
Under torchrun every rank runs its own replica of the workload (weak
scaling): the path has no exchange step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_kv_cache_177_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s and % of GB300 HBM peak; µs per decode step"
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20


def describe(sp: W.WorkloadSpec) -> str:
    if sp.lengths == "lognormal":
        lens = f"lognormal(median {sp.len_median:g}, sigma {sp.len_sigma:g}) clipped to [{sp.len_lo}, {sp.len_hi}]"
    elif sp.lengths == "sampling":
        lens = (f"{sp.num_prompts} prompts x {sp.samples_per_prompt} samples, prompt {sp.prompt_len} tokens + "
                f"suffix uniform [{sp.len_lo}, {sp.len_hi}]")
    elif sp.lengths == "explicit":
        lens = f"explicit lengths {list(sp.lengths_list)}"
    else:
        lens = f"uniform int [{sp.len_lo}, {sp.len_hi}]"
    pool = f"pool {sp.pool_blocks} blocks" if sp.pool_blocks else f"pool {sp.pool_factor:g}x the blocks needed"
    return (f"{sp.name}: {sp.num_seqs} seqs, {sp.num_q_heads} q / {sp.num_kv_heads} kv heads, head_dim "
            f"{sp.head_dim}, {sp.dtype}, block 16, {lens}, shuffled {pool}")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Committed ncu summaries that hold a kernel's DRAM traffic per launch on a
# workload, valid while the source the kernel is built and launched from is
# unchanged: a sha256 over the definitions each kernel depends on (its own
# code, the device helpers and per-block steps it calls, the host code that
# encodes its tensor maps and launches it), comments and whitespace removed.
# A change anywhere else in the same files leaves the capture valid.
PROFILED = {
    ("mha13b", "decode_bf16_persistent_kernel"): "decode_bf16_persistent_kernel_mha13b.md",
    ("gqa8b", "decode_bf16_persistent_kernel"): "decode_bf16_persistent_kernel_gqa8b.md",
    ("long_context", "decode_bf16_kernel"): "decode_bf16_kernel_long_context.md",
}
_CSRC = "paged_kv_cache_177_gb300/csrc/"
_DEVICE_COMMON = ["kBlock", "kSplitBlocks", "g_dev_error", "raise_error", "to_out", "DecodeParams", "seq_len",
                  "WarpAttn", "WarpAttnScalar"]
_HOST_COMMON = ["PKV_MHA_CUDA_CORES", "kMhaCudaCores", "kCounterBytes", "kSmemLimit", "launch_pdl", "encode_fn",
                "encode_cache_map", "max_parts_for", "sm_count", "decode_dispatch", "pkv_decode_partition_tokens",
                "pkv_decode_workspace_bytes", "grid_workspace_bytes", "input_dtype", "use_persistent"]
KERNEL_SPANS = {
    "decode_bf16_persistent_kernel": {
        "include/pagedkv.h": None, _CSRC + "pkv_ptx.cuh": None,
        _CSRC + "pkv_kernels.cuh": _DEVICE_COMMON + ["PersistCfg", "Cursor", "cursor_advance", "merge_segments",
                                                     "decode_bf16_persistent_kernel"],
        _CSRC + "pkv.cu": _HOST_COMMON + ["PKV_PERSIST_WARPS", "PKV_PERSIST_STAGES_D128", "PKV_PERSIST_STAGES_D64",
                                          "PKV_PERSIST_MAX_SEQS", "kPersistWarps", "kPersistMaxCtas",
                                          "kPersistMaxSeqs", "persist_workspace_bytes", "launch_persistent",
                                          "persistent_by_shape"],
    },
    "decode_bf16_kernel": {
        "include/pagedkv.h": None, _CSRC + "pkv_ptx.cuh": None,
        _CSRC + "pkv_kernels.cuh": _DEVICE_COMMON + ["Bf16Cfg", "grid_produce", "grid_consume",
                                                     "decode_bf16_kernel", "block_reduce", "lse_reduce_kernel"],
        _CSRC + "pkv.cu": _HOST_COMMON + ["PKV_GRID_STAGES", "PKV_GRID_CONSUMERS", "kNstage", "kNcw",
                                          "launch_bf16", "grid_by_shape", "launch_reduce"],
    },
}


def _strip_comments(text: str) -> str:
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    return re.sub(r"//[^\n]*", " ", text)


def _matching(text: str, i: int, open_c: str, close_c: str) -> int:
    """Index just past the bracket that closes the one at text[i]."""
    depth = 0
    for j in range(i, len(text)):
        if text[j] == open_c:
            depth += 1
        elif text[j] == close_c:
            depth -= 1
            if depth == 0:
                return j + 1
    raise ValueError("unbalanced source")


def definition_spans(text: str, name: str):
    """The definitions of ``name`` in C++ source ``text`` (comments removed):
    a struct or class body, a function body, a constant or variable up to its
    semicolon, or a #define line. Calls and declarations are not definitions."""
    spans = []
    for m in re.finditer(r"\b%s\b" % re.escape(name), text):
        i, j = m.start(), m.end()
        line_start = text.rfind("\n", 0, i) + 1
        before = text[line_start:i]
        if before.strip() == "#define":
            spans.append(text[line_start:text.find("\n", j)])
            continue
        if re.search(r"\b(struct|class)\s*$", before):
            brace, semi = text.find("{", j), text.find(";", j)
            if brace != -1 and (semi == -1 or brace < semi):
                spans.append(text[i:_matching(text, brace, "{", "}")])
            continue
        k = j
        while k < len(text) and text[k].isspace():
            k += 1
        if k < len(text) and text[k] == "(":
            close = _matching(text, k, "(", ")")
            rest = re.match(r"\s*(const\s*)?\{", text[close:])
            if rest and not re.search(r"[=(,]\s*$", before):
                brace = close + rest.end() - 1
                spans.append(text[i:_matching(text, brace, "{", "}")])
            continue
        if k < len(text) and text[k] in "=[" and re.search(r"\b(constexpr|__device__|const)\b", before):
            spans.append(text[line_start:text.find(";", j) + 1])
    return spans


def kernel_source_sha256(kernel: str) -> str:
    """sha256 of the source spans ``kernel`` is built and launched from."""
    import hashlib
    h = hashlib.sha256()
    for f, names in KERNEL_SPANS[kernel].items():
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            text = _strip_comments(fh.read())
        parts = [text] if names is None else []
        for n in names or ():
            found = definition_spans(text, n)
            if not found:
                raise KeyError(f"{n} has no definition in {f}")
            parts.extend(found)
        for part in parts:
            h.update(" ".join(part.split()).encode())
    return h.hexdigest()


def f32_kernel_name(sp) -> str:
    """The fp32 decode kernel for a workload's group size (tensor cores past four heads)."""
    return "decode_f32_tc_kernel" if sp.num_q_heads // sp.num_kv_heads > 4 else "decode_f32_staged_kernel"


def profiled_traffic(workload: str, kernel: str):
    """(DRAM bytes per launch, summary file) from the committed ncu summary, or
    (None, reason) when there is none or the kernel changed since it was taken."""
    name = PROFILED.get((workload, kernel))
    if name is None:
        return None, "no ncu capture of this kernel on this workload"
    try:
        with open(os.path.join(ROOT, "profiles", name)) as f:
            fields = dict(line.split(": ", 1) for line in f.read().splitlines()
                          if line.startswith(("traffic_bytes_per_launch: ", "source_sha256: ")))
    except OSError:
        return None, f"profiles/{name} missing"
    if fields.get("source_sha256", "").strip() != kernel_source_sha256(kernel):
        return None, f"kernel sources changed since profiles/{name} was captured"
    return int(fields["traffic_bytes_per_launch"]), f"profiles/{name}"


def step_bytes(lay: W.Layout):
    """Algorithmic bytes of one step, by operation."""
    sp = lay.spec
    eb = 2 if sp.dtype == "bf16" else 4
    S, Hq, Hkv, D = sp.num_seqs, sp.num_q_heads, sp.num_kv_heads, sp.head_dim
    nblk = (lay.context_lens.astype(np.int64) + 15) // 16
    attn = lay.kv_bytes(eb) + 2 * S * Hq * D * eb + int(nblk.sum()) * 4 + S * 4
    T = len(lay.slot_mapping)
    append = T * Hkv * D * 2 * eb * 2 + T * 8
    n = len(lay.cow_pairs)
    copy = n * Hkv * 16 * D * eb * 2 * 2 + n * 16
    return {"attention": attn, "append": append, "copy": copy, "total": attn + append + copy}


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if self.proc is None or not self.lines:
            return None
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = max(smax, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, local, dist
    return 0, 1, 0, None


def max_over_ranks(x: float, dist, device) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, dist, device) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_sample(lay: W.Layout, host: dict, target_s: float, nthreads: int = 0):
    """Times the oracle (fp64, all host cores) on a bounded sample of the
    workload -- about ``target_s`` seconds of CPU work -- after applying the
    step's copies and appends on the host.  The sample grows by sequences
    until one pass takes a quarter of the budget (or covers the workload),
    then passes repeat until the budget is spent.  ``nthreads`` = 0 uses every
    host core.  Returns (GB/s, seconds, sequences, passes, sample bytes per pass)."""
    import oracle

    eb = 2 if lay.spec.dtype == "bf16" else 4
    oracle.copy_blocks(host["k_cache"], host["v_cache"], lay.cow_pairs)
    oracle.kv_append(host["k_new"], host["v_new"], lay.slot_mapping, host["k_cache"], host["v_cache"])
    order = np.random.default_rng(0).permutation(lay.spec.num_seqs)
    per_token = lay.spec.num_kv_heads * lay.spec.head_dim * 2 * eb

    def run(ids):
        t0 = time.perf_counter()
        oracle.paged_decode_attention(host["q"], host["k_cache"], host["v_cache"], lay.block_tables,
                                      lay.context_lens, 1.0 / math.sqrt(lay.spec.head_dim), lay.spec.num_kv_heads,
                                      seq_ids=ids, nthreads=nthreads or cpu_cores())
        return time.perf_counter() - t0

    n = min(len(order), max(1, (nthreads or cpu_cores()) // max(1, lay.spec.num_kv_heads)))
    dt = run(order[:n])
    while dt < target_s / 4 and n < len(order):
        n = min(len(order), max(n + 1, int(n * min(8.0, target_s / 4 / max(dt, 1e-4)))))
        dt = run(order[:n])
    ids = order[:n]
    total, passes = dt, 1
    while total < target_s:
        total += run(ids)
        passes += 1
    nbytes = int(lay.context_lens[ids].astype(np.int64).sum()) * per_token
    return nbytes * passes / total / 1e9, total, int(n), passes, nbytes


def full_parity(lay: W.Layout, host: dict, out: torch.Tensor, dtype: str, out32=None):
    """The timed step's output against the oracle on every sequence and head
    (the host caches already hold the step's copies and appends). ``out32``:
    the same attention call with fp32 output (bf16 inputs), whose error before
    rounding is reported against 2e-3 absolute alone."""
    import oracle

    ref = oracle.paged_decode_attention(host["q"], host["k_cache"], host["v_cache"], lay.block_tables,
                                        lay.context_lens, 1.0 / math.sqrt(lay.spec.head_dim), lay.spec.num_kv_heads,
                                        nthreads=cpu_cores())
    got = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    atol, rtol = (2e-3, 1e-2) if dtype == "bf16" else (1e-5, 1e-5)
    res = {"sample_seqs": int(lay.spec.num_seqs), "of_seqs": int(lay.spec.num_seqs), "elements": int(err.size),
           "max_abs_err": float(err.max()),
           "max_rel_err": float((err / np.maximum(np.abs(ref), 1e-30)).max()),
           "bound": f"|gpu - ref| <= {atol:g} + {rtol:g} |ref| per element",
           "within_bound": bool(np.all(np.isfinite(got)) and np.all(err <= atol + rtol * np.abs(ref)))}
    if out32 is not None:
        g32 = out32.cpu().numpy().astype(np.float64)
        e32 = np.abs(g32 - ref)
        res["unrounded"] = {
            "max_abs_err": float(e32.max()), "bound": "2e-3 absolute",
            "within_bound": bool(np.all(np.isfinite(g32)) and e32.max() <= 2e-3),
            "rounds_to_output": bool(torch.equal(out32.to(torch.bfloat16).cpu().view(torch.int16),
                                                 out.cpu().view(torch.int16))),
            "how": "the same attention call with fp32 output (PKV_BF16_OUT_F32): O / L before rounding to bf16"}
    return res


def unrounded_output(B, w, lay, pt, ws, stream):
    """fp32 output of the attention call on bf16 inputs, or None for fp32."""
    if w.q.dtype != torch.bfloat16:
        return None
    out32 = torch.empty(tuple(w.q.shape), dtype=torch.float32, device=w.q.device)
    B.paged_decode_attention(out32, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                             max_context_len=lay.max_context_len, partition_tokens=pt, workspace=ws, stream=stream)
    return out32


def config_summary(name: str, args, dev, B, evict) -> dict:
    """One more workload in the default run: its decode step (one
    paged_decode_step, replayed as a CUDA graph, L2 evicted between steps) and
    the attention call alone, timed with CUDA events; its output against the
    oracle on every sequence; and the oracle's rate on the host cores."""
    sp = W.spec(name)
    pt = sp.partition_tokens
    w = W.make_workload(sp, device=dev)
    lay = w.layout
    S, Hq, Hkv, D = sp.num_seqs, sp.num_q_heads, sp.num_kv_heads, sp.head_dim
    maxlen = lay.max_context_len
    nbytes = step_bytes(lay)
    ws = torch.zeros(max(B.workspace_bytes(S, Hq, Hkv, D, maxlen, pt), 16), dtype=torch.uint8, device=dev)
    out = torch.empty_like(w.q)
    stream = torch.cuda.Stream(dev)
    has_pairs = len(lay.cow_pairs) > 0
    persistent = B.decode_persistent(S, Hkv, pt, w.q.dtype)
    launches = B.decode_launches(S, Hkv, maxlen, pt, w.q.dtype)
    B.check_copy_pairs(lay.cow_pairs, lay.num_blocks)

    def step():
        B.paged_decode_step(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, w.k_new,
                            w.v_new, w.slot_mapping, w.cow_pairs if has_pairs else None, check=False,
                            max_context_len=maxlen, partition_tokens=pt, workspace=ws, stream=stream)

    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            evict.sum()
            step()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    n = args.config_steps
    attn_args = B.decode_args(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                              max_context_len=maxlen, partition_tokens=pt, workspace=ws, stream=stream)
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    aev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for i in range(n):
            evict.sum()
            sev[i][0].record(stream)
            g.replay()
            sev[i][1].record(stream)
        for i in range(n):
            evict.sum()
            aev[i][0].record(stream)
            B.decode_raw(attn_args)
            aev[i][1].record(stream)
        # warm: the attention call back to back with no eviction, so blocks that several
        # sequences share (parallel sampling) can stay in L2 between launches
        wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            wev[i][0].record(stream)
            B.decode_raw(attn_args)
            wev[i][1].record(stream)
        out32 = unrounded_output(B, w, lay, pt, ws, stream)
    torch.cuda.synchronize(dev)
    err = B.device_error(clear=True)
    if err:
        raise RuntimeError(f"{name}: device error word set: {err:#x}")
    t_warm = sum(a.elapsed_time(b) for a, b in wev) / n / 1e3
    step_ms = sorted(a.elapsed_time(b) for a, b in sev)
    attn_ms = [a.elapsed_time(b) for a, b in aev]
    t_step = sum(step_ms) / n / 1e3
    t_attn = sum(attn_ms) / n / 1e3
    peak, _ = peaks()
    host = {k: W.to_numpy(getattr(w, k)) for k in ("q", "k_cache", "v_cache", "k_new", "v_new")}
    gbs, secs, nseq, passes, sb = oracle_sample(lay, host, args.config_cpu_seconds)
    parity = full_parity(lay, host, out, sp.dtype, out32)
    kernel = ("decode_bf16_persistent_kernel" if persistent else
              ("decode_bf16_kernel" if sp.dtype == "bf16" else f32_kernel_name(sp)) +
              (" + lse_reduce_kernel" if launches == 2 else ""))
    res = {
        "workload": describe(sp),
        "partition_tokens": "balanced (persistent kernel)" if persistent else B.partition_tokens(S, Hkv, maxlen, pt),
        "us_per_step": round(t_step * 1e6, 2),
        "us_per_step_median": round(step_ms[n // 2] * 1e3, 2),
        "us_per_step_p10_p90": [round(step_ms[n // 10] * 1e3, 2), round(step_ms[(9 * n) // 10] * 1e3, 2)],
        "step_GBps": round(nbytes["total"] / t_step / 1e9, 2),
        "seqs_per_s": round(S / t_step, 1),
        "attention": {"kernel": kernel, "us": round(t_attn * 1e6, 2),
                      "warm_us": round(t_warm * 1e6, 2),
                      "GBps": round(nbytes["attention"] / t_attn / 1e9, 2),
                      "roofline_frac": round(nbytes["attention"] / t_attn / 1e9 / peak, 4),
                      "bytes_per_launch": nbytes["attention"]},
        "step_bytes": nbytes,
        "timed_steps": n,
        "parity": parity,
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{nseq} of {S} sequences ({sb / 1e6:.1f} MB of K/V, all heads) x {passes} "
                                   f"passes in {secs:.1f} s"},
    }
    del w, ws, out, g
    torch.cuda.empty_cache()
    return res


def run_reference(args, rank, world, dist):
    """The oracle, as it stands, on this host's cores: each step one bounded
    sample of the workload (the same sequences every step)."""
    if rank != 0:
        return
    import oracle

    sp = W.spec(args.workload)
    w = W.make_workload(sp, device="cpu")
    lay = w.layout
    host = {k: W.to_numpy(getattr(w, k)) for k in ("q", "k_cache", "v_cache", "k_new", "v_new")}
    oracle.copy_blocks(host["k_cache"], host["v_cache"], lay.cow_pairs)
    oracle.kv_append(host["k_new"], host["v_new"], lay.slot_mapping, host["k_cache"], host["v_cache"])
    eb = 2 if sp.dtype == "bf16" else 4
    per_token = sp.num_kv_heads * sp.head_dim * 2 * eb
    order = np.random.default_rng(0).permutation(sp.num_seqs)
    budget = args.reference_seconds / max(1, args.steps + args.warmup)
    # size the per-step sample from one timed probe
    n = max(1, min(len(order), cpu_cores()))
    t0 = time.perf_counter()
    oracle.paged_decode_attention(host["q"], host["k_cache"], host["v_cache"], lay.block_tables, lay.context_lens,
                                  w.scale, sp.num_kv_heads, seq_ids=order[:n], nthreads=cpu_cores())
    probe = time.perf_counter() - t0
    n = int(max(1, min(len(order), n * budget / max(probe, 1e-3))))
    ids = order[:n]
    nbytes = int(lay.context_lens[ids].astype(np.int64).sum()) * per_token
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.paged_decode_attention(host["q"], host["k_cache"], host["v_cache"], lay.block_tables,
                                      lay.context_lens, w.scale, sp.num_kv_heads, seq_ids=ids, nthreads=cpu_cores())
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    value = nbytes / t / 1e9
    sample = (f"{n} of {sp.num_seqs} sequences ({int(lay.context_lens[ids].sum())} tokens, all heads) per step, "
              f"fp64 C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(sp), "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def pack_inputs(tensors, dev):
    """Packs tensors into one pinned host buffer and one device buffer (each
    tensor 256-byte aligned); returns typed views into both and the buffers."""
    offs, off = [], 0
    for t in tensors:
        offs.append(off)
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(max(off, 256), dtype=torch.uint8, pin_memory=True)
    dev_buf = torch.empty(max(off, 256), dtype=torch.uint8, device=dev)
    host_views, dev_views = [], []
    for t, o in zip(tensors, offs):
        nb = t.numel() * t.element_size()
        hv = host_buf[o:o + nb].view(t.dtype).view(t.shape)
        hv.copy_(t.cpu())
        host_views.append(hv)
        dev_views.append(dev_buf[o:o + nb].view(t.dtype).view(t.shape))
    dev_buf.copy_(host_buf)
    return host_views, dev_views, host_buf, dev_buf


def run_ours(args, rank, world, local, dist):
    from paged_kv_cache_177_gb300 import build
    build.build_library()
    from paged_kv_cache_177_gb300 import binding as B

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    over = {"dtype": args.dtype} if args.dtype else {}
    sp = W.spec(args.workload, seed=W.spec(args.workload).seed + 7919 * rank, **over)
    pt = args.partition_tokens if args.partition_tokens is not None else sp.partition_tokens
    w = W.make_workload(sp, device=dev)
    lay = w.layout
    S, Hq, Hkv, D = sp.num_seqs, sp.num_q_heads, sp.num_kv_heads, sp.head_dim
    maxlen = lay.max_context_len
    nbytes = step_bytes(lay)
    ws_bytes = B.workspace_bytes(S, Hq, Hkv, D, maxlen, pt)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)   # zero-filled once, as required
    out = torch.empty_like(w.q)
    stream = torch.cuda.Stream(dev)
    has_pairs = len(lay.cow_pairs) > 0
    attn_launches = B.decode_launches(S, Hkv, maxlen, pt, w.q.dtype)
    persistent = B.decode_persistent(S, Hkv, pt, w.q.dtype)
    launches_per_step = (1 if has_pairs else 0) + 1 + attn_launches
    B.check_copy_pairs(lay.cow_pairs, lay.num_blocks)
    # per-step inputs live in buffers of their own, so the end-to-end run can
    # refill them from pinned host memory; the step rewrites the same slots and
    # blocks every time, so repeating it is idempotent
    # one step's inputs packed into one staging buffer (each 256-byte aligned):
    # pinned on the host, and on the device, where the calls read typed views
    host_in, dev_in, host_buf, dev_buf = pack_inputs(
        [w.q, w.k_new, w.v_new, w.slot_mapping, w.block_tables, w.context_lens, w.cow_pairs], dev)
    q, k_new, v_new, slots, tables, lens, pairs = dev_in
    evict = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev).fill_(1.0)

    def flush_l2():
        evict.sum()           # reads 256 MiB: evicts K/V lines without leaving dirty ones

    def step():
        # the whole step in one library call: copies, append, then attention (whose set-up overlaps the append)
        B.paged_decode_step(out, q, w.k_cache, w.v_cache, tables, lens, w.scale, k_new, v_new, slots,
                            pairs if has_pairs else None, check=False, max_context_len=maxlen, partition_tokens=pt,
                            workspace=ws, stream=stream)

    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2()
            step()
    torch.cuda.synchronize(dev)
    if B.device_error(clear=True):
        raise RuntimeError("device error word set during warm-up")

    # the step as a CUDA graph: a decode loop replays it without host launch work
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        step()
    torch.cuda.synchronize(dev)

    steps = args.steps
    if steps is None:
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(20):
                flush_l2()
                g_step.replay()
        torch.cuda.synchronize(dev)
        steps = int(min(20000, max(200, 1.5 / ((time.perf_counter() - t0) / 20))))

    def timed(graph, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for i in range(n):
                flush_l2()                 # untimed
                evs[i][0].record(stream)
                graph.replay()
                evs[i][1].record(stream)
        return evs

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        wall0 = time.perf_counter()
        ev = timed(g_step, steps)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    # the attention call alone, launched straight through the C ABI with its
    # arguments marshalled once (the eviction read in front of each call keeps
    # the GPU busy while the host enqueues, so host time is not in the window)
    attn_args = B.decode_args(out, q, w.k_cache, w.v_cache, tables, lens, w.scale, max_context_len=maxlen,
                              partition_tokens=pt, workspace=ws, stream=stream)
    n_attn = min(steps, 2000)
    aev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_attn)]
    with torch.cuda.stream(stream):
        for i in range(n_attn):
            flush_l2()
            aev[i][0].record(stream)
            B.decode_raw(attn_args)
            aev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    attn_ms = [a.elapsed_time(b) for a, b in aev]
    t_step = sum(step_ms) / len(step_ms) / 1e3
    t_attn = sum(attn_ms) / len(attn_ms) / 1e3
    t_step_max = max_over_ranks(t_step, dist, dev)
    total_bytes = sum_over_ranks(nbytes["total"], dist, dev)
    value = total_bytes / t_step_max / 1e9

    # ---- end to end: per-step inputs copied in from pinned host memory and the
    # output copied back, inside the timed region (one copy each way) ----
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = host_buf.numel()
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = min(steps, 2000)
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    with torch.cuda.stream(stream):
        for i in range(args.warmup + e2e_steps):
            flush_l2()
            if i >= args.warmup:
                eev[i - args.warmup][0].record(stream)
            dev_buf.copy_(host_buf, non_blocking=True)
            g_step.replay()
            host_out.copy_(out, non_blocking=True)
            if i >= args.warmup:
                eev[i - args.warmup][1].record(stream)
    torch.cuda.synchronize(dev)
    t_ce = sum(a.elapsed_time(b) for a, b in eev) / e2e_steps / 1e3
    t_ce_max = max_over_ranks(t_ce, dist, dev)

    # ---- end to end in place: the step's kernels read this step's inputs from the
    # pinned host buffer and write the output into pinned host memory (over the
    # NVLink-C2C host link; no copy-engine round trips) ----
    hq, hk, hv, hslots, htables, hlens, hpairs = host_in
    zc_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

    def step_in_place():
        B.paged_decode_step(zc_out, hq, w.k_cache, w.v_cache, htables, hlens, w.scale, hk, hv, hslots,
                            hpairs if has_pairs else None, check=False, max_context_len=maxlen, partition_tokens=pt,
                            workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2()
            step_in_place()
    torch.cuda.synchronize(dev)
    if not torch.equal(zc_out.view(torch.uint8), out.cpu().view(torch.uint8)):
        raise RuntimeError("the in-place step's output differs from the device step's")
    g_zc = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_zc, stream=stream):
        step_in_place()
    torch.cuda.synchronize(dev)
    zev = timed(g_zc, e2e_steps)
    torch.cuda.synchronize(dev)
    t_zc = sum(a.elapsed_time(b) for a, b in zev) / e2e_steps / 1e3
    t_zc_max = max_over_ranks(t_zc, dist, dev)
    t_e2e_max = min(t_zc_max, t_ce_max)
    e2e_value = total_bytes / t_e2e_max / 1e9
    err = B.device_error(clear=True)
    if err:
        raise RuntimeError(f"device error word set during the timed steps: {err:#x}")

    if rank != 0:
        return
    peak, peak_kind = peaks()
    attn_gbs = nbytes["attention"] / t_attn / 1e9
    cpu = None
    parity = None
    if world == 1 and not args.no_cpu_baseline:
        # the device caches already hold the step's copies and appends; the oracle
        # re-applies them on the host (idempotent) before attending
        host = {k: W.to_numpy(getattr(w, k)) for k in ("q", "k_cache", "v_cache", "k_new", "v_new")}
        gbs, secs, nseq, passes, sb = oracle_sample(lay, host, args.cpu_seconds)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{nseq} of {S} sequences ({sb / 1e6:.1f} MB of K/V, all heads) x {passes} passes in "
                         f"{secs:.1f} s, fp64 C oracle, after the step's copies and appends"}
        g1, s1, n1, p1, b1 = oracle_sample(lay, host, min(3.0, args.cpu_seconds / 3), nthreads=1)
        cpu["single_thread"] = {"value": round(g1, 4), "unit": "GB/s", "cores": 1,
                                "sample": f"{n1} sequences ({b1 / 1e6:.1f} MB) x {p1} passes in {s1:.1f} s"}
        out32 = unrounded_output(B, w, lay, pt, ws, stream)
        torch.cuda.synchronize(dev)
        parity = full_parity(lay, host, out, sp.dtype, out32)
    configs = next_rows = None
    if world == 1 and args.all_configs:
        # the other configurations of the workload set, each measured and
        # checked the same way (the headline's buffers are released first)
        del g_step, g_zc
        torch.cuda.empty_cache()
        configs = {name: config_summary(name, args, dev, B, evict)
                   for name in W.CONFIG_ORDER if name != sp.name}
        configs["all_within_bound"] = bool(
            (parity is None or parity["within_bound"]) and
            all(c["parity"]["within_bound"] for c in configs.values() if isinstance(c, dict)))
        # the rows beyond the decode step: shared-prefix decode and prefill, each timed and checked
        next_rows = {"shared_prefix": shared_prefix_measure(max(args.config_steps // 10, 3), dev, B, evict),
                     "prefill": {name: prefill_measure(name, 30, dev, B, evict, oracle_seqs=2)
                                 for name in W.PREFILL_SPECS}}
    srt = sorted(step_ms)
    roof_kernel = ("decode_bf16_persistent_kernel" if persistent else
                   "decode_bf16_kernel" if sp.dtype == "bf16" else f32_kernel_name(sp))
    # the captures were taken on the workloads' default launch configuration
    traffic, traffic_src = profiled_traffic(sp.name if args.partition_tokens is None and args.dtype is None else "",
                                            roof_kernel)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_step_max * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if sp.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {
            "workload": describe(sp),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "step": "paged_decode_step: " + ("copy_blocks + " if has_pairs else "") +
                    "kv_append + paged_decode_attention (launched right after the append), replayed as one CUDA graph",
            "partition_tokens": "balanced (persistent kernel)" if persistent else B.partition_tokens(S, Hkv, maxlen, pt),
            "max_context_len": maxlen,
            "tokens": int(lay.context_lens.sum()),
            "step_bytes": nbytes,
            "l2": "evicted between steps by reading a 256 MiB buffer (untimed); K/V larger than L2",
        },
        "us_per_step": round(t_step_max * 1e6, 2),
        "us_per_step_median": round(srt[len(srt) // 2] * 1e3, 2),
        "us_per_step_p10_p90": [round(srt[len(srt) // 10] * 1e3, 2), round(srt[(9 * len(srt)) // 10] * 1e3, 2)],
        "seqs_per_s": round(S * world / t_step_max, 1),
        "pct_hbm_peak": {"measured": round(100 * value / world / peak, 2),
                         "nominal_7.9TBs": round(100 * value / world / NOMINAL_HBM_GBS, 2)},
        "roofline": {
            "kernel": "paged_decode_attention (" + (roof_kernel if persistent else
                                                    roof_kernel + (" + lse_reduce_kernel" if attn_launches == 2 else "")) + ")",
            "bound": "hbm", "achieved": round(attn_gbs, 2), "peak": peak, "unit": "GB/s",
            "frac": round(attn_gbs / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
            "traffic": traffic, "traffic_source": traffic_src,
            "us_per_launch": round(t_attn * 1e6, 2), "timed_launches": len(attn_ms),
            "bytes_per_launch": nbytes["attention"],
        },
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(t_e2e_max * 1e3, 4),
                "transfer": "in place" if t_zc_max <= t_ce_max else "copy engine",
                "in_place": {"value": round(total_bytes / t_zc_max / 1e9, 2), "ms_per_step": round(t_zc_max * 1e3, 4),
                             "how": "the step's kernels read its inputs from the pinned host buffer and write the "
                                    "output to pinned host memory (NVLink-C2C), one CUDA graph per step"},
                "copy_engine": {"value": round(total_bytes / t_ce_max / 1e9, 2), "ms_per_step": round(t_ce_max * 1e3, 4),
                                "how": "one cudaMemcpyAsync of the packed inputs in, the step's graph, one of the "
                                       "output back"}},
        "gpu_launches": launches_per_step * steps,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
        "parity": parity,
        "wall_s_timed_region": round(wall, 3),
        "configs": configs,
        "next_rows": next_rows,
    }
    print(json.dumps(line), flush=True)


def run_op(args, rank, world, local, dist):
    """Secondary measurements (one JSON line each, rank 0 only):
    --op swap: swap-out (device pool -> pinned host pool) and swap-in (back to
      fresh device blocks) of the blocks of a quarter of the workload's
      sequences, as preemption does; GB/s of block bytes moved each way.
    --op append_layers: kv_append of one token per sequence into every layer's
      caches (40 layers) in one launch, against one launch per layer.
    --op shared_prefix: shared-prefix decode on a workload with shared
      prompts, against plain decode of the same batch.
    --op prefill: a prefill step (multi-token kv_append of every new token,
      then causal prefill attention) on --prefill-workload; TFLOP/s of the
      attention against the measured bf16 tensor peak."""
    from paged_kv_cache_177_gb300 import build
    build.build_library()
    from paged_kv_cache_177_gb300 import binding as B

    if rank != 0:
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.op == "prefill":
        return run_prefill(args, dev, B)
    if args.op == "shared_prefix":
        evict = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev).fill_(1.0)
        res = shared_prefix_measure(args.steps or 50, dev, B, evict)
        if not res["parity"]["within_bound"]:
            raise RuntimeError(f"shared-prefix output outside the bound: {res['parity']}")
        line = {"metric": "shared-prefix decode attention, logical KV GB/s", "unit": "GB/s",
                "value": res["shared_prefix"]["logical_GBps"], "higher_is_better": True,
                "config": {"workload": res["workload"], "groups": res["groups"],
                           "shared_blocks": res["shared_blocks"]},
                "op": "shared_prefix", "n_gpus": 1, "dtype": "bf16", "data": "synthetic"}
        line.update({k: v for k, v in res.items() if k not in ("workload", "groups", "shared_blocks")})
        print(json.dumps(line), flush=True)
        return
    sp = W.spec(args.workload)
    w = W.make_workload(sp, device=dev)
    lay = w.layout
    eb = 2 if sp.dtype == "bf16" else 4
    block_bytes = sp.num_kv_heads * 16 * sp.head_dim * eb
    evict = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev).fill_(1.0)
    stream = torch.cuda.current_stream(dev)

    def time_it(fn, n):
        """Median device time of fn, captured once as a CUDA graph and replayed."""
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            fn()                                   # warm-up outside the capture
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            evict.sum()
            evs[i][0].record(stream)
            g.replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        t = sorted(a.elapsed_time(b) for a, b in evs)
        return t[len(t) // 2] / 1e3

    if args.op == "swap":
        seqs = np.arange(0, sp.num_seqs, 4)
        nblk = (lay.context_lens.astype(np.int64) + 15) // 16
        blocks = np.concatenate([lay.block_tables[s, :nblk[s]] for s in seqs]).astype(np.int64)
        n = len(blocks)
        hk = torch.empty((n,) + tuple(w.k_cache.shape[1:]), dtype=w.k_cache.dtype, pin_memory=True)
        hv = torch.empty_like(hk).pin_memory()
        out_pairs = np.stack([blocks, np.arange(n)], 1)
        back = np.random.default_rng(0).permutation(lay.num_blocks)[:n]
        in_pairs = np.stack([np.arange(n), back], 1)
        po, pi = torch.from_numpy(out_pairs).to(dev), torch.from_numpy(in_pairs).to(dev)
        dk, dv = torch.empty_like(w.k_cache), torch.empty_like(w.v_cache)
        B.check_swap_pairs(out_pairs, lay.num_blocks, n)
        B.check_swap_pairs(in_pairs, n, lay.num_blocks)
        t_out = time_it(lambda: B.swap_blocks(hk, hv, w.k_cache, w.v_cache, po, check=False), args.steps or 50)
        t_in = time_it(lambda: B.swap_blocks(dk, dv, hk, hv, pi, check=False), args.steps or 50)
        torch.cuda.synchronize(dev)
        src, dst = torch.from_numpy(blocks).to(dev), torch.from_numpy(back).to(dev)
        for a_, b_ in ((dk, w.k_cache), (dv, w.v_cache)):  # the round trip is a byte copy
            if not torch.equal(a_[dst].view(torch.uint8), b_[src].view(torch.uint8)):
                raise RuntimeError("swap round trip is not bit-exact")
        if B.device_error(clear=True):
            raise RuntimeError("device error word set during the swap benchmark")
        moved = 2 * n * block_bytes
        line = {"metric": "swap_blocks GB/s (block bytes moved per direction)", "unit": "GB/s",
                "value": round(moved / t_out / 1e9, 2),
                "swap_out": {"GB/s": round(moved / t_out / 1e9, 2), "us": round(t_out * 1e6, 2)},
                "swap_in": {"GB/s": round(moved / t_in / 1e9, 2), "us": round(t_in * 1e6, 2)},
                "blocks": int(n), "bytes_per_direction": int(moved), "higher_is_better": True,
                "config": {"workload": describe(sp), "host_pool": "pinned host memory addressed by the kernel"}}
    else:
        L = 40
        T = sp.num_seqs
        slots = w.slot_mapping
        kn = [torch.randn(w.k_new.shape, device=dev).to(w.k_new.dtype) for _ in range(L)]
        vn = [torch.randn(w.v_new.shape, device=dev).to(w.v_new.dtype) for _ in range(L)]
        # L layers' caches: views of one pool cut into L equal block ranges; one
        # token per sequence, each in a block of its own
        per = lay.num_blocks // L
        assert T <= per
        slots = torch.arange(T, device=dev, dtype=torch.int64) * 16 + 3
        kc = [w.k_cache[l * per:(l + 1) * per] for l in range(L)]
        vc = [w.v_cache[l * per:(l + 1) * per] for l in range(L)]
        ptrs = tuple(B.layer_pointers(x) for x in (kn, vn, kc, vc))
        t_one = time_it(lambda: B.kv_append_layers(kn, vn, slots, kc, vc, ptrs=ptrs), args.steps or 50)
        t_each = time_it(lambda: [B.kv_append(kn[l], vn[l], slots, kc[l], vc[l]) for l in range(L)], args.steps or 50)
        torch.cuda.synchronize(dev)
        for l in (0, L // 2, L - 1):  # token t's rows sit in block t, slot 3 of every layer's cache
            for new, cache in ((kn[l], kc[l]), (vn[l], vc[l])):
                if not torch.equal(cache[:T, :, 3].view(torch.uint8), new.view(torch.uint8)):
                    raise RuntimeError(f"layer {l}: appended rows differ from the new tokens")
        if B.device_error(clear=True):
            raise RuntimeError("device error word set during the multi-layer append benchmark")
        moved = L * T * sp.num_kv_heads * sp.head_dim * eb * 2 * 2
        line = {"metric": "kv_append over 40 layers, GB/s (read + write of the appended K/V)", "unit": "GB/s",
                "value": round(moved / t_one / 1e9, 2),
                "one_launch": {"GB/s": round(moved / t_one / 1e9, 2), "us": round(t_one * 1e6, 2)},
                "one_launch_per_layer": {"GB/s": round(moved / t_each / 1e9, 2), "us": round(t_each * 1e6, 2)},
                "timing": "each variant captured once as a CUDA graph and replayed",
                "higher_is_better": True, "config": {"workload": describe(sp), "layers": L, "tokens": T}}
    line.update({"op": args.op, "n_gpus": 1, "dtype": sp.dtype, "data": "synthetic"})
    print(json.dumps(line), flush=True)


def graph_time(fn, n, dev, evict):
    """Median device time of fn, captured once as a CUDA graph and replayed
    after an L2 eviction each time (at least once)."""
    n = max(n, 1)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        fn()                                   # warm-up outside the capture
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fn()
    stream = torch.cuda.current_stream(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        evict.sum()
        evs[i][0].record(stream)
        g.replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t = sorted(a.elapsed_time(b) for a, b in evs)
    return t[len(t) // 2] / 1e3


def tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def prefill_measure(name: str, n: int, dev, B, evict, oracle_seqs: int = 0) -> dict:
    """One prefill step (kv_append of every new token, then causal prefill
    attention) on workload ``name``: both timed as CUDA graphs (median of ``n``
    replays after an L2 eviction), each prompt's last row checked against the
    decode kernels, and the ``oracle_seqs`` shortest prompts against the
    oracle (every row, every head)."""
    w = W.make_prefill(name, device=dev)
    sp = w.spec
    host = ({k: W.to_numpy(getattr(w, k)) for k in ("q", "k_cache", "v_cache", "k_new", "v_new")}
            if oracle_seqs else None)
    out = torch.empty_like(w.q)
    mq, mc = w.max_query_len, w.max_context_len

    def attention():
        B.paged_prefill_attention(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.query_start,
                                  w.scale, max_query_len=mq, max_context_len=mc)

    def step():
        B.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)
        attention()

    t_step = graph_time(step, n, dev, evict)
    t_attn = graph_time(attention, n, dev, evict)
    # Each prompt's last query row attends its whole context: the decode kernels (CUDA cores or
    # mma.sync, no code shared with the tcgen05 prefill kernel) must give the same row.
    torch.cuda.synchronize(dev)
    if not bool(torch.isfinite(out.float()).all()):
        raise RuntimeError("non-finite prefill attention output")
    qs = w.query_start.to(torch.int64)
    has = (qs[1:] > qs[:-1]).nonzero().flatten()
    last = qs[1:][has] - 1
    dec = torch.empty((len(has),) + tuple(w.q.shape[1:]), dtype=w.q.dtype, device=dev)
    B.paged_decode_attention(dec, w.q[last].contiguous(), w.k_cache, w.v_cache, w.block_tables[has].contiguous(),
                             w.context_lens[has].contiguous(), w.scale, max_context_len=mc)
    torch.cuda.synchronize(dev)
    diff = float((out[last].float() - dec.float()).abs().max())
    if diff > 4e-3 + 2e-2 * float(dec.float().abs().max()):
        raise RuntimeError(f"prefill's last rows differ from decode by {diff}")
    if B.device_error(clear=True):
        raise RuntimeError("device error word set during the prefill benchmark")
    T = int(w.q.shape[0])
    flops = w.flops()
    peak, kind = tensor_peak()
    tflops = flops / t_attn / 1e12
    res = {"workload": f"{sp.name}: {sp.num_seqs} seqs, {sp.num_q_heads} q / {sp.num_kv_heads} kv heads, head_dim "
                       f"{sp.head_dim}, bf16, block 16, new tokens {sp.new_lengths} [{sp.new_lo}, {sp.new_hi}], "
                       f"prior context [{sp.prior_lo}, {sp.prior_hi}]",
           "attention": {"us": round(t_attn * 1e6, 2), "TFLOP/s": round(tflops, 2),
                         "frac_of_peak": round(tflops / peak, 4), "peak": peak, "peak_kind": kind},
           "step": {"us": round(t_step * 1e6, 2), "tokens_per_s": round(T / t_step, 1),
                    "what": "kv_append of every new token + prefill attention"},
           "flops": int(flops), "new_tokens": T,
           "check": {"last_rows_vs_decode_max_abs_diff": diff, "rows": int(len(has))}}
    if oracle_seqs:
        import oracle
        hs = w.host
        oracle.kv_append(host["k_new"], host["v_new"], hs["slot_mapping"], host["k_cache"], host["v_cache"])
        nq = np.diff(hs["query_start"])
        seqs = [int(i) for i in np.argsort(nq, kind="stable") if nq[i] > 0][:oracle_seqs]
        rows = np.concatenate([np.arange(hs["query_start"][i], hs["query_start"][i + 1]) for i in seqs])
        sub_qs = np.concatenate([[0], np.cumsum([nq[i] for i in seqs])]).astype(np.int32)
        ref = oracle.paged_prefill_attention(np.ascontiguousarray(host["q"][rows]), host["k_cache"],
                                             host["v_cache"], np.ascontiguousarray(hs["block_tables"][seqs]),
                                             np.ascontiguousarray(hs["context_lens"][seqs]), sub_qs, w.scale,
                                             sp.num_kv_heads, nthreads=cpu_cores())
        got = out[torch.from_numpy(rows).to(dev)].float().cpu().numpy().astype(np.float64)
        err = np.abs(got - ref)
        res["parity"] = {"sequences": seqs, "rows": int(len(rows)), "max_abs_err": float(err.max()),
                         "bound": "|gpu - ref| <= 0.002 + 0.01 |ref| per element",
                         "within_bound": bool(np.all(err <= 2e-3 + 1e-2 * np.abs(ref)))}
    del w, out, dec
    torch.cuda.empty_cache()
    return res


def shared_prefix_measure(n: int, dev, B, evict) -> dict:
    """Shared-prefix decode on parallel_sampling (32 prompts x 4 samples): the
    call that reads each group's shared prompt blocks once, timed as a CUDA
    graph against plain decode of the same batch, and checked against the
    oracle on every sequence and head."""
    import oracle
    sp = W.spec("parallel_sampling")
    w = W.make_workload(sp, device=dev)
    lay = w.layout
    host = {k: W.to_numpy(getattr(w, k)) for k in ("q", "k_cache", "v_cache", "k_new", "v_new")}
    H = sp.num_q_heads
    groups = torch.from_numpy(lay.group_members).to(dev)
    shared = torch.from_numpy(lay.shared_blocks).to(dev)
    out_c, out_p = torch.empty_like(w.q), torch.empty_like(w.q)
    maxlen = lay.max_context_len
    ws_c = torch.empty(B.shared_prefix_workspace_bytes(sp.num_seqs, H, sp.head_dim, maxlen, groups.shape[1]),
                       dtype=torch.uint8, device=dev)
    ws_p = torch.zeros(max(16, B.workspace_bytes(sp.num_seqs, H, sp.num_kv_heads, sp.head_dim, maxlen)),
                       dtype=torch.uint8, device=dev)
    # the step's writes, in the step's order: copy-on-write copies, then the new tokens
    B.copy_blocks(w.k_cache, w.v_cache, w.cow_pairs, host_pairs=lay.cow_pairs)
    B.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)
    t_c = graph_time(lambda: B.paged_decode_attention_shared_prefix(
        out_c, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, groups, shared,
        max_context_len=maxlen, workspace=ws_c), n, dev, evict)
    t_p = graph_time(lambda: B.paged_decode_attention(
        out_p, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, max_context_len=maxlen,
        workspace=ws_p), n, dev, evict)
    torch.cuda.synchronize(dev)
    if B.device_error(clear=True):
        raise RuntimeError("device error word set during the shared-prefix benchmark")
    oracle.copy_blocks(host["k_cache"], host["v_cache"], lay.cow_pairs)
    oracle.kv_append(host["k_new"], host["v_new"], lay.slot_mapping, host["k_cache"], host["v_cache"])
    ref = oracle.paged_decode_attention(host["q"], host["k_cache"], host["v_cache"], lay.block_tables,
                                        lay.context_lens, w.scale, sp.num_kv_heads, nthreads=cpu_cores())
    got = out_c.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    eb = 2
    logical, unique = lay.kv_bytes(eb), lay.unique_kv_bytes(eb)
    peak, kind = peaks()
    res = {"workload": describe(sp), "groups": int(groups.shape[0]), "shared_blocks": int(lay.shared_blocks[0]),
           "shared_prefix": {"us": round(t_c * 1e6, 2), "logical_GBps": round(logical / t_c / 1e9, 2),
                             "unique_GBps": round(unique / t_c / 1e9, 2),
                             "unique_frac_of_peak": round(unique / t_c / 1e9 / peak, 4)},
           "plain_decode": {"us": round(t_p * 1e6, 2), "logical_GBps": round(logical / t_p / 1e9, 2)},
           "speedup": round(t_p / t_c, 3), "logical_bytes": int(logical), "unique_bytes": int(unique),
           "parity": {"sample_seqs": int(sp.num_seqs), "max_abs_err": float(err.max()),
                      "bound": "|gpu - ref| <= 0.002 + 0.01 |ref| per element",
                      "within_bound": bool(np.all(np.isfinite(got)) and np.all(err <= 2e-3 + 1e-2 * np.abs(ref)))},
           "peak": peak, "peak_kind": kind}
    del w, out_c, out_p, ws_c, ws_p
    torch.cuda.empty_cache()
    return res


def run_prefill(args, dev, B):
    evict = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev).fill_(1.0)
    res = prefill_measure(args.prefill_workload, args.steps or 30, dev, B, evict)
    line = {"metric": "prefill attention TFLOP/s (causal, algorithmic FLOPs)", "unit": "TFLOP/s",
            "value": res["attention"]["TFLOP/s"], "tokens_per_s": res["step"]["tokens_per_s"],
            "attention": res["attention"], "step": res["step"], "flops": res["flops"],
            "new_tokens": res["new_tokens"], "bound": "tensor", "check": res["check"], "higher_is_better": True,
            "timing": "each variant captured once as a CUDA graph, median of replays after an L2 eviction",
            "config": {"workload": res["workload"]}, "op": "prefill", "n_gpus": 1, "dtype": "bf16",
            "data": "synthetic"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for about 1.5 s of device time)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, choices=list(W.SPECS),
                    help="the workload to time (default mha13b, the headline, followed by every other "
                         "configuration in a 'configs' object)")
    ap.add_argument("--config-steps", type=int, default=300, help="timed steps per extra configuration")
    ap.add_argument("--config-cpu-seconds", type=float, default=3.0,
                    help="oracle seconds per extra configuration's cpu_baseline")
    ap.add_argument("--no-configs", action="store_true", help="time the headline workload only")
    ap.add_argument("--partition-tokens", type=int, default=None)
    ap.add_argument("--dtype", choices=["bf16", "f32"], default=None,
                    help="cache dtype (default: the workload's own); f32 runs the fp32 path")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-workload", default="prefill13b", choices=list(W.PREFILL_SPECS))
    ap.add_argument("--op", choices=["step", "swap", "append_layers", "shared_prefix", "prefill"], default="step",
                    help="step: the decode step (the benchmark line); swap / append_layers: secondary measurements")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.impl == "reference" and args.steps is None:
        args.steps = 5
    args.all_configs = (args.workload is None and not args.no_configs and args.partition_tokens is None
                        and args.dtype is None)
    if args.workload is None:
        args.workload = "mha13b"
    rank, world, local, dist = dist_setup(args)
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world, dist)
        elif args.op != "step":
            run_op(args, rank, world, local, dist)
        else:
            run_ours(args, rank, world, local, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
