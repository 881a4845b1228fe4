"""Seeded synthetic inputs for paged decode.

This module holds no part of the method's arithmetic: it draws context
lengths, lays sequences out on a shuffled physical block pool, fills the
caches with N(0, 1) values rounded to the storage dtype, poisons everything a
correct kernel must never read with NaN, and lists the KV-append slots and the
copy-on-write pairs of one decode step.  Both the CUDA path and the oracle
consume what it produces; neither is imported here.

Workloads (the shapes of the pages' serving scenarios: 13B-class heads,
right-skewed context lengths, shared prompts for parallel sampling):

=================  =====  =========  ====  =====  ===================================
name               seqs   Hq / Hkv   d     dtype  context lengths
=================  =====  =========  ====  =====  ===================================
tiny               4      8 / 8      64    f32    uniform int [1, 64]; pool 32 blocks
mha13b             64     40 / 40    128   bf16   lognormal(ln 400, 1.0) in [16, 2048];
                                                  pool 8192 blocks
gqa8b              256    32 / 8     128   bf16   lognormal(ln 1000, 0.8) in [32, 4096];
                                                  pool 1.1x the blocks needed
parallel_sampling  128    40 / 40    128   bf16   32 prompts x 4 samples, prompt 1000
                                                  tokens + suffix uniform [0, 256]
long_context       8      64 / 8     128   bf16   uniform int [32768, 131072];
                                                  512-token partitions
=================  =====  =========  ====  =====  ===================================

One decode step of a workload = copy-on-write block copies (``cow_pairs``),
then the KV append of this step's tokens (``slot_mapping``, ``k_new``,
``v_new``), then attention over ``context_lens`` tokens (which include the
appended ones).  Before the step, every slot the append will write and every
copy-on-write destination block hold NaN, so a skipped write shows up.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                      # "f32" or "bf16"
    lengths: str                    # recipe: "uniform", "lognormal", "sampling"
    len_lo: int
    len_hi: int
    len_median: float = 0.0         # lognormal median
    len_sigma: float = 0.0          # lognormal sigma
    pool_blocks: int = 0            # fixed pool size, 0 = pool_factor x needed
    pool_factor: float = 1.1
    partition_tokens: int = 0       # 0 = library heuristic
    seed: int = 0
    # parallel sampling
    num_prompts: int = 0
    samples_per_prompt: int = 0
    prompt_len: int = 0
    # extra copy pairs (tiny workload: two pairs into free blocks)
    extra_copy_pairs: int = 0
    # lengths recipe "explicit": one context length per sequence
    lengths_list: tuple = ()


SPECS = {
    "tiny": WorkloadSpec("tiny", 4, 8, 8, 64, "f32", "uniform", 1, 64, pool_blocks=32, seed=1001,
                         extra_copy_pairs=2),
    "mha13b": WorkloadSpec("mha13b", 64, 40, 40, 128, "bf16", "lognormal", 16, 2048, 400.0, 1.0,
                           pool_blocks=8192, seed=1002),
    "gqa8b": WorkloadSpec("gqa8b", 256, 32, 8, 128, "bf16", "lognormal", 32, 4096, 1000.0, 0.8,
                          pool_factor=1.1, seed=1003),
    "parallel_sampling": WorkloadSpec("parallel_sampling", 128, 40, 40, 128, "bf16", "sampling", 0, 256,
                                      pool_factor=1.1, seed=1004, num_prompts=32, samples_per_prompt=4,
                                      prompt_len=1000),
    "long_context": WorkloadSpec("long_context", 8, 64, 8, 128, "bf16", "uniform", 32768, 131072,
                                 pool_factor=1.1, partition_tokens=512, seed=1005),
}

# The bench workload and the order the configurations are usually listed in.
CONFIG_ORDER = ["tiny", "mha13b", "gqa8b", "parallel_sampling", "long_context"]


def spec(name: str, **overrides) -> WorkloadSpec:
    s = SPECS[name]
    if "lengths_list" in overrides:
        overrides.setdefault("lengths", "explicit")
        overrides.setdefault("num_seqs", len(overrides["lengths_list"]))
    s = dataclasses.replace(s, **overrides) if overrides else s
    if s.lengths == "sampling" and s.num_seqs != s.num_prompts * s.samples_per_prompt:
        s = dataclasses.replace(s, num_seqs=s.num_prompts * s.samples_per_prompt)
    return s


@dataclass
class Layout:
    """Host-side description of one decode step (numpy)."""
    spec: WorkloadSpec
    context_lens: np.ndarray          # int32 [S], after this step's append
    block_tables: np.ndarray          # int32 [S, maxB], unused entries -> a poisoned block
    num_blocks: int
    slot_mapping: np.ndarray          # int64 [T]
    cow_pairs: np.ndarray             # int64 [n, 2] (src, dst)
    used_blocks: np.ndarray           # bool [NB]: referenced by some table after the step
    valid_tokens: np.ndarray          # int32 [NB]: tokens a reader may read in each block
    poison_slots: list = field(default_factory=list)   # (block, first_slot) pairs: NaN from slot on
    # sequences sharing leading blocks (parallel sampling): int32 [groups, members] and [groups]
    group_members: np.ndarray = field(default_factory=lambda: np.zeros((0, 1), dtype=np.int32))
    shared_blocks: np.ndarray = field(default_factory=lambda: np.zeros((0,), dtype=np.int32))

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0

    def kv_bytes(self, elem_bytes: int) -> int:
        """Algorithmic K+V bytes one attention pass reads (every sequence's
        context, shared blocks counted once per reader)."""
        s = self.spec
        return int(self.context_lens.astype(np.int64).sum()) * s.num_kv_heads * s.head_dim * 2 * elem_bytes

    def unique_kv_bytes(self, elem_bytes: int) -> int:
        """K+V bytes of the distinct valid tokens read (shared blocks once)."""
        s = self.spec
        return int(self.valid_tokens.astype(np.int64).sum()) * s.num_kv_heads * s.head_dim * 2 * elem_bytes


def _lengths(sp: WorkloadSpec, rng: np.random.Generator) -> np.ndarray:
    if sp.lengths == "explicit":
        if len(sp.lengths_list) != sp.num_seqs:
            raise ValueError("lengths_list must hold one length per sequence")
        return np.array(sp.lengths_list, dtype=np.int64)
    if sp.lengths == "uniform":
        return rng.integers(sp.len_lo, sp.len_hi + 1, size=sp.num_seqs).astype(np.int64)
    if sp.lengths == "lognormal":
        raw = rng.lognormal(mean=math.log(sp.len_median), sigma=sp.len_sigma, size=sp.num_seqs)
        return np.clip(np.rint(raw), sp.len_lo, sp.len_hi).astype(np.int64)
    raise ValueError(sp.lengths)


def _blocks_for(n: int) -> int:
    return -(-n // BLOCK_SIZE)


def make_layout(sp: WorkloadSpec) -> Layout:
    rng = np.random.default_rng(sp.seed)
    if sp.lengths == "sampling":
        return _sampling_layout(sp, rng)
    lens = _lengths(sp, rng)
    need = np.array([_blocks_for(int(n)) for n in lens], dtype=np.int64)
    total = int(need.sum())
    nb = sp.pool_blocks or int(math.ceil(sp.pool_factor * total))
    nb = max(nb, total + 1 + sp.extra_copy_pairs)       # keep free blocks for poison and copies
    perm = rng.permutation(nb)
    max_b = int(need.max()) if need.size else 1
    tables = np.empty((sp.num_seqs, max(max_b, 1)), dtype=np.int64)
    used = np.zeros(nb, dtype=bool)
    valid = np.zeros(nb, dtype=np.int64)
    pos = 0
    for s in range(sp.num_seqs):
        ids = perm[pos:pos + need[s]]
        pos += need[s]
        tables[s, :need[s]] = ids
        used[ids] = True
        valid[ids] = BLOCK_SIZE
        if need[s]:
            valid[ids[-1]] = int(lens[s]) - BLOCK_SIZE * (need[s] - 1)
    free = perm[pos:]
    poison_block = int(free[0])
    for s in range(sp.num_seqs):
        tables[s, need[s]:] = poison_block
    # this step appends each sequence's last token
    slots = []
    poison = []
    for s in range(sp.num_seqs):
        n = int(lens[s])
        if n == 0:
            continue
        b = int(tables[s, (n - 1) // BLOCK_SIZE])
        slots.append(b * BLOCK_SIZE + (n - 1) % BLOCK_SIZE)
        poison.append((b, (n - 1) % BLOCK_SIZE))       # last token and the tail: NaN before the step
    pairs = np.zeros((0, 2), dtype=np.int64)
    if sp.extra_copy_pairs:
        src = tables[:sp.extra_copy_pairs, 0]
        dst = free[1:1 + sp.extra_copy_pairs]
        pairs = np.stack([src, dst], axis=1).astype(np.int64)
    return Layout(sp, lens.astype(np.int32), tables.astype(np.int32), nb, np.array(slots, dtype=np.int64),
                  pairs, used, valid.astype(np.int32), poison)


def _sampling_layout(sp: WorkloadSpec, rng: np.random.Generator) -> Layout:
    """Parallel sampling: every prompt's blocks are shared by its samples; the
    partly filled last prompt block is copied on write by each sample that
    writes into it while another reference to it remains (the last writer
    writes in place); samples that have not generated still share it."""
    P, G, L = sp.num_prompts, sp.samples_per_prompt, sp.prompt_len
    S = P * G
    suffix = rng.integers(sp.len_lo, sp.len_hi + 1, size=S).astype(np.int64)
    lens = L + suffix
    tail = L % BLOCK_SIZE
    prompt_blocks = _blocks_for(L)
    # blocks needed: prompt blocks once per prompt, at most one copy per sample,
    # and each sample's blocks past the prompt
    past_prompt = sum(max(0, _blocks_for(int(n)) - prompt_blocks) for n in lens)
    total = P * prompt_blocks + S + past_prompt
    nb = int(math.ceil(sp.pool_factor * total)) + 1
    perm = list(rng.permutation(nb))
    max_b = int(max(_blocks_for(int(n)) for n in lens))
    tables = np.empty((S, max_b), dtype=np.int64)
    used = np.zeros(nb, dtype=bool)
    valid = np.zeros(nb, dtype=np.int64)
    pairs, slots, poison = [], [], []
    cursor = 0

    def take():
        nonlocal cursor
        b = int(perm[cursor])
        cursor += 1
        return b

    for p in range(P):
        pblocks = [take() for _ in range(prompt_blocks)]
        members = list(range(p * G, (p + 1) * G))
        for s in members:
            tables[s, :prompt_blocks] = pblocks
        for b in pblocks:
            used[b] = True
            valid[b] = BLOCK_SIZE
        if tail:
            shared = pblocks[-1]
            valid[shared] = tail
            poison.append((shared, tail))
            refs = len(members)
            for s in members:
                if suffix[s] == 0:
                    continue
                if refs > 1:
                    dst = take()
                    pairs.append((shared, dst))
                    poison.append((dst, 0))                # fresh block: NaN until the copy
                    tables[s, prompt_blocks - 1] = dst
                    used[dst] = True
                    refs -= 1
                    blk = dst
                else:
                    blk = shared                           # last reference: write in place
                # tokens of this sample that land in the copied block are appended this step
                last_in_blk = min(int(lens[s]), prompt_blocks * BLOCK_SIZE)
                for t in range(L, last_in_blk):
                    slots.append(blk * BLOCK_SIZE + t % BLOCK_SIZE)
                valid[blk] = max(valid[blk], last_in_blk - (prompt_blocks - 1) * BLOCK_SIZE)
        for s in members:
            n = int(lens[s])
            nblk = _blocks_for(n)
            for j in range(prompt_blocks, nblk):
                b = take()
                tables[s, j] = b
                used[b] = True
                valid[b] = min(BLOCK_SIZE, n - j * BLOCK_SIZE)
            if nblk > prompt_blocks:
                b = int(tables[s, nblk - 1])
                slots.append(b * BLOCK_SIZE + (n - 1) % BLOCK_SIZE)
                poison.append((b, (n - 1) % BLOCK_SIZE))
    free = [int(b) for b in perm[cursor:]]
    poison_block = free[0]
    for s in range(S):
        tables[s, _blocks_for(int(lens[s])):] = poison_block
    groups = np.arange(S, dtype=np.int32).reshape(P, G)
    shared = np.full(P, L // BLOCK_SIZE, dtype=np.int32)      # the full prompt blocks every sample shares
    return Layout(sp, lens.astype(np.int32), tables.astype(np.int32), nb, np.array(slots, dtype=np.int64),
                  np.array(pairs, dtype=np.int64).reshape(-1, 2), used, valid.astype(np.int32), poison, groups, shared)


TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}
NAN_BITS = {"f32": 0x7FC00000, "bf16": 0x7FC0}


@dataclass
class Workload:
    """Tensors of one decode step, on ``device``; see the module docstring."""
    layout: Layout
    q: torch.Tensor               # [S, Hq, d]
    k_cache: torch.Tensor         # [NB, Hkv, 16, d], state before the step
    v_cache: torch.Tensor
    k_new: torch.Tensor           # [T, Hkv, d]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor    # int64 [T]
    block_tables: torch.Tensor    # int32 [S, maxB]
    context_lens: torch.Tensor    # int32 [S]
    cow_pairs: torch.Tensor       # int64 [n, 2]
    scale: float

    @property
    def spec(self) -> WorkloadSpec:
        return self.layout.spec

    def to(self, device) -> "Workload":
        f = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in self.__dict__.items()}
        return Workload(**f)


def _randn(shape, dtype, gen, device, chunk_elems=1 << 27):
    """N(0,1) rounded to ``dtype``, drawn in chunks so the fp32 temporary stays small."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for lo in range(0, n, chunk_elems):
        hi = min(n, lo + chunk_elems)
        flat[lo:hi] = torch.randn(hi - lo, generator=gen, device=device, dtype=torch.float32).to(dtype)
    return out


def _nan_fill(t: torch.Tensor, dtype_name: str):
    if dtype_name == "bf16":
        t.view(torch.int16).fill_(NAN_BITS["bf16"])
    else:
        t.view(torch.int32).fill_(NAN_BITS["f32"])


def make_workload(name_or_spec, device="cpu", **overrides) -> Workload:
    sp = spec(name_or_spec, **overrides) if isinstance(name_or_spec, str) else name_or_spec
    lay = make_layout(sp)
    dt = TORCH_DTYPE[sp.dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(sp.seed)
    S, Hq, Hkv, d = sp.num_seqs, sp.num_q_heads, sp.num_kv_heads, sp.head_dim
    q = _randn((S, Hq, d), dt, gen, device)
    k_cache = _randn((lay.num_blocks, Hkv, BLOCK_SIZE, d), dt, gen, device)
    v_cache = _randn((lay.num_blocks, Hkv, BLOCK_SIZE, d), dt, gen, device)
    T = lay.slot_mapping.shape[0]
    k_new = _randn((T, Hkv, d), dt, gen, device)
    v_new = _randn((T, Hkv, d), dt, gen, device)
    # poison: unreferenced blocks, tails past the readable tokens, append targets, copy destinations
    unused = torch.from_numpy(np.nonzero(~lay.used_blocks)[0]).to(device)
    for c in (k_cache, v_cache):
        if unused.numel():
            sub = c.index_select(0, unused)
            _nan_fill(sub, sp.dtype)
            c.index_copy_(0, unused, sub)
        for b, first in lay.poison_slots:
            _nan_fill(c[b, :, first:, :], sp.dtype)
    return Workload(
        layout=lay, q=q, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        slot_mapping=torch.from_numpy(lay.slot_mapping.copy()).to(device),
        block_tables=torch.from_numpy(lay.block_tables.copy()).to(device),
        context_lens=torch.from_numpy(lay.context_lens.copy()).to(device),
        cow_pairs=torch.from_numpy(lay.cow_pairs.copy()).to(device),
        scale=1.0 / math.sqrt(d),
    )


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """CPU numpy view of a tensor; bf16 comes back as uint16 bit patterns."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def from_numpy_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    """Inverse of ``to_numpy``: uint16 arrays are read as bf16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(a.copy()).to(device)


# ---- prefill steps ------------------------------------------------------------------------
#
# A prefill step writes n_s new tokens per sequence into the cache (a whole
# prompt, or a chunk of one after `prior` tokens already cached) and attends
# each new token causally over the sequence's tokens up to itself.
#
# =============  =====  =========  ====  =====================================  ==================
# name           seqs   Hq / Hkv   d     new tokens n_s                         prior context
# =============  =====  =========  ====  =====================================  ==================
# prefill13b     32     40 / 40    128   lognormal(ln 500, 0.8) in [16, 2048]   0 (whole prompts)
# chunked_gqa    16     32 / 8     128   uniform int [1, 512]                   uniform [0, 2048]
# long_prefix    8      32 / 8     128   512 (one chunk)                        uniform [16384, 32768]
# =============  =====  =========  ====  =====================================  ==================

@dataclass(frozen=True)
class PrefillSpec:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    new_lengths: str                # "lognormal", "uniform" or "explicit"
    new_lo: int
    new_hi: int
    new_median: float = 0.0
    new_sigma: float = 0.0
    prior_lo: int = 0
    prior_hi: int = 0
    pool_factor: float = 1.1
    seed: int = 0
    new_list: tuple = ()            # explicit n_s
    prior_list: tuple = ()          # explicit prior context (with new_list)


PREFILL_SPECS = {
    "prefill13b": PrefillSpec("prefill13b", 32, 40, 40, 128, "lognormal", 16, 2048, 500.0, 0.8, seed=2001),
    "chunked_gqa": PrefillSpec("chunked_gqa", 16, 32, 8, 128, "uniform", 1, 512, prior_lo=0, prior_hi=2048,
                               seed=2002),
    "long_prefix": PrefillSpec("long_prefix", 8, 32, 8, 128, "uniform", 512, 512, prior_lo=16384,
                               prior_hi=32768, seed=2003),
}


@dataclass
class PrefillWorkload:
    """One prefill step, on ``device``: kv_append of ``k_new``/``v_new`` at
    ``slot_mapping`` (every new token of every sequence, in query order), then
    causal attention of ``q`` over the cache."""
    spec: PrefillSpec
    q: torch.Tensor               # bf16 [T, Hq, d]
    k_cache: torch.Tensor         # bf16 [NB, Hkv, 16, d]; new-token slots NaN before the append
    v_cache: torch.Tensor
    k_new: torch.Tensor           # bf16 [T, Hkv, d]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor    # int64 [T]
    block_tables: torch.Tensor    # int32 [S, maxB]
    context_lens: torch.Tensor    # int32 [S] = prior + n_s
    query_start: torch.Tensor     # int32 [S + 1]
    scale: float
    host: dict                    # numpy copies of the index arrays

    @property
    def max_query_len(self) -> int:
        n = np.diff(self.host["query_start"])
        return int(n.max()) if n.size else 0

    @property
    def max_context_len(self) -> int:
        return int(self.host["context_lens"].max()) if self.host["context_lens"].size else 0

    def pairs(self) -> int:
        """(query, key) pairs the causal attention scores, per query head."""
        n = np.diff(self.host["query_start"]).astype(np.int64)
        prior = self.host["context_lens"].astype(np.int64) - n
        return int(np.sum(n * prior + n * (n + 1) // 2))

    def flops(self) -> int:
        """Algorithmic FLOPs: 2 d for q.k and 2 d for p v per scored pair and query head."""
        return 4 * self.spec.head_dim * self.spec.num_q_heads * self.pairs()

    def to(self, device) -> "PrefillWorkload":
        f = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in self.__dict__.items()}
        return PrefillWorkload(**f)


def prefill_spec(name: str, **overrides) -> PrefillSpec:
    s = PREFILL_SPECS[name]
    if "new_list" in overrides:
        overrides.setdefault("new_lengths", "explicit")
        overrides.setdefault("num_seqs", len(overrides["new_list"]))
    return dataclasses.replace(s, **overrides) if overrides else s


def make_prefill(name_or_spec, device="cpu", **overrides) -> PrefillWorkload:
    sp = prefill_spec(name_or_spec, **overrides) if isinstance(name_or_spec, str) else name_or_spec
    rng = np.random.default_rng(sp.seed)
    S = sp.num_seqs
    if sp.new_lengths == "explicit":
        new = np.array(sp.new_list, dtype=np.int64)
        prior = np.array(sp.prior_list or (0,) * S, dtype=np.int64)
        if len(new) != S or len(prior) != S:
            raise ValueError("new_list and prior_list need one entry per sequence")
    else:
        if sp.new_lengths == "lognormal":
            raw = rng.lognormal(mean=math.log(sp.new_median), sigma=sp.new_sigma, size=S)
            new = np.clip(np.rint(raw), sp.new_lo, sp.new_hi).astype(np.int64)
        elif sp.new_lengths == "uniform":
            new = rng.integers(sp.new_lo, sp.new_hi + 1, size=S).astype(np.int64)
        else:
            raise ValueError(sp.new_lengths)
        prior = rng.integers(sp.prior_lo, sp.prior_hi + 1, size=S).astype(np.int64)
    lens = prior + new
    need = np.array([_blocks_for(int(n)) for n in lens], dtype=np.int64)
    total = int(need.sum())
    nb = max(int(math.ceil(sp.pool_factor * total)), total + 1)
    perm = rng.permutation(nb)
    max_b = max(int(need.max()) if S else 1, 1)
    tables = np.empty((S, max_b), dtype=np.int64)
    used = np.zeros(nb, dtype=bool)
    pos = 0
    for s in range(S):
        tables[s, :need[s]] = perm[pos:pos + need[s]]
        used[perm[pos:pos + need[s]]] = True
        pos += need[s]
    poison_block = int(perm[pos])
    for s in range(S):
        tables[s, need[s]:] = poison_block
    slots = []
    for s in range(S):
        for t in range(int(prior[s]), int(lens[s])):
            slots.append(int(tables[s, t // BLOCK_SIZE]) * BLOCK_SIZE + t % BLOCK_SIZE)
    slots = np.array(slots, dtype=np.int64)
    qs = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    T = int(qs[-1])
    gen = torch.Generator(device=device)
    gen.manual_seed(sp.seed)
    Hq, Hkv, d = sp.num_q_heads, sp.num_kv_heads, sp.head_dim
    dt = torch.bfloat16
    q = _randn((T, Hq, d), dt, gen, device)
    k_cache = _randn((nb, Hkv, BLOCK_SIZE, d), dt, gen, device)
    v_cache = _randn((nb, Hkv, BLOCK_SIZE, d), dt, gen, device)
    k_new = _randn((T, Hkv, d), dt, gen, device)
    v_new = _randn((T, Hkv, d), dt, gen, device)
    # poison: unreferenced blocks, slots past each sequence's end, the new tokens' slots
    unused = torch.from_numpy(np.nonzero(~used)[0]).to(device)
    for c in (k_cache, v_cache):
        if unused.numel():
            sub = c.index_select(0, unused)
            _nan_fill(sub, "bf16")
            c.index_copy_(0, unused, sub)
        for s in range(S):
            if lens[s] % BLOCK_SIZE:
                _nan_fill(c[int(tables[s, need[s] - 1]), :, int(lens[s] % BLOCK_SIZE):, :], "bf16")
        if slots.size:
            flat = c.view(nb * 1, Hkv, BLOCK_SIZE, d)
            idx = torch.from_numpy(slots).to(device)
            blk, off = idx // BLOCK_SIZE, idx % BLOCK_SIZE
            flat[blk, :, off, :] = float("nan")
    host = {"block_tables": tables.astype(np.int32), "context_lens": lens.astype(np.int32), "query_start": qs,
            "slot_mapping": slots, "num_blocks": nb}
    return PrefillWorkload(
        spec=sp, q=q, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        slot_mapping=torch.from_numpy(slots.copy()).to(device),
        block_tables=torch.from_numpy(host["block_tables"].copy()).to(device),
        context_lens=torch.from_numpy(host["context_lens"].copy()).to(device),
        query_start=torch.from_numpy(qs.copy()).to(device),
        scale=1.0 / math.sqrt(d), host=host)
