"""Seeded synthetic inputs for the decode-attention and gather workloads.

This module is shared by both sides of every comparison: it feeds the CPU oracle
and the CUDA path the same numbers. It holds workload recipes and random draws
only -- no softmax, no paging arithmetic, no planning. Every draw comes from a
NumPy PCG64 generator with an explicit seed.

Workload shapes (model head counts and context lengths) follow the pages:
Qwen3-4B and Qwen2.5-32B shapes from "Tangram: Unlocking Non-Uniform KV Cache
for Efficient Multi-turn LLM Serving" (Figs. 1, 5, 6, 11), the fragmented
block pool from "KV-RM: Regularizing KV-Cache Movement for Static-Graph LLM
Serving" (Figs. 1-3), and batch 8 x 122k sparse decode with Llama-3-8B shapes
from "KVDrive" (Fig. 5). The datasets those pages use are not needed: values
are N(0, 1) rounded to the storage type.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

FULL = 1 << 30  # a budget this large keeps every token of any sequence


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------- rounding
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even);
    returns the 16-bit patterns. NaN stays NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 array holding values exactly representable in `dtype`."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))
    raise ValueError(dtype)


def normal(g: np.random.Generator, shape, dtype: str) -> np.ndarray:
    return round_to(g.standard_normal(shape, dtype=np.float64).astype(np.float32), dtype)


# ---------------------------------------------------------- kept-set draws
def kept_random(g: np.random.Generator, L: int, n: int) -> np.ndarray:
    """A seeded random set of n positions of [0, L), ascending."""
    if n >= L:
        return np.arange(L, dtype=np.int32)
    return np.sort(g.choice(L, size=n, replace=False)).astype(np.int32)


def kept_sink_recent(L: int, sinks: int, recent: int) -> np.ndarray:
    """The first `sinks` and the last `recent` positions (union, ascending)."""
    s = set(range(min(sinks, L))) | set(range(max(0, L - recent), L))
    return np.array(sorted(s), dtype=np.int32)


# ----------------------------------------------------------- dense cases
@dataclass
class DenseCase:
    """A decode-attention problem held densely: every head of every sequence
    has K/V rows for all positions, plus the set of positions it keeps."""
    B: int
    Hq: int
    Hkv: int
    D: int
    dtype: str
    seq_len: np.ndarray            # int32 [B]
    q: np.ndarray                  # float32 [B][Hq][D] (values of `dtype`)
    k: np.ndarray                  # float32 [B][Hkv][Lmax][D]
    v: np.ndarray                  # float32 [B][Hkv][Lmax][D]
    kept: list                     # B*Hkv arrays of kept positions
    budget: np.ndarray             # int32 [B][Hkv] budget handed to the library
    head_group: np.ndarray         # int32 [Hkv]
    P: int = 16
    meta: dict = field(default_factory=dict)

    @property
    def n(self) -> np.ndarray:
        return np.array([len(x) for x in self.kept], dtype=np.int32).reshape(self.B, self.Hkv)


def dense_case(B, Hq, Hkv, D, seq_len, n_keep, dtype="bf16", seed=0, P=16,
               head_group=None, full_budget=FULL, kept_mode="random"):
    """Dense seeded case. n_keep: [B][Hkv] kept counts (values >= L mean 'all';
    those heads get `full_budget` as their library budget).
    Draw order: q, k, v, then kept sets (b-major, h-minor)."""
    g = rng(seed)
    seq_len = np.asarray(seq_len, dtype=np.int32)
    Lmax = int(seq_len.max())
    q = normal(g, (B, Hq, D), dtype)
    k = normal(g, (B, Hkv, Lmax, D), dtype)
    v = normal(g, (B, Hkv, Lmax, D), dtype)
    kept, budget = [], np.zeros((B, Hkv), dtype=np.int32)
    n_keep = np.asarray(n_keep).reshape(B, Hkv)
    for b in range(B):
        L = int(seq_len[b])
        for h in range(Hkv):
            n = int(n_keep[b, h])
            if n >= L:
                kept.append(np.arange(L, dtype=np.int32))
                budget[b, h] = full_budget
            else:
                kept.append(kept_random(g, L, n) if kept_mode == "random"
                            else np.arange(L - n, L, dtype=np.int32))
                budget[b, h] = n
    if head_group is None:
        head_group = np.arange(Hkv, dtype=np.int32)
    return DenseCase(B, Hq, Hkv, D, dtype, seq_len, q, k, v, kept, budget,
                     np.asarray(head_group, dtype=np.int32), P)


def tiny(seed=0, grouping="per_head"):
    """1 layer, 4 query / 2 KV heads, head_dim 64, batch 2, seq_len {37, 100};
    KV head 0 keeps everything, KV head 1 keeps the first 4 (sink) and the 16
    most recent tokens; page 16; fp32 N(0,1). grouping: 'per_head' gives the
    groups {h0}, {h1}; 'one' puts both heads in one group."""
    B, Hq, Hkv, D = 2, 4, 2, 64
    seq_len = np.array([37, 100], dtype=np.int32)
    g = rng(seed)
    Lmax = 100
    q = normal(g, (B, Hq, D), "f32")
    k = normal(g, (B, Hkv, Lmax, D), "f32")
    v = normal(g, (B, Hkv, Lmax, D), "f32")
    kept, budget = [], np.zeros((B, Hkv), dtype=np.int32)
    for b in range(B):
        L = int(seq_len[b])
        kept.append(np.arange(L, dtype=np.int32))
        budget[b, 0] = FULL
        ks = kept_sink_recent(L, 4, 16)
        kept.append(ks)
        budget[b, 1] = len(ks)
    hg = np.array([0, 1] if grouping == "per_head" else [0, 0], dtype=np.int32)
    return DenseCase(B, Hq, Hkv, D, "f32", seq_len, q, k, v, kept, budget, hg, 16,
                     meta={"name": "tiny", "grouping": grouping})


# ------------------------------------------------- decode config recipes
@dataclass
class DecodeConfig:
    """Shapes, sequence lengths, per-layer budgets and head groups of one
    decode workload. Token values are drawn separately (see value_table)."""
    name: str
    layers: int
    B: int
    Hq: int
    Hkv: int
    D: int
    P: int
    dtype: str
    seq_len: np.ndarray     # int32 [B]
    n: np.ndarray           # int32 [layers][B][Hkv] kept tokens per head
    budget: np.ndarray      # int32 [layers][B][Hkv] budget handed to the library
    head_group: np.ndarray  # int32 [layers][Hkv]
    num_groups: int
    note: str = ""

    def kv_bytes_layer(self, layer: int) -> int:
        """Algorithmic KV bytes of one layer: kept tokens x (K+V) x D x dtype."""
        es = 2 if self.dtype == "bf16" else 4
        return int(self.n[layer].astype(np.int64).sum()) * 2 * self.D * es

    def kv_bytes_step(self) -> int:
        return sum(self.kv_bytes_layer(l) for l in range(self.layers))


def groups_by_budget(rate: np.ndarray, cuts) -> np.ndarray:
    """Sort KV heads by retention rate (descending; ties to the lower head id)
    and cut the ranking into contiguous groups of the given sizes."""
    order = sorted(range(len(rate)), key=lambda h: (-rate[h], h))
    hg = np.zeros(len(rate), dtype=np.int32)
    pos = 0
    for gi, c in enumerate(cuts):
        for h in order[pos:pos + c]:
            hg[h] = gi
        pos += c
    return hg


def regroup(cfg: "DecodeConfig", heads_per_group: int) -> "DecodeConfig":
    """The same workload with head groups of `heads_per_group` KV heads each:
    per layer, heads sorted by retention (descending, ties to the lower id) and
    cut into equal groups. heads_per_group = Hkv is one unified page over all
    heads; 1 gives every head its own page table."""
    import copy
    G = heads_per_group
    if cfg.Hkv % G:
        raise ValueError("heads_per_group must divide Hkv")
    out = copy.copy(cfg)
    hg = np.zeros_like(cfg.head_group)
    for layer in range(cfg.layers):
        rate = cfg.n[layer].astype(np.float64).sum(0) / cfg.seq_len.astype(np.float64).sum()
        hg[layer] = groups_by_budget(rate, [G] * (cfg.Hkv // G))
    out.head_group = hg
    out.num_groups = cfg.Hkv // G
    out.name = f"{cfg.name}_G{G}"
    return out


def _rate_to_count(rate: float, L: int) -> int:
    return min(L, max(1, int(math.ceil(rate * L))))


def decode_config(name: str, seed: int = 0, layers: int | None = None,
                  batch: int | None = None) -> DecodeConfig:
    """Recipes of the decode workloads:

    qwen3_4b      36 layers, 32/8 heads, D 128, bf16, batch 16, L ~ U{8192..32768};
                  per layer 2 random KV heads keep everything, the other 6 keep a
                  rate ~ U[0.10, 0.50] of each sequence; 3 groups [2|3|3]; page 16.
    qwen3_4b_32k  the same with every L = 32768.
    qwen25_32b    64 layers, 40/8 heads, D 128, bf16, batch 64,
                  L = clip(round(exp(N(ln 4096, 1))), 16, 65536), L[0] = 65536;
                  per layer 4 random KV heads keep everything, 4 keep 12.5%;
                  4 groups of 2; page 32.
    llama3_sparse 32 layers, 32/8 heads, D 128, bf16, batch 8, L = 122000,
                  every head keeps 2176 tokens (top 2048 by score + 128 recent);
                  one group; page 16.
    tiny          1 layer, 4/2 heads, D 64, fp32, batch 2, L {37, 100}; KV head 0
                  keeps everything, KV head 1 keeps 20 tokens (4 sink + 16
                  recent); groups {h0}, {h1}; page 16 (the shapes of tiny()).
    """
    if name == "tiny":
        L = np.array([37, 100], dtype=np.int32)
        n = np.array([[[37, 20], [100, 20]]], dtype=np.int32)
        budget = np.array([[[FULL, 20], [FULL, 20]]], dtype=np.int32)
        hg = np.array([[0, 1]], dtype=np.int32)
        if layers and layers > 1:
            n, budget, hg = (np.repeat(a, layers, axis=0) for a in (n, budget, hg))
        return DecodeConfig("tiny", layers or 1, 2, 4, 2, 64, 16, "f32", L, n, budget, hg, 2)
    g = rng(seed)
    if name in ("qwen3_4b", "qwen3_4b_32k"):
        nl, B, Hq, Hkv, D, P = 36, 16, 32, 8, 128, 16
        B = batch or B
        if name == "qwen3_4b":
            L = g.integers(8192, 32768, size=B, endpoint=True).astype(np.int32)
        else:
            L = np.full(B, 32768, dtype=np.int32)
        cuts = [2, 3, 3]
    elif name == "qwen25_32b":
        nl, B, Hq, Hkv, D, P = 64, 64, 40, 8, 128, 32
        B = batch or B
        L = np.clip(np.round(np.exp(g.normal(math.log(4096.0), 1.0, size=B))), 16,
                    65536).astype(np.int32)
        L[0] = 65536
        cuts = [2, 2, 2, 2]
    elif name == "llama3_sparse":
        nl, B, Hq, Hkv, D, P = 32, 8, 32, 8, 128, 16
        B = batch or B
        L = np.full(B, 122000, dtype=np.int32)
        cuts = [8]
    else:
        raise ValueError(name)
    nl = layers or nl
    n = np.zeros((nl, B, Hkv), dtype=np.int32)
    budget = np.zeros_like(n)
    hg = np.zeros((nl, Hkv), dtype=np.int32)
    for layer in range(nl):
        if name.startswith("qwen3_4b"):
            full = g.choice(Hkv, size=2, replace=False)
            rate = g.uniform(0.10, 0.50, size=Hkv)
            rate[full] = 1.0
        elif name == "qwen25_32b":
            full = g.choice(Hkv, size=4, replace=False)
            rate = np.full(Hkv, 0.125)
            rate[full] = 1.0
        else:
            rate = np.zeros(Hkv)
        for b in range(B):
            for h in range(Hkv):
                if name == "llama3_sparse":
                    n[layer, b, h] = min(int(L[b]), 2176)
                    budget[layer, b, h] = 2176
                elif rate[h] >= 1.0:
                    n[layer, b, h] = int(L[b])
                    budget[layer, b, h] = FULL
                else:
                    n[layer, b, h] = _rate_to_count(float(rate[h]), int(L[b]))
                    budget[layer, b, h] = n[layer, b, h]
        hg[layer] = groups_by_budget(rate, cuts)
    return DecodeConfig(name, nl, B, Hq, Hkv, D, P, "bf16", L, n, budget, hg, len(cuts))


# ------------------------------------------------------------ value table
def value_table(seed: int, n_elems: int, dtype: str = "bf16") -> np.ndarray:
    """A table of n_elems N(0,1) values rounded to dtype: uint16 bf16 patterns
    for 'bf16', float32 for 'f32'. Large pools are filled by tiling it."""
    g = rng(seed)
    x = g.standard_normal(n_elems, dtype=np.float32)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def tile_offsets(seed: int, count: int, table_len: int, align: int) -> np.ndarray:
    """Seeded start offsets (multiples of `align`) into a value table."""
    g = rng(seed)
    return (g.integers(0, table_len // align, size=count) * align).astype(np.int64)


def page_permutation(seed: int, total_pages: int) -> np.ndarray:
    """Seeded permutation of physical page ids (a fragmented pool)."""
    return rng(seed).permutation(total_pages).astype(np.int32)


# ---------------------------------------------------------- gather recipes
@dataclass
class GatherConfig:
    name: str
    S: int
    max_blocks: int
    nb: np.ndarray          # int32 [S] live blocks per sequence
    bt: np.ndarray          # int32 [S][max_blocks] physical ids (-1 past nb)
    num_phys: int
    block_bytes: int
    row_bytes: int
    seq_tokens: np.ndarray  # int32 [S]

    def live_bytes(self) -> int:
        return int(self.nb.astype(np.int64).sum()) * self.block_bytes


def gather_config(seed=0, S=256, Lmin=512, Lmax=16384, block_tokens=16,
                  token_bytes=8 * 128 * 2, num_phys=655360, extents=False,
                  max_extent=64) -> GatherConfig:
    """KV-RM movement workload: S sequences with lengths ~ U{Lmin..Lmax}
    tokens, blocks of `block_tokens` tokens x 8 KV heads x 128 dims bf16,
    each sequence's blocks drawn without replacement from a seeded random
    permutation of the pool (extents=False), or as extents of 1..max_extent
    physically consecutive blocks (extents=True)."""
    g = rng(seed)
    L = g.integers(Lmin, Lmax, size=S, endpoint=True).astype(np.int32)
    nb = ((L + block_tokens - 1) // block_tokens).astype(np.int32)
    max_blocks = Lmax // block_tokens
    bt = np.full((S, max_blocks), -1, dtype=np.int32)
    if not extents:
        perm = g.permutation(num_phys).astype(np.int32)
        if int(nb.sum()) > num_phys:
            raise ValueError("pool too small")
        pos = 0
        for s in range(S):
            bt[s, :nb[s]] = perm[pos:pos + nb[s]]
            pos += int(nb[s])
    else:
        nchunks = num_phys // max_extent
        chunks = g.permutation(nchunks)
        ci = 0
        for s in range(S):
            j = 0
            while j < nb[s]:
                ln = int(min(g.integers(1, max_extent, endpoint=True), nb[s] - j))
                base = int(chunks[ci]) * max_extent
                ci += 1
                bt[s, j:j + ln] = np.arange(base, base + ln, dtype=np.int32)
                j += ln
    return GatherConfig("kvrm_extents" if extents else "kvrm", S, max_blocks, nb, bt,
                        num_phys, block_tokens * token_bytes,
                        max_blocks * block_tokens * token_bytes, L)


def block_stamp_pool(num_phys: int, block_bytes: int, seed: int = 0) -> np.ndarray:
    """A small pool whose blocks are distinguishable: the first 8 bytes of each
    block hold its id (little-endian int64); the rest is seeded random bytes."""
    g = rng(seed)
    pool = g.integers(0, 256, size=(num_phys, block_bytes), dtype=np.uint8)
    ids = np.arange(num_phys, dtype=np.int64).view(np.uint8).reshape(num_phys, 8)
    pool[:, :8] = ids
    return pool
