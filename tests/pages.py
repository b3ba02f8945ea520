"""Test input preparation: lays dense kept rows out in head-group pages.

Layout ("Tangram: Unlocking Non-Uniform KV Cache for Efficient Multi-turn LLM
Serving", Fig. 8(b), Head Group Page): each head group G has its own pool of
pages, [pages][|G|][P][D] per K and per V, and its own page table per
sequence. All heads of a group walk the same pages; head h of G owns slot
row r(h) (its rank within G, ascending head order) of every page. Token t of
head (b, h) -- the head's t-th kept token in ascending position -- lives at
page page_table[G][b][t // P], row r(h), slot t % P. A page is laid out
[|G|][P][D] (head-major) or [P][|G|][D] (token-major, the block layout of
"KV-RM: Regularizing KV-Cache Movement for Static-Graph LLM Serving"). Slots
past a head's kept count are padding and are never read.

These helpers assign physical pages to sequences (any permutation of a group's
pages is valid: the result does not depend on where pages sit) and pack dense
kept rows into pools, following the page layout that the kvx C ABI documents
for kvx_decode_attn. They prepare GPU inputs for tests only: the library never
imports them, and the oracle never sees pages.
"""
from __future__ import annotations

import numpy as np


def head_rows(head_group: np.ndarray) -> np.ndarray:
    """Row of every KV head within its group (rank in ascending head order)."""
    hg = np.asarray(head_group, dtype=np.int32)
    rows = np.zeros_like(hg)
    seen: dict[int, int] = {}
    for h, g in enumerate(hg.tolist()):
        rows[h] = seen.get(g, 0)
        seen[g] = rows[h] + 1
    return rows


def group_sizes(head_group: np.ndarray) -> np.ndarray:
    hg = np.asarray(head_group, dtype=np.int32)
    return np.bincount(hg, minlength=int(hg.max()) + 1).astype(np.int32)


def assign_pages(group_pages: np.ndarray, perms=None, spare_pages: int = 0):
    """Page tables for every group.

    group_pages: int [G][B] pages each group needs per sequence.
    perms: optional list of G permutations of range(total pages of the group)
           (a fragmented pool); None keeps pages in order.
    Returns (page_tables, pool_pages): page_tables[g] is int32 [B][stride]
    with -1 past the pages a sequence uses; pool_pages[g] is the pool size.
    """
    gp = np.asarray(group_pages, dtype=np.int64)
    G, B = gp.shape
    tables, sizes = [], []
    for g in range(G):
        total = int(gp[g].sum()) + int(spare_pages)
        ids = np.arange(total, dtype=np.int32) if perms is None else np.asarray(perms[g],
                                                                                dtype=np.int32)
        if ids.size < int(gp[g].sum()):
            raise ValueError("permutation shorter than the pages needed")
        stride = max(1, int(gp[g].max()))
        pt = np.full((B, stride), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            k = int(gp[g, b])
            pt[b, :k] = ids[off:off + k]
            off += k
        tables.append(pt)
        sizes.append(max(total, 1))
    return tables, sizes


def pack_pools(k_dense, v_dense, kept, head_group, page_tables, pool_pages, P,
               out_dtype=np.float32, fill=np.nan, token_major=False):
    """Scatter dense kept rows into head-group pools.

    k_dense, v_dense: [B][Hkv][Lmax][D] arrays already holding values of the
    storage type; kept: B*Hkv index arrays (ascending positions kept by each
    head); out_dtype: np.float32, or np.uint16 for bf16 bit patterns (then
    k_dense / v_dense must be uint16 too). Padding slots get `fill`.
    Returns a list of (k_pool, v_pool), each [pool_pages][|G|][P][D]
    (head-major) or [pool_pages][P][|G|][D] (token_major=True).
    """
    B, Hkv, _, D = k_dense.shape
    hg = np.asarray(head_group, dtype=np.int32)
    rows, sizes = head_rows(hg), group_sizes(hg)
    pools = []
    for g in range(len(page_tables)):
        shape = ((pool_pages[g], P, int(sizes[g]), D) if token_major
                 else (pool_pages[g], int(sizes[g]), P, D))
        if out_dtype == np.uint16:
            fillv = np.uint16(0x7FC0) if (isinstance(fill, float) and np.isnan(fill)) else np.uint16(fill)
            kp = np.full(shape, fillv, dtype=np.uint16)
        else:
            kp = np.full(shape, fill, dtype=out_dtype)
        pools.append((kp, kp.copy()))
    for b in range(B):
        for h in range(Hkv):
            g, r = int(hg[h]), int(rows[h])
            ix = np.asarray(kept[b * Hkv + h])
            t = np.arange(ix.size)
            pages = page_tables[g][b, t // P]
            if np.any(pages < 0):
                raise ValueError("page table shorter than the kept tokens")
            kp, vp = pools[g]
            if token_major:
                kp[pages, t % P, r] = k_dense[b, h, ix]
                vp[pages, t % P, r] = v_dense[b, h, ix]
            else:
                kp[pages, r, t % P] = k_dense[b, h, ix]
                vp[pages, r, t % P] = v_dense[b, h, ix]
    return pools
