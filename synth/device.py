"""Materialise large synthetic pools on the GPU from a seeded value table.

Full-size workloads (tens of GB) are not generated value by value on the
host. Instead a seeded table of N(0,1) values (bf16-rounded) is drawn once on
the host, uploaded, and every pool row is a row of that table picked by a
seeded offset: row i of a pool holds table row (shift + i) mod table_rows.
The host can therefore rebuild any row it wants to check from the same
table, without reading the GPU. Holds input generation only.
"""
from __future__ import annotations

import numpy as np
import torch

import synth


class ValueTable:
    def __init__(self, seed: int, rows: int, D: int, dtype: str = "bf16", device="cuda"):
        self.rows, self.D, self.dtype = rows, D, dtype
        vals = synth.value_table(seed, rows * D, dtype)
        self.host_raw = vals.reshape(rows, D)  # bf16 bit patterns (uint16) or float32
        if dtype == "bf16":
            self.host = synth.bf16_bits_to_f32(vals).reshape(rows, D)
            t = torch.from_numpy(vals.view(np.int16)).view(torch.bfloat16)
        else:
            self.host = vals.reshape(rows, D)
            t = torch.from_numpy(vals)
        self.dev = t.reshape(rows, D).to(device)

    def fill(self, pool: torch.Tensor, shift: int) -> None:
        """Fill pool (any shape, rows of D elements) with table rows
        (shift + i) mod rows, by device copies of contiguous table slices."""
        flat = pool.view(-1, self.D)
        n = flat.shape[0]
        i = 0
        while i < n:
            start = (shift + i) % self.rows
            k = min(self.rows - start, n - i)
            flat[i:i + k].copy_(self.dev[start:start + k])
            i += k

    def host_rows(self, shift: int, row_ids: np.ndarray) -> np.ndarray:
        """float32 values of pool rows `row_ids` of a pool filled with `shift`."""
        return self.host[(shift + np.asarray(row_ids, dtype=np.int64)) % self.rows]

    def host_raw_rows(self, shift: int, row_ids: np.ndarray) -> np.ndarray:
        """Stored element patterns (uint16 for bf16) of pool rows `row_ids`."""
        return self.host_raw[(shift + np.asarray(row_ids, dtype=np.int64)) % self.rows]


def torch_dtype(dtype: str):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def page_tables_for(group_pages: np.ndarray, seed: int, spare: int = 0):
    """Seeded fragmented page tables: group g's pages are a random permutation
    of its pool, dealt to sequences in order; -1 past each sequence's pages."""
    gp = np.asarray(group_pages, dtype=np.int64)
    G, B = gp.shape
    tables, sizes = [], []
    for g in range(G):
        total = int(gp[g].sum()) + spare
        perm = synth.page_permutation(seed * 7919 + g, max(total, 1))
        stride = max(1, int(gp[g].max()))
        pt = np.full((B, stride), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            k = int(gp[g, b])
            pt[b, :k] = perm[off:off + k]
            off += k
        tables.append(pt)
        sizes.append(max(total, 1))
    return tables, sizes


def rows_in_group(head_group: np.ndarray) -> np.ndarray:
    """Slot row of each KV head inside its group: rank in ascending head order."""
    hg = np.asarray(head_group)
    return np.array([int(np.sum(hg[:h] == hg[h])) for h in range(hg.size)], dtype=np.int64)


class TableLayer:
    """One layer of a DecodeConfig on the GPU: head-group pools filled from a
    ValueTable, fragmented page tables, q, budgets and lengths."""

    def __init__(self, cfg, layer: int, table: ValueTable, group_pages: np.ndarray,
                 seed: int = 0, spare: int = 0, device="cuda"):
        self.cfg, self.layer, self.table = cfg, layer, table
        hg = cfg.head_group[layer]
        self.rows = rows_in_group(hg)
        self.gsize = np.bincount(hg, minlength=cfg.num_groups)
        self.tables, self.pool_pages = page_tables_for(group_pages, seed * 131 + layer, spare)
        g = synth.rng(seed * 1009 + layer)
        self.shifts = g.integers(0, table.rows, size=(cfg.num_groups, 2)).astype(np.int64)
        dt = torch_dtype(cfg.dtype)
        self.k_pools, self.v_pools = [], []
        for gi in range(cfg.num_groups):
            shape = (self.pool_pages[gi], int(self.gsize[gi]), cfg.P, cfg.D)
            kp = torch.empty(shape, dtype=dt, device=device)
            vp = torch.empty(shape, dtype=dt, device=device)
            table.fill(kp, int(self.shifts[gi, 0]))
            table.fill(vp, int(self.shifts[gi, 1]))
            self.k_pools.append(kp)
            self.v_pools.append(vp)
        self.pt = [torch.from_numpy(t).to(device) for t in self.tables]
        self.strides = [t.shape[1] for t in self.tables]
        qv = synth.normal(g, (cfg.B, cfg.Hq, cfg.D), cfg.dtype)
        self.q_host = qv
        if cfg.dtype == "bf16":
            self.q = torch.from_numpy(synth.f32_to_bf16_bits(qv).view(np.int16)).view(
                torch.bfloat16).to(device)
        else:
            self.q = torch.from_numpy(qv).to(device)
        self.budget = torch.from_numpy(np.ascontiguousarray(cfg.budget[layer].reshape(-1),
                                                            dtype=np.int32)).to(device)
        self.seq_len = torch.from_numpy(np.ascontiguousarray(cfg.seq_len, np.int32)).to(device)

    def pool_row_ids(self, b: int, h: int) -> np.ndarray:
        """Pool row index (in units of D elements) of each kept token of (b, h)."""
        cfg = self.cfg
        gi = int(cfg.head_group[self.layer][h])
        n = int(cfg.n[self.layer][b, h])
        t = np.arange(n, dtype=np.int64)
        page = self.tables[gi][b, t // cfg.P].astype(np.int64)
        return (page * int(self.gsize[gi]) + int(self.rows[h])) * cfg.P + t % cfg.P

    def host_kv(self, b: int, h: int):
        """float32 K and V rows of the kept tokens of head (b, h), in order."""
        gi = int(self.cfg.head_group[self.layer][h])
        ids = self.pool_row_ids(b, h)
        return (self.table.host_rows(int(self.shifts[gi, 0]), ids),
                self.table.host_rows(int(self.shifts[gi, 1]), ids))
