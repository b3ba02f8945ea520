"""CPU oracle for the non-uniform paged decode-attention path and the KV gather.

TEST INFRASTRUCTURE ONLY: the product (``paged_non_uniform_gb300``) never imports
this package. It is used by ``tests/``, by ``__graft_entry__.smoke()`` and by the
CPU-baseline leg of ``bench.py``.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double). This module only
compiles it with gcc and marshals NumPy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(out: str = _LIB, mutant: int = 0, openmp: bool = True) -> str:
    """Compile oracle.c into a shared library (gcc, -O2, no fast-math)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", out, "-lm"]
    if openmp:
        cmd.insert(1, "-fopenmp")
    if mutant:
        cmd.insert(1, f"-DORACLE_MUTANT={int(mutant)}")
    subprocess.run(cmd, check=True)
    return out


def _needs_build() -> bool:
    if not os.path.exists(_LIB):
        return True
    return os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC),
                                        os.path.getmtime(os.path.join(_HERE, "oracle.h")))


_I32 = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_I64 = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_F64 = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_U8 = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_c = ctypes


class Oracle:
    """ctypes view of one compiled oracle library (the real one or a mutant)."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_resolve_budget.argtypes = [_c.c_int, _c.c_int, _I32, _I32, _I32]
        lib.oracle_attn_head.argtypes = [_c.c_int, _c.c_int, _c.c_int, _F64, _F64, _F64,
                                         _c.c_int, _I32, _c.c_double, _F64, _c.c_void_p]
        lib.oracle_decode_attn.argtypes = [_c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,
                                           _I32, _F64, _F64, _F64, _I64, _I32,
                                           _c.c_double, _F64]
        lib.oracle_group_pages.argtypes = [_c.c_int, _c.c_int, _I32, _I32, _c.c_int,
                                           _c.c_int, _I32]
        lib.oracle_footprint_bytes.argtypes = [_c.c_int, _c.c_int, _I32, _I32, _c.c_int,
                                               _c.c_int, _c.c_int, _c.c_int, _I64]
        lib.oracle_plan_coverage.argtypes = [_c.c_int, _I32, _c.c_int, _c.c_int,
                                             _c.c_void_p, _I32]
        lib.oracle_plan_coverage.restype = _c.c_int64
        lib.oracle_runs.argtypes = [_c.c_int, _c.c_int, _I32, _I32, _I32, _I32]
        lib.oracle_runs.restype = _c.c_int64
        lib.oracle_gather.argtypes = [_c.c_int, _c.c_int, _I32, _I32, _U8, _c.c_int64,
                                      _c.c_int64, _U8, _c.c_int64, _c.c_int]
        lib.oracle_select_topk.argtypes = [_c.c_int, _c.c_int, _c.c_int, _F64, _F64, _c.c_int,
                                           _c.c_int, _I32, _c.c_void_p]
        lib.oracle_num_threads.restype = _c.c_int
        lib.oracle_frame_new.argtypes = [_c.c_int, _c.c_int, _c.c_int32]
        lib.oracle_frame_new.restype = _c.c_void_p
        lib.oracle_frame_free.argtypes = [_c.c_void_p]
        lib.oracle_frame_reserve.argtypes = [_c.c_void_p, _c.c_int, _c.c_int, _c.c_void_p]
        lib.oracle_frame_alias.argtypes = [_c.c_void_p] + [_c.c_int] * 5
        lib.oracle_frame_trim.argtypes = [_c.c_void_p, _c.c_int, _c.c_int, _c.c_int]
        lib.oracle_frame_state.argtypes = [_c.c_void_p, _I32, _I32, _c.c_void_p]
        self.lib = lib

    # -- attention -------------------------------------------------------
    def resolve_budget(self, budget, seq_len):
        budget = np.ascontiguousarray(budget, dtype=np.int32)
        seq_len = np.ascontiguousarray(seq_len, dtype=np.int32)
        B = seq_len.shape[0]
        Hkv = budget.size // max(B, 1)
        n = np.zeros(B * Hkv, dtype=np.int32)
        if self.lib.oracle_resolve_budget(B, Hkv, budget.reshape(-1), seq_len, n) != 0:
            raise ValueError("oracle_resolve_budget: invalid arguments")
        return n.reshape(B, Hkv)

    def attn_head(self, q, k, v, idx, scale, want_weights=False):
        """q: [g][D]; k, v: [L][D]; idx: kept positions. Returns out [g][D] (and w)."""
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        g, D = q.shape
        L = k.shape[0]
        out = np.zeros((g, D), dtype=np.float64)
        w = np.zeros((g, idx.size), dtype=np.float64) if want_weights else None
        rc = self.lib.oracle_attn_head(D, g, L, q, k, v, idx.size, idx, float(scale), out,
                                       w.ctypes.data if w is not None else None)
        if rc != 0:
            raise ValueError("oracle_attn_head: invalid arguments")
        return (out, w) if want_weights else out

    def decode_attn(self, q, k, v, seq_len, kept, scale):
        """q: [B][Hq][D]; k, v: [B][Hkv][Lmax][D]; kept: list (len B*Hkv) of index arrays."""
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        B, Hq, D = q.shape
        Hkv, Lmax = k.shape[1], k.shape[2]
        seq_len = np.ascontiguousarray(seq_len, dtype=np.int32)
        off = np.zeros(B * Hkv + 1, dtype=np.int64)
        off[1:] = np.cumsum([len(x) for x in kept])
        idx = (np.concatenate([np.asarray(x, dtype=np.int32) for x in kept])
               if off[-1] else np.zeros(1, np.int32))
        out = np.zeros((B, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_decode_attn(B, Hq, Hkv, D, Lmax, seq_len, q, k, v, off,
                                         np.ascontiguousarray(idx), float(scale), out)
        if rc != 0:
            raise ValueError("oracle_decode_attn: invalid arguments")
        return out

    # -- head-group pages ------------------------------------------------
    def group_pages(self, n, head_group, P):
        n = np.ascontiguousarray(n, dtype=np.int32)
        B, Hkv = n.shape
        hg = np.ascontiguousarray(head_group, dtype=np.int32)
        G = int(hg.max()) + 1
        pages = np.zeros((G, B), dtype=np.int32)
        if self.lib.oracle_group_pages(B, Hkv, n.reshape(-1), hg, G, P, pages) != 0:
            raise ValueError("oracle_group_pages: invalid arguments")
        return pages

    def footprint_bytes(self, n, head_group, P, D, dtype_bytes):
        n = np.ascontiguousarray(n, dtype=np.int32)
        B, Hkv = n.shape
        hg = np.ascontiguousarray(head_group, dtype=np.int32)
        G = int(hg.max()) + 1
        out = np.zeros(B, dtype=np.int64)
        if self.lib.oracle_footprint_bytes(B, Hkv, n.reshape(-1), hg, G, P, D,
                                           dtype_bytes, out) != 0:
            raise ValueError("oracle_footprint_bytes: invalid arguments")
        return out

    # -- plan coverage ---------------------------------------------------
    def plan_coverage(self, n, items):
        """n: [nheads]; items: [nitems][4] int32. Returns (violations, count)."""
        n = np.ascontiguousarray(n, dtype=np.int32).reshape(-1)
        items = np.ascontiguousarray(items, dtype=np.int32).reshape(-1, 4)
        maxn = int(n.max()) if n.size else 0
        maxn = max(maxn, int(items[:, 2].max()) if items.size else 0)
        count = np.zeros((n.size, max(maxn, 1)), dtype=np.int32)
        bad = self.lib.oracle_plan_coverage(n.size, n, max(maxn, 1), items.shape[0],
                                            items.ctypes.data if items.size else None, count)
        if bad < 0:
            raise ValueError("oracle_plan_coverage: invalid arguments")
        return int(bad), count

    # -- gather ----------------------------------------------------------
    def runs(self, bt, nb):
        bt = np.ascontiguousarray(bt, dtype=np.int32)
        nb = np.ascontiguousarray(nb, dtype=np.int32)
        S, mb = bt.shape
        cnt = np.zeros(S, dtype=np.int32)
        runs = np.zeros((S, max(mb, 1), 3), dtype=np.int32)
        tot = self.lib.oracle_runs(S, mb, bt, nb, cnt, runs)
        if tot < 0:
            raise ValueError("oracle_runs: invalid arguments")
        return int(tot), cnt, runs

    def gather(self, bt, nb, pool, staging, zero_tail=False):
        """pool: uint8 [num_phys][block_bytes]; staging: uint8 [S][row_bytes] (updated)."""
        bt = np.ascontiguousarray(bt, dtype=np.int32)
        nb = np.ascontiguousarray(nb, dtype=np.int32)
        assert pool.dtype == np.uint8 and pool.flags.c_contiguous
        assert staging.dtype == np.uint8 and staging.flags.c_contiguous
        S, mb = bt.shape
        rc = self.lib.oracle_gather(S, mb, bt, nb, pool.reshape(-1), pool.shape[0],
                                    pool.shape[1], staging.reshape(-1), staging.shape[1],
                                    int(bool(zero_tail)))
        if rc != 0:
            raise ValueError("oracle_gather: invalid arguments")
        return staging

    # -- sparse selection --------------------------------------------
    def select_topk(self, q, k, top, recent, want_scores=False):
        """q: [g][D]; k: [L][D]. Returns ascending kept positions (and scores)."""
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        g, D = q.shape
        L = k.shape[0]
        kept = np.zeros(max(top + recent, 1), dtype=np.int32)
        sc = np.zeros(L, dtype=np.float64) if want_scores else None
        n = self.lib.oracle_select_topk(L, D, g, q, k, int(top), int(recent), kept,
                                        sc.ctypes.data if sc is not None else None)
        if n < 0:
            raise ValueError("oracle_select_topk: invalid arguments")
        return (kept[:n], sc) if want_scores else kept[:n]

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    # -- KV-RM block pager -------------------------------------------------
    def frame(self, S, max_blocks, num_phys):
        return OracleFrame(self, S, max_blocks, num_phys)


class OracleFrame:
    """The oracle's block pager: one logical view per sequence over
    refcounted physical blocks, edited by Reserve / Alias / Trim. Each edit
    returns the oracle's code (0, -1 bad argument, -2 range, -3 no space)."""

    def __init__(self, orc: Oracle, S: int, max_blocks: int, num_phys: int):
        self.lib, self.S, self.M, self.N = orc.lib, S, max_blocks, num_phys
        self.h = self.lib.oracle_frame_new(S, max_blocks, num_phys)
        if not self.h:
            raise ValueError("oracle_frame_new: invalid arguments")

    def __del__(self):
        if getattr(self, "h", None):
            self.lib.oracle_frame_free(self.h)
            self.h = None

    def reserve(self, s, c):
        out = np.zeros(max(int(c), 1), dtype=np.int32)
        rc = self.lib.oracle_frame_reserve(self.h, int(s), int(c), out.ctypes.data)
        return rc, out[:max(int(c), 0)] if rc == 0 else out[:0]

    def alias(self, dst, dj, src, sj, c):
        return self.lib.oracle_frame_alias(self.h, int(dst), int(dj), int(src), int(sj), int(c))

    def trim(self, s, begin, end):
        return self.lib.oracle_frame_trim(self.h, int(s), int(begin), int(end))

    def state(self):
        """(table [S][max_blocks] with -1 past the view, nb [S], refcount [N])."""
        table = np.zeros((self.S, self.M), dtype=np.int32)
        nb = np.zeros(self.S, dtype=np.int32)
        rc = np.zeros(self.N, dtype=np.int32)
        self.lib.oracle_frame_state(self.h, table.reshape(-1), nb, rc.ctypes.data)
        return table, nb, rc


_default: Oracle | None = None


def load() -> Oracle:
    """The oracle library, compiled on first use if missing or stale."""
    global _default
    if _default is None:
        if _needs_build():
            build()
        _default = Oracle(_LIB)
    return _default


def load_mutant(k: int) -> Oracle:
    """A copy of the oracle with planted mistake number k (tests only)."""
    d = tempfile.mkdtemp(prefix="oracle_mutant_")
    path = build(os.path.join(d, f"liboracle_m{k}.so"), mutant=k, openmp=False)
    return Oracle(path)
