"""Runs the kvx decode path on a synthetic case and the oracle beside it.

Test infrastructure: builds the plan through the C ABI, assigns physical pages
with a seeded permutation, packs the dense kept rows into head-group pools,
uploads everything with torch and calls kvx_decode_attn through the binding.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import synth
from paged_non_uniform_gb300 import kvx
import pages


def num_groups(case) -> int:
    return int(np.asarray(case.head_group).max()) + 1


def make_plan(case, num_ctas=0, policy=kvx.KVX_PLAN_BALANCED, kernel=kvx.KVX_KERNEL_AUTO,
              upload=True, layout=kvx.KVX_LAYOUT_HEAD_MAJOR):
    dtype = kvx.KVX_BF16 if case.dtype == "bf16" else kvx.KVX_F32
    plan = kvx.kvx_plan_create(case.B, case.Hq, case.Hkv, case.D, case.P, num_groups(case),
                               dtype, case.budget, case.seq_len, case.head_group, num_ctas,
                               policy, kernel, layout)
    if upload:
        kvx.kvx_plan_upload(plan)
    return plan


class DeviceCase:
    """Device copies of a DenseCase laid out in head-group pages."""

    def __init__(self, case, plan, perm_seed=1, spare_pages=3, fill=float("nan"),
                 dense_override=None):
        self.case, self.plan = case, plan
        G = num_groups(case)
        gp = plan.group_pages()
        perms = [synth.page_permutation(perm_seed * 1000 + g, int(gp[g].sum()) + spare_pages)
                 for g in range(G)]
        self.tables, self.pool_pages = pages.assign_pages(gp, perms, spare_pages)
        k, v = (case.k, case.v) if dense_override is None else dense_override
        tm = plan.shape.layout == kvx.KVX_LAYOUT_TOKEN_MAJOR
        if case.dtype == "bf16":
            kb, vb = synth.f32_to_bf16_bits(k), synth.f32_to_bf16_bits(v)
            pools = pages.pack_pools(kb, vb, case.kept, case.head_group, self.tables,
                                     self.pool_pages, case.P, np.uint16, fill, token_major=tm)
            conv = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
            self.q = conv(synth.f32_to_bf16_bits(case.q))
        else:
            pools = pages.pack_pools(k, v, case.kept, case.head_group, self.tables,
                                     self.pool_pages, case.P, np.float32, fill, token_major=tm)
            conv = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
            self.q = conv(case.q)
        self.k_pools = [conv(kp) for kp, _ in pools]
        self.v_pools = [conv(vp) for _, vp in pools]
        self.pt = [torch.from_numpy(t).cuda() for t in self.tables]
        self.strides = [t.shape[1] for t in self.tables]
        self.budget = torch.from_numpy(np.ascontiguousarray(case.budget.reshape(-1),
                                                            dtype=np.int32)).cuda()
        self.seq_len = torch.from_numpy(np.ascontiguousarray(case.seq_len, np.int32)).cuda()
        self.out = torch.full((case.B, case.Hq, case.D), float("nan"), device="cuda")
        nbytes = plan.workspace_bytes()
        self.ws = torch.zeros(max(nbytes, 256) // 4 + 64, dtype=torch.int32, device="cuda")

    def run(self, scale=0.0, budget=None, stream=None) -> np.ndarray:
        kvx.kvx_decode_attn(self.plan, self.q, self.k_pools, self.v_pools, self.pool_pages,
                            self.pt, self.strides, self.budget if budget is None else budget,
                            self.seq_len, scale, self.out, self.ws, stream=stream)
        torch.cuda.synchronize()
        return self.out.cpu().numpy().astype(np.float64)

    def status(self) -> int:
        return kvx.kvx_workspace_status(self.ws)


def oracle_out(case, scale=None) -> np.ndarray:
    orc = oracle.load()
    s = 1.0 / math.sqrt(case.D) if scale is None else scale
    return orc.decode_attn(case.q.astype(np.float64), case.k.astype(np.float64),
                           case.v.astype(np.float64), case.seq_len, case.kept, s)


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


def oracle_layer(orc, cfg, lay, max_rows=1 << 19) -> np.ndarray:
    """The oracle's output for every (sequence, query head) of one layer held
    by a synth.device.TableLayer: each head's kept K/V rows are rebuilt on
    the host from the value table, compacted to positions 0..n-1, and the
    oracle runs over groups of sequences (at most max_rows rows per tensor
    per call, so that its OpenMP loop spans many heads)."""
    B, Hq, Hkv, D = cfg.B, cfg.Hq, cfg.Hkv, cfg.D
    n = cfg.n[lay.layer]
    out = np.zeros((B, Hq, D))
    scale = 1.0 / math.sqrt(D)
    b0 = 0
    while b0 < B:
        b1 = b0 + 1
        while b1 < B and (b1 + 1 - b0) * Hkv * int(n[b0:b1 + 1].max()) <= max_rows:
            b1 += 1
        nmax = int(n[b0:b1].max())
        k = np.zeros((b1 - b0, Hkv, nmax, D))
        v = np.zeros_like(k)
        kept = []
        for b in range(b0, b1):
            for h in range(Hkv):
                kh, vh = lay.host_kv(b, h)
                k[b - b0, h, :kh.shape[0]] = kh
                v[b - b0, h, :vh.shape[0]] = vh
                kept.append(np.arange(kh.shape[0], dtype=np.int32))
        out[b0:b1] = orc.decode_attn(lay.q_host[b0:b1].astype(np.float64), k, v,
                                     np.full(b1 - b0, nmax, np.int32), kept, scale)
        b0 = b1
    return out
