"""Full-size workloads in the launch configuration the benchmark times
(balanced plan over two persistent blocks per SM, tensor-core kernel): every
(sequence, query head) of the layer against the fp64 oracle, and the tokens
the kernel actually consumed (its coverage record) against the oracle's
count array of the plan."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import oracle_layer
from synth.device import TableLayer, ValueTable
from paged_non_uniform_gb300 import kvx
import pages

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def table():
    return ValueTable(seed=11, rows=1 << 19, D=128, dtype="bf16")


def _plan(cfg, layer, policy=kvx.KVX_PLAN_BALANCED):
    plan = kvx.kvx_plan_create(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.P, cfg.num_groups,
                               kvx.KVX_BF16, cfg.budget[layer], cfg.seq_len,
                               cfg.head_group[layer], 0, policy)
    kvx.kvx_plan_upload(plan)
    return plan


def _run(plan, lay, cfg, cover=None):
    out = torch.full((cfg.B, cfg.Hq, cfg.D), float("nan"), device="cuda")
    ws = torch.zeros(plan.workspace_bytes() // 4 + 64, dtype=torch.int32, device="cuda")
    if cover is not None:
        plan.set_coverage_record(cover, cover.shape[1])
    kvx.kvx_decode_attn(plan, lay.q, lay.k_pools, lay.v_pools, lay.pool_pages, lay.pt,
                        lay.strides, lay.budget, lay.seq_len, 0.0, out, ws)
    torch.cuda.synchronize()
    if cover is not None:
        plan.set_coverage_record(None)
    assert kvx.kvx_workspace_status(ws) == 0
    return out.cpu().numpy().astype(np.float64)


def check_coverage(plan, cover):
    """The kernel's count of consumed tokens equals, bit for bit, the oracle's
    count array of the plan's items, and that array has no violation (every
    kept token once, nothing past n)."""
    items, _ = plan.items()
    n = plan.kept().reshape(-1)
    bad, count = oracle.load().plan_coverage(n, items)
    assert bad == 0
    got = cover.cpu().numpy()
    assert got.shape == count.shape
    assert np.array_equal(got, count)
    assert int(got.sum()) == int(n.sum())


def every_head(name, table, policy=kvx.KVX_PLAN_BALANCED, cfg=None):
    cfg = cfg or synth.decode_config(name, seed=0, layers=1)
    plan = _plan(cfg, 0, policy)
    lay = TableLayer(cfg, 0, table, plan.group_pages(), seed=0)
    cover = torch.zeros((cfg.B * cfg.Hkv, max(1, int(cfg.n[0].max()))), dtype=torch.int32,
                        device="cuda")
    got = _run(plan, lay, cfg, cover)
    check_coverage(plan, cover)
    assert np.all(np.isfinite(got))
    ref = oracle_layer(oracle.load(), cfg, lay)
    err = float(np.abs(got - ref).max())
    st = plan.stats()
    print(f"{cfg.name} layer 0, policy {policy}: {st['num_ctas']} blocks, "
          f"{st['num_items']} items, {st['num_split_heads']} split heads; "
          f"{cfg.B * cfg.Hq} (sequence, query head) outputs, max abs err {err:.3e}")
    assert err <= TOL, err
    return plan, lay, cfg


@pytest.mark.parametrize("name", ["qwen3_4b", "qwen3_4b_32k", "qwen25_32b", "llama3_sparse"])
def test_full_size_every_head_and_coverage(name, table):
    every_head(name, table)


def test_full_size_uniform_split_every_head_and_coverage(table):
    """The uniform-split plan (Tangram, Fig. 4(c)) on the same layer."""
    every_head("qwen3_4b", table, kvx.KVX_PLAN_UNIFORM)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_full_size_group_sweep_every_head(G, table):
    """The head-group sweep's configurations (Qwen3-4B layer 0 regrouped into
    groups of G KV heads; G = 8 is the unified page), as the benchmark's group
    sweep runs them: every head against the oracle, coverage exact."""
    every_head(None, table, cfg=synth.regroup(synth.decode_config("qwen3_4b", seed=0, layers=1),
                                              G))


def test_full_size_sparse_with_selected_tokens(table):
    """Llama-3-8B shapes, batch 8 x 122k: sampled heads keep the top 2048
    tokens by score plus the 128 most recent, selected from dense keys."""
    cfg = synth.decode_config("llama3_sparse", seed=0, layers=1)
    plan = _plan(cfg, 0)
    lay = TableLayer(cfg, 0, table, plan.group_pages(), seed=0)
    g = cfg.Hq // cfg.Hkv
    L = int(cfg.seq_len[0])
    dense = {}
    for b, h in [(0, 0), (3, 5), (7, 7)]:
        gen = synth.rng(5000 + b * cfg.Hkv + h)
        K = synth.normal(gen, (L, cfg.D), "bf16")
        V = synth.normal(gen, (L, cfg.D), "bf16")
        qh = lay.q_host[b, h * g:(h + 1) * g]
        kept = oracle.load().select_topk(qh, K, 2048, 128)
        assert kept.size == cfg.n[0][b, h] == 2176
        ids = torch.from_numpy(lay.pool_row_ids(b, h)).cuda()
        gi = int(cfg.head_group[0][h])
        for pool, src in ((lay.k_pools[gi], K), (lay.v_pools[gi], V)):
            rows = torch.from_numpy(synth.f32_to_bf16_bits(src[kept]).view(np.int16)).view(
                torch.bfloat16).cuda()
            pool.view(-1, cfg.D).index_copy_(0, ids, rows)
        dense[(b, h)] = (qh, K, V, kept)
    got = _run(plan, lay, cfg)
    orc = oracle.load()
    for (b, h), (qh, K, V, kept) in dense.items():
        ref = orc.attn_head(qh, K, V, kept, 1.0 / math.sqrt(cfg.D))
        err = float(np.abs(got[b, h * g:(h + 1) * g] - ref).max())
        assert err <= TOL, (b, h, err)


def test_full_size_gpu_selection_every_head(table):
    """Batch 8 x 122k dense keys (Llama-3-8B shapes, one layer, tiled from the
    value table): the GPU kept set of every head against the oracle's
    selection, outside the fp32 error band around the cut."""
    from test_select_gpu import check_head
    cfg = synth.decode_config("llama3_sparse", seed=0, layers=1)
    B, Hq, Hkv, D, L = cfg.B, cfg.Hq, cfg.Hkv, cfg.D, int(cfg.seq_len[0])
    top, recent = 2048, 128
    keys = torch.empty((B, Hkv, L, D), dtype=torch.bfloat16, device="cuda")
    table.fill(keys, 4242)
    q = synth.normal(synth.rng(99), (B, Hq, D), "bf16")
    qd = torch.from_numpy(synth.f32_to_bf16_bits(q).view(np.int16)).view(torch.bfloat16).cuda()
    kept = torch.zeros((B * Hkv, top + recent), dtype=torch.int32, device="cuda")
    cnt = torch.zeros(B * Hkv, dtype=torch.int32, device="cuda")
    ws = torch.zeros(kvx.kvx_select_workspace_bytes(B, Hkv, L) // 4 + 64, dtype=torch.int32,
                     device="cuda")
    kvx.kvx_select_topk(keys, qd, torch.from_numpy(cfg.seq_len).cuda(), B, Hq, Hkv, D, L, top,
                        recent, kept, cnt, ws)
    torch.cuda.synchronize()
    kept, cnt = kept.cpu().numpy(), cnt.cpu().numpy()
    assert np.all(cnt == top + recent)
    orc = oracle.load()
    g = Hq // Hkv
    for b, h in [(b, h) for b in range(B) for h in range(Hkv)]:
        bh = b * Hkv + h
        kh = table.host_rows(4242, bh * L + np.arange(L, dtype=np.int64))
        check_head(orc, q[b, h * g:(h + 1) * g], kh, top, recent, kept[bh])


def test_full_size_select_pack_attend(table):
    """The benchmark's sparse pipeline at full size (Llama-3-8B shapes, batch 8
    x 122k, one layer): GPU selection, packing of the kept rows into
    head-group pages, attention over them. Every head: packed slots equal the
    dense rows bit for bit, and the output equals the oracle's attention over
    the same kept set; attention straight over the kept rows
    (kvx_decode_attn_kept, same plan) gives the same bits."""
    cfg = synth.decode_config("llama3_sparse", seed=0, layers=1)
    B, Hq, Hkv, D, L, P = cfg.B, cfg.Hq, cfg.Hkv, cfg.D, int(cfg.seq_len[0]), cfg.P
    top, recent = 2048, 128
    keys = torch.empty((B, Hkv, L, D), dtype=torch.bfloat16, device="cuda")
    vals = torch.empty_like(keys)
    table.fill(keys, 777)
    table.fill(vals, 31337)
    q = synth.normal(synth.rng(98), (B, Hq, D), "bf16")
    qd = torch.from_numpy(synth.f32_to_bf16_bits(q).view(np.int16)).view(torch.bfloat16).cuda()
    kept = torch.zeros((B * Hkv, top + recent), dtype=torch.int32, device="cuda")
    cnt = torch.zeros(B * Hkv, dtype=torch.int32, device="cuda")
    sl = torch.from_numpy(cfg.seq_len).cuda()
    ws = torch.zeros(kvx.kvx_select_workspace_bytes(B, Hkv, L) // 4 + 64, dtype=torch.int32,
                     device="cuda")
    kvx.kvx_select_topk(keys, qd, sl, B, Hq, Hkv, D, L, top, recent, kept, cnt, ws)
    torch.cuda.synchronize()
    n = cnt.cpu().numpy().reshape(B, Hkv)
    assert np.all(n == top + recent)
    hg = np.zeros(Hkv, np.int32)
    plan = kvx.kvx_plan_create(B, Hq, Hkv, D, P, 1, kvx.KVX_BF16, n, cfg.seq_len, hg, 0)
    kvx.kvx_plan_upload(plan)
    gp = plan.group_pages()
    tables, npages = pages.assign_pages(gp, [synth.page_permutation(7, int(gp[0].sum()) + 2)], 2)
    kp = torch.zeros((npages[0], Hkv, P, D), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    pt = torch.from_numpy(tables[0]).cuda()
    aws = torch.zeros(plan.workspace_bytes() // 4 + 64, dtype=torch.int32, device="cuda")
    kvx.kvx_pack_kept(plan, keys, vals, L, kept, top + recent, [kp], [vp], npages, [pt],
                      [tables[0].shape[1]], aws)
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    kvx.kvx_decode_attn(plan, qd, [kp], [vp], npages, [pt], [tables[0].shape[1]],
                        torch.from_numpy(n.reshape(-1).copy()).cuda(), sl, 0.0, out, aws)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(aws) == 0
    got = out.cpu().numpy().astype(np.float64)
    # the same plan straight over the kept rows of the dense cache: the same bits
    out2 = torch.full((B, Hq, D), float("nan"), device="cuda")
    kvx.kvx_decode_attn_kept(plan, qd, keys, vals, L, kept, top + recent,
                             torch.from_numpy(n.reshape(-1).copy()).cuda(), sl, 0.0, out2, aws)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(aws) == 0
    assert np.array_equal(out2.cpu().numpy().astype(np.float64), got)
    kept_h = kept.cpu().numpy()
    orc = oracle.load()
    g = Hq // Hkv
    for b, h in [(b, h) for b in range(B) for h in range(Hkv)]:
        bh = b * Hkv + h
        idx = kept_h[bh]
        rows = bh * L + idx.astype(np.int64)
        kh = table.host_rows(777, rows)
        vh = table.host_rows(31337, rows)
        # packed slots: token i of head h at page tables[0][b, i // P], slot row h
        t = np.arange(idx.size)
        pg = tables[0][b, t // P]
        slots = kp[torch.from_numpy(pg).cuda(), h, torch.from_numpy(t % P).cuda()]
        assert np.array_equal(slots.float().cpu().numpy(), kh), (b, h)
        ref = orc.attn_head(q[b, h * g:(h + 1) * g], kh, vh, np.arange(idx.size, dtype=np.int32),
                            1.0 / math.sqrt(D))
        assert float(np.abs(got[b, h * g:(h + 1) * g] - ref).max()) <= TOL, (b, h)
