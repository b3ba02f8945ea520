"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and its host-only planner agrees with the oracle."""
import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvx():
    from paged_non_uniform_gb300 import build
    build.build()
    from paged_non_uniform_gb300 import kvx as k
    return k


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvx.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvx_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("kvx_plan_create", "kvx_decode_attn", "kvx_gather_coalesce",
                 "kvx_plan_destroy", "kvx_plan_upload", "kvx_plan_workspace_bytes"):
        assert must in names


def test_library_exports_every_declared_symbol(kvx):
    missing = [n for n in declared_functions() if not hasattr(kvx.lib, n)]
    assert not missing, missing


def test_status_strings(kvx):
    for code in (0, -1, -2, -3, -4, -5, -6, -99):
        assert isinstance(kvx.kvx_status_string(code), str)


def _plan(kvx, case, num_ctas=0, policy=0, kernel=0):
    dtype = kvx.KVX_BF16 if case.dtype == "bf16" else kvx.KVX_F32
    G = int(case.head_group.max()) + 1
    return kvx.kvx_plan_create(case.B, case.Hq, case.Hkv, case.D, case.P, G, dtype,
                               case.budget, case.seq_len, case.head_group, num_ctas, policy,
                               kernel)


CASES = {
    "tiny_per_head": lambda: synth.tiny(0, "per_head"),
    "tiny_one_group": lambda: synth.tiny(0, "one"),
    "mixed": lambda: synth.dense_case(3, 12, 4, 64, [40, 300, 1000],
                                      [[40, 5, 17, 33], [300, 100, 1, 64], [900, 1000, 31, 32]],
                                      "f32", seed=2, head_group=[0, 1, 1, 2]),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("policy", [0, 1, 2])
@pytest.mark.parametrize("num_ctas", [1, 3, 7, 152])
def test_plan_coverage_matches_oracle(kvx, orc, name, policy, num_ctas):
    case = CASES[name]()
    plan = _plan(kvx, case, num_ctas=num_ctas, policy=policy)
    n_oracle = orc.resolve_budget(case.budget, case.seq_len)
    assert np.array_equal(plan.kept(), n_oracle)
    assert np.array_equal(plan.kept(), case.n)
    items, off = plan.items()
    bad, count = orc.plan_coverage(n_oracle.reshape(-1), items)
    assert bad == 0
    assert np.array_equal(plan.coverage(), count)  # kvx_plan_coverage, bit for bit
    st = plan.stats()
    assert off[0] == 0 and off[-1] == len(items) and np.all(np.diff(off) >= 0)
    assert st["total_tokens"] == int(n_oracle.sum())
    # partial slots: every item of a split head has a distinct slot, others -1
    per_head = np.bincount(items[:, 0], minlength=case.B * case.Hkv)
    split = per_head[items[:, 0]] > 1
    assert np.all(items[~split, 3] == -1)
    slots = items[split, 3]
    assert sorted(slots.tolist()) == list(range(st["num_slots"]))
    # items start at multiples of the cut granularity, min(P, 32) tokens
    assert np.all(items[:, 1] % min(case.P, 32) == 0)


@pytest.mark.parametrize("name", sorted(CASES))
def test_group_pages_and_footprint_match_oracle(kvx, orc, name):
    case = CASES[name]()
    plan = _plan(kvx, case, num_ctas=4)
    pages = orc.group_pages(case.n, case.head_group, case.P)
    assert np.array_equal(plan.group_pages(), pages)
    st = plan.stats()
    fp = orc.footprint_bytes(case.n, case.head_group, case.P, case.D, 4)
    # footprint = allocated token slots x 2 (K, V) x D x bytes
    assert st["slots_allocated"] * 2 * case.D * 4 == int(fp.sum())
    assert st["slots_used"] == int(case.n.sum())


def test_balanced_plan_is_balanced(kvx):
    cfg = synth.decode_config("qwen3_4b", seed=0, layers=2)
    for layer in range(cfg.layers):
        plan = kvx.kvx_plan_create(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.P, cfg.num_groups,
                                   kvx.KVX_BF16, cfg.budget[layer], cfg.seq_len,
                                   cfg.head_group[layer], 152)
        t = plan.cta_tokens()
        st = plan.stats()
        assert t.sum() == cfg.n[layer].sum()
        # max load within one item overhead + one stage of the mean
        assert t.max() <= t.mean() + st["item_overhead"] + 32 + 1, (t.max(), t.mean())
        naive = kvx.kvx_plan_create(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.P, cfg.num_groups,
                                    kvx.KVX_BF16, cfg.budget[layer], cfg.seq_len,
                                    cfg.head_group[layer], 152, kvx.KVX_PLAN_PER_HEAD)
        assert naive.stats()["max_cta_tokens"] > 2 * st["max_cta_tokens"]


@pytest.mark.parametrize("bad", ["budget0", "seq0", "group_range", "empty_group", "gqa",
                                 "head_dim", "page", "mma_f32", "policy"])
def test_plan_rejects_bad_arguments(kvx, bad):
    B, Hq, Hkv, D, P, G = 2, 8, 2, 64, 16, 2
    budget, seq, hg = np.array([[4, 5], [6, 7]]), np.array([10, 20]), np.array([0, 1])
    dtype, kernel, policy = kvx.KVX_BF16, 0, 0
    if bad == "budget0":
        budget = np.array([[0, 5], [6, 7]])
    elif bad == "seq0":
        seq = np.array([0, 20])
    elif bad == "group_range":
        hg = np.array([0, 2])
    elif bad == "empty_group":
        hg = np.array([0, 0])
    elif bad == "gqa":
        Hq = 7
    elif bad == "head_dim":
        D = 96
    elif bad == "page":
        P = 12
    elif bad == "mma_f32":
        dtype, kernel = kvx.KVX_F32, kvx.KVX_KERNEL_MMA
    elif bad == "policy":
        policy = 9
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_plan_create(B, Hq, Hkv, D, P, G, dtype, budget, seq, hg, 4, policy, kernel)
    assert e.value.status in (kvx.KVX_EINVAL, kvx.KVX_EUNSUPPORTED)


def test_decode_rejects_before_upload(kvx):
    case = synth.tiny(0)
    plan = _plan(kvx, case, num_ctas=2)
    rc = kvx.lib.kvx_decode_attn(plan.handle, 16, (kvx._vp * 2)(16, 16), (kvx._vp * 2)(16, 16),
                                 np.array([1, 1], np.int64).ctypes.data,
                                 (kvx._vp * 2)(16, 16), np.array([8, 8], np.int32).ctypes.data,
                                 16, 16, 0.0, 16, 256, 1 << 20, None)
    assert rc == kvx.KVX_ESTATE


def test_gather_rejects_bad_arguments(kvx):
    p = (kvx._vp * 1)(4096)
    ws = kvx.kvx_gather_workspace_bytes(2, 4)
    assert ws > kvx.KVX_WS_HEADER_BYTES
    # block_bytes not a multiple of 16
    rc = kvx.lib.kvx_gather_coalesce(256, 256, 2, 4, 1, p, 8, 40, p, 160, 0, 256, ws, None)
    assert rc == kvx.KVX_EINVAL
    # workspace too small
    rc = kvx.lib.kvx_gather_coalesce(256, 256, 2, 4, 1, p, 8, 32, p, 128, 0, 256, 16, None)
    assert rc == kvx.KVX_EINVAL
    # unknown flag
    rc = kvx.lib.kvx_gather_coalesce(256, 256, 2, 4, 1, p, 8, 32, p, 128, 8, 256, ws, None)
    assert rc == kvx.KVX_EINVAL


def test_group_size_trades_fragmentation_for_tables(kvx, orc):
    """Larger head groups mean fewer page-table entries but more padding slots;
    the planner's counts follow the oracle's page counts for every G."""
    cfg = synth.decode_config("qwen3_4b", seed=0, layers=1)
    frag, entries = [], []
    for G in (1, 2, 4, 8):
        c = synth.regroup(cfg, G)
        plan = kvx.kvx_plan_create(c.B, c.Hq, c.Hkv, c.D, c.P, c.num_groups, kvx.KVX_BF16,
                                   c.budget[0], c.seq_len, c.head_group[0], 152)
        pages = orc.group_pages(c.n[0], c.head_group[0], c.P)
        assert np.array_equal(plan.group_pages(), pages)
        st = plan.stats()
        frag.append(1 - st["slots_used"] / st["slots_allocated"])
        entries.append(int(pages.sum()))
    assert frag == sorted(frag) and frag[0] < frag[-1]
    assert entries == sorted(entries, reverse=True)


def test_early_kv_setter(kvx):
    """kvx_plan_set_early_kv takes 0 or 1 on a plan; anything else is
    KVX_EINVAL (a NULL plan too)."""
    case = synth.tiny(0)
    plan = _plan(kvx, case, num_ctas=2)
    assert kvx.lib.kvx_plan_set_early_kv(plan.handle, 1) == kvx.KVX_OK
    assert kvx.lib.kvx_plan_set_early_kv(plan.handle, 0) == kvx.KVX_OK
    assert kvx.lib.kvx_plan_set_early_kv(plan.handle, 2) == kvx.KVX_EINVAL
    assert kvx.lib.kvx_plan_set_early_kv(plan.handle, -1) == kvx.KVX_EINVAL
    assert kvx.lib.kvx_plan_set_early_kv(None, 1) == kvx.KVX_EINVAL


def test_select_and_pack_reject_bad_arguments(kvx):
    ws = kvx.kvx_select_workspace_bytes(2, 2, 101)
    # header | histograms [4][2048] | group maxima u16 [4][16] | scores [4][104],
    # each section 256-aligned (13 groups of 8 rounded up to 16; 101 scores to 104)
    al = lambda x: (x + 255) // 256 * 256
    gmax = al(kvx.KVX_WS_HEADER_BYTES + 4 * 2048 * 4)
    scores = al(gmax + 4 * 2 * 16)
    assert ws == al(scores + 4 * 4 * 104)
    rc = kvx.lib.kvx_select_topk(256, 256, 256, 2, 8, 2, 96, 100, 10, 4, 256, 256, 256, ws, None)
    assert rc == kvx.KVX_EUNSUPPORTED
    rc = kvx.lib.kvx_select_topk(256, 256, 256, 2, 7, 2, 128, 100, 10, 4, 256, 256, 256, ws, None)
    assert rc == kvx.KVX_EINVAL
    rc = kvx.lib.kvx_select_topk(256, 256, 256, 2, 8, 2, 128, 100, 10, 4, 256, 256, 256, 16, None)
    assert rc == kvx.KVX_EINVAL
    case = synth.tiny(0)
    plan = _plan(kvx, case, num_ctas=2)
    p = (kvx._vp * 2)(256, 256)
    rc = kvx.lib.kvx_pack_kept(plan.handle, 256, 256, 100, 256, 100, p, p,
                               np.array([4, 4], np.int64).ctypes.data, p,
                               np.array([8, 8], np.int32).ctypes.data, 256, 256, None)
    assert rc == kvx.KVX_ESTATE


def test_kept_row_attention_rejects_bad_arguments(kvx):
    case = synth.tiny(0)
    plan = _plan(kvx, case, num_ctas=2)
    f = kvx.lib.kvx_decode_attn_kept
    # null dense caches or kept list, then a plan that was never uploaded
    assert f(plan.handle, 256, None, 256, 100, 256, 100, 256, 256, 0.0, 256, 256, 1 << 20,
             None) == kvx.KVX_EINVAL
    assert f(plan.handle, 256, 256, 256, 100, None, 100, 256, 256, 0.0, 256, 256, 1 << 20,
             None) == kvx.KVX_EINVAL
    assert f(None, 256, 256, 256, 100, 256, 100, 256, 256, 0.0, 256, 256, 1 << 20,
             None) == kvx.KVX_EINVAL
    assert f(plan.handle, 256, 256, 256, 100, 256, 100, 256, 256, 0.0, 256, 256, 1 << 20,
             None) == kvx.KVX_ESTATE


@pytest.mark.parametrize("name", ["qwen3_4b", "llama3_sparse", "qwen25_32b"])
@pytest.mark.parametrize("num_ctas", [152, 304, 1000])
def test_balanced_plan_cap(kvx, name, num_ctas):
    """Every block of the balanced plan costs (tokens + item charge per item)
    at most one item charge plus two stages above the ideal share (cut
    rounding and the no-sliver rule leave less than a cut each, and a block
    may close one item short); pieces are whole multiples of the cut
    granularity min(P, 32) except a head's last piece; at most one head is
    cut at each block boundary."""
    cfg = synth.decode_config(name, seed=0, layers=1)
    plan = kvx.kvx_plan_create(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.P, cfg.num_groups,
                               kvx.KVX_BF16, cfg.budget[0], cfg.seq_len, cfg.head_group[0],
                               num_ctas)
    st = plan.stats()
    c0 = st["item_overhead"]
    items, off = plan.items()
    n = cfg.n[0].reshape(-1)
    cost = [int((items[off[c]:off[c + 1], 2] - items[off[c]:off[c + 1], 1]).sum())
            + c0 * int(off[c + 1] - off[c]) for c in range(num_ctas)]
    # ideal share: tokens, an item charge per head, and one more per block
    # boundary (where a head can be cut)
    ideal = (int(n.sum()) + c0 * n.size + c0 * (num_ctas - 1)) / num_ctas
    assert max(cost) <= ideal + c0 + 2 * 32 + 1, (max(cost), ideal)
    T = min(cfg.P, 32)  # cut granularity
    for bh, b, e in items[:, :3]:
        assert b % T == 0 and (e % T == 0 or e == n[bh]), (bh, b, e)
    # a head cut across blocks: its pieces sit in consecutive blocks
    cta_of = np.repeat(np.arange(num_ctas), np.diff(off))
    for bh in np.unique(items[:, 0]):
        ctas = np.sort(cta_of[items[:, 0] == bh])
        assert np.all(np.diff(ctas) == 1), (bh, ctas)


@pytest.mark.parametrize("seed", range(40))
def test_balanced_plan_random_shapes(kvx, orc, seed):
    """Seeded random shapes, budgets, groupings and block counts, down to
    heads shorter than a stage and more blocks than stages. The balanced plan
    covers every kept token once (oracle count array) and resolves budgets as
    the oracle does. Pieces are whole cuts (min(P, 32) tokens) except a head's
    last. A cut head's pieces sit in consecutive blocks and run before the
    block's whole heads. No block costs more than one item charge plus two
    stages above the ideal share. Every piece of a cut head holds at least
    one cut.
    """
    g = np.random.default_rng(1000 + seed)
    Hkv = int(g.choice([1, 2, 3, 4, 8]))
    gqa = int(g.choice([1, 2, 4, 8]))
    B = int(g.integers(1, 7))
    P = int(g.choice([8, 16, 32, 64, 128]))
    L = g.integers(1, 6001, size=B).astype(np.int32)
    budget = g.integers(1, 8001, size=(B, Hkv)).astype(np.int32)
    G = int(g.integers(1, min(Hkv, 4) + 1))
    hg = np.concatenate([np.arange(G), g.integers(0, G, size=Hkv - G)]).astype(np.int32)
    g.shuffle(hg)
    num_ctas = int(g.choice([1, 2, 3, 7, 50, 152, 304, 900]))
    plan = kvx.kvx_plan_create(B, gqa * Hkv, Hkv, 128, P, G, kvx.KVX_BF16, budget, L, hg,
                               num_ctas)
    n = orc.resolve_budget(budget, L).reshape(-1)
    assert np.array_equal(plan.kept().reshape(-1), n)
    items, off = plan.items()
    assert len(off) == num_ctas + 1 and off[0] == 0 and off[-1] == len(items)
    bad, count = orc.plan_coverage(n, items)
    assert bad == 0
    assert np.array_equal(plan.coverage(), count)
    T, c0 = min(P, 32), plan.stats()["item_overhead"]  # cut granularity, item charge
    for bh, b, e in items[:, :3]:
        assert b % T == 0 and (e % T == 0 or e == n[bh]), (bh, b, e)
    pieces = np.bincount(items[:, 0], minlength=n.size)
    cta_of = np.repeat(np.arange(num_ctas), np.diff(off))
    for bh in np.flatnonzero(pieces > 1):
        mine = items[:, 0] == bh
        assert np.all(np.diff(np.sort(cta_of[mine])) == 1), bh
        # no sliver: every piece of a cut head holds at least one cut
        assert np.all(items[mine, 2] - items[mine, 1] >= T), (bh, items[mine])
    cost = []
    for c in range(num_ctas):
        blk = items[off[c]:off[c + 1]]
        split = pieces[blk[:, 0]] > 1
        assert not np.any(split[1:] & ~split[:-1]), (c, blk)  # split pieces first
        cost.append(int((blk[:, 2] - blk[:, 1]).sum()) + c0 * len(blk))
    ideal = (int(n.sum()) + c0 * n.size + c0 * (num_ctas - 1)) / num_ctas
    assert max(cost) <= ideal + c0 + 2 * T + 1, (max(cost), ideal)


def test_coverage_record_stride_is_checked(kvx):
    """kvx_plan_set_coverage_record needs a row per head at least as long as
    the longest kept set; no device memory is touched by the call."""
    case = synth.tiny(0)
    plan = _plan(kvx, case, num_ctas=2)
    assert int(plan.kept().max()) == 100
    with pytest.raises(kvx.KvxError) as e:
        plan.set_coverage_record(1 << 20, 99)
    assert e.value.status == kvx.KVX_ERANGE
    plan.set_coverage_record(1 << 20, 100)
    plan.set_coverage_record(None)


CLUSTER_POLICIES = {2: 3, 4: 4, 8: 5}  # cluster size -> KVX_PLAN_CLUSTER_*


def check_cluster_plan(orc, plan, n, C, num_ctas):
    """Structure of a cluster layout: exact coverage (oracle count array); a
    cut head's pieces lie on blocks of one cluster, at most C of them, each
    the last item of its block and at most one per block; cuts fall on stage
    boundaries except at a head's end."""
    items, off = plan.items()
    assert len(off) == num_ctas + 1 and off[-1] == len(items)
    bad, count = orc.plan_coverage(n, items)
    assert bad == 0
    assert np.array_equal(plan.coverage(), count)
    assert plan.stats()["cluster"] == C and plan.stats()["num_slots"] == 0
    cta_of = np.repeat(np.arange(num_ctas), np.diff(off))
    pieces = np.bincount(items[:, 0], minlength=n.size)
    is_last = np.zeros(len(items), bool)
    is_last[off[1:][np.diff(off) > 0] - 1] = True
    per_block = np.zeros(num_ctas, int)
    for i, (bh, b, e, slot) in enumerate(items):
        assert slot == -1
        if pieces[bh] > 1:
            assert is_last[i], (bh, i)
            per_block[cta_of[i]] += 1
            assert b % 32 == 0 and (e % 32 == 0 or e == n[bh]), (bh, b, e)
    assert per_block.max(initial=0) <= 1
    for bh in np.flatnonzero(pieces > 1):
        blocks = cta_of[items[:, 0] == bh]
        assert 2 <= blocks.size <= C
        assert len(set((blocks // C).tolist())) == 1, (bh, blocks)
    return items, off, pieces


@pytest.mark.parametrize("C", [2, 4, 8])
def test_cluster_layout_on_the_sparse_workload(kvx, orc, C):
    """Llama-3-8B sparse layer (64 heads of 2176 kept tokens) on 304 blocks:
    every head is cut inside one cluster; with clusters of 4 or 8 every block
    of a used cluster streams 544 tokens (one head per four blocks)."""
    cfg = synth.decode_config("llama3_sparse", seed=0, layers=1)
    plan = kvx.kvx_plan_create(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.P, cfg.num_groups,
                               kvx.KVX_BF16, cfg.budget[0], cfg.seq_len, cfg.head_group[0],
                               304, CLUSTER_POLICIES[C])
    n = cfg.n[0].reshape(-1)
    items, off, pieces = check_cluster_plan(orc, plan, n, C, 304)
    assert np.all(pieces > 1)
    if C >= 4:
        assert plan.stats()["max_cta_tokens"] == 544


@pytest.mark.parametrize("seed", range(30))
def test_cluster_layout_random_shapes(kvx, orc, seed):
    """Seeded random shapes, budgets and block counts under every cluster
    size: the layout's structure and exact coverage."""
    g = np.random.default_rng(5000 + seed)
    C = int(g.choice([2, 4, 8]))
    Hkv = int(g.choice([1, 2, 4, 8]))
    B = int(g.integers(1, 9))
    L = g.integers(1, 9001, size=B).astype(np.int32)
    budget = g.integers(1, 12001, size=(B, Hkv)).astype(np.int32)
    G = int(g.integers(1, min(Hkv, 3) + 1))
    hg = np.concatenate([np.arange(G), g.integers(0, G, size=Hkv - G)]).astype(np.int32)
    num_ctas = C * int(g.integers(1, 40))
    plan = kvx.kvx_plan_create(B, 4 * Hkv, Hkv, 128, 16, G, kvx.KVX_BF16, budget, L, hg,
                               num_ctas, CLUSTER_POLICIES[C])
    n = orc.resolve_budget(budget, L).reshape(-1)
    check_cluster_plan(orc, plan, n, C, num_ctas)


def test_cluster_layout_rejects_bad_arguments(kvx):
    case = synth.tiny(0)
    for num_ctas, kernel, want in ((6, 0, kvx.KVX_EINVAL),   # not a multiple of 4 (fp32: SIMT)
                                   (8, 0, kvx.KVX_EUNSUPPORTED)):  # fp32 runs on the SIMT kernel
        with pytest.raises(kvx.KvxError) as e:
            _plan(kvx, case, num_ctas=num_ctas, policy=kvx.KVX_PLAN_CLUSTER_4, kernel=kernel)
        assert e.value.status in (want, kvx.KVX_EUNSUPPORTED)
    bf = synth.dense_case(2, 8, 2, 64, [37, 100], [[37, 20], [100, 20]], "bf16", seed=0)
    with pytest.raises(kvx.KvxError) as e:
        _plan(kvx, bf, num_ctas=6, policy=kvx.KVX_PLAN_CLUSTER_4)
    assert e.value.status == kvx.KVX_EINVAL
