"""Pins that tie the CPU oracle to facts fixed outside itself.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with: a hand-worked example under tests/golden/, a closed form, a
library routine (torch's scaled-dot-product attention in float64), or an
invariant of the definition. The same pins run against the real oracle
(test_oracle_pins.py) and against copies with planted mistakes
(test_oracle_mutants.py), which shows that each plausible mistake is caught.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append(vals)
    return rows


def _floats(v):
    return np.array([float(x) for x in v], dtype=np.float64)


def _ints(v):
    return np.array([int(x) for x in v], dtype=np.int32)


# ------------------------------------------------------------- attention
def pin_golden_two_token(orc):
    g = read_golden("attn_two_token.txt")
    D, L = int(g["D"][0][0]), int(g["L"][0][0])
    q = _floats(g["q"][0]).reshape(1, D)
    k = np.stack([_floats(r) for r in g["k"]])
    v = np.stack([_floats(r) for r in g["v"]])
    out, w = orc.attn_head(q, k, v, _ints(g["kept"][0]), float(g["scale"][0][0]), True)
    assert np.allclose(out[0], _floats(g["out"][0]), rtol=0, atol=1e-13), out
    assert np.allclose(w[0], _floats(g["weights"][0]), rtol=0, atol=1e-15), w


def pin_golden_kept_subset(orc):
    g = read_golden("attn_kept_subset.txt")
    D = int(g["D"][0][0])
    q = _floats(g["q"][0]).reshape(1, D)
    k = np.stack([_floats(r) for r in g["k"]])
    v = np.stack([_floats(r) for r in g["v"]])
    out, w = orc.attn_head(q, k, v, _ints(g["kept"][0]), float(g["scale"][0][0]), True)
    assert np.allclose(out[0], _floats(g["out"][0]), rtol=0, atol=1e-13), out
    assert np.allclose(w[0], _floats(g["weights"][0]), rtol=0, atol=1e-15), w


def _case(seed=3, B=2, Hq=8, Hkv=2, D=64, L=(29, 70)):
    gen = synth.rng(seed)
    Lmax = max(L)
    q = gen.standard_normal((B, Hq, D))
    k = gen.standard_normal((B, Hkv, Lmax, D))
    v = gen.standard_normal((B, Hkv, Lmax, D))
    return q, k, v, np.array(L, dtype=np.int32)


def pin_full_budget_equals_sdpa(orc):
    """Every token kept: the oracle must equal dense, unpaged attention as
    torch computes it (float64, grouped-query heads expanded by torch)."""
    q, k, v, L = _case()
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    for b in range(B):
        Lb = int(L[b])
        kept = [np.arange(Lb, dtype=np.int32)] * Hkv
        got = orc.decode_attn(q[b:b + 1], k[b:b + 1, :, :Lb], v[b:b + 1, :, :Lb],
                              L[b:b + 1], kept, 1.0 / math.sqrt(D))
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[b:b + 1, :, None, :]), torch.from_numpy(k[b:b + 1, :, :Lb]),
            torch.from_numpy(v[b:b + 1, :, :Lb]), enable_gqa=True).numpy()[:, :, 0, :]
        assert np.abs(got - ref).max() <= 1e-12, np.abs(got - ref).max()


def pin_subset_equals_sdpa_on_kept_rows(orc):
    """Random kept subsets: equal to torch attention over just the kept rows,
    with every other row set to NaN in the oracle's input."""
    q, k, v, L = _case(seed=5)
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    gen = synth.rng(11)
    kept = []
    for b in range(B):
        for h in range(Hkv):
            n = int(gen.integers(1, L[b] + 1))
            kept.append(synth.kept_random(gen, int(L[b]), n))
    kn, vn = np.full_like(k, np.nan), np.full_like(v, np.nan)
    for b in range(B):
        for h in range(Hkv):
            ix = kept[b * Hkv + h]
            kn[b, h, ix] = k[b, h, ix]
            vn[b, h, ix] = v[b, h, ix]
    got = orc.decode_attn(q, kn, vn, L, kept, 1.0 / math.sqrt(D))
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hkv):
            ix = kept[b * Hkv + h]
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[b, h * g:(h + 1) * g, None, :]),
                torch.from_numpy(k[b, h][ix][None].repeat(g, 0)),
                torch.from_numpy(v[b, h][ix][None].repeat(g, 0))).numpy()[:, 0, :]
            d = np.abs(got[b, h * g:(h + 1) * g] - ref).max()
            assert d <= 1e-12, (b, h, d)


def pin_single_token(orc):
    """n = 1: the weight is 1, the output is that token's value row, exactly."""
    gen = synth.rng(1)
    D, L = 16, 9
    q = gen.standard_normal((3, D))
    k = gen.standard_normal((L, D)) * 10
    v = gen.standard_normal((L, D))
    for t in (0, 4, 8):
        out = orc.attn_head(q, k, v, np.array([t], np.int32), 0.25)
        assert np.array_equal(out, np.repeat(v[t][None], 3, 0)), (t, out)


def pin_equal_keys_give_mean(orc):
    gen = synth.rng(2)
    D, L = 8, 12
    q = gen.standard_normal((2, D))
    k = np.repeat(gen.standard_normal((1, D)), L, 0)
    v = gen.standard_normal((L, D))
    idx = np.array([1, 2, 5, 11], np.int32)
    out = orc.attn_head(q, k, v, idx, 0.3)
    assert np.abs(out - v[idx].mean(0)).max() <= 1e-13


def pin_constant_values(orc):
    gen = synth.rng(4)
    D, L = 8, 10
    q = gen.standard_normal((2, D)) * 3
    k = gen.standard_normal((L, D)) * 3
    c = gen.standard_normal(D)
    v = np.repeat(c[None], L, 0)
    out = orc.attn_head(q, k, v, np.array([0, 3, 4, 9], np.int32), 1.0)
    assert np.abs(out - c[None]).max() <= 1e-13


def pin_zero_query_gives_mean(orc):
    gen = synth.rng(6)
    D, L = 8, 10
    k = gen.standard_normal((L, D)) * 5
    v = gen.standard_normal((L, D))
    idx = np.array([0, 2, 3, 7, 8], np.int32)
    out = orc.attn_head(np.zeros((1, D)), k, v, idx, 0.5)
    assert np.abs(out[0] - v[idx].mean(0)).max() <= 1e-13


def pin_dominant_key(orc):
    """One kept key aligned with q at a huge score: its weight is 1 to within
    exp(-gap); the output is its value row (and nothing overflows)."""
    gen = synth.rng(7)
    D, L = 8, 6
    q = gen.standard_normal((1, D))
    k = gen.standard_normal((L, D))
    k[3] = q[0] * 1e3
    v = gen.standard_normal((L, D))
    out = orc.attn_head(q, k, v, np.arange(L, dtype=np.int32), 1.0 / math.sqrt(D))
    assert np.all(np.isfinite(out))
    assert np.abs(out[0] - v[3]).max() <= 1e-12


def pin_weights_sum_to_one(orc):
    gen = synth.rng(8)
    for D, L, n in ((64, 300, 120), (128, 50, 50), (8, 7, 1)):
        q = gen.standard_normal((4, D)) * 2
        k = gen.standard_normal((L, D)) * 2
        v = gen.standard_normal((L, D))
        idx = synth.kept_random(gen, L, n)
        _, w = orc.attn_head(q, k, v, idx, 1.0 / math.sqrt(D), True)
        assert np.all(w >= 0)
        assert np.abs(w.sum(1) - 1.0).max() <= 1e-12


def pin_scale_invariance(orc):
    """(lambda q, scale / lambda) gives the same scores, so the same output."""
    gen = synth.rng(9)
    D, L = 32, 40
    q = gen.standard_normal((2, D))
    k = gen.standard_normal((L, D))
    v = gen.standard_normal((L, D))
    idx = synth.kept_random(gen, L, 17)
    a = orc.attn_head(q, k, v, idx, 0.2)
    b = orc.attn_head(q * 4.0, k, v, idx, 0.05)
    assert np.abs(a - b).max() <= 1e-13


def pin_gqa_mapping(orc):
    """Each KV head carries its own constant value row: query head j must
    return the constant of KV head floor(j / g) (contiguous grouping, as
    torch's grouped-query attention maps heads)."""
    B, Hq, Hkv, D, L = 1, 8, 4, 4, 6
    gen = synth.rng(10)
    q = gen.standard_normal((B, Hq, D))
    k = gen.standard_normal((B, Hkv, L, D))
    v = np.zeros((B, Hkv, L, D))
    for h in range(Hkv):
        v[0, h] = float(h + 1)
    kept = [np.arange(L, dtype=np.int32)] * Hkv
    out = orc.decode_attn(q, k, v, np.array([L], np.int32), kept, 0.5)
    for j in range(Hq):
        assert np.abs(out[0, j] - (j // (Hq // Hkv) + 1)).max() <= 1e-13, (j, out[0, j])


def pin_budget_resolution(orc):
    """n = min(L, budget): a budget above the length keeps the whole sequence."""
    budget = np.array([[5, 1 << 30], [40, 7]], np.int32)
    L = np.array([10, 30], np.int32)
    n = orc.resolve_budget(budget, L)
    assert np.array_equal(n, np.array([[5, 10], [30, 7]], np.int32)), n


# ---------------------------------------------------------- head groups
def pin_group_pages(orc):
    """Group pages = ceil(max kept count of the group's heads / P)."""
    n = np.array([[17, 5, 16, 1], [3, 33, 32, 64]], np.int32)
    per_head = orc.group_pages(n, [0, 1, 2, 3], 16)
    assert np.array_equal(per_head, np.array([[2, 1], [1, 3], [1, 2], [1, 4]], np.int32))
    one = orc.group_pages(n, [0, 0, 0, 0], 16)
    assert np.array_equal(one, np.array([[2, 4]], np.int32))
    two = orc.group_pages(n, [0, 1, 0, 1], 16)
    # group 0 = heads {0, 2}: max(17, 16) -> 2 pages, max(3, 32) -> 2 pages
    # group 1 = heads {1, 3}: max(5, 1) -> 1 page,   max(33, 64) -> 4 pages
    assert np.array_equal(two, np.array([[2, 2], [1, 4]], np.int32)), two


def pin_footprint(orc):
    """One group over all heads is the unified page: pages x Hkv x P x 2 x D x bytes."""
    n = np.array([[37, 20], [100, 20]], np.int32)
    one = orc.footprint_bytes(n, [0, 0], 16, 64, 4)
    assert np.array_equal(one, np.array([3 * 2 * 16 * 2 * 64 * 4, 7 * 2 * 16 * 2 * 64 * 4]))
    per = orc.footprint_bytes(n, [0, 1], 16, 64, 4)
    assert np.array_equal(per, np.array([(3 + 2) * 16 * 2 * 64 * 4, (7 + 2) * 16 * 2 * 64 * 4]))


# ----------------------------------------------------------- plan cover
def pin_plan_coverage(orc):
    n = np.array([5, 3], np.int32)
    ok = [[0, 0, 3, 0], [0, 3, 5, 1], [1, 0, 3, -1]]
    bad, count = orc.plan_coverage(n, ok)
    assert bad == 0 and count[0, :5].tolist() == [1] * 5
    assert orc.plan_coverage(n, [[0, 0, 2, 0], [0, 3, 5, 1], [1, 0, 3, -1]])[0] == 1  # gap
    assert orc.plan_coverage(n, [[0, 0, 3, 0], [0, 2, 5, 1], [1, 0, 3, -1]])[0] == 1  # overlap
    assert orc.plan_coverage(n, [[0, 0, 5, -1], [1, 0, 4, -1]])[0] == 1  # past n
    assert orc.plan_coverage(n, [[0, 0, 5, -1], [1, 0, 3, -1], [1, 2, 2, 0]])[0] == 1  # empty
    assert orc.plan_coverage(n, [[0, 0, 5, -1]])[0] == 3  # head 1 uncovered


# ---------------------------------------------------------------- gather
def _gather_golden():
    g = read_golden("gather_tiny.txt")
    S, mb = int(g["S"][0][0]), int(g["max_blocks"][0][0])
    bb, nphys = int(g["block_bytes"][0][0]), int(g["num_phys"][0][0])
    fill = int(g["fill"][0][0])
    nb = _ints(g["nb"][0])
    bt = np.stack([_ints(r) for r in g["bt"]])
    pool = np.arange(nphys * bb, dtype=np.uint8).reshape(nphys, bb)
    rows = np.stack([np.array([int(x) for x in r], np.uint8) for r in g["row"]])
    runs = [_ints(r).reshape(-1, 3) for r in g["runs"]]
    return S, mb, bb, fill, nb, bt, pool, rows, runs, int(g["run_total"][0][0])


def pin_gather_golden(orc):
    S, mb, bb, fill, nb, bt, pool, rows, _, _ = _gather_golden()
    st = np.full((S, mb * bb), fill, dtype=np.uint8)
    orc.gather(bt, nb, pool, st)
    assert np.array_equal(st, rows), st
    st = np.full((S, mb * bb), fill, dtype=np.uint8)
    orc.gather(bt, nb, pool, st, zero_tail=True)
    assert np.array_equal(st, np.where(rows == fill, 0, rows).astype(np.uint8))


def pin_runs_golden(orc):
    S, mb, bb, fill, nb, bt, pool, rows, runs, total = _gather_golden()
    tot, cnt, got = orc.runs(bt, nb)
    assert tot == total
    for s in range(S):
        assert cnt[s] == len(runs[s])
        assert np.array_equal(got[s, :cnt[s]], runs[s]), (s, got[s, :cnt[s]])


def pin_runs_closed_form(orc):
    """Run count = breaks in physical contiguity + non-empty rows; the runs
    tile each row exactly and each is physically contiguous."""
    cfg = synth.gather_config(seed=3, S=12, Lmin=16, Lmax=640, num_phys=4096, extents=True,
                              max_extent=9)
    tot, cnt, runs = orc.runs(cfg.bt, cfg.nb)
    breaks = 0
    for s in range(cfg.S):
        row = cfg.bt[s, :cfg.nb[s]].astype(np.int64)
        breaks += int(np.count_nonzero(np.diff(row) != 1))
        covered = 0
        for r in runs[s, :cnt[s]]:
            assert r[1] == covered
            assert np.array_equal(cfg.bt[s, r[1]:r[1] + r[2]], r[0] + np.arange(r[2]))
            covered += r[2]
        assert covered == cfg.nb[s]
    assert tot == breaks + int(np.count_nonzero(cfg.nb))


def pin_gather_stamped_blocks(orc):
    """Blocks carry their own id in their first 8 bytes: every staging block
    must name the physical block the table points at."""
    cfg = synth.gather_config(seed=4, S=6, Lmin=16, Lmax=256, block_tokens=16,
                              token_bytes=4, num_phys=128)
    pool = synth.block_stamp_pool(cfg.num_phys, cfg.block_bytes, seed=1)
    st = np.zeros((cfg.S, cfg.row_bytes), np.uint8)
    orc.gather(cfg.bt, cfg.nb, pool, st)
    for s in range(cfg.S):
        blocks = st[s].reshape(cfg.max_blocks, cfg.block_bytes)
        ids = blocks[:, :8].copy().view(np.int64)[:, 0]
        assert np.array_equal(ids[:cfg.nb[s]], cfg.bt[s, :cfg.nb[s]])
        assert np.array_equal(blocks[:cfg.nb[s]], pool[cfg.bt[s, :cfg.nb[s]]])
        assert not blocks[cfg.nb[s]:].any()


# ------------------------------------------------------ sparse selection
def pin_select_closed_form(orc):
    """Keys along one axis with known scores: the kept set is the top positions
    by that coordinate plus the recent window, ascending."""
    L, D, top, recent = 40, 8, 5, 3
    q = np.zeros((2, D))
    q[0, 2], q[1, 2] = 1.5, 0.5          # Q = 2 e_2 (sum of the two query heads)
    c = synth.rng(13).permutation(L).astype(np.float64)
    k = np.zeros((L, D))
    k[:, 2] = c
    kept = orc.select_topk(q, k, top, recent)
    cand = np.arange(L - recent)
    best = cand[np.argsort(-c[cand])[:top]]
    expect = np.sort(np.concatenate([best, np.arange(L - recent, L)]))
    assert np.array_equal(kept, expect), (kept, expect)


def pin_select_ties_and_edges(orc):
    D = 4
    q = np.array([[1.0, -2.0, 0.5, 0.0], [-1.0, 2.0, -0.5, 0.0]])  # Q = 0: every score ties
    k = synth.rng(14).standard_normal((30, D))
    assert np.array_equal(orc.select_topk(q, k, 4, 2), [0, 1, 2, 3, 28, 29])
    # budget at least the candidates: everything is kept
    assert np.array_equal(orc.select_topk(q, k, 40, 2), np.arange(30))
    # sequence shorter than the recent window: everything is kept
    assert np.array_equal(orc.select_topk(q, k[:3], 4, 5), np.arange(3))


def pin_select_permutation_equivariance(orc):
    """Relabelling token positions (away from the recent window) relabels the
    selection; the recent window stays."""
    gen = synth.rng(15)
    L, D, top, recent = 60, 16, 7, 4
    q = gen.standard_normal((4, D))
    k = gen.standard_normal((L, D))
    perm = np.concatenate([gen.permutation(L - recent), np.arange(L - recent, L)])
    a = orc.select_topk(q, k, top, recent)
    inv = np.argsort(perm)
    b = orc.select_topk(q, k[perm], top, recent)
    assert np.array_equal(np.sort(perm[b]), a)


# ------------------------------------------------ KV-RM block pager
def read_frame_golden():
    """(S, max_blocks, num_phys, steps, refcount) of tests/golden/frame_edits.txt;
    a step is (op, args, code, views, free)."""
    cfg, steps, rc = None, [], None
    with open(os.path.join(GOLDEN, "frame_edits.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("config"):
                cfg = [int(x) for x in line.split()[1:]]
            elif line.startswith("refcount"):
                rc = [int(x) for x in line.split()[1:]]
            elif line.startswith("step"):
                cols = [c.strip() for c in line[len("step"):].split("|")]
                op, *args = cols[0].split()
                ints = lambda c: [] if c == "-" else [int(x) for x in c.split()]
                steps.append((op, [int(x) for x in args], int(cols[1]),
                              [ints(c) for c in cols[2:-1]], ints(cols[-1])))
    return cfg[0], cfg[1], cfg[2], steps, rc


def pager_views(pager):
    table, nb, rc = pager.state()
    return [list(table[s, :nb[s]]) for s in range(table.shape[0])], table, nb, rc


def replay_frame_golden(pager, S, M, N, steps, rc_final):
    """Replays the hand-worked edit sequence on any pager with reserve / alias /
    trim / state and checks every intermediate state."""
    for i, (op, args, code, views, free) in enumerate(steps):
        before = pager_views(pager)[0]
        if op == "reserve":
            got, ids = pager.reserve(*args)
        else:
            got = getattr(pager, op)(*args)
        assert got == code, (i, op, args, got, code)
        now, table, nb, rc = pager_views(pager)
        assert now == views, (i, op, args, now, views)
        assert list(np.flatnonzero(rc == 0)) == free, (i, op, np.flatnonzero(rc == 0), free)
        assert np.all(table[np.arange(M)[None, :] >= nb[:, None]] == -1)
        if op == "reserve" and code == 0:
            s = args[0]
            assert list(ids) == now[s][len(before[s]):], (i, ids)
    assert list(pager_views(pager)[3]) == rc_final


def pin_frame_golden(orc):
    S, M, N, steps, rc = read_frame_golden()
    replay_frame_golden(orc.frame(S, M, N), S, M, N, steps, rc)


def pin_frame_closed_form(orc):
    """On a fresh pool, consecutive reserves lay the sequences end to end;
    ending every sequence frees the whole pool, after which one reserve of
    the whole pool takes blocks 0..N-1 in order."""
    S, M, N = 5, 12, 40
    f = orc.frame(S, M, N)
    sizes = [3, 7, 1, 12, 5]
    off = 0
    for s, c in enumerate(sizes):
        code, ids = f.reserve(s, c)
        assert code == 0 and list(ids) == list(range(off, off + c)), (s, ids)
        off += c
    views, table, nb, rc = pager_views(f)
    assert list(nb) == sizes and rc.sum() == sum(sizes)
    assert np.all(rc[:off] == 1) and np.all(rc[off:] == 0)
    for s in range(S):
        assert f.trim(s, 0, 0) == 0
    assert not pager_views(f)[3].any()
    g = orc.frame(1, N, N)
    code, ids = g.reserve(0, N)
    assert code == 0 and list(ids) == list(range(N))
    assert g.reserve(0, 1)[0] == -2  # view full
    h = orc.frame(2, 4, 3)
    assert h.reserve(0, 4)[0] == -3 and h.reserve(0, 3)[0] == 0


def pin_frame_invariants(orc):
    """Random edit streams: every block's reference count equals the number of
    view entries naming it, free blocks are exactly the unreferenced ones, a
    failed edit changes nothing, Trim keeps exactly the asked slice, Alias
    copies the source entries as they were, and Reserve hands out free blocks
    only, distinct, appended in order."""
    gen = synth.rng(77)
    S, M, N = 6, 12, 40
    f = orc.frame(S, M, N)
    for it in range(600):
        views, table, nb, rc = pager_views(f)
        op = gen.integers(0, 3)
        if op == 0:
            s, c = int(gen.integers(0, S)), int(gen.integers(0, 5))
            code, ids = f.reserve(s, c)
            ok = nb[s] + c <= M and c <= int((rc == 0).sum())
            assert (code == 0) == ok, (it, code)
            if ok:
                assert len(set(ids.tolist())) == c and np.all(rc[ids] == 0)
        elif op == 1:
            dst, src = int(gen.integers(0, S)), int(gen.integers(0, S))
            c = int(gen.integers(0, 4))
            sj, dj = int(gen.integers(0, nb[src] + 2)), int(gen.integers(0, nb[dst] + 2))
            code = f.alias(dst, dj, src, sj, c)
            ok = sj + c <= nb[src] and dj <= nb[dst] and dj + c <= M
            assert (code == 0) == ok, (it, code)
            if ok:
                now = pager_views(f)[0]
                assert now[dst][dj:dj + c] == views[src][sj:sj + c]
                assert now[dst][:dj] == views[dst][:dj]
                assert now[dst][dj + c:] == views[dst][dj + c:]
        else:
            s = int(gen.integers(0, S))
            b = int(gen.integers(0, nb[s] + 2))
            e = int(gen.integers(0, nb[s] + 2))
            code = f.trim(s, b, e)
            ok = b <= e <= nb[s]
            assert (code == 0) == ok, (it, code)
            if ok:
                assert pager_views(f)[0][s] == views[s][b:e]
        now, table2, nb2, rc2 = pager_views(f)
        if code != 0:
            assert now == views and np.array_equal(rc2, rc)
        count = np.bincount(np.concatenate([np.asarray(v, np.int64) for v in now] + [[]]).astype(
            np.int64), minlength=N)
        assert np.array_equal(count, rc2), it
        edited = s if op != 1 else dst
        for r in range(S):
            if r != edited:
                assert now[r] == views[r], (it, r)


ALL_PINS = [
    pin_golden_two_token, pin_golden_kept_subset, pin_full_budget_equals_sdpa,
    pin_subset_equals_sdpa_on_kept_rows, pin_single_token, pin_equal_keys_give_mean,
    pin_constant_values, pin_zero_query_gives_mean, pin_dominant_key,
    pin_weights_sum_to_one, pin_scale_invariance, pin_gqa_mapping,
    pin_budget_resolution, pin_group_pages, pin_footprint, pin_plan_coverage,
    pin_gather_golden, pin_runs_golden, pin_runs_closed_form, pin_gather_stamped_blocks,
    pin_select_closed_form, pin_select_ties_and_edges, pin_select_permutation_equivariance,
    pin_frame_golden, pin_frame_closed_form, pin_frame_invariants,
]
