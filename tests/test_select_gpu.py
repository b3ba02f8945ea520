"""Sparse kept-set selection (kvx_select_topk), page packing (kvx_pack_kept)
and attention over the packed pages, against the fp64 oracle.

The cut is decided on fp32 scores, the oracle decides it on fp64 scores. The
unique part is compared exactly: every position whose score lies outside the
fp32 error band around the cut must be kept or dropped as the oracle decides;
positions inside the band may be exchanged, and the counts must agree. The
band is rigorous: for <k, Q> with Q = sum_j q_j summed in fp32,
|fl(score) - score| <= gamma_D * sum_d |k_d Q_d| + 3u * sum_d |k_d| sum_j |q_jd|,
u = 2^-24, gamma_D = D u / (1 - D u).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from paged_non_uniform_gb300 import kvx
import pages

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


def _bf16(a):
    return torch.from_numpy(synth.f32_to_bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()


def make(seed, B, Hq, Hkv, D, L, const_keys=False):
    g = synth.rng(seed)
    Lmax = int(max(L))
    q = synth.normal(g, (B, Hq, D), "bf16")
    k = synth.normal(g, (B, Hkv, Lmax, D), "bf16")
    v = synth.normal(g, (B, Hkv, Lmax, D), "bf16")
    if const_keys:
        k[:] = k[:, :, :1]
    return q, k, v, np.asarray(L, np.int32)


def gpu_select(q, k, L, top, recent):
    B, Hq, D = q.shape
    Hkv, Lmax = k.shape[1], k.shape[2]
    kept = torch.full((B * Hkv, top + recent), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(B * Hkv, dtype=torch.int32, device="cuda")
    ws = torch.zeros(kvx.kvx_select_workspace_bytes(B, Hkv, Lmax) // 4 + 64, dtype=torch.int32,
                     device="cuda")
    kvx.kvx_select_topk(_bf16(k), _bf16(q), torch.from_numpy(L).cuda(), B, Hq, Hkv, D, Lmax,
                        top, recent, kept, cnt, ws)
    torch.cuda.synchronize()
    return kept.cpu().numpy(), cnt.cpu().numpy()


def check_head(orc, qh, kh, top, recent, got):
    """got: GPU kept positions of one head. Returns True if equal to the oracle's."""
    ref, sc = orc.select_topk(qh, kh, top, recent, want_scores=True)
    assert got.size == ref.size
    assert np.all(np.diff(got) > 0)
    L = kh.shape[0]
    n = max(0, L - recent)
    assert np.array_equal(got[got >= n], np.arange(n, L))
    if np.array_equal(got, ref):
        return True
    D = kh.shape[1]
    Q = qh.astype(np.float64).sum(0)
    gam = D * U / (1 - D * U)
    eps = gam * np.abs(kh[:n]) @ np.abs(Q) + 3 * U * np.abs(kh[:n]) @ np.abs(qh).sum(0)
    thr = np.sort(sc[:n])[::-1][min(top, n) - 1]
    amb = np.abs(sc[:n] - thr) <= eps + eps.max()
    diff = np.setxor1d(got, ref)
    assert np.all(amb[diff]), diff[~amb[diff]]
    return False


@pytest.mark.parametrize("D", [128, 64])
def test_selection_matches_oracle(D):
    q, k, v, L = make(1, 3, 16, 4, D, [5000, 3100, 700])
    top, recent = 300, 64
    kept, cnt = gpu_select(q, k, L, top, recent)
    orc = oracle.load()
    same = 0
    for b in range(3):
        for h in range(4):
            bh = b * 4 + h
            c = int(cnt[bh])
            assert c == min(top, L[b] - recent) + min(recent, L[b])
            assert np.all(kept[bh, c:] == -1)
            same += check_head(orc, q[b, 4 * h:4 * h + 4], k[b, h, :L[b]], top, recent,
                               kept[bh, :c])
    assert same >= 10


def test_selection_ties_and_edges():
    orc = oracle.load()
    # all keys of a head equal: every score ties, the lowest positions win
    q, k, v, L = make(2, 2, 8, 2, 128, [900, 400], const_keys=True)
    kept, cnt = gpu_select(q, k, L, 50, 10)
    for bh in range(4):
        b = bh // 2
        exp = np.concatenate([np.arange(50), np.arange(L[b] - 10, L[b])])
        assert np.array_equal(kept[bh, :cnt[bh]], exp)
    # budget >= candidates, sequence shorter than the window, no top at all
    q, k, v, L = make(3, 3, 8, 2, 128, [120, 5, 300])
    for top, recent in ((200, 16), (0, 16), (10, 0)):
        kept, cnt = gpu_select(q, k, L, top, recent)
        for bh in range(6):
            b = bh // 2
            h = bh % 2
            ref = orc.select_topk(q[b, 4 * h:4 * h + 4], k[b, h, :L[b]], top, recent)
            assert cnt[bh] == ref.size
            check_head(orc, q[b, 4 * h:4 * h + 4], k[b, h, :L[b]], top, recent,
                       kept[bh, :cnt[bh]])


@pytest.mark.parametrize("layout", [kvx.KVX_LAYOUT_HEAD_MAJOR, kvx.KVX_LAYOUT_TOKEN_MAJOR])
def test_select_pack_attend_end_to_end(layout):
    """GPU selection -> packing into head-group pages -> attention, against the
    oracle's selection and attention, head by head where the kept sets agree;
    the packed slots are compared bit for bit with the dense rows, and
    attention straight over the kept rows (kvx_decode_attn_kept, same plan)
    with the packed path's output."""
    B, Hq, Hkv, D, P = 2, 32, 8, 128, 16
    top, recent = 512, 64
    q, k, v, L = make(4, B, Hq, Hkv, D, [6000, 4000])
    kept, cnt = gpu_select(q, k, L, top, recent)
    n = cnt.reshape(B, Hkv)
    hg = np.array([0, 0, 0, 0, 1, 1, 1, 1], np.int32)
    plan = kvx.kvx_plan_create(B, Hq, Hkv, D, P, 2, kvx.KVX_BF16, n, L, hg, 11, layout=layout)
    kvx.kvx_plan_upload(plan)
    gp = plan.group_pages()
    tables, npages = pages.assign_pages(gp, [synth.page_permutation(40 + i, int(gp[i].sum()) + 2)
                                             for i in range(2)], 2)
    sizes = pages.group_sizes(hg)
    shape = (lambda i: (npages[i], P, int(sizes[i]), D)) if layout else \
        (lambda i: (npages[i], int(sizes[i]), P, D))
    kp = [torch.zeros(shape(i), dtype=torch.bfloat16, device="cuda") for i in range(2)]
    vp = [torch.zeros(shape(i), dtype=torch.bfloat16, device="cuda") for i in range(2)]
    pt = [torch.from_numpy(t).cuda() for t in tables]
    ws = torch.zeros(plan.workspace_bytes() // 4 + 64, dtype=torch.int32, device="cuda")
    kd, vd = _bf16(k), _bf16(v)
    kvx.kvx_pack_kept(plan, kd, vd, k.shape[2], torch.from_numpy(kept).cuda(), top + recent, kp,
                      vp, npages, pt, [t.shape[1] for t in tables], ws)
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    kvx.kvx_decode_attn(plan, _bf16(q), kp, vp, npages, pt, [t.shape[1] for t in tables],
                        torch.from_numpy(n.reshape(-1).copy()).cuda(),
                        torch.from_numpy(L).cuda(), 0.0, out, ws)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(ws) == 0
    got = out.cpu().numpy().astype(np.float64)
    # the same plan straight over the kept rows of the dense cache (no
    # packing): the same bits
    out2 = torch.full((B, Hq, D), float("nan"), device="cuda")
    kvx.kvx_decode_attn_kept(plan, _bf16(q), kd, vd, k.shape[2], torch.from_numpy(kept).cuda(),
                             top + recent, torch.from_numpy(n.reshape(-1).copy()).cuda(),
                             torch.from_numpy(L).cuda(), 0.0, out2, ws)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(ws) == 0
    assert np.array_equal(out2.cpu().numpy().astype(np.float64), got)
    # packed slots: bit-exact copies of the dense rows the GPU selected
    rows = pages.head_rows(hg)
    kbits = synth.f32_to_bf16_bits(k)
    kph = [p.view(torch.int16).cpu().numpy().view(np.uint16) for p in kp]
    for b in range(B):
        for h in range(Hkv):
            gi, r = int(hg[h]), int(rows[h])
            idx = kept[b * Hkv + h, :n[b, h]]
            t = np.arange(idx.size)
            pg = tables[gi][b, t // P]
            slots = kph[gi][pg, t % P, r] if layout else kph[gi][pg, r, t % P]
            assert np.array_equal(slots, kbits[b, h, idx])
    orc = oracle.load()
    g = Hq // Hkv
    agree = 0
    for b in range(B):
        for h in range(Hkv):
            qh, kh, vh = q[b, h * g:(h + 1) * g], k[b, h, :L[b]], v[b, h, :L[b]]
            if check_head(orc, qh, kh, top, recent, kept[b * Hkv + h, :n[b, h]]):
                agree += 1
                ref_idx = orc.select_topk(qh, kh, top, recent)
                ref = orc.attn_head(qh, kh, vh, ref_idx, 1.0 / math.sqrt(D))
                assert np.abs(got[b, h * g:(h + 1) * g] - ref).max() <= 2e-3
    assert agree >= 14


def test_selection_bucket_overflow_and_ragged():
    """All-equal keys put every candidate in the cut's bucket (more than a
    block keeps in shared memory, so the cut comes from scans of the scores
    in global memory); ragged lengths end inside a float4, a bitmask word
    and a block's share of the words."""
    orc = oracle.load()
    q, k, v, L = make(5, 1, 8, 2, 128, [20001], const_keys=True)
    kept, cnt = gpu_select(q, k, L, 300, 7)
    exp = np.concatenate([np.arange(300), np.arange(20001 - 7, 20001)])
    for bh in range(2):
        assert np.array_equal(kept[bh, :cnt[bh]], exp)
    q, k, v, L = make(6, 3, 8, 2, 64, [8197 + 3, 4101, 33])
    for top, recent in ((1000, 3), (4095, 1), (31, 2)):
        kept, cnt = gpu_select(q, k, L, top, recent)
        for bh in range(6):
            b, h = bh // 2, bh % 2
            ref = orc.select_topk(q[b, 4 * h:4 * h + 4], k[b, h, :L[b]], top, recent)
            assert cnt[bh] == ref.size
            assert np.all(kept[bh, cnt[bh]:] == -1)
            check_head(orc, q[b, 4 * h:4 * h + 4], k[b, h, :L[b]], top, recent,
                       kept[bh, :cnt[bh]])


def test_selection_longest_rows():
    """Rows at the library's maximum length (262144) and just past 131072:
    each of the four blocks of a head's cut cluster then owns its largest
    share of bitmask words (2048)."""
    g = synth.rng(9)
    L = np.array([262144, 131200], np.int32)
    q = synth.normal(g, (2, 4, 128), "bf16")
    k = synth.normal(g, (2, 1, int(L.max()), 128), "bf16")
    top, recent = 2048, 128
    kept, cnt = gpu_select(q, k, L, top, recent)
    orc = oracle.load()
    for b in range(2):
        assert cnt[b] == top + recent
        check_head(orc, q[b], k[b, 0, :L[b]], top, recent, kept[b, :cnt[b]])


def test_selection_cut_bucket_beyond_first_chunk():
    """Every candidate score lies in one first-digit bucket (6436 entries),
    spread over all four blocks of the head's cut cluster: more than the
    blocks' warp lists hold, so the last two digits come from scans of the
    scores in global memory, and the equal keys at the cut cross block
    boundaries. The scores 4 (1 + m/128) are exact in fp32 and fp64, so the
    kept set is unique: the top 2048 with ties at the lower position, then
    the recent window."""
    B, Hq, Hkv, D, L = 1, 8, 2, 128, 6500
    top, recent = 2048, 64
    g = synth.rng(12)
    q = np.zeros((B, Hq, D), np.float32)
    q[:, :, 0] = 1.0
    k = np.zeros((B, Hkv, L, D), np.float32)
    k[..., 0] = 1.0 + g.integers(0, 26, size=(B, Hkv, L)) / 128.0
    kept, cnt = gpu_select(q, k, np.array([L], np.int32), top, recent)
    orc = oracle.load()
    for h in range(Hkv):
        ref = orc.select_topk(q[0, 4 * h:4 * h + 4], k[0, h], top, recent)
        assert cnt[h] == ref.size == top + recent
        assert np.array_equal(kept[h, :cnt[h]], ref)


def test_selection_many_equal_keys_at_the_cut():
    """About 500 scattered candidates score exactly 4.03125 and about 500
    score 4.0; the rest score 1.0. The bucket (about 1000 entries) fits the
    blocks' lists, so the cluster's leader finds the cut from their keys in
    its shared memory. More than 32 keys share the cut's top 22 bits, so the
    last digit comes from a histogram rather than one warp. The top 300 are
    the 300 lowest positions scoring 4.03125, taken across the four blocks.
    Every score is exact in fp32 and fp64, so the kept set is unique."""
    B, Hq, Hkv, D, L = 1, 8, 2, 128, 20000
    top, recent = 300, 16
    g = synth.rng(14)
    q = np.zeros((B, Hq, D), np.float32)
    q[:, :, 0] = 1.0
    k = np.zeros((B, Hkv, L, D), np.float32)
    u = g.random((B, Hkv, L))
    k[..., 0] = np.where(u < 0.025, 1.0078125, np.where(u < 0.05, 1.0, 0.25))
    kept, cnt = gpu_select(q, k, np.array([L], np.int32), top, recent)
    orc = oracle.load()
    for h in range(Hkv):
        n = L - recent
        hi = np.flatnonzero(k[0, h, :n, 0] == 1.0078125)
        assert hi.size > top
        exp = np.concatenate([hi[:top], np.arange(n, L)])
        ref = orc.select_topk(q[0, 4 * h:4 * h + 4], k[0, h], top, recent)
        assert np.array_equal(ref, exp)
        assert cnt[h] == exp.size
        assert np.array_equal(kept[h, :cnt[h]], exp)


def test_selection_back_to_back_calls_share_a_workspace():
    """Two calls on one stream with one workspace and no synchronisation in
    between, on different keys and into different outputs. The second call's
    histogram clearing and score pass start as programmatic dependents while
    the first call's cut may still run; both kept sets must match the
    oracle."""
    orc = oracle.load()
    B, Hq, Hkv, D = 2, 8, 2, 128
    L = np.array([5000, 3100], np.int32)
    top, recent = 700, 20
    runs = []
    for seed in (21, 22):
        q, k, v, _ = make(seed, B, Hq, Hkv, D, L)
        runs.append((q, k))
    Lmax = int(L.max())
    ws = torch.zeros(kvx.kvx_select_workspace_bytes(B, Hkv, Lmax) // 4 + 64, dtype=torch.int32,
                     device="cuda")
    dev = [(_bf16(k), _bf16(q)) for q, k in runs]
    sl = torch.from_numpy(L).cuda()
    outs = [(torch.full((B * Hkv, top + recent), -7, dtype=torch.int32, device="cuda"),
             torch.zeros(B * Hkv, dtype=torch.int32, device="cuda")) for _ in runs]
    torch.cuda.synchronize()
    for (kd, qd), (kept, cnt) in zip(dev, outs):
        kvx.kvx_select_topk(kd, qd, sl, B, Hq, Hkv, D, Lmax, top, recent, kept, cnt, ws)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(ws) == 0
    for (q, k), (kept, cnt) in zip(runs, outs):
        kept, cnt = kept.cpu().numpy(), cnt.cpu().numpy()
        for bh in range(B * Hkv):
            b, h = bh // Hkv, bh % Hkv
            ref = orc.select_topk(q[b, 4 * h:4 * h + 4], k[b, h, :L[b]], top, recent)
            assert cnt[bh] == ref.size
            check_head(orc, q[b, 4 * h:4 * h + 4], k[b, h, :L[b]], top, recent,
                       kept[bh, :cnt[bh]])


def test_selection_bad_length_flagged():
    """A length above Lmax selects nothing for its sequence and sets the
    status bit; the other sequences are unaffected."""
    q, k, v, L = make(7, 2, 8, 2, 128, [300, 200])
    B, Hq, D = q.shape
    Lmax = k.shape[2]
    top, recent = 40, 8
    bad = np.array([Lmax + 1, 200], np.int32)
    kept = torch.full((4, top + recent), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(kvx.kvx_select_workspace_bytes(B, 2, Lmax) // 4 + 64, dtype=torch.int32,
                     device="cuda")
    kvx.kvx_select_topk(_bf16(k), _bf16(q), torch.from_numpy(bad).cuda(), B, Hq, 2, D, Lmax,
                        top, recent, kept, cnt, ws)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(ws) == kvx.KVX_DEV_BAD_LENGTH
    c = cnt.cpu().numpy()
    kh = kept.cpu().numpy()
    assert c[0] == 0 and c[1] == 0 and np.all(kh[:2] == -1)
    orc = oracle.load()
    for h in range(2):
        ref = orc.select_topk(q[1, 4 * h:4 * h + 4], k[1, h, :200], top, recent)
        assert c[2 + h] == ref.size
        check_head(orc, q[1, 4 * h:4 * h + 4], k[1, h, :200], top, recent, kh[2 + h, :c[2 + h]])
