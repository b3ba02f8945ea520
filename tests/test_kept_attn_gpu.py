"""Decode attention straight over the kept rows of a dense cache
(kvx_decode_attn_kept) against the fp64 oracle, and against attention over the
same rows packed into head-group pages with the same plan, which it must equal
bit for bit ("KVDrive", Fig. 7: decode attends to each head's selected
entries; Tangram, Fig. 13: the plan's split).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import DeviceCase, make_plan, max_abs, oracle_out
from test_attn_gpu import BF16_CASES, EXTREME_CASES, TOL_BF16
from paged_non_uniform_gb300 import kvx

pytestmark = pytest.mark.gpu


def _bf16(a):
    return torch.from_numpy(synth.f32_to_bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()


class KeptCase:
    """Device copies of a DenseCase as dense bf16 K/V [B][Hkv][Lmax][D] and a
    kept list per head (ascending, or in a seeded random order)."""

    def __init__(self, case, plan, order_seed=None, kept=None):
        self.case, self.plan = case, plan
        self.keys, self.values = _bf16(case.k), _bf16(case.v)
        self.Lmax = case.k.shape[2]
        lists = case.kept if kept is None else kept
        self.stride = max(1, max(len(x) for x in lists))
        arr = np.full((len(lists), self.stride), -1, np.int32)
        for i, pos in enumerate(lists):
            pos = np.asarray(pos, np.int32)
            if order_seed is not None:
                pos = pos[synth.rng(order_seed * 1000 + i).permutation(pos.size)]
            arr[i, :pos.size] = pos
        self.kept_host = arr
        self.kept = torch.from_numpy(arr).cuda()
        self.q = _bf16(case.q)
        self.budget = torch.from_numpy(np.ascontiguousarray(case.budget.reshape(-1),
                                                            dtype=np.int32)).cuda()
        self.seq_len = torch.from_numpy(np.ascontiguousarray(case.seq_len, np.int32)).cuda()
        self.out = torch.full((case.B, case.Hq, case.D), float("nan"), device="cuda")
        self.ws = torch.zeros(max(plan.workspace_bytes(), 256) // 4 + 64, dtype=torch.int32,
                              device="cuda")

    def call(self, out=None, stream=None):
        kvx.kvx_decode_attn_kept(self.plan, self.q, self.keys, self.values, self.Lmax,
                                 self.kept, self.stride, self.budget, self.seq_len, 0.0,
                                 self.out if out is None else out, self.ws, stream=stream)

    def run(self) -> np.ndarray:
        self.call()
        torch.cuda.synchronize()
        return self.out.cpu().numpy().astype(np.float64)

    def status(self) -> int:
        return kvx.kvx_workspace_status(self.ws)


@pytest.mark.parametrize("name", sorted(BF16_CASES))
@pytest.mark.parametrize("num_ctas", [0, 7])
def test_kept_rows_match_oracle_and_packed_pages(name, num_ctas):
    """Same plan: attention over the kept rows equals attention over the
    packed head-group pages bit for bit, and both match the oracle."""
    case = BF16_CASES[name](3)
    plan = make_plan(case, num_ctas=num_ctas)
    kc = KeptCase(case, plan)
    got = kc.run()
    assert kc.status() == 0
    assert max_abs(got, oracle_out(case)) <= TOL_BF16
    paged = DeviceCase(case, plan).run()
    assert np.array_equal(got, paged)


@pytest.mark.parametrize("name", sorted(EXTREME_CASES))
def test_kept_rows_extreme_shapes(name):
    """64 KV heads without GQA (16 groups, 128-token pages), GQA 7 at D = 64
    (8-token pages), GQA 3: bit-equal to the packed pages, within tolerance of
    the oracle."""
    case = EXTREME_CASES[name]()
    plan = make_plan(case, num_ctas=0)
    kc = KeptCase(case, plan)
    got = kc.run()
    assert kc.status() == 0
    assert max_abs(got, oracle_out(case)) <= TOL_BF16
    assert np.array_equal(got, DeviceCase(case, plan).run())


@pytest.mark.parametrize("name", ["qwen3_like", "sparse_like", "p64"])
@pytest.mark.parametrize("policy,num_ctas", [(kvx.KVX_PLAN_PER_HEAD, 0),
                                             (kvx.KVX_PLAN_UNIFORM, 0),
                                             (kvx.KVX_PLAN_CLUSTER_2, 12),
                                             (kvx.KVX_PLAN_CLUSTER_4, 16)])
def test_kept_rows_under_every_plan_policy(name, policy, num_ctas):
    case = BF16_CASES[name](4)
    plan = make_plan(case, num_ctas=num_ctas, policy=policy)
    kc = KeptCase(case, plan)
    got = kc.run()
    assert kc.status() == 0
    assert max_abs(got, oracle_out(case)) <= TOL_BF16
    assert np.array_equal(got, DeviceCase(case, plan).run())


def test_kept_rows_in_any_order():
    """The kept list may be in any order: the result stays within the
    tolerance of the oracle (only fp32 rounding follows the order)."""
    case = BF16_CASES["qwen25_like"](5)
    plan = make_plan(case, num_ctas=9)
    got = KeptCase(case, plan, order_seed=7).run()
    assert max_abs(got, oracle_out(case)) <= TOL_BF16


def test_kept_rows_coverage_record():
    """The consumed-token record of the kept path equals the oracle's count
    array of the plan's items."""
    case = BF16_CASES["sparse_like"](6)
    plan = make_plan(case, num_ctas=0)
    kc = KeptCase(case, plan)
    n = plan.kept().reshape(-1)
    cover = torch.zeros((n.size, int(n.max())), dtype=torch.int32, device="cuda")
    plan.set_coverage_record(cover, cover.shape[1])
    got = kc.run()
    plan.set_coverage_record(None)
    items, _ = plan.items()
    bad, count = oracle.load().plan_coverage(n, items)
    assert bad == 0
    assert np.array_equal(cover.cpu().numpy(), count)
    assert max_abs(got, oracle_out(case)) <= TOL_BF16


def test_kept_index_outside_the_cache_reads_zeros_and_is_flagged():
    """An index outside [0, Lmax) is read as a zero row and reported; the
    result equals the same call with that entry pointing at a zero row."""
    case = BF16_CASES["qwen3_like"](8)
    plan = make_plan(case, num_ctas=5)
    lists = [np.array(x) for x in case.kept]
    bh, i = 9, 3
    L0 = case.k.shape[2]
    bad = [x.copy() for x in lists]
    bad[bh][i] = L0 + 17
    kc = KeptCase(case, plan, kept=bad)
    got = kc.run()
    assert kc.status() & kvx.KVX_DEV_BAD_BLOCK
    # reference: same lists, that entry naming a row zeroed in a copy of the cache
    b, h = divmod(bh, case.Hkv)
    z = int(lists[bh][i])
    k0, v0 = case.k.copy(), case.v.copy()
    k0[b, h, z] = 0.0
    v0[b, h, z] = 0.0
    zc = KeptCase(case, plan)
    zc.keys, zc.values = _bf16(k0), _bf16(v0)
    ref = zc.run()
    assert zc.status() == 0
    assert np.array_equal(got, ref)


def test_kept_rows_back_to_back_and_in_a_graph():
    """Layers launched back to back (programmatic dependent launches) and a
    captured graph of them give the bits of separate calls."""
    cases = [BF16_CASES[n](11 + i) for i, n in enumerate(["qwen3_like", "sparse_like", "g8_p8"])]
    kcs = [KeptCase(c, make_plan(c, num_ctas=nc)) for c, nc in zip(cases, (0, 40, 3))]
    ref = [kc.run() for kc in kcs]
    for _ in range(3):
        for kc in kcs:
            kc.out.fill_(float("nan"))
        torch.cuda.synchronize()
        for kc in kcs:
            kc.call()
        torch.cuda.synchronize()
        for kc, r in zip(kcs, ref):
            assert kc.status() == 0
            assert np.array_equal(kc.out.cpu().numpy(), r)
    outs = [torch.full_like(kc.out, float("nan")) for kc in kcs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = torch.cuda.current_stream()
        for kc, o in zip(kcs, outs):
            kc.call(out=o, stream=st)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for o, r in zip(outs, ref):
            assert np.array_equal(o.cpu().numpy(), r)


def test_kept_rows_wait_runs_out_and_is_reported():
    """Failure detection without a GPU fault: one block's first stage gets no
    copies, its consumers' wait runs out after the plan's limit, the call
    reports KVX_DEV_TIMEOUT and the context stays usable."""
    case = BF16_CASES["sparse_like"](12)
    plan = make_plan(case, num_ctas=8)
    plan.inject_stall(2, 20_000_000)
    kc = KeptCase(case, plan)
    kc.run()
    assert kc.status() & kvx.KVX_DEV_TIMEOUT
    plan.inject_stall(-1, 2_000_000_000)
    kvx.kvx_workspace_clear(kc.ws)
    got = kc.run()
    assert kc.status() == 0
    assert max_abs(got, oracle_out(case)) <= TOL_BF16
