"""Decode attention with the cluster layout: split heads merged through
distributed shared memory inside thread-block clusters (this GPU only).

Tangram's ahead-of-time split (AOT Load Balancing, Fig. 13) cuts heads across
thread blocks; in the cluster layout every cut head stays inside one cluster
and its pieces are merged by the block of its first piece, reading the other
pieces' (m, l, o) from their blocks' shared memory. Results must match the
oracle like any other layout, cover every kept token once (coverage record),
repeat bit for bit, survive graph capture, and report a wait that runs out
instead of hanging.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import DeviceCase, make_plan, max_abs, oracle_out
from test_attn_gpu import BF16_CASES, TOL_BF16
from paged_non_uniform_gb300 import kvx

pytestmark = pytest.mark.gpu
POLICY = {2: kvx.KVX_PLAN_CLUSTER_2, 4: kvx.KVX_PLAN_CLUSTER_4, 8: kvx.KVX_PLAN_CLUSTER_8}


def run_checked(case, plan):
    """Output with the coverage record on; the record must equal the oracle's
    count array of the plan's items."""
    dev = DeviceCase(case, plan)
    n = plan.kept().reshape(-1)
    cover = torch.zeros((n.size, max(1, int(n.max()))), dtype=torch.int32, device="cuda")
    plan.set_coverage_record(cover, cover.shape[1])
    got = dev.run()
    plan.set_coverage_record(None)
    assert dev.status() == 0
    items, _ = plan.items()
    bad, count = oracle.load().plan_coverage(n, items)
    assert bad == 0 and np.array_equal(cover.cpu().numpy(), count)
    return got, dev


def pieces_per_head(plan):
    items, _ = plan.items()
    n = plan.kept().reshape(-1)
    return np.bincount(items[:, 0], minlength=n.size)


@pytest.mark.parametrize("name", sorted(BF16_CASES))
@pytest.mark.parametrize("C", [2, 4, 8])
@pytest.mark.parametrize("clusters", [1, 3, 9])
def test_cluster_layout_parity(name, C, clusters):
    case = BF16_CASES[name](0)
    plan = make_plan(case, num_ctas=C * clusters, policy=POLICY[C])
    assert plan.stats()["cluster"] == C
    got, _ = run_checked(case, plan)
    assert max_abs(got, oracle_out(case)) <= TOL_BF16


@pytest.mark.parametrize("k", range(2, 9))
def test_head_cut_into_k_pieces(k):
    """One head of 32k kept tokens on one cluster of 8 blocks: the smallest
    cost cap cuts it into exactly k one-stage pieces, merged by piece 0."""
    n = 32 * k
    case = synth.dense_case(1, 4, 1, 128, [n + 5], [[n]], "bf16", seed=30 + k, P=16)
    plan = make_plan(case, num_ctas=8, policy=kvx.KVX_PLAN_CLUSTER_8)
    assert pieces_per_head(plan).tolist() == [k]
    got, _ = run_checked(case, plan)
    assert max_abs(got, oracle_out(case)) <= TOL_BF16


def test_whole_heads_and_cut_heads_together():
    """Short heads stay whole on one block, long heads are cut inside a
    cluster; both kinds in one launch."""
    n = [[2000, 40, 700, 1, 33, 1500, 96, 5], [64, 3000, 9, 1200, 480, 17, 2500, 250]]
    case = synth.dense_case(2, 16, 8, 128, [3100, 3200], n, "bf16", seed=41, P=16,
                            head_group=[0, 0, 1, 1, 2, 2, 3, 3])
    plan = make_plan(case, num_ctas=16, policy=kvx.KVX_PLAN_CLUSTER_4)
    pp = pieces_per_head(plan)
    assert (pp == 1).any() and (pp > 1).any()
    got, _ = run_checked(case, plan)
    assert max_abs(got, oracle_out(case)) <= TOL_BF16


@pytest.mark.parametrize("C", [2, 8])
def test_cluster_layout_repeats_bit_exact_and_replays_in_a_graph(C):
    case = BF16_CASES["qwen25_like"](3)
    plan = make_plan(case, num_ctas=4 * C, policy=POLICY[C])
    dev = DeviceCase(case, plan)
    first = dev.run()
    for _ in range(3):
        assert np.array_equal(dev.run(), first)
    out = torch.full_like(dev.out, float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kvx.kvx_decode_attn(plan, dev.q, dev.k_pools, dev.v_pools, dev.pool_pages, dev.pt,
                            dev.strides, dev.budget, dev.seq_len, 0.0, out, dev.ws,
                            stream=torch.cuda.current_stream())
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().astype(np.float64), first)
    assert dev.status() == 0
    assert max_abs(first, oracle_out(case)) <= TOL_BF16


@pytest.mark.parametrize("name", ["qwen3_like", "sparse_like"])
def test_cluster_layout_token_major_matches_head_major(name):
    case = BF16_CASES[name](5)
    hm = DeviceCase(case, make_plan(case, num_ctas=12, policy=kvx.KVX_PLAN_CLUSTER_4))
    tm = DeviceCase(case, make_plan(case, num_ctas=12, policy=kvx.KVX_PLAN_CLUSTER_4,
                                    layout=kvx.KVX_LAYOUT_TOKEN_MAJOR))
    a, b = hm.run(), tm.run()
    assert np.array_equal(a, b)
    assert max_abs(a, oracle_out(case)) <= TOL_BF16


def test_cluster_wait_runs_out_and_is_reported():
    """Failure detection without a GPU fault, cluster layout: one block's
    first stage is armed but never loaded; its wait runs out after 50 ms, it
    still signals its cluster's merging block, the call finishes with
    KVX_DEV_TIMEOUT, and the next call (workspace cleared, stall off) is
    correct."""
    import time
    case = BF16_CASES["sparse_like"](6)
    plan = make_plan(case, num_ctas=16, policy=kvx.KVX_PLAN_CLUSTER_4)
    dev = DeviceCase(case, plan)
    plan.inject_stall(5, 50_000_000)
    t0 = time.perf_counter()
    dev.run()
    assert time.perf_counter() - t0 < 5.0
    assert dev.status() & kvx.KVX_DEV_TIMEOUT
    plan.inject_stall(-1, 2_000_000_000)
    kvx.kvx_workspace_clear(dev.ws)
    got = dev.run()
    assert dev.status() == 0
    assert max_abs(got, oracle_out(case)) <= TOL_BF16


def test_balanced_policy_on_the_device_grid_merges_through_the_workspace():
    """The balanced policy on the device's own grid (num_ctas = 0) does not
    use clusters: split heads are merged through the workspace."""
    case = BF16_CASES["sparse_like"](7)
    plan = make_plan(case)
    assert plan.stats()["cluster"] == 1
    got, _ = run_checked(case, plan)
    assert max_abs(got, oracle_out(case)) <= TOL_BF16
