"""Parity of the CUDA decode-attention path against the fp64 oracle.

Tolerances: bf16 K/V with fp32 accumulation must stay within max-abs 2e-3 of
the oracle (the accuracy target of the method's GPU path). fp32 K/V: the
kernel's only approximations are fp32 rounding and the hardware exp2
(relative error ~2^-22), so 2e-5 is a safe bound for |o| <= ~4.
"""
import math

import numpy as np
import pytest
import torch

import synth
from harness import DeviceCase, make_plan, max_abs, oracle_out
from paged_non_uniform_gb300 import kvx

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-3
TOL_F32 = 2e-5


def qwen3_like(seed=0):
    L = [700, 2000, 3100]
    g = synth.rng(seed)
    rate = g.uniform(0.1, 0.5, size=8)
    rate[[1, 6]] = 1.0
    n = [[L[b] if rate[h] >= 1 else max(1, int(math.ceil(rate[h] * L[b]))) for h in range(8)]
         for b in range(3)]
    return synth.dense_case(3, 32, 8, 128, L, n, "bf16", seed=seed, P=16,
                            head_group=synth.groups_by_budget(rate, [2, 3, 3]))


def qwen25_like(seed=0):
    L = [2500, 90, 1000, 377]
    full = [0, 3, 4, 7]
    n = [[L[b] if h in full else max(1, int(math.ceil(0.125 * L[b]))) for h in range(8)]
         for b in range(4)]
    rate = np.array([1.0 if h in full else 0.125 for h in range(8)])
    return synth.dense_case(4, 40, 8, 128, L, n, "bf16", seed=seed, P=32,
                            head_group=synth.groups_by_budget(rate, [2, 2, 2, 2]))


def sparse_like(seed=0):
    return synth.dense_case(2, 32, 8, 128, [5000, 4100], [[2176] * 8] * 2, "bf16", seed=seed,
                            P=16, head_group=np.zeros(8, np.int32))


def d64_bf16(seed=0):
    return synth.dense_case(2, 4, 2, 64, [37, 100], [[37, 20], [100, 20]], "bf16", seed=seed,
                            P=16, head_group=[0, 1])


def g8_p8(seed=0):
    return synth.dense_case(2, 16, 2, 128, [300, 77], [[300, 40], [3, 77]], "bf16", seed=seed,
                            P=8, head_group=[0, 0])


def p64(seed=0):
    return synth.dense_case(2, 8, 4, 128, [600, 130], [[600, 1, 64, 65], [130, 2, 33, 129]],
                            "bf16", seed=seed, P=64, head_group=[0, 1, 1, 0])


BF16_CASES = {"qwen3_like": qwen3_like, "qwen25_like": qwen25_like, "sparse_like": sparse_like,
              "d64": d64_bf16, "g8_p8": g8_p8, "p64": p64}


@pytest.mark.parametrize("grouping", ["per_head", "one"])
@pytest.mark.parametrize("policy,num_ctas", [(0, 0), (0, 1), (0, 2), (0, 3), (0, 5),
                                             (1, 0), (2, 4)])
def test_tiny_fp32(grouping, policy, num_ctas):
    case = synth.tiny(0, grouping)
    plan = make_plan(case, num_ctas=num_ctas, policy=policy)
    dev = DeviceCase(case, plan)
    got = dev.run()
    ref = oracle_out(case)
    assert np.all(np.isfinite(got))
    err = max_abs(got, ref)
    assert err <= TOL_F32, err
    assert dev.status() == 0


@pytest.mark.parametrize("name", sorted(BF16_CASES))
@pytest.mark.parametrize("kernel", [kvx.KVX_KERNEL_MMA, kvx.KVX_KERNEL_SIMT])
@pytest.mark.parametrize("num_ctas", [0, 7])
def test_bf16_parity(name, kernel, num_ctas):
    case = BF16_CASES[name]()
    plan = make_plan(case, num_ctas=num_ctas, kernel=kernel)
    dev = DeviceCase(case, plan)
    got = dev.run()
    ref = oracle_out(case)
    assert np.all(np.isfinite(got))
    err = max_abs(got, ref)
    assert err <= TOL_BF16, err
    assert dev.status() == 0


@pytest.mark.parametrize("policy", [kvx.KVX_PLAN_PER_HEAD, kvx.KVX_PLAN_UNIFORM])
def test_naive_plans_match_oracle(policy):
    case = qwen3_like(1)
    dev = DeviceCase(case, make_plan(case, policy=policy))
    assert max_abs(dev.run(), oracle_out(case)) <= TOL_BF16


@pytest.mark.parametrize("kernel", [kvx.KVX_KERNEL_MMA, kvx.KVX_KERNEL_SIMT])
def test_page_permutation_is_bit_exact(kernel):
    """Same plan and page size, different physical page order: identical bits."""
    case = qwen3_like(2)
    plan = make_plan(case, num_ctas=11, kernel=kernel)
    a = DeviceCase(case, plan, perm_seed=1).run()
    b = DeviceCase(case, plan, perm_seed=2, spare_pages=17).run()
    assert np.array_equal(a, b)


def test_page_size_and_grouping_invariance():
    """P = 16 vs 32 and three group assignments: all within tolerance of the oracle."""
    base = qwen3_like(3)
    ref = oracle_out(base)
    for P in (16, 32):
        for hg in ([0, 1, 2, 3, 4, 5, 6, 7], [0, 0, 1, 1, 2, 2, 3, 3], [0, 0, 0, 0, 1, 1, 1, 1],
                   [0] * 8, list(base.head_group)):
            case = synth.dense_case(base.B, base.Hq, base.Hkv, base.D, base.seq_len, base.n,
                                    "bf16", seed=3, P=P, head_group=hg)
            got = DeviceCase(case, make_plan(case)).run()
            assert max_abs(got, ref) <= TOL_BF16, (P, hg)


def test_tokens_outside_kept_set_do_not_matter():
    """Dense rows a head does not keep, set to NaN, change nothing (bitwise);
    padding slots of partial pages hold NaN in every run here."""
    case = qwen25_like(4)
    plan = make_plan(case)
    a = DeviceCase(case, plan).run()
    k, v = case.k.copy(), case.v.copy()
    for b in range(case.B):
        for h in range(case.Hkv):
            mask = np.ones(k.shape[2], bool)
            mask[case.kept[b * case.Hkv + h]] = False
            k[b, h, mask] = np.nan
            v[b, h, mask] = np.nan
    b_ = DeviceCase(case, plan, dense_override=(k, v)).run()
    assert np.array_equal(a, b_)
    assert np.all(np.isfinite(a))


@pytest.mark.parametrize("kernel", [kvx.KVX_KERNEL_MMA, kvx.KVX_KERNEL_SIMT])
def test_single_token_heads_return_value_row(kernel):
    case = synth.dense_case(2, 16, 4, 128, [50, 70], [[1, 1, 50, 1], [1, 70, 1, 5]], "bf16",
                            seed=5, head_group=[0, 0, 1, 0])
    got = DeviceCase(case, make_plan(case, num_ctas=3, kernel=kernel)).run()
    g = case.Hq // case.Hkv
    for b in range(case.B):
        for h in range(case.Hkv):
            if case.n[b, h] == 1:
                t = case.kept[b * case.Hkv + h][0]
                for j in range(h * g, (h + 1) * g):
                    assert np.array_equal(got[b, j], case.v[b, h, t].astype(np.float64))


def test_device_flags_budget_mismatch():
    case = qwen3_like(6)
    dev = DeviceCase(case, make_plan(case))
    bad = dev.budget.clone()
    bad[5] = 1
    dev.run(budget=bad)
    assert dev.status() & kvx.KVX_DEV_BAD_BUDGET
    kvx.kvx_workspace_clear(dev.ws)
    torch.cuda.synchronize()
    dev.run()
    assert dev.status() == 0


@pytest.mark.parametrize("kernel", [kvx.KVX_KERNEL_MMA, kvx.KVX_KERNEL_SIMT])
def test_device_flags_page_outside_pool(kernel):
    """A page id past the pool is read as zeros and flagged; nothing faults."""
    case = qwen3_like(7)
    dev = DeviceCase(case, make_plan(case, kernel=kernel))
    pt = dev.pt[0]
    pt[0, 0] = dev.pool_pages[0] + 7
    got = dev.run()
    assert dev.status() & kvx.KVX_DEV_BAD_PAGE
    assert np.all(np.isfinite(got))


def test_custom_scale():
    case = d64_bf16(8)
    dev = DeviceCase(case, make_plan(case))
    got = dev.run(scale=0.05)
    assert max_abs(got, oracle_out(case, scale=0.05)) <= TOL_BF16


@pytest.mark.parametrize("kernel", [kvx.KVX_KERNEL_MMA, kvx.KVX_KERNEL_SIMT])
def test_repeated_calls_and_shared_workspace(kernel):
    """Split heads are merged in-kernel with per-head counters that return to
    zero after every call: repeated calls, and two plans taking turns on one
    workspace, give bit-identical results."""
    a_case, b_case = qwen3_like(9), qwen25_like(10)
    a = DeviceCase(a_case, make_plan(a_case, num_ctas=13, kernel=kernel))
    b = DeviceCase(b_case, make_plan(b_case, num_ctas=29, kernel=kernel))
    assert a.plan.stats()["num_split_heads"] > 0 and b.plan.stats()["num_split_heads"] > 0
    ws = torch.zeros(max(a.ws.numel(), b.ws.numel()), dtype=torch.int32, device="cuda")
    a.ws = b.ws = ws
    first_a, first_b = a.run(), b.run()
    for _ in range(3):
        assert np.array_equal(a.run(), first_a)
        assert np.array_equal(b.run(), first_b)
    assert a.status() == 0
    assert max_abs(first_a, oracle_out(a_case)) <= TOL_BF16
    assert max_abs(first_b, oracle_out(b_case)) <= TOL_BF16


@pytest.mark.parametrize("kernel", [kvx.KVX_KERNEL_MMA, kvx.KVX_KERNEL_SIMT])
def test_calls_captured_in_a_cuda_graph_replay_bit_exact(kernel):
    """Several layers' calls captured in one CUDA graph (after a first direct
    call per plan) replay to the same bits as direct calls, every replay."""
    cases = [qwen3_like(21), qwen25_like(22), sparse_like(23)]
    devs = [DeviceCase(c, make_plan(c, num_ctas=n, kernel=kernel))
            for c, n in zip(cases, (17, 0, 40))]
    direct = [d.run() for d in devs]
    outs = [torch.full_like(d.out, float("nan")) for d in devs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = torch.cuda.current_stream()
        for d, o in zip(devs, outs):
            kvx.kvx_decode_attn(d.plan, d.q, d.k_pools, d.v_pools, d.pool_pages, d.pt,
                                d.strides, d.budget, d.seq_len, 0.0, o, d.ws, stream=st)
    for _ in range(3):
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for ref, o, d in zip(direct, outs, devs):
            assert d.status() == 0
            assert np.array_equal(o.cpu().numpy().astype(np.float64), ref)
    for ref, c in zip(direct, cases):
        assert max_abs(ref, oracle_out(c)) <= TOL_BF16


def _early_kv_back_to_back(cases, devs):
    """Runs the layers once without early loads (reference bits, checked
    against the oracle), then with kvx_plan_set_early_kv on: three rounds of
    direct calls launched back to back on one stream (each a programmatic
    dependent of the one before) and three replays of a captured graph of
    them. Every output must equal the reference bit for bit."""
    ref = [d.run() for d in devs]
    for d, c, r in zip(devs, cases, ref):
        assert max_abs(r, oracle_out(c)) <= TOL_BF16
    for d in devs:
        d.plan.set_early_kv(True)
    st = torch.cuda.current_stream()
    for _ in range(3):
        for d in devs:
            d.out.fill_(float("nan"))
        torch.cuda.synchronize()
        for d in devs:  # no synchronisation between the layers
            kvx.kvx_decode_attn(d.plan, d.q, d.k_pools, d.v_pools, d.pool_pages, d.pt,
                                d.strides, d.budget, d.seq_len, 0.0, d.out, d.ws, stream=st)
        torch.cuda.synchronize()
        for d, r in zip(devs, ref):
            assert d.status() == 0
            assert np.array_equal(d.out.cpu().numpy(), r)
    outs = [torch.full_like(d.out, float("nan")) for d in devs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = torch.cuda.current_stream()
        for d, o in zip(devs, outs):
            kvx.kvx_decode_attn(d.plan, d.q, d.k_pools, d.v_pools, d.pool_pages, d.pt,
                                d.strides, d.budget, d.seq_len, 0.0, o, d.ws, stream=st)
    for _ in range(3):
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for o, r in zip(outs, ref):
            assert np.array_equal(o.cpu().numpy(), r)
    for d in devs:
        assert d.status() == 0


def test_early_kv_loads_are_bit_exact_back_to_back():
    """kvx_plan_set_early_kv: the load warps fill their rings before the
    preceding launch completes. Layers launched back to back give the same
    bits with early loads as without them, in direct calls and in a graph
    replay; the outputs match the oracle."""
    cases = [qwen3_like(31), sparse_like(32), qwen25_like(33), g8_p8(34), p64(35)]
    devs = [DeviceCase(c, make_plan(c, num_ctas=n)) for c, n in zip(cases, (0, 40, 17, 0, 9))]
    _early_kv_back_to_back(cases, devs)


def test_early_kv_loads_with_token_major_pages_and_cluster_layouts():
    """The same with KV-RM's token-major pages and with thread-block cluster
    layouts (their merging blocks wait on an inbox as well), mixed in one
    stream of back-to-back launches."""
    cases = [qwen3_like(41), sparse_like(42), qwen25_like(43), sparse_like(44), p64(45)]
    plans = [make_plan(cases[0], num_ctas=11, layout=kvx.KVX_LAYOUT_TOKEN_MAJOR),
             make_plan(cases[1], num_ctas=16, policy=kvx.KVX_PLAN_CLUSTER_4),
             make_plan(cases[2], num_ctas=16, policy=kvx.KVX_PLAN_CLUSTER_8),
             make_plan(cases[3], num_ctas=12, policy=kvx.KVX_PLAN_CLUSTER_2,
                       layout=kvx.KVX_LAYOUT_TOKEN_MAJOR),
             make_plan(cases[4], num_ctas=0)]
    devs = [DeviceCase(c, p) for c, p in zip(cases, plans)]
    _early_kv_back_to_back(cases, devs)


def test_pipeline_wait_runs_out_and_is_reported():
    """Failure detection without a GPU fault: one block's first stage is armed
    but never loaded, so its wait runs out after 50 ms. The call must return
    with KVX_DEV_TIMEOUT, and the next call on the same context, after the
    workspace is cleared and the stall removed, must be correct again."""
    import time
    case = qwen3_like(11)
    plan = make_plan(case, num_ctas=16, kernel=kvx.KVX_KERNEL_MMA)
    dev = DeviceCase(case, plan)
    plan.inject_stall(3, 50_000_000)
    t0 = time.perf_counter()
    dev.run()
    elapsed = time.perf_counter() - t0
    assert dev.status() & kvx.KVX_DEV_TIMEOUT
    assert elapsed < 5.0
    plan.inject_stall(-1, 2_000_000_000)
    kvx.kvx_workspace_clear(dev.ws)
    got = dev.run()
    assert dev.status() == 0
    assert max_abs(got, oracle_out(case)) <= TOL_BF16


def test_stall_hook_rejects_bad_limits():
    case = d64_bf16(12)
    plan = make_plan(case, upload=False)
    for bad in (0, 999_999, 20_000_000_000):
        with pytest.raises(kvx.KvxError):
            plan.inject_stall(0, bad)


@pytest.mark.parametrize("kernel", [kvx.KVX_KERNEL_MMA, kvx.KVX_KERNEL_SIMT])
@pytest.mark.parametrize("name", ["qwen3_like", "qwen25_like", "g8_p8", "p64", "d64"])
def test_token_major_pages_match_head_major_bit_for_bit(kernel, name):
    """KV-RM's token-major block layout and the head-major head-group page give
    the same bits: the kernels stage both into the same shared-memory tiles."""
    case = BF16_CASES[name]()
    a = DeviceCase(case, make_plan(case, num_ctas=9, kernel=kernel)).run()
    b = DeviceCase(case, make_plan(case, num_ctas=9, kernel=kernel,
                                   layout=kvx.KVX_LAYOUT_TOKEN_MAJOR), perm_seed=3).run()
    assert np.array_equal(a, b)
    assert max_abs(b, oracle_out(case)) <= TOL_BF16


def test_token_major_fp32_tiny():
    case = synth.tiny(0, "one")
    got = DeviceCase(case, make_plan(case, num_ctas=3, layout=kvx.KVX_LAYOUT_TOKEN_MAJOR)).run()
    assert max_abs(got, oracle_out(case)) <= TOL_F32


def mha_p128_16_groups(seed=0):
    """Limits: 64 KV heads (no GQA), 16 head groups, pages of 128 tokens."""
    g = synth.rng(seed + 50)
    L = [1000, 300]
    n = [[int(g.integers(1, L[b] + 1)) if h % 5 else L[b] for h in range(64)] for b in range(2)]
    return synth.dense_case(2, 64, 64, 128, L, n, "bf16", seed=seed, P=128,
                            head_group=np.arange(64, dtype=np.int32) % 16)


def g7_d64_p8(seed=0):
    """GQA factor 7, head dimension 64, pages of 8 tokens, 4 groups."""
    L = [257, 1031, 64]
    n = [[257, 31, 1, 200, 8, 9, 257, 100], [1031, 500, 17, 1030, 33, 1, 2, 64],
         [64, 64, 1, 63, 32, 33, 7, 64]]
    return synth.dense_case(3, 56, 8, 64, L, n, "bf16", seed=seed, P=8,
                            head_group=[0, 1, 2, 3, 0, 1, 2, 3])


def g3_p32(seed=0):
    """GQA factor 3, pages of 32 tokens."""
    return synth.dense_case(2, 12, 4, 128, [900, 33], [[900, 450, 31, 32], [33, 1, 33, 17]],
                            "bf16", seed=seed, P=32, head_group=[0, 0, 1, 1])


EXTREME_CASES = {"mha_p128_16_groups": mha_p128_16_groups, "g7_d64_p8": g7_d64_p8,
                 "g3_p32": g3_p32}


@pytest.mark.parametrize("name", sorted(EXTREME_CASES))
@pytest.mark.parametrize("kernel", [kvx.KVX_KERNEL_MMA, kvx.KVX_KERNEL_SIMT])
@pytest.mark.parametrize("layout", [kvx.KVX_LAYOUT_HEAD_MAJOR, kvx.KVX_LAYOUT_TOKEN_MAJOR])
def test_extreme_shapes(name, kernel, layout):
    case = EXTREME_CASES[name]()
    plan = make_plan(case, num_ctas=0, kernel=kernel, layout=layout)
    dev = DeviceCase(case, plan)
    got = dev.run()
    assert np.all(np.isfinite(got))
    err = max_abs(got, oracle_out(case))
    assert err <= TOL_BF16, err
    assert dev.status() == 0
