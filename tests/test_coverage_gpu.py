"""Token coverage as the attention kernels consume it.

Tangram's ahead-of-time plan (AOT Load Balancing, Fig. 13) cuts every head's
kept tokens across thread blocks; the cut may change only where a token is
read, never whether. With the coverage record on, a kernel adds one count per
token at the point where a consumer feeds it to the softmax. That array must
equal, bit for bit, the oracle's count array of the plan's items, which in
turn must be 1 on every kept token and 0 past it. The host entry point
kvx_plan_coverage must give the same array. Small cases here cover both
kernels, every plan policy and the extreme shapes; the full-size launches are
covered in test_full_size_gpu.py.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import DeviceCase, make_plan, max_abs, oracle_out
from test_attn_gpu import BF16_CASES, TOL_BF16, TOL_F32
from paged_non_uniform_gb300 import kvx

pytestmark = pytest.mark.gpu


def run_with_record(case, plan):
    dev = DeviceCase(case, plan)
    n = plan.kept().reshape(-1)
    cover = torch.zeros((n.size, max(1, int(n.max()))), dtype=torch.int32, device="cuda")
    plan.set_coverage_record(cover, cover.shape[1])
    got = dev.run()
    plan.set_coverage_record(None)
    assert dev.status() == 0
    items, _ = plan.items()
    bad, count = oracle.load().plan_coverage(n, items)
    assert bad == 0
    rec = cover.cpu().numpy()
    assert np.array_equal(rec, count)
    assert np.array_equal(plan.coverage(), count)
    return got, dev


@pytest.mark.parametrize("name", sorted(BF16_CASES))
@pytest.mark.parametrize("kernel", [kvx.KVX_KERNEL_MMA, kvx.KVX_KERNEL_SIMT])
@pytest.mark.parametrize("policy,num_ctas", [(0, 0), (0, 3), (0, 7), (1, 0), (2, 0)])
def test_bf16_coverage_record_is_exact(name, kernel, policy, num_ctas):
    case = BF16_CASES[name](0)
    plan = make_plan(case, num_ctas=num_ctas, policy=policy, kernel=kernel)
    got, _ = run_with_record(case, plan)
    assert max_abs(got, oracle_out(case)) <= TOL_BF16


@pytest.mark.parametrize("grouping", ["per_head", "one"])
@pytest.mark.parametrize("policy,num_ctas", [(0, 0), (0, 2), (0, 5), (1, 0), (2, 4)])
def test_fp32_coverage_record_is_exact(grouping, policy, num_ctas):
    case = synth.tiny(0, grouping)
    plan = make_plan(case, num_ctas=num_ctas, policy=policy)
    got, _ = run_with_record(case, plan)
    assert max_abs(got, oracle_out(case)) <= TOL_F32


@pytest.mark.parametrize("name", ["qwen3_like", "sparse_like", "p64"])
def test_coverage_record_is_exact_with_early_kv_loads(name):
    """Early K/V loads (kvx_plan_set_early_kv) change when the load warp
    issues a stage, not which tokens the consumers feed to the softmax."""
    case = BF16_CASES[name](2)
    plan = make_plan(case, num_ctas=0)
    plan.set_early_kv(True)
    got, _ = run_with_record(case, plan)
    assert max_abs(got, oracle_out(case)) <= TOL_BF16


def test_coverage_record_accumulates_and_turns_off():
    """Two calls with the record on count every kept token twice; a call with
    it off adds nothing."""
    case = BF16_CASES["qwen25_like"](1)
    plan = make_plan(case, num_ctas=9)
    dev = DeviceCase(case, plan)
    n = plan.kept().reshape(-1)
    cover = torch.zeros((n.size, int(n.max())), dtype=torch.int32, device="cuda")
    plan.set_coverage_record(cover, cover.shape[1])
    dev.run()
    dev.run()
    plan.set_coverage_record(None)
    dev.run()
    assert np.array_equal(cover.cpu().numpy(), 2 * plan.coverage())
