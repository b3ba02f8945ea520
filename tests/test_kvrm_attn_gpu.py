"""Fixed-shape attention over KV-RM's staging buffer ("KV-RM: Regularizing
KV-Cache Movement for Static-Graph LLM Serving", Figs. 2-3: the gathered
buffer feeds a fixed-shape attention kernel).

The staging buffer [S][max_tokens][8 heads][128] is a token-major paged pool
of S * max_blocks pages of 16 tokens with an identity page table; the same
kernel can also read the fragmented block pool directly, with the block table
as its page table. Both must match the oracle over each sequence's tokens and
each other bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from paged_non_uniform_gb300 import kvx

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _bf16_dev(a):
    return torch.from_numpy(synth.f32_to_bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()


def _attn(S, Hq, Hkv, D, L, q, k_pool, v_pool, pt, pool_pages):
    plan = kvx.kvx_plan_create(S, Hq, Hkv, D, 16, 1, kvx.KVX_BF16,
                               np.full((S, Hkv), synth.FULL, np.int32), L,
                               np.zeros(Hkv, np.int32), 0, layout=kvx.KVX_LAYOUT_TOKEN_MAJOR)
    kvx.kvx_plan_upload(plan)
    out = torch.full((S, Hq, D), float("nan"), device="cuda")
    ws = torch.zeros(plan.workspace_bytes() // 4 + 64, dtype=torch.int32, device="cuda")
    budget = torch.full((S * Hkv,), synth.FULL, dtype=torch.int32, device="cuda")
    kvx.kvx_decode_attn(plan, q, [k_pool], [v_pool], [pool_pages], [pt], [pt.shape[1]], budget,
                        torch.from_numpy(L).cuda(), 0.0, out, ws)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(ws) == 0
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("seed", [0, 1])
def test_attention_over_staging_and_over_fragmented_pool(seed):
    g = synth.rng(100 + seed)
    S, Hq, Hkv, D, max_blocks, num_phys = 6, 32, 8, 128, 24, 200
    L = g.integers(1, max_blocks * 16 + 1, size=S).astype(np.int32)
    L[0] = max_blocks * 16
    nb = ((L + 15) // 16).astype(np.int32)
    perm = g.permutation(num_phys).astype(np.int32)
    bt = np.full((S, max_blocks), -1, np.int32)
    pos = 0
    for s in range(S):
        bt[s, :nb[s]] = perm[pos:pos + nb[s]]
        pos += nb[s]
    kp = synth.normal(g, (num_phys, 16, Hkv, D), "bf16")
    vp = synth.normal(g, (num_phys, 16, Hkv, D), "bf16")
    q = synth.normal(g, (S, Hq, D), "bf16")
    k_dev, v_dev, q_dev = _bf16_dev(kp), _bf16_dev(vp), _bf16_dev(q)
    block_bytes = 16 * Hkv * D * 2
    row_bytes = max_blocks * block_bytes
    st_k = torch.zeros((S, max_blocks * 16, Hkv, D), dtype=torch.bfloat16, device="cuda")
    st_v = torch.zeros_like(st_k)
    ws = torch.zeros(kvx.kvx_gather_workspace_bytes(S, max_blocks) // 4 + 64, dtype=torch.int32,
                     device="cuda")
    kvx.kvx_gather_coalesce(torch.from_numpy(bt).cuda(), torch.from_numpy(nb).cuda(), S,
                            max_blocks, [k_dev, v_dev], num_phys, block_bytes, [st_k, st_v],
                            row_bytes, 0, ws)
    ident = torch.arange(S * max_blocks, dtype=torch.int32, device="cuda").view(S, max_blocks)
    over_staging = _attn(S, Hq, Hkv, D, L, q_dev, st_k, st_v, ident, S * max_blocks)
    direct = _attn(S, Hq, Hkv, D, L, q_dev, k_dev, v_dev, torch.from_numpy(bt).cuda(), num_phys)
    assert np.array_equal(over_staging, direct)
    # oracle: each sequence's tokens in logical order, dense
    Lmax = int(L.max())
    kd = np.zeros((S, Hkv, Lmax, D))
    vd = np.zeros((S, Hkv, Lmax, D))
    for s in range(S):
        t = np.arange(L[s])
        kd[s, :, :L[s]] = kp[bt[s, t // 16], t % 16].transpose(1, 0, 2)
        vd[s, :, :L[s]] = vp[bt[s, t // 16], t % 16].transpose(1, 0, 2)
    kept = [np.arange(L[s], dtype=np.int32) for s in range(S) for _ in range(Hkv)]
    ref = oracle.load().decode_attn(q, kd, vd, L, kept, 1.0 / math.sqrt(D))
    assert float(np.abs(over_staging - ref).max()) <= TOL


def test_full_size_kvrm_attention_sampled_sequences():
    """The benchmark's KV-RM workload at full size: 256 sequences of 512..16k
    tokens, 32 KB blocks randomly permuted over a 40 GiB K+V pool, gathered
    into [256][16384] staging rows; attention over the staging rows and
    directly over the pool must agree bit for bit everywhere, and match the
    oracle on sampled sequences (rebuilt on the host from the value table)."""
    from synth.device import ValueTable
    cfg = synth.gather_config(seed=0)
    S, Hq, Hkv, D, mb = cfg.S, 32, 8, 128, cfg.max_blocks
    table = ValueTable(seed=21, rows=1 << 18, D=D, dtype="bf16")
    shifts = [7, 1007]
    pools, stagings = [], []
    for t in range(2):
        p = torch.empty((cfg.num_phys, 16, Hkv, D), dtype=torch.bfloat16, device="cuda")
        table.fill(p, shifts[t])
        pools.append(p)
        stagings.append(torch.zeros((S, mb * 16, Hkv, D), dtype=torch.bfloat16, device="cuda"))
    bt = torch.from_numpy(cfg.bt).cuda()
    ws = torch.zeros(kvx.kvx_gather_workspace_bytes(S, mb) // 4 + 64, dtype=torch.int32,
                     device="cuda")
    kvx.kvx_gather_coalesce(bt, torch.from_numpy(cfg.nb).cuda(), S, mb, pools, cfg.num_phys,
                            cfg.block_bytes, stagings, cfg.row_bytes, 0, ws)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(ws) == 0
    L = np.ascontiguousarray(cfg.seq_tokens, dtype=np.int32)
    q = synth.normal(synth.rng(77), (S, Hq, D), "bf16")
    q_dev = _bf16_dev(q)
    ident = torch.arange(S * mb, dtype=torch.int32, device="cuda").view(S, mb)
    over_staging = _attn(S, Hq, Hkv, D, L, q_dev, stagings[0], stagings[1], ident, S * mb)
    direct = _attn(S, Hq, Hkv, D, L, q_dev, pools[0], pools[1], bt, cfg.num_phys)
    assert np.array_equal(over_staging, direct)
    orc = oracle.load()
    rows_per_block = 16 * Hkv
    for s in sorted({0, S - 1, int(np.argmax(L)), int(np.argmin(L)), 17, 101}):
        tok = np.arange(L[s])
        blk = cfg.bt[s, tok // 16].astype(np.int64)
        # pool row of (token, head): block * 128 + (token % 16) * 8 + head
        ids = (blk * rows_per_block + (tok % 16) * Hkv)[:, None] + np.arange(Hkv)
        kd = table.host_rows(shifts[0], ids.reshape(-1)).reshape(L[s], Hkv, D).transpose(1, 0, 2)
        vd = table.host_rows(shifts[1], ids.reshape(-1)).reshape(L[s], Hkv, D).transpose(1, 0, 2)
        kept = [np.arange(L[s], dtype=np.int32)] * Hkv
        ref = orc.decode_attn(q[s:s + 1], kd[None], vd[None], L[s:s + 1], kept, 1.0 / math.sqrt(D))
        assert float(np.abs(over_staging[s] - ref[0]).max()) <= TOL, s
