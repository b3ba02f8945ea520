"""The allocation-free gather entry point (kvx_gather_coalesce_noalloc).

It serves callers that cannot call cudaMalloc (host callbacks, allocator
paths, runtimes with a fixed, pre-planned device footprint): its scratch lives
in a static device array inside the library instead of a caller workspace.
These tests call it through the C ABI and check that it writes exactly what
the workspace entry point writes, on two calls in a row with different
inputs (the shared scratch keeps the previous call's contents). This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from paged_non_uniform_gb300 import kvx

pytestmark = pytest.mark.gpu


def _u(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _both(cfg, pools_h, flags, bt=None, nb=None):
    bt = cfg.bt if bt is None else bt
    nb = cfg.nb if nb is None else nb
    pools = [_u(p) for p in pools_h]
    init = synth.rng(5).integers(0, 256, size=(cfg.S, cfg.row_bytes), dtype=np.uint8)
    ref_st = [_u(init) for _ in pools]
    new_st = [_u(init) for _ in pools]
    ws = torch.zeros(kvx.kvx_gather_workspace_bytes(cfg.S, cfg.max_blocks) // 4 + 64,
                     dtype=torch.int32, device="cuda")
    kvx.kvx_gather_coalesce(_u(bt), _u(nb), cfg.S, cfg.max_blocks, pools, cfg.num_phys,
                            cfg.block_bytes, ref_st, cfg.row_bytes, flags, ws)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvx.kvx_gather_coalesce_noalloc(_u(bt), _u(nb), cfg.S, cfg.max_blocks, pools, cfg.num_phys,
                                    cfg.block_bytes, new_st, cfg.row_bytes, flags, status)
    torch.cuda.synchronize()
    return ([s.cpu().numpy() for s in ref_st], [s.cpu().numpy() for s in new_st],
            kvx.kvx_workspace_status(ws), int(status.item()))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    for call, (seed, extents) in enumerate(((3, False), (4, True))):
        cfg = synth.gather_config(seed=seed, S=24, Lmin=1, Lmax=2048, token_bytes=64,
                                  num_phys=4096, extents=extents, max_extent=9)
        pools = [synth.block_stamp_pool(cfg.num_phys, cfg.block_bytes, seed=seed + t)
                 for t in range(2)]
        ref, got, ws_status, status = _both(cfg, pools, 0)
        assert ws_status == 0 and status == 0, call
        init = synth.rng(5).integers(0, 256, size=(cfg.S, cfg.row_bytes), dtype=np.uint8)
        for t in range(2):
            assert np.array_equal(ref[t], got[t]), (call, t)
            # and on its own against the oracle's brute-force gather
            exp = oracle.load().gather(cfg.bt, cfg.nb, pools[t], init.copy())
            assert np.array_equal(got[t], exp), (call, t)


def test_noalloc_zero_tail_and_error_bits():
    cfg = synth.gather_config(seed=6, S=10, Lmin=1, Lmax=1024, token_bytes=32, num_phys=512)
    pools = [synth.block_stamp_pool(cfg.num_phys, cfg.block_bytes, seed=9)]
    bt, nb = cfg.bt.copy(), cfg.nb.copy()
    s = 1 + int(np.argmax(nb[1:]))
    bt[s, 0] = cfg.num_phys + 1
    nb[0] = cfg.max_blocks + 2
    ref, got, ws_status, status = _both(cfg, pools, kvx.KVX_ZERO_TAIL, bt=bt, nb=nb)
    assert ws_status == status == (kvx.KVX_DEV_BAD_BLOCK | kvx.KVX_DEV_BAD_LENGTH)
    assert np.array_equal(ref[0], got[0])


def test_noalloc_rejects_problems_beyond_its_scratch():
    p = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_gather_coalesce_noalloc(p, p, 4096, 4096, [p], 1, 16, [p], 16 * 4096, 0)
    assert e.value.status == kvx.KVX_ESCRATCH


def _largest_fitting_max_blocks(S):
    cap = 8 << 20  # KVX_GATHER_NOALLOC_SCRATCH_BYTES
    lo, hi = 1, 1 << 16
    assert kvx.kvx_gather_workspace_bytes(S, lo) <= cap < kvx.kvx_gather_workspace_bytes(S, hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if kvx.kvx_gather_workspace_bytes(S, mid) <= cap:
            lo = mid
        else:
            hi = mid
    return lo


def test_noalloc_at_the_scratch_limit():
    """S = 256 (the KV-RM shape) with the largest table the 8 MiB scratch
    holds, short rows: equal to the workspace entry point and to the oracle.
    One more block per row is rejected with KVX_ESCRATCH before any launch."""
    S = 256
    mb = _largest_fitting_max_blocks(S)
    assert mb >= 1024  # the KV-RM workload's table (16k tokens / 16) fits
    g = synth.rng(17)
    num_phys, bb = 4096, 16
    nb = g.integers(0, 9, size=S).astype(np.int32)
    bt = np.full((S, mb), -1, np.int32)
    for s in range(S):
        bt[s, :nb[s]] = g.choice(num_phys, size=nb[s], replace=False)
    cfg = synth.GatherConfig("limit", S, mb, nb, bt, num_phys, bb, 8 * bb, nb * 16)
    pools = [synth.block_stamp_pool(num_phys, bb, seed=21)]
    ref, got, ws_status, status = _both(cfg, pools, 0)
    assert ws_status == status == 0
    assert np.array_equal(ref[0], got[0])
    init = synth.rng(5).integers(0, 256, size=(S, 8 * bb), dtype=np.uint8)
    assert np.array_equal(got[0], oracle.load().gather(bt, nb, pools[0], init.copy()))
    p = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_gather_coalesce_noalloc(p, p, S, mb + 1, [p], num_phys, bb, [p], 8 * bb, 0)
    assert e.value.status == kvx.KVX_ESCRATCH


def test_noalloc_setup_call_with_no_rows():
    """S = 0 only prepares the device (address lookup, header clear)."""
    p = torch.zeros(64, dtype=torch.uint8, device="cuda")
    kvx.kvx_gather_coalesce_noalloc(p, p, 0, 0, [p], 1, 16, [p], 16, 0)
    torch.cuda.synchronize()
