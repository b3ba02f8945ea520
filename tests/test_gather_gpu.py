"""Bit-exact parity of the CUDA gather (run merge + coalesced copy) against
the oracle's brute-force index copy and run list."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import ValueTable
from paged_non_uniform_gb300 import kvx

pytestmark = pytest.mark.gpu


def _dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gather(cfg, pools, stagings, flags=0, nb=None, bt=None):
    nb = cfg.nb if nb is None else nb
    bt = cfg.bt if bt is None else bt
    ws = torch.zeros(kvx.kvx_gather_workspace_bytes(cfg.S, cfg.max_blocks) // 4 + 64,
                     dtype=torch.int32, device="cuda")
    kvx.kvx_gather_coalesce(_dev_u8(bt), _dev_u8(nb), cfg.S, cfg.max_blocks, pools,
                            cfg.num_phys, cfg.block_bytes, stagings, cfg.row_bytes, flags, ws)
    torch.cuda.synchronize()
    return ws


def small_cfg(seed, extents, S=12, Lmax=640, num_phys=512, token_bytes=4):
    return synth.gather_config(seed=seed, S=S, Lmin=1, Lmax=Lmax, block_tokens=16,
                               token_bytes=token_bytes, num_phys=num_phys, extents=extents,
                               max_extent=7)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("extents", [False, True])
@pytest.mark.parametrize("zero_tail", [False, True])
def test_small_gather_bit_exact(seed, extents, zero_tail):
    cfg = small_cfg(seed, extents)
    orc = oracle.load()
    pools = [synth.block_stamp_pool(cfg.num_phys, cfg.block_bytes, seed=seed + t) for t in (0, 1)]
    init = synth.rng(99).integers(0, 256, size=(cfg.S, cfg.row_bytes), dtype=np.uint8)
    dp = [_dev_u8(p) for p in pools]
    ds = [_dev_u8(init) for _ in pools]
    ws = run_gather(cfg, dp, ds, kvx.KVX_ZERO_TAIL if zero_tail else 0)
    assert kvx.kvx_workspace_status(ws) == 0
    for t in range(2):
        ref = orc.gather(cfg.bt, cfg.nb, pools[t], init.copy(), zero_tail=zero_tail)
        assert np.array_equal(ds[t].cpu().numpy(), ref)
    total, cnt, runs = orc.runs(cfg.bt, cfg.nb)
    gcnt, gruns = kvx.kvx_gather_read_runs(ws, cfg.S, cfg.max_blocks)
    assert np.array_equal(gcnt, cnt)
    for s in range(cfg.S):
        assert np.array_equal(gruns[s, :cnt[s]], runs[s, :cnt[s]])


def test_gather_golden_layout_with_16_byte_blocks():
    """The hand-worked table of tests/golden/gather_tiny.txt, with each block
    widened to 16 bytes."""
    bt = np.array([[7, 8, 2, 11, -1], [0, 1, 2, 3, 15], [4, -1, -1, -1, -1]], np.int32)
    nb = np.array([3, 5, 0], np.int32)
    pool = (np.arange(16 * 16) % 256).astype(np.uint8).reshape(16, 16)
    cfg = synth.GatherConfig("golden", 3, 5, nb, bt, 16, 16, 80, nb * 16)
    st = _dev_u8(np.full((3, 80), 238, np.uint8))
    ws = run_gather(cfg, [_dev_u8(pool)], [st])
    got = st.cpu().numpy()
    exp = np.full((3, 80), 238, np.uint8)
    exp[0, :48] = np.concatenate([pool[7], pool[8], pool[2]])
    exp[1, :80] = np.concatenate([pool[0], pool[1], pool[2], pool[3], pool[15]])
    assert np.array_equal(got, exp)
    cnt, runs = kvx.kvx_gather_read_runs(ws, 3, 5)
    assert cnt.tolist() == [2, 2, 0]
    assert runs[0, :2].tolist() == [[7, 0, 2], [2, 2, 1]]
    assert runs[1, :2].tolist() == [[0, 0, 4], [15, 4, 1]]


def test_gather_flags_bad_entries_and_copies_the_rest():
    cfg = small_cfg(5, False)
    orc = oracle.load()
    pool = synth.block_stamp_pool(cfg.num_phys, cfg.block_bytes, seed=3)
    bt, nb = cfg.bt.copy(), cfg.nb.copy()
    s_bad_block = 1 + int(np.argmax(nb[1:]))
    assert nb[s_bad_block] >= 2
    bt[s_bad_block, 1] = cfg.num_phys + 3          # outside the pool
    nb[0] = cfg.max_blocks + 1                      # longer than the table
    init = np.zeros((cfg.S, cfg.row_bytes), np.uint8)
    st = _dev_u8(init)
    ws = run_gather(cfg, [_dev_u8(pool)], [st], nb=nb, bt=bt)
    status = kvx.kvx_workspace_status(ws)
    assert status & kvx.KVX_DEV_BAD_BLOCK and status & kvx.KVX_DEV_BAD_LENGTH
    got = st.cpu().numpy()
    assert not got[0].any()                        # rejected row untouched
    good_nb, good_bt = nb.copy(), bt.copy()
    good_nb[0] = 0
    good_bt[s_bad_block, 1] = 0
    ref = orc.gather(good_bt, good_nb, pool, init.copy())
    ref[s_bad_block, cfg.block_bytes:2 * cfg.block_bytes] = 0   # the bad block is not copied
    assert np.array_equal(got, ref)


def _row_blocks_u8(table, shift, ids, block_bytes):
    """Host copy of pool blocks `ids` of a pool filled from `table` with
    `shift` whose first 8 bytes were stamped with the block id: the bytes the
    gather must copy, uint8 [len(ids)][block_bytes]."""
    rows_per_block = block_bytes // 256
    blk = table.host_raw_rows(shift, (ids[:, None].astype(np.int64) * rows_per_block
                                      + np.arange(rows_per_block)).reshape(-1))
    blk = np.ascontiguousarray(blk).reshape(ids.size, block_bytes // 2)
    blk.view(np.int64)[:, 0] = ids
    return blk.view(np.uint8).reshape(ids.size, block_bytes)


@pytest.mark.parametrize("extents", [False, True])
def test_full_size_gather_every_row(extents):
    """256 sequences, 16..16k tokens, 32 KB blocks, 40 GB fragmented K+V pool,
    two 8 GiB staging tensors: all 512 staging rows (256 per tensor) bit-exact
    against the oracle's gather of the same blocks, and the run list exact."""
    cfg = synth.gather_config(seed=0, extents=extents)
    orc = oracle.load()
    table = ValueTable(seed=21, rows=1 << 18, D=128, dtype="bf16")
    pools, stagings, shifts = [], [], [12345, 777777]
    for t in range(2):
        p = torch.empty((cfg.num_phys, cfg.block_bytes // 2), dtype=torch.bfloat16, device="cuda")
        table.fill(p, shifts[t])
        p.view(torch.int64)[:, 0] = torch.arange(cfg.num_phys, device="cuda", dtype=torch.int64)
        pools.append(p)
        stagings.append(torch.zeros((cfg.S, cfg.row_bytes // 2), dtype=torch.bfloat16,
                                    device="cuda"))
    ws = run_gather(cfg, pools, stagings)
    assert kvx.kvx_workspace_status(ws) == 0
    total, cnt, runs = orc.runs(cfg.bt, cfg.nb)
    gcnt, gruns = kvx.kvx_gather_read_runs(ws, cfg.S, cfg.max_blocks)
    assert np.array_equal(gcnt, cnt) and int(gcnt.sum()) == total
    for s in range(cfg.S):
        assert np.array_equal(gruns[s, :cnt[s]], runs[s, :cnt[s]])
    checked = 0
    for t in range(2):
        for s in range(cfg.S):
            ids = cfg.bt[s, :cfg.nb[s]]
            mini = _row_blocks_u8(table, shifts[t], ids, cfg.block_bytes)
            ref = np.zeros((1, cfg.row_bytes), np.uint8)
            orc.gather(np.arange(ids.size, dtype=np.int32)[None, :],
                       np.array([ids.size], np.int32), mini, ref)
            got = stagings[t][s].view(torch.uint8).cpu().numpy()
            assert np.array_equal(got, ref[0]), (t, s)
            checked += 1
    assert checked == 2 * cfg.S == 512


def test_medium_gather_all_rows():
    """32 sequences, 32 KB blocks, 1 GiB pool per tensor (K and V): every row
    bit-exact against the oracle (inputs larger than L2)."""
    cfg = synth.gather_config(seed=7, S=32, num_phys=32768)
    orc = oracle.load()
    table = ValueTable(seed=23, rows=1 << 18, D=128, dtype="bf16")
    pools, stagings, shifts = [], [], [5, 99991]
    for t in range(2):
        p = torch.empty((cfg.num_phys, cfg.block_bytes // 2), dtype=torch.bfloat16, device="cuda")
        table.fill(p, shifts[t])
        p.view(torch.int64)[:, 0] = torch.arange(cfg.num_phys, device="cuda", dtype=torch.int64)
        pools.append(p)
        stagings.append(torch.full((cfg.S, cfg.row_bytes // 2), 3.0, dtype=torch.bfloat16,
                                   device="cuda"))
    ws = run_gather(cfg, pools, stagings)
    assert kvx.kvx_workspace_status(ws) == 0
    for t in range(2):
        got = stagings[t].view(torch.uint8).cpu().numpy()
        for s in range(cfg.S):
            ids = cfg.bt[s, :cfg.nb[s]]
            mini = _row_blocks_u8(table, shifts[t], ids, cfg.block_bytes)
            init = np.full((1, cfg.row_bytes // 2), 0x4040, np.uint16)  # bf16 3.0
            ref = orc.gather(np.arange(ids.size, dtype=np.int32)[None, :],
                             np.array([ids.size], np.int32), mini,
                             init.view(np.uint8).reshape(1, -1).copy())
            assert np.array_equal(got[s], ref[0]), (t, s)
