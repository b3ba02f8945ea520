"""KV-RM Frame commit on the GPU: after every commit the active device
descriptor equals the oracle pager's state entry for entry, and the coalesced
gather through it equals the oracle's gather of that state."""
import numpy as np
import pytest
import torch

import oracle
import synth
from paged_non_uniform_gb300 import kvx

pytestmark = pytest.mark.gpu


class _DevArray:
    """Zero-copy view of a device address the library owns."""

    def __init__(self, ptr, shape):
        self.__cuda_array_interface__ = {"data": (ptr, False), "shape": tuple(shape),
                                         "typestr": "<i4", "version": 2}


def active(frame):
    bt, nb = frame.active()
    return (torch.as_tensor(_DevArray(bt, (frame.S, frame.M)), device="cuda"),
            torch.as_tensor(_DevArray(nb, (frame.S,)), device="cuda"))


def edit_stream(gen, S, nb, ops):
    for _ in range(ops):
        op = int(gen.integers(0, 10))
        if op < 5:
            yield "reserve", (int(gen.integers(0, S)), int(gen.integers(0, 5)))
        elif op < 8:
            dst, src = int(gen.integers(0, S)), int(gen.integers(0, S))
            yield "alias", (dst, int(gen.integers(0, nb()[dst] + 1)), src,
                            int(gen.integers(0, nb()[src] + 1)), int(gen.integers(0, 4)))
        else:
            s = int(gen.integers(0, S))
            n = int(nb()[s])
            b = int(gen.integers(0, n + 1))
            yield "trim", (s, b, int(gen.integers(b, n + 1)))


@pytest.mark.parametrize("S,M,N,edits_per_frame", [(8, 40, 300, 7), (32, 64, 1500, 40),
                                                   (5, 20, 90, 1)])
def test_commit_matches_oracle_every_frame(S, M, N, edits_per_frame):
    gen = synth.rng(S * 31 + N)
    f = kvx.Frame(S, M, N)
    o = oracle.load().frame(S, M, N)
    stream = torch.cuda.Stream()
    bufs = set()
    for frame in range(60):
        for op, args in edit_stream(gen, S, lambda: o.state()[1], edits_per_frame):
            if op == "reserve":
                a, ida = f.reserve(*args)
                b, idb = o.reserve(*args)
                assert np.array_equal(ida, idb)
            else:
                a, b = getattr(f, op)(*args), getattr(o, op)(*args)
            assert (a == kvx.KVX_OK) == (b == 0), (frame, op, args)
        f.commit(stream)
        stream.synchronize()
        bt, nb = active(f)
        bufs.add(f.active()[0])
        table, onb, _ = o.state()
        assert np.array_equal(nb.cpu().numpy(), onb), frame
        assert np.array_equal(bt.cpu().numpy(), table), frame
    assert len(bufs) == 2          # the two descriptors alternate
    assert f.stats()["commits"] == 60


def test_commit_without_edits_and_first_use():
    f = kvx.Frame(4, 8, 32)
    bt, nb = active(f)             # before any commit: empty views
    assert np.all(bt.cpu().numpy() == -1) and not nb.cpu().numpy().any()
    f.reserve(1, 3)
    f.commit()
    torch.cuda.synchronize()
    st = f.stats()
    assert st["launches"] == 1 and st["last_records"] == 4
    f.commit()                     # brings the other descriptor up to date
    f.commit()                     # nothing changed in two frames: no copy, no launch
    torch.cuda.synchronize()
    st = f.stats()
    assert st["launches"] == 2 and st["last_records"] == 0
    bt, nb = active(f)
    assert list(nb.cpu().numpy()) == [0, 3, 0, 0]
    assert list(bt.cpu().numpy()[1, :4]) == [0, 1, 2, -1]


def test_gather_through_committed_descriptors():
    """Movement step of a decode loop: edits, one Frame commit, then the
    coalesced gather of the active descriptor, all on one stream, for several
    frames; every staging buffer is checked against the oracle's gather of the
    oracle pager's state in that frame."""
    S, M, N, block_bytes = 12, 48, 400, 64
    gen = synth.rng(5)
    f = kvx.Frame(S, M, N)
    o = oracle.load().frame(S, M, N)
    orc = oracle.load()
    pool = synth.block_stamp_pool(N, block_bytes, seed=3)
    dpool = torch.from_numpy(pool).cuda()
    row = M * block_bytes
    ws = torch.zeros(kvx.kvx_gather_workspace_bytes(S, M) // 4 + 64, dtype=torch.int32,
                     device="cuda")
    stream = torch.cuda.Stream()
    stagings, expect = [], []
    for frame in range(6):
        for op, args in edit_stream(gen, S, lambda: o.state()[1], 15):
            if op == "reserve":
                f.reserve(*args)
                o.reserve(*args)
            else:
                getattr(f, op)(*args)
                getattr(o, op)(*args)
        f.commit(stream)
        bt, nb = f.active()
        st = torch.zeros((S, row), dtype=torch.uint8, device="cuda")
        kvx.kvx_gather_coalesce(bt, nb, S, M, [dpool], N, block_bytes, [st], row,
                                kvx.KVX_ZERO_TAIL, ws, stream=stream)
        table, onb, _ = o.state()
        expect.append(orc.gather(table, onb, pool, np.zeros((S, row), np.uint8), zero_tail=True))
        stagings.append(st)
    stream.synchronize()
    assert kvx.kvx_workspace_status(ws) == 0
    for frame, (st, ref) in enumerate(zip(stagings, expect)):
        assert np.array_equal(st.cpu().numpy(), ref), frame


def test_full_size_churn_matches_oracle():
    """The benchmark's churn on its full pool (256 sequences, at most 1024
    blocks each, 655 360 physical blocks): per step every sequence gains a
    token, sequences end (Trim) and are replaced by new prompts that share a
    live prefix (Alias) or not, full windows drop their oldest block (Trim),
    blocks are reserved 8 at a time; one commit per step. The committed
    device descriptor equals the oracle pager's state at sampled steps."""
    cfg = synth.gather_config(seed=0)
    S, M, N, bt_tok, look = cfg.S, cfg.max_blocks, cfg.num_phys, 16, 8
    f = kvx.Frame(S, M, N)
    o = oracle.load().frame(S, M, N)
    gen = synth.rng(4242)
    tokens = cfg.seq_tokens.astype(np.int64).copy()
    nbv = np.zeros(S, np.int64)

    def both(op, *args):
        if op == "reserve":
            a, ia = f.reserve(*args)
            b, ib = o.reserve(*args)
            assert np.array_equal(ia, ib), (op, args)
        else:
            a, b = getattr(f, op)(*args), getattr(o, op)(*args)
        assert (a == kvx.KVX_OK) == (b == 0), (op, args, a, b)
        return b

    def need(t):
        return int(min(M, -(-int(t) // bt_tok)))

    def grow(s):
        want = need(tokens[s])
        if want > nbv[s]:
            c = int(min(M - nbv[s], max(want - nbv[s], look)))
            assert both("reserve", s, c) == 0
            nbv[s] += c

    for s in range(S):
        grow(s)
    stream = torch.cuda.Stream()
    for step in range(120):
        tokens += 1
        for s in np.flatnonzero(gen.random(S) < 1.0 / 100):
            s = int(s)
            assert both("trim", s, 0, 0) == 0
            nbv[s] = 0
            tokens[s] = int(gen.integers(512, M * bt_tok - 512))
            r = int(gen.integers(0, S))
            k = int(min(nbv[r], need(tokens[s]) // 2))
            if gen.random() < 0.25 and r != s and k > 0:
                assert both("alias", s, 0, r, 0, k) == 0
                nbv[s] = k
        for s in np.flatnonzero(tokens > M * bt_tok):
            s = int(s)
            assert both("trim", s, 1, int(nbv[s])) == 0
            nbv[s] -= 1
            tokens[s] -= bt_tok
        for s in range(S):
            grow(s)
        f.commit(stream)
        if step % 20 == 19:
            stream.synchronize()
            bt, nb = active(f)
            table, onb, _ = o.state()
            assert np.array_equal(nb.cpu().numpy(), onb), step
            assert np.array_equal(bt.cpu().numpy(), table), step
