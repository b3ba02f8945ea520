"""KV-RM block pager of the library (kvx_frame_*): host-side edits against the
oracle's pager, entry for entry. No GPU: edits and the host view only (device
descriptors are allocated on first commit)."""
import numpy as np
import pytest

import oracle
import synth
from oracle_pins import read_frame_golden, replay_frame_golden
from paged_non_uniform_gb300 import kvx

# the library's status codes, named as the oracle names them
CODE = {kvx.KVX_OK: 0, kvx.KVX_EINVAL: -1, kvx.KVX_ERANGE: -2, kvx.KVX_ENOBLOCKS: -3}


class Coded:
    """A kvx.Frame whose edits report the oracle's codes."""

    def __init__(self, f):
        self.f = f

    def reserve(self, *a):
        c, ids = self.f.reserve(*a)
        return CODE[c], ids

    def alias(self, *a):
        return CODE[self.f.alias(*a)]

    def trim(self, *a):
        return CODE[self.f.trim(*a)]

    def state(self):
        return self.f.state()


def test_frame_golden_sequence():
    S, M, N, steps, rc = read_frame_golden()
    replay_frame_golden(Coded(kvx.Frame(S, M, N)), S, M, N, steps, rc)


def random_edits(gen, S, M, nb, big=False):
    """One random edit (op, args) given the current view lengths nb."""
    op = int(gen.integers(0, 10))
    if op < 4:
        c = int(gen.integers(0, 200 if big else 6))
        return "reserve", (int(gen.integers(0, S)), c)
    if op < 7:
        dst, src = int(gen.integers(0, S)), int(gen.integers(0, S))
        c = int(gen.integers(0, 8))
        return "alias", (dst, int(gen.integers(0, nb[dst] + 2)), src,
                         int(gen.integers(0, nb[src] + 2)), c)
    s = int(gen.integers(0, S))
    if op == 7:
        return "trim", (s, 0, 0)
    return "trim", (s, int(gen.integers(0, nb[s] + 2)), int(gen.integers(0, nb[s] + 2)))


@pytest.mark.parametrize("S,M,N,big", [(8, 32, 200, False), (16, 512, 5000, True),
                                       (3, 70, 130, False)])
def test_frame_random_edits_match_oracle(S, M, N, big):
    gen = synth.rng(1000 + N)
    lib_f = Coded(kvx.Frame(S, M, N))
    orc_f = oracle.load().frame(S, M, N)
    for it in range(2500):
        _, nb, _ = orc_f.state()
        op, args = random_edits(gen, S, M, nb, big)
        if op == "reserve":
            a, ida = lib_f.reserve(*args)
            b, idb = orc_f.reserve(*args)
            assert np.array_equal(ida, idb), (it, op, args)
        else:
            a, b = getattr(lib_f, op)(*args), getattr(orc_f, op)(*args)
        assert a == b, (it, op, args, a, b)
        if it % 25 == 0 or it > 2450:
            for x, y in zip(lib_f.state(), orc_f.state()):
                assert np.array_equal(x, y), (it, op, args)


def test_frame_pool_edges():
    # pool not a multiple of 64 blocks; a run that spans bitmap words
    f = kvx.Frame(2, 200, 130)
    rc, ids = f.reserve(0, 130)
    assert rc == kvx.KVX_OK and np.array_equal(ids, np.arange(130))
    assert f.reserve(1, 1)[0] == kvx.KVX_ENOBLOCKS
    assert f.trim(0, 60, 70) == kvx.KVX_OK        # frees 0..59 and 70..129
    rc, ids = f.reserve(1, 61)                    # the run 70..130 is 60 long: 0..60 is not
    assert rc == kvx.KVX_OK and np.array_equal(ids, np.r_[0:60, 70]), ids
    rc, ids = f.reserve(1, 59)
    assert rc == kvx.KVX_OK and np.array_equal(ids, np.arange(71, 130))
    assert f.stats()["free_blocks"] == 0


def test_frame_pending_accounting():
    f = kvx.Frame(4, 16, 64)
    f.reserve(0, 3)
    f.reserve(1, 2)
    f.alias(2, 0, 0, 0, 3)
    st = f.stats()
    assert st["pending_entries"] == 8 and st["pending_rows"] == 3
    assert st["commits"] == 0 and st["free_blocks"] == 59
    f.trim(2, 0, 0)                                # same entries again: not counted twice
    assert f.stats()["pending_entries"] == 8


def test_frame_create_errors():
    h = kvx._vp()
    assert kvx.lib.kvx_frame_create(0, 4, 4, kvx._c.byref(h)) == kvx.KVX_EINVAL
    assert kvx.lib.kvx_frame_create(4, 0, 4, kvx._c.byref(h)) == kvx.KVX_EINVAL
    assert kvx.lib.kvx_frame_create(4, 4, 0, kvx._c.byref(h)) == kvx.KVX_EINVAL
    assert kvx.lib.kvx_frame_create(1 << 16, 1 << 15, 4, kvx._c.byref(h)) == kvx.KVX_ERANGE
    f = kvx.Frame(2, 4, 8)
    assert f.reserve(2, 1)[0] == kvx.KVX_EINVAL
    assert f.reserve(0, -1)[0] == kvx.KVX_EINVAL
    assert f.reserve(0, 5)[0] == kvx.KVX_ERANGE
    assert f.alias(0, 1, 1, 0, 1) == kvx.KVX_ERANGE  # src view empty; dst_block past nb
    assert f.trim(0, 1, 0) == kvx.KVX_ERANGE


def test_batch_edit_matches_single_edits():
    """kvx_frame_edit applies a batch exactly as the single-edit calls would,
    failed edits included (they change nothing and report their status)."""
    gen = synth.rng(31)
    S, M, N = 10, 40, 300
    a, b = kvx.Frame(S, M, N), kvx.Frame(S, M, N)
    for it in range(40):
        ops, want = [], []
        for _ in range(25):
            _, nb, _ = b.state()
            op, args = random_edits(gen, S, M, nb)
            kind = {"reserve": kvx.KVX_EDIT_RESERVE, "alias": kvx.KVX_EDIT_ALIAS,
                    "trim": kvx.KVX_EDIT_TRIM}[op]
            ops.append([kind, *args] + [0] * (5 - len(args)))
            if op == "reserve":
                single, got_ids = b.reserve(*args)
                want.extend(got_ids.tolist())
            else:
                single = getattr(b, op)(*args)
            ops[-1].append(single)
        ops = np.array(ops, np.int32)
        if it % 2:
            st, ids = a.edit(ops[:, :6], want_ids=True)
            assert ids.tolist() == want, it
        else:
            st = a.edit(ops[:, :6])
        assert np.array_equal(st, ops[:, 6]), it
        for x, y in zip(a.state(), b.state()):
            assert np.array_equal(x, y), it
    assert a.edit(np.array([[7, 0, 0, 0, 0, 0]], np.int32))[0] == kvx.KVX_EINVAL


def test_batch_edit_ids_capacity():
    f = kvx.Frame(2, 16, 64)
    ops = np.array([[kvx.KVX_EDIT_RESERVE, 0, 3, 0, 0, 0],
                    [kvx.KVX_EDIT_RESERVE, 1, 4, 0, 0, 0]], np.int32)
    ids = np.zeros(5, np.int32)
    st = np.zeros(2, np.int32)
    nw = kvx._c.c_int64(0)
    rc = kvx.lib.kvx_frame_edit(f.handle, ops.ctypes.data, 2, st.ctypes.data, ids.ctypes.data,
                                5, kvx._c.byref(nw))
    # the second Reserve does not fit in the id buffer: refused, nothing applied
    assert rc == kvx.KVX_ERANGE and list(st) == [kvx.KVX_OK, kvx.KVX_ERANGE] and nw.value == 3
    assert list(ids[:3]) == [0, 1, 2] and list(f.state()[1]) == [3, 0]
