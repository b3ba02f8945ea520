"""Thin ctypes binding of the kvx C ABI (include/kvx.h).

Argument marshalling only: every step of the decode-attention and gather
path runs in the library's CUDA kernels. Device buffers may be passed as
torch tensors (their ``data_ptr()``) or raw integer addresses; host arrays as
NumPy arrays. Importing this module fails if ``libkvx.so`` has not been built
(``python -m paged_non_uniform_gb300.build``): there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_LIB_PATH = os.environ.get("KVX_LIBRARY") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libkvx.so")

KVX_OK = 0
KVX_EINVAL = -1
KVX_ERANGE = -2
KVX_ENOMEM = -3
KVX_ECUDA = -4
KVX_EUNSUPPORTED = -5
KVX_ESTATE = -6
KVX_ESCRATCH = -7
KVX_ENOBLOCKS = -8
KVX_EDIT_RESERVE = 0
KVX_EDIT_ALIAS = 1
KVX_EDIT_TRIM = 2

KVX_DEV_BAD_PAGE = 1
KVX_DEV_BAD_BUDGET = 2
KVX_DEV_TIMEOUT = 4
KVX_DEV_BAD_BLOCK = 8
KVX_DEV_BAD_LENGTH = 16

KVX_F32 = 0
KVX_BF16 = 1
KVX_PLAN_BALANCED = 0
KVX_PLAN_PER_HEAD = 1
KVX_PLAN_UNIFORM = 2
KVX_PLAN_CLUSTER_2 = 3
KVX_PLAN_CLUSTER_4 = 4
KVX_PLAN_CLUSTER_8 = 5
KVX_KERNEL_AUTO = 0
KVX_KERNEL_MMA = 1
KVX_KERNEL_SIMT = 2
KVX_ZERO_TAIL = 1
KVX_LAYOUT_HEAD_MAJOR = 0
KVX_LAYOUT_TOKEN_MAJOR = 1
KVX_MAX_GROUPS = 16
KVX_WS_HEADER_BYTES = 256


class KvxError(RuntimeError):
    def __init__(self, what: str, status: int):
        self.status = status
        super().__init__(f"{what}: {kvx_status_string(status)} (status {status}, "
                         f"cuda error {kvx_last_cuda_error()})")


if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with "
                      "`python -m paged_non_uniform_gb300.build` (nvcc, sm_103a)")

lib = ctypes.CDLL(_LIB_PATH)
_c = ctypes
_vp = _c.c_void_p


class kvx_shape(_c.Structure):
    _fields_ = [("B", _c.c_int32), ("Hq", _c.c_int32), ("Hkv", _c.c_int32), ("D", _c.c_int32),
                ("page_size", _c.c_int32), ("num_groups", _c.c_int32), ("dtype", _c.c_int32),
                ("layout", _c.c_int32)]


class kvx_plan_stats(_c.Structure):
    _fields_ = [("num_ctas", _c.c_int32), ("num_items", _c.c_int32), ("num_slots", _c.c_int32),
                ("num_split_heads", _c.c_int32), ("kernel", _c.c_int32), ("policy", _c.c_int32),
                ("total_tokens", _c.c_int64), ("max_cta_tokens", _c.c_int64),
                ("mean_cta_tokens", _c.c_double), ("slots_allocated", _c.c_int64),
                ("slots_used", _c.c_int64), ("plan_us", _c.c_double),
                ("item_overhead", _c.c_int32), ("cluster", _c.c_int32)]


lib.kvx_status_string.restype = _c.c_char_p
lib.kvx_status_string.argtypes = [_c.c_int]
lib.kvx_last_cuda_error.restype = _c.c_int
lib.kvx_device_sm_count.argtypes = [_vp]
lib.kvx_plan_create.argtypes = [_c.POINTER(kvx_shape), _vp, _vp, _vp, _c.c_int32, _c.c_int32,
                                _c.c_int32, _c.POINTER(_vp)]
lib.kvx_plan_upload.argtypes = [_vp, _vp]
lib.kvx_plan_workspace_bytes.argtypes = [_vp, _c.POINTER(_c.c_size_t)]
lib.kvx_plan_get_stats.argtypes = [_vp, _c.POINTER(kvx_plan_stats)]
lib.kvx_plan_kept.argtypes = [_vp, _vp]
lib.kvx_plan_group_pages.argtypes = [_vp, _vp]
lib.kvx_plan_items.argtypes = [_vp, _vp, _vp]
lib.kvx_plan_cta_tokens.argtypes = [_vp, _vp]
lib.kvx_plan_set_trace.argtypes = [_vp, _vp]
lib.kvx_plan_coverage.argtypes = [_vp, _vp]
lib.kvx_plan_set_coverage_record.argtypes = [_vp, _vp, _c.c_int32]
lib.kvx_plan_inject_stall.argtypes = [_vp, _c.c_int32, _c.c_uint64]
lib.kvx_plan_set_early_kv.argtypes = [_vp, _c.c_int32]
lib.kvx_plan_destroy.argtypes = [_vp]
lib.kvx_plan_destroy.restype = None
lib.kvx_decode_attn.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c.c_float, _vp,
                                _vp, _c.c_size_t, _vp]
lib.kvx_workspace_status.argtypes = [_vp, _c.POINTER(_c.c_uint32)]
lib.kvx_workspace_clear.argtypes = [_vp, _c.c_size_t, _vp]
lib.kvx_gather_workspace_bytes.argtypes = [_c.c_int32, _c.c_int32, _c.POINTER(_c.c_size_t)]
lib.kvx_gather_coalesce.argtypes = [_vp, _vp, _c.c_int32, _c.c_int32, _c.c_int32, _vp,
                                    _c.c_int64, _c.c_int64, _vp, _c.c_int64, _c.c_int32, _vp,
                                    _c.c_size_t, _vp]
lib.kvx_gather_read_runs.argtypes = [_vp, _c.c_int32, _c.c_int32, _vp, _vp]
lib.kvx_select_workspace_bytes.argtypes = [_c.c_int32, _c.c_int32, _c.c_int32,
                                           _c.POINTER(_c.c_size_t)]
lib.kvx_select_topk.argtypes = [_vp, _vp, _vp, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32,
                                _c.c_int32, _c.c_int32, _c.c_int32, _vp, _vp, _vp, _c.c_size_t,
                                _vp]
lib.kvx_pack_kept.argtypes = [_vp, _vp, _vp, _c.c_int32, _vp, _c.c_int32, _vp, _vp, _vp, _vp,
                              _vp, _vp, _c.c_size_t, _vp]
lib.kvx_decode_attn_kept.argtypes = [_vp, _vp, _vp, _vp, _c.c_int32, _vp, _c.c_int32, _vp,
                                     _vp, _c.c_float, _vp, _vp, _c.c_size_t, _vp]

class kvx_frame_stats(_c.Structure):
    _fields_ = [("commits", _c.c_int64), ("free_blocks", _c.c_int64),
                ("pending_entries", _c.c_int64), ("pending_rows", _c.c_int64),
                ("last_records", _c.c_int64), ("last_bytes", _c.c_int64),
                ("launches", _c.c_int64), ("wait_ns", _c.c_int64)]


lib.kvx_frame_create.argtypes = [_c.c_int32, _c.c_int32, _c.c_int32, _c.POINTER(_vp)]
lib.kvx_frame_destroy.argtypes = [_vp]
lib.kvx_frame_reserve.argtypes = [_vp, _c.c_int32, _c.c_int32, _vp]
lib.kvx_frame_alias.argtypes = [_vp] + [_c.c_int32] * 5
lib.kvx_frame_trim.argtypes = [_vp, _c.c_int32, _c.c_int32, _c.c_int32]
lib.kvx_frame_edit.argtypes = [_vp, _vp, _c.c_int32, _vp, _vp, _c.c_int64,
                               _c.POINTER(_c.c_int64)]
lib.kvx_frame_commit.argtypes = [_vp, _vp]
lib.kvx_frame_active.argtypes = [_vp, _c.POINTER(_vp), _c.POINTER(_vp)]
lib.kvx_frame_view.argtypes = [_vp, _vp, _vp, _vp]
lib.kvx_frame_get_stats.argtypes = [_vp, _c.POINTER(kvx_frame_stats)]
lib.kvx_gather_coalesce_noalloc.argtypes = [_vp, _vp, _c.c_int32, _c.c_int32, _c.c_int32, _vp,
                                            _c.c_int64, _c.c_int64, _vp, _c.c_int64,
                                            _c.c_int32, _vp, _vp]


def kvx_status_string(status: int) -> str:
    return lib.kvx_status_string(int(status)).decode()


def kvx_last_cuda_error() -> int:
    return int(lib.kvx_last_cuda_error())


def _check(rc: int, what: str) -> None:
    if rc != KVX_OK:
        raise KvxError(what, rc)


def _dptr(x) -> int | None:
    """Device address of a torch tensor or an integer address."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return int(torch.cuda.current_stream().cuda_stream)
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def kvx_device_sm_count() -> int:
    v = _c.c_int32(0)
    _check(lib.kvx_device_sm_count(_c.byref(v)), "kvx_device_sm_count")
    return int(v.value)


class Plan:
    """Owner of one kvx_plan handle."""

    def __init__(self, handle: int, shape: kvx_shape):
        self.handle = handle
        self.shape = shape

    @property
    def g(self) -> int:
        return self.shape.Hq // self.shape.Hkv

    def stats(self) -> dict:
        st = kvx_plan_stats()
        _check(lib.kvx_plan_get_stats(self.handle, _c.byref(st)), "kvx_plan_get_stats")
        return {name: getattr(st, name) for name, _ in kvx_plan_stats._fields_}

    def workspace_bytes(self) -> int:
        return kvx_plan_workspace_bytes(self)

    def kept(self) -> np.ndarray:
        n = np.zeros(self.shape.B * self.shape.Hkv, dtype=np.int32)
        _check(lib.kvx_plan_kept(self.handle, n.ctypes.data), "kvx_plan_kept")
        return n.reshape(self.shape.B, self.shape.Hkv)

    def group_pages(self) -> np.ndarray:
        pg = np.zeros(self.shape.num_groups * self.shape.B, dtype=np.int32)
        _check(lib.kvx_plan_group_pages(self.handle, pg.ctypes.data), "kvx_plan_group_pages")
        return pg.reshape(self.shape.num_groups, self.shape.B)

    def items(self):
        st = self.stats()
        items = np.zeros((max(st["num_items"], 1), 4), dtype=np.int32)
        off = np.zeros(st["num_ctas"] + 1, dtype=np.int32)
        _check(lib.kvx_plan_items(self.handle, items.ctypes.data, off.ctypes.data),
               "kvx_plan_items")
        return items[:st["num_items"]], off

    def cta_tokens(self) -> np.ndarray:
        st = self.stats()
        t = np.zeros(max(st["num_ctas"], 1), dtype=np.int64)
        _check(lib.kvx_plan_cta_tokens(self.handle, t.ctypes.data), "kvx_plan_cta_tokens")
        return t[:st["num_ctas"]]

    def set_early_kv(self, enable: bool) -> None:
        """kvx_plan_set_early_kv: let the load warp fill its ring before the
        dependency wait (see the header for the precondition)."""
        _check(lib.kvx_plan_set_early_kv(self.handle, 1 if enable else 0), "kvx_plan_set_early_kv")

    def set_trace(self, dev_trace) -> None:
        _check(lib.kvx_plan_set_trace(self.handle, _dptr(dev_trace)), "kvx_plan_set_trace")

    def coverage(self) -> np.ndarray:
        """kvx_plan_coverage: int32 [B*Hkv][max_n] count of items per token."""
        mx = max(1, int(self.kept().max()))
        c = np.zeros((self.shape.B * self.shape.Hkv, mx), dtype=np.int32)
        _check(lib.kvx_plan_coverage(self.handle, c.ctypes.data), "kvx_plan_coverage")
        return c

    def set_coverage_record(self, dev_count, stride: int = 0) -> None:
        """kvx_plan_set_coverage_record (None turns it off)."""
        _check(lib.kvx_plan_set_coverage_record(self.handle, _dptr(dev_count), int(stride)),
               "kvx_plan_set_coverage_record")

    def inject_stall(self, block: int, wait_limit_ns: int) -> None:
        """Failure-detection test hook: see kvx_plan_inject_stall."""
        _check(lib.kvx_plan_inject_stall(self.handle, int(block), int(wait_limit_ns)),
               "kvx_plan_inject_stall")

    def destroy(self) -> None:
        if self.handle:
            lib.kvx_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def kvx_plan_create(B, Hq, Hkv, D, page_size, num_groups, dtype, head_budget, seq_len,
                    head_group, num_ctas=0, policy=KVX_PLAN_BALANCED,
                    kernel=KVX_KERNEL_AUTO, layout=KVX_LAYOUT_HEAD_MAJOR) -> Plan:
    shape = kvx_shape(B, Hq, Hkv, D, page_size, num_groups, dtype, layout)
    hb, sl, hg = _i32(head_budget).reshape(-1), _i32(seq_len).reshape(-1), _i32(head_group)
    h = _vp()
    rc = lib.kvx_plan_create(_c.byref(shape), hb.ctypes.data, sl.ctypes.data, hg.ctypes.data,
                             int(num_ctas), int(policy), int(kernel), _c.byref(h))
    _check(rc, "kvx_plan_create")
    return Plan(h.value, shape)


def kvx_plan_upload(plan: Plan, stream=None) -> None:
    _check(lib.kvx_plan_upload(plan.handle, _stream(stream)), "kvx_plan_upload")


def kvx_plan_workspace_bytes(plan: Plan) -> int:
    v = _c.c_size_t(0)
    _check(lib.kvx_plan_workspace_bytes(plan.handle, _c.byref(v)), "kvx_plan_workspace_bytes")
    return int(v.value)


def _ptr_array(xs) -> ctypes.Array:
    return (_vp * max(len(xs), 1))(*[_dptr(x) for x in xs])


def kvx_decode_attn(plan: Plan, q, k_pools, v_pools, pool_pages, page_tables,
                    page_table_stride, head_budget, seq_len, scale, out, workspace,
                    workspace_bytes=None, stream=None) -> None:
    kp, vp, pt = _ptr_array(k_pools), _ptr_array(v_pools), _ptr_array(page_tables)
    pp = np.ascontiguousarray(np.asarray(pool_pages, dtype=np.int64))
    ps = _i32(page_table_stride)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib.kvx_decode_attn(plan.handle, _dptr(q), kp, vp, pp.ctypes.data, pt, ps.ctypes.data,
                             _dptr(head_budget), _dptr(seq_len), float(scale), _dptr(out),
                             _dptr(workspace), int(workspace_bytes), _stream(stream))
    _check(rc, "kvx_decode_attn")


def kvx_workspace_status(workspace) -> int:
    v = _c.c_uint32(0)
    _check(lib.kvx_workspace_status(_dptr(workspace), _c.byref(v)), "kvx_workspace_status")
    return int(v.value)


def kvx_workspace_clear(workspace, nbytes=None, stream=None) -> None:
    """Zero the first `nbytes` bytes of a workspace (default: all of a tensor)."""
    if nbytes is None:
        nbytes = workspace.numel() * workspace.element_size()
    _check(lib.kvx_workspace_clear(_dptr(workspace), int(nbytes), _stream(stream)),
           "kvx_workspace_clear")


def kvx_gather_workspace_bytes(S: int, max_blocks: int) -> int:
    v = _c.c_size_t(0)
    _check(lib.kvx_gather_workspace_bytes(int(S), int(max_blocks), _c.byref(v)),
           "kvx_gather_workspace_bytes")
    return int(v.value)


def kvx_gather_coalesce(block_table, num_blocks, S, max_blocks, pools, num_phys_blocks,
                        block_bytes, stagings, staging_row_bytes, flags, workspace,
                        workspace_bytes=None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib.kvx_gather_coalesce(_dptr(block_table), _dptr(num_blocks), int(S), int(max_blocks),
                                 len(pools), _ptr_array(pools), int(num_phys_blocks),
                                 int(block_bytes), _ptr_array(stagings), int(staging_row_bytes),
                                 int(flags), _dptr(workspace), int(workspace_bytes),
                                 _stream(stream))
    _check(rc, "kvx_gather_coalesce")


def kvx_gather_read_runs(workspace, S: int, max_blocks: int):
    cnt = np.zeros(max(S, 1), dtype=np.int32)
    runs = np.zeros((max(S, 1), max(max_blocks, 1), 3), dtype=np.int32)
    _check(lib.kvx_gather_read_runs(_dptr(workspace), int(S), int(max_blocks), cnt.ctypes.data,
                                    runs.ctypes.data), "kvx_gather_read_runs")
    return cnt[:S], runs[:S]


def kvx_select_workspace_bytes(B: int, Hkv: int, Lmax: int) -> int:
    v = _c.c_size_t(0)
    _check(lib.kvx_select_workspace_bytes(int(B), int(Hkv), int(Lmax), _c.byref(v)),
           "kvx_select_workspace_bytes")
    return int(v.value)


def kvx_select_topk(keys, q, seq_len, B, Hq, Hkv, D, Lmax, top, recent, kept_idx, kept_count,
                    workspace, workspace_bytes=None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib.kvx_select_topk(_dptr(keys), _dptr(q), _dptr(seq_len), int(B), int(Hq), int(Hkv),
                             int(D), int(Lmax), int(top), int(recent), _dptr(kept_idx),
                             _dptr(kept_count), _dptr(workspace), int(workspace_bytes),
                             _stream(stream))
    _check(rc, "kvx_select_topk")


def kvx_pack_kept(plan: Plan, keys, values, Lmax, kept_idx, kept_stride, k_pools, v_pools,
                  pool_pages, page_tables, page_table_stride, workspace, workspace_bytes=None,
                  stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    pp = np.ascontiguousarray(np.asarray(pool_pages, dtype=np.int64))
    ps = _i32(page_table_stride)
    rc = lib.kvx_pack_kept(plan.handle, _dptr(keys), _dptr(values), int(Lmax), _dptr(kept_idx),
                           int(kept_stride), _ptr_array(k_pools), _ptr_array(v_pools),
                           pp.ctypes.data, _ptr_array(page_tables), ps.ctypes.data,
                           _dptr(workspace), int(workspace_bytes), _stream(stream))
    _check(rc, "kvx_pack_kept")


def kvx_decode_attn_kept(plan: Plan, q, keys, values, Lmax, kept_idx, kept_stride, head_budget,
                         seq_len, scale, out, workspace, workspace_bytes=None,
                         stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib.kvx_decode_attn_kept(plan.handle, _dptr(q), _dptr(keys), _dptr(values), int(Lmax),
                                  _dptr(kept_idx), int(kept_stride), _dptr(head_budget),
                                  _dptr(seq_len), float(scale), _dptr(out), _dptr(workspace),
                                  int(workspace_bytes), _stream(stream))
    _check(rc, "kvx_decode_attn_kept")


def kvx_gather_coalesce_noalloc(block_table, num_blocks, S, max_blocks, pools, num_phys_blocks,
                                block_bytes, stagings, staging_row_bytes, flags, status=None,
                                stream=None) -> None:
    """kvx_gather_coalesce for callers that cannot allocate device memory: no
    workspace argument; the library's static device scratch is used instead.
    `status` is an optional device uint32/int32 tensor that collects
    device-detected error bits."""
    rc = lib.kvx_gather_coalesce_noalloc(_dptr(block_table), _dptr(num_blocks), int(S),
                                         int(max_blocks), len(pools), _ptr_array(pools),
                                         int(num_phys_blocks), int(block_bytes),
                                         _ptr_array(stagings), int(staging_row_bytes), int(flags),
                                         _dptr(status), _stream(stream))
    _check(rc, "kvx_gather_coalesce_noalloc")


class Frame:
    """KV-RM block pager with double-buffered device descriptors
    (kvx_frame_*). Edits return the library's status code; commit raises."""

    def __init__(self, S: int, max_blocks: int, num_phys_blocks: int):
        h = _vp()
        _check(lib.kvx_frame_create(int(S), int(max_blocks), int(num_phys_blocks),
                                    _c.byref(h)), "kvx_frame_create")
        self.handle, self.S, self.M, self.N = h, int(S), int(max_blocks), int(num_phys_blocks)

    def __del__(self):
        if getattr(self, "handle", None):
            lib.kvx_frame_destroy(self.handle)
            self.handle = None

    def reserve(self, seq: int, count: int):
        ids = np.zeros(max(int(count), 1), dtype=np.int32)
        rc = lib.kvx_frame_reserve(self.handle, int(seq), int(count), ids.ctypes.data)
        return rc, (ids[:max(int(count), 0)] if rc == KVX_OK else ids[:0])

    def alias(self, dst: int, dst_block: int, src: int, src_block: int, count: int) -> int:
        return lib.kvx_frame_alias(self.handle, int(dst), int(dst_block), int(src),
                                   int(src_block), int(count))

    def trim(self, seq: int, begin_block: int, end_block: int) -> int:
        return lib.kvx_frame_trim(self.handle, int(seq), int(begin_block), int(end_block))

    def edit(self, ops, want_ids: bool = False):
        """Applies ops ([n][6] int32, KVX_EDIT_* rows) in order; returns the
        status of every edit (and, with want_ids, the reserved block ids in
        edit order)."""
        ops = np.ascontiguousarray(ops, dtype=np.int32).reshape(-1, 6)
        st = np.zeros(max(len(ops), 1), dtype=np.int32)
        if not want_ids:
            lib.kvx_frame_edit(self.handle, ops.ctypes.data, len(ops), st.ctypes.data, None, 0,
                               None)
            return st[:len(ops)]
        cap = int(np.maximum(ops[ops[:, 0] == KVX_EDIT_RESERVE, 2], 0).sum())
        ids = np.zeros(max(cap, 1), dtype=np.int32)
        nw = _c.c_int64(0)
        lib.kvx_frame_edit(self.handle, ops.ctypes.data, len(ops), st.ctypes.data,
                           ids.ctypes.data, cap, _c.byref(nw))
        return st[:len(ops)], ids[:nw.value]

    def commit(self, stream=None) -> None:
        _check(lib.kvx_frame_commit(self.handle, _stream(stream)), "kvx_frame_commit")

    def active(self):
        """Device addresses (block_table, num_blocks) of the active descriptor."""
        bt, nb = _vp(), _vp()
        _check(lib.kvx_frame_active(self.handle, _c.byref(bt), _c.byref(nb)),
               "kvx_frame_active")
        return int(bt.value), int(nb.value)

    def state(self):
        """Host view: (block_table [S][max_blocks], num_blocks [S], refcount [N])."""
        bt = np.zeros((self.S, self.M), dtype=np.int32)
        nb = np.zeros(self.S, dtype=np.int32)
        rc = np.zeros(self.N, dtype=np.int32)
        _check(lib.kvx_frame_view(self.handle, bt.ctypes.data, nb.ctypes.data, rc.ctypes.data),
               "kvx_frame_view")
        return bt, nb, rc

    def stats(self) -> dict:
        st = kvx_frame_stats()
        _check(lib.kvx_frame_get_stats(self.handle, _c.byref(st)), "kvx_frame_get_stats")
        return {k: int(getattr(st, k)) for k, _ in kvx_frame_stats._fields_}
