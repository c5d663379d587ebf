"""Python binding of libsarathi (ctypes): the mixed-batch paged-attention step
of chunked prefill with stall-free batching on one sm_103a GPU.

Argument marshalling only: every step of the path runs in the C/CUDA library
(``csrc/``), whose ABI is ``include/sarathi.h``.  The function names match the
C entry points.  If the shared library is missing this module raises: there is
no fallback.  PyTorch supplies device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

OK, ERR_INVALID_ARG, ERR_CAPACITY, WARN_OVER_BUDGET_DECODES = 0, 1, 2, 3
ERR_CUDA, ERR_UNSUPPORTED, ERR_DEVICE_CHECK = 4, 5, 6
DECODE, PREFILL_RUNNING, PREFILL_WAITING = 0, 1, 2
ABI_VERSION = 6   # SARATHI_ABI_VERSION of include/sarathi.h
ROPE_ROTATE_HALF, ROPE_INTERLEAVED = 0, 1
ITEM_INTS = 24    # SARATHI_ITEM_INTS

EXPORTED = ("sarathi_plan_bounds", "sarathi_plan", "sarathi_plan_ex", "sarathi_advance", "sarathi_split_metadata",
            "sarathi_rope_table", "sarathi_qkv_proj",
            "sarathi_mixed_attn", "sarathi_mixed_attn_host",
            "sarathi_mixed_attn_noalloc", "sarathi_noalloc_status", "sarathi_workspace_status", "sarathi_last_error",
            "sarathi_abi_version")


class SarathiError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: status {status}: {msg}")
        self.status = status


class Request(ctypes.Structure):
    _fields_ = [("state", ctypes.c_int32), ("prompt_len", ctypes.c_int32), ("num_computed", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("pages", ctypes.POINTER(ctypes.c_int32))]


POLICY_STALL_FREE, POLICY_DECODE_MAXIMAL = 0, 1


class PlanPolicy(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("token_budget", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("chunk_align", ctypes.c_int32)]


class MetaSet(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("rows", "tokens", "token_offset", "nnz_pages", "first_row",
                                              "off_qo_indptr", "off_kv_page_indptr", "off_kv_page_indices",
                                              "off_kv_last_page_len")]


class QkvArgs(ctypes.Structure):
    pass


class Shape(ctypes.Structure):
    _fields_ = [("num_heads_q", ctypes.c_int32), ("num_heads_kv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32)]


QkvArgs._fields_ = [("x", ctypes.c_void_p), ("w", ctypes.c_void_p), ("q", ctypes.c_void_p),
                    ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("tokens", ctypes.c_int32),
                    ("hidden", ctypes.c_int32), ("shape", Shape), ("workspace", ctypes.c_void_p)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_sched", "num_decodes", "num_tokens", "nnz_pages", "n_items",
                                             "n_partials", "n_merge", "max_kv_len")] + \
               [("pairs", ctypes.c_int64), ("history_tokens", ctypes.c_int64)] + \
               [(n, ctypes.c_int32) for n in ("off_req_index", "off_num_new", "off_last_chunk", "off_qo_indptr",
                                             "off_kv_page_indptr", "off_kv_page_indices", "off_kv_last_page_len",
                                             "off_req_aux", "off_items", "packed_ints")] + \
               [("workspace_bytes", ctypes.c_int64), ("n_first", ctypes.c_int32), ("first_sms", ctypes.c_int32)]


class AttnArgs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("plan", ctypes.c_void_p), ("info", ctypes.POINTER(PlanInfo)),
                ("rope_table", ctypes.c_void_p), ("rope_max_pos", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_int64),
                ("shape", Shape), ("sm_scale", ctypes.c_float), ("rope_style", ctypes.c_int32),
                ("plan_host", ctypes.c_void_p)]


class HostIO(ctypes.Structure):
    _fields_ = [("q_host", ctypes.c_void_p), ("k_host", ctypes.c_void_p), ("v_host", ctypes.c_void_p),
                ("out_host", ctypes.c_void_p), ("wait_event", ctypes.c_void_p), ("done_event", ctypes.c_void_p)]


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libsarathi.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and _build.stale():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise ImportError(f"libsarathi.so not built at {_build.LIB}")
    lib = ctypes.CDLL(_build.LIB)
    lib.sarathi_plan_bounds.restype = ctypes.c_int32
    lib.sarathi_plan_bounds.argtypes = [ctypes.POINTER(Request), ctypes.c_int32, ctypes.c_int32,
                                        ctypes.POINTER(Shape), ctypes.c_int32,
                                        ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]
    lib.sarathi_plan.restype = ctypes.c_int32
    lib.sarathi_plan.argtypes = [ctypes.POINTER(Request), ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(Shape),
                                 ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(PlanInfo)]
    lib.sarathi_qkv_proj.restype = ctypes.c_int32
    lib.sarathi_qkv_proj.argtypes = [ctypes.POINTER(QkvArgs), ctypes.c_void_p]
    lib.sarathi_split_metadata.restype = ctypes.c_int32
    lib.sarathi_split_metadata.argtypes = [ctypes.POINTER(PlanInfo), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                           ctypes.POINTER(MetaSet), ctypes.POINTER(MetaSet)]
    lib.sarathi_advance.restype = ctypes.c_int32
    lib.sarathi_advance.argtypes = [ctypes.POINTER(Request), ctypes.c_int32, ctypes.POINTER(PlanInfo),
                                    ctypes.c_void_p]
    lib.sarathi_plan_ex.restype = ctypes.c_int32
    lib.sarathi_plan_ex.argtypes = [ctypes.POINTER(Request), ctypes.c_int32, ctypes.POINTER(PlanPolicy),
                                    ctypes.POINTER(Shape), ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                                    ctypes.POINTER(PlanInfo)]
    lib.sarathi_rope_table.restype = ctypes.c_int32
    lib.sarathi_rope_table.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                       ctypes.c_void_p]
    lib.sarathi_mixed_attn.restype = ctypes.c_int32
    lib.sarathi_mixed_attn.argtypes = [ctypes.POINTER(AttnArgs), ctypes.c_void_p]
    lib.sarathi_mixed_attn_host.restype = ctypes.c_int32
    lib.sarathi_mixed_attn_host.argtypes = [ctypes.POINTER(AttnArgs), ctypes.POINTER(HostIO), ctypes.c_void_p]
    lib.sarathi_mixed_attn_noalloc.restype = ctypes.c_int32
    lib.sarathi_mixed_attn_noalloc.argtypes = [ctypes.POINTER(AttnArgs), ctypes.c_void_p]
    lib.sarathi_noalloc_status.restype = ctypes.c_int32
    lib.sarathi_noalloc_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    lib.sarathi_workspace_status.restype = ctypes.c_int32
    lib.sarathi_workspace_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    lib.sarathi_last_error.restype = ctypes.c_char_p
    lib.sarathi_last_error.argtypes = []
    lib.sarathi_abi_version.restype = ctypes.c_int32
    lib.sarathi_abi_version.argtypes = []
    _lib = lib
    return lib


def sarathi_last_error() -> str:
    return load().sarathi_last_error().decode()


def sarathi_abi_version() -> int:
    return int(load().sarathi_abi_version())


def _check(st: int, where: str, allow=(OK,)):
    if st not in allow:
        raise SarathiError(st, where, sarathi_last_error())
    return st


# sarathi_request as a numpy record (4 int32, then the page pointer at byte 16)
_REQ_DTYPE = np.dtype({"names": ["state", "prompt_len", "num_computed", "num_pages", "pages"],
                       "formats": ["<i4", "<i4", "<i4", "<i4", "<u8"], "offsets": [0, 4, 8, 12, 16],
                       "itemsize": ctypes.sizeof(Request)})
assert ctypes.sizeof(Request) == 24 and Request.pages.offset == 16


def make_requests(states, prompt_len, num_computed, block_tables):
    """ctypes request array plus what it points into (keep both alive while
    the array is in use).  The array is a view of a numpy record array filled
    column by column, and the block tables are concatenated once, so the cost
    does not grow with a Python loop per request."""
    n = len(states)
    lens = np.fromiter(map(len, block_tables), dtype=np.int64, count=n)
    if n and int(lens.sum()):
        pages = np.ascontiguousarray(np.concatenate(block_tables), dtype=np.int32)
        if pages.ndim != 1 or pages.size != int(lens.sum()):
            raise ValueError("block tables must be 1-D sequences of page ids")
    else:
        pages = np.zeros(1, np.int32)
    rec = np.zeros(max(n, 1), dtype=_REQ_DTYPE)
    if n:
        rec["state"][:n] = states
        rec["prompt_len"][:n] = prompt_len
        rec["num_computed"][:n] = num_computed
        rec["num_pages"][:n] = lens
        starts = np.zeros(n, np.int64)
        np.cumsum(lens[:-1], out=starts[1:])
        rec["pages"][:n] = pages.ctypes.data + 4 * starts
    arr = (Request * max(n, 1)).from_buffer(rec)
    return arr, (rec, pages)


def sarathi_plan_bounds(reqs, n_reqs: int, token_budget: int, shape: Shape, num_sms: int):
    hb, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load().sarathi_plan_bounds(reqs, n_reqs, token_budget, ctypes.byref(shape), num_sms,
                                      ctypes.byref(hb), ctypes.byref(wb)), "sarathi_plan_bounds")
    return int(hb.value), int(wb.value)


def sarathi_plan(reqs, n_reqs: int, token_budget: int, shape: Shape, num_sms: int,
                 host_buf: np.ndarray | None = None):
    """Returns (status, PlanInfo, packed int32 array).  Raises on errors; the
    over-budget-decodes warning is returned as a status."""
    if host_buf is None:
        hb, _ = sarathi_plan_bounds(reqs, n_reqs, token_budget, shape, num_sms)
        host_buf = np.zeros(hb // 4 + 4, dtype=np.int32)
    info = PlanInfo()
    st = load().sarathi_plan(reqs, n_reqs, token_budget, ctypes.byref(shape), num_sms,
                             host_buf.ctypes.data, host_buf.nbytes, ctypes.byref(info))
    _check(st, "sarathi_plan", allow=(OK, WARN_OVER_BUDGET_DECODES))
    return st, info, host_buf[:info.packed_ints]

def sarathi_split_metadata(info: PlanInfo, packed: np.ndarray):
    """The plan's decode and prefill metadata sets: returns (decode, prefill),
    each a dict of qo_indptr / kv_page_indptr / kv_page_indices /
    kv_last_page_len plus rows, tokens, token_offset, first_row."""
    packed = np.ascontiguousarray(packed, dtype=np.int32)
    out = np.zeros(3 * info.n_sched + 4 + info.nnz_pages, dtype=np.int32)
    d, p = MetaSet(), MetaSet()
    _check(load().sarathi_split_metadata(ctypes.byref(info), packed.ctypes.data, out.ctypes.data, out.nbytes,
                                         ctypes.byref(d), ctypes.byref(p)), "sarathi_split_metadata")

    def view(m):
        return dict(rows=m.rows, tokens=m.tokens, token_offset=m.token_offset, first_row=m.first_row,
                    qo_indptr=out[m.off_qo_indptr:m.off_qo_indptr + m.rows + 1].copy(),
                    kv_page_indptr=out[m.off_kv_page_indptr:m.off_kv_page_indptr + m.rows + 1].copy(),
                    kv_page_indices=out[m.off_kv_page_indices:m.off_kv_page_indices + m.nnz_pages].copy(),
                    kv_last_page_len=out[m.off_kv_last_page_len:m.off_kv_last_page_len + m.rows].copy())
    return view(d), view(p)


def sarathi_advance(reqs, n_reqs: int, info: PlanInfo, packed: np.ndarray) -> None:
    """Apply the step's plan to the ctypes request array in place."""
    packed = np.ascontiguousarray(packed, dtype=np.int32)
    _check(load().sarathi_advance(reqs, n_reqs, ctypes.byref(info), packed.ctypes.data), "sarathi_advance")


def sarathi_plan_ex(reqs, n_reqs: int, policy: PlanPolicy, shape: Shape, num_sms: int,
                    host_buf: np.ndarray | None = None):
    """sarathi_plan with a batch policy; returns (status, PlanInfo, packed int32 array)."""
    if host_buf is None:
        hb, _ = sarathi_plan_bounds(reqs, n_reqs, policy.token_budget, shape, num_sms)
        host_buf = np.zeros(hb // 4 + 4, dtype=np.int32)
    info = PlanInfo()
    st = load().sarathi_plan_ex(reqs, n_reqs, ctypes.byref(policy), ctypes.byref(shape), num_sms,
                                host_buf.ctypes.data, host_buf.nbytes, ctypes.byref(info))
    _check(st, "sarathi_plan_ex", allow=(OK, WARN_OVER_BUDGET_DECODES))
    return st, info, host_buf[:info.packed_ints]


def plan_arrays(info: PlanInfo, packed: np.ndarray) -> dict:
    """Views of the packed plan buffer by name."""
    n = info.n_sched

    def view(off, count):
        return packed[off:off + count]
    return dict(
        n_sched=n, num_decodes=info.num_decodes, num_tokens=info.num_tokens, nnz_pages=info.nnz_pages,
        req_index=view(info.off_req_index, n), num_new=view(info.off_num_new, n),
        last_chunk=view(info.off_last_chunk, n), qo_indptr=view(info.off_qo_indptr, n + 1),
        kv_page_indptr=view(info.off_kv_page_indptr, n + 1),
        kv_page_indices=view(info.off_kv_page_indices, info.nnz_pages),
        kv_last_page_len=view(info.off_kv_last_page_len, n), req_aux=view(info.off_req_aux, n),
        items=view(info.off_items, info.n_items * ITEM_INTS).reshape(info.n_items, ITEM_INTS),
    )


def _stream_ptr(stream) -> int:
    if stream is None:
        return 0
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def sarathi_rope_table(table, max_pos: int, head_dim: int, rope_theta: float, stream=None) -> None:
    """Fill ``table`` (torch float64 CUDA tensor of 2*max_pos*head_dim elements)."""
    _check(load().sarathi_rope_table(table.data_ptr(), max_pos, head_dim, rope_theta, _stream_ptr(stream)),
           "sarathi_rope_table")


def _attn_args(q, k, v, k_cache, v_cache, out, plan_dev, info, rope_table, rope_max_pos, workspace, shape,
               sm_scale, rope_style, plan_host) -> AttnArgs:
    a = AttnArgs()
    if plan_host is not None:
        a.plan_host = plan_host.data_ptr() if hasattr(plan_host, "data_ptr") else plan_host.ctypes.data
    a.q, a.k, a.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    a.k_cache, a.v_cache, a.out = k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr()
    a.plan = plan_dev.data_ptr()
    a.info = ctypes.pointer(info)
    a.rope_table = rope_table.data_ptr()
    a.rope_max_pos = int(rope_max_pos)
    a.num_pages = int(k_cache.shape[0])
    a.workspace = workspace.data_ptr()
    a.workspace_bytes = int(workspace.numel() * workspace.element_size())
    a.shape = shape
    a.sm_scale = float(sm_scale)
    a.rope_style = int(rope_style)
    return a


def sarathi_mixed_attn(q, k, v, k_cache, v_cache, out, plan_dev, info: PlanInfo, rope_table, rope_max_pos: int,
                       workspace, shape: Shape, sm_scale: float, stream=None, rope_style: int = ROPE_ROTATE_HALF,
                       plan_host=None) -> None:
    """Enqueue one step (one kernel) on ``stream`` (torch.cuda.Stream or raw handle).
    plan_host: optional host tensor or array holding the packed plan; the call
    then copies it into plan_dev first (same stream)."""
    a = _attn_args(q, k, v, k_cache, v_cache, out, plan_dev, info, rope_table, rope_max_pos, workspace, shape,
                   sm_scale, rope_style, plan_host)
    _check(load().sarathi_mixed_attn(ctypes.byref(a), _stream_ptr(stream)), "sarathi_mixed_attn")


def _event_ptr(ev, stream) -> int:
    """Raw cudaEvent_t of a torch.cuda.Event (created by recording it once on
    ``stream`` if torch has not created it yet), of a raw handle, or 0."""
    if ev is None:
        return 0
    if hasattr(ev, "cuda_event"):
        if not ev.cuda_event:
            ev.record(stream)
        return int(ev.cuda_event)
    return int(ev)


def sarathi_mixed_attn_host(q_host, k_host, v_host, out_host, q, k, v, k_cache, v_cache, out, plan_dev,
                            info: PlanInfo, rope_table, rope_max_pos: int, workspace, shape: Shape,
                            sm_scale: float, stream=None, rope_style: int = ROPE_ROTATE_HALF, plan_host=None,
                            wait_event=None, done_event=None) -> None:
    """The step end to end from host buffers on ``stream``: q_host, k_host,
    v_host (pinned host tensors) copied into the device q, k, v; the plan from
    plan_host into plan_dev; a wait for ``wait_event``; the kernel;
    ``done_event`` recorded; out copied into out_host (pinned)."""
    a = _attn_args(q, k, v, k_cache, v_cache, out, plan_dev, info, rope_table, rope_max_pos, workspace, shape,
                   sm_scale, rope_style, plan_host)
    io = HostIO(q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), out_host.data_ptr(),
                _event_ptr(wait_event, stream), _event_ptr(done_event, stream))
    _check(load().sarathi_mixed_attn_host(ctypes.byref(a), ctypes.byref(io), _stream_ptr(stream)),
           "sarathi_mixed_attn_host")


def sarathi_mixed_attn_noalloc(q, k, v, k_cache, v_cache, out, plan_dev, info: PlanInfo, rope_table,
                               rope_max_pos: int, shape: Shape, sm_scale: float, stream=None,
                               rope_style: int = ROPE_ROTATE_HALF) -> None:
    """Enqueue one step without a caller workspace: the library's built-in
    scratch array is used (see include/sarathi.h for its limits)."""
    a = AttnArgs()
    a.q, a.k, a.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    a.k_cache, a.v_cache, a.out = k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr()
    a.plan = plan_dev.data_ptr()
    a.info = ctypes.pointer(info)
    a.rope_table = rope_table.data_ptr()
    a.rope_max_pos = int(rope_max_pos)
    a.num_pages = int(k_cache.shape[0])
    a.workspace = None
    a.workspace_bytes = 0
    a.shape = shape
    a.sm_scale = float(sm_scale)
    a.rope_style = int(rope_style)
    _check(load().sarathi_mixed_attn_noalloc(ctypes.byref(a), _stream_ptr(stream)), "sarathi_mixed_attn_noalloc")


def sarathi_qkv_proj(x, w, q, k, v, shape: Shape, workspace, stream=None) -> None:
    """Enqueue Y = X W^T split into q, k, v (bf16 device tensors: x [T][hidden],
    w [(H_q + 2 H_kv) d][hidden], q [T][H_q][d], k / v [T][H_kv][d])."""
    a = QkvArgs()
    a.x, a.w, a.q, a.k, a.v = x.data_ptr(), w.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr()
    a.tokens = int(x.shape[0])
    a.hidden = int(x.shape[1])
    a.shape = shape
    a.workspace = workspace.data_ptr()
    _check(load().sarathi_qkv_proj(ctypes.byref(a), _stream_ptr(stream)), "sarathi_qkv_proj")


def sarathi_noalloc_status(stream=None) -> int:
    """Synchronise, read and clear the error word of the built-in scratch array
    of sarathi_mixed_attn_noalloc on the current device (0 = fine)."""
    err = ctypes.c_int32(0)
    st = load().sarathi_noalloc_status(_stream_ptr(stream), ctypes.byref(err))
    if st not in (OK, ERR_DEVICE_CHECK):
        _check(st, "sarathi_noalloc_status")
    return int(err.value)


def sarathi_workspace_status(workspace, stream=None) -> int:
    """Synchronise, read and clear the kernel's error word; returns it (0 = fine)."""
    err = ctypes.c_int32(0)
    st = load().sarathi_workspace_status(workspace.data_ptr(), _stream_ptr(stream), ctypes.byref(err))
    if st not in (OK, ERR_DEVICE_CHECK):
        _check(st, "sarathi_workspace_status")
    return int(err.value)
