"""The oracle: a plain fp64 CPU restatement of the mixed-batch paged-attention
step (chunked prefill with stall-free batching).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg import this package.  The CUDA library never
links or calls it, and it never imports the CUDA library: the two share no code.
The arithmetic lives in ``sarathi_oracle.c`` (built with gcc on first use); this
module is argument marshalling only.

Pages followed (titles as printed on them):
  "Sarathi-Serve 完全拆解：分块 Prefill 与无停顿批处理如何兼顾吞吐和尾延迟"
  "Chunked Prefill 与 PD 分离：切片混批，还是拆开两个池"
  "分块预填充与 Stall-free 调度：把 LLM 推理的吞吐-延迟权衡算清楚"
Each C function's comment names the section it restates.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sarathi_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, INVALID, CAPACITY, OVER_BUDGET_DECODES = 0, 1, 2, 3
DECODE, PREFILL_RUNNING, PREFILL_WAITING = 0, 1, 2

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc, -O2, OpenMP)."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    lib.oracle_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_rope.restype = None
    lib.oracle_rope.argtypes = [_f64p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, _f64p]
    lib.oracle_rope_styled.restype = None
    lib.oracle_rope_styled.argtypes = [_f64p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_int, _f64p]
    lib.oracle_plan.restype = ctypes.c_int
    lib.oracle_plan.argtypes = [ctypes.c_int, _i32p, _i32p, _i32p, _i32p, _i32p,
                                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                _i32p, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p]
    lib.oracle_advance.restype = ctypes.c_int
    lib.oracle_advance.argtypes = [ctypes.c_int, _i32p, _i32p, _i32p, ctypes.c_int, _i32p, _i32p]
    lib.oracle_plan_policy.restype = ctypes.c_int
    lib.oracle_plan_policy.argtypes = [ctypes.c_int, _i32p, _i32p, _i32p, _i32p, _i32p,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int,
                                       _i32p, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p]
    lib.oracle_append_styled.restype = None
    lib.oracle_append.restype = None
    lib.oracle_append.argtypes = [ctypes.c_int, _i32p, _i32p, _i32p, _i32p, _u16p, _u16p,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                  _u16p, _u16p]
    lib.oracle_attend_styled.restype = None
    lib.oracle_attend.restype = None
    lib.oracle_attend.argtypes = [ctypes.c_int, _i32p, _i32p, _i32p, _i32p, _u16p,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_double, _u16p, _u16p, ctypes.c_int, _i32p, _i32p,
                                  _f64p, _f64p]
    lib.oracle_append_styled.argtypes = [ctypes.c_int, _i32p, _i32p, _i32p, _i32p, _u16p, _u16p,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                         _u16p, _u16p]
    lib.oracle_attend_styled.argtypes = [ctypes.c_int, _i32p, _i32p, _i32p, _i32p, _u16p,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_double, ctypes.c_int, _u16p, _u16p, ctypes.c_int, _i32p, _i32p,
                                         _f64p, _f64p]
    lib.oracle_pairs.restype = ctypes.c_int64
    lib.oracle_pairs.argtypes = [ctypes.c_int, _i32p, _i32p, _i32p, ctypes.c_int]
    lib.oracle_reread_tokens.restype = ctypes.c_int64
    lib.oracle_reread_tokens.argtypes = [ctypes.c_int, _i32p, _i32p, _i32p, ctypes.c_int]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_set_num_threads.restype = None
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the OpenMP loops from now on."""
    _load().oracle_set_num_threads(int(n))


def bf16_rne(x) -> np.ndarray:
    """Round each double to bf16 (ties to even, one rounding); returns uint16 bits."""
    lib = _load()
    flat = np.asarray(x, dtype=np.float64).ravel()
    out = np.fromiter((lib.oracle_bf16_rne(float(v)) for v in flat), dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(x))


def bf16_to_double(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


ROTATE_HALF, INTERLEAVED = 0, 1


def rope(x, pos: int, base: float = 10000.0, style: int = ROTATE_HALF) -> np.ndarray:
    """RoPE of one vector at absolute position ``pos``, fp64; style ROTATE_HALF
    pairs (j, j + d/2), INTERLEAVED pairs (2j, 2j + 1)."""
    lib = _load()
    xv = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty_like(xv)
    if style == ROTATE_HALF:
        lib.oracle_rope(xv, xv.size, int(pos), float(base), out)
    else:
        lib.oracle_rope_styled(xv, xv.size, int(pos), float(base), int(style), out)
    return out


STALL_FREE, DECODE_MAXIMAL = 0, 1


def plan(states, prompt_len, num_computed, block_tables, budget: int, page_size: int,
         policy: int | None = None, max_batch: int = 0, align: int = 1):
    """Budgeted batch; returns (status, dict of metadata arrays).  policy None:
    stall-free through oracle_plan; otherwise oracle_plan_policy with the given
    policy (STALL_FREE / DECODE_MAXIMAL: budget = chunk size), max_batch (B,
    decode-maximal only, 0 = no limit) and chunk alignment."""
    lib = _load()
    n = len(states)
    bt_indptr = np.zeros(n + 1, dtype=np.int32)
    for i, t in enumerate(block_tables):
        bt_indptr[i + 1] = bt_indptr[i] + len(t)
    bt = _i32(np.concatenate([np.asarray(t, dtype=np.int32) for t in block_tables]) if n else [])
    if bt.size == 0:
        bt = np.zeros(1, dtype=np.int32)
    cap_pages = int(bt_indptr[-1]) + 1
    req_index = np.zeros(max(n, 1), np.int32)
    num_new = np.zeros(max(n, 1), np.int32)
    last_chunk = np.zeros(max(n, 1), np.int32)
    qo = np.zeros(n + 1, np.int32)
    kvp = np.zeros(n + 1, np.int32)
    kvi = np.zeros(cap_pages, np.int32)
    last = np.zeros(max(n, 1), np.int32)
    counts = np.zeros(4, np.int32)
    reqs = (_i32(states) if n else np.zeros(1, np.int32), _i32(prompt_len) if n else np.zeros(1, np.int32),
            _i32(num_computed) if n else np.zeros(1, np.int32), bt_indptr, bt)
    outs = (req_index, num_new, last_chunk, qo, kvp, kvi, last, counts)
    if policy is None:
        st = lib.oracle_plan(n, *reqs, int(budget), int(page_size), cap_pages, *outs)
    else:
        st = lib.oracle_plan_policy(n, *reqs, int(policy), int(budget), int(max_batch), int(align),
                                    int(page_size), cap_pages, *outs)
    ns = int(counts[0])
    meta = dict(
        n_sched=ns, num_decodes=int(counts[1]), nnz_pages=int(counts[2]), num_tokens=int(counts[3]),
        req_index=req_index[:ns].copy(), num_new=num_new[:ns].copy(), last_chunk=last_chunk[:ns].copy(),
        qo_indptr=qo[:ns + 1].copy(), kv_page_indptr=kvp[:ns + 1].copy(),
        kv_page_indices=kvi[:int(counts[2])].copy(), kv_last_page_len=last[:ns].copy(),
    )
    return int(st), meta


def advance(states, prompt_len, num_computed, meta):
    """Request state after the step the plan `meta` describes: returns (status,
    new states, new num_computed) as lists."""
    lib = _load()
    n = len(states)
    st_a = _i32(states).copy() if n else np.zeros(1, np.int32)
    pl = _i32(prompt_len) if n else np.zeros(1, np.int32)
    nc = _i32(num_computed).copy() if n else np.zeros(1, np.int32)
    ns = int(meta["n_sched"])
    ri = _i32(meta["req_index"]) if ns else np.zeros(1, np.int32)
    nn = _i32(meta["num_new"]) if ns else np.zeros(1, np.int32)
    st = lib.oracle_advance(n, st_a, pl, nc, ns, ri, nn)
    return int(st), st_a[:n].tolist(), nc[:n].tolist()


def _meta_arrays(meta):
    ns = int(meta["n_sched"]) if "n_sched" in meta else len(meta["qo_indptr"]) - 1
    kvi = _i32(meta["kv_page_indices"])
    if kvi.size == 0:
        kvi = np.zeros(1, np.int32)
    last = _i32(meta["kv_last_page_len"])
    if last.size == 0:
        last = np.zeros(1, np.int32)
    return ns, _i32(meta["qo_indptr"]), _i32(meta["kv_page_indptr"]), kvi, last


def append(meta, k_bits, v_bits, H_kv: int, d: int, page_size: int, base: float,
           k_cache: np.ndarray, v_cache: np.ndarray, style: int = ROTATE_HALF) -> None:
    """Write the step's new K (rotated, bf16) and V into the caches, in place.
    Caches: uint16 [num_pages][H_kv][page_size][d]."""
    lib = _load()
    ns, qo, kvp, kvi, last = _meta_arrays(meta)
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
    kb = np.ascontiguousarray(k_bits, dtype=np.uint16).reshape(-1)
    vb = np.ascontiguousarray(v_bits, dtype=np.uint16).reshape(-1)
    if kb.size == 0:
        return
    lib.oracle_append_styled(ns, qo, kvp, kvi, last, kb, vb, H_kv, d, page_size, float(base), int(style),
                      k_cache.reshape(-1), v_cache.reshape(-1))


def attend(meta, q_bits, H_q: int, H_kv: int, d: int, page_size: int, base: float,
           k_cache: np.ndarray, v_cache: np.ndarray, rows_t=None, rows_hq=None, style: int = ROTATE_HALF):
    """fp64 attention outputs for (row, q-head) pairs (all pairs if None).
    Returns (out [n_pairs][d], lse [n_pairs], rows_t, rows_hq)."""
    lib = _load()
    ns, qo, kvp, kvi, last = _meta_arrays(meta)
    T = int(qo[-1]) if qo.size else 0
    if rows_t is None:
        rows_t = np.repeat(np.arange(T, dtype=np.int32), H_q)
        rows_hq = np.tile(np.arange(H_q, dtype=np.int32), T)
    rows_t = _i32(rows_t)
    rows_hq = _i32(rows_hq)
    n = rows_t.size
    out = np.zeros((max(n, 1), d), np.float64)
    lse = np.zeros(max(n, 1), np.float64)
    if n:
        qb = np.ascontiguousarray(q_bits, dtype=np.uint16).reshape(-1)
        lib.oracle_attend_styled(ns, qo, kvp, kvi, last, qb, H_q, H_kv, d, page_size, float(base), int(style),
                          np.ascontiguousarray(k_cache).reshape(-1), np.ascontiguousarray(v_cache).reshape(-1),
                          n, rows_t, rows_hq, out.reshape(-1), lse)
    return out[:n], lse[:n], rows_t, rows_hq


def step(meta, q_bits, k_bits, v_bits, H_q: int, H_kv: int, d: int, page_size: int,
         base: float, k_cache: np.ndarray, v_cache: np.ndarray, style: int = ROTATE_HALF):
    """One whole step: append every new token, then attend every (row, q head).
    Returns out [T][H_q][d] (fp64); the caches are updated in place."""
    append(meta, k_bits, v_bits, H_kv, d, page_size, base, k_cache, v_cache, style)
    out, _, _, _ = attend(meta, q_bits, H_q, H_kv, d, page_size, base, k_cache, v_cache, style=style)
    T = int(meta["qo_indptr"][-1])
    return out.reshape(T, H_q, d)


def pairs(meta, page_size: int) -> int:
    lib = _load()
    ns, qo, kvp, _, last = _meta_arrays(meta)
    return int(lib.oracle_pairs(ns, qo, kvp, last, page_size))


def reread_tokens(meta, page_size: int) -> int:
    lib = _load()
    ns, qo, kvp, _, last = _meta_arrays(meta)
    return int(lib.oracle_reread_tokens(ns, qo, kvp, last, page_size))


def qkv_proj(x_bits, w_bits, H_q: int, H_kv: int, d: int):
    """The Q/K/V projection of the step's tokens, in fp64: Y = X W^T with X
    bf16 [T][hidden] and W bf16 [(H_q + 2 H_kv) d][hidden] (rows: q heads, then
    k heads, then v heads); returns q [T][H_q][d], k, v [T][H_kv][d].
    "Sarathi：让解码搭上 prefill 的顺风车" §"Decode-maximal batching：顺车的账本":
    the linear layer of all the batch's tokens is one matrix product."""
    x = bf16_to_double(np.asarray(x_bits))
    w = bf16_to_double(np.asarray(w_bits))
    y = x @ w.T
    T = x.shape[0]
    nq, nk = H_q * d, H_kv * d
    return (y[:, :nq].reshape(T, H_q, d), y[:, nq:nq + nk].reshape(T, H_kv, d),
            y[:, nq + nk:nq + 2 * nk].reshape(T, H_kv, d))
