"""Seeded synthetic inputs for the mixed-batch paged-attention step.

This module only draws inputs: request states, block tables (page ids) and
bf16 values.  It holds none of the step's arithmetic (no planning, no RoPE, no
attention), so both the oracle's tests and the CUDA path's tests and benchmark
can use it without sharing any of the method with each other.

Workload shapes follow the configurations the step is measured on:

  tiny      1 layer, 4 q / 4 kv heads, d_h 64, page 16; 2 decodes (context 100
            and 37) and one 200-token prompt prefilled in chunks of 64 over 4
            steps under a 66-token budget.
  mistral   32 q / 8 kv heads, d_h 128; budget 512 = 80 decodes (context
            uniform 256..4096) + running prefill P (300 tokens left, no
            history) + running prefill Q (900 left after 768 of history).
  llama7b   32 / 32 heads, d_h 128; one 8192-token prompt under budget 2048
            next to 64 decodes (context uniform 512..8192).
  llama70b  64 q / 8 kv heads; budget 1536 = 200 decodes (context lognormal,
            median 2048, sigma 1, cap 16384) + running A (12288 history, 500
            left) + running B (4096 history, 600 left) + waiting C (2000-token
            prompt).
  yi34b     56 q / 8 kv heads; 256 decodes (context 4096) + one 256-token chunk
            after 3840 of history, budget 512; physical pages randomly permuted.

Values: every q, k, v and history K/V element is N(0,1) rounded to bf16.
Seeds: tiny 0, mistral 1, llama7b 2, llama70b 3, yi34b 4.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

DECODE, PREFILL_RUNNING, PREFILL_WAITING = 0, 1, 2
PAGE = 16


@dataclass
class Shape:
    H_q: int
    H_kv: int
    d: int
    page_size: int = PAGE
    rope_base: float = 10000.0


@dataclass
class Request:
    state: int
    prompt_len: int
    num_computed: int
    pages: np.ndarray  # int32 physical page ids (the block table)


@dataclass
class Workload:
    name: str
    shape: Shape
    budget: int
    requests: list
    num_pages: int
    seed: int
    notes: dict = field(default_factory=dict)

    def arrays(self):
        """Flat request arrays: states, prompt_len, num_computed, block tables."""
        st = np.array([r.state for r in self.requests], np.int32)
        pl = np.array([r.prompt_len for r in self.requests], np.int32)
        nc = np.array([r.num_computed for r in self.requests], np.int32)
        return st, pl, nc, [r.pages for r in self.requests]


SHAPES = {
    "tiny": Shape(4, 4, 64),
    "mistral": Shape(32, 8, 128),
    "llama7b": Shape(32, 32, 128),
    "llama70b": Shape(64, 8, 128),
    "yi34b": Shape(56, 8, 128),
}
SEEDS = {"tiny": 0, "mistral": 1, "llama7b": 2, "llama70b": 3, "yi34b": 4}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (input drawing only)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16))
    return r.astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


class _PagePool:
    """Hands out physical page ids: contiguous, or through a fixed permutation."""

    def __init__(self, total: int, rng: np.random.Generator | None = None):
        self.total = total
        self.next = 0
        self.perm = rng.permutation(total).astype(np.int32) if rng is not None else None

    def take(self, n: int) -> np.ndarray:
        if self.next + n > self.total:
            raise ValueError("page pool exhausted")
        ids = np.arange(self.next, self.next + n, dtype=np.int32)
        self.next += n
        return self.perm[ids] if self.perm is not None else ids


def _pages_for(tokens: int, page_size: int = PAGE) -> int:
    return (tokens + page_size - 1) // page_size


def _build(name, shape, budget, specs, seed, permute=False, spare_pages=0, notes=None):
    """specs: list of (state, prompt_len, num_computed, kv_capacity_tokens)."""
    total = sum(_pages_for(cap, shape.page_size) for (_, _, _, cap) in specs) + spare_pages
    rng = np.random.default_rng(seed + 1000)
    pool = _PagePool(total, rng if permute else None)
    reqs = [Request(st, pl, nc, pool.take(_pages_for(cap, shape.page_size))) for (st, pl, nc, cap) in specs]
    return Workload(name, shape, budget, reqs, total, seed, notes or {})


def tiny(step: int = 0) -> Workload:
    """Step ``step`` (0..3) of the tiny schedule: decodes at context 100+step and
    37+step; the 200-token prompt has 64*step tokens computed."""
    shape = SHAPES["tiny"]
    L = 200
    specs = [
        (DECODE, 0, 100 + step, 100 + 4 + 1),
        (DECODE, 0, 37 + step, 37 + 4 + 1),
        (PREFILL_WAITING if step == 0 else PREFILL_RUNNING, L, 64 * step, L),
    ]
    return _build("tiny", shape, 66, specs, SEEDS["tiny"], notes={"step": step, "prompt_len": L})


def mistral() -> Workload:
    shape = SHAPES["mistral"]
    seed = SEEDS["mistral"]
    rng = np.random.default_rng(seed)
    ctx = rng.integers(256, 4096, size=80, endpoint=True)
    specs = [(PREFILL_RUNNING, 300, 0, 300)]
    specs += [(DECODE, 0, int(c), int(c) + 1) for c in ctx[:40]]
    specs += [(PREFILL_RUNNING, 768 + 900, 768, 768 + 900)]
    specs += [(DECODE, 0, int(c), int(c) + 1) for c in ctx[40:]]
    return _build("mistral", shape, 512, specs, seed)


def llama7b(chunk_step: int = 3, budget: int = 2048, n_decodes: int = 64, prompt: int = 8192) -> Workload:
    """The 8192-token prompt with ``computed`` = (budget - n_decodes) * chunk_step
    tokens already prefilled (clipped to the prompt), next to the decodes."""
    shape = SHAPES["llama7b"]
    seed = SEEDS["llama7b"]
    rng = np.random.default_rng(seed)
    ctx = rng.integers(512, 8192, size=n_decodes, endpoint=True)
    per = budget - n_decodes
    computed = min(prompt, per * chunk_step) if per > 0 else 0
    state = PREFILL_WAITING if computed == 0 else PREFILL_RUNNING
    specs = [(DECODE, 0, int(c), int(c) + 1) for c in ctx]
    specs.append((state, prompt, computed, prompt))
    return _build("llama7b", shape, budget, specs, seed,
                  notes={"chunk_step": chunk_step, "history": computed})


def llama7b_prefill_only(chunk: int, step: int, prompt: int = 8192) -> Workload:
    """Prefill-only sweep: the 8192-token prompt alone, budget = chunk; step k
    has k*chunk tokens computed."""
    shape = SHAPES["llama7b"]
    computed = min(prompt, chunk * step)
    state = PREFILL_WAITING if computed == 0 else PREFILL_RUNNING
    return _build("llama7b_prefill", shape, chunk, [(state, prompt, computed, prompt)], SEEDS["llama7b"],
                  notes={"chunk": chunk, "step": step})


def llama70b() -> Workload:
    shape = SHAPES["llama70b"]
    seed = SEEDS["llama70b"]
    rng = np.random.default_rng(seed)
    ctx = np.floor(rng.lognormal(mean=np.log(2048.0), sigma=1.0, size=200)).astype(np.int64)
    ctx = np.clip(ctx, 1, 16384)
    specs = [(DECODE, 0, int(c), int(c) + 1) for c in ctx]
    specs.append((PREFILL_RUNNING, 12288 + 500, 12288, 12288 + 500))
    specs.append((PREFILL_RUNNING, 4096 + 600, 4096, 4096 + 600))
    specs.append((PREFILL_WAITING, 2000, 0, 2000))
    return _build("llama70b", shape, 1536, specs, seed)


def yi34b() -> Workload:
    shape = SHAPES["yi34b"]
    seed = SEEDS["yi34b"]
    specs = [(DECODE, 0, 4096, 4097) for _ in range(256)]
    specs.append((PREFILL_RUNNING, 4096, 3840, 4096))
    return _build("yi34b", shape, 512, specs, seed, permute=True)


WORKLOADS = {
    "tiny": tiny,
    "mistral": mistral,
    "llama7b": llama7b,
    "llama70b": llama70b,
    "yi34b": yi34b,
}


def new_token_values(T: int, shape: Shape, seed: int):
    """bf16 bits for the step's new tokens: q [T][H_q][d], k, v [T][H_kv][d]."""
    rng = np.random.default_rng(seed + 7919)
    q = normal_bf16(rng, (T, shape.H_q, shape.d))
    k = normal_bf16(rng, (T, shape.H_kv, shape.d))
    v = normal_bf16(rng, (T, shape.H_kv, shape.d))
    return q, k, v


def history_cache_numpy(num_pages: int, shape: Shape, seed: int):
    """Host K/V page pools filled with N(0,1) bf16 (uint16 bits)."""
    rng = np.random.default_rng(seed + 104729)
    dims = (num_pages, shape.H_kv, shape.page_size, shape.d)
    return normal_bf16(rng, dims), normal_bf16(rng, dims)


def history_cache_torch(num_pages: int, shape: Shape, seed: int, device):
    """Device K/V page pools filled with N(0,1) bf16 drawn by torch's generator
    on ``device`` (fast for multi-GB pools)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed + 104729)
    dims = (num_pages, shape.H_kv, shape.page_size, shape.d)
    out = []
    for _ in range(2):
        t = torch.empty(dims, dtype=torch.bfloat16, device=device)
        flat = t.view(num_pages, -1)
        step = max(1, (64 << 20) // flat.shape[1])  # about 64 M elements per draw
        for p0 in range(0, num_pages, step):
            blk = flat[p0:p0 + step]
            blk.copy_(torch.randn(blk.shape, generator=g, device=device, dtype=torch.float32))
        out.append(t)
    return out[0], out[1]


# ---------------------------------------------------------------- arrival traces
# Stand-ins for the pages' two request-length distributions (a chat set and a
# summarisation set, whose prompts are much longer and outputs shorter): the
# datasets are not used; lengths are drawn lognormal with the medians below.
TRACE_KINDS = {
    #               prompt median, sigma, clip        output median, sigma, clip
    "chat": ((800, 0.8, (32, 6000)), (150, 0.8, (8, 600))),
    "summarization": ((5000, 0.5, (1000, 14000)), (100, 0.5, (16, 400))),
}


@dataclass
class Arrival:
    iteration: int      # step at which the request becomes visible to the scheduler
    prompt_len: int
    max_new: int        # output tokens (the first comes with the last prefill chunk)


def arrival_trace(kind: str, n: int, mean_gap: float, seed: int) -> list[Arrival]:
    """n requests; gaps between arrivals (in steps) exponential with the given
    mean, rounded down; lengths as TRACE_KINDS[kind]."""
    (pm, ps, (plo, phi)), (om, os_, (olo, ohi)) = TRACE_KINDS[kind]
    rng = np.random.default_rng(seed + 65537)
    t = 0.0
    out = []
    for _ in range(n):
        pl = int(np.clip(np.exp(np.log(pm) + ps * rng.standard_normal()), plo, phi))
        mn = int(np.clip(np.exp(np.log(om) + os_ * rng.standard_normal()), olo, ohi))
        out.append(Arrival(int(t), pl, mn))
        t += rng.exponential(mean_gap)
    return out
