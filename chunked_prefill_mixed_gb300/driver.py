"""A multi-step serving loop around the step: requests arrive on a trace, each
iteration plans a batch (sarathi_plan / sarathi_plan_ex), runs the step kernel
on synthetic q/k/v for the scheduled tokens, and applies the plan to the
requests (sarathi_advance).  A request yields one output token per step in
which it decodes or finishes its prompt; it leaves when it has produced its
max_new tokens, and its pages go back to the pool.

This is the loop of "Sarathi-Serve 完全拆解" §"一个 512-token 预算的例子" run
for many steps, used to measure how uniform the iterations are (§"流水并行收益
来自方差，不只来自均值").  Only the attention step runs on the GPU; the linear
layers are not part of it."""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

import numpy as np
import torch

from . import DECODE, PREFILL_WAITING, PlanPolicy, make_requests, plan_arrays, sarathi_advance


class PageAllocator:
    """Free list of page ids of one pool."""

    def __init__(self, num_pages: int):
        self.free = deque(range(num_pages))

    def alloc(self, n: int) -> np.ndarray:
        if n > len(self.free):
            raise MemoryError(f"page pool exhausted: need {n}, have {len(self.free)}")
        return np.array([self.free.popleft() for _ in range(n)], dtype=np.int32)

    def release(self, pages) -> None:
        self.free.extend(int(p) for p in pages)


@dataclass
class ServeRequest:
    rid: int
    prompt_len: int
    max_new: int
    pages: np.ndarray
    state: int = PREFILL_WAITING
    num_computed: int = 0
    generated: int = 0


@dataclass
class StepRecord:
    iteration: int
    tokens: int
    decodes: int
    prefill_tokens: int
    chunks: int
    kernel_us: float
    active: int
    plan: dict | None = field(default=None, repr=False)


class MultiStepDriver:
    """runner: a StepRunner for the shape; k_cache / v_cache: the device pools;
    trace: workloads.Arrival list; policy: PlanPolicy or None (stall-free with
    `budget`); values(iteration, T) -> (q, k, v) for the step's tokens, as bf16
    bit arrays (uint16) or bf16 device tensors."""

    def __init__(self, runner, k_cache, v_cache, num_pages: int, trace, values, budget: int = 512,
                 policy: PlanPolicy | None = None, page_size: int = 16):
        self.runner = runner
        self.kc, self.vc = k_cache, v_cache
        self.pages = PageAllocator(num_pages)
        self.trace = sorted(trace, key=lambda a: a.iteration)
        self.next_arrival = 0
        self.values = values
        self.budget = budget
        self.policy = policy
        self.page_size = page_size
        self.active: list[ServeRequest] = []
        self.done: list[ServeRequest] = []
        self.iteration = 0
        self.device = runner.device

    def _admit(self):
        while self.next_arrival < len(self.trace) and self.trace[self.next_arrival].iteration <= self.iteration:
            a = self.trace[self.next_arrival]
            need = -(-(a.prompt_len + a.max_new) // self.page_size)
            self.active.append(ServeRequest(self.next_arrival, a.prompt_len, a.max_new, self.pages.alloc(need)))
            self.next_arrival += 1

    def finished(self) -> bool:
        return self.next_arrival >= len(self.trace) and not self.active

    def step(self, keep: bool = False) -> StepRecord:
        """One iteration.  keep=True also returns the plan arrays, the inputs and
        the output in the record (for checking against the oracle)."""
        self._admit()
        act = self.active
        states = [r.state for r in act]
        prompt = [r.prompt_len for r in act]
        computed = [r.num_computed for r in act]
        tables = [r.pages for r in act]
        rec = StepRecord(self.iteration, 0, 0, 0, 0, 0.0, len(act))
        if act:
            st, info, packed = self.runner.plan(states, prompt, computed, tables, self.budget, policy=self.policy)
            packed = packed.copy()
            T = info.num_tokens
            rec.tokens, rec.decodes = T, info.num_decodes
            m = plan_arrays(info, packed)
            rec.chunks = int(info.n_sched - info.num_decodes)
            rec.prefill_tokens = T - info.num_decodes
            if T > 0:
                q, k, v = self.values(self.iteration, T)
                if isinstance(q, torch.Tensor):
                    qd, kd, vd = q, k, v   # already bf16 on the device
                else:
                    bf = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(
                        torch.bfloat16).to(self.device)
                    qd, kd, vd = bf(q), bf(k), bf(v)
                out = torch.empty((T, qd.shape[1], qd.shape[2]), dtype=torch.bfloat16, device=self.device)
                pd = self.runner.upload(packed)
                stream = self.runner.stream
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                self.runner.run(qd, kd, vd, self.kc, self.vc, out, pd, info)
                b.record(stream)
                b.synchronize()
                rec.kernel_us = 1e3 * a.elapsed_time(b)
                if self.runner.status() != 0:
                    raise RuntimeError(f"device error at iteration {self.iteration}")
                if keep:
                    rec.plan = dict(meta=m, states=states, prompt=prompt, computed=computed,
                                    tables=[t.copy() for t in tables], q=q, k=k, v=v, out=out)
                # the plan applied to the requests
                reqs, _keep = make_requests(states, prompt, computed, tables)
                sarathi_advance(reqs, len(act), info, packed)
                produced = set()
                for s in range(int(info.n_sched)):
                    i = int(m["req_index"][s])
                    if act[i].state == DECODE or m["last_chunk"][s]:
                        produced.add(i)
                for i, r in enumerate(act):
                    r.state, r.num_computed = int(reqs[i].state), int(reqs[i].num_computed)
                    if i in produced:
                        r.generated += 1
                if keep:
                    rec.plan["after_states"] = [r.state for r in act]
                    rec.plan["after_computed"] = [r.num_computed for r in act]
                still = []
                for r in act:
                    if r.generated >= r.max_new:
                        self.pages.release(r.pages)
                        self.done.append(r)
                    else:
                        still.append(r)
                self.active = still
        self.iteration += 1
        return rec
