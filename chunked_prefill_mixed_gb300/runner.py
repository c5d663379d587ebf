"""A small host-side driver around the C ABI: owns the RoPE table and the
workspace on one device, plans a step, copies the packed plan to the device
and enqueues the step kernel.  PyTorch is used for device memory and streams
only; all computation runs in libsarathi."""
from __future__ import annotations

import math

import numpy as np
import torch

from . import (ERR_CAPACITY, PlanInfo, PlanPolicy, SarathiError, Shape, make_requests, sarathi_mixed_attn,
               sarathi_mixed_attn_host,
               sarathi_plan, sarathi_plan_bounds, sarathi_plan_ex, sarathi_rope_table, sarathi_workspace_status)


class StepRunner:
    def __init__(self, H_q: int, H_kv: int, d: int, max_pos: int, device="cuda", rope_theta: float = 10000.0,
                 page_size: int = 16, stream=None, rope_style: int = 0):
        self.shape = Shape(H_q, H_kv, d, page_size)
        self.device = torch.device(device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.num_sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        self.sm_scale = 1.0 / math.sqrt(d)
        self.rope_style = rope_style  # 0 rotate-half, 1 interleaved
        self.max_pos = int(max_pos)
        self.rope = torch.empty(2 * self.max_pos * d, dtype=torch.float64, device=self.device)
        sarathi_rope_table(self.rope, self.max_pos, d, rope_theta, self.stream)
        self.workspace = torch.zeros(1 << 16, dtype=torch.uint8, device=self.device)
        # the packed plan is written straight into pinned memory, so that its
        # copy to the device is one asynchronous DMA from there; PLAN_BUFFERS
        # buffers in turn, so that the host can plan up to two steps ahead of
        # the GPU without waiting
        n = self.PLAN_BUFFERS
        self._host_ts = [torch.empty(0, dtype=torch.int32) for _ in range(n)]
        self._cur = 0
        # a device copy of each: a step's plan buffers are free again once the
        # event recorded after its step call has passed
        self._plan_devs = [torch.empty(0, dtype=torch.int32, device=self.device) for _ in range(n)]
        self._upload_evts = [torch.cuda.Event() for _ in range(n)]
        self._uploaded = [False] * n  # a copy out of buffer i may be in flight (_upload_evts[i])

    PLAN_BUFFERS = 3

    def plan(self, states, prompt_len, num_computed, block_tables, budget: int, policy: PlanPolicy | None = None):
        """Plans into one of three pinned host buffers the runner keeps (taken
        in turn, grown when a batch needs more); the returned packed array is a
        view of it, valid until the next call.  The buffer's previous use
        (three plans ago) is waited for, not the last one, so a step can be
        planned while the steps before it run.  policy: a PlanPolicy
        for sarathi_plan_ex (its token_budget is used); None plans with
        sarathi_plan and `budget`."""
        reqs, keep = make_requests(states, prompt_len, num_computed, block_tables)
        return self.plan_requests(reqs, len(states), budget, policy)

    def plan_requests(self, reqs, n_reqs: int, budget: int, policy: PlanPolicy | None = None):
        """plan() from a request table the caller keeps (the ctypes array of
        make_requests, with its block tables alive; a serving loop advances it
        in place with sarathi_advance between steps)."""
        tb = policy.token_budget if policy is not None else budget
        self._cur = (self._cur + 1) % self.PLAN_BUFFERS
        c = self._cur
        if self._uploaded[c]:
            self._upload_evts[c].synchronize()  # that plan's copy has left the buffer
            self._uploaded[c] = False
        host_buf = self._host_ts[c].numpy()
        for attempt in range(2):
            try:
                if policy is not None:
                    return sarathi_plan_ex(reqs, n_reqs, policy, self.shape, self.num_sms, host_buf)
                return sarathi_plan(reqs, n_reqs, budget, self.shape, self.num_sms, host_buf)
            except SarathiError as e:
                if e.status != ERR_CAPACITY or attempt:
                    raise
                # host_buf too small, or a block table too short: size the
                # buffer by the bounds and plan again (the bounds call fails
                # the same way in the second case)
                hb, _ = sarathi_plan_bounds(reqs, n_reqs, tb, self.shape, self.num_sms)
                if host_buf.nbytes >= hb:
                    raise
                self._host_ts[c] = torch.empty(max(hb // 4 + 4, 2 * host_buf.size), dtype=torch.int32,
                                               pin_memory=True)
                host_buf = self._host_ts[c].numpy()

    def upload_plan(self, info: PlanInfo) -> torch.Tensor:
        """Enqueues on the runner's stream the copy of the packed plan of the
        last plan() call (pinned memory) into a device buffer the runner
        keeps; returns that buffer, valid until the next upload_plan."""
        n = int(info.packed_ints)
        c = self._cur
        dev = self._plan_device_buffer(n)
        # (the buffer is pinned once plan() has sized it)
        if torch.cuda.current_stream(self.device) == self.stream:
            dev[:n].copy_(self._host_ts[c][:n], non_blocking=True)
        else:
            with torch.cuda.stream(self.stream):
                dev[:n].copy_(self._host_ts[c][:n], non_blocking=True)
        self._upload_evts[c].record(self.stream)
        self._uploaded[c] = True
        return dev

    def _plan_device_buffer(self, n: int) -> torch.Tensor:
        c = self._cur
        if self._plan_devs[c].numel() < n + 4:
            torch.cuda.synchronize(self.device)  # the old buffer may be in use by an enqueued step
            self._plan_devs[c] = torch.empty(max(n + 4, 2 * self._plan_devs[c].numel()), dtype=torch.int32,
                                             device=self.device)
        return self._plan_devs[c]

    def ensure_workspace(self, nbytes: int):
        if self.workspace.numel() < nbytes:
            # rare: wait for every stream that may run a step on the old one
            torch.cuda.synchronize(self.device)
            self.workspace = torch.zeros(max(nbytes, 2 * self.workspace.numel()), dtype=torch.uint8,
                                         device=self.device)
            torch.cuda.synchronize(self.device)

    def upload(self, packed: np.ndarray) -> torch.Tensor:
        src = torch.from_numpy(np.ascontiguousarray(packed))
        dev = torch.empty(src.numel() + 4, dtype=torch.int32, device=self.device)
        dev[:src.numel()].copy_(src)
        self.stream.wait_stream(torch.cuda.current_stream(self.device))
        return dev

    def run(self, q, k, v, k_cache, v_cache, out, plan_dev: torch.Tensor, info: PlanInfo, plan_host=None) -> None:
        self.ensure_workspace(int(info.workspace_bytes))
        if info.max_kv_len > self.max_pos:
            raise ValueError(f"RoPE table covers {self.max_pos} positions, batch needs {info.max_kv_len}")
        sarathi_mixed_attn(q, k, v, k_cache, v_cache, out, plan_dev, info, self.rope, self.max_pos,
                           self.workspace, self.shape, self.sm_scale, self.stream, self.rope_style, plan_host)

    def run_planned(self, q, k, v, k_cache, v_cache, out, info: PlanInfo) -> None:
        """Enqueues the step planned by the last plan() call: one library call
        copies the packed plan from the runner's pinned buffer into its device
        buffer and launches the kernel."""
        c = self._cur
        dev = self._plan_device_buffer(int(info.packed_ints))
        self.run(q, k, v, k_cache, v_cache, out, dev, info, plan_host=self._host_ts[c])
        self._upload_evts[c].record(self.stream)
        self._uploaded[c] = True

    def run_host(self, q_host, k_host, v_host, out_host, q, k, v, k_cache, v_cache, out, info: PlanInfo,
                 stream=None, wait_event=None, done_event=None) -> None:
        """Enqueues the step planned by the last plan() call end to end from
        host buffers (one library call, sarathi_mixed_attn_host) on ``stream``
        (default: the runner's): q_host, k_host, v_host (pinned) into the
        device q, k, v, the plan into the runner's device buffer, a wait for
        ``wait_event``, the kernel, ``done_event``, out into out_host
        (pinned).  Alternating two streams, each with its own q, k, v, out
        and host buffers and the other's last done_event as wait_event,
        overlaps one step's copies and the host's planning of the next with
        the kernel before it."""
        stream = self.stream if stream is None else stream
        self.ensure_workspace(int(info.workspace_bytes))
        if info.max_kv_len > self.max_pos:
            raise ValueError(f"RoPE table covers {self.max_pos} positions, batch needs {info.max_kv_len}")
        c = self._cur
        dev = self._plan_device_buffer(int(info.packed_ints))
        sarathi_mixed_attn_host(q_host, k_host, v_host, out_host, q, k, v, k_cache, v_cache, out, dev, info,
                                self.rope, self.max_pos, self.workspace, self.shape, self.sm_scale, stream,
                                self.rope_style, self._host_ts[c], wait_event, done_event)
        self._upload_evts[c].record(stream)
        self._uploaded[c] = True

    def status(self) -> int:
        return sarathi_workspace_status(self.workspace, self.stream)
