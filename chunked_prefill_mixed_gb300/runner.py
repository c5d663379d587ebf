"""A small host-side driver around the C ABI: owns the RoPE table and the
workspace on one device, plans a step, copies the packed plan to the device
and enqueues the step kernel.  PyTorch is used for device memory and streams
only; all computation runs in libsarathi."""
from __future__ import annotations

import math

import numpy as np
import torch

from . import (PlanInfo, PlanPolicy, Shape, make_requests, sarathi_mixed_attn, sarathi_plan, sarathi_plan_bounds,
               sarathi_plan_ex, sarathi_rope_table, sarathi_workspace_status)


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
        self._host_buf = np.zeros(0, dtype=np.int32)

    def plan(self, states, prompt_len, num_computed, block_tables, budget: int, policy: PlanPolicy | None = None):
        """Plans into a host buffer the runner keeps (grown when a batch needs
        more); the returned packed array is a view of it, valid until the
        next call.  policy: a PlanPolicy for sarathi_plan_ex (its token_budget
        is used); None plans with sarathi_plan and `budget`."""
        reqs, keep = make_requests(states, prompt_len, num_computed, block_tables)
        tb = policy.token_budget if policy is not None else budget
        hb, _ = sarathi_plan_bounds(reqs, len(states), tb, self.shape, self.num_sms)
        if self._host_buf.nbytes < hb:
            self._host_buf = np.zeros(max(hb // 4 + 4, 2 * self._host_buf.size), dtype=np.int32)
        if policy is not None:
            return sarathi_plan_ex(reqs, len(states), policy, self.shape, self.num_sms, self._host_buf)
        return sarathi_plan(reqs, len(states), budget, self.shape, self.num_sms, self._host_buf)

    def ensure_workspace(self, nbytes: int):
        if self.workspace.numel() < nbytes:
            torch.cuda.current_stream(self.device).wait_stream(self.stream)
            self.workspace = torch.zeros(max(nbytes, 2 * self.workspace.numel()), dtype=torch.uint8,
                                         device=self.device)
            self.stream.wait_stream(torch.cuda.current_stream(self.device))

    def upload(self, packed: np.ndarray) -> torch.Tensor:
        src = torch.from_numpy(np.ascontiguousarray(packed))
        dev = torch.empty(src.numel() + 4, dtype=torch.int32, device=self.device)
        dev[:src.numel()].copy_(src)
        self.stream.wait_stream(torch.cuda.current_stream(self.device))
        return dev

    def run(self, q, k, v, k_cache, v_cache, out, plan_dev: torch.Tensor, info: PlanInfo) -> None:
        self.ensure_workspace(int(info.workspace_bytes))
        if info.max_kv_len > self.max_pos:
            raise ValueError(f"RoPE table covers {self.max_pos} positions, batch needs {info.max_kv_len}")
        sarathi_mixed_attn(q, k, v, k_cache, v_cache, out, plan_dev, info, self.rope, self.max_pos,
                           self.workspace, self.shape, self.sm_scale, self.stream, self.rope_style)

    def status(self) -> int:
        return sarathi_workspace_status(self.workspace, self.stream)
