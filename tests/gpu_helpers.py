"""Shared pieces of the GPU parity tests: run a workload's step through the C
ABI on the device and compute the oracle's answer on the same inputs."""
from __future__ import annotations

import numpy as np

import oracle
import workloads as W

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def to_u16(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_u16(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


class GpuStep:
    """One workload step on the GPU: history caches, new-token values, plan."""

    def __init__(self, wl: W.Workload, runner=None, seed_offset: int = 0, host_history: bool | None = None,
                 max_pos: int | None = None, policy: tuple | None = None, rope_style: int = 0):
        """policy: (kind, token_budget, max_batch, chunk_align) to plan with
        sarathi_plan_ex (and the oracle's same policy) instead of the workload's
        stall-free budget."""
        import torch
        from chunked_prefill_mixed_gb300.runner import StepRunner
        self.wl = wl
        self.rope_style = rope_style
        sh = wl.shape
        self.dev = torch.device("cuda")
        if policy is None:
            self.st_o, self.meta = oracle.plan(*wl.arrays(), wl.budget, sh.page_size)
        else:
            kind, tb, mb, al = policy
            self.st_o, self.meta = oracle.plan(*wl.arrays(), tb, sh.page_size, policy=kind, max_batch=mb, align=al)
        T = self.meta["num_tokens"]
        self.q, self.k, self.v = W.new_token_values(T, sh, wl.seed + seed_offset)
        elems = wl.num_pages * sh.H_kv * sh.page_size * sh.d
        small = elems < (64 << 20) if host_history is None else host_history
        if small:
            kc, vc = W.history_cache_numpy(wl.num_pages, sh, wl.seed)
            self.kc0, self.vc0 = kc, vc
            self.kc_dev, self.vc_dev = from_u16(kc, self.dev), from_u16(vc, self.dev)
        else:
            self.kc_dev, self.vc_dev = W.history_cache_torch(wl.num_pages, sh, wl.seed, self.dev)
            self.kc0, self.vc0 = to_u16(self.kc_dev), to_u16(self.vc_dev)
        self.runner = runner or StepRunner(sh.H_q, sh.H_kv, sh.d, max_pos or self._max_pos(), device=self.dev,
                                           rope_theta=sh.rope_base, rope_style=rope_style)
        if policy is None:
            self.status, self.info, self.packed = self.runner.plan(*wl.arrays(), wl.budget)
        else:
            from chunked_prefill_mixed_gb300 import PlanPolicy
            self.status, self.info, self.packed = self.runner.plan(*wl.arrays(), 0, policy=PlanPolicy(*policy))
        self.packed = self.packed.copy()  # the runner's buffer is reused by its next plan
        self.plan_dev = self.runner.upload(self.packed)
        self.q_dev, self.k_dev, self.v_dev = (from_u16(x, self.dev) for x in (self.q, self.k, self.v))
        self.out = torch.full((T, sh.H_q, sh.d), float("nan"), dtype=torch.bfloat16, device=self.dev)

    def _max_pos(self):
        m = self.meta
        if m["n_sched"] == 0:
            return 16
        kv = (np.diff(m["kv_page_indptr"]) - 1) * 16 + m["kv_last_page_len"]
        return int(kv.max()) + 16

    def run(self):
        import torch
        self.runner.run(self.q_dev, self.k_dev, self.v_dev, self.kc_dev, self.vc_dev, self.out, self.plan_dev,
                        self.info)
        torch.cuda.synchronize()
        self.last_header = self.runner.workspace[:64].view(torch.int32).cpu().numpy().copy()
        err = self.runner.status()
        torch.cuda.synchronize()
        return err

    def oracle_caches(self):
        sh = self.wl.shape
        kc, vc = self.kc0.copy(), self.vc0.copy()
        oracle.append(self.meta, self.k, self.v, sh.H_kv, sh.d, sh.page_size, sh.rope_base, kc, vc,
                      style=self.rope_style)
        return kc, vc

    def oracle_rows(self, kc, vc, rows_t=None, rows_hq=None):
        sh = self.wl.shape
        out, lse, rt, rh = oracle.attend(self.meta, self.q, sh.H_q, sh.H_kv, sh.d, sh.page_size, sh.rope_base,
                                         kc, vc, rows_t, rows_hq, style=self.rope_style)
        return out, rt, rh

    def sample_rows(self, n_random: int, seed: int = 0):
        """Every prefill chunk's first and last rows (all heads), the first
        decodes, plus random (row, head) pairs."""
        sh = self.wl.shape
        m = self.meta
        rng = np.random.default_rng(seed)
        qo = m["qo_indptr"]
        rows = []
        for s in range(m["n_sched"]):
            n = qo[s + 1] - qo[s]
            picks = {qo[s], qo[s + 1] - 1} if n > 1 else ({qo[s]} if s < 8 else set())
            for t in picks:
                for hq in range(sh.H_q):
                    rows.append((int(t), hq))
        T = int(qo[-1])
        for _ in range(n_random):
            rows.append((int(rng.integers(0, T)), int(rng.integers(0, sh.H_q))))
        rows = sorted(set(rows))
        return np.array([r[0] for r in rows], np.int32), np.array([r[1] for r in rows], np.int32)


def assert_close(gpu_rows: np.ndarray, ref_rows: np.ndarray, what: str = ""):
    g = gpu_rows.astype(np.float64)
    diff = np.abs(g - ref_rows)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU outputs"
    mx, mean = float(diff.max()), float(diff.mean())
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max-abs {mx:.3e} mean-abs {mean:.3e}"
    return mx, mean
