"""Benchmark of the mixed-batch paged-attention step (one kernel launch per step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama7b]
                    [--impl ours|reference]

Prints ONE JSON line on rank 0.  ``value`` is tokens/s over the whole job: the
step's new tokens (decodes + prefill chunk tokens) divided by the kernel's
device time (CUDA events on the launching stream, L2 flushed before every
timed step).  ``e2e`` is the same metric through the public API with the
step's inputs in pinned host memory: host planning, host->device copies, the
kernel and the device->host read of the outputs inside the timed region.
``--impl reference`` times the oracle (plain fp64 CPU code) on a bounded
sample of the same workload.  Under torchrun every rank runs its own replica
(the step needs no exchange between GPUs).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "mixed-batch paged attn: μs/step, tokens/s, % of roofline (HBM or TC)"
UNIT = "tokens/s"
DESCR = {
    "mistral": "Mistral-7B-like attention layer (32 q / 8 kv heads, d 128, page 16), budget 512: "
               "80 decodes (context U[256,4096]) + running prefill P (300 left, no history) + "
               "running prefill Q (132 of 900 left, 768 history)",
    "llama7b": "Llama-2-7B-like MHA layer (32/32 heads, d 128), budget 2048: 64 decodes (context U[512,8192]) "
               "+ 1984-token chunk of an 8192-token prompt after 5952 history",
    "llama70b": "LLaMA2-70B-like GQA layer (64 q / 8 kv, d 128), budget 1536: 200 decodes (lognormal context) + "
                "chunks (12288,500), (4096,600), (0,236)",
    "yi34b": "Yi-34B-like layer (56 q / 8 kv, d 128), budget 512, fragmented pages: 256 decodes (context 4096) + "
             "256-token chunk after 3840 history",
    "tiny": "tiny layer (4/4 heads, d 64), budget 66: 2 decodes + 64-token chunk",
    "llama7b_oneshot": "Llama-2-7B-like MHA layer, prefill-only: one 8192-token prompt in one shot",
    "llama7b_c512": "Llama-2-7B-like MHA layer, prefill-only: last 512-token chunk of an 8192-token prompt",
    "llama7b_c2048": "Llama-2-7B-like MHA layer, prefill-only: last 2048-token chunk of an 8192-token prompt",
}


def make_workload(name: str) -> W.Workload:
    if name == "llama7b":
        return W.llama7b(chunk_step=3)
    if name == "llama7b_oneshot":
        return W.llama7b_prefill_only(8192, 0)
    if name.startswith("llama7b_c"):
        c = int(name[len("llama7b_c"):])
        return W.llama7b_prefill_only(c, 8192 // c - 1)
    return W.WORKLOADS[name]()


def algorithmic(wl: W.Workload, meta) -> dict:
    """Algorithmic FLOP and bytes of one step: FLOP = 4 d H_q pairs; bytes =
    Q in + raw K,V in + K,V page writes + history K,V read once per request + O out."""
    sh = wl.shape
    n = np.diff(meta["qo_indptr"]).astype(np.int64)
    kv = (np.diff(meta["kv_page_indptr"]).astype(np.int64) - 1) * 16 + meta["kv_last_page_len"].astype(np.int64)
    h = kv - n
    T = int(n.sum())
    pairs = int((n * h + n * (n + 1) // 2).sum())
    flop = 4.0 * sh.d * sh.H_q * pairs
    byt = (2.0 * T * sh.H_q * sh.d + 4.0 * T * sh.H_kv * sh.d + 4.0 * T * sh.H_kv * sh.d
           + 4.0 * float(h.sum()) * sh.H_kv * sh.d + 2.0 * T * sh.H_q * sh.d)
    return {"T": T, "pairs": pairs, "flop": flop, "bytes": byt, "history": int(h.sum())}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


def _code_only(src: str) -> str:
    """C++ source without comments or blank lines, so that a profile stays keyed to
    the code that ran when only the comments change.  String literals are kept as
    they are."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(l.rstrip() for l in "".join(out).splitlines() if l.strip())


def kernel_source_sha(read=None) -> str:
    """Hash of the code (comments stripped) of the three sources that make the
    step kernel and its plan."""
    h = hashlib.sha256()
    for f in ("mixed_attn.cu", "sarathi_internal.h", "plan.cpp"):
        rel = os.path.join("chunked_prefill_mixed_gb300", "csrc", f)
        src = read(rel) if read else open(os.path.join(ROOT, rel)).read()
        h.update(_code_only(src).encode())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel source as it is now."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        e = json.load(open(p)).get(workload)
        if e and e.get("src_sha") == kernel_source_sha():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        return None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def clocks_summary(nvml: dict, smi: dict) -> dict:
    """The NVML samples taken inside the timed region when there are any (the
    nvidia-smi samples, every 100 ms around it, beside them), else nvidia-smi's."""
    if nvml.get("samples"):
        out = dict(nvml)
        out["reasons"] = sorted(set(nvml["reasons"]) | set(smi.get("reasons") or []))
        out["nvidia_smi"] = smi
        return out
    return smi


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (the driver's
    libnvidia-ml, by ctypes) every half millisecond while the timed region
    runs, so that a region of a few milliseconds still holds samples; read-only.
    Any failure leaves it empty (the nvidia-smi sampler still reports)."""

    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, index: int, uuid: str | None = None):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.ok = False
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            got = False
            if uuid:
                u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                got = nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0
            if not got and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
                return
            try:
                self.get_reasons = nv.nvmlDeviceGetCurrentClocksEventReasons
            except AttributeError:
                self.get_reasons = nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nv, self.h, self.ct = nv, h, ctypes
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
                self.max_mhz = float(mx.value)
            self.ok = True
        except Exception:
            self.ok = False

    def __enter__(self):
        if self.ok:
            self._stop = False
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        return self

    def _run(self):
        nv, h, ct = self.nv, self.h, self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self._stop:
            try:
                if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0:
                    self.samples.append(float(clk.value))
                if self.get_reasons(h, ct.byref(rs)) == 0:
                    for bit, name in self.REASONS.items():
                        if rs.value & bit:
                            self.reasons.add(name)
            except Exception:
                return
            time.sleep(0.0005)

    def __exit__(self, *a):
        if self.ok:
            self._stop = True
            self.thread.join(timeout=2)

    def summary(self):
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples), "source": "nvml, every 0.5 ms"}


def reduce_max(values, world: int, device=None):
    """Max over ranks of per-rank timings (all_reduce MAX); the job is as slow
    as its slowest replica."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tokens_per_s(tokens_per_step: int, world: int, seconds_per_step: float) -> float:
    """Whole-job throughput: every replica processes its own step's tokens."""
    return world * tokens_per_step / seconds_per_step


def oracle_sample_time(wl: W.Workload, meta, q, k, v, kc, vc, budget_s: float, seed: int = 0):
    """Time the oracle on a bounded sample of the step: every append plus the
    attention of random (row, head) pairs, until ~budget_s of CPU work; scale
    to the full step by the share of query-key pairs the sample covered.
    Returns (estimated seconds per full step, cores, description)."""
    import oracle
    sh = wl.shape
    n = np.diff(meta["qo_indptr"])
    kvl = (np.diff(meta["kv_page_indptr"]) - 1) * 16 + meta["kv_last_page_len"]
    h = kvl - n
    row_keys = np.concatenate([np.arange(h[s] + 1, h[s] + n[s] + 1) for s in range(len(n))]).astype(np.int64)
    total_pairs = int(row_keys.sum()) * sh.H_q
    kcw, vcw = kc.copy(), vc.copy()
    t0 = time.perf_counter()
    oracle.append(meta, k, v, sh.H_kv, sh.d, 16, sh.rope_base, kcw, vcw)
    t_append = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    T = int(meta["qo_indptr"][-1])
    done_pairs, t_attn, batches = 0, 0.0, 0
    batch = max(oracle.num_threads() * 4, 16)
    while t_attn < budget_s and done_pairs < total_pairs:
        rt = rng.integers(0, T, size=batch).astype(np.int32)
        rh = rng.integers(0, sh.H_q, size=batch).astype(np.int32)
        t1 = time.perf_counter()
        oracle.attend(meta, q, sh.H_q, sh.H_kv, sh.d, 16, sh.rope_base, kcw, vcw, rt, rh)
        t_attn += time.perf_counter() - t1
        done_pairs += int(row_keys[rt].sum())
        batches += 1
    est = t_append + t_attn * (total_pairs / max(done_pairs, 1))
    desc = (f"all {T} appends + {batches * batch} random (row, q-head) attention outputs "
            f"({done_pairs / total_pairs:.2%} of the step's query-key pairs), scaled by pairs")
    return est, oracle.num_threads(), desc


def setup_inputs(wl: W.Workload):
    """The oracle's own plan of the workload and the step's new-token values
    (the oracle legs: the reference arm and the CPU baseline)."""
    import oracle
    st, meta = oracle.plan(*wl.arrays(), wl.budget, 16)
    q, k, v = W.new_token_values(meta["num_tokens"], wl.shape, wl.seed)
    return meta, q, k, v


def max_positions(wl: W.Workload) -> int:
    """An upper bound on the KV length of any row the workload can schedule."""
    m = 1
    for r in wl.requests:
        m = max(m, r.num_computed + 1 if r.state == W.DECODE else r.prompt_len)
    return m


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step = a bounded sample of the workload."""
    if rank != 0:
        return None
    wl = make_workload(args.workload)
    meta, q, k, v = setup_inputs(wl)
    kc, vc = W.history_cache_numpy(wl.num_pages, wl.shape, wl.seed)
    alg = algorithmic(wl, meta)
    per_step = max(1.0, args.ref_seconds / max(args.steps + args.warmup, 1))
    times, cores, desc = [], 1, ""
    for i in range(args.warmup + args.steps):
        est, cores, desc = oracle_sample_time(wl, meta, q, k, v, kc, vc, per_step, seed=i)
        if i >= args.warmup:
            times.append(est)
    sec = statistics.mean(times)
    value = alg["T"] / sec
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": DESCR[args.workload]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_ours(args, rank, world, local_rank):
    import torch
    import chunked_prefill_mixed_gb300 as S
    from chunked_prefill_mixed_gb300.runner import StepRunner
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    S.load()
    wl = make_workload(args.workload)
    sh = wl.shape
    kc, vc = W.history_cache_torch(wl.num_pages, sh, wl.seed, dev)
    stream = torch.cuda.Stream(dev)
    runner = StepRunner(sh.H_q, sh.H_kv, sh.d, max_positions(wl) + 16, device=dev, rope_theta=sh.rope_base,
                        stream=stream)
    st, info, packed = runner.plan(*wl.arrays(), wl.budget)
    packed = packed.copy()  # the runner's buffer is reused by its next plan
    runner.ensure_workspace(int(info.workspace_bytes))
    # the roofline's algorithmic bytes and FLOP come from the library's own
    # plan of the step, the metadata the timed kernel runs
    meta = S.plan_arrays(info, packed)
    alg = algorithmic(wl, meta)
    T = alg["T"]
    q, k, v = W.new_token_values(info.num_tokens, sh, wl.seed)

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    # the step's new-token q, k, v side by side in one pinned buffer and one
    # device buffer (so that their host-to-device copy is one DMA)
    nq, nk = q.size, k.size
    qkv_h = torch.cat([bf(x).reshape(-1) for x in (q, k, v)]).pin_memory()
    qkv_d = qkv_h.to(dev)
    q_h, k_h, v_h = qkv_h[:nq].view(q.shape), qkv_h[nq:nq + nk].view(k.shape), qkv_h[nq + nk:].view(v.shape)
    q_d, k_d, v_d = qkv_d[:nq].view(q.shape), qkv_d[nq:nq + nk].view(k.shape), qkv_d[nq + nk:].view(v.shape)
    out = torch.empty((T, sh.H_q, sh.d), dtype=torch.bfloat16, device=dev)
    out_h = torch.empty((T, sh.H_q, sh.d), dtype=torch.bfloat16).pin_memory()
    plan_pin = torch.empty(info.packed_ints + 64, dtype=torch.int32).pin_memory()
    plan_dev = torch.empty(info.packed_ints + 64, dtype=torch.int32, device=dev)
    plan_pin[:info.packed_ints].copy_(torch.from_numpy(packed))
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        plan_dev[:info.packed_ints].copy_(plan_pin[:info.packed_ints], non_blocking=True)
    stream.synchronize()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # > 129 MB L2

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            runner.run(q_d, k_d, v_d, kc, vc, out, plan_dev, info)
    torch.cuda.synchronize(dev)
    hdr = runner.workspace[:64].view(torch.int32).cpu().tolist()
    if runner.status() != 0:
        raise RuntimeError(f"device error during warm-up: workspace header {hdr[:12]}")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    nvml = NvmlSampler(dev.index if dev.index is not None else 0, uuid)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk, nvml:
        t_wall0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush.zero_()
                starts[i].record(stream)
                runner.run(q_d, k_d, v_d, kc, vc, out, plan_dev, info)
                ends[i].record(stream)
        stream.synchronize()
        t_wall = time.perf_counter() - t_wall0
    barrier()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    torch.cuda.synchronize(dev)
    # context only: the same launch with L2 left warm (no flush between launches)
    warm = []
    with torch.cuda.stream(stream):
        for i in range(8):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            runner.run(q_d, k_d, v_d, kc, vc, out, plan_dev, info)
            b.record(stream)
            warm.append((a, b))
    stream.synchronize()
    warm_ms = statistics.median([a.elapsed_time(b) for a, b in warm[3:]])
    hdr = runner.workspace[:64].view(torch.int32).cpu().tolist()
    if runner.status() != 0:
        raise RuntimeError(f"device error in the timed region: workspace header {hdr[:12]}")

    # e2e through the public API: pinned H2D of q, k, v (one copy, enqueued
    # first: it does not depend on the plan), the plan on the host meanwhile
    # (straight into the runner's pinned buffer), its H2D, the kernel, D2H
    h2d = qkv_h.numel() * 2 + info.packed_ints * 4
    d2h = out.numel() * 2
    e2e_times = []
    barrier()
    for i in range(args.steps):
        with torch.cuda.stream(stream):
            flush.zero_()
        stream.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            qkv_d.copy_(qkv_h, non_blocking=True)
            st2, info2, packed2 = runner.plan(*wl.arrays(), wl.budget)
            runner.run_planned(q_d, k_d, v_d, kc, vc, out, info2)
            out_h.copy_(out, non_blocking=True)
        stream.synchronize()
        e2e_times.append(time.perf_counter() - t0)
    barrier()

    # e2e pipelined as a serving loop drives it, through the host-buffer entry
    # (sarathi_mixed_attn_host: q, k, v in, the plan in, the kernel, out back,
    # all enqueued by one library call): two streams in turn, each with its
    # own device buffers, each step's kernel waiting for the one before it;
    # the host plans and enqueues step i, then reads step i - 2's result
    # (three pinned output buffers in turn), so step i's copies and plan
    # overlap the kernels before it.
    streams = [stream, torch.cuda.Stream(dev)]
    dbufs = [(q_d, k_d, v_d, out)] + [tuple(torch.empty_like(x) for x in (q_d, k_d, v_d, out))]
    out_hs = [out_h] + [torch.empty(out_h.shape, dtype=out_h.dtype, pin_memory=True) for _ in range(2)]
    k_done = [torch.cuda.Event(), torch.cuda.Event()]
    o_done = [torch.cuda.Event() for _ in range(3)]
    # the request table, kept across steps as a serving loop keeps it (there
    # it is advanced in place by sarathi_advance; this loop repeats one step)
    reqs_t, keep_t = S.make_requests(*wl.arrays())
    n_reqs = len(wl.requests)
    checks = []
    n_pipe = max(args.steps, 8)
    with torch.cuda.stream(stream):
        flush.zero_()
    barrier()
    t0 = time.perf_counter()
    for i in range(n_pipe):
        b, o = i & 1, i % 3
        st2, info2, packed2 = runner.plan_requests(reqs_t, n_reqs, wl.budget)
        runner.run_host(q_h, k_h, v_h, out_hs[o], *dbufs[b][:3], kc, vc, dbufs[b][3], info2, stream=streams[b],
                        wait_event=k_done[b ^ 1] if i else None, done_event=k_done[b])
        o_done[o].record(streams[b])
        if i >= 2:
            o_done[(i - 2) % 3].synchronize()  # step i - 2's result is on the host
            checks.append(float(out_hs[(i - 2) % 3].view(-1)[0]))
    for i in range(max(n_pipe - 2, 0), n_pipe):
        o_done[i % 3].synchronize()
        checks.append(float(out_hs[i % 3].view(-1)[0]))
    t_pipe = (time.perf_counter() - t0) / n_pipe
    torch.cuda.synchronize(dev)
    barrier()
    if not all(np.isfinite(checks)) or not (torch.equal(out_hs[0], out_hs[1]) and torch.equal(out_hs[0], out_hs[2])):
        raise RuntimeError("pipelined e2e steps disagree")

    ms_per, e2e_s, e2e_serial_s = reduce_max(
        [float(sum(ms)) / args.steps, t_pipe, float(np.mean(e2e_times))], world, device=dev)
    if rank != 0:
        return None
    hbm, tc, tc_sus, peak_kind = load_peaks()
    t_hbm = alg["bytes"] / (hbm * 1e9)
    t_tc = alg["flop"] / (tc * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    sec = ms_per / 1e3
    if bound == "hbm":
        achieved, peak, unit_r = alg["bytes"] / sec / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit_r = alg["flop"] / sec / 1e12, tc, "TFLOP/s"
    res = {
        "metric": METRIC, "value": job_tokens_per_s(T, world, sec), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per, "us_per_step": ms_per * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": DESCR[args.workload], "name": args.workload, "tokens_per_step": T,
                   "l2": "flushed (512 MB write) before every timed step", "replicas": world},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit_r, "frac": achieved / peak,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json, burst)",
                     "roofline_us": max(t_hbm, t_tc) * 1e6, "algorithmic_bytes": alg["bytes"],
                     "algorithmic_flop": alg["flop"], "traffic": committed_traffic(args.workload)},
        "e2e": {"value": job_tokens_per_s(T, world, e2e_s), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "us_per_step": e2e_s * 1e6, "steps": n_pipe,
                "l2": f"not flushed between pipelined steps: a step reads {alg['bytes'] / 1e6:.0f} MB "
                      "(the L2 holds 129 MB)",
                "includes": "per step: the host plan (StepRunner.plan_requests on the kept request table), "
                            "then one library call "
                            "(sarathi_mixed_attn_host) enqueuing pinned H2D of q, k, v and the plan, the kernel "
                            "and D2H of out into pinned memory, and a host read of the result; two streams in "
                            "turn, the host two steps ahead, so a step's copies and plan overlap the kernels "
                            "before it",
                "serial": {"value": job_tokens_per_s(T, world, e2e_serial_s), "us_per_step": e2e_serial_s * 1e6,
                           "includes": "the same, one step at a time (synchronised after each step)"}},
        "clocks": clocks_summary(nvml.summary(), clk.summary()),
        "gpu_launches": args.steps,
        "timing": {"kernel_ms_min": min(ms), "kernel_ms_median": statistics.median(ms), "wall_s": t_wall,
                   "kernel_ms_median_warm_l2": warm_ms},
    }
    if not args.no_cpu_baseline:
        kc_h = kc.view(torch.int16).cpu().numpy().view(np.uint16)
        vc_h = vc.view(torch.int16).cpu().numpy().view(np.uint16)
        # the device caches already hold this step's appends; the oracle
        # re-appends the same values, so the sample sees the same state; the
        # oracle runs its own plan of the step
        meta_o, q, k, v = setup_inputs(wl)
        est, cores, desc = oracle_sample_time(wl, meta_o, q, k, v, kc_h, vc_h, args.cpu_seconds)
        res["cpu_baseline"] = {"value": T / est, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
        # the same oracle on one core, on a smaller sample
        import oracle
        oracle.set_num_threads(1)
        est1, _, desc1 = oracle_sample_time(wl, meta_o, q, k, v, kc_h, vc_h, args.cpu_seconds / 4, seed=1)
        oracle.set_num_threads(cores)
        res["cpu_baseline"]["one_core"] = {"value": T / est1, "unit": UNIT, "sample": desc1}
    return res


def policy_sweep(dev, flush):
    """The Mistral-7B-like request set (80 decodes, prefills P and Q) planned by
    each batch policy: the stall-free 512-token budget, the same with chunks
    aligned to 32, and decode-maximal batching with one 432-token chunk (no
    batch limit) or one 256-token chunk beside at most 47 decodes (B = 48).
    Step time: CUDA events, L2 flushed before each launch, median of 5."""
    import torch
    import chunked_prefill_mixed_gb300 as S
    from chunked_prefill_mixed_gb300.runner import StepRunner
    wl = W.mistral()
    sh = wl.shape
    kc, vc = W.history_cache_torch(wl.num_pages, sh, wl.seed, dev)
    runner = StepRunner(sh.H_q, sh.H_kv, sh.d, 8192, device=dev)
    res = {}
    for label, pol in (("stall_free_512", S.PlanPolicy(S.POLICY_STALL_FREE, 512, 0, 1)),
                       ("stall_free_512_align32", S.PlanPolicy(S.POLICY_STALL_FREE, 512, 0, 32)),
                       ("decode_maximal_c432", S.PlanPolicy(S.POLICY_DECODE_MAXIMAL, 432, 0, 1)),
                       ("decode_maximal_c256_b48", S.PlanPolicy(S.POLICY_DECODE_MAXIMAL, 256, 48, 1))):
        st, info, packed = runner.plan(*wl.arrays(), 0, policy=pol)
        pd = runner.upload(packed)
        n = info.num_tokens
        q, k, v = W.new_token_values(n, sh, wl.seed)

        def bf(x):
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
        qd, kd, vd = bf(q), bf(k), bf(v)
        out = torch.empty((n, sh.H_q, sh.d), dtype=torch.bfloat16, device=dev)
        ms = []
        for i in range(7):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            runner.run(qd, kd, vd, kc, vc, out, pd, info)
            b.record()
            b.synchronize()
            if i >= 2:
                ms.append(a.elapsed_time(b))
        if runner.status() != 0:
            raise RuntimeError("device error in the policy sweep")
        us = 1e3 * statistics.median(ms)
        res[label] = {"tokens": n, "decodes": info.num_decodes, "prefill_tokens": n - info.num_decodes,
                      "us": round(us, 1), "tokens_per_s": round(n / us * 1e6)}
    return res


def run_qkv(args):
    """The QKV projection as one tcgen05 GEMM over the step's concatenated
    tokens (weights read once), against the same tokens projected in two
    GEMMs, decodes alone and the prefill chunk alone (weights read twice):
    the Mistral-7B-like layer (hidden 4096, 32 q / 8 kv heads, d 128) at its
    512-token budget step (80 decodes + 432 prefill tokens) and the
    Llama-2-7B-like layer (hidden 4096, 32 / 32 heads) at its 2048-token step
    (64 decodes + 1984).  CUDA events, L2 flushed before each launch, median of
    7 after 3 warm-ups; torch.matmul (cuBLAS) on the same operands for context."""
    import torch
    import chunked_prefill_mixed_gb300 as S
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    S.load()
    hbm, tc, tc_sus, peak_kind = load_peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(17)

    def timed(fn):
        ms = []
        for i in range(10):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            if i >= 3:
                ms.append(a.elapsed_time(b))
        return 1e3 * statistics.median(ms)

    out = {"qkv": "QKV projection of a mixed batch, one tcgen05 GEMM (bf16 in, fp32 accumulate, bf16 out)",
           "peak": {"tflops": tc, "hbm_gbs": hbm, "source": peak_kind}, "cases": {}}
    for name, hidden, Hq, Hkv, d, n_dec, n_pf in (("mistral_budget512", 4096, 32, 8, 128, 80, 432),
                                                  ("llama7b_budget2048", 4096, 32, 32, 128, 64, 1984)):
        N = (Hq + 2 * Hkv) * d
        T = n_dec + n_pf
        x = torch.randn((T, hidden), generator=gen, device=dev).to(torch.bfloat16)
        w = (torch.randn((N, hidden), generator=gen, device=dev) / hidden ** 0.5).to(torch.bfloat16)
        q = torch.empty((T, Hq, d), dtype=torch.bfloat16, device=dev)
        k = torch.empty((T, Hkv, d), dtype=torch.bfloat16, device=dev)
        v = torch.empty((T, Hkv, d), dtype=torch.bfloat16, device=dev)
        shp = S.Shape(Hq, Hkv, d, 16)

        def proj(r0, r1):
            S.sarathi_qkv_proj(x[r0:r1], w, q[r0:r1], k[r0:r1], v[r0:r1], shp, ws)
        fused = timed(lambda: proj(0, T))
        dec = timed(lambda: proj(0, n_dec))
        pf = timed(lambda: proj(n_dec, T))
        cub = timed(lambda: torch.matmul(x, w.t()))
        if S.sarathi_workspace_status(ws) != 0:
            raise RuntimeError("device error in the QKV projection")
        flop = 2.0 * T * N * hidden
        byt = 2.0 * (T * hidden + N * hidden + T * N)
        out["cases"][name] = {
            "tokens": T, "decodes": n_dec, "prefill_tokens": n_pf, "N": N, "hidden": hidden,
            "fused_us": round(fused, 2), "fused_tflops": round(flop / fused / 1e6, 1),
            "fused_frac_of_tensor_peak": round(flop / fused / 1e6 / tc, 3),
            "roofline_us": round(max(flop / (tc * 1e12), byt / (hbm * 1e9)) * 1e6, 2),
            "separate_us": round(dec + pf, 2), "decode_only_us": round(dec, 2), "prefill_only_us": round(pf, 2),
            "weight_bytes": 2 * N * hidden, "cublas_us": round(cub, 2)}
    print(json.dumps(out), flush=True)
    return None


def run_serve(args):
    """Many steps over an arrival trace (chunked_prefill_mixed_gb300.driver):
    the Mistral-7B-like layer under Sarathi-Serve's stall-free 512-token
    budget, under mixed batching with no chunking (a budget no prompt
    reaches), and under decode-maximal batching with 512-token chunks.  Per
    iteration the step kernel is timed with CUDA events (inputs already on the
    device); reported: distribution of iteration times and tokens/s over the
    whole trace."""
    import torch
    import chunked_prefill_mixed_gb300 as S
    from chunked_prefill_mixed_gb300.driver import MultiStepDriver
    from chunked_prefill_mixed_gb300.runner import StepRunner
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    S.load()
    sh = W.SHAPES["mistral"]
    num_pages = 30000
    gen = torch.Generator(device=dev)

    def values(it, T):
        gen.manual_seed(5000 + it)
        mk = lambda h: torch.randn((T, h, sh.d), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
        return mk(sh.H_q), mk(sh.H_kv), mk(sh.H_kv)

    out = {"serve": "Mistral-7B-like attention layer (32 q / 8 kv heads, d 128), synthetic arrival traces",
           "traces": {}}
    for kind, n_req, gap in (("chat", 48, 3.0), ("summarization", 24, 8.0)):
        trace = W.arrival_trace(kind, n_req, gap, seed=11)
        res = {}
        for label, budget, pol in (("sarathi_serve_budget512", 512, None),
                                   ("mixed_no_chunking", 1 << 20, None),
                                   ("decode_maximal_chunk512", 0, S.PlanPolicy(S.POLICY_DECODE_MAXIMAL, 512, 0, 1))):
            # every page a step reads was written earlier in the trace: zeroed pools
            dims = (num_pages, sh.H_kv, sh.page_size, sh.d)
            kc = torch.zeros(dims, dtype=torch.bfloat16, device=dev)
            vc = torch.zeros(dims, dtype=torch.bfloat16, device=dev)
            runner = StepRunner(sh.H_q, sh.H_kv, sh.d, 16384 + 1024, device=dev)
            drv = MultiStepDriver(runner, kc, vc, num_pages, trace, values, budget=budget, policy=pol)
            recs = []
            while not drv.finished() and len(recs) < 5000:
                recs.append(drv.step())
            us = np.array([r.kernel_us for r in recs if r.tokens > 0])
            toks = sum(r.tokens for r in recs)
            res[label] = {"iterations": len(recs), "tokens": int(toks),
                          "us_mean": round(float(us.mean()), 1), "us_p50": round(float(np.percentile(us, 50)), 1),
                          "us_p99": round(float(np.percentile(us, 99)), 1), "us_max": round(float(us.max()), 1),
                          "us_cv": round(float(us.std() / us.mean()), 3),
                          "tokens_per_s": round(toks / (us.sum() * 1e-6)),
                          "max_prefill_tokens_in_a_step": int(max(r.prefill_tokens for r in recs))}
            del kc, vc, runner, drv
            torch.cuda.empty_cache()
        out["traces"][kind] = {"requests": n_req, "mean_gap_steps": gap, "policies": res}
    print(json.dumps(out), flush=True)
    return None


def run_sweep(args):
    """Whole-prompt prefill of the 8192-token Llama-2-7B-like prompt in chunks
    of 512 / 1024 / 2048 and in one shot (the history re-read of chunked
    prefill), and single chunks of 128/129, 256/257, 512/513 tokens after
    4096 tokens of history (tile quantisation).  Kernel time per step: CUDA
    events, L2 flushed before each timed launch, median of 5."""
    import torch
    import chunked_prefill_mixed_gb300 as S
    from chunked_prefill_mixed_gb300.runner import StepRunner
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    S.load()
    sh = W.SHAPES["llama7b"]
    L = 8192
    base = W.llama7b_prefill_only(L, 0)
    kc, vc = W.history_cache_torch(base.num_pages, sh, base.seed, dev)
    q, k, v = W.new_token_values(L, sh, base.seed)

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
    qd, kd, vd = bf(q), bf(k), bf(v)
    runner = StepRunner(sh.H_q, sh.H_kv, sh.d, L + 64, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    reps = 1 if args.sweep_once else 7

    def time_step(wl, t0):
        st, info, packed = runner.plan(*wl.arrays(), wl.budget)
        pd = runner.upload(packed)
        n = info.num_tokens
        out = torch.empty((n, sh.H_q, sh.d), dtype=torch.bfloat16, device=dev)
        ms = []
        for i in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            runner.run(qd[t0:t0 + n], kd[t0:t0 + n], vd[t0:t0 + n], kc, vc, out, pd, info)
            b.record()
            b.synchronize()
            if i >= 2 or reps == 1:
                ms.append(a.elapsed_time(b))
        if runner.status() != 0:
            raise RuntimeError("device error in the sweep")
        return statistics.median(ms), n, info

    chunks = {}
    for c in (512, 1024, 2048, L):
        done, steps, reread = 0, [], 0
        while done < L:
            wl = W.llama7b_prefill_only(c, done // c)
            ms, n, info = time_step(wl, done)
            steps.append(ms)
            reread += info.history_tokens
            done += n
        chunks[c] = {"prompt_us": 1e3 * sum(steps), "steps": len(steps), "history_tokens_reread": int(reread),
                     "reread_bytes": int(reread) * 4 * sh.H_kv * sh.d, "step_us": [round(1e3 * x, 1) for x in steps]}
    one = chunks[L]["prompt_us"]
    for c in chunks:
        chunks[c]["overhead_vs_one_shot"] = chunks[c]["prompt_us"] / one - 1.0
    if args.sweep_once:
        # one launch per chunk step, for a DRAM-traffic capture of each (ncu)
        print(json.dumps({"sweep_once": {str(c): v["steps"] for c, v in chunks.items()}}), flush=True)
        return None
    tq = {}
    for n in (128, 129, 256, 257, 512, 513):
        wl = W._build("tq", sh, n, [(W.PREFILL_RUNNING, 4096 + n, 4096, 4096 + n)], base.seed)
        ms, _, _ = time_step(wl, 0)
        tq[n] = round(1e3 * ms, 2)
    res = {"sweep": "chunked prefill of one 8192-token prompt (Llama-2-7B-like layer, 32/32 heads, d 128)",
           "chunks": {str(c): v for c, v in chunks.items()},
           "tile_quantisation_us_after_4096_history": {str(k): v for k, v in tq.items()},
           "ratio_257_over_256": tq[257] / tq[256], "ratio_129_over_128": tq[129] / tq[128],
           "ratio_513_over_512": tq[513] / tq[512],
           "plan_policies": policy_sweep(dev, flush)}
    print(json.dumps(res), flush=True)
    return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama7b", choices=sorted(DESCR))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="chunk-size / tile-quantisation sweep (own JSON line)")
    ap.add_argument("--serve", action="store_true", help="multi-step loop over arrival traces (own JSON line)")
    ap.add_argument("--qkv", action="store_true", help="QKV projection GEMM, fused vs separate (own JSON line)")
    ap.add_argument("--sweep-once", action="store_true",
                    help="with --sweep: one launch per chunk step and nothing else (for ncu traffic captures)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    if args.sweep:
        run_sweep(args)
        return
    if args.serve:
        run_serve(args)
        return
    if args.qkv:
        run_qkv(args)
        return
    res = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world, local_rank)
    if res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
