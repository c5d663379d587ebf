"""The step entry point for callers that cannot allocate device memory.

Some callers -- a plugin inside a process whose allocator already owns the
GPU's memory, or a serving loop that forbids allocation after start-up --
cannot provide a workspace.  sarathi_mixed_attn_noalloc runs the same step with
the library's own fixed scratch array.  These tests check that it gives the
same pages and outputs as the workspace entry point, on two calls in a row (the
array keeps the previous call's contents), and that batches needing more
scratch than the array holds are refused.  The file is named so that pytest
collects it last."""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as W
import chunked_prefill_mixed_gb300 as S


def test_noalloc_refuses_batches_beyond_the_scratch_limit():
    info = S.PlanInfo()
    info.n_items = 1
    info.workspace_bytes = (8 << 20) + 256
    a = S.AttnArgs()
    a.info = ctypes.pointer(info)
    st = S.load().sarathi_mixed_attn_noalloc(ctypes.byref(a), None)
    assert st == S.ERR_CAPACITY
    assert "scratch" in S.sarathi_last_error()


def test_noalloc_refuses_inconsistent_plan_info_before_any_cuda_call():
    """A plan info whose counters (n_sched, n_merge) would not fit the
    workspace it states is refused before anything is enqueued, so the
    clearing of the array can never run past its end."""
    for n_sched, n_merge, n_partials in ((1 << 28, 0, 0), (4, 1 << 27, 0), (4, 0, 1 << 20), (0, 0, 0)):
        info = S.PlanInfo()
        info.n_items = 1
        info.n_sched = n_sched
        info.n_merge = n_merge
        info.n_partials = n_partials
        info.workspace_bytes = 1024
        a = S.AttnArgs()
        a.info = ctypes.pointer(info)
        a.shape = S.Shape(32, 8, 128, 16)
        st = S.load().sarathi_mixed_attn_noalloc(ctypes.byref(a), None)
        assert st == S.ERR_INVALID_ARG, (n_sched, n_merge, n_partials, st)
        assert "inconsistent plan info" in S.sarathi_last_error()


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import torch
    from gpu_helpers import GpuStep, assert_close, to_u16
    # a few very long decodes are split across CTAs, so the scratch holds merge
    # tickets and partial results; the prefill chunk uses the append counters
    shape = W.SHAPES["mistral"]
    specs = [(W.DECODE, 0, 12000 + 37 * i, 12001 + 37 * i) for i in range(6)]
    specs.append((W.PREFILL_RUNNING, 900, 700, 900))
    gs = GpuStep(W._build("noalloc", shape, 256, specs, 7))
    assert gs.info.n_partials > 0 and gs.info.workspace_bytes <= (8 << 20)
    k0, v0 = gs.kc_dev.clone(), gs.vc_dev.clone()
    assert gs.run() == 0
    ref_out = oracle.bf16_to_double(to_u16(gs.out))
    ref_k, ref_v = to_u16(gs.kc_dev), to_u16(gs.vc_dev)
    r = gs.runner
    for call in range(2):
        gs.kc_dev.copy_(k0)
        gs.vc_dev.copy_(v0)
        out = torch.full_like(gs.out, float("nan"))
        S.sarathi_mixed_attn_noalloc(gs.q_dev, gs.k_dev, gs.v_dev, gs.kc_dev, gs.vc_dev, out, gs.plan_dev, gs.info,
                                     r.rope, r.max_pos, r.shape, r.sm_scale, r.stream)
        torch.cuda.synchronize()
        assert np.array_equal(to_u16(gs.kc_dev), ref_k), f"call {call}: K pages differ"
        assert np.array_equal(to_u16(gs.vc_dev), ref_v), f"call {call}: V pages differ"
        assert_close(oracle.bf16_to_double(to_u16(out)), ref_out, f"no-alloc call {call}")


@pytest.mark.gpu
def test_noalloc_error_word_is_reported_and_the_next_call_is_clean():
    """A bounded wait that runs out inside a no-allocation step sets the error
    word of the built-in array; sarathi_noalloc_status reports it (and clears
    it), and the next call on a correct plan gives the oracle's pages and
    outputs.  The failure is made in the metadata (a row's first APPEND item
    replaced by a copy of its second, so the first block's ready flag is never
    set), as in the workspace entry point's failure test."""
    import torch
    from gpu_helpers import GpuStep, assert_close, to_u16
    shape = W.Shape(8, 2, 64)
    specs = [(W.DECODE, 0, 40, 41), (W.DECODE, 0, 70, 71), (W.PREFILL_RUNNING, 200, 64, 200)]
    gs = GpuStep(W._build("noalloc_fail", shape, 100, specs, 9, spare_pages=2))
    k0, v0 = gs.kc_dev.clone(), gs.vc_dev.clone()
    r = gs.runner
    bad = gs.packed.copy()
    s = gs.meta["n_sched"] - 1
    items = bad[gs.info.off_items:gs.info.off_items + gs.info.n_items * 24].reshape(-1, 24)
    app = [i for i in range(len(items)) if items[i, 0] == 0 and items[i, 1] == s]
    assert len(app) >= 2 and items[app[0], 3] < items[app[-1], 3]
    items[app[0]] = items[app[-1]]
    out = torch.full_like(gs.out, float("nan"))
    plan_bad = r.upload(bad)  # (the runner's stream waits for the work above)
    S.sarathi_mixed_attn_noalloc(gs.q_dev, gs.k_dev, gs.v_dev, gs.kc_dev, gs.vc_dev, out, plan_bad, gs.info,
                                 r.rope, r.max_pos, r.shape, r.sm_scale, r.stream)
    assert S.sarathi_noalloc_status(r.stream) == 1
    assert S.sarathi_noalloc_status(r.stream) == 0   # read once, then cleared
    gs.kc_dev.copy_(k0)
    gs.vc_dev.copy_(v0)
    out = torch.full_like(gs.out, float("nan"))
    plan_ok = r.upload(gs.packed)
    S.sarathi_mixed_attn_noalloc(gs.q_dev, gs.k_dev, gs.v_dev, gs.kc_dev, gs.vc_dev, out, plan_ok, gs.info,
                                 r.rope, r.max_pos, r.shape, r.sm_scale, r.stream)
    assert S.sarathi_noalloc_status(r.stream) == 0
    kc, vc = gs.oracle_caches()
    assert np.array_equal(to_u16(gs.kc_dev), kc) and np.array_equal(to_u16(gs.vc_dev), vc)
    ref, rt, rh = gs.oracle_rows(kc, vc)
    assert_close(oracle.bf16_to_double(to_u16(out))[rt, rh], ref, "no-alloc call after an error")
