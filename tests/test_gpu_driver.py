"""The multi-step loop (plan -> step -> advance over an arrival trace) on the
GPU against the oracle run step by step on the same trace: every iteration's
plan is bit-identical, the outputs agree within tolerance, the request states
advance alike, and the page pools end bit-identical."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_helpers import assert_close, to_u16

pytestmark = pytest.mark.gpu


def _trace():
    return [W.Arrival(0, 70, 4), W.Arrival(0, 23, 3), W.Arrival(1, 150, 5), W.Arrival(3, 9, 2),
            W.Arrival(5, 64, 6), W.Arrival(6, 130, 3)]


@pytest.mark.parametrize("policy", [None, (1, 48, 4, 1)], ids=["stall_free_64", "decode_maximal"])
def test_multi_step_loop_matches_oracle(policy):
    import torch
    import chunked_prefill_mixed_gb300 as S
    from chunked_prefill_mixed_gb300.driver import MultiStepDriver
    from chunked_prefill_mixed_gb300.runner import StepRunner
    sh = W.SHAPES["tiny"]
    dev = torch.device("cuda")
    num_pages = 64
    dims = (num_pages, sh.H_kv, sh.page_size, sh.d)
    kc = torch.zeros(dims, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros(dims, dtype=torch.bfloat16, device=dev)
    okc, ovc = np.zeros(dims, np.uint16), np.zeros(dims, np.uint16)
    runner = StepRunner(sh.H_q, sh.H_kv, sh.d, 512, device=dev, rope_theta=sh.rope_base)
    pol = S.PlanPolicy(*policy) if policy else None
    drv = MultiStepDriver(runner, kc, vc, num_pages, _trace(), lambda it, T: W.new_token_values(T, sh, 1000 + it),
                          budget=64, policy=pol)
    steps = 0
    while not drv.finished() and steps < 200:
        rec = drv.step(keep=True)
        steps += 1
        if rec.plan is None:
            continue
        p = rec.plan
        if policy is None:
            st, om = oracle.plan(p["states"], p["prompt"], p["computed"], p["tables"], 64, 16)
        else:
            st, om = oracle.plan(p["states"], p["prompt"], p["computed"], p["tables"], policy[1], 16,
                                 policy=policy[0], max_batch=policy[2], align=policy[3])
        for key in ("req_index", "num_new", "last_chunk", "qo_indptr", "kv_page_indptr", "kv_page_indices",
                    "kv_last_page_len"):
            assert np.array_equal(np.asarray(om[key]), np.asarray(p["meta"][key])), (rec.iteration, key)
        oo = oracle.step(om, p["q"], p["k"], p["v"], sh.H_q, sh.H_kv, sh.d, 16, sh.rope_base, okc, ovc)
        assert_close(oracle.bf16_to_double(to_u16(p["out"])), oo, f"iteration {rec.iteration}")
        st, ostates, ocomp = oracle.advance(p["states"], p["prompt"], p["computed"], om)
        assert st == oracle.OK
        assert ostates == p["after_states"] and ocomp == p["after_computed"], rec.iteration
    assert drv.finished(), "the trace did not drain"
    assert len(drv.done) == len(_trace())
    assert np.array_equal(to_u16(kc), okc) and np.array_equal(to_u16(vc), ovc)
