"""Failure detection on the GPU without faulting it.

Every wait in the step kernel gives up after a bounded time and page ids are
checked before they are used; both end in an error word the host reads back.
These tests feed metadata that the kernel's own checks must catch and then
check that the same context still runs a correct step."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_helpers import GpuStep, assert_close, to_u16

pytestmark = pytest.mark.gpu


def _fresh_run_is_correct(gs):
    gs.runner.workspace.zero_()
    gs.plan_dev = gs.runner.upload(gs.packed)
    gs.kc_dev.copy_(gs._k0)
    gs.vc_dev.copy_(gs._v0)
    assert gs.run() == 0
    kc, vc = gs.oracle_caches()
    assert np.array_equal(to_u16(gs.kc_dev), kc)
    ref, rt, rh = gs.oracle_rows(kc, vc)
    assert_close(oracle.bf16_to_double(to_u16(gs.out))[rt, rh], ref, "after recovery")


def _small_mixed():
    shape = W.Shape(8, 2, 64)
    specs = [(W.DECODE, 0, 40, 41), (W.DECODE, 0, 70, 71), (W.PREFILL_RUNNING, 200, 64, 200)]
    return W._build("fail", shape, 100, specs, 9, spare_pages=2)


def test_wait_that_runs_out_is_reported_and_context_stays_usable():
    gs = GpuStep(_small_mixed())
    gs._k0, gs._v0 = gs.kc_dev.clone(), gs.vc_dev.clone()
    bad = gs.packed.copy()
    s = gs.meta["n_sched"] - 1                     # the prefill row
    # the row's two APPEND items (positions 64-127 and 128-199): the first is
    # replaced by a copy of the second, so the first block's ready flag is
    # never set and the tiles' wait for it runs out
    items = bad[gs.info.off_items:gs.info.off_items + gs.info.n_items * 24].reshape(-1, 24)
    app = [i for i in range(len(items)) if items[i, 0] == 0 and items[i, 1] == s]
    assert len(app) == 2 and items[app[0], 3] < items[app[1], 3]
    items[app[0]] = items[app[1]]
    gs.plan_dev = gs.runner.upload(bad)
    err = gs.run()
    assert err == 1, f"expected a bounded-wait error, got {err}"
    assert gs.last_header[3] == -1 - s
    _fresh_run_is_correct(gs)


def test_page_id_outside_the_pool_is_reported_not_written():
    gs = GpuStep(_small_mixed())
    gs._k0, gs._v0 = gs.kc_dev.clone(), gs.vc_dev.clone()
    bad = gs.packed.copy()
    # last page of the first decode: its K/V append would land there
    p = gs.info.off_kv_page_indices + gs.meta["kv_page_indptr"][1] - 1
    bad[p] = gs.wl.num_pages + 5
    gs.plan_dev = gs.runner.upload(bad)
    err = gs.run()
    assert err == 2, f"expected a bounds error, got {err}"
    assert gs.last_header[3] == gs.wl.num_pages + 5
    # nothing outside the pool was written, and the pool itself is intact
    # apart from the other rows' appends
    _fresh_run_is_correct(gs)
