"""GPU parity: the CUDA step (through the C ABI) against the oracle on the same
seeded inputs.  KV pages must match bit for bit (bf16 of the fp64 RoPE);
outputs within max-abs 2e-2 and mean-abs 2e-3 of the fp64 oracle."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_helpers import GpuStep, assert_close, from_u16, to_u16

pytestmark = pytest.mark.gpu


def _check_step(gs: GpuStep, rows="all", n_random=256):
    err = gs.run()
    assert err == 0, f"device error {err}, header {gs.last_header[:12].tolist()}"
    kc, vc = gs.oracle_caches()
    assert np.array_equal(to_u16(gs.kc_dev), kc), "K pages differ from the oracle"
    assert np.array_equal(to_u16(gs.vc_dev), vc), "V pages differ from the oracle"
    outd = oracle.bf16_to_double(to_u16(gs.out))
    if rows == "all":
        ref, rt, rh = gs.oracle_rows(kc, vc)
    else:
        rt, rh = gs.sample_rows(n_random)
        ref, rt, rh = gs.oracle_rows(kc, vc, rt, rh)
    return assert_close(outd[rt, rh], ref, gs.wl.name)


def test_tiny_single_step():
    _check_step(GpuStep(W.tiny(0)))


def test_mistral_budget_512_all_rows():
    _check_step(GpuStep(W.mistral()))


@pytest.mark.parametrize("policy", [(1, 256, 48, 32), (0, 512, 0, 32)], ids=["decode_maximal", "aligned"])
def test_mistral_request_set_under_other_plan_policies(policy):
    """The same requests planned by decode-maximal batching (one 256-token
    chunk, at most 47 decodes) and by the stall-free rule with 32-aligned
    chunks: the kernel follows whatever metadata the plan emits."""
    gs = GpuStep(W.mistral(), policy=policy)
    m = gs.meta
    if policy[0] == 1:
        assert m["num_decodes"] == 47 and list(m["num_new"][47:]) == [256]
    else:
        assert list(m["num_new"][80:]) == [300, 128]
    _check_step(gs)


@pytest.mark.parametrize("make", [lambda: W.tiny(1), W.mistral, W.llama70b], ids=["tiny", "mistral", "llama70b"])
def test_interleaved_rope_option(make):
    """The interleaved RoPE pairing (x[2j], x[2j+1]): appended pages bit-exact
    and outputs within tolerance of the oracle's interleaved step."""
    wl = make()
    gs = GpuStep(wl, rope_style=1)
    _check_step(gs, rows="all" if wl.name in ("tiny", "mistral") else "sample")


@pytest.mark.parametrize("k", [0, 3, 4])
def test_llama7b_budget_2048_sampled(k):
    _check_step(GpuStep(W.llama7b(chunk_step=k)), rows="sample")


@pytest.mark.parametrize("chunk", [128, 512])
def test_llama7b_last_prefill_chunk_sampled(chunk):
    """The last chunk of an 8192-token prompt alone in the step (its items
    fill fewer than half the SMs); sampled rows against the oracle."""
    _check_step(GpuStep(W.llama7b_prefill_only(chunk, 8192 // chunk - 1)), rows="sample")


@pytest.mark.parametrize("seed", range(6))
def test_random_request_sets_sampled(seed):
    """Random mixed batches: a GQA shape, 0-48 decodes with contexts 0-3000,
    0-4 prefill chunks (running with a random history, or waiting), a random
    budget and scattered pages; sampled rows and the pages against the
    oracle."""
    rng = np.random.default_rng(1234 + seed)
    H_q, H_kv, d = [(32, 8, 128), (8, 1, 64), (28, 4, 128), (16, 16, 64), (64, 8, 128), (12, 2, 128)][seed]
    specs = []
    for _ in range(int(rng.integers(0, 49))):
        c = int(rng.integers(0, 3001))
        specs.append((W.DECODE, 0, c, c + 1))
    for _ in range(int(rng.integers(0 if specs else 1, 5))):
        if rng.random() < 0.5:
            h = int(rng.integers(1, 4000))
            pl = h + int(rng.integers(1, 900))
            specs.append((W.PREFILL_RUNNING, pl, h, pl))
        else:
            pl = int(rng.integers(1, 1200))
            specs.append((W.PREFILL_WAITING, pl, 0, pl))
    order = rng.permutation(len(specs))
    specs = [specs[i] for i in order]
    budget = int(rng.integers(len([x for x in specs if x[0] == W.DECODE]) + 1, 2600))
    _check_step(GpuStep(_custom(W.Shape(H_q, H_kv, d), specs, budget, seed=seed, name=f"random{seed}")),
                rows="sample")


@pytest.mark.parametrize("make,num_sms", [(W.mistral, 1), (W.mistral, 7), (W.llama70b, 400)],
                         ids=["mistral-1", "mistral-7", "llama70b-400"])
def test_work_queues_planned_for_another_sm_count(make, num_sms):
    """A plan sized for another SM count than the device's: with 1 SM every
    CTA starts on the second queue (APPEND items and decodes) and moves to the
    tiles; with 400 the planner's partition (221 CTAs) exceeds the grid and the
    launcher keeps one CTA on the second queue.  The step ends without a
    device error and matches the oracle."""
    import torch
    from chunked_prefill_mixed_gb300.runner import StepRunner
    wl = make()
    sh = wl.shape
    st, meta = oracle.plan(*wl.arrays(), wl.budget, sh.page_size)
    max_pos = int(((np.diff(meta["kv_page_indptr"]) - 1) * 16 + meta["kv_last_page_len"]).max()) + 16
    runner = StepRunner(sh.H_q, sh.H_kv, sh.d, max_pos, device="cuda", rope_theta=sh.rope_base)
    runner.num_sms = num_sms
    gs = GpuStep(wl, runner=runner)
    assert 0 < gs.info.n_first < gs.info.n_items
    if num_sms == 400:
        assert gs.info.first_sms >= torch.cuda.get_device_properties(0).multi_processor_count
    _check_step(gs, rows="sample")


def _plan_with_pieces(wl, sh, want_split):
    """The first SM count for which the planner cuts some tiles of the step
    into want_split key pieces."""
    import chunked_prefill_mixed_gb300 as S
    reqs, keep = S.make_requests(*wl.arrays())
    shp = S.Shape(sh.H_q, sh.H_kv, sh.d, 16)
    for nsm in range(2, 152):
        st, info, packed = S.sarathi_plan(reqs, len(wl.requests), wl.budget, shp, nsm)
        items = packed[info.off_items:info.off_items + info.n_items * 24].reshape(-1, 24)
        if want_split in set(items[(items[:, 0] == 1), 7].tolist()):
            return nsm
    return None


@pytest.mark.parametrize("H_q,H_kv,d,hist,chunk,nsplit", [
    (32, 8, 128, 2300, 300, 3), (56, 8, 128, 2300, 300, 4), (32, 32, 128, 2300, 300, 3), (8, 1, 64, 4300, 400, 3),
    (7, 1, 128, 2300, 300, 2), (7, 1, 128, 2300, 300, 4)])
def test_key_pieces_of_split_tiles_all_rows(H_q, H_kv, d, hist, chunk, nsplit):
    """A chunk after thousands of tokens of history, alone in the step, so
    every tile runs ~20-40 key blocks: planned for a small SM count the last
    tiles come as 2-4 key pieces that write fp32 partials and are merged by
    the last piece to finish (odd groups place their partials on an even
    slot; d = 64 and 128).  Every output row matches the oracle and the pages
    match bit for bit."""
    from chunked_prefill_mixed_gb300.runner import StepRunner
    sh = W.Shape(H_q, H_kv, d)
    L = hist + chunk
    wl = _custom(sh, [(W.PREFILL_RUNNING, L, hist, L)], chunk, name=f"pieces{H_q}x{H_kv}x{d}")
    num_sms = _plan_with_pieces(wl, sh, nsplit)
    assert num_sms is not None, f"no SM count gives {nsplit} pieces"
    runner = StepRunner(sh.H_q, sh.H_kv, sh.d, L + 16, device="cuda", rope_theta=sh.rope_base)
    runner.num_sms = num_sms
    gs = GpuStep(wl, runner=runner)
    items = gs.packed[gs.info.off_items:gs.info.off_items + gs.info.n_items * 24].reshape(-1, 24)
    assert nsplit in set(items[(items[:, 0] == 1), 7].tolist())
    _check_step(gs)
    # whichever piece of a tile finishes last merges, in piece order: the
    # bits do not depend on the arrival order, which varies launch to launch
    first = to_u16(gs.out).copy()
    for _ in range(3):
        gs.out.fill_(float("nan"))
        assert gs.run() == 0
        assert np.array_equal(to_u16(gs.out), first)


def _plan_where(wl, sh, pred):
    """The first SM count whose plan of the step satisfies pred(info, items)."""
    import chunked_prefill_mixed_gb300 as S
    reqs, keep = S.make_requests(*wl.arrays())
    shp = S.Shape(sh.H_q, sh.H_kv, sh.d, 16)
    for nsm in range(2, 153):
        st, info, packed = S.sarathi_plan(reqs, len(wl.requests), wl.budget, shp, nsm)
        items = packed[info.off_items:info.off_items + info.n_items * 24].reshape(-1, 24)
        if pred(info, items):
            return nsm
    return None


@pytest.mark.parametrize("H_q,H_kv,d,hist,chunk", [
    (32, 8, 128, 4000, 300), (8, 1, 64, 6000, 500), (7, 1, 128, 4000, 300), (32, 32, 128, 3000, 300),
    (56, 8, 128, 3840, 256)])
def test_appends_on_a_second_queue_beside_the_tiles(H_q, H_kv, d, hist, chunk):
    """A chunk after thousands of tokens of history, alone in the step, planned
    for an SM count where the APPEND items make up a second queue that a few
    CTAs start on while the others take the tiles (which wait at the chunk's
    blocks for the ready flags).  Every output row matches the oracle and the
    pages match bit for bit."""
    from chunked_prefill_mixed_gb300.runner import StepRunner
    sh = W.Shape(H_q, H_kv, d)
    L = hist + chunk
    wl = _custom(sh, [(W.PREFILL_RUNNING, L, hist, L)], chunk, name=f"appq{H_q}x{H_kv}x{d}")

    def second_queue(info, items):
        return info.n_first < info.n_items and (items[info.n_first:, 0] == 0).all()
    num_sms = _plan_where(wl, sh, second_queue)
    assert num_sms is not None, "no SM count gives that layout"
    runner = StepRunner(sh.H_q, sh.H_kv, sh.d, L + 16, device="cuda", rope_theta=sh.rope_base)
    runner.num_sms = num_sms
    gs = GpuStep(wl, runner=runner)
    items = gs.packed[gs.info.off_items:gs.info.off_items + gs.info.n_items * 24].reshape(-1, 24)
    assert second_queue(gs.info, items)
    _check_step(gs)


def test_llama70b_budget_1536_sampled():
    _check_step(GpuStep(W.llama70b()), rows="sample")


def test_yi34b_fragmented_sampled():
    _check_step(GpuStep(W.yi34b()), rows="sample")


def _custom(shape, specs, budget, seed=5, permute=True, name="custom"):
    return W._build(name, shape, budget, specs, seed, permute=permute, spare_pages=3)


@pytest.mark.parametrize("H_q,H_kv,d", [(8, 2, 64), (7, 1, 128), (16, 1, 64), (4, 4, 128), (8, 1, 128)])
def test_edge_shapes_ragged_chunks(H_q, H_kv, d):
    shape = W.Shape(H_q, H_kv, d)
    specs = [
        (W.DECODE, 0, 0, 1),        # first decode token: attends only to itself
        (W.DECODE, 0, 15, 16),      # fills a page exactly (last page length 16)
        (W.DECODE, 0, 16, 17),      # opens a new page (last page length 1)
        (W.DECODE, 0, 333, 334),
        (W.PREFILL_RUNNING, 40, 39, 40),     # chunk of one token after history
        (W.PREFILL_RUNNING, 100, 31, 100),   # ragged history, chunk 69
        (W.PREFILL_RUNNING, 64, 16, 64),     # history an exact page multiple
        (W.PREFILL_WAITING, 17, 0, 17),
        (W.PREFILL_WAITING, 300, 0, 300),    # takes what is left (several tiles, ragged tail)
    ]
    _check_step(GpuStep(_custom(shape, specs, budget=400)))


def test_repeat_launch_is_deterministic_and_leaves_workspace_clean():
    import torch
    gs = GpuStep(W.mistral())
    k0, v0 = gs.kc_dev.clone(), gs.vc_dev.clone()
    assert gs.run() == 0
    out1, k1 = gs.out.clone(), gs.kc_dev.clone()
    gs.kc_dev.copy_(k0)
    gs.vc_dev.copy_(v0)
    gs.out.fill_(float("nan"))
    assert gs.run() == 0
    assert np.array_equal(to_u16(gs.out), to_u16(out1))
    assert np.array_equal(to_u16(gs.kc_dev), to_u16(k1))
    hdr = gs.runner.workspace[:64].view(torch.int32).cpu().numpy()
    assert np.all(hdr[:3] == 0)


def test_plan_copied_inside_the_step_call_gives_the_same_bits():
    """StepRunner.run_planned: the packed plan goes from the runner's pinned
    buffer to the device inside sarathi_mixed_attn (args.plan_host); the step
    equals the one launched with a plan already on the device."""
    import torch
    gs = GpuStep(W.mistral())
    k0, v0 = gs.kc_dev.clone(), gs.vc_dev.clone()
    assert gs.run() == 0
    out1, k1 = gs.out.clone(), gs.kc_dev.clone()
    gs.kc_dev.copy_(k0)
    gs.vc_dev.copy_(v0)
    gs.out.fill_(float("nan"))
    r = gs.runner
    st, info, packed = r.plan(*gs.wl.arrays(), gs.wl.budget)
    r.run_planned(gs.q_dev, gs.k_dev, gs.v_dev, gs.kc_dev, gs.vc_dev, gs.out, info)
    torch.cuda.synchronize()
    assert r.status() == 0
    assert np.array_equal(to_u16(gs.out), to_u16(out1))
    assert np.array_equal(to_u16(gs.kc_dev), to_u16(k1))


def test_tiny_chunked_schedule_equals_one_shot_and_oracle():
    """The 200-token prompt in chunks of 64 over 4 steps next to 2 decodes, then
    the same prompt in one shot: same KV pages, outputs within tolerance, and
    every step matches the oracle."""
    import torch
    from chunked_prefill_mixed_gb300.runner import StepRunner
    shape = W.SHAPES["tiny"]
    L = 200
    pq, pk, pv = W.new_token_values(L, shape, 100)
    wl0 = W.tiny(0)
    kc_h, vc_h = W.history_cache_numpy(wl0.num_pages, shape, 0)
    dev = torch.device("cuda")
    kc, vc = from_u16(kc_h, dev), from_u16(vc_h, dev)
    okc, ovc = kc_h.copy(), vc_h.copy()
    runner = StepRunner(shape.H_q, shape.H_kv, shape.d, 256, device=dev)
    prompt_out = np.zeros((L, shape.H_q, shape.d))
    done = 0
    for s in range(4):
        wl = W.tiny(s)
        st, meta = oracle.plan(*wl.arrays(), wl.budget, 16)
        n = int(meta["num_new"][2])
        dq, dk, dv = W.new_token_values(2, shape, 200 + s)
        q = np.concatenate([dq, pq[done:done + n]])
        k = np.concatenate([dk, pk[done:done + n]])
        v = np.concatenate([dv, pv[done:done + n]])
        status, info, packed = runner.plan(*wl.arrays(), wl.budget)
        out = torch.empty((2 + n, shape.H_q, shape.d), dtype=torch.bfloat16, device=dev)
        runner.run(from_u16(q, dev), from_u16(k, dev), from_u16(v, dev), kc, vc, out, runner.upload(packed), info)
        assert runner.status() == 0
        oo = oracle.step(meta, q, k, v, shape.H_q, shape.H_kv, shape.d, 16, shape.rope_base, okc, ovc)
        assert np.array_equal(to_u16(kc), okc) and np.array_equal(to_u16(vc), ovc)
        assert_close(oracle.bf16_to_double(to_u16(out)), oo, f"tiny step {s}")
        prompt_out[done:done + n] = oracle.bf16_to_double(to_u16(out))[2:]
        done += n
    assert done == L
    # one shot: the same prompt into a fresh copy of the history pools
    table = wl0.requests[2].pages
    wl1 = W._build("tiny_oneshot", shape, L, [(W.PREFILL_WAITING, L, 0, L)], 0)
    wl1.requests[0].pages = table
    kc2, vc2 = from_u16(kc_h, dev), from_u16(vc_h, dev)
    status, info, packed = runner.plan(*wl1.arrays(), L)
    out = torch.empty((L, shape.H_q, shape.d), dtype=torch.bfloat16, device=dev)
    runner.run(from_u16(pq, dev), from_u16(pk, dev), from_u16(pv, dev), kc2, vc2, out, runner.upload(packed), info)
    assert runner.status() == 0
    ptab = table[: (L + 15) // 16]
    assert np.array_equal(to_u16(kc2)[ptab], to_u16(kc)[ptab])
    assert np.array_equal(to_u16(vc2)[ptab], to_u16(vc)[ptab])
    diff = np.abs(oracle.bf16_to_double(to_u16(out)) - prompt_out)
    assert diff.max() <= 2e-2


@pytest.mark.parametrize("chunk", [512, 1024, 2048])
def test_llama7b_prefill_chunk_sweep_against_oracle_and_one_shot(chunk):
    """The 8192-token prompt prefilled alone in chunks of 512, 1024 and 2048
    tokens ("Sarathi-Serve 完全拆解", §"先验证数值与状态正确性": chunked prefill
    must equal one-shot prefill, checked at the long-context boundaries).
    After every chunk step the whole page pool equals the oracle's, bit for
    bit; every step's sampled rows (the chunk's first, second, middle and last
    two rows over all heads, plus random pairs) match the oracle; the final
    pages equal the one-shot step's, and each chunk's outputs agree with the
    one-shot outputs of the same rows."""
    import torch
    L = 8192
    one = GpuStep(W.llama7b_prefill_only(L, 0))
    assert one.run() == 0
    sh = one.wl.shape
    pages = one.wl.requests[0].pages
    kc_one, vc_one = one.oracle_caches()
    assert np.array_equal(to_u16(one.kc_dev), kc_one) and np.array_equal(to_u16(one.vc_dev), vc_one)
    rt = np.array([0, 1, 511, 512, 513, 4095, 4096, 8190, 8191], np.int32)
    rh = np.array([0, 31, 5, 17, 3, 9, 30, 2, 31], np.int32)
    ref, _, _ = one.oracle_rows(kc_one, vc_one, rt, rh)
    assert_close(oracle.bf16_to_double(to_u16(one.out))[rt, rh], ref, "one-shot 8192")

    dev = one.dev
    runner = one.runner
    kc, vc = from_u16(one.kc0, dev), from_u16(one.vc0, dev)
    okc, ovc = one.kc0.copy(), one.vc0.copy()
    rng = np.random.default_rng(chunk)
    done, step = 0, 0
    while done < L:
        wl = W.llama7b_prefill_only(chunk, step)
        st_o, meta = oracle.plan(*wl.arrays(), wl.budget, 16)
        st, info, packed = runner.plan(*wl.arrays(), wl.budget)
        n = info.num_tokens
        assert n == meta["num_tokens"] == min(chunk, L - done)
        out = torch.full((n, sh.H_q, sh.d), float("nan"), dtype=torch.bfloat16, device=dev)
        runner.run(one.q_dev[done:done + n], one.k_dev[done:done + n], one.v_dev[done:done + n],
                   kc, vc, out, runner.upload(packed.copy()), info)
        torch.cuda.synchronize()
        assert runner.status() == 0, f"chunk {chunk} step {step}: device error"
        q, k, v = one.q[done:done + n], one.k[done:done + n], one.v[done:done + n]
        oracle.append(meta, k, v, sh.H_kv, sh.d, 16, sh.rope_base, okc, ovc)
        assert np.array_equal(to_u16(kc), okc), f"chunk {chunk} step {step}: K pages differ from the oracle"
        assert np.array_equal(to_u16(vc), ovc), f"chunk {chunk} step {step}: V pages differ from the oracle"
        local = sorted({0, 1, n // 2, n - 2, n - 1})
        st_rows = [(t, hq) for t in local for hq in range(sh.H_q)]
        st_rows += [(int(rng.integers(0, n)), int(rng.integers(0, sh.H_q))) for _ in range(64)]
        st_rows = sorted(set(st_rows))
        srt = np.array([r[0] for r in st_rows], np.int32)
        srh = np.array([r[1] for r in st_rows], np.int32)
        sref, _, _, _ = oracle.attend(meta, q, sh.H_q, sh.H_kv, sh.d, 16, sh.rope_base, okc, ovc, srt, srh)
        got = oracle.bf16_to_double(to_u16(out))
        assert_close(got[srt, srh], sref, f"chunk {chunk} step {step}")
        diff = (out.float() - one.out[done:done + n].float()).abs()
        assert float(diff.max()) <= 2e-2, f"chunk {chunk} step {step}: differs from the one-shot outputs"
        done += n
        step += 1
    assert np.array_equal(to_u16(kc)[pages], to_u16(one.kc_dev)[pages])
    assert np.array_equal(to_u16(vc)[pages], to_u16(one.vc_dev)[pages])


def test_repeated_launches_with_long_prefill_tiles():
    """Several launches in a row of a step whose prefill tiles run ~100 key
    blocks (the softmax warps can then run a block ahead of the MMA issuer):
    every launch ends without a device error and gives the same bits."""
    gs = GpuStep(W.llama70b())
    k0, v0 = gs.kc_dev.clone(), gs.vc_dev.clone()
    outs = []
    for _ in range(4):
        gs.kc_dev.copy_(k0)
        gs.vc_dev.copy_(v0)
        err = gs.run()
        assert err == 0, f"device error {err}, header {gs.last_header[:12].tolist()}"
        outs.append(to_u16(gs.out))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_host_buffer_steps_on_two_streams_give_the_same_bits():
    """StepRunner.run_host (sarathi_mixed_attn_host): four steps from pinned
    host buffers, alternating two streams with their own device buffers,
    each waiting for the step before it; every step's host output and the
    pages equal the step launched from device buffers."""
    import torch
    gs = GpuStep(W.mistral())
    k0, v0 = gs.kc_dev.clone(), gs.vc_dev.clone()
    assert gs.run() == 0
    out1, k1, v1 = to_u16(gs.out), to_u16(gs.kc_dev), to_u16(gs.vc_dev)
    gs.kc_dev.copy_(k0)
    gs.vc_dev.copy_(v0)
    torch.cuda.synchronize()
    r = gs.runner
    pin = lambda t: t.cpu().pin_memory()
    q_h, k_h, v_h = pin(gs.q_dev), pin(gs.k_dev), pin(gs.v_dev)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    dq = [[torch.empty_like(x) for x in (gs.q_dev, gs.k_dev, gs.v_dev, gs.out)] for _ in range(2)]
    out_hs = [torch.full(gs.out.shape, float("nan"), dtype=gs.out.dtype).pin_memory() for _ in range(2)]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    results = []
    for i in range(4):
        b = i & 1
        if i >= 2:
            streams[b].synchronize()
            results.append(to_u16(out_hs[b]).copy())
            out_hs[b].fill_(float("nan"))
        st, info, packed = r.plan(*gs.wl.arrays(), gs.wl.budget)
        q, k, v, out = dq[b]
        r.run_host(q_h, k_h, v_h, out_hs[b], q, k, v, gs.kc_dev, gs.vc_dev, out, info, stream=streams[b],
                   wait_event=done[b ^ 1] if i else None, done_event=done[b])
    torch.cuda.synchronize()
    results += [to_u16(out_hs[0]), to_u16(out_hs[1])]
    assert r.status() == 0
    for res in results:
        assert np.array_equal(res, out1)
    assert np.array_equal(to_u16(gs.kc_dev), k1) and np.array_equal(to_u16(gs.vc_dev), v1)


def test_host_buffer_step_with_an_empty_batch_records_its_event():
    """An empty step (no items) copies and runs nothing but still records its
    done event after the event it waits for."""
    import ctypes
    import torch
    import chunked_prefill_mixed_gb300 as S
    s = torch.cuda.Stream()
    before, done = torch.cuda.Event(), torch.cuda.Event()
    with torch.cuda.stream(s):
        torch.cuda._sleep(1000)
    before.record(s)
    info = S.PlanInfo()
    a = S.AttnArgs()
    a.info = ctypes.pointer(info)
    a.shape = S.Shape(32, 8, 128, 16)
    buf = torch.empty(16, dtype=torch.int16).pin_memory()
    io = S.HostIO(buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), S._event_ptr(before, s),
                  S._event_ptr(done, s))
    other = torch.cuda.Stream()
    assert S.load().sarathi_mixed_attn_host(ctypes.byref(a), ctypes.byref(io), other.cuda_stream) == S.OK
    other.synchronize()
    assert done.query() and before.query()
