"""CPU tests of the library's host side: the C ABI loads and exports every
declared symbol; sarathi_plan's metadata equals the oracle's plan bit for bit;
the kernel work list covers every output row, token and page exactly once."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads as W
import chunked_prefill_mixed_gb300 as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_library_exports_every_declared_function():
    text = open(os.path.join(ROOT, "include", "sarathi.h")).read()
    declared = set(re.findall(r"^\s*(?:int32_t|const char\*)\s+(sarathi_\w+)\s*\(", text, re.M))
    assert declared == set(S.EXPORTED)
    lib = S.load()
    for name in declared:
        assert hasattr(lib, name), name
    assert S.sarathi_abi_version() == S.ABI_VERSION
    for name, value in (("SARATHI_ABI_VERSION", S.ABI_VERSION), ("SARATHI_ITEM_INTS", S.ITEM_INTS)):
        assert re.search(rf"#define {name} {value}\b", text), name


def _product_plan(states, prompt, computed, tables, budget, shape, num_sms=148):
    reqs, keep = S.make_requests(states, prompt, computed, tables)
    st, info, packed = S.sarathi_plan(reqs, len(states), budget, S.Shape(shape.H_q, shape.H_kv, shape.d, 16), num_sms)
    return st, info, S.plan_arrays(info, packed)


def _compare(st_o, mo, st_p, mp):
    assert st_o == st_p
    for key in ("req_index", "num_new", "last_chunk", "qo_indptr", "kv_page_indptr", "kv_page_indices",
                "kv_last_page_len"):
        assert np.array_equal(np.asarray(mo[key]), np.asarray(mp[key])), key
    assert mo["num_decodes"] == mp["num_decodes"] and mo["num_tokens"] == mp["num_tokens"]


def _workload_cases():
    yield W.tiny(0)
    yield W.tiny(3)
    yield W.mistral()
    for k in range(5):
        yield W.llama7b(chunk_step=k)
    yield W.llama70b()
    yield W.yi34b()
    yield W.llama7b_prefill_only(512, 3)


@pytest.mark.parametrize("wl", list(_workload_cases()), ids=lambda w: f"{w.name}-{w.notes}")
def test_plan_matches_oracle_on_workloads(wl):
    st_o, mo = oracle.plan(*wl.arrays(), wl.budget, 16)
    st_p, info, mp = _product_plan(*wl.arrays(), wl.budget, wl.shape)
    _compare(st_o, mo, st_p, mp)
    _check_work_list(info, mp, wl.shape)
    assert info.pairs == oracle.pairs(mo, 16)


def test_plan_matches_oracle_random_request_sets():
    rng = np.random.default_rng(123)
    shape = W.Shape(8, 2, 64)
    for trial in range(60):
        n = int(rng.integers(0, 12))
        states, prompt, computed, tables = [], [], [], []
        for i in range(n):
            stt = int(rng.integers(0, 3))
            if stt == W.DECODE:
                h = int(rng.integers(0, 300))
                pl = 0
                cap = h + 1
            else:
                pl = int(rng.integers(1, 400))
                h = 0 if stt == W.PREFILL_WAITING and rng.random() < 0.7 else int(rng.integers(0, pl + 1))
                cap = pl
            npages = (cap + 15) // 16 + int(rng.integers(0, 3))
            states.append(stt)
            prompt.append(pl)
            computed.append(h)
            tables.append(rng.permutation(5000)[:npages].astype(np.int32))
        budget = int(rng.integers(1, 600))
        st_o, mo = oracle.plan(states, prompt, computed, tables, budget, 16)
        nsm = int(rng.integers(1, 200))
        st_p, info, mp = _product_plan(states, prompt, computed, tables, budget, shape, num_sms=nsm)
        _compare(st_o, mo, st_p, mp)
        _check_work_list(info, mp, shape, nsm)


def _check_work_list(info, m, shape, num_sms=148):
    """Every (row, q head) is produced once; every new token's K/V is appended
    once per kv head; decode splits tile each decode's pages; the first queue
    holds the prefill tiles and the second the decode splits; the appends lead
    the second queue (the first when it holds everything), so a CTA that waits
    on one never holds up the CTAs that take them.  A tile split along its keys
    comes as pieces whose 128-key block ranges tile [0, nblk) in order, with
    partial slots of their own."""
    G = shape.H_q // shape.H_kv
    n = m["n_sched"]
    qo, kvp = m["qo_indptr"], m["kv_page_indptr"]
    items = m["items"]
    T = int(qo[-1]) if n else 0
    covered = np.zeros((T, shape.H_q), np.int32)
    appended = np.zeros((T, shape.H_kv), np.int32)
    seen_slots = set()
    pages_cov = {}
    pieces = {}
    spt = -(-128 // G)
    spt += spt & (G & 1)
    kvi, last = m["kv_page_indices"], m["kv_last_page_len"]
    kinds = items[:, 0] if len(items) else np.zeros(0, np.int32)
    nf = info.n_first
    assert 0 <= nf <= info.n_items == len(items)
    has_dec = bool((kinds == 2).any())
    assert not (kinds[:nf] == 2).any() and not (kinds[nf:] == 1).any()
    # the APPEND items lead the second queue when it holds items, else the first
    app_q = kinds[nf:] if nf < info.n_items else kinds[:nf]
    n_app = int((kinds == 0).sum())
    assert (app_q[:n_app] == 0).all() and not (app_q[n_app:] == 0).any()
    if nf == 0:
        assert info.first_sms == 0
    elif nf == info.n_items:
        assert info.first_sms == num_sms
    else:
        assert 0 <= info.first_sms < num_sms
        # CTAs past the tiles would find the first queue empty at once
        assert info.first_sms <= int((kinds == 1).sum())
    for idx, it in enumerate(items):
        kind, s, g, start, count, slot, merge, nsplit = (int(x) for x in it[:8])
        nn = qo[s + 1] - qo[s]
        np_ = kvp[s + 1] - kvp[s]
        # the row's metadata copied into the item, and the page ids it carries
        assert list(it[8:13]) == [qo[s], nn, kvp[s], np_, 16 * (np_ - 1) + last[s]]
        b0, b1, piece = (int(x) for x in it[13:16])
        if kind != 1 or nsplit == 1:
            assert b0 == b1 == piece == 0
        ids = it[16:24]
        if kind == 0:
            assert not ids.any()
        elif kind == 1:
            p0 = 8 * b0
            k = max(min(8, np_ - p0), 0)
            assert list(ids[:k]) == list(kvi[kvp[s] + p0:kvp[s] + p0 + k]) and not ids[k:].any()
        else:
            k = min(8, count)
            assert list(ids[:k]) == list(kvi[kvp[s] + start:kvp[s] + start + k]) and not ids[k:].any()
        if kind == 0:
            # up to 2 kv heads, tokens whose positions share one 128-position block
            assert nn >= 2 and g % 2 == 0 and 0 < count <= 128
            h = 16 * (np_ - 1) + last[s] - nn
            assert (h + start) // 128 == (h + start + count - 1) // 128
            appended[qo[s] + start: qo[s] + start + count, g:g + 2] += 1
        elif kind == 1:
            # one Q tile of up to 128 // G tokens, starting on a tile boundary
            tpi = 128 // G
            assert 0 < count <= tpi and start % tpi == 0 and start + count <= nn
            if nsplit > 1:
                h = 16 * (np_ - 1) + last[s] - nn
                nblk = -(-(h + start + count) // 128)
                assert 2 <= nsplit <= 4 and 0 <= b0 < b1 <= nblk and 0 <= piece < nsplit
                assert 0 <= merge < info.n_merge and slot >= 0 and (slot % 2 == 0 or G % 2 == 0)
                pieces.setdefault((slot, merge), []).append((piece, b0, b1, nblk, nsplit, s, g, start))
                for q in range(spt):
                    assert slot + piece * spt + q not in seen_slots
                    seen_slots.add(slot + piece * spt + q)
                if piece != 0:
                    continue
            else:
                assert slot == -1 and merge == -1
            for t in range(start, start + count):
                covered[qo[s] + t, g * G:(g + 1) * G] += 1
        else:
            # a page range of one decode for up to 2 kv heads
            assert nn == 1 and g % 2 == 0
            ngh = min(2, shape.H_kv - g)
            per = -(-np_ // nsplit)
            for h in range(ngh):
                pages_cov.setdefault((s, g + h), []).append((start, count))
            if start + count == np_:
                appended[qo[s], g:g + ngh] += 1
                covered[qo[s], g * G:(g + ngh) * G] += 1
            if nsplit > 1:
                k = start // per
                assert start == k * per
                for h in range(ngh):
                    assert (slot + k * ngh + h) not in seen_slots
                    seen_slots.add(slot + k * ngh + h)
                assert 0 <= merge < info.n_merge
            else:
                assert slot == -1 and merge == -1
    assert np.all(covered == 1)
    assert np.all(appended == 1)
    for (s, g), spans in pages_cov.items():
        spans.sort()
        pos = 0
        for a, c in spans:
            assert a == pos and c > 0
            pos += c
        assert pos == kvp[s + 1] - kvp[s]
    for key, ps in pieces.items():
        ps.sort()
        assert [p[0] for p in ps] == list(range(ps[0][4]))
        assert len({p[3:] for p in ps}) == 1
        assert ps[0][1] == 0 and ps[-1][2] == ps[0][3]
        assert all(ps[i][2] == ps[i + 1][1] for i in range(len(ps) - 1))
    assert len(seen_slots) <= info.n_partials and (not seen_slots or max(seen_slots) < info.n_partials)
    assert info.n_partials - len(seen_slots) <= 1
    # each prefill row's ready flags (one per 128-position block and group of 2
    # kv heads) follow the previous row's, from req_aux on
    aux = m["req_aux"]
    groups = -(-shape.H_kv // 2)
    nxt = 0
    for s in range(n):
        nn = qo[s + 1] - qo[s]
        if nn >= 2:
            h = 16 * (kvp[s + 1] - kvp[s] - 1) + last[s] - nn
            assert aux[s] == nxt
            nxt += ((h + nn - 1) // 128 - h // 128 + 1) * groups
    assert nxt <= (int(qo[-1]) // 128 + 2 * n) * groups if n else True


def test_plan_reports_errors_and_warning():
    shape = W.Shape(4, 4, 64)
    t = [np.arange(2, dtype=np.int32)]
    with pytest.raises(S.SarathiError) as e:
        _product_plan([W.PREFILL_WAITING], [100], [0], t, 64, shape)
    assert e.value.status == S.ERR_CAPACITY
    with pytest.raises(S.SarathiError) as e:
        _product_plan([W.DECODE], [0], [3], t, 0, shape)
    assert e.value.status == S.ERR_INVALID_ARG
    with pytest.raises(S.SarathiError) as e:
        _product_plan([W.DECODE], [0], [3], t, 4, W.Shape(4, 4, 96))
    assert e.value.status == S.ERR_UNSUPPORTED
    with pytest.raises(S.SarathiError) as e:
        _product_plan([W.DECODE], [0], [3], t, 4, W.Shape(64, 2, 128))
    assert e.value.status == S.ERR_UNSUPPORTED
    tables = [np.arange(4, dtype=np.int32) + 4 * i for i in range(11)]
    st, info, m = _product_plan([W.DECODE] * 10 + [W.PREFILL_WAITING], [0] * 10 + [40], [20] * 10 + [0], tables, 8,
                                shape)
    assert st == S.WARN_OVER_BUDGET_DECODES and m["n_sched"] == 10


def test_plan_bounds_cover_actual_sizes():
    for wl in (W.mistral(), W.llama70b(), W.yi34b(), W.tiny(1)):
        reqs, keep = S.make_requests(*wl.arrays())
        shp = S.Shape(wl.shape.H_q, wl.shape.H_kv, wl.shape.d, 16)
        hb, wb = S.sarathi_plan_bounds(reqs, len(wl.requests), wl.budget, shp, 148)
        st, info, packed = S.sarathi_plan(reqs, len(wl.requests), wl.budget, shp, 148)
        assert info.packed_ints * 4 <= hb and info.workspace_bytes <= wb


# ------------------------------------------------------------ plan policies

def _random_policy_set(rng):
    n = int(rng.integers(0, 14))
    states, prompt, computed, tables = [], [], [], []
    for i in range(n):
        stt = int(rng.integers(0, 3))
        if stt == W.DECODE:
            h, pl, cap = int(rng.integers(0, 300)), 0, 0
            cap = h + 1
        else:
            pl = int(rng.integers(1, 700))
            h = 0 if stt == W.PREFILL_WAITING and rng.random() < 0.7 else int(rng.integers(0, pl + 1))
            cap = pl
        states.append(stt)
        prompt.append(pl)
        computed.append(h)
        tables.append(rng.permutation(5000)[:(cap + 15) // 16 + int(rng.integers(0, 3))].astype(np.int32))
    return states, prompt, computed, tables


def test_plan_policies_match_oracle_random_request_sets():
    rng = np.random.default_rng(321)
    shape = W.Shape(8, 2, 64)
    shp = S.Shape(8, 2, 64, 16)
    for trial in range(200):
        states, prompt, computed, tables = _random_policy_set(rng)
        kind = int(rng.integers(0, 2))
        budget = int(rng.integers(1, 600))
        max_batch = int(rng.integers(0, 8)) if kind == S.POLICY_DECODE_MAXIMAL else 0
        align = int(rng.choice([1, 1, 8, 32, 128]))
        st_o, mo = oracle.plan(states, prompt, computed, tables, budget, 16, policy=kind, max_batch=max_batch,
                               align=align)
        reqs, keep = S.make_requests(states, prompt, computed, tables)
        pol = S.PlanPolicy(kind, budget, max_batch, align)
        hb, wb = S.sarathi_plan_bounds(reqs, len(states), budget, shp, 148)
        nsm = int(rng.integers(1, 200))
        st_p, info, packed = S.sarathi_plan_ex(reqs, len(states), pol, shp, nsm)
        mp = S.plan_arrays(info, packed)
        _compare(st_o, mo, st_p, mp)
        _check_work_list(info, mp, shape, nsm)
        assert info.packed_ints * 4 <= hb


@pytest.mark.parametrize("wl", [W.mistral(), W.llama70b(), W.yi34b()], ids=lambda w: w.name)
def test_plan_policies_match_oracle_on_workloads(wl):
    shp = S.Shape(wl.shape.H_q, wl.shape.H_kv, wl.shape.d, 16)
    reqs, keep = S.make_requests(*wl.arrays())
    for kind, budget, B, align in ((S.POLICY_STALL_FREE, wl.budget, 0, 32),
                                   (S.POLICY_DECODE_MAXIMAL, 256, 0, 1),
                                   (S.POLICY_DECODE_MAXIMAL, 512, 64, 32)):
        st_o, mo = oracle.plan(*wl.arrays(), budget, 16, policy=kind, max_batch=B, align=align)
        st_p, info, packed = S.sarathi_plan_ex(reqs, len(wl.requests), S.PlanPolicy(kind, budget, B, align), shp, 148)
        mp = S.plan_arrays(info, packed)
        _compare(st_o, mo, st_p, mp)
        _check_work_list(info, mp, wl.shape)


def test_plan_ex_rejects_bad_policies():
    wl = W.tiny(0)
    shp = S.Shape(wl.shape.H_q, wl.shape.H_kv, wl.shape.d, 16)
    reqs, keep = S.make_requests(*wl.arrays())
    buf = np.zeros(1 << 16, np.int32)
    for pol in (S.PlanPolicy(2, 64, 0, 1), S.PlanPolicy(0, 64, 3, 1), S.PlanPolicy(1, 64, -1, 1),
                S.PlanPolicy(0, 64, 0, 0), S.PlanPolicy(1, 0, 4, 1)):
        info = S.PlanInfo()
        st = S.load().sarathi_plan_ex(reqs, len(wl.requests), ctypes.byref(pol), ctypes.byref(shp), 148,
                                      buf.ctypes.data, buf.nbytes, ctypes.byref(info))
        assert st == S.ERR_INVALID_ARG, (pol.kind, pol.token_budget, pol.max_batch, pol.chunk_align)


# ------------------------------------------------------------ separate metadata sets

def test_split_metadata_equals_oracle_plans_of_each_class():
    """The decode set equals the oracle's plan of the decode requests alone, and
    the prefill set the oracle's plan of the prefill requests alone with the
    budget the decodes left (the stall-free rule fills prefills from what is
    left): the separate sets an executor with two attention calls builds."""
    rng = np.random.default_rng(77)
    shp = S.Shape(8, 2, 64, 16)
    for trial in range(150):
        states, prompt, computed, tables = _random_policy_set(rng)
        budget = int(rng.integers(1, 800))
        reqs, keep = S.make_requests(states, prompt, computed, tables)
        st, info, packed = S.sarathi_plan(reqs, len(states), budget, shp, 148)
        dec, pre = S.sarathi_split_metadata(info, packed)
        full = S.plan_arrays(info, packed)
        assert dec["rows"] == info.num_decodes and dec["rows"] + pre["rows"] == info.n_sched
        assert dec["token_offset"] == 0 and pre["token_offset"] == dec["tokens"]
        di = [i for i in range(len(states)) if states[i] == W.DECODE]
        pi = [i for i in range(len(states)) if states[i] != W.DECODE]
        sub = lambda idx: ([states[i] for i in idx], [prompt[i] for i in idx], [computed[i] for i in idx],
                           [tables[i] for i in idx])
        if di:
            _, od = oracle.plan(*sub(di), max(len(di), 1), 16)
            for key in ("qo_indptr", "kv_page_indptr", "kv_page_indices", "kv_last_page_len"):
                assert np.array_equal(np.asarray(od[key]), dec[key]), key
        left = budget - len(di)
        if pi and left > 0:
            _, op = oracle.plan(*sub(pi), left, 16)
            for key in ("qo_indptr", "kv_page_indptr", "kv_page_indices", "kv_last_page_len"):
                assert np.array_equal(np.asarray(op[key]), pre[key]), key
            assert [pi[i] for i in op["req_index"]] == list(full["req_index"][pre["first_row"]:])
        else:
            assert pre["rows"] == 0


def test_host_buffer_step_rejects_missing_host_side_before_any_cuda_call():
    """sarathi_mixed_attn_host checks its host side first: a NULL io or NULL
    host pointer is INVALID_ARG, returned before the library touches CUDA
    (so this runs without a GPU)."""
    import ctypes
    lib = S.load()
    a = S.AttnArgs()
    st = lib.sarathi_mixed_attn_host(ctypes.byref(a), None, None)
    assert st == S.ERR_INVALID_ARG and b"io" in lib.sarathi_last_error()
    buf = np.zeros(16, np.uint16)
    io = S.HostIO(buf.ctypes.data, buf.ctypes.data, 0, buf.ctypes.data, 0, 0)
    st = lib.sarathi_mixed_attn_host(ctypes.byref(a), ctypes.byref(io), None)
    assert st == S.ERR_INVALID_ARG and b"host pointer" in lib.sarathi_last_error()


@pytest.mark.parametrize("wl,lo,hi", [(W.llama7b(chunk_step=3), 46, 62), (W.llama70b(), 56, 96),
                                      (W.mistral(), 16, 80)], ids=lambda x: getattr(x, "name", str(x)))
def test_sm_partition_lies_in_the_measured_flat_range(wl, lo, hi):
    """The planner's share of SMs for the prefill tiles (first_sms, 152 SMs)
    lies where a sweep of it on GB300 measured the step within about 2% of
    its best: Llama-2-7B-like 46-62 (788 us at 48, 792 at 56, 803 at 64, 829
    at 40), LLaMA2-70B-like 56-96 (578-602 us, no clear optimum), Mistral-7B-like
    16-80 (133-135 us; 138 at 40, 148 at 120)."""
    st, info, mp = _product_plan(*wl.arrays(), wl.budget, wl.shape, num_sms=152)
    assert lo <= info.first_sms <= hi, info.first_sms


def test_prefill_only_steps_choose_where_the_appends_run():
    """In a step without decodes the planner starts the APPEND items on a
    second queue (a few CTAs append while the tiles stream their history)
    where every tile has more history to read than an APPEND item takes, and
    keeps them at the head of the one queue where the tiles need the new keys
    at once.  Last 512-token chunk of an 8192-token prompt on 152 SMs: 128
    tiles on the first queue, the 64 APPEND items on the second, 24 CTAs
    starting there; the one-shot prompt (no history): one queue."""
    wl = W.llama7b_prefill_only(512, 15)
    st, info, mp = _product_plan(*wl.arrays(), wl.budget, wl.shape, num_sms=152)
    kinds = mp["items"][:, 0]
    assert info.n_first == int((kinds == 1).sum()) == 128 and (kinds[info.n_first:] == 0).all()
    assert info.first_sms == 128
    _check_work_list(info, mp, wl.shape, 152)
    wl = W.llama7b_prefill_only(8192, 0)
    st, info, mp = _product_plan(*wl.arrays(), wl.budget, wl.shape, num_sms=152)
    kinds = mp["items"][:, 0]
    assert info.n_first == info.n_items and info.first_sms == 152
    assert (kinds[:int((kinds == 0).sum())] == 0).all()


@pytest.mark.parametrize("chunk,app_sms,pieces", [(512, 24, 0), (1024, 38, 0), (2048, 76, 0), (8192, 0, 0)])
def test_prefill_only_layout_is_the_measured_best(chunk, app_sms, pieces):
    """The last chunk of an 8192-token prompt on 152 SMs gets the layout that
    timed fastest on GB300 among those tried: APPEND items on a second queue
    started by 24 CTAs at 512 tokens (70.4 us; 81.8 with them at the head of
    the one queue), 38 at 1024 (125.6; 24: 131.7, 57: 144.0, 76: 142.0, one
    queue with 38 x 2 key pieces: 137.9), 76 at 2048 (223.9; 66: 224.9, 49:
    228.5, one queue with 76 x 2 pieces: 228.0), and one queue without
    pieces for the one-shot prompt, whose tiles need the new keys at once."""
    wl = W.llama7b_prefill_only(chunk, 8192 // chunk - 1)
    st, info, mp = _product_plan(*wl.arrays(), wl.budget, wl.shape, num_sms=152)
    kinds = mp["items"][:, 0]
    assert info.first_sms == 152 - app_sms
    assert (info.n_first < info.n_items) == (app_sms > 0)
    assert int(((kinds == 1) & (mp["items"][:, 7] > 1)).sum()) == pieces
    _check_work_list(info, mp, wl.shape, 152)
