"""Pins for the oracle: each test ties it to something other than itself —
values the pages print, closed forms, library routines on special cases, brute
force on tiny inputs, and invariants the pages state.  CPU only."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_matches_library_on_float32_values():
    # For values a float32 holds exactly, round-to-nearest-even to bf16 is what
    # torch's float32 -> bfloat16 cast does.
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(4000).astype(np.float32),
                        (rng.standard_normal(1000) * 1e-30).astype(np.float32),
                        (rng.standard_normal(1000) * 1e30).astype(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_rne(x.astype(np.float64))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("x,expect", [
    (1.0 + 2.0**-8, 0x3F80),                  # exact tie between 1 and 1+2^-7 -> even (1.0)
    (1.0 + 2.0**-8 + 2.0**-40, 0x3F81),       # just above the tie: a double rounding via float would give 1.0
    (1.0 + 2.0**-8 - 2.0**-40, 0x3F80),
    (1.0 + 3 * 2.0**-8, 0x3F82),              # tie with odd lower neighbour -> up to even
    (-(1.0 + 2.0**-8 + 2.0**-40), 0xBF81),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (2.0**-130, 0x0008),                      # bf16 subnormal: 2^-130 = 8 * 2^-133
    (float.fromhex("0x1.FEp127"), 0x7F7F),    # bf16 max
    (float.fromhex("0x1.FFp127"), 0x7F80),    # tie above max rounds to even -> infinity
])
def test_bf16_single_rounding_cases(x, expect):
    assert int(oracle.bf16_rne(np.array([x]))[0]) == expect


# ---------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal(128)
    assert np.array_equal(oracle.rope(x, 0), x)


def test_rope_closed_form_unit_vectors():
    # rotate-half: pair (j, j+d/2) turns by pos * base^(-2j/d)
    d, base, pos = 8, 100.0, 37
    for j in range(d // 2):
        th = pos * base ** (-2.0 * j / d)
        e = np.zeros(d); e[j] = 1.0
        r = oracle.rope(e, pos, base)
        want = np.zeros(d); want[j] = math.cos(th); want[j + d // 2] = math.sin(th)
        assert np.allclose(r, want, atol=1e-15, rtol=0)
        e = np.zeros(d); e[j + d // 2] = 1.0
        r = oracle.rope(e, pos, base)
        want = np.zeros(d); want[j] = -math.sin(th); want[j + d // 2] = math.cos(th)
        assert np.allclose(r, want, atol=1e-15, rtol=0)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(128)
    r = oracle.rope(x, 12345)
    n0 = x[:64] ** 2 + x[64:] ** 2
    n1 = r[:64] ** 2 + r[64:] ** 2
    assert np.allclose(n0, n1, rtol=1e-13, atol=0)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    base_dot = oracle.rope(q, 900) @ oracle.rope(k, 100)
    for shift in (1, 17, 5000):
        assert abs(oracle.rope(q, 900 + shift) @ oracle.rope(k, 100 + shift) - base_dot) < 1e-9


# ---------------------------------------------------------------- plan

def _plan_from_lists(states, prompt, computed, tables, budget, page=16):
    return oracle.plan(states, prompt, computed, tables, budget, page)


def test_plan_worked_example_512():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_512.json")))
    s1 = g["step1"]
    budget = g["budget"]
    ctx = np.random.default_rng(5).integers(256, 4096, size=s1["decodes"], endpoint=True)
    # caller order deliberately mixes classes: the plan must put decodes first
    states = [W.PREFILL_RUNNING] + [W.DECODE] * 40 + [W.PREFILL_RUNNING] + [W.DECODE] * 40
    prompt = [300] + [0] * 40 + [768 + 900] + [0] * 40
    computed = [0] + list(ctx[:40]) + [768] + list(ctx[40:])
    tables = [np.arange(2000, dtype=np.int32) + 2000 * i for i in range(len(states))]
    st, m = _plan_from_lists(states, prompt, computed, tables, budget)
    assert st == oracle.OK
    assert m["num_decodes"] == 80 and m["n_sched"] == 82
    assert list(m["num_new"][:80]) == [1] * 80
    assert all(states[i] == W.DECODE for i in m["req_index"][:80])
    assert m["req_index"][80] == 0 and m["num_new"][80] == s1["P"]["expect_new"]
    assert m["last_chunk"][80] == s1["P"]["expect_last_chunk"]
    assert m["req_index"][81] == 41 and m["num_new"][81] == s1["Q"]["expect_new"]
    assert m["last_chunk"][81] == s1["Q"]["expect_last_chunk"]
    assert m["num_tokens"] == s1["expect_total"]
    # step 2: P became a decode; Q continues
    s2 = g["step2"]
    states2 = [W.DECODE] + [W.DECODE] * 40 + [W.PREFILL_RUNNING] + [W.DECODE] * 40
    computed2 = [300] + list(ctx[:40] + 1) + [768 + 132] + list(ctx[40:] + 1)
    st, m2 = _plan_from_lists(states2, prompt, computed2, tables, budget)
    assert st == oracle.OK
    assert m2["num_decodes"] == s2["decodes"]
    assert m2["num_new"][-1] == s2["Q"]["expect_new"]
    assert m2["num_tokens"] == s2["expect_total"]


def test_plan_class_order_waiting_after_running():
    # P waiting, Q running: the running chunk is served first and takes the rest
    ctx = [300] * 80
    states = [W.PREFILL_WAITING] + [W.DECODE] * 80 + [W.PREFILL_RUNNING]
    prompt = [300] + [0] * 80 + [1668]
    computed = [0] + ctx + [768]
    tables = [np.arange(200, dtype=np.int32) + 200 * i for i in range(len(states))]
    st, m = _plan_from_lists(states, prompt, computed, tables, 512)
    assert st == oracle.OK
    assert m["n_sched"] == 81
    assert m["req_index"][-1] == 81 and m["num_new"][-1] == 432


def test_plan_small_by_hand():
    g = json.load(open(os.path.join(GOLDEN, "plan_small_by_hand.json")))
    rq = g["requests"]
    st, m = _plan_from_lists([r["state"] for r in rq], [r["prompt_len"] for r in rq],
                             [r["num_computed"] for r in rq], [np.array(r["pages"], np.int32) for r in rq],
                             g["budget"], g["page_size"])
    e = g["expect"]
    assert st == e["status"]
    for key in ("req_index", "num_new", "last_chunk", "qo_indptr", "kv_page_indptr",
                "kv_page_indices", "kv_last_page_len"):
        assert list(m[key]) == e[key], key


def test_plan_tiny_schedule_chunks_64_64_64_8():
    chunks = []
    for s in range(4):
        wl = W.tiny(s)
        st, m = oracle.plan(*wl.arrays(), wl.budget, 16)
        assert st == oracle.OK
        assert m["num_decodes"] == 2 and list(m["num_new"][:2]) == [1, 1]
        chunks.append(int(m["num_new"][2]))
        assert m["last_chunk"][2] == (1 if s == 3 else 0)
    assert chunks == [64, 64, 64, 8]


def test_plan_decodes_over_budget_all_admitted():
    states = [W.DECODE] * 10 + [W.PREFILL_WAITING]
    tables = [np.arange(4, dtype=np.int32) + 4 * i for i in range(11)]
    st, m = _plan_from_lists(states, [0] * 10 + [40], [20] * 10 + [0], tables, 8)
    assert st == oracle.OVER_BUDGET_DECODES
    assert m["n_sched"] == 10 and m["num_tokens"] == 10


def test_plan_errors():
    t = [np.arange(2, dtype=np.int32)]
    assert _plan_from_lists([W.PREFILL_WAITING], [100], [0], t, 64)[0] == oracle.CAPACITY
    assert _plan_from_lists([W.DECODE], [0], [3], t, 0)[0] == oracle.INVALID
    assert _plan_from_lists([7], [0], [3], t, 8)[0] == oracle.INVALID
    assert _plan_from_lists([W.PREFILL_RUNNING], [4], [9], t, 8)[0] == oracle.INVALID


def test_plan_exact_page_boundary():
    # history 15 + 1 new = 16 tokens: exactly one full page, last page length 16
    st, m = _plan_from_lists([W.DECODE], [0], [15], [np.array([5, 6], np.int32)], 4)
    assert st == oracle.OK
    assert list(m["kv_page_indices"]) == [5] and list(m["kv_last_page_len"]) == [16]
    st, m = _plan_from_lists([W.DECODE], [0], [16], [np.array([5, 6], np.int32)], 4)
    assert list(m["kv_page_indices"]) == [5, 6] and list(m["kv_last_page_len"]) == [1]


# ---------------------------------------------------------------- attention

def _run_chunks(L, chunks, shape, seed, history_pages=None):
    """Prefill one L-token prompt through the oracle in the given chunk sizes.
    Returns (k_cache, v_cache, out [L][H_q][d])."""
    q, k, v = W.new_token_values(L, shape, seed)
    npages = (L + 15) // 16 + 2
    table = np.random.default_rng(seed).permutation(npages).astype(np.int32)
    kc = np.zeros((npages, shape.H_kv, 16, shape.d), np.uint16)
    vc = np.zeros_like(kc)
    out = np.zeros((L, shape.H_q, shape.d))
    done = 0
    for c in chunks:
        state = W.PREFILL_WAITING if done == 0 else W.PREFILL_RUNNING
        st, m = oracle.plan([state], [L], [done], [table], c, 16)
        assert st == oracle.OK and m["num_new"][0] == min(c, L - done)
        n = int(m["num_new"][0])
        o = oracle.step(m, q[done:done + n], k[done:done + n], v[done:done + n],
                        shape.H_q, shape.H_kv, shape.d, 16, shape.rope_base, kc, vc)
        out[done:done + n] = o
        done += n
    assert done == L
    return kc, vc, out, (q, k, v, table)


def test_chunk_invariance_bit_exact():
    # "chunking never changes attention semantics": any split gives the same
    # KV cache and the same outputs as one-shot prefill.
    shape = W.Shape(4, 2, 64)
    L = 83
    kc1, vc1, o1, _ = _run_chunks(L, [L], shape, 11)
    for chunks in ([16] * 6, [1, 15, 16, 17, 34], [40, 43], [64, 19]):
        kc2, vc2, o2, _ = _run_chunks(L, chunks, shape, 11)
        assert np.array_equal(kc1, kc2) and np.array_equal(vc1, vc2)
        assert np.array_equal(o1, o2)


def _dense_reference(q_rot, K, V, positions, scale):
    """Textbook dense masked softmax attention in numpy fp64.
    q_rot [n][d], K/V [kv_len][d], positions [n]: row i sees keys 0..positions[i]."""
    S = (q_rot @ K.T) * scale
    mask = np.arange(K.shape[0])[None, :] > positions[:, None]
    S = np.where(mask, -np.inf, S)
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    P /= P.sum(axis=1, keepdims=True)
    return P @ V


def test_attention_matches_dense_brute_force_with_history_and_gqa():
    shape = W.Shape(4, 2, 64)
    L = 70
    chunks = [32, 38]
    kc, vc, out, (q, k, v, table) = _run_chunks(L, chunks, shape, 21)
    group = shape.H_q // shape.H_kv
    # gather the final cache for the prompt (as the oracle wrote it)
    for hq in range(shape.H_q):
        g = hq // group
        K = np.concatenate([oracle.bf16_to_double(kc[p, g]) for p in table])[:L]
        V = np.concatenate([oracle.bf16_to_double(vc[p, g]) for p in table])[:L]
        q_rot = np.stack([oracle.rope(oracle.bf16_to_double(q[i, hq]), i) for i in range(L)])
        ref = _dense_reference(q_rot, K, V, np.arange(L), 1 / math.sqrt(shape.d))
        assert np.max(np.abs(ref - out[:, hq])) < 1e-12


def test_attention_decode_row_is_single_row_softmax():
    # a decode at history h attends its h+1 keys (history + its own new key)
    shape = W.Shape(2, 1, 64)
    h = 45
    rng = np.random.default_rng(9)
    table = np.array([3, 0, 2, 1], np.int32)
    kc = W.normal_bf16(rng, (4, 1, 16, 64))
    vc = W.normal_bf16(rng, (4, 1, 16, 64))
    q, k, v = W.new_token_values(1, shape, 9)
    st, m = oracle.plan([W.DECODE], [0], [h], [table], 8, 16)
    out = oracle.step(m, q, k, v, 2, 1, 64, 16, 10000.0, kc, vc)
    K = np.concatenate([oracle.bf16_to_double(kc[p, 0]) for p in table])[:h + 1]
    V = np.concatenate([oracle.bf16_to_double(vc[p, 0]) for p in table])[:h + 1]
    # the new key sits at position h, rotated by h
    assert np.array_equal(K[h], oracle.bf16_to_double(oracle.bf16_rne(oracle.rope(oracle.bf16_to_double(k[0, 0]), h))))
    assert np.array_equal(V[h], oracle.bf16_to_double(v[0, 0]))
    for hq in range(2):
        q_rot = oracle.rope(oracle.bf16_to_double(q[0, hq]), h)[None, :]
        ref = _dense_reference(q_rot, K, V, np.array([h]), 1 / 8.0)
        assert np.max(np.abs(ref[0] - out[0, hq])) < 1e-12


def test_attention_uniform_keys_average_values():
    # identical keys -> uniform weights over exactly the p+1 visible keys
    shape = W.Shape(1, 1, 64)
    L = 37
    kc = np.zeros((4, 1, 16, 64), np.uint16)
    vc = np.zeros_like(kc)
    table = np.arange(4, dtype=np.int32)
    rng = np.random.default_rng(4)
    q = W.normal_bf16(rng, (L, 1, 64))
    k = np.zeros((L, 1, 64), np.uint16)          # all-zero keys: every score is 0
    v = W.normal_bf16(rng, (L, 1, 64))
    st, m = oracle.plan([W.PREFILL_WAITING], [L], [0], [table], 64, 16)
    out = oracle.step(m, q, k, v, 1, 1, 64, 16, 10000.0, kc, vc)
    vd = oracle.bf16_to_double(v[:, 0])
    for i in range(L):
        assert np.max(np.abs(out[i, 0] - vd[:i + 1].mean(axis=0))) < 1e-13


# ---------------------------------------------------------------- counters

@pytest.mark.parametrize("L,chunks", [(200, [64, 64, 64, 8]), (83, [1, 15, 16, 17, 34]), (50, [50])])
def test_pairs_equal_triangle_for_any_split(L, chunks):
    total, done = 0, 0
    table = np.arange((L + 15) // 16, dtype=np.int32)
    for c in chunks:
        st, m = oracle.plan([W.PREFILL_RUNNING], [L], [done], [table], c, 16)
        total += oracle.pairs(m, 16)
        done += int(m["num_new"][0])
    assert total == L * (L + 1) // 2


@pytest.mark.parametrize("c,expect", [(512, 61440), (1024, 28672), (2048, 12288), (8192, 0)])
def test_reread_closed_form_8192(c, expect):
    # equal chunks c, K = L/c: history re-read = c*K*(K-1)/2 tokens
    L = 8192
    K = L // c
    assert expect == c * K * (K - 1) // 2
    table = np.arange(L // 16, dtype=np.int32)
    total, done = 0, 0
    while done < L:
        st, m = oracle.plan([W.PREFILL_RUNNING], [L], [done], [table], c, 16)
        total += oracle.reread_tokens(m, 16)
        done += int(m["num_new"][0])
    assert total == expect


# ---------------------------------------------------------------- plan policies
# Decode-maximal batching ("Sarathi：让解码搭上 prefill 的顺风车", section
# "Decode-maximal batching：顺车的账本") and chunk alignment ("Sarathi-Serve
# 完全拆解", section "257 为什么可能比 256 慢 32%").

def _random_request_set(rng, n_dec_max=12, n_pf_max=4):
    n_dec = int(rng.integers(0, n_dec_max + 1))
    n_pf = int(rng.integers(0, n_pf_max + 1))
    states, prompt, computed = [], [], []
    for _ in range(n_dec):
        states.append(W.DECODE); prompt.append(0); computed.append(int(rng.integers(0, 3000)))
    for _ in range(n_pf):
        st = W.PREFILL_RUNNING if rng.random() < 0.5 else W.PREFILL_WAITING
        L = int(rng.integers(1, 2500))
        h = int(rng.integers(1, L + 1)) - 1 if st == W.PREFILL_RUNNING else 0
        states.append(st); prompt.append(L); computed.append(h)
    order = rng.permutation(len(states))
    states = [states[i] for i in order]; prompt = [prompt[i] for i in order]; computed = [computed[i] for i in order]
    tables = [np.arange(300, dtype=np.int32) + 300 * i for i in range(len(states))]
    return states, prompt, computed, tables


def test_decode_maximal_table2_example():
    g = json.load(open(os.path.join(GOLDEN, "decode_maximal_table2.json")))
    B, C, L, ctx = g["batch_size_B"], g["chunk_tokens"], g["prompt_len"], g["decode_context"]
    # more decodes are waiting than fit: the batch takes the first B - 1 of them
    states = [W.DECODE] * 2 + [W.PREFILL_WAITING] + [W.DECODE] * 3
    prompt = [0, 0, L, 0, 0, 0]
    computed = [ctx, ctx, 0, ctx, ctx, ctx]
    tables = [np.arange(100, dtype=np.int32) + 100 * i for i in range(6)]
    st, m = oracle.plan(states, prompt, computed, tables, C, 16, policy=oracle.DECODE_MAXIMAL, max_batch=B)
    assert st == oracle.OK
    e = g["expect"]
    assert m["num_decodes"] == e["decodes"] and list(m["req_index"][:3]) == [0, 1, 3]
    assert m["req_index"][3] == 2 and m["num_new"][3] == e["chunk"] and m["last_chunk"][3] == 0
    assert m["num_tokens"] == e["total_tokens"]
    # next step: the prompt's last 3 tokens ride with 3 decodes
    computed2 = [ctx + 1, ctx + 1, C, ctx + 1, ctx, ctx]
    states2 = [W.DECODE, W.DECODE, W.PREFILL_RUNNING, W.DECODE, W.DECODE, W.DECODE]
    st, m2 = oracle.plan(states2, prompt, computed2, tables, C, 16, policy=oracle.DECODE_MAXIMAL, max_batch=B)
    n = g["next_step"]
    assert m2["num_new"][-1] == n["chunk"] and m2["last_chunk"][-1] == 1
    assert m2["num_decodes"] == n["decodes"] and m2["num_tokens"] == n["total_tokens"]


def test_decode_maximal_one_chunk_and_decode_cap_on_random_sets():
    rng = np.random.default_rng(21)
    for _ in range(300):
        states, prompt, computed, tables = _random_request_set(rng)
        C = int(rng.integers(1, 1500))
        B = int(rng.integers(0, 10))
        st, m = oracle.plan(states, prompt, computed, tables, C, 16, policy=oracle.DECODE_MAXIMAL, max_batch=B)
        assert st == oracle.OK
        pending = [i for c in (W.PREFILL_RUNNING, W.PREFILL_WAITING) for i in range(len(states))
                   if states[i] == c and prompt[i] > computed[i]]
        rows = list(m["req_index"])
        chunks = [s for s, i in enumerate(rows) if states[i] != W.DECODE]
        # exactly one chunk when a prompt is pending: the first in-progress one, else the first new one
        assert len(chunks) == (1 if pending else 0)
        if pending:
            s = chunks[0]
            assert s == len(rows) - 1 and rows[s] == pending[0]
            assert m["num_new"][s] == min(C, prompt[pending[0]] - computed[pending[0]])
        decs = [i for i in range(len(states)) if states[i] == W.DECODE]
        cap = len(decs) if B == 0 else min(len(decs), B - (1 if pending else 0))
        assert rows[:m["num_decodes"]] == decs[:cap] and m["num_decodes"] == cap


def test_decode_maximal_with_one_prompt_equals_stall_free():
    # one pending prompt and no batch limit: the stall-free plan with budget
    # decodes + C schedules exactly the same rows
    rng = np.random.default_rng(22)
    for _ in range(200):
        states, prompt, computed, tables = _random_request_set(rng, n_pf_max=0)
        L = int(rng.integers(1, 2500)); h = int(rng.integers(0, L))
        pos = int(rng.integers(0, len(states) + 1))
        states.insert(pos, W.PREFILL_RUNNING if h else W.PREFILL_WAITING)
        prompt.insert(pos, L); computed.insert(pos, h)
        tables = [np.arange(300, dtype=np.int32) + 300 * i for i in range(len(states))]
        C = int(rng.integers(1, 1500))
        n_dec = sum(1 for s in states if s == W.DECODE)
        st1, a = oracle.plan(states, prompt, computed, tables, C, 16, policy=oracle.DECODE_MAXIMAL, max_batch=0)
        st2, b = oracle.plan(states, prompt, computed, tables, n_dec + C, 16)
        assert st1 == st2 == oracle.OK
        for key in ("req_index", "num_new", "last_chunk", "qo_indptr", "kv_page_indptr", "kv_page_indices",
                    "kv_last_page_len"):
            assert np.array_equal(a[key], b[key]), key


def test_alignment_one_changes_nothing():
    rng = np.random.default_rng(23)
    for _ in range(200):
        states, prompt, computed, tables = _random_request_set(rng)
        budget = int(rng.integers(1, 3000))
        st1, a = oracle.plan(states, prompt, computed, tables, budget, 16)
        st2, b = oracle.plan(states, prompt, computed, tables, budget, 16, policy=oracle.STALL_FREE, align=1)
        assert st1 == st2
        for key in ("req_index", "num_new", "kv_page_indices"):
            assert np.array_equal(a[key], b[key]), key


def test_aligned_worked_example_512_by_hand():
    # the 512-token example with chunks aligned to 32: P's 300 tokens finish its
    # prompt and keep their size; Q's min(900, 132) = 132 is cut to 128
    ctx = np.random.default_rng(5).integers(256, 4096, size=80, endpoint=True)
    states = [W.DECODE] * 80 + [W.PREFILL_RUNNING, W.PREFILL_RUNNING]
    prompt = [0] * 80 + [300, 768 + 900]
    computed = list(ctx) + [0, 768]
    tables = [np.arange(2000, dtype=np.int32) + 2000 * i for i in range(82)]
    st, m = oracle.plan(states, prompt, computed, tables, 512, 16, policy=oracle.STALL_FREE, align=32)
    assert st == oracle.OK
    assert list(m["num_new"][80:]) == [300, 128] and list(m["last_chunk"][80:]) == [1, 0]
    assert m["num_tokens"] == 508
    # decode-maximal with the same alignment: C = 1021 leaves a 992-token chunk
    st, m = oracle.plan([W.PREFILL_WAITING], [1024], [0], [np.arange(100, dtype=np.int32)], 1021, 16,
                        policy=oracle.DECODE_MAXIMAL, align=32)
    assert list(m["num_new"]) == [992]


def test_aligned_chunks_are_multiples_unless_final():
    rng = np.random.default_rng(24)
    for _ in range(300):
        states, prompt, computed, tables = _random_request_set(rng)
        budget = int(rng.integers(1, 3000))
        align = int(rng.choice([8, 16, 32, 128]))
        for pol in (oracle.STALL_FREE, oracle.DECODE_MAXIMAL):
            st, m = oracle.plan(states, prompt, computed, tables, budget, 16, policy=pol, align=align)
            for s, i in enumerate(m["req_index"]):
                if states[i] == W.DECODE:
                    continue
                n = int(m["num_new"][s])
                assert n > 0
                assert m["last_chunk"][s] == 1 or n % align == 0
            n_dec = m["num_decodes"]
            if pol == oracle.STALL_FREE and n_dec <= budget:
                assert m["num_tokens"] <= budget


# ---------------------------------------------------------------- state after a step

def test_advance_turns_worked_example_step1_into_step2():
    """The 512-token example: after step 1, P (finished) decodes and Q continues,
    giving step 2's 81 decodes and Q's 431-token chunk (golden fixture)."""
    g = json.load(open(os.path.join(GOLDEN, "worked_example_512.json")))
    ctx = np.random.default_rng(5).integers(256, 4096, size=80, endpoint=True)
    states = [W.PREFILL_RUNNING] + [W.DECODE] * 40 + [W.PREFILL_RUNNING] + [W.DECODE] * 40
    prompt = [300] + [0] * 40 + [768 + 900] + [0] * 40
    computed = [0] + list(ctx[:40]) + [768] + list(ctx[40:])
    tables = [np.arange(2000, dtype=np.int32) + 2000 * i for i in range(len(states))]
    st, m1 = _plan_from_lists(states, prompt, computed, tables, g["budget"])
    st, states2, computed2 = oracle.advance(states, prompt, computed, m1)
    assert st == oracle.OK
    assert states2[0] == W.DECODE and computed2[0] == 300
    assert states2[41] == W.PREFILL_RUNNING and computed2[41] == 768 + 132
    assert computed2[1:41] == list(ctx[:40] + 1)
    st, m2 = _plan_from_lists(states2, prompt, computed2, tables, g["budget"])
    s2 = g["step2"]
    assert m2["num_decodes"] == s2["decodes"] and m2["num_new"][-1] == s2["Q"]["expect_new"]
    assert m2["num_tokens"] == s2["expect_total"]


def test_advance_waiting_prompt_runs_then_decodes():
    states, prompt, computed = [W.PREFILL_WAITING], [100], [0]
    tables = [np.arange(10, dtype=np.int32)]
    for expect_state, expect_h in ((W.PREFILL_RUNNING, 64), (W.DECODE, 100), (W.DECODE, 101)):
        st, m = oracle.plan(states, prompt, computed, tables, 64, 16)
        st, states, computed = oracle.advance(states, prompt, computed, m)
        assert st == oracle.OK and states == [expect_state] and computed == [expect_h]


# ---------------------------------------------------------------- interleaved RoPE
# The interleaved pairing (2j, 2j+1) of the original RoPE formulation (Su et
# al., RoFormer), as an option next to rotate-half.

def _perm_interleaved_to_half(d):
    # position 2j -> j, 2j+1 -> j + d/2
    p = np.empty(d, dtype=np.int64)
    p[0::2] = np.arange(d // 2)
    p[1::2] = np.arange(d // 2) + d // 2
    return p


def test_interleaved_rope_is_rotate_half_after_pairing_permutation():
    rng = np.random.default_rng(31)
    for d in (64, 128):
        perm = _perm_interleaved_to_half(d)
        for pos in (0, 1, 77, 4096, 16383):
            x = rng.standard_normal(d)
            xh = np.empty(d); xh[perm] = x          # x in rotate-half order
            yh = oracle.rope(xh, pos)
            yi = oracle.rope(x, pos, style=oracle.INTERLEAVED)
            assert np.array_equal(yi, yh[perm])


def test_interleaved_rope_closed_form_unit_vectors():
    d, pos, base = 64, 37, 10000.0
    for j in (0, 5, 31):
        x = np.zeros(d); x[2 * j] = 1.0
        th = pos * base ** (-2.0 * j / d)
        y = oracle.rope(x, pos, base, style=oracle.INTERLEAVED)
        expect = np.zeros(d); expect[2 * j] = np.cos(th); expect[2 * j + 1] = np.sin(th)
        assert np.max(np.abs(y - expect)) < 1e-15


def test_interleaved_step_equals_rotate_half_step_on_permuted_heads():
    """A whole step with interleaved RoPE equals the rotate-half step on inputs
    whose head dimensions were permuted, with the pages permuted back."""
    wl = W.tiny(1)
    sh = wl.shape
    st, m = oracle.plan(*wl.arrays(), wl.budget, 16)
    T = m["num_tokens"]
    q, k, v = W.new_token_values(T, sh, 5)
    kc, vc = W.history_cache_numpy(wl.num_pages, sh, wl.seed)
    perm = _perm_interleaved_to_half(sh.d)
    inv = np.argsort(perm)
    # interleaved step on (q, k, v) and caches as given
    kc_i, vc_i = kc.copy(), vc.copy()
    out_i = oracle.step(m, q, k, v, sh.H_q, sh.H_kv, sh.d, 16, sh.rope_base, kc_i, vc_i, style=oracle.INTERLEAVED)
    # rotate-half step on the same data with head dims reordered
    reord = lambda a: np.ascontiguousarray(a[..., inv])
    kc_h, vc_h = reord(kc), reord(vc)
    out_h = oracle.step(m, reord(q), reord(k), reord(v), sh.H_q, sh.H_kv, sh.d, 16, sh.rope_base, kc_h, vc_h)
    assert np.array_equal(kc_h[..., perm], kc_i) and np.array_equal(vc_h[..., perm], vc_i)
    assert np.max(np.abs(out_h[..., perm] - out_i)) < 1e-12


# ---------------------------------------------------------------- QKV projection

def test_qkv_proj_matches_a_brute_force_loop():
    rng = np.random.default_rng(41)
    T, hidden, Hq, Hkv, d = 3, 8, 2, 1, 4
    x = W.bf16_bits(rng.standard_normal((T, hidden)))
    w = W.bf16_bits(rng.standard_normal(((Hq + 2 * Hkv) * d, hidden)))
    q, k, v = oracle.qkv_proj(x, w, Hq, Hkv, d)
    xd, wd = oracle.bf16_to_double(x), oracle.bf16_to_double(w)
    y = [[sum(xd[t][i] * wd[n][i] for i in range(hidden)) for n in range(wd.shape[0])] for t in range(T)]
    for t in range(T):
        for n in range(wd.shape[0]):
            if n < Hq * d:
                got = q[t][n // d][n % d]
            elif n < (Hq + Hkv) * d:
                got = k[t][(n - Hq * d) // d][(n - Hq * d) % d]
            else:
                got = v[t][(n - (Hq + Hkv) * d) // d][(n - (Hq + Hkv) * d) % d]
            assert abs(got - y[t][n]) < 1e-12


def test_qkv_proj_permutation_weights_select_columns():
    # W row n = e_{perm[n]}: Y[:, n] = X[:, perm[n]] exactly, and the split puts
    # column n at the head and offset its position says
    rng = np.random.default_rng(42)
    T, hidden, Hq, Hkv, d = 5, 64, 4, 2, 8
    N = (Hq + 2 * Hkv) * d
    perm = rng.integers(0, hidden, size=N)
    w = np.zeros((N, hidden)); w[np.arange(N), perm] = 1.0
    x = W.bf16_bits(rng.standard_normal((T, hidden)))
    q, k, v = oracle.qkv_proj(x, W.bf16_bits(w), Hq, Hkv, d)
    xd = oracle.bf16_to_double(x)
    y = np.concatenate([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], axis=1)
    assert np.array_equal(y, xd[:, perm])
