"""The QKV projection (one tcgen05 GEMM over the concatenated tokens) against
the oracle's fp64 matrix product; then projection + step chained on the
Mistral-like batch against the oracle's chain.

Tolerance: each output is the bf16 rounding of an fp32 sum of exact bf16
products, so |gpu - y| <= 2^-8 |y| (half a bf16 step) plus the fp32
accumulation error; the test allows 2^-7 |y| + 1e-4."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_helpers import assert_close, from_u16, to_u16

pytestmark = pytest.mark.gpu


def _inputs(T, hidden, Hq, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    x = W.bf16_bits(rng.standard_normal((T, hidden)))
    w = W.bf16_bits(rng.standard_normal(((Hq + 2 * Hkv) * d, hidden)) / np.sqrt(hidden))
    return x, w


def _run(x, w, Hq, Hkv, d):
    import torch
    import chunked_prefill_mixed_gb300 as S
    dev = torch.device("cuda")
    T = x.shape[0]
    q = torch.full((T, Hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    k = torch.full((T, Hkv, d), float("nan"), dtype=torch.bfloat16, device=dev)
    v = torch.full((T, Hkv, d), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    S.sarathi_qkv_proj(from_u16(x, dev), from_u16(w, dev), q, k, v, S.Shape(Hq, Hkv, d, 16), ws)
    assert S.sarathi_workspace_status(ws) == 0
    return q, k, v


# The launcher picks the tile width from the product's shape: 128 for the small
# products, 192 for the Mistral-like 512 tokens x 6144 columns (and the
# Llama-like 2048-token product below), 256 for 19 M tiles x 2048 columns (152
# tiles: one whole wave).
@pytest.mark.parametrize("T,hidden,Hq,Hkv,d", [(1, 256, 4, 4, 64), (66, 256, 4, 4, 64), (200, 512, 8, 2, 64),
                                               (129, 1024, 16, 4, 128), (512, 4096, 32, 8, 128),
                                               (19 * 128, 512, 8, 4, 128)])
def test_qkv_proj_matches_oracle(T, hidden, Hq, Hkv, d):
    x, w = _inputs(T, hidden, Hq, Hkv, d, seed=T + hidden)
    gq, gk, gv = _run(x, w, Hq, Hkv, d)
    oq, ok, ov = oracle.qkv_proj(x, w, Hq, Hkv, d)
    for g, o, name in ((gq, oq, "q"), (gk, ok, "k"), (gv, ov, "v")):
        gd = oracle.bf16_to_double(to_u16(g))
        assert np.all(np.isfinite(gd)), name
        err = np.abs(gd - o)
        assert np.all(err <= 2.0 ** -7 * np.abs(o) + 1e-4), (name, float(err.max()))


def test_qkv_proj_llama7b_step_sampled_rows():
    """The Llama-2-7B-like 2048-token product (16 M tiles x 12288 columns),
    checked on 3 rows of every 128-row tile over all columns."""
    T, hidden, Hq, Hkv, d = 2048, 4096, 32, 32, 128
    x, w = _inputs(T, hidden, Hq, Hkv, d, seed=2048)
    gq, gk, gv = _run(x, w, Hq, Hkv, d)
    rows = np.array(sorted({r for m in range(T // 128) for r in (128 * m, 128 * m + 77, 128 * m + 127)}))
    oq, ok, ov = oracle.qkv_proj(x[rows], w, Hq, Hkv, d)
    for g, o, name in ((gq, oq, "q"), (gk, ok, "k"), (gv, ov, "v")):
        gd = oracle.bf16_to_double(to_u16(g[rows.tolist()]))
        assert np.all(np.isfinite(gd)), name
        err = np.abs(gd - o)
        assert np.all(err <= 2.0 ** -7 * np.abs(o) + 1e-4), (name, float(err.max()))


def test_projection_then_step_on_the_mistral_batch():
    import torch
    from gpu_helpers import GpuStep
    wl = W.mistral()
    sh = wl.shape
    hidden = 4096
    gs = GpuStep(wl)
    T = gs.meta["num_tokens"]
    x, w = _inputs(T, hidden, sh.H_q, sh.H_kv, sh.d, seed=99)
    gq, gk, gv = _run(x, w, sh.H_q, sh.H_kv, sh.d)
    gs.q_dev, gs.k_dev, gs.v_dev = gq, gk, gv
    assert gs.run() == 0
    # the oracle's chain: fp64 projection, rounded once to bf16, then the step
    oq, ok, ov = oracle.qkv_proj(x, w, sh.H_q, sh.H_kv, sh.d)
    gs.q, gs.k, gs.v = (oracle.bf16_rne(a) for a in (oq, ok, ov))
    kc, vc = gs.oracle_caches()
    rt, rh = gs.sample_rows(512)
    ref, rt, rh = gs.oracle_rows(kc, vc, rt, rh)
    assert_close(oracle.bf16_to_double(to_u16(gs.out))[rt, rh], ref, "projection + step")
