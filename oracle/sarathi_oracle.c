/*
 * sarathi_oracle.c -- the ORACLE for the mixed-batch paged-attention step of
 * chunked prefill with stall-free batching.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library: it is a plain, slow, obviously-correct restatement of what
 * the step computes, in fp64, with one loop per definition.
 *
 * Pages it follows (titles as the pages give them):
 *   [SS]  "Sarathi-Serve 完全拆解：分块 Prefill 与无停顿批处理如何兼顾吞吐和尾延迟"
 *   [CP]  "Chunked Prefill 与 PD 分离：切片混批，还是拆开两个池"
 *   [ST]  "分块预填充与 Stall-free 调度：把 LLM 推理的吞吐-延迟权衡算清楚"
 *   [SA]  "Sarathi：让解码搭上 prefill 的顺风车"
 *
 * Functions and the passages they restate:
 *   oracle_plan_policy  the two batch policies:
 *                     stall-free [CP] §3.1 (decode -> in-progress chunk -> new
 *                     request, the budget shared by several chunks);
 *                     decode-maximal [SA] §"Decode-maximal batching：顺车的账本"
 *                     (one prefill chunk plus as many decodes as fit, at most
 *                     B - 1 of them); optional chunk alignment, [SS] §"257 为什么
 *                     可能比 256 慢 32%" (candidate sizes aligned to 32).
 *   oracle_plan       stall-free without alignment:
 *                     [SS] §"一个 512-token 预算的例子" (budget filled in turn,
 *                     several chunks per batch allowed);
 *                     [ST] §六·补二 (chunk = min(remaining budget, remaining prompt));
 *                     [SS] §"混合批不是…" (qo_indptr / kv_page_indptr /
 *                     kv_page_indices / kv_last_page_len).
 *   oracle_advance    the request state after a step, [SS] §"一个 512-token 预算的
 *                     例子" and [CP] §3.1.
 *   oracle_rope(_styled)  RoPE at the ABSOLUTE position, [SS] §"分块不等于截断上下文"
 *                     and §"先验证数值与状态正确性" (positions never restart per
 *                     chunk).  The pages never spell RoPE out; the reading used is
 *                     rotate-half with theta_j = base^(-2j/d).
 *   oracle_bf16_rne   round-to-nearest-even to bfloat16 directly from the exact
 *                     double (one rounding, never via float).
 *   oracle_append     new tokens' K (rotated) and V written into the page
 *                     holding their position, [SS] §"分块不等于截断上下文".
 *   oracle_attend     o_i = sum_{j<=i} softmax_j(q_i.k_j / sqrt(d_h)) v_j over
 *                     history pages + current chunk, [SS] §"分块不等于截断上下文".
 *   oracle_pairs / oracle_reread_tokens   the triangle and re-read counts,
 *                     [SS] §"为什么总 FLOPs 近似不变，显存流量却增加".
 *
 * Pins (tests that tie this file to something other than itself) live in the
 * test suite: the 512-budget worked example, closed forms, brute force on tiny
 * inputs, chunk invariance.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_INVALID 1
#define ORC_CAPACITY 2
#define ORC_OVER_BUDGET_DECODES 3

#define ORC_DECODE 0
#define ORC_PREFILL_RUNNING 1
#define ORC_PREFILL_WAITING 2

#define ORC_POLICY_STALL_FREE 0
#define ORC_POLICY_DECODE_MAXIMAL 1

/* ------------------------------------------------------------------------- */
/* bf16 <-> double                                                            */
/* ------------------------------------------------------------------------- */

/* bf16 bits -> double: a bf16 is the top 16 bits of an IEEE float. */
double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round the exact double x to the nearest bfloat16, ties to even, in ONE
 * rounding step.  Written from the definition: x = m * 2^e with the integer
 * significand m rounded to 8 significant bits (1 implicit + 7 stored).
 * Normal range only for finite nonzero values of ordinary size; values below
 * the bf16 normal range are rounded on the subnormal grid 2^-133; overflow goes
 * to infinity.  NaN maps to the canonical quiet NaN. */
uint16_t oracle_bf16_rne(double x) {
    if (isnan(x)) return (uint16_t)0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);                /* a = f * 2^e with f in [0.5, 1) */
    /* bf16 normal numbers have unbiased exponent >= -126, i.e. e >= -125
     * in frexp's convention.  Below that the grid spacing is fixed. */
    int keep_e = e < -125 ? -125 : e;  /* grid: 2^(keep_e - 8) */
    double scaled = ldexp(a, 8 - keep_e);   /* exact: power-of-two scaling */
    /* nearbyint() in the default FE_TONEAREST mode rounds half to even. */
    double r = nearbyint(scaled);
    double y = ldexp(r, keep_e - 8);
    /* y is now exactly representable in bf16 unless it overflowed. */
    if (y > 0x1.FEp127) return (uint16_t)(sign | 0x7F80);  /* past bf16 max */
    float f = (float)y;                /* exact: y has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* ------------------------------------------------------------------------- */
/* RoPE (rotate-half, fp64)                                                   */
/* ------------------------------------------------------------------------- */

/* out = RoPE(x, pos): for j < d/2, theta = pos * base^(-2j/d),
 *   out_j       = x_j cos theta - x_{j+d/2} sin theta
 *   out_{j+d/2} = x_{j+d/2} cos theta + x_j sin theta
 * in fp64.  x and out may not alias. */
/* style 0, rotate-half: pair j is (x[j], x[j + d/2]).  style 1, interleaved:
 * pair j is (x[2j], x[2j+1]), the pairing of the original RoPE formulation
 * (Su et al., RoFormer, 2021, section 3.4.2).  Both rotate pair j by
 * pos * base^(-2j/d). */
void oracle_rope_styled(const double* x, int d, int64_t pos, double base, int style, double* out) {
    int half = d / 2;
    for (int j = 0; j < half; ++j) {
        double inv_freq = pow(base, -(2.0 * (double)j) / (double)d);
        double theta = (double)pos * inv_freq;
        double c = cos(theta), s = sin(theta);
        int i0 = style ? 2 * j : j, i1 = style ? 2 * j + 1 : j + half;
        double x0 = x[i0], x1 = x[i1];
        out[i0] = x0 * c - x1 * s;
        out[i1] = x1 * c + x0 * s;
    }
}
void oracle_rope(const double* x, int d, int64_t pos, double base, double* out) {
    oracle_rope_styled(x, d, pos, base, 0, out);
}

/* ------------------------------------------------------------------------- */
/* Plan                                                                       */
/* ------------------------------------------------------------------------- */

/* Inputs (caller order is kept inside each class):
 *   state[i], prompt_len[i], num_computed[i] (h: tokens already in cache),
 *   block table of request i = bt[bt_indptr[i] .. bt_indptr[i+1]).
 * Outputs (capacity: n_reqs rows, cap_pages page ids):
 *   req_index[n], num_new[n], last_chunk[n], qo_indptr[n+1],
 *   kv_page_indptr[n+1], kv_page_indices[...], kv_last_page_len[n];
 *   counts[0] = n scheduled, counts[1] = decodes, counts[2] = page ids written,
 *   counts[3] = tokens scheduled.
 * Returns ORC_OK, ORC_OVER_BUDGET_DECODES (output valid), ORC_CAPACITY,
 * ORC_INVALID. */
/* A chunk that does not finish its prompt is cut down to a multiple of
 * `align` tokens (align 1: no cut); the final chunk of a prompt keeps its size.
 * [SS] §"257 为什么可能比 256 慢 32%": the official code aligns candidate chunk
 * sizes to multiples of 32 -- an execution-shape choice, not a semantic one. */
static int aligned_take(int take, int rem, int align) {
    if (align > 1 && take < rem) take -= take % align;
    return take;
}

int oracle_plan_policy(int n_reqs, const int32_t* state, const int32_t* prompt_len,
                       const int32_t* num_computed, const int32_t* bt_indptr, const int32_t* bt,
                       int policy, int budget, int max_batch, int align, int page_size, int cap_pages,
                       int32_t* req_index, int32_t* num_new, int32_t* last_chunk,
                       int32_t* qo_indptr, int32_t* kv_page_indptr, int32_t* kv_page_indices,
                       int32_t* kv_last_page_len, int32_t* counts) {
    if (n_reqs < 0 || budget <= 0 || page_size <= 0 || align < 1 || max_batch < 0) return ORC_INVALID;
    if (policy != ORC_POLICY_STALL_FREE && policy != ORC_POLICY_DECODE_MAXIMAL) return ORC_INVALID;
    for (int i = 0; i < n_reqs; ++i) {
        if (state[i] < ORC_DECODE || state[i] > ORC_PREFILL_WAITING) return ORC_INVALID;
        if (num_computed[i] < 0) return ORC_INVALID;
        if (state[i] != ORC_DECODE && prompt_len[i] < num_computed[i]) return ORC_INVALID;
        if (bt_indptr[i + 1] < bt_indptr[i]) return ORC_INVALID;
    }
    int n = 0, decodes = 0;
    if (policy == ORC_POLICY_STALL_FREE) {
        int left = budget;
        /* 1) every running decode: one token each, [CP] §3.1 first class */
        for (int i = 0; i < n_reqs; ++i) {
            if (state[i] != ORC_DECODE) continue;
            req_index[n] = i; num_new[n] = 1; last_chunk[n] = 1;
            ++n; ++decodes; left -= 1;
        }
        /* 2) in-progress prefills, then 3) new prefills: min(remaining prompt,
         *    remaining budget) each, [ST] §六·补二; several chunks may share the
         *    budget, [SS] §"一个 512-token 预算的例子". */
        for (int cls = ORC_PREFILL_RUNNING; cls <= ORC_PREFILL_WAITING; ++cls) {
            for (int i = 0; i < n_reqs; ++i) {
                if (state[i] != cls) continue;
                int rem = prompt_len[i] - num_computed[i];
                int room = left > 0 ? left : 0;
                int take = aligned_take(rem < room ? rem : room, rem, align);
                if (take <= 0) continue;
                req_index[n] = i; num_new[n] = take;
                last_chunk[n] = (num_computed[i] + take == prompt_len[i]) ? 1 : 0;
                ++n; left -= take;
            }
        }
    } else {
        /* decode-maximal, [SA] §"Decode-maximal batching：顺车的账本": the batch
         * holds ONE prefill chunk of min(chunk size, remaining prompt) tokens --
         * from the first in-progress prefill, else the first new one -- and then
         * as many decodes as fit: at most B - 1 next to a chunk (its KV takes a
         * slot too), at most B without one; B = max_batch, 0 for no limit.
         * Decodes are listed first, in caller order, like every plan here. */
        int chunk_req = -1, chunk_take = 0;
        for (int cls = ORC_PREFILL_RUNNING; cls <= ORC_PREFILL_WAITING && chunk_req < 0; ++cls) {
            for (int i = 0; i < n_reqs; ++i) {
                if (state[i] != cls) continue;
                int rem = prompt_len[i] - num_computed[i];
                if (rem <= 0) continue;
                chunk_req = i;
                chunk_take = aligned_take(rem < budget ? rem : budget, rem, align);
                break;
            }
        }
        if (chunk_take <= 0) chunk_req = -1;
        int cap = max_batch > 0 ? max_batch - (chunk_req >= 0 ? 1 : 0) : n_reqs;
        for (int i = 0; i < n_reqs && decodes < cap; ++i) {
            if (state[i] != ORC_DECODE) continue;
            req_index[n] = i; num_new[n] = 1; last_chunk[n] = 1;
            ++n; ++decodes;
        }
        if (chunk_req >= 0) {
            req_index[n] = chunk_req; num_new[n] = chunk_take;
            last_chunk[n] = (num_computed[chunk_req] + chunk_take == prompt_len[chunk_req]) ? 1 : 0;
            ++n;
        }
    }
    /* metadata: kv_len = h + n, pages = ceil(kv_len / page), last-page length */
    int pages_out = 0, tokens = 0;
    qo_indptr[0] = 0; kv_page_indptr[0] = 0;
    for (int s = 0; s < n; ++s) {
        int i = req_index[s];
        int kv_len = num_computed[i] + num_new[s];
        int np = (kv_len + page_size - 1) / page_size;
        int have = bt_indptr[i + 1] - bt_indptr[i];
        if (np > have) return ORC_CAPACITY;
        if (pages_out + np > cap_pages) return ORC_CAPACITY;
        for (int p = 0; p < np; ++p) kv_page_indices[pages_out + p] = bt[bt_indptr[i] + p];
        pages_out += np;
        kv_last_page_len[s] = kv_len - page_size * (np - 1);
        tokens += num_new[s];
        qo_indptr[s + 1] = tokens;
        kv_page_indptr[s + 1] = pages_out;
    }
    counts[0] = n; counts[1] = decodes; counts[2] = pages_out; counts[3] = tokens;
    return (policy == ORC_POLICY_STALL_FREE && decodes > budget) ? ORC_OVER_BUDGET_DECODES : ORC_OK;
}

/* Stall-free with no alignment: [CP] §3.1, [ST] §六·补二, [SS] §"一个 512-token
 * 预算的例子". */
int oracle_plan(int n_reqs, const int32_t* state, const int32_t* prompt_len,
                const int32_t* num_computed, const int32_t* bt_indptr, const int32_t* bt,
                int budget, int page_size, int cap_pages,
                int32_t* req_index, int32_t* num_new, int32_t* last_chunk,
                int32_t* qo_indptr, int32_t* kv_page_indptr, int32_t* kv_page_indices,
                int32_t* kv_last_page_len, int32_t* counts) {
    return oracle_plan_policy(n_reqs, state, prompt_len, num_computed, bt_indptr, bt, ORC_POLICY_STALL_FREE,
                              budget, 0, 1, page_size, cap_pages, req_index, num_new, last_chunk, qo_indptr,
                              kv_page_indptr, kv_page_indices, kv_last_page_len, counts);
}

/* After the step: every scheduled request has num_new more tokens in its KV
 * cache; a prefill whose last chunk ran becomes a decode, one that ran a
 * chunk but has prompt left is in progress.  [SS] §"一个 512-token 预算的例子"
 * (P, finished, decodes in the next step; Q continues), [CP] §3.1 (the three
 * request classes). */
int oracle_advance(int n_reqs, int32_t* state, const int32_t* prompt_len, int32_t* num_computed,
                   int n_sched, const int32_t* req_index, const int32_t* num_new) {
    for (int s = 0; s < n_sched; ++s) {
        int i = req_index[s];
        if (i < 0 || i >= n_reqs || num_new[s] <= 0) return ORC_INVALID;
        num_computed[i] += num_new[s];
        if (state[i] == ORC_DECODE) continue;
        if (num_computed[i] > prompt_len[i]) return ORC_INVALID;
        state[i] = num_computed[i] == prompt_len[i] ? ORC_DECODE : ORC_PREFILL_RUNNING;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* KV append and attention                                                    */
/* ------------------------------------------------------------------------- */

/* Cache layout: cache[page][kv_head][slot][d] as bf16 bits.  This is just the
 * container the step writes into; its element order is the harness's choice. */
static size_t cache_off(int page, int g, int slot, int H_kv, int page_size, int d) {
    return (((size_t)page * H_kv + g) * page_size + slot) * (size_t)d;
}

/* Write every scheduled new token's K (rotated at its absolute position, then
 * rounded once to bf16) and V (copied) into page kv_page_indices[...][pos/page]
 * at slot pos%page, for every kv head.  k, v: bf16 bits [T][H_kv][d]. */
void oracle_append_styled(int n_sched, const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                          const int32_t* kv_page_indices, const int32_t* kv_last_page_len,
                          const uint16_t* k, const uint16_t* v, int H_kv, int d, int page_size,
                          double rope_base, int rope_style, uint16_t* k_cache, uint16_t* v_cache) {
    double* x = (double*)malloc(sizeof(double) * (size_t)d * 2);
    double* xr = x + d;
    for (int s = 0; s < n_sched; ++s) {
        int qo_len = qo_indptr[s + 1] - qo_indptr[s];
        int np = kv_page_indptr[s + 1] - kv_page_indptr[s];
        int kv_len = (np - 1) * page_size + kv_last_page_len[s];
        int h = kv_len - qo_len;  /* history: tokens cached before this step */
        for (int i = 0; i < qo_len; ++i) {
            int t = qo_indptr[s] + i;
            int pos = h + i;
            int page = kv_page_indices[kv_page_indptr[s] + pos / page_size];
            int slot = pos % page_size;
            for (int g = 0; g < H_kv; ++g) {
                const uint16_t* kr = k + ((size_t)t * H_kv + g) * d;
                const uint16_t* vr = v + ((size_t)t * H_kv + g) * d;
                for (int e = 0; e < d; ++e) x[e] = oracle_bf16_to_double(kr[e]);
                oracle_rope_styled(x, d, pos, rope_base, rope_style, xr);
                size_t off = cache_off(page, g, slot, H_kv, page_size, d);
                for (int e = 0; e < d; ++e) {
                    k_cache[off + e] = oracle_bf16_rne(xr[e]);
                    v_cache[off + e] = vr[e];
                }
            }
        }
    }
    free(x);
}

/* Attention for a list of (row t, q head hq) pairs, reading K/V from the pages
 * AFTER the step's append.  For the row's request r and its absolute position
 * p = h + (t - qo_indptr[r]):
 *   s_j = RoPE(q, p) . K[j] / sqrt(d)   for j = 0..p (causal: history + chunk)
 *   o   = sum_j e^{s_j - m} V[j] / sum_j e^{s_j - m},  m = max_j s_j
 * kv head of hq: g = hq / (H_q / H_kv) (contiguous GQA groups).
 * out: double [n_pairs][d]; lse (optional): double [n_pairs] = m + log(sum).
 * Rows are independent; OpenMP (if enabled) splits the list. */
void oracle_attend_styled(int n_sched, const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                          const int32_t* kv_page_indices, const int32_t* kv_last_page_len,
                          const uint16_t* q, int H_q, int H_kv, int d, int page_size, double rope_base,
                          int rope_style, const uint16_t* k_cache, const uint16_t* v_cache,
                          int n_pairs, const int32_t* row_t, const int32_t* row_hq,
                          double* out, double* lse) {
    int T = qo_indptr[n_sched];
    int group = H_q / H_kv;
    double scale = 1.0 / sqrt((double)d);
    #pragma omp parallel
    {
        double* qx = (double*)malloc(sizeof(double) * (size_t)d * 2);
        double* qr = qx + d;
        size_t cap = 1024;
        double* sc = (double*)malloc(sizeof(double) * cap);
        #pragma omp for schedule(dynamic, 1)
        for (int w = 0; w < n_pairs; ++w) {
            int t = row_t[w], hq = row_hq[w];
            double* o = out + (size_t)w * d;
            if (t < 0 || t >= T || hq < 0 || hq >= H_q) {
                for (int e = 0; e < d; ++e) o[e] = NAN;
                if (lse) lse[w] = NAN;
                continue;
            }
            /* request owning row t */
            int r = 0;
            while (!(qo_indptr[r] <= t && t < qo_indptr[r + 1])) ++r;
            int qo_len = qo_indptr[r + 1] - qo_indptr[r];
            int np = kv_page_indptr[r + 1] - kv_page_indptr[r];
            int kv_len = (np - 1) * page_size + kv_last_page_len[r];
            int h = kv_len - qo_len;
            int p = h + (t - qo_indptr[r]);
            int g = hq / group;
            const uint16_t* qrow = q + ((size_t)t * H_q + hq) * d;
            for (int e = 0; e < d; ++e) qx[e] = oracle_bf16_to_double(qrow[e]);
            oracle_rope_styled(qx, d, p, rope_base, rope_style, qr);
            if ((size_t)(p + 1) > cap) {
                cap = (size_t)(p + 1);
                sc = (double*)realloc(sc, sizeof(double) * cap);
            }
            double m = -INFINITY;
            for (int j = 0; j <= p; ++j) {
                int page = kv_page_indices[kv_page_indptr[r] + j / page_size];
                const uint16_t* kj = k_cache + cache_off(page, g, j % page_size, H_kv, page_size, d);
                double acc = 0.0;
                for (int e = 0; e < d; ++e) acc += qr[e] * oracle_bf16_to_double(kj[e]);
                sc[j] = acc * scale;
                if (sc[j] > m) m = sc[j];
            }
            double denom = 0.0;
            for (int e = 0; e < d; ++e) o[e] = 0.0;
            for (int j = 0; j <= p; ++j) {
                double wj = exp(sc[j] - m);
                denom += wj;
                int page = kv_page_indices[kv_page_indptr[r] + j / page_size];
                const uint16_t* vj = v_cache + cache_off(page, g, j % page_size, H_kv, page_size, d);
                for (int e = 0; e < d; ++e) o[e] += wj * oracle_bf16_to_double(vj[e]);
            }
            for (int e = 0; e < d; ++e) o[e] /= denom;
            if (lse) lse[w] = m + log(denom);
        }
        free(qx);
        free(sc);
    }
}

void oracle_append(int n_sched, const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                   const int32_t* kv_page_indices, const int32_t* kv_last_page_len,
                   const uint16_t* k, const uint16_t* v, int H_kv, int d, int page_size,
                   double rope_base, uint16_t* k_cache, uint16_t* v_cache) {
    oracle_append_styled(n_sched, qo_indptr, kv_page_indptr, kv_page_indices, kv_last_page_len, k, v, H_kv, d,
                         page_size, rope_base, 0, k_cache, v_cache);
}
void oracle_attend(int n_sched, const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                   const int32_t* kv_page_indices, const int32_t* kv_last_page_len,
                   const uint16_t* q, int H_q, int H_kv, int d, int page_size, double rope_base,
                   const uint16_t* k_cache, const uint16_t* v_cache,
                   int n_pairs, const int32_t* row_t, const int32_t* row_hq,
                   double* out, double* lse) {
    oracle_attend_styled(n_sched, qo_indptr, kv_page_indptr, kv_page_indices, kv_last_page_len, q, H_q, H_kv, d,
                         page_size, rope_base, 0, k_cache, v_cache, n_pairs, row_t, row_hq, out, lse);
}

/* ------------------------------------------------------------------------- */
/* Counters                                                                   */
/* ------------------------------------------------------------------------- */

/* Query-key pairs the step scores: sum over requests of n*h + n(n+1)/2 (each
 * new query at position h+i sees h+i+1 keys).  For one prompt of length L split
 * at any boundaries this sums to L(L+1)/2, [SS] §"为什么总 FLOPs 近似不变". */
int64_t oracle_pairs(int n_sched, const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                     const int32_t* kv_last_page_len, int page_size) {
    int64_t total = 0;
    for (int s = 0; s < n_sched; ++s) {
        int64_t n = qo_indptr[s + 1] - qo_indptr[s];
        int np = kv_page_indptr[s + 1] - kv_page_indptr[s];
        int64_t kv_len = (int64_t)(np - 1) * page_size + kv_last_page_len[s];
        int64_t h = kv_len - n;
        for (int64_t i = 0; i < n; ++i) total += h + i + 1;
    }
    return total;
}

/* History tokens re-read by multi-token chunks this step: sum of h over the
 * requests with more than one new token. */
int64_t oracle_reread_tokens(int n_sched, const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                             const int32_t* kv_last_page_len, int page_size) {
    int64_t total = 0;
    for (int s = 0; s < n_sched; ++s) {
        int64_t n = qo_indptr[s + 1] - qo_indptr[s];
        if (n <= 1) continue;
        int np = kv_page_indptr[s + 1] - kv_page_indptr[s];
        int64_t kv_len = (int64_t)(np - 1) * page_size + kv_last_page_len[s];
        total += kv_len - n;
    }
    return total;
}

/* Threads the OpenMP loops use from now on (timing on one core). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
