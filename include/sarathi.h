/*
 * sarathi.h -- C ABI of libsarathi: the mixed-batch paged-attention step of
 * chunked prefill with stall-free batching, on one sm_103a GPU.
 *
 * Two calls make the step:
 *   sarathi_plan        (host only) fills a per-iteration token budget --
 *                       decodes first, then in-progress prefill chunks, then new
 *                       prefills -- and emits the ragged-batch metadata
 *                       qo_indptr / kv_page_indptr / kv_page_indices /
 *                       kv_last_page_len plus the kernel's work list, packed in
 *                       one int32 buffer for a single host-to-device copy.
 *   sarathi_mixed_attn  enqueues ONE kernel on the caller's stream: RoPE at
 *                       absolute positions and K/V append into pages, causal
 *                       attention of every prefill chunk over history pages plus
 *                       the chunk, split-KV decode attention and its
 *                       log-sum-exp merge.
 *
 * Conventions for every function here:
 *   - returns an int32 sarathi_status; 0 is success; nothing throws;
 *   - sarathi_last_error() gives a thread-local message for the last failure;
 *   - the caller owns every buffer (host and device); the library keeps no
 *     device allocation across calls;
 *   - "device pointer" means CUDA global memory of the current device.
 *
 * Sources (pages, by title):
 *   [SS] "Sarathi-Serve 完全拆解：分块 Prefill 与无停顿批处理如何兼顾吞吐和尾延迟"
 *   [CP] "Chunked Prefill 与 PD 分离：切片混批，还是拆开两个池"
 *   [ST] "分块预填充与 Stall-free 调度：把 LLM 推理的吞吐-延迟权衡算清楚"
 *   [SA] "Sarathi：让解码搭上 prefill 的顺风车"
 */
#ifndef SARATHI_H_
#define SARATHI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SARATHI_ABI_VERSION 6
/* int32 words of one kernel work item in the packed plan.  Items are kernel
 * bookkeeping: their layout is private to the library and may change with
 * SARATHI_ABI_VERSION; callers copy the packed plan as a whole. */
#define SARATHI_ITEM_INTS 24

/* Status codes. */
#define SARATHI_OK 0
#define SARATHI_ERR_INVALID_ARG 1          /* bad pointer, size, state or metadata */
#define SARATHI_ERR_CAPACITY 2             /* block table too short or buffer too small */
#define SARATHI_WARN_OVER_BUDGET_DECODES 3 /* decodes alone exceed the budget; output valid */
#define SARATHI_ERR_CUDA 4                 /* a CUDA runtime/driver call failed */
#define SARATHI_ERR_UNSUPPORTED 5          /* head_dim / group size / page size not built */
#define SARATHI_ERR_DEVICE_CHECK 6         /* the kernel flagged an error (see below) */

/* Request states, [CP] §3.1: running decodes, in-progress prefills, new requests. */
#define SARATHI_DECODE 0
#define SARATHI_PREFILL_RUNNING 1
#define SARATHI_PREFILL_WAITING 2

/* One request as the scheduler sees it ([SS] §"分块不等于截断上下文": processed
 * prompt length, block table).  The plan never writes to it; after the step the
 * caller advances num_computed by the scheduled num_new, and a request whose
 * last chunk ran becomes SARATHI_DECODE ([SS] §"一个 512-token 预算的例子"). */
typedef struct sarathi_request {
    int32_t state;          /* SARATHI_DECODE / _PREFILL_RUNNING / _PREFILL_WAITING   */
    int32_t prompt_len;     /* prefill: total prompt tokens; decode: ignored         */
    int32_t num_computed;   /* h: tokens already in the KV cache                      */
    int32_t num_pages;      /* length of the block table                              */
    const int32_t* pages;   /* host pointer: physical page ids in logical order       */
} sarathi_request;

/* Model shape of the attention layer.  Built: page_size 16, head_dim 64 or 128,
 * num_heads_q a multiple of num_heads_kv with group size 1..16. */
typedef struct sarathi_shape {
    int32_t num_heads_q;
    int32_t num_heads_kv;
    int32_t head_dim;
    int32_t page_size;
} sarathi_shape;

/* What sarathi_plan produced.  Offsets count int32 elements from the start of
 * the packed buffer; the same offsets hold for its device copy. */
typedef struct sarathi_plan_info {
    int32_t n_sched;            /* scheduled requests = rows of qo_indptr - 1          */
    int32_t num_decodes;        /* the first num_decodes scheduled rows are decodes   */
    int32_t num_tokens;         /* T = qo_indptr[n_sched]                              */
    int32_t nnz_pages;          /* entries of kv_page_indices                           */
    int32_t n_items;            /* kernel work items                                    */
    int32_t n_partials;         /* split-KV partial slots the kernel writes             */
    int32_t n_merge;            /* split-KV merge groups                                */
    int32_t max_kv_len;         /* longest h + n in the batch (RoPE table must cover it) */
    int64_t pairs;              /* query-key pairs scored: sum n*h + n(n+1)/2           */
    int64_t history_tokens;     /* sum of h over scheduled requests (KV read once each)  */
    int32_t off_req_index;      /* [n_sched] caller index of each scheduled request     */
    int32_t off_num_new;        /* [n_sched] new tokens this step                       */
    int32_t off_last_chunk;     /* [n_sched] 1 if sampling is valid for the row         */
    int32_t off_qo_indptr;      /* [n_sched+1]                                          */
    int32_t off_kv_page_indptr; /* [n_sched+1]                                          */
    int32_t off_kv_page_indices;/* [nnz_pages]                                          */
    int32_t off_kv_last_page_len;/* [n_sched] in 1..page_size                            */
    int32_t off_req_aux;        /* [n_sched] kernel bookkeeping (first K/V ready flag)  */
    int32_t off_items;          /* [n_items][SARATHI_ITEM_INTS] kernel work list         */
    int32_t packed_ints;        /* int32 elements to copy to the device                  */
    int64_t workspace_bytes;    /* device workspace sarathi_mixed_attn needs             */
    int32_t n_first;            /* the work list's first n_first items form the first    */
                                /*   queue (prefill tiles), the rest the second (decodes) */
    int32_t first_sms;          /* CTAs that take from the first queue before the second */
} sarathi_plan_info;

/* Upper bounds for the buffers of sarathi_plan on this request set at ANY
 * budget <= token_budget: host packed buffer bytes and device workspace bytes.
 * Either output pointer may be NULL. */
int32_t sarathi_plan_bounds(const sarathi_request* reqs, int32_t n_reqs, int32_t token_budget,
                            const sarathi_shape* shape, int32_t num_sms,
                            size_t* host_buf_bytes, size_t* device_workspace_bytes);

/* Build the step's batch.  Budget order ([CP] §3.1; [ST] §六·补二; [SS]
 * §"一个 512-token 预算的例子"): every SARATHI_DECODE request gets 1 token (in
 * caller order), then every SARATHI_PREFILL_RUNNING request gets
 * min(prompt_len - num_computed, budget left), then every
 * SARATHI_PREFILL_WAITING request likewise; requests that get 0 are left out.
 * When the decodes alone exceed the budget all of them are still scheduled,
 * prefills get nothing and the return is SARATHI_WARN_OVER_BUDGET_DECODES
 * (decodes never stall, [CP] §3.1).
 * Metadata ([SS] §"混合批不是…"): for scheduled row s with history h and n new
 * tokens, kv_len = h + n, its pages are the first ceil(kv_len/page_size) entries
 * of the block table, and kv_last_page_len = kv_len - page_size*(pages-1).
 * num_sms sizes the split-KV work (pass the device's SM count).
 * host_buf: caller-allocated, >= host_buf_bytes, 4-byte aligned.
 * Errors: INVALID_ARG (bad state, h > prompt_len, budget <= 0, NULL pointers),
 * CAPACITY (a block table too short, or host_buf too small: info->packed_ints
 * then holds the size needed), UNSUPPORTED (shape not built). */
int32_t sarathi_plan(const sarathi_request* reqs, int32_t n_reqs, int32_t token_budget,
                     const sarathi_shape* shape, int32_t num_sms,
                     int32_t* host_buf, size_t host_buf_bytes, sarathi_plan_info* info);

/* Batch policies for sarathi_plan_ex. */
#define SARATHI_POLICY_STALL_FREE 0     /* the rule of sarathi_plan above              */
#define SARATHI_POLICY_DECODE_MAXIMAL 1 /* [SA] §"Decode-maximal batching：顺车的账本"  */

typedef struct sarathi_plan_policy {
    int32_t kind;          /* SARATHI_POLICY_*                                          */
    int32_t token_budget;  /* stall-free: tokens per step; decode-maximal: chunk size  */
    int32_t max_batch;     /* decode-maximal: B, requests per batch (0 = no limit);    */
                           /*   stall-free: must be 0                                  */
    int32_t chunk_align;   /* >= 1: a chunk that does not finish its prompt is cut     */
                           /*   down to a multiple of this ([SS] §"257 为什么可能比 256 */
                           /*   慢 32%": candidate sizes aligned to 32); 1 = no cut     */
} sarathi_plan_policy;

/* sarathi_plan with a choice of batch policy.
 * SARATHI_POLICY_STALL_FREE: exactly sarathi_plan, except that chunks are
 *   aligned as chunk_align says (a request whose aligned share is 0 is left out).
 * SARATHI_POLICY_DECODE_MAXIMAL ([SA] §"Decode-maximal batching：顺车的账本"):
 *   ONE prefill chunk of min(token_budget, prompt_len - num_computed) tokens,
 *   aligned, from the first SARATHI_PREFILL_RUNNING request with tokens left,
 *   else the first SARATHI_PREFILL_WAITING one; then as many SARATHI_DECODE
 *   requests as fit, in caller order: at most max_batch - 1 next to a chunk,
 *   max_batch without one (0: all).  Decodes that do not fit are left out
 *   for this step.  Rows are listed decodes first, then the chunk.
 * Metadata, buffers and errors are those of sarathi_plan (INVALID_ARG also for
 * an unknown kind, chunk_align < 1, max_batch < 0, or max_batch != 0 with
 * stall-free).  sarathi_plan_bounds with token_budget = policy->token_budget
 * bounds the buffers of either policy. */
int32_t sarathi_plan_ex(const sarathi_request* reqs, int32_t n_reqs, const sarathi_plan_policy* policy,
                        const sarathi_shape* shape, int32_t num_sms,
                        int32_t* host_buf, size_t host_buf_bytes, sarathi_plan_info* info);

/* One of the two metadata sets of a step, as an executor that runs prefill
 * and decode attention separately builds them ([SS] §"混合批不是把两类注意力强行
 * 做成同一个形状": separate qo_indptr / kv_page_indptr / kv_page_indices /
 * kv_last_page_len for prefill and for decode requests).  Offsets count int32
 * elements of the caller's output buffer. */
typedef struct sarathi_meta_set {
    int32_t rows;                /* requests in the set                                 */
    int32_t tokens;              /* query rows: qo_indptr[rows]                          */
    int32_t token_offset;        /* the set's first query row in the step's q / out     */
    int32_t nnz_pages;           /* kv_page_indptr[rows]                                 */
    int32_t first_row;           /* the set's first row in the combined plan            */
    int32_t off_qo_indptr;       /* [rows + 1], from 0                                   */
    int32_t off_kv_page_indptr;  /* [rows + 1], from 0                                   */
    int32_t off_kv_page_indices; /* [nnz_pages]                                          */
    int32_t off_kv_last_page_len;/* [rows]                                               */
} sarathi_meta_set;

/* Split a plan's metadata into its decode set (the first num_decodes rows) and
 * its prefill set (the rest, chunks in plan order).  host_buf / info: as
 * returned by sarathi_plan or sarathi_plan_ex.  out: >= 4 * (3 * n_sched + 4 +
 * nnz_pages) bytes, 4-byte aligned.  Host only.  Errors: INVALID_ARG (NULL
 * pointer), CAPACITY (out too small). */
int32_t sarathi_split_metadata(const sarathi_plan_info* info, const int32_t* host_buf, int32_t* out,
                               size_t out_bytes, sarathi_meta_set* decode, sarathi_meta_set* prefill);

/* Apply a step's plan to the requests ([SS] §"一个 512-token 预算的例子";
 * [CP] §3.1): every scheduled request's num_computed grows by its num_new; a
 * prefill whose last chunk ran becomes SARATHI_DECODE, one with prompt left
 * becomes SARATHI_PREFILL_RUNNING.  reqs: the array (same order) the plan was
 * made from, updated in place.  host_buf / info: the packed plan and the info
 * that sarathi_plan or sarathi_plan_ex returned.  Host only.
 * Errors: INVALID_ARG (NULL pointer, a row index out of range, a chunk past
 * its prompt); on error reqs may be partly updated. */
int32_t sarathi_advance(sarathi_request* reqs, int32_t n_reqs, const sarathi_plan_info* info,
                        const int32_t* host_buf);

/* Fill the RoPE table on the device: {cos(p*f_j), sin(p*f_j)} in fp64 for
 * p < max_pos, j < head_dim/2, f_j = rope_theta^(-2j/head_dim) (rotate-half
 * RoPE at absolute positions, [SS] §"分块不等于截断上下文"), followed by the same
 * values split into float pairs (hi + lo) for the kernel's fp32 fast path.
 * table: device pointer to 2*max_pos*head_dim doubles (16*max_pos*head_dim
 * bytes): double[max_pos][head_dim/2][2] {cos, sin}, then
 * float[max_pos][4][head_dim/2]: per position the planes cos_hi, sin_hi,
 * cos_lo, sin_lo over the pairs (cos = cos_hi + cos_lo, likewise sin; the
 * hi planes first, so that one tensor-map box fetches them for many rows).
 * head_dim must be a multiple of 16 (UNSUPPORTED otherwise).
 * Asynchronous on `cuda_stream` (a cudaStream_t; NULL = legacy default stream). */
int32_t sarathi_rope_table(double* table, int32_t max_pos, int32_t head_dim, double rope_theta,
                           void* cuda_stream);

/* RoPE pairing of the head dimensions; pair j turns by pos * theta^(-2j/d) in
 * both.  Rotate-half pairs (x[j], x[j + d/2]) (the reading of the pages used
 * by default); interleaved pairs (x[2j], x[2j+1]), the pairing of the
 * original RoPE formulation (Su et al., RoFormer). */
#define SARATHI_ROPE_ROTATE_HALF 0
#define SARATHI_ROPE_INTERLEAVED 1

/* Arguments of one step.  All pointers are device pointers unless noted. */
typedef struct sarathi_attn_args {
    const void* q;              /* bf16 [T][H_q][d]  new tokens' queries, before RoPE   */
    const void* k;              /* bf16 [T][H_kv][d] new tokens' keys, before RoPE      */
    const void* v;              /* bf16 [T][H_kv][d] new tokens' values                 */
    void* k_cache;              /* bf16 [num_pages][H_kv][page_size][d], rotated keys    */
    void* v_cache;              /* bf16 [num_pages][H_kv][page_size][d]                 */
    void* out;                  /* bf16 [T][H_q][d] attention outputs                   */
    const int32_t* plan;        /* device copy of the packed plan buffer                */
    const sarathi_plan_info* info; /* HOST pointer: the info sarathi_plan returned      */
    const double* rope_table;   /* from sarathi_rope_table, max_pos >= info->max_kv_len, */
                                /*   16-byte aligned                                    */
    int32_t rope_max_pos;
    int32_t num_pages;          /* pages in each cache pool                             */
    void* workspace;            /* >= info->workspace_bytes, 256-byte aligned, ZEROED    */
    int64_t workspace_bytes;    /*   once before first use; every launch leaves it so   */
    sarathi_shape shape;
    float sm_scale;             /* softmax scale, normally 1/sqrt(head_dim)             */
    int32_t rope_style;         /* SARATHI_ROPE_ROTATE_HALF or SARATHI_ROPE_INTERLEAVED */
    const int32_t* plan_host;   /* optional HOST copy of the packed plan (pinned memory */
                                /*   for an asynchronous copy): when not NULL the call  */
                                /*   first enqueues its copy into `plan` (packed_ints    */
                                /*   int32), so that it must not change until the copy   */
                                /*   has run on the stream; NULL: `plan` already holds it */
} sarathi_attn_args;

/* Enqueue the step on `cuda_stream` (a cudaStream_t): one kernel launch, no
 * host synchronisation, no allocation.  Writes the new tokens' rotated K and V
 * into their pages and every out row.  The history pages must already hold
 * the earlier tokens of each request.  Attention for row i of a request with
 * history h: softmax over keys 0..h+i of RoPE(q_i, h+i).K_j * sm_scale,
 * weights applied to V_j ([SS] §"分块不等于截断上下文").  Keys are the bf16
 * pages; scores and sums in fp32.
 * q, k, v, out, k_cache, v_cache, plan and rope_table must be 16-byte aligned.
 * Launches using one workspace must not overlap in time.  A launch that hits a
 * device-side check (a wait that ran out, a page id outside the pool) sets an
 * error word in the workspace; read it with sarathi_workspace_status.
 * Errors (before anything is enqueued): INVALID_ARG, CAPACITY (workspace or
 * RoPE table too small), UNSUPPORTED, CUDA. */
int32_t sarathi_mixed_attn(const sarathi_attn_args* args, void* cuda_stream);

/* Host side of one step for sarathi_mixed_attn_host.  q_host, k_host, v_host
 * and out_host are HOST pointers, in the layouts of sarathi_attn_args' q, k, v
 * and out (num_tokens = info->num_tokens rows); page-locked memory makes the
 * copies asynchronous, pageable memory makes the call wait for them.  The
 * events are cudaEvent_t handles owned by the caller, or NULL. */
typedef struct sarathi_host_io {
    const void* q_host;         /* bf16 [T][H_q][d]                                       */
    const void* k_host;         /* bf16 [T][H_kv][d]                                      */
    const void* v_host;         /* bf16 [T][H_kv][d]                                      */
    void* out_host;             /* bf16 [T][H_q][d], written when the stream reaches it   */
    void* wait_event;           /* the kernel starts after this event (the step before:   */
                                /*   it wrote the pages this step reads), or NULL         */
    void* done_event;           /* recorded right after the kernel, or NULL               */
} sarathi_host_io;

/* sarathi_mixed_attn from host buffers, end to end on `cuda_stream`: copies
 * q, k, v from the host into args->q, k, v (device), the plan from
 * args->plan_host into args->plan when plan_host is set, waits for
 * io->wait_event, runs the step kernel, records io->done_event, and copies
 * args->out into io->out_host.  The copies in ahead of the wait let a caller
 * that alternates two streams (each with its own q, k, v, out, plan buffers,
 * one workspace shared) overlap one step's copies with the other's kernel,
 * passing each step the event of the step before it.  The host must not
 * change q_host, k_host, v_host or plan_host, nor read out_host, before the
 * stream has passed them.  The pages define the step itself (see
 * sarathi_mixed_attn); this host-side packaging is the library's own.
 * Errors: as sarathi_mixed_attn, and INVALID_ARG for a NULL io or host
 * pointer, all before anything is enqueued; a CUDA error from one of the
 * enqueued calls returns SARATHI_ERR_CUDA with the calls before it already
 * enqueued. */
int32_t sarathi_mixed_attn_host(const sarathi_attn_args* args, const sarathi_host_io* io, void* cuda_stream);

/* The same step as sarathi_mixed_attn, for callers that cannot allocate device
 * memory when they run it -- for example a plugin inside a process whose
 * allocator already owns the GPU's memory, or a serving loop that allows no
 * allocation after start-up.  The pages have no counterpart to this call.
 * The scratch (args->workspace and args->workspace_bytes are ignored) comes
 * from an 8 MiB array inside the library that every GPU loading the library
 * holds until the process exits; a batch whose info->workspace_bytes exceeds
 * 8 MiB is rejected with SARATHI_ERR_CAPACITY before anything is enqueued.
 * The call allocates nothing: it clears the array's counters with
 * cudaMemsetAsync on `cuda_stream` and enqueues the step kernel.  The first
 * call on each device looks up the array's device address; with lazy module
 * loading (the CUDA default) that first lookup is also when the device
 * reserves the array, so make the first call on each device before a host
 * allocator claims the GPU's memory, and before any stream capture.  The
 * address is kept per device index for the life of the process: do not use
 * this call after cudaDeviceReset on that device.  All calls share the one
 * array, so calls whose work overlaps on the GPU (other streams, other
 * threads) race and give wrong results.  The device error word lives in the
 * shared array: a bounded wait that runs out or a page id outside the pool
 * leaves the outputs and pages partly written while the call still returned
 * SARATHI_OK; read the word with sarathi_noalloc_status (the next call clears
 * the array's counters itself).
 * Errors, all before anything is enqueued: CAPACITY when
 * info->workspace_bytes exceeds the array; INVALID_ARG when the plan info is
 * inconsistent (n_sched <= 0, negative counts, or counters and partial slots
 * larger than info->workspace_bytes); then as sarathi_mixed_attn. */
int32_t sarathi_mixed_attn_noalloc(const sarathi_attn_args* args, void* cuda_stream);

/* sarathi_workspace_status for the built-in array of sarathi_mixed_attn_noalloc
 * on the current device: synchronise `cuda_stream`, then read and clear the
 * device error word of the last call there.  Allocates nothing.  Returns
 * SARATHI_OK, SARATHI_ERR_DEVICE_CHECK when the word was nonzero
 * (*device_error: 1 a bounded wait ran out, 2 a bounds check failed), or
 * SARATHI_ERR_CUDA / INVALID_ARG. */
int32_t sarathi_noalloc_status(void* cuda_stream, int32_t* device_error);

/* The Q/K/V projection of a step's tokens as ONE GEMM over the concatenated
 * ragged batch ([SA] §"Decode-maximal batching：顺车的账本": the linear layers of
 * the prefill chunk and of the decodes run as one matrix product, so the
 * weights are read once for both; [SS] §"混合批不是把两类注意力强行做成同一个形状":
 * the linear-layer inputs are concatenated along the token dimension).
 *   Y = X W^T, X: bf16 [tokens][hidden], W: bf16 [N][hidden], N = (H_q + 2 H_kv) d;
 *   q[t][h][:] = Y[t][h d ...], k = the next H_kv d columns, v the last H_kv d.
 * fp32 accumulation, bf16 outputs (round to nearest even).  The outputs are the
 * q / k / v of sarathi_attn_args for the same token order.  All pointers are
 * device pointers, 16-byte aligned. */
typedef struct sarathi_qkv_args {
    const void* x;          /* bf16 [tokens][hidden] hidden states, plan token order    */
    const void* w;          /* bf16 [(H_q + 2 H_kv) d][hidden] stacked Q, K, V weights   */
    void* q;                /* bf16 [tokens][H_q][d]                                     */
    void* k;                /* bf16 [tokens][H_kv][d]                                    */
    void* v;                /* bf16 [tokens][H_kv][d]                                    */
    int32_t tokens;         /* >= 1                                                      */
    int32_t hidden;         /* multiple of 64                                            */
    sarathi_shape shape;    /* num_heads_q, num_heads_kv, head_dim (multiple of 32)      */
    void* workspace;        /* >= 256 bytes, ZEROED once; holds the device error word   */
} sarathi_qkv_args;

/* Enqueue the projection (one kernel) on `cuda_stream`.  A bounded wait that
 * runs out sets the workspace's error word (read it with
 * sarathi_workspace_status).  Errors: INVALID_ARG, CUDA. */
int32_t sarathi_qkv_proj(const sarathi_qkv_args* args, void* cuda_stream);

/* Synchronise `cuda_stream`, then read and clear the device error word of a
 * workspace.  *device_error receives 0 or the kernel's error code (1: a
 * bounded wait ran out; 2: a bounds check failed).  Returns SARATHI_OK, or
 * SARATHI_ERR_DEVICE_CHECK when the word was nonzero (the rest of the
 * workspace must then be zeroed again before the next launch), or
 * SARATHI_ERR_CUDA. */
int32_t sarathi_workspace_status(void* workspace, void* cuda_stream, int32_t* device_error);

/* Thread-local text of the last error; never NULL. */
const char* sarathi_last_error(void);

/* SARATHI_ABI_VERSION of the loaded library. */
int32_t sarathi_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SARATHI_H_ */
