// mixed_attn.cu -- the step kernel of libsarathi (sm_103a) and its launcher.
//
// One persistent launch runs the whole mixed-batch attention step that chunked
// prefill with stall-free batching produces ("Sarathi-Serve 完全拆解", §"混合批不是
// 把两类注意力强行做成同一个形状": one ragged batch, attention split back per
// request through qo_indptr / kv_page_indptr / kv_page_indices /
// kv_last_page_len).  CTAs pull work items from the planner's two queues
// (prefill tiles; APPEND items and decode splits) through an atomic head
// counter each, longest items first; CTAs below first_sms start on the first
// queue, the others on the second, and each moves to the other queue once its
// own is empty:
//
//   APPEND   new prefill tokens of one 128-position block, 2 kv heads: K rotated
//            at its ABSOLUTE position and rounded once to bf16 as from the fp64
//            value, V copied, both into the pages that hold the positions
//            ("Sarathi-Serve 完全拆解", §"分块不等于截断上下文": RoPE never restarts
//            per chunk; the chunk's K/V land in the paged cache); then a ready
//            flag for the block.
//   PREFILL  one tile of up to 128 query rows (token x q-head of one GQA group)
//            of a chunk: causal attention over every history page plus the
//            chunk's own keys (ibid.: o_i = sum_{j<=i} softmax(q_i.k_j/sqrt d) v_j),
//            128-key blocks streamed into shared memory with TMA; a block of the
//            chunk's own keys waits (bounded) for its ready flag.  The last tiles
//            of a step without decodes may come as key pieces, merged by
//            log-sum-exp by the last piece to arrive.
//   DECODE   one split of a decode's pages for two kv heads (four warps a
//            head): per-warp TMA page pipelines, warp-level MMA for the GQA
//            group, online softmax, in-CTA merge per head, and across splits a
//            log-sum-exp merge done by the last split to arrive (atomic ticket,
//            no spinning).  The split that owns the last page also appends the
//            decode token's K/V.
//
// No CTA waits on a CTA that took a later item, and the only cross-CTA wait
// (a PREFILL block on its APPEND item's ready flag; the APPEND items lead the
// second queue, or, in a step without decodes, the one queue or all of the
// second, and some CTA starts on them at launch) is bounded by a timer; a wait
// that runs out sets an error word in the workspace.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "sarathi.h"
#include "sarathi_internal.h"

namespace sarathi {

// ----------------------------------------------------------------------------
// Kernel parameters
// ----------------------------------------------------------------------------
struct KParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    __nv_bfloat16* k_cache;
    __nv_bfloat16* v_cache;
    __nv_bfloat16* out;
    const int32_t* plan;
    int off_qo, off_kvp, off_kvi, off_last, off_aux, off_items;
    int n_items, n_sched;
    int n_flags;              // ready-flag words after the header (merge tickets follow them)
    int n_first, first_sms;   // the work list's two queues (see the kernel's claim loop)
    const double2* rope;  // [max_pos][d/2] {cos, sin} in fp64
    const float* ropef;   // [max_pos][4][d/2]: cos_hi, sin_hi, cos_lo, sin_lo rows (cos = hi + lo to ~2^-48)
    int rope_max_pos;
    int32_t* ws_int;      // header, append counters, merge tickets
    float* ws_part;       // split partials
    int Hq, Hkv, group, num_pages;
    float scale_log2;     // sm_scale * log2(e)
    int slot_floats;
};

constexpr int kThreads = 384;                                  // 12 warps
constexpr int kDecWarps = 8;                                   // warps that stream decode pages
constexpr int kDecStages = 3;                                  // per-warp page ring
constexpr int kPageHalfBytes = kPage * 128;                    // 16 rows x 64 bf16
constexpr int kDecStageBytes = 2 * 2 * kPageHalfBytes;         // K+V page-head, d=128
constexpr int kSmemStages = kDecWarps * kDecStages * kDecStageBytes;  // 192 KB
constexpr int kSmemDecQ = kSmemStages;                         // 16 x 128 bf16
constexpr int kSmemStash = kSmemDecQ + 8192;                   // new K/V of a decode item's heads
constexpr int kSmemBars = kSmemStash + 1024;                  // mbarriers, initialised once
constexpr int kDecBar0 = 0;                                    // [warp][stage] decode rings
constexpr int kSmemBytes = kSmemBars + 512;
constexpr int kSmemAlloc = kSmemBytes + 1024;                  // + alignment slack
static_assert(kDecWarps * 16 * 128 * 4 + 2 * kDecWarps * 16 * 4 <= kSmemStages, "merge scratch");
static_assert(kSmemAlloc <= 227 * 1024, "shared memory per CTA");

constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s bound on any wait
constexpr uint32_t kWaitSleepNs = 200000u;             // longest sleep of one suspended try-wait

// ----------------------------------------------------------------------------
// PTX helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// The same with a suspend-time hint: a thread whose phase is not complete
// sleeps (up to the hint, in ns) until it completes instead of spinning, so a
// waiting thread takes no issue slots from the warps that share its SM
// sub-partition.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kWaitSleepNs)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// 3-D box: coordinates {x, y, z} innermost first.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
// 5-D box: coordinates {x0..x4} innermost first.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int x0, int x1, int x2, int x3,
                                            int x4, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, "
        "%6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x0), "r"(x1), "r"(x2), "r"(x3), "r"(x4), "r"(bar)
        : "memory");
}
// Plain (untiled) bulk copy global -> shared; both addresses 16-byte aligned,
// size a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }
// 2^x with the MUFU approximation (flushes subnormals; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Three-input max and two-lane fp32 FMA / add (one instruction each on
// sm_103a): the prefill softmax is bound by instruction issue.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
          "l"(*reinterpret_cast<uint64_t*>(&c)));
    return *reinterpret_cast<float2*>(&r);
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;"
        : "=l"(r)
        : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
    return *reinterpret_cast<float2*>(&r);
}

// Round a double to bf16 in ONE rounding (ties to even): round to float with
// round-to-odd (truncate, then force the last bit to 1 when inexact), then
// round that float to nearest-even bf16.  Round-to-odd at 16 extra bits makes
// the second rounding exact (Boldo & Melquiond, "Emulation of FMA and correctly
// rounded sums: proved algorithms using rounding to odd", IEEE TC 2008).
__device__ __forceinline__ uint16_t bf16_from_double(double x) {
    if (x != x) return 0x7FC0;
    float f = __double2float_rz(x);
    uint32_t u = __float_as_uint(f);
    if ((double)f != x) u |= 1u;
    if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16);  // +-inf stays
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// Shared-memory tiles use the 128-byte swizzle TMA writes: a tile is stored as
// (d/64) column halves of ROWS x 128 B, and the 16-byte chunk c of row r sits
// at chunk c ^ (r & 7).  Byte offset of element (row, col):
__device__ __forceinline__ uint32_t sw128_off(int rows, int row, int col) {
    int half = col >> 6, c = (col & 63) >> 3, w = col & 7;
    return (uint32_t)(half * rows * 128 + row * 128 + ((c ^ (row & 7)) << 4) + w * 2);
}
// Byte offset of the 16-byte chunk (row, chunk) where chunk counts 8 columns.
__device__ __forceinline__ uint32_t sw128_chunk(int rows, int row, int chunk) {
    int half = chunk >> 3, c = chunk & 7;
    return (uint32_t)(half * rows * 128 + row * 128 + ((c ^ (row & 7)) << 4));
}

// ----------------------------------------------------------------------------
// Error / abort
// ----------------------------------------------------------------------------
__device__ __forceinline__ void raise_error(const KParams& P, int code, int detail, int* s_abort) {
    if (atomicCAS(&P.ws_int[2], 0, code) == 0) P.ws_int[3] = detail;
    *(volatile int*)s_abort = 1;
}

// Bounded wait on an mbarrier phase; returns false (and flags the CTA) on
// timeout, recording the work item, the thread and the barrier's raw state in
// header words 3..11 for the host to read.  SLEEP: the thread suspends while it
// waits (for threads that wait long and share an SM sub-partition with warps
// that compute); otherwise it polls, which wakes sooner.
template <bool SLEEP>
__device__ __noinline__ bool mbar_wait_slow(const KParams& P, uint32_t bar, uint32_t parity, int* s_abort,
                                            int detail, const int* it) {
    if (!SLEEP)
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!(SLEEP ? mbar_try_wait_sleep(bar, parity) : mbar_try_wait(bar, parity))) {
        if (*(volatile int*)s_abort) return false;
        if (globaltimer() - t0 > kWaitNs) {
            if (atomicCAS(&P.ws_int[2], 0, kErrWait) == 0) {
                uint64_t raw;
                asm volatile("ld.shared.b64 %0, [%1];" : "=l"(raw) : "r"(bar) : "memory");
                P.ws_int[3] = detail;
                for (int i = 0; i < 5; ++i) P.ws_int[4 + i] = it[i];
                P.ws_int[9] = (int)threadIdx.x | ((int)parity << 16);
                P.ws_int[10] = (int)(uint32_t)raw;
                P.ws_int[11] = (int)(uint32_t)(raw >> 32);
            }
            *(volatile int*)s_abort = 1;
            return false;
        }
    }
    return true;
}
template <bool SLEEP = false>
__device__ __forceinline__ bool mbar_wait_bounded(const KParams& P, uint32_t bar, uint32_t parity, int* s_abort,
                                                  int detail, const int* it) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow<SLEEP>(P, bar, parity, s_abort, detail, it);
}

struct Row {
    int qo0, n, kvp0, np, kv_len, h;
};
// The row's geometry travels in the item (a copy of its metadata), so the
// first page can be fetched one load after the item is claimed.
__device__ __forceinline__ Row row_geom(const int* it) {
    Row r;
    r.qo0 = it[kQo0];
    r.n = it[kNNew];
    r.kvp0 = it[kKvp0];
    r.np = it[kNp];
    r.kv_len = it[kKvLen];
    r.h = r.kv_len - r.n;
    return r;
}

// Physical page id of a request-local page, checked against the pool.
__device__ __forceinline__ int checked_page(const KParams& P, int page, int* s_abort) {
    if (page < 0 || page >= P.num_pages) {
        raise_error(P, kErrBounds, page, s_abort);
        return 0;
    }
    return page;
}
__device__ __forceinline__ int page_id(const KParams& P, const Row& R, int lp, int* s_abort) {
    const int page = P.plan[P.off_kvi + R.kvp0 + lp];
    if (page < 0 || page >= P.num_pages) {
        raise_error(P, kErrBounds, page, s_abort);
        return 0;
    }
    return page;
}

// bf16 of y = a*p + b*q where the fp64 evaluation rounds each product and
// the sum once (no contraction) and then rounds once to bf16 -- the RoPE of a
// key at an absolute position (y0 = x0 cos - x1 sin, y1 = x1 cos + x0 sin).
//
// Fast path in fp32: with p = p_hi + p_lo, q = q_hi + q_lo, the products
// a*p_hi and b*q_hi are split exactly by FMA (a, b have 8 significant bits)
// and summed by TwoSum, so y = S + small with an error below 2^-46 (|a p| +
// |b q|).  The fp64 evaluation differs from the exact value by at most about
// 2^-52 (|a p| + |b q|).  When S + small lies farther than 2^-34 (|a p| +
// |b q|) from both bf16 rounding boundaries around its nearest bf16 value w,
// every value within those errors rounds to w, so w is the answer.  Otherwise
// (about one element in 10^8) the fp64 evaluation runs as written.  A cheaper
// single-FMA test (below) settles most elements before the double-float step.
__device__ __forceinline__ uint16_t rope_bf16(float a, float b, float p_hi, float p_lo, float q_hi, float q_lo,
                                             const double2* pq) {
    // First, one fused multiply-add: u = fl(a p_hi + fl(b q_hi)).  With
    // |p - p_hi| <= 2^-24 |p_hi| (and the same for q), |u - y| <= 3.1 2^-24
    // (|a p_hi| + |b q_hi|) for the fp64 value y, i.e. at most 1.55 m / 2^E
    // units of u's last place (2^E the power of two at or below |u|, m that
    // magnitude sum).  The bf16 rounding boundaries lie where u's low 16 bits
    // are 0x8000; when u is more than 8 m / 2^E units from them (and the
    // cancellation m / |u| is below 2^10, so that the nearest boundary is in
    // u's binade), y rounds to the same bf16 value as u.  About one element in
    // 10^3 goes on to the double-float step below.
    {
        const float t = b * q_hi;
        const float u = fmaf(a, p_hi, t);
        const float m = fabsf(a * p_hi) + fabsf(t);
        const uint32_t ub = __float_as_uint(u);
        const float e2 = __uint_as_float(ub & 0x7F800000u);  // 0 for zero and subnormal u
        const int low = (int)(ub & 0xFFFFu) - 0x8000;
        const float dist = __uint_as_float(0x4B000000u | (uint32_t)abs(low)) - 8388608.f;  // |low|, exactly
        if (dist * e2 > 8.f * m && 1024.f * e2 > m && e2 < 1e30f)
            return (uint16_t)((ub + 0x7FFFu + ((ub >> 16) & 1u)) >> 16);
    }
    const float P1 = a * p_hi, E1 = fmaf(a, p_hi, -P1);
    const float P2 = b * q_hi, E2 = fmaf(b, q_hi, -P2);
    const float S = P1 + P2;
    const float bb = S - P1;
    const float T = (P1 - (S - bb)) + (P2 - bb);
    const float small = ((E1 + E2) + T) + fmaf(a, p_lo, b * q_lo);
    const float u = S + small;
    const float mag = fabsf(P1) + fabsf(P2);
    const uint32_t ub = __float_as_uint(u);
    const uint16_t w = (uint16_t)((ub + 0x7FFFu + ((ub >> 16) & 1u)) >> 16);
    const uint32_t wb = (uint32_t)w;
    const float wf = __uint_as_float(wb << 16);
    const float awf = fabsf(wf);
    if (mag > 0.f && awf > 1e-30f && awf < 1e30f) {
        // neighbours of w toward +inf and -inf (w away from zero and inf)
        const uint32_t up = (wb & 0x8000u) ? wb - 1u : wb + 1u;
        const uint32_t dn = (wb & 0x8000u) ? wb + 1u : wb - 1u;
        const float m1 = 0.5f * (wf + __uint_as_float(up << 16));   // exact: short significands
        const float m0 = 0.5f * (wf + __uint_as_float(dn << 16));
        const float margin = mag * 0x1p-34f;
        const float d1 = (m1 - S) - small;   // m1 - S is exact (Sterbenz)
        const float d0 = (S - m0) + small;
        if (d1 > margin && d0 > margin) return w;
    }
    const double2 c = *pq;  // fp64 {cos, sin}: read only on this rare path
    return bf16_from_double(__dadd_rn(__dmul_rn((double)a, c.x), __dmul_rn((double)b, c.y)));
}
// fp32 RoPE table: each position's row holds cos_hi[d/2], sin_hi[d/2],
// cos_lo[d/2], sin_lo[d/2], so that the hi parts the queries need are the
// first half of the row (one TMA box fetches them for a whole Q tile).
template <int HALF>
__device__ __forceinline__ float4 rope_row_pair(const float* row, int j) {
    return make_float4(row[j], row[2 * HALF + j], row[HALF + j], row[3 * HALF + j]);  // {cos_hi, cos_lo, sin_hi, sin_lo}
}
__device__ __forceinline__ void rope_pair(float x0, float x1, float4 cf, const double2* cs, uint16_t& y0,
                                          uint16_t& y1) {
    y0 = rope_bf16(x0, -x1, cf.x, cf.y, cf.z, cf.w, cs);
    y1 = rope_bf16(x1, x0, cf.x, cf.y, cf.z, cf.w, cs);
}
// Interleaved pairing: a holds dims 2j0..2j0+7 (pairs j0..j0+3), b the next
// eight (pairs j0+4..j0+7); the outputs replace them in place.
template <int HALF>
__device__ __forceinline__ void rope8_interleaved(uint4 a, uint4 b, const float* ch, const double2* fb, uint4& oa,
                                                  uint4& ob) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        uint16_t y0, y1;
        rope_pair(__uint_as_float(w[p] << 16), __uint_as_float(w[p] & 0xFFFF0000u), rope_row_pair<HALF>(ch, p), fb + p,
                  y0, y1);
        o[p] = (uint32_t)y0 | ((uint32_t)y1 << 16);
    }
    oa = make_uint4(o[0], o[1], o[2], o[3]);
    ob = make_uint4(o[4], o[5], o[6], o[7]);
}
// Eight consecutive pairs (x0 = a, x1 = b, 8 bf16 each) of one key row:
// lo = first-half outputs, hi = second-half outputs.
template <int HALF>
__device__ __forceinline__ void rope8(uint4 a, uint4 b, const float* ch, const double2* fb, uint4& lo, uint4& hi) {
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
    uint32_t w0[4], w1[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
        uint16_t lo0, lo1, hi0, hi1;
        rope_pair(__uint_as_float(aw[e2] << 16), __uint_as_float(bw[e2] << 16), rope_row_pair<HALF>(ch, 2 * e2),
                  fb + 2 * e2, lo0, lo1);
        rope_pair(__uint_as_float(aw[e2] & 0xFFFF0000u), __uint_as_float(bw[e2] & 0xFFFF0000u), rope_row_pair<HALF>(ch, 2 * e2 + 1),
                  fb + 2 * e2 + 1, hi0, hi1);
        w0[e2] = (uint32_t)lo0 | ((uint32_t)hi0 << 16);
        w1[e2] = (uint32_t)lo1 | ((uint32_t)hi1 << 16);
    }
    lo = make_uint4(w0[0], w0[1], w0[2], w0[3]);
    hi = make_uint4(w1[0], w1[1], w1[2], w1[3]);
}

// Key rotation for the APPEND items, branch-free.  For one output y = a p +
// b q (p, q = cos, sin of the angle, |p|, |q| <= 1) the fp32 value
// u = fl(fma(a, p_hi, fl(b q_hi))) lies within 3.1 2^-24 (|a| + |b|) of the
// fp64 evaluation v (the lo parts of p and q, the two roundings, and the fp64
// evaluation's own error, which is below 2^-52 (|a| + |b|)); eb = 3.25 2^-24
// (|a| + |b|) in fp32 bounds it strictly.  Rounding to nearest even changes
// bf16 value only at the midpoints between bf16 numbers.  m, u's fp32 encoding
// with its low 16 bits set to 0x8000, is the midpoint inside u's bf16 interval
// (u - m is exact: same sign and exponent); the neighbouring intervals'
// midpoints lie at least a quarter bf16 ulp of u, so at least |u| 2^-10, from
// u.  Hence |u - m| > eb and |u| >= 1024 eb mean that no midpoint lies between
// u and v: both round to the same bf16 -- all but about one output in 10^3;
// the others are queued and redone by rope_bf16.
__device__ __forceinline__ float rope_fast(float a, float b, float p_hi, float q_hi, float eb, float ebk, bool& sure) {
    const float u = fmaf(a, p_hi, b * q_hi);
    const float m = __uint_as_float((__float_as_uint(u) & 0xFFFF0000u) | 0x8000u);
    sure = (fabsf(u - m) > eb) & (fabsf(u) >= ebk);
    return u;
}
constexpr float kRopeErrScale = 3.25f / 16777216.f;  // 3.25 2^-24
// Fix-up queue entry: where the output goes (byte offset in shared memory), its
// pair and token (pair j, output 0 or 1, item-local token), and x0, x1.
struct RopeFix {
    uint32_t off;   // kRopeFixNone: a slot of a run that did not fit the queue
    uint32_t code;  // j | which << 7 | tl << 8 | page of the pair << 15
    float x0, x1;
};
constexpr int kRopeFixCap = 256;            // entries (4 KB)
constexpr uint32_t kRopeFixNone = 0xFFFFFFFFu;

// Element e (0..7) of eight packed bf16 values.
__device__ __forceinline__ void set_bf16(uint32_t (&w)[4], int e, uint16_t v) {
    w[e >> 1] = (e & 1) ? ((w[e >> 1] & 0xFFFFu) | ((uint32_t)v << 16)) : ((w[e >> 1] & 0xFFFF0000u) | v);
}

// Eight pairs of one key row, rotated and rounded to bf16 exactly as the fp64
// evaluation is.  Rotate-half (IL false): a = x0 and b = x1 of pairs j0..j0+7,
// lo / hi = their outputs.  Interleaved: a = dims 2j0..2j0+7, b = the next
// eight, outputs in place.  hrow: cos_hi and sin_hi of pairs j0..j0+7 (planes
// HALF floats apart).  The rare uncertain outputs are appended to the fix-up
// queue (off_lo / off_hi: byte offsets in shared memory where lo / hi will be
// stored; code_tl: the token and page bits of the entry's code); if the queue
// is full they are redone here with rope_bf16 (grow: the full fp32 table row at
// pair j0, fb: its fp64 values).
template <int HALF, bool IL>
__device__ __forceinline__ void rope8_key(uint4 a, uint4 b, const float* hrow, int j0, uint32_t off_lo,
                                          uint32_t off_hi, uint32_t code_tl, RopeFix* fixq, int* fix_n,
                                          const float* grow, const double2* fb, uint4& lo, uint4& hi) {
    float ch[8], sh[8];
    {
        const float4* vc = reinterpret_cast<const float4*>(hrow);
        const float4* vs = reinterpret_cast<const float4*>(hrow + HALF);
        const float4 c0 = vc[0], c1 = vc[1], s0 = vs[0], s1 = vs[1];
        ch[0] = c0.x; ch[1] = c0.y; ch[2] = c0.z; ch[3] = c0.w; ch[4] = c1.x; ch[5] = c1.y; ch[6] = c1.z; ch[7] = c1.w;
        sh[0] = s0.x; sh[1] = s0.y; sh[2] = s0.z; sh[3] = s0.w; sh[4] = s1.x; sh[5] = s1.y; sh[6] = s1.z; sh[7] = s1.w;
    }
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
    float x0[8], x1[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (!IL) {
            x0[2 * q] = __uint_as_float(aw[q] << 16);
            x0[2 * q + 1] = __uint_as_float(aw[q] & 0xFFFF0000u);
            x1[2 * q] = __uint_as_float(bw[q] << 16);
            x1[2 * q + 1] = __uint_as_float(bw[q] & 0xFFFF0000u);
        } else {
            x0[q] = __uint_as_float(aw[q] << 16);
            x1[q] = __uint_as_float(aw[q] & 0xFFFF0000u);
            x0[4 + q] = __uint_as_float(bw[q] << 16);
            x1[4 + q] = __uint_as_float(bw[q] & 0xFFFF0000u);
        }
    }
    float y0[8], y1[8];
    uint32_t unsure = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const float eb = (fabsf(x0[p]) + fabsf(x1[p])) * kRopeErrScale, ebk = eb * 1024.f;
        bool s0, s1;
        y0[p] = rope_fast(x0[p], -x1[p], ch[p], sh[p], eb, ebk, s0);
        y1[p] = rope_fast(x1[p], x0[p], ch[p], sh[p], eb, ebk, s1);
        unsure |= (s0 ? 0u : 1u << p) | (s1 ? 0u : 0x100u << p);
    }
    uint32_t wl[4], wh[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (!IL) {
            wl[q] = pack_bf16(y0[2 * q], y0[2 * q + 1]);
            wh[q] = pack_bf16(y1[2 * q], y1[2 * q + 1]);
        } else {
            wl[q] = pack_bf16(y0[q], y1[q]);
            wh[q] = pack_bf16(y0[4 + q], y1[4 + q]);
        }
    }
    if (unsure) {
        // rare: queue the uncertain outputs (a run of consecutive entries)
        const int need = __popc(unsure);
        const int k0 = atomicAdd(fix_n, need);
        if (k0 + need <= kRopeFixCap) {
            int k = k0;
            for (uint32_t m = unsure; m; m &= m - 1, ++k) {
                const int bit = __ffs(m) - 1;
                const int p = bit & 7, which = bit >> 3;
                // where that output sits in lo / hi (two bytes per element)
                const uint32_t off = IL ? ((p < 4 ? off_lo : off_hi) + (uint32_t)(4 * (p & 3) + 2 * which))
                                        : ((which ? off_hi : off_lo) + (uint32_t)(2 * p));
                float px0 = 0.f, px1 = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (e == p) {
                        px0 = x0[e];
                        px1 = x1[e];
                    }
                fixq[k] = RopeFix{off, (uint32_t)(j0 + p) | ((uint32_t)which << 7) | code_tl, px0, px1};
            }
        } else {
            // the queue is full (never with ordinary inputs): mark this run's
            // slots that fit, and redo the outputs here
            for (int k = k0; k < kRopeFixCap; ++k) fixq[k].off = kRopeFixNone;
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const float4 cf = rope_row_pair<HALF>(grow, p);
                if (unsure & (1u << p)) {
                    const uint16_t r = rope_bf16(x0[p], -x1[p], cf.x, cf.y, cf.z, cf.w, fb + p);
                    if (!IL) set_bf16(wl, p, r); else set_bf16(p < 4 ? wl : wh, 2 * (p & 3), r);
                }
                if (unsure & (0x100u << p)) {
                    const uint16_t r = rope_bf16(x1[p], x0[p], cf.x, cf.y, cf.z, cf.w, fb + p);
                    if (!IL) set_bf16(wh, p, r); else set_bf16(p < 4 ? wl : wh, 2 * (p & 3) + 1, r);
                }
            }
        }
    }
    lo = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    hi = make_uint4(wh[0], wh[1], wh[2], wh[3]);
}

// Eight pairs of one query row in fp32, rounded to bf16 (Q feeds the MMA in
// bf16; its rotation needs no certified rounding).  Rotate-half: a = x0 and
// b = x1 of pairs j0..j0+7, lo / hi = their outputs.  Interleaved: a = dims
// 2j0..2j0+7, b = the next eight, outputs in place.  c, s: cos_hi and sin_hi
// of pairs j0..j0+7.
__device__ __forceinline__ void rope_q8(uint4 a, uint4 b, const float (&c)[8], const float (&s)[8], bool interleaved,
                                        uint4& lo, uint4& hi) {
    const __nv_bfloat16* xa = reinterpret_cast<const __nv_bfloat16*>(&a);
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(&b);
    uint32_t ylo[4], yhi[4];
    if (!interleaved) {
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const float a0 = __bfloat162float(xa[e]), a1 = __bfloat162float(xa[e + 1]);
            const float b0 = __bfloat162float(xb[e]), b1 = __bfloat162float(xb[e + 1]);
            ylo[e >> 1] = pack_bf16(a0 * c[e] - b0 * s[e], a1 * c[e + 1] - b1 * s[e + 1]);
            yhi[e >> 1] = pack_bf16(b0 * c[e] + a0 * s[e], b1 * c[e + 1] + a1 * s[e + 1]);
        }
    } else {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float x0 = __bfloat162float(xa[2 * p]), x1 = __bfloat162float(xa[2 * p + 1]);
            const float z0 = __bfloat162float(xb[2 * p]), z1 = __bfloat162float(xb[2 * p + 1]);
            ylo[p] = pack_bf16(x0 * c[p] - x1 * s[p], x1 * c[p] + x0 * s[p]);
            yhi[p] = pack_bf16(z0 * c[p + 4] - z1 * s[p + 4], z1 * c[p + 4] + z0 * s[p + 4]);
        }
    }
    lo = make_uint4(ylo[0], ylo[1], ylo[2], ylo[3]);
    hi = make_uint4(yhi[0], yhi[1], yhi[2], yhi[3]);
}
// cos_hi and sin_hi of pairs j0..j0+7 of one table row (global or shared
// memory; the row's first d/2 floats are cos_hi, the next d/2 sin_hi).
template <int HALF>
__device__ __forceinline__ void load_rope_hi(const float* row, int j0, float (&c)[8], float (&s)[8]) {
    const float4* vc = reinterpret_cast<const float4*>(row + j0);
    const float4* vs = reinterpret_cast<const float4*>(row + HALF + j0);
    const float4 c0 = vc[0], c1 = vc[1], s0 = vs[0], s1 = vs[1];
    c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w; c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
    s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w; s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
}

// ----------------------------------------------------------------------------
// APPEND: rotate + store the K/V of the prefill tokens of one 128-position
// block (up to 8 pages), for up to kAppendHeads kv heads
// ----------------------------------------------------------------------------
// Every page's rows arrive at once: per page, lane k of warp 0 issues three TMA
// boxes -- the page's K rows and V rows from k's and v's [token][kv head][d]
// layout as [head][16 tokens][d] (the order of a page's slots), and the cos_hi /
// sin_hi planes of the page's positions -- on one mbarrier per page, and stores
// the V rows to the page as soon as they land.  The threads rotate the K rows in
// place as their pages land (certified rounding, the rare uncertain outputs
// redone from a queue), then lane k stores page k's K rows.  The item then sets
// its ready flag, which the prefill tiles of its kv heads wait for before they
// load the block.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
template <int D, bool IL>
__device__ void run_append(const KParams& P, const CUtensorMap* tmKin, const CUtensorMap* tmVin,
                           const CUtensorMap* tmRA, const int* it, uint8_t* smem, uint32_t bar0, uint32_t* s_phase,
                           int* s_abort, int* s_fix) {
    const int tid = threadIdx.x;
    const int s = it[kS], g0 = it[kG], t0 = it[kStart], cnt = it[kCount];
    const Row R = row_geom(it);
    const int Hkv = P.Hkv;
    constexpr int HALF = D / 2;
    constexpr int ROW = D * 2;                           // bytes of one (token, head) row
    constexpr int KBOX = kAppendHeads * kPage * ROW;     // one page's K (or V) rows, [head][slot][d]
    constexpr int TROW = D * 4;                          // cos_hi, sin_hi of one position
    constexpr int TBOX = kPage * TROW;                   // ... of one page's positions
    constexpr int kMaxPg = kTileRows / kPage;            // pages of a 128-position block
    constexpr int VBASE = kMaxPg * KBOX;
    constexpr int TBASE = 2 * kMaxPg * KBOX;
    static_assert(TBASE + kMaxPg * TBOX <= kSmemStages && kAppendBufs >= kMaxPg && kMaxPg <= 32,
                  "APPEND shared memory");
    const int ng = min(kAppendHeads, Hkv - g0);          // heads of this item
    const int pos0 = R.h + t0;                           // position of the item's first token
    const int pg0 = pos0 / kPage;
    const int npg = (pos0 + cnt - 1) / kPage - pg0 + 1;
    const int32_t* pages = P.plan + P.off_kvi + R.kvp0;
    // every page id and the RoPE table bound checked up front (all threads alike)
    bool ok = pos0 + cnt <= P.rope_max_pos;
    int bad = pos0 + cnt - 1;
    for (int k = 0; k < npg && ok; ++k) {
        bad = pages[pg0 + k];
        ok = bad >= 0 && bad < P.num_pages;
    }
    RopeFix* fixq = reinterpret_cast<RopeFix*>(smem + kSmemDecQ);  // idle during APPEND items
    static_assert(kRopeFixCap * sizeof(RopeFix) <= 2 * kPageHalfBytes, "fix-up queue");
    const uint32_t ph = *s_phase;  // completed-phase parities of the pages' barriers
    // lane k of warp 0 runs page k's copies: its slots' positions [lo, hi)
    const int lane_pg = tid < 32 ? tid : 0;
    const int pa = (pg0 + lane_pg) * kPage;
    const int lo_pos = max(pos0, pa), hi_pos = min(pos0 + cnt, pa + kPage);
    const uint32_t pbar = bar0 + 8u * (uint32_t)lane_pg;
    const bool copier = ok && tid < npg;
    const size_t pdst = (((size_t)pages[pg0 + (copier ? lane_pg : 0)] * Hkv + g0) * kPage + lo_pos % kPage) * D;
    const uint32_t prow = (uint32_t)((lo_pos % kPage) * ROW), pbytes = (uint32_t)((hi_pos - lo_pos) * ROW);
    if (!ok) {
        if (tid == 0) raise_error(P, kErrBounds, bad, s_abort);
    } else {
        if (copier) {
            // the page's 16 slots: the boxes start at the slot of the page's
            // first position (rows outside the item are loaded, not used)
            mbar_expect_tx(pbar, (uint32_t)(2 * KBOX + TBOX));
            tma_load_3d(smem_u32(smem + lane_pg * KBOX), tmKin, 0, R.qo0 + t0 + (pa - pos0), g0, pbar);
            tma_load_3d(smem_u32(smem + VBASE + lane_pg * KBOX), tmVin, 0, R.qo0 + t0 + (pa - pos0), g0, pbar);
            tma_load_2d(smem_u32(smem + TBASE + lane_pg * TBOX), tmRA, 0, pa, pbar);
            // V goes straight back out to the page
            if (mbar_wait_bounded(P, pbar, (ph >> lane_pg) & 1u, s_abort, 11000 + lane_pg, it)) {
                const uint32_t src = smem_u32(smem + VBASE + lane_pg * KBOX) + prow;
                for (int g = 0; g < ng; ++g)
                    bulk_store(P.v_cache + pdst + (size_t)g * kPage * D, src + (uint32_t)(g * kPage * ROW), pbytes);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
        }
        // K: eight pairs of one (token, head) row per unit, in token order
        int* fix_n = s_fix;
        const int units = cnt * ng * (HALF / 8);
        int seen = -1;  // pages whose loads this thread has waited for: 0..seen
        for (int u = tid; u < units; u += kThreads) {
            const int c = u % (HALF / 8), h = (u / (HALF / 8)) % ng, tl = u / (ng * (HALF / 8));
            const int pos = pos0 + tl;
            const int k = pos / kPage - pg0, slot = pos % kPage;
            while (seen < k) {
                ++seen;
                if (!mbar_wait_bounded(P, bar0 + 8u * (uint32_t)seen, (ph >> seen) & 1u, s_abort, 10000 + seen, it))
                    break;
            }
            if (*(volatile int*)s_abort) break;
            uint16_t* krow = reinterpret_cast<uint16_t*>(smem + k * KBOX + (h * kPage + slot) * ROW);
            const float* trow = reinterpret_cast<const float*>(smem + TBASE + k * TBOX + slot * TROW);
            const float* grow = P.ropef + (size_t)pos * 4 * HALF;  // the full fp32 row (rare path)
            // pairs 8c .. 8c + 7: dims (j, j + d/2), or (2j, 2j + 1) interleaved
            const int d0 = IL ? 16 * c : 8 * c;
            const int d1 = IL ? 16 * c + 8 : HALF + 8 * c;
            uint4 lo, hi;
            rope8_key<HALF, IL>(*reinterpret_cast<const uint4*>(krow + d0), *reinterpret_cast<const uint4*>(krow + d1),
                                trow + c * 8, 8 * c, smem_u32(krow + d0), smem_u32(krow + d1), (uint32_t)tl << 8,
                                fixq, fix_n, grow + c * 8, P.rope + (size_t)pos * HALF + c * 8, lo, hi);
            *reinterpret_cast<uint4*>(krow + d0) = lo;
            *reinterpret_cast<uint4*>(krow + d1) = hi;
        }
        __syncthreads();
        if (!*(volatile int*)s_abort) {
            // the queued uncertain outputs, redone in full (about one in 10^3);
            // the row's four values load together
            const int nfix = min(*(volatile int*)fix_n, kRopeFixCap);
            for (int e = tid; e < nfix; e += kThreads) {
                const RopeFix f = fixq[e];
                if (f.off == kRopeFixNone) continue;
                const int j = (int)(f.code & 127u), which = (int)((f.code >> 7) & 1u);
                const int pos = pos0 + (int)((f.code >> 8) & 127u);
                const float4 cf = rope_row_pair<HALF>(P.ropef + (size_t)pos * 4 * HALF, j);
                const double2* fb = P.rope + (size_t)pos * HALF + j;
                const uint16_t r = which ? rope_bf16(f.x1, f.x0, cf.x, cf.y, cf.z, cf.w, fb)
                                         : rope_bf16(f.x0, -f.x1, cf.x, cf.y, cf.z, cf.w, fb);
                asm volatile("st.shared.u16 [%0], %1;" ::"r"(f.off), "h"(r) : "memory");
            }
        }
        fence_proxy_async_shared();  // the rotated rows are read by the bulk stores (async proxy)
        __syncthreads();
        if (tid == 0) *fix_n = 0;    // every thread read it before the barrier
        if (copier && !*(volatile int*)s_abort) {
            const uint32_t src = smem_u32(smem + lane_pg * KBOX) + prow;
            for (int g = 0; g < ng; ++g)
                bulk_store(P.k_cache + pdst + (size_t)g * kPage * D, src + (uint32_t)(g * kPage * ROW), pbytes);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        if (copier) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // the page's V and K are written
    }
    // publish: the pages are read next by TMA (async proxy) in other CTAs
    fence_proxy_async_global();
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int blk = pos0 / kTileRows - R.h / kTileRows;
        atomicExch(&P.ws_int[kHdrInts + P.plan[P.off_aux + s] + blk * kv_groups(Hkv) + g0 / kAppendHeads], 1);
        // each page's barrier completed one phase (a thread that gave up on a
        // wait has flagged the CTA, which stops taking items)
        if (ok) *s_phase = ph ^ ((1u << npg) - 1u);
    }
}

// ----------------------------------------------------------------------------
// tcgen05 / TMEM helpers (inline PTX)
// ----------------------------------------------------------------------------
// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, M = 128.
__host__ __device__ constexpr uint32_t umma_idesc(int n, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Same with the A operand read from tensor memory.
__device__ __forceinline__ void umma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Phase parities of the prefill pipeline, one word per thread, carried across
// work items; each role only flips the bits of the barriers it waits on.  Only
// parities are needed: a barrier's n-th completion is waited for with parity
// n & 1, and a fresh barrier passes a wait on parity 1 at once (the phase
// before its first), which is how a producer's first wait on an empty slot
// returns.
struct PfPhase {
    uint32_t bits;
};
constexpr int kPfStagesMax = 4;
constexpr int kPhKFill = 0;    // 4: producer, loads issued into each K stage
constexpr int kPhVFill = 4;    // 4: producer, loads issued into each V stage
constexpr int kPhKUse = 8;     // 4: MMA issuer, K loads consumed
constexpr int kPhVUse = 12;    // 4: MMA issuer, V loads consumed
constexpr int kPhPFull = 16;   // 2: MMA issuer, P of each buffer consumed
constexpr int kPhSUse = 18;    // 2: softmax, S of each buffer consumed
constexpr int kPhOUp = 20;     // 2: softmax, P.V groups of each P buffer waited for
constexpr int kPhODone = 22;   // 1: softmax, items completed before this one
constexpr int kPhVSeen = 23;   // 4: softmax, V loads into each stage (last-block clean-up)
constexpr int kPhSFree = 27;   // 2: QK issuer, S of each buffer loaded by the softmax
constexpr int kPhQ = 29;       // 1: Q writers, Q tiles loaded
__device__ __forceinline__ uint32_t ph_get(const PfPhase& ph, int bit) { return (ph.bits >> bit) & 1u; }
__device__ __forceinline__ void ph_flip(PfPhase& ph, int bit) { ph.bits ^= 1u << bit; }

// TMEM loads without the wait, so that two can be in flight; tmem_wait_ld
// then also pins the destination registers after the wait.
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, float* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]),
          "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]),
          "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]),
          "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
        : "r"(taddr));
}
template <int N>
__device__ __forceinline__ void tmem_wait_ld(float (&v)[N]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+f"(v[i]));
}
// 16 consecutive 32-bit columns of this thread's TMEM lane; completes at tmem_wait_st.
__device__ __forceinline__ void tmem_st16_nw(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 16 consecutive 32-bit columns of this thread's TMEM lane, waited for.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(v[i]));
}

// ----------------------------------------------------------------------------
// PREFILL item on the 5th-generation tensor cores: one Q tile of up to 128
// query rows (token-major, q-head-in-group minor) of one chunk for one kv
// head, causal over every history page and the chunk ("Sarathi-Serve 完全拆解",
// §"分块不等于截断上下文"), over all its 128-key blocks or, for a key piece of a
// split tile, over a range of them.  K and V blocks stream through shared
// memory rings; tensor memory holds two score buffers, two P buffers and O:
//   S(j) = Q K(j)^T: tcgen05.mma (M 128, N 128, K 16 steps, both operands in
//       shared memory), fp32 into S buffer j & 1 (columns [128 b, 128 b + 128));
//   softmax (warps 0-7: warps q and q + 4 hold rows 32 q .. 32 q + 31, the TMEM
//       lanes of their SM sub-partition, one thread a row, each warp one half
//       of the block's keys; the pair agrees on the block's max through shared
//       memory), lazy rescale of O (only when the max grows by more than 2^8),
//       bf16 P into P buffer j & 1 (64 columns at 384 + 64 b);
//   O += P(j) V(j): tcgen05.mma with A = P from tensor memory and V read as an
//       MN-major operand straight from the TMA-loaded pages; O in columns
//       [256, 256 + d) until the end of the item.
// Two threads issue the MMAs: warp 11 runs S(j) as soon as the softmax has
// loaded S(j - 2) (so the tensor pipe holds the next block's scores while the
// softmax works), warp 10 runs P(j).V(j) once all eight softmax warps have
// stored P(j).  The groups of different issuers do not complete in a known
// order, so each P.V group signals its P buffer's barrier, which the softmax
// waits for before it overwrites that buffer or rescales O.
// Roles: warps 8 and 9 are the TMA producers of the K and V rings (one box per
// block when the block's pages are consecutive in the pool, else one box per
// page and 64-column half), warps 0-7 run the softmax and the epilogue, warps
// 0-7, 10 and 11 rotate Q at the item's start.
// ----------------------------------------------------------------------------
constexpr int kTcKeys = 128;                     // keys per block
static_assert(kTcKeys == kTileRows, "a K/V block and a Q tile have the same shape");
template <int D>
struct PfLayout {
    static constexpr int kTile = kTileRows * D * 2;    // bytes of the Q tile or of one K/V block
    static constexpr int kKStages = D == 128 ? 3 : 4;  // K ring (runs two blocks ahead of V)
    static constexpr int kVStages = D == 128 ? 2 : 4;  // V ring
    static constexpr int kQ = 0;                       // Q tile: [d/64][128 rows][128 B]
    static constexpr int kK = kTile;
    static constexpr int kV = kK + kKStages * kTile;
    static_assert(kV + kVStages * kTile <= kSmemStages, "prefill shared memory");
    static_assert(kKStages <= kPfStagesMax && kVStages <= kPfStagesMax, "phase bits");
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;     // S of block parity b at 128 b
constexpr uint32_t kTmemO = 256;   // O
constexpr uint32_t kTmemP = 384;   // bf16 P of block parity b at 384 + 64 b
constexpr int kBarKFull = kDecWarps * kDecStages;   // kPfStagesMax
constexpr int kBarKEmpty = kBarKFull + kPfStagesMax;
constexpr int kBarVFull = kBarKEmpty + kPfStagesMax;
constexpr int kBarVEmpty = kBarVFull + kPfStagesMax;
constexpr int kBarSFull = kBarVEmpty + kPfStagesMax;  // 2 (per S buffer)
constexpr int kBarPFull = kBarSFull + 2;               // 2 (per P buffer, 256 arrivals each)
constexpr int kBarSFree = kBarPFull + 2;               // 2 (per S buffer: loaded by the softmax, 256 arrivals)
constexpr int kBarOUp = kBarSFree + 2;                 // 2 (per P buffer: its P.V group done)
constexpr int kBarODone = kBarOUp + 2;                 // 1 (one completion per item: its last P.V)
constexpr int kBarDrain = kBarODone + 1;               // 2 (one per MMA-issuing thread)
constexpr int kBarAppend = kBarDrain + 2;              // kAppendBufs (one per page of an APPEND item)
constexpr int kBarQ = kBarAppend + kAppendBufs;        // 1 (the Q tile's TMA boxes)
constexpr int kNumBars = kBarQ + 1;
static_assert(kNumBars * 8 <= 512, "barrier area");

template <int D, bool IL>
__device__ void run_prefill(const KParams& P, const CUtensorMap* tmK, const CUtensorMap* tmV,
                            const CUtensorMap* tmK5, const CUtensorMap* tmV5, const CUtensorMap* tmQ,
                            const CUtensorMap* tmR, const int* it,
                            uint8_t* smem,
                            int* s_abort, PfPhase& ph, uint32_t tmem) {
    using L = PfLayout<D>;
    constexpr int HALVES = D / 64;
    constexpr int HALF = D / 2;
    constexpr int BLK_HALF = kTcKeys * 128;      // one 64-column half of a 128-key block
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = it[kS], g = it[kG], t0 = it[kStart], cnt = it[kCount];
    const Row R = row_geom(it);
    const int G = P.group;
    const int kv_hi = R.h + t0 + cnt;            // keys [0, kv_hi) are visible to some row
    const int nblk = (kv_hi + kTcKeys - 1) / kTcKeys;
    const int pages_hi = (kv_hi + kPage - 1) / kPage;
    // a tile split along its keys runs blocks [kb0, kb1) here (j below is
    // the block, jj its place in this item's pipeline); else every block
    const int kb0 = it[kB0], kb1 = it[kB1] > 0 ? min(it[kB1], nblk) : nblk;
    const int nb = kb1 - kb0;
    const uint32_t bars = smem_u32(smem + kSmemBars);
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };

    // The TMA producers (warps 8 and 9) start on the history pages at once; only
    // the blocks holding the chunk's own keys wait for this request's APPENDs.
    // Meanwhile warps 0-7, 10 and 11 write the Q tile and meet on named barrier 5.
    const bool q_writer = warp < 8 || warp >= 10;
    const int qtid = warp >= 10 ? 256 + (warp - 10) * 32 + lane : tid;
    constexpr int kQThreads = 320;
    constexpr int kQUnits = kTileRows * (HALF / 8);
    // Q tile: two TMA boxes (one per 64-column half) bring the raw rows
    // [tokens][heads of the group][d] of the item straight into the swizzled
    // tile, and one more box brings the hi parts (cos_hi, sin_hi) of the RoPE
    // table rows of the tile's positions into the V ring, still idle then (the
    // V producer joins the writers' barrier before its first load).  The
    // writers then rotate their 16-byte chunks in place in fp32: one memory
    // round trip for the whole tile.
    constexpr int kQBar = kQThreads + 32;
    const int tpt = kTileRows / G;
    const float* rtab = reinterpret_cast<const float*>(smem + L::kV);  // [tpt][cos_hi[d/2], sin_hi[d/2]]
    if (warp == 11 && lane == 0) {
        mbar_expect_tx(bar(kBarQ), (uint32_t)(HALVES * tpt * G * 128 + tpt * HALF * 8));
        for (int hf = 0; hf < HALVES; ++hf)
            tma_load_3d(smem_u32(smem + L::kQ + hf * kTileRows * 128), tmQ, hf * 64, g * G, R.qo0 + t0, bar(kBarQ));
        tma_load_2d(smem_u32(smem + L::kV), tmR, 0, R.h + t0, bar(kBarQ));
    }
    if (q_writer) {
        const int rows_valid = cnt * G;
        mbar_wait_bounded(P, bar(kBarQ), ph_get(ph, kPhQ), s_abort, 500, it);
        ph_flip(ph, kPhQ);
        uint8_t* qtile = smem + L::kQ;
        for (int i = qtid; i < kQUnits; i += kQThreads) {
            const int row = i / (HALF / 8), c = i % (HALF / 8);
            // 16-byte chunks holding pairs 8c..8c+7
            const int c0 = IL ? 2 * c : c, c1 = IL ? 2 * c + 1 : c + HALF / 8;
            uint4* p0 = reinterpret_cast<uint4*>(qtile + sw128_chunk(kTileRows, row, c0));
            uint4* p1 = reinterpret_cast<uint4*>(qtile + sw128_chunk(kTileRows, row, c1));
            uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
            if (row < rows_valid) {
                float cs[8], sn[8];
                load_rope_hi<HALF>(rtab + (row / G) * HALF * 2, c * 8, cs, sn);
                rope_q8(*p0, *p1, cs, sn, IL, lo, hi);
            }
            *p0 = lo;
            *p1 = hi;
        }
        fence_proxy_async_shared();  // Q is read by the tensor cores (async proxy)
        tc_fence_before();
        asm volatile("bar.sync 5, %0;" ::"n"(kQBar) : "memory");
        tc_fence_after();
    } else if (warp == 9) {
        // the V ring holds the table rows until the Q tile is written
        asm volatile("bar.sync 5, %0;" ::"n"(kQBar) : "memory");
    }

    if (warp == 8 || warp == 9) {
        // ---------------- TMA producers: warp 8 fills the K ring, warp 9 the V ring ----------------
        const bool is_v = warp == 9;
        const int NST = is_v ? L::kVStages : L::kKStages;
        // lane 8 hf + q holds the id of page q of the block; when the block's
        // pages are not consecutive in the pool it issues the box of that page
        // and column half hf
        const int hf = lane >> 3, pq = lane & 7;
        const bool issuer = hf < HALVES;
        const CUtensorMap* map = is_v ? tmV : tmK;
        const CUtensorMap* map5 = is_v ? tmV5 : tmK5;
        const int full0 = is_v ? kBarVFull : kBarKFull;
        const int empty0 = is_v ? kBarVEmpty : kBarKEmpty;
        const int fill = is_v ? kPhVFill : kPhKFill;
        uint8_t* ring = smem + (is_v ? L::kV : L::kK);
        const int32_t* kvi = P.plan + P.off_kvi + R.kvp0;
        int id = kb0 * 8 + pq < pages_hi ? it[kIds + pq] : 0;  // the first block's ids come with the item
        const int j_chunk = R.h / kTcKeys;  // first block with a key of the chunk
        for (int jj = 0; jj < nb; ++jj) {
            const int j = kb0 + jj;
            if (j >= j_chunk) {
                // the block's new K/V must be in the pages: the ready flag its
                // APPEND item sets for this tile's group of kv heads
                const int* ctr = &P.ws_int[kHdrInts + P.plan[P.off_aux + s] + (j - j_chunk) * kv_groups(P.Hkv) +
                                           g / kAppendHeads];
                if (lane == 0 && ld_acquire(ctr) == 0) {
                    const uint64_t w0 = globaltimer();
                    while (ld_acquire(ctr) == 0) {
                        if (globaltimer() - w0 > kWaitNs / 2) {  // first to give up: names the cause
                            raise_error(P, kErrWait, -1 - s, s_abort);
                            break;
                        }
                        __nanosleep(100);
                    }
                }
                __syncwarp();
                (void)ld_acquire(ctr);      // every issuing lane acquires for itself
                fence_proxy_async_global();  // ... and orders the TMA reads after it
            }
            if (*(volatile int*)s_abort) break;
            const int st = jj % NST;
            const int nxt = (j + 1) * 8 + pq < pages_hi ? kvi[(j + 1) * 8 + pq] : 0;
            const int npg = min(kTcKeys / kPage, pages_hi - j * 8);
            // one box for the whole block when its pages are consecutive and in the pool
            const int id0 = __shfl_sync(0xffffffffu, id, 0);
            const bool ok_page = pq >= npg || (id == id0 + pq && id >= 0 && id < P.num_pages);
            const bool one_box = __all_sync(0xffffffffu, ok_page);
            mbar_wait_bounded<true>(P, bar(empty0 + st), ph_get(ph, fill + st) ^ 1u, s_abort,
                                    (is_v ? 2000 : 1000) + j, it);
            uint8_t* dst = ring + st * L::kTile;
            if (one_box) {
                if (lane == 0) {
                    mbar_expect_tx(bar(full0 + st), (uint32_t)L::kTile);
                    tma_load_5d(smem_u32(dst), map5, 0, 0, g, id0, 0, bar(full0 + st));
                }
            } else {
                if (lane == 0) mbar_expect_tx(bar(full0 + st), (uint32_t)(npg * HALVES) * kPageHalfBytes);
                __syncwarp();
                if (issuer && pq < npg) {
                    int page = id;
                    if (page < 0 || page >= P.num_pages) {
                        raise_error(P, kErrBounds, page, s_abort);
                        page = 0;
                    }
                    tma_load_2d(smem_u32(dst + hf * BLK_HALF + pq * kPageHalfBytes), map, hf * 64,
                                (page * P.Hkv + g) * kPage, bar(full0 + st));
                }
            }
            __syncwarp();
            ph_flip(ph, fill + st);
            id = nxt;
        }
    } else if (warp == 11) {
        // ---------------- QK issuer: S(j) = Q K(j)^T into S buffer j & 1 ----------------
        // S buffer j & 1 is free once the softmax has loaded block j - 2's scores
        // (P has buffers of its own), so S(j) runs while block j - 2's softmax does
        if (lane == 0) {
            constexpr uint32_t idesc_s = umma_idesc(kTcKeys, false);
            const uint64_t qd = umma_desc(smem_u32(smem + L::kQ), 16, 1024);
            for (int jj = 0; jj < nb; ++jj) {
                const int j = kb0 + jj;
                const int b = jj & 1;
                if (jj >= 2) {
                    mbar_wait_bounded<true>(P, bar(kBarSFree + b), ph_get(ph, kPhSFree + b), s_abort, 4000 + j, it);
                    ph_flip(ph, kPhSFree + b);
                }
                const int st = jj % L::kKStages;
                mbar_wait_bounded<true>(P, bar(kBarKFull + st), ph_get(ph, kPhKUse + st), s_abort, 3000 + j, it);
                ph_flip(ph, kPhKUse + st);
                tc_fence_after();
                const uint64_t kd = umma_desc(smem_u32(smem + L::kK + st * L::kTile), 16, 1024);
                const uint32_t sd = tmem + kTmemS + (uint32_t)(b * kTcKeys);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // start addresses advance in 16-byte units inside the descriptors
                    const uint64_t off = (uint64_t)(((kk >> 2) * kTileRows * 128 + (kk & 3) * 32) >> 4);
                    const uint64_t koff = (uint64_t)(((kk >> 2) * BLK_HALF + (kk & 3) * 32) >> 4);
                    umma_f16(sd, qd + off, kd + koff, idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(bar(kBarSFull + b));
                umma_commit(bar(kBarKEmpty + st));
            }
            // the loads of the item's last two blocks were not waited for here
            for (int jj = max(nb - 2, 0); jj < nb; ++jj) ph_flip(ph, kPhSFree + (jj & 1));
        }
    } else if (warp == 10) {
        // ---------------- P.V issuer: O += P(j) V(j) ----------------
        if (lane == 0) {
            constexpr uint32_t idesc_o = umma_idesc(D, true);
            for (int jj = 0; jj < nb; ++jj) {
                const int j = kb0 + jj;
                const int b = jj & 1;
                const int vst = jj % L::kVStages;
                mbar_wait_bounded<true>(P, bar(kBarVFull + vst), ph_get(ph, kPhVUse + vst), s_abort, 5000 + j, it);
                ph_flip(ph, kPhVUse + vst);
                mbar_wait_bounded<true>(P, bar(kBarPFull + b), ph_get(ph, kPhPFull + b), s_abort, 4500 + j, it);
                ph_flip(ph, kPhPFull + b);
                tc_fence_after();
                const uint64_t vd = umma_desc(smem_u32(smem + L::kV + vst * L::kTile), BLK_HALF, 1024);
                const uint32_t pa = tmem + kTmemP + (uint32_t)(b * (kTcKeys / 2));
#pragma unroll
                for (int kk = 0; kk < kTcKeys / 16; ++kk) {
                    // A = P from TMEM (16 keys = 8 columns per step); B = V (MN-major:
                    // d contiguous, keys as rows) straight from the TMA-loaded pages
                    umma_f16_ts(tmem + kTmemO, pa + (uint32_t)(kk * 8), vd + (uint64_t)((kk * 16 * 128) >> 4), idesc_o,
                                (jj > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(bar(kBarVEmpty + vst));
                umma_commit(bar(kBarOUp + b));
                if (jj == nb - 1) umma_commit(bar(kBarODone));
            }
        }
    } else if (warp < 8) {
        // ---------------- softmax + epilogue: warps q and q + 4 share query rows 32 q .. 32 q + 31 ----------------
        // (a warp reaches the TMEM lanes of its SM sub-partition, so both see
        // the same rows); warp q takes keys 0-63 of each block, warp q + 4 keys
        // 64-127, and the pair agree on the exponent base through shared memory
        const int hs = warp >> 2;                    // key half of the block (and of P, and of O's columns)
        const int quad = warp & 3;
        const int r = quad * 32 + lane;              // query row = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const int rows_valid = cnt * G;
        const int tt = r < rows_valid ? r / G : cnt - 1;  // item-local token of the row
        const int pos_r = R.h + t0 + tt;
        const float sl2 = P.scale_log2;
        // [block parity][key half][row] maxima, then [key half][row] sums
        float* xmax = reinterpret_cast<float*>(smem + kSmemDecQ);
        float* xsum = xmax + 2 * 2 * kTileRows;
        const uint32_t pair_bar = 6u + (uint32_t)quad;   // named barrier of warps q and q + 4
        constexpr int OCOLS = D / 2;                 // O columns this warp rescales and stores
        float m_run = -INFINITY, l_run = 0.f;
        for (int jj = 0; jj < nb; ++jj) {
            const int j = kb0 + jj;
            const int b = jj & 1;
            const int kc = j * kTcKeys + hs * 64;    // first key of this warp's half
            const uint32_t s_col = kTmemS + (uint32_t)(b * kTcKeys + hs * 64);
            const uint32_t p_col = kTmemP + (uint32_t)(b * (kTcKeys / 2) + hs * 32);
            mbar_wait_bounded(P, bar(kBarSFull + b), ph_get(ph, kPhSUse + b), s_abort, 6000 + j, it);
            ph_flip(ph, kPhSUse + b);
            tc_fence_after();
            float v[64];
            tmem_ld32_nw(lane_base + s_col, v);
            tmem_ld32_nw(lane_base + s_col + 32u, v + 32);
            tmem_wait_ld(v);
            // the scores are in registers: S buffer b may take S(j + 2)
            tc_fence_before();
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kBarSFree + b)) : "memory");
            if (kc + 63 > pos_r) {
#pragma unroll
                for (int e = 0; e < 64; ++e) v[e] = kc + e <= pos_r ? v[e] : -INFINITY;
            }
            // the half's max in four independent chains
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < 64; e += 8) {
#pragma unroll
                for (int c = 0; c < 4; ++c) mq[c] = fmax3(mq[c], v[e + 2 * c], v[e + 2 * c + 1]);
            }
            const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            xmax[(b * 2 + hs) * kTileRows + r] = mx;
            asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
            const float mxs = fmaxf(mx, xmax[(b * 2 + (hs ^ 1)) * kTileRows + r]) * sl2;  // the scale (> 0) applied to the max
            // lazy rescaling: the exponent base moves only when the block's max
            // exceeds it by more than 2^8 (both warps of the pair decide alike)
            const float m_use = mxs > m_run + 8.f ? mxs : m_run;
            if (jj >= 2) {
                // P buffer b was read by P(j - 2).V, issued by another thread
                // than this block's S: wait for it before overwriting
                mbar_wait_bounded(P, bar(kBarOUp + b), ph_get(ph, kPhOUp + b), s_abort, 6500 + j, it);
                ph_flip(ph, kPhOUp + b);
                tc_fence_after();
            }
            // P = 2^(s - m) in bf16, two keys per column
            float2 sum2 = make_float2(0.f, 0.f);
            const float2 sl2v = make_float2(sl2, sl2);
            // (a row of a later key piece may see no key yet: base 0, P = 0)
            const float m_exp = m_use == -INFINITY ? 0.f : m_use;
            const float2 nmv = make_float2(-m_exp, -m_exp);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 x = ffma2(make_float2(v[q * 32 + e], v[q * 32 + e + 1]), sl2v, nmv);
                    const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    sum2 = fadd2(sum2, pp);
                    pk[e >> 1] = pack_bf16(pp.x, pp.y);
                }
                tmem_st16_nw(lane_base + p_col + (uint32_t)(q * 16), pk);
            }
            tmem_wait_st();
            // O and l hold sums with base m_run: bring them to m_use.  O holds
            // the P.V groups of blocks before j; the last of them may still be
            // running, so wait for it first (rare: only when the base moves).
            // P(j - 3).V is done (block j - 1 waited for it) and P(j + 1).V is
            // not issued, so the wait on buffer (j - 1) & 1 is for P(j - 1).V;
            // block j + 1 waits for the same phase again and counts it.
            const bool moved = m_use != m_run;
            const float alpha = moved ? exp2f(m_run - m_use) : 1.f;
            if (jj > 0 && __any_sync(0xffffffffu, moved)) {
                mbar_wait_bounded(P, bar(kBarOUp + ((jj - 1) & 1)), ph_get(ph, kPhOUp + ((jj - 1) & 1)), s_abort,
                                  7000 + j, it);
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < OCOLS / 32; ++c) {
                    float o[32];
                    const uint32_t oc = kTmemO + (uint32_t)(hs * OCOLS + c * 32);
                    tmem_ld32(lane_base + oc, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tmem_st32(lane_base + oc, o);
                }
            }
            l_run = l_run * alpha + (sum2.x + sum2.y);
            m_run = m_use;
            // last block: V rows past kv_hi hold other bytes; zero them so 0 x V stays 0
            if (j == nblk - 1 && j * kTcKeys + kTcKeys > kv_hi) {
                const int vst = jj % L::kVStages;
                mbar_wait_bounded(P, bar(kBarVFull + vst),
                                  ph_get(ph, kPhVSeen + vst) ^ (uint32_t)((jj / L::kVStages) & 1), s_abort, 8000 + j,
                                  it);
                uint8_t* vb = smem + L::kV + vst * L::kTile;
                const int first = kv_hi - j * kTcKeys;
                for (int hf = 0; hf < HALVES; ++hf)
                    for (int i = first * 128 + tid * 16; i < kTcKeys * 128; i += 256 * 16)
                        *reinterpret_cast<uint4*>(vb + hf * BLK_HALF + i) = make_uint4(0, 0, 0, 0);
                fence_proxy_async_shared();
            }
            tc_fence_before();
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kBarPFull + b)) : "memory");
        }
        // epilogue: O / l -> bf16 once the last P.V group is done (a barrier of
        // its own: when it is waited for, two P.V groups may be outstanding,
        // which a parity wait on the per-buffer barriers cannot tell apart);
        // each warp of the pair adds the other's part of l and stores half of
        // the row's columns
        mbar_wait_bounded(P, bar(kBarODone), ph_get(ph, kPhODone), s_abort, 9000, it);
        ph_flip(ph, kPhODone);
        tc_fence_after();
        xsum[hs * kTileRows + r] = l_run;
        asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
        const float lt = l_run + xsum[(hs ^ 1) * kTileRows + r];
        __nv_bfloat16* dst =
            r < rows_valid ? P.out + ((size_t)(R.qo0 + t0 + tt) * P.Hq + g * G + r % G) * D + hs * OCOLS : nullptr;
        const int nsplit = it[kNSplit];
        if (nsplit <= 1) {
            const float inv = 1.f / lt;
#pragma unroll 1
            for (int c = 0; c < OCOLS / 32; ++c) {
                float o[32];
                tmem_ld32(lane_base + kTmemO + (uint32_t)(hs * OCOLS + c * 32), o);
                if (dst) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) =
                            make_uint4(pack_bf16(o[8 * q] * inv, o[8 * q + 1] * inv),
                                       pack_bf16(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                                       pack_bf16(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                                       pack_bf16(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
                }
            }
        } else {
            // one key piece of a split tile.  Its partial -- O / l in fp32
            // ([128 rows][d]), then the rows' base m[128] and sum l[128] -- goes
            // to global memory through a staging copy in the (now idle) ring
            // buffers, so that the stores are coalesced; the last piece to
            // arrive merges: out = sum_k O_k 2^(m_k - M) / sum_k l_k 2^(m_k - M),
            // its own O straight from TMEM and the others' copied into shared
            // memory with cp.async.  Shared rows hold 16-byte chunks in
            // XOR-swizzled order (chunk c of row r at c ^ (r & 7)): the row's
            // owner and a warp sweeping a row both access it conflict-free.
            constexpr int F4 = D / 4;              // 16-byte chunks per row
            constexpr int RPW = 32 / F4;           // rows per warp instruction when sweeping rows
            const int sub = lane / F4, c4 = lane % F4;
            const int piece = it[kPiece];
            const size_t piece_floats = (size_t)pf_piece_slots(G) * P.slot_floats;
            float* base = P.ws_part + (size_t)it[kSlot] * P.slot_floats;
            float* part = base + (size_t)piece * piece_floats;
            float4* stg = reinterpret_cast<float4*>(smem);
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll 1
            for (int c = 0; c < OCOLS / 32; ++c) {
                float o[32];
                tmem_ld32(lane_base + kTmemO + (uint32_t)(hs * OCOLS + c * 32), o);
                const int lc0 = (hs * OCOLS + c * 32) / 4;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    stg[r * F4 + ((lc0 + q) ^ (r & 7))] =
                        make_float4(o[4 * q] * inv, o[4 * q + 1] * inv, o[4 * q + 2] * inv, o[4 * q + 3] * inv);
            }
            if (hs == 0 && r < rows_valid) {
                __stcg(part + kTileRows * D + r, m_run);
                __stcg(part + kTileRows * D + kTileRows + r, lt);
            }
            __syncwarp();  // bar.sync wants converged warps
            asm volatile("bar.sync 10, 256;" ::: "memory");
            for (int rr = warp * RPW + sub; rr < rows_valid; rr += 8 * RPW)
                __stcg(reinterpret_cast<float4*>(part + (size_t)rr * D) + c4, stg[rr * F4 + (c4 ^ (rr & 7))]);
            int* s_last = reinterpret_cast<int*>(xsum + 2 * kTileRows);
            int* ticket = &P.ws_int[kHdrInts + P.n_flags + it[kMerge]];
            __threadfence();
            __syncwarp();  // bar.sync wants converged warps
            asm volatile("bar.sync 10, 256;" ::: "memory");
            if (tid == 0) {
                const int old = atomicAdd(ticket, 1);
                *s_last = old == nsplit - 1;
                if (old == nsplit - 1) __threadfence();
            }
            __syncwarp();  // bar.sync wants converged warps
            asm volatile("bar.sync 10, 256;" ::: "memory");
            if (*s_last) {
                // the other pieces' O / l into shared slots 0.. (the staging
                // copy is read out), and the m, l of this thread's row of every
                // piece.  The merge takes the pieces in index order, each from
                // its O / l (this piece's recomputed from TMEM: the same fp32
                // products it stored), so its bits do not depend on which
                // piece arrived last.
                float mk[kMaxPieces], lk[kMaxPieces];
#pragma unroll
                for (int k = 0; k < kMaxPieces; ++k) {
                    mk[k] = k == piece ? m_run : -INFINITY;
                    lk[k] = k == piece ? lt : 0.f;
                    if (k < nsplit && k != piece) {
                        const float* src = base + (size_t)k * piece_floats;
                        const uint32_t dsl = smem_u32(stg + (size_t)(k < piece ? k : k - 1) * kTileRows * F4);
                        for (int rr = warp * RPW + sub; rr < rows_valid; rr += 8 * RPW)
                            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                             dsl + (uint32_t)(rr * F4 + (c4 ^ (rr & 7))) * 16u),
                                         "l"(src + (size_t)rr * D + 4 * c4)
                                         : "memory");
                        if (r < rows_valid) {
                            mk[k] = __ldcg(src + kTileRows * D + r);
                            lk[k] = __ldcg(src + kTileRows * D + kTileRows + r);
                        }
                    }
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                __syncwarp();  // bar.sync wants converged warps
                asm volatile("bar.sync 10, 256;" ::: "memory");
                {
                    // every lane runs this (tcgen05.ld is warp-collective); only
                    // the rows of the tile's tokens are stored
                    float M = mk[0];
#pragma unroll
                    for (int k = 1; k < kMaxPieces; ++k) M = fmaxf(M, mk[k]);
                    float w[kMaxPieces], L = 0.f;
#pragma unroll
                    for (int k = 0; k < kMaxPieces; ++k) {
                        w[k] = mk[k] == -INFINITY ? 0.f : lk[k] * exp2f(mk[k] - M);
                        L += w[k];
                    }
                    const float invL = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
                    for (int k = 0; k < kMaxPieces; ++k) w[k] *= invL;
#pragma unroll 1
                    for (int c = 0; c < OCOLS / 32; ++c) {
                        float o[32];
                        tmem_ld32(lane_base + kTmemO + (uint32_t)(hs * OCOLS + c * 32), o);
                        const int lc0 = (hs * OCOLS + c * 32) / 4;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 own = make_float4(o[4 * q] * inv, o[4 * q + 1] * inv, o[4 * q + 2] * inv,
                                                           o[4 * q + 3] * inv);
                            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                            for (int k = 0; k < kMaxPieces; ++k) {
                                if (k < nsplit) {
                                    const float4 x =
                                        k == piece ? own
                                                   : stg[(size_t)(k < piece ? k : k - 1) * kTileRows * F4 + r * F4 +
                                                         ((lc0 + q) ^ (r & 7))];
                                    acc.x += x.x * w[k];
                                    acc.y += x.y * w[k];
                                    acc.z += x.z * w[k];
                                    acc.w += x.w * w[k];
                                }
                            }
                            o[4 * q] = acc.x;
                            o[4 * q + 1] = acc.y;
                            o[4 * q + 2] = acc.z;
                            o[4 * q + 3] = acc.w;
                        }
                        if (dst) {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) = make_uint4(
                                    pack_bf16(o[8 * q], o[8 * q + 1]), pack_bf16(o[8 * q + 2], o[8 * q + 3]),
                                    pack_bf16(o[8 * q + 4], o[8 * q + 5]), pack_bf16(o[8 * q + 6], o[8 * q + 7]));
                        }
                    }
                }
                if (tid == 0) *ticket = 0;
            }
        }
        tc_fence_before();
        // carried across items: the P.V groups not waited for above (the last
        // two blocks'), and the V loads per stage of this item
        for (int jj = max(nb - 2, 0); jj < nb; ++jj) ph_flip(ph, kPhOUp + (jj & 1));
#pragma unroll
        for (int st = 0; st < L::kVStages; ++st)
            if (((nb - st + L::kVStages - 1) / L::kVStages) & 1) ph_flip(ph, kPhVSeen + st);
    }
}

// ----------------------------------------------------------------------------
// DECODE split: pages [p0, p0+pc) of one decode for kv head g, all G q heads
// ----------------------------------------------------------------------------
template <int D, bool IL>
__device__ void run_decode(const KParams& P, const CUtensorMap* tmK, const CUtensorMap* tmV, const int* it,
                           uint8_t* smem, int* s_abort, int* s_flag, uint32_t& phase) {
    constexpr int HALVES = D / 64;
    constexpr int HALF = D / 2;
    constexpr int KPAGE = HALVES * kPageHalfBytes;  // one K page-head in smem
    constexpr int STAGE = 2 * KPAGE;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = it[kG], p0 = it[kStart], pc = it[kCount];
    const int slot_first = it[kSlot], merge = it[kMerge], nsplit = it[kNSplit];
    const Row R = row_geom(it);
    const int G = P.group;
    const int pos = R.kv_len - 1;   // the decode token's absolute position
    const bool last_owner = (p0 + pc == R.np);
    // the item's kv heads g .. g + ng - 1: warps WPH h .. WPH h + WPH - 1 stream
    // the pages of head g + h (warp place wq: pages p0 + wq, p0 + wq + WPH, ...)
    const int ng = min(kDecodeHeads, P.Hkv - g);
    constexpr int WPH = kDecWarps / kDecodeHeads;
    const int hw = warp / WPH, wq = warp % WPH;
    const bool streams = warp < kDecWarps && hw < ng;
    const int gh = g + (streams ? hw : 0);         // this warp's kv head
    constexpr int QBYTES = 16 * D * 2;              // one head's Q rows
    static_assert(kDecodeHeads * QBYTES <= kSmemStash - kSmemDecQ && kDecodeHeads * 2 * D * 2 <= kSmemBars - kSmemStash,
                  "decode Q tiles and stash");
    uint8_t* qtile = smem + kSmemDecQ + (streams ? hw : 0) * QBYTES;
    uint16_t* stash = reinterpret_cast<uint16_t*>(smem + kSmemStash) + (streams ? hw : 0) * 2 * D;
    uint8_t* wst = smem + warp * kDecStages * kDecStageBytes;
    const uint32_t wbar = smem_u32(smem + kSmemBars) + 8 * (kDecBar0 + kDecStages * warp);
    const int my_pages = (streams && pc > wq) ? (pc - wq + WPH - 1) / WPH : 0;

    // lane l holds the page id of this warp's page (32*window + l), so that
    // lane 0 never waits on a global load right before a TMA issue
    auto load_ids = [&](int base) -> int {
        const int k = base + lane;
        return k < my_pages ? page_id(P, R, p0 + wq + WPH * k, s_abort) : 0;
    };
    int ids = load_ids(0);
    auto issue = [&](int k, int page) {
        const int stg = k % kDecStages;
        const uint32_t dst = smem_u32(wst + stg * kDecStageBytes);
        const uint32_t bar = wbar + 8 * stg;
        mbar_expect_tx(bar, STAGE);
        const int y = (page * P.Hkv + gh) * kPage;
        if (HALVES == 2) {
            // one box per page-head: {64 columns, 16 rows, 2 halves} lands as
            // [half][16 rows][128 B], the same swizzled image as two 2-D boxes
            tma_load_3d(dst, tmK, 0, y, 0, bar);
            tma_load_3d(dst + KPAGE, tmV, 0, y, 0, bar);
        } else {
            tma_load_2d(dst, tmK, 0, y, bar);
            tma_load_2d(dst + KPAGE, tmV, 0, y, bar);
        }
    };
    // the first page id of every warp comes with the item: no load before it
    if (my_pages > 0 && lane == 0) issue(0, checked_page(P, it[kIds + wq], s_abort));
    for (int k = 1; k < my_pages && k < kDecStages; ++k) {
        const int pid = __shfl_sync(0xffffffffu, ids, k);
        if (lane == 0) issue(k, pid);
    }

    // Q rows of the group, RoPE'd in fp32, rows >= G zero: threads [0, QU) each
    // rotate 8 consecutive pairs (one round trip for the whole tile).
    constexpr int QU = 16 * (HALF / 8);
    static_assert(kDecodeHeads * QU <= kThreads, "decode prologue threads");
    if (tid < ng * QU) {
        const int h = tid / QU, t2 = tid % QU;
        const int row = t2 / (HALF / 8), c = t2 % (HALF / 8);
        const int c0 = IL ? 2 * c : c, c1 = IL ? 2 * c + 1 : c + HALF / 8;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
        if (row < G) {
            const uint4* qv = reinterpret_cast<const uint4*>(P.q + ((size_t)R.qo0 * P.Hq + (g + h) * G + row) * D);
            float cs[8], sn[8];
            load_rope_hi<HALF>(P.ropef + (size_t)pos * HALF * 4, c * 8, cs, sn);
            rope_q8(__ldg(qv + c0), __ldg(qv + c1), cs, sn, IL, lo, hi);
        }
        uint8_t* qt = smem + kSmemDecQ + h * QBYTES;
        *reinterpret_cast<uint4*>(qt + sw128_chunk(16, row, c0)) = lo;
        *reinterpret_cast<uint4*>(qt + sw128_chunk(16, row, c1)) = hi;
    }
    // the decode token's own K (fp64 RoPE, one rounding) and V: stash + page
    if (last_owner) {
        const int page = P.plan[P.off_kvi + R.kvp0 + pos / kPage];
        const bool ok = page >= 0 && page < P.num_pages && pos < P.rope_max_pos;
        uint16_t* stash0 = reinterpret_cast<uint16_t*>(smem + kSmemStash);
        for (int jh = tid; jh < ng * HALF; jh += kThreads) {
            const int h = jh / HALF, j = jh % HALF;
            const size_t off = (((size_t)(ok ? page : 0) * P.Hkv + g + h) * kPage + pos % kPage) * D;
            const uint16_t* kr = reinterpret_cast<const uint16_t*>(P.k) + ((size_t)R.qo0 * P.Hkv + g + h) * D;
            const int i0 = IL ? 2 * j : j, i1 = IL ? 2 * j + 1 : j + HALF;
            uint16_t y0 = 0, y1 = 0;
            if (ok) {
                const size_t ti = (size_t)pos * HALF + j;
                rope_pair(bf16_bits_to_float(kr[i0]), bf16_bits_to_float(kr[i1]),
                          rope_row_pair<HALF>(P.ropef + (size_t)pos * HALF * 4, j), P.rope + ti,
                          y0, y1);
                reinterpret_cast<uint16_t*>(P.k_cache)[off + i0] = y0;
                reinterpret_cast<uint16_t*>(P.k_cache)[off + i1] = y1;
            }
            stash0[h * 2 * D + i0] = y0;
            stash0[h * 2 * D + i1] = y1;
        }
        for (int eh = tid; eh < ng * D; eh += kThreads) {
            const int h = eh / D, e = eh % D;
            const size_t off = (((size_t)(ok ? page : 0) * P.Hkv + g + h) * kPage + pos % kPage) * D;
            const uint16_t vv = reinterpret_cast<const uint16_t*>(P.v)[((size_t)R.qo0 * P.Hkv + g + h) * D + e];
            stash0[h * 2 * D + D + e] = vv;
            if (ok) reinterpret_cast<uint16_t*>(P.v_cache)[off + e] = vv;
        }
        if (!ok && tid == 0) raise_error(P, kErrBounds, page, s_abort);
    }
    __syncthreads();

    const int mi = lane >> 3;
    // the Q fragments of every 16-wide k step, held for the whole item
    const int qrow = (mi & 1) * 8 + (lane & 7);
    uint32_t qf[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
        ldsm_x4(smem_u32(qtile + sw128_chunk(16, qrow, 2 * kk + (mi >> 1))), qf[kk][0], qf[kk][1], qf[kk][2],
                qf[kk][3]);
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    for (int k = 0; k < my_pages; ++k) {
        const int stg = k % kDecStages;
        mbar_wait_bounded(P, wbar + 8 * stg, (phase >> stg) & 1u, s_abort, k, it);
        phase ^= 1u << stg;
        uint8_t* kb = wst + stg * kDecStageBytes;
        uint8_t* vb = kb + KPAGE;
        const int lp = p0 + wq + WPH * k;
        const int key0 = lp * kPage;
        if (lp == R.np - 1) {
            // last page: put the new token in its slot, zero the slots past it
            const int slot = pos % kPage;
            for (int c = lane; c < 2 * kPage * (D / 8); c += 32) {
                const int which = c / (kPage * (D / 8));  // 0 = K, 1 = V
                const int rest = c % (kPage * (D / 8));
                const int row = rest / (D / 8), ch = rest % (D / 8);
                if (row < slot) continue;
                uint8_t* base = which ? vb : kb;
                uint4 val = make_uint4(0, 0, 0, 0);
                if (row == slot) val = *reinterpret_cast<const uint4*>(stash + which * D + ch * 8);
                *reinterpret_cast<uint4*>(base + sw128_chunk(kPage, row, ch)) = val;
            }
            __syncwarp();
        }
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int key = (mi >> 1) * 8 + (lane & 7);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(smem_u32(kb + sw128_chunk(kPage, key, 2 * kk + (mi & 1))), b0, b1, b2, b3);
            mma_bf16(sc[0], qf[kk], b0, b1);
            mma_bf16(sc[1], qf[kk], b2, b3);
        }
        float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + n * 8 + 2 * (lane & 3) + (e & 1);
                sc[n][e] = key < R.kv_len ? sc[n][e] * P.scale_log2 : -INFINITY;
            }
            mxA = fmaxf(mxA, fmaxf(sc[n][0], sc[n][1]));
            mxB = fmaxf(mxB, fmaxf(sc[n][2], sc[n][3]));
        }
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
        const float nmA = fmaxf(mA, mxA), nmB = fmaxf(mB, mxB);  // finite: every page has a key
        const float alA = exp2f(mA - nmA), alB = exp2f(mB - nmB);
        mA = nmA;
        mB = nmB;
        const float p00 = exp2f(sc[0][0] - nmA), p01 = exp2f(sc[0][1] - nmA);
        const float p02 = exp2f(sc[0][2] - nmB), p03 = exp2f(sc[0][3] - nmB);
        const float p10 = exp2f(sc[1][0] - nmA), p11 = exp2f(sc[1][1] - nmA);
        const float p12 = exp2f(sc[1][2] - nmB), p13 = exp2f(sc[1][3] - nmB);
        lA = lA * alA + (p00 + p01 + p10 + p11);
        lB = lB * alB + (p02 + p03 + p12 + p13);
        const uint32_t pa[4] = {pack_bf16(p00, p01), pack_bf16(p02, p03), pack_bf16(p10, p11), pack_bf16(p12, p13)};
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            o[n][0] *= alA;
            o[n][1] *= alA;
            o[n][2] *= alB;
            o[n][3] *= alB;
        }
#pragma unroll
        for (int np2 = 0; np2 < D / 16; ++np2) {
            const int key = (mi & 1) * 8 + (lane & 7);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(smem_u32(vb + sw128_chunk(kPage, key, 2 * np2 + (mi >> 1))), b0, b1, b2, b3);
            mma_bf16(o[2 * np2], pa, b0, b1);
            mma_bf16(o[2 * np2 + 1], pa, b2, b3);
        }
        __syncwarp();
        const int kn = k + kDecStages;
        if (kn < my_pages) {
            if ((kn & 31) == 0) ids = load_ids(kn);
            const int pid = __shfl_sync(0xffffffffu, ids, kn & 31);
            if (lane == 0) {
                fence_proxy_async_shared();
                issue(kn, pid);
            }
        }
    }
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);

    // in-CTA merge of the warps' (m, l, o) through the (now idle) stage memory
    __syncthreads();
    float* so = reinterpret_cast<float*>(smem);                 // [warp][16][D]
    float* sm = so + kDecWarps * 16 * D;                        // [warp][16]
    float* sl = sm + kDecWarps * 16;                            // [warp][16]
    if (warp < kDecWarps) {
        const int rA = lane >> 2, rB = rA + 8;
        float* ow = so + warp * 16 * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            const int col = n * 8 + 2 * (lane & 3);
            *reinterpret_cast<float2*>(ow + rA * D + col) = make_float2(o[n][0], o[n][1]);
            *reinterpret_cast<float2*>(ow + rB * D + col) = make_float2(o[n][2], o[n][3]);
        }
        if ((lane & 3) == 0) {
            sm[warp * 16 + rA] = mA;
            sm[warp * 16 + rB] = mB;
            sl[warp * 16 + rA] = lA;
            sl[warp * 16 + rB] = lB;
        }
    }
    __syncthreads();
    const bool single = slot_first < 0;
    const int ksplit = single ? 0 : p0 / ((R.np + nsplit - 1) / nsplit);
    // head h's streaming warps are WPH h .. WPH h + WPH - 1; split k of the
    // group writes head h's partial to slot slot_first + k ng + h
    for (int i = tid; i < ng * G * D; i += kThreads) {
        const int h = i / (G * D), row = (i / D) % G, col = i % D;
        float M = -INFINITY;
        for (int w = h * WPH; w < (h + 1) * WPH; ++w) M = fmaxf(M, sm[w * 16 + row]);
        float L = 0.f, acc = 0.f;
        for (int w = h * WPH; w < (h + 1) * WPH; ++w) {
            const float mw = sm[w * 16 + row];
            if (mw == -INFINITY) continue;
            const float sc = exp2f(mw - M);
            L += sl[w * 16 + row] * sc;
            acc += so[(w * 16 + row) * D + col] * sc;
        }
        const float val = acc / L;
        if (single) {
            P.out[((size_t)R.qo0 * P.Hq + (g + h) * G + row) * D + col] = __float2bfloat16_rn(val);
        } else {
            float* part = P.ws_part + (size_t)(slot_first + ksplit * ng + h) * P.slot_floats;
            part[row * (D + 2) + col] = val;
            if (col == 0) {
                part[row * (D + 2) + D] = M;
                part[row * (D + 2) + D + 1] = L;
            }
        }
    }
    if (single) return;
    // log-sum-exp merge across splits, done by the last split to arrive
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int old = atomicAdd(&P.ws_int[kHdrInts + P.n_flags + merge], 1);
        *s_flag = (old == nsplit - 1);
        if (*s_flag) __threadfence();
    }
    __syncthreads();
    if (!*s_flag) return;
    for (int i = tid; i < ng * G * D; i += kThreads) {
        const int h = i / (G * D), row = (i / D) % G, col = i % D;
        const float* base = P.ws_part + (size_t)(slot_first + h) * P.slot_floats;
        const size_t kstride = (size_t)ng * P.slot_floats;
        float M = -INFINITY;
        for (int k = 0; k < nsplit; ++k) M = fmaxf(M, __ldcg(base + k * kstride + row * (D + 2) + D));
        float L = 0.f, acc = 0.f;
        for (int k = 0; k < nsplit; ++k) {
            const float* pk = base + k * kstride + row * (D + 2);
            const float w = __ldcg(pk + D + 1) * exp2f(__ldcg(pk + D) - M);
            L += w;
            acc += __ldcg(pk + col) * w;
        }
        P.out[((size_t)R.qo0 * P.Hq + (g + h) * G + row) * D + col] = __float2bfloat16_rn(acc / L);
    }
    if (tid == 0) P.ws_int[kHdrInts + P.n_flags + merge] = 0;
}

// ----------------------------------------------------------------------------
// The persistent step kernel
// ----------------------------------------------------------------------------
// IL: interleaved RoPE pairing (x[2j], x[2j+1]) instead of rotate-half.
template <int D, bool IL>
__global__ void __launch_bounds__(kThreads, 1) mixed_step_kernel(const __grid_constant__ KParams P,
                                                                 const __grid_constant__ CUtensorMap tmK,
                                                                 const __grid_constant__ CUtensorMap tmV,
                                                                 const __grid_constant__ CUtensorMap tmK3,
                                                                 const __grid_constant__ CUtensorMap tmV3,
                                                                 const __grid_constant__ CUtensorMap tmK5,
                                                                 const __grid_constant__ CUtensorMap tmV5,
                                                                 const __grid_constant__ CUtensorMap tmQ,
                                                                 const __grid_constant__ CUtensorMap tmR,
                                                                 const __grid_constant__ CUtensorMap tmKin,
                                                                 const __grid_constant__ CUtensorMap tmVin,
                                                                 const __grid_constant__ CUtensorMap tmRA) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(16) int s_item[kItemInts];
    __shared__ int s_abort;
    __shared__ int s_flag;
    __shared__ uint32_t s_tmem;
    __shared__ uint32_t s_app_phase;
    __shared__ int s_fix[2];  // entries in the APPEND items' fix-up queue ([0]; [1] unused)
    const int tid = threadIdx.x;
    const uint32_t bars = smem_u32(smem + kSmemBars);
    if (tid == 0) {
        s_abort = 0;
        s_app_phase = 0;
        s_fix[0] = s_fix[1] = 0;
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t count = 1;
            if (i == kBarPFull || i == kBarPFull + 1 || i == kBarSFree || i == kBarSFree + 1)
                count = 256;  // the tile's softmax threads
            mbar_init(bars + 8 * i, count);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // tensor memory is taken when this CTA meets its first prefill item (one
    // CTA per SM: all of it); CTAs that only append and decode never hold it
    bool tmem_held = false;
    uint32_t tmem = 0;
    // completed-phase parities / counters, carried across work items
    uint32_t dec_phase = 0;
    PfPhase pf_phase = {};
    // CTAs below first_sms take items from the first queue (list positions
    // [0, n_first), head in header word 12) before the second (the rest, head
    // in word 0); the others the other way round.  A queue's head runs past its
    // end once it is empty; the last CTA out resets both.
    // The first round needs no atomic: CTA b takes item b of the queue it
    // prefers (b - first_sms of the second), and the heads count the claims
    // after those.
    const bool first_pref = (int)blockIdx.x < P.first_sms;
    const int n_second = P.n_items - P.n_first;
    const int stat1 = min(P.first_sms, P.n_first);                   // items of the first queue taken so
    const int stat2 = min((int)gridDim.x - P.first_sms, n_second);   // ... and of the second
    bool first_round = true;
    for (;;) {
        if (tid == 0) {
            int idx = -1;
            if (first_round) {
                const int b = (int)blockIdx.x;
                if (first_pref && b < P.n_first) idx = b;
                if (!first_pref && b - P.first_sms < n_second) idx = P.n_first + (b - P.first_sms);
            }
            for (int q = 0; q < 2 && idx < 0; ++q) {
                if ((q == 0) == first_pref) {
                    const int k = stat1 + atomicAdd(&P.ws_int[12], 1);
                    if (k < P.n_first) idx = k;
                } else {
                    const int k = stat2 + atomicAdd(&P.ws_int[0], 1);
                    if (k < n_second) idx = P.n_first + k;
                }
            }
            if (idx >= 0) {
                const int4* src = reinterpret_cast<const int4*>(P.plan + P.off_items + (size_t)idx * kItemInts);
                int4 v[kItemInts / 4];
#pragma unroll
                for (int i = 0; i < kItemInts / 4; ++i) v[i] = src[i];
#pragma unroll
                for (int i = 0; i < kItemInts / 4; ++i) reinterpret_cast<int4*>(s_item)[i] = v[i];
            } else {
                s_item[0] = -1;
            }
        }
        __syncthreads();
        first_round = false;
        const int* it = s_item;  // rewritten only after the end-of-item barrier
        if (it[0] < 0) break;
        if (it[0] == kAppend)
            run_append<D, IL>(P, &tmKin, &tmVin, &tmRA, it, smem, bars + 8 * kBarAppend, &s_app_phase, &s_abort, s_fix);
        else if (it[0] == kPrefill) {
            if (!tmem_held) {
                if (tid < 32) {
                    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                                     smem_u32(&s_tmem)),
                                 "r"(kTmemCols)
                                 : "memory");
                    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
                }
                tc_fence_before();
                __syncthreads();
                tc_fence_after();
                tmem_held = true;
                tmem = s_tmem;
            }
            run_prefill<D, IL>(P, &tmK, &tmV, &tmK5, &tmV5, &tmQ, &tmR, it, smem, &s_abort, pf_phase, tmem);
        }
        else
            run_decode<D, IL>(P, &tmK3, &tmV3, it, smem, &s_abort, &s_flag, dec_phase);
        // shared memory written through the generic proxy this item (tiles,
        // scratch, patched rows) is next overwritten by TMA
        fence_proxy_async_shared();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (s_abort) break;  // the error word is set; the workspace must be re-zeroed
    }
    if (tmem_held) {
        // no tensor-core work may be in flight when the tensor memory is released
        // (each MMA-issuing thread's commit covers the MMAs it issued)
        if (tid == 10 * 32 || tid == 11 * 32) {
            const uint32_t db = bars + 8 * (kBarDrain + (tid == 11 * 32 ? 1 : 0));
            umma_commit(db);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(db, 0))
                if (globaltimer() - t0 > kWaitNs) break;
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid < 32)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    if (s_abort) return;
    // the last CTA out leaves the counters at zero for the next launch
    if (tid == 0) {
        __threadfence();
        const int old = atomicAdd(&P.ws_int[1], 1);
        s_flag = (old == (int)gridDim.x - 1);
        if (s_flag) __threadfence();
    }
    __syncthreads();
    if (s_flag) {
        for (int i = tid; i < P.n_flags; i += kThreads) P.ws_int[kHdrInts + i] = 0;
        if (tid == 0) {
            P.ws_int[0] = 0;
            P.ws_int[1] = 0;
            P.ws_int[12] = 0;
        }
    }
}

// ----------------------------------------------------------------------------
// RoPE table: {cos, sin}(p * f_j) in fp64, f_j computed once on the host
// ----------------------------------------------------------------------------
struct InvFreq {
    double v[64];
};

__global__ void rope_table_kernel(double2* table, float* split, int max_pos, int half, const InvFreq f) {
    const int64_t total = (int64_t)max_pos * half;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int p = (int)(i / half), j = (int)(i % half);
        const double th = __dmul_rn((double)p, f.v[j]);
        double sn, cs;
        sincos(th, &sn, &cs);
        table[i] = make_double2(cs, sn);
        const float ch = __double2float_rn(cs), sh = __double2float_rn(sn);
        // row p: cos_hi[half], sin_hi[half], cos_lo[half], sin_lo[half]
        float* row = split + (size_t)p * half * 4;
        row[j] = ch;
        row[half + j] = sh;
        row[2 * half + j] = __double2float_rn(cs - (double)ch);
        row[3 * half + j] = __double2float_rn(sn - (double)sh);
    }
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
namespace {

int32_t cuda_fail(cudaError_t e, const char* what) {
    char msg[256];
    std::snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
    return fail(SARATHI_ERR_CUDA, msg);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D view of a page pool: rows = num_pages * H_kv * 16 tokens, columns = d.
// Box = 16 rows x 64 columns (one 128-byte swizzle span), 128-byte swizzle.
int32_t make_page_map(CUtensorMap* m, void* base, int num_pages, int Hkv, int d) {
    auto enc = encode_fn();
    if (!enc) return fail(SARATHI_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)num_pages * Hkv * kPage};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kPage};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[128];
        std::snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        return fail(SARATHI_ERR_CUDA, msg);
    }
    return SARATHI_OK;
}

// 3-D view of the same pool for d = 128: {64 columns, rows, 2 halves}, the
// halves 128 bytes apart.  Box = 64 x 16 x 2: one page-head (4 KB) per copy.
int32_t make_page_map3(CUtensorMap* m, void* base, int num_pages, int Hkv, int d) {
    auto enc = encode_fn();
    if (!enc) return fail(SARATHI_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[3] = {64, (cuuint64_t)num_pages * Hkv * kPage, (cuuint64_t)(d / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)kPage, (cuuint32_t)(d / 64)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[128];
        std::snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled (3-D page view) failed (%d)", (int)r);
        return fail(SARATHI_ERR_CUDA, msg);
    }
    return SARATHI_OK;
}

// 5-D view of the same pool: {64 columns, 16 slots, H_kv heads, pages, d/64
// halves} (strides 2 B, d*2, 16*d*2, H_kv*16*d*2 and 128 B).  Box = 64 x 16 x
// 1 x 8 x d/64: eight consecutive pages of one kv head (a whole 128-key block)
// in one copy, landing as [half][page][16 rows][128 B] like eight 2-D boxes.
int32_t make_page_map5(CUtensorMap* m, void* base, int num_pages, int Hkv, int d) {
    auto enc = encode_fn();
    if (!enc) return fail(SARATHI_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[5] = {64, (cuuint64_t)kPage, (cuuint64_t)Hkv, (cuuint64_t)num_pages, (cuuint64_t)(d / 64)};
    cuuint64_t strides[4] = {(cuuint64_t)d * 2, (cuuint64_t)kPage * d * 2, (cuuint64_t)Hkv * kPage * d * 2, 128};
    cuuint32_t box[5] = {64, (cuuint32_t)kPage, 1, (cuuint32_t)(kTileRows / kPage), (cuuint32_t)(d / 64)};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[128];
        std::snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled (5-D page view) failed (%d)", (int)r);
        return fail(SARATHI_ERR_CUDA, msg);
    }
    return SARATHI_OK;
}

// 3-D view of the step's queries q[T][H_q][d]: {d, H_q heads, T tokens}.  Box =
// 64 x G x (128 / G): the rows (token, q head of one GQA group) of one Q tile,
// token-major, landing as one 64-column half of the swizzled tile.
int32_t make_q_map(CUtensorMap* m, const void* q, int T, int Hq, int d, int G) {
    auto enc = encode_fn();
    if (!enc) return fail(SARATHI_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hq, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)Hq * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)tokens_per_tile(G)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[128];
        std::snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled (query view) failed (%d)", (int)r);
        return fail(SARATHI_ERR_CUDA, msg);
    }
    return SARATHI_OK;
}

// 2-D view of the fp32 RoPE table rows {max_pos rows, 2 d floats each}; box =
// the rows' first d floats (cos_hi and sin_hi) of `rows` (128 / G)
// consecutive positions: the table values one Q tile needs.
int32_t make_rope_map(CUtensorMap* m, const void* ropef, int max_pos, int d, int rows) {
    auto enc = encode_fn();
    if (!enc) return fail(SARATHI_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)d * 2, (cuuint64_t)max_pos};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2 * 4};
    cuuint32_t box[2] = {(cuuint32_t)d, (cuuint32_t)rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ropef), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[128];
        std::snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled (RoPE table view) failed (%d)", (int)r);
        return fail(SARATHI_ERR_CUDA, msg);
    }
    return SARATHI_OK;
}

// 3-D view of the step's new keys or values k[T][H_kv][d]: {d, T tokens, H_kv
// heads} (strides H_kv*d*2 and d*2 bytes).  Box = d x 16 x kAppendHeads: the
// rows of 16 tokens for a group of kv heads, landing head-major ([head][token]
// [d]) like the slots of a page.
int32_t make_kv_in_map(CUtensorMap* m, const void* x, int T, int Hkv, int d) {
    auto enc = encode_fn();
    if (!enc) return fail(SARATHI_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)Hkv};
    cuuint64_t strides[2] = {(cuuint64_t)Hkv * d * 2, (cuuint64_t)d * 2};
    cuuint32_t box[3] = {(cuuint32_t)d, (cuuint32_t)kPage, (cuuint32_t)kAppendHeads};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[128];
        std::snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled (new K/V view) failed (%d)", (int)r);
        return fail(SARATHI_ERR_CUDA, msg);
    }
    return SARATHI_OK;
}

// The step kernel instantiation for a head size and RoPE pairing.
const void* kernel_for(int d, int rope_style) {
    const bool il = rope_style == SARATHI_ROPE_INTERLEAVED;
    if (d == 128) return il ? (const void*)mixed_step_kernel<128, true> : (const void*)mixed_step_kernel<128, false>;
    return il ? (const void*)mixed_step_kernel<64, true> : (const void*)mixed_step_kernel<64, false>;
}

struct DevState {
    int sms = 0;
    bool smem_set[4] = {false, false, false, false};  // [d == 128][interleaved]
};
std::mutex g_mu;
DevState g_dev[128];

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace sarathi

using namespace sarathi;

extern "C" int32_t sarathi_rope_table(double* table, int32_t max_pos, int32_t head_dim, double rope_theta,
                                      void* cuda_stream) {
    if (!table || max_pos <= 0) return fail(SARATHI_ERR_INVALID_ARG, "table NULL or max_pos <= 0");
    if (head_dim <= 0 || (head_dim & 15) || head_dim / 2 > 64)
        return fail(SARATHI_ERR_UNSUPPORTED, "head_dim must be a multiple of 16 and <= 128");
    if (!(rope_theta > 0.0)) return fail(SARATHI_ERR_INVALID_ARG, "rope_theta must be positive");
    InvFreq f;
    std::memset(&f, 0, sizeof f);
    for (int j = 0; j < head_dim / 2; ++j) f.v[j] = std::pow(rope_theta, -(2.0 * (double)j) / (double)head_dim);
    const int64_t total = (int64_t)max_pos * (head_dim / 2);
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 8192);
    rope_table_kernel<<<blocks, 256, 0, (cudaStream_t)cuda_stream>>>(
        reinterpret_cast<double2*>(table), reinterpret_cast<float*>(table + (size_t)max_pos * head_dim), max_pos,
        head_dim / 2, f);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "rope_table launch");
    return SARATHI_OK;
}

namespace {
int32_t launch_step(const sarathi_attn_args* a, const sarathi_host_io* io, void* cuda_stream);
}

extern "C" int32_t sarathi_mixed_attn(const sarathi_attn_args* a, void* cuda_stream) {
    return launch_step(a, nullptr, cuda_stream);
}

extern "C" int32_t sarathi_mixed_attn_host(const sarathi_attn_args* a, const sarathi_host_io* io,
                                           void* cuda_stream) {
    if (!io) return fail(SARATHI_ERR_INVALID_ARG, "io is NULL");
    if (!io->q_host || !io->k_host || !io->v_host || !io->out_host)
        return fail(SARATHI_ERR_INVALID_ARG, "NULL host pointer");
    return launch_step(a, io, cuda_stream);
}

namespace {
int32_t launch_step(const sarathi_attn_args* a, const sarathi_host_io* io, void* cuda_stream) {
    if (!a) return fail(SARATHI_ERR_INVALID_ARG, "args is NULL");
    int32_t st = check_shape(&a->shape);
    if (st) return st;
    const sarathi_plan_info* in = a->info;
    if (!in) return fail(SARATHI_ERR_INVALID_ARG, "info is NULL");
    if (in->n_items == 0) {
        // an empty step: nothing to copy or run; its done event still follows the step before
        if (io && io->wait_event) {
            cudaError_t e = cudaStreamWaitEvent((cudaStream_t)cuda_stream, (cudaEvent_t)io->wait_event, 0);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
        }
        if (io && io->done_event) {
            cudaError_t e = cudaEventRecord((cudaEvent_t)io->done_event, (cudaStream_t)cuda_stream);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
        }
        return SARATHI_OK;
    }
    if (!a->q || !a->k || !a->v || !a->k_cache || !a->v_cache || !a->out || !a->plan || !a->rope_table ||
        !a->workspace)
        return fail(SARATHI_ERR_INVALID_ARG, "NULL device pointer");
    if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->out, 16) ||
        !aligned(a->k_cache, 16) || !aligned(a->v_cache, 16) || !aligned(a->plan, 16) || !aligned(a->rope_table, 16) ||
        !aligned(a->workspace, 256))
        return fail(SARATHI_ERR_INVALID_ARG, "misaligned pointer (tensors 16 B, workspace 256 B)");
    if (a->rope_style != SARATHI_ROPE_ROTATE_HALF && a->rope_style != SARATHI_ROPE_INTERLEAVED)
        return fail(SARATHI_ERR_INVALID_ARG, "rope_style must be SARATHI_ROPE_ROTATE_HALF or _INTERLEAVED");
    if (a->num_pages <= 0) return fail(SARATHI_ERR_INVALID_ARG, "num_pages must be positive");
    if (a->rope_max_pos < in->max_kv_len) return fail(SARATHI_ERR_CAPACITY, "RoPE table shorter than max_kv_len");
    if (a->workspace_bytes < in->workspace_bytes) return fail(SARATHI_ERR_CAPACITY, "workspace too small");
    if (in->n_sched <= 0 || in->packed_ints <= 0 || in->off_items < 0 || (in->off_items & 3) || in->n_first < 0 ||
        in->n_first > in->n_items || in->first_sms < 0)
        return fail(SARATHI_ERR_INVALID_ARG, "inconsistent plan info");
    const int d = a->shape.head_dim;
    const int Hkv = a->shape.num_heads_kv;
    if ((int64_t)a->num_pages * Hkv * kPage >= (int64_t)1 << 31)
        return fail(SARATHI_ERR_UNSUPPORTED, "page pool too large for 32-bit row coordinates");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 128) return fail(SARATHI_ERR_UNSUPPORTED, "device index >= 128");
    int sms = 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        DevState& ds = g_dev[dev];
        if (ds.sms == 0) {
            e = cudaDeviceGetAttribute(&ds.sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        }
        const int di = (d == 128 ? 2 : 0) + (a->rope_style == SARATHI_ROPE_INTERLEAVED ? 1 : 0);
        if (!ds.smem_set[di]) {
            const void* fn = kernel_for(d, a->rope_style);
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
            int resident = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, fn, kThreads, kSmemAlloc);
            if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
            if (resident < 1) return fail(SARATHI_ERR_CUDA, "step kernel does not fit one SM (registers/shared memory)");
            ds.smem_set[di] = true;
        }
        sms = ds.sms;
    }
    CUtensorMap tmK, tmV;
    st = make_page_map(&tmK, a->k_cache, a->num_pages, Hkv, d);
    if (st) return st;
    st = make_page_map(&tmV, a->v_cache, a->num_pages, Hkv, d);
    if (st) return st;
    CUtensorMap tmQ;
    st = make_q_map(&tmQ, a->q, in->num_tokens, a->shape.num_heads_q, d, a->shape.num_heads_q / Hkv);
    if (st) return st;
    CUtensorMap tmKin, tmVin, tmRA;
    st = make_kv_in_map(&tmKin, a->k, in->num_tokens, Hkv, d);
    if (st) return st;
    st = make_kv_in_map(&tmVin, a->v, in->num_tokens, Hkv, d);
    if (st) return st;
    st = make_rope_map(&tmRA, a->rope_table + (size_t)a->rope_max_pos * d, a->rope_max_pos, d, kPage);
    if (st) return st;
    CUtensorMap tmR;
    st = make_rope_map(&tmR, a->rope_table + (size_t)a->rope_max_pos * d, a->rope_max_pos, d,
                       tokens_per_tile(a->shape.num_heads_q / Hkv));
    if (st) return st;
    CUtensorMap tmK5, tmV5;
    st = make_page_map5(&tmK5, a->k_cache, a->num_pages, Hkv, d);
    if (st) return st;
    st = make_page_map5(&tmV5, a->v_cache, a->num_pages, Hkv, d);
    if (st) return st;
    CUtensorMap tmK3 = tmK, tmV3 = tmV;
    if (d == 128) {
        st = make_page_map3(&tmK3, a->k_cache, a->num_pages, Hkv, d);
        if (st) return st;
        st = make_page_map3(&tmV3, a->v_cache, a->num_pages, Hkv, d);
        if (st) return st;
    }

    KParams P;
    P.q = static_cast<const __nv_bfloat16*>(a->q);
    P.k = static_cast<const __nv_bfloat16*>(a->k);
    P.v = static_cast<const __nv_bfloat16*>(a->v);
    P.k_cache = static_cast<__nv_bfloat16*>(a->k_cache);
    P.v_cache = static_cast<__nv_bfloat16*>(a->v_cache);
    P.out = static_cast<__nv_bfloat16*>(a->out);
    P.plan = a->plan;
    P.off_qo = in->off_qo_indptr;
    P.off_kvp = in->off_kv_page_indptr;
    P.off_kvi = in->off_kv_page_indices;
    P.off_last = in->off_kv_last_page_len;
    P.off_aux = in->off_req_aux;
    P.off_items = in->off_items;
    P.n_items = in->n_items;
    P.n_first = in->n_first;
    P.n_sched = in->n_sched;
    P.n_flags = (int)flag_ints(in->n_sched, in->num_tokens, Hkv);
    P.rope = reinterpret_cast<const double2*>(a->rope_table);
    P.ropef = reinterpret_cast<const float*>(a->rope_table + (size_t)a->rope_max_pos * d);
    P.rope_max_pos = a->rope_max_pos;
    P.ws_int = static_cast<int32_t*>(a->workspace);
    P.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(a->workspace) +
                                         partial_offset_bytes(in->n_sched, in->n_merge, in->num_tokens, Hkv));
    P.Hq = a->shape.num_heads_q;
    P.Hkv = Hkv;
    P.group = a->shape.num_heads_q / Hkv;
    P.num_pages = a->num_pages;
    P.scale_log2 = a->sm_scale * 1.4426950408889634f;
    P.slot_floats = (int)partial_slot_floats(P.group, d);

    const int grid = std::min(sms, in->n_items);
    // at least one CTA prefers the second queue whenever it holds items (its
    // APPEND items must be taken while first-queue tiles may wait for them)
    P.first_sms = in->n_first < in->n_items ? std::min(in->first_sms, grid - 1) : grid;
    cudaStream_t stream = (cudaStream_t)cuda_stream;
    const size_t q_bytes = (size_t)in->num_tokens * a->shape.num_heads_q * d * 2;
    const size_t kv_bytes = (size_t)in->num_tokens * Hkv * d * 2;
    if (io) {
        // this step's new tokens, from the host
        e = cudaMemcpyAsync(const_cast<void*>(a->q), io->q_host, q_bytes, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(const_cast<void*>(a->k), io->k_host, kv_bytes, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(const_cast<void*>(a->v), io->v_host, kv_bytes, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "q, k, v copy to the device");
    }
    if (a->plan_host) {
        // the caller's host copy of the plan goes to the device first, on the same stream
        e = cudaMemcpyAsync(const_cast<int32_t*>(a->plan), a->plan_host, (size_t)in->packed_ints * 4,
                            cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "plan copy to the device");
    }
    if (io && io->wait_event) {
        e = cudaStreamWaitEvent(stream, (cudaEvent_t)io->wait_event, 0);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
    }
    const bool il = a->rope_style == SARATHI_ROPE_INTERLEAVED;
    if (d == 128 && !il)
        mixed_step_kernel<128, false><<<grid, kThreads, kSmemAlloc, stream>>>(P, tmK, tmV, tmK3, tmV3, tmK5, tmV5, tmQ, tmR, tmKin,
                                                                                  tmVin, tmRA);
    else if (d == 128)
        mixed_step_kernel<128, true><<<grid, kThreads, kSmemAlloc, stream>>>(P, tmK, tmV, tmK3, tmV3, tmK5, tmV5, tmQ, tmR, tmKin,
                                                                                  tmVin, tmRA);
    else if (!il)
        mixed_step_kernel<64, false><<<grid, kThreads, kSmemAlloc, stream>>>(P, tmK, tmV, tmK3, tmV3, tmK5, tmV5, tmQ, tmR, tmKin,
                                                                                  tmVin, tmRA);
    else
        mixed_step_kernel<64, true><<<grid, kThreads, kSmemAlloc, stream>>>(P, tmK, tmV, tmK3, tmV3, tmK5, tmV5, tmQ, tmR, tmKin,
                                                                                  tmVin, tmRA);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "mixed_step_kernel launch");
    if (io) {
        if (io->done_event) {
            e = cudaEventRecord((cudaEvent_t)io->done_event, stream);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
        }
        e = cudaMemcpyAsync(io->out_host, a->out, q_bytes, cudaMemcpyDeviceToHost, stream);
        if (e != cudaSuccess) return cuda_fail(e, "out copy to the host");
    }
    return SARATHI_OK;
}
}  // namespace

extern "C" int32_t sarathi_workspace_status(void* workspace, void* cuda_stream, int32_t* device_error) {
    if (!workspace || !device_error) return fail(SARATHI_ERR_INVALID_ARG, "NULL pointer");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)cuda_stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int32_t w = 0;
    e = cudaMemcpy(&w, static_cast<int32_t*>(workspace) + 2, sizeof w, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
    *device_error = w;
    if (w) {
        const int32_t zero = 0;
        e = cudaMemcpy(static_cast<int32_t*>(workspace) + 2, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
        return fail(SARATHI_ERR_DEVICE_CHECK, "the step kernel flagged an error; re-zero the workspace");
    }
    return SARATHI_OK;
}
