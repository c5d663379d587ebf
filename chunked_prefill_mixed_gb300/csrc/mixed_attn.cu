// mixed_attn.cu -- the step kernel of libsarathi (sm_103a) and its launcher.
//
// One persistent launch runs the whole mixed-batch attention step that chunked
// prefill with stall-free batching produces ("Sarathi-Serve 完全拆解", §"混合批不是
// 把两类注意力强行做成同一个形状": one ragged batch, attention split back per
// request through qo_indptr / kv_page_indptr / kv_page_indices /
// kv_last_page_len).  CTAs pull work items from the planner's list through an
// atomic head counter, longest items first:
//
//   APPEND   new prefill tokens: K rotated at its ABSOLUTE position in fp64 and
//            rounded once to bf16, V copied, both into the page that holds the
//            position ("Sarathi-Serve 完全拆解", §"分块不等于截断上下文": RoPE never
//            restarts per chunk; the chunk's K/V land in the paged cache).
//   PREFILL  one tile of up to 128 query rows (token x q-head of one GQA group)
//            of a chunk: causal attention over every history page plus the
//            chunk's own keys (ibid.: o_i = sum_{j<=i} softmax(q_i.k_j/sqrt d) v_j).
//            Waits (bounded) until the request's APPEND items are done, then
//            streams 64-key blocks of pages into shared memory with TMA.
//   DECODE   one split of a decode's pages for one kv head: per-warp TMA page
//            pipelines, warp-level MMA for the GQA group, online softmax,
//            in-CTA merge, and across splits a log-sum-exp merge done by the
//            last split to arrive (atomic ticket, no spinning).  The split that
//            owns the last page also appends the decode token's K/V.
//
// No CTA waits on a CTA that took a later item, and the only cross-CTA wait
// (PREFILL on its request's APPENDs, which precede it in the list) is bounded
// by a timer; a wait that runs out sets an error word in the workspace.
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
    const double2* rope;  // [max_pos][d/2] {cos, sin}
    int rope_max_pos;
    int32_t* ws_int;      // header, append counters, merge tickets
    float* ws_part;       // split partials
    int Hq, Hkv, group, num_pages;
    float scale_log2;     // sm_scale * log2(e)
    int slot_floats;
};

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kDecStages = 3;                                  // per-warp page ring
constexpr int kPageHalfBytes = kPage * 128;                    // 16 rows x 64 bf16
constexpr int kDecStageBytes = 2 * 2 * kPageHalfBytes;         // K+V page-head, d=128
constexpr int kSmemStages = kWarps * kDecStages * kDecStageBytes;  // 192 KB
constexpr int kSmemDecQ = kSmemStages;                         // 16 x 128 bf16
constexpr int kSmemStash = kSmemDecQ + 2 * kPageHalfBytes;     // new K/V (2 x 128 bf16)
constexpr int kSmemBars = kSmemStash + 512;                   // mbarriers, initialised once
constexpr int kDecBar0 = 0;                                    // [warp][stage] decode rings
constexpr int kPfBar0 = kWarps * kDecStages;                   // prefill ring
constexpr int kSmemBytes = kSmemBars + 256;
constexpr int kSmemAlloc = kSmemBytes + 1024;                  // + alignment slack
// prefill layout inside the stage region
constexpr int kPfBlockKeys = 64;
constexpr int kPfStages = 3;
constexpr int kPfQBytes = 2 * kTileRows * 128;                 // 128 rows x 128 bf16
constexpr int kPfStageBytes = 2 * 2 * kPfBlockKeys * 128;      // K+V, 64 keys x 128
static_assert(kPfQBytes + kPfStages * kPfStageBytes <= kSmemStages, "prefill smem");
static_assert(kWarps * 16 * 128 * 4 + 2 * kWarps * 16 * 4 <= kSmemStages, "merge scratch");
static_assert(kSmemAlloc <= 227 * 1024, "shared memory per CTA");

constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s bound on any wait

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
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
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
// header words 3..11 for the host to read.
__device__ bool mbar_wait_bounded(const KParams& P, uint32_t bar, uint32_t parity, int* s_abort, int detail,
                                  const int* it) {
    for (int i = 0; i < 256; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
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

struct Row {
    int qo0, n, kvp0, np, kv_len, h;
};
__device__ __forceinline__ Row row_geom(const KParams& P, int s) {
    Row r;
    const int32_t* pl = P.plan;
    r.qo0 = pl[P.off_qo + s];
    r.n = pl[P.off_qo + s + 1] - r.qo0;
    r.kvp0 = pl[P.off_kvp + s];
    r.np = pl[P.off_kvp + s + 1] - r.kvp0;
    r.kv_len = (r.np - 1) * kPage + pl[P.off_last + s];
    r.h = r.kv_len - r.n;
    return r;
}

// Physical page id of a request-local page, checked against the pool.
__device__ __forceinline__ int page_id(const KParams& P, const Row& R, int lp, int* s_abort) {
    const int page = P.plan[P.off_kvi + R.kvp0 + lp];
    if (page < 0 || page >= P.num_pages) {
        raise_error(P, kErrBounds, page, s_abort);
        return 0;
    }
    return page;
}

// Rotate (x0, x1) = (k_j, k_{j+d/2}) by the table angle in fp64, one rounding
// per product and sum (no contraction), exactly as written:
//   y0 = x0 cos - x1 sin,  y1 = x1 cos + x0 sin.
__device__ __forceinline__ void rope_pair_fp64(double x0, double x1, double2 cs, uint16_t& y0, uint16_t& y1) {
    double a = __dsub_rn(__dmul_rn(x0, cs.x), __dmul_rn(x1, cs.y));
    double b = __dadd_rn(__dmul_rn(x1, cs.x), __dmul_rn(x0, cs.y));
    y0 = bf16_from_double(a);
    y1 = bf16_from_double(b);
}

// ----------------------------------------------------------------------------
// APPEND: rotate + store the K/V of up to kAppendTokens prefill tokens
// ----------------------------------------------------------------------------
template <int D>
__device__ void run_append(const KParams& P, const int* it, int* s_abort) {
    const int tid = threadIdx.x;
    const int s = it[kS], t0 = it[kStart], cnt = it[kCount];
    const Row R = row_geom(P, s);
    const int Hkv = P.Hkv;
    constexpr int HALF = D / 2;
    const uint16_t* kin = reinterpret_cast<const uint16_t*>(P.k);
    uint16_t* kc = reinterpret_cast<uint16_t*>(P.k_cache);
    const int totk = cnt * Hkv * HALF;
    for (int i = tid; i < totk; i += kThreads) {
        const int j = i % HALF;
        const int rest = i / HALF;
        const int g = rest % Hkv;
        const int t = t0 + rest / Hkv;
        const int pos = R.h + t;
        const int page = P.plan[P.off_kvi + R.kvp0 + pos / kPage];
        if (page < 0 || page >= P.num_pages || pos >= P.rope_max_pos) {
            raise_error(P, kErrBounds, page, s_abort);
            continue;
        }
        const uint16_t* kr = kin + ((size_t)(R.qo0 + t) * Hkv + g) * D;
        uint16_t y0, y1;
        rope_pair_fp64((double)bf16_bits_to_float(kr[j]), (double)bf16_bits_to_float(kr[j + HALF]),
                       P.rope[(size_t)pos * HALF + j], y0, y1);
        uint16_t* dst = kc + (((size_t)page * Hkv + g) * kPage + pos % kPage) * D;
        dst[j] = y0;
        dst[j + HALF] = y1;
    }
    const int totv = cnt * Hkv * (D / 8);
    for (int i = tid; i < totv; i += kThreads) {
        const int c = i % (D / 8);
        const int rest = i / (D / 8);
        const int g = rest % Hkv;
        const int t = t0 + rest / Hkv;
        const int pos = R.h + t;
        const int page = P.plan[P.off_kvi + R.kvp0 + pos / kPage];
        if (page < 0 || page >= P.num_pages) continue;
        const uint4* src = reinterpret_cast<const uint4*>(P.v + ((size_t)(R.qo0 + t) * Hkv + g) * D) + c;
        uint4* dst = reinterpret_cast<uint4*>(P.v_cache + (((size_t)page * Hkv + g) * kPage + pos % kPage) * D) + c;
        *dst = __ldg(src);
    }
    // publish: the pages are read next by TMA (async proxy) in other CTAs
    fence_proxy_async_global();
    __threadfence();
    __syncthreads();
    if (tid == 0) atomicAdd(&P.ws_int[kHdrInts + s], 1);
}

// ----------------------------------------------------------------------------
// PREFILL tile: up to 128 rows (token-major, q-head-in-group minor) of one
// chunk for one kv head, causal over history pages + the chunk.
// ----------------------------------------------------------------------------
template <int D>
__device__ void run_prefill(const KParams& P, const CUtensorMap* tmK, const CUtensorMap* tmV, const int* it,
                            uint8_t* smem, int* s_abort, uint32_t& phase) {
    constexpr int HALVES = D / 64;
    constexpr int HALF = D / 2;
    constexpr int KBLK_HALF = kPfBlockKeys * 128;  // one column half of a 64-key block
    constexpr int K_BYTES = HALVES * KBLK_HALF;
    constexpr int STAGE = 2 * K_BYTES;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = it[kS], g = it[kG], t0 = it[kStart], cnt = it[kCount];
    const Row R = row_geom(P, s);
    const int G = P.group;
    const int rows_valid = cnt * G;
    const int kv_hi = R.h + t0 + cnt;                 // keys [0, kv_hi) are visible to some row
    const int nblk = (kv_hi + kPfBlockKeys - 1) / kPfBlockKeys;
    const int pages_hi = (kv_hi + kPage - 1) / kPage;
    uint8_t* qtile = smem;
    uint8_t* stages = smem + kPfQBytes;
    const uint32_t bars = smem_u32(smem + kSmemBars) + 8 * kPfBar0;

    // 1. the chunk's K/V must be in the pages: wait for this request's APPENDs
    if (tid == 0) {
        const int need = P.plan[P.off_aux + s];
        const int* ctr = &P.ws_int[kHdrInts + s];
        if (ld_acquire(ctr) < need) {
            const uint64_t w0 = globaltimer();
            while (ld_acquire(ctr) < need) {
                if (globaltimer() - w0 > kWaitNs) {
                    raise_error(P, kErrWait, -1 - s, s_abort);
                    break;
                }
                __nanosleep(100);
            }
        }
        fence_proxy_async_global();
    }
    __syncthreads();
    if (*(volatile int*)s_abort) return;

    auto issue = [&](int b) {
        const int stg = b % kPfStages;
        uint8_t* kb = stages + stg * STAGE;
        const uint32_t bar = bars + 8 * stg;
        int npg = 0;
        for (int i = 0; i < kPfBlockKeys / kPage; ++i) npg += (b * 4 + i < pages_hi);
        mbar_expect_tx(bar, npg * HALVES * kPageHalfBytes * 2);
        for (int i = 0; i < kPfBlockKeys / kPage; ++i) {
            const int lp = b * 4 + i;
            if (lp >= pages_hi) break;
            const int page = page_id(P, R, lp, s_abort);
            const int y = (page * P.Hkv + g) * kPage;
            for (int hf = 0; hf < HALVES; ++hf) {
                tma_load_2d(smem_u32(kb + hf * KBLK_HALF + i * kPageHalfBytes), tmK, hf * 64, y, bar);
                tma_load_2d(smem_u32(kb + K_BYTES + hf * KBLK_HALF + i * kPageHalfBytes), tmV, hf * 64, y, bar);
            }
        }
    };
    if (tid == 0)
        for (int b = 0; b < nblk && b < kPfStages; ++b) issue(b);

    // 2. Q rows, RoPE'd in fp32 at their absolute positions, into the tile
    for (int i = tid; i < kTileRows * HALF; i += kThreads) {
        const int row = i / HALF, j = i % HALF;
        float y0 = 0.f, y1 = 0.f;
        if (row < rows_valid) {
            const int t = t0 + row / G;
            const int hq = g * G + row % G;
            const int pos = R.h + t;
            const __nv_bfloat16* qr = P.q + ((size_t)(R.qo0 + t) * P.Hq + hq) * D;
            const float x0 = __bfloat162float(qr[j]), x1 = __bfloat162float(qr[j + HALF]);
            const double2 cs = P.rope[(size_t)pos * HALF + j];
            const float c = (float)cs.x, sn = (float)cs.y;
            y0 = x0 * c - x1 * sn;
            y1 = x1 * c + x0 * sn;
        }
        *reinterpret_cast<__nv_bfloat16*>(qtile + sw128_off(kTileRows, row, j)) = __float2bfloat16_rn(y0);
        *reinterpret_cast<__nv_bfloat16*>(qtile + sw128_off(kTileRows, row, j + HALF)) = __float2bfloat16_rn(y1);
    }
    __syncthreads();

    const int wrow0 = warp * 16;
    const bool active = wrow0 < rows_valid;
    const int mi = lane >> 3;
    uint32_t qa[D / 16][4];
    {
        const int row = wrow0 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            ldsm_x4(smem_u32(qtile + sw128_chunk(kTileRows, row, 2 * kk + (mi >> 1))), qa[kk][0], qa[kk][1],
                    qa[kk][2], qa[kk][3]);
    }
    // absolute positions of this thread's two rows (invalid rows mimic the last)
    const int rA = wrow0 + (lane >> 2), rB = rA + 8;
    const int posA = R.h + t0 + (rA < rows_valid ? rA / G : cnt - 1);
    const int posB = R.h + t0 + (rB < rows_valid ? rB / G : cnt - 1);
    const int pos_min = R.h + t0 + wrow0 / G;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    for (int b = 0; b < nblk; ++b) {
        const int stg = b % kPfStages;
        mbar_wait_bounded(P, bars + 8 * stg, (phase >> stg) & 1u, s_abort, b, it);
        phase ^= 1u << stg;
        uint8_t* kb = stages + stg * STAGE;
        uint8_t* vb = kb + K_BYTES;
        const int key0 = b * kPfBlockKeys;
        if (key0 + kPfBlockKeys > kv_hi) {
            // keys past kv_hi hold stale bytes: zero them so 0-weight x V stays 0
            const int first = kv_hi - key0;
            const int nbytes = (kPfBlockKeys - first) * 128;
            for (int hf = 0; hf < 2 * HALVES; ++hf) {
                uint8_t* base = kb + hf * KBLK_HALF + first * 128;
                for (int i = tid * 16; i < nbytes; i += kThreads * 16)
                    *reinterpret_cast<uint4*>(base + i) = make_uint4(0, 0, 0, 0);
            }
            __syncthreads();
        }
        if (active) {
            float sc[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
                for (int np2 = 0; np2 < 4; ++np2) {
                    const int key = np2 * 16 + (mi >> 1) * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_u32(kb + sw128_chunk(kPfBlockKeys, key, 2 * kk + (mi & 1))), b0, b1, b2, b3);
                    mma_bf16(sc[2 * np2], qa[kk], b0, b1);
                    mma_bf16(sc[2 * np2 + 1], qa[kk], b2, b3);
                }
            }
            const bool need_mask = key0 + kPfBlockKeys - 1 > pos_min;
            float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float v = sc[n][e] * P.scale_log2;
                    if (need_mask) {
                        const int key = key0 + n * 8 + 2 * (lane & 3) + (e & 1);
                        if (key > (e < 2 ? posA : posB)) v = -INFINITY;
                    }
                    sc[n][e] = v;
                }
                mxA = fmaxf(mxA, fmaxf(sc[n][0], sc[n][1]));
                mxB = fmaxf(mxB, fmaxf(sc[n][2], sc[n][3]));
            }
            mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
            mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
            mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
            mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
            const float nmA = fmaxf(mA, mxA), nmB = fmaxf(mB, mxB);
            // a row sees no key of a block only when it already saw block 0
            const float baseA = nmA == -INFINITY ? 0.f : nmA;
            const float baseB = nmB == -INFINITY ? 0.f : nmB;
            const float alA = exp2f(mA - baseA), alB = exp2f(mB - baseB);
            mA = nmA;
            mB = nmB;
            float sumA = 0.f, sumB = 0.f;
            uint32_t pa[4][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const float p0 = exp2f(sc[n][0] - baseA), p1 = exp2f(sc[n][1] - baseA);
                const float p2 = exp2f(sc[n][2] - baseB), p3 = exp2f(sc[n][3] - baseB);
                sumA += p0 + p1;
                sumB += p2 + p3;
                pa[n >> 1][(n & 1) * 2 + 0] = pack_bf16(p0, p1);
                pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2, p3);
            }
            lA = lA * alA + sumA;
            lB = lB * alB + sumB;
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                o[n][0] *= alA;
                o[n][1] *= alA;
                o[n][2] *= alB;
                o[n][3] *= alB;
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                for (int np2 = 0; np2 < D / 16; ++np2) {
                    const int key = ks * 16 + (mi & 1) * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_u32(vb + sw128_chunk(kPfBlockKeys, key, 2 * np2 + (mi >> 1))), b0, b1, b2, b3);
                    mma_bf16(o[2 * np2], pa[ks], b0, b1);
                    mma_bf16(o[2 * np2 + 1], pa[ks], b2, b3);
                }
            }
        }
        __syncthreads();
        if (tid == 0 && b + kPfStages < nblk) {
            fence_proxy_async_shared();
            issue(b + kPfStages);
        }
    }
    if (!active) return;
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    const float invA = 1.f / lA, invB = 1.f / lB;
    if (rA < rows_valid) {
        __nv_bfloat16* dst = P.out + ((size_t)(R.qo0 + t0 + rA / G) * P.Hq + g * G + rA % G) * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
            *reinterpret_cast<uint32_t*>(dst + n * 8 + 2 * (lane & 3)) = pack_bf16(o[n][0] * invA, o[n][1] * invA);
    }
    if (rB < rows_valid) {
        __nv_bfloat16* dst = P.out + ((size_t)(R.qo0 + t0 + rB / G) * P.Hq + g * G + rB % G) * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
            *reinterpret_cast<uint32_t*>(dst + n * 8 + 2 * (lane & 3)) = pack_bf16(o[n][2] * invB, o[n][3] * invB);
    }
}

// ----------------------------------------------------------------------------
// DECODE split: pages [p0, p0+pc) of one decode for kv head g, all G q heads
// ----------------------------------------------------------------------------
template <int D>
__device__ void run_decode(const KParams& P, const CUtensorMap* tmK, const CUtensorMap* tmV, const int* it,
                           uint8_t* smem, int* s_abort, int* s_flag, uint32_t& phase) {
    constexpr int HALVES = D / 64;
    constexpr int HALF = D / 2;
    constexpr int KPAGE = HALVES * kPageHalfBytes;  // one K page-head in smem
    constexpr int STAGE = 2 * KPAGE;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = it[kS], g = it[kG], p0 = it[kStart], pc = it[kCount];
    const int slot_first = it[kSlot], merge = it[kMerge], nsplit = it[kNSplit];
    const Row R = row_geom(P, s);
    const int G = P.group;
    const int pos = R.kv_len - 1;   // the decode token's absolute position
    const bool last_owner = (p0 + pc == R.np);
    uint8_t* qtile = smem + kSmemDecQ;
    uint16_t* stash = reinterpret_cast<uint16_t*>(smem + kSmemStash);
    uint8_t* wst = smem + warp * kDecStages * kDecStageBytes;
    const uint32_t wbar = smem_u32(smem + kSmemBars) + 8 * (kDecBar0 + kDecStages * warp);
    const int my_pages = pc > warp ? (pc - warp + kWarps - 1) / kWarps : 0;

    auto issue = [&](int k) {
        const int lp = p0 + warp + kWarps * k;
        const int page = page_id(P, R, lp, s_abort);
        const int stg = k % kDecStages;
        const uint32_t dst = smem_u32(wst + stg * kDecStageBytes);
        const uint32_t bar = wbar + 8 * stg;
        mbar_expect_tx(bar, STAGE);
        const int y = (page * P.Hkv + g) * kPage;
        for (int hf = 0; hf < HALVES; ++hf) {
            tma_load_2d(dst + hf * kPageHalfBytes, tmK, hf * 64, y, bar);
            tma_load_2d(dst + KPAGE + hf * kPageHalfBytes, tmV, hf * 64, y, bar);
        }
    };
    if (lane == 0)
        for (int k = 0; k < my_pages && k < kDecStages; ++k) issue(k);

    // Q rows of the group, RoPE'd in fp32, rows >= G zero
    for (int i = tid; i < 16 * HALF; i += kThreads) {
        const int row = i / HALF, j = i % HALF;
        float y0 = 0.f, y1 = 0.f;
        if (row < G) {
            const __nv_bfloat16* qr = P.q + ((size_t)R.qo0 * P.Hq + g * G + row) * D;
            const float x0 = __bfloat162float(qr[j]), x1 = __bfloat162float(qr[j + HALF]);
            const double2 cs = P.rope[(size_t)pos * HALF + j];
            const float c = (float)cs.x, sn = (float)cs.y;
            y0 = x0 * c - x1 * sn;
            y1 = x1 * c + x0 * sn;
        }
        *reinterpret_cast<__nv_bfloat16*>(qtile + sw128_off(16, row, j)) = __float2bfloat16_rn(y0);
        *reinterpret_cast<__nv_bfloat16*>(qtile + sw128_off(16, row, j + HALF)) = __float2bfloat16_rn(y1);
    }
    // the decode token's own K (fp64 RoPE, one rounding) and V: stash + page
    if (last_owner) {
        const int page = P.plan[P.off_kvi + R.kvp0 + pos / kPage];
        const bool ok = page >= 0 && page < P.num_pages && pos < P.rope_max_pos;
        const size_t off = (((size_t)(ok ? page : 0) * P.Hkv + g) * kPage + pos % kPage) * D;
        const uint16_t* kr = reinterpret_cast<const uint16_t*>(P.k) + ((size_t)R.qo0 * P.Hkv + g) * D;
        const uint16_t* vr = reinterpret_cast<const uint16_t*>(P.v) + ((size_t)R.qo0 * P.Hkv + g) * D;
        for (int j = tid; j < HALF; j += kThreads) {
            uint16_t y0 = 0, y1 = 0;
            if (ok) {
                rope_pair_fp64((double)bf16_bits_to_float(kr[j]), (double)bf16_bits_to_float(kr[j + HALF]),
                               P.rope[(size_t)pos * HALF + j], y0, y1);
                reinterpret_cast<uint16_t*>(P.k_cache)[off + j] = y0;
                reinterpret_cast<uint16_t*>(P.k_cache)[off + j + HALF] = y1;
            }
            stash[j] = y0;
            stash[j + HALF] = y1;
        }
        for (int e = tid; e < D; e += kThreads) {
            const uint16_t vv = vr[e];
            stash[D + e] = vv;
            if (ok) reinterpret_cast<uint16_t*>(P.v_cache)[off + e] = vv;
        }
        if (!ok && tid == 0) raise_error(P, kErrBounds, page, s_abort);
    }
    __syncthreads();

    const int mi = lane >> 3;
    uint32_t qa[D / 16][4];
    {
        const int row = (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            ldsm_x4(smem_u32(qtile + sw128_chunk(16, row, 2 * kk + (mi >> 1))), qa[kk][0], qa[kk][1], qa[kk][2],
                    qa[kk][3]);
    }
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
        const int lp = p0 + warp + kWarps * k;
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
            mma_bf16(sc[0], qa[kk], b0, b1);
            mma_bf16(sc[1], qa[kk], b2, b3);
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
        if (lane == 0 && k + kDecStages < my_pages) {
            fence_proxy_async_shared();
            issue(k + kDecStages);
        }
    }
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);

    // in-CTA merge of the warps' (m, l, o) through the (now idle) stage memory
    __syncthreads();
    float* so = reinterpret_cast<float*>(smem);                 // [warp][16][D]
    float* sm = so + kWarps * 16 * D;                           // [warp][16]
    float* sl = sm + kWarps * 16;                               // [warp][16]
    {
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
    float* part = single ? nullptr : P.ws_part + (size_t)(slot_first + ksplit) * P.slot_floats;
    for (int i = tid; i < G * D; i += kThreads) {
        const int row = i / D, col = i % D;
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm[w * 16 + row]);
        float L = 0.f, acc = 0.f;
        for (int w = 0; w < kWarps; ++w) {
            const float mw = sm[w * 16 + row];
            if (mw == -INFINITY) continue;
            const float sc = exp2f(mw - M);
            L += sl[w * 16 + row] * sc;
            acc += so[(w * 16 + row) * D + col] * sc;
        }
        const float val = acc / L;
        if (single) {
            P.out[((size_t)R.qo0 * P.Hq + g * G + row) * D + col] = __float2bfloat16_rn(val);
        } else {
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
        const int old = atomicAdd(&P.ws_int[kHdrInts + P.n_sched + merge], 1);
        *s_flag = (old == nsplit - 1);
        if (*s_flag) __threadfence();
    }
    __syncthreads();
    if (!*s_flag) return;
    const float* base = P.ws_part + (size_t)slot_first * P.slot_floats;
    for (int i = tid; i < G * D; i += kThreads) {
        const int row = i / D, col = i % D;
        float M = -INFINITY;
        for (int k = 0; k < nsplit; ++k) M = fmaxf(M, __ldcg(base + (size_t)k * P.slot_floats + row * (D + 2) + D));
        float L = 0.f, acc = 0.f;
        for (int k = 0; k < nsplit; ++k) {
            const float* pk = base + (size_t)k * P.slot_floats + row * (D + 2);
            const float w = __ldcg(pk + D + 1) * exp2f(__ldcg(pk + D) - M);
            L += w;
            acc += __ldcg(pk + col) * w;
        }
        P.out[((size_t)R.qo0 * P.Hq + g * G + row) * D + col] = __float2bfloat16_rn(acc / L);
    }
    if (tid == 0) P.ws_int[kHdrInts + P.n_sched + merge] = 0;
}

// ----------------------------------------------------------------------------
// The persistent step kernel
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads, 1) mixed_step_kernel(const __grid_constant__ KParams P,
                                                                 const __grid_constant__ CUtensorMap tmK,
                                                                 const __grid_constant__ CUtensorMap tmV) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ int s_item[kItemInts];
    __shared__ int s_abort;
    __shared__ int s_flag;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_abort = 0;
        const uint32_t bars = smem_u32(smem + kSmemBars);
        for (int i = 0; i < kPfBar0 + kPfStages; ++i) mbar_init(bars + 8 * i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // completed-phase parity of each ring stage, carried across work items
    uint32_t pf_phase = 0, dec_phase = 0;
    for (;;) {
        if (tid == 0) {
            const int idx = atomicAdd(&P.ws_int[0], 1);
            if (idx < P.n_items) {
                const int4* src = reinterpret_cast<const int4*>(P.plan + P.off_items + (size_t)idx * kItemInts);
                const int4 a = src[0], b = src[1];
                s_item[0] = a.x;
                s_item[1] = a.y;
                s_item[2] = a.z;
                s_item[3] = a.w;
                s_item[4] = b.x;
                s_item[5] = b.y;
                s_item[6] = b.z;
                s_item[7] = b.w;
            } else {
                s_item[0] = -1;
            }
        }
        __syncthreads();
        int it[kItemInts];
#pragma unroll
        for (int i = 0; i < kItemInts; ++i) it[i] = s_item[i];
        if (it[0] < 0) break;
        if (it[0] == kAppend)
            run_append<D>(P, it, &s_abort);
        else if (it[0] == kPrefill)
            run_prefill<D>(P, &tmK, &tmV, it, smem, &s_abort, pf_phase);
        else
            run_decode<D>(P, &tmK, &tmV, it, smem, &s_abort, &s_flag, dec_phase);
        // shared memory written through the generic proxy this item (tiles,
        // scratch, patched rows) is next overwritten by TMA
        fence_proxy_async_shared();
        __syncthreads();
        if (s_abort) return;  // the error word is set; the workspace must be re-zeroed
    }
    // the last CTA out leaves the counters at zero for the next launch
    if (tid == 0) {
        __threadfence();
        const int old = atomicAdd(&P.ws_int[1], 1);
        s_flag = (old == (int)gridDim.x - 1);
        if (s_flag) __threadfence();
    }
    __syncthreads();
    if (s_flag) {
        for (int i = tid; i < P.n_sched; i += kThreads) P.ws_int[kHdrInts + i] = 0;
        if (tid == 0) {
            P.ws_int[0] = 0;
            P.ws_int[1] = 0;
        }
    }
}

// ----------------------------------------------------------------------------
// RoPE table: {cos, sin}(p * f_j) in fp64, f_j computed once on the host
// ----------------------------------------------------------------------------
struct InvFreq {
    double v[64];
};

__global__ void rope_table_kernel(double2* table, int max_pos, int half, const InvFreq f) {
    const int64_t total = (int64_t)max_pos * half;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int p = (int)(i / half), j = (int)(i % half);
        const double th = __dmul_rn((double)p, f.v[j]);
        double sn, cs;
        sincos(th, &sn, &cs);
        table[i] = make_double2(cs, sn);
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

struct DevState {
    int sms = 0;
    bool smem_set[2] = {false, false};
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
    if (head_dim <= 0 || (head_dim & 1) || head_dim / 2 > 64)
        return fail(SARATHI_ERR_UNSUPPORTED, "head_dim must be even and <= 128");
    if (!(rope_theta > 0.0)) return fail(SARATHI_ERR_INVALID_ARG, "rope_theta must be positive");
    InvFreq f;
    std::memset(&f, 0, sizeof f);
    for (int j = 0; j < head_dim / 2; ++j) f.v[j] = std::pow(rope_theta, -(2.0 * (double)j) / (double)head_dim);
    const int64_t total = (int64_t)max_pos * (head_dim / 2);
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 8192);
    rope_table_kernel<<<blocks, 256, 0, (cudaStream_t)cuda_stream>>>(reinterpret_cast<double2*>(table), max_pos,
                                                                      head_dim / 2, f);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "rope_table launch");
    return SARATHI_OK;
}

extern "C" int32_t sarathi_mixed_attn(const sarathi_attn_args* a, void* cuda_stream) {
    if (!a) return fail(SARATHI_ERR_INVALID_ARG, "args is NULL");
    int32_t st = check_shape(&a->shape);
    if (st) return st;
    const sarathi_plan_info* in = a->info;
    if (!in) return fail(SARATHI_ERR_INVALID_ARG, "info is NULL");
    if (in->n_items == 0) return SARATHI_OK;
    if (!a->q || !a->k || !a->v || !a->k_cache || !a->v_cache || !a->out || !a->plan || !a->rope_table ||
        !a->workspace)
        return fail(SARATHI_ERR_INVALID_ARG, "NULL device pointer");
    if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->out, 16) ||
        !aligned(a->k_cache, 16) || !aligned(a->v_cache, 16) || !aligned(a->plan, 16) || !aligned(a->workspace, 256))
        return fail(SARATHI_ERR_INVALID_ARG, "misaligned pointer (tensors 16 B, workspace 256 B)");
    if (a->num_pages <= 0) return fail(SARATHI_ERR_INVALID_ARG, "num_pages must be positive");
    if (a->rope_max_pos < in->max_kv_len) return fail(SARATHI_ERR_CAPACITY, "RoPE table shorter than max_kv_len");
    if (a->workspace_bytes < in->workspace_bytes) return fail(SARATHI_ERR_CAPACITY, "workspace too small");
    if (in->n_sched <= 0 || in->packed_ints <= 0 || in->off_items < 0 || (in->off_items & 3))
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
        const int di = d == 128 ? 1 : 0;
        if (!ds.smem_set[di]) {
            e = d == 128 ? cudaFuncSetAttribute(mixed_step_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                kSmemAlloc)
                         : cudaFuncSetAttribute(mixed_step_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                kSmemAlloc);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
            ds.smem_set[di] = true;
        }
        sms = ds.sms;
    }
    CUtensorMap tmK, tmV;
    st = make_page_map(&tmK, a->k_cache, a->num_pages, Hkv, d);
    if (st) return st;
    st = make_page_map(&tmV, a->v_cache, a->num_pages, Hkv, d);
    if (st) return st;

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
    P.n_sched = in->n_sched;
    P.rope = reinterpret_cast<const double2*>(a->rope_table);
    P.rope_max_pos = a->rope_max_pos;
    P.ws_int = static_cast<int32_t*>(a->workspace);
    P.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(a->workspace) +
                                         partial_offset_bytes(in->n_sched, in->n_merge));
    P.Hq = a->shape.num_heads_q;
    P.Hkv = Hkv;
    P.group = a->shape.num_heads_q / Hkv;
    P.num_pages = a->num_pages;
    P.scale_log2 = a->sm_scale * 1.4426950408889634f;
    P.slot_floats = (int)partial_slot_floats(P.group, d);

    const int grid = std::min(sms, in->n_items);
    cudaStream_t stream = (cudaStream_t)cuda_stream;
    if (d == 128)
        mixed_step_kernel<128><<<grid, kThreads, kSmemAlloc, stream>>>(P, tmK, tmV);
    else
        mixed_step_kernel<64><<<grid, kThreads, kSmemAlloc, stream>>>(P, tmK, tmV);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "mixed_step_kernel launch");
    return SARATHI_OK;
}

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
