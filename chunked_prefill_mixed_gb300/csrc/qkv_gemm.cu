// qkv_gemm.cu -- the QKV projection of a mixed batch as ONE tensor-core GEMM.
//
// "Sarathi：让解码搭上 prefill 的顺风车" §"Decode-maximal batching：顺车的账本":
// the linear layers of the prefill chunk and of the decodes run as one matrix
// product over the concatenated tokens, so the weights are read from memory
// once for both ("Sarathi-Serve 完全拆解" §"混合批不是把两类注意力强行做成同一个
// 形状": the linear-layer inputs are concatenated along the token dimension
// into one ragged batch).  Here that product is the Q/K/V projection that feeds
// the step kernel:
//   Y[T][N] = X[T][hidden] . W[N][hidden]^T,  N = (H_q + 2 H_kv) d,
// with Y's columns [0, H_q d) written as q [T][H_q][d], the next H_kv d as k,
// the last H_kv d as v -- the step's input layouts.
//
// sm_103a design: a persistent kernel, one CTA per SM, 128 x 256 output tiles
// (tcgen05.mma M 128, N 256, K 16; fp32 accumulators in TMEM, two of 256
// columns so that the epilogue of one tile overlaps the MMAs of the next), a
// 4-stage ring of 64-wide K slices moved by TMA (A 16 KB + B 32 KB a stage, the
// 128-byte swizzle the MMA descriptors read).  Warp 0 issues the TMA loads,
// warp 1 the MMAs, warps 2-5 read the accumulators out (one row per thread)
// and store bf16.  Tiles go to CTAs round-robin, M fastest, so the CTAs
// running at the same time share one W slab through L2.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "sarathi.h"
#include "sarathi_internal.h"

namespace sarathi {
namespace qkv {

constexpr int kBM = 128, kBK = 64;             // tile rows and K slice
constexpr int kABytes = kBM * kBK * 2;         // 16 KB
constexpr int kThreads = 192;                  // 6 warps
constexpr unsigned long long kWaitNs = 2000000000ull;
// Tile width BN (128, 192 or 256): as many stages of A 16 KB + B BN x 128 B as
// fit 200 KB (6 at 128, 5 at 192, 4 at 256).
template <int BN>
struct Tile {
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = (200 * 1024) / kStageBytes;
    static constexpr int kSmemBars = kStages * kStageBytes;
    static constexpr int kSmemAlloc = kSmemBars + 256 + 1024;  // barriers + alignment slack
    // barriers: full / empty per stage, accumulator full / empty per TMEM buffer, drain
    static constexpr int kBarFull = 0, kBarEmpty = kStages, kBarAccFull = 2 * kStages;
    static constexpr int kBarAccEmpty = 2 * kStages + 2, kBarDrain = 2 * kStages + 4, kNumBars = kBarDrain + 1;
    static_assert(kSmemAlloc <= 227 * 1024, "shared memory per CTA");
    static_assert(kNumBars * 8 <= 256, "barrier area");
    static_assert(BN % 32 == 0 && BN <= 256 && 2 * BN <= 512, "MMA N and TMEM columns");
};

struct Params {
    __nv_bfloat16* q;
    __nv_bfloat16* k;
    __nv_bfloat16* v;
    int T, hidden, N, Nq, Nk;   // Nq = H_q d, Nk = H_kv d
    int mt, nt;                 // tiles along M and N
    int32_t* status;            // workspace error word (index 2) and detail (3)
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
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
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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
// Bounded wait: gives up after kWaitNs, records the wait's code and sets the
// CTA's abort flag; every later wait then returns at once.
__device__ __noinline__ bool wait_slow(const Params& P, uint32_t bar, uint32_t parity, int code, int* s_abort) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (*(volatile int*)s_abort) return false;
        if (globaltimer() - t0 > kWaitNs) {
            if (atomicCAS(&P.status[2], 0, kErrWait) == 0) P.status[3] = code;
            *(volatile int*)s_abort = 1;
            return false;
        }
    }
    return true;
}
__device__ __forceinline__ bool wait_bounded(const Params& P, uint32_t bar, uint32_t parity, int code, int* s_abort) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(P, bar, parity, code, s_abort);
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// Shared-memory matrix descriptor (start, leading / stride byte offsets in
// 16-byte units, descriptor version 1, 128-byte swizzle).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B (both
// K-major), N and M as given.
__host__ __device__ constexpr uint32_t umma_idesc(int n, int m) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]),
          "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]),
          "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]),
          "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) asm volatile("" : "+f"(v[i]));
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) qkv_kernel(const __grid_constant__ Params P,
                                                          const __grid_constant__ CUtensorMap tmX,
                                                          const __grid_constant__ CUtensorMap tmW) {
    using TL = Tile<BN>;
    constexpr int kBN = BN, kStages = TL::kStages, kStageBytes = TL::kStageBytes, kSmemBars = TL::kSmemBars;
    constexpr int kBarFull = TL::kBarFull, kBarEmpty = TL::kBarEmpty, kBarAccFull = TL::kBarAccFull;
    constexpr int kBarAccEmpty = TL::kBarAccEmpty, kBarDrain = TL::kBarDrain, kNumBars = TL::kNumBars;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bars = smem_u32(smem + kSmemBars);
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < kNumBars; ++i)
            mbar_init(bar(i), (i >= kBarAccEmpty && i < kBarAccEmpty + 2) ? 128u : 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&s_tmem))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int ntiles = P.mt * P.nt;
    const int ks_n = P.hidden / kBK;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            uint32_t it = 0;
            for (int tile = blockIdx.x; tile < ntiles && !*(volatile int*)&s_abort; tile += gridDim.x) {
                const int m = tile % P.mt, n = tile / P.mt;
                for (int ks = 0; ks < ks_n; ++ks, ++it) {
                    const int st = (int)(it % kStages);
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!wait_bounded(P, bar(kBarEmpty + st), ph ^ 1u, 1, &s_abort)) break;
                    uint8_t* a = smem + st * kStageBytes;
                    mbar_expect_tx(bar(kBarFull + st), kStageBytes);
                    tma_load_2d(smem_u32(a), &tmX, ks * kBK, m * kBM, bar(kBarFull + st));
                    tma_load_2d(smem_u32(a + kABytes), &tmW, ks * kBK, n * kBN, bar(kBarFull + st));
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc(kBN, kBM);
            uint32_t it = 0, tl = 0;
            for (int tile = blockIdx.x; tile < ntiles && !*(volatile int*)&s_abort; tile += gridDim.x, ++tl) {
                const uint32_t b = tl & 1u, aph = (tl >> 1) & 1u;
                wait_bounded(P, bar(kBarAccEmpty + b), aph ^ 1u, 2, &s_abort);
                tc_fence_after();
                const uint32_t d = tmem + b * kBN;
                for (int ks = 0; ks < ks_n; ++ks, ++it) {
                    const int st = (int)(it % kStages);
                    const uint32_t ph = (it / kStages) & 1u;
                    wait_bounded(P, bar(kBarFull + st), ph, 3, &s_abort);
                    tc_fence_after();
                    const uint8_t* a = smem + st * kStageBytes;
                    const uint64_t ad = umma_desc(smem_u32(a), 16, 1024);
                    const uint64_t bd = umma_desc(smem_u32(a + kABytes), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)  // 32 bytes a step inside the 128-byte swizzle span
                        umma_f16(d, ad + (uint64_t)((kk * 32) >> 4), bd + (uint64_t)((kk * 32) >> 4), idesc,
                                 (ks > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(bar(kBarEmpty + st));
                }
                umma_commit(bar(kBarAccFull + b));
            }
            // nothing of the tensor pipe may be in flight when TMEM is released
            umma_commit(bar(kBarDrain));
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(bar(kBarDrain), 0))
                if (globaltimer() - t0 > kWaitNs) break;
        }
    } else {
        // ---------------- epilogue: warps 2-5, one accumulator row per thread ----------------
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        uint32_t tl = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tl) {
            const int m = tile % P.mt, n = tile / P.mt;
            const uint32_t b = tl & 1u, ph = (tl >> 1) & 1u;
            if (!wait_bounded(P, bar(kBarAccFull + b), ph, 4, &s_abort)) break;
            tc_fence_after();
            const int row = m * kBM + r;
#pragma unroll 1
            for (int c = 0; c < kBN / 32; ++c) {
                float o[32];
                tmem_ld32(lane_base + b * kBN + (uint32_t)(c * 32), o);
                const int col = n * kBN + c * 32;
                if (row < P.T && col < P.N) {
                    // a 32-column chunk lies inside one head of one of q, k, v
                    __nv_bfloat16* dst = col < P.Nq ? P.q + (size_t)row * P.Nq + col
                                       : col < P.Nq + P.Nk ? P.k + (size_t)row * P.Nk + (col - P.Nq)
                                                           : P.v + (size_t)row * P.Nk + (col - P.Nq - P.Nk);
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd)
                        reinterpret_cast<uint4*>(dst)[qd] =
                            make_uint4(pack_bf16(o[8 * qd], o[8 * qd + 1]), pack_bf16(o[8 * qd + 2], o[8 * qd + 3]),
                                       pack_bf16(o[8 * qd + 4], o[8 * qd + 5]),
                                       pack_bf16(o[8 * qd + 6], o[8 * qd + 7]));
                }
            }
            tc_fence_before();
            mbar_arrive(bar(kBarAccEmpty + b));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
}

}  // namespace qkv
}  // namespace sarathi

// ----------------------------------------------------------------------------
// host
// ----------------------------------------------------------------------------
namespace {

using sarathi::fail;

int32_t cuda_err(cudaError_t e, const char* what) {
    char msg[192];
    std::snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
    return fail(SARATHI_ERR_CUDA, msg);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// Row-major bf16 [rows][cols] matrix; box = box_rows x 64 columns, 128-byte
// swizzle; rows past the end read as zero.
int32_t make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    auto enc = encoder();
    if (!enc) return fail(SARATHI_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[96];
        std::snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        return fail(SARATHI_ERR_CUDA, msg);
    }
    return SARATHI_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct Dev {
    int sms = 0;
    bool ready = false;
};
std::mutex g_mu;
Dev g_devs[128];

}  // namespace

extern "C" int32_t sarathi_qkv_proj(const sarathi_qkv_args* a, void* cuda_stream) {
    using namespace sarathi::qkv;
    if (!a || !a->x || !a->w || !a->q || !a->k || !a->v || !a->workspace)
        return fail(SARATHI_ERR_INVALID_ARG, "NULL pointer");
    const int Hq = a->shape.num_heads_q, Hkv = a->shape.num_heads_kv, d = a->shape.head_dim;
    if (Hq <= 0 || Hkv <= 0 || d <= 0 || d % 32 != 0)
        return fail(SARATHI_ERR_INVALID_ARG, "heads must be positive and head_dim a multiple of 32");
    if (a->tokens <= 0 || a->hidden <= 0 || a->hidden % kBK != 0)
        return fail(SARATHI_ERR_INVALID_ARG, "tokens must be positive and hidden a multiple of 64");
    if (!aligned16(a->x) || !aligned16(a->w) || !aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) ||
        !aligned16(a->workspace))
        return fail(SARATHI_ERR_INVALID_ARG, "misaligned pointer (16 bytes)");
    Params P;
    P.q = static_cast<__nv_bfloat16*>(a->q);
    P.k = static_cast<__nv_bfloat16*>(a->k);
    P.v = static_cast<__nv_bfloat16*>(a->v);
    P.T = a->tokens;
    P.hidden = a->hidden;
    P.Nq = Hq * d;
    P.Nk = Hkv * d;
    P.N = P.Nq + 2 * P.Nk;
    P.mt = (P.T + kBM - 1) / kBM;
    P.status = static_cast<int32_t*>(a->workspace);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
    if (dev < 0 || dev >= 128) return fail(SARATHI_ERR_UNSUPPORTED, "device index out of range");
    int sms;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        Dev& ds = g_devs[dev];
        if (!ds.ready) {
            e = cudaDeviceGetAttribute(&ds.sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return cuda_err(e, "cudaDeviceGetAttribute");
            for (int w = 0; w < 3; ++w) {
                const void* fn = w == 0 ? (const void*)qkv_kernel<128>
                               : w == 1 ? (const void*)qkv_kernel<192> : (const void*)qkv_kernel<256>;
                const int bytes = w == 0 ? Tile<128>::kSmemAlloc : w == 1 ? Tile<192>::kSmemAlloc : Tile<256>::kSmemAlloc;
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
                if (e != cudaSuccess) return cuda_err(e, "cudaFuncSetAttribute");
                int resident = 0;
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, fn, kThreads, bytes);
                if (e != cudaSuccess) return cuda_err(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
                if (resident < 1) return fail(SARATHI_ERR_CUDA, "QKV kernel does not fit one SM");
            }
            ds.ready = true;
        }
        sms = ds.sms;
    }
    // Tile width: the one whose waves of tiles over the SMs move the fewest
    // operand bytes per SM (a tile's K slice is 16 KB of X plus BN x 128 B of W),
    // the wider one on ties.  At 512 tokens x 6144 columns 192 fills one wave
    // with 128 tiles where 256 leaves 56 SMs idle.  (A 224-wide tile, four
    // stages deep, measured slower than both at 2048 tokens and is not used.)
    auto cost = [&](int bn) {
        const long long tiles = (long long)P.mt * ((P.N + bn - 1) / bn);
        return ((tiles + sms - 1) / sms) * (long long)(kABytes + bn * kBK * 2);
    };
    int BN = 256;
    for (int bn : {192, 128})
        if (cost(bn) < cost(BN)) BN = bn;
    P.nt = (P.N + BN - 1) / BN;
    CUtensorMap tmX, tmW;
    int32_t st = make_map(&tmX, a->x, P.T, P.hidden, kBM);
    if (st) return st;
    st = make_map(&tmW, a->w, P.N, P.hidden, BN);
    if (st) return st;
    const int tiles = P.mt * P.nt;
    const int grid = tiles < sms ? tiles : sms;
    cudaStream_t strm = (cudaStream_t)cuda_stream;
    if (BN == 128)
        qkv_kernel<128><<<grid, kThreads, Tile<128>::kSmemAlloc, strm>>>(P, tmX, tmW);
    else if (BN == 192)
        qkv_kernel<192><<<grid, kThreads, Tile<192>::kSmemAlloc, strm>>>(P, tmX, tmW);
    else
        qkv_kernel<256><<<grid, kThreads, Tile<256>::kSmemAlloc, strm>>>(P, tmX, tmW);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_err(e, "qkv_kernel launch");
    sarathi::set_error("");
    return SARATHI_OK;
}
