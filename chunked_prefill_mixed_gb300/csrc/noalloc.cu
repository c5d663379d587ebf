// noalloc.cu -- sarathi_mixed_attn_noalloc: the same step kernel, with its
// scratch memory (work-queue counters, split-KV partials) taken from a fixed
// array that the library owns, so the caller never has to allocate any.
//
// Some callers cannot allocate device memory at the moment they run the step:
// a plugin living inside a host process whose allocator has already claimed
// the GPU's memory, or a serving loop that forbids any allocation once it has
// started.  They still pass inputs and outputs; this entry point supplies the
// scratch.
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdio>
#include <mutex>

#include "sarathi.h"
#include "sarathi_internal.h"

namespace sarathi {
namespace {

constexpr size_t kStaticScratchBytes = (size_t)8 << 20;  // 8 MiB, held by every GPU that loads the library

// Host code must not use this name as an address: it is only a host-side
// stand-in.  The device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_step_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_dev[128] = {};  // device address of g_step_scratch, per device index

// The array's device address on the current device, looked up once per device.
int32_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SARATHI_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= 128) return fail(SARATHI_ERR_UNSUPPORTED, "device index >= 128");
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_dev[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_step_scratch);
        if (e != cudaSuccess || !p) {
            char msg[200];
            std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
            return fail(SARATHI_ERR_CUDA, msg);
        }
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return SARATHI_OK;
}

}  // namespace
}  // namespace sarathi

using namespace sarathi;

extern "C" int32_t sarathi_mixed_attn_noalloc(const sarathi_attn_args* args, void* cuda_stream) {
    if (!args || !args->info) return fail(SARATHI_ERR_INVALID_ARG, "args or args->info is NULL");
    const sarathi_plan_info* in = args->info;
    if (in->workspace_bytes < 0 || (uint64_t)in->workspace_bytes > kStaticScratchBytes) {
        char msg[200];
        std::snprintf(msg, sizeof msg,
                      "this batch needs %lld bytes of scratch but the built-in array holds %zu; "
                      "use sarathi_mixed_attn with a caller workspace",
                      (long long)in->workspace_bytes, kStaticScratchBytes);
        return fail(SARATHI_ERR_CAPACITY, msg);
    }
    if (in->n_items == 0) return SARATHI_OK;
    // The counters cleared below sit in front of the partial slots; their size
    // comes from n_sched and n_merge, so both are checked against the array
    // before anything is enqueued (an inconsistent plan info must not make the
    // memset run past the array).
    if (in->n_sched <= 0 || in->n_merge < 0 || in->n_partials < 0 || in->n_items < 0 || in->num_tokens < 0)
        return fail(SARATHI_ERR_INVALID_ARG, "inconsistent plan info (n_sched, n_merge, n_partials or n_items)");
    const int32_t st = check_shape(&args->shape);
    if (st) return st;
    const int64_t clear_bytes =
        partial_offset_bytes(in->n_sched, in->n_merge, in->num_tokens, args->shape.num_heads_kv);
    const int64_t need = clear_bytes + (int64_t)in->n_partials *
                                           partial_slot_floats(args->shape.num_heads_q / args->shape.num_heads_kv,
                                                               args->shape.head_dim) * 4;
    if (need > in->workspace_bytes)
        return fail(SARATHI_ERR_INVALID_ARG, "inconsistent plan info (counters and partials exceed its workspace_bytes)");
    void* scratch = nullptr;
    const int32_t sa = scratch_address(&scratch);
    if (sa) return sa;
    // The array keeps whatever the previous call left.  The counters, tickets
    // and error word must start at zero; the partial slots are always written
    // before they are read.
    const cudaError_t e = cudaMemsetAsync(scratch, 0, (size_t)clear_bytes, (cudaStream_t)cuda_stream);
    if (e != cudaSuccess) return fail(SARATHI_ERR_CUDA, cudaGetErrorString(e));
    sarathi_attn_args a = *args;
    a.workspace = scratch;
    a.workspace_bytes = (int64_t)kStaticScratchBytes;
    return sarathi_mixed_attn(&a, cuda_stream);
}

extern "C" int32_t sarathi_noalloc_status(void* cuda_stream, int32_t* device_error) {
    if (!device_error) return fail(SARATHI_ERR_INVALID_ARG, "NULL pointer");
    void* scratch = nullptr;
    const int32_t sa = scratch_address(&scratch);
    if (sa) return sa;
    return sarathi_workspace_status(scratch, cuda_stream, device_error);
}
