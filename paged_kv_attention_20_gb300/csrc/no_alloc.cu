// Allocation-free form of the split-KV forward.
//
// Some callers cannot hand this library a workspace: code embedded in a host
// runtime that owns every device allocation (a serving engine that carves all
// memory out of one fixed pool up front, a plugin whose host forbids stray
// allocations), or callers that must never pay cudaMalloc's implicit
// device-wide synchronisation in the middle of a decode loop.  For them the
// split partials live in one file-scope device array of
// PA_STATIC_SCRATCH_BYTES, reserved on every GPU where this file's device code
// is loaded and held there until the process exits.  The caller still passes its inputs and output.
//
// The array's host-side name is only a stand-in: host code must not pass it
// to a kernel.  Its device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) on the first call made on
// that device; make that first call before any stream capture.  A
// cudaDeviceReset unloads the module and may move the array, so the address
// kept from before a reset must not be used after it: a process that resets a
// device does not call this entry point on that device again.
//
// Every call shares the array and it keeps the previous call's contents.  The
// split kernels write every partial and log-sum-exp entry that the merge of
// the same call reads, so nothing needs clearing between calls.  Calls whose
// GPU work overlaps (different streams, or different host threads without
// ordering) race on the array: serialise them on one stream.

#include <mutex>

#include "pa_internal.h"

namespace {

__device__ __align__(256) unsigned char g_split_scratch[PA_STATIC_SCRATCH_BYTES];

std::mutex g_setup_mutex;
void *g_scratch_addr[64] = {nullptr};

// Device address of g_split_scratch on the current device (looked up once).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_split_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" pa_status paged_attn_forward_split_static(const pa_plan *plan, const void *q, const void *k_cache,
                                                     const void *v_cache, void *out, int32_t num_heads,
                                                     int32_t num_kv_heads, int32_t head_dim, int32_t value_dim,
                                                     float scale, int32_t causal, int32_t window, pa_dtype dtype,
                                                     int32_t splits, pa_stream_t stream) {
    // the same argument checks, in the same order, as the workspace form, so an
    // invalid call gets the status that form would give before any size check
    static const char kName[] = "paged_attn_forward_split_static";
    pa_status st = pa::check_attention_args(plan, num_heads, num_kv_heads, head_dim, value_dim, 0, scale, causal,
                                            window, dtype, false, kName);
    if (st != PA_OK) return st;
    int64_t counts[8];
    st = pa_plan_describe(plan, counts);
    if (st != PA_OK) return st;
    if (splits < 1 || splits > PA_MAX_SPLITS)
        return pa_fail_with(PA_ERR_SPLITS, "paged_attn_forward_split_static: splits must be in 1..64");
    const size_t need = pa_workspace_bytes((int32_t)counts[0], num_heads, value_dim, splits);
    if (need > (size_t)PA_STATIC_SCRATCH_BYTES) {
        return pa_fail_with(PA_ERR_WORKSPACE,
                            "paged_attn_forward_split_static: split partials need more than the "
                            "PA_STATIC_SCRATCH_BYTES static scratch; use fewer splits or "
                            "paged_attn_forward_split with a caller workspace");
    }
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return pa_fail_with(PA_ERR_CUDA, "paged_attn_forward_split_static: cudaGetSymbolAddress of the static "
                                         "scratch failed");
    return paged_attn_forward_split(plan, q, k_cache, v_cache, out, num_heads, num_kv_heads, head_dim, value_dim,
                                    scale, causal, window, dtype, scratch, (size_t)PA_STATIC_SCRATCH_BYTES, splits,
                                    stream);
}
