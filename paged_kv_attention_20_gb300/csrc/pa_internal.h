// Internal declarations shared by the host library and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "paged_attn.h"

namespace pa {

// Work-list constants of the plan.
constexpr int kPrefillTileM = 128;   // queries per tensor-core prefill tile
constexpr int kPrefillMinRun = 16;   // shorter runs of consecutive positions stay decode items

// Device view of an uploaded plan.  Every array lives in the caller's
// metadata buffer; offsets are fixed by the host plan (see plan.cpp).
struct PlanView {
    const int4 *qmeta;       // [queries] {seq, pos, physical slot, 0}
    const int32_t *seq_lens; // [sequences]
    const int32_t *table;    // [sequences * width]
    const int32_t *decode;   // [n_decode] query indices handled by the decode kernel
    const int4 *tiles;       // [n_tiles] {seq, first query, query count, first position}
    const int32_t *order;    // [queries] every query, longest visible history first
    int32_t queries;
    int32_t sequences;
    int32_t width;
    int32_t page_size;
    int32_t pages;
    int32_t n_decode;
    int32_t n_tiles;
};

// Arguments common to the attention kernels.
struct AttnArgs {
    PlanView plan;
    const void *q;        // [Q, Hq, D]
    const void *k;        // [pages, ps, Hkv, D]   (MLA: latent [pages, ps, 1, R])
    const void *v;        // [pages, ps, Hkv, Dv]  (MLA: same latent pointer)
    const void *qp;       // MLA position query [Q, Hq, P] or null
    const void *kp;       // MLA position cache [pages, ps, 1, P] or null
    void *out;            // [Q, Hq, Dv] in the operand dtype
    float *ws_o;          // split partials [S, Q, Hq, Dv] fp32 (null when unsplit)
    float *ws_lse;        // split lse      [S, Q, Hq]     fp32
    int32_t hq, hkv, d, dv, p;
    float scale;
    int32_t causal;
    int32_t window;       // sliding window (0 = none): keys pos - window + 1 and later
    int32_t splits;
    pa_dtype dtype;
    int32_t *status;      // device status word (bounded waits record timeouts here)
    int32_t max_ctas;     // persistent kernels: at most this many CTAs (0: as many as are resident at once)
};

// Keys a query at absolute position `pos` of a sequence holding `seq_len`
// keys may see: [lo, hi).  hi is pos + 1 (causal) or seq_len; a sliding
// window W > 0 (a layer's `window`, libmir-cuda 0.1.0,
// src/backend/attention/graph/mod.rs, `Geometry`) raises lo to pos - W + 1.
__host__ __device__ inline void visible_range(int pos, int seq_len, int causal, int window, int64_t &lo,
                                              int64_t &hi) {
    hi = causal ? (int64_t)pos + 1 : (int64_t)seq_len;
    lo = window > 0 ? (int64_t)pos - window + 1 : 0;
    if (lo < 0) lo = 0;
}

// Split s of `splits` over the visible keys [lo, hi): with base = lo rounded
// down to a page boundary and chunk = ceil((hi - base) / splits) rounded up to
// a page multiple, split s covers [max(lo, base + s*chunk), min(base + (s+1)*chunk, hi)).
// Every split but the first starts on a page boundary; an empty split has j0 == j1.
__host__ __device__ inline void split_bounds(int64_t lo, int64_t hi, int splits, int s, int ps, int64_t &j0,
                                             int64_t &j1) {
    if (splits == 1) {           // the whole range (what the rule below gives for one split)
        j0 = lo;
        j1 = hi > lo ? hi : lo;
        return;
    }
    // positions fit 32 bits (the plan checks slots against 2^31), so 32-bit division
    const int lo32 = (int)lo, hi32 = (int)hi;
    const int base = lo32 / ps * ps;
    int n = hi32 - base;
    if (n < 0) n = 0;
    int chunk = (n + splits - 1) / splits;
    chunk = (chunk + ps - 1) / ps * ps;
    int64_t b = base + (int64_t)s * chunk, e = b + chunk;
    if (b < lo) b = lo;
    if (b > hi) b = hi;
    if (e > hi) e = hi;
    if (e < b) e = b;
    j0 = b;
    j1 = e;
}

// The attention entry points' argument checks that need no device: plan,
// dtype, head counts and dims, scale, causal flag, window, MLA position dim
// and the size bounds.  PA_OK or the status (and message) the entry point
// named `name` returns for the first failing check.
pa_status check_attention_args(const pa_plan *plan, int32_t hq, int32_t hkv, int32_t d, int32_t dv, int32_t p,
                               float scale, int32_t causal, int32_t window, pa_dtype dtype, bool mla,
                               const char *name);

// Launchers (return cudaGetLastError() of the launch).
// use_decode_list: iterate over plan.decode (else over every query).
cudaError_t launch_kv_store(const PlanView &plan, const void *new_k, const void *new_v, void *k_cache,
                            void *v_cache, int heads, int d, int dv, int elem_bytes, cudaStream_t st);
cudaError_t launch_decode(const AttnArgs &a, bool use_decode_list, cudaStream_t st);
// Warp-independent TMA decode (bf16/f16, D == Dv in {64,128,256}, power-of-two pages).
bool decode_tma_supported(const AttnArgs &a);
cudaError_t launch_decode_tma(const AttnArgs &a, bool use_decode_list, cudaStream_t st);
bool decode_tc_supported(const AttnArgs &a);
cudaError_t launch_decode_tc(const AttnArgs &a, bool use_decode_list, cudaStream_t st);
cudaError_t launch_merge(const AttnArgs &a, bool use_decode_list, cudaStream_t st);
// Tensor-core prefill over plan.tiles; returns cudaErrorNotSupported when the
// shape/dtype is outside what the kernel covers (caller then uses decode for all).
bool prefill_supported(const AttnArgs &a);
cudaError_t launch_prefill(const AttnArgs &a, cudaStream_t st);
bool mla_supported(const AttnArgs &a);
cudaError_t launch_mla(const AttnArgs &a, bool use_decode_list, cudaStream_t st);

// One decode step forward on the device (pa_plan_advance).
cudaError_t launch_plan_advance(const PlanView &plan, int32_t *status, cudaStream_t st);

// Device status word (bounded waits record their timeouts here).
cudaError_t read_device_status(int32_t *code, bool clear);
// Device address of the status word on the current device (cached per device).
int32_t *device_status_ptr();

#ifdef __CUDACC__
// Programmatic dependent launch.  Every kernel of the library is launched
// with it allowed, so its CTAs may be scheduled before the kernel ahead of it
// in the stream has finished; each kernel therefore calls griddep_wait()
// before its first global-memory access (it returns once the preceding grid
// has completed and its writes are visible; without the launch attribute it
// returns at once).  A kernel calls griddep_launch() once its remaining work
// no longer needs SM room that a waiting dependent could take.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
#endif

}  // namespace pa

// Record `msg` as this thread's last error and return `status`.
pa_status pa_fail_with(pa_status status, const char *msg);
