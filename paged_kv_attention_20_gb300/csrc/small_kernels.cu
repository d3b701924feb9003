// Cache append, split merge and the device status word.
//
// Append: ruDNN 0.1.7, src/paged_attention/mod.rs, `append_with_report` --
// new rows [queries, heads, d|dv] land in the caches at the plan's positions,
// an elementwise kernel over queries * heads * max(d, dv).  Here each thread
// moves one 16-byte chunk (or one element when rows are not 16-byte multiples
// or not aligned); the destination slot comes precomputed in the plan.
//
// Merge: same page, `execute_attention_into` (merge launch when splits > 1)
// and `attention_into_split` (FP32 statistics): out = sum_s w_s o_s / sum_s w_s
// with w_s = exp(lse_s - max_s lse_s); empty splits (lse = -inf) weigh 0.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"

namespace pa {

__device__ int32_t g_device_status = 0;

template <typename U>
__global__ void kv_store_kernel(PlanView plan, const U *__restrict__ new_k, const U *__restrict__ new_v,
                                U *__restrict__ kc, U *__restrict__ vc, int heads, int uk, int uv,
                                int64_t total) {
    // One work unit = one U-sized piece of one row; K pieces then V pieces per (query, head).
    griddep_wait();
    griddep_launch();
    const int per_row = uk + uv;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        int64_t row = idx / per_row;          // (query, head)
        int u = (int)(idx - row * per_row);
        int64_t qi = row / heads;
        int h = (int)(row - qi * heads);
        int64_t slot = plan.qmeta[qi].z;
        if (u < uk) {
            kc[(slot * heads + h) * uk + u] = new_k[row * uk + u];
        } else {
            u -= uk;
            vc[(slot * heads + h) * uv + u] = new_v[row * uv + u];
        }
    }
}

cudaError_t launch_kv_store(const PlanView &plan, const void *new_k, const void *new_v, void *k_cache,
                            void *v_cache, int heads, int d, int dv, int elem_bytes, cudaStream_t st) {
    const int64_t kb = (int64_t)d * elem_bytes, vb = (int64_t)dv * elem_bytes;
    auto al = [](const void *p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
    int unit = elem_bytes;
    if (kb % 16 == 0 && vb % 16 == 0 && al(new_k, 16) && al(new_v, 16) && al(k_cache, 16) && al(v_cache, 16))
        unit = 16;
    const int uk = (int)(kb / unit), uv = (int)(vb / unit);
    const int64_t total = (int64_t)plan.queries * heads * (uk + uv);
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 152 * 32) blocks = 152 * 32;
    if (blocks < 1) blocks = 1;
    const dim3 grid((unsigned)blocks), block(threads);
    cudaError_t e;
    if (unit == 16)
        e = launch_pdl(kv_store_kernel<uint4>, grid, block, 0, st, plan, (const uint4 *)new_k, (const uint4 *)new_v,
                       (uint4 *)k_cache, (uint4 *)v_cache, heads, uk, uv, total);
    else if (unit == 4)
        e = launch_pdl(kv_store_kernel<uint32_t>, grid, block, 0, st, plan, (const uint32_t *)new_k,
                       (const uint32_t *)new_v, (uint32_t *)k_cache, (uint32_t *)v_cache, heads, uk, uv, total);
    else
        e = launch_pdl(kv_store_kernel<uint16_t>, grid, block, 0, st, plan, (const uint16_t *)new_k,
                       (const uint16_t *)new_v, (uint16_t *)k_cache, (uint16_t *)v_cache, heads, uk, uv, total);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T> __device__ __forceinline__ T from_float(float x);
template <> __device__ __forceinline__ float from_float<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// One warp per (query, head) row, eight rows per 256-thread block.  Every
// lane derives the split weights e^(lse_s - M) itself (M = max over splits,
// empty splits weigh 0) and holds VEC consecutive value columns of each
// 32*VEC-column chunk, read as one vector per split.
template <typename T, int VEC> struct OutVec;
template <typename T> struct OutVec<T, 1> {
    static __device__ __forceinline__ void store(T *p, const float *v) { p[0] = from_float<T>(v[0]); }
};
template <typename T> struct OutVec<T, 2> {
    static __device__ __forceinline__ void store(T *p, const float *v) {
        p[0] = from_float<T>(v[0]);
        p[1] = from_float<T>(v[1]);
    }
};
template <> struct OutVec<float, 4> {
    static __device__ __forceinline__ void store(float *p, const float *v) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <typename T> struct OutVec<T, 4> {
    static __device__ __forceinline__ void store(T *p, const float *v) {
        union { T h[4]; uint2 u; } x;
#pragma unroll
        for (int i = 0; i < 4; ++i) x.h[i] = from_float<T>(v[i]);
        *reinterpret_cast<uint2 *>(p) = x.u;
    }
};

template <int VEC> __device__ __forceinline__ void load_vec(const float *p, float *v) {
    if constexpr (VEC == 4) {
        const float4 x = *reinterpret_cast<const float4 *>(p);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else if constexpr (VEC == 2) {
        const float2 x = *reinterpret_cast<const float2 *>(p);
        v[0] = x.x; v[1] = x.y;
    } else {
        v[0] = p[0];
    }
}

template <typename T, int VEC>
__global__ void __launch_bounds__(256) merge_kernel(AttnArgs a, int use_list, int nrows) {
    griddep_wait();
    griddep_launch();
    const int wid = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (wid >= nrows) return;
    const int item = wid / a.hq, h = wid - item * a.hq;
    const int qi = use_list ? a.plan.decode[item] : item;
    const int S = a.splits;
    const int64_t rows = (int64_t)a.plan.queries * a.hq;
    const int64_t row = (int64_t)qi * a.hq + h;
    // lane l holds the weights of splits l and l + 32 (at most PA_MAX_SPLITS = 64)
    float m = -INFINITY;
    for (int s = lane; s < S; s += 32) m = fmaxf(m, a.ws_lse[s * rows + row]);
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float wl[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int s = lane + 32 * k;
        const float l = s < S ? a.ws_lse[s * rows + row] : -INFINITY;
        wl[k] = l == -INFINITY ? 0.f : __expf(l - m);
    }
    float tot = wl[0] + wl[1];
    for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    const float inv = 1.f / tot;
    T *out = static_cast<T *>(a.out) + row * a.dv;
    // every lane runs every chunk (the weights are shuffled in the loop); a lane
    // past the last column reads column 0 and stores nothing
    for (int c0 = 0; c0 < a.dv; c0 += 32 * VEC) {
        const bool live = c0 + lane * VEC < a.dv;
        const int c = live ? c0 + lane * VEC : 0;
        float acc[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
        // no branch on empty splits (their weight is 0 and their partial 0), so the
        // loads of several splits are in flight at once
#pragma unroll 8
        for (int s = 0; s < S; ++s) {
            const float ws = __shfl_sync(0xffffffffu, s < 32 ? wl[0] : wl[1], s & 31);
            float v[VEC];
            load_vec<VEC>(a.ws_o + (s * rows + row) * a.dv + c, v);
#pragma unroll
            for (int i = 0; i < VEC; ++i) acc[i] += ws * v[i];
        }
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[i] *= inv;
        if (live) OutVec<T, VEC>::store(out + c, acc);
    }
}

// Few rows or many splits: one 8-warp block per (query, head) row, warp w
// taking splits w, w + 8, ...; the eight partial sums meet in shared memory.
// Rows spread over every SM and all splits of a row are in flight at once,
// where one warp per row would walk its splits one after another.
template <typename T, int VEC>
__global__ void __launch_bounds__(256) merge_wide_kernel(AttnArgs a, int use_list) {
    griddep_wait();
    griddep_launch();
    extern __shared__ float part[];   // [8][dv]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int item = blockIdx.x / a.hq, h = blockIdx.x - item * a.hq;
    const int qi = use_list ? a.plan.decode[item] : item;
    const int S = a.splits;
    const int64_t rows = (int64_t)a.plan.queries * a.hq;
    const int64_t row = (int64_t)qi * a.hq + h;
    float m = -INFINITY;
    for (int s = lane; s < S; s += 32) m = fmaxf(m, a.ws_lse[s * rows + row]);
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float wl[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int s = lane + 32 * k;
        const float l = s < S ? a.ws_lse[s * rows + row] : -INFINITY;
        wl[k] = l == -INFINITY ? 0.f : __expf(l - m);
    }
    float tot = wl[0] + wl[1];
    for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    for (int c0 = 0; c0 < a.dv; c0 += 32 * VEC) {
        const bool live = c0 + lane * VEC < a.dv;
        const int c = live ? c0 + lane * VEC : 0;
        float acc[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
#pragma unroll 4
        for (int s = warp; s < S; s += 8) {
            const float ws = __shfl_sync(0xffffffffu, s < 32 ? wl[0] : wl[1], s & 31);
            float v[VEC];
            load_vec<VEC>(a.ws_o + (s * rows + row) * a.dv + c, v);
#pragma unroll
            for (int i = 0; i < VEC; ++i) acc[i] += ws * v[i];
        }
        if (live) {
#pragma unroll
            for (int i = 0; i < VEC; ++i) part[warp * a.dv + c + i] = acc[i];
        }
    }
    __syncthreads();
    const float inv = 1.f / tot;
    T *out = static_cast<T *>(a.out) + row * a.dv;
    for (int c = threadIdx.x; c < a.dv; c += 256) {
        float x = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) x += part[w * a.dv + c];
        out[c] = from_float<T>(x * inv);
    }
}

template <int VEC> cudaError_t launch_merge_vec(const AttnArgs &a, bool use_list, int nrows, cudaStream_t st) {
    const int ul = use_list ? 1 : 0;
    if (nrows < 1024 || a.splits >= 16) {
        // fewer rows than fill the GPU at 8 per block, or long split chains
        const dim3 grid((unsigned)nrows), block(256);
        const size_t smem = (size_t)8 * a.dv * sizeof(float);
        switch (a.dtype) {
            case PA_F32: return launch_pdl(merge_wide_kernel<float, VEC>, grid, block, smem, st, a, ul);
            case PA_F16: return launch_pdl(merge_wide_kernel<__half, VEC>, grid, block, smem, st, a, ul);
            default: return launch_pdl(merge_wide_kernel<__nv_bfloat16, VEC>, grid, block, smem, st, a, ul);
        }
    }
    const dim3 grid((unsigned)((nrows + 7) / 8)), block(256);
    switch (a.dtype) {
        case PA_F32: return launch_pdl(merge_kernel<float, VEC>, grid, block, 0, st, a, ul, nrows);
        case PA_F16: return launch_pdl(merge_kernel<__half, VEC>, grid, block, 0, st, a, ul, nrows);
        default: return launch_pdl(merge_kernel<__nv_bfloat16, VEC>, grid, block, 0, st, a, ul, nrows);
    }
}

cudaError_t launch_merge(const AttnArgs &a, bool use_list, cudaStream_t st) {
    const int items = use_list ? a.plan.n_decode : a.plan.queries;
    if (items == 0) return cudaSuccess;
    const int nrows = items * a.hq;
    // the workspace is 16-byte aligned and rows are dv floats apart; the output
    // takes 4-wide stores only when its base allows them
    const uintptr_t ob = reinterpret_cast<uintptr_t>(a.out);
    const uintptr_t esz = a.dtype == PA_F32 ? 4 : 2;
    cudaError_t e;
    if (a.dv % 4 == 0 && ob % (4 * esz) == 0)
        e = launch_merge_vec<4>(a, use_list, nrows, st);
    else if (a.dv % 2 == 0)
        e = launch_merge_vec<2>(a, use_list, nrows, st);
    else
        e = launch_merge_vec<1>(a, use_list, nrows, st);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Every query moves to the next position of its sequence: pos + 1, the write
// slot of that position from the block table, and a sequence length covering
// it.  A position the table does not map (past the row, or a negative or
// out-of-pool entry) leaves the query unchanged and records PA_DEVICE_RANGE.
__global__ void plan_advance_kernel(PlanView plan, int32_t *status) {
    griddep_wait();           // the previous kernel may still read the plan
    griddep_launch();
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= plan.queries) return;
    int4 *meta = const_cast<int4 *>(plan.qmeta) + q;
    const int4 m = *meta;
    const int64_t np = (int64_t)m.y + 1;
    if (np >= (int64_t)plan.width * plan.page_size) {
        atomicCAS(status, 0, PA_DEVICE_RANGE);
        return;
    }
    const int32_t pg = plan.table[(int64_t)m.x * plan.width + np / plan.page_size];
    if (pg < 0 || pg >= plan.pages) {
        atomicCAS(status, 0, PA_DEVICE_RANGE);
        return;
    }
    *meta = make_int4(m.x, (int)np, pg * plan.page_size + (int)(np % plan.page_size), 0);
    atomicMax(const_cast<int32_t *>(plan.seq_lens) + m.x, (int)(np + 1));
}

cudaError_t launch_plan_advance(const PlanView &plan, int32_t *status, cudaStream_t st) {
    const int threads = 128;
    cudaError_t e = launch_pdl(plan_advance_kernel, dim3((unsigned)((plan.queries + threads - 1) / threads)),
                               dim3(threads), 0, st, plan, status);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int32_t *device_status_ptr() {
    static int32_t *cached[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!cached[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        cached[dev] = static_cast<int32_t *>(p);
    }
    return cached[dev];
}

cudaError_t read_device_status(int32_t *code, bool clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(code, g_device_status, sizeof(int32_t));
    if (e != cudaSuccess) return e;
    if (clear) {
        int32_t zero = 0;
        e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int32_t));
    }
    return e;
}

}  // namespace pa
