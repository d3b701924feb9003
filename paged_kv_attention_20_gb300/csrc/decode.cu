// Paged decode attention on CUDA cores (bandwidth-bound path).
//
// ruDNN 0.1.7, src/paged_attention/mod.rs: `DevicePlan::attention` (packed Q
// [queries, Hq, D], K/V caches [pages, page_size, Hkv, D|Dv], causal at the
// plan's absolute positions), `execute_attention_into` (Hq a multiple of Hkv,
// no per-head repeat of the cache; launch over (queries, heads, splits)) and
// `attention_into_split` (split the visible history, FP32 statistics).
//
// Two kernels:
//  * decode_fast: bf16/f16, D == Dv in {64, 128, 256}.  One CTA of 128 threads
//    per (query, KV head, group of up to 8 query heads, split).  The query
//    heads that share a KV head are packed in one CTA so every page row is read
//    from HBM once.  Tiles of 32 (16 for D = 256) logical tokens are gathered
//    through the block table with 16-byte cp.async into a 4-stage shared-memory
//    ring; rows past the visible range are zero-filled, never read.  Scores use
//    several lanes per token with a transposing butterfly reduction; the online
//    softmax works in the log2 domain and only moves its reference maximum when
//    a tile's maximum exceeds it by more than 8 (weights stay <= 256, fp32
//    sums), so the accumulators are rarely rescaled.  P.V accumulates in fp32
//    registers split over token lanes and is reduced once at the end.
//  * decode_generic: any dtype and head dims up to 1024, MLA included (score
//    gets + qp . kp, the latent is the value).  One CTA per (query, head,
//    split); plain loads.  It is the correctness path for shapes the fast
//    kernels do not cover.
// Both write either the final output (one split) or per-split normalised fp32
// partials and natural-log lse into the workspace.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"

namespace pa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.f;  // log2 units


template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Eight packed 16-bit values -> floats.
template <typename T> __device__ __forceinline__ void unpack8(const uint4 &w, float (&f)[8]);
template <> __device__ __forceinline__ void unpack8<__nv_bfloat16>(const uint4 &w, float (&f)[8]) {
    f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xffff0000u);
    f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xffff0000u);
    f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xffff0000u);
}
template <> __device__ __forceinline__ void unpack8<__half>(const uint4 &w, float (&f)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = *reinterpret_cast<const __half2 *>(&u[i]);
        float2 t = __half22float2(h);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ int64_t physical_row(const int32_t *trow, int64_t j, int ps, int ps_shift) {
    if (ps_shift >= 0) return (int64_t)trow[j >> ps_shift] * ps + (j & (ps - 1));
    return (int64_t)trow[j / ps] * ps + j % ps;
}

template <typename T, int D, int GH>
struct FastCfg {
    static constexpr int NT = 128;
    static constexpr int TK = D <= 128 ? 32 : 16;          // tokens per tile
    static constexpr int NSTAGE = 4;
    static constexpr int CPR = D / 8;                       // 16-byte chunks per row
    static constexpr int CPT = TK * CPR / NT;               // chunks per thread per K (or V) tile
    static constexpr int DPL = (GH <= 4 && D >= 128) ? 16 : 8;  // dims per lane for the scores
    static constexpr int SUB = DPL / 8;                     // chunks per lane
    static constexpr int LPT = D / DPL;                     // lanes per token
    static constexpr int TPS = 32 / LPT;                    // tokens per warp step
    static constexpr int TPW = TK / 4;                      // tokens per warp per tile
    static constexpr int STEPS = TPW / TPS;
    static constexpr int NTL = NT / CPR;                    // token lanes of the P.V mapping
    static constexpr size_t RING = (size_t)NSTAGE * 2 * TK * D * 2;
    static constexpr size_t RED = (size_t)NTL * GH * D * 4;
    static constexpr size_t BIG = RING > RED ? RING : RED;
    static constexpr size_t SMEM = BIG + (size_t)TK * GH * 4 + 3 * 8 * 4;
    static_assert(CPT * NT == TK * CPR, "tile must split evenly over the threads");
    static_assert(STEPS * TPS == TPW, "tokens per warp must be whole steps");
    static_assert(GH <= LPT, "heads per CTA must not exceed lanes per token");
    static_assert(TK % NTL == 0, "token lanes must divide the tile");
};

// Sum GH per-lane partial scores over the LPT lanes of a token group, handing
// each head's total to a distinct sub-group (transposing butterfly).  Returns
// the total for head `head`; lanes with `writer` set hold a unique copy.
template <int GH, int LPT>
__device__ __forceinline__ float reduce_heads(float (&v)[GH], int glane, int &head, bool &writer) {
    int base = 0;
#pragma unroll
    for (int o = LPT / 2, n = GH; o >= 1; o >>= 1) {
        if (n > 1) {
            const int half = n / 2;
            const bool upper = (glane & o) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float send = upper ? v[i] : v[i + half];
                const float keep = upper ? v[i + half] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
            if (upper) base += half;
            n = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
    head = base;
    writer = (glane & (LPT / GH - 1)) == 0;
    return v[0];
}

template <typename T, int D, int GH>
__global__ void __launch_bounds__(128) decode_fast_kernel(AttnArgs a, int use_list, int groups, int ps_shift) {
    using C = FastCfg<T, D, GH>;
    extern __shared__ __align__(16) unsigned char smem[];
    float *sp = reinterpret_cast<float *>(smem + C::BIG);   // [TK][GH] scores, then weights
    float *m_sm = sp + C::TK * GH;                             // [8] reference max (log2)
    float *l_sm = m_sm + 8;                                    // [8] weight sums
    float *al_sm = l_sm + 8;                                   // [8] rescale factors

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int item = blockIdx.x;
    const int qi = use_list ? a.plan.decode[item] : item;
    const int4 meta = a.plan.qmeta[qi];
    const int seq = meta.x, pos = meta.y;
    const int ps = a.plan.page_size;
    int64_t lo, hi;
    visible_range(pos, a.plan.seq_lens[seq], a.causal, a.window, lo, hi);
    const int kvh = blockIdx.y / groups;
    const int h0 = kvh * (a.hq / a.hkv) + (blockIdx.y % groups) * GH;
    const int split = blockIdx.z;
    int64_t j0, j1;
    split_bounds(lo, hi, a.splits, split, ps, j0, j1);
    const int ntiles = (int)((j1 - j0 + C::TK - 1) / C::TK);
    const int32_t *trow = a.plan.table + (int64_t)seq * a.plan.width;
    const T *kg = static_cast<const T *>(a.k);
    const T *vg = static_cast<const T *>(a.v);

    if (tid < 8) {
        m_sm[tid] = -INFINITY;
        l_sm[tid] = 0.f;
        al_sm[tid] = 1.f;
    }

    // Gather one tile of keys/values into ring stage `stage`.
    const uint32_t ring = (uint32_t)__cvta_generic_to_shared(smem);
    auto load_tile = [&](int stage, int tile) {
        const int64_t tb = j0 + (int64_t)tile * C::TK;
        const uint32_t kdst = ring + (uint32_t)(stage * 2 * C::TK * D * 2);
        const uint32_t vdst = kdst + (uint32_t)(C::TK * D * 2);
#pragma unroll
        for (int k = 0; k < C::CPT; ++k) {
            const int c = tid + k * C::NT;
            const int t = c / C::CPR, part = c % C::CPR;
            const int64_t j = tb + t;
            const bool valid = j < j1;
            const T *ks = kg, *vs = vg;
            if (valid) {
                const int64_t row = physical_row(trow, j, ps, ps_shift);
                ks = kg + (row * a.hkv + kvh) * D + part * 8;
                vs = vg + (row * a.hkv + kvh) * D + part * 8;
            }
            cp_async16(kdst + c * 16, ks, valid);
            cp_async16(vdst + c * 16, vs, valid);
        }
    };

#pragma unroll
    for (int s = 0; s < C::NSTAGE - 1; ++s) {
        if (s < ntiles) load_tile(s, s);
        cp_async_commit();
    }

    // Query registers: lane covers chunks glane + c * LPT (bank-conflict free).
    const int glane = lane % C::LPT, tsub = lane / C::LPT;
    float qr[GH][C::DPL];
    {
        const float qs = a.scale * kLog2e;
        const T *qg = static_cast<const T *>(a.q) + ((int64_t)qi * a.hq + h0) * D;
#pragma unroll
        for (int g = 0; g < GH; ++g)
#pragma unroll
            for (int c = 0; c < C::SUB; ++c) {
                const uint4 w = *reinterpret_cast<const uint4 *>(qg + (int64_t)g * D + (glane + c * C::LPT) * 8);
                float f[8];
                unpack8<T>(w, f);
#pragma unroll
                for (int e = 0; e < 8; ++e) qr[g][c * 8 + e] = f[e] * qs;
            }
    }

    const int tl = tid / C::CPR, oc = tid % C::CPR;   // P.V mapping: token lane, column octet
    float acc[GH][8];
#pragma unroll
    for (int g = 0; g < GH; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;

    for (int it = 0; it < ntiles; ++it) {
        {
            const int nt = it + C::NSTAGE - 1;
            if (nt < ntiles) load_tile(nt % C::NSTAGE, nt);
            cp_async_commit();
        }
        cp_async_wait<C::NSTAGE - 1>();
        __syncthreads();
        const int stage = it % C::NSTAGE;
        const uint4 *Ks = reinterpret_cast<const uint4 *>(smem + (size_t)stage * 2 * C::TK * D * 2);
        const uint4 *Vs = Ks + C::TK * C::CPR;
        const int64_t tb = j0 + (int64_t)it * C::TK;

        // Scores of this tile for the GH heads.
#pragma unroll
        for (int step = 0; step < C::STEPS; ++step) {
            const int t = warp * C::TPW + step * C::TPS + tsub;
            float part[GH];
#pragma unroll
            for (int g = 0; g < GH; ++g) part[g] = 0.f;
#pragma unroll
            for (int c = 0; c < C::SUB; ++c) {
                float kf[8];
                unpack8<T>(Ks[t * C::CPR + glane + c * C::LPT], kf);
#pragma unroll
                for (int g = 0; g < GH; ++g)
#pragma unroll
                    for (int e = 0; e < 8; ++e) part[g] = fmaf(qr[g][c * 8 + e], kf[e], part[g]);
            }
            int head;
            bool writer;
            const float s = reduce_heads<GH, C::LPT>(part, glane, head, writer);
            if (writer) sp[t * GH + head] = (tb + t < j1) ? s : -INFINITY;
        }
        __syncthreads();

        // Online softmax update, one warp per head.
        for (int g = warp; g < GH; g += 4) {
            const float s = lane < C::TK ? sp[lane * GH + g] : -INFINITY;
            float mt = s;
#pragma unroll
            for (int o = 16; o; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
            const float mref = m_sm[g];
            const float nref = (mt > mref + kRescaleSlack) ? mt : mref;
            const float alpha = exp2f(mref - nref);
            const float p = exp2f(s - nref);
            float ps_ = p;
#pragma unroll
            for (int o = 16; o; o >>= 1) ps_ += __shfl_xor_sync(0xffffffffu, ps_, o);
            if (lane < C::TK) sp[lane * GH + g] = p;
            if (lane == 0) {
                l_sm[g] = l_sm[g] * alpha + ps_;
                m_sm[g] = nref;
                al_sm[g] = alpha;
            }
        }
        __syncthreads();

        // Rescale (rare) and accumulate P.V.
#pragma unroll
        for (int g = 0; g < GH; ++g) {
            const float al = al_sm[g];
            if (al != 1.f) {
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[g][e] *= al;
            }
        }
#pragma unroll
        for (int tt = tl; tt < C::TK; tt += C::NTL) {
            float vf[8];
            unpack8<T>(Vs[tt * C::CPR + oc], vf);
            float pg[GH];
            if constexpr (GH >= 4) {
#pragma unroll
                for (int g4 = 0; g4 < GH / 4; ++g4) {
                    const float4 w4 = reinterpret_cast<const float4 *>(sp + tt * GH)[g4];
                    pg[g4 * 4 + 0] = w4.x; pg[g4 * 4 + 1] = w4.y; pg[g4 * 4 + 2] = w4.z; pg[g4 * 4 + 3] = w4.w;
                }
            } else {
#pragma unroll
                for (int g = 0; g < GH; ++g) pg[g] = sp[tt * GH + g];
            }
#pragma unroll
            for (int g = 0; g < GH; ++g)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(pg[g], vf[e], acc[g][e]);
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    __syncthreads();

    // Reduce the token lanes and write the result.
    float *red = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int g = 0; g < GH; ++g) {
        float4 *dst = reinterpret_cast<float4 *>(red + ((size_t)(tl * GH + g) * D) + oc * 8);
        dst[0] = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
        dst[1] = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
    }
    __syncthreads();
    const int64_t rows = (int64_t)a.plan.queries * a.hq;
    for (int idx = tid; idx < GH * D; idx += C::NT) {
        const int g = idx / D, c = idx % D;
        float sum = 0.f;
#pragma unroll
        for (int t2 = 0; t2 < C::NTL; ++t2) sum += red[(size_t)(t2 * GH + g) * D + c];
        const float l = l_sm[g];
        const int64_t row = (int64_t)qi * a.hq + h0 + g;
        if (a.splits == 1) {
            static_cast<T *>(a.out)[row * D + c] = from_f<T>(sum / l);
        } else {
            a.ws_o[((int64_t)split * rows + row) * D + c] = l > 0.f ? sum / l : 0.f;
        }
    }
    if (a.splits > 1 && tid < GH) {
        const float l = l_sm[tid];
        const int64_t row = (int64_t)qi * a.hq + h0 + tid;
        a.ws_lse[(int64_t)split * rows + row] = l > 0.f ? (m_sm[tid] + log2f(l)) * kLn2 : -INFINITY;
    }
}

__device__ __forceinline__ float block_max128(float v, float *scratch) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    v = fmaxf(fmaxf(scratch[0], scratch[1]), fmaxf(scratch[2], scratch[3]));
    __syncthreads();
    return v;
}

__device__ __forceinline__ float block_sum128(float v, float *scratch) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    v = (scratch[0] + scratch[1]) + (scratch[2] + scratch[3]);
    __syncthreads();
    return v;
}

// Generic path: one CTA per (query, head, split), 128 threads, one key per thread.
template <typename T>
__global__ void __launch_bounds__(128) decode_generic_kernel(AttnArgs a, int use_list, int ps_shift) {
    extern __shared__ __align__(16) unsigned char smem[];
    long long *rows_sm = reinterpret_cast<long long *>(smem);        // [128]
    float *p_sm = reinterpret_cast<float *>(rows_sm + 128);           // [128]
    float *scratch = p_sm + 128;                                      // [8]
    float *qf = scratch + 8;                                          // [d]
    float *qpf = qf + a.d;                                            // [p]

    const int tid = threadIdx.x;
    const int item = blockIdx.x, h = blockIdx.y, split = blockIdx.z;
    const int qi = use_list ? a.plan.decode[item] : item;
    const int4 meta = a.plan.qmeta[qi];
    const int seq = meta.x, pos = meta.y;
    const int ps = a.plan.page_size;
    int64_t lo, hi;
    visible_range(pos, a.plan.seq_lens[seq], a.causal, a.window, lo, hi);
    const int kvh = h / (a.hq / a.hkv);
    int64_t j0, j1;
    split_bounds(lo, hi, a.splits, split, ps, j0, j1);
    const int32_t *trow = a.plan.table + (int64_t)seq * a.plan.width;
    const T *kg = static_cast<const T *>(a.k);
    const T *vg = static_cast<const T *>(a.v);
    const T *kpg = static_cast<const T *>(a.kp);
    const float qs = a.scale * kLog2e;
    {
        const T *qrow = static_cast<const T *>(a.q) + ((int64_t)qi * a.hq + h) * a.d;
        for (int i = tid; i < a.d; i += 128) qf[i] = to_f<T>(qrow[i]) * qs;
        if (a.p) {
            const T *qprow = static_cast<const T *>(a.qp) + ((int64_t)qi * a.hq + h) * a.p;
            for (int i = tid; i < a.p; i += 128) qpf[i] = to_f<T>(qprow[i]) * qs;
        }
    }
    __syncthreads();

    float m = -INFINITY, l = 0.f;
    float acc[PA_MAX_HEAD_DIM / 128];
#pragma unroll
    for (int i = 0; i < PA_MAX_HEAD_DIM / 128; ++i) acc[i] = 0.f;

    for (int64_t base = j0; base < j1; base += 128) {
        const int64_t j = base + tid;
        float s = -INFINITY;
        if (j < j1) {
            const int64_t row = physical_row(trow, j, ps, ps_shift);
            rows_sm[tid] = row;
            const T *kr = kg + (row * a.hkv + kvh) * a.d;
            float dot = 0.f;
            for (int e = 0; e < a.d; ++e) dot = fmaf(qf[e], to_f<T>(kr[e]), dot);
            if (a.p) {
                const T *kpr = kpg + row * a.p;
                for (int e = 0; e < a.p; ++e) dot = fmaf(qpf[e], to_f<T>(kpr[e]), dot);
            }
            s = dot;
        }
        const float mt = block_max128(s, scratch);
        const float nm = fmaxf(m, mt);
        const float alpha = exp2f(m - nm);
        const float p = (j < j1) ? exp2f(s - nm) : 0.f;
        p_sm[tid] = p;
        const float lt = block_sum128(p, scratch);   // its barriers also publish p_sm/rows_sm
        l = l * alpha + lt;
        m = nm;
        const int cnt = (int)((j1 - base) < 128 ? (j1 - base) : 128);
#pragma unroll
        for (int i = 0; i < PA_MAX_HEAD_DIM / 128; ++i) {
            const int c = tid + 128 * i;
            if (c < a.dv) {
                float x = acc[i] * alpha;
                for (int t = 0; t < cnt; ++t)
                    x = fmaf(p_sm[t], to_f<T>(vg[(rows_sm[t] * a.hkv + kvh) * a.dv + c]), x);
                acc[i] = x;
            }
        }
        __syncthreads();
    }

    const int64_t nrows = (int64_t)a.plan.queries * a.hq;
    const int64_t row = (int64_t)qi * a.hq + h;
#pragma unroll
    for (int i = 0; i < PA_MAX_HEAD_DIM / 128; ++i) {
        const int c = tid + 128 * i;
        if (c < a.dv) {
            if (a.splits == 1)
                static_cast<T *>(a.out)[row * a.dv + c] = from_f<T>(acc[i] / l);
            else
                a.ws_o[((int64_t)split * nrows + row) * a.dv + c] = l > 0.f ? acc[i] / l : 0.f;
        }
    }
    if (a.splits > 1 && tid == 0)
        a.ws_lse[(int64_t)split * nrows + row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

int ps_shift_of(int ps) {
    if (ps <= 0 || (ps & (ps - 1))) return -1;
    int s = 0;
    while ((1 << s) < ps) ++s;
    return s;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T, int D, int GH>
cudaError_t launch_fast_t(const AttnArgs &a, int items, int use_list, cudaStream_t st) {
    using C = FastCfg<T, D, GH>;
    static bool configured = false;  // attribute set once per process (single device use)
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_fast_kernel<T, D, GH>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int groups = (a.hq / a.hkv) / GH;
    dim3 grid(items, a.hkv * groups, a.splits);
    decode_fast_kernel<T, D, GH><<<grid, C::NT, C::SMEM, st>>>(a, use_list, groups, ps_shift_of(a.plan.page_size));
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_fast_d(const AttnArgs &a, int items, int use_list, cudaStream_t st) {
    const int G = a.hq / a.hkv;
    if (G % 8 == 0) return launch_fast_t<T, D, 8>(a, items, use_list, st);
    if (G % 4 == 0) return launch_fast_t<T, D, 4>(a, items, use_list, st);
    if (G % 2 == 0) return launch_fast_t<T, D, 2>(a, items, use_list, st);
    return launch_fast_t<T, D, 1>(a, items, use_list, st);
}

template <typename T>
cudaError_t launch_fast(const AttnArgs &a, int items, int use_list, cudaStream_t st) {
    switch (a.d) {
        case 64: return launch_fast_d<T, 64>(a, items, use_list, st);
        case 128: return launch_fast_d<T, 128>(a, items, use_list, st);
        default: return launch_fast_d<T, 256>(a, items, use_list, st);
    }
}

template <typename T>
cudaError_t launch_generic(const AttnArgs &a, int items, int use_list, cudaStream_t st) {
    const size_t smem = 128 * sizeof(long long) + 128 * 4 + 8 * 4 + (size_t)(a.d + a.p) * 4;
    dim3 grid(items, a.hq, a.splits);
    decode_generic_kernel<T><<<grid, 128, smem, st>>>(a, use_list, ps_shift_of(a.plan.page_size));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const AttnArgs &a, bool use_decode_list, cudaStream_t st) {
    const int items = use_decode_list ? a.plan.n_decode : a.plan.queries;
    if (items == 0) return cudaSuccess;
    if (decode_tc_supported(a)) return launch_decode_tc(a, use_decode_list, st);
    if (decode_tma_supported(a)) return launch_decode_tma(a, use_decode_list, st);
    const bool fast = a.dtype != PA_F32 && a.p == 0 && a.d == a.dv &&
                      (a.d == 64 || a.d == 128 || a.d == 256) && aligned16(a.q) && aligned16(a.k) &&
                      aligned16(a.v);
    const int ul = use_decode_list ? 1 : 0;
    if (fast) {
        return a.dtype == PA_BF16 ? launch_fast<__nv_bfloat16>(a, items, ul, st)
                                  : launch_fast<__half>(a, items, ul, st);
    }
    switch (a.dtype) {
        case PA_F32: return launch_generic<float>(a, items, ul, st);
        case PA_F16: return launch_generic<__half>(a, items, ul, st);
        default: return launch_generic<__nv_bfloat16>(a, items, ul, st);
    }
}

}  // namespace pa
