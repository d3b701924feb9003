// Paged decode attention, warp-independent TMA pipeline (CUDA cores).
//
// Same operation as decode.cu (ruDNN 0.1.7, src/paged_attention/mod.rs:
// `DevicePlan::attention`, `execute_attention_into`, `attention_into_split`),
// organised for GB300's HBM3e:
//  * one CTA of 4 warps per (query, KV head, group of up to 4 query heads,
//    split); the GQA heads of one KV head share the CTA (larger groups use
//    adjacent CTAs, whose second read of a page hits L2), so every page row
//    is read from HBM once;
//  * the split's keys are cut into 16-token tiles; warp w owns tiles w, w+4,
//    w+8, ... and runs its own online softmax over them, with no CTA-wide
//    barrier in the loop; the four warp states are merged once at the end;
//  * each warp streams its tiles with TMA: one lane issues one box per 16
//    tokens (or per page when pages are shorter) for K and one for V into a
//    3-stage per-warp ring, completion tracked by an mbarrier per stage;
//  * scores use a group of lanes per token and a transposing butterfly
//    reduction; the products run as packed fp32 pairs (fma.rn.f32x2);
//  * tokens past the visible range are masked in the scores and never enter
//    P.V (tail slots may hold anything, NaN included).
// Page sizes must be powers of two (other sizes use decode.cu).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
#include "sm103_tc.cuh"
#include "tma_host.h"

namespace pa {
namespace {

using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::smem_u32;
using tc::ffma2;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSlack = 8.f;


template <typename T> __device__ __forceinline__ float2 unpack2(uint32_t w);
template <> __device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <> __device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <int D, int GH>
struct Cfg {
    static constexpr int NW = 4;                               // warps per CTA
    static constexpr int NST = 2;                              // ring stages per warp
    static constexpr int TT = 16;                              // tokens per tile
    static constexpr int DPL = (GH <= 4 && D >= 128) ? 16 : 8; // dims per lane (scores)
    static constexpr int SUB = DPL / 8;                        // 16-byte chunks per lane
    static constexpr int LPT = D / DPL;                        // lanes per token
    static constexpr int TPS = 32 / LPT;                       // tokens per step
    static constexpr int STEPS = TT / TPS;
    static constexpr int CPL = D / 32;                         // value columns per lane
    static constexpr int ROW = D * 2;                          // bytes per cache row
    static constexpr int TILE = TT * ROW;                      // bytes of one K (or V) tile
    static constexpr int STAGE = 2 * TILE;
    static constexpr int WARP_RING = NST * STAGE;
    static constexpr int SP = 3 * TT * GH;                     // per-warp: weight pairs [2*TT*GH] + scores [TT*GH]
    // shared layout: [rings NW*WARP_RING][scores NW*SP][alpha NW*8][barriers NW*NST]
    static constexpr size_t RINGS = (size_t)NW * WARP_RING;
    static constexpr size_t MERGE = (size_t)NW * GH * (D + 2) * 4;  // final warp merge (reuses rings)
    static constexpr size_t BIG = RINGS > MERGE ? RINGS : MERGE;
    static constexpr size_t SMEM = BIG + (size_t)NW * SP * 4 + NW * 8 * 4 + NW * NST * 8 + 1024;
    static_assert(STEPS * TPS == TT, "tile must be whole steps");
    static_assert(GH <= LPT, "heads per CTA must not exceed lanes per token");
};

// Transposing butterfly: sum GH partials over LPT lanes, each head ending in a
// distinct lane sub-group.  Lanes with `writer` hold a unique copy of `head`.
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

struct TmaParams {
    int groups;       // head groups per KV head
    int ps_shift;     // log2(page_size)
    int box_rows;     // rows per TMA box (min(page_size, 16))
};

template <typename T, int D, int GH>
__global__ void __launch_bounds__(128) decode_tma_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                         const __grid_constant__ CUtensorMap tm_v, AttnArgs a,
                                                         int use_list, TmaParams tp) {
    using C = Cfg<D, GH>;
    griddep_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *ring = smem + (size_t)warp * C::WARP_RING;
    float *sp = reinterpret_cast<float *>(smem + C::BIG) + warp * C::SP;
    float *al = reinterpret_cast<float *>(smem + C::BIG + (size_t)C::NW * C::SP * 4) + warp * 8;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BIG + (size_t)C::NW * C::SP * 4 + C::NW * 8 * 4) +
                     warp * C::NST;

    // Flattened grid, item slowest: the plan lists decode items longest first,
    // so the heaviest (query, KV head, split) blocks start first.
    const int hg_count = a.hkv * tp.groups;
    const int hg = blockIdx.x % hg_count;
    const int rest = blockIdx.x / hg_count;
    const int split = rest % a.splits;
    const int item = rest / a.splits;
    const int qi = use_list ? a.plan.decode[item] : item;
    const int4 meta = a.plan.qmeta[qi];
    const int seq = meta.x, pos = meta.y;
    const int ps = a.plan.page_size;
    int64_t lo, hi;
    visible_range(pos, a.plan.seq_lens[seq], a.causal, a.window, lo, hi);
    const int kvh = hg / tp.groups;
    const int h0 = kvh * (a.hq / a.hkv) + (hg % tp.groups) * GH;
    int64_t j0, j1;
    split_bounds(lo, hi, a.splits, split, ps, j0, j1);
    // Tiles start on a multiple of TT (so no TMA box crosses a page); keys of the
    // first tile below j0 (only under a sliding window) are masked.
    const int64_t jb = j0 < j1 ? j0 / C::TT * C::TT : j0;
    const int ntiles = (int)((j1 - jb + C::TT - 1) / C::TT);
    const int mine = ntiles > warp ? (ntiles - warp + C::NW - 1) / C::NW : 0;
    const int32_t *trow = a.plan.table + (int64_t)seq * a.plan.width;
    const int used_pages = (a.plan.seq_lens[seq] + ps - 1) >> tp.ps_shift;
    const int oob_row = a.plan.pages * ps;

    if (lane == 0) {
        for (int s = 0; s < C::NST; ++s) mbar_init(&bars[s], 1);
        tc::fence_mbar_init();
    }
    __syncwarp();

    // Lane 0: gather my i-th tile (16 tokens) of K and V into stage i % NST.
    auto issue = [&](int i) {
        const int st = i % C::NST;
        uint8_t *kdst = ring + st * C::STAGE;
        uint8_t *vdst = kdst + C::TILE;
        const int64_t jt = jb + (int64_t)(warp + i * C::NW) * C::TT;
        mbar_arrive_expect_tx(&bars[st], C::STAGE);
        for (int b = 0; b < C::TT; b += tp.box_rows) {
            const int64_t j = jt + b;
            const int64_t lp = j >> tp.ps_shift;
            const int row = lp < used_pages ? trow[lp] * ps + (int)(j & (ps - 1)) : oob_row;
            tc::tma_load_3d(kdst + b * C::ROW, &tm_k, 0, kvh, row, &bars[st]);
            tc::tma_load_3d(vdst + b * C::ROW, &tm_v, 0, kvh, row, &bars[st]);
        }
    };
    if (lane == 0) {
        for (int i = 0; i < C::NST && i < mine; ++i) issue(i);
    }

    // Query registers (pre-scaled into the log2 domain), as fp32 pairs.
    const int glane = lane % C::LPT, tsub = lane / C::LPT;
    float2 q2[GH][C::DPL / 2];
    {
        const float qs = a.scale * kLog2e;
        const T *qg = static_cast<const T *>(a.q) + ((int64_t)qi * a.hq + h0) * D;
#pragma unroll
        for (int g = 0; g < GH; ++g)
#pragma unroll
            for (int c = 0; c < C::SUB; ++c) {
                const uint4 w = *reinterpret_cast<const uint4 *>(qg + (int64_t)g * D + (glane + c * C::LPT) * 8);
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = unpack2<T>(u[e]);
                    q2[g][c * 4 + e] = make_float2(f.x * qs, f.y * qs);
                }
            }
    }

    // Per-warp softmax state: lanes 0-15 carry heads 2k, lanes 16-31 heads 2k+1.
    constexpr int HP = (GH + 1) / 2;
    float m_ref[HP], l_run[HP];
#pragma unroll
    for (int k = 0; k < HP; ++k) {
        m_ref[k] = -INFINITY;
        l_run[k] = 0.f;
    }
    float2 acc[GH][C::CPL / 2];
#pragma unroll
    for (int g = 0; g < GH; ++g)
#pragma unroll
        for (int c = 0; c < C::CPL / 2; ++c) acc[g][c] = make_float2(0.f, 0.f);

    bool ok = true;
    for (int i = 0; i < mine; ++i) {
        const int st = i % C::NST;
        // warp-uniform outcome: the lanes go on to full-warp shuffles together
        ok = __all_sync(0xffffffffu, mbar_wait(&bars[st], (i / C::NST) & 1));
        if (!ok) break;
        const uint8_t *K = ring + st * C::STAGE;
        const uint8_t *V = K + C::TILE;
        const int64_t jt = jb + (int64_t)(warp + i * C::NW) * C::TT;
        const int valid = (int)((j1 - jt) < C::TT ? (j1 - jt) : C::TT);
        const int first = (int)(j0 > jt ? j0 - jt : 0);     // keys below j0 (first tile only)

        // scores
#pragma unroll
        for (int step = 0; step < C::STEPS; ++step) {
            const int t = step * C::TPS + tsub;
            float2 part2[GH];
#pragma unroll
            for (int g = 0; g < GH; ++g) part2[g] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < C::SUB; ++c) {
                const uint4 w = *reinterpret_cast<const uint4 *>(K + t * C::ROW + (glane + c * C::LPT) * 16);
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 kf = unpack2<T>(u[e]);
#pragma unroll
                    for (int g = 0; g < GH; ++g) part2[g] = ffma2(q2[g][c * 4 + e], kf, part2[g]);
                }
            }
            float part[GH];
#pragma unroll
            for (int g = 0; g < GH; ++g) part[g] = part2[g].x + part2[g].y;
            int head;
            bool writer;
            const float s = reduce_heads<GH, C::LPT>(part, glane, head, writer);
            if (writer) sp[2 * C::TT * GH + t * GH + head] = s;
        }
        __syncwarp();

        // online softmax, two heads per pass (one per half-warp).  Weights use
        // the current reference max; only when some score exceeds it by more
        // than 2^8 (the first tile, then rarely) does the half-warp reduce its
        // tile max and move the reference.  Weight sums stay per lane until the end.
        const int t16 = lane & 15;
#pragma unroll
        for (int k = 0; k < HP; ++k) {
            const int g = 2 * k + (lane >> 4);
            const bool gv = g < GH;
            const float s = (gv && t16 < valid && t16 >= first) ? sp[2 * C::TT * GH + t16 * GH + g] : -INFINITY;
            float alpha = 1.f;
            if (__any_sync(0xffffffffu, s > m_ref[k] + kSlack)) {
                float mt = s;
#pragma unroll
                for (int o = 8; o; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                if (mt > m_ref[k] + kSlack) {
                    alpha = exp2f(m_ref[k] - mt);
                    m_ref[k] = mt;
                    l_run[k] *= alpha;
                }
            }
            const float p = exp2f(s - m_ref[k]);
            l_run[k] += p;
            if (gv) {
                reinterpret_cast<float2 *>(sp)[t16 * GH + g] = make_float2(p, p);
                if (t16 == 0) al[g] = alpha;
            }
        }
        __syncwarp();

        // P.V over the visible tokens of the tile
#pragma unroll
        for (int g = 0; g < GH; ++g) {
            const float a_g = al[g];
            if (a_g != 1.f) {
#pragma unroll
                for (int c = 0; c < C::CPL / 2; ++c) acc[g][c] = make_float2(acc[g][c].x * a_g, acc[g][c].y * a_g);
            }
        }
        auto pv_token = [&](int t) {
            uint32_t vw[C::CPL / 2];
            if constexpr (C::CPL == 8) {
                const uint4 w = *reinterpret_cast<const uint4 *>(V + t * C::ROW + lane * 16);
                vw[0] = w.x; vw[1] = w.y; vw[2] = w.z; vw[3] = w.w;
            } else if constexpr (C::CPL == 4) {
                const uint2 w = *reinterpret_cast<const uint2 *>(V + t * C::ROW + lane * 8);
                vw[0] = w.x; vw[1] = w.y;
            } else {
                vw[0] = *reinterpret_cast<const uint32_t *>(V + t * C::ROW + lane * 4);
            }
            float2 pg[GH];   // {p, p} pairs written by the softmax
            if constexpr (GH >= 2) {
#pragma unroll
                for (int g2 = 0; g2 < GH / 2; ++g2) {
                    const float4 w4 = reinterpret_cast<const float4 *>(sp + 2 * t * GH)[g2];
                    pg[2 * g2] = make_float2(w4.x, w4.y);
                    pg[2 * g2 + 1] = make_float2(w4.z, w4.w);
                }
            } else {
                pg[0] = reinterpret_cast<const float2 *>(sp)[t];
            }
#pragma unroll
            for (int c = 0; c < C::CPL / 2; ++c) {
                const float2 vf = unpack2<T>(vw[c]);
#pragma unroll
                for (int g = 0; g < GH; ++g) acc[g][c] = ffma2(pg[g], vf, acc[g][c]);
            }
        };
        if (valid == C::TT) {
            // whole tile: unrolled, so the shared-memory loads of later tokens issue early
#pragma unroll
            for (int t = 0; t < C::TT; ++t) pv_token(t);
        } else {
            for (int t = 0; t < valid; ++t) pv_token(t);
        }
        __syncwarp();
        if (lane == 0 && i + C::NST < mine) {
            tc::fence_proxy_async_smem();
            issue(i + C::NST);
        }
    }
    if (!ok) atomicCAS(a.status, 0, PA_DEVICE_TIMEOUT_TMA);

    griddep_launch();
    // Merge the four warp states: M = max_w m_w, O = sum_w 2^(m_w-M) acc_w / sum_w 2^(m_w-M) l_w.
    __syncthreads();  // every ring is drained (each warp consumed all its tiles)
    float *mo = reinterpret_cast<float *>(smem);                    // [NW][GH][D] partial O
    float *ml = mo + (size_t)C::NW * GH * D;                         // [NW][GH][2] (m, l)
#pragma unroll
    for (int g = 0; g < GH; ++g)
#pragma unroll
        for (int c = 0; c < C::CPL / 2; ++c)
            reinterpret_cast<float2 *>(mo + ((size_t)warp * GH + g) * D + lane * C::CPL)[c] = acc[g][c];
#pragma unroll
    for (int k = 0; k < HP; ++k) {
        float lk = l_run[k];
#pragma unroll
        for (int o = 8; o; o >>= 1) lk += __shfl_xor_sync(0xffffffffu, lk, o);
        const int g = 2 * k + (lane >> 4);
        if (g < GH && (lane & 15) == 0) {
            ml[(warp * GH + g) * 2] = m_ref[k];
            ml[(warp * GH + g) * 2 + 1] = lk;
        }
    }
    __syncthreads();
    const int64_t rows = (int64_t)a.plan.queries * a.hq;
    for (int idx = threadIdx.x; idx < GH * D; idx += 128) {
        const int g = idx / D, c = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NW; ++w) M = fmaxf(M, ml[(w * GH + g) * 2]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < C::NW; ++w) {
                const float mw = ml[(w * GH + g) * 2];
                const float sc = mw == -INFINITY ? 0.f : exp2f(mw - M);
                L += sc * ml[(w * GH + g) * 2 + 1];
                O += sc * mo[((size_t)w * GH + g) * D + c];
            }
        }
        const int64_t row = (int64_t)qi * a.hq + h0 + g;
        if (a.splits == 1) {
            static_cast<T *>(a.out)[row * D + c] = from_f<T>(O / L);
        } else {
            a.ws_o[((int64_t)split * rows + row) * D + c] = L > 0.f ? O / L : 0.f;
            if (c == 0) a.ws_lse[(int64_t)split * rows + row] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
    }
}

int log2_exact(int v) {
    if (v <= 0 || (v & (v - 1))) return -1;
    int s = 0;
    while ((1 << s) < v) ++s;
    return s;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T, int D, int GH>
cudaError_t launch_t(const AttnArgs &a, int items, int use_list, const CUtensorMap &tk, const CUtensorMap &tv,
                     const TmaParams &tp, cudaStream_t st) {
    using C = Cfg<D, GH>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_tma_kernel<T, D, GH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    TmaParams p = tp;
    p.groups = (a.hq / a.hkv) / GH;
    const dim3 grid((unsigned)((int64_t)items * a.splits * a.hkv * p.groups));
    cudaError_t e = launch_pdl(decode_tma_kernel<T, D, GH>, grid, dim3(128), C::SMEM, st, tk, tv, a, use_list, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_d(const AttnArgs &a, int items, int use_list, const CUtensorMap &tk, const CUtensorMap &tv,
                     const TmaParams &tp, cudaStream_t st) {
    // At most 4 query heads per CTA: larger groups are covered by several CTAs
    // per KV head (adjacent blocks, so the second read of a page hits L2).  With
    // 8 heads in one CTA the kernel is issue-bound (about 8 flop per KV byte on
    // CUDA cores, twice the registers); two CTAs of 4 measured faster.
    const int G = a.hq / a.hkv;
    if (G % 4 == 0) return launch_t<T, D, 4>(a, items, use_list, tk, tv, tp, st);
    if (G % 2 == 0) return launch_t<T, D, 2>(a, items, use_list, tk, tv, tp, st);
    return launch_t<T, D, 1>(a, items, use_list, tk, tv, tp, st);
}

template <typename T>
cudaError_t launch_dt(const AttnArgs &a, int items, int use_list, const CUtensorMap &tk, const CUtensorMap &tv,
                      const TmaParams &tp, cudaStream_t st) {
    switch (a.d) {
        case 64: return launch_d<T, 64>(a, items, use_list, tk, tv, tp, st);
        case 128: return launch_d<T, 128>(a, items, use_list, tk, tv, tp, st);
        default: return launch_d<T, 256>(a, items, use_list, tk, tv, tp, st);
    }
}

}  // namespace

bool decode_tma_supported(const AttnArgs &a) {
    return (a.dtype == PA_BF16 || a.dtype == PA_F16) && a.p == 0 && a.d == a.dv &&
           (a.d == 64 || a.d == 128 || a.d == 256) && log2_exact(a.plan.page_size) >= 0 && aligned16(a.q) &&
           aligned16(a.k) && aligned16(a.v) && tma_available();
}

cudaError_t launch_decode_tma(const AttnArgs &a, bool use_decode_list, cudaStream_t st) {
    const int items = use_decode_list ? a.plan.n_decode : a.plan.queries;
    if (items == 0) return cudaSuccess;
    const bool bf16 = a.dtype == PA_BF16;
    const int ps = a.plan.page_size;
    TmaParams tp{};
    tp.ps_shift = log2_exact(ps);
    tp.box_rows = ps < 16 ? ps : 16;
    const uint64_t rows = (uint64_t)a.plan.pages * ps;
    CUtensorMap tk, tv;
    if (!encode_map_3d(&tk, a.k, bf16, a.d, a.hkv, rows, (uint64_t)a.d * 2, (uint64_t)a.d * 2 * a.hkv, a.d, 1,
                       tp.box_rows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map_3d(&tv, a.v, bf16, a.dv, a.hkv, rows, (uint64_t)a.dv * 2, (uint64_t)a.dv * 2 * a.hkv, a.dv, 1,
                       tp.box_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const int ul = use_decode_list ? 1 : 0;
    return bf16 ? launch_dt<__nv_bfloat16>(a, items, ul, tk, tv, tp, st)
                : launch_dt<__half>(a, items, ul, tk, tv, tp, st);
}

}  // namespace pa
