// Paged GQA decode on tcgen05 tensor cores, for groups of 8 or more query
// heads per KV head (head dim 128).
//
// Same operation as decode_tma.cu (ruDNN 0.1.7, src/paged_attention/mod.rs:
// `DevicePlan::attention`, `execute_attention_into`, `attention_into_split`):
// for query q and head h of KV head kv = h / G,
//   out[q, h, :] = sum_j softmax_j(scale * q[q,h,:] . K_j) V_j
// over the keys j the query sees.  With G query heads per KV head every KV
// byte feeds 2*G flops per dim; from G = 8 on, CUDA cores run out of issue
// slots before HBM runs out of bytes, so the contraction moves to the tensor
// core.  For each work unit (query, KV head, split) the group's G query rows
// go into the 128-row MMA tile C = 128 / R times (R = 32, 64 or 128 rows per
// copy; rows of a copy past G are zero and their results are never read) and
// runs, per 128-key tile,
//   S = Q . K^T   (M = 128, N = 128 keys, K = 128 dims; Q and K in shared memory)
//   O += P . V    (M = 128, N = 128 dims, K = 128 keys; P in TMEM, V in shared memory)
// Copy k runs its own online softmax over columns [k*128/C, (k+1)*128/C) of
// every tile and writes P there and zeros elsewhere, so its O rows collect
// only those keys; the copies merge at the end of the unit like split partials,
// through the Q buffer (the unit's S MMAs are done by then).  (With
// one copy, G = 8 rows in one warp's TMEM lanes, a single warp had to run the
// exponentials of every column on one SM sub-partition.)  The padding makes
// the tensor core do 128/G times the useful work, which still leaves it idle
// most of a tile's HBM time; the kernel stays bound by the KV bytes.
//
// The kernel is persistent: one CTA per SM walks the units in serpentine
// rounds, and the K/V ring streams from one unit into the next (one CTA per
// unit spent ~5.6 µs of every ~50 µs unit starting up and draining).
//
// Roles: warps 0-3 softmax/epilogue (thread r = MMA row r, TMEM lane r), warp 4
// TMA producer (128-key tiles of K and V, three stages; the lanes of the warp
// issue the boxes of a tile, so its page lookups run in parallel), warp 5 MMA
// issuer (P.V of tile t-1, then S of tile t: a stage goes back to the producer
// as soon as its own P.V has run; issued the other way round, a stage waited
// for the next tile's data as well and the kernel ran 2.5 % slower).  TMEM:
// three S/P buffers at columns 0, 128, 256, O at 384.  P is written
// back over its row of the S buffer as 16-bit pairs and read from there by
// P.V.  Keys outside the visible range score -inf; V rows past the visible
// end are zeroed before P.V (tail slots may hold anything).  Page sizes are
// powers of two from 8 on (each TMA box of at least 8 rows lands on a 1024-byte
// swizzle boundary).  All waits are bounded (timeout -> device status word).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
#include "sm103_tc.cuh"
#include "tma_host.h"

namespace pa {
namespace {

using namespace tc;

constexpr int kM = 128;                 // MMA rows: the group's heads, then zero rows
constexpr int kD = 128;                 // head dim = value dim
constexpr int kN = 128;                 // keys per tile
constexpr int kStages = 3;
constexpr int kCtasPerSm = 1;
constexpr int kSB = 3;                  // S/P buffers in TMEM
constexpr uint32_t kTmemCols = kSB * kN + kD <= 256 ? 256u : 512u;   // S/P buffers + O
static_assert(kSB * kN + kD <= 512, "TMEM holds the S/P buffers and O");
constexpr int kThreads = 192;           // 4 softmax warps + producer + MMA issuer
constexpr int kBlk = kN * 128;          // one 64-dim block of a 128-row tile (bytes)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSlack = 8.f;

struct Smem {
    uint8_t q[2][kM * 128];              // Q rows (group heads, then zeros), two 64-dim blocks
    uint8_t k[kStages][2][kBlk];         // key tiles, two 64-dim blocks each
    uint8_t v[kStages][2][kBlk];         // value tiles
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[kSB];                // S of tile kt in TMEM buffer kt % kSB
    uint64_t p_ready[kSB];               // P of tile kt written by every softmax thread -> p_ready[kt % kSB]
    uint64_t o_done[kSB];                // P.V of tile kt done -> o_done[kt % kSB]
    uint64_t q_ready;                    // Q rows of the CTA's current unit stored (phase = unit parity)
    uint64_t o_free;                     // the softmax warps have read O of the unit
    float ml[2 * kM];                    // per row (m, l) of the unit, for the merge of the copies
    uint32_t tmem_base;
};

// 1024-byte alignment for the swizzled operand tiles comes from the declared
// alignment of the dynamic shared memory (checked in the kernel).
constexpr size_t kSmemBytes = sizeof(Smem);
static_assert(kSmemBytes <= 232448, "decode shared memory above the per-block limit");

struct TcParams {
    int group;        // G = Hq / Hkv
    int ps_shift;     // log2(page_size)
    int box_rows;     // rows per TMA box: min(page_size, 128)
    float scale_log2;
    int bf16;
};

template <typename T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Named barrier over the four softmax warps (threads 0..127).
__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 128;\n" ::: "memory"); }

// AND of `pred` over the four softmax warps (a named-barrier reduction).
__device__ __forceinline__ bool __syncthreads_and_softmax(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

template <typename T, int CW>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     AttnArgs a, int use_list, TcParams tp) {
    griddep_wait();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if ((smem_u32(smem_raw) & 1023u) != 0u) {
        if (threadIdx.x == 0) atomicCAS(a.status, 0, PA_DEVICE_LAYOUT);
        return;
    }
    Smem &s = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = tp.group;
    const int ps = a.plan.page_size;

    // Persistent: each CTA walks its share of the units (item, split, KV head)
    // in that nesting, item slowest (the plan lists decode items longest
    // first).  Ring stages and S buffers follow one tile counter that runs on
    // across units, so the producer streams the next unit's tiles while the
    // current one finishes.
    const int items = use_list ? a.plan.n_decode : a.plan.queries;
    const int units = items * a.splits * a.hkv;
    struct Unit {
        int kvh, split, qi, seq_len, n_kt;
        int64_t j0, j1, jb;
        const int32_t *trow;
    };
    auto unit_at = [&](int u) -> Unit {
        Unit x;
        x.kvh = u % a.hkv;
        const int rest = u / a.hkv;
        x.split = rest % a.splits;
        const int item = rest / a.splits;
        x.qi = use_list ? a.plan.decode[item] : item;
        const int4 meta = a.plan.qmeta[x.qi];
        x.seq_len = a.plan.seq_lens[meta.x];
        int64_t lo, hi;
        visible_range(meta.y, x.seq_len, a.causal, a.window, lo, hi);
        split_bounds(lo, hi, a.splits, x.split, ps, x.j0, x.j1);
        // Tiles start on a TMA box boundary (no box crosses a page); keys of the
        // first tile below j0 (window or split start) are masked.
        x.jb = x.j0 < x.j1 ? x.j0 / tp.box_rows * tp.box_rows : x.j0;
        x.n_kt = (int)((x.j1 - x.jb + kN - 1) / kN);
        x.trow = a.plan.table + (int64_t)meta.x * a.plan.width;
        return x;
    };

    // The CTA's i-th unit: round i of grid-sized rounds, taken in serpentine
    // order (odd rounds from the last CTA down), so with units sorted by
    // decreasing size the CTAs' totals even out.  The last round may be
    // partial: a CTA whose slot in it lies past the end has no i-th unit.
    auto unit_of = [&](int i) -> int {
        const int g = (int)gridDim.x, b = (int)blockIdx.x;
        const int slot = (i & 1) ? g - 1 - b : b;
        const int u = i * g + slot;
        return (i * g < units && u < units) ? u : units;
    };

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.kv_full[i], 1);
            mbar_init(&s.kv_empty[i], 1);
        }
        for (int i = 0; i < kSB; ++i) {
            mbar_init(&s.s_full[i], 1);
            mbar_init(&s.p_ready[i], 128);
            mbar_init(&s.o_done[i], 1);
        }
        mbar_init(&s.q_ready, 128);
        mbar_init(&s.o_free, 128);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    auto tmem_s = [tmem](int b) -> uint32_t { return tmem + (uint32_t)kN * (uint32_t)b; };   // S / P buffers
    const uint32_t tmem_o = tmem + (uint32_t)(kSB * kN);

    if (warp == 4) {
        // ---------------------------------------------------- TMA producer --
        // Lane b issues the boxes of box b of a tile (its page lookup runs in
        // parallel with the other lanes'); lane 0 posts the expected bytes.
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        const int oob_row = a.plan.pages * ps;        // past the cache: TMA zero fill
        const int nb = kN / tp.box_rows;
        int gt = 0;                                   // tiles streamed so far (all units)
        bool ok = true;
        for (int i = 0; ok && unit_of(i) < units; ++i) {
            const Unit x = unit_at(unit_of(i));
            const int used_pages = (x.seq_len + ps - 1) >> tp.ps_shift;
            for (int kt = 0; kt < x.n_kt; ++kt, ++gt) {
                const int st = gt % kStages;
                if (gt >= kStages && !__all_sync(0xffffffffu, mbar_wait(&s.kv_empty[st], ((gt / kStages) - 1) & 1))) {
                    if (lane == 0) atomicCAS(a.status, 0, PA_DEVICE_TIMEOUT_TMA);
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&s.kv_full[st], 4u * kBlk);
                __syncwarp();
                const int64_t jt = x.jb + (int64_t)kt * kN;
                for (int bi = lane; bi < nb; bi += 32) {
                    const int b = bi * tp.box_rows;
                    const int64_t j = jt + b;
                    const int64_t lp = j >> tp.ps_shift;
                    const int row = lp < used_pages ? x.trow[lp] * ps + (int)(j & (ps - 1)) : oob_row;
                    for (int blk = 0; blk < 2; ++blk) {
                        tma_load_3d(s.k[st][blk] + b * 128, &tm_k, blk * 64, x.kvh, row, &s.kv_full[st]);
                        tma_load_3d(s.v[st][blk] + b * 128, &tm_v, blk * 64, x.kvh, row, &s.kv_full[st]);
                    }
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------ MMA issuer --
        // Per tile: P.V of the previous tile first (its stage goes back to the
        // producer as soon as its own P.V has run), then S of this tile.  The
        // first P.V of a unit overwrites O, so it waits until the softmax warps
        // have read O of the previous unit.
        if (lane == 0) {
            const uint32_t idesc_s = idesc_f16(kM, kN, tp.bf16 != 0, false, false);
            const uint32_t idesc_o = idesc_f16(kM, kD, tp.bf16 != 0, false, true);
            auto issue_pv = [&](int g, bool first) -> bool {     // g: global tile index
                if (!mbar_wait(&s.p_ready[g % kSB], (g / kSB) & 1)) return false;
                tc_fence_after();
                const int st = g % kStages;
                const uint32_t v_addr = smem_u32(s.v[st][0]);
                for (int ks = 0; ks < kN / 16; ++ks) {
                    const uint64_t b = smem_desc(v_addr + ks * 2048, kBlk, 1024, kLayoutSwizzle128B);
                    mma_f16_ts(tmem_o, tmem_s(g % kSB) + ks * 8, b, idesc_o, (!first || ks > 0) ? 1u : 0u);
                }
                mma_commit(&s.o_done[g % kSB]);
                mma_commit(&s.kv_empty[st]);
                return true;
            };
            bool ok = true;
            int gt = 0;
            for (int i = 0; ok && unit_of(i) < units; ++i) {
                const Unit x = unit_at(unit_of(i));
                if (!mbar_wait(&s.q_ready, i & 1)) { ok = false; break; }
                for (int kt = 0; kt < x.n_kt; ++kt, ++gt) {
                    if (kt > 0) {
                        if (kt == 1 && i > 0 && !mbar_wait(&s.o_free, (i - 1) & 1)) { ok = false; break; }
                        if (!issue_pv(gt - 1, kt == 1)) { ok = false; break; }
                    }
                    const int st = gt % kStages, sb = gt % kSB;
                    if (!mbar_wait(&s.kv_full[st], (gt / kStages) & 1)) { ok = false; break; }
                    // the buffer's previous tile (gt-kSB) must be through its P.V (P lives in it)
                    if (gt >= kSB && !mbar_wait(&s.o_done[sb], ((gt / kSB) - 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    for (int ks = 0; ks < kD / 16; ++ks) {
                        const int blk = ks / 4, k = ks % 4;
                        const uint64_t qa = smem_desc(smem_u32(s.q[blk]) + k * 32, 16, 1024, kLayoutSwizzle128B);
                        const uint64_t kb = smem_desc(smem_u32(s.k[st][blk]) + k * 32, 16, 1024, kLayoutSwizzle128B);
                        mma_f16_ss(tmem_s(sb), qa, kb, idesc_s, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(&s.s_full[sb]);
                }
                if (!ok) break;
                if (x.n_kt > 0) {
                    if (x.n_kt == 1 && i > 0 && !mbar_wait(&s.o_free, (i - 1) & 1)) { ok = false; break; }
                    if (!issue_pv(gt - 1, x.n_kt == 1)) { ok = false; break; }
                }
            }
            if (!ok) atomicCAS(a.status, 0, PA_DEVICE_TIMEOUT_MMA);
        }
    } else {
        // ---------------------------------------- softmax / epilogue rows --
        // Row r belongs to copy r / R of the group (R = 32, 64 or 128 rows per
        // copy, C = 128 / R copies) and is head r % R (a padding row when that
        // is >= G).  Copy k runs its own online softmax over columns
        // [k*CW, (k+1)*CW) of every tile and writes P there and zeros elsewhere,
        // so its O rows collect only those keys; the copies merge at the end of
        // each unit like split partials, through the Q buffer (S of the unit is
        // done by then) before the next unit's Q is written there.
        const int r = tid;
        constexpr int R = kM * CW / kN;                  // rows per copy
        constexpr int C = kN / CW;                       // copies
        const int copy = r / R, h = r - copy * R;
        const int c0 = copy * CW;
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        const int64_t rows = (int64_t)a.plan.queries * a.hq;
        bool ok = true;
        int gt = 0;                                      // tiles consumed so far (all units)
        float sc[CW];
        // Q rows into the two swizzled 64-dim blocks (16-byte chunk c of row at
        // chunk c ^ (row & 7)); each copy holds the group's heads, rows past G in
        // a copy are zero.  Thread tid moves chunk tid % 16 of rows tid / 16 + 8j:
        // load_q puts every load in flight, store_q writes them to the Q buffer.
        auto load_q = [&](const Unit &x, uint4 (&val)[kM / 8]) {
            const T *qsrc = static_cast<const T *>(a.q) + ((int64_t)x.qi * a.hq + (int64_t)x.kvh * G) * kD;
            const int c = tid & 15;
#pragma unroll
            for (int j = 0; j < kM / 8; ++j) {
                const int hr = ((tid >> 4) + 8 * j) % R;
                val[j] = hr < G ? reinterpret_cast<const uint4 *>(qsrc + (int64_t)hr * kD)[c] : make_uint4(0, 0, 0, 0);
            }
        };
        auto store_q = [&](const uint4 (&val)[kM / 8]) {
            const int c = tid & 15, blk = c >> 3, cc = c & 7;
#pragma unroll
            for (int j = 0; j < kM / 8; ++j) {
                const int row = (tid >> 4) + 8 * j;
                *reinterpret_cast<uint4 *>(s.q[blk] + row * 128 + ((cc ^ (row & 7)) * 16)) = val[j];
            }
            fence_proxy_async_smem();       // generic stores before the tensor core reads them
            mbar_arrive(&s.q_ready);
        };
        // The next unit's parameters and (below 128 columns per copy, where the
        // registers allow) its Q loads are issued before this unit's merge, so
        // their latency overlaps it.
        constexpr bool kPrefetchQ = CW < 128;
        Unit x = unit_of(0) < units ? unit_at(unit_of(0)) : Unit{};
        if (unit_of(0) < units) {
            uint4 val[kM / 8];
            load_q(x, val);
            store_q(val);
        }
        for (int i = 0; ok && unit_of(i) < units; ++i) {
            float m_ref = -INFINITY, l = 0.f;
            for (int kt = 0; ok && kt < x.n_kt; ++kt, ++gt) {
                const int pb = gt % kSB;
                const int64_t kbase = x.jb + (int64_t)kt * kN;
                const int valid = (int)((x.j1 - kbase) < kN ? (x.j1 - kbase) : kN);
                const int first = (int)(x.j0 > kbase ? x.j0 - kbase : 0);
                ok = __all_sync(0xffffffffu, mbar_wait(&s.s_full[pb], (gt / kSB) & 1));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < CW; c += 32) tmem_ld32f(tmem_s(pb) + lane_off + c0 + c, sc + c);
                tmem_wait_ld();
                if (valid < kN || first > 0) {
#pragma unroll
                    for (int c = 0; c < CW; ++c)
                        if (c0 + c >= valid || c0 + c < first) sc[c] = -INFINITY;
                }
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < CW; c += 8) {
                    mx[0] = fmax3(mx[0], sc[c], sc[c + 1]);
                    mx[1] = fmax3(mx[1], sc[c + 2], sc[c + 3]);
                    mx[2] = fmax3(mx[2], sc[c + 4], sc[c + 5]);
                    mx[3] = fmax3(mx[3], sc[c + 6], sc[c + 7]);
                }
                const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * tp.scale_log2;
                float alpha = 1.f;
                if (mt > m_ref + kSlack) {
                    alpha = exp2f(m_ref - mt);          // 0 while this copy had seen no key
                    m_ref = mt;
                }
                // rescaling O needs the previous P.V finished (rare: the row max moved by > 2^8)
                if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&s.o_done[(gt - 1) % kSB], ((gt - 1) / kSB) & 1));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < kD; c += 16) {
                        uint32_t v[16];
                        tmem_ld16(tmem_o + lane_off + c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                        tmem_st16(tmem_o + lane_off + c, v);
                    }
                    tmem_wait_st();
                }
                // P = exp2(s * scale - m_ref) over this copy's columns as 16-bit
                // pairs; zeros over the other copies' columns.  A copy that has
                // seen no visible key yet has only -inf scores (P = 0).
                const float mref = m_ref == -INFINITY ? 0.f : m_ref;
                const float2 sc2 = make_float2(tp.scale_log2, tp.scale_log2);
                const float2 nm2 = make_float2(-mref, -mref);
                const float2 *s2 = reinterpret_cast<const float2 *>(sc);
                float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < CW; c += 32) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 xx = ffma2(s2[c / 2 + i], sc2, nm2);
                        const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
                        ls[i & 1] = fadd2(ls[i & 1], pp);
                        pk[i] = pack2<T>(pp.x, pp.y);
                    }
                    tmem_st16(tmem_s(pb) + lane_off + (c0 + c) / 2, pk);
                }
                if (CW < kN) {
                    uint32_t zero[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) zero[i] = 0u;
#pragma unroll
                    for (int c = 0; c < kN; c += 32)
                        if (c < c0 || c >= c0 + CW) tmem_st16(tmem_s(pb) + lane_off + c / 2, zero);
                }
                tmem_wait_st();
                const float2 lsum = fadd2(ls[0], ls[1]);
                l = l * alpha + (lsum.x + lsum.y);
                // value rows past the visible end must not reach P.V (tail slots may hold NaN)
                if (valid < kN) {
                    const int st = gt % kStages;
                    ok = __all_sync(0xffffffffu, mbar_wait(&s.kv_full[st], (gt / kStages) & 1));
                    if (!ok) break;
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    for (int row = valid + tid; row < kN; row += 128)
#pragma unroll
                        for (int blk = 0; blk < 2; ++blk)
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                *reinterpret_cast<uint4 *>(s.v[st][blk] + row * 128 + i * 16) = z;
                    fence_proxy_async_smem();  // the zeroed rows before the tensor core reads them
                }
                tc_fence_before();
                mbar_arrive(&s.p_ready[pb]);
            }
            const bool more = unit_of(i + 1) < units;
            const Unit nx = more ? unit_at(unit_of(i + 1)) : x;
            uint4 qn[kM / 8];
            if (kPrefetchQ && more) load_q(nx, qn);
            if (ok && x.n_kt > 0)
                ok = __all_sync(0xffffffffu, mbar_wait(&s.o_done[(gt - 1) % kSB], ((gt - 1) / kSB) & 1));
            // every softmax thread reaches the merge barriers, whatever happened above
            ok = __syncthreads_and_softmax(ok);
            if (!ok) {
                atomicCAS(a.status, 0, PA_DEVICE_TIMEOUT_SOFTMAX);
                break;
            }
            const int64_t orow0 = (int64_t)x.qi * a.hq + (int64_t)x.kvh * G;      // output row of head 0
            if (x.n_kt == 0) {
                // empty split (only with splits > 1): zero partial, lse = -inf
                if (copy == 0 && h < G && a.splits > 1) {
                    float *dst = a.ws_o + ((int64_t)x.split * rows + orow0 + h) * kD;
                    for (int c = 0; c < kD; c += 4)
                        *reinterpret_cast<float4 *>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                    a.ws_lse[(int64_t)x.split * rows + orow0 + h] = -INFINITY;
                }
            } else {
                // Merge the copies: M = max_k m_k, w_k = 2^(m_k - M), L = sum_k w_k l_k,
                // O = sum_k w_k O_k / L.
                tc_fence_after();
                s.ml[2 * r] = m_ref;
                s.ml[2 * r + 1] = l;
                softmax_bar();
                float M = -INFINITY;
                for (int k = 0; k < C; ++k) M = fmaxf(M, s.ml[2 * (k * R + h)]);
                float L = 0.f;
                for (int k = 0; k < C; ++k) {
                    const float mk = s.ml[2 * (k * R + h)];
                    L += mk == -INFINITY ? 0.f : exp2f(mk - M) * s.ml[2 * (k * R + h) + 1];
                }
                const float wk = (m_ref == -INFINITY || !(L > 0.f)) ? 0.f : exp2f(m_ref - M) / L;
                if (copy == 0 && h < G && a.splits > 1)
                    a.ws_lse[(int64_t)x.split * rows + orow0 + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
                // one pass per 64 output columns; the scaled partials [C][G][64] fill the Q buffer
                float *ob = reinterpret_cast<float *>(s.q[0]);
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
#pragma unroll 1
                    for (int c = 0; c < 64; c += 16) {
                        uint32_t v[16];
                        tmem_ld16(tmem_o + lane_off + 64 * half + c, v);
                        tmem_wait_ld();
                        if (h < G) {
#pragma unroll
                            for (int i = 0; i < 16; i += 4)
                                *reinterpret_cast<float4 *>(ob + ((size_t)copy * G + h) * 64 + c + i) =
                                    make_float4(__uint_as_float(v[i]) * wk, __uint_as_float(v[i + 1]) * wk,
                                                __uint_as_float(v[i + 2]) * wk, __uint_as_float(v[i + 3]) * wk);
                        }
                    }
                    softmax_bar();
                    // sum the copies, 4 columns per thread and step
                    for (int idx = tid; idx < G * 16; idx += 128) {
                        const int hh = idx >> 4, c = (idx & 15) * 4;
                        float4 o = *reinterpret_cast<const float4 *>(ob + (size_t)hh * 64 + c);
                        for (int k = 1; k < C; ++k) {
                            const float4 y = *reinterpret_cast<const float4 *>(ob + ((size_t)k * G + hh) * 64 + c);
                            o.x += y.x; o.y += y.y; o.z += y.z; o.w += y.w;
                        }
                        const int col = 64 * half + c;
                        if (a.splits == 1) {
                            uint2 w;
                            w.x = pack2<T>(o.x, o.y);
                            w.y = pack2<T>(o.z, o.w);
                            *reinterpret_cast<uint2 *>(static_cast<T *>(a.out) + (orow0 + hh) * kD + col) = w;
                        } else {
                            *reinterpret_cast<float4 *>(a.ws_o + ((int64_t)x.split * rows + orow0 + hh) * kD + col) = o;
                        }
                    }
                    softmax_bar();      // the Q buffer is read before it is written again
                }
            }
            // O of this unit has been read: the next unit's first P.V may overwrite it
            tc_fence_before();
            mbar_arrive(&s.o_free);
            if (more) {
                // the merge has read the Q buffer (its last barrier): the next Q goes in
                if (!kPrefetchQ) load_q(nx, qn);
                store_q(qn);
            }
            x = nx;
        }
    }
    griddep_launch();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

int log2_exact(int v) {
    if (v <= 0 || (v & (v - 1))) return -1;
    int s = 0;
    while ((1 << s) < v) ++s;
    return s;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T, int CW>
cudaError_t launch_cw(const AttnArgs &a, int items, int use_list, const CUtensorMap &tk, const CUtensorMap &tv,
                      const TcParams &tp, cudaStream_t st) {
    // Persistent grid: as many CTAs as fit on the GPU at once (one per SM), or
    // fewer when the caller keeps SMs for a concurrent kernel.
    static int resident = 0;
    if (resident == 0) {
        cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<T, CW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        int per_sm = 0, dev = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_tc_kernel<T, CW>, kThreads, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        resident = per_sm * sms > 0 ? per_sm * sms : 1;
    }
    const int64_t units = (int64_t)items * a.splits * a.hkv;
    int64_t ctas = units < resident ? units : resident;
    if (a.max_ctas > 0 && a.max_ctas < ctas) ctas = a.max_ctas;
    const dim3 grid((unsigned)ctas);
    cudaError_t e = launch_pdl(decode_tc_kernel<T, CW>, grid, dim3(kThreads), kSmemBytes, st, tk, tv, a, use_list, tp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Copies of the group in the 128 MMA rows: 4 for G <= 32, 2 for G <= 64, 1 above;
// each copy's softmax covers 128 / copies columns of a tile.
template <typename T>
cudaError_t launch_t(const AttnArgs &a, int items, int use_list, const CUtensorMap &tk, const CUtensorMap &tv,
                     const TcParams &tp, cudaStream_t st) {
    if (tp.group <= 32) return launch_cw<T, 32>(a, items, use_list, tk, tv, tp, st);
    if (tp.group <= 64) return launch_cw<T, 64>(a, items, use_list, tk, tv, tp, st);
    return launch_cw<T, 128>(a, items, use_list, tk, tv, tp, st);
}

}  // namespace

bool decode_tc_supported(const AttnArgs &a) {
    const int G = a.hkv > 0 ? a.hq / a.hkv : 0;
    return (a.dtype == PA_BF16 || a.dtype == PA_F16) && a.p == 0 && a.d == kD && a.dv == kD && G >= 8 &&
           G <= kM && log2_exact(a.plan.page_size) >= 3 && aligned16(a.q) && aligned16(a.k) && aligned16(a.v) &&
           aligned16(a.out) && tma_available();
}

cudaError_t launch_decode_tc(const AttnArgs &a, bool use_decode_list, cudaStream_t st) {
    const int items = use_decode_list ? a.plan.n_decode : a.plan.queries;
    if (items == 0) return cudaSuccess;
    const bool bf16 = a.dtype == PA_BF16;
    const int ps = a.plan.page_size;
    TcParams tp{};
    tp.group = a.hq / a.hkv;
    tp.ps_shift = log2_exact(ps);
    tp.box_rows = ps < kN ? ps : kN;
    tp.scale_log2 = a.scale * kLog2e;
    tp.bf16 = bf16 ? 1 : 0;
    const uint64_t rows = (uint64_t)a.plan.pages * ps;
    CUtensorMap tk, tv;
    // caches viewed as [rows, Hkv, 128]; boxes of 64 dims x 1 head x box_rows rows, 128-byte swizzle
    if (!encode_map_3d(&tk, a.k, bf16, kD, a.hkv, rows, (uint64_t)kD * 2, (uint64_t)kD * 2 * a.hkv, 64, 1,
                       tp.box_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_3d(&tv, a.v, bf16, kD, a.hkv, rows, (uint64_t)kD * 2, (uint64_t)kD * 2 * a.hkv, 64, 1,
                       tp.box_rows, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int ul = use_decode_list ? 1 : 0;
    return bf16 ? launch_t<__nv_bfloat16>(a, items, ul, tk, tv, tp, st)
                : launch_t<__half>(a, items, ul, tk, tv, tp, st);
}

}  // namespace pa
