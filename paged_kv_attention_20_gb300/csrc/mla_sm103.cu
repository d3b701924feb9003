// MLA decode on tcgen05 tensor cores, one CTA pair per (query, 128 heads).
//
// ruDNN 0.1.7, src/paged_attention/mod.rs, doc of `DevicePlan::mla`: absorbed
// Q [queries, H, R] and position Q [queries, H, P] score against one shared
// latent head [pages, ps, 1, R] and a rotated position cache [pages, ps, 1, P];
// the latent is both key and value, so
//   s_j = scale * (q . c_j + qp . r_j),   out = sum_j softmax_j c_j   ([queries, H, R]).
// The scale comes from the model's original QK dims (caller supplied).
//
// The 128 x 512 fp32 output tile fills all of one SM's tensor memory, so the
// output columns are split over a CTA pair (a thread-block cluster of 2, which
// keeps the two on the GPU at the same time so the second reads each key tile
// from L2): CTA c accumulates output columns 256c..256c+255.  Each CTA computes
// the whole 128 x 64 score tile of every key tile itself (all 512 latent and 64
// position columns), so the pair exchanges nothing; the score contraction is
// done twice, which costs less tensor time than moving the partial scores
// between SMs (the SM-to-SM network carries only ~20 GB/s per SM each way).
//
// Tensor memory (512 columns): the CTA's own 256 latent Q columns (16-bit
// pairs, columns 0..127), two S/P buffers of 64 columns (128, 192), O (256..511).
// Shared memory: the other 256 latent Q columns and the 64 position columns
// (80 KB, the A operand of their part of Q.K^T), and two rings of key tiles:
//   w: the peer's latent half + the position columns, used by Q.K^T only and
//      released as soon as that part of the score MMA has run;
//   v: the CTA's own latent half, the K-major B operand of the rest of Q.K^T
//      and the MN-major B operand (V) of P.V, released after P.V.
// P (16-bit) is written back over its row of the S buffer and read from TMEM
// by P.V; two S/P buffers let the score MMAs of the next tile run during this
// tile's softmax.  One thread issues a tcgen05.mma only every ~100 cycles while
// the tensor core finishes a 128 x 64 x 16 step in about half of that, so the
// score MMAs of even and odd key tiles come from two threads (each into its
// own S buffer and ring slot) and a third issues every P.V in order.
//
// Roles per CTA: warps 0-3 softmax/epilogue (thread r = head r, TMEM lane r),
// warp 4 TMA producer of Q and the w ring, warps 5 and 7 score-MMA issuers
// (even / odd key tiles), warp 6 TMA producer of the v ring, warp 8 P.V
// issuer.  Key tiles are 64 keys, one page at page_size 64
// (several boxes for smaller pages).  Keys at or past the visible end score
// -inf and their latent rows are zeroed before P.V (tail slots may hold
// anything).  All waits are bounded (timeout -> device status word).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
#include "sm103_tc.cuh"
#include "tma_host.h"

namespace pa {
namespace {

using namespace tc;

constexpr int kHeads = 128;               // M: heads per CTA (TMEM lanes)
constexpr int kR = 512;                   // latent rank
constexpr int kP = 64;                    // rotary position dims
constexpr int kN = 64;                    // keys per tile
constexpr int kThreads = 288;             // 4 softmax + w producer + score MMA (even tiles) + v producer
                                          // + score MMA (odd tiles) + P.V MMA
constexpr int kBlk = kHeads * 128;        // one 64-column block of the Q tile (bytes)
constexpr int kKBlk = kN * 128;           // one 64-column block of a key tile (bytes)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSlack = 8.f;

struct Smem {
    uint8_t q[5][kBlk];                  // the peer half of latent Q (blocks 0..3) and position Q (block 4)
    uint8_t w[2][5][kKBlk];              // score-only key blocks: peer latent half (0..3), position (4)
    uint8_t v[2][4][kKBlk];              // own latent half: keys of Q.K^T and the V of P.V
    uint64_t q_full;                     // Q blocks landed
    uint64_t q_ready;                    // own latent Q rows stored in TMEM by the row threads
    uint64_t w_full[2], w_empty[2];
    uint64_t v_full[2], v_empty[2];
    uint64_t s_full[2];                  // S of tile kt in TMEM buffer kt % 2
    uint64_t p_ready[2];                 // P of tile kt in TMEM (all 128 rows) -> p_ready[kt % 2].  One
                                         // barrier per tile in flight: softmax warps are not in step,
                                         // and a warp already on tile kt+1 must not count toward kt
    uint64_t o_done[2];                  // P.V of tile kt done -> o_done[kt % 2]
    uint32_t tmem_base;
};

// The operand tiles need 1024-byte alignment (128-byte swizzle atoms); the
// dynamic shared memory is declared with that alignment and no slack is
// requested.  The kernel checks the alignment (PA_DEVICE_LAYOUT otherwise).
constexpr size_t kSmemBytes = sizeof(Smem);
static_assert(kSmemBytes <= 232448, "MLA shared memory above the per-block limit");

struct MlaParams {
    PlanView plan;
    void *out;
    const void *q;          // absorbed Q [queries, H, 512] (own half -> TMEM by the row threads)
    float *ws_o, *ws_lse;
    int32_t *status;
    int heads;              // H
    int head_blocks;        // ceil(H / 128)
    int use_list;
    int splits;
    int box_rows;           // rows per TMA box: min(page_size, 64)
    int ps_shift;
    float scale_log2;
    int causal;
    int window;
    int bf16;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}

template <typename T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <typename T>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
               const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_kp,
               MlaParams prm) {
    griddep_wait();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if ((smem_u32(smem_raw) & 1023u) != 0u) {
        if (threadIdx.x == 0) atomicCAS(prm.status, 0, PA_DEVICE_LAYOUT);
        return;
    }
    Smem &s = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank();
    const int own_col = (int)rank * 256, peer_col = (int)(rank ^ 1u) * 256;

    // CTA pair -> (item, head block, split)
    const int cl = blockIdx.x >> 1;
    const int hb = cl % prm.head_blocks;
    const int rest = cl / prm.head_blocks;
    const int item = rest % (prm.use_list ? prm.plan.n_decode : prm.plan.queries);
    const int split = rest / (prm.use_list ? prm.plan.n_decode : prm.plan.queries);
    const int qi = prm.use_list ? prm.plan.decode[item] : prm.plan.order[item];
    const int4 meta = prm.plan.qmeta[qi];
    const int seq = meta.x, pos = meta.y;
    const int ps = prm.plan.page_size;
    const int seq_len = prm.plan.seq_lens[seq];
    int64_t lo, hi;
    visible_range(pos, seq_len, prm.causal, prm.window, lo, hi);
    int64_t j0, j1;
    split_bounds(lo, hi, prm.splits, split, ps, j0, j1);
    // Key tiles start on a multiple of 64 (no TMA box crosses a page); keys of
    // the first tile below j0 (sliding window or split start) are masked.
    const int64_t jb = j0 < j1 ? j0 / kN * kN : j0;
    const int n_kt = (int)((j1 - jb + kN - 1) / kN);
    const int32_t *trow = prm.plan.table + (int64_t)seq * prm.plan.width;

    if (tid == 0) {
        mbar_init(&s.q_full, 1);
        mbar_init(&s.q_ready, kHeads);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.w_full[i], 1);
            mbar_init(&s.w_empty[i], 1);
            mbar_init(&s.v_full[i], 1);
            mbar_init(&s.v_empty[i], 1);
            mbar_init(&s.s_full[i], 1);
            mbar_init(&s.p_ready[i], kHeads);
            mbar_init(&s.o_done[i], 1);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    const uint32_t tmem_q = tmem;                                 // own latent Q: 256 x 16-bit = 128 columns
    auto tmem_s = [tmem](int b) -> uint32_t { return tmem + 128u + 64u * (uint32_t)b; };   // S / P buffers 0, 1
    const uint32_t tmem_o = tmem + 256;

    // cache row of key j (rows of pages the table does not cover read as TMA zero fill)
    const int used_pages = (seq_len + ps - 1) >> prm.ps_shift;
    const int oob_row = prm.plan.pages * ps;
    auto key_row = [&](int64_t j) -> int {
        const int64_t lp = j >> prm.ps_shift;
        return lp < used_pages ? trow[lp] * ps + (int)(j & (ps - 1)) : oob_row;
    };

    if (warp == 4 || warp == 6) {
        // ------------------------------------------------- TMA producers --
        // warp 4: Q blocks, then the w ring; warp 6: the v ring.
        if (lane == 0) {
            const bool w_ring = warp == 4;
            if (w_ring) {
                tma_prefetch_desc(&tm_lat);
                tma_prefetch_desc(&tm_kp);
                mbar_arrive_expect_tx(&s.q_full, 5 * kBlk);
                for (int blk = 0; blk < 4; ++blk)
                    tma_load_3d(s.q[blk], &tm_q, peer_col + blk * 64, hb * kHeads, qi, &s.q_full);
                tma_load_3d(s.q[4], &tm_qp, 0, hb * kHeads, qi, &s.q_full);
            }
            uint64_t *full = w_ring ? s.w_full : s.v_full;
            uint64_t *empty = w_ring ? s.w_empty : s.v_empty;
            const int col = w_ring ? peer_col : own_col;
            for (int kt = 0; kt < n_kt; ++kt) {
                const int slot = kt & 1;
                if (kt >= 2 && !mbar_wait(&empty[slot], ((kt / 2) - 1) & 1)) {
                    atomicCAS(prm.status, 0, PA_DEVICE_TIMEOUT_TMA);
                    break;
                }
                mbar_arrive_expect_tx(&full[slot], (uint32_t)(w_ring ? 5 : 4) * kKBlk);
                uint8_t *dst = w_ring ? s.w[slot][0] : s.v[slot][0];
                const int64_t jt = jb + (int64_t)kt * kN;
                for (int b = 0; b < kN; b += prm.box_rows) {
                    const int row = key_row(jt + b);
                    for (int blk = 0; blk < 4; ++blk)
                        tma_load_2d(dst + blk * kKBlk + b * 128, &tm_lat, col + blk * 64, row, &full[slot]);
                    if (w_ring) tma_load_2d(dst + 4 * kKBlk + b * 128, &tm_kp, 0, row, &full[slot]);
                }
            }
        }
    } else if (warp == 5 || warp == 7) {
        // ------------------------------------------------ score MMA issuers --
        // A thread issues a tcgen05.mma only every ~100 cycles, so a 64-key
        // tile's 36 score MMAs (20 with Q from shared memory, 16 with the own
        // latent half of Q from TMEM) take one thread three times as long as
        // the tensor core needs for them.  Warp 5 issues the scores of the even
        // key tiles into S buffer 0, warp 7 those of the odd tiles into buffer
        // 1; warp 8 issues every P.V.  A buffer is written again only once the
        // P.V of the tile before has read its P (o_done).
        if (lane == 0) {
            const int par = warp == 5 ? 0 : 1;              // tiles kt with kt % 2 == par, ring slot par
            const uint32_t idesc_s = idesc_f16(kHeads, kN, prm.bf16 != 0, false, false);
            bool ok = mbar_wait(&s.q_full, 0) && mbar_wait(&s.q_ready, 0);
            const uint32_t d_s = tmem_s(par);
            // descriptors of the operand bases; a K-step adds its byte offset / 16
            // to the start-address field (shared addresses stay below 256 KB)
            uint64_t qd[5];
#pragma unroll
            for (int blk = 0; blk < 5; ++blk) qd[blk] = smem_desc(smem_u32(s.q[blk]), 16, 1024, kLayoutSwizzle128B);
            for (int kt = par; ok && kt < n_kt; kt += 2) {
                const uint32_t ph = (uint32_t)(kt / 2) & 1u;
                if (!mbar_wait(&s.w_full[par], ph)) { ok = false; break; }
                // the buffer's previous tile (kt-2) must be through its P.V (P lives in it)
                if (kt >= 2 && !mbar_wait(&s.o_done[par], ph ^ 1u)) { ok = false; break; }
                tc_fence_after();
                // peer latent half and position columns: A (Q) from shared memory
#pragma unroll
                for (int blk = 0; blk < 5; ++blk) {
                    const uint64_t wd = smem_desc(smem_u32(s.w[par][blk]), 16, 1024, kLayoutSwizzle128B);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f16_ss(d_s, qd[blk] + (uint64_t)(k * 2), wd + (uint64_t)(k * 2), idesc_s,
                                   (blk > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&s.w_empty[par]);
                if (!mbar_wait(&s.v_full[par], ph)) { ok = false; break; }
                tc_fence_after();
                // own latent half: A (Q) from TMEM
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    const uint64_t vd = smem_desc(smem_u32(s.v[par][blk]), 16, 1024, kLayoutSwizzle128B);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f16_ts(d_s, tmem_q + blk * 32 + k * 8, vd + (uint64_t)(k * 2), idesc_s, 1u);
                }
                mma_commit(&s.s_full[par]);
            }
            if (!ok) atomicCAS(prm.status, 0, PA_DEVICE_TIMEOUT_MMA);
        }
    } else if (warp == 8) {
        // ------------------------------------------------------ P.V issuer --
        // O += P V for every key tile in order (one accumulator, one thread).
        // S of the tile has completed before its P exists, so the v stage that
        // both the score and this MMA read is free once this MMA has run.
        if (lane == 0) {
            const uint32_t idesc_o = idesc_f16(kHeads, 256, prm.bf16 != 0, false, true);
            bool ok = true;
            for (int kt = 0; ok && kt < n_kt; ++kt) {
                const int slot = kt & 1;
                const uint32_t ph = (uint32_t)(kt / 2) & 1u;
                if (!mbar_wait(&s.p_ready[slot], ph) || !mbar_wait(&s.v_full[slot], ph)) { ok = false; break; }
                tc_fence_after();
                const uint64_t vd = smem_desc(smem_u32(s.v[slot][0]), kKBlk, 1024, kLayoutSwizzle128B);
                const uint32_t p_tmem = tmem_s(slot);           // P (16-bit pairs) over the S columns
#pragma unroll
                for (int ks = 0; ks < kN / 16; ++ks)
                    mma_f16_ts(tmem_o, p_tmem + ks * 8, vd + (uint64_t)((ks * 2048) >> 4), idesc_o,
                               (kt > 0 || ks > 0) ? 1u : 0u);
                mma_commit(&s.o_done[slot]);
                mma_commit(&s.v_empty[slot]);
            }
            if (!ok) atomicCAS(prm.status, 0, PA_DEVICE_TIMEOUT_MMA);
        }
    } else if (warp < 4) {
        // ---------------------------------------- softmax / epilogue rows --
        const int r = tid;
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        {
            // own latent Q row (256 columns) into TMEM as 16-bit pairs; rows past H are zero
            const int h = hb * kHeads + r;
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const T *>(prm.q) +
                                                               ((int64_t)qi * prm.heads + h) * kR + own_col);
            // two rounds of 16 loads in flight (the row is 32 x 16 bytes)
#pragma unroll 1
            for (int c = 0; c < 128; c += 64) {
                uint32_t w[4][16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint4 v = h < prm.heads ? src[c / 4 + i] : make_uint4(0, 0, 0, 0);
                    w[i / 4][4 * (i % 4)] = v.x; w[i / 4][4 * (i % 4) + 1] = v.y;
                    w[i / 4][4 * (i % 4) + 2] = v.z; w[i / 4][4 * (i % 4) + 3] = v.w;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) tmem_st16(tmem_q + lane_off + c + 16 * k, w[k]);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&s.q_ready);
        }
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        float cur[kN];
        for (int kt = 0; ok && kt < n_kt; ++kt) {
            const int pb = kt & 1;         // S / P buffer and ring slot
            const int64_t kbase = jb + (int64_t)kt * kN;
            const int valid = (int)((j1 - kbase) < kN ? (j1 - kbase) : kN);
            const int first = (int)(j0 > kbase ? j0 - kbase : 0);      // keys below j0 (first tile only)
            ok = __all_sync(0xffffffffu, mbar_wait(&s.s_full[pb], (kt / 2) & 1));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kN; c += 32) tmem_ld32f(tmem_s(pb) + lane_off + c, cur + c);
            tmem_wait_ld();
            // online softmax; keys outside the visible range score -inf
            if (valid < kN || first > 0) {
#pragma unroll
                for (int c = 0; c < kN; ++c)
                    if (c >= valid || c < first) cur[c] = -INFINITY;
            }
            float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
            for (int c = 0; c < kN; c += 4) {
                ma = fmax3(ma, cur[c], cur[c + 1]);
                mb = fmax3(mb, cur[c + 2], cur[c + 3]);
            }
            const float mt = fmaxf(ma, mb) * prm.scale_log2;   // the scale is positive
            float alpha = 1.f;
            if (mt > m_ref + kSlack) {
                alpha = exp2f(m_ref - mt);
                m_ref = mt;
            }
            // rescaling O needs the previous P.V finished (rare: the row max moved by > 2^8)
            if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                ok = __all_sync(0xffffffffu, mbar_wait(&s.o_done[(kt - 1) & 1], ((kt - 1) / 2) & 1));
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 256; c += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem_o + lane_off + c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                    tmem_st16(tmem_o + lane_off + c, v);
                }
                tmem_wait_st();
            }
            // P = exp2(s * scale - m_ref) as 16-bit pairs over this row's S columns
            // (already read); every tile has a visible key, so m_ref is finite here
            const float2 sc2 = make_float2(prm.scale_log2, prm.scale_log2);
            const float2 nm2 = make_float2(-m_ref, -m_ref);
            const float2 *cur2 = reinterpret_cast<const float2 *>(cur);
            float2 ls2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kN; c += 32) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 x = ffma2(cur2[c / 2 + i], sc2, nm2);
                    const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                    ls2 = fadd2(ls2, pp);
                    pk[i] = pack2<T>(pp.x, pp.y);
                }
                tmem_st16(tmem_s(pb) + lane_off + c / 2, pk);
            }
            tmem_wait_st();
            l = l * alpha + (ls2.x + ls2.y);
            // latent rows past the visible range must not reach P.V (tail slots may hold NaN)
            if (valid < kN) {
                ok = __all_sync(0xffffffffu, mbar_wait(&s.v_full[pb], (kt / 2) & 1));
                if (!ok) break;
                if (r < kN && r >= valid) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk)
#pragma unroll
                        for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4 *>(s.v[pb][blk] + r * 128 + i * 16) = z;
                }
                fence_proxy_async_smem();  // the zeroed rows before the tensor core reads them
            }
            tc_fence_before();
            mbar_arrive(&s.p_ready[pb]);
        }
        if (ok && n_kt > 0)
            ok = __all_sync(0xffffffffu, mbar_wait(&s.o_done[(n_kt - 1) & 1], ((n_kt - 1) / 2) & 1));
        if (!ok) {
            atomicCAS(prm.status, 0, PA_DEVICE_TIMEOUT_SOFTMAX);
        } else if (n_kt == 0) {
            // empty split (only with splits > 1): zero partial, lse = -inf; O was never written
            const int h = hb * kHeads + r;
            if (h < prm.heads && prm.splits > 1) {
                const int64_t rows = (int64_t)prm.plan.queries * prm.heads;
                const int64_t orow = (int64_t)qi * prm.heads + h;
                float *dst = prm.ws_o + ((int64_t)split * rows + orow) * kR + own_col;
                for (int c = 0; c < 256; c += 4) *reinterpret_cast<float4 *>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                if (rank == 0) prm.ws_lse[(int64_t)split * rows + orow] = -INFINITY;
            }
        } else {
            tc_fence_after();
            const int h = hb * kHeads + r;
            const bool row_ok = h < prm.heads;
            const int64_t rows = (int64_t)prm.plan.queries * prm.heads;
            const int64_t orow = (int64_t)qi * prm.heads + h;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            // 64 columns per TMEM round trip; the 16-byte chunks are transposed across
            // each group of 8 lanes so that a warp's store writes whole 128-byte lines
            const int jj = lane & 7, g = lane & ~7;
#pragma unroll 1
            for (int c0 = 0; c0 < 256; c0 += 64) {
                uint32_t vv[64];
                tmem_ld32(tmem_o + lane_off + c0, vv);
                tmem_ld32(tmem_o + lane_off + c0 + 32, vv + 32);
                tmem_wait_ld();
                if (prm.splits == 1) {
                    uint32_t ch[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        ch[e] = pack2<T>(__uint_as_float(vv[2 * e]) * inv, __uint_as_float(vv[2 * e + 1]) * inv);
                    transpose_chunks8(ch, lane);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int hr = hb * kHeads + 32 * warp + g + c;      // the head this round stores
                        if (hr < prm.heads) {
                            T *dst = static_cast<T *>(prm.out) + ((int64_t)qi * prm.heads + hr) * kR + own_col + c0 + 8 * jj;
                            *reinterpret_cast<uint4 *>(dst) = make_uint4(ch[4 * c], ch[4 * c + 1], ch[4 * c + 2], ch[4 * c + 3]);
                        }
                    }
                } else {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t ch[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) ch[e] = __float_as_uint(__uint_as_float(vv[32 * hf + e]) * inv);
                        transpose_chunks8(ch, lane);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const int hr = hb * kHeads + 32 * warp + g + c;
                            if (hr < prm.heads) {
                                float *dst = prm.ws_o + ((int64_t)split * rows + (int64_t)qi * prm.heads + hr) * kR + own_col +
                                             c0 + 32 * hf + 4 * jj;
                                *reinterpret_cast<uint4 *>(dst) = make_uint4(ch[4 * c], ch[4 * c + 1], ch[4 * c + 2], ch[4 * c + 3]);
                            }
                        }
                    }
                }
            }
            if (prm.splits > 1 && rank == 0 && row_ok)
                prm.ws_lse[(int64_t)split * rows + orow] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
        }
    }
    griddep_launch();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int log2_exact(int v) {
    if (v <= 0 || (v & (v - 1))) return -1;
    int s = 0;
    while ((1 << s) < v) ++s;
    return s;
}

}  // namespace

bool mla_supported(const AttnArgs &a) {
    const int ps = a.plan.page_size;
    return (a.dtype == PA_BF16 || a.dtype == PA_F16) && a.p == kP && a.d == kR && a.dv == kR && a.hkv == 1 &&
           (a.hq <= kHeads || a.hq % kHeads == 0) && log2_exact(ps) >= 3 && aligned16(a.q) && aligned16(a.qp) &&
           aligned16(a.k) && aligned16(a.kp) && aligned16(a.out) && tma_available();
}

cudaError_t launch_mla(const AttnArgs &a, bool use_list, cudaStream_t st) {
    const int items = use_list ? a.plan.n_decode : a.plan.queries;
    if (items == 0) return cudaSuccess;
    const bool bf16 = a.dtype == PA_BF16;
    const int ps = a.plan.page_size;
    MlaParams prm{};
    prm.plan = a.plan;
    prm.q = a.q;
    prm.out = a.out;
    prm.ws_o = a.ws_o;
    prm.ws_lse = a.ws_lse;
    prm.status = a.status;
    prm.heads = a.hq;
    prm.head_blocks = (a.hq + kHeads - 1) / kHeads;
    prm.use_list = use_list ? 1 : 0;
    prm.splits = a.splits;
    prm.box_rows = ps < kN ? ps : kN;
    prm.ps_shift = log2_exact(ps);
    prm.scale_log2 = a.scale * kLog2e;
    prm.causal = a.causal;
    prm.window = a.window;
    prm.bf16 = bf16 ? 1 : 0;
    const uint64_t rows = (uint64_t)a.plan.pages * ps;
    CUtensorMap tq, tqp, tlat, tkp;
    // Q [queries, H, 512] and QP [queries, H, 64]: boxes of 64 columns x 128 heads x 1 query
    // (heads past H read as zero fill)
    if (!encode_map_3d(&tq, a.q, bf16, kR, a.hq, a.plan.queries, (uint64_t)kR * 2, (uint64_t)kR * 2 * a.hq, 64,
                       kHeads, 1, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_3d(&tqp, a.qp, bf16, kP, a.hq, a.plan.queries, (uint64_t)kP * 2, (uint64_t)kP * 2 * a.hq, 64,
                       kHeads, 1, CU_TENSOR_MAP_SWIZZLE_128B) ||
        // latent [rows, 512] and position cache [rows, 64]: boxes of 64 columns x box_rows keys
        !encode_map_2d(&tlat, a.k, bf16, kR, rows, (uint64_t)kR * 2, 64, prm.box_rows,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_2d(&tkp, a.kp, bf16, kP, rows, (uint64_t)kP * 2, 64, prm.box_rows,
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(2 * items * prm.head_blocks * a.splits));
    cudaError_t e;
    if (bf16) {
        static bool cfg = false;
        if (!cfg) {
            e = cudaFuncSetAttribute(mla_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
            if (e != cudaSuccess) return e;
            cfg = true;
        }
        e = launch_pdl(mla_kernel<__nv_bfloat16>, grid, dim3(kThreads), kSmemBytes, st, tq, tqp, tlat, tkp, prm);
        if (e != cudaSuccess) return e;
    } else {
        static bool cfg = false;
        if (!cfg) {
            e = cudaFuncSetAttribute(mla_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
            if (e != cudaSuccess) return e;
            cfg = true;
        }
        e = launch_pdl(mla_kernel<__half>, grid, dim3(kThreads), kSmemBytes, st, tq, tqp, tlat, tkp, prm);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace pa
