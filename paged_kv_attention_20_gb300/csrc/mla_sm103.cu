// MLA decode on tcgen05 tensor cores, one 2-CTA cluster per (query, 128 heads).
//
// ruDNN 0.1.7, src/paged_attention/mod.rs, doc of `DevicePlan::mla`: absorbed
// Q [queries, H, R] and position Q [queries, H, P] score against one shared
// latent head [pages, ps, 1, R] and a rotated position cache [pages, ps, 1, P];
// the latent is both key and value, so
//   s_j = scale * (q . c_j + qp . r_j),   out = sum_j softmax_j c_j   ([queries, H, R]).
// The scale comes from the model's original QK dims (caller supplied).
//
// The 128 x 512 fp32 output tile fills all of one SM's tensor memory, so the
// work is split over a CTA pair (thread-block cluster of 2):
//   CTA 0 contracts latent columns 0..255 plus the 64 position columns,
//   CTA 1 contracts latent columns 256..511;
// each writes its partial score tile to the peer through distributed shared
// memory, both add (a + b == b + a, so both get identical scores), run the
// same online softmax, and each accumulates its own 256-column half of O in
// TMEM with its own half of the latent tile as V.  Every latent byte is loaded
// once, by the CTA that owns its columns; the same 128-byte-swizzled tile is
// the K-major B operand of Q.K^T and the MN-major B operand of P.V.
//
// Roles per CTA: warps 0-3 softmax/epilogue (thread r = head r, TMEM lane r),
// warp 4 TMA producer (64-key tiles, 3 stages), warp 5 MMA issuer, warps 6-9
// senders: they read each partial score tile from TMEM and push it to the
// peer, so the SM-to-SM transfer (the slowest link: ~20 GB/s per SM each
// way) of tile kt+1 overlaps the softmax of tile kt; warp 10 releases the
// receive buffers to the peer.
// The CTA's 256 latent columns of Q live in TMEM (the A operand of Q.K^T is
// read from there), which leaves shared memory for three latent stages; the
// 64 position columns of Q stay in shared memory on CTA 0.  P (16-bit) is
// written back over its row of the S buffer in TMEM and read from there by
// the P.V MMA; two S/P buffers let S of the next tile be computed while the
// current tile's P waits for its P.V.  The peer's partial scores arrive by
// asynchronous remote stores that complete bytes on a local mbarrier, into a
// double-buffered, 16-byte-chunk-swizzled receive area.
// Key tiles are one page at page_size 64 (several boxes for smaller pages).
// Keys at or past the sequence end are masked and their latent rows zeroed
// before P.V.  All waits are bounded (timeout -> device status word).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
#include "sm103_tc.cuh"
#include "tma_host.h"

namespace pa {
namespace {

using namespace tc;

constexpr int kHeads = 128;               // M: heads per cluster (TMEM lanes)
constexpr int kR = 512;                   // latent rank
constexpr int kP = 64;                    // rotary position dims
constexpr int kN = 64;                    // keys per tile
constexpr int kStages = 3;
constexpr int kThreads = 352;              // 4 softmax + producer + MMA + 4 sender warps + releaser
constexpr int kBlk = kHeads * 128;        // one 64-column block of the Q tile (bytes)
constexpr int kKBlk = kN * 128;           // one 64-column block of a key tile (bytes)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSlack = 8.f;

struct Smem {
    uint8_t qp[kBlk];                    // rank 0: position Q block (the latent part of Q lives in TMEM)
    uint8_t kv[kStages][5][kKBlk];       // own latent blocks 0..3 (+ position block 4 on rank 0)
    float recv[2][kHeads * kN];          // peer's partial scores, double buffered, 16-byte chunks XOR-swizzled
    uint64_t q_full;                     // rank 0: position Q block landed
    uint64_t q_ready;                    // latent Q rows stored in TMEM by the row threads
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full[2];                  // S of tile kt in TMEM buffer kt % 2
    uint64_t s_sent[2];                  // the sender warps have read S of tile kt (P may overwrite it)
    uint64_t p_ready[2];                 // P of tile kt in TMEM (all 128 rows) -> p_ready[kt % 2].  One
                                         // barrier per tile in flight: softmax warps are not in step,
                                         // and a warp already on tile kt+1 must not count toward kt
    uint64_t o_done[2];                  // P.V of tile kt done -> o_done[kt % 2]
    uint64_t recv_full[2];               // local expect_tx + the peer's asynchronous stores (bytes)
    uint64_t can_send[2];                // arrived by the peer's releaser once the peer has read its recv[b]
    uint64_t recv_read[2];               // my 4 softmax warps have read recv[b] (local)
    uint32_t tmem_base;
    int32_t abort;
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct MlaParams {
    PlanView plan;
    const void *q;          // absorbed Q [queries, H, 512]
    void *out;
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

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t peer) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(local), "r"(peer));
    return r;
}

// Asynchronous store into the peer CTA's shared memory; its bytes complete a
// transaction on the peer's mbarrier (no fence on the sending side).
__device__ __forceinline__ void st_async_v4(uint32_t addr, float a, float b, float c, float d, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];\n" ::"r"(addr),
        "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
        : "memory");
}

__device__ __forceinline__ void arrive_remote(uint32_t remote_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(remote_bar) : "memory");
}

__device__ __forceinline__ bool try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool wait_cluster(uint64_t *bar, uint32_t parity, long long limit = 2000000000ll) {
    if (try_wait_cluster(bar, parity)) return true;
    const long long t0 = clock64();
    while (!try_wait_cluster(bar, parity))
        if (clock64() - t0 > limit) return false;
    return true;
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
    mla_kernel(const __grid_constant__ CUtensorMap tm_qp,
               const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_kp,
               MlaParams prm) {
    extern __shared__ uint8_t smem_raw[];
    Smem &s = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;

    // cluster -> (item, head block, split)
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
    // the first tile below j0 (only under a sliding window) are masked.
    const int64_t jb = j0 < j1 ? j0 / kN * kN : j0;
    const int n_kt = (int)((j1 - jb + kN - 1) / kN);
    const int32_t *trow = prm.plan.table + (int64_t)seq * prm.plan.width;

    if (tid == 0) {
        mbar_init(&s.q_full, 1);
        mbar_init(&s.q_ready, kHeads);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.kv_full[i], 1);
            mbar_init(&s.kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.s_full[i], 1);
            mbar_init(&s.s_sent[i], 4);
            mbar_init(&s.o_done[i], 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&s.p_ready[i], kHeads);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.recv_full[i], 1);
            mbar_init(&s.can_send[i], 1);
            mbar_init(&s.recv_read[i], 4);
        }
        s.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync();          // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    const uint32_t tmem_q = tmem;                                 // latent Q: 256 x 16-bit = 128 columns
    auto tmem_s = [tmem](int b) -> uint32_t { return tmem + 128u + 64u * (uint32_t)b; };   // S / P buffers 0, 1
    const uint32_t tmem_o = tmem + 256;

    if (warp == 4) {
        // ---------------------------------------------------- TMA producer --
        if (lane == 0) {
            tma_prefetch_desc(&tm_lat);
            if (rank == 0) {
                mbar_arrive_expect_tx(&s.q_full, kBlk);
                tma_load_3d(s.qp, &tm_qp, 0, hb * kHeads, qi, &s.q_full);
            }
            const int used_pages = (seq_len + ps - 1) >> prm.ps_shift;
            const int oob_row = prm.plan.pages * ps;
            for (int kt = 0; kt < n_kt; ++kt) {
                const int st = kt % kStages;
                if (kt >= kStages && !mbar_wait(&s.kv_empty[st], ((kt / kStages) - 1) & 1)) {
                    atomicExch(&s.abort, 1);
                    atomicCAS(prm.status, 0, PA_DEVICE_TIMEOUT_TMA);
                    break;
                }
                mbar_arrive_expect_tx(&s.kv_full[st], (uint32_t)(rank == 0 ? 5 : 4) * kKBlk);
                const int64_t jt = jb + (int64_t)kt * kN;
                for (int b = 0; b < kN; b += prm.box_rows) {
                    const int64_t j = jt + b;
                    const int64_t lp = j >> prm.ps_shift;
                    const int row = lp < used_pages ? trow[lp] * ps + (int)(j & (ps - 1)) : oob_row;
                    for (int blk = 0; blk < 4; ++blk)
                        tma_load_2d(s.kv[st][blk] + b * 128, &tm_lat, (int)(rank * 4 + blk) * 64, row,
                                    &s.kv_full[st]);
                    if (rank == 0) tma_load_2d(s.kv[st][4] + b * 128, &tm_kp, 0, row, &s.kv_full[st]);
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------ MMA issuer --
        if (lane == 0) {
            const uint32_t idesc_s = idesc_f16(kHeads, kN, prm.bf16 != 0, false, false);
            const uint32_t idesc_o = idesc_f16(kHeads, 256, prm.bf16 != 0, false, true);
            bool ok = (rank != 0 || mbar_wait(&s.q_full, 0)) && mbar_wait(&s.q_ready, 0);
            auto issue_pv = [&](int kt) -> bool {
                if (!mbar_wait(&s.p_ready[kt & 1], (kt / 2) & 1)) return false;
                tc_fence_after();
                const int st = kt % kStages;
                const uint32_t v_addr = smem_u32(s.kv[st][0]);
                const uint32_t p_tmem = tmem_s(kt & 1);           // P (16-bit pairs) over the S columns
                for (int ks = 0; ks < kN / 16; ++ks) {
                    const uint64_t b = smem_desc(v_addr + ks * 2048, kKBlk, 1024, kLayoutSwizzle128B);
                    mma_f16_ts(tmem_o, p_tmem + ks * 8, b, idesc_o, (kt > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(&s.o_done[kt & 1]);
                mma_commit(&s.kv_empty[st]);
                return true;
            };
            for (int kt = 0; ok && kt < n_kt; ++kt) {
                const int st = kt % kStages, sb = kt & 1;
                if (!mbar_wait(&s.kv_full[st], (kt / kStages) & 1)) { ok = false; break; }
                // the buffer's previous tile (kt-2) must be through its P.V (P lives in it)
                if (kt >= 2 && !mbar_wait(&s.o_done[sb], ((kt / 2) - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                for (int blk = 0; blk < 4; ++blk)            // latent columns: A from TMEM
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t b = smem_desc(smem_u32(s.kv[st][blk]) + k * 32, 16, 1024, kLayoutSwizzle128B);
                        mma_f16_ts(tmem_s(sb), tmem_q + blk * 32 + k * 8, b, idesc_s, (blk > 0 || k > 0) ? 1u : 0u);
                    }
                if (rank == 0)                                   // position columns: A from shared memory
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t a = smem_desc(smem_u32(s.qp) + k * 32, 16, 1024, kLayoutSwizzle128B);
                        const uint64_t b = smem_desc(smem_u32(s.kv[st][4]) + k * 32, 16, 1024, kLayoutSwizzle128B);
                        mma_f16_ss(tmem_s(sb), a, b, idesc_s, 1u);
                    }
                mma_commit(&s.s_full[sb]);
                if (kt > 0 && !issue_pv(kt - 1)) { ok = false; break; }
            }
            if (ok && n_kt > 0) ok = issue_pv(n_kt - 1);
            if (!ok) {
                atomicExch(&s.abort, 1);
                atomicCAS(prm.status, 0, PA_DEVICE_TIMEOUT_MMA);
            }
        }
    } else if (warp == 10) {
        // -------------------------------------------------------- releaser --
        // Tells the peer's senders that recv[b] may be overwritten.  The
        // softmax warps only arrive on a local barrier; the cluster-scope
        // release (ordered after their reads through this warp's acquire of
        // that barrier) is paid here, off the softmax path.
        bool ok = true;
        const uint32_t can_send_peer0 = peer_addr(smem_u32(&s.can_send[0]), peer);
        for (int kt = 0; ok && kt < n_kt; ++kt) {
            const int b = kt & 1;
            ok = mbar_wait(&s.recv_read[b], (kt / 2) & 1);
            if (ok && lane == 0) arrive_remote(can_send_peer0 + (uint32_t)b * 8u);
        }
        if (!ok) {
            atomicExch(&s.abort, 1);
            atomicCAS(prm.status, 0, PA_DEVICE_TIMEOUT_SOFTMAX);
        }
    } else if (warp >= 6) {
        // --------------------------------------------------------- senders --
        // Warp w reads TMEM lane quarter w % 4 (rows 32*(w%4)..): each partial
        // score tile goes to the peer's recv[kt & 1] by asynchronous remote
        // stores that complete bytes on the peer's recv_full barrier.
        const int q4 = warp & 3;
        const int r = 32 * q4 + lane;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const uint32_t recv_peer0 = peer_addr(smem_u32(&s.recv[0][r * kN]), peer);
        const uint32_t recv_full_peer0 = peer_addr(smem_u32(&s.recv_full[0]), peer);
        const int sw = r & 15;                   // chunk swizzle of row r
        bool ok = true;
        for (int kt = 0; ok && kt < n_kt; ++kt) {
            const int b = kt & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&s.s_full[b], (kt / 2) & 1));
            if (!ok) break;
            tc_fence_after();
            float sc[kN];
#pragma unroll
            for (int c = 0; c < kN; c += 32) tmem_ld32f(tmem_s(b) + lane_off + c, sc + c);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.s_sent[b]);
            // the peer has read what this buffer held two tiles ago
            if (kt >= 2) ok = __all_sync(0xffffffffu, wait_cluster(&s.can_send[b], ((kt / 2) - 1) & 1));
            if (!ok) break;
            const uint32_t dst = recv_peer0 + (uint32_t)b * (uint32_t)sizeof(s.recv[0]);
#pragma unroll
            for (int c = 0; c < kN / 4; ++c)
                st_async_v4(dst + ((c ^ sw) * 16), sc[4 * c], sc[4 * c + 1], sc[4 * c + 2], sc[4 * c + 3],
                            recv_full_peer0 + (uint32_t)b * 8u);
        }
        if (!ok) {
            atomicExch(&s.abort, 1);
            atomicCAS(prm.status, 0, PA_DEVICE_TIMEOUT_SOFTMAX);
        }
    } else {
        // ---------------------------------------- softmax / epilogue rows --
        // Per tile: own partial scores from TMEM plus the peer's from recv,
        // softmax, P into TMEM over the S columns (once the senders have read them).
        const int r = tid;
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        const int sw = r & 15;                   // chunk swizzle of row r
        {
            // latent Q row (this CTA's 256 columns) into TMEM as 16-bit pairs; rows past H are zero
            const int h = hb * kHeads + r;
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const T *>(prm.q) +
                                                               ((int64_t)qi * prm.heads + h) * kR + rank * 256);
#pragma unroll 1
            for (int c = 0; c < 128; c += 16) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = h < prm.heads ? src[c / 4 + i] : make_uint4(0, 0, 0, 0);
                    w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
                }
                tmem_st16(tmem_q + lane_off + c, w);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&s.q_ready);
        }
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        float cur[kN];
        for (int kt = 0; ok && kt < n_kt; ++kt) {
            const int sb = kt & 1;         // receive buffer
            const int pb = kt & 1;         // S / P buffer
            const int64_t kbase = jb + (int64_t)kt * kN;
            const int valid = (int)((j1 - kbase) < kN ? (j1 - kbase) : kN);
            const int first = (int)(j0 > kbase ? j0 - kbase : 0);      // keys below j0 (first tile only)
            if (r == 0) mbar_arrive_expect_tx(&s.recv_full[sb], kHeads * kN * 4);   // my receive of tile kt
            ok = __all_sync(0xffffffffu, mbar_wait(&s.s_full[pb], (kt / 2) & 1));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kN; c += 32) tmem_ld32f(tmem_s(pb) + lane_off + c, cur + c);
            tmem_wait_ld();
            ok = __all_sync(0xffffffffu, wait_cluster(&s.recv_full[sb], (kt / 2) & 1));
            if (!ok) break;
            const float *mine = &s.recv[sb][r * kN];
            float2 *cur2 = reinterpret_cast<float2 *>(cur);
#pragma unroll
            for (int c = 0; c < kN / 4; ++c) {
                const float4 o = *reinterpret_cast<const float4 *>(mine + ((c ^ sw) * 4));
                cur2[2 * c] = fadd2(cur2[2 * c], make_float2(o.x, o.y));
                cur2[2 * c + 1] = fadd2(cur2[2 * c + 1], make_float2(o.z, o.w));
            }
            // online softmax (identical on both CTAs); keys past the visible range score -inf
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
            // this warp's rows of recv[sb] are read (the releaser passes it on)
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.recv_read[sb]);
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
            // the senders must have read S before P overwrites it
            ok = __all_sync(0xffffffffu, mbar_wait(&s.s_sent[pb], (kt / 2) & 1));
            if (!ok) break;
            tc_fence_after();
            // P = exp2(s * scale - m_ref) as 16-bit pairs over this row's S columns
            // (already read); every tile has a visible key, so m_ref is finite here
            const float2 sc2 = make_float2(prm.scale_log2, prm.scale_log2);
            const float2 nm2 = make_float2(-m_ref, -m_ref);
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
                const int st = kt % kStages;
                ok = __all_sync(0xffffffffu, mbar_wait(&s.kv_full[st], (kt / kStages) & 1));
                if (!ok) break;
                if (r < kN && r >= valid) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk)
#pragma unroll
                        for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4 *>(s.kv[st][blk] + r * 128 + i * 16) = z;
                }
                fence_proxy_async_smem();  // the zeroed rows before the tensor core reads them
            }
            tc_fence_before();
            mbar_arrive(&s.p_ready[kt & 1]);
        }
        if (ok && n_kt > 0)
            ok = __all_sync(0xffffffffu, mbar_wait(&s.o_done[(n_kt - 1) & 1], ((n_kt - 1) / 2) & 1));
        if (!ok) {
            atomicExch(&s.abort, 1);
            atomicCAS(prm.status, 0, PA_DEVICE_TIMEOUT_SOFTMAX);
        } else if (n_kt == 0) {
            // empty split (only with splits > 1): zero partial, lse = -inf; O was never written
            const int h = hb * kHeads + r;
            if (h < prm.heads && prm.splits > 1) {
                const int64_t rows = (int64_t)prm.plan.queries * prm.heads;
                const int64_t orow = (int64_t)qi * prm.heads + h;
                float *dst = prm.ws_o + ((int64_t)split * rows + orow) * kR + (int)rank * 256;
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
#pragma unroll 1
            for (int c = 0; c < 256; c += 16) {
                uint32_t v[16];
                tmem_ld16(tmem_o + lane_off + c, v);
                tmem_wait_ld();
                if (!row_ok) continue;
                const int col = (int)rank * 256 + c;
                if (prm.splits == 1) {
                    uint4 w0, w1;
                    w0.x = pack2<T>(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv);
                    w0.y = pack2<T>(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv);
                    w0.z = pack2<T>(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv);
                    w0.w = pack2<T>(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv);
                    w1.x = pack2<T>(__uint_as_float(v[8]) * inv, __uint_as_float(v[9]) * inv);
                    w1.y = pack2<T>(__uint_as_float(v[10]) * inv, __uint_as_float(v[11]) * inv);
                    w1.z = pack2<T>(__uint_as_float(v[12]) * inv, __uint_as_float(v[13]) * inv);
                    w1.w = pack2<T>(__uint_as_float(v[14]) * inv, __uint_as_float(v[15]) * inv);
                    T *dst = static_cast<T *>(prm.out) + orow * kR + col;
                    reinterpret_cast<uint4 *>(dst)[0] = w0;
                    reinterpret_cast<uint4 *>(dst)[1] = w1;
                } else {
                    float *dst = prm.ws_o + ((int64_t)split * rows + orow) * kR + col;
#pragma unroll
                    for (int i = 0; i < 16; i += 4)
                        *reinterpret_cast<float4 *>(dst + i) =
                            make_float4(__uint_as_float(v[i]) * inv, __uint_as_float(v[i + 1]) * inv,
                                        __uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv);
                }
            }
            if (prm.splits > 1 && rank == 0 && row_ok)
                prm.ws_lse[(int64_t)split * rows + orow] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();          // the peer is done with my shared memory
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
    CUtensorMap tqp, tlat, tkp;
    // QP [queries, H, 64]: boxes of 64 columns x 128 heads x 1 query (latent Q is read by the row threads)
    if (!encode_map_3d(&tqp, a.qp, bf16, kP, a.hq, a.plan.queries, (uint64_t)kP * 2, (uint64_t)kP * 2 * a.hq, 64,
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
        mla_kernel<__nv_bfloat16><<<grid, kThreads, kSmemBytes, st>>>(tqp, tlat, tkp, prm);
    } else {
        static bool cfg = false;
        if (!cfg) {
            e = cudaFuncSetAttribute(mla_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
            if (e != cudaSuccess) return e;
            cfg = true;
        }
        mla_kernel<__half><<<grid, kThreads, kSmemBytes, st>>>(tqp, tlat, tkp, prm);
    }
    return cudaGetLastError();
}

}  // namespace pa
