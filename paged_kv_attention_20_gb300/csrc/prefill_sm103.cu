// Chunked causal prefill on tcgen05 tensor cores.
//
// ruDNN 0.1.7, src/paged_attention/mod.rs: module doc ("packed decode and
// chunked prefill") and `DevicePlan::attention` (causal at the plan's
// absolute positions, prefill chunks included).  A chunk is a run of
// consecutive positions of one sequence; query i of a chunk at position p_i
// sees keys 0..p_i: the cached context plus the chunk's earlier rows.
//
// Work unit: (tile of up to 128 consecutive queries, split, query head).  The
// kernel is persistent: one CTA per SM, walking
// the units (heaviest first) in serpentine rounds, so the K/V rings stream on from
// one unit into the next, Q of the next unit loads while the last tiles of
// the current one finish, and a CTA's start-up and teardown are paid once
// (as one CTA per unit, they cost ~4 µs of every 17-tile unit).  Per unit:
//   warps 0-7  softmax / O correction / epilogue: query row r (TMEM lane r) is
//              shared by warps r/32 and r/32+4, each taking 64 of the 128 key
//              (and output) columns; row maxima and sums cross over shared memory;
//   warps 8/10 TMA producers: Q of each unit and K tiles (warp 8, which also works
//              out each unit's parameters and leaves them in shared memory for
//              the other roles), V tiles (warp 10)
//              of 128 keys gathered page by page through the block table
//              (one box per page and 64-column half, 128-byte swizzle), each
//              through its own ring, so K is released once S is computed; the
//              block-table load of a tile's pages is issued one tile ahead;
//   warps 9/11 MMA issuers: warp 9 issues S = Q K^T into one of three TMEM
//              buffers, warp 11 issues O += P V with P read from tensor memory
//              (the softmax warps overwrite their row of the S buffer with P as
//              16-bit pairs); two issuers, because the tensor core takes only a
//              few MMAs ahead and one thread blocked on S noticed P late.
// K and V tiles use 3-stage shared-memory rings; P never touches shared memory.
// Each CTA loads its own tiles, from this GPU's memory only (no thread-block
// cluster, no multicast); the query heads of one KV head read the same tiles,
// which L2 serves after the first of them.
// Key tiles past the last query's position are never loaded; the diagonal
// tiles are masked per row.  Keys at or past the sequence length never reach
// P.V: their scores are masked and their V rows are zeroed in shared memory
// (tail slots may hold anything, NaN included).  The online softmax keeps a
// per-row reference maximum that only moves when a tile's maximum exceeds it
// by more than 8 (log2 units), so O in TMEM is rarely rescaled.
// Every wait is bounded; a timeout sets the library's device status word and
// the CTA stops issuing work.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"
#include "sm103_tc.cuh"
#include "tma_host.h"

namespace pa {
namespace {

using namespace tc;

constexpr int kM = 128;          // queries per tile (TMEM lanes)
constexpr int kN = 128;          // keys per tile
constexpr int kD = 128;          // head dim (== value dim)
constexpr int kStages = 3;
constexpr int kThreads = 384;        // 8 softmax warps + K producer + S issuer + V producer + P.V issuer
constexpr uint32_t kHalfBytes = kM * 128;          // one 64-column half of a 128-row tile
constexpr uint32_t kTileBytes = 2 * kHalfBytes;    // 32 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSlack = 8.f;

struct Smem {
    // 1024-byte aligned operand tiles (128-byte swizzle atoms)
    uint8_t q[kTileBytes];
    uint8_t k[kStages][kTileBytes];
    uint8_t v[kStages][kTileBytes];
    uint64_t q_full;               // Q of the CTA's current unit landed (phase = unit parity)
    uint64_t q_empty;              // every S MMA of the unit done: the Q buffer may be refilled
    uint64_t o_free;               // the softmax warps have read O of the unit (all 256 threads)
    uint64_t k_full[kStages];      // K tile landed
    uint64_t k_empty[kStages];     // S of the tile done (K free)
    uint64_t v_full[kStages];
    uint64_t v_empty[kStages];     // P.V of the tile done (V free)
    uint64_t s_full[3];            // S of tile kt in TMEM buffer kt % 3
    uint64_t p_ready[3];           // P of tile kt in TMEM (all 256 softmax threads) -> p_ready[kt % 3].
                                   // One barrier per tile in flight: S runs two tiles ahead, so warps
                                   // can be up to two tiles apart and must not count toward another tile
    uint64_t o_done[3];            // P.V of tile kt done -> o_done[kt % 3]
    float xred[2][2 * kM];         // row-max / row-sum exchange between the two warps of a row,
                                   // slot n % 2 for exchange n
    uint64_t xa[2][4];             // per slot and lane quarter: both warps' values written
    int32_t up[4][12];             // parameters of unit i in slot i % 4, written by the K producer
    uint64_t up_full[4];           // slot written
    uint64_t up_empty[4];          // slot read by every other role (11 arrivals)
    uint32_t tmem_base;
};

// The operand tiles need 1024-byte alignment (128-byte swizzle atoms); the
// dynamic shared memory is declared with that alignment, so no slack is
// requested (the struct fills the 227 KB a block may have).  The kernel checks
// the alignment and refuses to run (PA_DEVICE_LAYOUT) if it ever differs.
constexpr size_t kSmemBytes = sizeof(Smem);
static_assert(kSmemBytes <= 232448, "prefill shared memory above the per-block limit");

struct PrefillParams {
    PlanView plan;
    void *out;
    float *ws_o, *ws_lse;   // split partials (splits > 1): [S, Q, Hq, 128] and [S, Q, Hq]
    int32_t *status;
    int hq, hkv;
    float scale_log2;
    int causal;
    int window;
    int splits;
    int bf16;
};

__device__ __forceinline__ void set_timeout(Smem &s, int32_t *status, int code) {
    atomicCAS(status, 0, code);
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
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, PrefillParams prm) {
    griddep_wait();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if ((smem_u32(smem_raw) & 1023u) != 0u) {
        if (threadIdx.x == 0) atomicCAS(prm.status, 0, PA_DEVICE_LAYOUT);
        return;
    }
    Smem &s = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Persistent: each CTA walks its share of the units, a unit being (query
    // tile, split, query head) in the order unit = (tile * splits + split) *
    // Hq + head; the plan orders tiles by decreasing key count, so the
    // heaviest units go first.  Every role walks the same units; ring stages,
    // S buffers and their barrier phases follow one tile counter that runs on
    // across units, so the K/V rings stream without a break from one unit into
    // the next.
    const int cta = (int)blockIdx.x;
    const int n_ctas = (int)gridDim.x;
    const int units = prm.plan.n_tiles * prm.splits * prm.hq;
    const int ps = prm.plan.page_size;
    struct Unit {
        int split, h, kvh, q0, nq, pos0, seq_len, kt0, n_kt;
        const int32_t *trow;
    };
    // Keys of a row of the unit's split: its visible range [lo, hi) (causal
    // end, sliding window) cut by the split partition.  Without a window (or
    // split) both ends grow with the row's position, so the tile's key range
    // runs from the first row's lower end to the last row's upper end: key
    // tiles kt0 .. kt0 + n_kt - 1.
    auto row_keys = [&](const Unit &u, int pos, int64_t &j0, int64_t &j1) {
        int64_t lo, hi;
        visible_range(pos, u.seq_len, prm.causal, prm.window, lo, hi);
        split_bounds(lo, hi, prm.splits, u.split, ps, j0, j1);
    };
    auto unit_at = [&](int ui) -> Unit {
        Unit u;
        const int b = ui;
        const int tile_idx = b / (prm.hq * prm.splits);
        u.split = (b / prm.hq) % prm.splits;
        u.h = b % prm.hq;
        u.kvh = u.h / (prm.hq / prm.hkv);
        const int4 tile = prm.plan.tiles[tile_idx];
        const int seq = tile.x;
        u.q0 = tile.y;
        u.nq = tile.z;
        u.pos0 = tile.w;
        u.seq_len = prm.plan.seq_lens[seq];
        u.trow = prm.plan.table + (int64_t)seq * prm.plan.width;
        int64_t first_j0, first_j1, last_j0, last_j1;
        row_keys(u, u.pos0, first_j0, first_j1);
        row_keys(u, u.pos0 + u.nq - 1, last_j0, last_j1);
        if (prm.window > 0 && prm.splits > 1) {
            // With a window the split base (lo rounded down to a page) moves
            // along the tile, and a shorter page-rounded chunk after a move can
            // start split s > 1 earlier than it did for the rows before.  Rows
            // sharing a base form runs in which both ends only grow, so the
            // extremes lie at the runs' first and last rows.
            first_j0 = INT64_MAX;
            last_j1 = 0;
            for (int r = 0; r < u.nq;) {
                int64_t lo, hi;
                visible_range(u.pos0 + r, u.seq_len, prm.causal, prm.window, lo, hi);
                // first row whose lower end reaches the next page
                const int64_t next = (lo / ps + 1) * ps + prm.window - 1 - u.pos0;
                const int r_end = (int)(next < u.nq ? next : u.nq) - 1;
                int64_t a0, a1, b0, b1;
                row_keys(u, u.pos0 + r, a0, a1);
                row_keys(u, u.pos0 + r_end, b0, b1);
                first_j0 = a0 < first_j0 ? a0 : first_j0;
                last_j1 = b1 > last_j1 ? b1 : last_j1;
                r = r_end + 1;
            }
            if (first_j0 > last_j1) first_j0 = last_j1;
        }
        u.kt0 = (int)(first_j0 / kN);
        u.n_kt = last_j1 > first_j0 ? (int)((last_j1 + kN - 1) / kN) - u.kt0 : 0;
        return u;
    };

    // The CTA's i-th unit: round i of n_ctas-sized rounds, taken in serpentine
    // order (odd rounds from the last CTA down), so with units sorted by
    // decreasing size the CTAs' totals even out.  A CTA whose slot in the
    // last, partial round lies past the end has no i-th unit.
    auto unit_of = [&](int i) -> int {
        const int slot = (i & 1) ? n_ctas - 1 - cta : cta;
        const int ui = i * n_ctas + slot;
        return ui < units ? ui : units;
    };

    // Unit parameters come from dependent loads of plan metadata (~700 cycles).
    // The K producer, which runs furthest ahead, computes them and leaves them
    // in shared memory; every other role reads them from there.
    auto publish_unit = [&](int i, const Unit &u) -> bool {
        const int sl = i & 3;
        if (i >= 4 && !mbar_wait(&s.up_empty[sl], ((i >> 2) - 1) & 1)) return false;
        int32_t *p = s.up[sl];
        p[0] = u.split; p[1] = u.h; p[2] = u.kvh; p[3] = u.q0; p[4] = u.nq;
        p[5] = u.pos0; p[6] = u.seq_len; p[7] = u.kt0; p[8] = u.n_kt;
        const uint64_t t = reinterpret_cast<uint64_t>(u.trow);
        p[9] = (int32_t)(uint32_t)t;
        p[10] = (int32_t)(uint32_t)(t >> 32);
        mbar_arrive(&s.up_full[sl]);
        return true;
    };
    // every lane of the calling warp (or the one calling lane) waits and reads;
    // `one` arrives for the warp once all its lanes have read
    auto read_unit = [&](int i, Unit &u, bool whole_warp) -> bool {
        const int sl = i & 3;
        bool ok = mbar_wait(&s.up_full[sl], (i >> 2) & 1);
        if (whole_warp) ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        const int32_t *p = s.up[sl];
        u.split = p[0]; u.h = p[1]; u.kvh = p[2]; u.q0 = p[3]; u.nq = p[4];
        u.pos0 = p[5]; u.seq_len = p[6]; u.kt0 = p[7]; u.n_kt = p[8];
        u.trow = reinterpret_cast<const int32_t *>((uint64_t)(uint32_t)p[9] | ((uint64_t)(uint32_t)p[10] << 32));
        if (whole_warp) __syncwarp();
        if (!whole_warp || lane == 0) mbar_arrive(&s.up_empty[sl]);
        return true;
    };

    if (tid == 0) {
        mbar_init(&s.q_full, 1);
        mbar_init(&s.q_empty, 1);
        mbar_init(&s.o_free, 2 * kM);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.k_full[i], 1);
            mbar_init(&s.k_empty[i], 1);
            mbar_init(&s.v_full[i], 1);
            mbar_init(&s.v_empty[i], 1);
        }
        for (int i = 0; i < 3; ++i) mbar_init(&s.s_full[i], 1);
        for (int i = 0; i < 3; ++i) mbar_init(&s.p_ready[i], 2 * kM);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&s.xa[0][i], 64);
            mbar_init(&s.xa[1][i], 64);
        }
        for (int i = 0; i < 3; ++i) mbar_init(&s.o_done[i], 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&s.up_full[i], 1);
            mbar_init(&s.up_empty[i], 11);      // V producer, two MMA issuers, eight softmax warps
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
    auto tmem_s = [tmem](int b) -> uint32_t { return tmem + 128u * (uint32_t)b; };   // S / P buffers 0..2
    const uint32_t tmem_o = tmem + 384;

    if (warp == 8 || warp == 10) {
        // ------------------------------------------------- TMA producers --
        // Warp 8 streams K (and Q of each unit), warp 10 streams V, each through
        // its own 3-stage ring: a K stage is free as soon as S of its tile is
        // computed, a V stage only after P.V, so K runs ahead of V.  Lane 0 owns
        // the barriers; lanes 0..pages_per_tile-1 each gather one page (two
        // 64-column boxes).  Q of the next unit is loaded
        // once every S MMA of the previous unit has completed.
        const bool is_k = warp == 8;
        const int pages_per_tile = kN / ps;
        const CUtensorMap *tm = is_k ? &tm_k : &tm_v;
        uint64_t *full = is_k ? s.k_full : s.v_full;
        uint64_t *empty = is_k ? s.k_empty : s.v_empty;
        if (lane == 0) {
            tma_prefetch_desc(tm);
            if (is_k) tma_prefetch_desc(&tm_q);
        }
        const int oob_row = prm.plan.pages * ps;          // rows >= this read as zeros
        int gt = 0;                                        // tiles streamed so far (all units)
        bool go = true;
        for (int i = 0; go && unit_of(i) < units; ++i) {
            Unit u;
            if (is_k) {
                u = unit_at(unit_of(i));
                if (lane == 0 && !publish_unit(i, u)) {
                    set_timeout(s, prm.status, PA_DEVICE_TIMEOUT_TMA);
                    go = false;
                }
                go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
                if (!go) break;
            } else if (!read_unit(i, u, true)) {
                set_timeout(s, prm.status, PA_DEVICE_TIMEOUT_TMA);
                break;
            }
            if (is_k && lane == 0) {
                if (i > 0 && !mbar_wait(&s.q_empty, (i - 1) & 1)) {
                    set_timeout(s, prm.status, PA_DEVICE_TIMEOUT_TMA);
                    go = false;
                } else {
                    mbar_arrive_expect_tx(&s.q_full, kTileBytes);
                    tma_load_3d(s.q, &tm_q, 0, u.h, u.q0, &s.q_full);
                    tma_load_3d(s.q + kHalfBytes, &tm_q, 64, u.h, u.q0, &s.q_full);
                }
            }
            go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
            const int used_pages = (u.seq_len + ps - 1) / ps;
            // this lane's page of key tile kt; the block-table load of the next
            // tile is issued before the wait for a free stage, so its latency is
            // off the refill's critical path
            auto page_row = [&](int kt) -> int {
                const int lp = (u.kt0 + kt) * pages_per_tile + lane;
                return lp < used_pages ? u.trow[lp] * ps : oob_row;
            };
            int row_next = lane < pages_per_tile && u.n_kt > 0 ? page_row(0) : 0;
            for (int kt = 0; go && kt < u.n_kt; ++kt, ++gt) {
                const int row = row_next;
                if (lane < pages_per_tile && kt + 1 < u.n_kt) row_next = page_row(kt + 1);
                const int st = gt % kStages;
                uint8_t *ring = is_k ? s.k[st] : s.v[st];
                if (lane == 0) {
                    if (gt >= kStages && !mbar_wait(&empty[st], ((gt / kStages) - 1) & 1)) {
                        set_timeout(s, prm.status, PA_DEVICE_TIMEOUT_TMA);
                        go = false;
                    } else {
                        mbar_arrive_expect_tx(&full[st], kTileBytes);
                    }
                }
                go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
                if (!go) break;
                if (lane < pages_per_tile) {
                    const uint32_t off = (uint32_t)lane * ps * 128;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        tma_load_3d(ring + j * kHalfBytes + off, tm, j * 64, u.kvh, row, &full[st]);
                    }
                }
            }
        }
        // Do not leave while a load of this warp may still be landing (only a
        // timeout elsewhere can leave one unconsumed): wait, briefly, for the
        // last tiles issued.
        if (lane == 0) {
            for (int t = gt - kStages > 0 ? gt - kStages : 0; t < gt; ++t)
                mbar_wait(&full[t % kStages], (t / kStages) & 1, 2000000ll);
        }
    } else if (warp == 9 || warp == 11) {
        // ------------------------------------------------------ MMA issuers --
        // Two issuing threads: warp 9 issues S = Q K^T (three TMEM buffers, so
        // S runs up to two tiles ahead of P.V, into the next unit as well), warp
        // 11 issues O += P V as soon as P of a tile is in TMEM.  The tensor core
        // accepts only a few MMAs ahead, so a single issuer spends most of a tile
        // blocked on one kind and notices the other late.  The two touch
        // different TMEM (S buffers vs O) and shared memory (K vs V), and each
        // commits its own MMAs.  P.V of a unit's first tile overwrites O, so it
        // waits until the softmax warps have read O of the previous unit.
        if (lane == 0) {
            bool ok = true;
            int gt = 0;
            if (warp == 9) {
                const uint32_t idesc_s = idesc_f16(kM, kN, prm.bf16 != 0, false, false);
                const uint64_t q_desc = smem_desc(smem_u32(s.q), 16, 1024, kLayoutSwizzle128B);
                for (int i = 0; ok && unit_of(i) < units; ++i) {
                    Unit u;
                    if (!read_unit(i, u, false)) { ok = false; break; }
                    if (!mbar_wait(&s.q_full, i & 1)) { ok = false; break; }
                    for (int kt = 0; kt < u.n_kt; ++kt, ++gt) {
                        const int st = gt % kStages, sb = gt % 3;
                        if (!mbar_wait(&s.k_full[st], (gt / kStages) & 1)) { ok = false; break; }
                        // the buffer's previous tile (gt-3) must be through its P.V (P lives in it)
                        if (gt >= 3 && !mbar_wait(&s.o_done[sb], ((gt / 3) - 1) & 1)) { ok = false; break; }
                        tc_fence_after();
                        // stage descriptors; a K-step adds its byte offset / 16 to the
                        // start-address field (shared addresses are below 256 KB, so
                        // the field never carries)
                        const uint64_t k_desc = smem_desc(smem_u32(s.k[st]), 16, 1024, kLayoutSwizzle128B);
                        const uint32_t d_s = tmem_s(sb);
#pragma unroll
                        for (int ks = 0; ks < kD / 16; ++ks) {
                            const uint64_t o = (uint64_t)(((ks / 4) * kHalfBytes + (ks % 4) * 32) >> 4);
                            mma_f16_ss(d_s, q_desc + o, k_desc + o, idesc_s, ks > 0 ? 1u : 0u);
                        }
                        mma_commit(&s.s_full[sb]);
                        mma_commit(&s.k_empty[st]);
                    }
                    if (!ok) break;
                    mma_commit(&s.q_empty);        // Q is free once this unit's S MMAs are done
                }
            } else {
                const uint32_t idesc_o = idesc_f16(kM, kD, prm.bf16 != 0, false, true);
                for (int i = 0; ok && unit_of(i) < units; ++i) {
                    Unit u;
                    if (!read_unit(i, u, false)) { ok = false; break; }
                    if (i > 0 && !mbar_wait(&s.o_free, (i - 1) & 1)) { ok = false; break; }
                    for (int kt = 0; kt < u.n_kt; ++kt, ++gt) {
                        const int st = gt % kStages;
                        if (!mbar_wait(&s.p_ready[gt % 3], (gt / 3) & 1)) { ok = false; break; }
                        if (!mbar_wait(&s.v_full[st], (gt / kStages) & 1)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t v_desc = smem_desc(smem_u32(s.v[st]), kHalfBytes, 1024, kLayoutSwizzle128B);
                        const uint32_t p_tmem = tmem_s(gt % 3);          // P (16-bit pairs) over the S columns
#pragma unroll
                        for (int ks = 0; ks < kN / 16; ++ks)
                            mma_f16_ts(tmem_o, p_tmem + ks * 8, v_desc + (uint64_t)((ks * 2048) >> 4), idesc_o,
                                       (kt > 0 || ks > 0) ? 1u : 0u);
                        mma_commit(&s.o_done[gt % 3]);
                        mma_commit(&s.v_empty[st]);
                    }
                }
            }
            if (!ok) set_timeout(s, prm.status, PA_DEVICE_TIMEOUT_MMA);
        }
    } else {
        // ---------------------------------------- softmax / correction rows --
        // Warps w and w+4 share TMEM lanes 32*(w%4).. (query rows); warp w takes
        // key/value columns 0..63 of its rows and warp w+4 columns 64..127.
        const int q4 = warp & 3, h2 = warp >> 2;
        const int r = 32 * q4 + lane;            // query row == TMEM lane
        const int col0 = 64 * h2;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        bool ok = true;
        int xphase = 0;
        int gt = 0;                                // tiles consumed so far (all units)
        // value of the other warp of this row (bounded waits; false on timeout)
        // One barrier round per exchange: slot n % 2 is written again at exchange
        // n + 2 only after the partner arrived for exchange n + 1, which it does
        // after reading exchange n.
        auto exchange = [&](float v, float &other) -> bool {
            const int slot = xphase & 1;
            s.xred[slot][h2 * kM + r] = v;
            mbar_arrive(&s.xa[slot][q4]);
            if (!__all_sync(0xffffffffu, mbar_wait(&s.xa[slot][q4], (xphase >> 1) & 1))) return false;
            other = s.xred[slot][(1 - h2) * kM + r];
            ++xphase;
            return true;
        };
        // a unit's parameters come from the K producer through shared memory; the
        // next unit's are read before this unit's epilogue
        Unit u{};
        if (unit_of(0) < units) ok = read_unit(0, u, true);
        if (!ok) set_timeout(s, prm.status, PA_DEVICE_TIMEOUT_SOFTMAX);
        for (int i = 0; ok && unit_of(i) < units; ++i) {
            int64_t row_j0 = 0, row_j1 = 0;           // this row's keys in this split: [vis_lo, vis_end)
            if (r < u.nq) row_keys(u, u.pos0 + r, row_j0, row_j1);   // rows past the tile's queries see nothing
            const int vis_lo = (int)row_j0, vis_end = (int)row_j1;
            float m_ref = -INFINITY, l = 0.f;
            for (int kt = 0; kt < u.n_kt && ok; ++kt, ++gt) {
                const int sb = gt % 3;
                ok = __all_sync(0xffffffffu, mbar_wait(&s.s_full[sb], (gt / 3) & 1));
                if (!ok) break;
                tc_fence_after();
                const int kbase = (u.kt0 + kt) * kN + col0;
                // my 64 scores of the row into registers (two loads, one wait)
                uint32_t sv[64];
                tmem_ld32(tmem_s(sb) + lane_off + col0, sv);
                tmem_ld32(tmem_s(sb) + lane_off + col0 + 32, sv + 32);
                tmem_wait_ld();
                // keys outside the row's visible range score -inf (diagonal, sequence-end
                // and window-edge tiles only)
                if (kbase + 64 > vis_end || kbase < vis_lo) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (kbase + c >= vis_end || kbase + c < vis_lo) sv[c] = 0xff800000u;
                }
                // row maximum of the raw scores (the scale is positive, so it commutes with max)
                float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    ma = fmax3(ma, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
                    mb = fmax3(mb, __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
                }
                const float mine = fmaxf(ma, mb) * prm.scale_log2;
                float other;
                ok = exchange(mine, other);
                if (!ok) break;
                const float mt = fmaxf(mine, other);
                float alpha = 1.f;
                if (mt > m_ref + kSlack) {
                    alpha = exp2f(m_ref - mt);
                    m_ref = mt;
                }
                // rescaling O needs the previous P.V finished (rare: the row max moved by > 2^8)
                if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&s.o_done[(gt - 1) % 3], ((gt - 1) / 3) & 1));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 64; c += 16) {
                        uint32_t v[16];
                        tmem_ld16(tmem_o + lane_off + col0 + c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                        tmem_st16(tmem_o + lane_off + col0 + c, v);
                    }
                    tmem_wait_st();
                }
                // P = exp2(s * scale - m_ref) as 16-bit pairs over my S columns (already in
                // registers); masked keys hold -inf and give 0.  A row whose window has
                // not started yet still has m_ref = -inf: its weights are all 0.
                const float2 sc2 = make_float2(prm.scale_log2, prm.scale_log2);
                const float mr = m_ref == -INFINITY ? 0.f : m_ref;
                const float2 nm2 = make_float2(-mr, -mr);
                float2 ls2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < 64; c += 32) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 x = ffma2(make_float2(__uint_as_float(sv[c + 2 * i]), __uint_as_float(sv[c + 2 * i + 1])),
                                               sc2, nm2);
                        const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                        ls2 = fadd2(ls2, pp);
                        pk[i] = pack2<T>(pp.x, pp.y);
                    }
                    tmem_st16(tmem_s(sb) + lane_off + (col0 + c) / 2, pk);
                }
                tmem_wait_st();
                l = l * alpha + (ls2.x + ls2.y);
                // V rows at or past the sequence end (tail slots) must not reach the MMA
                if ((u.kt0 + kt) * kN + kN > u.seq_len) {
                    const int st = gt % kStages;
                    ok = __all_sync(0xffffffffu, mbar_wait(&s.v_full[st], (gt / kStages) & 1));
                    if (!ok) break;
                    if ((u.kt0 + kt) * kN + r >= u.seq_len) {
                        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            *reinterpret_cast<uint4 *>(s.v[st] + h2 * kHalfBytes + r * 128 + i * 16) = z;
                    }
                    fence_proxy_async_smem();  // the zeroed V rows before the tensor core reads them
                }
                tc_fence_before();
                mbar_arrive(&s.p_ready[gt % 3]);
            }
            const bool more = unit_of(i + 1) < units;
            Unit nu = u;
            if (more && ok) ok = read_unit(i + 1, nu, true);
            if (ok && u.n_kt > 0)
                ok = __all_sync(0xffffffffu, mbar_wait(&s.o_done[(gt - 1) % 3], ((gt - 1) / 3) & 1));
            float l_other = 0.f;
            if (ok) ok = exchange(l, l_other);
            if (!ok) {
                set_timeout(s, prm.status, PA_DEVICE_TIMEOUT_SOFTMAX);
            } else {
                // every lane loads (warp-collective); only rows of real queries store.
                // A row with no key in this split (only with splits > 1) writes a zero
                // partial and lse = -inf; O was not written for it.
                tc_fence_after();
                const float lsum = l + l_other;
                const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                const int64_t orow = (int64_t)(u.q0 + r) * prm.hq + u.h;
                const int jj = lane & 7, g = lane & ~7;   // lane in its group of 8, the group's first row
                if (prm.splits > 1) {
                    const int64_t rows = (int64_t)prm.plan.queries * prm.hq;
                    uint32_t vv[64];
                    if (u.n_kt > 0) {
                        tmem_ld32(tmem_o + lane_off + col0, vv);
                        tmem_ld32(tmem_o + lane_off + col0 + 32, vv + 32);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 64; ++e) vv[e] = 0u;
                    }
                    // fp32 partials: each half of the row's 64 columns is eight 16-byte chunks
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t ch[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            ch[e] = __float_as_uint(lsum > 0.f ? __uint_as_float(vv[32 * hf + e]) * inv : 0.f);
                        transpose_chunks8(ch, lane);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const int rr = 32 * q4 + g + c;
                            if (rr < u.nq) {
                                float *dst = prm.ws_o + ((int64_t)u.split * rows + (int64_t)(u.q0 + rr) * prm.hq + u.h) * kD +
                                             col0 + 32 * hf + 4 * jj;
                                *reinterpret_cast<uint4 *>(dst) = make_uint4(ch[4 * c], ch[4 * c + 1], ch[4 * c + 2], ch[4 * c + 3]);
                            }
                        }
                    }
                    if (r < u.nq && h2 == 0)
                        prm.ws_lse[(int64_t)u.split * rows + orow] =
                            lsum > 0.f ? (m_ref + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
                } else {
                uint32_t vv[64];
                tmem_ld32(tmem_o + lane_off + col0, vv);          // all 64 columns, one wait
                tmem_ld32(tmem_o + lane_off + col0 + 32, vv + 32);
                tmem_wait_ld();
                // the row's 64 output columns as eight 16-byte chunks of 16-bit pairs
                uint32_t ch[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    ch[e] = pack2<T>(__uint_as_float(vv[2 * e]) * inv, __uint_as_float(vv[2 * e + 1]) * inv);
                transpose_chunks8(ch, lane);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int rr = 32 * q4 + g + c;                // the row this round stores
                    if (rr < u.nq) {
                        T *dst = static_cast<T *>(prm.out) + ((int64_t)(u.q0 + rr) * prm.hq + u.h) * kD + col0 + 8 * jj;
                        *reinterpret_cast<uint4 *>(dst) = make_uint4(ch[4 * c], ch[4 * c + 1], ch[4 * c + 2], ch[4 * c + 3]);
                    }
                }
                }
                // O of this unit has been read: the next unit's first P.V may overwrite it
                tc_fence_before();
                mbar_arrive(&s.o_free);
            }
            u = nu;
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

// 3-D map over [rows, heads, 128] 16-bit elements; box = 64 columns x 1 head x box_rows rows.
bool make_map(CUtensorMap *m, const void *base, int heads, int64_t rows, int box_rows, bool bf16) {
    return encode_map_3d(m, base, bf16, kD, (uint64_t)heads, (uint64_t)rows, (uint64_t)kD * 2,
                         (uint64_t)kD * 2 * heads, 64, 1, (uint32_t)box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T>
cudaError_t launch_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &prm,
                     int units, int max_ctas, cudaStream_t st) {
    // Persistent grid: no more CTAs than can be resident at once (one per SM;
    // each walks its share of the units), so none waits for another to finish;
    // fewer when the caller keeps SMs free for a concurrent kernel.
    static int resident = 0;
    if (resident == 0) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        int per_sm = 0, dev = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prefill_kernel<T>, kThreads, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        resident = per_sm * sms > 0 ? per_sm * sms : 1;
    }
    int ctas = units < resident ? units : resident;
    if (max_ctas > 0 && max_ctas < ctas) ctas = max_ctas;
    const dim3 grid((unsigned)ctas);
    cudaError_t e = launch_pdl(prefill_kernel<T>, grid, dim3(kThreads), kSmemBytes, st, tq, tk, tv, prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool prefill_supported(const AttnArgs &a) {
    const int ps = a.plan.page_size;
    return (a.dtype == PA_BF16 || a.dtype == PA_F16) && a.p == 0 && a.d == kD && a.dv == kD &&
           (ps == 16 || ps == 32 || ps == 64 || ps == 128) && aligned16(a.q) && aligned16(a.k) &&
           aligned16(a.v) && aligned16(a.out) && a.plan.n_tiles > 0 && tma_available();
}

cudaError_t launch_prefill(const AttnArgs &a, cudaStream_t st) {
    const bool bf16 = a.dtype == PA_BF16;
    CUtensorMap tq, tk, tv;
    const int64_t cache_rows = (int64_t)a.plan.pages * a.plan.page_size;
    if (!make_map(&tq, a.q, a.hq, a.plan.queries, kM, bf16) ||
        !make_map(&tk, a.k, a.hkv, cache_rows, a.plan.page_size, bf16) ||
        !make_map(&tv, a.v, a.hkv, cache_rows, a.plan.page_size, bf16))
        return cudaErrorInvalidValue;
    PrefillParams prm{};
    prm.plan = a.plan;
    prm.out = a.out;
    prm.ws_o = a.ws_o;
    prm.ws_lse = a.ws_lse;
    prm.splits = a.splits;
    prm.status = a.status;
    prm.hq = a.hq;
    prm.hkv = a.hkv;
    prm.scale_log2 = a.scale * kLog2e;
    prm.causal = a.causal;
    prm.window = a.window;
    prm.bf16 = bf16 ? 1 : 0;
    const int64_t units = (int64_t)a.plan.n_tiles * a.splits * a.hq;
    if (units > INT32_MAX) return cudaErrorInvalidValue;
    return bf16 ? launch_t<__nv_bfloat16>(tq, tk, tv, prm, (int)units, a.max_ctas, st)
                : launch_t<__half>(tq, tk, tv, prm, (int)units, a.max_ctas, st);
}

}  // namespace pa
