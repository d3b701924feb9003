// Host side of the paged-attention library: schedule building and
// validation, argument checks, dispatch to the kernels, and the C ABI.
//
// Follows ruDNN 0.1.7, src/paged_attention/mod.rs: `HostPlan` /
// `DevicePlan::upload` (one small upload of u32 metadata, reusable while the
// schedule is unchanged), `check_tensor` / `bounded` and
// `execute_attention_into` (every check happens before any launch; zero
// queries is a successful no-op), `append_with_report` (`validate_writes`,
// then an elementwise append), and the split path (`attention_into_split`:
// attention over (item, head, split) then a merge when splits > 1).

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "pa_internal.h"

struct pa_plan {
    int32_t queries = 0, sequences = 0, width = 0, page_size = 0, pages = 0;
    int32_t n_decode = 0, n_tiles = 0, n_tile_queries = 0;
    int64_t max_seq_len = 0;          // longest sequence any decode item reads
    std::vector<int32_t> words;       // host copy of the device metadata
    size_t off_qmeta = 0, off_seqlen = 0, off_table = 0, off_decode = 0, off_tiles = 0, off_order = 0;
    const int32_t *dev = nullptr;     // caller's device copy (after upload)
    // visible keys of the prefill tiles' queries and of the decode items, without
    // a window, non-causal [0] and causal [1] (the mixed call's SM share needs them)
    double keys_tiles[2] = {0, 0}, keys_decode[2] = {0, 0};
};

namespace {

thread_local std::string g_error;
thread_local cudaEvent_t g_time_start = nullptr, g_time_stop = nullptr;  // pa_time_next_kernel

pa_status fail(pa_status st, const char *msg) {
    g_error = msg;
    return st;
}

pa_status fail_cuda(cudaError_t e, const char *what) {
    g_error = std::string(what) + ": " + cudaGetErrorString(e);
    return PA_ERR_CUDA;
}

size_t align_words(size_t n, size_t a) { return (n + a - 1) / a * a; }

bool valid_dtype(pa_dtype d) { return d == PA_F32 || d == PA_F16 || d == PA_BF16; }

int elem_bytes(pa_dtype d) { return d == PA_F32 ? 4 : 2; }

// A mixed call's decode items can run beside its prefill tiles: the tiles are
// bound by the tensor core and the softmax, the decode items by HBM, and one
// after the other they leave one of the two idle for the whole of the other.
// The decode kernel then runs on a second stream of the caller's thread (one
// per device, created on first use outside stream capture), forked from and
// joined back into the caller's stream with events, so the call stays one
// ordered step of that stream and can be captured into a graph.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    bool failed = false;
};

constexpr int kMaxSideDevices = 64;

SideStream *side_stream(cudaStream_t st) {
    thread_local SideStream side[kMaxSideDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDevices) return nullptr;
    SideStream &ss = side[dev];
    if (ss.stream) return &ss;
    if (ss.failed) return nullptr;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return nullptr;
    // kept for the life of the thread; on any failure the calls stay serial
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
        if (join) cudaEventDestroy(join);
        if (fork) cudaEventDestroy(fork);
        if (s) cudaStreamDestroy(s);
        (void)cudaGetLastError();
        ss.failed = true;
        return nullptr;
    }
    ss.stream = s;
    ss.fork = fork;
    ss.join = join;
    return &ss;
}

int device_sms() {
    static int sms[kMaxSideDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDevices) return 0;
    if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms[dev];
}

int decode_sms_beside_prefill(const pa_plan *plan, int hq, int hkv, int d, int dv, int causal, int window,
                              pa_dtype dtype, int sms);

// Visible keys summed over the prefill tiles' queries and over the decode items.
void visible_key_sums(const pa_plan *plan, int causal, int window, double &keys_tiles, double &keys_decode) {
    const int32_t *w = plan->words.data();
    auto visible = [&](int q) -> double {
        const int seq = w[plan->off_qmeta + 4 * (size_t)q], pos = w[plan->off_qmeta + 4 * (size_t)q + 1];
        int64_t lo, hi;
        pa::visible_range(pos, w[plan->off_seqlen + seq], causal, window, lo, hi);
        return (double)(hi > lo ? hi - lo : 0);
    };
    keys_tiles = keys_decode = 0;
    for (int t = 0; t < plan->n_tiles; ++t) {
        const int32_t *tile = w + plan->off_tiles + 4 * (size_t)t;
        for (int i = 0; i < tile[2]; ++i) keys_tiles += visible(tile[1] + i);
    }
    for (int i = 0; i < plan->n_decode; ++i) keys_decode += visible(w[plan->off_decode + i]);
}

pa::PlanView view_of(const pa_plan *p) {
    pa::PlanView v{};
    v.qmeta = reinterpret_cast<const int4 *>(p->dev + p->off_qmeta);
    v.seq_lens = p->dev + p->off_seqlen;
    v.table = p->dev + p->off_table;
    v.decode = p->dev + p->off_decode;
    v.tiles = reinterpret_cast<const int4 *>(p->dev + p->off_tiles);
    v.order = p->dev + p->off_order;
    v.queries = p->queries;
    v.sequences = p->sequences;
    v.width = p->width;
    v.page_size = p->page_size;
    v.pages = p->pages;
    v.n_decode = p->n_decode;
    v.n_tiles = p->n_tiles;
    return v;
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// True when `ptr` is device memory of the current device.  The kernels'
// tensor maps and loads address only this GPU's own memory, so host memory
// (pinned or not), managed memory and other GPUs' memory are refused.
bool on_current_device(const void *ptr, int dev) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice && at.device == dev;
}

// PA_OK when every non-null pointer of `ptrs` is device memory of the current
// device, else PA_ERR_ARG naming the operand.
pa_status operands_on_device(const void *const *ptrs, const char *const *names, int n, const char *call) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return fail(PA_ERR_CUDA, "no current CUDA device");
    }
    for (int i = 0; i < n; ++i) {
        if (ptrs[i] && !on_current_device(ptrs[i], dev)) {
            char msg[256];
            std::snprintf(msg, sizeof msg, "%s: %s is not device memory of the current device", call, names[i]);
            return fail(PA_ERR_ARG, msg);
        }
    }
    return PA_OK;
}


}  // namespace

pa_status pa_fail_with(pa_status status, const char *msg) { return fail(status, msg); }

extern "C" {

const char *pa_last_error(void) { return g_error.c_str(); }

const char *pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "PA_OK";
        case PA_ERR_ARG: return "PA_ERR_ARG";
        case PA_ERR_SHAPE: return "PA_ERR_SHAPE";
        case PA_ERR_DTYPE: return "PA_ERR_DTYPE";
        case PA_ERR_RANGE: return "PA_ERR_RANGE";
        case PA_ERR_WRITE_CONFLICT: return "PA_ERR_WRITE_CONFLICT";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_SPLITS: return "PA_ERR_SPLITS";
        case PA_ERR_LIMIT: return "PA_ERR_LIMIT";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_STATE: return "PA_ERR_STATE";
    }
    return "PA_UNKNOWN";
}

int32_t pa_abi_version(void) { return PA_ABI_VERSION; }

pa_status paged_attn_plan(const int32_t *seq_lens, int32_t num_seqs, const int32_t *block_table,
                          int32_t width, const int32_t *query_seq, const int32_t *query_pos,
                          int32_t num_queries, int32_t page_size, int32_t num_pages,
                          pa_plan **out_plan) {
    if (!out_plan) return fail(PA_ERR_ARG, "paged_attn_plan: out_plan is null");
    *out_plan = nullptr;
    if (num_seqs < 0 || width < 0 || num_queries < 0 || num_pages < 0)
        return fail(PA_ERR_ARG, "paged_attn_plan: negative count");
    if (page_size < 1) return fail(PA_ERR_ARG, "paged_attn_plan: page_size must be >= 1");
    if ((int64_t)num_pages * page_size > INT32_MAX)
        return fail(PA_ERR_RANGE, "paged_attn_plan: pages * page_size exceeds 32-bit slot indexing");
    if ((int64_t)num_seqs * width > INT32_MAX / 2)
        return fail(PA_ERR_RANGE, "paged_attn_plan: block table exceeds 32-bit indexing");
    if (num_seqs > 0 && !seq_lens) return fail(PA_ERR_ARG, "paged_attn_plan: seq_lens is null");
    if (num_seqs > 0 && width > 0 && !block_table)
        return fail(PA_ERR_ARG, "paged_attn_plan: block_table is null");
    if (num_queries > 0 && (!query_seq || !query_pos))
        return fail(PA_ERR_ARG, "paged_attn_plan: query arrays are null");

    // Sequences: length within the table, used table entries within the pool.
    for (int32_t s = 0; s < num_seqs; ++s) {
        int64_t n = seq_lens[s];
        if (n < 0) return fail(PA_ERR_RANGE, "paged_attn_plan: negative sequence length");
        if (n > (int64_t)width * page_size)
            return fail(PA_ERR_RANGE, "paged_attn_plan: sequence longer than its block-table row");
        int64_t used = (n + page_size - 1) / page_size;
        for (int64_t g = 0; g < used; ++g) {
            int32_t pg = block_table[(int64_t)s * width + g];
            if (pg < 0 || pg >= num_pages)
                return fail(PA_ERR_RANGE, "paged_attn_plan: block-table entry outside the page pool");
        }
    }
    // Queries: valid sequence, 0 <= pos < seq_len; distinct write slots.
    std::vector<int64_t> slots((size_t)num_queries);
    for (int32_t i = 0; i < num_queries; ++i) {
        int32_t s = query_seq[i], pos = query_pos[i];
        if (s < 0 || s >= num_seqs) return fail(PA_ERR_RANGE, "paged_attn_plan: query sequence out of range");
        if (pos < 0 || pos >= seq_lens[s])
            return fail(PA_ERR_RANGE, "paged_attn_plan: query position outside its sequence");
        int64_t pg = block_table[(int64_t)s * width + pos / page_size];
        slots[(size_t)i] = pg * page_size + pos % page_size;
    }
    {
        std::vector<int64_t> sorted = slots;
        std::sort(sorted.begin(), sorted.end());
        if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end())
            return fail(PA_ERR_WRITE_CONFLICT, "paged_attn_plan: two queries write the same cache slot");
    }

    pa_plan *p = new pa_plan();
    p->queries = num_queries;
    p->sequences = num_seqs;
    p->width = width;
    p->page_size = page_size;
    p->pages = num_pages;

    // Work lists: runs of consecutive positions of one sequence -> prefill
    // tiles of up to kPrefillTileM queries; all other queries -> decode items.
    std::vector<int32_t> decode;
    std::vector<int32_t> tiles;  // 4 words per tile
    int32_t i = 0;
    while (i < num_queries) {
        int32_t j = i + 1;
        while (j < num_queries && query_seq[j] == query_seq[i] && query_pos[j] == query_pos[j - 1] + 1) ++j;
        int32_t run = j - i;
        if (run >= pa::kPrefillMinRun) {
            for (int32_t b = i; b < j; b += pa::kPrefillTileM) {
                int32_t cnt = std::min(pa::kPrefillTileM, j - b);
                tiles.insert(tiles.end(), {query_seq[i], b, cnt, query_pos[b]});
                p->n_tile_queries += cnt;
            }
        } else {
            for (int32_t b = i; b < j; ++b) {
                decode.push_back(b);
                p->max_seq_len = std::max<int64_t>(p->max_seq_len, seq_lens[query_seq[b]]);
            }
        }
        i = j;
    }
    // Longest decode items first (visible keys of a causal query: pos + 1), so
    // the decode kernels' heaviest blocks start first.
    std::stable_sort(decode.begin(), decode.end(),
                     [&](int32_t a, int32_t b) { return query_pos[a] > query_pos[b]; });
    p->n_decode = (int32_t)decode.size();
    p->n_tiles = (int32_t)(tiles.size() / 4);
    {
        // Heaviest tiles first (most keys: largest last position), so the
        // tensor-core kernel's long CTAs start early and the tail is short.
        std::vector<int> order((size_t)p->n_tiles);
        for (int t = 0; t < p->n_tiles; ++t) order[(size_t)t] = t;
        auto last_pos = [&](int t) { return tiles[4 * (size_t)t + 3] + tiles[4 * (size_t)t + 2] - 1; };
        std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return last_pos(a) > last_pos(b); });
        std::vector<int32_t> sorted;
        sorted.reserve(tiles.size());
        for (int t : order) sorted.insert(sorted.end(), tiles.begin() + 4 * t, tiles.begin() + 4 * t + 4);
        tiles.swap(sorted);
    }

    // Word layout (int32 words; 16-byte aligned sections):
    //   [0..15]  header: magic, queries, sequences, width, page_size, pages,
    //            n_decode, n_tiles, and the five section offsets
    //   qmeta    queries x {seq, pos, slot, 0}
    //   seqlen   sequences
    //   table    sequences x width
    //   decode   n_decode query indices
    //   tiles    n_tiles x {seq, first query, count, first position}
    //   order    every query, longest visible history first
    size_t off = 16;
    p->off_qmeta = off;   off = align_words(off + 4 * (size_t)num_queries, 4);
    p->off_seqlen = off;  off = align_words(off + (size_t)num_seqs, 4);
    p->off_table = off;   off = align_words(off + (size_t)num_seqs * width, 4);
    p->off_decode = off;  off = align_words(off + decode.size(), 4);
    p->off_tiles = off;   off = align_words(off + tiles.size(), 4);
    p->off_order = off;   off = align_words(off + (size_t)num_queries, 4);
    p->words.assign(off, 0);
    int32_t *w = p->words.data();
    w[0] = 0x50414731;  // "PAG1"
    w[1] = num_queries; w[2] = num_seqs; w[3] = width; w[4] = page_size; w[5] = num_pages;
    w[6] = p->n_decode; w[7] = p->n_tiles;
    w[8] = (int32_t)p->off_qmeta; w[9] = (int32_t)p->off_seqlen; w[10] = (int32_t)p->off_table;
    w[11] = (int32_t)p->off_decode; w[12] = (int32_t)p->off_tiles; w[13] = (int32_t)off;
    for (int32_t q = 0; q < num_queries; ++q) {
        int32_t *m = w + p->off_qmeta + 4 * (size_t)q;
        m[0] = query_seq[q];
        m[1] = query_pos[q];
        m[2] = (int32_t)slots[(size_t)q];
        m[3] = 0;
    }
    if (num_seqs) std::memcpy(w + p->off_seqlen, seq_lens, sizeof(int32_t) * (size_t)num_seqs);
    // Entries past a sequence's pages are kept as given (e.g. -1, or pages
    // reserved ahead for pa_plan_advance); the attention kernels never read them.
    if ((int64_t)num_seqs * width > 0)
        std::memcpy(w + p->off_table, block_table, sizeof(int32_t) * (size_t)num_seqs * width);
    if (!decode.empty()) std::memcpy(w + p->off_decode, decode.data(), sizeof(int32_t) * decode.size());
    if (!tiles.empty()) std::memcpy(w + p->off_tiles, tiles.data(), sizeof(int32_t) * tiles.size());
    {
        std::vector<int32_t> order((size_t)num_queries);
        for (int32_t q = 0; q < num_queries; ++q) order[(size_t)q] = q;
        std::stable_sort(order.begin(), order.end(),
                         [&](int32_t a, int32_t b) { return query_pos[a] > query_pos[b]; });
        if (num_queries) std::memcpy(w + p->off_order, order.data(), sizeof(int32_t) * order.size());
    }
    for (int c = 0; c < 2; ++c) visible_key_sums(p, c, 0, p->keys_tiles[c], p->keys_decode[c]);
    *out_plan = p;
    return PA_OK;
}

size_t pa_plan_device_bytes(const pa_plan *plan) { return plan ? plan->words.size() * sizeof(int32_t) : 0; }

pa_status pa_plan_upload(pa_plan *plan, void *device_words, size_t bytes, pa_stream_t stream) {
    if (!plan || !device_words) return fail(PA_ERR_ARG, "pa_plan_upload: null argument");
    if (!aligned16(device_words)) return fail(PA_ERR_ARG, "pa_plan_upload: device buffer not 16-byte aligned");
    size_t need = pa_plan_device_bytes(plan);
    if (bytes < need) return fail(PA_ERR_ARG, "pa_plan_upload: device buffer too small");
    cudaError_t e = cudaMemcpyAsync(device_words, plan->words.data(), need, cudaMemcpyHostToDevice,
                                    (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e, "pa_plan_upload");
    plan->dev = static_cast<const int32_t *>(device_words);
    return PA_OK;
}

pa_status pa_plan_stage(pa_plan *plan, void *host_words, size_t host_bytes, void *device_words,
                        size_t device_bytes) {
    if (!plan || !host_words || !device_words) return fail(PA_ERR_ARG, "pa_plan_stage: null argument");
    if (!aligned16(device_words)) return fail(PA_ERR_ARG, "pa_plan_stage: device buffer not 16-byte aligned");
    const size_t need = pa_plan_device_bytes(plan);
    if (host_bytes < need || device_bytes < need) return fail(PA_ERR_ARG, "pa_plan_stage: buffer too small");
    std::memcpy(host_words, plan->words.data(), need);
    plan->dev = static_cast<const int32_t *>(device_words);
    return PA_OK;
}

void pa_plan_destroy(pa_plan *plan) { delete plan; }

pa_status pa_plan_describe(const pa_plan *plan, int64_t out[8]) {
    if (!plan || !out) return fail(PA_ERR_ARG, "pa_plan_describe: null argument");
    out[0] = plan->queries; out[1] = plan->sequences; out[2] = plan->width; out[3] = plan->page_size;
    out[4] = plan->pages; out[5] = plan->n_decode; out[6] = plan->n_tiles; out[7] = plan->n_tile_queries;
    return PA_OK;
}

size_t pa_workspace_bytes(int32_t queries, int32_t heads, int32_t value_dim, int32_t splits) {
    if (queries < 0 || heads < 1 || value_dim < 1 || splits < 1) return 0;
    size_t rows = (size_t)splits * (size_t)queries * (size_t)heads;
    size_t o = (rows * (size_t)value_dim * sizeof(float) + 255) / 256 * 256;
    size_t l = (rows * sizeof(float) + 255) / 256 * 256;
    return o + l;
}

int32_t paged_attn_split_heuristic(const pa_plan *plan, int32_t num_heads, int32_t num_kv_heads,
                                   int32_t window, int32_t num_sms) {
    if (!plan || num_heads < 1 || num_kv_heads < 1 || num_heads % num_kv_heads || num_sms < 1) return 1;
    if (plan->n_decode + plan->n_tiles == 0) return 1;
    int64_t group = num_heads / num_kv_heads;
    // decode CTAs (one per KV head and group of up to 4 query heads) plus the
    // prefill CTAs (one per tile and query head), per split
    int64_t blocks = (int64_t)plan->n_decode * num_kv_heads * ((group + 3) / 4) + (int64_t)plan->n_tiles * num_heads;
    // about four blocks per SM; a few long histories (fewer blocks than SMs)
    // get about eight, so the uneven split lengths still balance
    int64_t target = (blocks >= num_sms ? 4 : 8) * (int64_t)num_sms;
    int64_t s = (target + blocks - 1) / blocks;
    const int64_t longest = window > 0 ? std::min<int64_t>(plan->max_seq_len, window) : plan->max_seq_len;
    int64_t cap = std::max<int64_t>(1, longest / (4 * (int64_t)plan->page_size));
    if (group >= 8 && plan->n_tiles == 0) {
        // Groups of 8+ go to the persistent tensor-core decode: one CTA per SM
        // walks (query, split, KV head) units in rounds of num_sms.  Aim for about
        // four rounds and, within a quarter of that, prefer split counts that
        // fill the last round (a partial round leaves SMs idle at the end).
        const int64_t n = (int64_t)plan->n_decode * num_kv_heads;
        const int64_t base = std::max<int64_t>(1, (4 * (int64_t)num_sms + n - 1) / n);
        double best_fill = -1.0;
        int64_t best = base;
        for (int64_t c = std::max<int64_t>(1, base - base / 4); c <= base + base / 4; ++c) {
            if (c > cap || c > PA_MAX_SPLITS) break;
            const int64_t units = n * c;
            const int64_t rounds = (units + num_sms - 1) / num_sms;
            const double fill = (double)units / (double)(rounds * num_sms);
            if (fill > best_fill + 1e-9 || (fill > best_fill - 1e-9 && std::llabs(c - base) < std::llabs(best - base))) {
                best_fill = fill;
                best = c;
            }
        }
        s = best;
    }
    s = std::min<int64_t>(s, cap);
    s = std::max<int64_t>(1, std::min<int64_t>(s, PA_MAX_SPLITS));
    return (int32_t)s;
}

int32_t paged_attn_decode_sms_beside_prefill(const pa_plan *plan, int32_t num_heads, int32_t num_kv_heads,
                                              int32_t head_dim, int32_t value_dim, int32_t causal, int32_t window,
                                              pa_dtype dtype, int32_t num_sms) {
    if (!plan || num_heads < 1 || num_kv_heads < 1 || head_dim < 1 || value_dim < 1 || !valid_dtype(dtype) ||
        num_sms < 1)
        return 0;
    // only tiles on the tensor-core prefill kernel run beside the decode items
    const int ps = plan->page_size;
    if (dtype == PA_F32 || head_dim != 128 || value_dim != 128 || (ps != 16 && ps != 32 && ps != 64 && ps != 128))
        return 0;
    return decode_sms_beside_prefill(plan, num_heads, num_kv_heads, head_dim, value_dim, causal, window, dtype,
                                     num_sms);
}

int32_t paged_mla_split_heuristic(const pa_plan *plan, int32_t num_heads, int32_t window, int32_t num_sms) {
    if (!plan || num_heads < 1 || num_sms < 1 || plan->queries == 0) return 1;
    // One CTA pair per (query, 128 heads, split), one pair per two SMs; the
    // kernel is tensor-bound, so splits only pay for themselves when pairs
    // would sit idle or one history dwarfs a pair's share of the work (every
    // split adds fp32 partials and a merge).
    const int64_t blocks = (num_heads + 127) / 128;
    const int64_t pairs = (int64_t)plan->queries * blocks;
    const int64_t slots = std::max<int64_t>(1, num_sms / 2);
    int64_t longest = 0, total = 0;
    for (int32_t q = 0; q < plan->queries; ++q) {
        int64_t n = (int64_t)plan->words[plan->off_qmeta + 4 * (size_t)q + 1] + 1;
        if (window > 0) n = std::min<int64_t>(n, window);
        longest = std::max(longest, n);
        total += n * blocks;
    }
    int64_t s = (slots + pairs - 1) / pairs;                     // every pair slot gets work
    const double share = 1.25 * (double)total / (double)slots;  // a pair slot's load, with slack
    if ((double)longest > share) s = std::max<int64_t>(s, (int64_t)std::ceil((double)longest / share));
    const int64_t cap = std::max<int64_t>(1, longest / 256);   // splits of at least 4 tiles of 64 keys
    s = std::max<int64_t>(1, std::min<int64_t>(std::min(s, cap), PA_MAX_SPLITS));
    return (int32_t)s;
}

pa_status paged_kv_store(const pa_plan *plan, const void *new_k, const void *new_v, void *k_cache,
                         void *v_cache, int32_t num_heads, int32_t head_dim, int32_t value_dim,
                         pa_dtype dtype, pa_stream_t stream) {
    if (!plan) return fail(PA_ERR_ARG, "paged_kv_store: plan is null");
    if (!valid_dtype(dtype)) return fail(PA_ERR_DTYPE, "paged_kv_store: dtype must be F32, F16 or BF16");
    if (num_heads < 1 || head_dim < 1 || value_dim < 1)
        return fail(PA_ERR_SHAPE, "paged_kv_store: heads, head_dim and value_dim must be >= 1");
    if ((int64_t)plan->pages * plan->page_size * num_heads * std::max(head_dim, value_dim) > (int64_t)1 << 40)
        return fail(PA_ERR_RANGE, "paged_kv_store: cache too large");
    if (plan->queries == 0) return PA_OK;  // no-op append
    if (!plan->dev) return fail(PA_ERR_STATE, "paged_kv_store: plan not uploaded");
    if (!new_k || !new_v || !k_cache || !v_cache) return fail(PA_ERR_ARG, "paged_kv_store: null tensor");
    {
        const void *ptrs[] = {new_k, new_v, k_cache, v_cache};
        const char *names[] = {"new_k", "new_v", "k_cache", "v_cache"};
        pa_status on_dev = operands_on_device(ptrs, names, 4, "paged_kv_store");
        if (on_dev != PA_OK) return on_dev;
    }
    cudaError_t e = pa::launch_kv_store(view_of(plan), new_k, new_v, k_cache, v_cache, num_heads, head_dim,
                                        value_dim, elem_bytes(dtype), (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e, "paged_kv_store launch");
    return PA_OK;
}

}  // extern "C"

// The argument checks of the attention entry points that need no device
// (`execute_attention_into`, `check_tensor`, `bounded`), in the order the
// calls apply them.
pa_status pa::check_attention_args(const pa_plan *plan, int32_t hq, int32_t hkv, int32_t d, int32_t dv, int32_t p,
                                   float scale, int32_t causal, int32_t window, pa_dtype dtype, bool mla,
                                   const char *name) {
    char msg[256];
    auto bad = [&](pa_status s, const char *what) {
        std::snprintf(msg, sizeof msg, "%s: %s", name, what);
        return fail(s, msg);
    };
    if (!plan) return bad(PA_ERR_ARG, "plan is null");
    if (!valid_dtype(dtype)) return bad(PA_ERR_DTYPE, "dtype must be F32, F16 or BF16");
    if (hq < 1 || hkv < 1 || hq % hkv != 0) return bad(PA_ERR_SHAPE, "num_heads must be a positive multiple of num_kv_heads");
    if (d < 1 || dv < 1) return bad(PA_ERR_SHAPE, "head dims must be >= 1");
    if (d > PA_MAX_HEAD_DIM || dv > PA_MAX_HEAD_DIM) return bad(PA_ERR_LIMIT, "head dim above 1024");
    if (!std::isfinite(scale) || !(scale > 0.f)) return bad(PA_ERR_SHAPE, "scale must be finite and > 0");
    if (causal != 0 && causal != 1) return bad(PA_ERR_ARG, "causal must be 0 or 1");
    if (window < 0) return bad(PA_ERR_ARG, "window must be >= 0");
    if (mla) {
        if (p < 1 || p > PA_MAX_POS_DIM) return bad(PA_ERR_LIMIT, "MLA position dim must be in 1..256");
    }
    if (hq > 65535) return bad(PA_ERR_LIMIT, "num_heads above the launch grid limit");
    if ((int64_t)plan->queries * hq * std::max(d, dv) > ((int64_t)1 << 40))
        return bad(PA_ERR_RANGE, "tensor too large");
    return PA_OK;
}

namespace {

// Shared body of the attention entry points.
// SMs to leave to the decode items of a mixed call while its prefill tiles
// run on the others (0: run them one after the other).  Model, from runs of
// the mixed workload on GB300 (128-wide heads): the prefill kernel does
// kPrefillFlopsPerSm on each of its SMs; while it runs, the decode kernel
// reads kDecodeBytesPerSm on each of its own SMs but no more than
// kDecodeBesidePrefill in all (the prefill's own loads share HBM and L2);
// what is left of the decode then runs on the whole GPU at kHbmBytes.  The
// share with the shortest modelled call is taken when it saves at least 5 %
// and both halves are long enough for the fork and join to be noise.
int decode_sms_beside_prefill(const pa_plan *plan, int hq, int hkv, int d, int dv, int causal, int window,
                              pa_dtype dtype, int sms) {
    constexpr double kPrefillFlopsPerSm = 6.5e12, kDecodeBytesPerSm = 7.2e10, kDecodeBesidePrefill = 2.0e12,
                     kHbmBytes = 6.2e12;
    if (plan->n_decode == 0 || plan->n_tiles == 0 || sms < 8) return 0;
    double keys_p, keys_d;
    if (window == 0) {          // worked out when the plan was built
        keys_p = plan->keys_tiles[causal ? 1 : 0];
        keys_d = plan->keys_decode[causal ? 1 : 0];
    } else {
        visible_key_sums(plan, causal, window, keys_p, keys_d);
    }
    const double flops = keys_p * hq * 2.0 * (d + dv);
    const double bytes = keys_d * hkv * (double)(d + dv) * elem_bytes(dtype);
    const double t_prefill = flops / (kPrefillFlopsPerSm * sms), t_decode = bytes / kHbmBytes;
    if (t_prefill < 20e-6 || t_decode < 20e-6) return 0;
    const double serial = t_prefill + t_decode;
    double best = serial;
    int best_n = 0;
    for (int n = 1; n < sms / 2; ++n) {
        const double tp = flops / (kPrefillFlopsPerSm * (sms - n));
        const double beside = std::min(kDecodeBesidePrefill, kDecodeBytesPerSm * n) * tp;
        const double t = bytes > beside ? tp + (bytes - beside) / kHbmBytes : std::max(tp, bytes / kHbmBytes);
        if (t < best) {
            best = t;
            best_n = n;
        }
    }
    return best < 0.95 * serial ? best_n : 0;
}

pa_status attention(const pa_plan *plan, const void *q, const void *k, const void *v, const void *qp,
                    const void *kp, void *out, int32_t hq, int32_t hkv, int32_t d, int32_t dv, int32_t p,
                    float scale, int32_t causal, int32_t window, pa_dtype dtype, void *ws, size_t ws_bytes, int32_t splits,
                    bool split_call, bool mla, cudaStream_t st, const char *name) {
    char msg[256];
    auto bad = [&](pa_status s, const char *what) {
        std::snprintf(msg, sizeof msg, "%s: %s", name, what);
        return fail(s, msg);
    };
    pa_status checked = pa::check_attention_args(plan, hq, hkv, d, dv, p, scale, causal, window, dtype, mla, name);
    if (checked != PA_OK) return checked;
    if (split_call) {
        if (splits < 1 || splits > PA_MAX_SPLITS) return bad(PA_ERR_SPLITS, "splits must be in 1..64");
        if (splits > 1 || ws) {
            size_t need = pa_workspace_bytes(plan->queries, hq, dv, splits);
            if (need > PA_WORKSPACE_LIMIT_BYTES) return bad(PA_ERR_WORKSPACE, "workspace above the 1 GiB limit");
            if (splits > 1 && !ws) return bad(PA_ERR_WORKSPACE, "workspace is null");
            if (ws && ws_bytes < need) return bad(PA_ERR_WORKSPACE, "workspace too small");
            if (ws && !aligned16(ws)) return bad(PA_ERR_WORKSPACE, "workspace not 16-byte aligned");
        }
    } else {
        splits = 1;
    }
    if (plan->queries == 0) return PA_OK;  // nothing to launch
    if (!plan->dev) return bad(PA_ERR_STATE, "plan not uploaded");
    if (!q || !k || !v || !out || (mla && (!qp || !kp))) return bad(PA_ERR_ARG, "null tensor");
    {
        const void *ptrs[] = {q, k, v, out, qp, kp, splits > 1 ? ws : nullptr};
        const char *names[] = {"q", "the key cache", "the value cache", "out", "the position query",
                               "the position cache", "the workspace"};
        pa_status on_dev = operands_on_device(ptrs, names, 7, name);
        if (on_dev != PA_OK) return on_dev;
    }

    pa::AttnArgs a{};
    a.plan = view_of(plan);
    a.q = q; a.k = k; a.v = v; a.qp = qp; a.kp = kp; a.out = out;
    a.hq = hq; a.hkv = hkv; a.d = d; a.dv = dv; a.p = mla ? p : 0;
    a.scale = scale; a.causal = causal; a.window = window; a.splits = splits; a.dtype = dtype;
    a.status = pa::device_status_ptr();
    if (!a.status) return bad(PA_ERR_CUDA, "device status word unavailable");
    if (splits > 1) {
        size_t rows = (size_t)splits * plan->queries * hq;
        a.ws_o = static_cast<float *>(ws);
        a.ws_lse = reinterpret_cast<float *>(static_cast<char *>(ws) + (rows * dv * sizeof(float) + 255) / 256 * 256);
    }

    cudaError_t e = cudaSuccess;
    // optional profiling events around the call's main (first) kernel
    cudaEvent_t t0 = g_time_start, t1 = g_time_stop;
    g_time_start = g_time_stop = nullptr;
    auto mark = [&](cudaEvent_t ev) {
        if (ev && e == cudaSuccess) e = cudaEventRecord(ev, st);
    };
    if (mla) {
        bool fast = pa::mla_supported(a);
        mark(t0);
        e = fast ? pa::launch_mla(a, false, st) : pa::launch_decode(a, false, st);
        mark(t1);
        if (e == cudaSuccess && splits > 1) e = pa::launch_merge(a, false, st);
    } else {
        bool tiles = plan->n_tiles > 0 && pa::prefill_supported(a);
        if (tiles) {
            // with splits > 1 both kernels write partials and one merge covers every query
            const int sms = device_sms();
            const int beside =
                sms > 0 ? decode_sms_beside_prefill(plan, hq, hkv, d, dv, causal, window, dtype, sms) : 0;
            SideStream *side = beside > 0 ? side_stream(st) : nullptr;
            if (side) {
                // prefill on sms - beside persistent CTAs, launched first so that they
                // hold their SMs; the decode items fill the rest from the side stream
                e = cudaEventRecord(side->fork, st);
                if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
                pa::AttnArgs ap = a;
                ap.max_ctas = sms - beside;
                mark(t0);
                if (e == cudaSuccess) e = pa::launch_prefill(ap, st);
                mark(t1);
                pa::AttnArgs ad = a;
                ad.max_ctas = beside;
                if (e == cudaSuccess) e = pa::launch_decode(ad, true, side->stream);
                if (e == cudaSuccess) e = cudaEventRecord(side->join, side->stream);
                if (e == cudaSuccess) e = cudaStreamWaitEvent(st, side->join, 0);
            } else {
                mark(t0);
                e = pa::launch_prefill(a, st);
                mark(t1);
                if (e == cudaSuccess && plan->n_decode > 0) e = pa::launch_decode(a, true, st);
            }
            if (e == cudaSuccess && splits > 1) e = pa::launch_merge(a, false, st);
        } else {
            // every query is a decode item: use the (longest-first) decode list
            const bool all_decode = plan->n_tiles == 0;
            mark(t0);
            e = pa::launch_decode(a, all_decode, st);
            mark(t1);
            if (e == cudaSuccess && splits > 1) e = pa::launch_merge(a, all_decode, st);
        }
    }
    if (e != cudaSuccess) return fail_cuda(e, name);
    return PA_OK;
}

}  // namespace

extern "C" {

pa_status paged_attn_forward(const pa_plan *plan, const void *q, const void *k_cache, const void *v_cache,
                             void *out, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t value_dim, float scale, int32_t causal, int32_t window, pa_dtype dtype,
                             pa_stream_t stream) {
    return attention(plan, q, k_cache, v_cache, nullptr, nullptr, out, num_heads, num_kv_heads, head_dim,
                     value_dim, 0, scale, causal, window, dtype, nullptr, 0, 1, false, false, (cudaStream_t)stream,
                     "paged_attn_forward");
}

pa_status paged_attn_forward_split(const pa_plan *plan, const void *q, const void *k_cache,
                                   const void *v_cache, void *out, int32_t num_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t value_dim, float scale, int32_t causal,
                                   int32_t window, pa_dtype dtype, void *workspace, size_t workspace_bytes,
                                   int32_t splits, pa_stream_t stream) {
    if (!workspace) return fail(PA_ERR_WORKSPACE, "paged_attn_forward_split: workspace is null");
    return attention(plan, q, k_cache, v_cache, nullptr, nullptr, out, num_heads, num_kv_heads, head_dim,
                     value_dim, 0, scale, causal, window, dtype, workspace, workspace_bytes, splits, true, false,
                     (cudaStream_t)stream, "paged_attn_forward_split");
}

pa_status paged_mla_forward(const pa_plan *plan, const void *q, const void *qp, const void *latent_cache,
                            const void *pos_cache, void *out, int32_t num_heads, int32_t latent_dim,
                            int32_t pos_dim, float scale, int32_t causal, int32_t window, pa_dtype dtype,
                            void *workspace, size_t workspace_bytes, int32_t splits, pa_stream_t stream) {
    if (!workspace && splits != 1)
        return fail(PA_ERR_SPLITS, "paged_mla_forward: splits must be 1 without a workspace");
    return attention(plan, q, latent_cache, latent_cache, qp, pos_cache, out, num_heads, 1, latent_dim,
                     latent_dim, pos_dim, scale, causal, window, dtype, workspace, workspace_bytes, splits, true, true,
                     (cudaStream_t)stream, "paged_mla_forward");
}

pa_status pa_plan_advance(pa_plan *plan, pa_stream_t stream) {
    if (!plan) return fail(PA_ERR_ARG, "pa_plan_advance: plan is null");
    if (plan->n_tiles > 0)
        return fail(PA_ERR_STATE, "pa_plan_advance: plans with prefill tiles cannot advance");
    if (plan->queries == 0) return PA_OK;
    if (!plan->dev) return fail(PA_ERR_STATE, "pa_plan_advance: plan not uploaded");
    int32_t *status = pa::device_status_ptr();
    if (!status) return fail(PA_ERR_CUDA, "pa_plan_advance: device status word unavailable");
    cudaError_t e = pa::launch_plan_advance(view_of(plan), status, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e, "pa_plan_advance launch");
    // keep the host copy in step with one advance (graph replays advance only the device copy)
    int32_t *w = plan->words.data();
    for (int32_t q = 0; q < plan->queries; ++q) {
        int32_t *m = w + plan->off_qmeta + 4 * (size_t)q;
        const int64_t np = (int64_t)m[1] + 1;
        if (np >= (int64_t)plan->width * plan->page_size) continue;
        const int32_t pg = w[plan->off_table + (size_t)m[0] * plan->width + np / plan->page_size];
        if (pg < 0 || pg >= plan->pages) continue;
        m[1] = (int32_t)np;
        m[2] = pg * plan->page_size + (int32_t)(np % plan->page_size);
        int32_t &sl = w[plan->off_seqlen + m[0]];
        if (sl < np + 1) sl = (int32_t)(np + 1);
        plan->max_seq_len = std::max<int64_t>(plan->max_seq_len, sl);
    }
    return PA_OK;
}

pa_status pa_time_next_kernel(void *start_event, void *stop_event) {
    g_time_start = static_cast<cudaEvent_t>(start_event);
    g_time_stop = static_cast<cudaEvent_t>(stop_event);
    return PA_OK;
}

pa_status pa_device_status(int32_t *code, int32_t clear) {
    if (!code) return fail(PA_ERR_ARG, "pa_device_status: code is null");
    cudaError_t e = pa::read_device_status(code, clear != 0);
    if (e != cudaSuccess) return fail_cuda(e, "pa_device_status");
    return PA_OK;
}

}  // extern "C"
