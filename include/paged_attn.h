/*
 * paged_attn.h -- C ABI of libpagedattn.so, paged attention over a
 * block-table KV cache on one NVIDIA GB300 (sm_103a).
 *
 * The operation is the one stated by ruDNN 0.1.7, src/paged_attention/mod.rs
 * (module doc and `DevicePlan`): packed decode and chunked causal prefill at
 * absolute positions for MHA/GQA, the MLA latent-cache variant, a split-KV
 * path that merges FP32 partial outputs and log-sum-exp statistics from a
 * reusable workspace, and the cache append.
 *
 * Conventions shared by every call:
 *  - Pointers named *_cache, q, qp, new_*, out and workspace are DEVICE
 *    pointers; every other pointer is a host pointer.  All device tensors are
 *    dense, row-major ("contiguous") in the layout given per call.  The
 *    library allocates no device memory; the caller owns every buffer.
 *  - Every call that touches the GPU takes a stream (a cudaStream_t; NULL is
 *    the legacy default stream), only enqueues work on it and returns; no
 *    call synchronises the device or reads device memory back (module doc:
 *    no host tensor readback; `attention_into_split`: no CPU synchronisation).
 *  - Every call validates all arguments on the host first and returns a
 *    status other than PA_OK without launching anything when one is wrong
 *    (`PagedAttentionError` / `check_tensor` / `bounded`).  The message of
 *    the last failure on the calling thread is pa_last_error().
 *  - Inputs must be finite on the keys a query can see; NaN or Inf there
 *    propagates into that query's output and is not checked (module doc).
 *    Cache slots no query can see (pages no sequence references, slots past a
 *    sequence's length) are never read and may hold anything.
 *  - Every device pointer must be device memory of the current device
 *    (cudaMalloc or a pool allocator on it): host memory, pinned or mapped,
 *    managed memory and peer GPUs' memory are refused with PA_ERR_ARG before
 *    anything is launched (`check_tensor`: every operand on Q's device).
 *  - `out` must not overlap any input (`attention_into`, safety contract).
 *  - Element types: PA_F32, PA_F16, PA_BF16 for every floating operand of a
 *    call (one dtype per call, `check_tensor`); accumulation is fp32 and the
 *    output is rounded once to the operand dtype.  Split partials are fp32.
 */
#ifndef PAGED_ATTN_H
#define PAGED_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *pa_stream_t; /* identical to cudaStream_t */

typedef enum {
    PA_OK = 0,
    PA_ERR_ARG = 1,             /* null pointer where one is required, bad flag, misuse   */
    PA_ERR_SHAPE = 2,           /* shapes disagree with each other or with the plan       */
    PA_ERR_DTYPE = 3,           /* dtype not F32/F16/BF16                                 */
    PA_ERR_RANGE = 4,           /* index out of range: page id, position, u32 overflow    */
    PA_ERR_WRITE_CONFLICT = 5,  /* two queries of one plan write the same cache slot      */
    PA_ERR_WORKSPACE = 6,       /* workspace missing, too small or over the limit         */
    PA_ERR_SPLITS = 7,          /* split count outside 1..PA_MAX_SPLITS                   */
    PA_ERR_LIMIT = 8,           /* head dim > 1024, position dim > 256, grid limits       */
    PA_ERR_CUDA = 9,            /* a CUDA runtime call or kernel launch failed            */
    PA_ERR_STATE = 10           /* plan not uploaded                                      */
} pa_status;

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2 } pa_dtype;

#define PA_ABI_VERSION 3
#define PA_MAX_SPLITS 64                        /* `MAX_SPLITS` of the split workspace      */
#define PA_MAX_HEAD_DIM 1024                    /* d, dv <= 1024 (`execute_attention_into`) */
#define PA_MAX_POS_DIM 256                      /* MLA position dim P <= 256                */
#define PA_WORKSPACE_LIMIT_BYTES (1ull << 30)   /* `WORKSPACE_LIMIT_BYTES`                  */

/* Opaque schedule: host metadata plus the device copy the caller uploads. */
typedef struct pa_plan pa_plan;

/* Message of the last failed call on this thread ("" if none). */
const char *pa_last_error(void);
/* Short name of a status code. */
const char *pa_status_string(pa_status status);
/* PA_ABI_VERSION of the loaded library. */
int32_t pa_abi_version(void);

/*
 * Build and validate a schedule on the host (`HostPlan`, uploaded by
 * `DevicePlan::upload`).
 *
 *   seq_lens[num_seqs]            keys present in each sequence after this
 *                                 step's append (>= 1 for a sequence that a
 *                                 query names; 0 allowed otherwise)
 *   block_table[num_seqs*width]   row-major; entry [s][g] is the physical page
 *                                 holding keys g*page_size .. g*page_size+page_size-1
 *                                 of sequence s.  Entries for g >= ceil(seq_len/page_size)
 *                                 are ignored (may be -1).
 *   query_seq[num_queries]        sequence of each packed query
 *   query_pos[num_queries]        absolute position of each query (its own key
 *                                 is written there by paged_kv_store; causal
 *                                 queries see keys 0..pos, non-causal ones keys
 *                                 0..seq_len-1)
 *
 * Checks (PA_ERR_RANGE / PA_ERR_WRITE_CONFLICT / PA_ERR_ARG): counts >= 0,
 * page_size >= 1; every used table entry in [0, num_pages); 0 <= pos <
 * seq_len[seq]; seq_len <= width*page_size; no two queries map to the same
 * physical slot (page sharing for reads across sequences is allowed); every
 * size within u32 indexing.  num_queries == 0 is a valid empty plan.
 *
 * Besides per-query (seq, pos, slot) metadata the plan lists its work: runs of
 * consecutive positions of one sequence (>= 16 queries) become prefill tiles
 * of up to 128 queries for the tensor-core kernel; every other query is a
 * decode item.  On success *out_plan owns host memory only; release it with
 * pa_plan_destroy().
 */
pa_status paged_attn_plan(const int32_t *seq_lens, int32_t num_seqs, const int32_t *block_table,
                          int32_t width, const int32_t *query_seq, const int32_t *query_pos,
                          int32_t num_queries, int32_t page_size, int32_t num_pages,
                          pa_plan **out_plan);

/* Bytes of device memory the plan's metadata needs (a multiple of 16). */
size_t pa_plan_device_bytes(const pa_plan *plan);

/*
 * Enqueue one host-to-device copy of the plan's metadata into `device_words`
 * (caller-owned, >= pa_plan_device_bytes, 16-byte aligned, kept alive while the
 * plan is used) and bind it to the plan.  The plan stays valid and reusable
 * while the schedule is unchanged (`DevicePlan` doc).  The host words are
 * staged before this call returns, so the plan may be destroyed at any time
 * after it.
 */
pa_status pa_plan_upload(pa_plan *plan, void *device_words, size_t bytes, pa_stream_t stream);

/*
 * Stage a plan for a copy the caller makes: write its device image
 * (pa_plan_device_bytes bytes, the same bytes pa_plan_upload copies) into the
 * caller's host buffer `host_words` (typically pinned memory) and bind
 * `device_words` as the plan's device copy, without touching the device.  The
 * caller then moves host_words to device_words with its own stream-ordered
 * copy before the next call that uses the plan; a copy from pinned memory can
 * be captured in a CUDA graph, so one replay can refresh the schedule, append
 * and attend (the `DevicePlan` schedule re-sent each step with no host
 * synchronisation on the way).  Both buffers are caller-owned and at least
 * pa_plan_device_bytes long; device_words is 16-byte aligned and stays alive
 * while the plan is used.  PA_ERR_ARG on a null pointer, a short buffer or a
 * misaligned device buffer (nothing is written then).  A graph captured around
 * calls on this plan stays valid for images of plans with the same counts
 * (pa_plan_describe) and the same device buffer.
 */
pa_status pa_plan_stage(pa_plan *plan, void *host_words, size_t host_bytes, void *device_words,
                        size_t device_bytes);

/* Free the host side of a plan (does not touch the caller's device buffer). */
void pa_plan_destroy(pa_plan *plan);

/*
 * Counts of a plan: out[0] queries, [1] sequences, [2] table width,
 * [3] page size, [4] pages, [5] decode items, [6] prefill tiles,
 * [7] queries covered by prefill tiles.
 */
pa_status pa_plan_describe(const pa_plan *plan, int64_t out[8]);

/*
 * Workspace bytes for `splits` partials of `queries` x `heads` rows of
 * `value_dim` floats: fp32 [splits, queries, heads, value_dim] followed by
 * fp32 log-sum-exp [splits, queries, heads] (`SplitWorkspace`, an F32 tensor),
 * each part 256-byte aligned.  Returns 0 for invalid arguments.
 */
size_t pa_workspace_bytes(int32_t queries, int32_t heads, int32_t value_dim, int32_t splits);

/*
 * Split count for paged_attn_forward_split / paged_mla_forward on this plan
 * (libmir-cuda 0.1.0, src/backend/attention/graph/mod.rs enables a split
 * path above a `split_threshold`; its value is not given, this rule is ours):
 * enough blocks (decode: per item, KV head and group of up to 4 query heads;
 * prefill: per tile and query head) per split to give every SM about four
 * (eight when one split has fewer blocks than there are SMs), no split
 * shorter than 4 pages of the longest visible history (at most `window` keys
 * when window > 0), 1..PA_MAX_SPLITS.
 */
int32_t paged_attn_split_heuristic(const pa_plan *plan, int32_t num_heads, int32_t num_kv_heads,
                                   int32_t window, int32_t num_sms);

/*
 * Split count for paged_mla_forward (same source as above; the rule is ours):
 * the tensor-core MLA kernel runs one CTA pair per (query, 128 heads, split)
 * and is bound by the tensor pipe, so it splits only as far as needed to give
 * each of the num_sms / 2 SM pairs work, and to keep the longest history
 * (pos + 1 keys, at most `window` when window > 0) within 1.25x one pair's
 * share of all keys; each split keeps at least 256 keys, 1..PA_MAX_SPLITS.
 */
int32_t paged_mla_split_heuristic(const pa_plan *plan, int32_t num_heads, int32_t window, int32_t num_sms);

/*
 * SMs that paged_attn_forward / paged_attn_forward_split leave to the decode
 * items of this plan while its prefill tiles run on the others (0: the two
 * kernels run one after the other), on a GPU of num_sms SMs.  Only tiles on
 * the tensor-core prefill kernel (bf16 or fp16, head_dim = value_dim = 128,
 * pages of 16, 32, 64 or 128 rows) run beside the decode items.  The pages
 * describe one call for mixed prefill + decode batches and say nothing of
 * how its parts share the GPU; this rule is ours.  It models the prefill
 * kernel at a fixed rate per SM and the decode kernel at a fixed rate per SM
 * capped while the prefill runs, and keeps the share that shortens the call
 * by at least 5 %, when both parts would take at least 20 us alone.  The
 * calls run the decode kernel on a second stream of the calling thread
 * (created on the first such call that is not being captured and kept for
 * the thread's life, like the status word: a process that resets the device
 * must not call the library on it again), forked from and joined back into
 * the caller's stream with events.  Pure host function
 * of the plan; 0 for invalid arguments.
 */
int32_t paged_attn_decode_sms_beside_prefill(const pa_plan *plan, int32_t num_heads, int32_t num_kv_heads,
                                              int32_t head_dim, int32_t value_dim, int32_t causal,
                                              int32_t window, pa_dtype dtype, int32_t num_sms);

/*
 * One decode step forward, on the device: every query of an uploaded plan
 * moves to position pos + 1 of its sequence, its write slot is taken from the
 * block table and its sequence length grows to cover the new position.  This
 * keeps the per-step schedule in device memory, so a CUDA graph captured
 * around pa_plan_advance + paged_kv_store + an attention call replays a
 * decode loop step after step without re-capture (libmir-cuda 0.1.0,
 * `CapturedDecodeAttentionBf16`; boostr 0.1.0, `DeviceScalars::update`: write
 * at seq_len, attend over seq_len + 1, updated stream-ordered with no host
 * synchronisation).  The caller reserves the pages ahead in the block table
 * given to paged_attn_plan (entries past a sequence's current pages are not
 * validated there).  A position the table does not map leaves that query
 * unchanged and sets PA_DEVICE_RANGE in the device status word.  Plans with
 * prefill tiles are refused (PA_ERR_STATE); the host copy advances with each
 * call, but graph replays advance only the device copy.
 */
pa_status pa_plan_advance(pa_plan *plan, pa_stream_t stream);

/*
 * Cache append (`DevicePlan::append_with_report`): for every query q and head
 * h, new_k[q, h, :] is copied bit-for-bit into k_cache[page, row, h, :] and
 * new_v[q, h, :] into v_cache[page, row, h, :], where page =
 * block_table[query_seq[q]][query_pos[q] / page_size] and row =
 * query_pos[q] % page_size.
 *
 *   new_k   [queries, heads, head_dim]           new_v   [queries, heads, value_dim]
 *   k_cache [pages, page_size, heads, head_dim]  v_cache [pages, page_size, heads, value_dim]
 *
 * head_dim and value_dim may differ (MLA: latent rows into the latent cache and
 * rotated position rows into the position cache, heads = 1).  A plan with zero
 * queries enqueues nothing.  The plan's write-conflict check guarantees that
 * no two queries write one slot.
 */
pa_status paged_kv_store(const pa_plan *plan, const void *new_k, const void *new_v, void *k_cache,
                         void *v_cache, int32_t num_heads, int32_t head_dim, int32_t value_dim,
                         pa_dtype dtype, pa_stream_t stream);

/*
 * Paged MHA/GQA attention (`DevicePlan::attention` / `attention_into`):
 * for query q and head h, with kv = h / (num_heads / num_kv_heads),
 *   out[q, h, :] = sum_j softmax_j(scale * q[q,h,:] . K_j) V_j
 * over the keys j that q sees (causal: 0..pos; else 0..seq_len-1), K_j / V_j
 * gathered through the block table from head kv.  window > 0 is a sliding
 * window: the keys start at pos - window + 1 (a layer's `window`, libmir-cuda
 * 0.1.0, src/backend/attention/graph/mod.rs, `Geometry`; the pages name the
 * field only, this reading is ours); window == 0 is no window; < 0 is
 * PA_ERR_ARG.
 *
 *   q       [queries, num_heads, head_dim]
 *   k_cache [pages, page_size, num_kv_heads, head_dim]
 *   v_cache [pages, page_size, num_kv_heads, value_dim]
 *   out     [queries, num_heads, value_dim]
 *
 * Requires num_heads % num_kv_heads == 0, 1 <= head_dim, value_dim <= 1024,
 * finite scale > 0 (`execute_attention_into`).  Zero queries: PA_OK, no launch.
 */
pa_status paged_attn_forward(const pa_plan *plan, const void *q, const void *k_cache,
                             const void *v_cache, void *out, int32_t num_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t value_dim,
                             float scale, int32_t causal, int32_t window, pa_dtype dtype,
                             pa_stream_t stream);

/*
 * Split-KV form (`attention_into_split`): the visible history [lo, hi) of
 * every query -- decode items and each row of a prefill tile alike -- is cut
 * into `splits` contiguous ranges (base = lo rounded down to a page boundary,
 * chunk = ceil((hi - base) / splits) rounded up to a multiple of page_size,
 * split s covers [max(lo, base + s*chunk), min(base + (s+1)*chunk, hi));
 * lo = 0 without a window); each range writes its normalised fp32 partial
 * output and natural-log log-sum-exp into `workspace`, then a merge kernel
 * writes out.  The workspace
 * (>= pa_workspace_bytes(queries, num_heads, value_dim, splits), 16-byte
 * aligned) may be reused by later calls on the same stream with any plan;
 * calls on different streams need different workspaces.  splits == 1 is
 * allowed.  Same shapes and checks as paged_attn_forward.
 */
pa_status paged_attn_forward_split(const pa_plan *plan, const void *q, const void *k_cache,
                                   const void *v_cache, void *out, int32_t num_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t value_dim,
                                   float scale, int32_t causal, int32_t window, pa_dtype dtype,
                                   void *workspace, size_t workspace_bytes, int32_t splits,
                                   pa_stream_t stream);

/*
 * MLA attention (`DevicePlan::mla`, `mla_with_workspace`): one shared latent
 * head is both key and value and a rotated position cache adds a second score
 * term:  out[q, h, :] = sum_j softmax_j(scale * (q[q,h,:] . c_j + qp[q,h,:] . r_j)) c_j.
 *
 *   q            [queries, num_heads, latent_dim]   (absorbed query)
 *   qp           [queries, num_heads, pos_dim]      (position query)
 *   latent_cache [pages, page_size, 1, latent_dim]
 *   pos_cache    [pages, page_size, 1, pos_dim]
 *   out          [queries, num_heads, latent_dim]
 *
 * `scale` comes from the model's original QK head dims, not the latent rank.
 * 1 <= latent_dim <= 1024, 1 <= pos_dim <= 256.  workspace may be NULL (then
 * splits must be 1); otherwise the split rules of paged_attn_forward_split
 * apply with value_dim = latent_dim.  `window` as for paged_attn_forward.
 */
pa_status paged_mla_forward(const pa_plan *plan, const void *q, const void *qp,
                            const void *latent_cache, const void *pos_cache, void *out,
                            int32_t num_heads, int32_t latent_dim, int32_t pos_dim, float scale,
                            int32_t causal, int32_t window, pa_dtype dtype, void *workspace,
                            size_t workspace_bytes, int32_t splits, pa_stream_t stream);

/*
 * Split-KV forward that allocates nothing.  The pages have no counterpart for
 * this call; it serves callers that cannot hand the library a workspace --
 * code inside a host runtime that owns every device allocation (a serving
 * engine with one fixed memory pool, a plugin host that forbids stray
 * allocations) or that cannot afford cudaMalloc's implicit device-wide
 * synchronisation in a decode loop.  Same arguments, checks and result as
 * paged_attn_forward_split, but the split partials live in a file-scope device
 * array of PA_STATIC_SCRATCH_BYTES that every GPU loading the library holds
 * until the process exits.  The caller still owns q, the caches and out.
 *
 * The argument checks of paged_attn_forward_split run first and return the
 * same statuses; then any plan/heads/value_dim/splits whose
 * pa_workspace_bytes exceeds PA_STATIC_SCRATCH_BYTES is rejected
 * (PA_ERR_WORKSPACE).  Calls no cudaMalloc, cudaFree or allocating library
 * routine.  The first call on a device looks up the array's device address
 * with that device current and keeps it; make that call before any stream
 * capture, and do not call this entry point on a device after a
 * cudaDeviceReset of it (the reset may move the array).  All calls share the
 * array and it keeps the last call's
 * contents (each call writes every entry it later reads, so nothing needs
 * clearing); calls whose GPU work overlaps race on it -- serialise them on one
 * stream.
 */
#define PA_STATIC_SCRATCH_BYTES (16u << 20)
pa_status paged_attn_forward_split_static(const pa_plan *plan, const void *q, const void *k_cache,
                                          const void *v_cache, void *out, int32_t num_heads,
                                          int32_t num_kv_heads, int32_t head_dim, int32_t value_dim,
                                          float scale, int32_t causal, int32_t window, pa_dtype dtype,
                                          int32_t splits, pa_stream_t stream);

/*
 * Profiling hook: the next attention call made on this thread records
 * `start_event` on its stream just before launching its main kernel (the
 * decode, MLA or prefill kernel -- the first one the call launches) and
 * `stop_event` right after it.  Both are caller-created cudaEvent_t handles;
 * the hook is consumed by that one call.  It changes no result; the benchmark
 * uses it to time the dominant kernel alone.
 */
pa_status pa_time_next_kernel(void *start_event, void *stop_event);

/*
 * Device-side status word.  Kernels that wait on hardware (mbarriers, tensor
 * memory) bound every wait; a wait that runs out sets this word to a non-zero
 * code (PA_DEVICE_TIMEOUT_*) and the kernel returns early, leaving the context
 * usable.  This call synchronises the current device, reads the word and
 * optionally clears it; it is a diagnostic, not part of the hot path.  The
 * word's device address is looked up once per device and kept, so a process
 * that calls cudaDeviceReset must not use the library on that device again.
 */
#define PA_DEVICE_TIMEOUT_TMA 1
#define PA_DEVICE_TIMEOUT_MMA 2
#define PA_DEVICE_TIMEOUT_SOFTMAX 3
#define PA_DEVICE_RANGE 4
#define PA_DEVICE_LAYOUT 5   /* a kernel found its shared memory misplaced and did nothing */
pa_status pa_device_status(int32_t *code, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H */
