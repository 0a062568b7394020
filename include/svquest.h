/*
 * svquest.h -- C ABI of libsvquest.so: query-aware (Quest-style) sparse decode
 * attention over a paged KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The three calls map the cache-manager hooks of the "add-sparse-method"
 * skill page (section "Placement Rules", items 3-5) and the SparseEngine
 * summary page (section "method key points": CacheManager, AttentionView):
 *   on_kv_stored(...)      -> sv_quest_update_meta  (store K/V, refresh page metadata)
 *   build_decode_view(q)   -> sv_quest_select       (query-aware page selection)
 *   generic attention      -> sv_sparse_decode      (attention over the view)
 * and sv_quest_decode_step runs the last two in one call.
 *
 * Conventions common to every call
 *  - Every buffer argument is a DEVICE pointer, allocated and owned by the
 *    caller; the library never allocates, frees or retains it.  One
 *    exception: the per-step inputs and results of sv_quest_decode_step (q,
 *    page_table, seq_lens, out, lse) may be page-locked host memory that the
 *    GPU addresses under unified addressing (e.g. from cudaHostAlloc).  Its
 *    kernels then read those inputs and write those results across the
 *    host link themselves, with no separate copy.
 *  - q, k_new, v_new, out, the pools, the metadata, the fp8 scales and the
 *    workspaces of sv_sparse_decode(_ex) and sv_quest_decode_step must be
 *    16-byte aligned (SV_ERR_INVALID_ARG otherwise): kernels move them 16
 *    bytes at a time.
 *  - bf16 means IEEE bfloat16 stored as 16-bit words.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls enqueue kernels and return; they never synchronise.
 *  - Kernels are launched with programmatic dependent launch.  The scoring,
 *    top-K and attention kernels read the call's q, page_table and seq_lens,
 *    and the append kernel its slot_mapping, k_new and v_new, as soon as
 *    they start, possibly while the kernel enqueued just before them is
 *    still running.  Pools, metadata and workspace are touched only
 *    after that kernel has completed.  So the kernel that produces a
 *    call's inputs must not release its dependents early
 *    (griddepcontrol.launch_dependents): an ordinary kernel, a copy, or any
 *    work enqueued earlier is fine.
 *  - The page metadata and the K/V tiles a call streams are read through an
 *    L2 evict-first policy, so that they displace little else: what a call
 *    reuses (page tables, scores, selections, split partials) and the
 *    caller's other data tend to stay in L2 across calls.
 *  - Arguments are checked on the host before anything is launched.  A
 *    failed check returns a nonzero sv_status and launches nothing.  Values
 *    that live on the device (page tables, slot mappings, selected indices)
 *    cannot be checked on the host: kernels bounds-check them, skip any
 *    access they would make out of range and record the fault in a device
 *    error word read by sv_get_device_error().
 *  - Geometry: page_size must be 16 and head_dim 128 (SV_ERR_UNSUPPORTED
 *    otherwise); num_q_heads must be a multiple of num_kv_heads with at most
 *    8 query heads per kv head; query head h reads kv head h / (Hq / Hkv).
 *
 * Layouts (row-major, innermost last)
 *   k_pool, v_pool  bf16 [num_phys_pages][num_kv_heads][16][128]   (e4m3: see sv_cache)
 *   meta            bf16 [num_phys_pages][num_kv_heads][2][128]
 *                        [..][0][:] = per-channel key minimum of the page,
 *                        [..][1][:] = per-channel key maximum
 *   q               bf16 [B][num_q_heads][128]
 *   page_table      int32 [B][max_pages]   logical page -> physical page
 *   seq_lens        int32 [B]              tokens of each request, >= 1;
 *                        request b has n_b = ceil(seq_lens[b] / 16) pages,
 *                        the last holding seq_lens[b] - 16 (n_b - 1) tokens
 *   sel_idx         int32 [B][num_kv_heads][budget_pages]
 *   sel_cnt         int32 [B][num_kv_heads]
 */
#ifndef SVQUEST_H
#define SVQUEST_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum sv_status {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1,   /* NULL pointer, negative or inconsistent size */
    SV_ERR_UNSUPPORTED = 2,   /* geometry this build does not support */
    SV_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than required */
    SV_ERR_CUDA = 4           /* a kernel launch or device query failed */
};

/* Device error-word bits (sv_get_device_error). */
#define SV_DEVERR_PAGE_TABLE 0x1u   /* page_table entry outside [0, num_phys_pages) */
#define SV_DEVERR_SEL_IDX    0x2u   /* sel_idx entry outside [0, n_b) or sel_cnt out of range */
#define SV_DEVERR_SLOT       0x4u   /* slot_mapping entry outside the pool */
#define SV_DEVERR_SEQ_LEN    0x8u   /* seq_lens[b] < 1 or needs more than max_pages pages */
#define SV_DEVERR_TIMEOUT    0x10u  /* a kernel gave up a wait on its own bulk copies after
                                       2^28 SM clock cycles */

/* K/V pool formats (sv_cache.kv_format). */
#define SV_KV_BF16     0   /* k_pool, v_pool bf16 [pages][Hkv][16][128] */
#define SV_KV_FP8_E4M3 1   /* k_pool, v_pool e4m3 bytes [pages][Hkv][16][128], one fp32 scale per row */

/*
 * The paged pool and its metadata: caller-owned device buffers.
 *
 * SV_KV_FP8_E4M3 (the pages name a quantized attention view but define no
 * codec; the one used here): every (token, kv head) row of K and of V is 128
 * e4m3 codes (sign, 4 exponent bits biased by 7, 3 mantissa bits, largest
 * finite 448) and one fp32 scale s = max |x| / 448 over the row's bf16
 * values; x is stored as e4m3(x / s), rounded to nearest with ties to even and
 * saturated to +-448 (an all-zero row stores s = 0 and zero codes), and reads
 * back as value(code) * s.  The metadata stays bf16 and holds the min / max
 * of the keys as appended (before coding), so page selection is the same as
 * for bf16 pools; only attention reads the coded rows.  All calls accept both
 * formats.
 */
typedef struct sv_cache {
    void* k_pool;             /* [num_phys_pages][num_kv_heads][16][128] of the format's element */
    void* v_pool;
    void* meta;               /* bf16 [num_phys_pages][num_kv_heads][2][128]  */
    int64_t num_phys_pages;
    int32_t num_kv_heads;
    int32_t page_size;        /* must be 16 */
    int32_t head_dim;         /* must be 128 */
    int32_t kv_format;        /* SV_KV_BF16 (zero) or SV_KV_FP8_E4M3 */
    void* k_scale;            /* SV_KV_FP8_E4M3: fp32 [num_phys_pages][num_kv_heads][16]; else unused */
    void* v_scale;
} sv_cache;

/*
 * sv_quest_update_meta -- the on_kv_stored hook ("add-sparse-method" page,
 * "Placement Rules" item 3: metadata is updated after KV is written).
 * Writes T new tokens' key and value rows into the pool at
 * slot = physical_page * 16 + offset, and refreshes the touched pages'
 * per-channel key min/max: a page whose run of new tokens starts at offset 0
 * restarts its metadata from those tokens; otherwise the new tokens are
 * folded into the stored min/max.  min/max of bf16 values are bf16 values,
 * so the metadata is exact.
 *   k_new, v_new   bf16 [T][num_kv_heads][128]
 *   slot_mapping   int32 [T]
 * Contract: within one call, the tokens of one page are consecutive in the
 * token list with increasing offsets; across calls, each page fills from
 * offset 0 without holes.  T == 0 is a no-op.
 */
int sv_quest_update_meta(const sv_cache* cache, const void* k_new, const void* v_new,
                         const int32_t* slot_mapping, int64_t num_tokens, void* stream);

/*
 * sv_quest_score -- the page-scoring half of build_decode_view.  For every
 * request b, kv head g and logical page p < n_b:
 *   scores[b][g][p] = sum over the query heads h of group g, over channels i,
 *                     of max(q[h][i] * kmax[i], q[h][i] * kmin[i])
 * computed in fp32 as sum_i Qp[i] * kmax[i] + Qn[i] * kmin[i] with
 * Qp = sum_h max(q_h, 0) and Qn = sum_h min(q_h, 0), which is the same sum
 * regrouped by the sign of each q.  Entries p >= n_b are not written.
 *   scores   fp32 [B][num_kv_heads][max_pages]
 */
int sv_quest_score(const sv_cache* cache, const void* q, int32_t num_q_heads,
                   const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                   int32_t max_pages, float* scores, void* stream);

/*
 * sv_quest_topk -- the selection half of build_decode_view ("Quest's
 * query-relevant page selection", SparseEngine page, "method key points").
 * For each (b, g) keeps the K_b = min(budget_pages, n_b) pages with the
 * highest score; among equal scores the lower logical page index wins.
 * Writes their logical indices in ascending order to sel_idx[b][g][0..K_b),
 * -1 to the rest of the row, and K_b to sel_cnt[b][g].  Scores compare as
 * fp32 values, except that -0.0 ranks below +0.0 and NaN above +inf
 * (sv_quest_score produces neither from finite inputs).
 * max_pages <= 32768.
 */
int sv_quest_topk(const float* scores, const int32_t* seq_lens, int32_t batch,
                  int32_t num_kv_heads, int32_t max_pages, int32_t budget_pages,
                  int32_t* sel_idx, int32_t* sel_cnt, void* stream);

/*
 * sv_quest_select -- build_decode_view in one call: sv_quest_score then
 * sv_quest_topk.  Scores go to scores_out when it is non-NULL (fp32
 * [B][num_kv_heads][max_pages]), else to the workspace, which must then hold
 * sv_quest_select_workspace_size(...) bytes (ws may be NULL when scores_out
 * is given).
 */
int sv_quest_select(const sv_cache* cache, const void* q, int32_t num_q_heads,
                    const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                    int32_t max_pages, int32_t budget_pages, int32_t* sel_idx, int32_t* sel_cnt,
                    float* scores_out, void* workspace, size_t workspace_bytes, void* stream);

size_t sv_quest_select_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t max_pages);

/*
 * sv_sparse_decode -- exact softmax attention of each query head over the
 * tokens of its kv head's selected pages (the AttentionView consumed by a
 * generic attention backend; SparseEngine page, "method key points").
 * With sel_idx == NULL every page 0..n_b-1 is read (dense decode).
 *   z_t = (q_h . k_t) * softmax_scale over the valid tokens t of the pages,
 *   out[b][h] = sum_t softmax(z)_t v_t        bf16 [B][num_q_heads][128]
 *   lse[b][h] = ln(sum_t exp(z_t))            fp32 [B][num_q_heads]
 * A head with no token gets out = 0, lse = -inf.  Split-K: each (request,
 * kv head) is cut into page ranges whose partial (max, sum, output) go to
 * the workspace and are merged by a log-sum-exp combine.
 * budget_pages is the row length of sel_idx (ignored when dense).
 */
int sv_sparse_decode(const sv_cache* cache, const void* q, int32_t num_q_heads,
                     const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                     int32_t max_pages, const int32_t* sel_idx, const int32_t* sel_cnt,
                     int32_t budget_pages, float softmax_scale, void* out, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream);

/* pages = budget_pages for sparse decode, max_pages for dense decode. */
size_t sv_sparse_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t pages);

/*
 * Selection options (the pages describe none of these policies; each is a
 * switch on the selection, off when zero):
 *   per_q_head    0: one page set per kv head, scored with the bound summed
 *                 over its query heads (the base method);
 *                 1: one page set per query head, scored with that head's
 *                 own bound against its kv head's metadata.  sel_idx then
 *                 holds R = num_q_heads rows per request ([B][Hq][K],
 *                 sel_cnt [B][Hq], scores [B][Hq][max_pages]) and each
 *                 query head attends only its own row's pages.
 *   sink_pages,   the first sink_pages and the last window_pages logical
 *   window_pages  pages of every request are always selected: they rank
 *                 above every scored page, among themselves by lower page
 *                 index, and count toward budget_pages.  Their entries in
 *                 scores_out are +inf.
 *   layer,        a layer with layer < dense_layers attends densely:
 *   dense_layers  sv_quest_select_ex returns SV_OK without launching or
 *                 writing anything, and sv_sparse_decode_ex ignores sel_idx
 *                 and reads every page.
 * Negative values, or per_q_head other than 0 / 1, are SV_ERR_INVALID_ARG.
 * A NULL opts pointer means all zero.
 */
typedef struct sv_quest_opts {
    int32_t per_q_head;
    int32_t sink_pages;
    int32_t window_pages;
    int32_t layer;
    int32_t dense_layers;
} sv_quest_opts;

/* sv_quest_select with options; R = num_q_heads rows per request when
 * per_q_head, else num_kv_heads.  The scores workspace (when scores_out is
 * NULL) is sv_quest_select_ex_workspace_size(...) bytes. */
int sv_quest_select_ex(const sv_cache* cache, const void* q, int32_t num_q_heads,
                       const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                       int32_t max_pages, int32_t budget_pages, const sv_quest_opts* opts,
                       int32_t* sel_idx, int32_t* sel_cnt, float* scores_out,
                       void* workspace, size_t workspace_bytes, void* stream);

size_t sv_quest_select_ex_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t max_pages, const sv_quest_opts* opts);

/* sv_sparse_decode with options: sel_idx / sel_cnt in the layout
 * sv_quest_select_ex wrote for the same options; batch * R <= 65535.  The
 * workspace is sv_sparse_decode_workspace_size(...) bytes, as without options. */
int sv_sparse_decode_ex(const sv_cache* cache, const void* q, int32_t num_q_heads,
                        const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                        int32_t max_pages, const int32_t* sel_idx, const int32_t* sel_cnt,
                        int32_t budget_pages, const sv_quest_opts* opts, float softmax_scale,
                        void* out, float* lse, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * sv_sparse_decode_static_scratch -- sv_sparse_decode without a caller
 * workspace; the paper has no counterpart to this call.  It is for callers
 * that cannot allocate device memory: plugins inside a host framework that
 * owns every device allocation and forbids cudaMalloc, or serving loops that
 * reserved nearly all of HBM for the KV cache up front.  The split-K
 * partials go to a 16 MiB array compiled into the library (every GPU that
 * loads the library holds it until the process exits).  The call allocates
 * nothing; inputs and outputs are still the caller's.
 *  - The first call on a device looks up that device's address of the array
 *    (a runtime symbol query); make that first call before any stream capture.
 *  - Every call shares the one array: calls whose kernels may overlap on the
 *    GPU (other streams, other threads) race on it and must be serialised by
 *    the caller.  Nothing in it needs to start at zero.
 *  - Returns SV_ERR_WORKSPACE, launching nothing, when
 *    sv_sparse_decode_workspace_size(batch, num_q_heads, num_kv_heads, pages)
 *    exceeds SV_STATIC_SCRATCH_BYTES (e.g. batch 8 x 32 query heads fits at
 *    any budget; batch 32 x 32 heads fits up to 248 pages, not beyond).
 * Arguments and results are those of sv_sparse_decode.
 */
#define SV_STATIC_SCRATCH_BYTES (16u << 20)
int sv_sparse_decode_static_scratch(const sv_cache* cache, const void* q, int32_t num_q_heads,
                                    const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                                    int32_t max_pages, const int32_t* sel_idx, const int32_t* sel_cnt,
                                    int32_t budget_pages, float softmax_scale, void* out, float* lse,
                                    void* stream);

/*
 * sv_quest_decode_step -- one decode step in one call: build_decode_view
 * (page scores + top-K, exactly sv_quest_select) followed by attention over
 * the view (exactly sv_sparse_decode), the decode-time hooks of the
 * SparseEngine page ("method key points": query-relevant page selection
 * before attention, then attention over the selected pages only).  It
 * enqueues four kernels back to back with programmatic dependent launch:
 * page scores, top-K, split-K attention, log-sum-exp combine.
 *  - budget_pages >= 1 is the row length of sel_idx, as in sv_quest_select.
 *  - softmax_scale > 0, as in sv_sparse_decode.
 *  - workspace: sv_quest_decode_step_workspace_size(...) bytes, not shared
 *    with a call that may run at the same time; nothing in it needs to start
 *    at zero.
 *  - A q in page-locked host memory is first copied into the workspace by
 *    one small kernel (each of its bytes crosses the host link once; every
 *    scoring CTA of a request reads that request's query), and the
 *    kernels then read the copy.
 */
int sv_quest_decode_step(const sv_cache* cache, const void* q, int32_t num_q_heads,
                         const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                         int32_t max_pages, int32_t budget_pages, float softmax_scale,
                         int32_t* sel_idx, int32_t* sel_cnt, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of sv_quest_decode_step. */
size_t sv_quest_decode_step_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t max_pages, int32_t budget_pages);

/* Reads (and with reset != 0 clears) the current device's error word; the
 * read synchronises the device.  Returns SV_OK or SV_ERR_CUDA. */
int sv_get_device_error(uint32_t* flags, int reset);

const char* sv_status_string(int status);
int sv_version(void);   /* major * 10000 + minor * 100 + patch */

#ifdef __cplusplus
}
#endif

#endif /* SVQUEST_H */
