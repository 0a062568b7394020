// C ABI of libsvquest.so (include/svquest.h): host-side argument checks,
// launch-shape choices and dispatch to the kernels, plus the small kernel that
// stages a host-resident query for the one-call step.  Nothing here
// allocates, frees or synchronises, except sv_get_device_error which reads
// device words.
#include <climits>

#include "svq_common.cuh"

namespace svq {
int read_error_meta(uint32_t* flags, int reset);
int read_error_select(uint32_t* flags, int reset);
int read_error_decode(uint32_t* flags, int reset);
int launch_update_meta(const sv_cache* c, const void* k_new, const void* v_new, const int32_t* slot_mapping,
                       int64_t num_tokens, cudaStream_t stream);
int launch_score(const sv_cache* c, const void* q, int num_q_heads, const int32_t* page_table,
                 const int32_t* seq_lens, int batch, int max_pages, bool per_q_head, int sink, int window,
                 float* scores, int sm_count, cudaStream_t stream, int q_after_wait);
int launch_topk(const float* scores, const int32_t* seq_lens, int batch, int num_kv_heads, int max_pages,
                int budget_pages, int32_t* sel_idx, int32_t* sel_cnt, cudaStream_t stream);
int launch_decode(const sv_cache* c, const void* q, int num_q_heads, const int32_t* page_table,
                  const int32_t* seq_lens, int batch, int max_pages, const int32_t* sel_idx,
                  const int32_t* sel_cnt, int budget_pages, bool per_q_head, float softmax_scale, void* out,
                  float* lse, void* workspace, size_t workspace_bytes, int sm_count, cudaStream_t stream);
int decode_max_splits(int pages);
size_t decode_workspace_bytes(int batch, int num_q_heads, int splits);
int read_error_decode_fp8(uint32_t* flags, int reset);

constexpr int kMaxTopkPages = 32768;

namespace {

int sm_count_of_current_device(int* out) {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    if (dev >= 0 && dev < 64) {
        const int c = cached[dev].load(std::memory_order_acquire);
        if (c > 0) {
            *out = c;
            return SV_OK;
        }
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return SV_ERR_CUDA;
    if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_release);
    *out = n;
    return SV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cache(const sv_cache* c) {
    if (!c || !c->k_pool || !c->v_pool || !c->meta) return SV_ERR_INVALID_ARG;
    if (c->num_phys_pages < 1 || c->num_kv_heads < 1) return SV_ERR_INVALID_ARG;
    if (c->num_phys_pages > INT_MAX) return SV_ERR_UNSUPPORTED;
    if (c->page_size != kPage || c->head_dim != kHeadDim) return SV_ERR_UNSUPPORTED;
    if (!aligned16(c->k_pool) || !aligned16(c->v_pool) || !aligned16(c->meta)) return SV_ERR_INVALID_ARG;
    if (c->kv_format != SV_KV_BF16 && c->kv_format != SV_KV_FP8_E4M3) return SV_ERR_UNSUPPORTED;
    if (c->kv_format == SV_KV_FP8_E4M3 && (!c->k_scale || !c->v_scale || !aligned16(c->k_scale) ||
                                           !aligned16(c->v_scale)))
        return SV_ERR_INVALID_ARG;
    return SV_OK;
}

int check_heads(const sv_cache* c, int num_q_heads) {
    if (num_q_heads < 1 || num_q_heads % c->num_kv_heads != 0) return SV_ERR_INVALID_ARG;
    if (num_q_heads / c->num_kv_heads > kMaxGroup) return SV_ERR_UNSUPPORTED;
    return SV_OK;
}

int check_batch(const void* q, const int32_t* page_table, const int32_t* seq_lens, int batch, int max_pages) {
    if (!q || !page_table || !seq_lens) return SV_ERR_INVALID_ARG;
    if (batch < 1 || max_pages < 1) return SV_ERR_INVALID_ARG;
    if (batch > 65535) return SV_ERR_UNSUPPORTED;
    if (!aligned16(q)) return SV_ERR_INVALID_ARG;
    return SV_OK;
}

size_t scores_bytes(int batch, int rows_per_req, int max_pages) {
    return (static_cast<size_t>(batch) * rows_per_req * max_pages * sizeof(float) + 255) / 256 * 256;
}
size_t query_bytes(int batch, int num_q_heads) {
    return (static_cast<size_t>(batch) * num_q_heads * 128 * 2 + 255) / 256 * 256;
}

// True when p is page-locked host memory.  Device, managed and unregistered
// memory answer false; a failed query also answers false and its error is
// cleared, so that it does not surface in the caller's next error check.
bool is_pinned_host(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

// Copies a query that lives in page-locked host memory into the workspace,
// so that each of its bytes crosses the host link once (the scoring kernel
// reads a request's query from each of that request's CTAs).  The loads come
// before the wait on the kernel before, which may still read the previous
// copy; the stores come after it.
__global__ void __launch_bounds__(256) stage_query_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                          int64_t n16) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const uint4 v = i < n16 ? src[i] : make_uint4(0u, 0u, 0u, 0u);
    svq::pdl_wait();
    svq::pdl_launch_dependents();
    if (i < n16) dst[i] = v;
}

const sv_quest_opts kBaseOpts = {0, 0, 0, 0, 0};

int check_opts(const sv_quest_opts* o) {
    if (o->per_q_head != 0 && o->per_q_head != 1) return SV_ERR_INVALID_ARG;
    if (o->sink_pages < 0 || o->window_pages < 0 || o->layer < 0 || o->dense_layers < 0) return SV_ERR_INVALID_ARG;
    return SV_OK;
}

int rows_per_request(const sv_cache* c, int num_q_heads, const sv_quest_opts* o) {
    return o->per_q_head ? num_q_heads : c->num_kv_heads;
}

int select_impl(const sv_cache* cache, const void* q, int32_t num_q_heads, const int32_t* page_table,
                const int32_t* seq_lens, int32_t batch, int32_t max_pages, int32_t budget_pages,
                const sv_quest_opts* opts, int32_t* sel_idx, int32_t* sel_cnt, float* scores_out, void* workspace,
                size_t workspace_bytes, void* stream) {
    int st = check_cache(cache);
    if (st) return st;
    if ((st = check_heads(cache, num_q_heads))) return st;
    if ((st = check_batch(q, page_table, seq_lens, batch, max_pages))) return st;
    if ((st = check_opts(opts))) return st;
    if (!sel_idx || !sel_cnt || budget_pages < 1) return SV_ERR_INVALID_ARG;
    if (max_pages > kMaxTopkPages) return SV_ERR_UNSUPPORTED;
    if (opts->layer < opts->dense_layers) return SV_OK;   // dense layer: no selection
    const int rows = rows_per_request(cache, num_q_heads, opts);
    float* scores = scores_out;
    if (!scores) {
        if (!workspace || workspace_bytes < scores_bytes(batch, rows, max_pages)) return SV_ERR_WORKSPACE;
        scores = static_cast<float*>(workspace);
    }
    int sms = 0;
    if ((st = sm_count_of_current_device(&sms))) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = launch_score(cache, q, num_q_heads, page_table, seq_lens, batch, max_pages, opts->per_q_head != 0,
                           opts->sink_pages, opts->window_pages, scores, sms, s, 0)))
        return st;
    return launch_topk(scores, seq_lens, batch, rows, max_pages, budget_pages, sel_idx, sel_cnt, s);
}

int decode_impl(const sv_cache* cache, const void* q, int32_t num_q_heads, const int32_t* page_table,
                const int32_t* seq_lens, int32_t batch, int32_t max_pages, const int32_t* sel_idx,
                const int32_t* sel_cnt, int32_t budget_pages, const sv_quest_opts* opts, float softmax_scale,
                void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    int st = check_cache(cache);
    if (st) return st;
    if ((st = check_heads(cache, num_q_heads))) return st;
    if ((st = check_batch(q, page_table, seq_lens, batch, max_pages))) return st;
    if ((st = check_opts(opts))) return st;
    if (!out || !lse || !aligned16(out)) return SV_ERR_INVALID_ARG;
    if (opts->layer < opts->dense_layers) sel_idx = nullptr;   // dense layer: every page
    if (sel_idx && (!sel_cnt || budget_pages < 1)) return SV_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || softmax_scale == INFINITY) return SV_ERR_INVALID_ARG;
    const int rows = sel_idx ? rows_per_request(cache, num_q_heads, opts) : cache->num_kv_heads;
    if (static_cast<int64_t>(batch) * rows > 65535) return SV_ERR_UNSUPPORTED;
    if (!workspace) return SV_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SV_ERR_INVALID_ARG;   // partials are read 16 bytes at a time
    int sms = 0;
    if ((st = sm_count_of_current_device(&sms))) return st;
    return launch_decode(cache, q, num_q_heads, page_table, seq_lens, batch, max_pages, sel_idx, sel_cnt,
                         budget_pages, opts->per_q_head != 0, softmax_scale, out, lse, workspace, workspace_bytes,
                         sms, static_cast<cudaStream_t>(stream));
}


}  // namespace
}  // namespace svq

using namespace svq;

extern "C" {

int sv_quest_update_meta(const sv_cache* cache, const void* k_new, const void* v_new,
                         const int32_t* slot_mapping, int64_t num_tokens, void* stream) {
    int st = check_cache(cache);
    if (st) return st;
    if (num_tokens < 0) return SV_ERR_INVALID_ARG;
    if (num_tokens == 0) return SV_OK;
    if (!k_new || !v_new || !slot_mapping) return SV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return SV_ERR_INVALID_ARG;
    return launch_update_meta(cache, k_new, v_new, slot_mapping, num_tokens, static_cast<cudaStream_t>(stream));
}

int sv_quest_score(const sv_cache* cache, const void* q, int32_t num_q_heads, const int32_t* page_table,
                   const int32_t* seq_lens, int32_t batch, int32_t max_pages, float* scores, void* stream) {
    int st = check_cache(cache);
    if (st) return st;
    if ((st = check_heads(cache, num_q_heads))) return st;
    if ((st = check_batch(q, page_table, seq_lens, batch, max_pages))) return st;
    if (!scores) return SV_ERR_INVALID_ARG;
    int sms = 0;
    if ((st = sm_count_of_current_device(&sms))) return st;
    return launch_score(cache, q, num_q_heads, page_table, seq_lens, batch, max_pages, false, 0, 0, scores, sms,
                        static_cast<cudaStream_t>(stream), 0);
}

int sv_quest_topk(const float* scores, const int32_t* seq_lens, int32_t batch, int32_t num_kv_heads,
                  int32_t max_pages, int32_t budget_pages, int32_t* sel_idx, int32_t* sel_cnt, void* stream) {
    if (!scores || !seq_lens || !sel_idx || !sel_cnt) return SV_ERR_INVALID_ARG;
    if (batch < 1 || num_kv_heads < 1 || max_pages < 1 || budget_pages < 1) return SV_ERR_INVALID_ARG;
    if (max_pages > kMaxTopkPages) return SV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(batch) * num_kv_heads > INT_MAX) return SV_ERR_UNSUPPORTED;
    return launch_topk(scores, seq_lens, batch, num_kv_heads, max_pages, budget_pages, sel_idx, sel_cnt,
                       static_cast<cudaStream_t>(stream));
}

size_t sv_quest_select_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t max_pages) {
    if (batch < 1 || num_kv_heads < 1 || max_pages < 1) return 0;
    return scores_bytes(batch, num_kv_heads, max_pages);
}

int sv_quest_select(const sv_cache* cache, const void* q, int32_t num_q_heads, const int32_t* page_table,
                    const int32_t* seq_lens, int32_t batch, int32_t max_pages, int32_t budget_pages,
                    int32_t* sel_idx, int32_t* sel_cnt, float* scores_out, void* workspace,
                    size_t workspace_bytes, void* stream) {
    return select_impl(cache, q, num_q_heads, page_table, seq_lens, batch, max_pages, budget_pages, &kBaseOpts,
                       sel_idx, sel_cnt, scores_out, workspace, workspace_bytes, stream);
}

int sv_quest_select_ex(const sv_cache* cache, const void* q, int32_t num_q_heads, const int32_t* page_table,
                       const int32_t* seq_lens, int32_t batch, int32_t max_pages, int32_t budget_pages,
                       const sv_quest_opts* opts, int32_t* sel_idx, int32_t* sel_cnt, float* scores_out,
                       void* workspace, size_t workspace_bytes, void* stream) {
    return select_impl(cache, q, num_q_heads, page_table, seq_lens, batch, max_pages, budget_pages,
                       opts ? opts : &kBaseOpts, sel_idx, sel_cnt, scores_out, workspace, workspace_bytes, stream);
}

size_t sv_quest_select_ex_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t max_pages, const sv_quest_opts* opts) {
    if (batch < 1 || num_q_heads < 1 || num_kv_heads < 1 || max_pages < 1) return 0;
    const bool per_head = opts && opts->per_q_head;
    return scores_bytes(batch, per_head ? num_q_heads : num_kv_heads, max_pages);
}

size_t sv_sparse_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t pages) {
    if (batch < 1 || num_q_heads < 1 || num_kv_heads < 1 || pages < 1) return 0;
    return decode_workspace_bytes(batch, num_q_heads, decode_max_splits(pages));
}

int sv_sparse_decode(const sv_cache* cache, const void* q, int32_t num_q_heads, const int32_t* page_table,
                     const int32_t* seq_lens, int32_t batch, int32_t max_pages, const int32_t* sel_idx,
                     const int32_t* sel_cnt, int32_t budget_pages, float softmax_scale, void* out, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream) {
    return decode_impl(cache, q, num_q_heads, page_table, seq_lens, batch, max_pages, sel_idx, sel_cnt, budget_pages,
                       &kBaseOpts, softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

int sv_sparse_decode_ex(const sv_cache* cache, const void* q, int32_t num_q_heads, const int32_t* page_table,
                        const int32_t* seq_lens, int32_t batch, int32_t max_pages, const int32_t* sel_idx,
                        const int32_t* sel_cnt, int32_t budget_pages, const sv_quest_opts* opts,
                        float softmax_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                        void* stream) {
    return decode_impl(cache, q, num_q_heads, page_table, seq_lens, batch, max_pages, sel_idx, sel_cnt, budget_pages,
                       opts ? opts : &kBaseOpts, softmax_scale, out, lse, workspace, workspace_bytes, stream);
}

size_t sv_quest_decode_step_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t max_pages, int32_t budget_pages) {
    if (batch < 1 || num_q_heads < 1 || num_kv_heads < 1 || max_pages < 1 || budget_pages < 1) return 0;
    // Scores, room for a copy of a host-resident query, split-K partials.
    return scores_bytes(batch, num_kv_heads, max_pages) + query_bytes(batch, num_q_heads) +
           decode_workspace_bytes(batch, num_q_heads, decode_max_splits(budget_pages));
}

}  // extern "C"

namespace {
int step_checks(const sv_cache* cache, const void* q, int32_t num_q_heads, const int32_t* page_table,
                const int32_t* seq_lens, int32_t batch, int32_t max_pages, int32_t budget_pages, float softmax_scale,
                const int32_t* sel_idx, const int32_t* sel_cnt, const void* out, const float* lse,
                const void* workspace, size_t workspace_bytes) {
    int st = check_cache(cache);
    if (st) return st;
    if ((st = check_heads(cache, num_q_heads))) return st;
    if ((st = check_batch(q, page_table, seq_lens, batch, max_pages))) return st;
    if (!sel_idx || !sel_cnt || !out || !lse || budget_pages < 1 || !aligned16(out)) return SV_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || softmax_scale == INFINITY) return SV_ERR_INVALID_ARG;
    if (max_pages > kMaxTopkPages) return SV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(batch) * cache->num_kv_heads > 65535) return SV_ERR_UNSUPPORTED;
    if (!workspace ||
        workspace_bytes < sv_quest_decode_step_workspace_size(batch, num_q_heads, cache->num_kv_heads, max_pages,
                                                              budget_pages))
        return SV_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SV_ERR_INVALID_ARG;   // a staged query and the partials are read 16 bytes at a time
    return SV_OK;
}
}  // namespace

extern "C" {

int sv_quest_decode_step(const sv_cache* cache, const void* q, int32_t num_q_heads, const int32_t* page_table,
                         const int32_t* seq_lens, int32_t batch, int32_t max_pages, int32_t budget_pages,
                         float softmax_scale, int32_t* sel_idx, int32_t* sel_cnt, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, void* stream) {
    int st = step_checks(cache, q, num_q_heads, page_table, seq_lens, batch, max_pages, budget_pages, softmax_scale,
                         sel_idx, sel_cnt, out, lse, workspace, workspace_bytes);
    if (st) return st;
    int sms = 0;
    if ((st = sm_count_of_current_device(&sms))) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Workspace: scores, a copy of the query when it lives in page-locked
    // host memory, then the split-K partials.
    const int hkv = cache->num_kv_heads;
    const size_t sb = scores_bytes(batch, hkv, max_pages);
    const size_t qb = query_bytes(batch, num_q_heads);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    float* scores = reinterpret_cast<float*>(ws);
    const void* qd = q;
    const bool staged = is_pinned_host(q);
    if (staged) {
        const int64_t n16 = static_cast<int64_t>(batch) * num_q_heads * 128 * 2 / 16;
        if (launch_pdl(stage_query_kernel, dim3(static_cast<unsigned>((n16 + 255) / 256)), dim3(256), 0, s,
                       static_cast<const uint4*>(q), reinterpret_cast<uint4*>(ws + sb), n16) != cudaSuccess)
            return SV_ERR_CUDA;
        qd = ws + sb;
    }
    if ((st = launch_score(cache, qd, num_q_heads, page_table, seq_lens, batch, max_pages, false, 0, 0, scores, sms, s,
                           staged ? 1 : 0)))
        return st;
    if ((st = launch_topk(scores, seq_lens, batch, hkv, max_pages, budget_pages, sel_idx, sel_cnt, s)))
        return st;
    return launch_decode(cache, qd, num_q_heads, page_table, seq_lens, batch, max_pages, sel_idx, sel_cnt,
                         budget_pages, false, softmax_scale, out, lse, ws + sb + qb, workspace_bytes - sb - qb, sms, s);
}

int sv_get_device_error(uint32_t* flags, int reset) {
    if (!flags) return SV_ERR_INVALID_ARG;
    *flags = 0;
    int st;
    if ((st = read_error_meta(flags, reset))) return st;
    if ((st = read_error_select(flags, reset))) return st;
    if ((st = read_error_decode_fp8(flags, reset))) return st;
    return read_error_decode(flags, reset);
}

const char* sv_status_string(int status) {
    switch (status) {
        case SV_OK: return "SV_OK";
        case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG: null pointer, misaligned buffer or bad size";
        case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED: geometry not supported by this build";
        case SV_ERR_WORKSPACE: return "SV_ERR_WORKSPACE: workspace missing or too small";
        case SV_ERR_CUDA: return "SV_ERR_CUDA: CUDA launch or device query failed";
        default: return "unknown sv_status";
    }
}

int sv_version(void) { return 100; }

}  // extern "C"
