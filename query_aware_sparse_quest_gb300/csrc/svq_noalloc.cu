// sv_sparse_decode_static_scratch: sparse decode whose scratch (the split-K
// partials) lives in a fixed device array compiled into this library, for
// callers that are not allowed to allocate device memory themselves.
//
// Callers of this kind include plugins hosted inside a framework that owns
// every device allocation through its own pool and forbids calls to
// cudaMalloc, and serving loops that have pre-reserved nearly all of HBM
// for the KV cache and must not grow or fragment it at decode time.  Such
// callers still provide inputs and outputs; only the scratch comes from the
// library.
#include <mutex>

#include "svq_common.cuh"

namespace svq {

// Largest scratch this entry point can use: 16 MiB.  Every GPU that loads the
// library reserves this array until the process exits.
static_assert(SV_STATIC_SCRATCH_BYTES == (16u << 20), "header and array size must agree");
static __device__ __align__(256) unsigned char g_decode_scratch[SV_STATIC_SCRATCH_BYTES];

namespace {
std::mutex g_setup_mutex;
void* g_scratch_ptr[64] = {};

// The array's name is a host-side stand-in in host code, not a device
// address: ask the runtime for the current device's address of it, once per
// device, with that device current.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (dev >= 0 && dev < 64 && g_scratch_ptr[dev]) {
        *out = g_scratch_ptr[dev];
        return SV_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return SV_ERR_CUDA;
    if (dev >= 0 && dev < 64) g_scratch_ptr[dev] = p;
    *out = p;
    return SV_OK;
}
}  // namespace
}  // namespace svq

extern "C" int sv_sparse_decode_static_scratch(const sv_cache* cache, const void* q, int32_t num_q_heads,
                                               const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                                               int32_t max_pages, const int32_t* sel_idx, const int32_t* sel_cnt,
                                               int32_t budget_pages, float softmax_scale, void* out, float* lse,
                                               void* stream) {
    if (!cache || num_q_heads < 1 || batch < 1 || max_pages < 1) return SV_ERR_INVALID_ARG;
    const int32_t pages = sel_idx ? budget_pages : max_pages;
    if (pages < 1) return SV_ERR_INVALID_ARG;
    // Reject, before touching the device, any problem whose partials could
    // exceed the array (the bound is the one sv_sparse_decode_workspace_size
    // reports).
    const size_t need = sv_sparse_decode_workspace_size(batch, num_q_heads, cache->num_kv_heads, pages);
    if (need == 0) return SV_ERR_INVALID_ARG;
    if (need > SV_STATIC_SCRATCH_BYTES) return SV_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int st = svq::scratch_address(&scratch);
    if (st != SV_OK) return st;
    // Every split writes its own partial before the combine reads it, so
    // nothing in the array needs to start at zero.
    return sv_sparse_decode(cache, q, num_q_heads, page_table, seq_lens, batch, max_pages, sel_idx, sel_cnt,
                            budget_pages, softmax_scale, out, lse, scratch, SV_STATIC_SCRATCH_BYTES, stream);
}
