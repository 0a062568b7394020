// sv_quest_update_meta: append K/V rows into the paged pool and refresh the
// per-page, per-channel key min/max (the on_kv_stored hook of the
// "add-sparse-method" skill page, "Placement Rules" item 3).
#include "svq_common.cuh"

namespace svq {

SVQ_DEFINE_ERROR_WORD(read_error_meta)

// One warp per (token t, kv head h).  Lanes 0-15 copy the key row, lanes
// 16-31 the value row, 16 bytes each.  The warp of the last token of a run
// of consecutive tokens bound for one page also rebuilds that page's
// metadata for head h: lane l < 16 produces kmin of channels 8l..8l+7, lane
// l >= 16 kmax of channels 8(l-16)..; the run's first offset decides whether
// the stored min/max are kept (offset > 0) or restarted (offset 0).
__global__ void __launch_bounds__(256) append_kv_meta_kernel(
    __nv_bfloat16* __restrict__ k_pool, __nv_bfloat16* __restrict__ v_pool, __nv_bfloat16* __restrict__ meta,
    int64_t num_phys_pages, int num_kv_heads, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, const int32_t* __restrict__ slot_mapping, int64_t num_tokens) {
    const int lane = threadIdx.x & 31;
    const int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (item >= num_tokens * num_kv_heads) return;
    const int64_t t = item / num_kv_heads;
    const int h = static_cast<int>(item % num_kv_heads);
    const int64_t pool_slots = num_phys_pages * kPage;

    const int32_t slot = slot_mapping[t];
    if (slot < 0 || slot >= pool_slots) {
        if (lane == 0) svq_flag(SV_DEVERR_SLOT);
        return;
    }
    const int64_t page = slot / kPage;
    const int off = slot % kPage;
    const int chunk = lane & 15;

    // Row copy.
    {
        const __nv_bfloat16* src = (lane < 16 ? k_new : v_new) + (t * num_kv_heads + h) * kHeadDim + chunk * 8;
        __nv_bfloat16* dst = (lane < 16 ? k_pool : v_pool) +
                             ((page * num_kv_heads + h) * kPage + off) * kHeadDim + chunk * 8;
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    }

    // Is t the last token of its page's run in this call?
    if (t + 1 < num_tokens) {
        const int32_t nxt = slot_mapping[t + 1];
        if (nxt >= 0 && nxt / kPage == page) return;
    }
    // Walk back over the run (at most one page of tokens).
    int64_t first = t;
    while (first > 0 && t - first < kPage - 1) {
        const int32_t prev = slot_mapping[first - 1];
        const int32_t cur = slot_mapping[first];
        if (prev < 0 || prev / kPage != page || prev % kPage >= cur % kPage) break;
        --first;
    }
    const int first_off = slot_mapping[first] % kPage;
    const bool is_max = lane >= 16;
    __nv_bfloat162 acc[4];
    int64_t j = first;
    {
        uint4 w = *reinterpret_cast<const uint4*>(k_new + (j * num_kv_heads + h) * kHeadDim + chunk * 8);
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = p[i];
    }
    for (++j; j <= t; ++j) {
        uint4 w = *reinterpret_cast<const uint4*>(k_new + (j * num_kv_heads + h) * kHeadDim + chunk * 8);
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = is_max ? __hmax2(acc[i], p[i]) : __hmin2(acc[i], p[i]);
    }
    __nv_bfloat16* mdst = meta + ((page * num_kv_heads + h) * 2 + (is_max ? 1 : 0)) * kHeadDim + chunk * 8;
    if (first_off > 0) {
        uint4 w = *reinterpret_cast<const uint4*>(mdst);
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = is_max ? __hmax2(acc[i], p[i]) : __hmin2(acc[i], p[i]);
    }
    *reinterpret_cast<uint4*>(mdst) = *reinterpret_cast<const uint4*>(acc);
}

int launch_update_meta(const sv_cache* c, const void* k_new, const void* v_new, const int32_t* slot_mapping,
                       int64_t num_tokens, cudaStream_t stream) {
    const int64_t items = num_tokens * c->num_kv_heads;
    const int64_t blocks = (items * 32 + 255) / 256;
    if (blocks > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
    append_kv_meta_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<__nv_bfloat16*>(c->k_pool), static_cast<__nv_bfloat16*>(c->v_pool),
        static_cast<__nv_bfloat16*>(c->meta), c->num_phys_pages, c->num_kv_heads,
        static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new), slot_mapping,
        num_tokens);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace svq
