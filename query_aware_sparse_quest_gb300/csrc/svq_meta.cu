// sv_quest_update_meta: append K/V rows into the paged pool and refresh the
// per-page, per-channel key min/max (the on_kv_stored hook of the
// "add-sparse-method" skill page, "Placement Rules" item 3).
#include "svq_common.cuh"

namespace svq {

SVQ_DEFINE_ERROR_WORD(read_error_meta)

// One warp per (token t, kv head h).  Lanes 0-15 copy the key row, lanes
// 16-31 the value row, 16 bytes (8 values) each.  FP8 pools: each half-warp
// takes the row's max |x| (4 shuffles), stores the fp32 scale s = max / 448
// and the row's codes e4m3(x / s) (IEEE division, round to nearest even,
// saturating), 8 bytes per lane.  The warp of the last token of a run
// of consecutive tokens bound for one page also rebuilds that page's
// metadata for head h: lane l < 16 produces kmin of channels 8l..8l+7, lane
// l >= 16 kmax of channels 8(l-16)..; the run's first offset decides whether
// the stored min/max are kept (offset > 0) or restarted (offset 0).
template <bool FP8>
__global__ void __launch_bounds__(256) append_kv_meta_kernel(
    void* __restrict__ k_pool, void* __restrict__ v_pool, __nv_bfloat16* __restrict__ meta,
    float* __restrict__ k_scale, float* __restrict__ v_scale,
    int64_t num_phys_pages, int num_kv_heads, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, const int32_t* __restrict__ slot_mapping, int64_t num_tokens) {
    const int lane = threadIdx.x & 31;
    const int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    // The kernel before may still read the pool and the metadata: wait for
    // it before writing.  The scoring kernel that usually follows may then
    // be scheduled and load its page-table entries and query meanwhile.
    pdl_wait();
    pdl_launch_dependents();
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

    // Row copy (bf16) or row coding (fp8).
    {
        const __nv_bfloat16* src = (lane < 16 ? k_new : v_new) + (t * num_kv_heads + h) * kHeadDim + chunk * 8;
        const int64_t row = (page * num_kv_heads + h) * kPage + off;
        const uint4 w = *reinterpret_cast<const uint4*>(src);
        if (!FP8) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(lane < 16 ? k_pool : v_pool) + row * kHeadDim + chunk * 8;
            *reinterpret_cast<uint4*>(dst) = w;
        } else {
            const uint32_t x[4] = {w.x, w.y, w.z, w.w};
            float f[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[2 * e] = bf16lo(x[e]);
                f[2 * e + 1] = bf16hi(x[e]);
            }
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float sc = __fdiv_rn(amax, 448.f);
            uint32_t packed[2] = {0u, 0u};
            if (sc > 0.f) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t code = __nv_cvt_float_to_fp8(__fdiv_rn(f[e], sc), __NV_SATFINITE, __NV_E4M3);
                    packed[e >> 2] |= code << (8 * (e & 3));
                }
            }
            unsigned char* dst = static_cast<unsigned char*>(lane < 16 ? k_pool : v_pool) + row * kHeadDim + chunk * 8;
            *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
            if (chunk == 0) (lane < 16 ? k_scale : v_scale)[row] = sc;
        }
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
    const auto kn = static_cast<const __nv_bfloat16*>(k_new);
    const auto vn = static_cast<const __nv_bfloat16*>(v_new);
    auto* meta = static_cast<__nv_bfloat16*>(c->meta);
    cudaError_t e;
    if (c->kv_format == SV_KV_FP8_E4M3)
        e = launch_pdl(append_kv_meta_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                       c->k_pool, c->v_pool, meta, static_cast<float*>(c->k_scale), static_cast<float*>(c->v_scale),
                       c->num_phys_pages, c->num_kv_heads, kn, vn, slot_mapping, num_tokens);
    else
        e = launch_pdl(append_kv_meta_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                       c->k_pool, c->v_pool, meta, static_cast<float*>(nullptr), static_cast<float*>(nullptr),
                       c->num_phys_pages, c->num_kv_heads, kn, vn, slot_mapping, num_tokens);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace svq
