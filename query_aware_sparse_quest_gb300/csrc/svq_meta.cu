// sv_quest_update_meta: append K/V rows into the paged pool and refresh the
// per-page, per-channel key min/max (the on_kv_stored hook of the
// "add-sparse-method" skill page, "Placement Rules" item 3).
#include "svq_common.cuh"

namespace svq {

SVQ_DEFINE_ERROR_WORD(read_error_meta)

// One warp per (token t, kv head h); only the warps whose token starts a
// page run (the tokens bound for one page, consecutive in the token list with
// increasing offsets, at most 16) do work, for the whole run:
//  1. lanes 1..15 look at tokens t+1 .. t+15 and a ballot gives the run
//     length R (each further token must be in the same page, one offset on);
//  2. the run's K and V rows are loaded at once (lane l: 16-byte chunk l % 16
//     of rows l / 16, l / 16 + 2, ...: 8 loads of K and 8 of V in flight) and
//     stored to the pool (bf16), or coded (fp8: each half-warp takes a row's
//     max |x| by 4 shuffles, stores s = max / 448 and e4m3(x / s), IEEE
//     division, round to nearest even, saturating);
//  3. the same registers give the run's per-channel key min / max (one
//     shuffle joins the two half-warps); a run that starts past offset 0
//     folds in the stored min / max, one starting at offset 0 replaces them.
// The warps of the run's other tokens return at once.
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
    auto in_pool = [&](int32_t sl) { return sl >= 0 && sl < pool_slots; };

    const int32_t slot = slot_mapping[t];
    if (!in_pool(slot)) {
        if (lane == 0) svq_flag(SV_DEVERR_SLOT);
        return;
    }
    const int64_t page = slot / kPage;
    const int off = slot % kPage;
    if (t > 0) {   // token t continues the previous token's run: that run's warp does the work
        const int32_t prev = slot_mapping[t - 1];
        if (in_pool(prev) && prev / kPage == page && prev % kPage < off) return;
    }
    // 1. run length.  Lane i in 1..15: token t + i continues the run from t + i - 1.
    int32_t si = slot, sp = 0;   // lane i < 16: the slot of token t + i
    if (lane >= 1 && lane < kPage && t + lane < num_tokens) {
        si = slot_mapping[t + lane];
        sp = slot_mapping[t + lane - 1];
    }
    const bool cont = lane >= 1 && lane < kPage && t + lane < num_tokens && in_pool(si) && si / kPage == page &&
                      in_pool(sp) && sp / kPage == page && sp % kPage < si % kPage;
    const uint32_t mask = __ballot_sync(0xffffffffu, cont);
    const int R = __ffs(~(mask >> 1));   // 1 + the leading run of continuing tokens

    // 2. rows: lane l moves chunk c = l % 16 of rows r = l / 16 + 2 k.
    const int c = lane & 15, half = lane >> 4;
    uint4 kw[kPage / 2], vw[kPage / 2];
#pragma unroll
    for (int k = 0; k < kPage / 2; ++k) {
        const int r = half + 2 * k;
        kw[k] = vw[k] = make_uint4(0u, 0u, 0u, 0u);
        if (r < R) {
            const int64_t src = ((t + r) * num_kv_heads + h) * kHeadDim + c * 8;
            kw[k] = *reinterpret_cast<const uint4*>(k_new + src);
            vw[k] = *reinterpret_cast<const uint4*>(v_new + src);
        }
    }
#pragma unroll
    for (int k = 0; k < kPage / 2; ++k) {
        const int r = half + 2 * k;
        if (r >= (R + 1) / 2 * 2) break;   // warp-uniform: both half-warps stay for the shuffles
        const bool live = r < R;
        const int off_r = __shfl_sync(0xffffffffu, si, r & 31) % kPage;   // row r's own offset in the page
        const int64_t row = (page * num_kv_heads + h) * kPage + off_r;
        if (!FP8) {
            if (live) {
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(k_pool) + row * kHeadDim + c * 8) = kw[k];
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(v_pool) + row * kHeadDim + c * 8) = vw[k];
            }
        } else {
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint4 w = which ? vw[k] : kw[k];
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
                if (live) {
                    unsigned char* dst = static_cast<unsigned char*>(which ? v_pool : k_pool) + row * kHeadDim + c * 8;
                    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
                    if (c == 0) (which ? v_scale : k_scale)[row] = sc;
                }
            }
        }
    }

    // 3. the run's key min / max per channel (bf16 min / max are exact).
    __nv_bfloat162 mn[4], mx[4];
    {
        const __nv_bfloat162* p0 = reinterpret_cast<const __nv_bfloat162*>(&kw[0]);
#pragma unroll
        for (int i = 0; i < 4; ++i) mn[i] = mx[i] = p0[i];   // row `half` (R >= 2 when half == 1 uses it)
    }
    const bool have = half < R;
#pragma unroll
    for (int k = 1; k < kPage / 2; ++k) {
        if (half + 2 * k < R) {
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&kw[k]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mn[i] = __hmin2(mn[i], p[i]);
                mx[i] = __hmax2(mx[i], p[i]);
            }
        }
    }
    // Join the half-warps: lane c and lane c + 16 hold the same channels.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t a = *reinterpret_cast<uint32_t*>(&mn[i]), b = *reinterpret_cast<uint32_t*>(&mx[i]);
        const uint32_t oa = __shfl_xor_sync(0xffffffffu, a, 16), ob = __shfl_xor_sync(0xffffffffu, b, 16);
        const bool other_has = (half ^ 1) < R;
        if (other_has && have) {
            mn[i] = __hmin2(mn[i], *reinterpret_cast<const __nv_bfloat162*>(&oa));
            mx[i] = __hmax2(mx[i], *reinterpret_cast<const __nv_bfloat162*>(&ob));
        } else if (other_has) {
            mn[i] = *reinterpret_cast<const __nv_bfloat162*>(&oa);
            mx[i] = *reinterpret_cast<const __nv_bfloat162*>(&ob);
        }
    }
    // Lanes 0-15 write kmin of chunk c, lanes 16-31 kmax of chunk c.
    const bool is_max = half == 1;
    __nv_bfloat162 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = is_max ? mx[i] : mn[i];
    __nv_bfloat16* mdst = meta + ((page * num_kv_heads + h) * 2 + (is_max ? 1 : 0)) * kHeadDim + c * 8;
    if (off > 0) {
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
