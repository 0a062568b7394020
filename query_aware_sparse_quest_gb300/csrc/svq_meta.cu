// sv_quest_update_meta: append K/V rows into the paged pool and refresh the
// per-page, per-channel key min/max (the on_kv_stored hook of the
// "add-sparse-method" skill page, "Placement Rules" item 3).
#include "svq_common.cuh"

namespace svq {

SVQ_DEFINE_ERROR_WORD(read_error_meta)

// Two warps per (window of `win` tokens, kv head h), win = 1 or 16: one for
// the keys, one for the values.  A page run is the tokens bound for one page,
// consecutive in the token list with increasing offsets (at most 16); each
// warp handles, one after another, its side of every run that starts in its
// window:
//  1. lane i loads the slot of token t0 + i (i < 32: the window and what
//     follows it, since a run starting in the window may go on for 15 more
//     tokens); a token continues a run when its predecessor is in the pool,
//     in the same page, at a lower offset; a ballot gives the runs that start
//     in the window and each run's length;
//  2. the run's rows are moved (append_run);
//  3. the key warp takes the run's per-channel key min / max from the same
//     registers (one shuffle joins the two half-warps); a run that starts
//     past offset 0 folds in the stored min / max, one starting at offset 0
//     replaces them.
// Long calls (a prefill chunk of page-aligned consecutive slots: one run per
// 16-token window) take win = 16, so every warp of the grid has a run; short
// ones (a decode step's one token per request, each its own run) take win = 1,
// one warp pair per token, so that their runs proceed side by side.
// One bulk copy (TMA) shared -> global, waited for in full, so that the
// shared source may be reused and the rows are written when the CTA retires.
__device__ __forceinline__ void bulk_store_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Lane-wise min / max of two bf16 pairs held in 32-bit words (the
// instructions behind __hmin2 / __hmax2; bf16 min / max are exact).
__device__ __forceinline__ uint32_t min_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// One side (keys, or values) of one run: the rows are loaded at once (lane
// l: 16-byte chunk l % 16 of rows l / 16, l / 16 + 2, ...: 8 loads in
// flight) and stored to the pool (bf16), or coded (fp8: each half-warp takes
// a row's max |x| by 4 shuffles, stores s = max / 448 and e4m3(x / s), IEEE
// division, round to nearest even, saturating).  The key side then refreshes
// the page's min / max from the same registers.
template <bool FP8>
__device__ __forceinline__ void append_run(void* __restrict__ pool, float* __restrict__ scale,
                                           __nv_bfloat16* __restrict__ meta, bool is_key, int num_kv_heads, int h,
                                           const __nv_bfloat16* __restrict__ rows_new, int64_t t, int R, int32_t si,
                                           int first, const uint4* staged) {
    const int lane = threadIdx.x & 31;
    const int32_t slot = __shfl_sync(0xffffffffu, si, first);
    const int64_t page = slot / kPage;
    const int off = slot % kPage;
    const int c = lane & 15, half = lane >> 4;
    uint4 kw[kPage / 2];
#pragma unroll
    for (int k = 0; k < kPage / 2; ++k) {
        const int r = half + 2 * k;
        kw[k] = make_uint4(0u, 0u, 0u, 0u);
        if (r < R)
            kw[k] = staged ? staged[32 * k]
                           : *reinterpret_cast<const uint4*>(rows_new + ((t + r) * num_kv_heads + h) * kHeadDim + c * 8);
    }
    // A whole page from offset 0 with its rows staged in shared memory (row
    // r at byte 256 r: the staging layout is row-major): one bulk store.
    const bool whole = !FP8 && staged && R == kPage && off == 0;
    if (whole) {
        fence_proxy_async_smem();   // this lane's staged rows, for the bulk copy engine
        __syncwarp();
        if (lane == 0)
            bulk_store_s2g(static_cast<__nv_bfloat16*>(pool) + (page * num_kv_heads + h) * kPage * kHeadDim,
                           smem_addr(staged - lane), kPage * kHeadDim * 2);
        __syncwarp();
    }
#pragma unroll
    for (int k = 0; k < kPage / 2; ++k) {
        if (whole) break;
        const int r = half + 2 * k;
        if (r >= (R + 1) / 2 * 2) break;   // warp-uniform: both half-warps stay for the shuffles
        const bool live = r < R;
        const int off_r = __shfl_sync(0xffffffffu, si, (first + r) & 31) % kPage;   // row r's own offset
        const int64_t row = (page * num_kv_heads + h) * kPage + off_r;
        if (!FP8) {
            if (live) *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(pool) + row * kHeadDim + c * 8) = kw[k];
        } else {
            const uint32_t x[4] = {kw[k].x, kw[k].y, kw[k].z, kw[k].w};
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
                unsigned char* dst = static_cast<unsigned char*>(pool) + row * kHeadDim + c * 8;
                *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
                if (c == 0) scale[row] = sc;
            }
        }
    }
    if (!is_key) return;

    // The run's key min / max per channel.
    uint32_t mn[4], mx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) mn[i] = mx[i] = word_of(kw[0], i);   // row `half` (R >= 2 when half == 1 uses it)
    const bool have = half < R;
#pragma unroll
    for (int k = 1; k < kPage / 2; ++k) {
        if (half + 2 * k < R) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mn[i] = min_bf16x2(mn[i], word_of(kw[k], i));
                mx[i] = max_bf16x2(mx[i], word_of(kw[k], i));
            }
        }
    }
    // Join the half-warps: lane c and lane c + 16 hold the same channels.
    const bool other_has = (half ^ 1) < R;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t oa = __shfl_xor_sync(0xffffffffu, mn[i], 16);
        const uint32_t ob = __shfl_xor_sync(0xffffffffu, mx[i], 16);
        if (other_has && have) {
            mn[i] = min_bf16x2(mn[i], oa);
            mx[i] = max_bf16x2(mx[i], ob);
        } else if (other_has) {
            mn[i] = oa;
            mx[i] = ob;
        }
    }
    // Lanes 0-15 write kmin of chunk c, lanes 16-31 kmax of chunk c.
    const bool is_max = half == 1;
    uint32_t acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = is_max ? mx[i] : mn[i];
    __nv_bfloat16* mdst = meta + ((page * num_kv_heads + h) * 2 + (is_max ? 1 : 0)) * kHeadDim + c * 8;
    if (off > 0) {
        const uint4 w = *reinterpret_cast<const uint4*>(mdst);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = is_max ? max_bf16x2(acc[i], word_of(w, i)) : min_bf16x2(acc[i], word_of(w, i));
    }
    *reinterpret_cast<uint4*>(mdst) = make_uint4(acc[0], acc[1], acc[2], acc[3]);
}

constexpr int kAppendThreads = 128;
constexpr int64_t kLongAppend = 2048;   // calls of at least this many tokens use 16-token windows

template <bool FP8>
__global__ void __launch_bounds__(kAppendThreads, FP8 ? 5 : 7) append_kv_meta_kernel(
    void* __restrict__ k_pool, void* __restrict__ v_pool, __nv_bfloat16* __restrict__ meta,
    float* __restrict__ k_scale, float* __restrict__ v_scale, int64_t num_phys_pages, int num_kv_heads,
    const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new,
    const int32_t* __restrict__ slot_mapping, int64_t num_tokens, int win) {
    const int lane = threadIdx.x & 31;
    const int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t windows = (num_tokens + win - 1) / win;
    const bool active = item < windows * num_kv_heads * 2;
    const bool is_key = (item & 1) == 0;                        // even items: keys, odd: values
    const int64_t t0 = (item / 2 / num_kv_heads) * win;
    const int h = static_cast<int>((item / 2) % num_kv_heads);
    const int64_t pool_slots = num_phys_pages * kPage;
    auto in_pool = [&](int32_t sl) { return sl >= 0 && sl < pool_slots; };
    const __nv_bfloat16* rows_new = is_key ? k_new : v_new;

    // The slots and new rows are inputs of the call, so they load before the
    // wait for the kernel before (which may still read or write the pool and
    // the metadata): in a chunked prefill a chunk's loads then overlap the
    // previous chunk's stores.  With 16-token windows the rows of a run
    // starting at the window's first token (a prefill window's only run) go
    // to shared memory by async copies (lane l: chunk l % 16 of rows
    // l / 16 + 2 k), which hold no registers; other runs, and every run of a
    // one-token window (mostly one row long), load theirs when handled.
    __shared__ __align__(16) uint4 s_rows[kAppendThreads / 32][kPage / 2][32];
    uint4* const my_rows = &s_rows[threadIdx.x >> 5][0][lane];
    {
        const int c = lane & 15, half = lane >> 4;
#pragma unroll
        for (int k = 0; k < kPage / 2; ++k) {
            const int64_t t = t0 + half + 2 * k;
            const bool ok = active && win == kPage && t < num_tokens;
            cp_async16(smem_addr(my_rows + 32 * k), ok ? rows_new + (t * num_kv_heads + h) * kHeadDim + c * 8 : rows_new,
                       ok ? 16u : 0u);
        }
        cp_async_commit();
    }
    // 1. slots of tokens t0 .. t0 + 31 and of t0 - 1; runs that start in the window.
    const int64_t ti = t0 + lane;
    const int32_t si = active && ti < num_tokens ? slot_mapping[ti] : -1;
    const int32_t s_before = (active && lane == 0 && t0 > 0) ? slot_mapping[t0 - 1] : -1;
    cp_async_wait<0>();   // each lane reads back only its own copies
    // The kernel before may still read the pool and the metadata: wait for
    // it before writing.  The scoring kernel that usually follows may then
    // be scheduled and load its page-table entries and query meanwhile.
    pdl_wait();
    pdl_launch_dependents();
    if (!active) return;
    if (lane < win && ti < num_tokens && !in_pool(si) && h == 0 && is_key) svq_flag(SV_DEVERR_SLOT);
    int32_t sp = __shfl_up_sync(0xffffffffu, si, 1);   // the predecessor's slot
    if (lane == 0) sp = s_before;
    const bool valid = ti < num_tokens && in_pool(si);
    const bool cont = valid && in_pool(sp) && sp / kPage == si / kPage && sp % kPage < si % kPage;
    const uint32_t cont_mask = __ballot_sync(0xffffffffu, cont);
    uint32_t starts = __ballot_sync(0xffffffffu, lane < win && valid && !cont);
    while (starts) {
        const int r = __ffs(starts) - 1;
        starts &= starts - 1u;
        const int R = __ffs(~(cont_mask >> (r + 1)));   // 1 + the continuing tokens after r (r + R <= 31)
        append_run<FP8>(is_key ? k_pool : v_pool, is_key ? k_scale : v_scale, meta, is_key, num_kv_heads, h,
                        rows_new, t0 + r, R, si, r, r == 0 && win == kPage ? my_rows : nullptr);
    }
}

int launch_update_meta(const sv_cache* c, const void* k_new, const void* v_new, const int32_t* slot_mapping,
                       int64_t num_tokens, cudaStream_t stream) {
    const int win = num_tokens >= kLongAppend ? kPage : 1;
    const int64_t items = (num_tokens + win - 1) / win * c->num_kv_heads * 2;   // (window, kv head, K or V)
    const int64_t blocks = (items * 32 + kAppendThreads - 1) / kAppendThreads;
    if (blocks > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
    const auto kn = static_cast<const __nv_bfloat16*>(k_new);
    const auto vn = static_cast<const __nv_bfloat16*>(v_new);
    auto* meta = static_cast<__nv_bfloat16*>(c->meta);
    cudaError_t e;
    if (c->kv_format == SV_KV_FP8_E4M3)
        e = launch_pdl(append_kv_meta_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(kAppendThreads), 0, stream,
                       c->k_pool, c->v_pool, meta, static_cast<float*>(c->k_scale), static_cast<float*>(c->v_scale),
                       c->num_phys_pages, c->num_kv_heads, kn, vn, slot_mapping, num_tokens, win);
    else
        e = launch_pdl(append_kv_meta_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(kAppendThreads), 0, stream,
                       c->k_pool, c->v_pool, meta, static_cast<float*>(nullptr), static_cast<float*>(nullptr),
                       c->num_phys_pages, c->num_kv_heads, kn, vn, slot_mapping, num_tokens, win);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace svq
