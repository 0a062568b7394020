// Query-aware page selection (the build_decode_view hook of the
// "add-sparse-method" skill page; Quest's query-relevant page selection on
// the SparseEngine summary page, section "method key points").
//
//   score_pages_kernel : upper-bound score of every (request, kv head, page)
//   topk_pages_kernel  : top-K pages per (request, kv head), ties to the lower
//                        page index, emitted in ascending page order
#include "svq_common.cuh"

namespace svq {

SVQ_DEFINE_ERROR_WORD(read_error_select)

// ---------------------------------------------------------------- scoring
//
// Regrouping the bound by the sign of each query element,
//   sum_h sum_i max(q_hi kmax_i, q_hi kmin_i) = sum_i Qp_i kmax_i + Qn_i kmin_i,
//   Qp_i = sum_h max(q_hi, 0),  Qn_i = sum_h min(q_hi, 0),
// turns the score into one fp32 multiply-add per metadata element (1 flop per
// byte), which keeps the kernel bound by HBM rather than by the ALUs.
//
// A page's metadata for all kv heads is contiguous (HKV x 512 bytes).  Lane l
// reads 16 bytes of every head j: chunk l of [kmin(128) | kmax(128)], so its
// coefficients are fixed for the kernel's lifetime (Qn for l < 16, Qp for
// l >= 16, channels 8 (l & 15) .. + 7).  Each warp keeps U pages x HKV heads of
// 16-byte loads in flight and folds the U*HKV lane partials with a transposed
// butterfly (one shuffle per score).

#ifndef SVQ_SCORE_WARPS
#define SVQ_SCORE_WARPS 16
#endif
#ifndef SVQ_SCORE_STAGE_BYTES
#define SVQ_SCORE_STAGE_BYTES 4096   // metadata bytes per ring stage (a group of pages)
#endif
#ifndef SVQ_SCORE_STAGES
#define SVQ_SCORE_STAGES 3           // stages in flight per warp
#endif
constexpr int kScoreWarps = SVQ_SCORE_WARPS;
constexpr int kScoreThreads = kScoreWarps * 32;

template <int HKV>
struct ScoreShape {
    static constexpr int kPageBytes = HKV * 2 * kHeadDim * 2;              // metadata of one page, all kv heads
    static constexpr int kGroupRaw = SVQ_SCORE_STAGE_BYTES / kPageBytes;   // pages per stage
    static constexpr int G = kGroupRaw < 1 ? 1 : (kGroupRaw > 8 ? 8 : kGroupRaw);
    static constexpr int kStages = SVQ_SCORE_STAGES;
    static constexpr int kStageBytes = G * kPageBytes;
    static constexpr int kSmemBytes = kScoreWarps * kStages * kStageBytes;
    static constexpr int L = 32 / HKV;      // lanes per kv head
    static constexpr int kChunks = HKV;     // 16-byte chunks of a head's 512-byte row per lane
    static_assert(32 % HKV == 0, "kv heads per page must divide 32");
    static_assert(32 % G == 0, "pages per stage must divide 32");
};

// Each warp streams a contiguous run of one request's pages through a ring of
// kStages stages of G pages in shared memory.  Lanes 0..G-1 each move one
// page's metadata (all kv heads, contiguous) with a bulk copy; the copies of
// a stage complete on one mbarrier.  Lane (j, k) = (lane / L, lane % L) owns
// kv head j and the 16-byte chunks k, k + L, k + 2L, ... of that head's
// 512-byte [kmin | kmax] row, so a page's score is one register accumulation
// per lane followed by a log2(L)-level shuffle sum among the L lanes of the
// head.  Physical page numbers are fetched 32 at a time, one batch ahead.
template <int HKV>
__global__ void __launch_bounds__(kScoreThreads, 1) score_pages_kernel(
    const __nv_bfloat16* __restrict__ meta, int64_t num_phys_pages, const __nv_bfloat16* __restrict__ q,
    int group, const int32_t* __restrict__ page_table, const int32_t* __restrict__ seq_lens, int max_pages,
    int pages_per_cta, float* __restrict__ scores) {
    using S = ScoreShape<HKV>;
    constexpr int kStages = S::kStages, G = S::G, L = S::L, C = S::kChunks;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ float coef[HKV][2][kHeadDim];   // [j][0] = Qn (pairs kmin), [j][1] = Qp (pairs kmax)
    __shared__ __align__(8) uint64_t bars[kScoreWarps][kStages];

    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int hj = lane / L;        // kv head of this lane
    const int hk = lane % L;        // first chunk of this lane

    if (lane == 0) {
        for (int st = 0; st < kStages; ++st) mbar_init(smem_addr(&bars[warp][st]), 1);
        mbar_init_fence();
    }
    // Fold the group's query heads into Qp / Qn (q is an input of the step).
    const int hq = HKV * group;
    for (int idx = threadIdx.x; idx < HKV * kHeadDim; idx += kScoreThreads) {
        const int j = idx / kHeadDim, ch = idx % kHeadDim;
        float qp = 0.f, qn = 0.f;
        for (int h = 0; h < group; ++h) {
            const float v = __bfloat162float(q[(static_cast<int64_t>(b) * hq + j * group + h) * kHeadDim + ch]);
            qp += fmaxf(v, 0.f);
            qn += fminf(v, 0.f);
        }
        coef[j][0][ch] = qn;
        coef[j][1][ch] = qp;
    }
    pdl_wait();   // metadata may come from an append launched just before
    __syncthreads();

    const int len = seq_lens[b];
    int n = (len + kPage - 1) / kPage;
    if (len < 1 || n > max_pages) {
        if (threadIdx.x == 0 && blockIdx.x == 0) svq_flag(SV_DEVERR_SEQ_LEN);
        n = len < 1 ? 0 : max_pages;
    }
    const int cta_begin = blockIdx.x * pages_per_cta;
    const int cta_end = min(n, cta_begin + pages_per_cta);
    const int span = max(0, cta_end - cta_begin);
    const int per_warp = (span + kScoreWarps - 1) / kScoreWarps;
    const int w_begin = cta_begin + min(span, warp * per_warp);
    const int count = max(0, min(cta_end, w_begin + per_warp) - w_begin);
    const int n_groups = (count + G - 1) / G;

    // Chunk t of this lane is chunk hk + L t of the head's row: kmin channels
    // for chunks < 16, kmax channels for chunks >= 16.
    float c[C][8];
#pragma unroll
    for (int t = 0; t < C; ++t) {
        const int chunk = hk + L * t;
#pragma unroll
        for (int i = 0; i < 8; ++i) c[t][i] = coef[hj][chunk >> 4][(chunk & 15) * 8 + i];
    }

    const int32_t* pt_row = page_table + static_cast<int64_t>(b) * max_pages + w_begin;
    float* score_row = scores + (static_cast<int64_t>(b) * HKV + hj) * max_pages + w_begin;
    const unsigned char* meta_bytes = reinterpret_cast<const unsigned char*>(meta);
    const unsigned char* ring_w = ring + warp * (kStages * S::kStageBytes);
    const uint32_t ring_s = smem_addr(ring_w);
    const uint32_t bar0 = smem_addr(&bars[warp][0]);

    auto load_pt = [&](int base) -> int {
        const int p = base + lane;
        int v = p < count ? pt_row[p] : -1;
        if (p < count && static_cast<uint32_t>(v) >= static_cast<uint64_t>(num_phys_pages)) {
            svq_flag(SV_DEVERR_PAGE_TABLE);
            v = -1;
        }
        return v;
    };
    int pt_base = 0;
    int pt_cur = load_pt(0);
    int pt_nxt = load_pt(32);
    uint32_t stage_ok[kStages];   // bit u: page u of the stage is real (uniform across the warp)
#pragma unroll
    for (int st = 0; st < kStages; ++st) stage_ok[st] = 0u;
    // Issues group gi (warp-uniform, increasing) into ring stage `stage`.
    auto issue = [&](int gi, int stage) -> uint32_t {
        const int p0 = gi * G;
        if (p0 >= pt_base + 32) {   // G divides 32, so a group never straddles two batches
            pt_base += 32;
            pt_cur = pt_nxt;
            pt_nxt = load_pt(pt_base + 32);
        }
        const int mine = __shfl_sync(0xffffffffu, pt_cur, (p0 - pt_base + (lane % G)) & 31);
        const uint32_t ok = __ballot_sync(0xffffffffu, lane < G && mine >= 0) & ((1u << G) - 1u);
        const uint32_t bar = bar0 + stage * 8;
        if (lane == 0) {
            if (ok) mbar_arrive_expect_tx(bar, __popc(ok) * S::kPageBytes);
            else mbar_arrive(bar);
        }
        __syncwarp();
        if (lane < G && mine >= 0)
            bulk_copy_g2s(ring_s + stage * S::kStageBytes + lane * S::kPageBytes,
                          meta_bytes + static_cast<int64_t>(mine) * S::kPageBytes, S::kPageBytes, bar);
        return ok;
    };

    __syncwarp();   // barriers initialised before any use
    int issued = 0;
#pragma unroll
    for (int st = 0; st < kStages; ++st)
        if (st < n_groups) stage_ok[st] = issue(st, st), ++issued;
    bool timed_out = false;
    int consumed = 0;
    const unsigned char* lane_base = ring_w + hj * 512 + hk * 16;
    for (int gi = 0; gi < n_groups; ++gi) {
        const int stage = gi % kStages;
        const bool ok = mbar_wait_bounded(bar0 + stage * 8, (gi / kStages) & 1);
        if (__any_sync(0xffffffffu, !ok)) {
            timed_out = true;
            break;
        }
        consumed = gi + 1;
        uint32_t okm = 0;
#pragma unroll
        for (int st = 0; st < kStages; ++st) okm = st == stage ? stage_ok[st] : okm;
        float acc[G];
#pragma unroll
        for (int u = 0; u < G; ++u) {
            uint4 w[C];
#pragma unroll
            for (int t = 0; t < C; ++t)
                w[t] = *reinterpret_cast<const uint4*>(lane_base + stage * S::kStageBytes + u * S::kPageBytes +
                                                       t * L * 16);
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int t = 0; t < C; ++t) {
                const uint32_t x[4] = {w[t].x, w[t].y, w[t].z, w[t].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a0 = fmaf(c[t][2 * e], bf16lo(x[e]), a0);
                    a1 = fmaf(c[t][2 * e + 1], bf16hi(x[e]), a1);
                }
            }
            acc[u] = (okm & (1u << u)) ? a0 + a1 : 0.f;
        }
        __syncwarp();   // every lane has read the stage before it is refilled
        if (gi + kStages < n_groups) {
            const uint32_t nok = issue(gi + kStages, stage);
#pragma unroll
            for (int st = 0; st < kStages; ++st) stage_ok[st] = st == stage ? nok : stage_ok[st];
            ++issued;
        }
#pragma unroll
        for (int u = 0; u < G; ++u) {
#pragma unroll
            for (int m = 1; m < L; m <<= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], m);
        }
        if (hk < G) {
            // Lane (j, u) writes page u's score for head j.
            float v = acc[0];
#pragma unroll
            for (int u = 1; u < G; ++u) v = hk == u ? acc[u] : v;
            const int p = gi * G + hk;
            if (p < count) score_row[p] = v;
        }
    }
    if (timed_out) {
        // Give the copies this warp still has in flight a bounded chance to land
        // before the CTA's shared memory is released.
        if (lane == 0) svq_flag(SV_DEVERR_TIMEOUT);
        for (int gi = consumed; gi < issued; ++gi)
            (void)mbar_wait_bounded(bar0 + (gi % kStages) * 8, (gi / kStages) & 1);
    }
    pdl_launch_dependents();
}

template <int HKV>
int launch_score_hkv(const sv_cache* c, const __nv_bfloat16* q, int group, const int32_t* page_table,
                     const int32_t* seq_lens, int batch, int max_pages, float* scores, int sm_count,
                     cudaStream_t stream) {
    using S = ScoreShape<HKV>;
    static bool attr_set[64] = {};
    const int dev = current_device();
    if (dev < 0) return SV_ERR_CUDA;
    if (dev >= 64 || !attr_set[dev]) {
        if (cudaFuncSetAttribute(score_pages_kernel<HKV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 S::kSmemBytes) != cudaSuccess)
            return SV_ERR_CUDA;
        if (dev < 64) attr_set[dev] = true;
    }
    // One CTA per SM over the (batch x max_pages) page grid, whole warps of pages.
    int64_t ppc = (static_cast<int64_t>(batch) * max_pages + sm_count - 1) / sm_count;
    ppc = ((ppc + kScoreWarps - 1) / kScoreWarps) * kScoreWarps;
    if (ppc < kScoreWarps) ppc = kScoreWarps;
    const int ctas = ceil_div(max_pages, ppc);
    const cudaError_t e = launch_pdl(score_pages_kernel<HKV>, dim3(ctas, batch), dim3(kScoreThreads),
                                     S::kSmemBytes, stream, static_cast<const __nv_bfloat16*>(c->meta),
                                     c->num_phys_pages, q, group, page_table, seq_lens, max_pages,
                                     static_cast<int>(ppc), scores);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

int launch_score(const sv_cache* c, const void* q, int num_q_heads, const int32_t* page_table,
                 const int32_t* seq_lens, int batch, int max_pages, float* scores, int sm_count,
                 cudaStream_t stream) {
    const int group = num_q_heads / c->num_kv_heads;
    const auto* qq = static_cast<const __nv_bfloat16*>(q);
    switch (c->num_kv_heads) {
        case 1: return launch_score_hkv<1>(c, qq, group, page_table, seq_lens, batch, max_pages, scores, sm_count, stream);
        case 2: return launch_score_hkv<2>(c, qq, group, page_table, seq_lens, batch, max_pages, scores, sm_count, stream);
        case 4: return launch_score_hkv<4>(c, qq, group, page_table, seq_lens, batch, max_pages, scores, sm_count, stream);
        case 8: return launch_score_hkv<8>(c, qq, group, page_table, seq_lens, batch, max_pages, scores, sm_count, stream);
        default: return SV_ERR_UNSUPPORTED;
    }
}

// ---------------------------------------------------------------- top-K
//
// One CTA per (request, kv head).  Scores become order-preserving 32-bit
// keys in shared memory.  The threshold search is a selection, not a sort:
//  1. one histogram over [min key, max key] in 2048 power-of-two-wide bins
//     (a bin index is a right shift of key - min, so bins are monotone in the
//     score) locates the bin b* holding the K-th best key;
//  2. if b* holds few keys (<= kCandCap), each of them gets its exact rank in
//     (key desc, page asc) order by comparing against the others, which gives
//     the threshold key T and how many keys equal to T are taken;
//     otherwise three radix passes (11, 11, 10 bits) over all keys find T.
// A block-wide scan over contiguous index segments then emits, in ascending
// index order, every page above T and the lowest-indexed pages equal to T.

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kRadixBins = 2048;
constexpr int kLoadItems = 8;
constexpr int kCandCap = 256;

__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide inclusive scan of one value per thread (1024 threads).
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint32_t t = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += x;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    const uint32_t add = warp > 0 ? warp_tot[warp - 1] : 0u;
    __syncthreads();   // warp_tot may be reused right after
    return v + add;
}

// Finds, over a 2048-bin histogram, the bin holding the `remaining`-th key
// counted from the top, and how many keys of that bin are still needed.
__device__ __forceinline__ void find_bin_from_top(const uint32_t* hist, uint32_t remaining, uint32_t* warp_tot,
                                                  uint32_t* s_bin, uint32_t* s_rem) {
    const int tid = threadIdx.x;
    const uint32_t hi_bin = kRadixBins - 1 - 2 * tid;   // thread t owns bins 2047-2t, 2046-2t
    const uint32_t c0 = hist[hi_bin], c1 = hist[hi_bin - 1];
    const uint32_t incl = block_inclusive_scan(c0 + c1, warp_tot);
    const uint32_t excl = incl - c0 - c1;
    if (excl < remaining && remaining <= excl + c0) {
        *s_bin = hi_bin;
        *s_rem = remaining - excl;
    } else if (excl + c0 < remaining && remaining <= excl + c0 + c1) {
        *s_bin = hi_bin - 1;
        *s_rem = remaining - excl - c0;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kTopkThreads) topk_pages_kernel(const float* __restrict__ scores,
                                                                  const int32_t* __restrict__ seq_lens,
                                                                  int num_kv_heads, int max_pages, int K,
                                                                  int32_t* __restrict__ sel_idx,
                                                                  int32_t* __restrict__ sel_cnt) {
    extern __shared__ uint32_t keys[];   // [max_pages]
    __shared__ uint32_t hist[kRadixBins];
    __shared__ uint32_t warp_tot[kTopkWarps];
    __shared__ uint32_t warp_lo[kTopkWarps], warp_hi[kTopkWarps];
    __shared__ uint32_t cand_key[kCandCap];
    __shared__ int32_t cand_idx[kCandCap];
    __shared__ uint32_t s_bin, s_rem, s_cand, s_T, s_take, s_lo, s_shift;
    __shared__ int32_t s_Tidx;

    const int bg = blockIdx.x;
    const int b = bg / num_kv_heads;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int len = seq_lens[b];
    int n = (len + kPage - 1) / kPage;
    if (len < 1 || n > max_pages) {
        if (tid == 0) svq_flag(SV_DEVERR_SEQ_LEN);
        n = len < 1 ? 0 : max_pages;
    }
    const int m = min(K, n);
    int32_t* out = sel_idx + static_cast<int64_t>(bg) * K;
    pdl_wait();   // scores come from the scoring kernel launched just before
    if (n <= K) {
        for (int i = tid; i < K; i += kTopkThreads) out[i] = i < n ? i : -1;
        if (tid == 0) sel_cnt[bg] = n;
        pdl_launch_dependents();
        return;
    }

    // 1. keys (all loads of a round issued before any use), min and max.
    const float* row = scores + static_cast<int64_t>(bg) * max_pages;
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int base = 0; base < n; base += kTopkThreads * kLoadItems) {
        float f[kLoadItems];
#pragma unroll
        for (int r = 0; r < kLoadItems; ++r) {
            const int i = base + r * kTopkThreads + tid;
            f[r] = i < n ? row[i] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < kLoadItems; ++r) {
            const int i = base + r * kTopkThreads + tid;
            if (i < n) {
                const uint32_t k = order_key(f[r]);
                keys[i] = k;
                lo = min(lo, k);
                hi = max(hi, k);
            }
        }
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) {
        warp_lo[warp] = lo;
        warp_hi[warp] = hi;
    }
    for (int i = tid; i < kRadixBins; i += kTopkThreads) hist[i] = 0u;
    if (tid == 0) s_cand = 0u;
    __syncthreads();
    if (warp == 0) {
        lo = __reduce_min_sync(0xffffffffu, warp_lo[lane]);
        hi = __reduce_max_sync(0xffffffffu, warp_hi[lane]);
        if (lane == 0) {
            const uint32_t range = hi - lo;
            const int bits = range == 0 ? 0 : 32 - __clz(range);   // range < 2^bits
            s_lo = lo;
            s_shift = bits > 11 ? bits - 11 : 0;                    // (range >> shift) < 2048
        }
    }
    __syncthreads();
    lo = s_lo;
    const uint32_t shift = s_shift;

    // 2. histogram of (key - lo) >> shift; bin of the m-th best key.
    for (int i = tid; i < n; i += kTopkThreads) atomicAdd(&hist[(keys[i] - lo) >> shift], 1u);
    __syncthreads();
    find_bin_from_top(hist, static_cast<uint32_t>(m), warp_tot, &s_bin, &s_rem);
    const uint32_t bstar = s_bin, need = s_rem;
    uint32_t T, take;
    if (hist[bstar] <= kCandCap) {
        // 3a. exact rank of each key of bin b* among the others.
        for (int i = tid; i < n; i += kTopkThreads) {
            const uint32_t k = keys[i];
            if (((k - lo) >> shift) == bstar) {
                const uint32_t pos = atomicAdd(&s_cand, 1u);
                cand_key[pos] = k;
                cand_idx[pos] = i;
            }
        }
        __syncthreads();
        const int nc = static_cast<int>(s_cand);
        if (tid < nc) {
            const uint32_t k = cand_key[tid];
            const int idx = cand_idx[tid];
            uint32_t rank = 0;
            for (int j = 0; j < nc; ++j) {
                const uint32_t kj = cand_key[j];
                rank += (kj > k) || (kj == k && cand_idx[j] < idx);
            }
            if (rank == need - 1) {
                s_T = k;
                s_Tidx = idx;
            }
        }
        if (tid == 0) s_take = 0u;
        __syncthreads();
        if (tid < nc && cand_key[tid] == s_T && cand_idx[tid] <= s_Tidx) atomicAdd(&s_take, 1u);
        __syncthreads();
        T = s_T;
        take = s_take;
    } else {
        // 3b. many keys crowd one bin (e.g. equal scores): exact radix select.
        uint32_t prefix = 0, remaining = static_cast<uint32_t>(m);
        constexpr int kShift[3] = {21, 10, 0};
        constexpr int kBits[3] = {11, 11, 10};
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
            const int sh = kShift[pass];
            const uint32_t nbins = 1u << kBits[pass];
            const uint32_t hi_mask = (pass == 0) ? 0u : ~((1u << (sh + kBits[pass])) - 1u);
            __syncthreads();
            for (int i = tid; i < kRadixBins; i += kTopkThreads) hist[i] = 0u;
            __syncthreads();
            for (int i = tid; i < n; i += kTopkThreads) {
                const uint32_t k = keys[i];
                if ((k & hi_mask) == prefix) atomicAdd(&hist[(k >> sh) & (nbins - 1u)], 1u);
            }
            __syncthreads();
            find_bin_from_top(hist, remaining, warp_tot, &s_bin, &s_rem);
            prefix |= s_bin << sh;
            remaining = s_rem;
        }
        T = prefix;
        take = remaining;
    }

    // 4. ordered compaction over contiguous index segments.
    const int seg = (n + kTopkThreads - 1) / kTopkThreads;
    const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
    uint32_t gt = 0, eq = 0;
    for (int i = s0; i < s1; ++i) {
        const uint32_t k = keys[i];
        gt += k > T;
        eq += k == T;
    }
    const uint32_t packed = (gt << 16) | eq;   // n <= 32768 keeps both halves in 16 bits
    const uint32_t excl = block_inclusive_scan(packed, warp_tot) - packed;
    uint32_t eq_seen = excl & 0xffffu;
    uint32_t pos = (excl >> 16) + min(eq_seen, take);
    for (int i = s0; i < s1; ++i) {
        const uint32_t k = keys[i];
        bool sel = k > T;
        if (k == T) {
            sel = eq_seen < take;
            ++eq_seen;
        }
        if (sel) {
            if (pos < static_cast<uint32_t>(m)) out[pos] = i;
            ++pos;
        }
    }
    for (int i = m + tid; i < K; i += kTopkThreads) out[i] = -1;
    if (tid == 0) sel_cnt[bg] = m;
    pdl_launch_dependents();
}

int launch_topk(const float* scores, const int32_t* seq_lens, int batch, int num_kv_heads, int max_pages,
                int budget_pages, int32_t* sel_idx, int32_t* sel_cnt, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(max_pages) * sizeof(uint32_t);
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(topk_pages_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return SV_ERR_CUDA;
    }
    const cudaError_t e = launch_pdl(topk_pages_kernel, dim3(batch * num_kv_heads), dim3(kTopkThreads), smem,
                                     stream, scores, seq_lens, num_kv_heads, max_pages, budget_pages, sel_idx,
                                     sel_cnt);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace svq
