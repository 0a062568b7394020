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

constexpr int kScoreThreads = 256;
constexpr int kScoreWarps = kScoreThreads / 32;

// Sums N partials over the warp; afterwards lane l holds the full sum of
// value index l >> (5 - log2 N).
template <int N>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[N], int lane) {
    static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two <= 32");
    int s = 16;
#pragma unroll
    for (int n = N; n > 1; n >>= 1, s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
#pragma unroll
    for (; s >= 1; s >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], s);
    return v[0];
}

template <int HKV>
__global__ void __launch_bounds__(kScoreThreads, 2) score_pages_kernel(
    const __nv_bfloat16* __restrict__ meta, int64_t num_phys_pages, const __nv_bfloat16* __restrict__ q,
    int group, const int32_t* __restrict__ page_table, const int32_t* __restrict__ seq_lens, int max_pages,
    int pages_per_cta, float* __restrict__ scores) {
    constexpr int U = (HKV >= 8) ? 2 : (HKV >= 4 ? 4 : (HKV == 2 ? 8 : 8));
    constexpr int N = U * HKV;
    __shared__ float coef[HKV][2][kHeadDim];   // [j][0] = Qn (pairs kmin), [j][1] = Qp (pairs kmax)

    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int len = seq_lens[b];
    int n = (len + kPage - 1) / kPage;
    if (len < 1 || n > max_pages) {
        if (threadIdx.x == 0 && blockIdx.x == 0) svq_flag(SV_DEVERR_SEQ_LEN);
        n = len < 1 ? 0 : max_pages;
    }
    const int cta_begin = blockIdx.x * pages_per_cta;
    if (cta_begin >= n) return;
    const int cta_end = min(n, cta_begin + pages_per_cta);

    // Fold the group's query heads into Qp / Qn.
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
    __syncthreads();
    float c[HKV][8];
#pragma unroll
    for (int j = 0; j < HKV; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) c[j][i] = coef[j][lane >> 4][(lane & 15) * 8 + i];

    // Contiguous slice of the CTA's pages for this warp.
    const int span = cta_end - cta_begin;
    const int per_warp = (span + kScoreWarps - 1) / kScoreWarps;
    const int w_begin = cta_begin + warp * per_warp;
    const int w_end = min(cta_end, w_begin + per_warp);
    const int32_t* pt_row = page_table + static_cast<int64_t>(b) * max_pages;
    float* score_row = scores + static_cast<int64_t>(b) * HKV * max_pages;

    for (int base = w_begin; base < w_end; base += 32) {
        const int cnt = min(32, w_end - base);
        int phys_l = lane < cnt ? pt_row[base + lane] : 0;
        if (static_cast<uint32_t>(phys_l) >= static_cast<uint64_t>(num_phys_pages)) {
            svq_flag(SV_DEVERR_PAGE_TABLE);
            phys_l = -1;
        }
        for (int u0 = 0; u0 < cnt; u0 += U) {
            uint4 w[U][HKV];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int phys = __shfl_sync(0xffffffffu, phys_l, (u0 + u) & 31);
                const bool ok = (u0 + u < cnt) && phys >= 0;
#pragma unroll
                for (int j = 0; j < HKV; ++j) {
                    if (ok) {
                        w[u][j] = ld_stream_v4(meta + (static_cast<int64_t>(phys) * HKV + j) * 2 * kHeadDim + lane * 8);
                    } else {
                        w[u][j] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            float part[N];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int j = 0; j < HKV; ++j) {
                    const uint32_t* x = reinterpret_cast<const uint32_t*>(&w[u][j]);
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc = fmaf(c[j][2 * i], bf16lo(x[i]), acc);
                        acc = fmaf(c[j][2 * i + 1], bf16hi(x[i]), acc);
                    }
                    part[u * HKV + j] = acc;
                }
            const float s = warp_transpose_reduce<N>(part, lane);
            constexpr int kLanesPerValue = 32 / N;
            if ((lane % kLanesPerValue) == 0) {
                const int idx = lane / kLanesPerValue;
                const int u = idx / HKV, j = idx % HKV;
                if (u0 + u < cnt) score_row[static_cast<int64_t>(j) * max_pages + base + u0 + u] = s;
            }
        }
    }
}

int score_pages_ctas_per_request(int batch, int max_pages, int sm_count, int* pages_per_cta) {
    // One wave of two CTAs per SM over the (batch x max_pages) page grid.
    const int64_t target = static_cast<int64_t>(sm_count) * 2;
    int64_t ppc = (static_cast<int64_t>(batch) * max_pages + target - 1) / target;
    ppc = ((ppc + kScoreWarps - 1) / kScoreWarps) * kScoreWarps;
    if (ppc < kScoreWarps) ppc = kScoreWarps;
    *pages_per_cta = static_cast<int>(ppc);
    return ceil_div(max_pages, ppc);
}

int launch_score(const sv_cache* c, const void* q, int num_q_heads, const int32_t* page_table,
                 const int32_t* seq_lens, int batch, int max_pages, float* scores, int sm_count,
                 cudaStream_t stream) {
    const int group = num_q_heads / c->num_kv_heads;
    int ppc = 0;
    const int ctas = score_pages_ctas_per_request(batch, max_pages, sm_count, &ppc);
    dim3 grid(ctas, batch);
    const auto* meta = static_cast<const __nv_bfloat16*>(c->meta);
    const auto* qq = static_cast<const __nv_bfloat16*>(q);
    switch (c->num_kv_heads) {
        case 1: score_pages_kernel<1><<<grid, kScoreThreads, 0, stream>>>(meta, c->num_phys_pages, qq, group, page_table, seq_lens, max_pages, ppc, scores); break;
        case 2: score_pages_kernel<2><<<grid, kScoreThreads, 0, stream>>>(meta, c->num_phys_pages, qq, group, page_table, seq_lens, max_pages, ppc, scores); break;
        case 4: score_pages_kernel<4><<<grid, kScoreThreads, 0, stream>>>(meta, c->num_phys_pages, qq, group, page_table, seq_lens, max_pages, ppc, scores); break;
        case 8: score_pages_kernel<8><<<grid, kScoreThreads, 0, stream>>>(meta, c->num_phys_pages, qq, group, page_table, seq_lens, max_pages, ppc, scores); break;
        default: return SV_ERR_UNSUPPORTED;
    }
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// ---------------------------------------------------------------- top-K
//
// One CTA per (request, kv head).  Scores become order-preserving 32-bit
// keys in shared memory; three radix passes (11, 11, 10 bits, most
// significant first) locate the exact key T of the K-th best page and how
// many pages equal to T still fit.  A single block-wide scan over contiguous
// per-thread index segments then emits, in ascending index order, every page
// above T and the lowest-indexed pages equal to T.

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kRadixBins = 2048;

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

__global__ void __launch_bounds__(kTopkThreads) topk_pages_kernel(const float* __restrict__ scores,
                                                                  const int32_t* __restrict__ seq_lens,
                                                                  int num_kv_heads, int max_pages, int K,
                                                                  int32_t* __restrict__ sel_idx,
                                                                  int32_t* __restrict__ sel_cnt) {
    extern __shared__ uint32_t keys[];   // [max_pages]
    __shared__ uint32_t hist[kRadixBins];
    __shared__ uint32_t warp_tot[kTopkWarps];
    __shared__ uint32_t s_prefix, s_remaining;

    const int bg = blockIdx.x;
    const int b = bg / num_kv_heads;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int len = seq_lens[b];
    int n = (len + kPage - 1) / kPage;
    if (len < 1 || n > max_pages) {
        if (tid == 0) svq_flag(SV_DEVERR_SEQ_LEN);
        n = len < 1 ? 0 : max_pages;
    }
    const int m = min(K, n);
    int32_t* out = sel_idx + static_cast<int64_t>(bg) * K;
    if (n <= K) {
        for (int i = tid; i < K; i += kTopkThreads) out[i] = i < n ? i : -1;
        if (tid == 0) sel_cnt[bg] = n;
        return;
    }

    const float* row = scores + static_cast<int64_t>(bg) * max_pages;
    for (int i = tid; i < n; i += kTopkThreads) keys[i] = order_key(row[i]);

    if (tid == 0) {
        s_prefix = 0u;
        s_remaining = static_cast<uint32_t>(m);
    }
    uint32_t prefix = 0, remaining = static_cast<uint32_t>(m);
    constexpr int kShift[3] = {21, 10, 0};
    constexpr int kBits[3] = {11, 11, 10};
#pragma unroll
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = kShift[pass];
        const uint32_t nbins = 1u << kBits[pass];
        const uint32_t hi_mask = (pass == 0) ? 0u : ~((1u << (shift + kBits[pass])) - 1u);
        for (int i = tid; i < kRadixBins; i += kTopkThreads) hist[i] = 0u;
        __syncthreads();
        for (int base = 0; base < n; base += kTopkThreads) {
            const int i = base + tid;
            uint32_t bin = 0xffffffffu;
            if (i < n) {
                const uint32_t k = keys[i];
                if ((k & hi_mask) == prefix) bin = (k >> shift) & (nbins - 1u);
            }
            const uint32_t peers = __match_any_sync(0xffffffffu, bin);
            if (bin != 0xffffffffu && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
        }
        __syncthreads();
        // Thread t owns bins 2047-2t and 2046-2t (descending); a scan gives the
        // count of candidates in strictly higher bins.
        const uint32_t hi_bin = kRadixBins - 1 - 2 * tid;
        const uint32_t c0 = hist[hi_bin], c1 = hist[hi_bin - 1];
        const uint32_t incl = block_inclusive_scan(c0 + c1, warp_tot);
        const uint32_t excl = incl - c0 - c1;
        if (excl < remaining && remaining <= excl + c0) {
            s_prefix = prefix | (hi_bin << shift);
            s_remaining = remaining - excl;
        } else if (excl + c0 < remaining && remaining <= excl + c0 + c1) {
            s_prefix = prefix | ((hi_bin - 1) << shift);
            s_remaining = remaining - excl - c0;
        }
        __syncthreads();
        prefix = s_prefix;
        remaining = s_remaining;
        __syncthreads();
    }
    const uint32_t T = prefix;   // key of the m-th best page; `remaining` pages equal to T are taken

    // Ordered compaction over contiguous index segments.
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
    uint32_t pos = (excl >> 16) + min(eq_seen, remaining);
    for (int i = s0; i < s1; ++i) {
        const uint32_t k = keys[i];
        bool take = k > T;
        if (k == T) {
            take = eq_seen < remaining;
            ++eq_seen;
        }
        if (take) {
            if (pos < static_cast<uint32_t>(m)) out[pos] = i;
            ++pos;
        }
    }
    for (int i = m + tid; i < K; i += kTopkThreads) out[i] = -1;
    if (tid == 0) sel_cnt[bg] = m;
}

int launch_topk(const float* scores, const int32_t* seq_lens, int batch, int num_kv_heads, int max_pages,
                int budget_pages, int32_t* sel_idx, int32_t* sel_cnt, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(max_pages) * sizeof(uint32_t);
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(topk_pages_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return SV_ERR_CUDA;
    }
    topk_pages_kernel<<<batch * num_kv_heads, kTopkThreads, smem, stream>>>(
        scores, seq_lens, num_kv_heads, max_pages, budget_pages, sel_idx, sel_cnt);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace svq
