// Exact top-K of one score row by 256 threads (page selection of one
// (request, kv head)), shared by the stand-alone top-K kernel and the fused
// step kernel.
//
// Keeps the m = min(K, n) highest scores, ties to the lower page index, and
// writes their indices in ascending order, -1 after them.  Thread t holds keys
// 32t .. 32t+31 in registers.  Steps: a lower bound on the m-th largest key
// (from per-thread maxima of 4 groups of 8 keys); an adaptive 2048-bin
// histogram of the keys at or above it, over [bound, max]; the bin holding the
// m-th key; exact ranks of that bin's keys (three radix passes over all keys
// when it holds more than 256); ordered compaction by a block scan.
#pragma once

#include "svq_common.cuh"

namespace svq {

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowItems = 32;                          // keys per thread
constexpr int kRowMaxPages = kRowThreads * kRowItems;  // 8192
constexpr int kRowBins = 2048;
constexpr int kRowCandCap = 256;

// Order-preserving map of a float to u32 (larger float -> larger key).
__device__ __forceinline__ uint32_t row_order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int kBar>
__device__ __forceinline__ void row_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(kBar), "n"(kRowThreads) : "memory");
}

// Keeps the m = min(K, n) highest scores (ties to the lower page index) and
// writes their indices in ascending order.  The row is staged through shared
// memory with coalesced loads; thread t then holds keys 32t .. 32t+31.  A
// lower bound on the m-th largest key (the smallest j-th largest key over
// threads, for the smallest j in 1..4 with enough keys at or above it) trims
// the adaptive histogram to the top of the row; the boundary bin's keys are
// ranked exactly (radix passes when the bin holds more than 256 keys); the
// compaction follows the index order.
struct RowTopkScratch {
    uint32_t hist[kRowBins];
    uint32_t warp_tot[kRowWarps];
    uint32_t warp_red[6][kRowWarps];
    uint32_t cand_key[kRowCandCap];
    int32_t cand_idx[kRowCandCap];
    uint32_t bin, rem, cand, T, take;
};

// Run by threads 0 .. 255 of a CTA (named barrier kBar, 256 threads).
// row: the n scores of the row (L2 loads: the scores may come from other CTAs
// of the same launch, read after an acquire).  With kVec the row start is
// 16-byte aligned and readable up to n rounded up to 4 (16-byte loads);
// otherwise it is read one float per thread per step.  stage: 8192 floats of
// shared memory.  Writes out[0 .. K) and *cnt_out.
template <int kBar, bool kVec>
__device__ void topk_row_256(const float* row, int n, int K, int32_t* out, int32_t* cnt_out, RowTopkScratch& sc,
                             float* stage) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = min(K, n);
    if (n <= K) {
        for (int i = tid; i < K; i += kRowThreads) out[i] = i < n ? i : -1;
        if (tid == 0) *cnt_out = n < 0 ? 0 : n;
        return;
    }
    // Coalesced loads -> shared memory, where thread t's 32 keys sit in 16-byte
    // chunks swizzled by t % 8 (conflict-free both ways) -> registers.
    if (kVec) {
#pragma unroll
        for (int e = 0; e < kRowItems / 4; ++e) {
            const int idx = 4 * tid + 4 * kRowThreads * e;
            const float4 v = idx < n ? __ldcg(reinterpret_cast<const float4*>(row + idx))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            const int owner = (tid >> 3) + (kRowThreads / 8) * e;
            const int chunk = tid & 7;
            *reinterpret_cast<float4*>(stage + owner * 32 + 4 * (chunk ^ (owner & 7))) = v;
        }
    } else {
#pragma unroll 8
        for (int e = 0; e < kRowItems; ++e) {
            const int idx = tid + kRowThreads * e;
            const float v = idx < n ? __ldcg(row + idx) : 0.f;
            const int owner = warp + kRowWarps * e;
            stage[owner * 32 + 4 * ((lane >> 2) ^ (owner & 7)) + (lane & 3)] = v;
        }
    }
    row_sync<kBar>();
    const int i0 = kRowItems * tid;
    uint32_t key[kRowItems];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(stage + tid * 32 + 4 * (c ^ (tid & 7)));
        key[4 * c] = row_order_key(v.x);
        key[4 * c + 1] = row_order_key(v.y);
        key[4 * c + 2] = row_order_key(v.z);
        key[4 * c + 3] = row_order_key(v.w);
    }
    // Row minimum / maximum and, per thread, the maxima of its four groups of
    // 8 keys sorted (q1 >= q2 >= q3 >= q4): the thread holds at least j keys
    // >= qj, one from each of j groups.
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    uint32_t qmax[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < kRowItems; ++e) {
        const bool v = i0 + e < n;
        kmin = min(kmin, v ? key[e] : 0xffffffffu);
        qmax[e >> 3] = max(qmax[e >> 3], v ? key[e] : 0u);
    }
    kmax = max(max(qmax[0], qmax[1]), max(qmax[2], qmax[3]));
    {
        uint32_t x;
#define SVQ_CSWAP(i, j) x = min(qmax[i], qmax[j]); qmax[i] = max(qmax[i], qmax[j]); qmax[j] = x;
        SVQ_CSWAP(0, 1) SVQ_CSWAP(2, 3) SVQ_CSWAP(0, 2) SVQ_CSWAP(1, 3) SVQ_CSWAP(1, 2)
#undef SVQ_CSWAP
    }
    const bool full = i0 + kRowItems <= n;   // only threads with 32 valid keys give bounds
    uint32_t red[6] = {kmin, kmax, full ? qmax[0] : 0xffffffffu, full ? qmax[1] : 0xffffffffu,
                       full ? qmax[2] : 0xffffffffu, full ? qmax[3] : 0xffffffffu};
    for (int i = tid; i < kRowBins; i += kRowThreads) sc.hist[i] = 0u;
#pragma unroll
    for (int r = 0; r < 6; ++r) {
        const uint32_t v = r == 1 ? __reduce_max_sync(0xffffffffu, red[r]) : __reduce_min_sync(0xffffffffu, red[r]);
        if (lane == 0) sc.warp_red[r][warp] = v;
    }
    row_sync<kBar>();
#pragma unroll
    for (int r = 0; r < 6; ++r) {
        const uint32_t v = lane < kRowWarps ? sc.warp_red[r][lane] : (r == 1 ? 0u : 0xffffffffu);
        red[r] = r == 1 ? __reduce_max_sync(0xffffffffu, v) : __reduce_min_sync(0xffffffffu, v);
    }
    // Lower bound on the m-th largest key: the full threads each hold j keys
    // >= the minimum over them of qj, so that minimum is a bound once
    // j * (number of full threads) >= m; the smallest such j gives the tightest.
    uint32_t lo = red[0];
    const int full_threads = min(kRowThreads, n / kRowItems);
#pragma unroll
    for (int j = 4; j >= 1; --j)
        if (j * full_threads >= m) lo = red[1 + j];
    const uint32_t hi = red[1];
    const uint32_t range = hi - lo;
    const int rbits = range == 0 ? 0 : 32 - __clz(range);
    const uint32_t shift = rbits > 11 ? rbits - 11 : 0;
#pragma unroll
    for (int e = 0; e < kRowItems; ++e)
        if (i0 + e < n && key[e] >= lo) atomicAdd(&sc.hist[(key[e] - lo) >> shift], 1u);
    row_sync<kBar>();
    auto find_bin = [&](uint32_t remaining) {
        constexpr int kBpt = kRowBins / kRowThreads;
        const uint32_t top = kRowBins - 1 - kBpt * tid;
        uint32_t cnt[kBpt];
        uint32_t sum = 0;
#pragma unroll
        for (int i = 0; i < kBpt; ++i) {
            cnt[i] = sc.hist[top - i];
            sum += cnt[i];
        }
        uint32_t v = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        if (lane == 31) sc.warp_tot[warp] = v;
        row_sync<kBar>();
        uint32_t add = 0;
        for (int w2 = 0; w2 < warp; ++w2) add += sc.warp_tot[w2];
        uint32_t before = v + add - sum;
#pragma unroll
        for (int i = 0; i < kBpt; ++i) {
            if (before < remaining && remaining <= before + cnt[i]) {
                sc.bin = top - i;
                sc.rem = remaining - before;
            }
            before += cnt[i];
        }
        row_sync<kBar>();
    };
    find_bin(static_cast<uint32_t>(m));
    const uint32_t bstar = sc.bin, need = sc.rem;
    uint32_t T, take;
    if (sc.hist[bstar] <= kRowCandCap) {
        // Keys of the boundary bin: per-thread mask, positions by a block scan.
        uint32_t cmask = 0;
#pragma unroll
        for (int e = 0; e < kRowItems; ++e)
            cmask |= ((i0 + e < n && key[e] >= lo && ((key[e] - lo) >> shift) == bstar) ? 1u : 0u) << e;
        const uint32_t cnt = __popc(cmask);
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) sc.warp_tot[warp] = incl;
        row_sync<kBar>();
        uint32_t pos = incl - cnt;
        uint32_t total = 0;
#pragma unroll
        for (int w2 = 0; w2 < kRowWarps; ++w2) {
            const uint32_t t = sc.warp_tot[w2];
            pos += w2 < warp ? t : 0u;
            total += t;
        }
#pragma unroll
        for (int e = 0; e < kRowItems; ++e) {   // static indices keep key[] in registers
            if ((cmask >> e) & 1u) {
                sc.cand_key[pos] = key[e];
                sc.cand_idx[pos] = i0 + e;
                ++pos;
            }
        }
        if (tid == 0) sc.cand = total;
        row_sync<kBar>();
        const int nc = static_cast<int>(sc.cand);
        if (tid < nc) {
            const uint32_t my_k = sc.cand_key[tid];
            const int my_i = sc.cand_idx[tid];
            uint32_t above = 0, tied_before = 0;
            for (int j = 0; j < nc; ++j) {
                const uint32_t kj = sc.cand_key[j];
                above += kj > my_k;
                tied_before += (kj == my_k && sc.cand_idx[j] < my_i);
            }
            if (above + tied_before == need - 1) {
                sc.T = my_k;
                sc.take = need - above;
            }
        }
        row_sync<kBar>();
        T = sc.T;
        take = sc.take;
    } else {
        // Radix select on the full keys: 11 + 11 + 10 bits.
        uint32_t prefix = 0, remaining = static_cast<uint32_t>(m);
        for (int pass = 0; pass < 3; ++pass) {
            const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
            const int nbits = pass == 2 ? 10 : 11;
            const uint32_t nbins = 1u << nbits;
            const uint32_t hi_mask = pass == 0 ? 0u : ~((1u << (sh + nbits)) - 1u);
            row_sync<kBar>();
            for (int i = tid; i < kRowBins; i += kRowThreads) sc.hist[i] = 0u;
            row_sync<kBar>();
#pragma unroll
            for (int e = 0; e < kRowItems; ++e)
                if (i0 + e < n && (key[e] & hi_mask) == prefix) atomicAdd(&sc.hist[(key[e] >> sh) & (nbins - 1u)], 1u);
            row_sync<kBar>();
            find_bin(remaining);
            prefix |= sc.bin << sh;
            remaining = sc.rem;
        }
        T = prefix;
        take = remaining;
    }
    uint32_t gt_mask = 0, eq_mask = 0;
#pragma unroll
    for (int e = 0; e < kRowItems; ++e) {
        if (i0 + e < n) {
            gt_mask |= (key[e] > T ? 1u : 0u) << e;
            eq_mask |= (key[e] == T ? 1u : 0u) << e;
        }
    }
    const uint32_t packed = (static_cast<uint32_t>(__popc(gt_mask)) << 16) | __popc(eq_mask);
    uint32_t v = packed;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) sc.warp_tot[warp] = v;
    row_sync<kBar>();
    uint32_t add = 0;
    for (int w2 = 0; w2 < warp; ++w2) add += sc.warp_tot[w2];
    const uint32_t excl = v + add - packed;
    const uint32_t eq_before = excl & 0xffffu;
    uint32_t sel_mask = gt_mask;
    uint32_t eq_take = take > eq_before ? min(take - eq_before, static_cast<uint32_t>(__popc(eq_mask))) : 0u;
    uint32_t eqm = eq_mask;
    while (eq_take--) {
        const uint32_t low = eqm & (0u - eqm);
        sel_mask |= low;
        eqm ^= low;
    }
    uint32_t pos = (excl >> 16) + min(eq_before, take);
    while (sel_mask) {
        const int e = __ffs(sel_mask) - 1;
        sel_mask &= sel_mask - 1u;
        if (pos < static_cast<uint32_t>(m)) out[pos] = i0 + e;
        ++pos;
    }
    for (int i = m + tid; i < K; i += kRowThreads) out[i] = -1;
    if (tid == 0) *cnt_out = m;
}

}  // namespace svq
