// Query-aware page selection (the build_decode_view hook of the
// "add-sparse-method" skill page; Quest's query-relevant page selection on
// the SparseEngine summary page, section "method key points").
//
//   score_pages_kernel : upper-bound score of every (request, kv head, page)
//   topk_pages_kernel  : top-K pages per (request, kv head), ties to the lower
//                        page index, emitted in ascending page order
#include <algorithm>

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
// A page's metadata for all kv heads is contiguous (HKV x 512 bytes) and
// reaches shared memory as one bulk copy; a consumer lane's coefficients
// (its request's Qp or Qn over its channels) stay in registers for the
// CTA's whole run of pages.

#ifndef SVQ_SCORE_CONSUMERS
#define SVQ_SCORE_CONSUMERS 8
#endif
#ifndef SVQ_SCORE_RING_BYTES
#define SVQ_SCORE_RING_BYTES (128 * 1024)
#endif
constexpr int kScoreConsumers = SVQ_SCORE_CONSUMERS;
constexpr int kScoreThreads = (kScoreConsumers + 1) * 32;
constexpr int kScoreProducer = kScoreConsumers;   // warp index of the producer

// The scoring grid over a batch of (possibly very different) request lengths:
// with a one-dimensional grid of X >= B CTAs, request b gets
// k_b = 1 + floor((X - B) n_b / N) CTAs (N = the batch's pages; sum k_b <= X)
// that split its n_b pages evenly, so a CTA's load is at most about N / (X - B)
// pages whatever the length mix; the CTAs past sum k_b have nothing to do.
// Every warp works this out itself from the lengths (one coalesced load).
// With equal lengths k_b = floor(X / B), the split of a two-dimensional grid.
struct ScoreRun {
    int b;       // request, -1: no pages for this CTA
    int begin;   // first logical page
    int span;    // pages
    int n;       // the request's page count
};

constexpr int kLenSlots = 8;   // lengths a lane holds: the split by length serves up to 256 requests

__device__ __forceinline__ int pages_of(int len, int max_pages, bool flag) {
    int n = (len + kPage - 1) / kPage;
    if (len < 1 || n > max_pages) {
        if (flag) svq_flag(SV_DEVERR_SEQ_LEN);
        n = len < 1 ? 0 : max_pages;
    }
    return n;
}

// lens[i] = the length of request lane + 32 i (loaded by the caller).
__device__ __forceinline__ ScoreRun run_by_length(const int (&lens)[kLenSlots], int batch, int max_pages, int cta,
                                                  int ctas, int lane, bool flag) {
    int n_of[kLenSlots];
    int64_t total = 0;
#pragma unroll
    for (int i = 0; i < kLenSlots; ++i) {
        n_of[i] = lane + 32 * i < batch ? pages_of(lens[i], max_pages, flag) : 0;
        total += n_of[i];
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    ScoreRun run = {-1, 0, 0, 0};
    int before = 0;   // CTAs of the requests before this chunk
#pragma unroll
    for (int i = 0; i < kLenSlots; ++i) {
        if (32 * i >= batch || run.b >= 0) break;   // warp-uniform
        const int r = 32 * i + lane;
        const int n = n_of[i];
        const int k = r < batch ? 1 + (total > 0 ? static_cast<int>(static_cast<int64_t>(ctas - batch) * n / total) : 0)
                                : 0;
        int incl = k;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const bool mine = r < batch && cta >= before + incl - k && cta < before + incl;
        const uint32_t hit = __ballot_sync(0xffffffffu, mine);
        if (hit) {
            const int src = __ffs(hit) - 1;
            const int x = cta - (before + __shfl_sync(0xffffffffu, incl - k, src));
            const int kb = __shfl_sync(0xffffffffu, k, src);
            const int nb = __shfl_sync(0xffffffffu, n, src);
            const int per = (nb + kb - 1) / kb;
            run.b = 32 * i + src;
            run.n = nb;
            run.begin = x * per;
            run.span = max(0, min(nb, run.begin + per) - run.begin);
        }
        before += __shfl_sync(0xffffffffu, incl, 31);
    }
    return run;
}

template <int HKV>
struct ScoreShape {
    static constexpr int kPageBytes = HKV * 2 * kHeadDim * 2;           // metadata of one page, all kv heads
    static constexpr int kSlotsRaw = SVQ_SCORE_RING_BYTES / kPageBytes;
    static constexpr int kSlots = kSlotsRaw >= 128 ? 128 : (kSlotsRaw < 32 ? 32 : kSlotsRaw / 32 * 32);   // multiple of 32
    static constexpr int kSmemBytes = kSlots * kPageBytes;
    static constexpr int L = 32 / HKV;      // lanes per kv head
    static constexpr int C = HKV;           // 16-byte chunks of a head's 512-byte row per lane
    static_assert(32 % HKV == 0, "kv heads per page must divide 32");
    // Each ring slot must always be consumed by the same warp: a second warp
    // waiting on the slot's barrier for a later phase would see that phase's
    // parity as already complete.
    static_assert(kSlots % kScoreConsumers == 0, "ring slots must be a multiple of the consumer warps");
    static_assert(kSlots <= kScoreThreads, "one thread initialises each slot's barriers");
};

// Warp-specialised streaming of page metadata.  Each CTA owns a contiguous
// run of one request's pages.  Producer lane l handles pages l, l + 32, ...
// of the run: it waits until the ring slot (page mod kSlots) is free, then
// moves the page's metadata (all kv heads, contiguous) with one bulk copy
// that completes on the slot's "full" mbarrier; the 32 lanes keep up to 32
// copies being issued at once.  Consumer warp c scores pages c, c + C, ...:
// lane (j, k) = (lane / L, lane % L) owns kv head j and the 16-byte chunks
// k, k + L, ... of that head's 512-byte [kmin | kmax] row, so a page's score
// is one register accumulation per lane plus a log2(L)-level shuffle sum;
// the warp then releases the slot on its "empty" mbarrier.
//
// PER_HEAD: one score row per query head (no sum over the group): lane (u, k)
// = (lane / 4, lane % 4) scores query head u of every kv head j over channels
// 32k .. 32k+31 with the bound's per-channel form, q >= 0 ? q kmax : q kmin
// (the larger of the two products), and the four channel quarters are summed
// by two shuffles.  Rows are [B][Hkv * group][max_pages].
// Forced pages (the first `sink` and last `window` pages of a request) get
// the score +inf, which the top-K ranks first, ties to the lower index.
template <int HKV, bool PER_HEAD>
__global__ void __launch_bounds__(kScoreThreads, 1) score_pages_kernel(
    const __nv_bfloat16* __restrict__ meta, int64_t num_phys_pages, const __nv_bfloat16* __restrict__ q,
    int group, const int32_t* __restrict__ page_table, const int32_t* __restrict__ seq_lens, int max_pages,
    int pages_per_cta, int sink, int window, float* __restrict__ scores, int batch, int q_after_wait) {
    using S = ScoreShape<HKV>;
    constexpr int kSlots = S::kSlots, L = S::L, C = S::C;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ float coef[HKV][2][kHeadDim];   // [j][0] = Qn (pairs kmin), [j][1] = Qp (pairs kmax)
    __shared__ __align__(8) uint64_t full_bar[kSlots];
    __shared__ __align__(8) uint64_t empty_bar[kSlots];
    __shared__ unsigned char slot_ok[kSlots];
    __shared__ __align__(16) __nv_bfloat16 qstage[HKV * kMaxGroup * kHeadDim];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t full0 = smem_addr(&full_bar[0]);
    const uint32_t empty0 = smem_addr(&empty_bar[0]);

    // A two-dimensional grid gives request blockIdx.y the runs of
    // pages_per_cta pages; a one-dimensional grid splits the batch by length
    // (run_by_length), and pages_per_cta is then the run its CTA has when all
    // requests are full (floor(X / B) runs each), the guess under which the
    // first page-table entries and the query are fetched before the lengths
    // are known.
    const bool by_length = gridDim.y == 1 && batch > 1;
    int b = blockIdx.y;
    int cta_begin = blockIdx.x * pages_per_cta;
    if (by_length) {
        const int per_req = gridDim.x / batch;
        b = blockIdx.x / per_req;
        cta_begin = (blockIdx.x % per_req) * pages_per_cta;
        if (b >= batch) b = batch - 1, cta_begin = max_pages;   // no guess: fetched after the lengths
    }
    const int guess_b = b, guess_begin = cta_begin;
    // Consumers fetch the (guessed) request's query, Hq x 128 bf16 (at most
    // 16 KB), with 16-byte loads now, and keep it if the guess holds.
    constexpr int kConsumerThreads = kScoreConsumers * 32;
    constexpr int kQVecs = (HKV * kMaxGroup * kHeadDim / 8 + kConsumerThreads - 1) / kConsumerThreads;
    const int hq = HKV * group;
    uint4 qpre[kQVecs];
    if (warp != kScoreProducer && !q_after_wait) {
        const uint4* qsrc = reinterpret_cast<const uint4*>(q + static_cast<int64_t>(b) * hq * kHeadDim);
#pragma unroll
        for (int i = 0; i < kQVecs; ++i) {
            const int v = threadIdx.x + i * kConsumerThreads;
            qpre[i] = v < hq * kHeadDim / 8 ? qsrc[v] : make_uint4(0u, 0u, 0u, 0u);
        }
    }

    // The page table, like q and the lengths, is an input of the step.  The
    // producer's first 32 entries (inside the table's row whatever the
    // request's length) load together with the length, so the first copies
    // wait for one memory round trip, not two.
    const int32_t* pt_row = page_table + static_cast<int64_t>(b) * max_pages + cta_begin;
    int nxt = (warp == kScoreProducer && cta_begin + lane < max_pages) ? pt_row[lane] : 0;
    const int len = seq_lens[b];
    int lens[kLenSlots];
#pragma unroll
    for (int i = 0; i < kLenSlots; ++i) lens[i] = by_length && lane + 32 * i < batch ? seq_lens[lane + 32 * i] : 0;

    if (threadIdx.x < kSlots) {
        mbar_init(full0 + threadIdx.x * 8, 1);
        mbar_init(empty0 + threadIdx.x * 8, 1);
        mbar_init_fence();
    }
    __syncthreads();
    // The top-K kernel that follows may be scheduled now; its CTAs land as
    // this kernel's CTAs retire, and wait for its completion to read scores.
    pdl_launch_dependents();

    int n, span;
    bool all_full = by_length;   // every request fills the table's row: the guess is the split
    if (by_length) {
#pragma unroll
        for (int i = 0; i < kLenSlots; ++i)
            if (lane + 32 * i < batch) all_full &= lens[i] >= 1 && (lens[i] + kPage - 1) / kPage == max_pages;
        all_full = __all_sync(0xffffffffu, all_full);
    }
    if (all_full) {
        n = max_pages;
        span = max(0, min(n, cta_begin + pages_per_cta) - cta_begin);
    } else if (by_length) {
        const ScoreRun run = run_by_length(lens, batch, max_pages, blockIdx.x, gridDim.x, lane,
                                           warp == 0 && blockIdx.x == 0);
        n = run.n;
        span = run.span;
        b = run.b < 0 ? guess_b : run.b;
        cta_begin = run.begin;
        if (warp == kScoreProducer && (b != guess_b || cta_begin != guess_begin)) {
            // Another split than the guess (unequal lengths): fetch the entries now.
            pt_row = page_table + static_cast<int64_t>(b) * max_pages + cta_begin;
            nxt = lane < span ? pt_row[lane] : 0;
        }
    } else {
        n = (len + kPage - 1) / kPage;
        if (len < 1 || n > max_pages) {
            if (threadIdx.x == 0 && blockIdx.x == 0) svq_flag(SV_DEVERR_SEQ_LEN);
            n = len < 1 ? 0 : max_pages;
        }
        span = max(0, min(n, cta_begin + pages_per_cta) - cta_begin);
    }

    if (warp != kScoreProducer) {
        // Consumers stage this request's query in shared memory and fold each
        // kv group's query heads into Qp / Qn, while the producer already
        // streams metadata.  q is an input of the step, so this also overlaps
        // the previous kernel.
        // With q_after_wait the query is written by the kernel launched just
        // before (a copy of a host-resident query): wait for it first.
        if (q_after_wait) pdl_wait();
        {
            const uint4* qsrc = reinterpret_cast<const uint4*>(q + static_cast<int64_t>(b) * hq * kHeadDim);
            uint4* qdst = reinterpret_cast<uint4*>(qstage);
            const bool kept = b == guess_b && !q_after_wait;
#pragma unroll
            for (int i = 0; i < kQVecs; ++i) {
                const int v = threadIdx.x + i * kConsumerThreads;
                if (v < hq * kHeadDim / 8) qdst[v] = kept ? qpre[i] : qsrc[v];
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
        for (int idx = threadIdx.x; idx < HKV * kHeadDim; idx += kConsumerThreads) {
            const int j = idx / kHeadDim, ch = idx % kHeadDim;
            float qp = 0.f, qn = 0.f;
            for (int h = 0; h < group; ++h) {
                const float v = __bfloat162float(qstage[(j * group + h) * kHeadDim + ch]);
                qp += fmaxf(v, 0.f);
                qn += fminf(v, 0.f);
            }
            coef[j][0][ch] = qn;
            coef[j][1][ch] = qp;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
    }
    // Metadata may come from an append launched just before, and the previous
    // step's top-K may still read the score buffer.
    pdl_wait();

    if (warp == kScoreProducer) {
        const unsigned char* meta_bytes = reinterpret_cast<const unsigned char*>(meta);
        const uint32_t ring_s = smem_addr(ring);
        int issued_last = -1;   // highest page this lane issued
        bool failed = false;
        const uint64_t policy = l2_evict_first_policy();
        for (int p = lane; p < span; p += 32) {
            const int phys = nxt;
            if (p + 32 < span) nxt = pt_row[p + 32];
            const int slot = p % kSlots;
            if (p >= kSlots && !mbar_wait_bounded(empty0 + slot * 8, ((p / kSlots) - 1) & 1)) {
                failed = true;
                break;
            }
            const uint32_t fb = full0 + slot * 8;
            const bool ok = static_cast<uint32_t>(phys) < static_cast<uint64_t>(num_phys_pages);
            slot_ok[slot] = ok ? 1 : 0;
            if (ok) {
                mbar_arrive_expect_tx(fb, S::kPageBytes);
                bulk_copy_g2s_hint(ring_s + slot * S::kPageBytes,
                                   meta_bytes + static_cast<int64_t>(phys) * S::kPageBytes, S::kPageBytes, fb, policy);
            } else {
                svq_flag(SV_DEVERR_PAGE_TABLE);
                mbar_arrive(fb);
            }
            issued_last = p;
        }
        if (failed) svq_flag(SV_DEVERR_TIMEOUT);
        // This lane's copies land before the CTA (and its shared memory) retires.
        for (int p = issued_last; p >= 0 && p > issued_last - kSlots; p -= 32)
            (void)mbar_wait_bounded(full0 + (p % kSlots) * 8, (p / kSlots) & 1);
        return;
    }

    // ---------------- consumer warps
    auto forced = [&](int lp) { return lp < sink || lp >= n - window; };
    if constexpr (PER_HEAD) {
        const int u = lane >> 2, kq = lane & 3;
        const bool active = u < group;
        uint4 qreg[HKV][4];   // query head u of kv head j, channels 32 kq .. 32 kq + 31
#pragma unroll
        for (int j = 0; j < HKV; ++j) {
            const __nv_bfloat16* qrow = qstage + (j * group + (active ? u : 0)) * kHeadDim + kq * 32;
#pragma unroll
            for (int t = 0; t < 4; ++t) qreg[j][t] = *reinterpret_cast<const uint4*>(qrow + t * 8);
        }
        const int rows = HKV * group;
        for (int p = warp; p < span; p += kScoreConsumers) {
            const int slot = p % kSlots;
            const bool okw = mbar_wait_bounded(full0 + slot * 8, (p / kSlots) & 1);
            if (__any_sync(0xffffffffu, !okw)) {
                if (lane == 0) svq_flag(SV_DEVERR_TIMEOUT);
                break;
            }
            const unsigned char* page = ring + slot * S::kPageBytes;
            float acc[HKV];
#pragma unroll
            for (int j = 0; j < HKV; ++j) {
                const unsigned char* mrow = page + j * 512 + kq * 64;   // kmin at +0, kmax at +256
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint4 mn = *reinterpret_cast<const uint4*>(mrow + t * 16);
                    const uint4 mx = *reinterpret_cast<const uint4*>(mrow + 256 + t * 16);
                    const uint32_t a[4] = {mn.x, mn.y, mn.z, mn.w};
                    const uint32_t bb[4] = {mx.x, mx.y, mx.z, mx.w};
                    const uint32_t c4[4] = {qreg[j][t].x, qreg[j][t].y, qreg[j][t].z, qreg[j][t].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float q0 = bf16lo(c4[e]), q1 = bf16hi(c4[e]);
                        s0 = fmaf(q0, q0 >= 0.f ? bf16lo(bb[e]) : bf16lo(a[e]), s0);
                        s1 = fmaf(q1, q1 >= 0.f ? bf16hi(bb[e]) : bf16hi(a[e]), s1);
                    }
                }
                acc[j] = s0 + s1;
            }
            const bool real = slot_ok[slot] != 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + slot * 8);
            const int lp = cta_begin + p;
            const bool f = forced(lp);
#pragma unroll
            for (int j = 0; j < HKV; ++j) {
                float v = acc[j] + __shfl_xor_sync(0xffffffffu, acc[j], 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                if (kq == 0 && active)
                    scores[(static_cast<int64_t>(b) * rows + j * group + u) * max_pages + lp] =
                        f ? INFINITY : (real ? v : 0.f);
            }
        }
        return;
    }
    const int hj = lane / L;        // kv head of this lane
    const int hk = lane % L;        // first chunk of this lane
    float c[C][8];
#pragma unroll
    for (int t = 0; t < C; ++t) {
        const int chunk = hk + L * t;   // chunks < 16 hold kmin channels, >= 16 kmax
#pragma unroll
        for (int i = 0; i < 8; ++i) c[t][i] = coef[hj][chunk >> 4][(chunk & 15) * 8 + i];
    }
    float* score_row = scores + (static_cast<int64_t>(b) * HKV + hj) * max_pages + cta_begin;
    const unsigned char* lane_base = ring + hj * 512 + hk * 16;
    for (int p = warp; p < span; p += kScoreConsumers) {
        const int slot = p % kSlots;
        const bool okw = mbar_wait_bounded(full0 + slot * 8, (p / kSlots) & 1);
        if (__any_sync(0xffffffffu, !okw)) {
            if (lane == 0) svq_flag(SV_DEVERR_TIMEOUT);
            break;
        }
        uint4 w[C];
#pragma unroll
        for (int t = 0; t < C; ++t)
            w[t] = *reinterpret_cast<const uint4*>(lane_base + slot * S::kPageBytes + t * L * 16);
        const bool real = slot_ok[slot] != 0;
        __syncwarp();   // every lane has read the slot before it is released
        if (lane == 0) mbar_arrive(empty0 + slot * 8);
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
        float acc = real ? a0 + a1 : 0.f;
#pragma unroll
        for (int m = 1; m < L; m <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (hk == 0) score_row[p] = forced(cta_begin + p) ? INFINITY : acc;
    }
}

template <int HKV, bool PER_HEAD>
int launch_score_hkv(const sv_cache* c, const __nv_bfloat16* q, int group, const int32_t* page_table,
                     const int32_t* seq_lens, int batch, int max_pages, int sink, int window, float* scores,
                     int sm_count, cudaStream_t stream, int q_after_wait) {
    using S = ScoreShape<HKV>;
    static std::atomic<bool> attr_set[64];
    const int st = once_per_device(attr_set, [] {
        return cudaFuncSetAttribute(score_pages_kernel<HKV, PER_HEAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    S::kSmemBytes) == cudaSuccess
                   ? SV_OK
                   : SV_ERR_CUDA;
    });
    if (st) return st;
    // At most one wave of one CTA per SM.  Up to SM-count requests: a
    // one-dimensional grid of X CTAs (at least 32 pages each when the
    // requests are full) that the kernel splits by the actual lengths, and
    // the run a CTA has when all requests are full (the kernel's guess).
    // More requests: one CTA each, in waves.
    dim3 grid;
    int64_t ppc;
    if (batch > 1 && batch <= sm_count && batch <= 32 * kLenSlots) {
        const int64_t want = (static_cast<int64_t>(batch) * max_pages + 31) / 32;
        const int X = static_cast<int>(std::min<int64_t>(sm_count, std::max<int64_t>(batch, want)));
        const int per_req = X / batch;
        ppc = (static_cast<int64_t>(max_pages) + per_req - 1) / per_req;
        grid = dim3(X, 1);
    } else {
        const int per_req = max(1, sm_count / batch);
        ppc = (static_cast<int64_t>(max_pages) + per_req - 1) / per_req;
        if (ppc < 32) ppc = 32;
        grid = dim3(ceil_div(max_pages, ppc), batch);
    }
    const cudaError_t e = launch_pdl(score_pages_kernel<HKV, PER_HEAD>, grid, dim3(kScoreThreads), S::kSmemBytes,
                                     stream, static_cast<const __nv_bfloat16*>(c->meta), c->num_phys_pages, q, group,
                                     page_table, seq_lens, max_pages, static_cast<int>(ppc), sink, window, scores,
                                     batch, q_after_wait);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

int launch_score(const sv_cache* c, const void* q, int num_q_heads, const int32_t* page_table,
                 const int32_t* seq_lens, int batch, int max_pages, bool per_q_head, int sink, int window,
                 float* scores, int sm_count, cudaStream_t stream, int q_after_wait) {
    const int group = num_q_heads / c->num_kv_heads;
    const auto* qq = static_cast<const __nv_bfloat16*>(q);
#define SVQ_SCORE_CASE(H)                                                                                      \
    case H:                                                                                                    \
        return per_q_head ? launch_score_hkv<H, true>(c, qq, group, page_table, seq_lens, batch, max_pages,   \
                                                      sink, window, scores, sm_count, stream, q_after_wait)   \
                          : launch_score_hkv<H, false>(c, qq, group, page_table, seq_lens, batch, max_pages,  \
                                                       sink, window, scores, sm_count, stream, q_after_wait);
    switch (c->num_kv_heads) {
        SVQ_SCORE_CASE(1)
        SVQ_SCORE_CASE(2)
        SVQ_SCORE_CASE(4)
        SVQ_SCORE_CASE(8)
        default: return SV_ERR_UNSUPPORTED;
    }
#undef SVQ_SCORE_CASE
}

// ---------------------------------------------------------------- top-K
//
// One CTA per (request, kv head).  Scores become order-preserving 32-bit
// keys held in registers (each thread a run of consecutive pages).  The
// threshold search is a selection, not a sort:
//  1. one histogram over [min key, max key] in 2048 power-of-two-wide bins
//     (a bin index is a right shift of key - min, so bins are monotone in the
//     score) locates the bin b* holding the K-th best key; forced pages (+inf)
//     stay out of the max and join the top bin, so that a few of them do not
//     squeeze every scored page into a handful of bins;
//  2. if b* holds few keys (<= kCandCap), each of them gets its exact rank in
//     (key desc, page asc) order by comparing against the others, which gives
//     the threshold key T and how many keys equal to T are taken;
//     otherwise three radix passes (11, 11, 10 bits) over all keys find T.
// A block-wide scan over contiguous index segments then emits, in ascending
// index order, every page above T and the lowest-indexed pages equal to T.

#ifndef SVQ_TOPK_THREADS
#define SVQ_TOPK_THREADS 1024
#endif
constexpr int kTopkThreads = SVQ_TOPK_THREADS;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kRadixBins = 2048;
constexpr int kBinsPerThread = kRadixBins / kTopkThreads;
constexpr int kCandCap = 256;
static_assert(kRadixBins % kTopkThreads == 0 && kTopkWarps <= 32, "top-K block shape");

__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide inclusive scan of one value per thread: a warp scan, then each
// warp adds up the totals of the warps before it, read after one barrier.
// With reuse = false the caller promises that warp_tot is not written again
// before the block's next barrier, which saves a second one.
template <bool reuse = true>
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    const uint32_t add = __reduce_add_sync(0xffffffffu, lane < warp ? warp_tot[lane] : 0u);
    if (reuse) __syncthreads();   // warp_tot may be reused right after
    return v + add;
}

// Finds, over a 2048-bin histogram, the bin holding the `remaining`-th key
// counted from the top, and how many keys of that bin are still needed.
__device__ __forceinline__ void find_bin_from_top(const uint32_t* hist, uint32_t remaining, uint32_t* warp_tot,
                                                  uint32_t* s_bin, uint32_t* s_rem) {
    const int tid = threadIdx.x;
    // Thread t owns kBinsPerThread consecutive bins counted down from the top.
    const uint32_t top = kRadixBins - 1 - kBinsPerThread * tid;
    uint32_t cnt[kBinsPerThread];
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < kBinsPerThread; ++i) {
        cnt[i] = hist[top - i];
        sum += cnt[i];
    }
    // warp_tot is next written after the barrier that ends this function.
    uint32_t before = block_inclusive_scan<false>(sum, warp_tot) - sum;   // keys in strictly higher bins
#pragma unroll
    for (int i = 0; i < kBinsPerThread; ++i) {
        if (before < remaining && remaining <= before + cnt[i]) {
            *s_bin = top - i;
            *s_rem = remaining - before;
        }
        before += cnt[i];
    }
    __syncthreads();
}

// Keys live in registers: thread t holds the ITEMS consecutive pages
// [ITEMS t, ITEMS t + ITEMS) of the row (n <= ITEMS * kTopkThreads), so the
// final compaction emits in ascending page order from per-thread bit masks.
template <int ITEMS>
__global__ void __launch_bounds__(kTopkThreads) topk_pages_kernel(const float* __restrict__ scores,
                                                                  const int32_t* __restrict__ seq_lens,
                                                                  int num_kv_heads, int max_pages, int K,
                                                                  int32_t* __restrict__ sel_idx,
                                                                  int32_t* __restrict__ sel_cnt) {
    static_assert(ITEMS <= 32, "selection masks are 32 bits");
    __shared__ uint32_t hist[kRadixBins];
    __shared__ uint32_t warp_tot[kTopkWarps];
    __shared__ uint32_t warp_lo[kTopkWarps], warp_hi[kTopkWarps];
    __shared__ uint32_t cand_key[kCandCap];
    __shared__ int32_t cand_idx[kCandCap];
    __shared__ uint32_t s_bin, s_rem, s_cand, s_T, s_take;

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
    for (int i = tid; i < kRadixBins; i += kTopkThreads) hist[i] = 0u;
    if (tid == 0) s_cand = 0u;
    // The attention kernel that follows may start now: its CTAs set up and
    // load q while this one runs, and wait for its completion before they
    // read the selection.
    pdl_launch_dependents();
    pdl_wait();   // scores come from the scoring kernel launched just before
    if (n <= K) {
        for (int i = tid; i < K; i += kTopkThreads) out[i] = i < n ? i : -1;
        if (tid == 0) sel_cnt[bg] = n;
        return;
    }

    // 1. this thread's keys, min and max.
    const float* row = scores + static_cast<int64_t>(bg) * max_pages;
    const int i0 = ITEMS * tid;
    float f[ITEMS];
    if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0 && i0 + ITEMS <= n) {
#pragma unroll
        for (int e = 0; e < ITEMS; e += 4) {
            const float4 v = *reinterpret_cast<const float4*>(row + i0 + e);
            f[e] = v.x; f[e + 1] = v.y; f[e + 2] = v.z; f[e + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < ITEMS; ++e) f[e] = i0 + e < n ? row[i0 + e] : 0.f;
    }
    // Forced pages score +inf; they stay out of the maximum, so that the
    // histogram spans the scored pages, and land in the top bin.
    constexpr uint32_t kForcedKey = 0xff800000u;   // order_key(+inf)
    uint32_t key[ITEMS];
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int e = 0; e < ITEMS; ++e) {
        key[e] = order_key(f[e]);
        if (i0 + e < n) {
            lo = min(lo, key[e]);
            if (key[e] != kForcedKey) hi = max(hi, key[e]);
        }
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) {
        warp_lo[warp] = lo;
        warp_hi[warp] = hi;
    }
    __syncthreads();
    // Every warp folds the per-warp values itself (no second barrier).
    lo = __reduce_min_sync(0xffffffffu, lane < kTopkWarps ? warp_lo[lane] : 0xffffffffu);
    hi = __reduce_max_sync(0xffffffffu, lane < kTopkWarps ? warp_hi[lane] : 0u);
    hi = max(hi, lo);   // every page forced
    const uint32_t range = hi - lo;
    const int range_bits = range == 0 ? 0 : 32 - __clz(range);            // range < 2^bits
    const uint32_t shift = range_bits > 11 ? range_bits - 11 : 0;        // (range >> shift) < 2048
    // Bins are monotone in the key; keys above hi (forced pages) join the top bin.
    auto bin_of = [&](uint32_t k) { return min((k - lo) >> shift, static_cast<uint32_t>(kRadixBins - 1)); };

    // 2. histogram of the bins; bin of the m-th best key.
#pragma unroll
    for (int e = 0; e < ITEMS; ++e)
        if (i0 + e < n) atomicAdd(&hist[bin_of(key[e])], 1u);
    __syncthreads();
    find_bin_from_top(hist, static_cast<uint32_t>(m), warp_tot, &s_bin, &s_rem);
    const uint32_t bstar = s_bin, need = s_rem;
    uint32_t T, take;
    if (hist[bstar] <= kCandCap) {
        // 3a. exact rank of each key of bin b* among the others.
#pragma unroll
        for (int e = 0; e < ITEMS; ++e) {
            if (i0 + e < n && bin_of(key[e]) == bstar) {
                const uint32_t pos = atomicAdd(&s_cand, 1u);
                cand_key[pos] = key[e];
                cand_idx[pos] = i0 + e;
            }
        }
        __syncthreads();
        const int nc = static_cast<int>(s_cand);
        // rank = keys above mine + equal keys at lower pages; the candidate
        // ranked need - 1 is the threshold T, and the keys equal to T that are
        // taken are those ranked at or before it: need - (keys above T).
        auto rank = [&](int c, uint32_t& my_k, uint32_t& above) {
            my_k = cand_key[c];
            const int my_i = cand_idx[c];
            uint32_t tied_before = 0;
            above = 0;
            for (int j = 0; j < nc; ++j) {
                const uint32_t kj = cand_key[j];
                above += kj > my_k;
                tied_before += (kj == my_k && cand_idx[j] < my_i);
            }
            return above + tied_before == need - 1;
        };
        if (nc <= 32) {
            // Few candidates (the usual case): every warp ranks them all, one
            // per lane, so the threshold needs no further barrier.
            uint32_t my_k = 0, above = 0;
            const bool hit = lane < nc && rank(lane, my_k, above);
            const int src = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;   // exactly one candidate hits
            T = __shfl_sync(0xffffffffu, my_k, src);
            take = need - __shfl_sync(0xffffffffu, above, src);
        } else {
            if (tid < nc) {
                uint32_t my_k, above;
                if (rank(tid, my_k, above)) {
                    s_T = my_k;
                    s_take = need - above;
                }
            }
            __syncthreads();
            T = s_T;
            take = s_take;
        }
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
#pragma unroll
            for (int e = 0; e < ITEMS; ++e)
                if (i0 + e < n && (key[e] & hi_mask) == prefix) atomicAdd(&hist[(key[e] >> sh) & (nbins - 1u)], 1u);
            __syncthreads();
            find_bin_from_top(hist, remaining, warp_tot, &s_bin, &s_rem);
            prefix |= s_bin << sh;
            remaining = s_rem;
        }
        T = prefix;
        take = remaining;
    }

    // 4. ordered compaction: every key above T, and the `take` lowest-indexed keys equal to T.
    uint32_t gt_mask = 0, eq_mask = 0;
#pragma unroll
    for (int e = 0; e < ITEMS; ++e) {
        if (i0 + e < n) {
            gt_mask |= (key[e] > T ? 1u : 0u) << e;
            eq_mask |= (key[e] == T ? 1u : 0u) << e;
        }
    }
    const uint32_t gt = __popc(gt_mask), eq = __popc(eq_mask);
    const uint32_t packed = (gt << 16) | eq;   // n <= 32768 keeps both halves in 16 bits
    const uint32_t excl = block_inclusive_scan<false>(packed, warp_tot) - packed;
    const uint32_t eq_before = excl & 0xffffu;
    uint32_t sel_mask = gt_mask;
    uint32_t eq_take = take > eq_before ? min(take - eq_before, eq) : 0u;
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
    for (int i = m + tid; i < K; i += kTopkThreads) out[i] = -1;
    if (tid == 0) sel_cnt[bg] = m;
}

int launch_topk(const float* scores, const int32_t* seq_lens, int batch, int num_kv_heads, int max_pages,
                int budget_pages, int32_t* sel_idx, int32_t* sel_cnt, cudaStream_t stream) {
    cudaError_t e;
    const dim3 grid(batch * num_kv_heads), block(kTopkThreads);
    if (max_pages <= 8 * kTopkThreads)
        e = launch_pdl(topk_pages_kernel<8>, grid, block, 0, stream, scores, seq_lens, num_kv_heads, max_pages,
                       budget_pages, sel_idx, sel_cnt);
    else if (max_pages <= 16 * kTopkThreads)
        e = launch_pdl(topk_pages_kernel<16>, grid, block, 0, stream, scores, seq_lens, num_kv_heads, max_pages,
                       budget_pages, sel_idx, sel_cnt);
    else if (max_pages <= 32 * kTopkThreads)
        e = launch_pdl(topk_pages_kernel<32>, grid, block, 0, stream, scores, seq_lens, num_kv_heads, max_pages,
                       budget_pages, sel_idx, sel_cnt);
    else
        return SV_ERR_UNSUPPORTED;
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace svq
