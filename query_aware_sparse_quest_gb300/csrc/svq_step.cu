// sv_quest_decode_step: the whole decode step -- page scoring, top-K page
// selection, split-K attention over the selected pages and the log-sum-exp
// combine -- as one persistent, cooperative launch (two CTAs per SM, all
// co-resident).
//
// Every CTA has eight compute warps, a producer warp (TMA) and a control warp
// that does all of the CTA's cross-CTA signalling (work claims, readiness
// waits, releases), so compute warps never stall on a global round trip.
// Roles, by CTA index:
//   score     : stream, request by request, this CTA's slice of the page
//               metadata (bulk copies into a shared-memory ring) and write the
//               page scores; the control warp publishes "slice of request b
//               scored" once all eight compute warps are past it.
//   selector  : per (request, kv head) of its share, wait until every score
//               CTA has published the request, run the top-K over the score row
//               and publish the selection.
//   then all  : a request-major queue of attention items -- (request, kv head,
//               split) page ranges of the selection, then one combine item per
//               (request, kv head), placed one request later.  The control warp
//               claims an item and waits for its inputs, the producer streams
//               the split's K/V boxes while the compute warps still work on the
//               previous item, and the compute warps run the tensor-core flash
//               decode loop; a combine item merges the splits by log-sum-exp.
// So the selection and attention of request b overlap the scoring of b+1, ...
// Every cross-CTA wait is bounded and waits on work that a co-resident CTA
// owns and finishes without waiting on the waiter: score CTAs wait on nothing,
// selectors on score CTAs, attention items on selectors, combine items on
// attention items of lower queue index.

#include <cuda.h>
#include <cudaTypedefs.h>

#include "svq_common.cuh"
#include "svq_topk.cuh"

namespace svq {

SVQ_DEFINE_ERROR_WORD(read_error_step)

constexpr int kStepConsumers = 8;                          // compute warps
constexpr int kStepProducer = kStepConsumers;              // warp 8
constexpr int kStepControl = kStepConsumers + 1;           // warp 9
constexpr int kStepThreads = (kStepConsumers + 2) * 32;    // 320
constexpr int kComputeThreads = kStepConsumers * 32;       // 256
constexpr int kStepRingBytes = 64 * 1024;
constexpr int kBox = kPage * 64 * 2;                       // 16 x 64 bf16 TMA box (2 KB)
constexpr int kKvStage = 4 * kBox;                         // K lo | K hi | V lo | V hi
constexpr int kKvStages = kStepRingBytes / kKvStage;       // 8: stage s is consumed by warp s
constexpr int kStepMaxPages = kRowMaxPages;               // 8192 pages (131072 tokens) per request
constexpr int kStepMaxSplits = 64;
constexpr uint32_t kSpinLimit = 1u << 24;                  // polls of a cross-CTA counter before giving up
// Merge area for the eight warps' partial outputs: o [8][8 heads][128] + m, l [8][8].
constexpr int kMergeBytes = kStepConsumers * kMaxGroup * (kHeadDim + 2) * 4;
static_assert(kKvStages == kStepConsumers, "each ring stage belongs to one compute warp");
static_assert(kStepMaxPages * 4 <= kStepRingBytes, "a score row must fit the ring for the top-K");
static_assert(kComputeThreads == kRowThreads, "the compute warps run the row top-K");

#ifndef SVQ_STEP_PAGES_PER_SPLIT
#define SVQ_STEP_PAGES_PER_SPLIT 16
#endif
#ifndef SVQ_STEP_SCORE_PERMILLE
#define SVQ_STEP_SCORE_PERMILLE 0   // 0: one score CTA per SM
#endif
#ifndef SVQ_STEP_SELECTORS_PER_HEAD
#define SVQ_STEP_SELECTORS_PER_HEAD 4
#endif
#ifndef SVQ_STEP_POLL_NS
#define SVQ_STEP_POLL_NS 256   // sleep between polls of a cross-CTA counter
#endif
#ifndef SVQ_STEP_IDLE_NS
#define SVQ_STEP_IDLE_NS 128   // sleep between polls of an idle warp waiting for its next item
#endif

struct StepArgs {
    const __nv_bfloat16* meta;
    int64_t num_phys_pages;
    const __nv_bfloat16* q;
    int num_q_heads;
    int group;
    const int32_t* page_table;
    const int32_t* seq_lens;
    int batch;
    int max_pages;
    int K;
    float scale_log2;
    float* scores;            // [B][Hkv][score_stride]
    int score_stride;         // max_pages rounded up to 32
    int32_t* sel_idx;         // [B][Hkv][K]
    int32_t* sel_cnt;         // [B][Hkv]
    float* o_part;            // [B][Hq][splits][128]
    float2* ml_part;          // [B][Hq][splits]
    __nv_bfloat16* out;       // [B][Hq][128]
    float* lse;               // [B][Hq]
    int score_ctas;           // CTAs [0, score_ctas) score
    int sel_ctas;             // CTAs [score_ctas, score_ctas + sel_ctas) select
    int splits;               // attention items per (request, kv head)
    uint32_t* ctr;            // [0] next queue item, [1 + b] score CTAs done with request b,
                              // [1 + B + bg] selection of bg published, [1 + B + BH + bg] splits done
};

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ float step_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// 128-byte swizzle of a 16 x 64 bf16 box (chunk = 16 bytes).
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
// Barrier of the eight compute warps only.
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kComputeThreads) : "memory"); }

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Data that other CTAs of this launch wrote is read after an acquire (by this
// thread, or by another thread followed by a barrier) with L2 loads (__ldcg),
// which the compiler may batch; L1 may hold stale copies, L2 does not.
__device__ __forceinline__ int ld_relaxed_i32(const int32_t* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Adds v to a global counter, ordered after every write this thread has
// observed (its own and, through barriers, its CTA's).
__device__ __forceinline__ void red_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_cta_smem(uint32_t* p, uint32_t v) {
    asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_cta_smem(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}

// Polls a counter written by other CTAs until it reaches `target` (acquire;
// bounded).
__device__ __forceinline__ bool wait_counter(const uint32_t* p, uint32_t target) {
    for (uint32_t it = 0; it < kSpinLimit; ++it) {
        if (ld_acquire_gpu(p) >= target) return true;
        __nanosleep(SVQ_STEP_POLL_NS);
    }
    return false;
}

// Waits for an item-slot phase; the waiting warps sleep between polls so
// that they take few issue slots from the CTA that shares their SM.
__device__ __forceinline__ bool wait_item(uint32_t bar, uint32_t parity) {
    for (uint32_t it = 0; it < kMbarPollLimit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (SVQ_STEP_IDLE_NS > 0) __nanosleep(SVQ_STEP_IDLE_NS);
    }
    return false;
}

__device__ __forceinline__ int pages_of(const StepArgs& a, int b, int& len) {
    len = a.seq_lens[b];
    int n = (len + kPage - 1) / kPage;
    if (len < 1 || n > a.max_pages) {
        svq_flag(SV_DEVERR_SEQ_LEN);
        n = len < 1 ? 0 : a.max_pages;
    }
    return n;
}

template <int HKV>
struct StepScoreShape {
    static constexpr int kPageBytes = HKV * 2 * kHeadDim * 2;          // one page's metadata, all kv heads
    static constexpr int kSlots = kStepRingBytes / kPageBytes;          // 128 / 64 / 32 / 16 for HKV 1 / 2 / 4 / 8
    static constexpr int R = kSlots < 32 ? kSlots : 32;                 // pages issued per producer round
    static constexpr int L = 32 / HKV;                                  // compute lanes per kv head
    static constexpr int C = HKV;                                       // 16-byte chunks per lane per page
    static constexpr int kQBufBytes = kMaxGroup * HKV * kHeadDim * 2;   // one request's queries, at most
    static_assert(kSlots % R == 0 && kSlots % kStepConsumers == 0, "score ring shape");
    static_assert(2 * kQBufBytes <= kMergeBytes, "query buffers live in the merge area");
};

// ---------------------------------------------------------------- queue items
// Request-major: F(0), F(1), C(0), F(2), C(1), ..., F(B-1), C(B-2), C(B-1),
// where F(b) = Hkv * splits attention items and C(b) = Hkv combine items.
struct QueueItem {
    int kind;   // 0 stop, 1 attention, 2 combine
    int b, g, split;
};
template <int HKV>
__device__ __forceinline__ QueueItem decode_item(const StepArgs& a, int item) {
    QueueItem it{0, 0, 0, 0};
    const int nf = HKV * a.splits;
    const int total = a.batch * (nf + HKV);
    if (item < 0 || item >= total) return it;
    int j, r;
    if (item < nf) {
        j = 0;
        r = item;
    } else {
        const int x = item - nf;
        j = 1 + x / (nf + HKV);
        r = x - (j - 1) * (nf + HKV);
    }
    if (j < a.batch && r < nf) {
        it.kind = 1;
        it.b = j;
        it.g = r / a.splits;
        it.split = r - it.g * a.splits;
    } else {
        it.kind = 2;
        it.b = j - 1;
        it.g = j < a.batch ? r - nf : r;
    }
    return it;
}

// ---------------------------------------------------------------- top-K of one score row
// (svq_topk.cuh; the compute warps are threads 0 .. 255, barrier 1)
__device__ __forceinline__ void select_row(const StepArgs& a, RowTopkScratch& sc, float* stage, int bg, int n) {
    topk_row_256<1, true>(a.scores + static_cast<int64_t>(bg) * a.score_stride, n, a.K,
                          a.sel_idx + static_cast<int64_t>(bg) * a.K, a.sel_cnt + bg, sc, stage);
}

// ---------------------------------------------------------------- score role
// Producer: streams this CTA's slices of all requests as one flat sequence of
// pages, request-major, into ring slots (slot = sequence % slots), one page per
// lane per round; the page-table entries of the next round are loaded while
// the current round waits for free slots.  Compute warp w takes sequence
// numbers = w (mod 8), so each slot has one waiting warp.  Control warp:
// copies request b + 2's queries into q buffer b % 2 once the compute warps
// have folded request b's, and publishes request b once all eight compute
// warps are past it.
template <int HKV>
__device__ __forceinline__ void score_role(const StepArgs& a, unsigned char* ring, uint32_t ring_s, uint32_t full0,
                                           uint32_t empty0, unsigned char* slot_ok, const __nv_bfloat16* qbuf,
                                           uint32_t qbuf_s, uint32_t qfull0, uint32_t qempty0, uint32_t* req_done) {
    using SS = StepScoreShape<HKV>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    if (warp == kStepControl) {
        if (lane == 0) {
            const uint32_t q_bytes = static_cast<uint32_t>(a.num_q_heads) * kHeadDim * 2;
            const unsigned char* q_src = reinterpret_cast<const unsigned char*>(a.q);
            auto stage_q = [&](int b) {
                const int qb = b & 1;
                mbar_arrive_expect_tx(qfull0 + qb * 8, q_bytes);
                bulk_copy_g2s(qbuf_s + qb * SS::kQBufBytes, q_src + static_cast<int64_t>(b) * q_bytes, q_bytes,
                              qfull0 + qb * 8);
            };
            stage_q(0);
            if (a.batch > 1) stage_q(1);
            uint32_t* sdone = a.ctr + 1;
            for (int b = 0; b < a.batch; ++b) {
                if (b + 2 < a.batch) {
                    if (mbar_wait_bounded(qempty0 + (b & 1) * 8, (static_cast<uint32_t>(b) >> 1) & 1))
                        stage_q(b + 2);
                    else
                        svq_flag(SV_DEVERR_TIMEOUT);
                }
                bool ok = false;
                for (uint32_t it = 0; it < kSpinLimit; ++it) {
                    if (ld_acquire_cta_smem(req_done) >= static_cast<uint32_t>(kStepConsumers) * (b + 1)) {
                        ok = true;
                        break;
                    }
                    __nanosleep(32);
                }
                if (!ok) svq_flag(SV_DEVERR_TIMEOUT);
                red_release_gpu(sdone + b, 1u);
            }
        }
        return;
    }
    if (warp == kStepProducer) {
        // Lane l streams the pages at flat positions l, l + R, l + 2R, ... on its
        // own (no warp-wide rounds), so each slot is refilled as soon as its
        // page is consumed; the page-table entry of the lane's next page is
        // loaded before it waits for the current slot.
        if (lane >= SS::R) return;
        const unsigned char* meta_bytes = reinterpret_cast<const unsigned char*>(a.meta);
        const int B = a.batch;
        // Slice [lo, hi) of request b (clamped like pages_of, which flags).
        auto slice = [&](int b, int& lo, int& hi) {
            const int len = __ldg(a.seq_lens + b);
            const int n = len < 1 ? 0 : min(a.max_pages, (len + kPage - 1) / kPage);
            const int spp = (n + a.score_ctas - 1) / a.score_ctas;
            lo = min(n, c * spp);
            hi = min(n, lo + spp);
        };
        // Moves cursor (b, p) t pages forward in the flat sequence; b = B past the end.
        auto advance = [&](int& b, int& p, int t) {
            int lo = 0, hi = 0;
            if (b < B) slice(b, lo, hi);
            while (b < B && p + t >= hi) {
                t -= hi - p;
                if (++b < B) {
                    slice(b, lo, hi);
                    p = lo;
                }
            }
            p += t;
        };
        auto fetch = [&](int b, int p) -> int {
            return b < B ? __ldg(a.page_table + static_cast<int64_t>(b) * a.max_pages + p) : -1;
        };
        int cb = 0, cp;
        {
            int lo, hi;
            slice(0, lo, hi);
            cp = lo;
        }
        advance(cb, cp, lane);
        int phys = fetch(cb, cp);
        bool ok = true;
        for (uint32_t f = lane; cb < B; f += SS::R) {
            int nb = cb, np = cp;
            advance(nb, np, SS::R);
            const int phys_next = fetch(nb, np);
            const int slot = f % SS::kSlots;
            if (f >= SS::kSlots) ok = mbar_wait_bounded(empty0 + slot * 8, ((f / SS::kSlots) - 1) & 1);
            if (!ok) break;
            const uint32_t fb = full0 + slot * 8;
            const bool real = phys >= 0 && phys < a.num_phys_pages;
            slot_ok[slot] = real ? 1 : 0;
            if (real) {
                mbar_arrive_expect_tx(fb, SS::kPageBytes);
                bulk_copy_g2s(ring_s + slot * SS::kPageBytes, meta_bytes + static_cast<int64_t>(phys) * SS::kPageBytes,
                              SS::kPageBytes, fb);
            } else {
                svq_flag(SV_DEVERR_PAGE_TABLE);
                mbar_arrive(fb);
            }
            cb = nb;
            cp = np;
            phys = phys_next;
        }
        if (!ok) svq_flag(SV_DEVERR_TIMEOUT);
        return;
    }
    const int hj = lane / SS::L, hk = lane % SS::L;
    const unsigned char* lane_base = ring + hj * 512 + hk * 16;
    uint32_t seq = 0;
    bool failed = false;
    for (int b = 0; b < a.batch; ++b) {
        int len;
        const int n = pages_of(a, b, len);
        const int spp = (n + a.score_ctas - 1) / a.score_ctas;
        const int lo = min(n, c * spp), hi = min(n, lo + spp);
        // Chunk hk + L t of kv head hj holds 8 channels of kmin (chunks 0-15,
        // coefficient Qn = sum_h min(q_h, 0)) or of kmax (chunks 16-31,
        // coefficient Qp = sum_h max(q_h, 0)).
        const int qb = b & 1;
        if (!failed) {
            const bool okq = mbar_wait_bounded(qfull0 + qb * 8, (static_cast<uint32_t>(b) >> 1) & 1);
            if (__any_sync(0xffffffffu, !okq)) {
                if (lane == 0) svq_flag(SV_DEVERR_TIMEOUT);
                failed = true;
            }
        }
        float cf[SS::C][8];
#pragma unroll
        for (int t = 0; t < SS::C; ++t) {
            const int chunk = hk + SS::L * t;
            const bool is_max = chunk >= 16;
            const __nv_bfloat16* qp = qbuf + qb * (SS::kQBufBytes / 2) + hj * a.group * kHeadDim + (chunk & 15) * 8;
#pragma unroll
            for (int e = 0; e < 8; ++e) cf[t][e] = 0.f;
#pragma unroll
            for (int h = 0; h < kMaxGroup; ++h) {
                if (h < a.group && !failed) {
                    const uint4 w = *reinterpret_cast<const uint4*>(qp + h * kHeadDim);
                    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float v0 = bf16lo(x[e]), v1 = bf16hi(x[e]);
                        cf[t][2 * e] += is_max ? fmaxf(v0, 0.f) : fminf(v0, 0.f);
                        cf[t][2 * e + 1] += is_max ? fmaxf(v1, 0.f) : fminf(v1, 0.f);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && !failed) mbar_arrive(qempty0 + qb * 8);
        float* score_row = a.scores + (static_cast<int64_t>(b) * HKV + hj) * a.score_stride;
        const int first = lo + (warp - static_cast<int>(seq % kStepConsumers) + kStepConsumers) % kStepConsumers;
        for (int p = first; p < hi && !failed; p += kStepConsumers) {
            const uint32_t sq = seq + (p - lo);
            const int slot = sq % SS::kSlots;
            const bool okw = mbar_wait_bounded(full0 + slot * 8, (sq / SS::kSlots) & 1);
            if (__any_sync(0xffffffffu, !okw)) {
                if (lane == 0) svq_flag(SV_DEVERR_TIMEOUT);
                failed = true;
                break;
            }
            // At most 4 chunks in flight per lane (register budget at 8 kv heads).
            constexpr int kHalf = SS::C < 4 ? SS::C : 4;
            const unsigned char* src = lane_base + slot * SS::kPageBytes;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int t0 = 0; t0 < SS::C; t0 += kHalf) {
                uint4 w[kHalf];
#pragma unroll
                for (int t = 0; t < kHalf; ++t) w[t] = *reinterpret_cast<const uint4*>(src + (t0 + t) * SS::L * 16);
#pragma unroll
                for (int t = 0; t < kHalf; ++t) {
                    const uint32_t x[4] = {w[t].x, w[t].y, w[t].z, w[t].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        a0 = fmaf(cf[t0 + t][2 * e], bf16lo(x[e]), a0);
                        a1 = fmaf(cf[t0 + t][2 * e + 1], bf16hi(x[e]), a1);
                    }
                }
            }
            const bool real = slot_ok[slot] != 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + slot * 8);
            float acc = real ? a0 + a1 : 0.f;
#pragma unroll
            for (int mm = 1; mm < SS::L; mm <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, mm);
            if (hk == 0) score_row[p] = acc;
        }
        seq += hi - lo;
        // This warp is past request b: count it for the control warp.
        __syncwarp();
        if (lane == 0) red_release_cta_smem(req_done, 1u);
    }
}

// ---------------------------------------------------------------- attention items
// Page range of split `split` of the selection of (b, g).
struct SplitRange {
    int j0, count;
};
__device__ __forceinline__ SplitRange split_range(const StepArgs& a, int bg, int split, int n) {
    const int cnt = ld_relaxed_i32(a.sel_cnt + bg);
    const int total = max(0, min(cnt, min(a.K, n)));
    const int chunk = (total + a.splits - 1) / a.splits;
    const int j0 = min(total, split * chunk);
    return {j0, min(total, j0 + chunk) - j0};
}

// Producer side of one attention item: lane group u (lanes 4u .. 4u+3) feeds
// stage u -- the item's pages whose sequence number is u mod 8, one 2 KB box
// per lane (K lo, K hi, V lo, V hi).  Groups run on their own (no warp-wide
// rounds); each lane resolves its group's next page while it waits for the
// stage of the current one.
template <int HKV>
__device__ __forceinline__ void produce_split(const StepArgs& a, const QueueItem& it, const CUtensorMap* tmap_k,
                                              const CUtensorMap* tmap_v, uint32_t ring_s, uint32_t kvf0,
                                              uint32_t kve0, int* stage_valid, uint32_t& fseq) {
    const int lane = threadIdx.x & 31;
    const int bg = it.b * HKV + it.g;
    int len;
    const int n = pages_of(a, it.b, len);
    const SplitRange sr = split_range(a, bg, it.split, n);
    const int my_count = sr.count;
    const int32_t* sel_row = a.sel_idx + static_cast<int64_t>(bg) * a.K + sr.j0;
    const int32_t* pt_row = a.page_table + static_cast<int64_t>(it.b) * a.max_pages;
    const int u = lane >> 2, box = lane & 3;
    const void* tmap = box < 2 ? static_cast<const void*>(tmap_k) : static_cast<const void*>(tmap_v);
    // Physical page and valid rows of item page i (phys -1: skip and zero-fill).
    auto resolve = [&](int i, int& phys_out, int& valid_out) {
        phys_out = -1;
        valid_out = 0;
        if (i < my_count) {
            const int lp = __ldcg(sel_row + i);
            if (lp < 0 || lp >= n) {
                svq_flag(SV_DEVERR_SEL_IDX);
            } else {
                const int ph = __ldg(pt_row + lp);
                if (ph < 0 || ph >= a.num_phys_pages) {
                    svq_flag(SV_DEVERR_PAGE_TABLE);
                } else {
                    phys_out = ph;
                    valid_out = (lp == n - 1) ? len - kPage * (n - 1) : kPage;
                }
            }
        }
    };
    const int first = (u - static_cast<int>(fseq % kKvStages) + kKvStages) % kKvStages;
    int phys, valid;
    resolve(first, phys, valid);
    bool ok = true;
    for (int i = first; i < my_count; i += kKvStages) {
        int phys_next, valid_next;
        resolve(i + kKvStages, phys_next, valid_next);
        const uint32_t sq = fseq + i;   // sq % 8 == u
        if (sq >= kKvStages) ok = mbar_wait_bounded(kve0 + u * 8, ((sq / kKvStages) - 1) & 1);
        if (!ok) break;
        const uint32_t fb = kvf0 + u * 8;
        if (box == 0) {
            stage_valid[u] = phys >= 0 ? valid : 0;
            if (phys >= 0) mbar_arrive_expect_tx(fb, kKvStage);
            else mbar_arrive(fb);
        }
        if (phys >= 0) {
            const int y = static_cast<int>((static_cast<int64_t>(phys) * HKV + it.g) * kPage);
            tma_load_2d(ring_s + u * kKvStage + box * kBox, tmap, (box & 1) * 64, y, fb);
        }
        phys = phys_next;
        valid = valid_next;
    }
    if (!ok) svq_flag(SV_DEVERR_TIMEOUT);
    __syncwarp();
    fseq += my_count;
}

// Compute side of one attention item: flash decode over the warp's pages
// (stage = this warp), merge of the 8 warps through `merge`, partial (o, m, l)
// of the split to the workspace.
template <int HKV>
__device__ __forceinline__ void attend_split(const StepArgs& a, const QueueItem& it, unsigned char* ring,
                                             uint32_t ring_s, uint32_t kvf0, uint32_t kve0, const int* stage_valid,
                                             float* merge, uint32_t& fseq) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int b = it.b, g = it.g;
    const int bg = b * HKV + g;
    int len;
    const int n = pages_of(a, b, len);
    const int my_count = split_range(a, bg, it.split, n).count;
    const int quad = lane & 3, row = lane >> 2;
    uint32_t qf[8][2];
    {
        const bool hv = row < a.group;
        const __nv_bfloat16* qh =
            a.q + (static_cast<int64_t>(b) * a.num_q_heads + g * a.group + (hv ? row : 0)) * kHeadDim;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            qf[kk][0] = hv ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 2 * quad) : 0u;
            qf[kk][1] = hv ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 8 + 2 * quad) : 0u;
        }
    }
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    const int mat = lane >> 3, rr8 = lane & 7;
    const int krow = rr8 + 8 * (mat & 1);
    const int vrow = rr8 + 8 * (mat >> 1);
    const int first = (warp - static_cast<int>(fseq % kKvStages) + kKvStages) % kKvStages;
    for (int i = first; i < my_count; i += kStepConsumers) {
        const uint32_t sq = fseq + i;
        const bool okw = mbar_wait_bounded(kvf0 + warp * 8, (sq / kKvStages) & 1);
        if (__any_sync(0xffffffffu, !okw)) {
            if (lane == 0) svq_flag(SV_DEVERR_TIMEOUT);
            break;
        }
        const uint32_t st_s = ring_s + warp * kKvStage;
        const int valid = stage_valid[warp];
        if (valid < kPage) {
            // Rows past the last token: V rows to zero (their weights are 0,
            // but the pool bytes there are arbitrary), logits masked below.
            unsigned char* vb = ring + warp * kKvStage + 2 * kBox;
            for (int cc = lane; cc < (kPage - valid) * 16; cc += 32) {
                const int rr = valid + (cc >> 4);
                *reinterpret_cast<uint4*>(vb + ((cc & 8) ? kBox : 0) + swz128(rr, cc & 7)) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        // S^T (16 tokens x 8 heads) = K (16 x 128) . Q^T, two accumulators.
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t addr = st_s + (kk >> 2) * kBox + swz128(krow, 2 * (kk & 3) + (mat >> 1));
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(addr, a0, a1, a2, a3);
            if (kk & 1) mma_bf16_16816(sb, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
            else mma_bf16_16816(sa, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        }
        const float x0 = row < valid ? (sa[0] + sb[0]) * a.scale_log2 : -INFINITY;
        const float x1 = row < valid ? (sa[1] + sb[1]) * a.scale_log2 : -INFINITY;
        const float x2 = row + 8 < valid ? (sa[2] + sb[2]) * a.scale_log2 : -INFINITY;
        const float x3 = row + 8 < valid ? (sa[3] + sb[3]) * a.scale_log2 : -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int s2 = 4; s2 < 32; s2 <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, s2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, s2));
        }
        const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
        const float base0 = mn0 == -INFINITY ? 0.f : mn0;
        const float base1 = mn1 == -INFINITY ? 0.f : mn1;
        const float alpha0 = step_exp2(m_run[0] - base0), alpha1 = step_exp2(m_run[1] - base1);
        const float p0 = step_exp2(x0 - base0), p1 = step_exp2(x1 - base1);
        const float p2 = step_exp2(x2 - base0), p3 = step_exp2(x3 - base1);
        m_run[0] = mn0;
        m_run[1] = mn1;
        l_run[0] = l_run[0] * alpha0 + p0 + p2;
        l_run[1] = l_run[1] * alpha1 + p1 + p3;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            o[mt][0] *= alpha0;
            o[mt][1] *= alpha1;
            o[mt][2] *= alpha0;
            o[mt][3] *= alpha1;
        }
        // P^T fragment (tokens x heads) from the S^T accumulators of 2 lanes.
        const uint32_t plo = pack_bf16x2(p0, p1);
        const uint32_t phi = pack_bf16x2(p2, p3);
        const int src0 = (2 * quad) * 4 + (row >> 1);
        const int src1 = (2 * quad + 1) * 4 + (row >> 1);
        const uint32_t lo0 = __shfl_sync(0xffffffffu, plo, src0);
        const uint32_t lo1 = __shfl_sync(0xffffffffu, plo, src1);
        const uint32_t hi0 = __shfl_sync(0xffffffffu, phi, src0);
        const uint32_t hi1 = __shfl_sync(0xffffffffu, phi, src1);
        const uint32_t selector = (row & 1) ? 0x7632u : 0x5410u;
        const uint32_t pb0 = __byte_perm(lo0, lo1, selector);
        const uint32_t pb1 = __byte_perm(hi0, hi1, selector);
        // O^T (128 channels x 8 heads) += V^T . P^T
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const uint32_t addr = st_s + (2 + (mt >> 2)) * kBox + swz128(vrow, 2 * (mt & 3) + (mat & 1));
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4_trans(addr, a0, a1, a2, a3);
            mma_bf16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(kve0 + warp * 8);
    }
    fseq += my_count;
#pragma unroll
    for (int s2 = 4; s2 < 32; s2 <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], s2);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], s2);
    }
    compute_sync();   // the previous item's readers of the merge area are done
    float* sm_o = merge;
    float* sm_m = sm_o + kStepConsumers * kMaxGroup * kHeadDim;
    float* sm_l = sm_m + kStepConsumers * kMaxGroup;
    {
        float* ow = sm_o + warp * kMaxGroup * kHeadDim;
        const int h0 = 2 * quad, h1 = 2 * quad + 1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            ow[h0 * kHeadDim + 16 * mt + row] = o[mt][0];
            ow[h1 * kHeadDim + 16 * mt + row] = o[mt][1];
            ow[h0 * kHeadDim + 16 * mt + row + 8] = o[mt][2];
            ow[h1 * kHeadDim + 16 * mt + row + 8] = o[mt][3];
        }
        if (row == 0) {
            sm_m[warp * kMaxGroup + h0] = m_run[0];
            sm_m[warp * kMaxGroup + h1] = m_run[1];
            sm_l[warp * kMaxGroup + h0] = l_run[0];
            sm_l[warp * kMaxGroup + h1] = l_run[1];
        }
    }
    compute_sync();
    const int S = a.splits;
    const int64_t qbase = static_cast<int64_t>(b) * a.num_q_heads + g * a.group;
    for (int idx = tid; idx < a.group * kHeadDim; idx += kComputeThreads) {
        const int h = idx / kHeadDim, d = idx % kHeadDim;
        float M = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < kStepConsumers; ++w2) M = fmaxf(M, sm_m[w2 * kMaxGroup + h]);
        float Lsum = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w2 = 0; w2 < kStepConsumers; ++w2) {
                const float e = step_exp2(sm_m[w2 * kMaxGroup + h] - M);
                Lsum += sm_l[w2 * kMaxGroup + h] * e;
                O += sm_o[(w2 * kMaxGroup + h) * kHeadDim + d] * e;
            }
        }
        a.o_part[((qbase + h) * S + it.split) * kHeadDim + d] = O;
        if (d == 0) a.ml_part[(qbase + h) * S + it.split] = make_float2(M, Lsum);
    }
}

// Log-sum-exp combine of the splits of (b, g) into out / lse (compute warps).
__device__ __forceinline__ void combine_splits(const StepArgs& a, int b, int g) {
    constexpr int kU = 8;   // splits loaded per batch
    const int S = a.splits;
    const int64_t qbase = static_cast<int64_t>(b) * a.num_q_heads + g * a.group;
    for (int idx = threadIdx.x; idx < a.group * kHeadDim; idx += kComputeThreads) {
        const int h = idx / kHeadDim, d = idx % kHeadDim;
        const int64_t qh = qbase + h;
        const float2* ml = a.ml_part + qh * S;
        const float* op = a.o_part + qh * S * kHeadDim + d;
        float M = -INFINITY;
        for (int s0 = 0; s0 < S; s0 += kU) {
            float mx[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) mx[u] = s0 + u < S ? __ldcg(&ml[s0 + u].x) : -INFINITY;
#pragma unroll
            for (int u = 0; u < kU; ++u) M = fmaxf(M, mx[u]);
        }
        float Lsum = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int s0 = 0; s0 < S; s0 += kU) {
                float2 v[kU];
                float ov[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    v[u] = s0 + u < S ? __ldcg(&ml[s0 + u]) : make_float2(-INFINITY, 0.f);
                    ov[u] = s0 + u < S ? __ldcg(op + (s0 + u) * kHeadDim) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const float e = step_exp2(v[u].x - M);
                    Lsum += v[u].y * e;
                    O += ov[u] * e;
                }
            }
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        a.out[qh * kHeadDim + d] = __float2bfloat16_rn(O * inv);
        if (d == 0) a.lse[qh] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
    }
}

// ---------------------------------------------------------------- the step kernel
template <int HKV>
__global__ void __launch_bounds__(kStepThreads, 2) quest_step_kernel(const __grid_constant__ StepArgs a,
                                                                   const __grid_constant__ CUtensorMap tmap_k,
                                                                   const __grid_constant__ CUtensorMap tmap_v) {
    using SS = StepScoreShape<HKV>;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[SS::kSlots];
    __shared__ __align__(8) uint64_t empty_bar[SS::kSlots];
    __shared__ __align__(8) uint64_t kv_full[kKvStages];
    __shared__ __align__(8) uint64_t kv_empty[kKvStages];
    __shared__ __align__(8) uint64_t q_full[2];
    __shared__ __align__(8) uint64_t q_empty[2];
    __shared__ __align__(8) uint64_t item_full[2];
    __shared__ __align__(8) uint64_t item_empty[2];
    __shared__ unsigned char slot_ok[SS::kSlots];
    __shared__ int stage_valid[kKvStages];
    __shared__ int item_slot[2];
    __shared__ uint32_t req_done;
    __shared__ RowTopkScratch sc;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tid = threadIdx.x;
    // Dynamic shared memory: [ring 64 KB, 1024-aligned][merge area / query buffers].
    const uint32_t raw_s = smem_addr(smem_raw);
    const uint32_t ring_s = (raw_s + 1023u) & ~1023u;   // 128-byte swizzle wants 1024-byte alignment
    unsigned char* ring = smem_raw + (ring_s - raw_s);
    float* merge = reinterpret_cast<float*>(ring + kStepRingBytes);
    const uint32_t full0 = smem_addr(&full_bar[0]), empty0 = smem_addr(&empty_bar[0]);
    const uint32_t kvf0 = smem_addr(&kv_full[0]), kve0 = smem_addr(&kv_empty[0]);
    const uint32_t itf0 = smem_addr(&item_full[0]), ite0 = smem_addr(&item_empty[0]);

    if (tid == 0) {
        for (int i = 0; i < SS::kSlots; ++i) {
            mbar_init(full0 + i * 8, 1);
            mbar_init(empty0 + i * 8, 1);
        }
        for (int i = 0; i < kKvStages; ++i) {
            mbar_init(kvf0 + i * 8, 1);
            mbar_init(kve0 + i * 8, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&q_full[i]), 1);
            mbar_init(smem_addr(&q_empty[i]), kStepConsumers);
            mbar_init(itf0 + i * 8, 1);
            mbar_init(ite0 + i * 8, 1 + kStepConsumers);   // producer + compute warps
        }
        req_done = 0u;
        mbar_init_fence();
    }
    if (warp == kStepProducer && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    __syncthreads();

    const int cta = blockIdx.x;
    if (cta < a.score_ctas) {
        score_role<HKV>(a, ring, ring_s, full0, empty0, slot_ok, reinterpret_cast<const __nv_bfloat16*>(merge),
                        smem_addr(merge), smem_addr(&q_full[0]), smem_addr(&q_empty[0]), &req_done);
    } else if (cta < a.score_ctas + a.sel_ctas && warp < kStepConsumers) {
        const int s = cta - a.score_ctas;
        const int g = s % HKV;
        const int reps = a.sel_ctas / HKV;
        for (int b = s / HKV; b < a.batch; b += reps) {
            int len;
            const int n = pages_of(a, b, len);
            if (tid == 0 && !wait_counter(a.ctr + 1 + b, static_cast<uint32_t>(a.score_ctas)))
                svq_flag(SV_DEVERR_TIMEOUT);
            compute_sync();
            const int bg = b * HKV + g;
            select_row(a, sc, reinterpret_cast<float*>(ring), bg, n);
            compute_sync();
            if (tid == 0)
                asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a.ctr + 1 + a.batch + bg), "r"(1u) : "memory");
        }
    }
    fence_proxy_async_smem();   // generic accesses to the ring before the TMA writes below
    __syncthreads();

    // ============================================ attention queue (every CTA)
    const int BH = a.batch * HKV;
    uint32_t* const ctr_next = a.ctr;
    uint32_t* const ctr_tdone = a.ctr + 1 + a.batch;
    uint32_t* const ctr_fdone = a.ctr + 1 + a.batch + BH;
    if (warp == kStepControl) {
        if (lane != 0) return;
        // Claims items one ahead of the compute warps, waits for each item's
        // inputs and publishes it in item slot k % 2.  Retiring item j (waiting
        // until the producer and compute warps are done with it) releases an
        // attention item's "split done".  Before a combine item waits for the
        // splits of its (b, g), this CTA retires all of its own items, so it
        // never waits on a release it holds itself.
        int kind_of[2] = {0, 0}, bg_of[2] = {0, 0};
        uint32_t k = 0, retired = 0;
        auto retire_next = [&]() {
            const uint32_t j = retired++;
            const int s = j & 1;
            if (!mbar_wait_bounded(ite0 + s * 8, (j >> 1) & 1)) svq_flag(SV_DEVERR_TIMEOUT);
            if (kind_of[s] == 1) red_release_gpu(ctr_fdone + bg_of[s], 1u);
        };
        for (;;) {
            const int item = static_cast<int>(atomicAdd(ctr_next, 1u));
            const QueueItem it = decode_item<HKV>(a, item);
            while (retired + 2 <= k) retire_next();       // slot k % 2 must be free
            if (it.kind == 2)
                while (retired < k) retire_next();
            const int bg = it.b * HKV + it.g;
            if (it.kind == 1 && !wait_counter(ctr_tdone + bg, 1u)) svq_flag(SV_DEVERR_TIMEOUT);
            if (it.kind == 2 && !wait_counter(ctr_fdone + bg, static_cast<uint32_t>(a.splits)))
                svq_flag(SV_DEVERR_TIMEOUT);
            const int s = k & 1;
            item_slot[s] = it.kind == 0 ? -1 : item;
            kind_of[s] = it.kind;
            bg_of[s] = bg;
            mbar_arrive(itf0 + s * 8);
            ++k;
            if (it.kind == 0) break;
        }
        while (retired + 1 < k) retire_next();            // everything before the stop marker
        return;
    }
    uint32_t fseq = 0;   // K/V pages this CTA has streamed (stage = fseq % 8)
    for (uint32_t k = 0;; ++k) {
        const int s = k & 1;
        if (!wait_item(itf0 + s * 8, (k >> 1) & 1)) {
            svq_flag(SV_DEVERR_TIMEOUT);
            break;
        }
        const int item = item_slot[s];
        const QueueItem it = decode_item<HKV>(a, item);
        if (it.kind == 1) {
            if (warp == kStepProducer)
                produce_split<HKV>(a, it, &tmap_k, &tmap_v, ring_s, kvf0, kve0, stage_valid, fseq);
            else
                attend_split<HKV>(a, it, ring, ring_s, kvf0, kve0, stage_valid, merge, fseq);
        } else if (it.kind == 2 && warp != kStepProducer) {
            combine_splits(a, it.b, it.g);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(ite0 + s * 8);
        if (it.kind == 0) break;
    }
}

// ---------------------------------------------------------------- host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 step_tensor_map_encoder() {
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_entry());
}

bool step_pool_map(CUtensorMap* map, const void* pool, int64_t rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = step_tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kPage)};
    const cuuint32_t estride[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct StepLayout {
    size_t scores, o_part, ml_part, ctr, total;
    int splits, stride;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

constexpr int kStepSmem = 1024 + kStepRingBytes + kMergeBytes;   // alignment slack + ring + merge area

StepLayout step_layout(int batch, int num_q_heads, int num_kv_heads, int max_pages, int budget_pages) {
    StepLayout L;
    const int kb = min(budget_pages, max_pages);
    L.splits = max(1, min(kStepMaxSplits, (kb + SVQ_STEP_PAGES_PER_SPLIT - 1) / SVQ_STEP_PAGES_PER_SPLIT));
    L.stride = (max_pages + 31) / 32 * 32;
    const size_t bh = static_cast<size_t>(batch) * num_kv_heads;
    const size_t heads = static_cast<size_t>(batch) * num_q_heads * L.splits;
    L.scores = 0;
    L.o_part = align256(bh * L.stride * sizeof(float));
    L.ml_part = L.o_part + align256(heads * kHeadDim * sizeof(float));
    L.ctr = L.ml_part + align256(heads * sizeof(float2));
    L.total = L.ctr + align256((1 + batch + 2 * bh) * sizeof(uint32_t));
    return L;
}

}  // namespace

size_t step_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int max_pages, int budget_pages) {
    return step_layout(batch, num_q_heads, num_kv_heads, max_pages, budget_pages).total;
}

template <int HKV>
int launch_step_hkv(const sv_cache* c, const void* q, int num_q_heads, const int32_t* page_table,
                    const int32_t* seq_lens, int batch, int max_pages, int budget_pages, int32_t* sel_idx,
                    int32_t* sel_cnt, float softmax_scale, void* out, float* lse, void* workspace, size_t ws_bytes,
                    int sm_count, cudaStream_t stream) {
    static std::atomic<int> per_sm_cache[64];
    const int dev = current_device();
    if (dev < 0) return SV_ERR_CUDA;
    int per_sm = dev < 64 ? per_sm_cache[dev].load(std::memory_order_acquire) : 0;
    if (per_sm == 0) {
        if (cudaFuncSetAttribute(quest_step_kernel<HKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, kStepSmem) !=
            cudaSuccess)
            return SV_ERR_CUDA;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quest_step_kernel<HKV>, kStepThreads, kStepSmem) !=
                cudaSuccess ||
            per_sm < 1)
            return SV_ERR_CUDA;
        per_sm = min(per_sm, 2);
        if (dev < 64) per_sm_cache[dev].store(per_sm, std::memory_order_release);
    }
    if (max_pages > kStepMaxPages) return SV_ERR_UNSUPPORTED;
    const StepLayout Ly = step_layout(batch, num_q_heads, c->num_kv_heads, max_pages, budget_pages);
    if (!workspace || ws_bytes < Ly.total) return SV_ERR_WORKSPACE;
    const int64_t rows = c->num_phys_pages * c->num_kv_heads * kPage;
    if (rows > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
    CUtensorMap tmap_k, tmap_v;
    if (!step_pool_map(&tmap_k, c->k_pool, rows) || !step_pool_map(&tmap_v, c->v_pool, rows)) return SV_ERR_CUDA;

    const int grid = per_sm * sm_count;
    const int sel_ctas = HKV * max(1, min(batch, SVQ_STEP_SELECTORS_PER_HEAD));
    if (grid < sel_ctas + 1) return SV_ERR_UNSUPPORTED;
    // Score CTAs take the first wave (one per SM, so every score CTA streams at
    // the same rate); selectors and attention-only CTAs the rest.
    int score_ctas = sm_count;
    if (SVQ_STEP_SCORE_PERMILLE > 0) score_ctas = static_cast<int>(static_cast<int64_t>(grid) * SVQ_STEP_SCORE_PERMILLE / 1000);
    score_ctas = max(1, min(grid - sel_ctas, score_ctas));

    unsigned char* ws = static_cast<unsigned char*>(workspace);
    StepArgs a;
    a.meta = static_cast<const __nv_bfloat16*>(c->meta);
    a.num_phys_pages = c->num_phys_pages;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.num_q_heads = num_q_heads;
    a.group = num_q_heads / c->num_kv_heads;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.batch = batch;
    a.max_pages = max_pages;
    a.K = budget_pages;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.scores = reinterpret_cast<float*>(ws + Ly.scores);
    a.score_stride = Ly.stride;
    a.sel_idx = sel_idx;
    a.sel_cnt = sel_cnt;
    a.o_part = reinterpret_cast<float*>(ws + Ly.o_part);
    a.ml_part = reinterpret_cast<float2*>(ws + Ly.ml_part);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.score_ctas = score_ctas;
    a.sel_ctas = sel_ctas;
    a.splits = Ly.splits;
    a.ctr = reinterpret_cast<uint32_t*>(ws + Ly.ctr);

    const size_t ctr_bytes = (1 + batch + 2 * static_cast<size_t>(batch) * c->num_kv_heads) * sizeof(uint32_t);
    if (cudaMemsetAsync(a.ctr, 0, ctr_bytes, stream) != cudaSuccess) return SV_ERR_CUDA;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = kStepSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs co-resident, or no launch
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, quest_step_kernel<HKV>, a, tmap_k, tmap_v) != cudaSuccess) return SV_ERR_CUDA;
    return SV_OK;
}

int launch_step(const sv_cache* c, const void* q, int num_q_heads, const int32_t* page_table, const int32_t* seq_lens,
                int batch, int max_pages, int budget_pages, int32_t* sel_idx, int32_t* sel_cnt, float softmax_scale,
                void* out, float* lse, void* workspace, size_t ws_bytes, int sm_count, cudaStream_t stream) {
#define SVQ_STEP_CASE(H)                                                                                            \
    case H:                                                                                                         \
        return launch_step_hkv<H>(c, q, num_q_heads, page_table, seq_lens, batch, max_pages, budget_pages, sel_idx, \
                                  sel_cnt, softmax_scale, out, lse, workspace, ws_bytes, sm_count, stream);
    switch (c->num_kv_heads) {
        SVQ_STEP_CASE(1)
        SVQ_STEP_CASE(2)
        SVQ_STEP_CASE(4)
        SVQ_STEP_CASE(8)
        default: return SV_ERR_UNSUPPORTED;
    }
#undef SVQ_STEP_CASE
}

}  // namespace svq
