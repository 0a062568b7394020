// sv_quest_decode_step: the whole decode step -- page scoring, top-K page
// selection, split-K attention over the selected pages and the log-sum-exp
// combine -- as one persistent, cooperative launch (two CTAs per SM, all
// co-resident).
//
// Work split:
//   scoring   : CTAs 0 .. score_ctas-1 stream, for request 0, 1, ..., B-1 in
//               turn, their slice of the request's page metadata (TMA bulk copies
//               into a shared-memory ring; producer warp + eight consumer warps)
//               and write the page scores, with no drain between requests.
//   queue     : request-major items -- per request, one top-K selection item
//               per kv head, then (kv head, split) attention items.  The other
//               CTAs take items from the start; score CTAs join when their
//               scoring is done.  A selection item waits until every score CTA
//               has finished the request; an attention item waits for its kv
//               head's selection, streams the split's K/V boxes by TMA and runs
//               the tensor-core flash-decode loop; the CTA that finishes the
//               last split of a (request, kv head) combines the splits by
//               log-sum-exp.
// So request b's selection and attention overlap the scoring of requests
// b+1, ..., and HBM stays busy through the latency-bound top-K.  Every
// cross-CTA wait is bounded and is on work owned by a co-resident CTA that
// does not wait on the waiter.

#include <cuda.h>
#include <cudaTypedefs.h>

#include "svq_common.cuh"

namespace svq {

SVQ_DEFINE_ERROR_WORD(read_error_step)

constexpr int kStepConsumers = 8;
constexpr int kStepThreads = (kStepConsumers + 1) * 32;
constexpr int kStepProducer = kStepConsumers;
constexpr int kStepRingBytes = 64 * 1024;
constexpr int kStepSmem = kStepRingBytes + 1024;          // + slack for 1024-byte alignment
constexpr int kBox = kPage * 64 * 2;                      // 16 x 64 bf16 TMA box (2 KB)
constexpr int kKvStage = 4 * kBox;                        // K lo | K hi | V lo | V hi
constexpr int kKvStages = kStepRingBytes / kKvStage;      // 8: stage s is consumed by warp s
constexpr int kTopkThreadsStep = kStepConsumers * 32;     // 256
constexpr int kTopkItemsStep = 32;                        // rows up to 8192 pages
constexpr int kStepBins = 2048;
constexpr int kStepCandCap = 256;
constexpr uint32_t kSpinLimit = 1u << 24;                 // polls of a cross-CTA counter before giving up
constexpr int kStepMaxSplits = 64;
constexpr int kStepMaxPages = kTopkThreadsStep * kTopkItemsStep;   // 8192 pages (131072 tokens) per request
static_assert(kKvStages == kStepConsumers, "each ring stage belongs to one consumer warp");

struct StepArgs {
    const __nv_bfloat16* meta;
    int64_t num_phys_pages;
    int num_kv_heads;
    const __nv_bfloat16* q;
    int num_q_heads;
    int group;
    const int32_t* page_table;
    const int32_t* seq_lens;
    int batch;
    int max_pages;
    int K;
    float scale_log2;
    float* scores;            // [B][Hkv][max_pages]
    int32_t* sel_idx;         // [B][Hkv][K]
    int32_t* sel_cnt;         // [B][Hkv]
    float* o_part;            // [B][Hq][splits][128]
    float2* ml_part;          // [B][Hq][splits]
    __nv_bfloat16* out;       // [B][Hq][128]
    float* lse;               // [B][Hq]
    int score_ctas;           // CTAs 0 .. score_ctas-1 score; the rest decode
    int splits;               // decode items per (request, kv head)
    uint32_t* ctr;            // [0] next decode item, [1 + b] score slices done,
                              // [1 + B + bg] selection ready, [1 + B + BH + bg] splits done
};

__device__ __forceinline__ float step_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t step_order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kTopkThreadsStep) : "memory"); }

// Polls a counter written by other CTAs until it reaches `target` (bounded).
__device__ __forceinline__ bool wait_counter(const uint32_t* p, uint32_t target) {
    for (uint32_t it = 0; it < kSpinLimit; ++it) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v >= target) return true;
        __nanosleep(64);
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
    static constexpr int L = 32 / HKV;                                  // consumer lanes per kv head
    static constexpr int C = HKV;                                       // 16-byte chunks per lane per page
    static constexpr int kQBufBytes = kMaxGroup * HKV * kHeadDim * 2;   // one request's queries, at most
    static_assert(kSlots % R == 0 && kSlots % kStepConsumers == 0, "score ring shape");
};

// ---------------------------------------------------------------- top-K (256 consumer threads)
// Same selection as topk_pages_kernel: keys in registers (32 consecutive pages
// per thread), min/max-adaptive histogram, exact rank among the boundary
// bin's keys (radix fallback), ordered compaction from bit masks.
struct TopkScratch {
    uint32_t hist[kStepBins];
    uint32_t warp_tot[kStepConsumers];
    uint32_t warp_lo[kStepConsumers], warp_hi[kStepConsumers];
    uint32_t cand_key[kStepCandCap];
    int32_t cand_idx[kStepCandCap];
    uint32_t bin, rem, cand, T, take;
};

__device__ void step_topk(const StepArgs& a, TopkScratch& sc, int bg, int n) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K;
    const int m = min(K, n);
    int32_t* out = a.sel_idx + static_cast<int64_t>(bg) * K;
    if (n <= K) {
        for (int i = tid; i < K; i += kTopkThreadsStep) out[i] = i < n ? i : -1;
        if (tid == 0) a.sel_cnt[bg] = n;
        return;
    }
    const float* row = a.scores + static_cast<int64_t>(bg) * a.max_pages;
    const int i0 = kTopkItemsStep * tid;
    uint32_t key[kTopkItemsStep];
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int e = 0; e < kTopkItemsStep; ++e) {
        float f;
        asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(f) : "l"(row + min(i0 + e, a.max_pages - 1)) : "memory");
        key[e] = step_order_key(f);
        if (i0 + e < n) {
            lo = min(lo, key[e]);
            hi = max(hi, key[e]);
        }
    }
    for (int i = tid; i < kStepBins; i += kTopkThreadsStep) sc.hist[i] = 0u;
    if (tid == 0) sc.cand = 0u;
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) {
        sc.warp_lo[warp] = lo;
        sc.warp_hi[warp] = hi;
    }
    consumers_sync();
    lo = __reduce_min_sync(0xffffffffu, lane < kStepConsumers ? sc.warp_lo[lane] : 0xffffffffu);
    hi = __reduce_max_sync(0xffffffffu, lane < kStepConsumers ? sc.warp_hi[lane] : 0u);
    const uint32_t range = hi - lo;
    const int rbits = range == 0 ? 0 : 32 - __clz(range);
    const uint32_t shift = rbits > 11 ? rbits - 11 : 0;
#pragma unroll
    for (int e = 0; e < kTopkItemsStep; ++e)
        if (i0 + e < n) atomicAdd(&sc.hist[(key[e] - lo) >> shift], 1u);
    consumers_sync();
    auto find_bin = [&](uint32_t remaining) {
        constexpr int kBpt = kStepBins / kTopkThreadsStep;
        const uint32_t top = kStepBins - 1 - kBpt * tid;
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
            const uint32_t t2 = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t2;
        }
        if (lane == 31) sc.warp_tot[warp] = v;
        consumers_sync();
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
        consumers_sync();
    };
    find_bin(static_cast<uint32_t>(m));
    const uint32_t bstar = sc.bin, need = sc.rem;
    uint32_t T, take;
    if (sc.hist[bstar] <= kStepCandCap) {
#pragma unroll
        for (int e = 0; e < kTopkItemsStep; ++e) {
            if (i0 + e < n && ((key[e] - lo) >> shift) == bstar) {
                const uint32_t pos = atomicAdd(&sc.cand, 1u);
                sc.cand_key[pos] = key[e];
                sc.cand_idx[pos] = i0 + e;
            }
        }
        consumers_sync();
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
        consumers_sync();
        T = sc.T;
        take = sc.take;
    } else {
        uint32_t prefix = 0, remaining = static_cast<uint32_t>(m);
        const int kSh[3] = {21, 10, 0};
        const int kBi[3] = {11, 11, 10};
        for (int pass = 0; pass < 3; ++pass) {
            const int sh = kSh[pass];
            const uint32_t nbins = 1u << kBi[pass];
            const uint32_t hi_mask = (pass == 0) ? 0u : ~((1u << (sh + kBi[pass])) - 1u);
            consumers_sync();
            for (int i = tid; i < kStepBins; i += kTopkThreadsStep) sc.hist[i] = 0u;
            consumers_sync();
#pragma unroll
            for (int e = 0; e < kTopkItemsStep; ++e)
                if (i0 + e < n && (key[e] & hi_mask) == prefix) atomicAdd(&sc.hist[(key[e] >> sh) & (nbins - 1u)], 1u);
            consumers_sync();
            find_bin(remaining);
            prefix |= sc.bin << sh;
            remaining = sc.rem;
        }
        T = prefix;
        take = remaining;
    }
    uint32_t gt_mask = 0, eq_mask = 0;
#pragma unroll
    for (int e = 0; e < kTopkItemsStep; ++e) {
        if (i0 + e < n) {
            gt_mask |= (key[e] > T ? 1u : 0u) << e;
            eq_mask |= (key[e] == T ? 1u : 0u) << e;
        }
    }
    const uint32_t packed = (static_cast<uint32_t>(__popc(gt_mask)) << 16) | __popc(eq_mask);
    uint32_t v = packed;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t2 = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t2;
    }
    consumers_sync();   // everyone has read warp_tot of the last find_bin
    if (lane == 31) sc.warp_tot[warp] = v;
    consumers_sync();
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
    for (int i = m + tid; i < K; i += kTopkThreadsStep) out[i] = -1;
    if (tid == 0) a.sel_cnt[bg] = m;
}

// ---------------------------------------------------------------- score role
// Streams this CTA's slice of every request's page metadata through the ring
// (slot = sequence % slots; consumer warp = sequence % 8, so each slot has
// one waiting warp) and writes the page scores.  The producer issues the pages
// of one round from different lanes, each lane on its own slot.
template <int HKV>
__device__ __forceinline__ void score_role(const StepArgs& a, unsigned char* ring, uint32_t ring_s, uint32_t full0,
                                           uint32_t empty0, unsigned char* slot_ok, const __nv_bfloat16* qbuf,
                                           uint32_t qbuf_s, uint32_t qfull0, uint32_t qempty0, uint32_t* ctr_sdone) {
    using SS = StepScoreShape<HKV>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const uint32_t q_bytes = static_cast<uint32_t>(a.num_q_heads) * kHeadDim * 2;
    if (warp == kStepProducer) {
        const unsigned char* meta_bytes = reinterpret_cast<const unsigned char*>(a.meta);
        const unsigned char* q_src = reinterpret_cast<const unsigned char*>(a.q);
        uint32_t seq = 0;
        bool failed = false;
        for (int b = 0; b < a.batch && !failed; ++b) {
            // Request b's queries (num_q_heads x 128 bf16, contiguous) into q
            // buffer b % 2, once the consumers have folded request b - 2's.
            if (lane == 0) {
                const int qb = b & 1;
                const uint32_t use = static_cast<uint32_t>(b) >> 1;
                bool okq = true;
                if (use >= 1) okq = mbar_wait_bounded(qempty0 + qb * 8, (use - 1) & 1);
                if (okq) {
                    mbar_arrive_expect_tx(qfull0 + qb * 8, q_bytes);
                    bulk_copy_g2s(qbuf_s + qb * SS::kQBufBytes, q_src + static_cast<int64_t>(b) * q_bytes, q_bytes,
                                  qfull0 + qb * 8);
                } else {
                    failed = true;
                }
            }
            failed = __shfl_sync(0xffffffffu, failed, 0);
            if (failed) break;
            int len;
            const int n = pages_of(a, b, len);
            const int spp = (n + a.score_ctas - 1) / a.score_ctas;
            const int lo = min(n, c * spp), hi = min(n, lo + spp);
            const int32_t* pt_row = a.page_table + static_cast<int64_t>(b) * a.max_pages;
            for (int base = lo; base < hi; base += SS::R) {
                const int p = base + lane;
                bool ok = true;
                if (lane < SS::R && p < hi) {
                    const uint32_t sq = seq + (p - lo);
                    const int slot = sq % SS::kSlots;
                    if (sq >= SS::kSlots) ok = mbar_wait_bounded(empty0 + slot * 8, ((sq / SS::kSlots) - 1) & 1);
                    if (ok) {
                        const int phys = pt_row[p];
                        const uint32_t fb = full0 + slot * 8;
                        const bool real = phys >= 0 && phys < a.num_phys_pages;
                        slot_ok[slot] = real ? 1 : 0;
                        if (real) {
                            mbar_arrive_expect_tx(fb, SS::kPageBytes);
                            bulk_copy_g2s(ring_s + slot * SS::kPageBytes,
                                          meta_bytes + static_cast<int64_t>(phys) * SS::kPageBytes, SS::kPageBytes, fb);
                        } else {
                            svq_flag(SV_DEVERR_PAGE_TABLE);
                            mbar_arrive(fb);
                        }
                    }
                }
                if (__any_sync(0xffffffffu, !ok)) {
                    failed = true;
                    break;
                }
            }
            seq += hi - lo;
        }
        if (failed && lane == 0) svq_flag(SV_DEVERR_TIMEOUT);
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
        // Chunk hk + L t of kv head hj: 8 channels of kmin (chunks 0-15,
        // coefficient Qn) or of kmax (chunks 16-31, coefficient Qp), folded
        // from the staged queries of request b.
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
        float* score_row = a.scores + (static_cast<int64_t>(b) * HKV + hj) * a.max_pages;
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
                for (int t = 0; t < kHalf; ++t)
                    w[t] = *reinterpret_cast<const uint4*>(src + (t0 + t) * SS::L * 16);
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
        // This warp's share of request b is written: count it (release).
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            atomicAdd(ctr_sdone + b, 1u);
        }
    }
}

// ---------------------------------------------------------------- one attention split
// Pages [j0, j0 + my_count) of the selection of (b, g): K/V boxes by TMA into
// the 8-stage ring (stage = sequence % 8, consumed by warp = stage), tensor-core
// flash decode per page, merge of the 8 warps, partial (o, m, l) to the workspace.
template <int HKV>
__device__ __forceinline__ void attend_split(const StepArgs& a, int b, int g, int split, int n, int len,
                                             const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                             unsigned char* ring, uint32_t ring_s, uint32_t kvf0, uint32_t kve0,
                                             int* stage_valid, uint32_t& fseq) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int bg = b * HKV + g;
    int count;
    {
        int cnt;
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(cnt) : "l"(a.sel_cnt + bg) : "memory");
        count = max(0, min(cnt, min(a.K, n)));
    }
    const int chunk = (count + a.splits - 1) / a.splits;
    const int j0 = min(count, split * chunk);
    const int my_count = min(count, j0 + chunk) - j0;
    const int32_t* sel_row = a.sel_idx + static_cast<int64_t>(bg) * a.K;
    const int32_t* pt_row = a.page_table + static_cast<int64_t>(b) * a.max_pages;

    if (warp == kStepProducer) {
        // Lane group u (lanes 4u .. 4u+3) feeds stage u: of every 8 consecutive
        // pages it issues the one whose sequence number is u mod 8, one 2 KB
        // box per lane (K lo, K hi, V lo, V hi).
        const int u = lane >> 2, box = lane & 3;
        const void* tmap = box < 2 ? static_cast<const void*>(tmap_k) : static_cast<const void*>(tmap_v);
        auto resolve = [&](int base, int& phys_out, int& valid_out) {
            const int ii = base + lane;
            phys_out = -1;
            valid_out = 0;
            if (ii < my_count) {
                int lp;
                asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(lp) : "l"(sel_row + j0 + ii) : "memory");
                if (lp < 0 || lp >= n) {
                    svq_flag(SV_DEVERR_SEL_IDX);
                } else {
                    const int ph = pt_row[lp];
                    if (ph < 0 || ph >= a.num_phys_pages) {
                        svq_flag(SV_DEVERR_PAGE_TABLE);
                    } else {
                        phys_out = ph;
                        valid_out = (lp == n - 1) ? len - kPage * (n - 1) : kPage;
                    }
                }
            }
        };
        int cur_phys, cur_valid, nxt_phys, nxt_valid;
        resolve(0, cur_phys, cur_valid);
        bool failed = false;
        const int rot = static_cast<int>(fseq % kKvStages);
        for (int base = 0; base < my_count && !failed; base += 32) {
            resolve(base + 32, nxt_phys, nxt_valid);
            for (int r8 = 0; r8 < 32 && base + r8 < my_count; r8 += 8) {
                const int t = (u - rot + kKvStages) % kKvStages;
                const int i = base + r8 + t;
                const int phys = __shfl_sync(0xffffffffu, cur_phys, r8 + t);
                const int valid = __shfl_sync(0xffffffffu, cur_valid, r8 + t);
                bool ok = true;
                if (i < my_count) {
                    const uint32_t sq = fseq + i;   // sq % 8 == u
                    if (sq >= kKvStages) ok = mbar_wait_bounded(kve0 + u * 8, ((sq / kKvStages) - 1) & 1);
                    if (ok) {
                        const uint32_t fb = kvf0 + u * 8;
                        if (box == 0) {
                            stage_valid[u] = phys >= 0 ? valid : 0;
                            if (phys >= 0) mbar_arrive_expect_tx(fb, kKvStage);
                            else mbar_arrive(fb);
                        }
                        if (phys >= 0) {
                            const int y = static_cast<int>((static_cast<int64_t>(phys) * HKV + g) * kPage);
                            tma_load_2d(ring_s + u * kKvStage + box * kBox, tmap, (box & 1) * 64, y, fb);
                        }
                    }
                }
                if (__any_sync(0xffffffffu, !ok)) {
                    failed = true;
                    break;
                }
            }
            cur_phys = nxt_phys;
            cur_valid = nxt_valid;
        }
        if (failed && lane == 0) svq_flag(SV_DEVERR_TIMEOUT);
        fseq += my_count;
        return;
    }

    const int quad = lane & 3, row = lane >> 2;
    uint32_t qf[8][2];
    {
        const bool hv = row < a.group;
        const __nv_bfloat16* qh = a.q + (static_cast<int64_t>(b) * a.num_q_heads + g * a.group + (hv ? row : 0)) * kHeadDim;
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
    // Merge the 8 consumer warps through shared memory (every stage has been
    // consumed, so the ring is free).
    consumers_sync();
    float* sm_o = reinterpret_cast<float*>(ring);
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
    consumers_sync();
    const int S = a.splits;
    const int64_t qbase = static_cast<int64_t>(b) * a.num_q_heads + g * a.group;
    for (int idx = tid; idx < a.group * kHeadDim; idx += kTopkThreadsStep) {
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
        a.o_part[((qbase + h) * S + split) * kHeadDim + d] = O;
        if (d == 0) a.ml_part[(qbase + h) * S + split] = make_float2(M, Lsum);
    }
    // The ring is written next by TMA: order these generic writes first.
    fence_proxy_async_smem();
}

// Log-sum-exp combine of the splits of (b, g) into out / lse.
__device__ __forceinline__ void combine_splits(const StepArgs& a, int b, int g) {
    const int S = a.splits;
    const int64_t qbase = static_cast<int64_t>(b) * a.num_q_heads + g * a.group;
    for (int idx = threadIdx.x; idx < a.group * kHeadDim; idx += kStepThreads) {
        const int h = idx / kHeadDim, d = idx % kHeadDim;
        const int64_t qh = qbase + h;
        float M = -INFINITY;
        for (int s2 = 0; s2 < S; ++s2) {
            float mx;
            asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(mx) : "l"(a.ml_part + qh * S + s2) : "memory");
            M = fmaxf(M, mx);
        }
        float Lsum = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int s2 = 0; s2 < S; ++s2) {
                float mx, lx, ov;
                asm volatile("ld.relaxed.gpu.global.v2.f32 {%0, %1}, [%2];" : "=f"(mx), "=f"(lx) : "l"(a.ml_part + qh * S + s2) : "memory");
                asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(ov) : "l"(a.o_part + (qh * S + s2) * kHeadDim + d) : "memory");
                const float e = step_exp2(mx - M);
                Lsum += lx * e;
                O += ov * e;
            }
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        a.out[qh * kHeadDim + d] = __float2bfloat16_rn(O * inv);
        if (d == 0) a.lse[qh] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
    }
}

// ---------------------------------------------------------------- the step kernel
// Work queue, request-major: for request b, HKV selection items (one per kv
// head) and then HKV * splits attention items.  CTAs below score_ctas first
// score every request, then join the queue; the others take queue items from
// the start.  A selection item waits for the scores of its request (written by
// score CTAs, which wait on nothing); an attention item waits for a selection
// item of a lower queue index, already taken by a running CTA.  All CTAs are
// co-resident, so every wait ends.
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
    __shared__ __align__(128) __nv_bfloat16 qbuf[SS::kQBufBytes];   // two buffers
    __shared__ unsigned char slot_ok[SS::kSlots];
    __shared__ int stage_valid[kKvStages];
    __shared__ int s_item, s_flag;
    __shared__ TopkScratch sc;

    const int warp = threadIdx.x >> 5;
    const int tid = threadIdx.x;
    const uint32_t raw_s = smem_addr(smem_raw);
    const uint32_t ring_s = (raw_s + 1023u) & ~1023u;   // 128-byte swizzle wants 1024-byte alignment
    unsigned char* ring = smem_raw + (ring_s - raw_s);
    const uint32_t full0 = smem_addr(&full_bar[0]), empty0 = smem_addr(&empty_bar[0]);
    const uint32_t kvf0 = smem_addr(&kv_full[0]), kve0 = smem_addr(&kv_empty[0]);
    const int BH = a.batch * HKV;
    uint32_t* const ctr_next = a.ctr;
    uint32_t* const ctr_sdone = a.ctr + 1;
    uint32_t* const ctr_tdone = a.ctr + 1 + a.batch;
    uint32_t* const ctr_fdone = a.ctr + 1 + a.batch + BH;

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
        }
        mbar_init_fence();
    }
    if (warp == kStepProducer && (threadIdx.x & 31) == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    __syncthreads();

    if (static_cast<int>(blockIdx.x) < a.score_ctas) {
        score_role<HKV>(a, ring, ring_s, full0, empty0, slot_ok, qbuf, smem_addr(qbuf), smem_addr(&q_full[0]),
                        smem_addr(&q_empty[0]), ctr_sdone);
        fence_proxy_async_smem();
        __syncthreads();
    }

    const int per_req = HKV + HKV * a.splits;
    const int n_items = a.batch * per_req;
    const uint32_t scored = static_cast<uint32_t>(a.score_ctas) * kStepConsumers;
    uint32_t fseq = 0;
    for (;;) {
        if (tid == 0) s_item = static_cast<int>(atomicAdd(ctr_next, 1u));
        __syncthreads();
        const int item = s_item;
        if (item >= n_items) break;
        const int b = item / per_req;
        const int r = item - b * per_req;
        int len;
        const int n = pages_of(a, b, len);
        if (r < HKV) {
            // Selection of kv head r of request b.
            const int bg = b * HKV + r;
            if (tid == 0) {
                if (!wait_counter(ctr_sdone + b, scored)) svq_flag(SV_DEVERR_TIMEOUT);
                __threadfence();
            }
            __syncthreads();
            if (warp != kStepProducer) {
                step_topk(a, sc, bg, n);
                consumers_sync();
                if (tid == 0) {
                    __threadfence();
                    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ctr_tdone + bg), "r"(1u) : "memory");
                }
            }
        } else {
            const int f = r - HKV;
            const int g = f / a.splits, split = f - g * a.splits;
            const int bg = b * HKV + g;
            if (tid == 0) {
                if (!wait_counter(ctr_tdone + bg, 1u)) svq_flag(SV_DEVERR_TIMEOUT);
                __threadfence();
            }
            __syncthreads();
            attend_split<HKV>(a, b, g, split, n, len, &tmap_k, &tmap_v, ring, ring_s, kvf0, kve0, stage_valid, fseq);
            __syncthreads();
            // The CTA that completes the last split of (b, g) combines.
            if (tid == 0) {
                __threadfence();
                const uint32_t old = atomicAdd(ctr_fdone + bg, 1u);
                s_flag = (old == static_cast<uint32_t>(a.splits) - 1u) ? 1 : 0;
                if (s_flag) __threadfence();
            }
            __syncthreads();
            if (s_flag) combine_splits(a, b, g);
        }
        __syncthreads();   // item boundary
    }
}

// ---------------------------------------------------------------- host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 step_tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
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
    int splits;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

#ifndef SVQ_STEP_PAGES_PER_SPLIT
#define SVQ_STEP_PAGES_PER_SPLIT 16
#endif
#ifndef SVQ_STEP_SCORE_PERMILLE
#define SVQ_STEP_SCORE_PERMILLE 0   // 0: CTAs split by the bytes each role reads
#endif

StepLayout step_layout(int batch, int num_q_heads, int num_kv_heads, int max_pages, int budget_pages) {
    StepLayout L;
    const int kb = min(budget_pages, max_pages);
    L.splits = max(1, min(kStepMaxSplits, (kb + SVQ_STEP_PAGES_PER_SPLIT - 1) / SVQ_STEP_PAGES_PER_SPLIT));
    const size_t bh = static_cast<size_t>(batch) * num_kv_heads;
    const size_t heads = static_cast<size_t>(batch) * num_q_heads * L.splits;
    L.scores = 0;
    L.o_part = align256(bh * max_pages * sizeof(float));
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
    static int per_sm_cache[64] = {};
    const int dev = current_device();
    if (dev < 0) return SV_ERR_CUDA;
    int per_sm = dev < 64 ? per_sm_cache[dev] : 0;
    if (per_sm == 0) {
        if (cudaFuncSetAttribute(quest_step_kernel<HKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, kStepSmem) !=
            cudaSuccess)
            return SV_ERR_CUDA;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quest_step_kernel<HKV>, kStepThreads, kStepSmem) !=
                cudaSuccess ||
            per_sm < 1)
            return SV_ERR_CUDA;
        per_sm = min(per_sm, 2);
        if (dev < 64) per_sm_cache[dev] = per_sm;
    }
    if (max_pages > kStepMaxPages) return SV_ERR_UNSUPPORTED;
    const StepLayout Ly = step_layout(batch, num_q_heads, c->num_kv_heads, max_pages, budget_pages);
    if (!workspace || ws_bytes < Ly.total) return SV_ERR_WORKSPACE;
    const int64_t rows = c->num_phys_pages * c->num_kv_heads * kPage;
    if (rows > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
    CUtensorMap tmap_k, tmap_v;
    if (!step_pool_map(&tmap_k, c->k_pool, rows) || !step_pool_map(&tmap_v, c->v_pool, rows)) return SV_ERR_CUDA;

    const int grid = per_sm * sm_count;
    int score_ctas;
    if (SVQ_STEP_SCORE_PERMILLE > 0) {
        score_ctas = static_cast<int>(static_cast<int64_t>(grid) * SVQ_STEP_SCORE_PERMILLE / 1000);
    } else {
        // Metadata bytes per request vs selected K/V bytes per request.
        const double score_b = static_cast<double>(max_pages) * HKV * 2 * kHeadDim * 2;
        const double attend_b = static_cast<double>(min(budget_pages, max_pages)) * HKV * 2 * kPage * kHeadDim * 2;
        score_ctas = static_cast<int>(grid * score_b / (score_b + attend_b) + 0.5);
    }
    score_ctas = max(1, min(grid, score_ctas));

    unsigned char* ws = static_cast<unsigned char*>(workspace);
    StepArgs a;
    a.meta = static_cast<const __nv_bfloat16*>(c->meta);
    a.num_phys_pages = c->num_phys_pages;
    a.num_kv_heads = c->num_kv_heads;
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
    a.sel_idx = sel_idx;
    a.sel_cnt = sel_cnt;
    a.o_part = reinterpret_cast<float*>(ws + Ly.o_part);
    a.ml_part = reinterpret_cast<float2*>(ws + Ly.ml_part);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.score_ctas = score_ctas;
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
