// Exact softmax attention over the selected pages of a paged KV cache (the
// attention backend consuming the Quest view; SparseEngine summary page,
// section "method key points": AttentionView), as split-K flash decoding:
//
//   flash_decode_split_kernel : one CTA per (split, request, kv head); each
//       warp streams its share of the split's pages through shared memory and
//       keeps an online softmax; the CTA merges its warps into one partial
//   lse_combine_kernel        : merges the splits' partials by log-sum-exp
//
// Tensor cores: for one kv head the group's query heads (<= 8) share every
// key and value, so a page is a dense (16 tokens x 128) x (128 x 8 heads)
// product.  The token dimension is the MMA's M side: S^T = K Q^T
// (m16n8k16, 8 k-steps) and O^T += V^T P^T (8 m-tiles of 16 channels).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "svq_common.cuh"

namespace svq {

SVQ_DEFINE_ERROR_WORD(read_error_decode)

constexpr int kConsumers = 4;                     // consumer warps; warp w takes pages w, w + 4, ... of its split
constexpr int kDecodeThreads = (kConsumers + 1) * 32;
constexpr int kProducer = kConsumers;             // warp index of the producer
constexpr int kStages = 8;                        // pages in flight per CTA (one producer lane group each)
static_assert(kStages % kConsumers == 0, "each ring stage must belong to one consumer warp");
constexpr int kBoxBytes = kPage * 64 * 2;         // one TMA box: 16 rows x 64 channels (2 KB)
constexpr int kStageBytes = 4 * kBoxBytes;        // K lo | K hi | V lo | V hi
constexpr int kDecodeSmem = kStages * kStageBytes + 1024;   // + slack for 1024-byte alignment
constexpr int kMaxSplits = 64;
#ifndef SVQ_DECODE_WAVE_PERMILLE
#define SVQ_DECODE_WAVE_PERMILLE 1000   // split CTAs as a fraction of one full wave
#endif
constexpr int kMinPagesPerSplit = 8;       // workspace bound: at most ceil(pages / 8) splits
// Pages per split below which a split costs more (its setup, merge and partial,
// and the combine's read of it) than its parallelism saves once the GPU is
// full (bf16 / e4m3 pools).
constexpr int kSplitPagesBf16 = 24;
constexpr int kSplitPagesFp8 = 16;
// Online softmax with a lazily moved base: a head's running base moves only
// when one of the page's logits exceeds it by more than this many log2 units.
// Most pages then skip the warp max, the correction factors and the rescale
// of the 32 output registers; the weights stay at most 2^kRescaleSlack (bf16
// holds that with room to spare), and sums and outputs share the base, so the
// result is the same softmax.
constexpr float kRescaleSlack = 8.f;

struct DecodeArgs {
    int64_t num_phys_pages;
    int num_kv_heads;
    const __nv_bfloat16* q;
    int num_q_heads;
    int group;                // query heads of one selection row
    int rows_per_req;         // selection rows per request (kv heads, or query heads)
    int kv_div;               // selection row r reads kv head r / kv_div
    const int32_t* page_table;
    const int32_t* seq_lens;
    int max_pages;
    const int32_t* sel_idx;   // nullptr => dense
    const int32_t* sel_cnt;
    int K;
    int num_splits;
    float scale_log2;         // softmax_scale * log2(e)
    float* o_part;            // [B][Hq][S][128] unnormalised partial outputs
    float2* ml_part;          // [B][Hq][S] (base m in log2 units, at most kRescaleSlack below the max; sum of exp2(x - m))
};

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of (row, 16-byte chunk) inside a 128B-swizzled TMA box whose
// rows are 128 bytes (64 bf16): chunk c of row r sits at chunk c ^ (r & 7).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// One CTA per (split, request, kv head).  The K and V pools are seen as 3-D
// tensors (64 channels, pages * kv heads * 16 rows, 2 channel halves); a
// page's 16 x 128 tile of one kv head is one box that lands as two 16 x 64
// halves, 128-byte swizzled (so ldmatrix reads are conflict-free).  Producer
// lane group u (lanes 4u .. 4u+3) owns ring stage u and the split's pages
// u, u + 8, ...: after the consumers free the stage, lane 4u publishes the
// page's valid-token count, arms the stage's "full" mbarrier for 8 KB and
// moves the K tile; lane 4u + 2 moves the V tile.  Consumer warp w takes the
// split's pages w, w + 4, ... whole: the page's logits S^T = K Q^T for the
// query group, the online softmax update and O^T += V^T P^T over all 128
// channels, then it arrives on the stage's "empty" mbarrier.  The four warps'
// running (max, sum, output) are merged through shared memory into the CTA's
// partial.
__global__ void __launch_bounds__(kDecodeThreads) flash_decode_split_kernel(const __grid_constant__ DecodeArgs a,
                                                                          const __grid_constant__ CUtensorMap tmap_k,
                                                                          const __grid_constant__ CUtensorMap tmap_v) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ int s_valid[kStages];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];

    const int split = blockIdx.x;
    const int bg = blockIdx.y;                 // selection row of the whole batch
    const int b = bg / a.rows_per_req;
    const int g = bg % a.rows_per_req;          // row in the request: query heads g * group ..
    const int kvh = g / a.kv_div;               // kv head the row reads
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t raw_s = smem_addr(smem_raw);
    const uint32_t ring_s = (raw_s + 1023u) & ~1023u;      // 128B swizzle wants 1024-byte aligned boxes
    unsigned char* ring = smem_raw + (ring_s - raw_s);
    const uint32_t full0 = smem_addr(&full_bar[0]);
    const uint32_t empty0 = smem_addr(&empty_bar[0]);

    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(full0 + st * 8, 1);
            mbar_init(empty0 + st * 8, 1);   // stage s is consumed by warp s % kConsumers alone
        }
        mbar_init_fence();
    }
    __syncthreads();

    const int len = a.seq_lens[b];
    int n = (len + kPage - 1) / kPage;
    if (len < 1 || n > a.max_pages) {
        if (threadIdx.x == 0 && split == 0) svq_flag(SV_DEVERR_SEQ_LEN);
        n = len < 1 ? 0 : a.max_pages;
    }

    if (warp == kProducer) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        const int32_t* pt_row = a.page_table + static_cast<int64_t>(b) * a.max_pages;
        const int32_t* sel_row = a.sel_idx ? a.sel_idx + static_cast<int64_t>(bg) * a.K : nullptr;
        pdl_wait();   // sel_idx / sel_cnt come from the top-K kernel launched just before
        int count = n;
        int spec_lp = -1;        // this lane's first list entry, fetched with the count
        bool spec_ok = false;    // true when the count is the one guessed below
        if (a.sel_idx) {
            // The top-K writes min(K, n) entries; guess that count so that the
            // first list entries load in the same round trip as the count.
            const int guess = min(a.K, n);
            const int chunk_g = (guess + a.num_splits - 1) / a.num_splits;
            const int j0_g = min(guess, split * chunk_g);
            const int my_g = min(guess, j0_g + chunk_g) - j0_g;
            spec_lp = lane < my_g ? sel_row[j0_g + lane] : -1;
            count = a.sel_cnt[bg];
            spec_ok = count == guess;
            if (count < 0 || count > a.K || count > n) {
                if (lane == 0 && split == 0) svq_flag(SV_DEVERR_SEL_IDX);
                count = max(0, min(count, min(a.K, n)));
            }
        }
        const int chunk = (count + a.num_splits - 1) / a.num_splits;
        const int j0 = min(count, split * chunk);
        const int my_count = min(count, j0 + chunk) - j0;
        const int u = lane >> 2, box = lane & 3;   // lane group u owns stage u
        const uint64_t policy = l2_evict_first_policy();
        const uint32_t fb = full0 + u * 8;
        const uint32_t eb = empty0 + u * 8;
        const void* tmap = box < 2 ? static_cast<const void*>(&tmap_k) : static_cast<const void*>(&tmap_v);
        const bool mover = (box & 1) == 0;         // lanes 4u (K) and 4u + 2 (V)
        const uint32_t dst = ring_s + u * kStageBytes + box * kBoxBytes;
        // Lane l resolves list position base + l to (physical page, valid
        // tokens); the next 32 are resolved while the current 32 are issued.
        auto resolve = [&](int base, int& phys_out, int& valid_out) {
            const int ii = base + lane;
            phys_out = -1;
            valid_out = 0;
            if (ii < my_count) {
                const int lp = sel_row ? (base == 0 && spec_ok ? spec_lp : sel_row[j0 + ii]) : j0 + ii;
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
        int last = -1;
        bool failed = false;
        for (int base = 0; base < my_count && !failed; base += 32) {
            resolve(base + 32, nxt_phys, nxt_valid);
            for (int sub = 0; sub < 32 && base + sub < my_count; sub += kStages) {
                // Lane group u issues list position i = base + sub + u into stage u.
                const int i = base + sub + u;
                const int phys = __shfl_sync(0xffffffffu, cur_phys, sub + u);
                const int valid = __shfl_sync(0xffffffffu, cur_valid, sub + u);
                bool ok = true;
                if (i < my_count) {
                    if (i >= kStages) ok = mbar_wait_bounded(eb, ((i / kStages) - 1) & 1);
                    if (ok) {
                        if (box == 0) {
                            s_valid[u] = phys >= 0 ? valid : 0;
                            if (phys >= 0) mbar_arrive_expect_tx(fb, kStageBytes);
                            else mbar_arrive(fb);
                        }
                        if (phys >= 0 && mover) {
                            const int y = static_cast<int>((static_cast<int64_t>(phys) * a.num_kv_heads + kvh) * kPage);
                            tma_load_3d_hint(dst, tmap, 0, y, 0, fb, policy);
                        }
                        last = i;
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
        if (failed) svq_flag(SV_DEVERR_TIMEOUT);
        // This group's copies land before the CTA (and its shared memory) retires.
        if (last >= 0) (void)mbar_wait_bounded(fb, (last / kStages) & 1);
        pdl_launch_dependents();
        return;
    }

    // ---------------- consumer warps: warp w takes the split's pages w, w + 4, ...
    const int quad = lane & 3;      // column pair of the accumulator fragments
    const int row = lane >> 2;      // row of the accumulator fragments
    // Q^T fragments (B operand): head `row` of the group, channels 16kk + 2 quad (+8).
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
    pdl_wait();
    // The producer's page count for this CTA (same formula, computed again here).
    int count = n;
    if (a.sel_idx) count = max(0, min(a.sel_cnt[bg], min(a.K, n)));
    const int chunk = (count + a.num_splits - 1) / a.num_splits;
    const int j0 = min(count, split * chunk);
    const int my_count = min(count, j0 + chunk) - j0;

    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};   // heads 2 quad, 2 quad + 1 (log2 units)
    float l_run[2] = {0.f, 0.f};               // lane-partial sums
    const int mat = lane >> 3, r8 = lane & 7;
    const int krow = r8 + 8 * (mat & 1);       // ldmatrix row of the key tile
    const int vrow = r8 + 8 * (mat >> 1);      // ldmatrix row of the value tile
    for (int i = warp; i < my_count; i += kConsumers) {
        const int stage = i % kStages;
        const bool ok = mbar_wait_bounded(full0 + stage * 8, (i / kStages) & 1);
        if (__any_sync(0xffffffffu, !ok)) {
            if (lane == 0) svq_flag(SV_DEVERR_TIMEOUT);
            break;
        }
        const uint32_t st_s = ring_s + stage * kStageBytes;
        const int valid = s_valid[stage];
        if (valid < kPage) {
            // Value rows past the fill hold whatever the pool holds there; zero
            // them so that P = 0 never meets a NaN.  (Key rows are masked on
            // the logits.)
            unsigned char* vb = ring + stage * kStageBytes + 2 * kBoxBytes;
            for (int c = lane; c < (kPage - valid) * 16; c += 32) {
                const int rr = valid + (c >> 4);
                *reinterpret_cast<uint4*>(vb + (c & 8 ? kBoxBytes : 0) + swz(rr, c & 7)) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }

        // S^T (16 tokens x 8 heads) = K (16 x 128) Q^T (128 x 8), two accumulation chains.
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t addr = st_s + (kk >> 2) * kBoxBytes + swz(krow, 2 * (kk & 3) + (mat >> 1));
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(addr, a0, a1, a2, a3);
            if (kk & 1) mma_bf16_16816(sb, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
            else mma_bf16_16816(sa, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        }
        // Scaled logits in log2 units; tokens past the page's fill are masked.
        const float x0 = row < valid ? (sa[0] + sb[0]) * a.scale_log2 : -INFINITY;       // token row,   head 2q
        const float x1 = row < valid ? (sa[1] + sb[1]) * a.scale_log2 : -INFINITY;       // token row,   head 2q+1
        const float x2 = row + 8 < valid ? (sa[2] + sb[2]) * a.scale_log2 : -INFINITY;   // token row+8, head 2q
        const float x3 = row + 8 < valid ? (sa[3] + sb[3]) * a.scale_log2 : -INFINITY;   // token row+8, head 2q+1
        // The base moves (warp max, correction of sums and outputs) only when
        // some lane holds a logit more than kRescaleSlack above it.
        const bool grow = x0 > m_run[0] + kRescaleSlack || x2 > m_run[0] + kRescaleSlack ||
                          x1 > m_run[1] + kRescaleSlack || x3 > m_run[1] + kRescaleSlack;
        if (__any_sync(0xffffffffu, grow)) {
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int s = 4; s < 32; s <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, s));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, s));
            }
            const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
            const float alpha0 = fast_exp2(m_run[0] - (mn0 == -INFINITY ? 0.f : mn0));
            const float alpha1 = fast_exp2(m_run[1] - (mn1 == -INFINITY ? 0.f : mn1));
            m_run[0] = mn0;
            m_run[1] = mn1;
            l_run[0] *= alpha0;
            l_run[1] *= alpha1;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                o[mt][0] *= alpha0;
                o[mt][1] *= alpha1;
                o[mt][2] *= alpha0;
                o[mt][3] *= alpha1;
            }
        }
        const float base0 = m_run[0] == -INFINITY ? 0.f : m_run[0];
        const float base1 = m_run[1] == -INFINITY ? 0.f : m_run[1];
        const float p0 = fast_exp2(x0 - base0), p1 = fast_exp2(x1 - base1);
        const float p2 = fast_exp2(x2 - base0), p3 = fast_exp2(x3 - base1);
        l_run[0] += p0 + p2;
        l_run[1] += p1 + p3;

        // P^T as the B operand: lane needs P[token 2 quad + {0,1} (+8)][head row].
        const uint32_t lo = pack_bf16x2(p0, p1);   // token row:   heads 2q, 2q+1
        const uint32_t hi = pack_bf16x2(p2, p3);   // token row+8: heads 2q, 2q+1
        const int src0 = (2 * quad) * 4 + (row >> 1);
        const int src1 = (2 * quad + 1) * 4 + (row >> 1);
        const uint32_t lo0 = __shfl_sync(0xffffffffu, lo, src0);
        const uint32_t lo1 = __shfl_sync(0xffffffffu, lo, src1);
        const uint32_t hi0 = __shfl_sync(0xffffffffu, hi, src0);
        const uint32_t hi1 = __shfl_sync(0xffffffffu, hi, src1);
        const uint32_t selector = (row & 1) ? 0x7632u : 0x5410u;
        const uint32_t pb0 = __byte_perm(lo0, lo1, selector);
        const uint32_t pb1 = __byte_perm(hi0, hi1, selector);

        // O^T (128 channels x 8) += V^T (128 x 16) P^T (16 x 8)
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const uint32_t addr = st_s + (2 + (mt >> 2)) * kBoxBytes + swz(vrow, 2 * (mt & 3) + (mat & 1));
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4_trans(addr, a0, a1, a2, a3);
            mma_bf16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
        }
        __syncwarp();   // every lane has read the stage before it is released
        if (lane == 0) mbar_arrive(empty0 + stage * 8);
    }

    // Full per-head sums over the 8 lanes sharing a head.
#pragma unroll
    for (int s = 4; s < 32; s <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], s);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], s);
    }

    // Merge the consumer warps through shared memory (the ring is idle: every
    // page of this CTA has been consumed, so no copy is in flight).
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
    float* sm_o = reinterpret_cast<float*>(ring);                   // [warp][8][128]
    float* sm_m = sm_o + kConsumers * kMaxGroup * kHeadDim;         // [warp][8]
    float* sm_l = sm_m + kConsumers * kMaxGroup;                    // [warp][8]
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
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
    const int S = a.num_splits;
    const int64_t qbase = static_cast<int64_t>(b) * a.num_q_heads + g * a.group;
    for (int idx = threadIdx.x; idx < a.group * kHeadDim; idx += kConsumers * 32) {
        const int h = idx / kHeadDim, d = idx % kHeadDim;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, sm_m[w * kMaxGroup + h]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) {
                const float e = fast_exp2(sm_m[w * kMaxGroup + h] - M);
                L += sm_l[w * kMaxGroup + h] * e;
                O += sm_o[(w * kMaxGroup + h) * kHeadDim + d] * e;
            }
        }
        a.o_part[((qbase + h) * S + split) * kHeadDim + d] = O;
        if (d == 0) a.ml_part[(qbase + h) * S + split] = make_float2(M, L);
    }
}

// One warp per (request, query head); lane l owns channels 4l .. 4l+3.
// The split statistics (one split per lane) and the first 16 splits' partial
// outputs are requested together, so the common case costs one round trip.
constexpr int kCombineThreads = 128;
constexpr int kCombineBatch = 16;

__global__ void __launch_bounds__(kCombineThreads) lse_combine_kernel(const float* __restrict__ o_part,
                                                                      const float2* __restrict__ ml_part,
                                                                      int num_splits, int64_t total_heads,
                                                                      __nv_bfloat16* __restrict__ out,
                                                                      float* __restrict__ lse) {
    const int64_t qh = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    pdl_wait();   // partials come from the split kernel launched just before
    if (qh >= total_heads) return;
    const float2* ml = ml_part + qh * num_splits;
    const float* ob = o_part + qh * num_splits * kHeadDim + 4 * lane;
    const float2 v0 = lane < num_splits ? ml[lane] : make_float2(-INFINITY, 0.f);
    const float2 v1 = lane + 32 < num_splits ? ml[lane + 32] : make_float2(-INFINITY, 0.f);
    // The first kCombineBatch splits' partials go to shared memory with async
    // copies issued back to back, so they arrive in the round trip of the
    // statistics above.
    __shared__ __align__(16) float4 stash[kCombineThreads / 32][kCombineBatch][32];
    float4* mine = &stash[threadIdx.x >> 5][0][lane];
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u)
        cp_async16(smem_addr(mine + u * 32), ob + u * kHeadDim, u < num_splits ? 16u : 0u);
    cp_async_commit();
    float M = fmaxf(v0.x, v1.x);
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, s));
    const float e0 = M == -INFINITY ? 0.f : exp2f(v0.x - M);   // exp2(-inf) = 0 for empty splits
    const float e1 = M == -INFINITY ? 0.f : exp2f(v1.x - M);
    float L = v0.y * e0 + v1.y * e1;
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) L += __shfl_xor_sync(0xffffffffu, L, s);

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](const float4& x, int s) {
        const float e = __shfl_sync(0xffffffffu, s < 32 ? e0 : e1, s & 31);
        if (s < num_splits) {
            acc.x += x.x * e;
            acc.y += x.y * e;
            acc.z += x.z * e;
            acc.w += x.w * e;
        }
    };
    cp_async_wait<0>();
    __syncwarp();
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) add(mine[u * 32], u);
    for (int s0 = kCombineBatch; s0 < num_splits; s0 += 8) {
        float4 r[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            r[u] = s0 + u < num_splits ? *reinterpret_cast<const float4*>(ob + (s0 + u) * kHeadDim)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 8; ++u) add(r[u], s0 + u);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat162 r01 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 r23 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&r01);
    packed.y = *reinterpret_cast<uint32_t*>(&r23);
    *reinterpret_cast<uint2*>(out + qh * kHeadDim + 4 * lane) = packed;
    if (lane == 0) lse[qh] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

int decode_max_splits(int pages) {
    const int cap = (pages + kMinPagesPerSplit - 1) / kMinPagesPerSplit;
    return max(1, min(kMaxSplits, cap));
}

// Most splits per row: rows of split_pages pages each when that many CTAs
// still put one on every SM; otherwise (few rows) the finer bound, so that
// idle SMs take the extra splits.
int split_cap(int pages, int64_t rows, int sm_count, int split_pages) {
    const int coarse = (pages + split_pages - 1) / split_pages;
    const int fine = decode_max_splits(pages);
    return static_cast<int64_t>(coarse) * rows >= sm_count ? max(1, min(fine, coarse)) : fine;
}

size_t decode_workspace_bytes(int batch, int num_q_heads, int splits) {
    const size_t heads = static_cast<size_t>(batch) * num_q_heads * splits;
    const size_t o_bytes = ((heads * kHeadDim * sizeof(float)) + 255) / 256 * 256;
    return o_bytes + heads * sizeof(float2);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_entry());
}

// A pool bf16 [pages][kv heads][16][128] seen as a 3-D tensor: 64 channels
// (contiguous), pages * kv heads * 16 rows (256 bytes apart), 2 channel
// halves (128 bytes apart).  A box of 64 x 16 x 2 is one page's tile of one
// kv head; in shared memory it lands as the low half's 16 rows, then the high
// half's, each row of 128 bytes swizzled (128-byte swizzle).
bool encode_pool_map(CUtensorMap* map, const void* pool, int64_t rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), 2};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kPage), 2};
    const cuuint32_t estride[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int decode_fp8_splits(const sv_cache* c, int batch, int rows_per_req, int pages, int sm_count, int max_splits);
int launch_decode_fp8_split(const sv_cache* c, const void* q, int num_q_heads, const int32_t* page_table,
                            const int32_t* seq_lens, int batch, int max_pages, const int32_t* sel_idx,
                            const int32_t* sel_cnt, int budget_pages, bool per_head, float softmax_scale, int splits,
                            float* o_part, float2* ml_part, cudaStream_t stream);

int launch_decode(const sv_cache* c, const void* q, int num_q_heads, const int32_t* page_table,
                  const int32_t* seq_lens, int batch, int max_pages, const int32_t* sel_idx,
                  const int32_t* sel_cnt, int budget_pages, bool per_q_head, float softmax_scale, void* out,
                  float* lse, void* workspace, size_t workspace_bytes, int sm_count, cudaStream_t stream) {
    static std::atomic<bool> attr_set[64];
    const int st0 = once_per_device(attr_set, [] {
        return cudaFuncSetAttribute(flash_decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kDecodeSmem) == cudaSuccess
                   ? SV_OK
                   : SV_ERR_CUDA;
    });
    if (st0) return st0;
    const int pages = sel_idx ? budget_pages : max_pages;
    if (c->kv_format == SV_KV_FP8_E4M3) {
        const bool per_head8 = per_q_head && sel_idx;
        const int rows8 = per_head8 ? num_q_heads : c->num_kv_heads;
        const int cap8 = split_cap(pages, static_cast<int64_t>(batch) * rows8, sm_count, kSplitPagesFp8);
        const int splits8 = decode_fp8_splits(c, batch, rows8, pages, sm_count, cap8);
        if (splits8 < 1) return SV_ERR_CUDA;
        if (decode_workspace_bytes(batch, num_q_heads, splits8) > workspace_bytes) return SV_ERR_WORKSPACE;
        const size_t heads8 = static_cast<size_t>(batch) * num_q_heads * splits8;
        float* o_part8 = static_cast<float*>(workspace);
        float2* ml_part8 = reinterpret_cast<float2*>(static_cast<unsigned char*>(workspace) +
                                                     ((heads8 * kHeadDim * sizeof(float)) + 255) / 256 * 256);
        int st = launch_decode_fp8_split(c, q, num_q_heads, page_table, seq_lens, batch, max_pages, sel_idx, sel_cnt,
                                         budget_pages, per_head8, softmax_scale, splits8, o_part8, ml_part8, stream);
        if (st) return st;
        const int64_t total_heads8 = static_cast<int64_t>(batch) * num_q_heads;
        const int64_t blocks8 = (total_heads8 * 32 + kCombineThreads - 1) / kCombineThreads;
        return launch_pdl(lse_combine_kernel, dim3(static_cast<unsigned>(blocks8)), dim3(kCombineThreads), 0, stream,
                          static_cast<const float*>(o_part8), static_cast<const float2*>(ml_part8), splits8,
                          total_heads8, static_cast<__nv_bfloat16*>(out), lse) == cudaSuccess
                   ? SV_OK
                   : SV_ERR_CUDA;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, flash_decode_split_kernel, kDecodeThreads,
                                                      kDecodeSmem) != cudaSuccess || per_sm < 1)
        return SV_ERR_CUDA;
    // Selection rows: one per kv head (its query heads share the page list),
    // or one per query head.  Dense decode always works per kv head.
    const bool per_head = per_q_head && sel_idx;
    const int rows_per_req = per_head ? num_q_heads : c->num_kv_heads;
    const int bh = batch * rows_per_req;
    int splits = static_cast<int>((static_cast<int64_t>(sm_count) * per_sm * SVQ_DECODE_WAVE_PERMILLE / 1000) / bh);
    splits = max(1, min(splits, split_cap(pages, bh, sm_count, kSplitPagesBf16)));
    if (decode_workspace_bytes(batch, num_q_heads, splits) > workspace_bytes) return SV_ERR_WORKSPACE;

    // TMA row coordinates are 32-bit.
    const int64_t rows = c->num_phys_pages * c->num_kv_heads * kPage;
    if (rows > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
    CUtensorMap tmap_k, tmap_v;
    if (!encode_pool_map(&tmap_k, c->k_pool, rows) || !encode_pool_map(&tmap_v, c->v_pool, rows)) return SV_ERR_CUDA;

    DecodeArgs a;
    a.num_phys_pages = c->num_phys_pages;
    a.num_kv_heads = c->num_kv_heads;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.num_q_heads = num_q_heads;
    a.group = per_head ? 1 : num_q_heads / c->num_kv_heads;
    a.rows_per_req = rows_per_req;
    a.kv_div = per_head ? num_q_heads / c->num_kv_heads : 1;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.max_pages = max_pages;
    a.sel_idx = sel_idx;
    a.sel_cnt = sel_cnt;
    a.K = sel_idx ? budget_pages : 0;
    a.num_splits = splits;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    const size_t heads = static_cast<size_t>(batch) * num_q_heads * splits;
    a.o_part = static_cast<float*>(workspace);
    a.ml_part = reinterpret_cast<float2*>(static_cast<unsigned char*>(workspace) +
                                          ((heads * kHeadDim * sizeof(float)) + 255) / 256 * 256);
    if (launch_pdl(flash_decode_split_kernel, dim3(splits, bh), dim3(kDecodeThreads), kDecodeSmem, stream, a, tmap_k,
                   tmap_v) != cudaSuccess)
        return SV_ERR_CUDA;
    const int64_t total_heads = static_cast<int64_t>(batch) * num_q_heads;
    const int64_t blocks = (total_heads * 32 + kCombineThreads - 1) / kCombineThreads;
    if (launch_pdl(lse_combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kCombineThreads), 0, stream,
                   static_cast<const float*>(a.o_part), static_cast<const float2*>(a.ml_part), splits, total_heads,
                   static_cast<__nv_bfloat16*>(out), lse) != cudaSuccess)
        return SV_ERR_CUDA;
    return SV_OK;
}

}  // namespace svq
