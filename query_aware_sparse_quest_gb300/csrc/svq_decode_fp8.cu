// Split-K flash decode over FP8 (e4m3) K/V pages (sv_cache.kv_format =
// SV_KV_FP8_E4M3): the same exact softmax attention over the selected pages
// (SparseEngine page, "method key points": the AttentionView consumed by the
// attention backend) with K and V rows stored as e4m3 codes and one fp32
// scale per (token, kv head) row.
//
// Per CTA: one producer warp and four consumer warps over an 8-stage ring.  A
// stage holds one page of one kv head: the K tile and the V tile, each a
// 16 x 128-byte TMA box with the 128-byte swizzle (2 KB), plus the page's 16
// K scales and 16 V scales (128 B, bulk copies) in a separate scale ring.
// Producer lanes 4u and 4u+1 feed stage u (K, V): the pages whose list
// position is u mod 8, each lane group on its own.
//
// The tensor cores read the codes without a staging pass.  e4m3 values are
// exact in f16, so codes convert to f16 pairs (cvt e4m3x2 -> f16x2) and feed
// mma.sync m16n8k16 with f16 operands (q is converted once; P is f16):
//  - K as the A operand of S^T = K Q^T: ldmatrix on the byte tile as 16-bit
//    elements hands lane (g, q) four consecutive channels 4q .. 4q+3 of token
//    rows g and g + 8 of a 16-channel block.  The MMA's k index is mapped to
//    channels as (2q, 2q+1) -> (4q, 4q+1) and (2q+8, 2q+9) -> (4q+2, 4q+3); a
//    dot product does not depend on the channel order, so the q fragments
//    (B operand) use the same map.
//  - V as the A operand of O^T += V^T P^T: the transposing byte ldmatrix
//    (m16n16 .b8) hands lane (g, q) tokens 4q .. 4q+3 of channels g and g + 8
//    of a 16-channel block, two tokens of one channel per 16-bit half, which
//    is what the pairwise conversion takes; the MMA's k slots (2q, 2q+1) and
//    (2q+8, 2q+9) are then tokens (4q, 4q+1) and (4q+2, 4q+3).  The logit
//    tile's rows are permuted to match (token_of_row), so that the weights
//    reach their B-operand lanes through the same four shuffles.
// Scales: the logit of token t is s_k(t) * (q . codes_t); the value weight of
// token t is p_t * s_v(t) (the softmax sum uses p_t).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "svq_common.cuh"

namespace svq {

SVQ_DEFINE_ERROR_WORD(read_error_decode_fp8)

constexpr int kF8Consumers = 4;
constexpr int kF8Threads = (kF8Consumers + 1) * 32;
constexpr int kF8Producer = kF8Consumers;
// Pages in flight per CTA.  Eight stages (34 KB of shared memory) let four
// CTAs share an SM, which the registers allow: sixteen consumer warps per SM
// and finer splits; sixteen stages left room for three.
constexpr int kF8Stages = 8;
constexpr int kF8LanesPerStage = 32 / kF8Stages; // producer lanes per stage: the first moves K, the second V
constexpr int kF8Box = kPage * kHeadDim;         // 16 rows x 128 e4m3 = 2 KB
constexpr int kF8Stage = 2 * kF8Box;             // K box | V box
constexpr int kF8ScaleBytes = 2 * kPage * 4;     // 16 K scales | 16 V scales
constexpr int kF8Smem = 1024 + kF8Stages * kF8Stage + kF8Stages * kF8ScaleBytes;
static_assert(kF8Stages % kF8Consumers == 0, "each ring stage must belong to one consumer warp");
static_assert(32 % kF8Stages == 0 && kF8LanesPerStage >= 2, "at least two producer lanes per stage");
static_assert(kF8Stages * kF8Stage >= (kF8Consumers * kMaxGroup * kHeadDim + 2 * kF8Consumers * kMaxGroup) * 4,
              "the warps merge through the ring");

struct DecodeF8Args {
    int64_t num_phys_pages;
    int num_kv_heads;
    const __nv_bfloat16* q;
    int num_q_heads;
    int group;                // query heads of one selection row
    int rows_per_req;         // selection rows per request
    int kv_div;               // row r reads kv head r / kv_div
    const int32_t* page_table;
    const int32_t* seq_lens;
    int max_pages;
    const int32_t* sel_idx;   // nullptr => dense
    const int32_t* sel_cnt;
    int K;
    int num_splits;
    float scale_log2;
    const float* k_scale;     // [pages][Hkv][16]
    const float* v_scale;
    float* o_part;            // [B][Hq][S][128]
    float2* ml_part;          // [B][Hq][S]
};

__device__ __forceinline__ float f8_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Two e4m3 codes (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes & 0xffffu), __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}
__device__ __forceinline__ uint32_t swz8(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
// Token held by row m of the S^T = K Q^T tile.  The value MMA reads tokens
// 4q .. 4q+3 as its k slots (2q, 2q+1, 2q+8, 2q+9), so the logit tile puts
// tokens 4q, 4q+1 in rows 2q, 2q+1 and tokens 4q+2, 4q+3 in rows 2q+8, 2q+9:
// the weights then reach their B-operand lanes through the usual shuffles.
__device__ __forceinline__ int token_of_row(int m) { return 4 * ((m & 7) >> 1) + (m & 1) + 2 * (m >> 3); }
// Two 16 x 16 byte tiles transposed: lane 4c + j receives bytes (rows 4j .. 4j+3,
// column c) in r0 and (rows 4j .. 4j+3, column c + 8) in r1 of tile 0, and the
// same of tile 1 in r2, r3.  Lanes 0-15 address tile 0's rows, lanes 16-31
// tile 1's.
__device__ __forceinline__ void ldmatrix_b8_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                     uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__global__ void __launch_bounds__(kF8Threads, 4) flash_decode_fp8_kernel(const __grid_constant__ DecodeF8Args a,
                                                                    const __grid_constant__ CUtensorMap tmap_k,
                                                                    const __grid_constant__ CUtensorMap tmap_v) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ int s_valid[kF8Stages];
    __shared__ __align__(8) uint64_t full_bar[kF8Stages];
    __shared__ __align__(8) uint64_t empty_bar[kF8Stages];

    const int split = blockIdx.x;
    const int bg = blockIdx.y;
    const int b = bg / a.rows_per_req;
    const int g = bg % a.rows_per_req;
    const int kvh = g / a.kv_div;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t raw_s = smem_addr(smem_raw);
    const uint32_t ring_s = (raw_s + 1023u) & ~1023u;   // 128-byte swizzle wants 1024-byte aligned boxes
    unsigned char* ring = smem_raw + (ring_s - raw_s);
    const uint32_t scale_s = ring_s + kF8Stages * kF8Stage;
    const float* scale_ring = reinterpret_cast<const float*>(ring + kF8Stages * kF8Stage);
    const uint32_t full0 = smem_addr(&full_bar[0]);
    const uint32_t empty0 = smem_addr(&empty_bar[0]);

    if (threadIdx.x == 0) {
        for (int st = 0; st < kF8Stages; ++st) {
            mbar_init(full0 + st * 8, 1);
            mbar_init(empty0 + st * 8, 1);   // stage s is consumed by warp s % kF8Consumers alone
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

    if (warp == kF8Producer) {
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
        const int u = lane / kF8LanesPerStage, part = lane % kF8LanesPerStage;   // stage u; part 0 moves K, part 1 V
        const uint64_t policy = l2_evict_first_policy();
        const bool mover = part < 2;
        const uint32_t fb = full0 + u * 8;
        const uint32_t eb = empty0 + u * 8;
        const void* tmap = part == 1 ? static_cast<const void*>(&tmap_v) : static_cast<const void*>(&tmap_k);
        const float* scale_src = part == 1 ? a.v_scale : a.k_scale;
        // Lane l resolves list position base + l to (physical page, valid
        // tokens); the next 32 are resolved while the current 32 are issued.
        auto resolve = [&](int base, int& phys_out, int& valid_out) {
            const int i = base + lane;
            phys_out = -1;
            valid_out = 0;
            if (i < my_count) {
                const int lp = sel_row ? (base == 0 && spec_ok ? spec_lp : sel_row[j0 + i]) : j0 + i;
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
        bool ok = true;
        for (int base = 0; base < my_count && ok; base += 32) {
            resolve(base + 32, nxt_phys, nxt_valid);
            for (int sub = 0; sub < 32 && base + sub < my_count; sub += kF8Stages) {
                // Lane group u issues list position i = base + sub + u into stage u.
                const int i = base + sub + u;
                const int phys = __shfl_sync(0xffffffffu, cur_phys, sub + u);
                const int valid = __shfl_sync(0xffffffffu, cur_valid, sub + u);
                bool mine_ok = true;
                if (mover && i < my_count) {
                    if (i >= kF8Stages) mine_ok = mbar_wait_bounded(eb, ((i / kF8Stages) - 1) & 1);
                    if (mine_ok) {
                        if (part == 0) {
                            s_valid[u] = phys >= 0 ? valid : 0;
                            if (phys >= 0) mbar_arrive_expect_tx(fb, kF8Stage + kF8ScaleBytes);
                            else mbar_arrive(fb);
                        }
                        if (phys >= 0) {
                            const int64_t head_row = static_cast<int64_t>(phys) * a.num_kv_heads + kvh;
                            tma_load_2d_hint(ring_s + u * kF8Stage + part * kF8Box, tmap, 0,
                                             static_cast<int>(head_row * kPage), fb, policy);
                            bulk_copy_g2s_hint(scale_s + u * kF8ScaleBytes + part * (kPage * 4),
                                               scale_src + head_row * kPage, kPage * 4, fb, policy);
                        }
                        last = i;
                    }
                }
                if (__any_sync(0xffffffffu, !mine_ok)) {
                    ok = false;
                    break;
                }
            }
            cur_phys = nxt_phys;
            cur_valid = nxt_valid;
        }
        if (!ok) svq_flag(SV_DEVERR_TIMEOUT);
        // This lane's copies land before the CTA (and its shared memory) retires.
        if (last >= 0) (void)mbar_wait_bounded(fb, (last / kF8Stages) & 1);
        pdl_launch_dependents();
        return;
    }

    // ---------------- consumer warps: warp w takes the split's pages w, w + 4, ...
    const int quad = lane & 3;
    const int row = lane >> 2;
    // Q^T fragments (f16, B operand) for the 8 MMAs over 16-channel blocks
    // c0 = 16 mm: k pair (2 quad, +1) -> channels c0 + 4 quad, +1; k pair
    // (2 quad + 8, +9) -> channels c0 + 4 quad + 2, +3.
    uint32_t qf[8][2];
    {
        const bool hv = row < a.group;
        const __nv_bfloat16* qh =
            a.q + (static_cast<int64_t>(b) * a.num_q_heads + g * a.group + (hv ? row : 0)) * kHeadDim;
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) {
            const int c = 16 * mm + 4 * quad;
            const uint2 w = hv ? *reinterpret_cast<const uint2*>(qh + c) : make_uint2(0u, 0u);
            qf[mm][0] = pack_half2(bf16lo(w.x), bf16hi(w.x));
            qf[mm][1] = pack_half2(bf16lo(w.y), bf16hi(w.y));
        }
    }
    pdl_wait();
    int count = n;
    if (a.sel_idx) count = max(0, min(a.sel_cnt[bg], min(a.K, n)));
    const int chunk = (count + a.num_splits - 1) / a.num_splits;
    const int j0 = min(count, split * chunk);
    const int my_count = min(count, j0 + chunk) - j0;

    float o[8][4];   // o[mt]: output channels 16 mt + r (and + 8), heads 2 quad, 2 quad + 1
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    const int mat = lane >> 3, r8 = lane & 7;
    const int ktok = token_of_row(r8 + 8 * (mat & 1));   // K: matrices (rows 0-7 | 8-15) x (chunk 2kp | 2kp+1)
    const int kchunk_off = mat >> 1;
    const int tok0 = token_of_row(row), tok1 = token_of_row(row + 8);   // tokens of this lane's logits
    for (int i = warp; i < my_count; i += kF8Consumers) {
        const int stage = i % kF8Stages;
        const bool okw = mbar_wait_bounded(full0 + stage * 8, (i / kF8Stages) & 1);
        if (__any_sync(0xffffffffu, !okw)) {
            if (lane == 0) svq_flag(SV_DEVERR_TIMEOUT);
            break;
        }
        const uint32_t st_s = ring_s + stage * kF8Stage;
        const int valid = s_valid[stage];
        if (valid < kPage) {
            // Value rows past the fill hold whatever the pool holds there (NaN
            // codes included): zero them.  Key rows are masked on the logits.
            unsigned char* vb = ring + stage * kF8Stage + kF8Box;
            for (int c = lane; c < (kPage - valid) * 8; c += 32) {
                const int rr = valid + (c >> 3);
                *reinterpret_cast<uint4*>(vb + swz8(rr, c & 7)) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        const float* ks = scale_ring + stage * (kF8ScaleBytes / 4);
        const float* vs = ks + kPage;

        // S^T (16 tokens x 8 heads) = K Q^T over 128 channels.
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
            uint32_t r0, r1, r2, r3;
            ldmatrix_x4(st_s + swz8(ktok, 2 * kp + kchunk_off), r0, r1, r2, r3);
            mma_f16_16816(sa, e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r0 >> 16),
                          e4m3x2_to_f16x2(r1 >> 16), qf[2 * kp][0], qf[2 * kp][1]);
            mma_f16_16816(sb, e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r2 >> 16),
                          e4m3x2_to_f16x2(r3 >> 16), qf[2 * kp + 1][0], qf[2 * kp + 1][1]);
        }
        const bool v0 = tok0 < valid, v1 = tok1 < valid;
        const float ks0 = v0 ? ks[tok0] : 0.f, ks1 = v1 ? ks[tok1] : 0.f;
        const float x0 = v0 ? (sa[0] + sb[0]) * ks0 * a.scale_log2 : -INFINITY;   // token tok0, head 2q
        const float x1 = v0 ? (sa[1] + sb[1]) * ks0 * a.scale_log2 : -INFINITY;   // token tok0, head 2q+1
        const float x2 = v1 ? (sa[2] + sb[2]) * ks1 * a.scale_log2 : -INFINITY;   // token tok1, head 2q
        const float x3 = v1 ? (sa[3] + sb[3]) * ks1 * a.scale_log2 : -INFINITY;   // token tok1, head 2q+1
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int s = 4; s < 32; s <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, s));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, s));
        }
        const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
        const float base0 = mn0 == -INFINITY ? 0.f : mn0;
        const float base1 = mn1 == -INFINITY ? 0.f : mn1;
        const float alpha0 = f8_exp2(m_run[0] - base0), alpha1 = f8_exp2(m_run[1] - base1);
        const float p0 = f8_exp2(x0 - base0), p1 = f8_exp2(x1 - base1);
        const float p2 = f8_exp2(x2 - base0), p3 = f8_exp2(x3 - base1);
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
        // Value weights p_t * s_v(t) as P^T (k slots x heads, f16): lane (g, q)
        // needs tokens 4q, 4q+1 (slots 2q, 2q+1) and 4q+2, 4q+3 (slots 2q+8,
        // 2q+9) of head g, held by the lanes of rows 2q and 2q+1.
        const float vs0 = v0 ? vs[tok0] : 0.f, vs1 = v1 ? vs[tok1] : 0.f;
        const uint32_t lo = pack_half2(p0 * vs0, p1 * vs0);   // token tok0: heads 2q, 2q+1
        const uint32_t hi = pack_half2(p2 * vs1, p3 * vs1);   // token tok1: heads 2q, 2q+1
        const int src0 = (2 * quad) * 4 + (row >> 1);
        const int src1 = (2 * quad + 1) * 4 + (row >> 1);
        const uint32_t lo0 = __shfl_sync(0xffffffffu, lo, src0);
        const uint32_t lo1 = __shfl_sync(0xffffffffu, lo, src1);
        const uint32_t hi0 = __shfl_sync(0xffffffffu, hi, src0);
        const uint32_t hi1 = __shfl_sync(0xffffffffu, hi, src1);
        const uint32_t selector = (row & 1) ? 0x7632u : 0x5410u;
        const uint32_t pb0 = __byte_perm(lo0, lo1, selector);
        const uint32_t pb1 = __byte_perm(hi0, hi1, selector);

        // O^T += V^T P^T, 32 channels per transposing byte ldmatrix: lane
        // (g, q) gets tokens 4q .. 4q+3 of channels 16 mt + g and 16 mt + g + 8,
        // two tokens of one channel per 16-bit half, as the conversion wants.
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            uint32_t r0, r1, r2, r3;
            ldmatrix_b8_x2_trans(st_s + kF8Box + swz8(lane & 15, 2 * cb + (lane >> 4)), r0, r1, r2, r3);
            mma_f16_16816(o[2 * cb], e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r0 >> 16),
                          e4m3x2_to_f16x2(r1 >> 16), pb0, pb1);
            mma_f16_16816(o[2 * cb + 1], e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r2 >> 16),
                          e4m3x2_to_f16x2(r3 >> 16), pb0, pb1);
        }
        __syncwarp();   // every lane has read the stage before it is released
        if (lane == 0) mbar_arrive(empty0 + stage * 8);
    }

#pragma unroll
    for (int s = 4; s < 32; s <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], s);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], s);
    }

    // Merge the consumer warps through shared memory (every page of this CTA
    // has been consumed, so no copy is in flight into the ring).
    asm volatile("bar.sync 1, %0;" ::"n"(kF8Consumers * 32) : "memory");
    float* sm_o = reinterpret_cast<float*>(ring);                   // [warp][8][128]
    float* sm_m = sm_o + kF8Consumers * kMaxGroup * kHeadDim;       // [warp][8]
    float* sm_l = sm_m + kF8Consumers * kMaxGroup;                  // [warp][8]
    {
        float* ow = sm_o + warp * kMaxGroup * kHeadDim;
        const int h0 = 2 * quad, h1 = 2 * quad + 1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int ch = 16 * mt + row;
            ow[h0 * kHeadDim + ch] = o[mt][0];
            ow[h1 * kHeadDim + ch] = o[mt][1];
            ow[h0 * kHeadDim + ch + 8] = o[mt][2];
            ow[h1 * kHeadDim + ch + 8] = o[mt][3];
        }
        if (row == 0) {
            sm_m[warp * kMaxGroup + h0] = m_run[0];
            sm_m[warp * kMaxGroup + h1] = m_run[1];
            sm_l[warp * kMaxGroup + h0] = l_run[0];
            sm_l[warp * kMaxGroup + h1] = l_run[1];
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kF8Consumers * 32) : "memory");
    const int S = a.num_splits;
    const int64_t qbase = static_cast<int64_t>(b) * a.num_q_heads + g * a.group;
    for (int idx = threadIdx.x; idx < a.group * kHeadDim; idx += kF8Consumers * 32) {
        const int h = idx / kHeadDim, d = idx % kHeadDim;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kF8Consumers; ++w) M = fmaxf(M, sm_m[w * kMaxGroup + h]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kF8Consumers; ++w) {
                const float e = f8_exp2(sm_m[w * kMaxGroup + h] - M);
                L += sm_l[w * kMaxGroup + h] * e;
                O += sm_o[(w * kMaxGroup + h) * kHeadDim + d] * e;
            }
        }
        a.o_part[((qbase + h) * S + split) * kHeadDim + d] = O;
        if (d == 0) a.ml_part[(qbase + h) * S + split] = make_float2(M, L);
    }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 f8_tensor_map_encoder() {
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_entry());
}

// An e4m3 pool [pages][kv heads][16][128] as a 2-D byte tensor
// [pages * kv heads * 16 rows][128], read in 16 x 128-byte boxes with the
// 128-byte swizzle.
bool encode_f8_pool_map(CUtensorMap* map, const void* pool, int64_t rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = f8_tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kHeadDim), static_cast<cuuint32_t>(kPage)};
    const cuuint32_t estride[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int decode_fp8_splits(const sv_cache* c, int batch, int rows_per_req, int pages, int sm_count, int max_splits) {
    static std::atomic<bool> attr_set[64];
    if (once_per_device(attr_set, [] {
            return cudaFuncSetAttribute(flash_decode_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kF8Smem) == cudaSuccess
                       ? SV_OK
                       : SV_ERR_CUDA;
        }) != SV_OK)
        return -1;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, flash_decode_fp8_kernel, kF8Threads, kF8Smem) !=
            cudaSuccess ||
        per_sm < 1)
        return -1;
    (void)c;
    (void)pages;
    const int bh = batch * rows_per_req;
#ifndef SVQ_DECODE_WAVE_PERMILLE
#define SVQ_DECODE_WAVE_PERMILLE 1000   // split CTAs as a fraction of one full wave
#endif
    const int splits = static_cast<int>((static_cast<int64_t>(sm_count) * per_sm * SVQ_DECODE_WAVE_PERMILLE / 1000) / bh);
    return max(1, min(splits, max_splits));
}

int launch_decode_fp8_split(const sv_cache* c, const void* q, int num_q_heads, const int32_t* page_table,
                            const int32_t* seq_lens, int batch, int max_pages, const int32_t* sel_idx,
                            const int32_t* sel_cnt, int budget_pages, bool per_head, float softmax_scale, int splits,
                            float* o_part, float2* ml_part, cudaStream_t stream) {
    const int64_t rows = c->num_phys_pages * c->num_kv_heads * kPage;
    if (rows > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
    CUtensorMap tmap_k, tmap_v;
    if (!encode_f8_pool_map(&tmap_k, c->k_pool, rows) || !encode_f8_pool_map(&tmap_v, c->v_pool, rows))
        return SV_ERR_CUDA;
    DecodeF8Args a;
    a.num_phys_pages = c->num_phys_pages;
    a.num_kv_heads = c->num_kv_heads;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.num_q_heads = num_q_heads;
    a.group = per_head ? 1 : num_q_heads / c->num_kv_heads;
    a.rows_per_req = per_head ? num_q_heads : c->num_kv_heads;
    a.kv_div = per_head ? num_q_heads / c->num_kv_heads : 1;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.max_pages = max_pages;
    a.sel_idx = sel_idx;
    a.sel_cnt = sel_cnt;
    a.K = sel_idx ? budget_pages : 0;
    a.num_splits = splits;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.k_scale = static_cast<const float*>(c->k_scale);
    a.v_scale = static_cast<const float*>(c->v_scale);
    a.o_part = o_part;
    a.ml_part = ml_part;
    const int bh = batch * a.rows_per_req;
    return launch_pdl(flash_decode_fp8_kernel, dim3(splits, bh), dim3(kF8Threads), kF8Smem, stream, a, tmap_k,
                      tmap_v) == cudaSuccess
               ? SV_OK
               : SV_ERR_CUDA;
}

}  // namespace svq
