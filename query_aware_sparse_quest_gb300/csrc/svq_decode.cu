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
#include "svq_common.cuh"

namespace svq {

SVQ_DEFINE_ERROR_WORD(read_error_decode)

constexpr int kDecodeWarps = 4;
constexpr int kDecodeThreads = kDecodeWarps * 32;
constexpr int kStages = 3;                        // pages in flight per warp
constexpr int kTileBytes = kPage * kHeadDim * 2;  // 4 KB: one page of K (or V) for one kv head
constexpr int kStageBytes = 2 * kTileBytes;       // K + V
constexpr int kDecodeSmem = kDecodeWarps * kStages * kStageBytes;
constexpr int kMaxSplits = 64;
constexpr int kMinPagesPerSplit = 8;

struct DecodeArgs {
    const __nv_bfloat16* k_pool;
    const __nv_bfloat16* v_pool;
    int64_t num_phys_pages;
    int num_kv_heads;
    const __nv_bfloat16* q;
    int num_q_heads;
    int group;
    const int32_t* page_table;
    const int32_t* seq_lens;
    int max_pages;
    const int32_t* sel_idx;   // nullptr => dense
    const int32_t* sel_cnt;
    int K;
    int num_splits;
    float scale_log2;         // softmax_scale * log2(e)
    float* o_part;            // [B][Hq][S][128] unnormalised partial outputs
    float2* ml_part;          // [B][Hq][S] (running max in log2 units, sum of exp2)
};

__global__ void __launch_bounds__(kDecodeThreads) flash_decode_split_kernel(const DecodeArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_valid[kDecodeWarps][kStages];

    const int split = blockIdx.x;
    const int bg = blockIdx.y;
    const int b = bg / a.num_kv_heads;
    const int g = bg % a.num_kv_heads;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quad = lane & 3;      // column pair of the accumulator fragments
    const int row = lane >> 2;      // row of the accumulator fragments

    const int len = a.seq_lens[b];
    int n = (len + kPage - 1) / kPage;
    if (len < 1 || n > a.max_pages) {
        if (threadIdx.x == 0 && split == 0) svq_flag(SV_DEVERR_SEQ_LEN);
        n = len < 1 ? 0 : a.max_pages;
    }
    int count = n;
    if (a.sel_idx) {
        count = a.sel_cnt[bg];
        if (count < 0 || count > a.K || count > n) {
            if (threadIdx.x == 0 && split == 0) svq_flag(SV_DEVERR_SEL_IDX);
            count = max(0, min(count, min(a.K, n)));
        }
    }
    const int chunk = (count + a.num_splits - 1) / a.num_splits;
    const int j0 = min(count, split * chunk);
    const int j1 = min(count, j0 + chunk);
    // Pages of this warp: list positions j0 + warp + kDecodeWarps * i.
    const int my_count = (j1 - j0 > warp) ? (j1 - j0 - warp + kDecodeWarps - 1) / kDecodeWarps : 0;

    unsigned char* wbuf = smem + warp * kStages * kStageBytes;
    const uint32_t wbuf_s = smem_addr(wbuf);

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

    const int32_t* pt_row = a.page_table + static_cast<int64_t>(b) * a.max_pages;
    const int32_t* sel_row = a.sel_idx ? a.sel_idx + static_cast<int64_t>(bg) * a.K : nullptr;

    auto issue = [&](int i, int stage) {
        const int j = j0 + warp + kDecodeWarps * i;
        int lp = sel_row ? sel_row[j] : j;
        int valid = 0;
        int64_t phys = 0;
        if (lp < 0 || lp >= n) {
            if (lane == 0) svq_flag(SV_DEVERR_SEL_IDX);
        } else {
            phys = pt_row[lp];
            if (phys < 0 || phys >= a.num_phys_pages) {
                if (lane == 0) svq_flag(SV_DEVERR_PAGE_TABLE);
                phys = 0;
            } else {
                valid = (lp == n - 1) ? len - kPage * (n - 1) : kPage;
            }
        }
        if (lane == 0) s_valid[warp][stage] = valid;
        const int64_t tile = (phys * a.num_kv_heads + g) * (kPage * kHeadDim);
        const unsigned char* ksrc = reinterpret_cast<const unsigned char*>(a.k_pool + tile);
        const unsigned char* vsrc = reinterpret_cast<const unsigned char*>(a.v_pool + tile);
        const uint32_t kdst = wbuf_s + stage * kStageBytes;
        const uint32_t vdst = kdst + kTileBytes;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int c = lane + 32 * r;      // 16-byte chunk of the 4 KB tile
            const int trow = c >> 4, tch = c & 15;
            const uint32_t nbytes = trow < valid ? 16u : 0u;
            cp_async16(kdst + tile_offset(trow, tch), ksrc + c * 16, nbytes);
            cp_async16(vdst + tile_offset(trow, tch), vsrc + c * 16, nbytes);
        }
    };

#pragma unroll
    for (int st = 0; st < kStages; ++st) {
        if (st < my_count) issue(st, st);
        cp_async_commit();
    }

    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};   // heads 2 quad, 2 quad + 1 (log2 units)
    float l_run[2] = {0.f, 0.f};               // lane-partial sums

    for (int i = 0; i < my_count; ++i) {
        const int stage = i % kStages;
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const uint32_t ks = wbuf_s + stage * kStageBytes;
        const uint32_t vs = ks + kTileBytes;
        const int valid = s_valid[warp][stage];

        // S^T (16 tokens x 8 heads) = K (16 x 128) Q^T (128 x 8)
        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int mat = lane >> 3, r = lane & 7;
            const int trow = r + 8 * (mat & 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4(ks + tile_offset(trow, 2 * kk + (mat >> 1)), a0, a1, a2, a3);
                mma_bf16_16816(sacc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
            }
        }
        // Scaled logits in log2 units; tokens past the page's fill are masked.
        float x0 = row < valid ? sacc[0] * a.scale_log2 : -INFINITY;       // token row,   head 2q
        float x1 = row < valid ? sacc[1] * a.scale_log2 : -INFINITY;       // token row,   head 2q+1
        float x2 = row + 8 < valid ? sacc[2] * a.scale_log2 : -INFINITY;   // token row+8, head 2q
        float x3 = row + 8 < valid ? sacc[3] * a.scale_log2 : -INFINITY;   // token row+8, head 2q+1
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int s = 4; s < 32; s <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, s));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, s));
        }
        const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
        const float base0 = mn0 == -INFINITY ? 0.f : mn0;
        const float base1 = mn1 == -INFINITY ? 0.f : mn1;
        const float alpha0 = exp2f(m_run[0] - base0), alpha1 = exp2f(m_run[1] - base1);
        const float p0 = exp2f(x0 - base0), p1 = exp2f(x1 - base1);
        const float p2 = exp2f(x2 - base0), p3 = exp2f(x3 - base1);
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

        // O^T (128 x 8) += V^T (128 x 16) P^T (16 x 8)
        {
            const int mat = lane >> 3, r = lane & 7;
            const int trow = r + 8 * (mat >> 1);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4_trans(vs + tile_offset(trow, 2 * mt + (mat & 1)), a0, a1, a2, a3);
                mma_bf16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
            }
        }
        __syncwarp();
        if (i + kStages < my_count) issue(i + kStages, stage);
        cp_async_commit();
    }
    cp_async_wait<0>();

    // Full per-head sums over the 8 lanes sharing a head.
#pragma unroll
    for (int s = 4; s < 32; s <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], s);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], s);
    }

    // Merge the warps of this CTA through shared memory (reusing the page buffers).
    __syncthreads();
    float* sm_o = reinterpret_cast<float*>(smem);                              // [warp][8][128]
    float* sm_m = sm_o + kDecodeWarps * kMaxGroup * kHeadDim;                  // [warp][8]
    float* sm_l = sm_m + kDecodeWarps * kMaxGroup;                             // [warp][8]
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
    __syncthreads();
    const int S = a.num_splits;
    for (int idx = threadIdx.x; idx < a.group * kHeadDim; idx += kDecodeThreads) {
        const int h = idx / kHeadDim, d = idx % kHeadDim;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, sm_m[w * kMaxGroup + h]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kDecodeWarps; ++w) {
                const float e = exp2f(sm_m[w * kMaxGroup + h] - M);
                L += sm_l[w * kMaxGroup + h] * e;
                O += sm_o[(w * kMaxGroup + h) * kHeadDim + d] * e;
            }
        }
        const int64_t qh = static_cast<int64_t>(b) * a.num_q_heads + g * a.group + h;
        a.o_part[(qh * S + split) * kHeadDim + d] = O;
        if (d == 0) a.ml_part[qh * S + split] = make_float2(M, L);
    }
}

// One warp per (request, query head); lane l owns channels 4l .. 4l+3.
__global__ void __launch_bounds__(256) lse_combine_kernel(const float* __restrict__ o_part,
                                                          const float2* __restrict__ ml_part, int num_splits,
                                                          int64_t total_heads, __nv_bfloat16* __restrict__ out,
                                                          float* __restrict__ lse) {
    const int64_t qh = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (qh >= total_heads) return;
    const float2* ml = ml_part + qh * num_splits;
    float M = -INFINITY;
    for (int s = lane; s < num_splits; s += 32) M = fmaxf(M, ml[s].x);
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, s));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < num_splits; ++s) {
            const float2 v = ml[s];
            const float e = exp2f(v.x - M);   // exp2(-inf) = 0 for empty splits
            L += v.y * e;
            const float4 p = *reinterpret_cast<const float4*>(o_part + (qh * num_splits + s) * kHeadDim + 4 * lane);
            acc.x += p.x * e;
            acc.y += p.y * e;
            acc.z += p.z * e;
            acc.w += p.w * e;
        }
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

size_t decode_workspace_bytes(int batch, int num_q_heads, int splits) {
    const size_t heads = static_cast<size_t>(batch) * num_q_heads * splits;
    const size_t o_bytes = ((heads * kHeadDim * sizeof(float)) + 255) / 256 * 256;
    return o_bytes + heads * sizeof(float2);
}

int launch_decode(const sv_cache* c, const void* q, int num_q_heads, const int32_t* page_table,
                  const int32_t* seq_lens, int batch, int max_pages, const int32_t* sel_idx,
                  const int32_t* sel_cnt, int budget_pages, float softmax_scale, void* out, float* lse,
                  void* workspace, size_t workspace_bytes, int sm_count, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(flash_decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kDecodeSmem) != cudaSuccess)
            return SV_ERR_CUDA;
        attr_set[dev] = true;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, flash_decode_split_kernel, kDecodeThreads,
                                                      kDecodeSmem) != cudaSuccess || per_sm < 1)
        return SV_ERR_CUDA;
    const int pages = sel_idx ? budget_pages : max_pages;
    const int bh = batch * c->num_kv_heads;
    int splits = static_cast<int>((static_cast<int64_t>(sm_count) * per_sm) / bh);
    splits = max(1, min(splits, decode_max_splits(pages)));
    if (decode_workspace_bytes(batch, num_q_heads, splits) > workspace_bytes) return SV_ERR_WORKSPACE;

    DecodeArgs a;
    a.k_pool = static_cast<const __nv_bfloat16*>(c->k_pool);
    a.v_pool = static_cast<const __nv_bfloat16*>(c->v_pool);
    a.num_phys_pages = c->num_phys_pages;
    a.num_kv_heads = c->num_kv_heads;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.num_q_heads = num_q_heads;
    a.group = num_q_heads / c->num_kv_heads;
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
    dim3 grid(splits, bh);
    flash_decode_split_kernel<<<grid, kDecodeThreads, kDecodeSmem, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    const int64_t total_heads = static_cast<int64_t>(batch) * num_q_heads;
    const int64_t blocks = (total_heads * 32 + 255) / 256;
    lse_combine_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        a.o_part, a.ml_part, splits, total_heads, static_cast<__nv_bfloat16*>(out), lse);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace svq
