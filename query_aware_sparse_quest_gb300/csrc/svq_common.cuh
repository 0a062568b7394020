// Device helpers shared by the svquest kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "svquest.h"

namespace svq {

constexpr int kPage = 16;      // tokens per page
constexpr int kHeadDim = 128;  // channels per head
constexpr int kMaxGroup = 8;   // query heads per kv head handled by one MMA n-tile

// ---------------------------------------------------------------- error word
// Each translation unit owns one device word; the host reads and clears it
// through the TU's reader (see svq_api.cu).
#define SVQ_DEFINE_ERROR_WORD(reader)                                              \
    static __device__ unsigned int svq_error_word = 0u;                            \
    static __device__ __forceinline__ void svq_flag(unsigned int bit) {            \
        atomicOr(&svq_error_word, bit);                                            \
    }                                                                              \
    int reader(uint32_t* flags, int reset) {                                       \
        unsigned int v = 0;                                                        \
        if (cudaMemcpyFromSymbol(&v, svq_error_word, sizeof v) != cudaSuccess)     \
            return SV_ERR_CUDA;                                                    \
        *flags |= v;                                                               \
        if (reset) {                                                               \
            unsigned int z = 0;                                                    \
            if (cudaMemcpyToSymbol(svq_error_word, &z, sizeof z) != cudaSuccess)   \
                return SV_ERR_CUDA;                                                \
        }                                                                          \
        return SV_OK;                                                              \
    }

// ---------------------------------------------------------------- loads
// 16-byte streaming load that bypasses L1 (data read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---------------------------------------------------------------- cp.async
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Copies 16 bytes global -> shared; src_bytes == 0 writes 16 zero bytes
// without reading the source.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- tensor-core tiles
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D(16x8 fp32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Page tile in shared memory: 16 rows of 256 bytes (16 chunks of 16 B).
// Chunk c of row r lives at chunk c ^ (r & 7), so that the 8 rows read by one
// ldmatrix phase hit 8 distinct 16-byte bank groups.
__device__ __forceinline__ uint32_t tile_offset(int row, int chunk) {
    return static_cast<uint32_t>(row * 256 + ((chunk ^ (row & 7)) << 4));
}

inline int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

}  // namespace svq
