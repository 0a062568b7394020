// Device helpers shared by the svquest kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

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

// ---------------------------------------------------------------- TMA bulk copies + mbarriers
// A bulk copy moves a contiguous run of bytes global -> shared through the
// tensor memory accelerator and reports completion (bytes) on an mbarrier;
// it holds no registers and no per-thread request slots while in flight.
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t arrivals) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(arrivals) : "memory");
}
// Makes initialised mbarriers visible to the async proxy.
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Every wait in these kernels gives up after kWaitLimitCycles SM clock cycles
// (about 0.27 s at 1 GHz; no legitimate wait comes near it: copies land in
// microseconds and a step lasts well under a millisecond), and after
// kMbarPollLimit polls whatever the clock says.  The clock is read every
// 16th poll only, so that a waiting warp still notices a completed phase
// within a few cycles.
constexpr long long kWaitLimitCycles = 1ll << 28;
constexpr uint32_t kMbarPollLimit = 1u << 22;
__device__ __forceinline__ bool waited_too_long(uint32_t it, long long t0) {
    return (it & 15u) == 15u && clock64() - t0 > kWaitLimitCycles;
}
// Waits for the phase with the given parity to complete; false when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 0; it < kMbarPollLimit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (waited_too_long(it, t0)) return false;
    }
    return false;
}
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// 2-D tiled tensor copy (TMA) global -> shared through a tensor map that is a
// __grid_constant__ kernel parameter; x is the innermost coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
// An L2 policy for data read once per call (metadata, K/V tiles): those lines
// are evicted first, so that the small structures the kernels reuse (page
// tables, scores, selection lists, split partials, the query) stay in L2
// while a call streams far more than L2 holds past them.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_copy_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                                   uint64_t policy) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* tmap, int x, int y, uint32_t bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void* tmap, int x, int y, int z, uint32_t bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;"
        ::"r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

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

// D(16x8 fp32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
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

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels of one step are launched so that the next kernel's CTAs may start
// while the previous kernel drains.  Every CTA of every kernel waits
// (griddepcontrol.wait) before it touches memory an earlier kernel of the
// library writes and before it exits, so a kernel completes only after its
// predecessor has, and ordering stays transitive.  Where a kernel lets its
// dependents launch (griddepcontrol.launch_dependents) only decides when
// their CTAs may be scheduled, never what they may read.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline int current_device() {
    int dev = 0;
    return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

// One-time host set-up per device (a kernel attribute, a device query).  A
// slot per device index below 64 remembers that it succeeded; larger indices
// run it on every call.  The slots are atomics, so first calls from several
// host threads at once each run the idempotent set-up without a data race.
template <typename F>
inline int once_per_device(std::atomic<bool> (&done)[64], F&& setup) {
    const int dev = current_device();
    if (dev < 0) return SV_ERR_CUDA;
    if (dev < 64 && done[dev].load(std::memory_order_acquire)) return SV_OK;
    const int st = setup();
    if (st == SV_OK && dev < 64) done[dev].store(true, std::memory_order_release);
    return st;
}

// The driver's cuTensorMapEncodeTiled (ABI version 12000), looked up once per
// process (a function-local static, initialised thread-safely); null if the
// driver does not provide it.
inline void* tensor_map_encode_entry() {
    static void* const fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        const bool ok = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                                         &qr) == cudaSuccess &&
                        qr == cudaDriverEntryPointSuccess;
        return ok ? p : nullptr;
    }();
    return fn;
}

}  // namespace svq
