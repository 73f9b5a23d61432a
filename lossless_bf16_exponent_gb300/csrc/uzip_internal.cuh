// uzip_internal.cuh -- shared definitions of the libuzip CUDA sources: stream
// layout arithmetic, small PTX helpers and the error-return macro.
//
// Stream format version 1 is specified in include/uzip.h; the layout function
// below is its arithmetic (header, sign-mantissa bytes, packed codes, chunk
// offsets, escape blocks; the first four parts padded to 16 bytes).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "uzip.h"

namespace uzip {

constexpr uint32_t kStreamMagic = 0x31505A55u;    // "UZP1" little endian
constexpr uint32_t kStreamMagicE5 = 0x31455A55u;  // "UZE1": the FP8 E5M2 stream
constexpr uint32_t kStreamMagicS = 0x31535A55u;   // "UZS1": the Top-15 + sentinel stream
constexpr uint32_t kCodebookMagic = 0x42435A55u;  // "UZCB" little endian

__host__ __device__ __forceinline__ uint64_t pad16(uint64_t v) { return (v + 15) & ~uint64_t(15); }

struct Layout {
    uint64_t n, nc, off_a, off_b, off_c, off_d;
};

__host__ __device__ __forceinline__ Layout layout_of(uint64_t n, uint32_t chunk) {
    Layout L;
    L.n = n;
    L.nc = (n + chunk - 1) / chunk;
    L.off_a = UZIP_HEADER_BYTES;
    L.off_b = L.off_a + pad16(n);
    L.off_c = L.off_b + pad16((n + 1) / 2);
    L.off_d = L.off_c + pad16(4 * (L.nc + 1));
    return L;
}

// Stream formats: BF16 (the codec of the page's §3), FP8 E5M2 (§4.2 /
// appendix C: the same Top-16 framework on E5M2 bytes; three bits of sign and
// mantissa per value, eight values per 3 bytes) and BF16 Top-15 + sentinel
// (§3.4, Table 6: code 15 marks an escape, one byte per escape, no positions).
enum Format : uint32_t { kBF16 = 0, kE5M2 = 1, kSentinel = 2 };

__host__ __device__ __forceinline__ Layout layout_e5m2_of(uint64_t n, uint32_t chunk) {
    Layout L;
    L.n = n;
    L.nc = (n + chunk - 1) / chunk;
    L.off_a = UZIP_HEADER_BYTES;
    L.off_b = L.off_a + pad16(3 * ((n + 7) / 8));
    L.off_c = L.off_b + pad16((n + 1) / 2);
    L.off_d = L.off_c + pad16(4 * (L.nc + 1));
    return L;
}

__host__ __device__ __forceinline__ Layout layout_for(uint32_t fmt, uint64_t n, uint32_t chunk) {
    return fmt == kE5M2 ? layout_e5m2_of(n, chunk) : layout_of(n, chunk);
}

__host__ __device__ __forceinline__ bool chunk_valid(uint32_t chunk) {
    return chunk >= UZIP_MIN_CHUNK && chunk <= UZIP_MAX_CHUNK && chunk % 8 == 0;
}

__host__ __forceinline__ bool aligned16(const void* p) {
    return (reinterpret_cast<uintptr_t>(p) & 15) == 0;
}

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const unsigned long long* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Programmatic dependent launch (PTX griddepcontrol): let the next kernel of
// the stream launch now / wait until the previous kernel has completed and
// its writes are visible (a no-op when not launched as a dependent).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// 16-byte streaming load through the non-coherent path (data read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// L2 eviction priority (PTX createpolicy): data a later kernel of the same
// call reads back is stored with evict_last so the streamed tensor does not
// push it out of L2 first.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void st_u32_keep(void* p, uint32_t v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol) : "memory");
}

// Launchers shared by the entry points (calibrate.cu, encode.cu).
int calibrate_impl(const void* d_sample_bf16, size_t n_sample, void* d_codebook, cudaStream_t stream,
                   uint32_t fmt = kBF16);
int encode_impl(const void* d_in_bf16, size_t n, uint32_t chunk, const void* d_codebook, void* d_out,
                size_t out_capacity, void* d_workspace, size_t workspace_bytes, size_t* h_out_bytes,
                uzip_stream_t stream, uint32_t fmt = kBF16);

}  // namespace uzip

#define UZIP_CUDA_TRY(expr)                          \
    do {                                             \
        cudaError_t _e = (expr);                     \
        if (_e != cudaSuccess) return UZIP_ERR_CUDA; \
    } while (0)

