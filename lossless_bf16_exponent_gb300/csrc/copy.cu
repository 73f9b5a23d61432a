// copy.cu -- moving a stream whose length only the device knows yet.
//
// SplitZip review page, appendix B: compression, transfer and decompression
// are pipelined. A sender learns an encoded stream's length from its header,
// which the encoder writes on the device; copying exactly that many bytes on
// the device (rather than reading the header back to the host first) keeps
// the host out of the pipeline. The kernel reads the header, checks it, and
// copies [0, total) bytes with 16-byte vectors; either end may be pinned host
// memory (a copy over the host link), in which case a small grid with four
// loads in flight per thread fills the link and leaves the SMs to the codec.
#include <algorithm>

#include "uzip_internal.cuh"

namespace uzip {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) stream_copy_kernel(const uint8_t* __restrict__ src,
                                                                   uint8_t* __restrict__ dst, uint64_t capacity,
                                                                   unsigned long long* copied) {
    const uint4* h = reinterpret_cast<const uint4*>(src);
    const uint4 h0 = h[0], h3 = h[3];
    uint64_t total = 0;
    const bool magic = h0.x == kStreamMagic || h0.x == kStreamMagicE5 || h0.x == kStreamMagicS;
    if (magic && (h0.y & 0xFFFF) == UZIP_VERSION) total = (uint64_t)h3.x | ((uint64_t)h3.y << 32);
    if (total < UZIP_HEADER_BYTES || total > capacity) total = 0;  // not a whole stream: copy nothing
    if (copied && blockIdx.x == 0 && threadIdx.x == 0) *copied = total;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    const uint64_t vecs = total / 16;
    const uint64_t stride = (uint64_t)gridDim.x * kCopyThreads;
    for (uint64_t base = (uint64_t)blockIdx.x * kCopyThreads + threadIdx.x; base < vecs;
         base += stride * kCopyUnroll) {
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int j = 0; j < kCopyUnroll; j++)
            if (base + j * stride < vecs) v[j] = s4[base + j * stride];
#pragma unroll
        for (int j = 0; j < kCopyUnroll; j++)
            if (base + j * stride < vecs) d4[base + j * stride] = v[j];
    }
    if (blockIdx.x == 0 && threadIdx.x < total % 16) dst[vecs * 16 + threadIdx.x] = src[vecs * 16 + threadIdx.x];
}

// Where a pointer lives: kDevice (device or managed memory), kPinned (page-
// locked host memory, which a kernel reaches over the host link) or kOther
// (pageable host memory or an unknown address: no kernel may touch it).
enum Where { kDevice, kPinned, kOther };

Where where_is(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the error
        return kOther;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return kDevice;
    return a.type == cudaMemoryTypeHost ? kPinned : kOther;
}

}  // namespace
}  // namespace uzip

using namespace uzip;

extern "C" UZIP_API int uzip_stream_copy(const void* src_stream, void* dst, size_t capacity,
                                         unsigned long long* d_copied, uzip_stream_t stream) {
    if (!src_stream || !dst) return UZIP_ERR_ARG;
    if (!aligned16(src_stream) || !aligned16(dst) || (reinterpret_cast<uintptr_t>(d_copied) & 7)) return UZIP_ERR_ALIGN;
    if (capacity < UZIP_HEADER_BYTES) return UZIP_ERR_CAPACITY;
    int dev = 0, sms = 0;
    UZIP_CUDA_TRY(cudaGetDevice(&dev));
    UZIP_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const Where ws = where_is(src_stream), wd = where_is(dst);
    if (ws == kOther || wd == kOther || (d_copied && where_is(d_copied) == kOther)) return UZIP_ERR_ARG;
    const bool host_end = ws == kPinned || wd == kPinned;
    const uint64_t per_cta = (uint64_t)kCopyThreads * kCopyUnroll * 16;
    const uint64_t want = std::max<uint64_t>(1, (capacity + per_cta - 1) / per_cta);
    const uint64_t grid = std::min<uint64_t>(want, host_end ? 32 : (uint64_t)sms * 4);
    stream_copy_kernel<<<(unsigned)grid, kCopyThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(src_stream), static_cast<uint8_t*>(dst), capacity, d_copied);
    UZIP_CUDA_TRY(cudaGetLastError());
    return UZIP_OK;
}
