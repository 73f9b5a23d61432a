// api.cu -- host-only entry points of libuzip: exact stream sizes, header
// inspection and status text.
#include "uzip_internal.cuh"

using namespace uzip;

extern "C" UZIP_API size_t uzip_compressed_size(size_t n, size_t n_escapes, uint32_t chunk) {
    if (!chunk_valid(chunk) || n > UZIP_MAX_N || n_escapes > n) return 0;
    return (size_t)(layout_of(n, chunk).off_d + 3 * (uint64_t)n_escapes);
}

extern "C" UZIP_API int uzip_stream_info(const void* d_stream, size_t stream_bytes, uzip_info_t* h_info,
                                         uzip_stream_t stream) {
    if (!d_stream || !h_info) return UZIP_ERR_ARG;
    if (!aligned16(d_stream)) return UZIP_ERR_ALIGN;
    if (stream_bytes < UZIP_HEADER_BYTES) return UZIP_ERR_CORRUPT;
    uint8_t h[UZIP_HEADER_BYTES];
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    UZIP_CUDA_TRY(cudaMemcpyAsync(h, d_stream, sizeof(h), cudaMemcpyDeviceToHost, s));
    UZIP_CUDA_TRY(cudaStreamSynchronize(s));
    auto rd = [&](int off, int bytes) {
        uint64_t v = 0;
        for (int b = bytes - 1; b >= 0; b--) v = (v << 8) | h[off + b];
        return v;
    };
    h_info->version = (uint32_t)rd(4, 2);
    h_info->flags = (uint32_t)rd(6, 2);
    h_info->n = rd(8, 8);
    h_info->chunk = (uint32_t)rd(16, 4);
    h_info->nc = (uint32_t)rd(20, 4);
    h_info->escapes = rd(24, 8);
    for (int k = 0; k < 16; k++) h_info->exps[k] = h[32 + k];
    h_info->total_bytes = rd(48, 8);
    const uint32_t magic = (uint32_t)rd(0, 4);
    const uint32_t fmt = magic == kStreamMagicE5 ? kE5M2 : magic == kStreamMagicS ? kSentinel : kBF16;
    h_info->format = fmt;
    // The page's size: dense bytes, packed codes, escape bytes.
    const uint64_t dense = fmt == kE5M2 ? 3 * ((h_info->n + 7) / 8) : h_info->n;
    const uint64_t per_escape = fmt == kSentinel ? 1 : 3;
    h_info->payload_bytes = dense + (h_info->n + 1) / 2 + per_escape * h_info->escapes;
    if ((magic != kStreamMagic && magic != kStreamMagicE5 && magic != kStreamMagicS) ||
        h_info->version != UZIP_VERSION)
        return UZIP_ERR_CORRUPT;
    if (!chunk_valid(h_info->chunk) || h_info->n > UZIP_MAX_N || h_info->escapes > h_info->n)
        return UZIP_ERR_CORRUPT;
    const Layout L = layout_for(fmt, h_info->n, h_info->chunk);
    if (h_info->nc != L.nc || h_info->total_bytes != L.off_d + per_escape * h_info->escapes ||
        h_info->total_bytes > stream_bytes)
        return UZIP_ERR_CORRUPT;
    return UZIP_OK;
}

extern "C" UZIP_API const char* uzip_status_string(int status) {
    switch (status) {
        case UZIP_OK: return "ok";
        case UZIP_ERR_ARG: return "invalid argument";
        case UZIP_ERR_ALIGN: return "device pointer not 16-byte aligned";
        case UZIP_ERR_CHUNK: return "chunk must be a multiple of 8 in [8, 65536]";
        case UZIP_ERR_CAPACITY: return "output or workspace buffer too small";
        case UZIP_ERR_CORRUPT: return "corrupt or inconsistent stream";
        case UZIP_ERR_TIMEOUT: return "device-side wait timed out (not produced by this version)";
        case UZIP_ERR_CUDA: return "CUDA runtime error";
        default: return "unknown status";
    }
}

extern "C" UZIP_API int uzip_version(void) { return UZIP_VERSION; }
