/* A plain C client of libuzip: no Python, no PyTorch. It fills a BF16 buffer
 * with a deterministic pattern (a linear congruential generator over bit
 * patterns of values around 1, about 6 % of them given any exponent, so that
 * rare exponents fall outside the Top-16 and escape),
 * calibrates on it, encodes (asking for the exact stream size), decodes with
 * a status word and checks the round trip bit for bit. Exit status 0 on
 * success; the failing step is printed otherwise. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "uzip.h"

#define CHECK(what, cond)                                  \
    do {                                                   \
        if (!(cond)) {                                     \
            fprintf(stderr, "roundtrip: %s failed\n", what); \
            return 1;                                      \
        }                                                  \
    } while (0)

int main(int argc, char **argv) {
    const size_t n = argc > 1 ? (size_t)strtoull(argv[1], NULL, 10) : 1000003;
    const uint32_t chunk = argc > 2 ? (uint32_t)strtoul(argv[2], NULL, 10) : 1024;
    uint16_t *h_in = (uint16_t *)malloc(n * sizeof(uint16_t) + 1);
    uint16_t *h_out = (uint16_t *)malloc(n * sizeof(uint16_t) + 1);
    CHECK("host allocation", h_in && h_out);
    uint32_t state = 12345u;
    for (size_t i = 0; i < n; i++) {
        state = state * 1664525u + 1013904223u;
        uint16_t x = (uint16_t)(0x3E00u + ((state >> 8) & 0x03FFu)); /* exponents 124..131 */
        if ((state >> 28) == 0)                                        /* about 6 %: any exponent */
            x = (uint16_t)((x & 0x807Fu) | (((state >> 18) & 0xFFu) << 7));
        if ((state >> 27) & 1u) x |= 0x8000u;                          /* sign */
        h_in[i] = x;
    }
    const size_t cap = uzip_compressed_size(n, n, chunk);
    const size_t wsb = uzip_encode_workspace_bytes(n, chunk);
    CHECK("sizes", cap > 0 && wsb > 0);
    void *d_in = NULL, *d_out = NULL, *d_stream = NULL, *d_ws = NULL, *d_cb = NULL;
    uint32_t *d_status = NULL;
    CHECK("cudaMalloc", cudaMalloc(&d_in, n * 2 + 16) == cudaSuccess && cudaMalloc(&d_out, n * 2 + 16) == cudaSuccess &&
                            cudaMalloc(&d_stream, cap) == cudaSuccess && cudaMalloc(&d_ws, wsb) == cudaSuccess &&
                            cudaMalloc(&d_cb, UZIP_CODEBOOK_BYTES) == cudaSuccess &&
                            cudaMalloc((void **)&d_status, sizeof(uint32_t)) == cudaSuccess);
    CHECK("copy in", cudaMemcpy(d_in, h_in, n * 2, cudaMemcpyHostToDevice) == cudaSuccess);

    CHECK("uzip_calibrate", uzip_calibrate(d_in, n, d_cb, NULL) == UZIP_OK);
    size_t nbytes = 0;
    CHECK("uzip_encode", uzip_encode(d_in, n, chunk, d_cb, d_stream, cap, d_ws, wsb, &nbytes, NULL) == UZIP_OK);
    CHECK("stream size", nbytes >= uzip_compressed_size(n, 0, chunk) && nbytes <= cap);
    uzip_info_t info;
    CHECK("uzip_stream_info", uzip_stream_info(d_stream, nbytes, &info, NULL) == UZIP_OK);
    CHECK("stream header", info.n == n && info.chunk == chunk && info.total_bytes == nbytes &&
                               uzip_compressed_size(n, info.escapes, chunk) == nbytes);
    CHECK("some escapes", n < 100000 || info.escapes > 0); /* rare exponents outside the Top-16 */
    CHECK("uzip_decode", uzip_decode(d_stream, nbytes, d_out, n, d_status, NULL) == UZIP_OK);
    uint32_t status = 1;
    CHECK("copy out", cudaMemcpy(&status, d_status, sizeof(status), cudaMemcpyDeviceToHost) == cudaSuccess &&
                          cudaMemcpy(h_out, d_out, n * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK("decode status", status == UZIP_OK);
    CHECK("bit-exact round trip", memcmp(h_in, h_out, n * 2) == 0);
    printf("roundtrip ok: n=%zu chunk=%u bytes=%zu escapes=%llu\n", n, chunk, nbytes,
           (unsigned long long)info.escapes);
    cudaFree(d_in);
    cudaFree(d_out);
    cudaFree(d_stream);
    cudaFree(d_ws);
    cudaFree(d_cb);
    cudaFree(d_status);
    free(h_in);
    free(h_out);
    return 0;
}
