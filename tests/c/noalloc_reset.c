/* uzip_encode_noalloc across a cudaDeviceReset, from plain C. The no-alloc
 * encoder's workspace is a device array built into the library, and host
 * code reaches it only through an address looked up at run time. A reset
 * destroys the context the library's device code was loaded in; the next call
 * runs in a new one, where the array (and every kernel attribute) may differ.
 * The program encodes the same input with uzip_encode (caller workspace) and
 * uzip_encode_noalloc, resets the device, uploads the input again and encodes
 * it both ways once more; the four streams must be byte-identical. Exit
 * status 0 on success; the failing step is printed otherwise. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "uzip.h"

#define CHECK(what, cond)                                      \
    do {                                                       \
        if (!(cond)) {                                         \
            fprintf(stderr, "noalloc_reset: %s failed\n", what); \
            return 1;                                          \
        }                                                      \
    } while (0)

/* Encode h_in both ways on a fresh set of device buffers; the two streams go
 * to h_a and h_b (cap bytes each), their sizes to *na and *nb. */
static int encode_both(const uint16_t *h_in, size_t n, uint32_t chunk, size_t cap, uint8_t *h_a, uint8_t *h_b,
                       size_t *na, size_t *nb) {
    const size_t wsb = uzip_encode_workspace_bytes(n, chunk);
    void *d_in = NULL, *d_cb = NULL, *d_s1 = NULL, *d_s2 = NULL, *d_ws = NULL;
    CHECK("cudaMalloc", cudaMalloc(&d_in, n * 2 + 16) == cudaSuccess && cudaMalloc(&d_cb, UZIP_CODEBOOK_BYTES) == cudaSuccess &&
                            cudaMalloc(&d_s1, cap) == cudaSuccess && cudaMalloc(&d_s2, cap) == cudaSuccess &&
                            cudaMalloc(&d_ws, wsb) == cudaSuccess);
    CHECK("copy in", cudaMemcpy(d_in, h_in, n * 2, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK("clear", cudaMemset(d_s1, 0, cap) == cudaSuccess && cudaMemset(d_s2, 0, cap) == cudaSuccess);
    CHECK("uzip_calibrate", uzip_calibrate(d_in, n, d_cb, NULL) == UZIP_OK);
    CHECK("uzip_encode", uzip_encode(d_in, n, chunk, d_cb, d_s1, cap, d_ws, wsb, na, NULL) == UZIP_OK);
    CHECK("uzip_encode_noalloc", uzip_encode_noalloc(d_in, n, chunk, d_cb, d_s2, cap, nb, NULL) == UZIP_OK);
    CHECK("copy out", cudaMemcpy(h_a, d_s1, cap, cudaMemcpyDeviceToHost) == cudaSuccess &&
                          cudaMemcpy(h_b, d_s2, cap, cudaMemcpyDeviceToHost) == cudaSuccess);
    cudaFree(d_in);
    cudaFree(d_cb);
    cudaFree(d_s1);
    cudaFree(d_s2);
    cudaFree(d_ws);
    return 0;
}

int main(int argc, char **argv) {
    const size_t n = argc > 1 ? (size_t)strtoull(argv[1], NULL, 10) : 3000017;
    const uint32_t chunk = argc > 2 ? (uint32_t)strtoul(argv[2], NULL, 10) : 1024;
    CHECK("size within the no-alloc limit", n <= UZIP_NOALLOC_MAX_N);
    uint16_t *h_in = (uint16_t *)malloc(n * sizeof(uint16_t) + 1);
    const size_t cap = uzip_compressed_size(n, n, chunk);
    uint8_t *h[4];
    for (int i = 0; i < 4; i++) h[i] = (uint8_t *)malloc(cap);
    CHECK("host allocation", h_in && h[0] && h[1] && h[2] && h[3] && cap > 0);
    uint32_t state = 777u;
    for (size_t i = 0; i < n; i++) { /* values around 1, about 3 % with any exponent (escapes) */
        state = state * 1664525u + 1013904223u;
        uint16_t x = (uint16_t)(0x3E00u + ((state >> 8) & 0x03FFu));
        if ((state >> 27) == 0) x = (uint16_t)((x & 0x807Fu) | (((state >> 18) & 0xFFu) << 7));
        if ((state >> 26) & 1u) x |= 0x8000u;
        h_in[i] = x;
    }
    size_t n0 = 0, n1 = 0, n2 = 0, n3 = 0;
    if (encode_both(h_in, n, chunk, cap, h[0], h[1], &n0, &n1)) return 1;
    CHECK("cudaDeviceReset", cudaDeviceReset() == cudaSuccess);
    if (encode_both(h_in, n, chunk, cap, h[2], h[3], &n2, &n3)) return 1;
    CHECK("equal sizes", n0 == n1 && n0 == n2 && n0 == n3 && n0 > 0 && n0 <= cap);
    CHECK("streams before the reset", memcmp(h[0], h[1], cap) == 0);
    CHECK("streams after the reset", memcmp(h[0], h[2], cap) == 0 && memcmp(h[0], h[3], cap) == 0);
    printf("noalloc_reset ok: n=%zu chunk=%u bytes=%zu\n", n, chunk, n0);
    for (int i = 0; i < 4; i++) free(h[i]);
    free(h_in);
    return 0;
}
