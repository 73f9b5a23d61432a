/*
 * uzip.h -- C ABI of libuzip, a fixed-length lossless BF16 exponent codec for
 * NVIDIA GB300 (sm_103a).
 *
 * The method is SplitZip's, as the review page "SplitZip: Ultra Fast Lossless
 * KV Compression for Disaggregated LLM Serving" states it:
 *   §3.2  each BF16 bit pattern x is split into an 8-bit exponent
 *         e = (x >> 7) & 0xff and an exact sign-mantissa byte
 *         a = ((x >> 8) & 0x80) | (x & 0x7f); e is mapped through a Top-16
 *         codebook to a 4-bit code (two codes per byte); exponents outside the
 *         Top-16 are escapes, stored as a 16-bit position inside their chunk plus
 *         the raw 8-bit exponent; size N + N/2 + 3M bytes for M escapes.
 *         Decoding unpacks the codes, looks them up in a 16-entry table,
 *         rebuilds x = ((a & 0x80) << 8) | (e << 7) | (a & 0x7f), then overwrites
 *         each escape with its exact exponent.
 *   §3.3  the Top-16 codebook is calibrated once, offline, from the exponent
 *         histogram of a representative sample, giving three lookup tables.
 *   §3.4  all 16 codes are real exponents; an escape carries a dummy code.
 *
 * Conventions for every entry point:
 *   - Pointers named d_* are device memory owned by the caller; h_* are host
 *     memory owned by the caller. The library allocates nothing, keeps no
 *     global state between calls and is safe to call from several host threads
 *     on different streams with different buffers.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and is asynchronous unless an entry point says it synchronises.
 *   - BF16 data are raw 16-bit patterns (any value, including NaN, Inf,
 *     subnormals and -0, round-trips bit-exactly).
 *   - Device pointers must be 16-byte aligned (UZIP_ERR_ALIGN otherwise).
 *   - Errors found on the host return at once and enqueue nothing. Errors found
 *     on the device are reported through a status word (see each call); no
 *     kernel traps or waits on another block.
 *
 * Compressed stream format, version 1 (all integers little endian; every part
 * before the escape section starts on a 16-byte boundary and is padded with
 * zero bytes to one):
 *   header  64 B   [0,4) "UZP1" | [4,6) u16 version = 1 | [6,8) u16 status
 *                  flags (0 = valid) | [8,16) u64 n | [16,20) u32 chunk |
 *                  [20,24) u32 nc = ceil(n / chunk) | [24,32) u64 M escapes |
 *                  [32,48) u8 exps[16] (code k <-> exponent exps[k]) |
 *                  [48,56) u64 total stream bytes | [56,64) zero
 *   A       n B    sign-mantissa bytes a_i
 *   B  ceil(n/2) B 4-bit codes, element 2j in the low nibble of byte j; an
 *                  escape carries the dummy code 0; a missing last high
 *                  nibble is 0
 *   C  4(nc+1) B   u32 offsets[c] = number of escapes in chunks < c
 *                  (offsets[nc] = M)
 *   D  3M B        chunk c's escape block starts at byte 3 * offsets[c]: its
 *                  k = offsets[c+1] - offsets[c] positions (u16, element index
 *                  minus c * chunk, ascending), then its k raw exponents
 *   total = 64 + pad16(n) + pad16(ceil(n/2)) + pad16(4(nc+1)) + 3M.
 * The page's size N + N/2 + 3M is the A + B + D payload; header, offsets and
 * padding are the metadata.
 */
#ifndef UZIP_H
#define UZIP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define UZIP_API __attribute__((visibility("default")))
#else
#define UZIP_API
#endif

/* Same type as cudaStream_t, so no CUDA header is needed to use this one. */
typedef struct CUstream_st *uzip_stream_t;

enum uzip_status {
    UZIP_OK = 0,
    UZIP_ERR_ARG = 1,       /* null pointer, size out of range, bad codebook  */
    UZIP_ERR_ALIGN = 2,     /* a device pointer is not 16-byte aligned         */
    UZIP_ERR_CHUNK = 3,     /* chunk not a multiple of 8 in [8, 65536]         */
    UZIP_ERR_CAPACITY = 4,  /* output or workspace buffer too small            */
    UZIP_ERR_CORRUPT = 5,   /* stream header or escape data inconsistent       */
    UZIP_ERR_TIMEOUT = 6,   /* reserved: no entry point waits on the device    */
    UZIP_ERR_CUDA = 7       /* a CUDA runtime call failed                      */
};

#define UZIP_VERSION 1
#define UZIP_HEADER_BYTES 64
#define UZIP_CODEBOOK_BYTES 4096
#define UZIP_MIN_CHUNK 8
#define UZIP_MAX_CHUNK 65536
#define UZIP_MAX_N 0xFFFFFFFFull /* offsets and M are stored in 32 bits */

/* Header status flags, set by the encoder's kernels. */
#define UZIP_FLAG_CAPACITY 0x1u /* the escapes did not fit in out_capacity   */

/* Codebook blob (UZIP_CODEBOOK_BYTES of device memory, written by
 * uzip_calibrate or uzip_codebook_from_exps):
 *   [0,4) "UZCB" | [4,8) u32 version 1 | [8,16) u64 calibration sample size |
 *   [16,32) u8 exps[16], most frequent first | [32,48) u8 decode table
 *   (code -> exponent, equal to exps) | [48,304) u8 encode table
 *   (exponent -> code, 0 for an escape) | [304,560) u8 escape table
 *   (exponent -> 1 if not in the Top-16) | [1024,3072) u64 histogram[256] of
 *   the calibration sample (zero for uzip_codebook_from_exps) | [3072,3088)
 *   working space of uzip_calibrate, zero when it has finished. */
#define UZIP_CB_EXPS 16
#define UZIP_CB_DEC 32
#define UZIP_CB_ENC 48
#define UZIP_CB_ESC 304
#define UZIP_CB_HIST 1024

/* Offline calibration (§3.3): histogram of all exponents of the sample, the 16
 * most frequent exponents (code k = k-th most frequent; equal counts -> the
 * smaller exponent first; exponents the sample lacks fill the remaining codes
 * in ascending order), then the three lookup tables.
 *   d_sample_bf16  n_sample BF16 values (n_sample may be 0: codes 0..15 map to
 *                  exponents 0..15).
 *   d_codebook     UZIP_CODEBOOK_BYTES, overwritten.
 * Returns UZIP_ERR_ARG / UZIP_ERR_ALIGN / UZIP_ERR_CUDA, else UZIP_OK. Async. */
UZIP_API int uzip_calibrate(const void *d_sample_bf16, size_t n_sample, void *d_codebook,
                            uzip_stream_t stream);

/* Codebook from 16 given exponents (host array, code k -> h_exps16[k]); the
 * values must be distinct (UZIP_ERR_ARG otherwise). Builds the same three
 * tables as uzip_calibrate, histogram zero. Async; h_exps16 may be reused as
 * soon as the call returns. */
UZIP_API int uzip_codebook_from_exps(const uint8_t *h_exps16, void *d_codebook,
                                     uzip_stream_t stream);

/* Exact stream bytes for n values of which n_escapes are escapes (see the
 * format above); n_escapes = n gives the worst case. Returns 0 for an invalid
 * chunk, n > UZIP_MAX_N or n_escapes > n. Host only. */
UZIP_API size_t uzip_compressed_size(size_t n, size_t n_escapes, uint32_t chunk);

/* Device workspace bytes uzip_encode needs for (n, chunk): about n/4 bytes
 * (per 2048 values: an escape count, a list of up to 64 escape entries and
 * 256 escape-mask bytes; plus one total per segment of 64 or more such units);
 * 0 for an invalid chunk or n. Host only. */
UZIP_API size_t uzip_encode_workspace_bytes(size_t n, uint32_t chunk);

/* Encode n BF16 values (§3.2), reading the input from HBM once: a dense kernel
 * (sign-mantissa bytes, packed codes, per-unit escape lists and counts) and an
 * escape kernel (chunk offsets from the escape-count prefix, escape blocks in
 * ascending element order, header). Each call launches, on `stream`, a
 * one-block kernel that clears the per-segment escape totals (inputs of more
 * than 64 units of 2048 values only) and the two kernels; the later launches
 * start early (programmatic dependent launch) and wait on the device for the
 * data they need.
 *   d_in_bf16      n BF16 values (may be NULL when n == 0).
 *   chunk          escape-position chunk, a multiple of 8 in [8, 65536].
 *   d_codebook     from uzip_calibrate / uzip_codebook_from_exps.
 *   d_out          stream buffer of out_capacity bytes. out_capacity must hold
 *                  at least uzip_compressed_size(n, 0, chunk) (UZIP_ERR_CAPACITY
 *                  at once otherwise); uzip_compressed_size(n, n, chunk) can
 *                  never overflow. If the escapes do not fit, the kernel writes
 *                  none past out_capacity and sets UZIP_FLAG_CAPACITY in the
 *                  header.
 *   d_workspace    at least uzip_encode_workspace_bytes(n, chunk) bytes, 16-byte
 *                  aligned, any contents (the call clears what it accumulates
 *                  into and writes everything else before reading it); must not
 *                  be shared with a call that may overlap on the GPU.
 *   h_out_bytes    NULL: fully asynchronous; read the total from the header.
 *                  Non-NULL: the call synchronises `stream`, stores the exact
 *                  stream size and returns UZIP_ERR_CAPACITY if the kernels
 *                  set that header flag.
 * Bytes of d_out past the stream's total are not written. */
UZIP_API int uzip_encode(const void *d_in_bf16, size_t n, uint32_t chunk, const void *d_codebook,
                         void *d_out, size_t out_capacity, void *d_workspace,
                         size_t workspace_bytes, size_t *h_out_bytes, uzip_stream_t stream);

/* uzip_encode for callers that cannot allocate device memory for the
 * workspace -- for example code that runs where a framework's caching
 * allocator already holds the device memory, or latency-critical paths that
 * must not call cudaMalloc, which can synchronise the device. The page has no
 * counterpart: this is a library convenience, not part of the method.
 *   The workspace is a device array built into the library, sized for at most
 *   UZIP_NOALLOC_MAX_N values (about 8.1 MiB, held on every GPU that loads the
 *   library until the process exits); n above that returns UZIP_ERR_CAPACITY
 *   before any CUDA call. Nothing is allocated: each call looks up the
 *   array's address for the device and context current at the call (so a
 *   cudaDeviceReset between calls is harmless); the first call on a device
 *   may load the library's device code, so make it before any stream
 *   capture. All calls share the one array; the call
 *   clears what must start at zero, but calls that overlap on the GPU (other
 *   streams, other host threads) race on it and corrupt each other's output,
 *   so serialise them. Arguments, output and errors are otherwise those of
 *   uzip_encode, and the stream is byte-identical to uzip_encode's. */
#define UZIP_NOALLOC_MAX_N (1ull << 25)
UZIP_API int uzip_encode_noalloc(const void *d_in_bf16, size_t n, uint32_t chunk, const void *d_codebook,
                                 void *d_out, size_t out_capacity, size_t *h_out_bytes,
                                 uzip_stream_t stream);

/* Encode with a codebook built from the input itself (§4.3, Table 7: the
 * "dynamic Top-16" alternative to offline calibration): the histogram of all
 * n exponents, the Top-16 and the three tables are written to d_codebook
 * (exactly what uzip_calibrate(d_in_bf16, n, d_codebook) writes), then the
 * input is encoded with them; the input is read twice.
 *   d_codebook     UZIP_CODEBOOK_BYTES of device memory, overwritten.
 * Other arguments, output and errors are those of uzip_encode; the stream is
 * byte-identical to uzip_encode's with that codebook. */
UZIP_API int uzip_encode_dynamic(const void *d_in_bf16, size_t n, uint32_t chunk, void *d_codebook,
                                 void *d_out, size_t out_capacity, void *d_workspace,
                                 size_t workspace_bytes, size_t *h_out_bytes, uzip_stream_t stream);

/* Decode a stream produced by uzip_encode (§3.2): dense unpack and lookup,
 * then the escape fix-up, fused per tile so each output byte is written once.
 *   d_stream       stream_bytes bytes (at least the header's total).
 *   d_out_bf16     n BF16 values; n must equal the header's n.
 *   d_status       NULL or one device uint32_t that receives UZIP_OK or the
 *                  error code. The kernel checks the header (magic, version,
 *                  status flags, n, chunk, nc, M, total <= stream_bytes) before
 *                  it writes any output; with a bad header it writes no output
 *                  and stores UZIP_ERR_CORRUPT. The rest of the stream must
 *                  follow the format: offsets[0] = 0, offsets[nc] = M, the
 *                  offsets rising, no chunk holding more escapes than values,
 *                  and in each block positions inside the chunk that rise
 *                  strictly (one entry per escape). A stream that breaks any
 *                  of these also gives UZIP_ERR_CORRUPT (its output is then
 *                  not trustworthy); a stream that keeps every rule is
 *                  accepted. No read or write leaves the buffers.
 * Returns host-detected errors only (UZIP_ERR_ARG, UZIP_ERR_ALIGN,
 * UZIP_ERR_CAPACITY if stream_bytes < 64, UZIP_ERR_CUDA). Async. */
UZIP_API int uzip_decode(const void *d_stream, size_t stream_bytes, void *d_out_bf16, size_t n,
                         uint32_t *d_status, uzip_stream_t stream);

/* Copy one encoded stream, exactly its header's total bytes, without the
 * host learning its length first (a sender in the encode -> transfer ->
 * decode pipeline of appendix B). The kernel reads the header at src_stream;
 * if it is a stream header of this version (any format: BF16, E5M2 or
 * Top-15 + sentinel) and its total is at most
 * capacity, bytes [0, total) are copied to dst, else nothing is.
 *   src_stream     16-byte aligned, at least capacity readable bytes; device
 *                  memory or pinned (mapped) host memory.
 *   dst            16-byte aligned, at least capacity writable bytes; device
 *                  or pinned host memory.
 *   capacity       at least UZIP_HEADER_BYTES.
 *   d_copied       NULL or one 8-byte aligned device (or pinned host) word
 *                  that receives the bytes copied (0 when nothing was).
 * When either end is host memory the copy uses a small grid that fills the
 * host link and leaves the SMs to concurrent codec kernels.
 * Returns UZIP_ERR_ARG (a NULL end, or an end or d_copied in pageable host
 * memory or at an address CUDA does not know; nothing is launched) /
 * UZIP_ERR_ALIGN / UZIP_ERR_CAPACITY / UZIP_ERR_CUDA, else UZIP_OK. Async. */
UZIP_API int uzip_stream_copy(const void *src_stream, void *dst, size_t capacity,
                              unsigned long long *d_copied, uzip_stream_t stream);

/* ------------------------------------------------------------ FP8 E5M2
 * The same Top-16 framework on FP8 E5M2 values (§4.2, appendix C: "a further
 * 1.14x on FP8 KV"). An E5M2 byte x splits into its 5-bit exponent
 * e = (x >> 2) & 0x1f and a 3-bit sign-mantissa field a = sign << 2 | mantissa;
 * the stream is laid out as for BF16 with magic "UZE1" and a sign-mantissa
 * section of 3 * ceil(n / 8) bytes (the 3-bit fields of values 8j .. 8j+7 form
 * the 24-bit little-endian word sum(a_{8j+i} << 3i) at bytes 3j .. 3j+2);
 * codes, offsets and escape blocks (raw 5-bit exponent in a byte) as for
 * BF16. Size 64 + A16(3 ceil(n/8)) + A16(ceil(n/2)) + A16(4(nc+1)) + 3M.
 * Codebook blobs have the BF16 layout (exponents 0..31 only); a workspace of
 * uzip_encode_workspace_bytes(n, chunk) bytes serves uzip_e5m2_encode. */

/* Calibrate a codebook from n_sample E5M2 bytes (as uzip_calibrate). */
UZIP_API int uzip_e5m2_calibrate(const void *d_sample_e5m2, size_t n_sample, void *d_codebook,
                                 uzip_stream_t stream);

/* Exact E5M2 stream bytes for n values with n_escapes escapes; 0 on invalid
 * arguments. Host only. */
UZIP_API size_t uzip_e5m2_compressed_size(size_t n, size_t n_escapes, uint32_t chunk);

/* Encode n E5M2 values (16-byte aligned bytes); arguments, output and errors
 * as uzip_encode's. */
UZIP_API int uzip_e5m2_encode(const void *d_in_e5m2, size_t n, uint32_t chunk, const void *d_codebook,
                              void *d_out, size_t out_capacity, void *d_workspace, size_t workspace_bytes,
                              size_t *h_out_bytes, uzip_stream_t stream);

/* Decode an E5M2 stream into n bytes; arguments, checks and errors as
 * uzip_decode's (a BF16 stream is refused as corrupt, and vice versa). */
UZIP_API int uzip_e5m2_decode(const void *d_stream, size_t stream_bytes, void *d_out_e5m2, size_t n,
                              uint32_t *d_status, uzip_stream_t stream);

/* ----------------------------------------------------- Top-15 + sentinel
 * The alternative the page measures and rejects (§3.4, Table 6): the 15 most
 * frequent exponents get codes 0..14, code 15 marks an escape and only the
 * escape's raw exponent is stored (no position), so the decoder finds escapes
 * by scanning the code stream. Stream: magic "UZS1", the BF16 layout, the
 * codebook bytes = the 15 exponents then 0, u32 per-chunk offsets, then one
 * byte per escape in ascending element order (chunk c's values at byte
 * offsets[c] of that section). Size 64 + A16(n) + A16(ceil(n/2)) +
 * A16(4(nc+1)) + M. */

/* Turn a codebook (uzip_calibrate / uzip_codebook_from_exps) into the
 * Top-15 + sentinel codebook of its first 15 exponents, in place. Async. */
UZIP_API int uzip_codebook_make_sentinel(void *d_codebook, uzip_stream_t stream);

/* Exact sentinel stream bytes for n values with n_escapes escapes. Host only. */
UZIP_API size_t uzip_sentinel_compressed_size(size_t n, size_t n_escapes, uint32_t chunk);

/* Encode BF16 values with a sentinel codebook; arguments, output and errors
 * as uzip_encode's. */
UZIP_API int uzip_sentinel_encode(const void *d_in_bf16, size_t n, uint32_t chunk, const void *d_codebook,
                                  void *d_out, size_t out_capacity, void *d_workspace, size_t workspace_bytes,
                                  size_t *h_out_bytes, uzip_stream_t stream);

/* Decode a sentinel stream; arguments and errors as uzip_decode's. Besides
 * the header, a chunk holding more or fewer code 15s than its offsets give
 * values, or offsets that do not run from 0 to M, give UZIP_ERR_CORRUPT. */
UZIP_API int uzip_sentinel_decode(const void *d_stream, size_t stream_bytes, void *d_out_bf16, size_t n,
                                  uint32_t *d_status, uzip_stream_t stream);

/* Host view of a stream header. */
typedef struct {
    uint64_t n;
    uint64_t escapes;     /* M */
    uint64_t total_bytes; /* whole stream */
    uint64_t payload_bytes; /* the page's size: n + ceil(n/2) + 3M for BF16,
                               3 ceil(n/8) + ceil(n/2) + 3M for E5M2,
                               n + ceil(n/2) + M for Top-15 + sentinel */
    uint32_t chunk;
    uint32_t nc;
    uint32_t version;
    uint32_t flags;       /* UZIP_FLAG_* */
    uint8_t exps[16];
    uint32_t format;      /* UZIP_FORMAT_* from the magic */
    uint32_t reserved;
} uzip_info_t;

enum uzip_format {
    UZIP_FORMAT_BF16 = 0,     /* "UZP1" */
    UZIP_FORMAT_E5M2 = 1,     /* "UZE1" */
    UZIP_FORMAT_SENTINEL = 2  /* "UZS1" */
};

/* Copy the header of a stream of any format to the host (synchronises
 * `stream`) and check it. Returns
 * UZIP_ERR_CORRUPT for a bad magic, version or inconsistent sizes, else
 * UZIP_OK (h_info is filled in both cases when the header was readable). */
UZIP_API int uzip_stream_info(const void *d_stream, size_t stream_bytes, uzip_info_t *h_info,
                              uzip_stream_t stream);

/* Static text for a status code. */
UZIP_API const char *uzip_status_string(int status);

/* UZIP_VERSION of the loaded library. */
UZIP_API int uzip_version(void);

#ifdef __cplusplus
}
#endif

#endif /* UZIP_H */
