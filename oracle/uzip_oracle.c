/*
 * uzip_oracle.c -- plain, slow, scalar CPU oracle for the fixed-length lossless
 * BF16 exponent codec ("SplitZip").
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's
 * CPU-baseline / reference arm are the only callers. The GPU library shares no
 * code, header, table or constant with this file: everything here is restated
 * from the page below, independently of the CUDA path.
 *
 * Source page: "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated
 * LLM Serving" (paper review), sections cited per function:
 *   §3.2  bit split e = (x >> 7) & 0xff, a = ((x >> 8) & 0x80) | (x & 0x7f),
 *         rebuild x = ((a & 0x80) << 8) | (e << 7) | (a & 0x7f);
 *         encode = (1) dense transform: store a verbatim, map e through the
 *         Top-16 code table, pack two 4-bit codes per byte; (2) scan the
 *         exponent stream and push exponents outside the Top-16 into chunked
 *         escape position / value arrays (16-bit position relative to the
 *         chunk, 8-bit raw exponent); size B = N + N/2 + 3M bytes;
 *         decode = (1) unpack codes, 16-entry decode table, rebuild every
 *         value; (2) overwrite every recorded escape with its exact exponent.
 *   §3.3  offline calibration: histogram of all exponents of a sample, pick the
 *         Top-16, build the encode, decode and escape-membership tables.
 *   §3.4  all 16 codes are real exponents; escapes carry a dummy code in the
 *         dense stream and are fixed through the explicit position array.
 *   §4.1  chunk size 1024 (the default; any multiple of 8 in [8, 65536] here).
 *
 * Readings of points the page leaves open (each one is a choice, not a fact
 * of the page):
 *   - code k is the k-th most frequent exponent; equal counts are ordered by
 *     the smaller exponent value first; unseen exponents fill the codebook in
 *     ascending value order;
 *   - the dummy code of an escape is 0;
 *   - code of element 2j sits in the low nibble of byte j, element 2j+1 in the
 *     high nibble; an odd element count leaves the last high nibble 0;
 *   - escapes are stored in ascending element order; chunk c's escape block is
 *     its k_c positions (u16, little endian) followed by its k_c values, and
 *     starts at byte 3 * offsets[c] of the escape section, where offsets[] is
 *     the exclusive prefix sum of the per-chunk escape counts (u32, nc + 1
 *     entries, offsets[nc] = M);
 *   - so a decoder accepts only offsets that rise from 0 to M and blocks whose
 *     positions lie inside their chunk and rise strictly (one entry per
 *     escape: a repeated or falling position is not a stream of this format);
 *   - the stream is: a 64-byte header, then the sign-mantissa bytes, the packed
 *     codes, the chunk offsets and the escape blocks, each of the first four
 *     parts padded with zero bytes to a multiple of 16 bytes.
 *
 * Header (little endian): [0,4) "UZP1"; [4,6) version 1; [6,8) status 0;
 * [8,16) n; [16,20) chunk; [20,24) nc; [24,32) M; [32,48) the 16 codebook
 * exponents (code k -> exps[k]); [48,56) total stream bytes; [56,64) zero.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_CHUNK = 3, ORC_ERR_CAPACITY = 4, ORC_ERR_CORRUPT = 5 };

/* ---------------------------------------------------------------- §3.2 split */

static uint8_t exponent_of(uint16_t x) { return (uint8_t)((x >> 7) & 0xFF); }

static uint8_t sign_mantissa_of(uint16_t x) { return (uint8_t)(((x >> 8) & 0x80) | (x & 0x7F)); }

static uint16_t rebuild(uint8_t a, uint8_t e)
{
    return (uint16_t)(((unsigned)(a & 0x80) << 8) | ((unsigned)e << 7) | (unsigned)(a & 0x7F));
}

void orc_split(const uint16_t *x, uint64_t n, uint8_t *e, uint8_t *a)
{
    for (uint64_t i = 0; i < n; i++) {
        e[i] = exponent_of(x[i]);
        a[i] = sign_mantissa_of(x[i]);
    }
}

void orc_merge(const uint8_t *a, const uint8_t *e, uint64_t n, uint16_t *x)
{
    for (uint64_t i = 0; i < n; i++) x[i] = rebuild(a[i], e[i]);
}

/* ---------------------------------------------------------- §3.3 calibration */

/* Frequency of every exponent value over the sample. */
void orc_histogram(const uint16_t *x, uint64_t n, uint64_t *hist)
{
    for (int v = 0; v < 256; v++) hist[v] = 0;
    for (uint64_t i = 0; i < n; i++) hist[exponent_of(x[i])]++;
}

/* The 16 most frequent exponents, most frequent first; ties -> smaller value
 * first. Plain insertion sort of the 256 values, which starts in ascending
 * value order and only moves a value past one with a strictly smaller count,
 * so equal counts keep ascending value order. */
void orc_top16(const uint64_t *hist, uint8_t *exps)
{
    int order[256];
    for (int v = 0; v < 256; v++) order[v] = v;
    for (int i = 1; i < 256; i++) {
        int v = order[i];
        int j = i - 1;
        while (j >= 0 && hist[order[j]] < hist[v]) {
            order[j + 1] = order[j];
            j--;
        }
        order[j + 1] = v;
    }
    for (int k = 0; k < 16; k++) exps[k] = (uint8_t)order[k];
}

/* The three lookup tables of §3.3: exponent -> 4-bit code (dummy 0 for an
 * escape), code -> exponent, exponent -> "is an escape". */
void orc_luts(const uint8_t *exps, uint8_t *enc, uint8_t *dec, uint8_t *esc)
{
    for (int v = 0; v < 256; v++) {
        enc[v] = 0;
        esc[v] = 1;
    }
    for (int k = 0; k < 16; k++) {
        enc[exps[k]] = (uint8_t)k;
        esc[exps[k]] = 0;
        dec[k] = exps[k];
    }
}

void orc_calibrate(const uint16_t *x, uint64_t n, uint8_t *exps)
{
    uint64_t hist[256];
    orc_histogram(x, n, hist);
    orc_top16(hist, exps);
}

/* ------------------------------------------------------------ stream layout */

static uint64_t pad16(uint64_t v) { return (v + 15) / 16 * 16; }

static int chunk_ok(uint32_t chunk) { return chunk >= 8 && chunk <= 65536 && chunk % 8 == 0; }

typedef struct {
    uint64_t n, nc, off_a, off_b, off_c, off_d;
} layout_t;

static layout_t layout_of(uint64_t n, uint32_t chunk)
{
    layout_t L;
    L.n = n;
    L.nc = (n + chunk - 1) / chunk;
    L.off_a = 64;
    L.off_b = L.off_a + pad16(n);
    L.off_c = L.off_b + pad16((n + 1) / 2);
    L.off_d = L.off_c + pad16(4 * (L.nc + 1));
    return L;
}

/* Exact stream bytes for n values with m escapes. */
uint64_t orc_stream_bytes(uint64_t n, uint64_t m, uint32_t chunk)
{
    if (!chunk_ok(chunk)) return 0;
    return layout_of(n, chunk).off_d + 3 * m;
}

uint64_t orc_count_escapes(const uint16_t *x, uint64_t n, const uint8_t *exps)
{
    uint8_t enc[256], dec[16], esc[256];
    orc_luts(exps, enc, dec, esc);
    uint64_t m = 0;
    for (uint64_t i = 0; i < n; i++) m += esc[exponent_of(x[i])];
    return m;
}

static void put_u16(uint8_t *p, uint32_t v)
{
    p[0] = (uint8_t)(v & 0xFF);
    p[1] = (uint8_t)((v >> 8) & 0xFF);
}

static void put_u32(uint8_t *p, uint32_t v)
{
    for (int b = 0; b < 4; b++) p[b] = (uint8_t)((v >> (8 * b)) & 0xFF);
}

static void put_u64(uint8_t *p, uint64_t v)
{
    for (int b = 0; b < 8; b++) p[b] = (uint8_t)((v >> (8 * b)) & 0xFF);
}

static uint32_t get_u16(const uint8_t *p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8); }

static uint32_t get_u32(const uint8_t *p)
{
    uint32_t v = 0;
    for (int b = 3; b >= 0; b--) v = (v << 8) | p[b];
    return v;
}

static uint64_t get_u64(const uint8_t *p)
{
    uint64_t v = 0;
    for (int b = 7; b >= 0; b--) v = (v << 8) | p[b];
    return v;
}

/* --------------------------------------------------------------- §3.2 encode */

int orc_encode(const uint16_t *x, uint64_t n, uint32_t chunk, const uint8_t *exps, uint8_t *out,
               uint64_t cap, uint64_t *out_bytes)
{
    if (!chunk_ok(chunk)) return ORC_ERR_CHUNK;
    if (n >= ((uint64_t)1 << 32)) return ORC_ERR_ARG;
    if (n > 0 && x == NULL) return ORC_ERR_ARG;
    if (out == NULL || exps == NULL) return ORC_ERR_ARG;

    uint8_t enc[256], dec[16], esc[256];
    orc_luts(exps, enc, dec, esc);

    layout_t L = layout_of(n, chunk);
    uint64_t m = orc_count_escapes(x, n, exps);
    uint64_t total = L.off_d + 3 * m;
    if (out_bytes) *out_bytes = total;
    if (total > cap) return ORC_ERR_CAPACITY;
    memset(out, 0, total);

    /* Stage 1, the dense transform: sign-mantissa byte verbatim, exponent
     * through the code table, two codes per byte. */
    uint8_t *A = out + L.off_a;
    uint8_t *B = out + L.off_b;
    for (uint64_t i = 0; i < n; i++) {
        uint8_t e = exponent_of(x[i]);
        A[i] = sign_mantissa_of(x[i]);
        uint8_t code = enc[e];
        if (i % 2 == 0)
            B[i / 2] = code;
        else
            B[i / 2] = (uint8_t)(B[i / 2] | (code << 4));
    }

    /* Stage 2, the escape scan: walk the exponent stream chunk by chunk and
     * append every exponent outside the Top-16 to that chunk's block. */
    uint8_t *C = out + L.off_c;
    uint8_t *D = out + L.off_d;
    uint64_t running = 0;
    for (uint64_t c = 0; c < L.nc; c++) {
        uint64_t start = c * chunk;
        uint64_t end = start + chunk < n ? start + chunk : n;
        uint64_t k = 0;
        for (uint64_t i = start; i < end; i++) k += esc[exponent_of(x[i])];
        put_u32(C + 4 * c, (uint32_t)running);
        uint8_t *block = D + 3 * running;
        uint64_t j = 0;
        for (uint64_t i = start; i < end; i++) {
            uint8_t e = exponent_of(x[i]);
            if (!esc[e]) continue;
            put_u16(block + 2 * j, (uint32_t)(i - start));
            block[2 * k + j] = e;
            j++;
        }
        running += k;
    }
    put_u32(C + 4 * L.nc, (uint32_t)running);

    memcpy(out, "UZP1", 4);
    out[4] = 1;
    out[5] = 0;
    put_u64(out + 8, n);
    put_u32(out + 16, chunk);
    put_u32(out + 20, (uint32_t)L.nc);
    put_u64(out + 24, m);
    memcpy(out + 32, exps, 16);
    put_u64(out + 48, total);
    return ORC_OK;
}

/* --------------------------------------------------------------- §3.2 decode */

int orc_decode(const uint8_t *in, uint64_t in_bytes, uint16_t *x, uint64_t n)
{
    if (in == NULL || (n > 0 && x == NULL)) return ORC_ERR_ARG;
    if (in_bytes < 64) return ORC_ERR_CORRUPT;
    if (memcmp(in, "UZP1", 4) != 0 || get_u16(in + 4) != 1 || get_u16(in + 6) != 0)
        return ORC_ERR_CORRUPT;
    uint64_t hn = get_u64(in + 8);
    uint32_t chunk = get_u32(in + 16);
    uint64_t nc = get_u32(in + 20);
    uint64_t m = get_u64(in + 24);
    uint64_t total = get_u64(in + 48);
    if (hn != n || !chunk_ok(chunk) || n >= ((uint64_t)1 << 32)) return ORC_ERR_CORRUPT;
    layout_t L = layout_of(n, chunk);
    if (nc != L.nc || m > n || total != L.off_d + 3 * m || total > in_bytes) return ORC_ERR_CORRUPT;

    const uint8_t *dec = in + 32;
    const uint8_t *A = in + L.off_a;
    const uint8_t *B = in + L.off_b;
    const uint8_t *C = in + L.off_c;
    const uint8_t *D = in + L.off_d;

    /* Offsets must rise from 0 to M. */
    if (get_u32(C) != 0 || get_u32(C + 4 * nc) != m) return ORC_ERR_CORRUPT;
    for (uint64_t c = 0; c < nc; c++)
        if (get_u32(C + 4 * c) > get_u32(C + 4 * (c + 1))) return ORC_ERR_CORRUPT;

    /* Stage 1, dense: unpack each code, look it up, rebuild every value
     * (escapes come out with the dummy code's exponent for now). */
    for (uint64_t i = 0; i < n; i++) {
        uint8_t code = (uint8_t)((B[i / 2] >> (4 * (i % 2))) & 0x0F);
        x[i] = rebuild(A[i], dec[code]);
    }

    /* Stage 2, sparse fix-up: overwrite each recorded escape with its exact
     * exponent. */
    for (uint64_t c = 0; c < nc; c++) {
        uint64_t o = get_u32(C + 4 * c);
        uint64_t k = get_u32(C + 4 * (c + 1)) - o;
        uint64_t start = c * chunk;
        uint64_t len = start + chunk < n ? chunk : n - start;
        if (k > len) return ORC_ERR_CORRUPT;
        const uint8_t *block = D + 3 * o;
        for (uint64_t j = 0; j < k; j++) {
            uint64_t pos = get_u16(block + 2 * j);
            if (pos >= len) return ORC_ERR_CORRUPT;
            /* Escapes are stored in ascending element order, one entry each:
             * a position that does not rise past the one before is corrupt. */
            if (j > 0 && pos <= get_u16(block + 2 * (j - 1))) return ORC_ERR_CORRUPT;
            x[start + pos] = rebuild(A[start + pos], block[2 * k + j]);
        }
    }
    return ORC_OK;
}

/* ====================================================== FP8 E5M2 variant
 *
 * Source page §4.2 and appendix C: the same Top-16 framework applied to FP8
 * E5M2 KV values compresses them a further 1.14x. An E5M2 value is one byte:
 * sign (bit 7), 5-bit exponent (bits 6..2), 2-bit mantissa (bits 1..0).
 * Readings (choices, not facts of the page):
 *   - split e = (x >> 2) & 0x1f and a 3-bit sign-mantissa field
 *     a = ((x >> 5) & 4) | (x & 3); rebuild x = ((a & 4) << 5) | (e << 2) | (a & 3);
 *   - the Top-16 of the 5-bit exponents is chosen with the same rules as for
 *     BF16 (count descending, smaller exponent first; unseen exponents fill in
 *     ascending order), over a 256-bin histogram whose bins 32..255 stay 0;
 *   - the 3-bit fields of values 8j .. 8j+7 form the 24-bit little-endian
 *     word sum(a_{8j+i} << 3i) at bytes 3j .. 3j+2 (a partial last group
 *     padded with zero fields): 3 bytes per 8 values, so 7 bits per value with
 *     the 4-bit code, i.e. 8/7 = 1.14x before escapes;
 *   - codes, chunk offsets and escape blocks exactly as for BF16, the raw
 *     exponent of an escape in a whole byte;
 *   - the stream is a 64-byte header with magic "UZE1" (otherwise as for
 *     BF16), the packed fields, the codes, the offsets and the escape blocks,
 *     the first four parts padded with zeros to a multiple of 16 bytes. */

static uint8_t e5m2_exponent(uint8_t x) { return (uint8_t)((x >> 2) & 0x1F); }

static uint8_t e5m2_sign_mantissa(uint8_t x) { return (uint8_t)(((x >> 5) & 4) | (x & 3)); }

static uint8_t e5m2_rebuild(uint8_t a, uint8_t e) { return (uint8_t)(((a & 4) << 5) | ((e & 0x1F) << 2) | (a & 3)); }

void orc_e5m2_split(const uint8_t *x, uint64_t n, uint8_t *e, uint8_t *a)
{
    for (uint64_t i = 0; i < n; i++) {
        e[i] = e5m2_exponent(x[i]);
        a[i] = e5m2_sign_mantissa(x[i]);
    }
}

void orc_e5m2_merge(const uint8_t *a, const uint8_t *e, uint64_t n, uint8_t *x)
{
    for (uint64_t i = 0; i < n; i++) x[i] = e5m2_rebuild(a[i], e[i]);
}

void orc_e5m2_histogram(const uint8_t *x, uint64_t n, uint64_t *hist)
{
    for (int b = 0; b < 256; b++) hist[b] = 0;
    for (uint64_t i = 0; i < n; i++) hist[e5m2_exponent(x[i])]++;
}

void orc_e5m2_calibrate(const uint8_t *x, uint64_t n, uint8_t *exps)
{
    uint64_t hist[256];
    orc_e5m2_histogram(x, n, hist);
    orc_top16(hist, exps);
}

static layout_t e5m2_layout_of(uint64_t n, uint32_t chunk)
{
    layout_t L;
    L.n = n;
    L.nc = (n + chunk - 1) / chunk;
    L.off_a = 64;
    L.off_b = L.off_a + pad16(3 * ((n + 7) / 8));
    L.off_c = L.off_b + pad16((n + 1) / 2);
    L.off_d = L.off_c + pad16(4 * (L.nc + 1));
    return L;
}

uint64_t orc_e5m2_stream_bytes(uint64_t n, uint64_t m, uint32_t chunk)
{
    if (!chunk_ok(chunk)) return 0;
    return e5m2_layout_of(n, chunk).off_d + 3 * m;
}

int orc_e5m2_encode(const uint8_t *x, uint64_t n, uint32_t chunk, const uint8_t *exps, uint8_t *out, uint64_t cap,
                    uint64_t *out_bytes)
{
    if (!chunk_ok(chunk)) return ORC_ERR_CHUNK;
    if (n >= ((uint64_t)1 << 32)) return ORC_ERR_ARG;
    if (n > 0 && x == NULL) return ORC_ERR_ARG;
    if (out == NULL || exps == NULL) return ORC_ERR_ARG;
    uint8_t enc[256], dec[16], esc[256];
    orc_luts(exps, enc, dec, esc);
    layout_t L = e5m2_layout_of(n, chunk);
    uint64_t m = 0;
    for (uint64_t i = 0; i < n; i++) m += esc[e5m2_exponent(x[i])];
    uint64_t total = L.off_d + 3 * m;
    if (out_bytes) *out_bytes = total;
    if (total > cap) return ORC_ERR_CAPACITY;
    memset(out, 0, total);

    /* Dense: each 3-bit field into its group's 24-bit word, each exponent
     * through the code table, two codes per byte. */
    uint8_t *A = out + L.off_a;
    uint8_t *B = out + L.off_b;
    for (uint64_t i = 0; i < n; i++) {
        uint32_t bit = 3 * (uint32_t)(i % 8);
        uint8_t *w = A + 3 * (i / 8);
        uint32_t word = (uint32_t)w[0] | ((uint32_t)w[1] << 8) | ((uint32_t)w[2] << 16);
        word |= (uint32_t)e5m2_sign_mantissa(x[i]) << bit;
        w[0] = (uint8_t)(word & 0xFF);
        w[1] = (uint8_t)((word >> 8) & 0xFF);
        w[2] = (uint8_t)((word >> 16) & 0xFF);
        uint8_t code = enc[e5m2_exponent(x[i])];
        if (i % 2 == 0)
            B[i / 2] = code;
        else
            B[i / 2] = (uint8_t)(B[i / 2] | (code << 4));
    }

    /* Escapes, chunk by chunk, as for BF16. */
    uint8_t *C = out + L.off_c;
    uint8_t *D = out + L.off_d;
    uint64_t running = 0;
    for (uint64_t c = 0; c < L.nc; c++) {
        uint64_t start = c * chunk;
        uint64_t end = start + chunk < n ? start + chunk : n;
        uint64_t k = 0;
        for (uint64_t i = start; i < end; i++) k += esc[e5m2_exponent(x[i])];
        put_u32(C + 4 * c, (uint32_t)running);
        uint8_t *block = D + 3 * running;
        uint64_t j = 0;
        for (uint64_t i = start; i < end; i++) {
            uint8_t e = e5m2_exponent(x[i]);
            if (!esc[e]) continue;
            put_u16(block + 2 * j, (uint32_t)(i - start));
            block[2 * k + j] = e;
            j++;
        }
        running += k;
    }
    put_u32(C + 4 * L.nc, (uint32_t)running);

    memcpy(out, "UZE1", 4);
    out[4] = 1;
    out[5] = 0;
    put_u64(out + 8, n);
    put_u32(out + 16, chunk);
    put_u32(out + 20, (uint32_t)L.nc);
    put_u64(out + 24, m);
    memcpy(out + 32, exps, 16);
    put_u64(out + 48, total);
    return ORC_OK;
}

int orc_e5m2_decode(const uint8_t *in, uint64_t in_bytes, uint8_t *x, uint64_t n)
{
    if (in == NULL || (n > 0 && x == NULL)) return ORC_ERR_ARG;
    if (in_bytes < 64) return ORC_ERR_CORRUPT;
    if (memcmp(in, "UZE1", 4) != 0 || get_u16(in + 4) != 1 || get_u16(in + 6) != 0) return ORC_ERR_CORRUPT;
    uint64_t hn = get_u64(in + 8);
    uint32_t chunk = get_u32(in + 16);
    uint64_t nc = get_u32(in + 20);
    uint64_t m = get_u64(in + 24);
    uint64_t total = get_u64(in + 48);
    if (hn != n || !chunk_ok(chunk) || n >= ((uint64_t)1 << 32)) return ORC_ERR_CORRUPT;
    layout_t L = e5m2_layout_of(n, chunk);
    if (nc != L.nc || m > n || total != L.off_d + 3 * m || total > in_bytes) return ORC_ERR_CORRUPT;
    const uint8_t *dec = in + 32;
    const uint8_t *A = in + L.off_a;
    const uint8_t *B = in + L.off_b;
    const uint8_t *C = in + L.off_c;
    const uint8_t *D = in + L.off_d;
    if (get_u32(C) != 0 || get_u32(C + 4 * nc) != m) return ORC_ERR_CORRUPT;
    for (uint64_t c = 0; c < nc; c++)
        if (get_u32(C + 4 * c) > get_u32(C + 4 * (c + 1))) return ORC_ERR_CORRUPT;

    /* Dense: field and code of every value, rebuilt with the decoded exponent. */
    for (uint64_t i = 0; i < n; i++) {
        const uint8_t *w = A + 3 * (i / 8);
        uint32_t word = (uint32_t)w[0] | ((uint32_t)w[1] << 8) | ((uint32_t)w[2] << 16);
        uint8_t a = (uint8_t)((word >> (3 * (i % 8))) & 7);
        uint8_t code = (uint8_t)((B[i / 2] >> (4 * (i % 2))) & 0x0F);
        x[i] = e5m2_rebuild(a, dec[code]);
    }
    /* Sparse fix-up of the escapes. */
    for (uint64_t c = 0; c < nc; c++) {
        uint64_t o = get_u32(C + 4 * c);
        uint64_t k = get_u32(C + 4 * (c + 1)) - o;
        uint64_t start = c * chunk;
        uint64_t len = start + chunk < n ? chunk : n - start;
        if (k > len) return ORC_ERR_CORRUPT;
        const uint8_t *block = D + 3 * o;
        for (uint64_t j = 0; j < k; j++) {
            uint64_t pos = get_u16(block + 2 * j);
            if (pos >= len) return ORC_ERR_CORRUPT;
            if (j > 0 && pos <= get_u16(block + 2 * (j - 1))) return ORC_ERR_CORRUPT; /* ascending, as for BF16 */
            x[start + pos] = (uint8_t)((x[start + pos] & 0x83) | ((block[2 * k + j] & 0x1F) << 2));
        }
    }
    return ORC_OK;
}

/* ============================================= Top-15 + sentinel variant
 *
 * Source page §3.4 and §4.3 Table 6: the alternative the page rejects keeps
 * one code word as an explicit escape token -- the Top-15 exponents get codes
 * 0..14, code 15 marks an escape -- so the decoder finds escapes in the code
 * stream and no positions are stored (a slightly higher ratio, 1.331x on the
 * page, and a slower decode). Readings (choices, not facts of the page):
 *   - the Top-15 are the first 15 of the Top-16 ranking (same rules);
 *   - an escape stores only its raw exponent byte, in ascending element order;
 *     u32 offsets[nc + 1] (exclusive prefix of per-chunk escape counts) are
 *     kept so every chunk decodes on its own: chunk c's values start at byte
 *     offsets[c] of the value section;
 *   - the stream is a 64-byte header with magic "UZS1" (codebook bytes: the 15
 *     exponents, then 0), the sign-mantissa bytes, the codes, the offsets and
 *     the values, the first four parts padded with zeros to 16 bytes. */

void orc_sentinel_luts(const uint8_t *exps, uint8_t *enc, uint8_t *dec, uint8_t *esc)
{
    for (int v = 0; v < 256; v++) {
        enc[v] = 15;
        esc[v] = 1;
    }
    for (int k = 0; k < 15; k++) {
        enc[exps[k]] = (uint8_t)k;
        esc[exps[k]] = 0;
        dec[k] = exps[k];
    }
    dec[15] = 0;
}

uint64_t orc_sentinel_stream_bytes(uint64_t n, uint64_t m, uint32_t chunk)
{
    if (!chunk_ok(chunk)) return 0;
    return layout_of(n, chunk).off_d + m;
}

int orc_sentinel_encode(const uint16_t *x, uint64_t n, uint32_t chunk, const uint8_t *exps, uint8_t *out,
                        uint64_t cap, uint64_t *out_bytes)
{
    if (!chunk_ok(chunk)) return ORC_ERR_CHUNK;
    if (n >= ((uint64_t)1 << 32)) return ORC_ERR_ARG;
    if (n > 0 && x == NULL) return ORC_ERR_ARG;
    if (out == NULL || exps == NULL) return ORC_ERR_ARG;
    uint8_t enc[256], dec[16], esc[256];
    orc_sentinel_luts(exps, enc, dec, esc);
    layout_t L = layout_of(n, chunk);
    uint64_t m = 0;
    for (uint64_t i = 0; i < n; i++) m += esc[exponent_of(x[i])];
    uint64_t total = L.off_d + m;
    if (out_bytes) *out_bytes = total;
    if (total > cap) return ORC_ERR_CAPACITY;
    memset(out, 0, total);

    /* Dense: as for Top-16, with code 15 for every escape. */
    uint8_t *A = out + L.off_a;
    uint8_t *B = out + L.off_b;
    for (uint64_t i = 0; i < n; i++) {
        A[i] = sign_mantissa_of(x[i]);
        uint8_t code = enc[exponent_of(x[i])];
        B[i / 2] = (uint8_t)(B[i / 2] | (code << (4 * (i % 2))));
    }
    /* Escape values only, chunk by chunk, behind per-chunk offsets. */
    uint8_t *C = out + L.off_c;
    uint8_t *D = out + L.off_d;
    uint64_t running = 0;
    for (uint64_t c = 0; c < L.nc; c++) {
        uint64_t start = c * chunk;
        uint64_t end = start + chunk < n ? start + chunk : n;
        put_u32(C + 4 * c, (uint32_t)running);
        for (uint64_t i = start; i < end; i++) {
            uint8_t e = exponent_of(x[i]);
            if (esc[e]) D[running++] = e;
        }
    }
    put_u32(C + 4 * L.nc, (uint32_t)running);

    memcpy(out, "UZS1", 4);
    out[4] = 1;
    out[5] = 0;
    put_u64(out + 8, n);
    put_u32(out + 16, chunk);
    put_u32(out + 20, (uint32_t)L.nc);
    put_u64(out + 24, m);
    memcpy(out + 32, exps, 15);
    out[47] = 0;
    put_u64(out + 48, total);
    return ORC_OK;
}

int orc_sentinel_decode(const uint8_t *in, uint64_t in_bytes, uint16_t *x, uint64_t n)
{
    if (in == NULL || (n > 0 && x == NULL)) return ORC_ERR_ARG;
    if (in_bytes < 64) return ORC_ERR_CORRUPT;
    if (memcmp(in, "UZS1", 4) != 0 || get_u16(in + 4) != 1 || get_u16(in + 6) != 0) return ORC_ERR_CORRUPT;
    uint64_t hn = get_u64(in + 8);
    uint32_t chunk = get_u32(in + 16);
    uint64_t nc = get_u32(in + 20);
    uint64_t m = get_u64(in + 24);
    uint64_t total = get_u64(in + 48);
    if (hn != n || !chunk_ok(chunk) || n >= ((uint64_t)1 << 32)) return ORC_ERR_CORRUPT;
    layout_t L = layout_of(n, chunk);
    if (nc != L.nc || m > n || total != L.off_d + m || total > in_bytes) return ORC_ERR_CORRUPT;
    const uint8_t *dec = in + 32;
    const uint8_t *A = in + L.off_a;
    const uint8_t *B = in + L.off_b;
    const uint8_t *C = in + L.off_c;
    const uint8_t *D = in + L.off_d;
    if (get_u32(C) != 0 || get_u32(C + 4 * nc) != m) return ORC_ERR_CORRUPT;
    /* Each chunk on its own: a code 15 takes the chunk's next value. */
    for (uint64_t c = 0; c < nc; c++) {
        uint64_t o = get_u32(C + 4 * c), o1 = get_u32(C + 4 * (c + 1));
        if (o > o1) return ORC_ERR_CORRUPT;
        uint64_t start = c * chunk;
        uint64_t end = start + chunk < n ? start + chunk : n;
        uint64_t next = o;
        for (uint64_t i = start; i < end; i++) {
            uint8_t code = (uint8_t)((B[i / 2] >> (4 * (i % 2))) & 0x0F);
            uint8_t e;
            if (code == 15) {
                if (next >= o1) return ORC_ERR_CORRUPT;
                e = D[next++];
            } else {
                e = dec[code];
            }
            x[i] = rebuild(A[i], e);
        }
        if (next != o1) return ORC_ERR_CORRUPT;
    }
    return ORC_OK;
}
