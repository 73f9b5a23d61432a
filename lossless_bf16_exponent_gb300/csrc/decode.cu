// decode.cu -- SplitZip decoder for sm_103a.
//
// SplitZip review page, §3.2: decoding unpacks each byte into two 4-bit codes,
// looks every code up in the 16-entry decode table, rebuilds the BF16 value
// from the stored sign-mantissa byte, and then a sparse fix-up overwrites the
// exponent of every recorded escape with its exact raw value. §3.4: the dense
// path is the same table lookup for every value (no sentinel test).
//
// Persistent CTAs (header checked and layout derived once per CTA) walk tiles
// of 8192 values; the two stages are fused so each output byte is written
// once:
//   1. every thread issues its dense loads (8 sign-mantissa bytes + one word
//      of eight codes per group of eight values) into registers;
//   2. meanwhile the warps walk the escape blocks of the chunks that overlap
//      the tile and scatter (position -> raw exponent) into a shared-memory
//      bitmap + byte array;
//   3. each group is decoded with the 16-byte decode table held in four
//      registers and selected by byte permutes (three PRMTs per four values),
//      escapes are patched from shared memory, and 16 bytes are stored.
// The header is validated by every CTA before any output is written. The
// rest of a stream is checked as the oracle checks it: offsets that do not
// run from 0 to M or do not rise, and blocks whose positions leave their
// chunk or do not rise strictly, are skipped and reported as corrupt.
#include <algorithm>

#include <atomic>

#include "uzip_internal.cuh"

namespace uzip {
namespace {

// Tile shape (build-time tunables; the defaults are the measured best).
#ifndef UZIP_DEC_THREADS
#define UZIP_DEC_THREADS 256
#endif
#ifndef UZIP_DEC_GROUPS_PER_THREAD
#define UZIP_DEC_GROUPS_PER_THREAD 4
#endif
#ifndef UZIP_DEC_MIN_BLOCKS
#define UZIP_DEC_MIN_BLOCKS 6
#endif
constexpr int kThreads = UZIP_DEC_THREADS;
constexpr int kGroupsPerThread = UZIP_DEC_GROUPS_PER_THREAD;
constexpr uint32_t kTileGroups = kThreads * kGroupsPerThread;
constexpr uint32_t kTile = kTileGroups * 8;  // values per tile

struct Params {
    const uint8_t* s;
    uint64_t stream_bytes;
    uint16_t* out;
    uint64_t n;
    uint32_t* status;
};

// Eight codes (nibbles of a code word) -> eight exponent bytes (e_lo: values
// 0..3, e_hi: values 4..7). The selectors of both halves are formed once for
// the whole word; prmt reads only the low 16 bits of a selector.
__device__ __forceinline__ void lookup8(uint32_t cw, uint32_t d0, uint32_t d1, uint32_t d2, uint32_t d3,
                                        uint32_t& e_lo, uint32_t& e_hi) {
    const uint32_t sel = cw & 0x77777777u;                       // byte of the 8-entry half
    const uint32_t pick = ((cw >> 1) & 0x44444444u) | 0x32103210u;  // half per value
    const uint32_t sel_hi = sel >> 16, pick_hi = pick >> 16;
    e_lo = prmt(prmt(d0, d1, sel), prmt(d2, d3, sel), pick);
    e_hi = prmt(prmt(d0, d1, sel_hi), prmt(d2, d3, sel_hi), pick_hi);
}

// Four flag bits -> four byte masks (bit i set -> byte i = 0xFF): the four
// shifted copies of the multiply never overlap, and bit i lands at 8 i.
__device__ __forceinline__ uint32_t byte_mask4(uint32_t bits4) {
    return ((bits4 * 0x00204081u) & 0x01010101u) * 0xFFu;
}

// Four exponent bytes + four sign-mantissa bytes -> four BF16 values.
__device__ __forceinline__ uint2 rebuild4(uint32_t e4, uint32_t a4) {
    const uint32_t hi = (a4 & 0x80808080u) | ((e4 >> 1) & 0x7F7F7F7Fu);  // sign | exponent bits 7..1
    const uint32_t lo = ((e4 << 7) & 0x80808080u) | (a4 & 0x7F7F7F7Fu);  // exponent bit 0 | mantissa
    return make_uint2(prmt(lo, hi, 0x5140u), prmt(lo, hi, 0x7362u));
}

__device__ __forceinline__ uint32_t ld_u32_le(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// The stream's offsets must run from 0 (offsets[0]) to M (offsets[nc]); that
// they rise is checked chunk by chunk where each block is walked.
__device__ __forceinline__ bool offsets_span_ok(const uint8_t* C, uint64_t nc, uint64_t m) {
    return ld_u32_le(C) == 0 && ld_u32_le(C + 4 * nc) == m;
}

// Escape positions of a chunk's block rise strictly (one entry per escape,
// ascending). Lane l holds entry j0 + l; its predecessor's position comes from
// lane l - 1, or for lane 0 from `last` (entry j0 - 1, the previous step's
// lane 31). Every lane of the warp must call it.
__device__ __forceinline__ uint32_t rising_prev(uint32_t pos, uint32_t last, uint32_t lane) {
    const uint32_t up = __shfl_up_sync(0xffffffffu, pos, 1);
    return lane == 0 ? last : up;
}

__global__ void __launch_bounds__(kThreads, UZIP_DEC_MIN_BLOCKS) decode_kernel(const Params p) {
    static_assert(kGroupsPerThread == 4, "one 32-bit escape word per thread");
    // escape bitmap, double-buffered by tile parity: word w holds the four groups w + r * threads, bit
    // 8 r + i for value i of group r, so each thread reads one word per tile
    __shared__ uint32_t s_mask[2][kThreads];
    __shared__ __align__(16) uint8_t s_val[kTile];
    __shared__ int s_bad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4* h = reinterpret_cast<const uint4*>(p.s);
    const uint4 h0 = h[0], h1 = h[1], h2 = h[2], h3 = h[3];
    const uint64_t hn = (uint64_t)h0.z | ((uint64_t)h0.w << 32);
    const uint32_t chunk = h1.x;
    const uint64_t nc = h1.y;
    const uint64_t m = (uint64_t)h1.z | ((uint64_t)h1.w << 32);
    const uint64_t total = (uint64_t)h3.x | ((uint64_t)h3.y << 32);
    bool ok = h0.x == kStreamMagic && (h0.y & 0xFFFF) == 1 && (h0.y >> 16) == 0 && hn == p.n &&
              chunk_valid(chunk) && m <= hn;
    Layout L;
    if (ok) {
        L = layout_of(hn, chunk);
        ok = nc == L.nc && total == L.off_d + 3 * m && total <= p.stream_bytes;
    }
    if (!ok) {
        if (blockIdx.x == 0 && tid == 0 && p.status) *p.status = UZIP_ERR_CORRUPT;
        return;
    }
    // n < 2^32; sums that can pass n (a tile count, the end of a group or
    // chunk) are taken in 64 bits or relative to the tile.
    const uint32_t n32 = (uint32_t)p.n;
    const uint8_t* A = p.s + L.off_a;
    const uint8_t* B = p.s + L.off_b;
    const uint8_t* C = p.s + L.off_c;
    const uint8_t* D = p.s + L.off_d;
    const uint32_t d0 = h2.x, d1 = h2.y, d2 = h2.z, d3 = h2.w;  // decode table: code k -> byte k
    const uint32_t tiles = (uint32_t)(((uint64_t)n32 + kTile - 1) / kTile);

    s_mask[0][tid] = 0;
    if (tid == 0) s_bad = blockIdx.x == 0 && !offsets_span_ok(C, nc, m);
    __syncthreads();

    int par = 0;
    for (uint32_t t = blockIdx.x; t < tiles; t += gridDim.x, par ^= 1) {
        const uint32_t e0 = t * kTile;
        const uint32_t tlen = min(kTile, n32 - e0);
        const bool full = tlen == kTile;  // uniform: every group whole
        const uint32_t tgroups = (tlen + 7) / 8;
        const uint8_t* At = A + e0 + 8 * tid;
        const uint8_t* Bt = B + e0 / 2 + 4 * tid;

        // 1. dense loads first, so their latency overlaps the escape pass (the
        //    padded sections make whole-group loads safe at the ragged tail).
        uint2 av[kGroupsPerThread];
        uint32_t cv[kGroupsPerThread];
#pragma unroll
        for (int r = 0; r < kGroupsPerThread; r++) {
            if (full || tid + r * kThreads < tgroups) {
                av[r] = ld_stream_v2(At + 8 * r * kThreads);
                cv[r] = ld_stream_u32(Bt + 4 * r * kThreads);
            } else {
                av[r] = make_uint2(0, 0);
                cv[r] = 0;
            }
        }
        // 2. clear the other bitmap for the next tile; scatter this tile's
        //    escapes (chunks overlapping [e0, e0 + tlen)) into this one.
        s_mask[par ^ 1][tid] = 0;
        const uint32_t c_first = e0 / chunk, c_last = (e0 + tlen - 1) / chunk;
        bool bad = false;
        for (uint32_t c = c_first + warp; c <= c_last; c += kThreads / 32) {
            const uint32_t o = ld_u32_le(C + 4ull * c);
            const uint32_t o1 = ld_u32_le(C + 4ull * (c + 1));
            const uint32_t cbase = c * chunk;
            const uint32_t clen = min(chunk, n32 - cbase);
            if (o1 < o || o1 > m || o1 - o > clen) {
                bad = true;
                continue;
            }
            const uint32_t k = o1 - o;
            const uint8_t* blk = D + 3ull * o;
            uint32_t last = 0;  // position of entry j0 - 1 (read only when j0 > 0)
            for (uint32_t j0 = 0; j0 < k; j0 += 32) {  // uniform across the warp
                const uint32_t j = j0 + lane;
                const uint32_t pos = j < k ? (uint32_t)blk[2 * j] | ((uint32_t)blk[2 * j + 1] << 8) : 0u;
                const uint32_t prev = rising_prev(pos, last, lane);
                last = __shfl_sync(0xffffffffu, pos, 31);
                if (j >= k) continue;
                if (pos >= clen || (j > 0 && pos <= prev)) {
                    bad = true;
                    continue;
                }
                const uint32_t el = cbase + pos;
                if (el >= e0 && el < e0 + tlen) {
                    const uint32_t li = el - e0, g = li >> 3;
                    s_val[li] = blk[2 * k + j];
                    atomicOr(&s_mask[par][g % kThreads], 1u << (8 * (g / kThreads) + (li & 7)));
                }
            }
        }
        if (bad) s_bad = 1;
        __syncthreads();

        // 3. decode, patch, store.
        const uint32_t fix_all = s_mask[par][tid];
        uint16_t* out = p.out + e0 + 8 * tid;
#pragma unroll
        for (int r = 0; r < kGroupsPerThread; r++) {
            const uint32_t g = tid + r * kThreads;
            if (!full && g >= tgroups) continue;
            uint32_t e_lo, e_hi;
            lookup8(cv[r], d0, d1, d2, d3, e_lo, e_hi);
            const uint32_t fix = (fix_all >> (8 * r)) & 0xFF;
            if (fix) {  // the group's eight patch bytes at once; only the flagged ones are taken
                const uint2 sv = *reinterpret_cast<const uint2*>(s_val + 8 * g);
                const uint32_t m_lo = byte_mask4(fix & 0xF), m_hi = byte_mask4(fix >> 4);
                e_lo = (e_lo & ~m_lo) | (sv.x & m_lo);
                e_hi = (e_hi & ~m_hi) | (sv.y & m_hi);
            }
            const uint2 lo = rebuild4(e_lo, av[r].x);
            const uint2 hi = rebuild4(e_hi, av[r].y);
            if (full || 8 * g + 8 <= tlen) {
                *reinterpret_cast<uint4*>(out + 8 * r * kThreads) = make_uint4(lo.x, lo.y, hi.x, hi.y);
            } else {
                const uint32_t ge = e0 + 8 * g;
                const uint32_t w[4] = {lo.x, lo.y, hi.x, hi.y};
#pragma unroll
                for (uint32_t i = 0; i < 8; i++)
                    if (8 * g + i < tlen) p.out[ge + i] = (uint16_t)(w[i / 2] >> (16 * (i & 1)));
            }
        }
        __syncthreads();  // s_val and this bitmap are rewritten by the next tile
    }
    if (s_bad && tid == 0 && p.status) *p.status = UZIP_ERR_CORRUPT;
}

// ------------------------------------------------------------ FP8 E5M2

// The low twelve bits of packed 3-bit fields (four values, field i = sign << 2
// | mantissa at bits 3i..3i+2; higher bits ignored) -> four E5M2 bytes without
// their exponents: field i's sign at bit 8i + 7, its mantissa at 8i..8i+1. The
// bits that move by 5 or 15 (signs of fields 0 and 2, mantissas of fields 1
// and 3) take one multiply by 2^5 + 2^15; the bits that move by 0, 10 or 20
// (mantissas of fields 0 and 2, signs of fields 1 and 3) one by 2^0 + 2^10 +
// 2^20. Shifted copies that land on the same bit (only at bits 11 and 21 of
// the second product) carry into bits 12 and 22, which, like every other
// copy, the masks drop (checked for all 4096 field words).
__device__ __forceinline__ uint32_t spread_fields4(uint32_t f12) {
    return (((f12 & 0x71Cu) * 0x8020u) & 0x03800380u) | (((f12 & 0x8E3u) * 0x100401u) & 0x80038003u);
}

// Decoder for FP8 E5M2 streams (page §4.2 / appendix C): tiles of
// 256 * 32 * kE5Slots values, each thread taking kE5Slots slots of 32
// consecutive values (slot s = tid + 256 j: 12 bytes of packed sign-mantissa
// fields and 16 bytes of codes in, 32 bytes out), so a thread has
// 28 * kE5Slots bytes of loads in flight per tile; the escape fix-up goes
// through shared memory as for BF16.
#ifndef UZIP_E5_SLOTS
#define UZIP_E5_SLOTS 2
#endif
constexpr int kE5Slots = UZIP_E5_SLOTS;
constexpr uint32_t kE5Tile = kThreads * 32 * kE5Slots;

__global__ void __launch_bounds__(kThreads, UZIP_DEC_MIN_BLOCKS) decode_e5m2_kernel(const Params p) {
    __shared__ uint32_t s_mask[2][kE5Tile / 32];
    __shared__ __align__(16) uint8_t s_val[kE5Tile];
    __shared__ int s_bad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4* h = reinterpret_cast<const uint4*>(p.s);
    const uint4 h0 = h[0], h1 = h[1], h2 = h[2], h3 = h[3];
    const uint64_t hn = (uint64_t)h0.z | ((uint64_t)h0.w << 32);
    const uint32_t chunk = h1.x;
    const uint64_t nc = h1.y;
    const uint64_t m = (uint64_t)h1.z | ((uint64_t)h1.w << 32);
    const uint64_t total = (uint64_t)h3.x | ((uint64_t)h3.y << 32);
    bool ok = h0.x == kStreamMagicE5 && (h0.y & 0xFFFF) == 1 && (h0.y >> 16) == 0 && hn == p.n &&
              chunk_valid(chunk) && m <= hn;
    Layout L;
    if (ok) {
        L = layout_e5m2_of(hn, chunk);
        ok = nc == L.nc && total == L.off_d + 3 * m && total <= p.stream_bytes;
    }
    if (!ok) {
        if (blockIdx.x == 0 && tid == 0 && p.status) *p.status = UZIP_ERR_CORRUPT;
        return;
    }
    const uint32_t n32 = (uint32_t)p.n;
    const uint8_t* A = p.s + L.off_a;
    const uint8_t* B = p.s + L.off_b;
    const uint8_t* C = p.s + L.off_c;
    const uint8_t* D = p.s + L.off_d;
    uint8_t* out8 = reinterpret_cast<uint8_t*>(p.out);
    // decode table: code k -> its 5-bit exponent already at bits 2..6 of an E5M2 byte
    const uint32_t d0 = (h2.x << 2) & 0x7C7C7C7Cu, d1 = (h2.y << 2) & 0x7C7C7C7Cu;
    const uint32_t d2 = (h2.z << 2) & 0x7C7C7C7Cu, d3 = (h2.w << 2) & 0x7C7C7C7Cu;
    const uint32_t tiles = (uint32_t)(((uint64_t)n32 + kE5Tile - 1) / kE5Tile);

    for (uint32_t i = tid; i < kE5Tile / 32; i += kThreads) s_mask[0][i] = 0;
    if (tid == 0) s_bad = blockIdx.x == 0 && !offsets_span_ok(C, nc, m);
    __syncthreads();

    int par = 0;
    for (uint32_t t = blockIdx.x; t < tiles; t += gridDim.x, par ^= 1) {
        const uint32_t e0 = t * kE5Tile;
        const uint32_t tlen = min(kE5Tile, n32 - e0);
        // 1. dense loads of every slot (the padded sections keep a whole slot inside the stream)
        uint32_t f[kE5Slots][3];
        uint4 cv[kE5Slots];
#pragma unroll
        for (int j = 0; j < kE5Slots; j++) {
            const uint32_t sl = tid + j * kThreads, v0 = 32 * sl;
            f[j][0] = f[j][1] = f[j][2] = 0;
            cv[j] = make_uint4(0, 0, 0, 0);
            if (v0 < tlen) {
                const uint32_t* fa = reinterpret_cast<const uint32_t*>(A + (e0 / 8) * 3 + 12 * sl);
                f[j][0] = __ldg(fa);
                f[j][1] = __ldg(fa + 1);
                f[j][2] = __ldg(fa + 2);
                cv[j] = ld_stream_v4(B + e0 / 2 + 16 * sl);
            }
        }
        // 2. escapes of the chunks overlapping the tile -> shared memory
        for (uint32_t i = tid; i < kE5Tile / 32; i += kThreads) s_mask[par ^ 1][i] = 0;
        const uint32_t c_first = e0 / chunk, c_last = (e0 + tlen - 1) / chunk;
        bool bad = false;
        for (uint32_t c = c_first + warp; c <= c_last; c += kThreads / 32) {
            const uint32_t o = *reinterpret_cast<const uint32_t*>(C + 4ull * c);
            const uint32_t o1 = *reinterpret_cast<const uint32_t*>(C + 4ull * (c + 1));
            const uint32_t cbase = c * chunk;
            const uint32_t clen = min(chunk, n32 - cbase);
            if (o1 < o || o1 > m || o1 - o > clen) {
                bad = true;
                continue;
            }
            const uint32_t k = o1 - o;
            const uint8_t* blk = D + 3ull * o;
            uint32_t last = 0;
            for (uint32_t j0 = 0; j0 < k; j0 += 32) {  // uniform across the warp
                const uint32_t jj = j0 + lane;
                const uint32_t pos = jj < k ? (uint32_t)blk[2 * jj] | ((uint32_t)blk[2 * jj + 1] << 8) : 0u;
                const uint32_t prev = rising_prev(pos, last, lane);
                last = __shfl_sync(0xffffffffu, pos, 31);
                if (jj >= k) continue;
                if (pos >= clen || (jj > 0 && pos <= prev)) {
                    bad = true;
                    continue;
                }
                const uint32_t el = cbase + pos;
                if (el >= e0 && el < e0 + tlen) {
                    const uint32_t li = el - e0;
                    s_val[li] = blk[2 * k + jj];
                    atomicOr(&s_mask[par][li >> 5], 1u << (li & 31));
                }
            }
        }
        if (bad) s_bad = 1;
        __syncthreads();

        // 3. decode each slot's 32 values, patch, store
#pragma unroll
        for (int j = 0; j < kE5Slots; j++) {
            const uint32_t sl = tid + j * kThreads, v0 = 32 * sl;
            if (v0 >= tlen) continue;
            const uint32_t fix = s_mask[par][sl];
            const uint32_t cw[4] = {cv[j].x, cv[j].y, cv[j].z, cv[j].w};
            // the 24 field bits of group q start at bit 0 of g24[q]; bits above
            // 24 are the next group's, which spread_fields4 never reads
            const uint32_t g24[4] = {f[j][0], (f[j][0] >> 24) | (f[j][1] << 8), (f[j][1] >> 16) | (f[j][2] << 16),
                                     f[j][2] >> 8};
            uint32_t o[8];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                uint32_t e8[2];
                lookup8(cw[q], d0, d1, d2, d3, e8[0], e8[1]);
                const uint32_t fq = (fix >> (8 * q)) & 0xFF;
                if (fq) {  // the group's patch bytes at once; only the flagged ones are taken
                    const uint2 sv = *reinterpret_cast<const uint2*>(s_val + v0 + 8 * q);
                    const uint32_t m0 = byte_mask4(fq & 0xF), m1 = byte_mask4(fq >> 4);
                    e8[0] = (e8[0] & ~m0) | ((sv.x << 2) & 0x7C7C7C7Cu & m0);
                    e8[1] = (e8[1] & ~m1) | ((sv.y << 2) & 0x7C7C7C7Cu & m1);
                }
#pragma unroll
                for (int hh = 0; hh < 2; hh++) o[2 * q + hh] = spread_fields4(hh ? g24[q] >> 12 : g24[q]) | e8[hh];
            }
            const uint32_t ge = e0 + v0;
            if (v0 + 32 <= tlen) {
                uint4* dst = reinterpret_cast<uint4*>(out8 + ge);
                dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            } else {
#pragma unroll
                for (uint32_t i = 0; i < 32; i++)
                    if (v0 + i < tlen) out8[ge + i] = (uint8_t)(o[i / 4] >> (8 * (i & 3)));
            }
        }
        __syncthreads();  // s_val and this bitmap are rewritten by the next tile
    }
    if (s_bad && tid == 0 && p.status) *p.status = UZIP_ERR_CORRUPT;
}

// ------------------------------------------------------ Top-15 + sentinel

// Sentinel (code 15) flags of eight codes: bit 4i set when nibble i is 15.
__device__ __forceinline__ uint32_t sentinel_bits(uint32_t w) {
    return w & (w >> 1) & (w >> 2) & (w >> 3) & 0x11111111u;
}

// 16-byte asynchronous global -> shared copy (cp.async) and its wait.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

#ifndef UZIP_SDEC_MIN_BLOCKS
#define UZIP_SDEC_MIN_BLOCKS 4
#endif
#ifndef UZIP_SDEC_WINDOW
#define UZIP_SDEC_WINDOW 256
#endif

// Decoder for the Top-15 + sentinel format (page §3.4, Table 6). No escape
// positions are stored: the k-th code 15 of the stream takes value k of the
// value array (chunk c's values start at offsets[c]), so a tile's escapes are
// one contiguous run of values. Each CTA decodes one contiguous range of
// tiles of 8192 values and carries g0 -- the index of its tile's first
// escape -- from tile to tile; only its first tile derives g0 from the
// offsets (plus, when that tile's chunk began earlier, a count of the
// chunk's earlier code 15s). Groups of eight values as in decode_kernel
// (group g = tid + r * threads: coalesced loads and stores). Per tile
//   1. each thread loads its four groups and the tile's chunk offsets;
//   2. code-15 counts of the four group rows, packed two per word, are
//      scanned within each warp (shuffles); one barrier publishes the warp
//      totals, giving every thread the code 15s before each of its groups;
//   3. the next tile's run of values (a window of UZIP_SDEC_WINDOW bytes
//      from its g0) is requested with cp.async, so a tile's patch reads
//      shared memory (values past the window are read from global memory);
//   4. lookup, patch, rebuild, 16-byte stores.
// Shared buffers are double-buffered by tile parity: one barrier per tile.
// Checks, the oracle's: the header; offsets[0] = 0, offsets[nc] = M; every
// chunk holds as many code 15s as its offsets give values (checked in the
// tile where the chunk ends: its end offset must equal g0 + the code 15s
// before it), so a stream is refused exactly when the oracle refuses it.
// Every value index is checked against M before the read.
__global__ void __launch_bounds__(kThreads, UZIP_SDEC_MIN_BLOCKS) decode_sentinel_kernel(const Params p) {
    constexpr int kWarps = kThreads / 32;
    constexpr uint32_t kMaxOffs = kTile / UZIP_MIN_CHUNK + 2;  // offsets a tile can need
    constexpr uint32_t kWin = UZIP_SDEC_WINDOW + 16;           // window bytes from g0 rounded down to 16
    static_assert(kGroupsPerThread == 4, "two packed rows of two 16-bit counts");
    static_assert(kWin / 16 <= kThreads, "one 16-byte copy per thread");
    __shared__ uint32_t s_pre[2][2][kThreads];  // per thread: rows (0,1) and (2,3) of code 15s of earlier lanes
    __shared__ uint32_t s_wt[2][2][kWarps];     // per warp: the same, totals
    __shared__ uint32_t s_off[2][kMaxOffs];     // offsets[c_first ..]
    __shared__ __align__(16) uint8_t s_win[2][kWin];
    __shared__ uint32_t s_red[kWarps];
    __shared__ int s_bad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4* h = reinterpret_cast<const uint4*>(p.s);
    const uint4 h0 = h[0], h1 = h[1], h2 = h[2], h3 = h[3];
    const uint64_t hn = (uint64_t)h0.z | ((uint64_t)h0.w << 32);
    const uint32_t chunk = h1.x;
    const uint64_t nc = h1.y;
    const uint64_t m = (uint64_t)h1.z | ((uint64_t)h1.w << 32);
    const uint64_t total = (uint64_t)h3.x | ((uint64_t)h3.y << 32);
    bool ok = h0.x == kStreamMagicS && (h0.y & 0xFFFF) == 1 && (h0.y >> 16) == 0 && hn == p.n &&
              chunk_valid(chunk) && m <= hn;
    Layout L;
    if (ok) {
        L = layout_of(hn, chunk);
        ok = nc == L.nc && total == L.off_d + m && total <= p.stream_bytes;
    }
    if (!ok) {
        if (blockIdx.x == 0 && tid == 0 && p.status) *p.status = UZIP_ERR_CORRUPT;
        return;
    }
    const uint32_t n32 = (uint32_t)p.n;
    const uint32_t m32 = (uint32_t)m;
    const uint8_t* A = p.s + L.off_a;
    const uint8_t* B = p.s + L.off_b;
    const uint32_t* Cw = reinterpret_cast<const uint32_t*>(p.s + L.off_c);
    const uint8_t* D = p.s + L.off_d;
    const uint64_t d_room = p.stream_bytes - L.off_d;  // readable bytes from D on
    const uint32_t d0 = h2.x, d1 = h2.y, d2 = h2.z, d3 = h2.w;
    const uint32_t tiles = (uint32_t)(((uint64_t)n32 + kTile - 1) / kTile);
    const uint32_t t_begin = (uint32_t)((uint64_t)tiles * blockIdx.x / gridDim.x);
    const uint32_t t_end = (uint32_t)((uint64_t)tiles * (blockIdx.x + 1) / gridDim.x);
    if (tid == 0) s_bad = 0;
    if (t_begin >= t_end) return;  // uniform per CTA; no barrier has been passed

    // the window of values [w0, w0 + kWin) from index g into s_win[b] (16-byte copies inside the buffer)
    auto request_window = [&](uint32_t g, int b) {
        const uint64_t w0 = g & ~15u;
        if (tid < (int)(kWin / 16) && w0 + 16 * (tid + 1) <= d_room) cp_async16(&s_win[b][16 * tid], D + w0 + 16 * tid);
    };

    // g0 of the first tile: offsets[c_first] + the code 15s of chunk c_first before the tile
    uint32_t g0;
    {
        const uint32_t e0 = t_begin * kTile, c_first = e0 / chunk;
        uint32_t e = 0;
        for (uint32_t w = c_first * chunk / 8 + tid; w < e0 / 8; w += kThreads)
            e += __popc(sentinel_bits(__ldg(reinterpret_cast<const uint32_t*>(B) + w)));
        e = __reduce_add_sync(0xffffffffu, e);
        if (lane == 0) s_red[warp] = e;
        __syncthreads();
        g0 = __ldg(Cw + c_first);
#pragma unroll
        for (int w = 0; w < kWarps; w++) g0 += s_red[w];
        request_window(g0, 0);
    }

    int par = 0;
    for (uint32_t t = t_begin; t < t_end; t++, par ^= 1) {
        const uint32_t e0 = t * kTile;
        const uint32_t tlen = min(kTile, n32 - e0);
        const uint32_t tgroups = (tlen + 7) / 8;
        const uint32_t c_first = e0 / chunk, c_last = (e0 + tlen - 1) / chunk;

        // 1. loads (the padded sections make whole-group loads safe at the ragged tail)
        uint2 av[kGroupsPerThread];
        uint32_t cv[kGroupsPerThread];
#pragma unroll
        for (int r = 0; r < kGroupsPerThread; r++) {
            const uint32_t g = tid + r * kThreads;
            av[r] = make_uint2(0, 0);
            cv[r] = 0;
            if (g < tgroups) {
                av[r] = ld_stream_v2(A + e0 + 8 * g);
                cv[r] = ld_stream_u32(B + e0 / 2 + 4 * g);
            }
        }
        for (uint32_t k = tid; k <= c_last - c_first + 1; k += kThreads) s_off[par][k] = __ldg(Cw + c_first + k);

        // 2. counts, warp scans, one barrier
        uint32_t sb[kGroupsPerThread];
        uint32_t p01 = 0, p23 = 0;
#pragma unroll
        for (int r = 0; r < kGroupsPerThread; r++) {
            const uint32_t g = tid + r * kThreads;
            sb[r] = sentinel_bits(cv[r]);
            if (8 * g + 8 > tlen) sb[r] &= 8 * g < tlen ? (1u << (4 * (tlen - 8 * g))) - 1 : 0u;  // padding past n
            const uint32_t c = __popc(sb[r]) << (16 * (r & 1));
            if (r < 2) p01 += c;
            else p23 += c;
        }
        uint32_t i01 = p01, i23 = p23;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v01 = __shfl_up_sync(0xffffffffu, i01, o);
            const uint32_t v23 = __shfl_up_sync(0xffffffffu, i23, o);
            if (lane >= o) {
                i01 += v01;
                i23 += v23;
            }
        }
        s_pre[par][0][tid] = i01 - p01;
        s_pre[par][1][tid] = i23 - p23;
        if (lane == 31) {
            s_wt[par][0][warp] = i01;
            s_wt[par][1][warp] = i23;
        }
        cp_async_wait_all();  // this tile's window
        __syncthreads();

        uint32_t w01 = 0, w23 = 0, t01 = 0, t23 = 0;
#pragma unroll
        for (int w = 0; w < kWarps; w++) {
            const uint32_t x01 = s_wt[par][0][w], x23 = s_wt[par][1][w];
            if (w < warp) {
                w01 += x01;
                w23 += x23;
            }
            t01 += x01;
            t23 += x23;
        }
        // code 15s before each group row, in element order
        const uint32_t row1 = t01 & 0xFFFF, row2 = row1 + (t01 >> 16), row3 = row2 + (t23 & 0xFFFF);
        const uint32_t tile_total = row3 + (t23 >> 16);

        // 3. the next tile's window
        if (t + 1 < t_end) request_window(g0 + tile_total, par ^ 1);

        // code 15s of the tile before value f (f a multiple of 8, or f = tlen)
        auto before = [&](uint32_t f) {
            if (f >= tlen) return tile_total;
            const uint32_t G = f / 8, r = G / kThreads, tt = G % kThreads, ww = tt / 32;
            uint32_t x = s_pre[par][r >> 1][tt];
            for (uint32_t k = 0; k < ww; k++) x += s_wt[par][r >> 1][k];
            const uint32_t base = r == 0 ? 0u : r == 1 ? row1 : r == 2 ? row2 : row3;
            return base + ((x >> (16 * (r & 1))) & 0xFFFF);
        };
        // every chunk ending in the tile: its end offset against the code 15s before it
        for (uint32_t k = tid; k <= c_last - c_first; k += kThreads) {
            const uint32_t c = c_first + k;
            const uint32_t ce = (uint32_t)min((uint64_t)(c + 1) * chunk, (uint64_t)n32);
            const uint32_t o1 = s_off[par][k + 1];
            if (ce <= e0 + tlen && g0 + before(ce - e0) != o1) s_bad = 1;
            if ((c == 0 && s_off[par][k] != 0) || (c + 1 == nc && o1 != m32)) s_bad = 1;
        }

        // 4. decode, patch, store
        const uint32_t own01 = w01 + s_pre[par][0][tid], own23 = w23 + s_pre[par][1][tid];
        const uint32_t wbase = g0 & ~15u;
#pragma unroll
        for (int r = 0; r < kGroupsPerThread; r++) {
            const uint32_t g = tid + r * kThreads;
            if (g >= tgroups) continue;
            uint32_t e_lo, e_hi;
            lookup8(cv[r], d0, d1, d2, d3, e_lo, e_hi);
            uint32_t bits = sb[r];
            if (bits) {
                const uint32_t own = r == 0 ? (own01 & 0xFFFF) : r == 1 ? (own01 >> 16) + row1
                                   : r == 2 ? (own23 & 0xFFFF) + row2 : (own23 >> 16) + row3;
                uint32_t idx = g0 + own;
                do {
                    const uint32_t i = (__ffs(bits) - 1) / 4;  // value i of the group
                    bits &= bits - 1;
                    uint32_t ev = 0;
                    const uint32_t wo = idx - wbase;
                    if (idx >= m32) s_bad = 1;
                    else if (wo < kWin && wbase + 16 * (wo / 16 + 1) <= d_room) ev = s_win[par][wo];
                    else ev = D[idx];
                    idx++;
                    const uint32_t sh = 8 * (i & 3);
                    if (i < 4) e_lo = (e_lo & ~(0xFFu << sh)) | (ev << sh);
                    else e_hi = (e_hi & ~(0xFFu << sh)) | (ev << sh);
                } while (bits);
            }
            const uint2 lo = rebuild4(e_lo, av[r].x);
            const uint2 hi = rebuild4(e_hi, av[r].y);
            const uint32_t ge = e0 + 8 * g;
            if (8 * g + 8 <= tlen) {
                *reinterpret_cast<uint4*>(p.out + ge) = make_uint4(lo.x, lo.y, hi.x, hi.y);
            } else {
                const uint32_t wv[4] = {lo.x, lo.y, hi.x, hi.y};
#pragma unroll
                for (uint32_t i = 0; i < 8; i++)
                    if (8 * g + i < tlen) p.out[ge + i] = (uint16_t)(wv[i / 2] >> (16 * (i & 1)));
            }
        }
        g0 += tile_total;
    }
    cp_async_wait_all();
    __syncthreads();  // every thread's s_bad write before it is read
    if (s_bad && tid == 0 && p.status) *p.status = UZIP_ERR_CORRUPT;
}

}  // namespace
}  // namespace uzip

using namespace uzip;

namespace {

// SM count and each decoder's residency per device, looked up on the first
// call on that device (0 = not yet).
constexpr int kMaxCachedDevices = 64;
std::atomic<int> g_sms[kMaxCachedDevices];
std::atomic<int> g_per_sm[kMaxCachedDevices][3];

int decode_launch(void (*kernel)(Params), int slot, const void* d_stream, size_t stream_bytes, void* d_out,
                  size_t n, uint32_t* d_status, uzip_stream_t stream, uint32_t tile = kTile) {
    if (!d_stream || (n > 0 && !d_out) || n > UZIP_MAX_N) return UZIP_ERR_ARG;
    if (!aligned16(d_stream) || (n > 0 && !aligned16(d_out)) ||
        (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3)))
        return UZIP_ERR_ALIGN;
    if (stream_bytes < UZIP_HEADER_BYTES) return UZIP_ERR_CAPACITY;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (d_status) UZIP_CUDA_TRY(cudaMemsetAsync(d_status, 0, sizeof(uint32_t), s));
    Params p;
    p.s = static_cast<const uint8_t*>(d_stream);
    p.stream_bytes = stream_bytes;
    p.out = static_cast<uint16_t*>(d_out);
    p.n = n;
    p.status = d_status;
    int dev = 0;
    UZIP_CUDA_TRY(cudaGetDevice(&dev));
    const bool cached = dev < kMaxCachedDevices;
    int sms = cached ? g_sms[dev].load() : 0, per_sm = cached ? g_per_sm[dev][slot].load() : 0;
    if (sms < 1) {
        UZIP_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        if (cached) g_sms[dev].store(sms);
    }
    if (per_sm < 1) {
        UZIP_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0));
        if (per_sm < 1) return UZIP_ERR_CUDA;
        if (cached) g_per_sm[dev][slot].store(per_sm);
    }
    const uint64_t tiles = (n + tile - 1) / tile;
    const uint64_t grid = std::max<uint64_t>(1, std::min<uint64_t>(tiles, (uint64_t)sms * per_sm));
    kernel<<<(unsigned)grid, kThreads, 0, s>>>(p);
    UZIP_CUDA_TRY(cudaGetLastError());
    return UZIP_OK;
}

}  // namespace

extern "C" UZIP_API int uzip_decode(const void* d_stream, size_t stream_bytes, void* d_out_bf16, size_t n,
                                    uint32_t* d_status, uzip_stream_t stream) {
    return decode_launch(decode_kernel, 0, d_stream, stream_bytes, d_out_bf16, n, d_status, stream);
}

extern "C" UZIP_API int uzip_sentinel_decode(const void* d_stream, size_t stream_bytes, void* d_out_bf16, size_t n,
                                             uint32_t* d_status, uzip_stream_t stream) {
    return decode_launch(decode_sentinel_kernel, 1, d_stream, stream_bytes, d_out_bf16, n, d_status, stream);
}

extern "C" UZIP_API int uzip_e5m2_decode(const void* d_stream, size_t stream_bytes, void* d_out_e5m2, size_t n,
                                         uint32_t* d_status, uzip_stream_t stream) {
    return decode_launch(decode_e5m2_kernel, 2, d_stream, stream_bytes, d_out_e5m2, n, d_status, stream, kE5Tile);
}
