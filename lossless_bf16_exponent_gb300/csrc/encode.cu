// encode.cu -- SplitZip encoder for sm_103a: one pass over the input (a one-block
// clear of the segment totals, a dense kernel, an escape kernel; short inputs
// in one launch).
//
// SplitZip review page, §3.2: encoding is (1) a dense transform -- split each
// BF16 value into its exponent and sign-mantissa byte, store the latter
// verbatim, map the exponent through the Top-16 code table and pack two 4-bit
// codes per byte -- and (2) a scan of the exponent stream that pushes every
// exponent outside the Top-16 into chunked escape position / value arrays.
// Appendix A (Quad64): the dense work is fused into one pass over wide words;
// here each thread moves 16-byte vectors (eight values).
//
// The only serial dependency is the escape prefix (where each chunk's escape
// block starts), which a single-pass decoupled look-back resolves through a
// chain of inclusive prefixes; on GB300 that chain, not HBM, set the pace
// (one window of predecessors per loaded-L2 round trip). So the prefix is
// resolved by the kernel boundary instead:
//   dense kernel   warps take units of 2048 values in grid-stride order (all
//                  warps stream one compact window of the input, which keeps
//                  HBM rows open; contiguous per-warp spans measured 8 % slower):
//                  16-byte loads -> exponent and sign-mantissa bytes with byte
//                  permutes -> code + escape bit from a 256-byte shared table ->
//                  coalesced 8-byte sign-mantissa and 4-byte code stores. Its
//                  escapes go, in ascending order, into the unit's list of up to
//                  kListCap (position, exponent) entries in the workspace; a
//                  unit with more escapes stores its escape-mask bytes instead.
//                  It stores the unit's escape count and adds it to its
//                  segment's total (64 or more units per segment; the totals
//                  are zeroed by a one-block kernel launched just before,
//                  behind which the dense kernel launches at once and which
//                  it waits for only before its first total update).
//   escape kernel  launched as a programmatic dependent of the dense kernel (its
//                  launch overlaps the dense tail; it waits for the dense
//                  results before touching them). Each warp takes a range of
//                  whole chunks (up to 32 units, one per lane), adds the
//                  segment and unit totals before it into the range's first
//                  escape rank, writes the chunk offsets and then each escape's
//                  chunk-relative position and raw exponent in ascending
//                  element order, bounds-checked against out_capacity. The warp
//                  that owns the last range writes the tail and the header.
// The input is read from HBM once; the escape lists cost about 4 bytes per
// escape written and read. FP8 E5M2 input (page §4.2) has its own dense
// kernel (one lookup per exponent pair, 32 values per lane and step) and
// shares the escape kernel. Short inputs take one launch instead: up to 32
// units one CTA (encode_small_kernel), up to 256 units one thread-block
// cluster of up to 16 CTAs that meet through distributed shared memory
// (encode_cluster_kernel); both keep the escape lists in shared memory and
// use no workspace.
#include <algorithm>
#include <atomic>

#include "uzip_internal.cuh"

namespace uzip {
namespace {

constexpr uint32_t kUnit = 2048;              // values per counting unit (one warp)
constexpr uint32_t kUnitGroups = kUnit / 8;   // its mask bytes
constexpr int kThreads = 256;                 // both kernels
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kMaxSegments = 2048;       // segment totals (a block sums up to all of them)
constexpr uint32_t kListCap = 64;             // escape entries a unit keeps in its list
constexpr uint32_t kHeadEntries = 32;         // list entries a unit keeps in shared memory during the escape pass
static_assert(kHeadEntries == 32, "head_slot: eight 16-byte chunks per lane row");
constexpr uint32_t kMaxRangeUnits = 31;       // a range covers at most 31 units of values (32 overlapped)
constexpr uint32_t kStageBytes = 2560;        // per-warp staging of a range's escape blocks (853 escapes)
constexpr uint32_t kMaxRangeChunks = 256;     // bounds the per-warp chunk table
constexpr int kBatch = 4;                     // escape exponents re-read at once (mask units)
constexpr uint32_t kParallelAbove = 32;       // pass 2 goes escape-parallel when a unit has more escapes
                                              // (below, one lane per unit walking its list measured faster)
#ifndef UZIP_ENC_MIN_BLOCKS
#define UZIP_ENC_MIN_BLOCKS 4
#endif
#ifndef UZIP_ENC_E5_MIN_BLOCKS
#define UZIP_ENC_E5_MIN_BLOCKS 5  // E5M2 is issue-bound: 48 registers, a fifth CTA per SM
#endif
#ifndef UZIP_ENC_ITER_UNROLL
#define UZIP_ENC_ITER_UNROLL 2
#endif
#ifndef UZIP_ESC_MIN_BLOCKS
#define UZIP_ESC_MIN_BLOCKS 4
#endif
constexpr int kIterUnroll = UZIP_ENC_ITER_UNROLL;  // 2: both 4-load batches of a unit in flight per lane

// Workspace layout, a function of n only: segment totals (cleared by each
// call) | unit counts | unit lists | unit mask bytes. Every other word the
// escape kernel reads is written by the dense kernel of the same call.
struct Geometry {
    uint64_t units;      // counting units of kUnit values
    uint32_t seg_units;  // units per segment (power of two, >= 64)
    uint32_t nseg;       // segments
    uint64_t off_segs, off_counts, off_lists, off_masks, bytes;
};

__host__ __device__ constexpr uint64_t pad16c(uint64_t v) { return (v + 15) / 16 * 16; }

__host__ __device__ constexpr Geometry geometry_of(uint64_t n) {
    Geometry g{};
    g.units = (n + kUnit - 1) / kUnit;
    g.seg_units = 64;
    while ((g.units + g.seg_units - 1) / g.seg_units > kMaxSegments) g.seg_units *= 2;
    g.nseg = (uint32_t)((g.units + g.seg_units - 1) / g.seg_units);
    g.off_segs = 0;
    g.off_counts = g.off_segs + pad16c(4ull * g.nseg);
    g.off_lists = g.off_counts + pad16c(4ull * g.units);
    g.off_masks = g.off_lists + 4ull * kListCap * g.units;
    g.bytes = g.off_masks + (uint64_t)kUnitGroups * g.units;
    return g;
}

struct Params {
    const uint16_t* in;   // BF16 input
    const uint8_t* in8;   // FP8 E5M2 input
    uint32_t fmt;         // kBF16 or kE5M2
    uint64_t a_bytes;     // bytes of the sign-mantissa section (before its padding)
    uint64_t n;
    uint32_t chunk;
    uint32_t seg_units;   // units per segment
    uint32_t seg_shift;   // log2(seg_units)
    uint32_t nseg;        // segments
    uint32_t range_chunks;
    uint32_t chunk_shift;  // log2(chunk) when chunk is a power of two, else 32
    uint64_t units;
    uint64_t ranges;
    const uint8_t* cb;
    uint8_t* out;
    uint64_t cap;
    Layout L;
    uint32_t* segs;    // escapes per segment
    uint32_t* counts;  // escapes per unit
    uint32_t* lists;   // kListCap entries per unit: position | exponent << 16
    uint8_t* masks;    // kUnitGroups bytes per unit, written only when a unit overflows its list
};

// Programmatic dependent launch (PTX griddepcontrol): the dense kernel lets
// the escape kernel be scheduled early; the escape kernel waits until the
// dense grid has completed and its writes are visible.
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_for_prerequisite() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Eight values -> 8 sign-mantissa bytes (a_lo, a_hi), 8 packed codes (one
// word, value i in nibble i), the escape flags (bit 7 of byte i of esc_lo /
// esc_hi for value i / i + 4) and the 8 exponents.
__device__ __forceinline__ void encode_group(const uint4 v, const uint8_t* tab, uint32_t& a_lo,
                                             uint32_t& a_hi, uint32_t& codes, uint32_t& esc_lo, uint32_t& esc_hi,
                                             uint32_t& e_lo, uint32_t& e_hi) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed[2], esc[2], am[2], ex[2];
#pragma unroll
    for (int h = 0; h < 2; h++) {
        // Bytes of four values: high bytes (sign + exponent bits 7..1) and
        // low bytes (exponent bit 0 + mantissa).
        const uint32_t hi = prmt(w[2 * h], w[2 * h + 1], 0x7531);
        const uint32_t lo = prmt(w[2 * h], w[2 * h + 1], 0x6420);
        const uint32_t e4 = ((hi << 1) & 0xFEFEFEFEu) | ((lo >> 7) & 0x01010101u);
        am[h] = (hi & 0x80808080u) | (lo & 0x7F7F7F7Fu);
        ex[h] = e4;
        // Table byte = code | escape << 7.
        const uint32_t t0 = tab[e4 & 0xFF];
        const uint32_t t1 = tab[prmt(e4, 0, 0x4441)];
        const uint32_t t2 = tab[prmt(e4, 0, 0x4442)];
        const uint32_t t3 = tab[e4 >> 24];
        const uint32_t t4 = prmt(prmt(t0, t1, 0x0040), prmt(t2, t3, 0x0040), 0x5410);
        const uint32_t c = t4 & 0x0F0F0F0Fu;
        packed[h] = c | (c >> 4);  // byte 0 = c0 | c1 << 4, byte 2 = c2 | c3 << 4
        esc[h] = t4 & 0x80808080u;
    }
    a_lo = am[0];
    a_hi = am[1];
    e_lo = ex[0];
    e_hi = ex[1];
    esc_lo = esc[0];
    esc_hi = esc[1];
    codes = prmt(packed[0], packed[1], 0x6420);
}

// Escape flags (bit 7 of each byte) -> 8-bit mask, value i at bit i (the four
// shifted copies of the multiply never overlap).
__device__ __forceinline__ uint32_t escape_mask(uint32_t esc_lo, uint32_t esc_hi) {
    const uint32_t m_lo = (((esc_lo >> 7) * 0x204081u) >> 21) & 0xF;
    const uint32_t m_hi = (((esc_hi >> 7) * 0x204081u) >> 21) & 0xF;
    return m_lo | (m_hi << 4);
}

// Stream bytes for m escapes: 3 per escape (position + value), 1 for the
// sentinel format (value only).
__device__ __forceinline__ uint64_t stream_total(const Params& p, uint64_t m) {
    return p.L.off_d + (p.fmt == kSentinel ? m : 3 * m);
}

__device__ void write_header(const Params& p, uint64_t m, uint32_t flags) {
    uint4* h = reinterpret_cast<uint4*>(p.out);
    const uint64_t total = stream_total(p, m);
    uint4 exps = *reinterpret_cast<const uint4*>(p.cb + UZIP_CB_EXPS);
    if (p.fmt == kSentinel) exps.w &= 0x00FFFFFFu;  // only 15 exponents have codes
    const uint32_t magic = p.fmt == kE5M2 ? kStreamMagicE5 : p.fmt == kSentinel ? kStreamMagicS : kStreamMagic;
    h[0] = make_uint4(magic, 1u | (flags << 16), (uint32_t)p.n, (uint32_t)(p.n >> 32));
    h[1] = make_uint4(p.chunk, (uint32_t)p.L.nc, (uint32_t)m, (uint32_t)(m >> 32));
    h[2] = exps;
    h[3] = make_uint4((uint32_t)total, (uint32_t)(total >> 32), 0u, 0u);
}

// Zero bytes [from, to) of the stream, byte by byte (a few padding bytes).
__device__ void zero_bytes(uint8_t* out, uint64_t from, uint64_t to) {
    for (uint64_t o = from; o < to; o++) out[o] = 0;
}

// Zero bytes [from, to) of the stream, 4-byte aligned bounds.
__device__ void zero_words(uint8_t* out, uint64_t from, uint64_t to) {
    for (uint64_t o = from; o < to; o += 4) *reinterpret_cast<uint32_t*>(out + o) = 0;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) { return __reduce_add_sync(0xffffffffu, v); }

// Shared-memory slot of list entry j (< kHeadEntries) of lane L's unit (round
// rr): each lane owns a 128-byte row of eight 16-byte chunks, chunk c stored
// at c ^ (L & 7) so that lanes reading the same entry spread over the banks;
// for j < 32 that is entry j ^ ((L & 7) << 2) of the row.
__device__ __forceinline__ uint32_t head_slot(int rr, uint32_t L, uint32_t j) {
    return (uint32_t)rr * (kHeadEntries * 32) + L * kHeadEntries + (j ^ ((L & 7) << 2));
}

// 16-byte asynchronous global -> shared copy (cp.async) and its wait.
__device__ __forceinline__ void cp_async16(uint32_t* dst, const uint32_t* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// x / chunk (a shift for the power-of-two chunk sizes).
__device__ __forceinline__ uint32_t div_chunk(const Params& p, uint32_t x) {
    return p.chunk_shift < 32 ? x >> p.chunk_shift : x / p.chunk;
}

// Zero the segment totals. Its dependent (the dense kernel) may start at
// once: it waits for this grid only before its first total update.
__global__ void __launch_bounds__(256) clear_segments_kernel(uint32_t* segs, uint32_t words) {
    allow_dependent_launch();
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < words; i += gridDim.x * blockDim.x) segs[i] = 0;
}

// Stores of an E5M2 unit's escape list and mask words: to the global
// workspace with an L2 evict-last policy (the escape kernel reads them back),
// or, for the one-CTA encoder of short inputs, to shared memory.
template <bool kSmem>
__device__ __forceinline__ void put_u32(uint32_t* q, uint32_t v, uint64_t keep) {
    if (kSmem) *q = v;
    else st_u32_keep(q, v, keep);
}

// ------------------------------------------------------------ dense kernel

// The short-input encoders' unit of kUnit values, by the whole warp:
// sign-mantissa bytes and packed codes to the stream; the unit's escapes,
// ascending, to `list` (its row of the CTA's shared lists: up to kListCap
// (position, exponent) entries), or, past kListCap of them, its escape-mask
// bytes to `masks` (its row of the shared masks). Each row holding an escape ranks its
// escapes at once (the grid encoder's dense_unit_bf16 defers the ranking to
// the unit's end, which needs 2.3 KB of shared memory per warp). Returns the
// unit's escape count (the same in every lane).
__device__ __forceinline__ uint32_t dense_unit_bf16_shared(const Params& p, uint64_t u, const uint8_t* s_tab,
                                                           uint32_t* list, uint8_t* masks) {
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t ubase = u * kUnit;
    const uint32_t ulen = (uint32_t)min((uint64_t)kUnit, p.n - ubase);
    const uint4* src = reinterpret_cast<const uint4*>(p.in + ubase);
    uint8_t* dst_a = p.out + p.L.off_a + ubase;
    uint8_t* dst_b = p.out + p.L.off_b + ubase / 2;
    const bool full = ulen == kUnit;  // every unit but the tensor's last
    uint32_t cnt = 0;                 // escapes so far in this unit (uniform across the warp)
    uint32_t mbytes[2] = {0, 0};      // this lane's 8 mask bytes, in case the list overflows
#pragma unroll kIterUnroll
    for (int it = 0; it < 2; it++) {
        uint4 v[4];
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const uint32_t g = it * 128 + r * 32 + lane;
            v[r] = make_uint4(0, 0, 0, 0);
            if (full || 8 * g + 8 <= ulen) {
                v[r] = ld_stream_v4(src + g);
            } else if (8 * g < ulen) {  // ragged tail of the tensor (< 8 values)
                uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
                for (uint32_t i = 0; i < 8; i++)
                    if (8 * g + i < ulen) w[i / 2] |= (uint32_t)p.in[ubase + 8 * g + i] << (16 * (i & 1));
                v[r] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const uint32_t g = it * 128 + r * 32 + lane;
            uint32_t esc_lo = 0, esc_hi = 0, e_lo = 0, e_hi = 0;
            if (full || 8 * g < ulen) {
                uint32_t a_lo, a_hi, codes;
                encode_group(v[r], s_tab, a_lo, a_hi, codes, esc_lo, esc_hi, e_lo, e_hi);
                if (!full && 8 * g + 8 > ulen) {  // codes and escapes of real values only
                    const uint32_t valid = ulen - 8 * g;
                    const uint64_t live = (1ull << (8 * valid)) - 1;
                    esc_lo &= (uint32_t)live;
                    esc_hi &= (uint32_t)(live >> 32);
                    codes &= (1u << (4 * valid)) - 1;
                }
                *reinterpret_cast<uint2*>(dst_a + 8 * g) = make_uint2(a_lo, a_hi);
                *reinterpret_cast<uint32_t*>(dst_b + 4 * g) = codes;
            }
            // Escapes are rare: the mask and the ranking run only for rows
            // holding one. Groups g = it*128 + r*32 + lane come in
            // ascending order per (it, r) row, so a warp scan ranks the
            // row's escapes (the whole warp takes part).
            if (__any_sync(0xffffffffu, (esc_lo | esc_hi) != 0)) {
                const uint32_t mask = escape_mask(esc_lo, esc_hi);
                const uint32_t c = __popc(mask);
                uint32_t excl, total;
                if (!__any_sync(0xffffffffu, c > 1)) {  // sparse row: one ballot ranks it
                    const uint32_t b = __ballot_sync(0xffffffffu, c != 0);
                    excl = __popc(b & ((1u << lane) - 1));
                    total = __popc(b);
                } else {
                    uint32_t incl = c;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += t;
                    }
                    excl = incl - c;
                    total = __shfl_sync(0xffffffffu, incl, 31);
                }
                uint32_t j = cnt + excl;
                for (uint32_t bits = mask; bits; bits &= bits - 1, j++) {
                    const uint32_t b = __ffs(bits) - 1;
                    const uint32_t e = ((b < 4 ? e_lo : e_hi) >> (8 * (b & 3))) & 0xFF;
                    if (j < kListCap) list[j] = (8 * g + b) | (e << 16);
                }
                cnt += total;
                mbytes[it] |= mask << (8 * r);
            }
        }
    }
    if (cnt > kListCap) {  // the list overflowed: keep the masks instead
#pragma unroll
        for (int it = 0; it < 2; it++)
#pragma unroll
            for (int r = 0; r < 4; r++)
                masks[it * 128 + r * 32 + lane] = (uint8_t)(mbytes[it] >> (8 * r));
    }
    return cnt;
}

// The grid encoder's unit: as dense_unit_bf16_shared, but the list or mask
// words go to the workspace (row u, L2 evict-last policy `keep`), and rows
// holding an escape only note it (the row's escape-mask bytes, and the
// exponent bytes of the groups that escape) in the warp's shared memory
// s_flag / s_exb; the unit's escapes are ranked once, at its end, by one warp
// scan. Lane l then owns positions
// 64 l .. 64 l + 63 (groups 8 l .. 8 l + 7, all in row l / 4) and writes their
// list entries in position order. On escape-heavy inputs this replaces up to
// eight per-row scans and lane loops with one; the flags double as the mask
// bytes when the list overflows.
__device__ __forceinline__ uint32_t dense_unit_bf16(const Params& p, uint64_t u, const uint8_t* s_tab,
                                                    uint8_t* s_flag, uint8_t* s_exb, uint64_t keep) {
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t ubase = u * kUnit;
    const uint32_t ulen = (uint32_t)min((uint64_t)kUnit, p.n - ubase);
    const uint4* src = reinterpret_cast<const uint4*>(p.in + ubase);
    uint8_t* dst_a = p.out + p.L.off_a + ubase;
    uint8_t* dst_b = p.out + p.L.off_b + ubase / 2;
    const bool full = ulen == kUnit;
    uint32_t rows = 0;  // bit it * 4 + r: row (it, r), groups it*128 + r*32 + 0..31, holds an escape
#pragma unroll kIterUnroll
    for (int it = 0; it < 2; it++) {
        uint4 v[4];
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const uint32_t g = it * 128 + r * 32 + lane;
            v[r] = make_uint4(0, 0, 0, 0);
            if (full || 8 * g + 8 <= ulen) {
                v[r] = ld_stream_v4(src + g);
            } else if (8 * g < ulen) {  // ragged tail of the tensor (< 8 values)
                uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
                for (uint32_t i = 0; i < 8; i++)
                    if (8 * g + i < ulen) w[i / 2] |= (uint32_t)p.in[ubase + 8 * g + i] << (16 * (i & 1));
                v[r] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const uint32_t g = it * 128 + r * 32 + lane;
            uint32_t esc_lo = 0, esc_hi = 0, e_lo = 0, e_hi = 0;
            if (full || 8 * g < ulen) {
                uint32_t a_lo, a_hi, codes;
                encode_group(v[r], s_tab, a_lo, a_hi, codes, esc_lo, esc_hi, e_lo, e_hi);
                if (!full && 8 * g + 8 > ulen) {  // codes and escapes of real values only
                    const uint32_t valid = ulen - 8 * g;
                    const uint64_t live = (1ull << (8 * valid)) - 1;
                    esc_lo &= (uint32_t)live;
                    esc_hi &= (uint32_t)(live >> 32);
                    codes &= (1u << (4 * valid)) - 1;
                }
                *reinterpret_cast<uint2*>(dst_a + 8 * g) = make_uint2(a_lo, a_hi);
                *reinterpret_cast<uint32_t*>(dst_b + 4 * g) = codes;
            }
            if (__any_sync(0xffffffffu, (esc_lo | esc_hi) != 0)) {
                s_flag[g] = (uint8_t)escape_mask(esc_lo, esc_hi);
                if (esc_lo | esc_hi) *reinterpret_cast<uint2*>(s_exb + 8 * g) = make_uint2(e_lo, e_hi);
                rows |= 1u << (it * 4 + r);
            }
        }
    }
    if (rows == 0) return 0;  // uniform: rows is built from warp votes
    __syncwarp();
    uint2 fw = make_uint2(0, 0);
    if ((rows >> (lane >> 2)) & 1) fw = *reinterpret_cast<const uint2*>(s_flag + 8 * lane);
    const uint32_t c = __popc(fw.x) + __popc(fw.y);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const uint32_t cnt = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t* list = p.lists + u * kListCap;
    uint32_t j = incl - c;
    uint32_t lo = fw.x, hi = fw.y;
    while (lo | hi) {
        const bool in_lo = lo != 0;
        const uint32_t bp = (uint32_t)(__ffs(in_lo ? lo : hi) - 1) + (in_lo ? 0u : 32u);
        if (in_lo) lo &= lo - 1;
        else hi &= hi - 1;
        const uint32_t pos = 64 * lane + bp;
        if (j < kListCap) st_u32_keep(list + j, pos | ((uint32_t)s_exb[pos] << 16), keep);
        j++;
    }
    if (cnt > kListCap) {  // the list overflowed: keep the masks instead
        uint32_t* gm = reinterpret_cast<uint32_t*>(p.masks + u * kUnitGroups);
        st_u32_keep(gm + 2 * lane, fw.x, keep);
        st_u32_keep(gm + 2 * lane + 1, fw.y, keep);
    }
    __syncwarp();
    return cnt;
}

// Publish a unit for the escape kernel: its count, and its escapes added to
// its segment's total (zeroed by the launch before the dense kernel, which
// is waited for before the first total update).
__device__ __forceinline__ void publish_unit(const Params& p, uint64_t u, uint32_t cnt, uint64_t keep,
                                             bool& cleared) {
    if ((threadIdx.x & 31) == 0) {
        st_u32_keep(p.counts + u, cnt, keep);
        if (cnt) {
            if (!cleared) {
                wait_for_prerequisite();
                cleared = true;
            }
            atomicAdd(&p.segs[u >> p.seg_shift], cnt);
        }
    }
}

__global__ void __launch_bounds__(kThreads, UZIP_ENC_MIN_BLOCKS) encode_dense_kernel(const Params p) {
    __shared__ uint32_t s_tab_words[64];
    uint8_t* s_tab = reinterpret_cast<uint8_t*>(s_tab_words);
    s_tab[threadIdx.x] = p.cb[UZIP_CB_ENC + threadIdx.x] | (p.cb[UZIP_CB_ESC + threadIdx.x] ? 0x80 : 0);
    __syncthreads();
    allow_dependent_launch();

    const uint64_t stride = (uint64_t)gridDim.x * kWarps;
    const uint64_t keep = l2_policy_evict_last();  // counts, lists, masks: read by the escape kernel
    bool cleared = false;
    __shared__ __align__(16) uint8_t s_flag[kWarps][kUnitGroups];  // per warp: escape mask of each group
    __shared__ __align__(16) uint8_t s_exb[kWarps][kUnit];         // per warp: exponent bytes of escaping groups
    const uint32_t wid = threadIdx.x >> 5;
    for (uint64_t u = (uint64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); u < p.units; u += stride)
        publish_unit(p, u, dense_unit_bf16(p, u, s_tab, s_flag[wid], s_exb[wid], keep), keep, cleared);
    // The grid completes only after the clearing launch has (the escape
    // pass, which waits for this grid, reads the totals).
    if (threadIdx.x == 0) wait_for_prerequisite();
}

// ------------------------------------------------------- FP8 E5M2 dense kernel

// E5M2 exponents have 5 bits, so a table of every exponent pair fits in
// shared memory: the entry of (ea, eb) = code(ea) | code(eb) << 4 (the packed
// code byte of two neighbouring values) | esc(ea) << 8 | esc(eb) << 9. One
// lookup then encodes two values. Two layouts:
//  - wide (the grid encoder, 31.9 KB): the entry of (ea, eb) at byte offset
//    (ea << 2 | eb << 10) ^ (eb & 7) << 4, i.e. the exponent bits of the byte
//    pair in place, with eb's low three bits folded into the bank bits (in
//    place alone, the bank would be ea's, and the pairs of a warp that share
//    ea would queue on one bank); both pairs of a word take one mask, one
//    shift and one three-input operation;
//  - compact (the one-CTA encoder, whose shared memory holds its lists):
//    2 KB, the entry at byte offset 2 (ea | eb << 5).
constexpr uint32_t kPairEntries = 1024;
constexpr uint32_t kWidePairHalfwords = 0x7C7C / 2 + 2;  // largest offset / 2, + 1, rounded to a word
__host__ __device__ constexpr uint32_t wide_pair_offset(uint32_t ea, uint32_t eb) {
    return ((ea << 2) | (eb << 10)) ^ ((eb & 7) << 4);
}
// Every pair has its own halfword of the wide table, inside it.
constexpr bool wide_pairs_distinct() {
    bool used[kWidePairHalfwords] = {};
    for (uint32_t i = 0; i < kPairEntries; i++) {
        const uint32_t o = wide_pair_offset(i & 31, i >> 5);
        if (o % 2 || o / 2 >= kWidePairHalfwords || used[o / 2]) return false;
        used[o / 2] = true;
    }
    return true;
}
static_assert(wide_pairs_distinct(), "wide pair table: offsets must be distinct, even and in range");

// Eight E5M2 values (w0, w1: value i in byte i) -> their 8 codes (one word,
// value i in nibble i), their 3-bit sign-mantissa fields (24 bits, value i at
// bits 3i) and their escape flags (byte k: bit 0 for value 2k, bit 1 for
// value 2k + 1). `pair`: the wide pair table if kWide, else the compact one.
template <bool kWide>
__device__ __forceinline__ void encode_group_e5m2(uint32_t w0, uint32_t w1, const uint16_t* pair, uint32_t& codes,
                                                  uint32_t& fields, uint32_t& escs) {
    const uint32_t w[2] = {w0, w1};
    uint32_t t[4], f[2];
#pragma unroll
    for (int h = 0; h < 2; h++) {
        // Field i = sign << 2 | mantissa of byte i, at bits 20 + 3i..22 + 3i
        // (bits 0..19 are left over and dropped below): the bits that move
        // up by 15 or 5 (signs of values 0 and 2, mantissas of 1 and 3) take
        // one multiply by 2^15 + 2^5, those that move up by 20, 10 or 0
        // (mantissas of 0 and 2, signs of 1 and 3) one by 2^20 + 2^10 + 2^0;
        // no two copies meet at bits 20..31, and the others fall below them
        // or past bit 31 (checked for all 4096 sign-mantissa patterns).
        f[h] = ((w[h] & 0x03800380u) * 0x8020u) | ((w[h] & 0x80038003u) * 0x100401u);
        // Exponent bytes e0..e3 -> the byte offsets of the pairs (e0, e1) and
        // (e2, e3) in the table, in bits 0..15 and 16..31 (offsets rather
        // than indices: no scaling before the loads).
        const char* pb = reinterpret_cast<const char*>(pair);
        uint32_t o;
        if (kWide) {
            o = (w[h] & 0x7C7C7C7Cu) ^ ((w[h] >> 6) & 0x00700070u);  // wide_pair_offset of both pairs
        } else {
            const uint32_t e2 = (w[h] >> 1) & 0x3E3E3E3Eu;  // 2 e in each byte
            o = (e2 & 0x003E003Eu) | ((e2 >> 3) & 0x07C007C0u);  // 2 (e0 | e1 << 5), 2 (e2 | e3 << 5)
        }
        t[2 * h] = *reinterpret_cast<const uint16_t*>(pb + (o & 0xFFFFu));  // values 0, 1 of the word
        t[2 * h + 1] = *reinterpret_cast<const uint16_t*>(pb + (o >> 16));  // values 2, 3
    }
    const uint32_t x = prmt(t[0], t[1], 0x5140), y = prmt(t[2], t[3], 0x5140);
    codes = prmt(x, y, 0x5410);
    escs = prmt(x, y, 0x7632);
    fields = (f[0] >> 20) | ((f[1] >> 8) & 0x00FFF000u);  // the two 12-bit field words, side by side
}

// Escape flags of encode_group_e5m2 (pair k's two bits in byte k) -> 8-bit
// mask, value i at bit i: the multiply moves byte k's bits to 18 + 2k, and no
// two of its shifted copies overlap or carry into that window.
__device__ __forceinline__ uint32_t escape_mask_pairs(uint32_t escs) {
    return (((escs & 0x03030303u) * 0x41041u) >> 18) & 0xFFu;
}

// The dense pass for E5M2 input: as for BF16, one warp per unit of 2048
// values, but each lane takes 32 consecutive values per step (two 16-byte
// loads; 12 bytes of packed fields and 16 bytes of codes stored), so a row of
// the warp covers 1024 values in ascending lane order and its escapes are
// ranked with one scan; a unit whose list overflows keeps 32-bit mask words
// (word s = unit positions 32 s ..). s_pair: the table of exponent pairs
// (the wide layout for the workspace path, the compact one when kSmem); `row`:
// the unit's row of `lists` and `masks_all` (u itself for the workspace).
template <bool kSmem>
__device__ __forceinline__ uint32_t dense_unit_e5m2(const Params& p, uint64_t u, uint64_t row, const uint16_t* s_pair,
                                                    uint32_t* lists, uint8_t* masks_all, uint64_t keep) {
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t ubase = u * kUnit;
    const uint32_t ulen = (uint32_t)min((uint64_t)kUnit, p.n - ubase);
    const uint8_t* src = p.in8 + ubase;
    uint8_t* dst_a = p.out + p.L.off_a + u * (kUnit / 8 * 3);
    uint8_t* dst_b = p.out + p.L.off_b + u * (kUnit / 2);
    uint32_t* list = lists + row * kListCap;
    const bool full = ulen == kUnit;
    uint32_t cnt = 0;
    uint32_t mwords[2] = {0, 0};
    // both rows' loads first: a lane has 64 bytes in flight per unit
    uint32_t wall[2][8];
#pragma unroll
    for (int it = 0; it < 2; it++) {
        const uint32_t v0 = 32 * (it * 32 + lane);
        uint32_t* w = wall[it];
        if (full || v0 + 32 <= ulen) {
            const uint4 x0 = ld_stream_v4(src + v0), x1 = ld_stream_v4(src + v0 + 16);
            w[0] = x0.x, w[1] = x0.y, w[2] = x0.z, w[3] = x0.w;
            w[4] = x1.x, w[5] = x1.y, w[6] = x1.z, w[7] = x1.w;
        } else {  // the tensor's ragged tail
#pragma unroll
            for (int k = 0; k < 8; k++) w[k] = 0;
#pragma unroll
            for (uint32_t i = 0; i < 32; i++)
                if (v0 + i < ulen) w[i / 4] |= (uint32_t)src[v0 + i] << (8 * (i & 3));
        }
    }
#pragma unroll
    for (int it = 0; it < 2; it++) {
        const uint32_t slot = it * 32 + lane;
        const uint32_t v0 = 32 * slot;  // this lane's values v0 .. v0 + 31 of the unit
        const uint32_t* w = wall[it];
        uint32_t codes[4], fields[4], escs[4];
        uint32_t escany = 0;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            encode_group_e5m2<!kSmem>(w[2 * q], w[2 * q + 1], s_pair, codes[q], fields[q], escs[q]);
            escany |= escs[q];
        }
        const uint32_t valid = ulen > v0 ? min(ulen - v0, 32u) : 0u;
        if (valid < 32) {  // only real values have codes and fields (escapes: masked below)
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const uint32_t vq = valid > 8u * q ? min(valid - 8u * q, 8u) : 0u;
                if (vq < 8) {
                    codes[q] &= (1u << (4 * vq)) - 1;
                    fields[q] &= (1u << (3 * vq)) - 1;
                }
            }
        }
        // four 24-bit field words -> 12 bytes: one byte permute per 4 bytes
        const uint32_t f0 = prmt(fields[0], fields[1], 0x4210), f1 = prmt(fields[1], fields[2], 0x5421),
                       f2 = prmt(fields[2], fields[3], 0x6542);
        if (valid == 32) {
            *reinterpret_cast<uint4*>(dst_b + 16 * slot) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
            uint32_t* fa = reinterpret_cast<uint32_t*>(dst_a + 12 * slot);
            fa[0] = f0;
            fa[1] = f1;
            fa[2] = f2;
        } else if (valid > 0) {  // the last groups of the tensor: nothing past their bytes
            const uint32_t gv = (valid + 7) / 8;
#pragma unroll
            for (uint32_t q = 0; q < 4; q++)
                if (q < gv) *reinterpret_cast<uint32_t*>(dst_b + 16 * slot + 4 * q) = codes[q];
#pragma unroll
            for (uint32_t b = 0; b < 12; b++)
                if (b < 3 * gv) dst_a[12 * slot + b] = (uint8_t)((b < 4 ? f0 : b < 8 ? f1 : f2) >> (8 * (b & 3)));
        }
        // Escapes of this row (1024 values, lane-major): one scan ranks them.
        if (__any_sync(0xffffffffu, (escany & 0x03030303u) != 0)) {
            uint32_t emask = 0;
#pragma unroll
            for (int q = 0; q < 4; q++) emask |= escape_mask_pairs(escs[q]) << (8 * q);
            if (valid < 32) emask &= (1u << valid) - 1;  // (valid == 0: no bits)
            const uint32_t c = __popc(emask);
            uint32_t incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            uint32_t j = cnt + incl - c;
            for (uint32_t bits = emask; bits; bits &= bits - 1, j++) {
                const uint32_t b = __ffs(bits) - 1;
                const uint32_t k = b >> 2;  // input word of value b, chosen in registers
                const uint32_t lo = (k & 2) ? ((k & 1) ? w[3] : w[2]) : ((k & 1) ? w[1] : w[0]);
                const uint32_t hi = (k & 2) ? ((k & 1) ? w[7] : w[6]) : ((k & 1) ? w[5] : w[4]);
                const uint32_t e = (((k & 4) ? hi : lo) >> (8 * (b & 3) + 2)) & 0x1F;
                if (j < kListCap) put_u32<kSmem>(list + j, (v0 + b) | (e << 16), keep);
            }
            cnt += __shfl_sync(0xffffffffu, incl, 31);
            mwords[it] = emask;
        }
    }
    if (cnt > kListCap) {  // the list overflowed: keep the masks (word s = unit positions 32 s ..)
        uint8_t* masks = masks_all + row * kUnitGroups;
#pragma unroll
        for (int it = 0; it < 2; it++) put_u32<kSmem>(reinterpret_cast<uint32_t*>(masks) + it * 32 + lane, mwords[it], keep);
    }
    return cnt;
}

// The pair table (wide or compact layout) of the 1024 pairs, from the
// 32-entry table of code | escape << 7 in s_tab (built by the first 32
// threads). The wide table's other halfwords are never read.
template <bool kWide>
__device__ __forceinline__ void build_pair_table(const Params& p, uint8_t* s_tab, uint16_t* s_pair) {
    if (threadIdx.x < 32)
        s_tab[threadIdx.x] = p.cb[UZIP_CB_ENC + threadIdx.x] | (p.cb[UZIP_CB_ESC + threadIdx.x] ? 0x80 : 0);
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < kPairEntries; i += blockDim.x) {
        const uint32_t ta = s_tab[i & 31], tb = s_tab[i >> 5];
        s_pair[kWide ? wide_pair_offset(i & 31, i >> 5) / 2 : i] =
            (uint16_t)((ta & 0xF) | ((tb & 0xF) << 4) | ((ta >> 7) << 8) | ((tb >> 7) << 9));
    }
}

__global__ void __launch_bounds__(kThreads, UZIP_ENC_E5_MIN_BLOCKS) encode_dense_e5m2_kernel(const Params p) {
    __shared__ uint8_t s_tab[32];
    __shared__ __align__(16) uint16_t s_pair[kWidePairHalfwords];
    build_pair_table<true>(p, s_tab, s_pair);
    __syncthreads();
    allow_dependent_launch();

    const uint64_t stride = (uint64_t)gridDim.x * kWarps;
    const uint64_t keep = l2_policy_evict_last();
    bool cleared = false;
    for (uint64_t u = (uint64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); u < p.units; u += stride)
        publish_unit(p, u, dense_unit_e5m2<false>(p, u, u, s_pair, p.lists, p.masks, keep), keep, cleared);
    // The grid completes only after the clearing launch has (the escape
    // pass, which waits for this grid, reads the totals).
    if (threadIdx.x == 0) wait_for_prerequisite();
}

// ----------------------------------------------------------- escape kernel

// One lane's view of unit u's escapes at unit positions [plo, phi): from the
// unit's sorted list, or (a unit that overflowed its list) from its mask bytes
// with exponents re-read from the input.
struct UnitPart {
    uint32_t ubase;  // first value of the unit (n < 2^32)
    uint32_t cnt;    // all escapes of the unit
    uint32_t plo, phi;
    bool list;
};

// Bits of mask word w (unit positions 32 w ..) that lie in [lo, hi).
__device__ __forceinline__ uint32_t bits_in(uint32_t word, uint32_t w, uint32_t lo, uint32_t hi) {
    const uint32_t b0 = 32 * w;
    const uint32_t keep_hi = hi >= b0 + 32 ? 0xFFFFFFFFu : (hi <= b0 ? 0u : (1u << (hi - b0)) - 1);
    const uint32_t drop_lo = lo >= b0 + 32 ? 0xFFFFFFFFu : (lo <= b0 ? 0u : (1u << (lo - b0)) - 1);
    return word & keep_hi & ~drop_lo;
}

// A range's loads, issued together before any of them is used: per unit (one
// per lane and round) its count and first kHeadEntries list entries; the
// counts of the earlier units of u0's segment; the segment totals between the
// block's base segment and u0's segment.
constexpr int kPreLoads = 2;  // earlier-unit counts per lane, loaded up front (segments of 64 units)

// kRounds = 1 when every range overlaps at most 32 units (one per lane); 2 for
// the chunk sizes whose single chunk can overlap 33 units (longer than
// 32 * 2048 - 2040 values and not a multiple of 2048).
template <int kRounds>
struct RangeLoads {
    uint32_t c0, nq, s, e, u0, nu, seg;
    uint32_t cnt[kRounds];
    uint32_t pre_cnt[kPreLoads];
    uint32_t mid;
};

// Non-binding prefetch of a global line into L1.
__device__ __forceinline__ void prefetch_l1(const void* ptr) { asm volatile("prefetch.global.L1 [%0];" ::"l"(ptr)); }

template <int kRounds>
__device__ __forceinline__ void load_range(const Params& p, uint64_t r, uint32_t seg_first, RangeLoads<kRounds>& rl,
                                           uint32_t* s_head) {
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t C = p.chunk;
    rl.c0 = (uint32_t)(r * p.range_chunks);
    const uint32_t c1 = (uint32_t)min((uint64_t)rl.c0 + p.range_chunks, p.L.nc);
    rl.nq = c1 - rl.c0;
    rl.s = rl.c0 * C;  // < n < 2^32
    rl.e = (uint32_t)min((uint64_t)c1 * C, p.n);
    rl.u0 = rl.s / kUnit;
    rl.nu = (rl.e - 1) / kUnit - rl.u0 + 1;
    rl.seg = rl.u0 >> p.seg_shift;
#pragma unroll
    for (int rr = 0; rr < kRounds; rr++) {
        const uint32_t u = rl.u0 + 32 * rr + lane;
        const bool on = 32 * rr + lane < rl.nu;
        rl.cnt[rr] = on ? __ldg(p.counts + u) : 0;
        if (on) {  // the list's first 32-byte sector -> shared memory (the rest once the count is known)
            const uint32_t* list = p.lists + (uint64_t)u * kListCap;
            cp_async16(s_head + head_slot(rr, lane, 0), list);
            cp_async16(s_head + head_slot(rr, lane, 4), list + 4);
        }
    }
    cp_async_commit();
    const uint32_t first = rl.seg * p.seg_units;
#pragma unroll
    for (int j = 0; j < kPreLoads; j++) {
        const uint32_t i = first + 32 * j + lane;
        rl.pre_cnt[j] = i < rl.u0 ? __ldg(p.counts + i) : 0;
    }
    uint32_t mid = 0;
    for (uint32_t i = seg_first + lane; i < rl.seg; i += 32) mid += __ldg(p.segs + i);
    rl.mid = mid;
}

// One range: the chunk offsets c0 .. c0 + nq - 1 and the range's escape blocks
// (and, for the last range, offsets[nc], the padding and the header). base =
// escapes before the block's base segment.
template <int kRounds>
__device__ __forceinline__ void escape_range(const Params& p, const RangeLoads<kRounds>& rl, uint32_t base,
                                             uint8_t* stage, uint32_t* s_head, uint32_t* s_cp) {
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t C = p.chunk;
    const uint32_t c0 = rl.c0, nq = rl.nq, s = rl.s, e = rl.e, u0 = rl.u0, nu = rl.nu, seg = rl.seg;

    // Longer lists: their entries 8 .. kHeadEntries - 1 follow into shared
    // memory (entries past that are read from global memory, prefetched into
    // L1 here).
#pragma unroll
    for (int rr = 0; rr < kRounds; rr++) {
        if (32 * rr + lane < nu && rl.cnt[rr] > 8) {
            const uint32_t c = min(rl.cnt[rr], kListCap);
            const uint32_t* list = p.lists + (uint64_t)(u0 + 32 * rr + lane) * kListCap;
            for (uint32_t j = 8; j < min(c, kHeadEntries); j += 4)
                cp_async16(s_head + head_slot(rr, lane, j), list + j);
            for (uint32_t j = kHeadEntries; j < c; j += 8) prefetch_l1(list + j);  // one 32-byte sector each
        }
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncwarp();
    auto entry = [&](int rr, uint32_t ubase, uint32_t j) -> uint32_t {
        return j < kHeadEntries ? s_head[head_slot(rr, lane, j)]
                                : __ldg(p.lists + (uint64_t)(ubase / kUnit) * kListCap + j);
    };

    UnitPart up[kRounds];
    uint32_t n_lo[kRounds], n_in[kRounds];
#pragma unroll
    for (int rr = 0; rr < kRounds; rr++) {
        n_lo[rr] = n_in[rr] = 0;
        up[rr].list = true;
        if (32 * rr + lane < nu) {
            UnitPart& u = up[rr];
            const uint32_t uidx = u0 + 32 * rr + lane;
            u.ubase = uidx * kUnit;
            u.cnt = rl.cnt[rr];
            u.plo = s > u.ubase ? s - u.ubase : 0u;
            u.phi = min(kUnit, e - u.ubase);
            u.list = u.cnt <= kListCap;
            if (u.list) {
                const uint32_t ulen = (uint32_t)min((uint64_t)kUnit, p.n - u.ubase);
                if (u.plo == 0 && u.phi >= ulen) {
                    n_in[rr] = u.cnt;  // the whole unit lies in the range
                } else {
                    for (uint32_t j = 0; j < u.cnt; j++) {
                        const uint32_t pos = entry(rr, u.ubase, j) & 0xFFFF;
                        n_lo[rr] += pos < u.plo;
                        n_in[rr] += pos >= u.plo && pos < u.phi;
                    }
                }
            }
        }
    }
    // Units that overflowed their list are handled by the whole warp: lane
    // l takes mask words 2l and 2l+1 (unit positions 64l .. 64l+63).
    auto coop = [&](int rr, int o, uint64_t& ub, uint32_t& plo, uint32_t& phi, uint32_t& b0, uint32_t& b1) {
        ub = __shfl_sync(0xffffffffu, up[rr].ubase, o);
        plo = __shfl_sync(0xffffffffu, up[rr].plo, o);
        phi = __shfl_sync(0xffffffffu, up[rr].phi, o);
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(p.masks + (ub / kUnit) * kUnitGroups) + lane);
        b0 = bits_in(w.x, 2 * lane, plo, phi);
        b1 = bits_in(w.y, 2 * lane + 1, plo, phi);
        return w;
    };
#pragma unroll
    for (int rr = 0; rr < kRounds; rr++) {
        for (uint32_t ovf = __ballot_sync(0xffffffffu, !up[rr].list); ovf; ovf &= ovf - 1) {
            const int o = __ffs(ovf) - 1;
            uint64_t ub;
            uint32_t plo, phi, b0, b1;
            const uint2 w = coop(rr, o, ub, plo, phi, b0, b1);
            const uint32_t lo = warp_sum(__popc(bits_in(w.x, 2 * lane, 0, plo)) +
                                         __popc(bits_in(w.y, 2 * lane + 1, 0, plo)));
            const uint32_t in = warp_sum(__popc(b0) + __popc(b1));
            if (lane == (uint32_t)o) {
                n_lo[rr] = lo;
                n_in[rr] = in;
            }
        }
    }
    // Escapes before s: the block base, the segment totals up to u0's
    // segment, the earlier units of that segment, and unit u0's escapes
    // before s.
    uint32_t part = rl.mid;
#pragma unroll
    for (int j = 0; j < kPreLoads; j++) part += rl.pre_cnt[j];
    for (uint32_t i = seg * p.seg_units + 32 * kPreLoads + lane; i < u0; i += 32) part += __ldg(p.counts + i);
    const uint32_t pre = base + warp_sum(part) + __shfl_sync(0xffffffffu, n_lo[0], 0);

    // Pass 1: running rank of each unit's first in-range escape, and every
    // chunk's first rank. Chunk q starts at value s + q * C.
    __syncwarp();  // the previous range's chunk table is no longer read
    uint32_t first[kRounds];
    uint32_t carry = 0;
#pragma unroll
    for (int rr = 0; rr < kRounds; rr++) {
        uint32_t incl = n_in[rr];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        first[rr] = carry + incl - n_in[rr];
        carry += __shfl_sync(0xffffffffu, incl, 31);
        if (32 * rr + lane < nu && up[rr].list) {
            const UnitPart& u = up[rr];
            const uint32_t v_lo = u.ubase + u.plo - s;  // range offset of plo
            uint32_t q = div_chunk(p, v_lo + C - 1);
            uint32_t x = s + q * C - u.ubase;  // unit position of chunk q's start
            uint32_t i = n_lo[rr];
            const uint32_t iend = n_lo[rr] + n_in[rr];
            while (q < nq && x < u.phi) {
                // First entry at or past x: binary search (the list is ascending;
                // entries from n_lo on are at or past plo, so none is needed there).
                uint32_t hi = x > u.plo ? iend : i;
                while (i < hi) {
                    const uint32_t mid = (i + hi) >> 1;
                    if ((entry(rr, u.ubase, mid) & 0xFFFF) < x) i = mid + 1;
                    else hi = mid;
                }
                s_cp[q] = first[rr] + (i - n_lo[rr]);
                q++;
                x += C;
            }
        }
        for (uint32_t ovf = __ballot_sync(0xffffffffu, !up[rr].list); ovf; ovf &= ovf - 1) {
            const int o = __ffs(ovf) - 1;
            uint64_t ub;
            uint32_t plo, phi, b0, b1;
            coop(rr, o, ub, plo, phi, b0, b1);
            const uint32_t f = __shfl_sync(0xffffffffu, first[rr], o);
            const uint32_t c = __popc(b0) + __popc(b1);
            uint32_t ic = c;
#pragma unroll
            for (int k = 1; k < 32; k <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, ic, k);
                if (lane >= k) ic += t;
            }
            const uint32_t before = f + ic - c;  // rank of this lane's first escape
            const uint32_t lo = max(64 * lane, plo), hi = min(64 * lane + 64, phi);
            if (lo < hi) {
                const uint32_t v_lo = (uint32_t)(ub + lo) - s;
                uint32_t q = div_chunk(p, v_lo + C - 1);
                uint32_t x = (uint32_t)(s + q * C - ub);
                while (q < nq && x < hi) {
                    const uint32_t d = x - 64 * lane;  // 0..63
                    const uint32_t below = d < 32 ? __popc(b0 & ((1u << d) - 1))
                                                  : __popc(b0) + __popc(b1 & ((1u << (d - 32)) - 1));
                    s_cp[q] = before + below;
                    q++;
                    x += C;
                }
            }
        }
    }
    const uint32_t rtotal = carry;
    if (lane == 0) s_cp[nq] = rtotal;
    __syncwarp();

    uint8_t* offs = p.out + p.L.off_c;
    for (uint32_t q = lane; q < nq; q += 32)
        *reinterpret_cast<uint32_t*>(offs + 4ull * (c0 + q)) = pre + s_cp[q];
    if (c0 + nq == p.L.nc && lane == 0) {  // the last range: tail, padding, header
        const uint64_t m = (uint64_t)pre + rtotal;
        *reinterpret_cast<uint32_t*>(offs + 4 * p.L.nc) = (uint32_t)m;
        zero_words(p.out, p.L.off_c + 4 * (p.L.nc + 1), p.L.off_d);
        const uint64_t groups_all = (p.n + 7) / 8;
        zero_bytes(p.out, p.L.off_a + p.a_bytes, p.L.off_b);
        zero_words(p.out, p.L.off_b + 4 * groups_all, p.L.off_c);
        // Escape bytes are written only below out_capacity; the stream is
        // complete exactly when its total fits.
        write_header(p, m, stream_total(p, m) > p.cap ? UZIP_FLAG_CAPACITY : 0u);
    }
    if (rtotal == 0) return;

    // Pass 2: each escape's chunk-relative position and raw exponent. The
    // range's escape blocks are contiguous in the stream: assemble them in
    // this warp's stage -- shifted by the destination's offset within a
    // 16-byte piece, so whole pieces can be copied out -- and store them with
    // coalesced 16-byte stores, unless there are too many, then store them
    // directly.
    const bool sent = p.fmt == kSentinel;  // values only, at the escape's rank
    const uint64_t dbase = p.L.off_d + (sent ? (uint64_t)pre : 3ull * pre);
    const uint32_t dbytes = sent ? rtotal : 3 * rtotal;
    const uint32_t lead = (uint32_t)(dbase & 15);
    const bool staged = lead + dbytes <= kStageBytes;
    // One escape: its position bytes at block offset rel_pos, its value at rel_val.
    auto emit = [&](uint32_t rel_pos, uint32_t rel_val, uint32_t pos, uint32_t expo) {
        if (staged) {
            if (!sent) {
                stage[lead + rel_pos] = (uint8_t)(pos & 0xFF);
                stage[lead + rel_pos + 1] = (uint8_t)(pos >> 8);
            }
            stage[lead + rel_val] = (uint8_t)expo;
        } else if (sent) {
            if (dbase + rel_val < p.cap) p.out[dbase + rel_val] = (uint8_t)expo;
        } else if (dbase + rel_val < p.cap && dbase + rel_pos + 1 < p.cap) {
            p.out[dbase + rel_pos] = (uint8_t)(pos & 0xFF);
            p.out[dbase + rel_pos + 1] = (uint8_t)(pos >> 8);
            p.out[dbase + rel_val] = (uint8_t)expo;
        }
    };
    auto put = [&](uint32_t off, uint32_t rank_in_range, uint32_t q, uint32_t expo) {
        const uint32_t cstart = s_cp[q];
        const uint32_t k = s_cp[q + 1] - cstart;
        const uint32_t rank = rank_in_range - cstart;
        if (sent)
            emit(0, rank_in_range, 0, expo);
        else
            emit(3 * cstart + 2 * rank, 3 * cstart + 2 * k + rank, off - q * C, expo);
    };
    if (kRounds == 1 && __any_sync(0xffffffffu, n_in[0] > kParallelAbove)) {
        // Some unit has many escapes: go escape-parallel. Lane l takes range
        // ranks l, l + 32, ...; the unit
        // holding rank r is the last lane whose first rank is <= r (lanes
        // past the range's units never match).
        const uint32_t key = lane < nu ? first[0] : 0xFFFFFFFFu;
        const uint32_t nlo = n_lo[0], is_list = up[0].list ? 1u : 0u;
        for (uint32_t r0 = 0; r0 < rtotal; r0 += 32) {
            const uint32_t r = r0 + lane;
            uint32_t L = 0;
#pragma unroll
            for (uint32_t st = 16; st; st >>= 1) {
                const uint32_t kc = __shfl_sync(0xffffffffu, key, L + st);
                if (kc <= r) L += st;
            }
            const uint32_t fL = __shfl_sync(0xffffffffu, key, L);
            const uint32_t nloL = __shfl_sync(0xffffffffu, nlo, L);
            const uint32_t listL = __shfl_sync(0xffffffffu, is_list, L);
            if (r < rtotal && listL) {
                const uint32_t j = r - fL + nloL;  // index in unit L's list
                const uint32_t ent = j < kHeadEntries ? s_head[head_slot(0, L, j)]
                                                      : __ldg(p.lists + (uint64_t)(u0 + L) * kListCap + j);
                const uint32_t off = (u0 + L) * kUnit + (ent & 0xFFFF) - s;
                put(off, r, div_chunk(p, off), ent >> 16);
            }
        }
    } else {
#pragma unroll
        for (int rr = 0; rr < kRounds; rr++) {
            if (32 * rr + lane < nu && up[rr].list && n_in[rr]) {
                const UnitPart& u = up[rr];
                // Walk the unit's list chunk by chunk: one chunk-table lookup
                // per chunk, then each escape's bytes follow the previous
                // one's (positions 2 bytes on, values 1 byte on); the next
                // entry is read before the current escape is stored.
                uint32_t i = n_lo[rr];
                const uint32_t iend = i + n_in[rr];
                uint32_t rank = first[rr];
                if (staged && !sent && iend <= kHeadEntries) {
                    // The common case, specialised: every entry in shared
                    // memory, every byte into the stage.
                    const uint32_t* hrow = s_head + (uint32_t)rr * (kHeadEntries * 32) + lane * kHeadEntries;
                    const uint32_t hsw = (lane & 7) << 2;  // entry j of the row is hrow[j ^ hsw]
                    uint32_t ent = hrow[i ^ hsw];
                    uint32_t off = u.ubase + (ent & 0xFFFF) - s;
                    for (;;) {
                        const uint32_t q = div_chunk(p, off);
                        const uint32_t qbeg = q * C;
                        const uint32_t cstart = s_cp[q];
                        const uint32_t k = s_cp[q + 1] - cstart;
                        uint8_t* sp = stage + lead + 3 * cstart + 2 * (rank - cstart);
                        uint8_t* sv = stage + lead + 3 * cstart + 2 * k + (rank - cstart);
                        bool more;
                        for (;;) {
                            const uint32_t pos = off - qbeg, expo = ent >> 16;
                            i++;
                            rank++;
                            more = i < iend;
                            if (more) ent = hrow[i ^ hsw];
                            sp[0] = (uint8_t)(pos & 0xFF);
                            sp[1] = (uint8_t)(pos >> 8);
                            *sv = (uint8_t)expo;
                            sp += 2;
                            sv += 1;
                            if (!more) break;
                            off = u.ubase + (ent & 0xFFFF) - s;
                            if (off >= qbeg + C) break;  // the next escape opens another chunk
                        }
                        if (!more) break;
                    }
                    continue;
                }
                uint32_t ent = entry(rr, u.ubase, i);
                uint32_t off = u.ubase + (ent & 0xFFFF) - s;
                for (;;) {
                    const uint32_t q = div_chunk(p, off);
                    const uint32_t qbeg = q * C;
                    const uint32_t cstart = s_cp[q];
                    const uint32_t k = s_cp[q + 1] - cstart;
                    uint32_t rel_pos = 3 * cstart + 2 * (rank - cstart);
                    uint32_t rel_val = sent ? rank : 3 * cstart + 2 * k + (rank - cstart);
                    bool more;
                    for (;;) {
                        const uint32_t pos = off - qbeg, expo = ent >> 16;
                        i++;
                        rank++;
                        more = i < iend;
                        if (more) ent = entry(rr, u.ubase, i);
                        emit(rel_pos, rel_val, pos, expo);
                        rel_pos += 2;
                        rel_val += 1;
                        if (!more) break;
                        off = u.ubase + (ent & 0xFFFF) - s;
                        if (off >= qbeg + C) break;  // the next escape opens another chunk
                    }
                    if (!more) break;
                }
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < kRounds; rr++) {
        for (uint32_t ovf = __ballot_sync(0xffffffffu, !up[rr].list); ovf; ovf &= ovf - 1) {
            const int o = __ffs(ovf) - 1;
            uint64_t ub;
            uint32_t plo, phi, b0, b1;
            coop(rr, o, ub, plo, phi, b0, b1);
            const uint32_t f = __shfl_sync(0xffffffffu, first[rr], o);
            const uint32_t c = __popc(b0) + __popc(b1);
            uint32_t ic = c;
#pragma unroll
            for (int k = 1; k < 32; k <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, ic, k);
                if (lane >= k) ic += t;
            }
            uint32_t running = f + ic - c;
            // this lane's escapes, exponents re-read kBatch at a time
            while (b0 | b1) {
                uint32_t offs_b[kBatch], ex[kBatch];
                int got = 0;
#pragma unroll
                for (int t = 0; t < kBatch; t++) {
                    offs_b[t] = 0;
                    if (b0 | b1) {
                        const bool lo_word = b0 != 0;
                        const uint32_t bits = lo_word ? b0 : b1;
                        const uint32_t pos = 64 * lane + (lo_word ? 0 : 32) + (__ffs(bits) - 1);
                        if (lo_word) b0 &= b0 - 1;
                        else b1 &= b1 - 1;
                        offs_b[t] = (uint32_t)(ub + pos) - s;
                        got = t + 1;
                    }
                }
#pragma unroll
                for (int t = 0; t < kBatch; t++)
                    ex[t] = t >= got ? 0
                            : p.fmt == kE5M2 ? (__ldg(p.in8 + s + offs_b[t]) >> 2) & 0x1F
                                             : (__ldg(p.in + s + offs_b[t]) >> 7) & 0xFF;
#pragma unroll
                for (int t = 0; t < kBatch; t++)
                    if (t < got) put(offs_b[t], running++, div_chunk(p, offs_b[t]), ex[t]);
            }
        }
    }
    if (staged) {
        // Stage bytes [lead, lead + dbytes) go to the 16-byte aligned global
        // address gbase + the same index: whole 16-byte pieces as vectors,
        // the partial first and last pieces byte by byte.
        __syncwarp();
        const uint32_t end = lead + dbytes;
        const uint64_t gbase = dbase - lead;
        const bool fits = dbase + dbytes <= p.cap;
        for (uint32_t b0 = 16 * lane; b0 < end; b0 += 512) {
            if (fits && b0 >= lead && b0 + 16 <= end) {
                *reinterpret_cast<uint4*>(p.out + gbase + b0) = *reinterpret_cast<const uint4*>(stage + b0);
            } else {
                for (uint32_t i = max(b0, lead); i < min(b0 + 16, end); i++)
                    if (gbase + i < p.cap) p.out[gbase + i] = stage[i];
            }
        }
        __syncwarp();  // the stage is reused by the next range
    }
}

template <int kRounds>
__global__ void __launch_bounds__(kThreads, UZIP_ESC_MIN_BLOCKS) encode_escape_kernel(const Params p) {
    extern __shared__ __align__(16) uint32_t s_dyn[];
    __shared__ uint32_t s_red[kWarps];
    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Layout: per-warp escape staging | per-warp list heads | per-warp chunk tables.
    uint8_t* stage = reinterpret_cast<uint8_t*>(s_dyn) + warp * kStageBytes;
    uint32_t* s_head = s_dyn + kWarps * kStageBytes / 4 + warp * (kRounds * kHeadEntries * 32);
    uint32_t* s_cp = s_dyn + kWarps * (kStageBytes / 4 + kRounds * kHeadEntries * 32) + warp * (p.range_chunks + 1);

    wait_for_prerequisite();  // the dense kernel's stream and workspace are complete past this point

    const uint64_t stride = (uint64_t)gridDim.x * kWarps;
    for (uint64_t rb = (uint64_t)blockIdx.x * kWarps; rb < p.ranges; rb += stride) {
        // Ranges rb .. rb + 7, one per warp, in ascending order. The block's
        // base: escapes of the segments before the one holding range rb's
        // first unit (a block-wide sum of at most kMaxSegments totals).
        const uint64_t r = rb + warp;
        const bool active = r < p.ranges;
        const uint32_t seg_first = (uint32_t)(rb * p.range_chunks * p.chunk / kUnit) >> p.seg_shift;
        RangeLoads<kRounds> rl;
        __syncwarp();  // the previous range's list entries are no longer read
        if (active) load_range(p, r, seg_first, rl, s_head);
        uint32_t v = 0;
#pragma unroll
        for (int k = 0; k < (int)(kMaxSegments / kThreads); k++) {
            const uint32_t i = tid + k * kThreads;
            if (i < seg_first) v += __ldg(p.segs + i);
        }
        v = warp_sum(v);
        __syncthreads();  // the previous round's totals are read
        if (lane == 0) s_red[warp] = v;
        __syncthreads();
        uint32_t base = 0;
#pragma unroll
        for (int w = 0; w < kWarps; w++) base += s_red[w];
        if (active) escape_range<kRounds>(p, rl, base, stage, s_head, s_cp);
    }
}

// ------------------------------------------------------------ short inputs
//
// An input of at most kSmallUnits units and kSmallChunks chunks is encoded by
// one CTA in one launch. A warp per unit runs the dense pass with the unit's
// escape list (or mask bytes) in shared memory; after a barrier the CTA scans
// the unit counts, finds each chunk's first escape (a binary search of the
// chunk's start in its unit's list), writes the offsets and places every
// escape (a thread per escape: its unit from the unit prefixes, its chunk
// from its position). Nothing goes through the workspace: the input is read,
// the stream written, and a message costs one kernel launch instead of two.
#ifndef UZIP_SMALL_UNITS
#define UZIP_SMALL_UNITS 32
#endif
constexpr uint32_t kSmallUnits = UZIP_SMALL_UNITS;  // inputs of up to this many units of 2048 values
constexpr uint32_t kSmallChunks = 4096;  // chunk offsets held in shared memory
constexpr int kSmallThreads = 32 * kSmallUnits;

// Position in its unit of the j-th escape of a unit that kept mask bits
// (bit b of word w: position 32 w + b; j is below the unit's count, so the
// walk ends inside its kUnit / 32 words).
__device__ uint32_t nth_mask_bit(const uint32_t* words, uint32_t j) {
    for (uint32_t w = 0; w < kUnit / 32; w++) {
        uint32_t x = words[w];
        const uint32_t c = __popc(x);
        if (j < c) {
            for (; j; j--) x &= x - 1;
            return 32 * w + (__ffs(x) - 1);
        }
        j -= c;
    }
    return kUnit;  // not reached
}

// Escapes of a unit before its position x, from its list (cu <= kListCap
// entries, ascending positions) or its mask words.
__device__ __forceinline__ uint32_t escapes_before(const uint32_t* list, const uint32_t* masks, uint32_t cu,
                                                   uint32_t x) {
    uint32_t below = 0;
    if (cu <= kListCap) {
        uint32_t hi = cu;
        while (below < hi) {
            const uint32_t mid = (below + hi) >> 1;
            if ((list[mid] & 0xFFFF) < x) below = mid + 1;
            else hi = mid;
        }
    } else {
        for (uint32_t w = 0; w < x / 32; w++) below += __popc(masks[w]);
        if (x % 32) below += __popc(masks[x / 32] & ((1u << (x % 32)) - 1));
    }
    return below;
}

// The j-th escape of local unit i (count cu) of a short-input CTA, from the
// CTA's shared lists or mask words: its position in the unit and its
// exponent (re-read from the input for a unit that kept mask bits; ubase =
// the unit's first value).
template <bool kE5>
__device__ __forceinline__ void unit_escape(const Params& p, const uint32_t* list, const uint32_t* masks, uint32_t cu,
                                            uint32_t j, uint32_t ubase, uint32_t& pos, uint32_t& expo) {
    if (cu <= kListCap) {
        const uint32_t e = list[j];
        pos = e & 0xFFFF;
        expo = e >> 16;
    } else {
        pos = nth_mask_bit(masks, j);
        const uint32_t i = ubase + pos;
        expo = kE5 ? (p.in8[i] >> 2) & 0x1F : (p.in[i] >> 7) & 0xFF;
    }
}

// Escape gi (global rank) at value i, in chunk q with offsets o .. o1: its
// bytes in the stream (the sentinel format keeps the value only); every byte
// below out_capacity.
__device__ __forceinline__ void put_escape(const Params& p, uint32_t gi, uint32_t i, uint32_t q, uint32_t o,
                                           uint32_t o1, uint32_t expo) {
    const uint64_t dbase = p.L.off_d;
    if (p.fmt == kSentinel) {
        if (dbase + gi < p.cap) p.out[dbase + gi] = (uint8_t)expo;
    } else {
        const uint32_t r = gi - o, k = o1 - o, pq = i - q * p.chunk;
        const uint64_t bp = dbase + 3ull * o + 2 * r, bv = dbase + 3ull * o + 2 * k + r;
        if (bp < p.cap) p.out[bp] = (uint8_t)(pq & 0xFF);
        if (bp + 1 < p.cap) p.out[bp + 1] = (uint8_t)(pq >> 8);
        if (bv < p.cap) p.out[bv] = (uint8_t)expo;
    }
}

// A warp's inclusive scan.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, uint32_t lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= (uint32_t)o) v += t;
    }
    return v;
}

// The code tables of a short-input CTA (BF16 / sentinel: the 256-byte
// code | escape << 7 table; E5M2: the compact pair table).
template <bool kE5>
__device__ __forceinline__ void build_small_tables(const Params& p, uint8_t* s_tab, uint16_t* s_pair) {
    if (kE5) {
        build_pair_table<false>(p, s_tab, s_pair);
    } else if (threadIdx.x < 256) {
        s_tab[threadIdx.x] = p.cb[UZIP_CB_ENC + threadIdx.x] | (p.cb[UZIP_CB_ESC + threadIdx.x] ? 0x80 : 0);
    }
    __syncthreads();
}

// Padding and header, by one thread, once every escape is counted.
__device__ void finish_stream(const Params& p, uint32_t m) {
    zero_words(p.out, p.L.off_c + 4 * (p.L.nc + 1), p.L.off_d);
    zero_bytes(p.out, p.L.off_a + p.a_bytes, p.L.off_b);
    zero_words(p.out, p.L.off_b + 4 * ((p.n + 7) / 8), p.L.off_c);
    write_header(p, m, stream_total(p, m) > p.cap ? UZIP_FLAG_CAPACITY : 0u);
}

template <bool kE5>
__global__ void __launch_bounds__(kSmallThreads, 1) encode_small_kernel(const Params p) {
    __shared__ uint32_t s_list[kSmallUnits][kListCap];
    __shared__ __align__(16) uint32_t s_masks[kSmallUnits][kUnitGroups / 4];
    __shared__ uint32_t s_pre[kSmallUnits + 1];   // escapes before unit u; s_pre[units] = M
    __shared__ uint32_t s_off[kSmallChunks + 1];  // the chunk offsets
    __shared__ uint32_t s_tab_words[64];
    __shared__ uint16_t s_pair[kE5 ? kPairEntries : 2];
    uint8_t* s_tab = reinterpret_cast<uint8_t*>(s_tab_words);
    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    build_small_tables<kE5>(p, s_tab, s_pair);
    const uint32_t units = (uint32_t)p.units, nc = (uint32_t)p.L.nc;

    // 1. the dense pass, a warp per unit
    if (warp < units) {
        uint8_t* masks = reinterpret_cast<uint8_t*>(s_masks[warp]);
        const uint32_t cnt = kE5 ? dense_unit_e5m2<true>(p, warp, 0, s_pair, s_list[warp], masks, 0)
                                 : dense_unit_bf16_shared(p, warp, s_tab, s_list[warp], masks);
        if (lane == 0) s_pre[warp + 1] = cnt;
    }
    __syncthreads();
    // 2. the unit prefix
    if (warp == 0) {
        const uint32_t incl = warp_incl_scan(lane < units ? s_pre[lane + 1] : 0u, lane);
        if (lane < units) s_pre[lane + 1] = incl;
        if (lane == 0) s_pre[0] = 0;
    }
    __syncthreads();
    const uint32_t m = s_pre[units];
    // 3. each chunk's first escape: chunk q starts at position x of unit u
    for (uint32_t q = tid; q < nc; q += blockDim.x) {
        const uint32_t st = q * p.chunk, u = st / kUnit, x = st % kUnit;
        s_off[q] = s_pre[u] + escapes_before(s_list[u], s_masks[u], s_pre[u + 1] - s_pre[u], x);
    }
    if (tid == 0) s_off[nc] = m;
    __syncthreads();
    uint8_t* offs = p.out + p.L.off_c;
    for (uint32_t q = tid; q <= nc; q += blockDim.x) *reinterpret_cast<uint32_t*>(offs + 4ull * q) = s_off[q];
    // 4. every escape: its unit, its place in the unit, its chunk
    for (uint32_t gi = tid; gi < m; gi += blockDim.x) {
        uint32_t lo = 0, hi = units;  // s_pre[lo] <= gi < s_pre[hi]
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (s_pre[mid] <= gi) lo = mid;
            else hi = mid;
        }
        uint32_t pos, expo;
        unit_escape<kE5>(p, s_list[lo], s_masks[lo], s_pre[lo + 1] - s_pre[lo], gi - s_pre[lo], lo * kUnit, pos,
                         expo);
        const uint32_t i = lo * kUnit + pos, q = div_chunk(p, i);
        put_escape(p, gi, i, q, s_off[q], s_off[q + 1], expo);
    }
    // 5. padding and header
    if (tid == 0) finish_stream(p, m);
}

// ------------------------------------------------------------ mid-size inputs
//
// Inputs of more than kSmallUnits and at most kClusterUnits units (and at
// most kSmallChunks chunks) in one launch of one thread-block cluster: C <=
// kMaxCluster CTAs on C SMs, CTA b taking U units (b U .., a warp per unit,
// at least 256 threads; the grid is the cluster, C = ceil(units / U)).
// Each CTA runs the one-CTA encoder's dense pass and unit scan in its shared
// memory and counts, for every chunk that starts in its values, the escapes
// between its first value and that start. After a cluster barrier each CTA
// reads the others' escape totals from their shared memory (distributed
// shared memory, no global memory and no atomics), writes the offsets of the
// chunks that start in its values and places its own escapes; the offsets of
// the at most two chunks it shares with other CTAs (the one its first value
// lies in, the first one after its values) come from their owners' shared
// memory. A second cluster barrier, after the last of those reads, keeps every
// CTA's shared memory in place while others read it. Clusters of up to 16
// CTAs (above the portable 8, allowed per kernel; the host checks that such
// a cluster fits before taking this path): against the two-kernel path,
// 96-256 units encode 0.8-1.9 us sooner; from 256 units on, 16 SMs' share of
// the bandwidth is the limit and the two-kernel path is as fast.
#ifndef UZIP_MAX_CLUSTER
#define UZIP_MAX_CLUSTER 16
#endif
constexpr uint32_t kMaxCluster = UZIP_MAX_CLUSTER;
constexpr uint32_t kClusterUnits = 256;  // 524,288 values
static_assert(kMaxCluster <= 32, "the CTA totals are scanned by one warp");

__device__ __forceinline__ uint32_t shared_addr(const void* q) { return (uint32_t)__cvta_generic_to_shared(q); }

// The word at shared address a (this CTA's layout) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t a, uint32_t rank) {
    uint32_t r, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(r) : "memory");
    return v;
}

// Every thread of every CTA of the cluster; orders shared-memory writes
// before the barrier with reads after it, across the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <bool kE5>
__global__ void __launch_bounds__(kSmallThreads, 1) encode_cluster_kernel(const Params p, uint32_t U) {
    __shared__ uint32_t s_list[kSmallUnits][kListCap];
    __shared__ __align__(16) uint32_t s_masks[kSmallUnits][kUnitGroups / 4];
    __shared__ uint32_t s_pre[kSmallUnits + 1];    // escapes before this CTA's unit i, from its first value
    __shared__ uint32_t s_below[kSmallChunks];     // chunk qa + k: escapes from this CTA's first value to its start
    __shared__ uint32_t s_total;                   // this CTA's escapes (read by the others)
    __shared__ uint32_t s_cpre[kMaxCluster + 1];   // escapes before CTA c
    __shared__ uint32_t s_edge[2];                 // offsets of the chunks shared with other CTAs
    __shared__ uint32_t s_tab_words[64];
    __shared__ uint16_t s_pair[kE5 ? kPairEntries : 2];
    uint8_t* s_tab = reinterpret_cast<uint8_t*>(s_tab_words);
    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t b = blockIdx.x, C = gridDim.x;
    build_small_tables<kE5>(p, s_tab, s_pair);
    const uint32_t units = (uint32_t)p.units, nc = (uint32_t)p.L.nc, chunk = p.chunk, n32 = (uint32_t)p.n;
    const uint32_t span = U * kUnit;                        // values per CTA (< 2^20)
    const uint32_t u0 = b * U, nu = min(U, units - u0);     // C = ceil(units / U): nu >= 1
    const uint32_t v0 = u0 * kUnit, v1 = min(n32, v0 + nu * kUnit);

    // 1. the dense pass, a warp per unit
    if (warp < nu) {
        uint8_t* masks = reinterpret_cast<uint8_t*>(s_masks[warp]);
        const uint32_t cnt = kE5 ? dense_unit_e5m2<true>(p, u0 + warp, 0, s_pair, s_list[warp], masks, 0)
                                 : dense_unit_bf16_shared(p, u0 + warp, s_tab, s_list[warp], masks);
        if (lane == 0) s_pre[warp + 1] = cnt;
    }
    __syncthreads();
    // 2. this CTA's unit prefix
    if (warp == 0) {
        const uint32_t incl = warp_incl_scan(lane < nu ? s_pre[lane + 1] : 0u, lane);
        if (lane < nu) s_pre[lane + 1] = incl;
        if (lane == 0) s_pre[0] = 0;
    }
    __syncthreads();
    const uint32_t total = s_pre[nu];
    // 3. escapes from this CTA's first value to each chunk start in its values
    const uint32_t qa = (v0 + chunk - 1) / chunk, qb = (v1 + chunk - 1) / chunk;  // chunk starts in [v0, v1)
    for (uint32_t q = qa + tid; q < qb; q += blockDim.x) {
        const uint32_t st = q * chunk, i = st / kUnit - u0, x = st % kUnit;
        s_below[q - qa] = s_pre[i] + escapes_before(s_list[i], s_masks[i], s_pre[i + 1] - s_pre[i], x);
    }
    if (tid == 0) s_total = total;
    cluster_sync();
    // 4. escapes before each CTA; the shared chunks' offsets from their owners
    if (warp == 0) {
        const uint32_t incl = warp_incl_scan(lane < C ? ld_cluster_u32(shared_addr(&s_total), lane) : 0u, lane);
        if (lane < C) s_cpre[lane + 1] = incl;
        if (lane == 0) s_cpre[0] = 0;
        __syncwarp();
        if (lane < 2) {
            const uint32_t q = lane == 0 ? v0 / chunk : qb;  // the chunk holding v0; the first one after v1
            uint32_t o = s_cpre[C];                          // past the last chunk: M
            if (q < nc) {
                const uint32_t ob = q * chunk / span, oqa = (ob * span + chunk - 1) / chunk;
                o = s_cpre[ob] + (ob == b ? s_below[q - qa] : ld_cluster_u32(shared_addr(&s_below[q - oqa]), ob));
            }
            s_edge[lane] = o;
        }
    }
    cluster_sync();  // the last reads of other CTAs' shared memory are done
    const uint32_t cpre = s_cpre[b], m = s_cpre[C];
    uint8_t* offs = p.out + p.L.off_c;
    for (uint32_t q = qa + tid; q < qb; q += blockDim.x)
        *reinterpret_cast<uint32_t*>(offs + 4ull * q) = cpre + s_below[q - qa];
    if (b == C - 1 && tid == 0) *reinterpret_cast<uint32_t*>(offs + 4ull * nc) = m;
    // 5. this CTA's escapes: unit, place in the unit, chunk
    for (uint32_t r = tid; r < total; r += blockDim.x) {
        uint32_t lo = 0, hi = nu;  // s_pre[lo] <= r < s_pre[hi]
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (s_pre[mid] <= r) lo = mid;
            else hi = mid;
        }
        uint32_t pos, expo;
        unit_escape<kE5>(p, s_list[lo], s_masks[lo], s_pre[lo + 1] - s_pre[lo], r - s_pre[lo], (u0 + lo) * kUnit, pos,
                         expo);
        const uint32_t i = (u0 + lo) * kUnit + pos, q = div_chunk(p, i);
        const uint32_t o = q >= qa ? cpre + s_below[q - qa] : s_edge[0];
        const uint32_t o1 = q + 1 < qb ? cpre + s_below[q + 1 - qa] : s_edge[1];
        put_escape(p, cpre + r, i, q, o, o1, expo);
    }
    // 6. padding and header
    if (b == 0 && tid == 0) finish_stream(p, m);
}

// n == 0: header, offsets[0] = 0 and padding only.
__global__ void encode_empty_kernel(const Params p) {
    *reinterpret_cast<uint32_t*>(p.out + p.L.off_c) = 0;
    zero_words(p.out, p.L.off_c + 4, p.L.off_d);
    write_header(p, 0, 0);
}

}  // namespace
}  // namespace uzip

using namespace uzip;

extern "C" UZIP_API size_t uzip_encode_workspace_bytes(size_t n, uint32_t chunk) {
    if (!chunk_valid(chunk) || n > UZIP_MAX_N) return 0;
    return (size_t)geometry_of(n).bytes;
}

namespace uzip {
namespace {

#define CUDA_RET(x)                            \
    do {                                       \
        const cudaError_t e_ = (x);            \
        if (e_ != cudaSuccess) return e_;      \
    } while (0)

// Per-device launch facts, looked up on the first call on each device (the
// results are the same whichever thread gets there first).
struct DeviceFacts {
    int dev, sms, per_sm1, per_sm1e;
    bool cluster;  // a cluster of kMaxCluster CTAs of encode_cluster_kernel can run (both formats)
};
constexpr int kMaxFactDevices = 64;
std::atomic<int> g_facts_ready[kMaxFactDevices];
DeviceFacts g_facts[kMaxFactDevices];
// Escape-kernel residency per device, variant (one or two rounds) and
// largest chunk table (0 = not looked up yet).
std::atomic<int> g_escape_per_sm[kMaxFactDevices][2][kMaxRangeChunks + 1];

size_t escape_smem(uint32_t range_chunks, int rounds) {
    return (size_t)kWarps * (kStageBytes + 4ull * rounds * kHeadEntries * 32 + 4ull * (range_chunks + 1));
}

// Let both escape-kernel variants take their largest dynamic shared memory.
// A function attribute belongs to the current context, which a
// cudaDeviceReset replaces, so it is set again before every launch that
// needs it (a host-side call, no device work).
cudaError_t allow_escape_smem() {
    void (*esc[2])(Params) = {encode_escape_kernel<1>, encode_escape_kernel<2>};
    for (int k = 0; k < 2; k++) {
        const size_t smem_max = escape_smem(kMaxRangeChunks, k + 1);
        if (smem_max > 48 * 1024) {
            const cudaError_t e =
                cudaFuncSetAttribute(esc[k], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

int device_facts(DeviceFacts& f) {
    int dev = 0;
    UZIP_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < kMaxFactDevices && g_facts_ready[dev].load(std::memory_order_acquire)) {
        f = g_facts[dev];
        return UZIP_OK;
    }
    f.dev = dev;
    UZIP_CUDA_TRY(cudaDeviceGetAttribute(&f.sms, cudaDevAttrMultiProcessorCount, dev));
    UZIP_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&f.per_sm1, encode_dense_kernel, kThreads, 0));
    UZIP_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&f.per_sm1e, encode_dense_e5m2_kernel, kThreads, 0));
    UZIP_CUDA_TRY(allow_escape_smem());
    if (f.sms < 1 || f.per_sm1 < 1 || f.per_sm1e < 1) return UZIP_ERR_CUDA;
    // Whether a cluster of kMaxCluster CTAs of the cluster encoder can run
    // here; if not, mid-size inputs take the two-kernel path.
    f.cluster = true;
    void (*ck[2])(Params, uint32_t) = {encode_cluster_kernel<false>, encode_cluster_kernel<true>};
    for (int k = 0; k < 2; k++) {
        if (kMaxCluster > 8 &&
            cudaFuncSetAttribute(ck[k], cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
            (void)cudaGetLastError();  // not this call's error
            f.cluster = false;
            continue;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kMaxCluster);
        cfg.blockDim = dim3(kSmallThreads);
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = kMaxCluster;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, ck[k], &cfg) != cudaSuccess || clusters < 1) {
            (void)cudaGetLastError();  // not this call's error
            f.cluster = false;
        }
    }
    if (dev < kMaxFactDevices) {
        g_facts[dev] = f;
        g_facts_ready[dev].store(1, std::memory_order_release);
    }
    return UZIP_OK;
}

// Inputs of more than kSmallUnits and at most kClusterUnits units: one
// cluster of C CTAs of encode_cluster_kernel, U units each.
cudaError_t launch_cluster(const Params& p, const Geometry& g, uint32_t fmt, cudaStream_t s) {
    if (kMaxCluster > 8) {  // a cluster above the portable size: allowed per function and context
        cudaError_t e = cudaFuncSetAttribute(encode_cluster_kernel<false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(encode_cluster_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    const uint32_t U = (uint32_t)((g.units + kMaxCluster - 1) / kMaxCluster);
    const uint32_t C = (uint32_t)((g.units + U - 1) / U);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(std::max<uint32_t>(256, 32 * U));  // a warp per unit, at least the table's 256 threads
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return fmt == kE5M2 ? cudaLaunchKernelEx(&cfg, encode_cluster_kernel<true>, p, U)
                        : cudaLaunchKernelEx(&cfg, encode_cluster_kernel<false>, p, U);
}

// Longer inputs: the segment-total clear (when there are several segments),
// the dense kernel and the escape kernel, each a programmatic dependent of
// the one before.
cudaError_t launch_two_kernels(Params p, const Geometry& g, const Layout& L, const DeviceFacts& f, uint32_t fmt,
                               cudaStream_t s) {
    const uint32_t chunk = p.chunk;
    // Dense kernel: one resident wave.
    const uint64_t grid1 = std::min<uint64_t>((g.units + kWarps - 1) / kWarps,
                                              (uint64_t)f.sms * (fmt == kE5M2 ? f.per_sm1e : f.per_sm1));
    // Escape kernel: ranges of whole chunks, sized so every resident warp
    // gets at most one (the per-range cost is mostly load latency).
    const int two_rounds = chunk > 32 * kUnit - 2040 && chunk % kUnit != 0;
    const uint32_t rc_max =
        std::max<uint32_t>(1, std::min<uint32_t>(kMaxRangeChunks, kMaxRangeUnits * kUnit / chunk));
    // Residency at the largest chunk table this chunk size can need.
    int per_sm2 = f.dev < kMaxFactDevices ? g_escape_per_sm[f.dev][two_rounds][rc_max].load() : 0;
    if (per_sm2 < 1) {
        CUDA_RET(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm2, two_rounds ? encode_escape_kernel<2> : encode_escape_kernel<1>, kThreads,
            escape_smem(rc_max, two_rounds + 1)));
        if (per_sm2 > 0 && f.dev < kMaxFactDevices) g_escape_per_sm[f.dev][two_rounds][rc_max].store(per_sm2);
    }
    if (per_sm2 < 1) return cudaErrorInvalidConfiguration;
    const uint64_t warps2 = (uint64_t)f.sms * per_sm2 * kWarps;
    p.range_chunks = (uint32_t)std::min<uint64_t>(rc_max, std::max<uint64_t>(1, (L.nc + warps2 - 1) / warps2));
    p.ranges = (L.nc + p.range_chunks - 1) / p.range_chunks;
    const uint64_t grid2 = std::min<uint64_t>((p.ranges + kWarps - 1) / kWarps, (uint64_t)f.sms * per_sm2);

    // Segment totals start at zero; the last segment's is never read (no
    // escape lies after it), so a single-segment input (up to 64 units)
    // needs no clearing. The clearing kernel lets the dense kernel
    // launch behind it at once (programmatic dependent launch).
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg1 = {};
    cfg1.gridDim = dim3((unsigned)grid1);
    cfg1.blockDim = dim3(kThreads);
    cfg1.stream = s;
    if (g.nseg > 1) {
        clear_segments_kernel<<<1, 256, 0, s>>>(p.segs, g.nseg - 1);
        CUDA_RET(cudaGetLastError());
        cfg1.attrs = pdl;
        cfg1.numAttrs = 1;
    }
    CUDA_RET(cudaLaunchKernelEx(&cfg1, fmt == kE5M2 ? encode_dense_e5m2_kernel : encode_dense_kernel, p));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = escape_smem(p.range_chunks, two_rounds + 1);
    if (cfg.dynamicSmemBytes > 48 * 1024) CUDA_RET(allow_escape_smem());
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return two_rounds ? cudaLaunchKernelEx(&cfg, encode_escape_kernel<2>, p)
                      : cudaLaunchKernelEx(&cfg, encode_escape_kernel<1>, p);
}

}  // namespace

int encode_impl(const void* d_in_bf16, size_t n, uint32_t chunk, const void* d_codebook, void* d_out,
                size_t out_capacity, void* d_workspace, size_t workspace_bytes, size_t* h_out_bytes,
                uzip_stream_t stream, uint32_t fmt) {
    if (!chunk_valid(chunk)) return UZIP_ERR_CHUNK;
    if (n > UZIP_MAX_N || !d_out || !d_codebook || (n > 0 && !d_in_bf16) || !d_workspace) return UZIP_ERR_ARG;
    if (!aligned16(d_out) || !aligned16(d_codebook) || !aligned16(d_workspace) ||
        (n > 0 && !aligned16(d_in_bf16)))
        return UZIP_ERR_ALIGN;
    const Layout L = layout_for(fmt, n, chunk);
    if (out_capacity < L.off_d) return UZIP_ERR_CAPACITY;
    const Geometry g = geometry_of(n);
    if (workspace_bytes < g.bytes) return UZIP_ERR_CAPACITY;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    Params p;
    p.in = static_cast<const uint16_t*>(d_in_bf16);
    p.in8 = static_cast<const uint8_t*>(d_in_bf16);
    p.fmt = fmt;
    p.a_bytes = fmt == kE5M2 ? 3 * ((n + 7) / 8) : n;
    p.n = n;
    p.chunk = chunk;
    p.chunk_shift = (chunk & (chunk - 1)) == 0 ? (uint32_t)__builtin_ctz(chunk) : 32u;
    p.units = g.units;
    p.cb = static_cast<const uint8_t*>(d_codebook);
    p.out = static_cast<uint8_t*>(d_out);
    p.cap = out_capacity;
    p.L = L;
    p.seg_units = g.seg_units;
    p.seg_shift = (uint32_t)__builtin_ctz(g.seg_units);
    p.nseg = g.nseg;
    p.segs = reinterpret_cast<uint32_t*>(ws + g.off_segs);
    p.counts = reinterpret_cast<uint32_t*>(ws + g.off_counts);
    p.lists = reinterpret_cast<uint32_t*>(ws + g.off_lists);
    p.masks = ws + g.off_masks;

    if (n == 0) {
        encode_empty_kernel<<<1, 1, 0, s>>>(p);
        UZIP_CUDA_TRY(cudaGetLastError());
    } else if (g.units <= kSmallUnits && L.nc <= kSmallChunks) {  // one CTA, one launch
        // a warp per unit, and at least the 256 threads that build the code table
        const uint32_t threads = std::max<uint32_t>(256, 32 * (uint32_t)g.units);
        if (fmt == kE5M2) encode_small_kernel<true><<<1, threads, 0, s>>>(p);
        else encode_small_kernel<false><<<1, threads, 0, s>>>(p);
        UZIP_CUDA_TRY(cudaGetLastError());
    } else {
        DeviceFacts f;
        const int rc = device_facts(f);
        if (rc != UZIP_OK) return rc;
        UZIP_CUDA_TRY(f.cluster && g.units <= kClusterUnits && L.nc <= kSmallChunks
                          ? launch_cluster(p, g, fmt, s)                // one cluster, one launch
                          : launch_two_kernels(p, g, L, f, fmt, s));  // dense + escape kernels
    }
    if (h_out_bytes) {
        uint32_t hdr[16];
        UZIP_CUDA_TRY(cudaMemcpyAsync(hdr, d_out, sizeof(hdr), cudaMemcpyDeviceToHost, s));
        UZIP_CUDA_TRY(cudaStreamSynchronize(s));
        *h_out_bytes = (size_t)hdr[12] | ((size_t)hdr[13] << 32);
        const uint32_t flags = hdr[1] >> 16;
        if (flags & UZIP_FLAG_CAPACITY) return UZIP_ERR_CAPACITY;
    }
    return UZIP_OK;
}

}  // namespace uzip

extern "C" UZIP_API int uzip_encode(const void* d_in_bf16, size_t n, uint32_t chunk, const void* d_codebook,
                                    void* d_out, size_t out_capacity, void* d_workspace, size_t workspace_bytes,
                                    size_t* h_out_bytes, uzip_stream_t stream) {
    return encode_impl(d_in_bf16, n, chunk, d_codebook, d_out, out_capacity, d_workspace, workspace_bytes,
                       h_out_bytes, stream);
}

// ------------------------------------------------------------ FP8 E5M2

extern "C" UZIP_API int uzip_e5m2_encode(const void* d_in_e5m2, size_t n, uint32_t chunk, const void* d_codebook,
                                         void* d_out, size_t out_capacity, void* d_workspace, size_t workspace_bytes,
                                         size_t* h_out_bytes, uzip_stream_t stream) {
    return encode_impl(d_in_e5m2, n, chunk, d_codebook, d_out, out_capacity, d_workspace, workspace_bytes,
                       h_out_bytes, stream, kE5M2);
}

// ------------------------------------------------------ Top-15 + sentinel

extern "C" UZIP_API int uzip_sentinel_encode(const void* d_in_bf16, size_t n, uint32_t chunk,
                                             const void* d_codebook, void* d_out, size_t out_capacity,
                                             void* d_workspace, size_t workspace_bytes, size_t* h_out_bytes,
                                             uzip_stream_t stream) {
    return encode_impl(d_in_bf16, n, chunk, d_codebook, d_out, out_capacity, d_workspace, workspace_bytes,
                       h_out_bytes, stream, kSentinel);
}

extern "C" UZIP_API size_t uzip_sentinel_compressed_size(size_t n, size_t n_escapes, uint32_t chunk) {
    if (!chunk_valid(chunk) || n > UZIP_MAX_N || n_escapes > n) return 0;
    return (size_t)(layout_of(n, chunk).off_d + (uint64_t)n_escapes);
}

extern "C" UZIP_API size_t uzip_e5m2_compressed_size(size_t n, size_t n_escapes, uint32_t chunk) {
    if (!chunk_valid(chunk) || n > UZIP_MAX_N || n_escapes > n) return 0;
    return (size_t)(layout_e5m2_of(n, chunk).off_d + 3 * (uint64_t)n_escapes);
}

// ------------------------------------------------------ per-input codebook

// SplitZip review page, §4.3 Table 7 (dynamic Top-16): the codebook is rebuilt
// for every input -- the histogram of all n exponents, the Top-16, the tables
// -- and the input is then encoded with it. Two reads of the input: the
// histogram must be complete before the first code is chosen.
extern "C" UZIP_API int uzip_encode_dynamic(const void* d_in_bf16, size_t n, uint32_t chunk, void* d_codebook,
                                            void* d_out, size_t out_capacity, void* d_workspace,
                                            size_t workspace_bytes, size_t* h_out_bytes, uzip_stream_t stream) {
    if (!chunk_valid(chunk)) return UZIP_ERR_CHUNK;
    if (n > UZIP_MAX_N) return UZIP_ERR_ARG;
    const int rc = calibrate_impl(d_in_bf16, n, d_codebook, reinterpret_cast<cudaStream_t>(stream));
    if (rc != UZIP_OK) return rc;
    return encode_impl(d_in_bf16, n, chunk, d_codebook, d_out, out_capacity, d_workspace, workspace_bytes,
                       h_out_bytes, stream);
}

// ------------------------------------------------- encoding without allocation
//
// Some callers cannot allocate device memory for the encoder's workspace:
// code running where a framework's caching allocator has already reserved the
// device memory and hands out no raw buffers, or latency-critical paths that
// must not call cudaMalloc (which can synchronise the device). For them the
// workspace lives in a file-scope device array, fixed at load time: every GPU
// that loads this library holds kNoAllocScratchBytes (about 8.1 MiB) of it
// until the process exits. Host code cannot use the array's name as a device
// address, so every call looks the address up with cudaGetSymbolAddress, for
// the device and context current at the call, and passes it to the same
// kernels uzip_encode launches. The lookup is not cached: after a
// cudaDeviceReset, or under another context, the module is loaded again and
// the array may sit at another address.

namespace uzip {
namespace {

// Workspace bytes the encoder needs for n values (the geometry above, which
// depends on n only).
constexpr uint64_t workspace_bytes_for(uint64_t n) { return geometry_of(n).bytes; }

constexpr uint64_t kNoAllocScratchBytes = workspace_bytes_for(UZIP_NOALLOC_MAX_N);

}  // namespace
}  // namespace uzip

static __device__ __align__(256) uint8_t g_noalloc_scratch[uzip::kNoAllocScratchBytes];

extern "C" UZIP_API int uzip_encode_noalloc(const void* d_in_bf16, size_t n, uint32_t chunk,
                                            const void* d_codebook, void* d_out, size_t out_capacity,
                                            size_t* h_out_bytes, uzip_stream_t stream) {
    if (n > UZIP_NOALLOC_MAX_N) return UZIP_ERR_CAPACITY;  // beyond the built-in scratch
    if (!chunk_valid(chunk)) return UZIP_ERR_CHUNK;
    const uint64_t need = geometry_of(n).bytes;
    if (need > kNoAllocScratchBytes) return UZIP_ERR_CAPACITY;
    void* scratch = nullptr;
    UZIP_CUDA_TRY(cudaGetSymbolAddress(&scratch, g_noalloc_scratch));
    if (!scratch) return UZIP_ERR_CUDA;
    return encode_impl(d_in_bf16, n, chunk, d_codebook, d_out, out_capacity, scratch, (size_t)need, h_out_bytes,
                       stream);
}
