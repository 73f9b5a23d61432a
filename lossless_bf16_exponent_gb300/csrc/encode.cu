// encode.cu -- SplitZip encoder for sm_103a: one pass over the input, two kernels.
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
//   dense kernel   each warp owns fixed units of 2048 values (grid-stride, no
//                  tickets, no barriers): 16-byte loads -> exponent and
//                  sign-mantissa bytes with byte permutes -> code + escape bit
//                  from a 256-byte shared table -> coalesced 8-byte
//                  sign-mantissa and 4-byte code stores; one escape-mask byte
//                  per group of eight values into the workspace (N/8 bytes),
//                  the unit's escape count, and the count added to its
//                  segment's total (64+ units per segment).
//   escape kernel  every CTA scans the segment totals in shared memory; each
//                  warp takes ranges of whole chunks, finds the range's first
//                  escape rank from the segment prefix, unit counts and masks,
//                  writes the chunk offsets, and writes each escape's
//                  chunk-relative position and raw exponent (re-read from the
//                  input, eight loads in flight per lane) in ascending element
//                  order, bounds-checked against out_capacity. The last CTA to
//                  finish writes the 64-byte header.
// The input is read from HBM once; the masks add N/8 bytes written and read.
#include <algorithm>
#include <atomic>

#include "uzip_internal.cuh"

namespace uzip {
namespace {

constexpr uint32_t kUnit = 2048;              // values per counting unit (one warp)
constexpr uint32_t kUnitGroups = kUnit / 8;   // its mask bytes
constexpr int kThreads = 256;                 // both kernels
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kMaxSegments = 2048;       // segment totals one CTA scans
constexpr uint32_t kRangeValues = 16384;      // target values per escape-kernel range
constexpr uint32_t kMaxRangeChunks = 256;     // bounds the per-warp chunk table
constexpr int kBatch = 8;                     // escape exponents re-read per lane at once
#ifndef UZIP_ENC_MIN_BLOCKS
#define UZIP_ENC_MIN_BLOCKS 4
#endif
#ifndef UZIP_ENC_ITER_UNROLL
#define UZIP_ENC_ITER_UNROLL 2
#endif
constexpr int kIterUnroll = UZIP_ENC_ITER_UNROLL;  // 2: both 4-load batches of a unit in flight per lane

// Start of the caller's workspace.
struct WsHeader {
    unsigned int done;
    unsigned int flags;
    unsigned long long m;
    unsigned long long pad[6];
};
static_assert(sizeof(WsHeader) == 64, "workspace header is 64 bytes");

struct Geometry {
    uint64_t units;         // counting units of kUnit values
    uint32_t seg_units;     // units per segment (power of two, >= 64)
    uint32_t nseg;          // segments
    uint32_t range_chunks;  // chunks per escape-kernel range
    uint64_t ranges;
    uint64_t off_segs, off_counts, off_masks, bytes;  // workspace layout
};

__host__ Geometry geometry_of(uint64_t n, uint32_t chunk) {
    Geometry g;
    g.units = (n + kUnit - 1) / kUnit;
    g.seg_units = 64;
    while ((g.units + g.seg_units - 1) / g.seg_units > kMaxSegments) g.seg_units *= 2;
    g.nseg = (uint32_t)((g.units + g.seg_units - 1) / g.seg_units);
    g.range_chunks = std::max<uint32_t>(1, std::min<uint32_t>(kRangeValues / chunk, kMaxRangeChunks));
    const uint64_t nc = (n + chunk - 1) / chunk;
    g.ranges = (nc + g.range_chunks - 1) / g.range_chunks;
    g.off_segs = sizeof(WsHeader);
    g.off_counts = g.off_segs + pad16(4ull * g.nseg);
    g.off_masks = g.off_counts + pad16(4ull * g.units);
    g.bytes = g.off_masks + pad16((n + 7) / 8);
    return g;
}

struct Params {
    const uint16_t* in;
    uint64_t n;
    uint32_t chunk;
    uint32_t seg_units;
    uint32_t nseg;
    uint32_t range_chunks;
    uint64_t units;
    uint64_t ranges;
    const uint8_t* cb;
    uint8_t* out;
    uint64_t cap;
    Layout L;
    WsHeader* ws;
    uint32_t* segs;
    uint32_t* counts;
    uint8_t* masks;
};

// Eight values -> 8 sign-mantissa bytes (a_lo, a_hi), 8 packed codes (one
// word, value i in nibble i) and an 8-bit escape mask.
__device__ __forceinline__ void encode_group(const uint4 v, const uint8_t* tab, uint32_t& a_lo,
                                             uint32_t& a_hi, uint32_t& codes, uint32_t& mask) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed[2], esc[2], am[2];
#pragma unroll
    for (int h = 0; h < 2; h++) {
        // Bytes of four values: high bytes (sign + exponent bits 7..1) and
        // low bytes (exponent bit 0 + mantissa).
        const uint32_t hi = prmt(w[2 * h], w[2 * h + 1], 0x7531);
        const uint32_t lo = prmt(w[2 * h], w[2 * h + 1], 0x6420);
        const uint32_t e4 = ((hi << 1) & 0xFEFEFEFEu) | ((lo >> 7) & 0x01010101u);
        am[h] = (hi & 0x80808080u) | (lo & 0x7F7F7F7Fu);
        // Table byte = code | escape << 7.
        const uint32_t t0 = tab[e4 & 0xFF];
        const uint32_t t1 = tab[(e4 >> 8) & 0xFF];
        const uint32_t t2 = tab[(e4 >> 16) & 0xFF];
        const uint32_t t3 = tab[e4 >> 24];
        const uint32_t t4 = prmt(prmt(t0, t1, 0x0040), prmt(t2, t3, 0x0040), 0x5410);
        const uint32_t c = t4 & 0x0F0F0F0Fu;
        packed[h] = c | (c >> 4);  // byte 0 = c0 | c1 << 4, byte 2 = c2 | c3 << 4
        esc[h] = t4 & 0x80808080u;
    }
    a_lo = am[0];
    a_hi = am[1];
    codes = prmt(packed[0], packed[1], 0x6420);
    // Bit 7 of byte i -> bit i (the four shifted copies never overlap).
    const uint32_t m_lo = (((esc[0] >> 7) * 0x204081u) >> 21) & 0xF;
    const uint32_t m_hi = (((esc[1] >> 7) * 0x204081u) >> 21) & 0xF;
    mask = m_lo | (m_hi << 4);
}

__device__ void write_header(const Params& p, uint64_t m, uint32_t flags) {
    uint4* h = reinterpret_cast<uint4*>(p.out);
    const uint64_t total = p.L.off_d + 3 * m;
    const uint4 exps = *reinterpret_cast<const uint4*>(p.cb + UZIP_CB_EXPS);
    h[0] = make_uint4(kStreamMagic, 1u | (flags << 16), (uint32_t)p.n, (uint32_t)(p.n >> 32));
    h[1] = make_uint4(p.chunk, (uint32_t)p.L.nc, (uint32_t)m, (uint32_t)(m >> 32));
    h[2] = exps;
    h[3] = make_uint4((uint32_t)total, (uint32_t)(total >> 32), 0u, 0u);
}

// Zero bytes [from, to) of the stream, 4-byte aligned bounds.
__device__ void zero_words(uint8_t* out, uint64_t from, uint64_t to) {
    for (uint64_t o = from; o < to; o += 4) *reinterpret_cast<uint32_t*>(out + o) = 0;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) { return __reduce_add_sync(0xffffffffu, v); }

// ------------------------------------------------------------ dense kernel

__global__ void __launch_bounds__(kThreads, UZIP_ENC_MIN_BLOCKS) encode_dense_kernel(const Params p) {
    __shared__ uint32_t s_tab_words[64];
    uint8_t* s_tab = reinterpret_cast<uint8_t*>(s_tab_words);
    s_tab[threadIdx.x] = p.cb[UZIP_CB_ENC + threadIdx.x] | (p.cb[UZIP_CB_ESC + threadIdx.x] ? 0x80 : 0);
    __syncthreads();

    const uint32_t lane = threadIdx.x & 31;
    const uint64_t stride = (uint64_t)gridDim.x * kWarps;
    for (uint64_t u = (uint64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); u < p.units; u += stride) {
        const uint64_t ubase = u * kUnit;
        const uint32_t ulen = (uint32_t)min((uint64_t)kUnit, p.n - ubase);
        const uint4* src = reinterpret_cast<const uint4*>(p.in + ubase);
        uint8_t* dst_a = p.out + p.L.off_a + ubase;
        uint8_t* dst_b = p.out + p.L.off_b + ubase / 2;
        uint8_t* gmask = p.masks + u * kUnitGroups;
        uint32_t cnt = 0;
#pragma unroll kIterUnroll
        for (int it = 0; it < 2; it++) {
            uint4 v[4];
#pragma unroll
            for (int r = 0; r < 4; r++) {
                const uint32_t g = it * 128 + r * 32 + lane;
                v[r] = make_uint4(0, 0, 0, 0);
                if (8 * g + 8 <= ulen) {
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
                if (8 * g >= ulen) continue;
                uint32_t a_lo, a_hi, codes, mask;
                encode_group(v[r], s_tab, a_lo, a_hi, codes, mask);
                if (8 * g + 8 > ulen) {  // codes and escapes of real values only
                    const uint32_t valid = ulen - 8 * g;
                    mask &= (1u << valid) - 1;
                    codes &= (1u << (4 * valid)) - 1;
                }
                *reinterpret_cast<uint2*>(dst_a + 8 * g) = make_uint2(a_lo, a_hi);
                *reinterpret_cast<uint32_t*>(dst_b + 4 * g) = codes;
                gmask[g] = (uint8_t)mask;
                cnt += __popc(mask);
            }
        }
        cnt = warp_sum(cnt);
        if (lane == 0) {
            p.counts[u] = cnt;
            if (cnt) atomicAdd(&p.segs[u / p.seg_units], cnt);
        }
    }
}

// ----------------------------------------------------------- escape kernel

// Escapes before value s (s a multiple of 8): the segment prefix, the counts
// of the earlier units of its segment, the mask bytes of its own unit. A
// segment holds at most 64 units at this size, so each lane loads at most two
// counts and eight mask bytes, all at once.
__device__ uint64_t escapes_before(const Params& p, const uint32_t* s_segpref, uint32_t s) {
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t us = s / kUnit;
    const uint32_t seg = us / p.seg_units;
    uint32_t part = 0;
    uint32_t i = seg * p.seg_units + lane;
    for (; i + 32 < us; i += 64) part += p.counts[i] + p.counts[i + 32];
    if (i < us) part += p.counts[i];
    const uint32_t bend = s / 8;
    uint32_t b = us * kUnitGroups + lane;
    uint32_t m[8];
#pragma unroll
    for (int j = 0; j < 8; j++) m[j] = (b + 32 * j < bend) ? p.masks[b + 32 * j] : 0;
#pragma unroll
    for (int j = 0; j < 8; j++) part += __popc(m[j]);
    return (uint64_t)s_segpref[seg] + warp_sum(part);
}

constexpr uint32_t kWinValues = 16384;  // values per mask window (2 KiB of mask bytes)
constexpr int kVecPerLane = 5;           // 16-byte mask vectors per lane per window (128 + 2 slack)

// One lane's share of a window of mask bytes: the 16-byte vectors [v0, v1) of
// the aligned span around the window's bytes, bytes outside the window
// cleared, kept in shared memory transposed (word k of lane l at
// sw[k * 32 + l]) so a warp touching word k of every lane hits 32 different
// banks. Bit i of word k stands for value 8 * (a_first + 4 * k) + i.
constexpr int kLaneWords = kVecPerLane * 4;

struct LaneSpan {
    uint32_t a_first;  // byte address of the lane's word 0 in the mask section
    uint32_t nwords;   // words the lane holds (<= kLaneWords)
};

__device__ __forceinline__ LaneSpan load_lane_masks(const Params& p, uint32_t b0, uint32_t nb, uint32_t* sw) {
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t a0 = b0 & ~15u;
    const uint32_t nvec = (b0 + nb - a0 + 15) / 16;
    const uint32_t vpl = (nvec + 31) / 32;
    const uint32_t v0 = min(lane * vpl, nvec), v1 = min(v0 + vpl, nvec);
    LaneSpan sp;
    sp.a_first = a0 + 16 * v0;
    sp.nwords = 4 * (v1 - v0);
    const uint4* src = reinterpret_cast<const uint4*>(p.masks + a0);
    uint4 v[kVecPerLane];
#pragma unroll
    for (int j = 0; j < kVecPerLane; j++) v[j] = (v0 + j < v1) ? src[v0 + j] : make_uint4(0, 0, 0, 0);
    const uint32_t lo = b0, hi = b0 + nb;  // the window's bytes
#pragma unroll
    for (int j = 0; j < kVecPerLane; j++) {
        uint32_t vw[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
        const uint32_t a = sp.a_first + 16 * j;
        if (a < lo || a + 16 > hi) {  // an edge vector: clear bytes outside the window
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const uint32_t wa = a + 4 * k;
                const uint32_t from = lo > wa ? min(lo - wa, 4u) : 0u;  // first kept byte
                const uint32_t to = hi > wa ? min(hi - wa, 4u) : 0u;     // one past the last
                const uint32_t upto = to >= 4 ? 0xFFFFFFFFu : (1u << (8 * to)) - 1;
                const uint32_t below = from >= 4 ? 0xFFFFFFFFu : (1u << (8 * from)) - 1;
                vw[k] &= upto & ~below;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; k++) sw[(4 * j + k) * 32 + lane] = vw[k];
    }
    return sp;
}

__global__ void __launch_bounds__(kThreads, 3) encode_escape_kernel(const Params p) {
    extern __shared__ __align__(16) uint32_t s_dyn[];
    __shared__ uint32_t s_warp[kWarps];
    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Layout: per-warp mask words | segment prefix (nseg + 1) | per-warp chunk tables.
    uint32_t* sw = s_dyn + warp * (kLaneWords * 32);
    uint32_t* s_segpref = s_dyn + kWarps * kLaneWords * 32;
    uint32_t* s_cp = s_segpref + ((p.nseg + 1 + 3) & ~3u) + warp * (p.range_chunks + 1);

    // Segment prefix, one block scan (kMaxSegments / kThreads = 8 totals per
    // thread, loaded together).
    {
        constexpr int kPer = kMaxSegments / kThreads;
        uint32_t v[kPer];
        uint32_t sum = 0;
#pragma unroll
        for (int i = 0; i < kPer; i++) {
            const uint32_t idx = tid * kPer + i;
            v[i] = idx < p.nseg ? p.segs[idx] : 0;
        }
#pragma unroll
        for (int i = 0; i < kPer; i++) sum += v[i];
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        uint32_t run = incl - sum;
        for (uint32_t w = 0; w < warp; w++) run += s_warp[w];
#pragma unroll
        for (int i = 0; i < kPer; i++) {
            const uint32_t idx = tid * kPer + i;
            if (idx <= p.nseg) s_segpref[idx] = run;
            run += v[i];
        }
        __syncthreads();
    }

    const uint32_t C = p.chunk;
    bool overflow = false;
    const uint64_t stride = (uint64_t)gridDim.x * kWarps;
    for (uint64_t r = (uint64_t)blockIdx.x * kWarps + warp; r < p.ranges; r += stride) {
        const uint32_t c0 = (uint32_t)(r * p.range_chunks);
        const uint32_t c1 = (uint32_t)min((uint64_t)c0 + p.range_chunks, p.L.nc);
        const uint32_t nq = c1 - c0;
        const uint32_t s = c0 * C;
        const uint32_t e = (uint32_t)min((uint64_t)c1 * C, p.n);
        const bool one_window = e - s <= kWinValues;
        __syncwarp();  // the previous range's words are no longer read
        // The first window's masks and the range's prefix are loaded together.
        LaneSpan sp = load_lane_masks(p, s / 8, (min(s + kWinValues, e) - s + 7) / 8, sw);
        const uint64_t pre = escapes_before(p, s_segpref, s);

        // Pass 1: first escape rank (within the range) of every chunk. Chunk
        // q starts at value s + q * C, a mask-byte boundary.
        uint32_t base = 0, lexcl = 0;
        for (uint32_t ws = s; ws < e; ws += kWinValues) {
            const uint32_t we = min(ws + kWinValues, e);
            if (ws != s) {
                __syncwarp();  // the previous window's words are no longer read
                sp = load_lane_masks(p, ws / 8, (we - ws + 7) / 8, sw);
            }
            uint32_t cnt = 0;
#pragma unroll
            for (int k = 0; k < kLaneWords; k++) cnt += __popc(sw[k * 32 + lane]);
            uint32_t incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            lexcl = incl - cnt;
            // Chunk starts inside this lane's words, in value offsets from s
            // (the lane's first word may begin up to 120 values before s).
            const int32_t lv0 = 8 * (int32_t)sp.a_first - (int32_t)s;
            const int32_t lv1 = lv0 + 32 * (int32_t)sp.nwords;
            uint32_t q = lv0 <= 0 ? 0 : ((uint32_t)lv0 + C - 1) / C;
            int32_t cs = (int32_t)(q * C);  // next chunk start
            uint32_t running = base + lexcl;
            for (int k = 0; k < (int)sp.nwords; k++) {
                const uint32_t word = sw[k * 32 + lane];
                const int32_t wv = lv0 + 32 * k;  // value offset of bit 0 of word k
                while (q < nq && cs < wv + 32 && cs < lv1) {
                    s_cp[q++] = running + __popc(word & ((1u << (cs - wv)) - 1));
                    cs += (int32_t)C;
                }
                running += __popc(word);
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
        const uint32_t rtotal = base;
        if (lane == 0) s_cp[nq] = rtotal;
        __syncwarp();

        uint8_t* offs = p.out + p.L.off_c;
        for (uint32_t q = lane; q < nq; q += 32)
            *reinterpret_cast<uint32_t*>(offs + 4ull * (c0 + q)) = (uint32_t)(pre + s_cp[q]);
        if (r == p.ranges - 1 && lane == 0) {
            const uint64_t m = pre + rtotal;
            *reinterpret_cast<uint32_t*>(offs + 4 * p.L.nc) = (uint32_t)m;
            zero_words(p.out, p.L.off_c + 4 * (p.L.nc + 1), p.L.off_d);
            const uint64_t groups_all = (p.n + 7) / 8;
            zero_words(p.out, p.L.off_a + 8 * groups_all, p.L.off_b);
            zero_words(p.out, p.L.off_b + 4 * groups_all, p.L.off_c);
            p.ws->m = m;
        }
        if (rtotal == 0) {
            __syncwarp();
            continue;
        }

        // Pass 2: escapes, ascending, kBatch exponent re-reads in flight per
        // lane. A single-window range still holds its masks in registers.
        const uint64_t dbase = p.L.off_d + 3 * pre;
        base = 0;
        for (uint32_t ws = s; ws < e; ws += kWinValues) {
            const uint32_t we = min(ws + kWinValues, e);
            uint32_t wtotal = rtotal;
            if (!one_window) {
                __syncwarp();
                sp = load_lane_masks(p, ws / 8, (we - ws + 7) / 8, sw);
                uint32_t cnt = 0;
#pragma unroll
                for (int k = 0; k < kLaneWords; k++) cnt += __popc(sw[k * 32 + lane]);
                uint32_t incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                lexcl = incl - cnt;
                wtotal = __shfl_sync(0xffffffffu, incl, 31);
            }
            const int32_t lv0 = 8 * (int32_t)sp.a_first - (int32_t)s;
            uint32_t running = base + lexcl;
            uint32_t q = lv0 <= 0 ? 0 : (uint32_t)lv0 / C;  // chunk of the lane's first value
            uint32_t next = (q + 1) * C;
            const int kend = (int)sp.nwords;
            int k = 0;
            uint32_t bits = kend > 0 ? sw[lane] : 0;
            for (;;) {
                uint32_t el[kBatch], qq[kBatch], rk[kBatch];
                int got = 0;
                while (got < kBatch && k < kend) {
                    if (bits == 0) {
                        if (++k >= kend) break;
                        bits = sw[k * 32 + lane];
                        continue;
                    }
                    const uint32_t off = (uint32_t)(lv0 + 32 * k + (__ffs(bits) - 1));  // value offset in the range
                    bits &= bits - 1;
                    while (off >= next) {
                        q++;
                        next += C;
                    }
#pragma unroll
                    for (int i = 0; i < kBatch; i++)
                        if (i == got) {
                            el[i] = s + off;
                            qq[i] = q;
                            rk[i] = running;
                        }
                    running++;
                    got++;
                }
                if (got == 0) break;
                uint32_t ex[kBatch];
#pragma unroll
                for (int i = 0; i < kBatch; i++) ex[i] = i < got ? (p.in[el[i]] >> 7) & 0xFF : 0;
#pragma unroll
                for (int i = 0; i < kBatch; i++) {
                    if (i < got) {
                        const uint32_t cstart = s_cp[qq[i]];
                        const uint32_t kk = s_cp[qq[i] + 1] - cstart;
                        const uint32_t rank = rk[i] - cstart;
                        const uint32_t pos = el[i] - (c0 + qq[i]) * C;
                        const uint64_t blk = dbase + 3ull * cstart;
                        const uint64_t o_pos = blk + 2ull * rank, o_val = blk + 2ull * kk + rank;
                        if (o_val < p.cap && o_pos + 1 < p.cap) {
                            p.out[o_pos] = (uint8_t)(pos & 0xFF);
                            p.out[o_pos + 1] = (uint8_t)(pos >> 8);
                            p.out[o_val] = (uint8_t)ex[i];
                        } else {
                            overflow = true;
                        }
                    }
                }
            }
            base += wtotal;
        }
        __syncwarp();  // s_cp is reused by this warp's next range
    }
    if (overflow) atomicOr(&p.ws->flags, UZIP_FLAG_CAPACITY);

    // The last CTA to finish writes the header.
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&p.ws->done, 1u);
        if (prev == gridDim.x - 1) {
            __threadfence();
            const uint64_t m = *reinterpret_cast<volatile unsigned long long*>(&p.ws->m);
            const uint32_t flags = *reinterpret_cast<volatile unsigned int*>(&p.ws->flags);
            write_header(p, m, flags);
        }
    }
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
    return (size_t)geometry_of(n, chunk).bytes;
}

namespace uzip {

int encode_impl(const void* d_in_bf16, size_t n, uint32_t chunk, const void* d_codebook, void* d_out,
                size_t out_capacity, void* d_workspace, size_t workspace_bytes, size_t* h_out_bytes,
                uzip_stream_t stream) {
    if (!chunk_valid(chunk)) return UZIP_ERR_CHUNK;
    if (n > UZIP_MAX_N || !d_out || !d_codebook || (n > 0 && !d_in_bf16) || !d_workspace) return UZIP_ERR_ARG;
    if (!aligned16(d_out) || !aligned16(d_codebook) || !aligned16(d_workspace) ||
        (n > 0 && !aligned16(d_in_bf16)))
        return UZIP_ERR_ALIGN;
    const Layout L = layout_of(n, chunk);
    if (out_capacity < L.off_d) return UZIP_ERR_CAPACITY;
    const Geometry g = geometry_of(n, chunk);
    if (workspace_bytes < g.bytes) return UZIP_ERR_CAPACITY;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    Params p;
    p.in = static_cast<const uint16_t*>(d_in_bf16);
    p.n = n;
    p.chunk = chunk;
    p.seg_units = g.seg_units;
    p.nseg = g.nseg;
    p.range_chunks = g.range_chunks;
    p.units = g.units;
    p.ranges = g.ranges;
    p.cb = static_cast<const uint8_t*>(d_codebook);
    p.out = static_cast<uint8_t*>(d_out);
    p.cap = out_capacity;
    p.L = L;
    p.ws = reinterpret_cast<WsHeader*>(ws);
    p.segs = reinterpret_cast<uint32_t*>(ws + g.off_segs);
    p.counts = reinterpret_cast<uint32_t*>(ws + g.off_counts);
    p.masks = ws + g.off_masks;

    if (n == 0) {
        encode_empty_kernel<<<1, 1, 0, s>>>(p);
        UZIP_CUDA_TRY(cudaGetLastError());
    } else {
        int dev = 0, sms = 0, per_sm1 = 0, per_sm2 = 0;
        UZIP_CUDA_TRY(cudaGetDevice(&dev));
        UZIP_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        const size_t smem2 = 4 * ((size_t)kWarps * kLaneWords * 32 + ((size_t)g.nseg + 1 + 3) / 4 * 4 +
                                  (size_t)kWarps * (g.range_chunks + 1));
        UZIP_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm1, encode_dense_kernel, kThreads, 0));
        UZIP_CUDA_TRY(
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm2, encode_escape_kernel, kThreads, smem2));
        if (per_sm1 < 1 || per_sm2 < 1) return UZIP_ERR_CUDA;
        const uint64_t grid1 = std::min<uint64_t>((g.units + kWarps - 1) / kWarps, (uint64_t)sms * per_sm1);
        const uint64_t grid2 = std::min<uint64_t>((g.ranges + kWarps - 1) / kWarps, (uint64_t)sms * per_sm2);
        UZIP_CUDA_TRY(cudaMemsetAsync(ws, 0, g.off_counts, s));  // header + segment totals
        encode_dense_kernel<<<(unsigned)grid1, kThreads, 0, s>>>(p);
        UZIP_CUDA_TRY(cudaGetLastError());
        encode_escape_kernel<<<(unsigned)grid2, kThreads, smem2, s>>>(p);
        UZIP_CUDA_TRY(cudaGetLastError());
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

// ------------------------------------------------- encoding without allocation
//
// Some callers cannot allocate device memory for the encoder's workspace:
// code running where a framework's caching allocator has already reserved the
// device memory and hands out no raw buffers, or latency-critical paths that
// must not call cudaMalloc (which can synchronise the device). For them the
// workspace lives in a file-scope device array, fixed at load time: every GPU
// that loads this library holds kNoAllocScratchBytes (about 8.1 MiB) of it
// until the process exits. Host code cannot use the array's name as a device
// address, so its address is looked up once per device with
// cudaGetSymbolAddress (on the first call on that device, with the device
// current) and passed to the same two kernels uzip_encode launches.

namespace uzip {
namespace {

constexpr uint64_t cpad16(uint64_t v) { return (v + 15) / 16 * 16; }

// Workspace bytes the encoder needs for n values (the geometry above, which
// depends on n only).
constexpr uint64_t workspace_bytes_for(uint64_t n) {
    const uint64_t units = (n + kUnit - 1) / kUnit;
    uint64_t seg_units = 64;
    while ((units + seg_units - 1) / seg_units > kMaxSegments) seg_units *= 2;
    const uint64_t nseg = (units + seg_units - 1) / seg_units;
    return sizeof(WsHeader) + cpad16(4 * nseg) + cpad16(4 * units) + cpad16((n + 7) / 8);
}

constexpr uint64_t kNoAllocScratchBytes = workspace_bytes_for(UZIP_NOALLOC_MAX_N);

constexpr int kMaxCachedDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxCachedDevices];

}  // namespace
}  // namespace uzip

static __device__ __align__(256) uint8_t g_noalloc_scratch[uzip::kNoAllocScratchBytes];

extern "C" UZIP_API int uzip_encode_noalloc(const void* d_in_bf16, size_t n, uint32_t chunk,
                                            const void* d_codebook, void* d_out, size_t out_capacity,
                                            size_t* h_out_bytes, uzip_stream_t stream) {
    if (n > UZIP_NOALLOC_MAX_N) return UZIP_ERR_CAPACITY;  // beyond the built-in scratch
    if (!chunk_valid(chunk)) return UZIP_ERR_CHUNK;
    const uint64_t need = geometry_of(n, chunk).bytes;
    if (need > kNoAllocScratchBytes) return UZIP_ERR_CAPACITY;
    int dev = 0;
    UZIP_CUDA_TRY(cudaGetDevice(&dev));
    void* scratch = dev < kMaxCachedDevices ? g_scratch_addr[dev].load(std::memory_order_acquire) : nullptr;
    if (!scratch) {
        UZIP_CUDA_TRY(cudaGetSymbolAddress(&scratch, g_noalloc_scratch));
        if (!scratch) return UZIP_ERR_CUDA;
        if (dev < kMaxCachedDevices) g_scratch_addr[dev].store(scratch, std::memory_order_release);
    }
    return encode_impl(d_in_bf16, n, chunk, d_codebook, d_out, out_capacity, scratch, (size_t)need, h_out_bytes,
                       stream);
}
