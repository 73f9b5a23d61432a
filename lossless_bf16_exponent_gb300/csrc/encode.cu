// encode.cu -- fused single-pass SplitZip encoder for sm_103a.
//
// SplitZip review page, §3.2: encoding is (1) a dense transform -- split each
// BF16 value into its exponent and sign-mantissa byte, store the latter
// verbatim, map the exponent through the Top-16 code table and pack two 4-bit
// codes per byte -- and (2) a scan of the exponent stream that pushes every
// exponent outside the Top-16 into chunked escape position / value arrays.
// Appendix A (Quad64): both stages fused into one kernel over wide words; here
// each thread moves 16-byte vectors (eight values) instead of 64-bit words.
//
// One CTA encodes one "unit": a run of whole chunks (about 8192 values; one
// chunk when the chunk is longer, walked in 8192-value sub-tiles). Unit ids
// come from an atomic ticket, so a unit's predecessors are always held by CTAs
// that already run. Per unit:
//   dense   16-byte loads -> exponent / sign-mantissa bytes with byte permutes
//           -> code + escape bit from a 256-byte shared table -> 8-byte
//           sign-mantissa store + 4-byte code store, both coalesced; an 8-bit
//           escape mask per group of eight values goes to shared memory.
//   count   each thread sums the escape masks of a contiguous run of groups; a
//           block scan gives every run's escape rank inside the unit and every
//           chunk's first rank.
//   scan    decoupled look-back (one warp, 32 predecessors per step) over
//           64-bit unit descriptors {flag, count}: the unit publishes its
//           aggregate at once, sums predecessors' aggregates until it meets an
//           inclusive prefix, then publishes its own inclusive prefix. Every
//           wait is bounded by a time limit; running out sets a header flag.
//   write   chunk offsets (u32), then each escape: its chunk-relative position
//           into the chunk's position array and its raw exponent (re-read from
//           the input, which is still in L2) into the chunk's value array, in
//           ascending element order. Writes past out_capacity are dropped and
//           flagged.
//   finish  the last CTA to finish writes the 64-byte header and the padding.
#include "uzip_internal.cuh"

namespace uzip {
namespace {

constexpr int kThreads = 256;
constexpr int kGroupsPerThread = 4;                        // 16-byte groups per thread per sub-tile
constexpr int kSubGroups = kThreads * kGroupsPerThread;    // 1024 groups
constexpr uint32_t kSubElems = kSubGroups * 8;             // 8192 values

constexpr uint64_t kFlagAgg = 1ull << 62;
constexpr uint64_t kFlagInc = 2ull << 62;
constexpr uint64_t kValMask = (1ull << 62) - 1;

// Start of the caller's workspace; the unit descriptors follow at +64.
struct Workspace {
    unsigned int ticket;
    unsigned int done;
    unsigned int flags;
    unsigned int pad0;
    unsigned long long m;
    unsigned long long pad1[5];
};
static_assert(sizeof(Workspace) == 64, "workspace header is 64 bytes");

struct Geometry {
    uint32_t chunks_per_unit;  // whole chunks in a full unit
    uint32_t unit_elems;       // values in a full unit
    uint64_t units;
};

__host__ Geometry geometry_of(uint64_t n, uint32_t chunk) {
    Geometry g;
    g.chunks_per_unit = chunk <= kSubElems ? kSubElems / chunk : 1;
    g.unit_elems = g.chunks_per_unit * chunk;
    g.units = (n + g.unit_elems - 1) / g.unit_elems;
    return g;
}

struct Params {
    const uint16_t* in;
    uint64_t n;
    uint32_t chunk;
    uint32_t unit_elems;
    uint64_t units;
    const uint8_t* cb;
    uint8_t* out;
    uint64_t cap;
    Layout L;
    Workspace* ws;
    unsigned long long* desc;
    uint64_t timeout_ns;
    uint32_t withhold_first;  // failure-injection: unit 0 never publishes
};

// Eight values -> 8 sign-mantissa bytes (a_lo, a_hi), 8 packed codes (one
// word, value i in nibble i) and an 8-bit escape mask.
__device__ __forceinline__ void encode_group(const uint4 v, const uint8_t* tab, uint32_t& a_lo,
                                             uint32_t& a_hi, uint32_t& codes, uint32_t& mask) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed[2], esc[2];
#pragma unroll
    for (int h = 0; h < 2; h++) {
        // Bytes of four values: high bytes (sign + exponent bits 7..1) and
        // low bytes (exponent bit 0 + mantissa).
        const uint32_t hi = prmt(w[2 * h], w[2 * h + 1], 0x7531);
        const uint32_t lo = prmt(w[2 * h], w[2 * h + 1], 0x6420);
        const uint32_t e4 = ((hi << 1) & 0xFEFEFEFEu) | ((lo >> 7) & 0x01010101u);
        const uint32_t a4 = (hi & 0x80808080u) | (lo & 0x7F7F7F7Fu);
        if (h == 0) a_lo = a4; else a_hi = a4;
        // Table byte = code | escape << 7.
        const uint32_t t0 = tab[e4 & 0xFF];
        const uint32_t t1 = tab[(e4 >> 8) & 0xFF];
        const uint32_t t2 = tab[(e4 >> 16) & 0xFF];
        const uint32_t t3 = tab[e4 >> 24];
        const uint32_t t4 = t0 | (t1 << 8) | (t2 << 16) | (t3 << 24);
        const uint32_t c = t4 & 0x0F0F0F0Fu;
        packed[h] = c | (c >> 4);  // byte 0 = c0 | c1 << 4, byte 2 = c2 | c3 << 4
        esc[h] = t4 & 0x80808080u;
    }
    codes = prmt(packed[0], packed[1], 0x6420);
    // Bit 7 of byte i -> bit i (the four shifted copies never overlap).
    const uint32_t m_lo = (((esc[0] >> 7) * 0x204081u) >> 21) & 0xF;
    const uint32_t m_hi = (((esc[1] >> 7) * 0x204081u) >> 21) & 0xF;
    mask = m_lo | (m_hi << 4);
}

__device__ __forceinline__ void block_exclusive_scan(uint32_t v, uint32_t& excl, uint32_t& total,
                                                     uint32_t* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; w++) {
        const uint32_t s = s_warp[w];
        before += (w < warp) ? s : 0;
        all += s;
    }
    excl = before + incl - v;
    total = all;
}

// Decoupled look-back by warp 0; returns the unit's exclusive escape prefix.
__device__ uint64_t lookback(const Params& p, uint64_t u, uint32_t total) {
    const int lane = threadIdx.x & 31;
    if (u == 0) {
        if (lane == 0 && !p.withhold_first) st_relaxed_u64(p.desc, kFlagInc | total);
        return 0;
    }
    if (lane == 0) st_relaxed_u64(p.desc + u, kFlagAgg | total);
    uint64_t prefix = 0;
    int64_t nearest = (int64_t)u - 1;
    const uint64_t t0 = globaltimer_ns();
    bool timed_out = false;
    for (;;) {
        const int64_t idx = nearest - lane;
        uint64_t d;
        for (;;) {
            d = idx >= 0 ? ld_relaxed_u64(p.desc + idx) : kFlagInc;
            if (!__any_sync(0xffffffffu, (d >> 62) == 0)) break;
            if (__any_sync(0xffffffffu, globaltimer_ns() - t0 > p.timeout_ns)) {
                timed_out = true;
                break;
            }
            __nanosleep(32);
        }
        if (timed_out) break;
        const uint32_t inc = __ballot_sync(0xffffffffu, (d >> 62) == 2);
        const int stop = inc ? __ffs(inc) - 1 : 31;
        uint64_t val = lane <= stop ? (d & kValMask) : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) val += __shfl_xor_sync(0xffffffffu, val, o);
        prefix += val;
        if (inc) break;
        nearest -= 32;
    }
    if (lane == 0) {
        if (timed_out) atomicOr(&p.ws->flags, UZIP_FLAG_TIMEOUT);
        st_relaxed_u64(p.desc + u, kFlagInc | ((prefix + total) & kValMask));
    }
    return prefix;
}

__device__ __forceinline__ void put_byte(const Params& p, uint64_t off, uint8_t v, bool& overflow) {
    if (off < p.cap) p.out[off] = v;
    else overflow = true;
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

__global__ void __launch_bounds__(kThreads) encode_kernel(const Params p) {
    extern __shared__ __align__(16) uint8_t dyn[];
    __shared__ uint32_t s_tab_words[64];
    __shared__ uint32_t s_warp[kThreads / 32];
    __shared__ unsigned long long s_unit, s_prefix;

    const int tid = threadIdx.x;
    uint8_t* s_tab = reinterpret_cast<uint8_t*>(s_tab_words);
    uint8_t* s_mask = dyn;
    uint32_t* s_cpref = reinterpret_cast<uint32_t*>(dyn + pad16(p.unit_elems / 8));

    if (tid == 0) s_unit = atomicAdd(&p.ws->ticket, 1u);
    s_tab[tid] = p.cb[UZIP_CB_ENC + tid] | (p.cb[UZIP_CB_ESC + tid] ? 0x80 : 0);
    __syncthreads();

    const uint64_t u = s_unit;
    const uint64_t ubase = u * p.unit_elems;
    const uint32_t ulen = (uint32_t)min((uint64_t)p.unit_elems, p.n - ubase);
    const uint32_t ugroups = (ulen + 7) / 8;
    const uint4* in4 = reinterpret_cast<const uint4*>(p.in);

    // ---------------------------------------------------------------- dense
    for (uint32_t g0 = 0; g0 < ugroups; g0 += kSubGroups) {
        uint4 v[kGroupsPerThread];
#pragma unroll
        for (int r = 0; r < kGroupsPerThread; r++) {
            const uint32_t g = g0 + tid + r * kThreads;
            const uint64_t e0 = ubase + 8ull * g;
            v[r] = make_uint4(0, 0, 0, 0);
            if (g < ugroups) {
                if (e0 + 8 <= p.n) {
                    v[r] = ld_stream_v4(in4 + (e0 >> 3));
                } else {
                    uint32_t w[4] = {0, 0, 0, 0};
                    for (uint32_t i = 0; e0 + i < p.n; i++) w[i / 2] |= (uint32_t)p.in[e0 + i] << (16 * (i & 1));
                    v[r] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kGroupsPerThread; r++) {
            const uint32_t g = g0 + tid + r * kThreads;
            if (g >= ugroups) continue;
            const uint64_t e0 = ubase + 8ull * g;
            uint32_t a_lo, a_hi, codes, mask;
            encode_group(v[r], s_tab, a_lo, a_hi, codes, mask);
            if (e0 + 8 > p.n) {  // ragged tail: codes and escapes of real values only
                const uint32_t valid = (uint32_t)(p.n - e0);
                mask &= (1u << valid) - 1;
                codes &= (1u << (4 * valid)) - 1;
            }
            *reinterpret_cast<uint2*>(p.out + p.L.off_a + e0) = make_uint2(a_lo, a_hi);
            *reinterpret_cast<uint32_t*>(p.out + p.L.off_b + e0 / 2) = codes;
            s_mask[g] = (uint8_t)mask;
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- count
    const uint32_t run = (ugroups + kThreads - 1) / kThreads;
    const uint32_t gbeg = min(tid * run, ugroups), gend = min(gbeg + run, ugroups);
    uint32_t cnt = 0;
    for (uint32_t g = gbeg; g < gend; g++) cnt += __popc(s_mask[g]);
    uint32_t excl, total;
    block_exclusive_scan(cnt, excl, total, s_warp);
    {
        uint32_t running = excl;
        for (uint32_t g = gbeg; g < gend; g++) {
            const uint32_t el = 8 * g;
            if (el % p.chunk == 0) s_cpref[el / p.chunk] = running;
            running += __popc(s_mask[g]);
        }
    }
    const uint32_t uchunks = (ulen + p.chunk - 1) / p.chunk;
    if (tid == 0) s_cpref[uchunks] = total;

    // ----------------------------------------------------------------- scan
    if (tid < 32) {
        const uint64_t prefix = lookback(p, u, total);
        if (tid == 0) s_prefix = prefix;
    }
    __syncthreads();
    const uint64_t prefix = s_prefix;

    // ---------------------------------------------------------------- write
    const uint64_t c0 = ubase / p.chunk;
    uint8_t* offs = p.out + p.L.off_c;
    for (uint32_t ci = tid; ci < uchunks; ci += kThreads)
        *reinterpret_cast<uint32_t*>(offs + 4 * (c0 + ci)) = (uint32_t)(prefix + s_cpref[ci]);
    const bool last_unit = (u == p.units - 1);
    if (last_unit && tid == 0) {
        const uint64_t m = prefix + total;
        *reinterpret_cast<uint32_t*>(offs + 4 * p.L.nc) = (uint32_t)m;
        zero_words(p.out, p.L.off_c + 4 * (p.L.nc + 1), p.L.off_d);
        const uint64_t groups_all = (p.n + 7) / 8;
        zero_words(p.out, p.L.off_a + 8 * groups_all, p.L.off_b);
        zero_words(p.out, p.L.off_b + 4 * groups_all, p.L.off_c);
        p.ws->m = m;
    }
    bool overflow = false;
    if (total) {
        uint32_t running = excl;
        const uint64_t dbase = p.L.off_d + 3 * prefix;
        for (uint32_t g = gbeg; g < gend; g++) {
            uint32_t m8 = s_mask[g];
            while (m8) {
                const uint32_t b = __ffs(m8) - 1;
                m8 &= m8 - 1;
                const uint32_t el = 8 * g + b;
                const uint32_t ci = el / p.chunk;
                const uint32_t pos = el - ci * p.chunk;
                const uint32_t cstart = s_cpref[ci];
                const uint32_t k = s_cpref[ci + 1] - cstart;
                const uint32_t rank = running - cstart;
                const uint8_t e = (uint8_t)((p.in[ubase + el] >> 7) & 0xFF);
                const uint64_t blk = dbase + 3ull * cstart;
                put_byte(p, blk + 2ull * rank, (uint8_t)(pos & 0xFF), overflow);
                put_byte(p, blk + 2ull * rank + 1, (uint8_t)(pos >> 8), overflow);
                put_byte(p, blk + 2ull * k + rank, e, overflow);
                running++;
            }
        }
    }
    if (overflow) atomicOr(&p.ws->flags, UZIP_FLAG_CAPACITY);

    // --------------------------------------------------------------- finish
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&p.ws->done, 1u);
        if (prev == (unsigned)(p.units - 1)) {
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
    const Geometry g = geometry_of(n, chunk);
    return sizeof(Workspace) + 8 * (size_t)g.units;
}

namespace uzip {

int encode_impl(const void* d_in_bf16, size_t n, uint32_t chunk, const void* d_codebook, void* d_out,
                size_t out_capacity, void* d_workspace, size_t workspace_bytes, size_t* h_out_bytes,
                uzip_stream_t stream, uint64_t timeout_ns, uint32_t withhold_first) {
    if (!chunk_valid(chunk)) return UZIP_ERR_CHUNK;
    if (n > UZIP_MAX_N || !d_out || !d_codebook || (n > 0 && !d_in_bf16) || !d_workspace) return UZIP_ERR_ARG;
    if (!aligned16(d_out) || !aligned16(d_codebook) || !aligned16(d_workspace) ||
        (n > 0 && !aligned16(d_in_bf16)))
        return UZIP_ERR_ALIGN;
    const Layout L = layout_of(n, chunk);
    if (out_capacity < L.off_d) return UZIP_ERR_CAPACITY;
    const size_t ws_need = uzip_encode_workspace_bytes(n, chunk);
    if (workspace_bytes < ws_need) return UZIP_ERR_CAPACITY;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const Geometry g = geometry_of(n, chunk);
    Params p;
    p.in = static_cast<const uint16_t*>(d_in_bf16);
    p.n = n;
    p.chunk = chunk;
    p.unit_elems = g.unit_elems;
    p.units = g.units;
    p.cb = static_cast<const uint8_t*>(d_codebook);
    p.out = static_cast<uint8_t*>(d_out);
    p.cap = out_capacity;
    p.L = L;
    p.ws = static_cast<Workspace*>(d_workspace);
    p.desc = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(d_workspace) + sizeof(Workspace));
    p.timeout_ns = timeout_ns;
    p.withhold_first = withhold_first;

    if (n == 0) {
        encode_empty_kernel<<<1, 1, 0, s>>>(p);
        UZIP_CUDA_TRY(cudaGetLastError());
    } else {
        UZIP_CUDA_TRY(cudaMemsetAsync(d_workspace, 0, ws_need, s));
        const size_t smem = pad16(g.unit_elems / 8) + 4 * (size_t)(g.chunks_per_unit + 1);
        encode_kernel<<<(unsigned)g.units, kThreads, smem, s>>>(p);
        UZIP_CUDA_TRY(cudaGetLastError());
    }
    if (h_out_bytes) {
        uint32_t hdr[16];
        UZIP_CUDA_TRY(cudaMemcpyAsync(hdr, d_out, sizeof(hdr), cudaMemcpyDeviceToHost, s));
        UZIP_CUDA_TRY(cudaStreamSynchronize(s));
        *h_out_bytes = (size_t)hdr[12] | ((size_t)hdr[13] << 32);
        const uint32_t flags = hdr[1] >> 16;
        if (flags & UZIP_FLAG_TIMEOUT) return UZIP_ERR_TIMEOUT;
        if (flags & UZIP_FLAG_CAPACITY) return UZIP_ERR_CAPACITY;
    }
    return UZIP_OK;
}

}  // namespace uzip

extern "C" UZIP_API int uzip_encode(const void* d_in_bf16, size_t n, uint32_t chunk, const void* d_codebook,
                                    void* d_out, size_t out_capacity, void* d_workspace, size_t workspace_bytes,
                                    size_t* h_out_bytes, uzip_stream_t stream) {
    return encode_impl(d_in_bf16, n, chunk, d_codebook, d_out, out_capacity, d_workspace, workspace_bytes,
                       h_out_bytes, stream, kDefaultTimeoutNs, 0);
}
