// calibrate.cu -- offline codebook calibration of the SplitZip codec.
//
// SplitZip review page, §3.3: extract every exponent of a representative
// sample, count them, keep the 16 most frequent and build three lookup tables
// (exponent -> 4-bit code, code -> exponent, exponent -> escape membership).
// §3.4: all 16 codes are real exponents; an escape gets a dummy code (0 here).
//
// Kernels:
//   calibrate_kernel  a sample of up to 4 Mi values: blocks of 256 threads,
//                     each thread issuing its two 16-byte loads first, then
//                     counting into its warp's 256-bin shared histogram (BF16:
//                     one shared atomic per value; E5M2, whose values crowd
//                     onto a few of 32 bins: equal exponents of a warp merged
//                     with __match_any_sync first); per-block totals are added
//                     to the blob's u64 histogram. The last block to finish (a
//                     fence and a counter, no waiting) compacts the bins seen,
//                     ranks each against the others (count descending, exponent
//                     ascending; unseen bins follow in exponent order), keeps
//                     the 16 lowest ranks as the codebook and writes the three
//                     tables.
//   histogram_private_kernel  larger inputs (whole tensors), below.
//   luts_kernel       the same tables from 16 caller-given exponents.
#include <algorithm>
#include <atomic>

#include "uzip_internal.cuh"

namespace uzip {
namespace {

constexpr int kHistThreads = 256;
constexpr int kHistWarps = kHistThreads / 32;

// One value into the warp's shared histogram. BF16 (256 bins): a plain
// shared-memory atomic per value (measured faster than merging equal
// exponents first). E5M2 (32 bins, values crowd onto a few of them): lanes
// holding the same exponent add once, with their count.
template <int kFmt>
__device__ __forceinline__ void warp_hist_add(uint32_t* h, uint32_t e, bool valid) {
    if (kFmt != kE5M2) {
        if (valid) atomicAdd(&h[e], 1u);
        return;
    }
    const uint32_t key = valid ? e : (0x100u | (threadIdx.x & 31));
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    if (valid && (__ffs(peers) - 1) == (int)(threadIdx.x & 31)) atomicAdd(&h[e], __popc(peers));
}

constexpr int kLoadsPerThread = 2;  // 16-byte loads in flight per thread

// Block-done counter of calibrate_kernel, in the blob's reserved bytes after
// the histogram; cleared with the histogram before each launch.
constexpr uint32_t kCbCounter = UZIP_CB_HIST + 256 * 8;

__device__ void rank_and_write(uint8_t* cb, uint64_t n_sample);

// kFmt: kBF16 (8 values per 16-byte load, exponent bits 14..7) or kE5M2 (16
// values per load, exponent bits 6..2 of each byte).
template <int kFmt>
__global__ void __launch_bounds__(kHistThreads) calibrate_kernel(const void* __restrict__ xv, uint64_t n,
                                                                 uint8_t* __restrict__ cb) {
    constexpr uint32_t kPerVec = kFmt == kE5M2 ? 16 : 8;
    __shared__ uint32_t sh[kHistWarps][256];
    __shared__ bool s_last;
    unsigned long long* hist = reinterpret_cast<unsigned long long*>(cb + UZIP_CB_HIST);
    unsigned int* counter = reinterpret_cast<unsigned int*>(cb + kCbCounter);
    for (int i = threadIdx.x; i < kHistWarps * 256; i += kHistThreads) (&sh[0][0])[i] = 0;
    __syncthreads();
    uint32_t* h = sh[threadIdx.x / 32];

    const uint64_t groups = n / kPerVec;
    const uint64_t stride = (uint64_t)gridDim.x * kHistThreads * kLoadsPerThread;
    // Group g of a round is lane + 32 * (warp + kHistWarps * (j + kLoadsPerThread * block)); the
    // trip count is warp-uniform so __match_any_sync always sees the full warp.
    const uint64_t first =
        ((uint64_t)blockIdx.x * kLoadsPerThread * kHistWarps + threadIdx.x / 32) * 32 + (threadIdx.x & 31);
    for (uint64_t base = 0; base < groups; base += stride) {
        uint4 v[kLoadsPerThread];
        bool valid[kLoadsPerThread];
#pragma unroll
        for (int j = 0; j < kLoadsPerThread; j++) {
            const uint64_t g = base + first + (uint64_t)j * kHistThreads;
            valid[j] = g < groups;
            v[j] = valid[j] ? ld_stream_v4(static_cast<const uint8_t*>(xv) + 16 * g) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kLoadsPerThread; j++) {
            const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int q = 0; q < 4; q++) {
                if (kFmt == kE5M2) {
#pragma unroll
                    for (int b = 0; b < 4; b++) warp_hist_add<kFmt>(h, (w[q] >> (8 * b + 2)) & 0x1F, valid[j]);
                } else {
                    warp_hist_add<kFmt>(h, (w[q] >> 7) & 0xFF, valid[j]);
                    warp_hist_add<kFmt>(h, (w[q] >> 23) & 0xFF, valid[j]);
                }
            }
        }
    }
    // Ragged tail (< kPerVec values): block 0's first warp.
    if (blockIdx.x == 0 && threadIdx.x < 32) {
        const uint64_t i = groups * kPerVec + threadIdx.x;
        const bool valid = i < n && threadIdx.x < kPerVec;
        uint32_t e = 0;
        if (valid)
            e = kFmt == kE5M2 ? (static_cast<const uint8_t*>(xv)[i] >> 2) & 0x1F
                              : (static_cast<const uint16_t*>(xv)[i] >> 7) & 0xFF;
        warp_hist_add<kFmt>(h, e, valid);
    }
    __syncthreads();
    pdl_wait();  // the blob's totals and counter are zeroed by the launch before this one
    for (int b = threadIdx.x; b < 256; b += kHistThreads) {
        uint32_t s = 0;
#pragma unroll
        for (int w = 0; w < kHistWarps; w++) s += sh[w][b];
        if (s) atomicAdd(&hist[b], (unsigned long long)s);
    }
    // The last block ranks the totals.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(counter, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    rank_and_write(cb, n);
    if (threadIdx.x == 0) *counter = 0;
}

// Histogram of a large input (a whole tensor): the warp-merged shared
// histogram above spends most of its time in __match_any_sync, so for large
// inputs each thread counts into private 16-bit counters instead: thread t
// owns word (e >> 1) * kPrivThreads + t for bins e and e ^ 1 (low and high
// half), 192 KB of shared memory for 384 threads, one CTA per SM. Every
// access of a lane falls in bank t mod 32, so no two lanes of a warp meet in
// a bank whatever exponents they hold, and no two threads share a word. A
// value adds 1 to its half with a shared-memory atomic whose result is not
// used, so counting is never a read-modify-write chain through the shared
// memory's latency. Every 65,408 values per thread (before a half can carry
// into the other) the block folds the counters into per-bin totals and
// clears them. The next round's 16 loads per thread are issued before the
// current round is counted; whole rounds load without bounds tests, and every
// loaded vector is counted: the last round's out-of-range vectors are loaded
// as zeros, counted into bin 0 like any zero, and their number is taken off
// bin 0's total once (no test per vector). The last block ranks, as above.
constexpr int kPrivThreads = 384;
constexpr int kPrivLoads = 16;
constexpr uint32_t kEpochValues = 65408;  // per thread between folds, + one tail value < 65536
constexpr size_t kPrivSmem = (size_t)128 * kPrivThreads * sizeof(uint32_t);
#ifndef UZIP_HIST_PRIVATE_FROM
#define UZIP_HIST_PRIVATE_FROM (1u << 22)
#endif
constexpr uint64_t kPrivateFrom = UZIP_HIST_PRIVATE_FROM;  // inputs at least this long use it

__device__ __forceinline__ void count_one(uint32_t* col, uint32_t e) {
    atomicAdd(col + (e >> 1) * kPrivThreads, 1u << (16 * (e & 1)));
}

// A BF16 value's row (bin pair) is its high byte without the sign, its half
// (the bin's low bit) its bit 7. The row's byte offset, row * 4 kPrivThreads =
// row * 256 * 6, is the value's masked high byte times 6, and the half's
// increment, 1 or 2^16, is 1 + half * 0xFFFF: both multiply-adds, beside the
// saturated ALU pipe.
static_assert(4 * kPrivThreads == 6 * 256, "the row stride is 6 times 256 bytes");
__device__ __forceinline__ void count_bf16_pair(uint32_t* col, uint32_t x) {  // the two values of word x
    char* c = reinterpret_cast<char*>(col);
    atomicAdd(reinterpret_cast<uint32_t*>(c + (x & 0x7F00u) * 6u), ((x >> 7) & 1u) * 0xFFFFu + 1u);
    atomicAdd(reinterpret_cast<uint32_t*>(c + ((x >> 16) & 0x7F00u) * 6u), ((x >> 23) & 1u) * 0xFFFFu + 1u);
}

template <int kFmt>
__global__ void __launch_bounds__(kPrivThreads, 1) histogram_private_kernel(const void* __restrict__ xv, uint64_t n,
                                                                            uint8_t* __restrict__ cb) {
    constexpr uint32_t kPerVec = kFmt == kE5M2 ? 16 : 8;
#ifdef UZIP_HIST_EPOCH_ROUNDS
    constexpr uint32_t kRoundsPerEpoch = UZIP_HIST_EPOCH_ROUNDS;  // shorter epochs (tests of the fold)
    static_assert((kRoundsPerEpoch + 1) * kPrivLoads * kPerVec <= kEpochValues, "16-bit counters");
#else
    // one round short of the counters' limit: the last round's padding is counted too
    constexpr uint32_t kRoundsPerEpoch = kEpochValues / (kPrivLoads * kPerVec) - 1;
#endif
    extern __shared__ uint4 s_dyn[];
    const uint32_t* cnt = reinterpret_cast<const uint32_t*>(s_dyn);  // [bin pair][thread]
    __shared__ bool s_last;
    unsigned long long* hist = reinterpret_cast<unsigned long long*>(cb + UZIP_CB_HIST);
    unsigned int* counter = reinterpret_cast<unsigned int*>(cb + kCbCounter);
    const int tid = threadIdx.x;
    uint32_t* col = reinterpret_cast<uint32_t*>(s_dyn) + tid;
    const uint8_t* x8 = static_cast<const uint8_t*>(xv);

    auto clear = [&]() {
        for (uint32_t i = tid; i < kPrivSmem / 16; i += kPrivThreads) s_dyn[i] = make_uint4(0, 0, 0, 0);
    };
    auto count_vec = [&](const uint4 v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            if (kFmt == kE5M2) {
#pragma unroll
                for (int b = 0; b < 4; b++) count_one(col, (w[q] >> (8 * b + 2)) & 0x1F);
            } else {  // two values per word: rows from bits 8..14 and 24..30, halves bits 7 and 23
                count_bf16_pair(col, w[q]);
            }
        }
    };
    uint32_t total = 0;  // thread t < 256: bin t's block total
    auto fold = [&]() {
        __syncthreads();
        if (tid < 256) {  // bin tid: half tid & 1 of row tid >> 1, read from a rotated start (no bank meets twice)
            const uint32_t* row = cnt + (tid >> 1) * kPrivThreads;
            const uint32_t sh = 16 * (tid & 1);
            uint32_t j = tid % kPrivThreads;
            for (int k = 0; k < kPrivThreads; k++) {
                total += (row[j] >> sh) & 0xFFFF;
                j = j + 1 == kPrivThreads ? 0 : j + 1;
            }
        }
        __syncthreads();
    };

    __shared__ uint32_t s_pad;  // zero values counted for the padding of partial rounds
    clear();
    if (tid == 0) s_pad = 0;
    __syncthreads();
    const uint64_t groups = n / kPerVec;
    if (blockIdx.x == 0 && (uint64_t)tid < n - groups * kPerVec) {  // ragged tail: one value per thread
        const uint64_t i = groups * kPerVec + tid;
        const uint32_t e = kFmt == kE5M2 ? (x8[i] >> 2) & 0x1F : (static_cast<const uint16_t*>(xv)[i] >> 7) & 0xFF;
        count_one(col, e);
    }
    const uint64_t per_round = (uint64_t)gridDim.x * kPrivThreads * kPrivLoads;
    const uint64_t rounds = (groups + per_round - 1) / per_round;
    uint32_t pad = 0;
    auto load_round = [&](uint64_t r, uint4* v) {
        const uint64_t base = (r * gridDim.x + blockIdx.x) * (uint64_t)kPrivThreads * kPrivLoads + tid;
        const uint4* src = reinterpret_cast<const uint4*>(x8) + base;
        if (base + (uint64_t)(kPrivLoads - 1) * kPrivThreads < groups) {  // a whole round
#pragma unroll
            for (int j = 0; j < kPrivLoads; j++) v[j] = ld_stream_v4(src + j * kPrivThreads);
        } else {
#pragma unroll
            for (int j = 0; j < kPrivLoads; j++) {
                const bool in = base + (uint64_t)j * kPrivThreads < groups;
                v[j] = in ? ld_stream_v4(src + j * kPrivThreads) : make_uint4(0, 0, 0, 0);
                pad += in ? 0u : kPerVec;  // counted as zeros below (bin 0), taken off at the end
            }
        }
    };
    auto count_round = [&](const uint4* v) {
#pragma unroll
        for (int j = 0; j < kPrivLoads; j++) count_vec(v[j]);
    };
    uint4 v[kPrivLoads], nv[kPrivLoads];
    if (rounds) load_round(0, v);
    for (uint64_t r0 = 0; r0 < rounds; r0 += kRoundsPerEpoch) {
        const uint64_t r1 = min(rounds, r0 + kRoundsPerEpoch);
        for (uint64_t r = r0; r < r1; r++) {  // the next round's loads in flight while one is counted
            if (r + 1 < rounds) load_round(r + 1, nv);
            count_round(v);
#pragma unroll
            for (int j = 0; j < kPrivLoads; j++) v[j] = nv[j];
        }
        if (r1 < rounds) {  // fold before a counter can overflow
            fold();
            clear();
            __syncthreads();
        }
    }
    if (pad) atomicAdd(&s_pad, pad);
    fold();
    if (tid == 0) total -= s_pad;  // bin 0: the padding's zeros (fold ends with a barrier)
    pdl_wait();  // the blob's totals and counter are zeroed by the launch before this one
    if (tid < 256 && total) atomicAdd(&hist[tid], (unsigned long long)total);
    // The last block ranks the totals.
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(counter, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    rank_and_write(cb, n);
    if (tid == 0) *counter = 0;
}

// Zero the blob's histogram totals and block counter. Its dependent (the
// histogram kernel) may launch at once: it waits for this grid only before
// its first update of the totals.
__global__ void __launch_bounds__(256) clear_hist_kernel(uint8_t* __restrict__ cb) {
    pdl_launch_dependents();
    uint4* z = reinterpret_cast<uint4*>(cb + UZIP_CB_HIST);
    for (uint32_t i = threadIdx.x; i < (kCbCounter + 16 - UZIP_CB_HIST) / 16; i += blockDim.x)
        z[i] = make_uint4(0, 0, 0, 0);
}

// Tables from exps[16] (shared memory), written by a 256-thread CTA.
__device__ void write_tables(const uint8_t* exps, uint8_t* cb, uint64_t n_sample) {
    const int t = threadIdx.x;
    if (t >= 256) return;
    uint8_t code = 0, esc = 1;
#pragma unroll
    for (int k = 0; k < 16; k++)
        if (exps[k] == t) {
            code = (uint8_t)k;
            esc = 0;
        }
    cb[UZIP_CB_ENC + t] = code;
    cb[UZIP_CB_ESC + t] = esc;
    if (t < 16) {
        cb[UZIP_CB_EXPS + t] = exps[t];
        cb[UZIP_CB_DEC + t] = exps[t];
    }
    if (t == 0) {
        reinterpret_cast<uint32_t*>(cb)[0] = kCodebookMagic;
        reinterpret_cast<uint32_t*>(cb)[1] = 1;
        reinterpret_cast<uint64_t*>(cb)[1] = n_sample;
    }
}

// Rank the blob's 256 totals (count descending, exponent ascending) and write
// the codebook; the first 256 threads of the CTA, totals read from L2. The
// bins with a nonzero count are compacted first (in exponent order), so each
// of them is ranked against the nonzero bins only; a bin never seen ranks
// after all of them, in exponent order.
__device__ void rank_and_write(uint8_t* cb, uint64_t n_sample) {
    __shared__ unsigned long long nz_cnt[256];
    __shared__ uint32_t s_nz[8];
    __shared__ uint8_t exps[16];
    const int t = threadIdx.x;
    const unsigned long long* hist = reinterpret_cast<const unsigned long long*>(cb + UZIP_CB_HIST);
    const unsigned long long mine = t < 256 ? __ldcg(hist + t) : 0ull;
    const uint32_t lane = t & 31, warp = t >> 5;
    const uint32_t nzb = __ballot_sync(0xffffffffu, mine != 0);
    if (t < 256 && lane == 0) s_nz[warp] = __popc(nzb);
    __syncthreads();
    uint32_t pos = __popc(nzb & ((1u << lane) - 1)), nnz = 0;
#pragma unroll
    for (int w = 0; w < 8; w++) {
        pos += w < (int)warp ? s_nz[w] : 0u;
        nnz += s_nz[w];
    }
    if (t < 256 && mine) nz_cnt[pos] = mine;
    __syncthreads();
    if (t < 256) {
        uint32_t rank;
        if (mine) {
            rank = 0;
            for (uint32_t k = 0; k < nnz; k++) {
                const unsigned long long c = nz_cnt[k];
                rank += (c > mine) || (c == mine && k < pos);
            }
        } else {
            rank = nnz + ((uint32_t)t - pos);  // unseen: after every seen bin, in exponent order
        }
        if (rank < 16) exps[rank] = (uint8_t)t;
    }
    __syncthreads();
    write_tables(exps, cb, n_sample);
}

struct Exps16 {
    uint8_t v[16];
};

__global__ void __launch_bounds__(256) luts_kernel(Exps16 in, uint8_t* __restrict__ cb) {
    __shared__ uint8_t exps[16];
    if (threadIdx.x < 16) exps[threadIdx.x] = in.v[threadIdx.x];
    unsigned long long* hist = reinterpret_cast<unsigned long long*>(cb + UZIP_CB_HIST);
    hist[threadIdx.x] = 0;
    __syncthreads();
    write_tables(exps, cb, 0);
}

}  // namespace
}  // namespace uzip

using namespace uzip;

namespace uzip {
namespace {

// SM count and the histogram kernel's residency (BF16, E5M2) per device,
// looked up on the first call on that device (0 = not yet).
constexpr int kMaxCachedDevices = 64;
std::atomic<int> g_sms[kMaxCachedDevices];
std::atomic<int> g_per_sm[kMaxCachedDevices][2];

}  // namespace

int calibrate_impl(const void* d_sample_bf16, size_t n_sample, void* d_codebook, cudaStream_t s, uint32_t fmt) {
    if (!d_codebook || (n_sample > 0 && !d_sample_bf16)) return UZIP_ERR_ARG;
    if (!aligned16(d_codebook) || (n_sample > 0 && !aligned16(d_sample_bf16))) return UZIP_ERR_ALIGN;
    uint8_t* cb = static_cast<uint8_t*>(d_codebook);
    // Histogram totals and the block counter start at zero: a one-block
    // kernel clears them and the histogram kernel launches behind it at once.
    clear_hist_kernel<<<1, 256, 0, s>>>(cb);
    UZIP_CUDA_TRY(cudaGetLastError());
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    int dev = 0;
    UZIP_CUDA_TRY(cudaGetDevice(&dev));
    const bool cached = dev < kMaxCachedDevices;
    const int slot = fmt == kE5M2 ? 1 : 0;
    int sms = cached ? g_sms[dev].load() : 0, per_sm = cached ? g_per_sm[dev][slot].load() : 0;
    if (sms < 1) {
        UZIP_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        if (cached) g_sms[dev].store(sms);
    }
    if (n_sample >= kPrivateFrom) {  // a large input: private-column histogram, one CTA per SM
        auto* pk = fmt == kE5M2 ? histogram_private_kernel<kE5M2> : histogram_private_kernel<kBF16>;
        UZIP_CUDA_TRY(cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrivSmem));
        cfg.gridDim = dim3((unsigned)sms);
        cfg.blockDim = dim3(kPrivThreads);
        cfg.dynamicSmemBytes = kPrivSmem;
        UZIP_CUDA_TRY(cudaLaunchKernelEx(&cfg, pk, d_sample_bf16, (uint64_t)n_sample, cb));
        return UZIP_OK;
    }
    auto* kernel = fmt == kE5M2 ? calibrate_kernel<kE5M2> : calibrate_kernel<kBF16>;
    if (per_sm < 1) {
        UZIP_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kHistThreads, 0));
        if (cached && per_sm > 0) g_per_sm[dev][slot].store(per_sm);
    }
    // One block per kHistThreads * kLoadsPerThread 16-byte loads, up to a
    // full resident wave: a small sample is a latency chain, a whole tensor
    // is read at HBM speed.
    const uint64_t per_block = (uint64_t)kHistThreads * kLoadsPerThread * (fmt == kE5M2 ? 16 : 8);
    uint64_t blocks = (n_sample + per_block - 1) / per_block;
    blocks = std::min<uint64_t>(blocks, (uint64_t)sms * std::max(per_sm, 1));
    if (blocks == 0) blocks = 1;
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kHistThreads);
    UZIP_CUDA_TRY(cudaLaunchKernelEx(&cfg, kernel, d_sample_bf16, (uint64_t)n_sample, cb));
    return UZIP_OK;
}

}  // namespace uzip

extern "C" UZIP_API int uzip_calibrate(const void* d_sample_bf16, size_t n_sample, void* d_codebook,
                                       uzip_stream_t stream) {
    return calibrate_impl(d_sample_bf16, n_sample, d_codebook, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" UZIP_API int uzip_e5m2_calibrate(const void* d_sample_e5m2, size_t n_sample, void* d_codebook,
                                            uzip_stream_t stream) {
    return calibrate_impl(d_sample_e5m2, n_sample, d_codebook, reinterpret_cast<cudaStream_t>(stream), kE5M2);
}

namespace uzip {
namespace {

// Top-15 + sentinel tables from a codebook's exponents (page §3.4, Table 6):
// codes 0..14 for exps[0..14], code 15 for every other exponent (an escape),
// decode-table entry 15 = 0, blob version 2.
__global__ void __launch_bounds__(256) sentinel_tables_kernel(uint8_t* __restrict__ cb) {
    __shared__ uint8_t exps[16];
    const int t = threadIdx.x;
    if (t < 16) exps[t] = cb[UZIP_CB_EXPS + t];
    __syncthreads();
    uint8_t code = 15, esc = 1;
#pragma unroll
    for (int k = 0; k < 15; k++)
        if (exps[k] == t) {
            code = (uint8_t)k;
            esc = 0;
        }
    cb[UZIP_CB_ENC + t] = code;
    cb[UZIP_CB_ESC + t] = esc;
    if (t < 16) cb[UZIP_CB_DEC + t] = t < 15 ? exps[t] : 0;
    if (t == 0) reinterpret_cast<uint32_t*>(cb)[1] = 2;
}

}  // namespace
}  // namespace uzip

extern "C" UZIP_API int uzip_codebook_make_sentinel(void* d_codebook, uzip_stream_t stream) {
    if (!d_codebook) return UZIP_ERR_ARG;
    if (!aligned16(d_codebook)) return UZIP_ERR_ALIGN;
    sentinel_tables_kernel<<<1, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<uint8_t*>(d_codebook));
    UZIP_CUDA_TRY(cudaGetLastError());
    return UZIP_OK;
}

extern "C" UZIP_API int uzip_codebook_from_exps(const uint8_t* h_exps16, void* d_codebook,
                                                uzip_stream_t stream) {
    if (!h_exps16 || !d_codebook) return UZIP_ERR_ARG;
    if (!aligned16(d_codebook)) return UZIP_ERR_ALIGN;
    Exps16 e;
    bool seen[256] = {false};
    for (int k = 0; k < 16; k++) {
        if (seen[h_exps16[k]]) return UZIP_ERR_ARG;
        seen[h_exps16[k]] = true;
        e.v[k] = h_exps16[k];
    }
    luts_kernel<<<1, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(e, static_cast<uint8_t*>(d_codebook));
    UZIP_CUDA_TRY(cudaGetLastError());
    return UZIP_OK;
}
