// sz_histogram.cu -- exponent histogram and top-16 selection (calibration).
//
// The codebook is calibrated once, offline, from the exponent counts of a
// sample (SplitZip abstract, arXiv 2605.01708v2: an offline top-16 codebook
// removes online histogramming; technical summary, gist.science/es,
// "Resultados" > "Estudios de Ablacion" > "Calibracion").  The histogram can
// also be taken on the device per tensor, and the top-16 chosen there too
// (select_kernel), so that an encode can follow without a trip to the host;
// the ablation's price of such dynamic calibration is then measurable.
//
// The sample is made of whole 128-byte lines of the tensor (64 BF16 or 128
// E5M2 elements): with stride s, one line out of every run of s lines, at a
// hashed position in the run, so that a sparse sample costs 1/s of the DRAM
// traffic (a line is what one memory access fetches) and does not alias with
// the tensor's periodic layout (a fixed offset would always land on the same
// heads and channels).  Counts go into columns of a shared table, one column
// per lane (BF16: 256 bins x 32 columns) or per thread (E5M2: 32 bins x 256
// columns), so that the 32 lanes of one atomic never hit the same word or
// bank however few bins the exponents crowd into; the block adds its columns
// to the global counts at the end.
#include "sz_device.cuh"
#include "sz_params.h"

namespace sz {

namespace {
constexpr uint32_t kHistThreads = 256;
constexpr uint32_t kSelThreads = 256;
constexpr uint32_t kLineBytes = 128;             // the sample's unit
constexpr uint32_t kPieces = kLineBytes / 16;    // 16-byte pieces per line

// lowbias32 (C. Wellons, "hash-prospector"): a 32-bit integer hash.
__device__ __forceinline__ uint32_t lowbias32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

// The line that run w contributes: runs are `stride` lines long (the last
// one may be shorter, len lines), and the line sits at offset
// floor(lowbias32(w) * len / 2^32) of its run (multiply-shift range
// reduction).  Stride 1 takes every line.
__device__ __forceinline__ uint64_t sampled_line(uint32_t w, uint32_t stride, uint64_t lines) {
    const uint64_t first = (uint64_t)w * stride;
    if (stride == 1) return first;
    const uint64_t left = lines - first;
    const uint64_t len = left < stride ? left : stride;
    return first + (((uint64_t)lowbias32(w) * len) >> 32);
}

// Piece q (16 bytes) of a line as four words; returns its element count
// (BF16: up to 8, E5M2: up to 16; fewer at the end of the tensor).
template <bool BF16>
__device__ __forceinline__ uint32_t load_piece(const HistogramParams& p, bool vec, uint64_t line, uint32_t q,
                                               uint32_t (&w)[4]) {
    constexpr uint32_t kPer = BF16 ? 8u : 16u;
    const uint64_t e0 = line * (kLineBytes / (BF16 ? 2 : 1)) + q * kPer;
    w[0] = w[1] = w[2] = w[3] = 0;
    if (e0 >= p.n) return 0;
    const uint32_t cnt = p.n - e0 >= kPer ? kPer : (uint32_t)(p.n - e0);
    const uint8_t* src = p.in + e0 * (BF16 ? 2 : 1);
    if (vec && cnt == kPer) {
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
    } else {  // byte loads into two 64-bit halves (static register indexing)
        uint64_t lo = 0, hi = 0;
        const uint32_t bytes = cnt * (BF16 ? 2u : 1u);
        for (uint32_t j = 0; j < bytes; j++) {
            const uint64_t b = src[j];
            if (j < 8) lo |= b << (8 * j);
            else hi |= b << (8 * (j - 8));
        }
        w[0] = (uint32_t)lo, w[1] = (uint32_t)(lo >> 32), w[2] = (uint32_t)hi, w[3] = (uint32_t)(hi >> 32);
    }
    return cnt;
}
}  // namespace

// U: pieces each thread loads before it counts any (more loads in flight
// when the sample is sparse).
template <bool BF16, uint32_t U>
__global__ void __launch_bounds__(kHistThreads) histogram_kernel(const HistogramParams p) {
    constexpr uint32_t kBins = BF16 ? 256u : 32u;
    constexpr uint32_t kCols = BF16 ? 32u : kHistThreads;  // 32 KB either way
    constexpr uint32_t kPer = BF16 ? 8u : 16u;             // elements per piece
    __shared__ uint32_t s_hist[kBins * kCols];               // bin b, column c at b * kCols + c
    __shared__ unsigned long long s_part[kHistThreads];
    const uint32_t tid = threadIdx.x;
    for (uint32_t b = tid; b < kBins * kCols; b += kHistThreads) s_hist[b] = 0;
    __syncthreads();
    const uint64_t lines = (p.n * (BF16 ? 2 : 1) + kLineBytes - 1) / kLineBytes;
    const uint64_t pieces = (lines + p.stride - 1) / p.stride * kPieces;  // kPieces per run
    const uint64_t step = (uint64_t)gridDim.x * kHistThreads;
    const bool vec = (reinterpret_cast<uintptr_t>(p.in) % 16) == 0;
    uint32_t* h = s_hist + tid % kCols;
    for (uint64_t q0 = (uint64_t)blockIdx.x * kHistThreads + tid; q0 < pieces; q0 += U * step) {
        uint32_t w[U][4], cnt[U];
#pragma unroll
        for (uint32_t u = 0; u < U; u++) {
            const uint64_t q = q0 + u * step;
            cnt[u] = q < pieces ? load_piece<BF16>(p, vec, sampled_line((uint32_t)(q / kPieces), p.stride, lines),
                                                   (uint32_t)(q % kPieces), w[u])
                                : 0u;
        }
#pragma unroll
        for (uint32_t u = 0; u < U; u++) {
#pragma unroll
            for (uint32_t j = 0; j < kPer; j++) {
                if (j < cnt[u]) {
                    const uint32_t e = BF16 ? (w[u][j >> 1] >> (7 + 16 * (j & 1))) & 0xFFu
                                            : (w[u][j >> 2] >> (8 * (j & 3) + 2)) & 0x1Fu;
                    atomicAdd(h + e * kCols, 1u);
                }
            }
        }
    }
    __syncthreads();
    // Thread t sums 32 columns of bin t % kBins (slice t / kBins), in an order
    // rotated by the bin so that a warp's 32 reads fall in 32 banks; the
    // slices of a bin are added in shared memory, then once to global memory.
    const uint32_t b = tid % kBins, slice = tid / kBins;
    unsigned long long sum = 0;
#pragma unroll 8
    for (uint32_t c = 0; c < 32; c++) sum += s_hist[b * kCols + slice * 32 + ((c + b) & 31u)];
    s_part[tid] = sum;
    __syncthreads();
    if (tid < kBins) {
        unsigned long long total = 0;
        for (uint32_t k = 0; k < kHistThreads / kBins; k++) total += s_part[k * kBins + tid];
        if (total) atomicAdd(p.hist + tid, total);
    }
}

// Top-16 of `bins` counts, one block: sixteen rounds of a block-wide arg-max
// over the bins not yet taken, keyed (count + 1) << 8 | (255 - bin) so that
// the larger count wins and, between equal counts, the smaller exponent; bins
// with count 0 stay eligible.  The taken bins are then written in ascending
// order (code k = k-th smallest exponent).
__global__ void __launch_bounds__(kSelThreads) select_kernel(const unsigned long long* hist, uint32_t bins,
                                                            uint8_t* cb_out) {
    __shared__ unsigned long long s_key[kSelThreads / 32];
    __shared__ uint32_t s_win, s_rank[kSelThreads / 32];
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the counts are complete
    const unsigned long long count = tid < bins ? hist[tid] : 0ull;
    bool taken = false;
    for (int round = 0; round < kCodes; round++) {
        unsigned long long key = (tid < bins && !taken) ? ((count + 1ull) << 8) | (255u - tid) : 0ull;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, key, d);
            key = o > key ? o : key;
        }
        if (lane == 0) s_key[warp] = key;
        __syncthreads();
        if (tid == 0) {
            unsigned long long best = 0;
            for (uint32_t w = 0; w < kSelThreads / 32; w++) best = s_key[w] > best ? s_key[w] : best;
            s_win = 255u - (uint32_t)(best & 0xFFu);
        }
        __syncthreads();
        taken |= tid == s_win;
        __syncthreads();  // s_key and s_win are rewritten next round
    }
    const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, taken);
    if (lane == 0) s_rank[warp] = __popc(ballot);
    __syncthreads();
    if (taken) {
        uint32_t rank = __popc(ballot & ((1u << lane) - 1u));
        for (uint32_t w = 0; w < warp; w++) rank += s_rank[w];
        cb_out[rank] = (uint8_t)tid;
    }
}

cudaError_t launch_histogram(const HistogramParams& p, cudaStream_t s) {

    // Every line (stride 1): coalesced already; sparse samples load four
    // pieces at a time.
    const bool dense = p.stride == 1;
    const uint32_t U = dense ? 1u : 4u;
    const void* kern = p.bf16 ? (dense ? (const void*)histogram_kernel<true, 1> : (const void*)histogram_kernel<true, 4>)
                              : (dense ? (const void*)histogram_kernel<false, 1> : (const void*)histogram_kernel<false, 4>);
    int sms = 0, per_sm = 0;
    const cudaError_t err = kernel_fit(kern, kHistThreads, 0, &sms, &per_sm);
    if (err != cudaSuccess) return err;
    const uint64_t lines = (p.n * (p.bf16 ? 2 : 1) + kLineBytes - 1) / kLineBytes;
    const uint64_t pieces = (lines + p.stride - 1) / p.stride * kPieces;
    const uint64_t want = (pieces + kHistThreads * U - 1) / (kHistThreads * U);
    const uint64_t cap = (uint64_t)sms * (per_sm > 0 ? per_sm : 1);
    const uint32_t grid = (uint32_t)(want < 1 ? 1 : (want < cap ? want : cap));
    void* args[] = {const_cast<HistogramParams*>(&p)};
    return cudaLaunchKernel(kern, dim3(grid), dim3(kHistThreads), args, 0, s);
}

cudaError_t launch_select(const unsigned long long* hist, uint32_t bins, uint8_t* cb_out, cudaStream_t s) {
    // A programmatic dependent of the histogram kernel ahead of it.
    return launch_dependent(select_kernel, dim3(1), dim3(kSelThreads), 0, s, hist, bins, cb_out);
}

}  // namespace sz
