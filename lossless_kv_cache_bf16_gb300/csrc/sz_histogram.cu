// sz_histogram.cu -- exponent histogram and top-16 selection (calibration).
//
// The codebook is calibrated once, offline, from the exponent counts of a
// sample (SplitZip abstract, arXiv 2605.01708v2: an offline top-16 codebook
// removes online histogramming; technical summary, gist.science/es,
// "Resultados" > "Estudios de Ablacion" > "Calibracion").  The histogram can
// also be taken on the device per tensor, over every s-th group of 8
// elements, and the top-16 chosen there too (select_kernel), so that an
// encode can follow without a trip to the host; the ablation's price of such
// dynamic calibration is then measurable.  Each warp counts into its own
// shared-memory histogram (KV exponents crowd into a few bins, so per-warp
// copies cut atomic contention), then the block adds its totals to the
// global counts.
#include "sz_device.cuh"
#include "sz_params.h"

namespace sz {

namespace {
constexpr uint32_t kHistThreads = 256;
constexpr uint32_t kHistWarps = kHistThreads / 32;
constexpr uint32_t kSelThreads = 256;
}  // namespace

__global__ void __launch_bounds__(kHistThreads) histogram_kernel(const HistogramParams p) {
    __shared__ uint32_t s_hist[kHistWarps][256];
    const uint32_t tid = threadIdx.x, warp = tid >> 5;
    for (uint32_t b = tid; b < kHistWarps * 256; b += kHistThreads) (&s_hist[0][0])[b] = 0;
    __syncthreads();
    // Sampled groups of 8 elements: group g covers elements [8 g s, 8 g s + 8).
    const uint64_t groups = (p.n + 7) / 8;
    const uint64_t sampled = (groups + p.stride - 1) / p.stride;
    const uint64_t step = (uint64_t)gridDim.x * kHistThreads;
    const uint32_t esize = p.bf16 ? 2u : 1u;
    const bool vec = (reinterpret_cast<uintptr_t>(p.in) % (8 * esize)) == 0;
    uint32_t* h = s_hist[warp];
    for (uint64_t g = (uint64_t)blockIdx.x * kHistThreads + tid; g < sampled; g += step) {
        const uint64_t i0 = g * p.stride * 8;
        const uint32_t cnt = p.n - i0 >= 8 ? 8u : (uint32_t)(p.n - i0);
        if (p.bf16) {
            uint32_t w[4] = {0, 0, 0, 0};
            if (vec && cnt == 8) {
                const uint4 v = *reinterpret_cast<const uint4*>(p.in + 2 * i0);
                w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
            } else {
                for (uint32_t j = 0; j < cnt; j++)
                    w[j >> 1] |= ((uint32_t)p.in[2 * (i0 + j)] | ((uint32_t)p.in[2 * (i0 + j) + 1] << 8)) << (16 * (j & 1));
            }
#pragma unroll
            for (uint32_t j = 0; j < 8; j++)
                if (j < cnt) atomicAdd(&h[(w[j >> 1] >> (7 + 16 * (j & 1))) & 0xFFu], 1u);
        } else {
            uint32_t w[2] = {0, 0};
            if (vec && cnt == 8) {
                const uint2 v = *reinterpret_cast<const uint2*>(p.in + i0);
                w[0] = v.x, w[1] = v.y;
            } else {
                for (uint32_t j = 0; j < cnt; j++) w[j >> 2] |= (uint32_t)p.in[i0 + j] << (8 * (j & 3));
            }
#pragma unroll
            for (uint32_t j = 0; j < 8; j++)
                if (j < cnt) atomicAdd(&h[(w[j >> 2] >> (8 * (j & 3) + 2)) & 0x1Fu], 1u);
        }
    }
    __syncthreads();
    const uint32_t bins = p.bf16 ? 256u : 32u;
    for (uint32_t b = tid; b < bins; b += kHistThreads) {
        unsigned long long sum = 0;
#pragma unroll
        for (uint32_t w = 0; w < kHistWarps; w++) sum += s_hist[w][b];
        if (sum) atomicAdd(p.hist + b, sum);
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
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const uint64_t groups = ((p.n + 7) / 8 + p.stride - 1) / p.stride;
    const uint64_t want = (groups + kHistThreads - 1) / kHistThreads;
    const uint64_t cap = (uint64_t)sms * 8;
    const uint32_t grid = (uint32_t)(want < 1 ? 1 : (want < cap ? want : cap));
    histogram_kernel<<<grid, kHistThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_select(const unsigned long long* hist, uint32_t bins, uint8_t* cb_out, cudaStream_t s) {
    select_kernel<<<1, kSelThreads, 0, s>>>(hist, bins, cb_out);
    return cudaGetLastError();
}

}  // namespace sz
