// sz_histogram.cu -- exponent histogram for offline calibration.
//
// The codebook is calibrated once, offline, from the exponent counts of a
// sample (SplitZip abstract, arXiv 2605.01708v2: an offline top-16 codebook
// removes online histogramming; technical summary, gist.science/es,
// "Resultados" > "Estudios de Ablacion" > "Calibracion").  This kernel is not
// on the encode/decode path.  Each warp counts into its own shared-memory
// histogram (KV exponents crowd into a few bins, so per-warp copies cut
// atomic contention), then the block adds its totals to the global counts.
#include "sz_device.cuh"
#include "sz_params.h"

namespace sz {

namespace {
constexpr uint32_t kHistThreads = 256;
constexpr uint32_t kHistWarps = kHistThreads / 32;
}  // namespace

__global__ void __launch_bounds__(kHistThreads) histogram_kernel(const HistogramParams p) {
    __shared__ uint32_t s_hist[kHistWarps][256];
    const uint32_t tid = threadIdx.x, warp = tid >> 5;
    for (uint32_t b = tid; b < kHistWarps * 256; b += kHistThreads) (&s_hist[0][0])[b] = 0;
    __syncthreads();
    const uint64_t stride = (uint64_t)gridDim.x * kHistThreads;
    for (uint64_t i = (uint64_t)blockIdx.x * kHistThreads + tid; i < p.n; i += stride) {
        uint32_t e;
        if (p.bf16) {
            const uint32_t v = (uint32_t)p.in[2 * i] | ((uint32_t)p.in[2 * i + 1] << 8);
            e = (v >> 7) & 0xFFu;
        } else {
            e = ((uint32_t)p.in[i] >> 2) & 0x1Fu;
        }
        atomicAdd(&s_hist[warp][e], 1u);
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

cudaError_t launch_histogram(const HistogramParams& p, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const uint64_t want = (p.n + kHistThreads - 1) / kHistThreads;
    const uint64_t cap = (uint64_t)sms * 8;
    const uint32_t grid = (uint32_t)(want < 1 ? 1 : (want < cap ? want : cap));
    histogram_kernel<<<grid, kHistThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sz
