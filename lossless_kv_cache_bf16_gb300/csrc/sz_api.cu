// sz_api.cu -- the C ABI of splitzip.h: argument checks, stream layout and
// kernel launches.  Host code only; the kernels live in sz_bf16.cu,
// sz_e5m2.cu and sz_histogram.cu.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "splitzip.h"
#include "sz_params.h"

namespace {

using namespace sz;

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded in-kernel waits for asynchronous copies: 1 s

// An NVTX range around a public call, so that profilers can attribute the
// kernels it launches (free when no tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

bool dtype_ok(int dt) { return dt == SZ_BF16 || dt == SZ_FP8_E5M2; }
uint64_t cdiv(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
uint64_t dense_bytes(sz_dtype dt, uint64_t n) { return dt == SZ_BF16 ? n + cdiv(n, 2) : 7 * cdiv(n, 8); }
// Encode scan tiles (both dtypes): one escape count and one record staging
// area each in the workspace.
uint64_t scan_tiles_for(uint64_t n) { return std::max<uint64_t>(1, cdiv(n, kScanTile)); }

// The encoders stage up to this many escape records per scan tile in the
// workspace; the records of scan tiles with more are re-derived by the
// finish kernel.
uint32_t stage_recs_for(sz_dtype dt) { return dt == SZ_BF16 ? kStageRecsBf16 : kStageRecsE5; }
static_assert(kStageRecsBf16 % 16 == 0 && kStageRecsE5 % 16 == 0, "staged runs start 16-byte aligned");
uint64_t align16(uint64_t x) { return (x + 15) & ~15ull; }
// Workspace: [u32 count per scan tile][i32 error code per encode block (at
// most one block per scan tile)][u16 count per unit, 32 per scan tile][3 *
// cap bytes of records per scan tile].  Each section starts 16-byte aligned.
uint64_t error_words_offset(uint64_t tiles) { return align16(4 * tiles); }
uint64_t unit_counts_offset(uint64_t tiles) { return error_words_offset(tiles) + align16(4 * tiles); }
uint64_t staged_records_offset(uint64_t tiles) { return unit_counts_offset(tiles) + 2ull * kUnitsPerScan * tiles; }
uint64_t workspace_bytes(uint64_t n, uint32_t cap) {
    const uint64_t tiles = scan_tiles_for(n);
    return staged_records_offset(tiles) + 3ull * cap * tiles;
}
// Tiles of the decoder (independent of the encoder's scan tiles).
uint64_t decode_tiles_for(sz_dtype dt, uint64_t n) {
    return std::max<uint64_t>(1, cdiv(n, dt == SZ_BF16 ? kBf16Tile : kE5Tile));
}
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

StreamLayout layout_for(sz_dtype dt, uint64_t n) {
    StreamLayout L{};
    L.n = n;
    L.dense = dense_bytes(dt, n);
    L.nib_off = dt == SZ_BF16 ? n : 0;
    L.cb_off = L.dense;
    L.num_chunks = (uint32_t)cdiv(n, SZ_CHUNK_ELEMS);
    L.hdr_off = L.cb_off + SZ_CODEBOOK_SIZE;
    L.rec_off = L.hdr_off + 8ull * L.num_chunks;
    return L;
}

sz_status from_cuda(cudaError_t e) {
    switch (e) {
        case cudaSuccess:
            return SZ_OK;
        case cudaErrorNoKernelImageForDevice:
        case cudaErrorNoDevice:
        case cudaErrorInsufficientDriver:
            return SZ_ERR_UNSUPPORTED;
        default:
            return SZ_ERR_CUDA;
    }
}

// 16 distinct exponents that the dtype can hold.
bool codebook_ok(sz_dtype dt, const uint8_t* cb) {
    const unsigned limit = dt == SZ_BF16 ? 256u : 32u;
    bool seen[256] = {};
    for (int k = 0; k < SZ_CODEBOOK_SIZE; k++) {
        if (cb[k] >= limit || seen[cb[k]]) return false;
        seen[cb[k]] = true;
    }
    return true;
}

// Exactly one of h_cb (host codebook, checked here) and d_cb (device
// codebook, 16-byte aligned, checked by the kernels) is set.
sz_status encode_impl(sz_dtype dt, const sz_codebook* h_cb, const void* d_in, size_t n, void* d_out,
                      size_t out_capacity, unsigned long long* d_out_bytes, int* d_status, void* d_ws,
                      size_t ws_bytes, uint32_t skip_first, uint64_t wait_ns, cudaStream_t stream,
                      uint32_t stage_recs = 0, const uint8_t* d_cb = nullptr, PageMap pm = PageMap{}) {
    if (!dtype_ok(dt) || (!h_cb == !d_cb) || !d_out || !d_out_bytes || !d_ws) return SZ_ERR_INVALID_ARG;
    if ((n > 0 && !d_in) || (uint64_t)n >= (1ull << 32)) return SZ_ERR_INVALID_ARG;
    if (dt == SZ_BF16 && !aligned(d_in, 2)) return SZ_ERR_INVALID_ARG;
    if (!aligned(d_ws, 16) || !aligned(d_out_bytes, 8) || (d_status && !aligned(d_status, 4))) return SZ_ERR_INVALID_ARG;
    if (h_cb && !codebook_ok(dt, h_cb->exp)) return SZ_ERR_INVALID_ARG;
    if (d_cb && !aligned(d_cb, 16)) return SZ_ERR_INVALID_ARG;
    if (out_capacity < sz_encoded_size(dt, n, 0)) return SZ_ERR_CAPACITY;
    if (stage_recs == 0) stage_recs = stage_recs_for(dt);
    const uint64_t ws_need = workspace_bytes(n, stage_recs);
    if (ws_bytes < ws_need) return SZ_ERR_CAPACITY;

    EncodeParams p{};
    p.L = layout_for(dt, n);
    p.in = static_cast<const uint8_t*>(d_in);
    p.out = static_cast<uint8_t*>(d_out);
    p.capacity = out_capacity;
    p.num_tiles = (uint32_t)scan_tiles_for(n);
    p.ws_count = static_cast<uint32_t*>(d_ws);
    p.ws_err = reinterpret_cast<int*>(static_cast<uint8_t*>(d_ws) + error_words_offset(p.num_tiles));
    p.ws_unit = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(d_ws) + unit_counts_offset(p.num_tiles));
    p.ws_rec = static_cast<uint8_t*>(d_ws) + staged_records_offset(p.num_tiles);
    p.ws_cap = stage_recs;
    p.out_bytes = d_out_bytes;
    p.status = d_status;
    p.wait_limit_ns = wait_ns;
    if (h_cb) {
        std::memcpy(p.cb, h_cb->exp, SZ_CODEBOOK_SIZE);
        std::sort(p.cb, p.cb + SZ_CODEBOOK_SIZE);  // code k = k-th smallest exponent
        p.contig = p.cb[SZ_CODEBOOK_SIZE - 1] - p.cb[0] == SZ_CODEBOOK_SIZE - 1;
    }
    p.cb_dev = d_cb;
    p.pm = pm;
    p.skip_first = skip_first;
    if (dt == SZ_BF16)
        p.vec = aligned(d_in, 16) && aligned(d_out, 8) && aligned(static_cast<uint8_t*>(d_out) + n, 4);
    else
        p.vec = aligned(d_in, 16) && aligned(d_out, 16);

    // Neither the workspace nor *d_status needs clearing: the encoders
    // write every count and error word that the finish kernel reads, and the
    // finish kernel's last block writes *d_status once, after every other
    // block of the encode has reported.  (A reset of the status word would
    // cost the GPU an operation of its own, about 2.7 us.)
    const cudaError_t err = dt == SZ_BF16 ? launch_encode_bf16(p, stream) : launch_encode_e5m2(p, stream);
    return from_cuda(err);
}

// ---- encode without allocation ---------------------------------------------
// sz_encode_noalloc keeps its workspace in this file-scope device array
// instead of taking one from the caller.  Every GPU that loads the library
// holds the array until the process exits.  Sized for n up to 2^28 elements
// of either dtype, staging up to 256 escape records per scan tile (the rest
// are re-derived): 8,192 scan tiles x (4 + 4 + 64 + 768) bytes = 6,881,280
// bytes.
constexpr uint64_t kNoAllocMaxElems = 1ull << 28;
constexpr uint32_t kNoAllocStageRecs = 256;
static_assert(kNoAllocStageRecs <= kStageRecsE5 && kNoAllocStageRecs % 16 == 0, "within both encoders' staging");
constexpr uint64_t kNoAllocScratchBytes =
    (kNoAllocMaxElems / kScanTile) * (4 + 4 + 2ull * kUnitsPerScan + 3ull * kNoAllocStageRecs);
static_assert(kNoAllocScratchBytes == 6881280, "the size the header states");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Host code cannot use g_noalloc_scratch as a device address (in host code the
// name is a host-side stand-in), so its device address is looked up once per
// device, with that device current, and cached.  The address belongs to the
// device's primary context; a cudaDeviceReset would make it stale, which the
// header rules out.
constexpr int kMaxDevices = 128;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

sz_status noalloc_scratch_for_current_device(void** out) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return from_cuda(err);
    if (dev < 0 || dev >= kMaxDevices) return SZ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (err != cudaSuccess) return from_cuda(err);
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return SZ_OK;
}

}  // namespace

namespace sz {

namespace {
struct FitEntry {
    int dev;
    const void* kern;
    int threads;
    size_t smem;
    int sms, per_sm;
};
constexpr int kMaxFits = 128;
std::mutex g_fit_mu;
FitEntry g_fit[kMaxFits];
int g_fit_n = 0;
}  // namespace

cudaError_t kernel_fit(const void* kern, int threads, size_t smem, int* sms, int* per_sm) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    {
        std::lock_guard<std::mutex> lock(g_fit_mu);
        for (int k = 0; k < g_fit_n; k++) {
            const FitEntry& f = g_fit[k];
            if (f.dev == dev && f.kern == kern && f.threads == threads && f.smem == smem) {
                *sms = f.sms;
                *per_sm = f.per_sm;
                return cudaSuccess;
            }
        }
    }
    FitEntry f{dev, kern, threads, smem, 0, 0};
    if (smem > 0) err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&f.sms, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess) err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&f.per_sm, kern, threads, smem);
    if (err != cudaSuccess) return err;
    *sms = f.sms;
    *per_sm = f.per_sm;
    std::lock_guard<std::mutex> lock(g_fit_mu);
    if (g_fit_n < kMaxFits) g_fit[g_fit_n++] = f;  // a full table only costs the queries again
    return cudaSuccess;
}

}  // namespace sz

extern "C" {

size_t sz_encoded_size(sz_dtype dt, size_t n, size_t n_escapes) {
    if (!dtype_ok(dt)) return 0;
    return dense_bytes(dt, n) + SZ_CODEBOOK_SIZE + 8 * cdiv(n, SZ_CHUNK_ELEMS) + 3 * (uint64_t)n_escapes;
}

size_t sz_workspace_size(sz_dtype dt, size_t n) {
    if (!dtype_ok(dt)) return 0;
    return workspace_bytes(n, stage_recs_for(dt));
}

size_t sz_histogram_bins(sz_dtype dt) {
    if (!dtype_ok(dt)) return 0;
    return dt == SZ_BF16 ? 256 : 32;
}

sz_status sz_histogram(sz_dtype dt, const void* d_sample, size_t n, unsigned long long* d_hist,
                       cudaStream_t stream) {
    const NvtxRange range("sz_histogram");
    if (!dtype_ok(dt) || !d_hist || (n > 0 && !d_sample)) return SZ_ERR_INVALID_ARG;
    if (dt == SZ_BF16 && !aligned(d_sample, 2)) return SZ_ERR_INVALID_ARG;
    if (!aligned(d_hist, 8)) return SZ_ERR_INVALID_ARG;
    cudaError_t err = cudaMemsetAsync(d_hist, 0, sz_histogram_bins(dt) * sizeof(unsigned long long), stream);
    if (err != cudaSuccess) return from_cuda(err);
    if (n == 0) return SZ_OK;
    HistogramParams p{static_cast<const uint8_t*>(d_sample), n, d_hist, dt == SZ_BF16, 1u};
    return from_cuda(launch_histogram(p, stream));
}

sz_status sz_codebook_from_histogram_device(sz_dtype dt, const unsigned long long* d_hist, uint8_t* d_cb,
                                            cudaStream_t stream) {
    const NvtxRange range("sz_codebook_from_histogram_device");
    if (!dtype_ok(dt) || !d_hist || !d_cb || !aligned(d_hist, 8) || !aligned(d_cb, 16)) return SZ_ERR_INVALID_ARG;
    return from_cuda(launch_select(d_hist, (uint32_t)sz_histogram_bins(dt), d_cb, stream));
}

sz_status sz_calibrate_device(sz_dtype dt, const void* d_x, size_t n, uint32_t sample_stride,
                              unsigned long long* d_hist, uint8_t* d_cb, cudaStream_t stream) {
    const NvtxRange range("sz_calibrate_device");
    if (!dtype_ok(dt) || !d_hist || !d_cb || (n > 0 && !d_x) || sample_stride == 0) return SZ_ERR_INVALID_ARG;
    if (dt == SZ_BF16 && !aligned(d_x, 2)) return SZ_ERR_INVALID_ARG;
    if (!aligned(d_hist, 8) || !aligned(d_cb, 16)) return SZ_ERR_INVALID_ARG;
    cudaError_t err = cudaMemsetAsync(d_hist, 0, sz_histogram_bins(dt) * sizeof(unsigned long long), stream);
    if (err == cudaSuccess && n > 0) {
        HistogramParams p{static_cast<const uint8_t*>(d_x), n, d_hist, dt == SZ_BF16, sample_stride};
        err = launch_histogram(p, stream);
    }
    if (err == cudaSuccess) err = launch_select(d_hist, (uint32_t)sz_histogram_bins(dt), d_cb, stream);
    return from_cuda(err);
}

sz_status sz_codebook_from_histogram(sz_dtype dt, const unsigned long long* h_hist, sz_codebook* h_cb) {
    if (!dtype_ok(dt) || !h_hist || !h_cb) return SZ_ERR_INVALID_ARG;
    const int bins = (int)sz_histogram_bins(dt);
    int order[256];
    for (int e = 0; e < bins; e++) order[e] = e;
    // Most frequent first; equal counts keep the smaller exponent first.
    std::stable_sort(order, order + bins, [&](int a, int b) { return h_hist[a] > h_hist[b]; });
    uint8_t chosen[SZ_CODEBOOK_SIZE];
    for (int k = 0; k < SZ_CODEBOOK_SIZE; k++) chosen[k] = (uint8_t)order[k];
    std::sort(chosen, chosen + SZ_CODEBOOK_SIZE);
    std::memcpy(h_cb->exp, chosen, SZ_CODEBOOK_SIZE);
    return SZ_OK;
}

sz_status sz_ablation_sizes(sz_dtype dt, const unsigned long long* h_hist, size_t n, unsigned long long* h_sizes) {
    if (!dtype_ok(dt) || !h_hist || !h_sizes) return SZ_ERR_INVALID_ARG;
    const int bins = (int)sz_histogram_bins(dt);
    int order[256];
    for (int e = 0; e < bins; e++) order[e] = e;
    std::stable_sort(order, order + bins, [&](int a, int b) { return h_hist[a] > h_hist[b]; });
    // covered[k] = elements whose exponent is among the k most frequent.
    unsigned long long covered[17] = {};
    for (int k = 1; k <= 16; k++) covered[k] = covered[k - 1] + h_hist[order[k - 1]];
    const uint64_t chunks = cdiv(n, SZ_CHUNK_ELEMS);
    const uint64_t e16 = n - covered[16], e8 = n - covered[8], e15 = n - covered[15];
    const uint64_t codes8 = dt == SZ_BF16 ? n + 3 * cdiv(n, 8) : 3 * cdiv(n, 4);
    h_sizes[0] = sz_encoded_size(dt, n, e16);
    h_sizes[1] = codes8 + 3 * e8 + 8 + 8 * chunks;
    h_sizes[2] = dense_bytes(dt, n) + e15 + 15 + 8 * chunks;
    return SZ_OK;
}

sz_status sz_calibrate(sz_dtype dt, const void* d_sample, size_t n, unsigned long long* d_hist, sz_codebook* h_cb,
                       cudaStream_t stream) {
    const NvtxRange range("sz_calibrate");
    if (!h_cb) return SZ_ERR_INVALID_ARG;
    sz_status st = sz_histogram(dt, d_sample, n, d_hist, stream);
    if (st != SZ_OK) return st;
    unsigned long long h_hist[256];
    const size_t bins = sz_histogram_bins(dt);
    cudaError_t err = cudaMemcpyAsync(h_hist, d_hist, bins * sizeof(unsigned long long), cudaMemcpyDeviceToHost, stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return from_cuda(err);
    return sz_codebook_from_histogram(dt, h_hist, h_cb);
}

sz_status sz_encode(sz_dtype dt, const sz_codebook* h_cb, const void* d_in, size_t n, void* d_out,
                    size_t out_capacity, unsigned long long* d_out_bytes, int* d_status, void* d_ws, size_t ws_bytes,
                    cudaStream_t stream) {
    const NvtxRange range("sz_encode");
    return encode_impl(dt, h_cb, d_in, n, d_out, out_capacity, d_out_bytes, d_status, d_ws, ws_bytes, 0,
                       kWaitLimitNs, stream);
}

sz_status sz_encode_dcb(sz_dtype dt, const uint8_t* d_cb, const void* d_in, size_t n, void* d_out,
                        size_t out_capacity, unsigned long long* d_out_bytes, int* d_status, void* d_ws,
                        size_t ws_bytes, cudaStream_t stream) {
    const NvtxRange range("sz_encode_dcb");
    if (!d_cb) return SZ_ERR_INVALID_ARG;
    return encode_impl(dt, nullptr, d_in, n, d_out, out_capacity, d_out_bytes, d_status, d_ws, ws_bytes, 0,
                       kWaitLimitNs, stream, 0, d_cb);
}

sz_status sz_encode_noalloc(sz_dtype dt, const sz_codebook* h_cb, const void* d_in, size_t n, void* d_out,
                            size_t out_capacity, unsigned long long* d_out_bytes, int* d_status, cudaStream_t stream) {
    const NvtxRange range("sz_encode_noalloc");
    if (!dtype_ok(dt)) return SZ_ERR_INVALID_ARG;
    if ((uint64_t)n > kNoAllocMaxElems || workspace_bytes(n, kNoAllocStageRecs) > kNoAllocScratchBytes)
        return SZ_ERR_CAPACITY;  // beyond the static scratch
    void* ws = nullptr;
    const sz_status st = noalloc_scratch_for_current_device(&ws);
    if (st != SZ_OK) return st;
    // Nothing needs clearing: the encoders write every count that the finish
    // kernel reads.
    return encode_impl(dt, h_cb, d_in, n, d_out, out_capacity, d_out_bytes, d_status, ws, kNoAllocScratchBytes, 0,
                       kWaitLimitNs, stream, kNoAllocStageRecs);
}

sz_status sz_debug_encode_stalled(sz_dtype dt, const sz_codebook* h_cb, const void* d_in, size_t n, void* d_out,
                                  size_t out_capacity, unsigned long long* d_out_bytes, int* d_status, void* d_ws,
                                  size_t ws_bytes, unsigned long long wait_limit_ns, cudaStream_t stream) {
    if (!d_status || wait_limit_ns == 0 || wait_limit_ns > kWaitLimitNs) return SZ_ERR_INVALID_ARG;
    if (dt == SZ_FP8_E5M2) return SZ_ERR_UNSUPPORTED;  // the E5M2 encoder has no in-kernel wait
    return encode_impl(dt, h_cb, d_in, n, d_out, out_capacity, d_out_bytes, d_status, d_ws, ws_bytes, 1,
                       wait_limit_ns, stream);
}

// Streams with at least one escape per kDenseDecodeDiv elements count as
// dense in escapes for the decoder (a measured crossover: 2.5%).
constexpr uint64_t kDenseDecodeDiv = 40;

sz_status decode_impl(sz_dtype dt, const void* d_in, size_t in_bytes, size_t n, void* d_out, int* d_status,
                      cudaStream_t stream, PageMap pm) {
    if (!dtype_ok(dt) || !d_in || (n > 0 && !d_out) || (uint64_t)n >= (1ull << 32)) return SZ_ERR_INVALID_ARG;
    if (dt == SZ_BF16 && !aligned(d_out, 2)) return SZ_ERR_INVALID_ARG;
    if (d_status && !aligned(d_status, 4)) return SZ_ERR_INVALID_ARG;
    const uint64_t fixed = sz_encoded_size(dt, n, 0);
    if (in_bytes < fixed || (in_bytes - fixed) % 3 != 0) return SZ_ERR_CORRUPT;
    const uint64_t n_esc = (in_bytes - fixed) / 3;
    if (n_esc > n) return SZ_ERR_CORRUPT;  // at most one escape per element

    DecodeParams p{};
    p.L = layout_for(dt, n);
    p.in = static_cast<const uint8_t*>(d_in);
    p.out = static_cast<uint8_t*>(d_out);
    p.num_tiles = (uint32_t)decode_tiles_for(dt, n);
    p.n_esc = (uint32_t)n_esc;
    p.status = d_status;
    p.wait_limit_ns = kWaitLimitNs;
    p.pm = pm;
    if (dt == SZ_BF16)
        p.vec = aligned(d_in, 8) && aligned(static_cast<const uint8_t*>(d_in) + n, 4) && aligned(d_out, 16);
    else
        p.vec = aligned(d_in, 16) && aligned(d_out, 16);

    if (d_status) {
        const cudaError_t err = cudaMemsetAsync(d_status, 0, sizeof(int), stream);
        if (err != cudaSuccess) return from_cuda(err);
    }
    // A BF16 stream with escapes in at least 1 / kDenseDecodeDiv of its
    // elements (known here from its size) takes the decoder variant that
    // computes exponents by byte adds (decode_bf16_kernel's ADDS).
    const bool adds = dt == SZ_BF16 && !pm.ids && n_esc * kDenseDecodeDiv >= n;
    return from_cuda(dt == SZ_BF16 ? launch_decode_bf16(p, stream, false, adds) : launch_decode_e5m2(p, stream));
}

// A page pool: page_elems a power of two in [16, 2^30], the pool 16-byte
// aligned (so every page is), pool_pages in [1, 2^31).  Ids are checked on
// the device.
bool page_map_for(const void* d_pool, size_t pool_pages, size_t page_elems, const int32_t* d_ids, size_t n,
                  PageMap* pm) {
    if (page_elems < 16 || page_elems > (1ull << 30) || (page_elems & (page_elems - 1)) != 0) return false;
    if (pool_pages == 0 || pool_pages >= (1ull << 31) || !d_pool || !aligned(d_pool, 16)) return false;
    if (n > 0 && (!d_ids || !aligned(d_ids, 4))) return false;
    uint32_t lg = 0;
    while ((1ull << lg) < page_elems) lg++;
    pm->ids = d_ids;
    pm->pool_pages = (uint32_t)pool_pages;
    pm->lg = lg;
    return true;
}

sz_status sz_decode(sz_dtype dt, const void* d_in, size_t in_bytes, size_t n, void* d_out, int* d_status,
                    cudaStream_t stream) {
    const NvtxRange range("sz_decode");
    return decode_impl(dt, d_in, in_bytes, n, d_out, d_status, stream, PageMap{});
}

sz_status sz_encode_paged(sz_dtype dt, const sz_codebook* h_cb, const void* d_pool, size_t pool_pages,
                          size_t page_elems, const int32_t* d_block_ids, size_t n, void* d_out, size_t out_capacity,
                          unsigned long long* d_out_bytes, int* d_status, void* d_ws, size_t ws_bytes,
                          cudaStream_t stream) {
    const NvtxRange range("sz_encode_paged");
    PageMap pm{};
    if (!page_map_for(d_pool, pool_pages, page_elems, d_block_ids, n, &pm)) return SZ_ERR_INVALID_ARG;
    if (n > 0 && cdiv(n, page_elems) > (1ull << 31)) return SZ_ERR_INVALID_ARG;
    return encode_impl(dt, h_cb, d_pool, n, d_out, out_capacity, d_out_bytes, d_status, d_ws, ws_bytes, 0,
                       kWaitLimitNs, stream, 0, nullptr, pm);
}

sz_status sz_decode_paged(sz_dtype dt, const void* d_in, size_t in_bytes, size_t n, void* d_pool, size_t pool_pages,
                          size_t page_elems, const int32_t* d_block_ids, int* d_status, cudaStream_t stream) {
    const NvtxRange range("sz_decode_paged");
    PageMap pm{};
    if (!page_map_for(d_pool, pool_pages, page_elems, d_block_ids, n, &pm)) return SZ_ERR_INVALID_ARG;
    return decode_impl(dt, d_in, in_bytes, n, d_pool, d_status, stream, pm);
}

// ---- the codebook ablation's alternative codecs (BF16) ----------------------
namespace {
bool ablation_ok(int v) { return v == SZ_ABL_TOP8 || v == SZ_ABL_SENTINEL; }
uint32_t ablation_k(int v) { return v == SZ_ABL_TOP8 ? 8u : 15u; }
uint64_t ablation_dense(int v, uint64_t n) { return v == SZ_ABL_TOP8 ? n + 3 * cdiv(n, 8) : n + cdiv(n, 2); }
}  // namespace

size_t sz_ablation_encoded_size(int variant, size_t n, size_t n_escapes) {
    if (!ablation_ok(variant)) return 0;
    return ablation_dense(variant, n) + ablation_k(variant) + 8 * cdiv(n, SZ_CHUNK_ELEMS) +
           (variant == SZ_ABL_TOP8 ? 3 : 1) * (uint64_t)n_escapes;
}

sz_status sz_ablation_codebook(int variant, const unsigned long long* h_hist, uint8_t* h_cb) {
    if (!ablation_ok(variant) || !h_hist || !h_cb) return SZ_ERR_INVALID_ARG;
    int order[256];
    for (int e = 0; e < 256; e++) order[e] = e;
    std::stable_sort(order, order + 256, [&](int a, int b) { return h_hist[a] > h_hist[b]; });
    const uint32_t k = ablation_k(variant);
    for (uint32_t c = 0; c < k; c++) h_cb[c] = (uint8_t)order[c];
    std::sort(h_cb, h_cb + k);
    return SZ_OK;
}

size_t sz_ablation_workspace_size(size_t n) { return 8 * std::max<uint64_t>(1, cdiv(n, SZ_CHUNK_ELEMS)); }

sz_status sz_ablation_encode(int variant, const uint8_t* h_cb, const void* d_in, size_t n, void* d_out,
                             size_t out_capacity, unsigned long long* d_out_bytes, void* d_ws, size_t ws_bytes,
                             cudaStream_t stream) {
    const NvtxRange range("sz_ablation_encode");
    if (!ablation_ok(variant) || !h_cb || !d_out || !d_out_bytes || !d_ws) return SZ_ERR_INVALID_ARG;
    if ((n > 0 && !d_in) || (uint64_t)n >= (1ull << 32) || !aligned(d_in, 2) || !aligned(d_ws, 4) ||
        !aligned(d_out_bytes, 8))
        return SZ_ERR_INVALID_ARG;
    const uint32_t k = ablation_k(variant);
    bool seen[256] = {};
    for (uint32_t c = 0; c < k; c++) {
        if (seen[h_cb[c]]) return SZ_ERR_INVALID_ARG;
        seen[h_cb[c]] = true;
    }
    if (out_capacity < sz_ablation_encoded_size(variant, n, n)) return SZ_ERR_CAPACITY;
    if (ws_bytes < sz_ablation_workspace_size(n)) return SZ_ERR_CAPACITY;
    AblationParams p{};
    p.in = static_cast<const uint8_t*>(d_in);
    p.out = static_cast<uint8_t*>(d_out);
    p.n = n;
    p.chunks = (uint32_t)cdiv(n, SZ_CHUNK_ELEMS);
    p.k = k;
    p.top8 = variant == SZ_ABL_TOP8;
    p.cb_off = ablation_dense(variant, n);
    p.hdr_off = p.cb_off + k;
    p.rec_off = p.hdr_off + 8ull * p.chunks;
    p.counts = static_cast<uint32_t*>(d_ws);
    p.offsets = p.counts + std::max<uint32_t>(p.chunks, 1u);
    p.out_bytes = d_out_bytes;
    std::memcpy(p.cb, h_cb, k);
    return from_cuda(launch_ablation_encode(p, stream));
}

sz_status sz_ablation_decode(int variant, const void* d_in, size_t in_bytes, size_t n, void* d_out, int* d_status,
                             cudaStream_t stream) {
    const NvtxRange range("sz_ablation_decode");
    if (!ablation_ok(variant) || !d_in || (n > 0 && !d_out) || (uint64_t)n >= (1ull << 32)) return SZ_ERR_INVALID_ARG;
    if (!aligned(d_out, 2) || (d_status && !aligned(d_status, 4))) return SZ_ERR_INVALID_ARG;
    const uint64_t fixed = sz_ablation_encoded_size(variant, n, 0);
    const uint64_t per = variant == SZ_ABL_TOP8 ? 3 : 1;
    if (in_bytes < fixed || (in_bytes - fixed) % per != 0) return SZ_ERR_CORRUPT;
    const uint64_t n_esc = (in_bytes - fixed) / per;
    if (n_esc > n) return SZ_ERR_CORRUPT;
    DecodeParams p{};
    p.L.n = n;
    p.L.dense = ablation_dense(variant, n);
    p.L.nib_off = n;
    p.L.cb_off = p.L.dense;
    p.L.num_chunks = (uint32_t)cdiv(n, SZ_CHUNK_ELEMS);
    p.L.hdr_off = p.L.cb_off + ablation_k(variant);
    p.L.rec_off = p.L.hdr_off + 8ull * p.L.num_chunks;
    p.in = static_cast<const uint8_t*>(d_in);
    p.out = static_cast<uint8_t*>(d_out);
    p.num_tiles = (uint32_t)decode_tiles_for(SZ_BF16, n);
    p.n_esc = (uint32_t)n_esc;
    p.status = d_status;
    p.wait_limit_ns = kWaitLimitNs;
    // 16-byte input when the dense streams start 16-byte aligned; 16-byte output.
    p.vec = aligned(d_in, 16) && aligned(static_cast<const uint8_t*>(d_in) + n, 16) && aligned(d_out, 16);
    if (d_status) {
        const cudaError_t err = cudaMemsetAsync(d_status, 0, sizeof(int), stream);
        if (err != cudaSuccess) return from_cuda(err);
    }
    return from_cuda(variant == SZ_ABL_TOP8 ? launch_decode_bf16(p, stream, true) : launch_decode_sentinel(p, stream));
}

const char* sz_status_string(int status) {
    switch (status) {
        case SZ_OK: return "SZ_OK";
        case SZ_ERR_INVALID_ARG: return "SZ_ERR_INVALID_ARG";
        case SZ_ERR_UNSUPPORTED: return "SZ_ERR_UNSUPPORTED";
        case SZ_ERR_CAPACITY: return "SZ_ERR_CAPACITY";
        case SZ_ERR_CORRUPT: return "SZ_ERR_CORRUPT";
        case SZ_ERR_TIMEOUT: return "SZ_ERR_TIMEOUT";
        case SZ_ERR_CUDA: return "SZ_ERR_CUDA";
        default: return "SZ_ERR_UNKNOWN";
    }
}

}  // extern "C"
