// sz_params.h -- host/device launch parameters shared by the SplitZip kernels
// and the C ABI layer (not part of the public interface).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace sz {

// Byte offsets of the stream sections for n elements (see splitzip.h).
struct StreamLayout {
    uint64_t n;
    uint64_t dense;     // BF16: sm + nibbles; E5M2: packed groups
    uint64_t nib_off;   // BF16 only: start of the nibble stream (= n)
    uint64_t cb_off;    // codebook (16 bytes)
    uint64_t hdr_off;   // chunk headers (8 bytes each)
    uint64_t rec_off;   // escape records (3 bytes each)
    uint32_t num_chunks;
};

// Paged tensor (a block table over a pool of equal pages): element e lives in
// page ids[e >> lg] at offset e & (2^lg - 1); page q starts at byte
// (q << lg) * element size of the pool.  ids == nullptr: contiguous tensor.
struct PageMap {
    const int32_t* ids;
    uint32_t pool_pages;
    uint32_t lg;
};

struct EncodeParams {
    StreamLayout L;
    const uint8_t* in;
    uint8_t* out;
    uint64_t capacity;
    uint32_t num_tiles;      // scan tiles
    unsigned long long* out_bytes;
    int* status;             // nullable; written once, by the finish kernel
    uint64_t wait_limit_ns;
    int vec;                 // 1 when the aligned vector path may be used
    uint32_t grid;           // blocks of the encode kernel's launch
    uint32_t skip_first;     // test hook: a wait that never completes
    int contig;              // codebook is 16 consecutive exponents cb[0]..cb[0]+15
    uint32_t* ws_count;      // workspace: escapes per scan tile
    int* ws_err;             // workspace: each BF16 encode block's error code (0 = none); the
                             // finish kernel's last block turns them into *status
    uint16_t* ws_unit;       // workspace: escapes per 1,024-element unit, kUnitsPerScan per scan tile
    uint8_t* ws_rec;         // workspace: staged records, ws_cap per scan tile
    uint32_t ws_cap;         // records staged per scan tile
    const uint8_t* cb_dev;   // nullable: codebook in device memory instead of cb
    PageMap pm;              // paged input (in = the pool) when pm.ids is set
    uint8_t cb[16];          // ascending
};

struct DecodeParams {
    StreamLayout L;
    const uint8_t* in;
    uint8_t* out;
    uint32_t num_tiles;
    uint32_t n_esc;          // escape count implied by the stream size
    int* status;             // nullable
    int vec;
    uint64_t wait_limit_ns;  // bounded waits for in-kernel copies
    PageMap pm;              // paged output (out = the pool) when pm.ids is set
};

struct HistogramParams {
    const uint8_t* in;
    uint64_t n;
    unsigned long long* hist;
    int bf16;
    uint32_t stride;  // sample one 128-byte line per run of `stride` lines (1: all)
};

// The codebook ablation's alternative BF16 codecs (sz_ablation.cu).
struct AblationParams {
    const uint8_t* in;
    uint8_t* out;
    uint64_t n;
    uint32_t chunks;
    uint32_t k;                      // codebook entries: 8 (Top-8) or 15 (sentinel)
    int top8;
    uint64_t cb_off, hdr_off, rec_off;
    uint32_t* counts;                // workspace: escapes per chunk
    uint32_t* offsets;               // workspace: escapes before each chunk
    unsigned long long* out_bytes;
    uint8_t cb[16];                  // code c -> exponent, as given
};

// Tile sizes (elements).  Both divide the 65,536-element chunk.
constexpr uint32_t kBf16Threads = 256;
constexpr uint32_t kBf16PerThread = 32;
constexpr uint32_t kBf16Tile = kBf16Threads * kBf16PerThread;   // 8192
constexpr uint32_t kE5PerThread = 128;                          // E5M2 encode: 16 groups of 8 per thread
constexpr uint32_t kE5Tile = 16384;                             // E5M2 decode tile
// Encode (both dtypes): escape counts and staged records per scan tile.
constexpr uint32_t kScanTile = 32768;
// Records staged per scan tile by default: 2,048 (6.25% of the tile) for
// BF16 and 1,024 (3.1%) for E5M2, about 9.4% of the input bytes either way.
// EncodeParams::ws_cap is at most the encoder's default and a multiple of 16,
// so that every tile's staged run starts 16-byte aligned.
constexpr uint32_t kStageRecsBf16 = 2048;
constexpr uint32_t kStageRecsE5 = 1024;
// A scan tile is 32 units of 1,024 consecutive elements (BF16) or 8 units of
// 4,096 (E5M2, one encoder warp's share); for a scan tile with more escapes
// than it stages, the encoders record each unit's escape count, so that the
// remaining records can be re-derived unit by unit, in parallel, at known
// offsets.  The workspace has room for 32 counts per scan tile.
// The E5M2 encoder flags an error of its scan tile (a bad page id or device
// codebook) in bit 31 of the tile's escape count, which never exceeds 2^15.
constexpr uint32_t kCountError = 0x80000000u;
constexpr uint32_t kUnitElems = 1024;
constexpr uint32_t kUnitElemsE5 = 4096;
constexpr uint32_t kUnitsPerScan = kScanTile / kUnitElems;  // 32

// Launches kern as a programmatic dependent of the kernel before it in the
// stream: its blocks may be scheduled while that kernel finishes, and must
// execute griddepcontrol.wait before reading anything it wrote (the wait
// returns at once when there is no such kernel).  This hides launch gaps.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Launch shape of kernel `kern` with `threads` threads and `smem` bytes of
// dynamic shared memory on the current device: the SM count and how many
// blocks fit per SM.  The first query per device and kernel also raises the
// kernel's dynamic shared memory limit to `smem`; the answers are cached, so
// a call after that costs one cudaGetDevice and a table lookup.
cudaError_t kernel_fit(const void* kern, int threads, size_t smem, int* sms, int* per_sm);

cudaError_t launch_encode_bf16(const EncodeParams& p, cudaStream_t s);
// top8: the Top-8 layout of the codebook ablation (see sz_ablation_decode).
// adds: the stream is dense in escapes (decode_bf16_kernel's ADDS).
cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t s, bool top8 = false, bool adds = false);
cudaError_t launch_encode_e5m2(const EncodeParams& p, cudaStream_t s);
cudaError_t launch_decode_e5m2(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_histogram(const HistogramParams& p, cudaStream_t s);
// Top-16 of a device histogram -> 16 ascending exponents in device memory.
cudaError_t launch_select(const unsigned long long* hist, uint32_t bins, uint8_t* cb_out, cudaStream_t s);
cudaError_t launch_finish(const EncodeParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_ablation_encode(const AblationParams& p, cudaStream_t s);
cudaError_t launch_decode_sentinel(const DecodeParams& p, cudaStream_t s);

}  // namespace sz
