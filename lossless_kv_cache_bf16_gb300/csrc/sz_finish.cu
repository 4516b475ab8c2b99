// sz_finish.cu -- second phase of the SplitZip encode (both dtypes).
//
// The encode kernels stream the tensor and leave, per 32,768-element scan
// tile, the number of escapes and (up to ws_cap of) the tile's escape
// records in element order in the workspace.  This kernel places them:
//  * block b owns the contiguous scan-tile range [bT/F, (b+1)T/F); it sums
//    the counts of all earlier scan tiles (16-byte loads, several in flight
//    per thread), then scans its own counts in batches of 256, giving every
//    scan tile its escape offset;
//  * one warp per scan tile copies the staged records to offset * 3 in the
//    escape stream: 16-byte loads of the whole staged run into shared memory,
//    then aligned 4-byte stores (a funnel shift realigns the bytes) with at
//    most 3 single bytes at either end.  When the tile had more than ws_cap
//    escapes, the warp walks the tile's elements again in order and writes
//    the records directly;
//  * a chunk's last scan tile writes the chunk's header (offset = escapes
//    before the chunk, count = escapes in it); the last scan tile writes the
//    stream size.
// Escapes are (u16 position in the 65,536-element chunk, u8 exponent) pairs
// in element order (SplitZip technical summary, gist.science/es,
// "Metodologia: SplitZip" > "Flujo de Escape").
#include "sz_device.cuh"
#include "sz_params.h"

namespace sz {

namespace {

constexpr uint32_t kFinThreads = 256;
constexpr uint32_t kFinWarps = kFinThreads / 32;
constexpr uint32_t kScansPerChunk = kChunk / kScanTile;
constexpr uint32_t kStageBytes = 3 * kMaxStageRecs;      // staged records of one scan tile
constexpr uint32_t kStageLoads = kStageBytes / 512;       // 16-byte loads per lane
static_assert(kStageBytes % 512 == 0, "whole warp-wide 16-byte loads");
static_assert(kChunk % kScanTile == 0, "scan tiles must not straddle chunks");

// Exponent of element i (linear or paged input): bits 14..7 of a BF16, bits
// 6..2 of an E5M2 byte.
template <bool BF16, bool PAGED>
__device__ __forceinline__ uint32_t exponent_at(const EncodeParams& p, uint64_t i) {
    const uint8_t* e = p.in + elem_offset<PAGED>(p.pm, i, BF16 ? 2u : 1u, p.status);
    if (BF16) return (((uint32_t)e[0] | ((uint32_t)e[1] << 8)) >> 7) & 0xFFu;
    return ((uint32_t)e[0] >> 2) & 0x1Fu;
}

}  // namespace

template <bool BF16, bool PAGED>
__global__ void __launch_bounds__(kFinThreads) finish_kernel(const EncodeParams p) {
    __shared__ __align__(16) uint8_t s_stage[kFinWarps][kStageBytes + 16];  // +16: realignment reads past the end
    __shared__ uint32_t s_sum[kFinWarps];
    __shared__ uint32_t s_prefix[kFinThreads], s_count[kFinThreads];
    __shared__ uint8_t s_member[256];  // exponent is in the codebook
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t T = p.num_tiles, F = gridDim.x;
    const uint32_t t0 = (uint32_t)((uint64_t)blockIdx.x * T / F), t1 = (uint32_t)((uint64_t)(blockIdx.x + 1) * T / F);
    {
        uint8_t cb[16];
        bool contig;
        load_codebook(p.cb, p.cb_dev, BF16 ? 256u : 32u, cb, contig);
        uint32_t member = 0;
#pragma unroll
        for (int k = 0; k < kCodes; k++) member |= cb[k] == tid;
        s_member[tid] = (uint8_t)member;
    }
    // Escapes in all scan tiles before this block's range.  ws_count is
    // 16-byte aligned.
    uint32_t part = 0;
    {
        const uint4* c4 = reinterpret_cast<const uint4*>(p.ws_count);
        const uint32_t q_end = t0 / 4;
#pragma unroll 8
        for (uint32_t q = tid; q < q_end; q += kFinThreads) {
            const uint4 v = c4[q];
            part += v.x + v.y + v.z + v.w;
        }
        if (tid < (t0 & 3u)) part += p.ws_count[(t0 & ~3u) + tid];
    }
    part = __reduce_add_sync(0xFFFFFFFFu, part);
    if (lane == 0) s_sum[warp] = part;
    __syncthreads();
    uint32_t base = 0;
#pragma unroll
    for (uint32_t v = 0; v < kFinWarps; v++) base += s_sum[v];
    __syncthreads();

    uint8_t* const stage = s_stage[warp];
    for (uint32_t c0 = t0; c0 < t1; c0 += kFinThreads) {
        const uint32_t t = c0 + tid;
        const uint32_t cnt = t < t1 ? p.ws_count[t] : 0u;
        uint32_t incl = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= (uint32_t)d) incl += a;
        }
        if (lane == 31) s_sum[warp] = incl;
        __syncthreads();
        uint32_t wbase = 0, total = 0;
#pragma unroll
        for (uint32_t v = 0; v < kFinWarps; v++) {
            wbase += v < warp ? s_sum[v] : 0u;
            total += s_sum[v];
        }
        const uint32_t prefix = base + wbase + incl - cnt;
        s_prefix[tid] = prefix;
        s_count[tid] = cnt;
        if (t < t1) {
            const bool last = t == T - 1;
            if ((t % kScansPerChunk == kScansPerChunk - 1 || last) && p.L.num_chunks > 0) {
                // The chunk's earlier scan tiles: at most kScansPerChunk - 1.
                uint32_t before = 0;
                for (uint32_t k = t - t % kScansPerChunk; k < t; k++) before += p.ws_count[k];
                const uint32_t c = t / kScansPerChunk;
                store_u32_le(p.out + p.L.hdr_off + 8ull * c, prefix - before);
                store_u32_le(p.out + p.L.hdr_off + 8ull * c + 4, before + cnt);
            }
            if (last) {
                const unsigned long long size = p.L.rec_off + 3ull * (prefix + cnt);
                *p.out_bytes = size;
                if (size > p.capacity && p.status) atomicMax(p.status, kStatusCapacity);
            }
        }
        __syncthreads();
        // One warp per scan tile: copy the staged records, or re-derive them.
        const uint32_t batch = min(kFinThreads, t1 - c0);
        for (uint32_t j = warp; j < batch; j += kFinWarps) {
            const uint32_t st = c0 + j, c = s_count[j];
            const uint64_t dst = p.L.rec_off + 3ull * s_prefix[j];
            if (c <= p.ws_cap) {
                // Staged run: 3c bytes at a 16-byte aligned address, inside a
                // region of 3 * ws_cap bytes (a multiple of 16).
                const uint32_t nbytes = 3 * c;
                const uint4* src = reinterpret_cast<const uint4*>(p.ws_rec + (uint64_t)st * 3 * p.ws_cap);
                uint4 v[kStageLoads];
#pragma unroll
                for (uint32_t k = 0; k < kStageLoads; k++)
                    if (16 * lane + 512 * k < nbytes) v[k] = src[lane + 32 * k];
#pragma unroll
                for (uint32_t k = 0; k < kStageLoads; k++)
                    if (16 * lane + 512 * k < nbytes) reinterpret_cast<uint4*>(stage)[lane + 32 * k] = v[k];
                __syncwarp();
                // out + dst + head is 4-byte aligned; bytes before it, and the
                // 0..3 bytes after the last whole word, go one at a time.
                uint8_t* const o = p.out + dst;
                const uint32_t head = min((uint32_t)((4u - (uint32_t)(reinterpret_cast<uintptr_t>(o) & 3u)) & 3u), nbytes);
                const uint32_t words = (nbytes - head) / 4, tail = (nbytes - head) & 3u;
                const uint32_t* sw = reinterpret_cast<const uint32_t*>(stage);
                const uint32_t shift = 8u * (head & 3u);
                for (uint32_t w = lane; w < words; w += 32) {
                    const uint32_t off = head + 4 * w;
                    const uint32_t val = __funnelshift_r(sw[off >> 2], sw[(off >> 2) + 1], shift);
                    if (dst + off + 4 <= p.capacity) {
                        *reinterpret_cast<uint32_t*>(o + off) = val;
                    } else {
#pragma unroll
                        for (uint32_t b = 0; b < 4; b++)
                            if (dst + off + b < p.capacity) o[off + b] = (uint8_t)(val >> (8 * b));
                    }
                }
                if (lane < head + tail) {
                    const uint32_t off = lane < head ? lane : head + 4 * words + (lane - head);
                    if (dst + off < p.capacity) o[off] = stage[off];
                }
                __syncwarp();  // the buffer is reused by the warp's next scan tile
            } else {
                // More escapes than staged: walk the tile in element order,
                // 8 consecutive elements per lane, 256 per step.
                const uint64_t n = p.L.n, end = min((uint64_t)(st + 1) * kScanTile, n);
                uint64_t at = dst;
                for (uint64_t s0 = (uint64_t)st * kScanTile; s0 < end; s0 += 256) {
                    const uint64_t i0 = s0 + 8ull * lane;
                    uint32_t m = 0;
#pragma unroll
                    for (int jj = 0; jj < 8; jj++)
                        if (i0 + jj < end && !s_member[exponent_at<BF16, PAGED>(p, i0 + jj)]) m |= 1u << jj;
                    const uint32_t c8 = __popc(m);
                    uint32_t x = c8;
#pragma unroll
                    for (int d = 1; d < 32; d <<= 1) {
                        const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, x, d);
                        if (lane >= (uint32_t)d) x += a;
                    }
                    uint64_t r = at + 3ull * (x - c8);
                    while (m) {
                        const uint32_t jj = __ffs(m) - 1;
                        m &= m - 1;
                        const uint32_t pos = (uint32_t)(i0 + jj) & 0xFFFFu;
                        if (r + 3 <= p.capacity) {
                            p.out[r] = (uint8_t)pos;
                            p.out[r + 1] = (uint8_t)(pos >> 8);
                            p.out[r + 2] = (uint8_t)exponent_at<BF16, PAGED>(p, i0 + jj);
                        }
                        r += 3;
                    }
                    at += 3ull * __shfl_sync(0xFFFFFFFFu, x, 31);
                }
            }
        }
        base += total;
        __syncthreads();
    }
}

cudaError_t launch_finish(const EncodeParams& p, bool bf16, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    // Several blocks per SM: the record copies are latency bound.
    const uint64_t want = (uint64_t)4 * sms;
    const uint32_t grid = (uint32_t)(p.num_tiles < want ? p.num_tiles : want);
    const bool paged = p.pm.ids != nullptr;
    if (bf16)
        paged ? finish_kernel<true, true><<<grid, kFinThreads, 0, s>>>(p)
              : finish_kernel<true, false><<<grid, kFinThreads, 0, s>>>(p);
    else
        paged ? finish_kernel<false, true><<<grid, kFinThreads, 0, s>>>(p)
              : finish_kernel<false, false><<<grid, kFinThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sz
