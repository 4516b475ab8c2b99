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
//    most 3 single bytes at either end;
//  * a scan tile with more than ws_cap escapes has its ws_cap staged records
//    copied by its warp, which then walks the rest of the tile (after the
//    last staged position) again, in element order, 512 (BF16) or 1,024
//    (E5M2) elements per step: 16-byte loads (all of a step's in flight at
//    once), a warp scan of the escape counts, the step's records assembled
//    in the warp's staging buffer and written with the same aligned word
//    stores;
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

// Copy nbytes from shared memory (src, 4-byte aligned, readable up to 4 bytes
// past the end) to out + dst with aligned 4-byte stores; the 0..3 bytes
// before the first aligned word and after the last go one at a time.  Bytes
// at or beyond `capacity` are not written.  Threads tid = 0, step, 2 step, ...
// share the work.
__device__ __forceinline__ void copy_out(const uint8_t* src, uint32_t nbytes, uint8_t* out, uint64_t dst,
                                         uint64_t capacity, uint32_t tid, uint32_t step) {
    uint8_t* const o = out + dst;
    const uint32_t head = min((uint32_t)((4u - (uint32_t)(reinterpret_cast<uintptr_t>(o) & 3u)) & 3u), nbytes);
    const uint32_t words = (nbytes - head) / 4, tail = (nbytes - head) & 3u;
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(src);
    const uint32_t shift = 8u * (head & 3u);
    for (uint32_t w = tid; w < words; w += step) {
        const uint32_t off = head + 4 * w;
        const uint32_t val = __funnelshift_r(sw[off >> 2], sw[(off >> 2) + 1], shift);
        if (dst + off + 4 <= capacity) {
            *reinterpret_cast<uint32_t*>(o + off) = val;
        } else {
#pragma unroll
            for (uint32_t b = 0; b < 4; b++)
                if (dst + off + b < capacity) o[off + b] = (uint8_t)(val >> (8 * b));
        }
    }
    if (tid < head + tail) {
        const uint32_t off = tid < head ? tid : head + 4 * words + (tid - head);
        if (dst + off < capacity) o[off] = src[off];
    }
}

// The records of scan tile st, which has more escapes than the ws_cap it
// staged, written by one warp at byte offset dst of the stream (element
// order): the staged records first (they are the tile's first ws_cap
// escapes), then the ones after the last staged position, re-derived from
// the input.  A step covers kU pieces of 16 bytes per lane
// (piece u * 32 + lane of the step), all loaded before any is examined.
// buf: the warp's staging buffer (kStageBytes + 16 bytes, 16-byte aligned).
template <bool BF16, bool PAGED>
__device__ void rederive_tile(const EncodeParams& p, uint32_t st, uint64_t dst, const uint8_t* s_member, uint8_t* buf) {
    constexpr uint32_t kPer = BF16 ? 8u : 16u;  // elements in 16 bytes
    constexpr uint32_t kEsize = BF16 ? 2u : 1u;
    constexpr uint32_t kU = 2;
    constexpr uint32_t kStep = 32 * kU * kPer;  // 512 (BF16) or 1,024 (E5M2) elements
    static_assert(3 * kStep <= kStageBytes && kScanTile % kStep == 0, "a step's records fit the staging buffer");
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t n = p.L.n, begin = (uint64_t)st * kScanTile;
    const uint64_t end = min(begin + kScanTile, n);
    const bool vec = (reinterpret_cast<uintptr_t>(p.in) % 16) == 0;  // a paged pool is 16-byte aligned too
    auto exponent = [](const uint32_t (&w)[4], uint32_t j) {
        return BF16 ? (w[j >> 1] >> (7 + 16 * (j & 1))) & 0xFFu : (w[j >> 2] >> (8 * (j & 3) + 2)) & 0x1Fu;
    };
    uint64_t at = dst;
    uint64_t resume = begin;  // first element not covered by the staged records
    if (p.ws_cap > 0) {
        // 3 ws_cap bytes (a multiple of 16, at most kStageBytes) at a 16-byte
        // aligned address.
        const uint32_t nb = 3 * p.ws_cap;
        const uint4* src = reinterpret_cast<const uint4*>(p.ws_rec + (uint64_t)st * nb);
        for (uint32_t k = lane; k < nb / 16; k += 32) reinterpret_cast<uint4*>(buf)[k] = src[k];
        __syncwarp();
        const uint32_t last = (uint32_t)buf[nb - 3] | ((uint32_t)buf[nb - 2] << 8);
        resume = (begin & ~(uint64_t)(kChunk - 1)) + last + 1;
        copy_out(buf, nb, p.out, at, p.capacity, lane, 32);
        at += nb;
        __syncwarp();  // buf is reused below
    }
    for (uint64_t s0 = begin + (resume - begin) / kStep * kStep; s0 < end; s0 += kStep) {
        uint32_t w[kU][4], m[kU];
#pragma unroll
        for (uint32_t u = 0; u < kU; u++) {
            const uint64_t i0 = s0 + (uint64_t)(u * 32 + lane) * kPer;
            w[u][0] = w[u][1] = w[u][2] = w[u][3] = 0;
            m[u] = 0;
            if (i0 < end && i0 + kPer > resume) {
                const uint32_t valid = end - i0 >= kPer ? kPer : (uint32_t)(end - i0);
                // Elements [skip, valid) of the piece are examined.
                const uint32_t skip = resume > i0 ? (uint32_t)(resume - i0) : 0u;
                m[u] = valid | (skip << 8);  // until the mask replaces it
                if (vec && valid == kPer) {
                    // A piece of 16 bytes never straddles a page (pages are a
                    // power of two of at least 16 elements).
                    const uint4 v = *reinterpret_cast<const uint4*>(p.in + elem_offset<PAGED>(p.pm, i0, kEsize, p.status));
                    w[u][0] = v.x, w[u][1] = v.y, w[u][2] = v.z, w[u][3] = v.w;
                } else {
#pragma unroll
                    for (uint32_t j = 0; j < kPer; j++) {
                        if (j < valid) {
                            const uint8_t* e = p.in + elem_offset<PAGED>(p.pm, i0 + j, kEsize, p.status);
                            const uint32_t v = BF16 ? ((uint32_t)e[0] | ((uint32_t)e[1] << 8)) : (uint32_t)e[0];
                            w[u][j / (4 / kEsize)] |= v << (8 * kEsize * (j % (4 / kEsize)));
                        }
                    }
                }
            }
        }
        uint32_t before = 0;  // records of the step before slice u
#pragma unroll
        for (uint32_t u = 0; u < kU; u++) {
            const uint32_t valid = m[u] & 0xFFu, skip = m[u] >> 8;
            uint32_t mask = 0;
#pragma unroll
            for (uint32_t j = 0; j < kPer; j++)
                if (j >= skip && j < valid && !s_member[exponent(w[u], j)]) mask |= 1u << j;
            const uint32_t c = __popc(mask);
            uint32_t x = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, x, d);
                if (lane >= (uint32_t)d) x += a;
            }
            uint32_t r = 3 * (before + x - c);
            const uint32_t i0 = (uint32_t)(s0 + (uint64_t)(u * 32 + lane) * kPer);
#pragma unroll
            for (uint32_t j = 0; j < kPer; j++) {
                if ((mask >> j) & 1u) {
                    const uint32_t pos = (i0 + j) & 0xFFFFu;
                    buf[r] = (uint8_t)pos;
                    buf[r + 1] = (uint8_t)(pos >> 8);
                    buf[r + 2] = (uint8_t)exponent(w[u], j);
                    r += 3;
                }
            }
            before += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
        __syncwarp();
        copy_out(buf, 3 * before, p.out, at, p.capacity, lane, 32);
        at += 3ull * before;
        __syncwarp();  // buf is reused by the next step
    }
}

}  // namespace

template <bool BF16, bool PAGED>
__global__ void __launch_bounds__(kFinThreads, 4) finish_kernel(const EncodeParams p) {
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
    // The kernel is launched as a programmatic dependent of the encode
    // kernel, so the lines above overlap its tail; everything below reads
    // what it wrote, once it has finished (no wait without that launch).
    asm volatile("griddepcontrol.wait;" ::: "memory");
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
        // One warp per scan tile: copy its staged records, or re-derive them.
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
                copy_out(stage, nbytes, p.out, dst, p.capacity, lane, 32);
                __syncwarp();  // the buffer is reused by the warp's next scan tile
            } else {
                rederive_tile<BF16, PAGED>(p, st, dst, s_member, stage);
            }
        }
        base += total;
        __syncthreads();
    }
}

cudaError_t launch_finish(const EncodeParams& p, bool bf16, cudaStream_t s) {
    int sms = 0, per_sm = 0;
    cudaError_t err = kernel_fit((const void*)finish_kernel<true, false>, kFinThreads, 0, &sms, &per_sm);
    if (err != cudaSuccess) return err;
    // Several blocks per SM: the record copies are latency bound.
    const uint64_t want = (uint64_t)4 * sms;
    const uint32_t grid = (uint32_t)(p.num_tiles < want ? p.num_tiles : want);
    const bool paged = p.pm.ids != nullptr;
    auto kern = bf16 ? (paged ? finish_kernel<true, true> : finish_kernel<true, false>)
                     : (paged ? finish_kernel<false, true> : finish_kernel<false, false>);
    // A programmatic dependent of the encode kernel ahead of it.
    return launch_dependent(kern, dim3(grid), dim3(kFinThreads), 0, s, p);
}

}  // namespace sz
