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
//    escape stream: asynchronous 16-byte copies of the staged run into
//    shared memory (the next run's while this one leaves), then aligned
//    16-byte stores (funnel shifts realign the bytes) with at most 15 single
//    bytes at either end;
//  * a scan tile with more than ws_cap escapes has its ws_cap staged records
//    copied the same way; the rest are re-derived from the input unit by
//    unit (1,024 elements each for BF16, 4,096 for E5M2, whose escape counts
//    the encoders also left in the workspace, so every unit's first record
//    index is known).  The units holding unstaged records are spread over
//    all warps of the block: a warp loads its unit with all 16-byte loads in
//    flight, finds the escapes (byte arithmetic for a contiguous codebook,
//    a membership table otherwise) and ranks them (a warp scan), assembles
//    their records in its staging buffer and writes them with the same
//    aligned stores.  This path runs out of line, one call per heavy scan
//    tile and warp, so that it leaves the common path's registers alone;
//  * a chunk's last scan tile writes the chunk's header (offset = escapes
//    before the chunk, count = escapes in it); the last scan tile writes the
//    stream size;
//  * the last block writes the call's status word once: the largest error
//    code of the encode blocks and its own capacity check.
// Escapes are (u16 position in the 65,536-element chunk, u8 exponent) pairs
// in element order (SplitZip technical summary, gist.science/es,
// "Metodologia: SplitZip" > "Flujo de Escape").
#include "sz_device.cuh"
#include "sz_params.h"
#include "sz_pipeline.cuh"

namespace sz {

namespace {

constexpr uint32_t kFinThreads = 256;
constexpr uint32_t kFinWarps = kFinThreads / 32;
constexpr uint32_t kScansPerChunk = kChunk / kScanTile;
constexpr uint32_t kPieceRecs = 1024;                     // records a warp re-derives at a time
constexpr uint32_t kStageBytes = 3 * kPieceRecs;          // a warp's staging buffer
constexpr uint32_t kHalfRecs = kPieceRecs / 2;            // staged records per half of it
constexpr uint32_t kHalfStride = 3 * kHalfRecs + 16;      // second half: 16-byte aligned, a gap after the first
static_assert((3 * kHalfRecs) % 512 == 0 && kHalfStride % 16 == 0, "whole warp-wide 16-byte loads");
static_assert(kHalfStride + 3 * kHalfRecs + 16 <= kStageBytes + 32, "both halves, and the reads past them, fit");
static_assert(kChunk % kScanTile == 0, "scan tiles must not straddle chunks");

// Copy nbytes from shared memory (src, 4-byte aligned, readable up to 4 bytes
// past the end) to out + dst with aligned 16-byte stores (funnel shifts
// realign the bytes); the 0..15 bytes before the first aligned piece and
// after the last go one at a time.  Bytes at or beyond `capacity` are not
// written.  Threads tid = 0, step, 2 step, ... share the work.
__device__ __forceinline__ void copy_out(const uint8_t* src, uint32_t nbytes, uint8_t* out, uint64_t dst,
                                         uint64_t capacity, uint32_t tid, uint32_t step) {
    uint8_t* const o = out + dst;
    const uint32_t head = min((uint32_t)((16u - (uint32_t)(reinterpret_cast<uintptr_t>(o) & 15u)) & 15u), nbytes);
    const uint32_t pieces = (nbytes - head) / 16, tail = (nbytes - head) & 15u;
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(src);
    const uint32_t shift = 8u * (head & 3u);
    for (uint32_t c = tid; c < pieces; c += step) {
        const uint32_t off = head + 16 * c, i = off >> 2;
        const uint4 v = make_uint4(__funnelshift_r(sw[i], sw[i + 1], shift), __funnelshift_r(sw[i + 1], sw[i + 2], shift),
                                   __funnelshift_r(sw[i + 2], sw[i + 3], shift), __funnelshift_r(sw[i + 3], sw[i + 4], shift));
        if (dst + off + 16 <= capacity) {
            *reinterpret_cast<uint4*>(o + off) = v;
        } else {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (uint32_t b = 0; b < 16; b++)
                if (dst + off + b < capacity) o[off + b] = (uint8_t)(w[b >> 2] >> (8 * (b & 3)));
        }
    }
    for (uint32_t e = tid; e < head + tail; e += step) {
        const uint32_t off = e < head ? e : head + 16 * pieces + (e - head);
        if (dst + off < capacity) o[off] = src[off];
    }
}

// One warp copies a staged run of c records (run: 16-byte aligned, readable
// in whole 16-byte pieces up to 3 c rounded up) to out + dst, 1,024 records
// at a time through buf (the warp's whole staging buffer): every piece of a
// round is in flight at once.  Not inlined, like the re-derivation: it
// serves only runs longer than half the buffer.
__device__ __noinline__ void copy_run(const uint8_t* run, uint32_t c, uint8_t* out, uint64_t dst, uint64_t capacity,
                                      uint8_t* buf) {
    const uint32_t lane = threadIdx.x & 31u;
    for (uint32_t q = 0; q < c; q += kPieceRecs) {
        const uint32_t nbytes = 3 * min(kPieceRecs, c - q);
        for (uint32_t b = 16 * lane; b < nbytes; b += 512) cp_async16(buf + b, run + 3ull * q + b, 16);
        cp_async_commit();
        cp_async_wait_all();
        __syncwarp();
        copy_out(buf, nbytes, out, dst + 3ull * q, capacity, lane, 32);
        __syncwarp();  // buf is reused next
    }
}

// The 8 records of a group of 8 consecutive escaped elements, 24 bytes, at
// byte offset a of the staging buffer: record j is (pos0 + j as u16, the
// exponent in byte j & 3 of ex[j >> 2]).  pos0 is a multiple of 8, so the
// eight positions share their high byte and the low bytes do not carry.
// The words are assembled with byte permutes from two position pairs and
// the exponent words; a start that is not word aligned takes funnel shifts
// for the middle words and single bytes at both ends (those words are
// shared with the neighbouring records).
__device__ __forceinline__ void put_full_group(uint8_t* buf, uint32_t a, uint32_t pos0, uint32_t ex0, uint32_t ex1) {
    const uint32_t A = pos0 * 0x10001u + 0x10000u;  // pos0 | (pos0 + 1) << 16
    const uint32_t B = A + 0x20002u, C = A + 0x40004u, D = A + 0x60006u;
    const uint32_t w[6] = {__byte_perm(A, ex0, 0x2410), __byte_perm(B, ex0, 0x1051), __byte_perm(B, ex0, 0x7326),
                           __byte_perm(C, ex1, 0x2410), __byte_perm(D, ex1, 0x1051), __byte_perm(D, ex1, 0x7326)};
    uint32_t* bw = reinterpret_cast<uint32_t*>(buf) + (a >> 2);
    const uint32_t s = a & 3u;
    if (s == 0) {
#pragma unroll
        for (int k = 0; k < 6; k++) bw[k] = w[k];
    } else {
        const uint32_t sh = 8 * s;
#pragma unroll
        for (int k = 1; k < 6; k++) bw[k] = __funnelshift_l(w[k - 1], w[k], sh);
        for (uint32_t b = 0; b < 4 - s; b++) buf[a + b] = (uint8_t)(w[0] >> (8 * b));
        for (uint32_t b = 0; b < s; b++) buf[a + 24 - s + b] = (uint8_t)(w[5] >> (8 * (4 - s + b)));
    }
}

// The records of 1,024 elements of a scan tile that did not fit the staged
// ones, re-derived from the input and written by one warp at byte offset dst
// of the stream, in element order: those of local rank >= skip (the ones
// below are among the staged records).  Returns how many escapes the 1,024
// elements hold.  The
// unit is kU pieces of 16 bytes per lane (piece u * 32 + lane), all loaded
// before any is examined.  buf: the warp's staging buffer (kStageBytes + 32
// bytes, 16-byte aligned), which holds the 1,024 records a unit can have.
// cb_test (shared memory): {the codebook is cb0 .. cb0 + 15, cbk}.  With a
// contiguous codebook membership is tested with byte arithmetic instead of
// lookups in s_member (a byte per exponent, whose random banks conflict);
// cbk is (256 - cb0) mod 256 (BF16) or cb0 (E5M2) in every byte.
template <bool BF16, bool PAGED>
__device__ __forceinline__ uint32_t rederive_unit(const EncodeParams& p, uint64_t ubase, uint32_t skip, uint64_t dst,
                                               const uint8_t* s_member, const uint32_t* cb_test, uint8_t* buf) {
    constexpr uint32_t kPer = BF16 ? 8u : 16u;  // elements in 16 bytes
    constexpr uint32_t kEsize = BF16 ? 2u : 1u;
    constexpr uint32_t kU = kUnitElems / (32 * kPer);  // 4 (BF16) or 2 (E5M2)
    static_assert(3 * kUnitElems <= kStageBytes, "a unit's records fit the staging buffer");
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t n = p.L.n;
    const uint64_t end = min(ubase + kUnitElems, n);
    const bool vec = (reinterpret_cast<uintptr_t>(p.in) % 16) == 0;  // a paged pool is 16-byte aligned too
    uint32_t w[kU][4], valid[kU];
#pragma unroll
    for (uint32_t u = 0; u < kU; u++) {
        const uint64_t i0 = ubase + (uint64_t)(u * 32 + lane) * kPer;
        w[u][0] = w[u][1] = w[u][2] = w[u][3] = 0;
        valid[u] = i0 >= end ? 0u : (end - i0 >= kPer ? kPer : (uint32_t)(end - i0));
        if (vec && valid[u] == kPer) {
            // A piece of 16 bytes never straddles a page (pages are a power
            // of two of at least 16 elements).
            // A bad page id was already reported by the encode kernel.
            const uint4 v = ld_stream_v4(p.in + elem_offset<PAGED>(p.pm, i0, kEsize, nullptr));
            w[u][0] = v.x, w[u][1] = v.y, w[u][2] = v.z, w[u][3] = v.w;
        } else {
#pragma unroll
            for (uint32_t j = 0; j < kPer; j++) {
                if (j < valid[u]) {
                    const uint8_t* e = p.in + elem_offset<PAGED>(p.pm, i0 + j, kEsize, nullptr);
                    const uint32_t v = BF16 ? ((uint32_t)e[0] | ((uint32_t)e[1] << 8)) : (uint32_t)e[0];
                    w[u][j / (4 / kEsize)] |= v << (8 * kEsize * (j % (4 / kEsize)));
                }
            }
        }
    }
    uint32_t before = 0;  // records of the unit before piece row u
#pragma unroll
    for (uint32_t u = 0; u < kU; u++) {
        // The exponent bytes of the piece, four elements per word.
        uint32_t ex[kPer / 4];
        if (BF16) {
            // Element pairs: low byte = exponent bit 0 | mantissa, high byte
            // = sign | exponent bits 7..1.
#pragma unroll
            for (uint32_t g = 0; g < 2; g++) {
                const uint32_t lo = __byte_perm(w[u][2 * g], w[u][2 * g + 1], 0x6420);
                const uint32_t hi = __byte_perm(w[u][2 * g], w[u][2 * g + 1], 0x7531);
                ex[g] = ((hi << 1) & 0xFEFEFEFEu) | ((lo >> 7) & 0x01010101u);
            }
        } else {
#pragma unroll
            for (uint32_t g = 0; g < 4; g++) ex[g] = (w[u][g] >> 2) & 0x1F1F1F1Fu;
        }
        uint32_t mask = 0;
        if (cb_test[0]) {
            const uint32_t cbk = cb_test[1];
            // Per byte x = 128 + (exponent - cb0 modulo 256): the element is
            // in the codebook iff x lies in 128 .. 143, that is bit 7 set and
            // bits 4..6 clear.
#pragma unroll
            for (uint32_t g = 0; g < kPer / 4; g++) {
                const uint32_t e = ex[g];
                // BF16: a byte-wise add of (256 - cb0) without carries between
                // bytes (low 7 bits added, bit 7 by exclusive or), then bit 7
                // flipped.  E5M2: exponents <= 31 and cb0 <= 16 leave no
                // borrow.
                const uint32_t x = BF16 ? (((e & 0x7F7F7F7Fu) + (cbk & 0x7F7F7F7Fu)) ^ ((e ^ cbk) & 0x80808080u)) ^ 0x80808080u
                                        : (e | 0x80808080u) - cbk;
                const uint32_t hi3 = ((x & 0x70707070u) + 0x70707070u) & 0x80808080u;  // bits 4..6 not all clear
                const uint32_t out = (~x | hi3) & 0x80808080u;                            // bit 7: an escape
                mask |= (((out >> 7) * 0x00204081u) >> 21 & 0xFu) << (4 * g);            // bits 0, 8, 16, 24 -> 0..3
            }
            if (valid[u] < kPer) mask &= (1u << valid[u]) - 1u;
        } else {
#pragma unroll
            for (uint32_t j = 0; j < kPer; j++)
                if (j < valid[u] && !s_member[(ex[j >> 2] >> (8 * (j & 3))) & 0xFFu]) mask |= 1u << j;
        }
        const uint32_t c = __popc(mask);
        uint32_t x = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, x, d);
            if (lane >= (uint32_t)d) x += a;
        }
        uint32_t r = before + x - c;  // unit-local rank of this piece's first record
        const uint32_t pos0 = (uint32_t)(ubase + (uint64_t)(u * 32 + lane) * kPer) & 0xFFFFu;
        // Groups of 8 elements: when the group of every lane is 8 escapes
        // (all-escape data), each lane writes its 24 bytes as six words;
        // otherwise record by record.
#pragma unroll
        for (uint32_t g = 0; g < kPer / 8; g++) {
            const uint32_t m8 = (mask >> (8 * g)) & 0xFFu;
            // Only when every lane of the warp takes this path: lanes that
            // diverge would pay for both.
            if (__all_sync(0xFFFFFFFFu, m8 == 0xFFu && r >= skip)) {
                put_full_group(buf, 3 * (r - skip), pos0 + 8 * g, ex[2 * g], ex[2 * g + 1]);
                r += 8;
            } else {
#pragma unroll
                for (uint32_t j = 0; j < 8; j++) {
                    if ((m8 >> j) & 1u) {
                        if (r >= skip) {
                            const uint32_t pos = pos0 + 8 * g + j;
                            uint8_t* b = buf + 3 * (r - skip);
                            b[0] = (uint8_t)pos;
                            b[1] = (uint8_t)(pos >> 8);
                            b[2] = (uint8_t)(ex[2 * g + (j >> 2)] >> (8 * (j & 3)));
                        }
                        r++;
                    }
                }
            }
        }
        before += __shfl_sync(0xFFFFFFFFu, x, 31);
    }
    __syncwarp();
    copy_out(buf, before > skip ? 3 * (before - skip) : 0u, p.out, dst, p.capacity, lane, 32);
    __syncwarp();  // buf is reused by the warp's next unit
    return before;  // the escapes of these 1,024 elements
}

// The units of one heavy scan tile that this warp takes (every kFinWarps-th
// of those set in `units`, from the lowest): each unit's records of
// tile-local rank >= ws_cap go out, in steps of 1,024 elements (one step
// for a BF16 unit).  ufirst (lane u): the tile's escapes before unit u;
// prefix: the tile's first record index in the stream.  Not inlined: it
// runs only for scan tiles beyond their staging, and kept apart it leaves
// the registers of the kernel's common path alone.
template <bool BF16, bool PAGED>
__device__ __noinline__ void rederive_units(const EncodeParams& p, uint64_t tbase, uint32_t units, uint32_t ufirst,
                                            uint32_t prefix, const uint8_t* s_member, const uint32_t* cb_test,
                                            uint8_t* stage) {
    constexpr uint32_t kUnit = BF16 ? kUnitElems : kUnitElemsE5;
    while (units) {
        const uint32_t u = __ffs(units) - 1;
        for (uint32_t q = 0; q < kFinWarps && units; q++) units &= units - 1;  // the next one is 8 on
        const uint32_t f = __shfl_sync(0xFFFFFFFFu, ufirst, u);
        uint32_t done = 0;  // escapes of the unit's earlier steps
        for (uint32_t e = 0; e < kUnit; e += kUnitElems) {
            const uint32_t at = f + done;  // tile-local rank of the step's first escape
            const uint32_t skip = p.ws_cap > at ? p.ws_cap - at : 0u;
            const uint64_t dst = p.L.rec_off + 3ull * ((uint64_t)prefix + at + skip);
            done += rederive_unit<BF16, PAGED>(p, tbase + (uint64_t)u * kUnit + e, skip, dst, s_member, cb_test, stage);
        }
    }
}

}  // namespace

template <bool BF16, bool PAGED>
__global__ void __launch_bounds__(kFinThreads, 4) finish_kernel(const EncodeParams p) {
    __shared__ __align__(16) uint8_t s_stage[kFinWarps][kStageBytes + 32];  // +32: realignment reads past the end
    __shared__ uint32_t s_sum[kFinWarps];
    __shared__ uint32_t s_prefix[kFinThreads], s_count[kFinThreads];
    __shared__ uint8_t s_heavy[kFinThreads];  // the batch's heavy tiles, in order
    __shared__ uint32_t s_nheavy[kFinWarps];
    __shared__ uint8_t s_member[256];  // exponent is in the codebook
    __shared__ int s_err;              // last block: the capacity error, then the call's status
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t T = p.num_tiles, F = gridDim.x;
    const uint32_t t0 = (uint32_t)((uint64_t)blockIdx.x * T / F), t1 = (uint32_t)((uint64_t)(blockIdx.x + 1) * T / F);
    // The re-derivation's membership test: {contiguous codebook, its constant}
    // (see rederive_unit).
    __shared__ uint32_t s_cb_test[2];
    {
        uint8_t cb[16];
        bool contig;
        load_codebook(p.cb, p.cb_dev, BF16 ? 256u : 32u, cb, contig);
        if (tid == 0) {
            s_cb_test[0] = contig;
            s_cb_test[1] = 0x01010101u * (BF16 ? (256u - cb[0]) & 0xFFu : (uint32_t)cb[0]);
        }
        uint32_t member = 0;
#pragma unroll
        for (int k = 0; k < kCodes; k++) member |= cb[k] == tid;
        s_member[tid] = (uint8_t)member;
        if (tid == 0) s_err = 0;
    }
    // The kernel is launched as a programmatic dependent of the encode
    // kernel, so the lines above overlap its tail; everything below reads
    // what it wrote, once it has finished (no wait without that launch).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Escapes in all scan tiles before this block's range.  ws_count is
    // 16-byte aligned.  Bit 31 of a count is the E5M2 encoder's error flag
    // (kCountError); the last block, which reads every count, collects it.
    uint32_t part = 0, flags = 0;
    {
        const uint4* c4 = reinterpret_cast<const uint4*>(p.ws_count);
        const uint32_t q_end = t0 / 4;
#pragma unroll 8
        for (uint32_t q = tid; q < q_end; q += kFinThreads) {
            const uint4 v = c4[q];
            part += (v.x & ~kCountError) + (v.y & ~kCountError) + (v.z & ~kCountError) + (v.w & ~kCountError);
            flags |= v.x | v.y | v.z | v.w;
        }
        if (tid < (t0 & 3u)) {
            const uint32_t v = p.ws_count[(t0 & ~3u) + tid];
            part += v & ~kCountError;
            flags |= v;
        }
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
        const uint32_t cword = t < t1 ? p.ws_count[t] : 0u;
        const uint32_t cnt = cword & ~kCountError;
        flags |= cword;
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
                for (uint32_t k = t - t % kScansPerChunk; k < t; k++) before += p.ws_count[k] & ~kCountError;
                const uint32_t c = t / kScansPerChunk;
                store_u32_le(p.out + p.L.hdr_off + 8ull * c, prefix - before);
                store_u32_le(p.out + p.L.hdr_off + 8ull * c + 4, before + cnt);
            }
            if (last) {
                const unsigned long long size = p.L.rec_off + 3ull * (prefix + cnt);
                *p.out_bytes = size;
                if (size > p.capacity) s_err = kStatusCapacity;  // the last block's own
            }
        }
        // The batch's heavy tiles (more escapes than staged), in order.
        const uint32_t batch = min(kFinThreads, t1 - c0);
        const bool is_heavy = tid < batch && cnt > p.ws_cap;
        // The barrier that publishes s_prefix and s_count (and lets s_sum be
        // rewritten) also tells whether the batch has heavy tiles at all (the
        // common case has none).
        const bool any_heavy = __syncthreads_or(is_heavy);
        uint32_t nheavy = 0;
        if (any_heavy) {
            const uint32_t hb = __ballot_sync(0xFFFFFFFFu, is_heavy);
            if (lane == 0) s_nheavy[warp] = __popc(hb);
            __syncthreads();
            uint32_t hbefore = 0;
#pragma unroll
            for (uint32_t v = 0; v < kFinWarps; v++) {
                hbefore += v < warp ? s_nheavy[v] : 0u;
                nheavy += s_nheavy[v];
            }
            if (is_heavy) s_heavy[hbefore + __popc(hb & ((1u << lane) - 1u))] = (uint8_t)tid;
        }
        // One warp per scan tile: copy its staged records (all of them, or
        // the first ws_cap of a heavier tile).  The warp's staging buffer has
        // two halves of 512 records: a run that fits one (the common case)
        // arrives there by asynchronous copies while the warp writes out the
        // run before it, so a warp's runs cost one memory round trip instead
        // of one each.  A longer run takes the whole buffer, 1,024 records
        // (one round trip) at a time.
        auto fits = [&](uint32_t j) { return min(s_count[j], p.ws_cap) <= kHalfRecs; };
        auto prefetch = [&](uint32_t j, uint32_t h) {  // whole warp; one commit group
            const uint32_t nbytes = 3 * min(s_count[j], p.ws_cap);
            const uint8_t* run = p.ws_rec + (uint64_t)(c0 + j) * 3 * p.ws_cap;
            // Whole 16-byte pieces stay inside the run's region (3 ws_cap
            // bytes, a multiple of 16, starting 16-byte aligned).
            for (uint32_t b = 16 * lane; b < nbytes; b += 512) cp_async16(stage + h * kHalfStride + b, run + b, 16);
            cp_async_commit();
        };
        uint32_t h = 0;
        bool ready = warp < batch && fits(warp);  // run j is on its way into half h
        if (ready) prefetch(warp, 0);
        for (uint32_t j = warp; j < batch; j += kFinWarps) {
            const uint32_t c = min(s_count[j], p.ws_cap);
            const uint64_t dst = p.L.rec_off + 3ull * s_prefix[j];
            const uint32_t jn = j + kFinWarps;
            const bool next = jn < batch && fits(jn);
            if (ready) {
                if (next) prefetch(jn, h ^ 1u);
                if (next)
                    cp_async_wait_group<1>();
                else
                    cp_async_wait_all();
                __syncwarp();
                copy_out(stage + h * kHalfStride, 3 * c, p.out, dst, p.capacity, lane, 32);
                __syncwarp();  // the half is refilled two runs later
                h ^= 1u;
            } else {
                // A longer run takes the whole buffer (no copy is in flight
                // into it), 1,024 records at a time; the next run is fetched
                // afterwards.
                copy_run(p.ws_rec + (uint64_t)(c0 + j) * 3 * p.ws_cap, c, p.out, dst, p.capacity, stage);
                if (next) prefetch(jn, 0);
                h = 0;
            }
            ready = next;
        }
        if (any_heavy) __syncthreads();  // s_heavy complete (block-uniform)
        // The units that hold the heavy tiles' remaining records are
        // re-derived, spread over all warps of the block.  Every warp walks
        // the same list of such units in the same order (heavy tiles in tile
        // order, units in element order) and takes every kFinWarps-th one, so
        // the units of one tile run side by side.
        // Lane u of the warp holds the escape count of unit u of a heavy tile
        // (32 units of 1,024 elements for BF16, 8 of 4,096 for E5M2; units
        // past n were never written: 0); the next tile's counts are loaded
        // while this one's units are re-derived.
        constexpr uint32_t kUnit = BF16 ? kUnitElems : kUnitElemsE5;
        constexpr uint32_t kUnits = kScanTile / kUnit;
        auto unit_count = [&](uint32_t h) -> uint32_t {
            if (h >= nheavy) return 0u;
            const uint32_t st = c0 + s_heavy[h];
            const bool in_range = lane < kUnits && (uint64_t)st * kScanTile + (uint64_t)lane * kUnit < p.L.n;
            return in_range ? (uint32_t)p.ws_unit[(uint64_t)st * kUnitsPerScan + lane] : 0u;
        };
        uint32_t k = 0;  // running index of the units walked so far
        uint32_t uc_next = unit_count(0);
        for (uint32_t h = 0; h < nheavy; h++) {
            const uint32_t j = s_heavy[h];
            const uint64_t tbase = (uint64_t)(c0 + j) * kScanTile;
            const uint32_t uc = uc_next;
            uc_next = unit_count(h + 1);
            uint32_t incl = uc;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= (uint32_t)d) incl += a;
            }
            const uint32_t ufirst = incl - uc;  // escapes of the tile before this unit
            uint32_t units = __ballot_sync(0xFFFFFFFFu, uc > 0 && incl > p.ws_cap);
            // This warp's units of the tile: running index = warp mod kFinWarps.
            uint32_t skip_units = (warp - k % kFinWarps + kFinWarps) % kFinWarps;
            k += __popc(units);
            while (units && skip_units) {
                units &= units - 1;
                skip_units--;
            }
            if (units) rederive_units<BF16, PAGED>(p, tbase, units, ufirst, s_prefix[j], s_member, s_cb_test, stage);
        }
        base += total;
        __syncthreads();
    }
    // The call's status, written once, by the last block: the largest error
    // code of the encode (a timed-out wait, a bad device codebook, a bad page
    // id) and its own (capacity).  So the status word needs no reset before
    // the call.
    if (blockIdx.x == F - 1 && p.status) {
        // BF16: one error word per encode block (p.grid of them, a few
        // hundred); E5M2: the flags in the counts (p.grid is 0).
        int e = (flags & kCountError) ? kStatusInvalid : 0;
        for (uint32_t b = tid; b < p.grid; b += kFinThreads) e = max(e, p.ws_err[b]);
        e = __reduce_max_sync(0xFFFFFFFFu, e);
        if (lane == 0 && e) atomicMax(&s_err, e);
        __syncthreads();
        if (tid == 0) *p.status = s_err;
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
