// sz_bf16.cu -- SplitZip BF16 encode and decode kernels for sm_103a.
//
// Method: SplitZip technical summary (gist.science/es), "Metodologia:
// SplitZip", items "Estrategia de Codificacion" (split, top-16 4-bit codes,
// two per byte, (u16 position, u8 exponent) escapes) and "Estrategia de
// Decodificacion" (parallel LUT pass, then escape overwrite).
//
// Work layout.  A block of 256 threads owns a tile of 8192 elements (eight
// tiles per 65,536-element chunk).  Warp w owns tile elements
// [1024w, 1024w + 1024); inside it, lane l's k-th group of 8 elements starts
// at 1024w + 256k + 8l.  Every global access of a group is therefore one fully
// coalesced warp instruction: 16 B/lane of BF16 input or output, 8 B/lane of
// sign|mantissa bytes, 4 B/lane of nibbles.  The tile's element order is
// (k, lane, j) inside each warp, which is the order escapes are ranked in.
#include "sz_device.cuh"
#include "sz_params.h"

namespace sz {

namespace {

constexpr uint32_t kTilesPerChunk = kChunk / kBf16Tile;  // 8
static_assert(kChunk % kBf16Tile == 0, "tiles must not straddle chunks");
constexpr uint32_t kWarps = kBf16Threads / 32;

__device__ __forceinline__ uint64_t group_start(uint64_t base, uint32_t warp, uint32_t k, uint32_t lane) {
    return base + warp * 1024u + k * 256u + lane * 8u;
}

// sign|mantissa bytes of the two BF16 values in a 32-bit word, at bytes 0 and 2.
__device__ __forceinline__ uint32_t sm_pair(uint32_t w) {
    return (w & 0x007F007Fu) | ((w >> 8) & 0x00800080u);
}

}  // namespace

// ---------------------------------------------------------------------------
// Encode.  One pass: dense streams are stored as soon as they are computed;
// the tile's escapes are ranked (warp ballot/popc scans, then a block scan),
// staged in shared memory, and copied out once the decoupled look-back has
// given the number of escapes in all earlier tiles.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBf16Threads) encode_bf16_kernel(const EncodeParams p) {
    __shared__ uint8_t s_code[256];              // exponent -> code; 0x10 marks an escape
    __shared__ uint8_t s_rec[3 * kBf16Tile];     // this tile's escape records, in order
    __shared__ uint32_t s_warp_esc[kWarps];
    __shared__ uint32_t s_tile, s_prefix;
    __shared__ int s_failed;

    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    {
        uint32_t code = 0x10u;
#pragma unroll
        for (int k = 0; k < kCodes; k++)
            if (p.cb[k] == tid) code = (uint32_t)k;
        s_code[tid] = (uint8_t)code;
    }
    if (tid == 0) s_tile = atomicAdd(p.ticket, 1u);
    __syncthreads();
    const uint32_t tile = s_tile;
    if (tile >= p.num_tiles) return;  // only with the stalled-predecessor test hook
    const uint64_t n = p.L.n;
    const uint64_t base = (uint64_t)tile * kBf16Tile;

    // Load the four groups of 8 elements.
    uint32_t w[4][4];
    uint32_t cnt[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint64_t i0 = group_start(base, warp, k, lane);
        cnt[k] = i0 >= n ? 0u : (n - i0 >= 8 ? 8u : (uint32_t)(n - i0));
        if (p.vec && cnt[k] == 8) {
            const uint4 v = ld_stream_v4(p.in + 2 * i0);
            w[k][0] = v.x, w[k][1] = v.y, w[k][2] = v.z, w[k][3] = v.w;
        } else {
#pragma unroll
            for (int q = 0; q < 4; q++) w[k][q] = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if ((uint32_t)j < cnt[k]) {
                    const uint8_t* e = p.in + 2 * (i0 + j);
                    w[k][j >> 1] |= ((uint32_t)e[0] | ((uint32_t)e[1] << 8)) << (16 * (j & 1));
                }
            }
        }
    }

    // Split, code, pack, store; collect the escape mask of each group.
    uint32_t esc[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint64_t i0 = group_start(base, warp, k, lane);
        const uint32_t sm_lo = __byte_perm(sm_pair(w[k][0]), sm_pair(w[k][1]), 0x6420);
        const uint32_t sm_hi = __byte_perm(sm_pair(w[k][2]), sm_pair(w[k][3]), 0x6420);
        uint32_t nib = 0, m = 0;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const uint32_t e = (w[k][j >> 1] >> (7 + 16 * (j & 1))) & 0xFFu;
            const uint32_t c = s_code[e];
            nib |= (c & 0xFu) << (4 * j);
            m |= (c >> 4) << j;
        }
        const uint32_t valid = (1u << cnt[k]) - 1u;  // cnt <= 8
        m &= valid;
        if (cnt[k] < 8) nib &= (uint32_t)((1ull << (4 * cnt[k])) - 1ull);
        esc[k] = m;
        if (p.vec && cnt[k] == 8) {
            st_stream_v2(p.out + i0, make_uint2(sm_lo, sm_hi));
            st_stream_u32(p.out + p.L.nib_off + i0 / 2, nib);
        } else if (cnt[k] > 0) {
            const uint64_t smv = (uint64_t)sm_lo | ((uint64_t)sm_hi << 32);
            for (uint32_t j = 0; j < cnt[k]; j++) p.out[i0 + j] = (uint8_t)(smv >> (8 * j));
            for (uint32_t b = 0; b < (cnt[k] + 1) / 2; b++) p.out[p.L.nib_off + i0 / 2 + b] = (uint8_t)(nib >> (8 * b));
        }
    }

    // Rank escapes inside the warp in (k, lane, j) order: per-lane counts of
    // the four groups packed two per word, inclusive warp scans.
    uint32_t off[4] = {0, 0, 0, 0};
    uint32_t warp_total = 0;
    if (__any_sync(0xFFFFFFFFu, (esc[0] | esc[1] | esc[2] | esc[3]) != 0)) {
        const uint32_t c01 = __popc(esc[0]) | ((uint32_t)__popc(esc[1]) << 16);
        const uint32_t c23 = __popc(esc[2]) | ((uint32_t)__popc(esc[3]) << 16);
        uint32_t s01 = c01, s23 = c23;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, s01, d);
            const uint32_t b = __shfl_up_sync(0xFFFFFFFFu, s23, d);
            if (lane >= (uint32_t)d) s01 += a, s23 += b;
        }
        const uint32_t t01 = __shfl_sync(0xFFFFFFFFu, s01, 31);
        const uint32_t t23 = __shfl_sync(0xFFFFFFFFu, s23, 31);
        const uint32_t x01 = s01 - c01, x23 = s23 - c23;
        const uint32_t tot0 = t01 & 0xFFFFu, tot1 = t01 >> 16, tot2 = t23 & 0xFFFFu, tot3 = t23 >> 16;
        off[0] = x01 & 0xFFFFu;
        off[1] = tot0 + (x01 >> 16);
        off[2] = tot0 + tot1 + (x23 & 0xFFFFu);
        off[3] = tot0 + tot1 + tot2 + (x23 >> 16);
        warp_total = tot0 + tot1 + tot2 + tot3;
    }
    if (lane == 0) s_warp_esc[warp] = warp_total;
    __syncthreads();
    uint32_t warp_off = 0, tile_esc = 0;
#pragma unroll
    for (uint32_t v = 0; v < kWarps; v++) {
        const uint32_t c = s_warp_esc[v];
        if (v < warp) warp_off += c;
        tile_esc += c;
    }

    // Stage this tile's records (position inside the chunk, raw exponent).
    if (tile_esc != 0) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            if (esc[k] == 0) continue;
            const uint64_t i0 = group_start(base, warp, k, lane);
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if ((esc[k] >> j) & 1u) {
                    const uint32_t r = warp_off + off[k] + __popc(esc[k] & ((1u << j) - 1u));
                    const uint32_t pos = (uint32_t)(i0 + j) & 0xFFFFu;
                    const uint32_t e = (w[k][j >> 1] >> (7 + 16 * (j & 1))) & 0xFFu;
                    s_rec[3 * r + 0] = (uint8_t)pos;
                    s_rec[3 * r + 1] = (uint8_t)(pos >> 8);
                    s_rec[3 * r + 2] = (uint8_t)e;
                }
            }
        }
    }

    // Escapes in all earlier tiles (decoupled look-back by warp 0).
    if (warp == 0) {
        bool failed;
        const uint32_t prefix = lookback_prefix(p.tile_status, tile, tile_esc, p.wait_limit_ns, &failed);
        if (lane == 0) s_prefix = prefix, s_failed = failed;
    }
    __syncthreads();
    if (s_failed) {
        if (tid == 0 && p.status) atomicMax(p.status, kStatusTimeout);
        return;
    }
    const uint32_t prefix = s_prefix;

    // Copy the staged records to their final place (bytes, coalesced).
    if (tile_esc != 0) {
        const uint64_t dst = p.L.rec_off + 3ull * prefix;
        const uint32_t nbytes = 3u * tile_esc;
        for (uint32_t b = tid; b < nbytes; b += kBf16Threads)
            if (dst + b < p.capacity) p.out[dst + b] = s_rec[b];
    }

    if (tid == 0) {
        // The first tile of chunk c closes the header of chunk c - 1.
        if (tile % kTilesPerChunk == 0 && tile > 0) {
            const uint64_t wprev = wait_for_prefix(p.tile_status, tile - kTilesPerChunk, p.wait_limit_ns);
            if (status_flag(wprev) == kFlagError) {
                if (p.status) atomicMax(p.status, kStatusTimeout);
            } else {
                const uint32_t c = tile / kTilesPerChunk - 1;
                const uint32_t first = status_prefix(wprev);
                store_u32_le(p.out + p.L.hdr_off + 8ull * c, first);
                store_u32_le(p.out + p.L.hdr_off + 8ull * c + 4, prefix - first);
            }
        }
        // The last tile knows the total: stream size and the last header.
        if (tile == p.num_tiles - 1) {
            const uint32_t total = prefix + tile_esc;
            const unsigned long long size = p.L.rec_off + 3ull * total;
            *p.out_bytes = size;
            if (size > p.capacity && p.status) atomicMax(p.status, kStatusCapacity);
            if (p.L.num_chunks > 0) {
                const uint32_t c = p.L.num_chunks - 1;
                const uint32_t first_tile = c * kTilesPerChunk;
                uint32_t first = prefix;
                bool ok = true;
                if (first_tile != tile) {
                    const uint64_t wf = wait_for_prefix(p.tile_status, first_tile, p.wait_limit_ns);
                    ok = status_flag(wf) != kFlagError;
                    first = status_prefix(wf);
                }
                if (ok) {
                    store_u32_le(p.out + p.L.hdr_off + 8ull * c, first);
                    store_u32_le(p.out + p.L.hdr_off + 8ull * c + 4, total - first);
                } else if (p.status) {
                    atomicMax(p.status, kStatusTimeout);
                }
            }
        }
    }
    if (tile == 0 && tid < kCodes) p.out[p.L.cb_off + tid] = p.cb[tid];
}

// ---------------------------------------------------------------------------
// Decode.  Dense pass: nibble byte -> two exponents through a 256-entry
// shared LUT, joined with the sign|mantissa bytes.  Escapes of the tile (a
// contiguous run of the chunk's sorted records) are checked and spread into
// a shared bitmap + exponent table before the dense pass, so they are
// applied in registers and every output byte is stored once.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBf16Threads) decode_bf16_kernel(const DecodeParams p) {
    __shared__ uint32_t s_lut[256];
    __shared__ uint32_t s_bits[kBf16Threads];
    __shared__ uint8_t s_patch[kBf16Tile];
    __shared__ uint32_t s_cnt[6];
    __shared__ int s_bad;

    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t tile = blockIdx.x;
    const uint64_t n = p.L.n;
    const uint64_t base = (uint64_t)tile * kBf16Tile;
    const uint8_t* cb = p.in + p.L.cb_off;

    s_lut[tid] = ((uint32_t)cb[tid & 15u] << 7) | ((uint32_t)cb[tid >> 4] << 23);
    s_bits[tid] = 0;
    if (tid == 0) s_bad = 0;

    // Dense loads first, so they are in flight during the escape search.
    uint2 smv[4];
    uint32_t nibv[4], cnt[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint64_t i0 = group_start(base, warp, k, lane);
        cnt[k] = i0 >= n ? 0u : (n - i0 >= 8 ? 8u : (uint32_t)(n - i0));
        if (p.vec && cnt[k] == 8) {
            smv[k] = ld_stream_v2(p.in + i0);
            nibv[k] = ld_stream_u32(p.in + p.L.nib_off + i0 / 2);
        } else {
            uint64_t s = 0;
            uint32_t nb = 0;
            for (uint32_t j = 0; j < cnt[k]; j++) s |= (uint64_t)p.in[i0 + j] << (8 * j);
            for (uint32_t b = 0; b < (cnt[k] + 1) / 2; b++) nb |= (uint32_t)p.in[p.L.nib_off + i0 / 2 + b] << (8 * b);
            smv[k] = make_uint2((uint32_t)s, (uint32_t)(s >> 32));
            nibv[k] = nb;
        }
    }
    __syncthreads();  // s_bad initialised

    if (tid < kCodes) {  // a codebook is 16 distinct exponents
        bool dup = false;
        for (int k = 0; k < kCodes; k++) dup |= (k != (int)tid) && cb[k] == cb[tid];
        if (dup) s_bad = 1;
    }

    // Spread this tile's escapes into a bitmap (bit k*8+j of thread
    // warp*32+lane) and a per-element exponent table.
    for_each_tile_escape<kBf16Threads, kBf16Tile, false>(p, tile, s_cnt, &s_bad, [&](uint32_t q, uint32_t e) {
        s_patch[q] = (uint8_t)e;
        const uint32_t owner = (q >> 10) * 32u + ((q >> 3) & 31u);
        const uint32_t bit = ((q >> 8) & 3u) * 8u + (q & 7u);
        atomicOr(&s_bits[owner], 1u << bit);
    });

    const uint32_t bits = s_bits[tid];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint64_t i0 = group_start(base, warp, k, lane);
        uint32_t y[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const uint32_t smw = q < 2 ? smv[k].x : smv[k].y;
            const uint32_t t = __byte_perm(smw, 0, (q & 1) ? 0x4342 : 0x4140);
            y[q] = (t & 0x007F007Fu) | ((t & 0x00800080u) << 8) | s_lut[(nibv[k] >> (8 * q)) & 0xFFu];
        }
        const uint32_t gb = (bits >> (8 * k)) & 0xFFu;
        if (gb) {
            const uint32_t qbase = warp * 1024u + k * 256u + lane * 8u;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if ((gb >> j) & 1u) {
                    const uint32_t sh = 7 + 16 * (j & 1);
                    y[j >> 1] = (y[j >> 1] & ~(0xFFu << sh)) | ((uint32_t)s_patch[qbase + j] << sh);
                }
            }
        }
        if (p.vec && cnt[k] == 8) {
            st_stream_v4(p.out + 2 * i0, make_uint4(y[0], y[1], y[2], y[3]));
        } else {
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if ((uint32_t)j < cnt[k]) {
                    const uint32_t v = y[j >> 1] >> (16 * (j & 1));
                    p.out[2 * (i0 + j)] = (uint8_t)v;
                    p.out[2 * (i0 + j) + 1] = (uint8_t)(v >> 8);
                }
            }
        }
    }
    if (tid == 0 && s_bad && p.status) atomicMax(p.status, kStatusCorrupt);
}

cudaError_t launch_encode_bf16(const EncodeParams& p, cudaStream_t s) {
    encode_bf16_kernel<<<p.num_tiles, kBf16Threads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t s) {
    decode_bf16_kernel<<<p.num_tiles, kBf16Threads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sz
