// sz_e5m2.cu -- SplitZip FP8 E5M2 encode and decode kernels for sm_103a.
//
// Method: SplitZip technical summary (gist.science/es), "Contribuciones
// Clave", item 4 "Extensibilidad" (the codec extends to FP8 E5M2 KV caches),
// with the encode/decode steps of "Metodologia: SplitZip".  Each element
// becomes a 7-bit field code | (sign << 2 | mantissa) << 4; eight fields make
// a 56-bit little-endian word stored as 7 bytes; escapes use the same
// (u16 position, u8 exponent) stream as BF16.
//
// Work layout.  Thread t of a block owns 128 contiguous elements = 16 groups
// = 128 input bytes and 112 packed bytes.  A warp's 4 KB of elements and
// 3.5 KB of packed bytes move between global memory and registers through a
// per-warp shared-memory transpose, so every global access is a fully
// coalesced 16 B/lane instruction and every shared access is free of bank
// conflicts (XOR swizzle for 8-piece rows; the 7-piece rows need none
// because 7 is odd).  The encoder's block of 256 threads owns one
// 32,768-element scan tile; the decoder's block of 128 threads owns a
// 16,384-element tile.
#include "sz_device.cuh"
#include "sz_params.h"

namespace sz {

namespace {

static_assert(kChunk % kE5Tile == 0, "tiles must not straddle chunks");
constexpr uint32_t kWarps = kE5Threads / 32;           // decode warps
constexpr uint32_t kWarpElems = 32 * kE5PerThread;     // 4096
constexpr uint32_t kEncThreads = kScanTile / kE5PerThread;  // 256: one scan tile per encode block
constexpr uint32_t kEncWarps = kEncThreads / 32;

// 16-byte slot of piece s (0..7) of thread-row r in an 8-piece swizzled row set.
__device__ __forceinline__ uint32_t swz8(uint32_t r, uint32_t s) { return r * 8u + (s ^ (r & 7u)); }

// Four E5M2 bytes -> their four 7-bit fields (one per byte), for a codebook of
// 16 consecutive exponents cb0..cb0+15 (cb0 <= 16).  With add = 0x20 - cb0 in
// every byte, d = exponent + add has no carry between bytes, and bit 4 of d
// is set exactly when exponent - cb0 falls outside 0..15, i.e. for an escape,
// whose code is 0.  esc4 receives those bit-4 flags.  The parts of a field
// occupy disjoint bits, so the mantissa joins with a multiply-add.
__device__ __forceinline__ uint32_t fields4_contig(uint32_t w, uint32_t add, uint32_t& esc4) {
    const uint32_t d = ((w >> 2) & 0x1F1F1F1Fu) + add;
    esc4 = d & 0x10101010u;
    const uint32_t kill = (esc4 >> 4) * 0x0Fu;                     // 0x0F in escaped bytes
    const uint32_t code_sign = (d & 0x0F0F0F0Fu & ~kill) | ((w >> 1) & 0x40404040u);
    return (w & 0x03030303u) * 16u + code_sign;
}

// Four 7-bit fields held one per byte -> 28 bits, field 0 lowest.  Each step
// moves the upper half of every lane down by subtracting a multiple of it.
__device__ __forceinline__ uint32_t pack28(uint32_t f) {
    const uint32_t x = f - ((f >> 8) & 0x007F007Fu) * 128u;     // 16-bit lanes: f0 | f1 << 7
    return x - ((x >> 2) & 0x0FFFC000u) * 3u;                     // f0 | f1 << 7 | f2 << 14 | f3 << 21
}

// One group of 8 elements (two little-endian words of input bytes) -> the
// 56-bit packed word (lo: bits 0..31, hi: bits 32..55) and, in bits 24..31 of
// esc_hi, the escape mask (element j at bit 24 + j; the lower bits are junk).
// CONTIG: byte-parallel arithmetic, the eight bit-4 flags gathered by one
// multiply whose partial products land below bit 24 or above bit 31;
// otherwise a 256-entry table maps a byte to its field, with 0x80 marking an
// escape.
template <bool CONTIG>
__device__ __forceinline__ void code_group(uint32_t a, uint32_t b, uint32_t add, const uint8_t* field, uint32_t& lo,
                                           uint32_t& hi, uint32_t& esc_hi) {
    if (CONTIG) {
        uint32_t ea, eb;
        const uint32_t pa = pack28(fields4_contig(a, add, ea)), pb = pack28(fields4_contig(b, add, eb));
        lo = pb * (1u << 28) + pa;
        hi = pb >> 4;
        esc_hi = ((ea >> 4) | eb) * 0x01020408u;  // a_j at 8j, b_j at 8j + 4 -> bit 24 + j, 28 + j
    } else {
        lo = 0;
        hi = 0;
        uint32_t esc8 = 0;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const uint32_t f = field[((j < 4 ? a : b) >> (8 * (j & 3))) & 0xFFu];
            esc8 |= (f >> 7) << j;
            const uint32_t f7 = f & 0x7Fu;
            const int bit = 7 * j;
            if (bit + 7 <= 32) {
                lo |= f7 << bit;
            } else if (bit >= 32) {
                hi |= f7 << (bit - 32);
            } else {
                lo |= f7 << bit;
                hi |= f7 >> (32 - bit);
            }
        }
        esc_hi = esc8 << 24;
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Encode, first phase: one scan tile per block.  Each warp stages its 4 KB
// of input in shared memory (swizzled rows, one per thread), so that global
// loads stay coalesced while each thread codes its own 128 contiguous bytes.
// The packed bytes (7 pieces of 16 bytes per thread) reuse the same buffer
// once the whole warp has read its rows, and leave with coalesced stores.
// Before that, the tile's escape count and its first ws_cap records (element
// order: thread, then element; exponents read back from the rows) go to the
// workspace; finish_kernel (sz_finish.cu) places the records.
// ---------------------------------------------------------------------------
struct EncodeE5Smem {
    uint4 buf[kEncWarps][256];  // input: 8 swizzled pieces per thread; then output: 7 pieces per thread
    uint32_t warp_esc[kEncWarps];
    uint8_t field[256];         // byte -> field; 0x80 marks an escape
};

template <bool CONTIG>
__global__ void __launch_bounds__(kEncThreads, CONTIG ? 5 : 3) encode_e5m2_kernel(const EncodeParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    EncodeE5Smem& S = *reinterpret_cast<EncodeE5Smem*>(smem_raw);
    auto& s_field = S.field;
    auto& s_in = S.buf;
    auto& s_out = S.buf;
    auto& s_warp_esc = S.warp_esc;

    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    {
        const uint32_t x = tid, e = (x >> 2) & 31u;
        uint32_t code = 0xFFu;
#pragma unroll
        for (int k = 0; k < kCodes; k++)
            if (p.cb[k] == e) code = (uint32_t)k;
        const uint32_t sm3 = ((x >> 7) << 2) | (x & 3u);
        s_field[x] = (uint8_t)(code == 0xFFu ? (0x80u | (sm3 << 4)) : (code | (sm3 << 4)));
    }
    if (blockIdx.x == 0 && tid < kCodes) p.out[p.L.cb_off + tid] = p.cb[tid];
    __syncthreads();
    const uint32_t st = blockIdx.x;
    const uint64_t n = p.L.n;
    const uint64_t warp_base = (uint64_t)st * kScanTile + warp * kWarpElems;
    const uint64_t thread_base = warp_base + lane * kE5PerThread;
    const bool warp_full = p.vec && warp_base + kWarpElems <= n;
    const uint32_t cnt = thread_base >= n ? 0u : (n - thread_base >= kE5PerThread ? kE5PerThread : (uint32_t)(n - thread_base));

    // Input bytes into this thread's row.  Bytes past n read as exponent
    // cb[0] with sign and mantissa 0, which packs to field 0 and is no escape.
    if (warp_full) {
#pragma unroll
        for (uint32_t i = 0; i < 8; i++) {
            const uint32_t piece = lane + 32 * i;
            s_in[warp][swz8(piece >> 3, piece & 7u)] = ld_stream_v4(p.in + warp_base + 16 * piece);
        }
    } else {
        const uint32_t pad = (uint32_t)p.cb[0] << 2;
        for (uint32_t s = 0; s < 8; s++) {
            uint32_t w[4];
#pragma unroll
            for (uint32_t q = 0; q < 4; q++) {
                uint32_t v = 0;
#pragma unroll
                for (uint32_t t = 0; t < 4; t++) {
                    const uint32_t j = 16 * s + 4 * q + t;
                    v |= (j < cnt ? (uint32_t)p.in[thread_base + j] : pad) << (8 * t);
                }
                w[q] = v;
            }
            s_in[warp][swz8(lane, s)] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    __syncwarp();

    // Pack: four groups (224 bits) make seven 32-bit words; a thread's 16
    // groups make its 28 words = 7 pieces of 16 bytes.  escm[q] holds the
    // escape flags of elements 32q..32q+31 of the thread.
    uint32_t escm[4], words[28];
    {
        const uint32_t add = 0x20202020u - (uint32_t)p.cb[0] * 0x01010101u;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            uint32_t lo[4], hi[4], eh[4];
#pragma unroll
            for (int hs = 0; hs < 2; hs++) {
                const uint4 v = s_in[warp][swz8(lane, 2 * q + hs)];
                code_group<CONTIG>(v.x, v.y, add, s_field, lo[2 * hs], hi[2 * hs], eh[2 * hs]);
                code_group<CONTIG>(v.z, v.w, add, s_field, lo[2 * hs + 1], hi[2 * hs + 1], eh[2 * hs + 1]);
            }
            // Byte 3 of each group's eh, in group order.
            escm[q] = __byte_perm(__byte_perm(eh[0], eh[1], 0x0073u), __byte_perm(eh[2], eh[3], 0x7300u), 0x7610u);
            uint32_t* w = words + 7 * q;
            w[0] = lo[0];
            w[1] = lo[1] * (1u << 24) + hi[0];
            w[2] = __funnelshift_r(lo[1], hi[1], 8);
            w[3] = lo[2] * (1u << 16) + (hi[1] >> 8);
            w[4] = __funnelshift_r(lo[2], hi[2], 16);
            w[5] = lo[3] * (1u << 8) + (hi[2] >> 16);
            w[6] = __funnelshift_r(lo[3], hi[3], 24);
        }
    }

    // Rank escapes: thread order, then element order inside the thread.
    const uint32_t mine = __popc(escm[0]) + __popc(escm[1]) + __popc(escm[2]) + __popc(escm[3]);
    uint32_t incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= (uint32_t)d) incl += a;
    }
    if (lane == 31) s_warp_esc[warp] = incl;
    __syncthreads();
    uint32_t rank = incl - mine, tile_esc = 0;
#pragma unroll
    for (uint32_t v = 0; v < kEncWarps; v++) {
        const uint32_t c = s_warp_esc[v];
        if (v < warp) rank += c;
        tile_esc += c;
    }
    if (tid == 0) p.ws_count[st] = tile_esc;
    // Stage this thread's records (those ranked below ws_cap); the exponents
    // come from the thread's input row, still in shared memory.
    if (mine && rank < p.ws_cap) {
        const uint8_t* row = reinterpret_cast<const uint8_t*>(&s_in[warp][0]);
        uint8_t* dst = p.ws_rec + (uint64_t)st * 3 * p.ws_cap;
        const uint64_t limit = 3ull * p.ws_cap;
        uint64_t at = 3ull * rank;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            uint32_t m = escm[q];
            while (m) {
                const uint32_t j = 32 * q + __ffs(m) - 1;
                m &= m - 1;
                const uint32_t byte = row[swz8(lane, j >> 4) * 16u + (j & 15u)];
                const uint32_t pos = (uint32_t)(thread_base + j) & 0xFFFFu;
                if (at + 3 <= limit) {
                    dst[at] = (uint8_t)pos;
                    dst[at + 1] = (uint8_t)(pos >> 8);
                    dst[at + 2] = (uint8_t)((byte >> 2) & 31u);
                }
                at += 3;
            }
        }
    }

    // Every row of the warp has been read: the buffer takes the output.
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 7; k++)
        s_out[warp][lane * 7 + k] = make_uint4(words[4 * k], words[4 * k + 1], words[4 * k + 2], words[4 * k + 3]);
    __syncwarp();
    const uint64_t out_base = warp_base / 8 * 7;  // packed bytes before this warp
    if (warp_full) {
#pragma unroll
        for (uint32_t i = 0; i < 7; i++) {
            const uint32_t piece = lane + 32 * i;
            st_stream_v4(p.out + out_base + 16 * piece, s_out[warp][piece]);
        }
    } else if (cnt > 0) {
        const uint32_t nbytes = 7 * ((cnt + 7) / 8);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(&s_out[warp][lane * 7]);
        uint8_t* dst = p.out + out_base + lane * 112u;
        for (uint32_t b = 0; b < nbytes; b++) dst[b] = src[b];
    }
}

// ---------------------------------------------------------------------------
// Decode: packed groups -> fields -> bytes through a 128-entry LUT, staged in
// the warp's transpose buffer where the tile's escapes patch the exponent
// bits, then stored with coalesced 16-byte writes.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kE5Threads) decode_e5m2_kernel(const DecodeParams p) {
    __shared__ uint8_t s_dec[128];  // field -> E5M2 byte
    __shared__ __align__(16) uint4 s_xpose[kWarps][256];
    __shared__ uint32_t s_cnt[6];
    __shared__ int s_bad;

    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t tile = blockIdx.x;
    const uint64_t n = p.L.n;
    const uint64_t warp_base = (uint64_t)tile * kE5Tile + warp * kWarpElems;
    const uint64_t thread_base = warp_base + lane * kE5PerThread;
    const bool warp_full = p.vec && warp_base + kWarpElems <= n;
    const uint32_t cnt = thread_base >= n ? 0u : (n - thread_base >= kE5PerThread ? kE5PerThread : (uint32_t)(n - thread_base));
    const uint8_t* cb = p.in + p.L.cb_off;

    {
        const uint32_t f = tid;  // 128 threads, one field value each
        const uint32_t sm3 = f >> 4;
        s_dec[f] = (uint8_t)(((sm3 >> 2) << 7) | ((uint32_t)cb[f & 15u] << 2) | (sm3 & 3u));
    }
    if (tid == 0) s_bad = 0;

    // Packed bytes of this thread: 28 words (16 groups).
    uint32_t pw[28];
    const uint64_t in_base = warp_base / 8 * 7;
    if (warp_full) {
#pragma unroll
        for (uint32_t i = 0; i < 7; i++) {
            const uint32_t piece = lane + 32 * i;
            s_xpose[warp][piece] = ld_stream_v4(p.in + in_base + 16 * piece);
        }
        __syncwarp();
#pragma unroll
        for (uint32_t i = 0; i < 7; i++) {
            const uint4 v = s_xpose[warp][lane * 7 + i];
            pw[4 * i] = v.x, pw[4 * i + 1] = v.y, pw[4 * i + 2] = v.z, pw[4 * i + 3] = v.w;
        }
    } else {
        const uint32_t nbytes = 7 * ((cnt + 7) / 8);
        const uint8_t* src = p.in + in_base + lane * 112u;
#pragma unroll
        for (int k = 0; k < 28; k++) {
            uint32_t v = 0;
#pragma unroll
            for (int t = 0; t < 4; t++)
                if ((uint32_t)(4 * k + t) < nbytes) v |= (uint32_t)src[4 * k + t] << (8 * t);
            pw[k] = v;
        }
    }
    __syncthreads();  // s_dec, s_bad ready; transpose buffer free again

    if (tid < kCodes) {  // 16 distinct exponents that fit in 5 bits
        bool bad = cb[tid] >= 32;
        for (int k = 0; k < kCodes; k++) bad |= (k != (int)tid) && cb[k] == cb[tid];
        if (bad) s_bad = 1;
    }

    // Dense pass into the transpose buffer (this thread's row, swizzled).
#pragma unroll
    for (int s = 0; s < 8; s++) {
        uint32_t y[4];
#pragma unroll
        for (int w = 0; w < 4; w++) {
            uint32_t v = 0;
#pragma unroll
            for (int t = 0; t < 4; t++) {
                const int j = 16 * s + 4 * w + t;  // element inside the thread
                const int g = j / 8, bit = 7 * (j % 8);
                // 56-bit group value starts at byte 7g of the thread's packed bytes.
                const int byte0 = 7 * g + bit / 8, sh = bit % 8;
                const uint32_t lo = (pw[byte0 / 4] >> (8 * (byte0 % 4))) & 0xFFu;
                const int byte1 = byte0 + 1;
                const uint32_t hi = byte1 < 7 * (g + 1) ? (pw[byte1 / 4] >> (8 * (byte1 % 4))) & 0xFFu : 0u;
                const uint32_t f = ((lo | (hi << 8)) >> sh) & 0x7Fu;
                v |= (uint32_t)s_dec[f] << (8 * t);
            }
            y[w] = v;
        }
        s_xpose[warp][swz8(lane, s)] = make_uint4(y[0], y[1], y[2], y[3]);
    }

    // Escapes: patch the exponent bits of the staged bytes.
    uint8_t* staged = reinterpret_cast<uint8_t*>(&s_xpose[0][0]);
    for_each_tile_escape<kE5Threads, kE5Tile, true>(p, tile, s_cnt, &s_bad, [&](uint32_t q, uint32_t e) {
        const uint32_t t = q >> 7, b = q & 127u;  // owning thread of the tile, byte inside its row
        const uint32_t w = t >> 5, l = t & 31u;
        uint8_t* at = staged + (w * 256u + swz8(l, b >> 4)) * 16u + (b & 15u);
        *at = (uint8_t)((*at & 0x83u) | (e << 2));
    });
    __syncthreads();

    if (warp_full) {
#pragma unroll
        for (uint32_t i = 0; i < 8; i++) {
            const uint32_t piece = lane + 32 * i;
            st_stream_v4(p.out + warp_base + 16 * piece, s_xpose[warp][swz8(piece >> 3, piece & 7u)]);
        }
    } else {
        for (uint32_t b = 0; b < cnt; b++)
            p.out[thread_base + b] = staged[(warp * 256u + swz8(lane, b >> 4)) * 16u + (b & 15u)];
    }
    if (tid == 0 && s_bad && p.status) atomicMax(p.status, kStatusCorrupt);
}

cudaError_t launch_encode_e5m2(const EncodeParams& p, cudaStream_t s) {
    const size_t smem = sizeof(EncodeE5Smem);
    auto kern = p.contig ? encode_e5m2_kernel<true> : encode_e5m2_kernel<false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<p.num_tiles, kEncThreads, smem, s>>>(p);
    err = cudaGetLastError();
    return err != cudaSuccess ? err : launch_finish(p, false, s);
}

cudaError_t launch_decode_e5m2(const DecodeParams& p, cudaStream_t s) {
    decode_e5m2_kernel<<<p.num_tiles, kE5Threads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sz
