// sz_e5m2.cu -- SplitZip FP8 E5M2 encode and decode kernels for sm_103a.
//
// Method: SplitZip technical summary (gist.science/es), "Contribuciones
// Clave", item 4 "Extensibilidad" (the codec extends to FP8 E5M2 KV caches),
// with the encode/decode steps of "Metodologia: SplitZip".  Each element
// becomes a 7-bit field code | (sign << 2 | mantissa) << 4; eight fields make
// a 56-bit little-endian word stored as 7 bytes; escapes use the same
// (u16 position, u8 exponent) stream as BF16.
//
// Work layout.  Encoder: a block of 256 threads owns one 32,768-element scan
// tile, and thread t codes 128 contiguous elements of it (16 groups: 128
// input bytes, 112 packed bytes).  A warp's 4 KB of elements and 3.5 KB of
// packed bytes move between global memory and registers through a per-warp
// shared-memory transpose, so every global access is a fully coalesced
// 16 B/lane instruction and every shared access is free of bank conflicts
// (XOR swizzle for 8-piece rows; the 7-piece rows need none because 7 is
// odd).  Decoder: persistent blocks of 256 threads work through 16,384-element
// tiles, thread t decoding elements 64t..64t+63 of a tile (see below).
#include <algorithm>

#include "sz_device.cuh"
#include "sz_params.h"
#include "sz_pipeline.cuh"
#include "sz_records.cuh"

namespace sz {

namespace {

static_assert(kChunk % kE5Tile == 0, "tiles must not straddle chunks");
static_assert(32 * kE5PerThread == kUnitElemsE5, "an E5M2 unit is one encoder warp's elements");
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
    // Shifts of masked words as high multiplies, joins as multiply-adds (see
    // mad_hi): the coding is ALU-bound, the FMA pipe is not.
    const uint32_t d = mad_hi<0x40000000u>(w & 0x7C7C7C7Cu, add);   // exponent + add per byte
    esc4 = d & 0x10101010u;
    const uint32_t kill = mul_hi<0xF0000000u>(esc4);                 // 0x0F in escaped bytes
    const uint32_t code_sign = mad_hi<0x80000000u>(w & 0x80808080u, d & 0x0F0F0F0Fu & ~kill);  // sign to bit 6
    return mad_lo<16u>(w & 0x03030303u, code_sign);                  // mantissa to bits 4..5
}

// Four 7-bit fields held one per byte -> 28 bits, field 0 lowest.  Each step
// moves the upper half of every lane down by subtracting a multiple of it.
__device__ __forceinline__ uint32_t pack28(uint32_t f) {
    const uint32_t x = mad_lo<0xFFFFFF80u>(mul_hi<1u << 24>(f & 0x7F007F00u), f);  // f0 | f1 << 7 per 16-bit lane
    return mad_lo<0xFFFFFFFDu>(mul_hi<1u << 30>(x & 0x3FFF0000u), x);             // f0 | f1 << 7 | f2 << 14 | f3 << 21
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
        lo = mad_lo<1u << 28>(pb, pa);
        hi = mul_hi<1u << 28>(pb);                                  // pb >> 4
        esc_hi = mad_hi<1u << 28>(ea, eb) * 0x01020408u;  // a_j at 8j, b_j at 8j + 4 -> bit 24 + j, 28 + j
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
// Before that, the tile's escape count and its first ws_cap records
// (element order: thread, then element; exponents read back from the rows)
// go to the workspace, and, when the tile has more escapes than that, the
// count of each warp's 4,096 elements; finish_kernel (sz_finish.cu) places
// the records.
// ---------------------------------------------------------------------------
struct EncodeE5Smem {
    uint4 buf[kEncWarps][256];  // input: 8 swizzled pieces per thread; then output: 7 pieces per thread
    alignas(16) uint8_t rec[3 * kStageRecsE5];  // the scan tile's staged records
    uint32_t warp_esc[kEncWarps];
    int werr[kEncWarps];        // paged input: each warp's error code (bad page ids)
    uint8_t field[256];         // byte -> field; 0x80 marks an escape
};

// Everything after the input rows are in shared memory: coding, escape
// ranks, staged records, packed output.
// The block's error goes out with the tile's escape count, as its bit 31
// (kCountError): a bad device codebook (bad_codebook), or, with PAGED input,
// a bad page id reported by any warp in S.werr.
template <bool CONTIG, bool PAGED>
__device__ __forceinline__ void encode_e5m2_code(const EncodeParams& p, EncodeE5Smem& S, const uint8_t (&cb)[16],
                                                 uint64_t warp_base, uint64_t thread_base, bool warp_full,
                                                 uint32_t cnt, bool bad_codebook) {
    auto& s_field = S.field;
    auto& s_in = S.buf;
    auto& s_out = S.buf;
    auto& s_warp_esc = S.warp_esc;
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t st = blockIdx.x;

    // Pack: four groups (224 bits) make seven 32-bit words; a thread's 16
    // groups make its 28 words = 7 pieces of 16 bytes.  escm[q] holds the
    // escape flags of elements 32q..32q+31 of the thread.
    uint32_t escm[4], words[28];
    {
        const uint32_t add = 0x20202020u - (uint32_t)cb[0] * 0x01010101u;
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
            w[1] = mad_lo<1u << 24>(lo[1], hi[0]);
            w[2] = __funnelshift_r(lo[1], hi[1], 8);
            w[3] = mad_lo<1u << 16>(lo[2], mul_hi<1u << 24>(hi[1]));   // lo2 << 16 | hi1 >> 8
            w[4] = __funnelshift_r(lo[2], hi[2], 16);
            w[5] = mad_lo<1u << 8>(lo[3], mul_hi<1u << 16>(hi[2]));    // lo3 << 8 | hi2 >> 16
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
    if (tid == 0) {
        bool bad = bad_codebook;
        if (PAGED) {
#pragma unroll
            for (uint32_t v = 0; v < kEncWarps; v++) bad |= S.werr[v] != 0;
        }
        p.ws_count[st] = tile_esc | (bad ? kCountError : 0u);
    }
    // Only a scan tile with more escapes than it stages leaves the escape
    // count of each of its units (one warp's 4,096 elements each), from
    // which the finish kernel re-derives the rest.
    if (tile_esc > p.ws_cap && tid < kEncWarps) p.ws_unit[(uint64_t)st * kUnitsPerScan + tid] = (uint16_t)s_warp_esc[tid];
    // Stage this thread's records (those ranked below ws_cap); the exponents
    // come from the thread's input row, still in shared memory.
    // They are gathered in shared memory and leave in 16-byte stores.
    if (mine && rank < p.ws_cap) {
        const uint8_t* row = reinterpret_cast<const uint8_t*>(&s_in[warp][0]);
        uint8_t* dst = S.rec;
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

    __syncthreads();  // every record of the scan tile is in S.rec
    {
        // The workspace region (3 ws_cap bytes, a multiple of 16) starts
        // 16-byte aligned, so whole 16-byte pieces stay inside it.
        const uint32_t nbytes = 3 * min(tile_esc, p.ws_cap);
        uint8_t* dst = p.ws_rec + (uint64_t)st * 3 * p.ws_cap;
        for (uint32_t b = 16 * tid; b < nbytes; b += 16 * kEncThreads)
            *reinterpret_cast<uint4*>(dst + b) = *reinterpret_cast<const uint4*>(S.rec + b);
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
            st_v4(p.out + out_base + 16 * piece, s_out[warp][piece]);
        }
    } else if (cnt > 0) {
        const uint32_t nbytes = 7 * ((cnt + 7) / 8);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(&s_out[warp][lane * 7]);
        uint8_t* dst = p.out + out_base + lane * 112u;
        for (uint32_t b = 0; b < nbytes; b++) dst[b] = src[b];
    }
}

// MODE 0: codebook in the parameters, table coding; 1: in the parameters,
// contiguous; 2: in device memory, checked (a bad one is reported as
// SZ_ERR_INVALID_ARG), the coding chosen per block.  The device
// codebook is loaded first and examined only once this thread's input loads
// are in flight, so its latency hides behind theirs.
// PAGED: the input is a paged tensor (EncodeParams::pm).
template <int MODE, bool PAGED = false>
__global__ void __launch_bounds__(kEncThreads, MODE == 0 ? 3 : 4) encode_e5m2_kernel(const EncodeParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    EncodeE5Smem& S = *reinterpret_cast<EncodeE5Smem*>(smem_raw);
    auto& s_in = S.buf;
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    uint4 cbv = make_uint4(0, 0, 0, 0);
    if (MODE == 2) cbv = *reinterpret_cast<const uint4*>(p.cb_dev);
    const uint64_t n = p.L.n;
    const uint64_t warp_base = (uint64_t)blockIdx.x * kScanTile + warp * kWarpElems;
    const uint64_t thread_base = warp_base + lane * kE5PerThread;
    const bool warp_full = p.vec && warp_base + kWarpElems <= n;
    const uint32_t cnt = thread_base >= n ? 0u : (n - thread_base >= kE5PerThread ? kE5PerThread : (uint32_t)(n - thread_base));
    // Paged input: the warp's error word, cleared before any lane can report to it.
    int* const werr = PAGED ? &S.werr[warp] : nullptr;
    if (PAGED) {
        if (lane == 0) *werr = 0;
        __syncwarp();
    }

    // Input bytes into this thread's row.
    if (warp_full) {
        // A 16-element piece never straddles a page; the warp's 4,096
        // elements in one page take one lookup.
        const RunOffset<PAGED> run(p.pm, warp_base, 12, 1, werr);
#pragma unroll
        for (uint32_t i = 0; i < 8; i++) {
            const uint32_t piece = lane + 32 * i;
            s_in[warp][swz8(piece >> 3, piece & 7u)] = ld_stream_v4(p.in + run.at(p.pm, warp_base, 16 * piece, 1, werr));
        }
    }
    uint8_t cb[16];
    bool contig;
    bool ok;
    if (MODE == 2) {
        // 16 consecutive exponents cb0..cb0+15 with cb0 <= 16 (valid and
        // codable by arithmetic) are recognised word by word; anything else
        // takes the full check.  Every block runs this, so it is kept short.
        const uint32_t w[4] = {cbv.x, cbv.y, cbv.z, cbv.w};
        const uint32_t c0 = w[0] & 0xFFu, run = c0 * 0x01010101u + 0x03020100u;
        if (c0 <= 16 && w[0] == run && w[1] == run + 0x04040404u && w[2] == run + 0x08080808u &&
            w[3] == run + 0x0C0C0C0Cu) {
#pragma unroll
            for (int k = 0; k < 16; k++) cb[k] = (uint8_t)(c0 + k);
            contig = true;
            ok = true;
        } else {
            uint8_t dcb[16];
#pragma unroll
            for (int k = 0; k < 16; k++) dcb[k] = (uint8_t)(w[k >> 2] >> (8 * (k & 3)));
            ok = load_codebook(dcb, nullptr, 32u, cb, contig);
        }
    } else {
        ok = load_codebook(p.cb, nullptr, 32u, cb, contig);
    }
    if (blockIdx.x == 0 && tid == 0) {
#pragma unroll
        for (int k = 0; k < kCodes; k++) p.out[p.L.cb_off + k] = cb[k];
    }
    if (!warp_full) {
        // Bytes past n read as exponent cb[0] with sign and mantissa 0, which
        // packs to field 0 and is no escape.
        const uint32_t pad = (uint32_t)cb[0] << 2;
        for (uint32_t s = 0; s < 8; s++) {
            uint32_t w[4];
#pragma unroll
            for (uint32_t q = 0; q < 4; q++) {
                uint32_t v = 0;
#pragma unroll
                for (uint32_t t = 0; t < 4; t++) {
                    const uint32_t j = 16 * s + 4 * q + t;
                    v |= (j < cnt ? (uint32_t)p.in[elem_offset<PAGED>(p.pm, thread_base + j, 1, werr)] : pad)
                         << (8 * t);
                }
                w[q] = v;
            }
            s_in[warp][swz8(lane, s)] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    __syncwarp();
    // A contiguous run must also stay within 5 bits for the byte-parallel coding.
    const bool use_contig = MODE == 1 || (MODE == 2 && contig && cb[0] <= 16);
    if (use_contig) {
        encode_e5m2_code<true, PAGED>(p, S, cb, warp_base, thread_base, warp_full, cnt, MODE == 2 && !ok);
    } else {
        // The byte -> field table (block-uniform branch).
        const uint32_t x = tid, e = (x >> 2) & 31u;
        uint32_t code = 0xFFu;
#pragma unroll
        for (int k = 0; k < kCodes; k++)
            if (cb[k] == e) code = (uint32_t)k;
        const uint32_t sm3 = ((x >> 7) << 2) | (x & 3u);
        S.field[x] = (uint8_t)(code == 0xFFu ? (0x80u | (sm3 << 4)) : (code | (sm3 << 4)));
        __syncthreads();
        encode_e5m2_code<false, PAGED>(p, S, cb, warp_base, thread_base, warp_full, cnt, MODE == 2 && !ok);
    }
}

// ---------------------------------------------------------------------------
// Decode: a persistent kernel; block b owns the contiguous tile range
// [bT/G, (b+1)T/G) of 16,384-element tiles (4 per chunk).  The packed bytes
// of a tile (14,336) arrive through a 2-stage ring of TMA bulk copies (four
// blocks per SM keep eight tiles in flight per SM); thread
// t decodes elements 64t..64t+63 of the tile from its 56 bytes (7 8-byte
// shared loads, conflict-free because the 14-word row stride is an odd
// multiple of 2 words) into its row of the warp's output buffer (4 pieces of
// 16 bytes per row, XOR-swizzled so that the row writes are conflict-free).
// A field becomes a byte by arithmetic when the codebook is 16 consecutive
// exponents (exponent = cb0 + code), else through a 128-entry table.  The
// tile's records are walked as in the BF16 decoder (block search only where
// a range starts inside a chunk, then a cursor through record windows filled
// ahead by asynchronous copies, up to two records per thread per step); after
// the step's counting barrier the holders patch the exponent bits of their
// bytes in the output rows, and after a second barrier the rows leave with
// coalesced 16-byte stores.  Validation is
// the BF16 decoder's, plus exponents below 32 in the codebook and records.
// ---------------------------------------------------------------------------
namespace {

constexpr uint32_t kE5DecThreads = 256;
constexpr uint32_t kE5DecWarps = kE5DecThreads / 32;
constexpr uint32_t kE5DecTile = kE5Tile;                      // 16384 elements
constexpr uint32_t kE5DecPer = kE5DecTile / kE5DecThreads;    // 64 elements = 8 groups = 56 bytes
constexpr uint32_t kE5DecTileBytes = kE5DecTile / 8 * 7;      // 14336
constexpr uint32_t kE5DecStages = 2;
constexpr uint32_t kE5TilesPerChunk = kChunk / kE5DecTile;    // 4
constexpr uint32_t kE5R = 2;  // records a thread takes per step
constexpr uint32_t kE5StepRecs = kE5R * kE5DecThreads;
static_assert(kChunk % kE5DecTile == 0 && kE5DecTileBytes % 16 == 0, "tile layout");

struct DecodeE5Smem {
    alignas(128) uint8_t in[kE5DecStages][kE5DecTileBytes];
    alignas(16) uint4 out[kE5DecWarps][32 * 4];  // per warp: 32 rows of 4 swizzled pieces
    uint64_t full[kE5DecStages];
    uint8_t dec[128];                            // field -> byte
    alignas(16) uint8_t win[3][kWinBytes];       // record windows (RecordWindow)
    uint32_t hdr[2][2];                          // {offset, count} of a chunk, by chunk parity
    uint32_t scratch[8];
    int bad;
    int abort;
    int contig;
};
// Four blocks per SM: 4 x (this + 1 KB reserved) within 228 KB.
static_assert(sizeof(DecodeE5Smem) <= 56 * 1024, "decode shared memory");

// 16-byte slot of piece s (0..3) of row r in a 4-piece swizzled row set.
__device__ __forceinline__ uint32_t swz4(uint32_t r, uint32_t s) { return r * 4u + (s ^ ((r >> 1) & 3u)); }

// 28 bits holding four 7-bit fields -> the fields one per byte (inverse of
// the encoder's compaction): each step moves the upper half of every lane up.
__device__ __forceinline__ uint32_t spread28(uint32_t y) {
    const uint32_t x = y + (y & 0x0FFFC000u) * 3u;  // 16-bit lanes: f0 | f1 << 7
    return x + (x & 0x3F803F80u);                   // bytes: f0, f1, f2, f3
}

// Four fields (one per byte) -> four E5M2 bytes, codebook cb0..cb0+15:
// sign (field bit 6) to bit 7, exponent cb0 + code to bits 2..6, mantissa
// (field bits 4..5) to bits 0..1; the parts are disjoint, so they add.
__device__ __forceinline__ uint32_t bytes4_contig(uint32_t f, uint32_t cb0x4) {
    return (f & 0x40404040u) * 2u + ((f & 0x0F0F0F0Fu) + cb0x4) * 4u + ((f >> 4) & 0x03030303u);
}

// One group (56 bits: lo = bits 0..31, hi = bits 32..55) -> 8 bytes.
template <bool CONTIG>
__device__ __forceinline__ void decode_group(uint32_t lo, uint32_t hi, uint32_t cb0x4, const uint8_t* dec,
                                             uint32_t& y0, uint32_t& y1) {
    const uint32_t a = lo & 0x0FFFFFFFu, b = __funnelshift_r(lo, hi, 28) & 0x0FFFFFFFu;
    if (CONTIG) {
        y0 = bytes4_contig(spread28(a), cb0x4);
        y1 = bytes4_contig(spread28(b), cb0x4);
    } else {
        y0 = 0;
        y1 = 0;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            y0 |= (uint32_t)dec[(a >> (7 * j)) & 0x7Fu] << (8 * j);
            y1 |= (uint32_t)dec[(b >> (7 * j)) & 0x7Fu] << (8 * j);
        }
    }
}

// Byte j (0..6) of a group that starts at byte 7g of the 14 words pw.
template <int G>
__device__ __forceinline__ void group_words(const uint32_t (&pw)[14], uint32_t& lo, uint32_t& hi) {
    constexpr int b0 = 7 * G, w0 = b0 / 4, sh = 8 * (b0 % 4);
    const uint32_t x0 = pw[w0], x1 = w0 + 1 < 14 ? pw[w0 + 1] : 0u, x2 = w0 + 2 < 14 ? pw[w0 + 2] : 0u;
    lo = sh ? __funnelshift_r(x0, x1, sh) : x0;
    hi = (sh ? __funnelshift_r(x1, x2, sh) : x1) & 0x00FFFFFFu;
}

}  // namespace

template <bool CONTIG>
__device__ __forceinline__ void decode_rows(const uint32_t (&pw)[14], uint32_t cb0x4, const uint8_t* dec, uint4* rows,
                                            uint32_t lane) {
    uint32_t y[16];
#define SZ_E5_GROUP(G)                                                  \
    {                                                                   \
        uint32_t lo, hi;                                                \
        group_words<G>(pw, lo, hi);                                     \
        decode_group<CONTIG>(lo, hi, cb0x4, dec, y[2 * G], y[2 * G + 1]); \
    }
    SZ_E5_GROUP(0) SZ_E5_GROUP(1) SZ_E5_GROUP(2) SZ_E5_GROUP(3)
    SZ_E5_GROUP(4) SZ_E5_GROUP(5) SZ_E5_GROUP(6) SZ_E5_GROUP(7)
#undef SZ_E5_GROUP
#pragma unroll
    for (uint32_t s = 0; s < 4; s++) rows[swz4(lane, s)] = make_uint4(y[4 * s], y[4 * s + 1], y[4 * s + 2], y[4 * s + 3]);
}

// PAGED: the output is a paged tensor (DecodeParams::pm).
template <bool PAGED>
__global__ void __launch_bounds__(kE5DecThreads, 4) decode_e5m2_kernel(const DecodeParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // launched as a programmatic dependent
    extern __shared__ __align__(128) uint8_t smem_raw[];
    DecodeE5Smem& S = *reinterpret_cast<DecodeE5Smem*>(smem_raw);
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint64_t n = p.L.n;
    const uint32_t T = p.num_tiles, G = gridDim.x;
    const uint32_t t_begin = (uint32_t)((uint64_t)blockIdx.x * T / G);
    const uint32_t t_end = (uint32_t)((uint64_t)(blockIdx.x + 1) * T / G);
    const uint8_t* cb = p.in + p.L.cb_off;
    const uint8_t* rec = p.in + p.L.rec_off;
    const bool tma = p.vec && (reinterpret_cast<uintptr_t>(p.in) % 16 == 0);

    if (tid == 0) {
        for (uint32_t s = 0; s < kE5DecStages; s++) mbar_init(&S.full[s], 1);
        S.bad = 0;
        S.abort = 0;
        S.contig = 1;
        fence_mbar_init();
    }
    if (tid < 128) {
        const uint32_t sm3 = tid >> 4;
        S.dec[tid] = (uint8_t)(((sm3 >> 2) << 7) | ((uint32_t)cb[tid & 15u] << 2) | (sm3 & 3u));
    }
    __syncthreads();
    if (tid < kCodes) {  // 16 distinct exponents that fit in 5 bits
        bool bad = cb[tid] >= 32;
        for (int k = 0; k < kCodes; k++) bad |= (k != (int)tid) && cb[k] == cb[tid];
        if (bad) S.bad = 1;
        if ((uint32_t)cb[tid] != (uint32_t)cb[0] + tid) S.contig = 0;
    }
    __syncthreads();
    const bool contig = S.contig != 0;
    const uint32_t cb0x4 = (uint32_t)cb[0] * 0x01010101u;

    auto full_tile = [&](uint32_t t) { return tma && (uint64_t)(t + 1) * kE5DecTile <= n; };
    auto issue = [&](uint32_t slot, uint32_t t) {  // thread 0 only
        if (full_tile(t)) {
            mbar_arrive_expect_tx(&S.full[slot], kE5DecTileBytes);
            bulk_g2s(S.in[slot], p.in + (uint64_t)t * kE5DecTileBytes, kE5DecTileBytes, &S.full[slot]);
        } else {
            mbar_arrive(&S.full[slot]);
        }
    };
    uint32_t issued = 0, waited = 0;
    if (tid == 0)
        for (uint32_t t = t_begin; t < t_end && t < t_begin + kE5DecStages; t++, issued++)
            issue((t - t_begin) % kE5DecStages, t);

    auto tile_p0 = [&](uint32_t t) { return (t % kE5TilesPerChunk) * kE5DecTile; };
    auto tile_len_of = [&](uint32_t t) {
        const uint64_t b = (uint64_t)t * kE5DecTile;
        return n - b >= kE5DecTile ? kE5DecTile : (uint32_t)(n - b);
    };
    auto last_of_chunk = [&](uint32_t t) { return t % kE5TilesPerChunk == kE5TilesPerChunk - 1 || t == T - 1; };

    // Record windows and walk state (block-uniform).
    RecordWindow<kE5DecThreads> W(S.win, rec, p.n_esc);
    uint32_t chunk_o = 0, chunk_end = 0, cursor = 0;
    auto cover = [&](bool with_prev) {
        const uint32_t nb = min(kE5StepRecs, chunk_end - cursor);
        if (nb > 0) W.cover(with_prev ? cursor - 1 : cursor, cursor + nb);
    };
    // Chunk header checks and store (thread 0), as in the BF16 decoder.
    auto store_header = [&](uint32_t c, uint32_t o, uint32_t m, bool at_chunk_start, uint64_t prev_end) {
        const uint64_t rest = n - (uint64_t)c * kChunk;
        const uint64_t chunk_len = rest < kChunk ? rest : kChunk;
        bool bad = m > chunk_len || o > p.n_esc || m > p.n_esc - o;
        if (at_chunk_start) {
            bad |= (uint64_t)o != (c == 0 ? 0ull : prev_end);
            if (c == p.L.num_chunks - 1) bad |= (uint64_t)o + m != p.n_esc;
        }
        if (bad) S.bad = 1;
        S.hdr[c & 1][0] = o;
        S.hdr[c & 1][1] = bad ? 0u : m;
    };
    // One step: thread tid takes records cursor + tid + 256 k (k < kE5R)
    // while they lie below the tile's end; returns how many it took.  Good
    // ones leave their byte position q[k] in the tile and exponent e[k] for
    // the patch, flagged in bit k of ok.
    auto gather = [&](uint32_t tw, uint32_t prev, uint32_t& ok, uint32_t (&q)[kE5R], uint32_t (&e)[kE5R]) {
        ok = 0;
        const uint32_t p0 = tile_p0(tw);
        uint32_t took = 0;
#pragma unroll
        for (uint32_t k = 0; k < kE5R; k++) {
            // 64-bit: cursor + 511 may pass 2^32 near the end of 2^32 records.
            const uint64_t r64 = (uint64_t)cursor + tid + k * kE5DecThreads;
            if (r64 >= chunk_end) break;
            const uint32_t r = (uint32_t)r64;
            const uint8_t* rp = W.at(r);
            const uint32_t pos = (uint32_t)rp[0] | ((uint32_t)rp[1] << 8);
            if (pos >= p0 + kE5DecTile) break;
            took++;
            const uint32_t before = (tid == 0 && k == 0) ? prev : W.pos(r - 1);
            e[k] = rp[2];
            if (pos < p0 || pos - p0 >= tile_len_of(tw) || (before != 0xFFFFFFFFu && pos <= before) || e[k] >= 32) {
                S.bad = 1;
                continue;
            }
            ok |= 1u << k;
            q[k] = pos - p0;
        }
        return took;
    };
    // Byte q of the tile lives in row q / 64 (warp q / 2048), byte q % 64.
    auto patch = [&](uint32_t q, uint32_t e) {
        const uint32_t t = q >> 6, b = q & 63u;
        uint8_t* at = reinterpret_cast<uint8_t*>(&S.out[t >> 5][swz4(t & 31u, b >> 4)]) + (b & 15u);
        *at = (uint8_t)((*at & 0x83u) | (e << 2));
    };

    // Prologue: the first chunk's header and where the range's records start.
    if (p.L.num_chunks > 0) {
        const uint32_t c = t_begin / kE5TilesPerChunk;
        const bool at_start = t_begin % kE5TilesPerChunk == 0;
        if (tid == 0) {
            const uint8_t* h = p.in + p.L.hdr_off + 8ull * c;
            const uint64_t prev_end = (c > 0 && at_start) ? (uint64_t)load_u32_le(h - 8) + load_u32_le(h - 4) : 0ull;
            store_header(c, load_u32_le(h), load_u32_le(h + 4), at_start, prev_end);
        }
        __syncthreads();
        chunk_o = S.hdr[c & 1][0];
        chunk_end = chunk_o + S.hdr[c & 1][1];
        cursor = chunk_o;
        if (!at_start && chunk_end > chunk_o) {
            uint32_t a, b;
            const uint32_t p0 = tile_p0(t_begin);
            block_lower_bounds<kE5DecThreads>(rec, chunk_o, chunk_end - chunk_o, p0, p0, S.scratch, &a, &b);
            cursor = a;
        }
    }

    uint4* const rows = S.out[warp];
    bool aborted = false;
    uint32_t i = 0;
    for (uint32_t t = t_begin; t < t_end; t++, i++) {
        const uint32_t slot = i % kE5DecStages;
        const uint64_t base = (uint64_t)t * kE5DecTile;
        const uint32_t chunk = t / kE5TilesPerChunk;
        if (p.L.num_chunks > 0 && t % kE5TilesPerChunk == 0 && t != t_begin) {
            chunk_o = S.hdr[chunk & 1][0];
            chunk_end = chunk_o + S.hdr[chunk & 1][1];
            cursor = chunk_o;
        }
        // The next chunk's header, when tile t + 1 starts one: loaded now,
        // stored before this tile's second barrier.
        const bool prefetch = tid == 0 && p.L.num_chunks > 0 && t + 1 < t_end && (t + 1) % kE5TilesPerChunk == 0;
        uint32_t next_o = 0, next_m = 0;
        if (prefetch) {
            const uint8_t* h = p.in + p.L.hdr_off + 8ull * (chunk + 1);
            next_o = load_u32_le(h);
            next_m = load_u32_le(h + 4);
        }

        // Dense pass into this thread's output row.
        const bool failed_wait = !mbar_wait(&S.full[slot], (i / kE5DecStages) & 1u, p.wait_limit_ns);
        const uint64_t thread_base = base + (uint64_t)tid * kE5DecPer;
        const uint32_t cnt =
            thread_base >= n ? 0u : (n - thread_base >= kE5DecPer ? kE5DecPer : (uint32_t)(n - thread_base));
        if (!failed_wait) {
            waited = i + 1;
            uint32_t pw[14];
            if (full_tile(t)) {
                const uint2* src = reinterpret_cast<const uint2*>(S.in[slot] + 56u * tid);
#pragma unroll
                for (int k = 0; k < 7; k++) {
                    const uint2 v = src[k];
                    pw[2 * k] = v.x;
                    pw[2 * k + 1] = v.y;
                }
            } else {
                const uint32_t nbytes = 7 * ((cnt + 7) / 8);
                const uint8_t* src = p.in + thread_base / 8 * 7;
#pragma unroll
                for (int k = 0; k < 14; k++) {
                    uint32_t v = 0;
#pragma unroll
                    for (int b = 0; b < 4; b++)
                        if ((uint32_t)(4 * k + b) < nbytes) v |= (uint32_t)src[4 * k + b] << (8 * b);
                    pw[k] = v;
                }
            }
            if (contig)
                decode_rows<true>(pw, cb0x4, S.dec, rows, lane);
            else
                decode_rows<false>(pw, cb0x4, S.dec, rows, lane);
        }

        // This tile's records: one per thread, counted at the first barrier
        // (which also completes the rows); the holders then patch them.
        uint32_t ok = 0, q[kE5R] = {0, 0}, e[kE5R] = {0, 0};
        cover(false);
        const uint32_t mine = gather(t, 0xFFFFFFFFu, ok, q, e);
        if (failed_wait) S.abort = 1;
        uint32_t k = count_taken_sync<kE5DecThreads>(mine);
        if (S.abort) {
            aborted = true;
            break;
        }
        // The dense pass has consumed the ring slot: refill it now.
        if (tid == 0 && t + kE5DecStages < t_end) issue(slot, t + kE5DecStages), issued++;
#pragma unroll
        for (uint32_t j = 0; j < kE5R; j++)
            if ((ok >> j) & 1u) patch(q[j], e[j]);
        cursor += k;
        while (k == kE5StepRecs && cursor < chunk_end) {  // a full step: maybe more records
            const uint32_t prev = W.pos(cursor - 1);
            cover(true);
            const uint32_t more = gather(t, prev, ok, q, e);
            k = count_taken_sync<kE5DecThreads>(more);
#pragma unroll
            for (uint32_t j = 0; j < kE5R; j++)
                if ((ok >> j) & 1u) patch(q[j], e[j]);
            cursor += k;
        }
        if (last_of_chunk(t) && cursor != chunk_end && tid == 0) S.bad = 1;
        if (t == t_end - 1 && !last_of_chunk(t) && chunk_end > chunk_o) {
            const uint32_t end = tile_p0(t) + kE5DecTile;
            uint32_t a, b;
            block_lower_bounds<kE5DecThreads>(rec, chunk_o, chunk_end - chunk_o, end, end, S.scratch, &a, &b);
            if (tid == 0 && a != cursor) S.bad = 1;
        }
        if (prefetch) store_header(chunk + 1, next_o, next_m, true, chunk_end);
        __syncthreads();  // patches done

        // The warp's rows -> global memory.
        const uint64_t wbase = base + warp * (32u * kE5DecPer);
        if (p.vec && wbase + 32u * kE5DecPer <= n) {
            // 16 elements never straddle a page; the warp's 2,048 elements in
            // one page take one lookup.
            const RunOffset<PAGED> run(p.pm, wbase, 11, 1, p.status);
#pragma unroll
            for (uint32_t r = 0; r < 4; r++) {
                const uint32_t piece = lane + 32 * r;
                st_v4(p.out + run.at(p.pm, wbase, 16 * piece, 1, p.status), rows[swz4(piece >> 2, piece & 3u)]);
            }
        } else {
            const uint8_t* row = reinterpret_cast<const uint8_t*>(rows);
            for (uint32_t b = 0; b < cnt; b++)
                p.out[elem_offset<PAGED>(p.pm, thread_base + b, 1, p.status)] = row[swz4(lane, b >> 4) * 16u + (b & 15u)];
        }
        __syncwarp();  // the rows are rewritten by the next tile
    }
    if (tid == 0 && aborted) {
        for (uint32_t k = waited; k < issued; k++)
            mbar_wait(&S.full[k % kE5DecStages], (k / kE5DecStages) & 1u, p.wait_limit_ns);
        if (p.status) atomicMax(p.status, kStatusTimeout);
    }
    W.drain();
    __syncthreads();
    if (tid == 0 && S.bad && p.status) atomicMax(p.status, kStatusCorrupt);
}

cudaError_t launch_encode_e5m2(const EncodeParams& p, cudaStream_t s) {
    const size_t smem = sizeof(EncodeE5Smem);
    const bool paged = p.pm.ids != nullptr;  // host codebooks only
    auto kern = p.cb_dev   ? encode_e5m2_kernel<2>
                : p.contig ? (paged ? encode_e5m2_kernel<1, true> : encode_e5m2_kernel<1>)
                           : (paged ? encode_e5m2_kernel<0, true> : encode_e5m2_kernel<0>);
    int sms = 0, per_sm = 0;  // one block per scan tile; only the shared memory limit matters
    cudaError_t err = kernel_fit((const void*)kern, kEncThreads, smem, &sms, &per_sm);
    if (err != cudaSuccess) return err;
    kern<<<p.num_tiles, kEncThreads, smem, s>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    EncodeParams q = p;
    q.grid = 0;  // no error words: the E5M2 blocks flag errors in their counts
    return launch_finish(q, false, s);
}

cudaError_t launch_decode_e5m2(const DecodeParams& p, cudaStream_t s) {
    const size_t smem = sizeof(DecodeE5Smem);
    auto kern = p.pm.ids ? decode_e5m2_kernel<true> : decode_e5m2_kernel<false>;
    int sms = 0, per_sm = 0;
    cudaError_t err = kernel_fit((const void*)kern, kE5DecThreads, smem, &sms, &per_sm);
    if (err != cudaSuccess) return err;
    const uint32_t grid = (uint32_t)std::min<uint64_t>(p.num_tiles, (uint64_t)std::max(per_sm, 1) * sms);
    // A programmatic dependent of whatever kernel precedes it (the stream's
    // producer): only the launch overlaps, the kernel waits first thing.
    return launch_dependent(kern, dim3(grid), dim3(kE5DecThreads), smem, s, p);
}

}  // namespace sz
