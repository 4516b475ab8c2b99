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
#include "sz_pipeline.cuh"
#include "sz_records.cuh"

#include <algorithm>
#include <type_traits>

namespace sz {

namespace {

constexpr uint32_t kTilesPerChunk = kChunk / kBf16Tile;  // 8
static_assert(kChunk % kBf16Tile == 0, "tiles must not straddle chunks");
constexpr uint32_t kWarps = kBf16Threads / 32;

}  // namespace

// ---------------------------------------------------------------------------
// Encode, in two kernels.
//
// 1. encode_bf16_kernel streams the tensor: a persistent kernel whose blocks
//    take 32,768-element "scan tiles" (four 8,192-element sub-tiles) in
//    round-robin order.  Sub-tiles arrive through a 2-stage ring of TMA bulk
//    copies; per sub-tile the block splits, codes and packs, stores the dense
//    streams, and ranks the escapes (ballot/popc warp scans, then a block
//    scan).  Each scan tile's escape count and its first ws_cap records, in
//    element order, go to the workspace, and, for a scan tile with more
//    escapes than that, the count of each of its 1,024-element units (one per
//    warp and sub-tile).  Blocks never wait for each other.
// 2. finish_kernel (sz_finish.cu) turns the counts into escape offsets,
//    copies the staged records into the stream, writes the chunk headers and
//    the stream size, and re-derives the records of any scan tile beyond its
//    first ws_cap from the input, unit by unit.
// The records cost 6 extra bytes of traffic per escape (staged, read back),
// a small price for a streaming pass without inter-block waits.
// ---------------------------------------------------------------------------
namespace {

#ifndef SZ_ENC_STAGES
#define SZ_ENC_STAGES 2
#endif
#ifndef SZ_ENC_MIN_BLOCKS
#define SZ_ENC_MIN_BLOCKS 4
#endif
constexpr uint32_t kEncStages = SZ_ENC_STAGES;   // input ring depth (16 KB sub-tiles)
constexpr uint32_t kSubsPerScan = 4;
constexpr uint32_t kComputeThreads = kBf16Threads;           // 256
constexpr uint32_t kTileBytes = kBf16Tile * 2;               // 16 KB of BF16 per sub-tile
static_assert(kBf16Tile * kSubsPerScan == kScanTile, "four sub-tiles per scan tile");
static_assert(kBf16Tile / kWarps == kUnitElems, "a unit is one warp's share of a sub-tile");

struct EncodeSmem {
    alignas(128) uint8_t in[kEncStages][kTileBytes];
    uint64_t full[kEncStages];        // TMA -> compute: sub-tile landed
    alignas(16) uint32_t warp_esc[kSubsPerScan][kWarps];  // warp totals of the scan tile's sub-tiles
    alignas(16) uint8_t rec[3 * kStageRecsBf16];  // the scan tile's staged records
    uint8_t code[256];                // exponent -> code; 0x10 marks an escape
    int err;                          // the block's error code (paged input: bad page ids)
};

struct GroupOut {
    uint32_t sm_lo, sm_hi, nib, esc;
    uint32_t ex0, ex1;  // the exponent bytes of elements 0..3 and 4..7
};

// Split and code one group of 8 elements (four 32-bit words of BF16 pairs).
// The low bytes (exponent bit 0 | mantissa) and high bytes (sign | exponent
// bits 7..1) of four elements are gathered with byte permutes; the
// sign|mantissa bytes then take one 3-input op, and the four exponents two
// shifts and one 3-input op.
// CONTIG (codebook cb0..cb0+15): d = exponent - cb0 mod 256 per byte, with a
// carry-free byte-wise add; the element is in the codebook iff d < 16, and d
// is then its code.  Escaped elements are rare, so their nibbles are fixed in
// a separate branch.
template <bool CONTIG, bool FULL>
__device__ __forceinline__ GroupOut code_group(const uint32_t (&w)[4], uint32_t cnt, uint32_t sub_lo,
                                               const uint8_t* s_code) {
    GroupOut o;
    const uint32_t L0 = __byte_perm(w[0], w[1], 0x6420), H0 = __byte_perm(w[0], w[1], 0x7531);
    const uint32_t L1 = __byte_perm(w[2], w[3], 0x6420), H1 = __byte_perm(w[2], w[3], 0x7531);
    o.sm_lo = (H0 & 0x80808080u) | (L0 & 0x7F7F7F7Fu);
    o.sm_hi = (H1 & 0x80808080u) | (L1 & 0x7F7F7F7Fu);
    // Exponent byte = (high byte << 1) | (low byte >> 7): both shifts as
    // multiplies (FMA pipe; the coding is ALU-bound), then one 3-input op
    // keeps bits 1..7 of the first and bit 0 of the second in every byte.
    const uint32_t e0 = (mad_lo<2u>(H0, 0u) & 0xFEFEFEFEu) | (mul_hi<1u << 25>(L0) & 0x01010101u);  // exponents 0..3
    const uint32_t e1 = (mad_lo<2u>(H1, 0u) & 0xFEFEFEFEu) | (mul_hi<1u << 25>(L1) & 0x01010101u);  // exponents 4..7
    uint32_t m = 0;
    if (CONTIG) {
        // sub_lo = (256 - cb0) mod 256 in every byte.
        const uint32_t b7 = sub_lo & 0x7F7F7F7Fu, b8 = sub_lo & 0x80808080u;
        const uint32_t d0 = ((e0 & 0x7F7F7F7Fu) + b7) ^ (e0 & 0x80808080u) ^ b8;
        const uint32_t d1 = ((e1 & 0x7F7F7F7Fu) + b7) ^ (e1 & 0x80808080u) ^ b8;
        uint32_t c0 = d0, c1 = d1;
        if ((d0 | d1) & 0xF0F0F0F0u) {
            // Escapes: bytes with d >= 16, flagged in their bit 7 (adding
            // 0x70 to the low 7 bits carries into bit 7 from 16 up; a set
            // bit 7 is an escape already).  Codes of escaped bytes are zeroed
            // (g >> 7 as a high multiply, times 0xFF), and the flags gathered
            // into the mask by one high multiply: bit 8j + 7 lands on bit j,
            // every other partial product below bit 32 or above bit 35.
            const uint32_t g0 = (((d0 & 0x7F7F7F7Fu) + 0x70707070u) | d0) & 0x80808080u;
            const uint32_t g1 = (((d1 & 0x7F7F7F7Fu) + 0x70707070u) | d1) & 0x80808080u;
            c0 &= ~(mul_hi<1u << 25>(g0) * 0xFFu);
            c1 &= ~(mul_hi<1u << 25>(g1) * 0xFFu);
            m = mad_lo<16u>(mul_hi<0x02040810u>(g1) & 0xFu, mul_hi<0x02040810u>(g0) & 0xFu);
        }
        // Bytes 0, 2: code pairs (every byte of c is < 16, so c + (c >> 4) = c | (c >> 4)).
        const uint32_t p0 = mad_hi<1u << 28>(c0, c0), p1 = mad_hi<1u << 28>(c1, c1);
        o.nib = __byte_perm(p0, p1, 0x6420);
    } else {
        uint32_t nib = 0, flags = 0;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const uint32_t c = s_code[((j < 4 ? e0 : e1) >> (8 * (j & 3))) & 0xFFu];
            nib |= (c & 0xFu) << (4 * j);
            flags |= (c & 0x10u) << j;  // bit 4 + j set for an escape
        }
        m = (flags >> 4) & 0xFFu;
        o.nib = nib;
    }
    if (!FULL && cnt < 8) {
        m &= (1u << cnt) - 1u;
        o.nib &= (uint32_t)((1ull << (4 * cnt)) - 1ull);
    }
    o.esc = m;
    o.ex0 = e0;
    o.ex1 = e1;
    return o;
}

// Escape ranks inside one warp's 1024 elements, in (k, lane, j) order:
// off[k] = escapes of this warp before lane's group k; returns the warp total.
__device__ __forceinline__ uint32_t warp_escape_ranks(const uint32_t (&esc)[4], uint32_t lane, uint32_t (&off)[4]) {
    off[0] = off[1] = off[2] = off[3] = 0;
    if (!__any_sync(0xFFFFFFFFu, (esc[0] | esc[1] | esc[2] | esc[3]) != 0)) return 0;
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
    return tot0 + tot1 + tot2 + tot3;
}

}  // namespace

// Loads lane's 4 groups of 8 elements of one warp's 1,024 elements starting
// at element `base` (= sub-tile start + 1024 warp), from global memory.
// A group of 8 never straddles a page (pages hold a power of two >= 16
// elements), so one page lookup serves the whole group.
template <bool PAGED>
__device__ __forceinline__ void load_groups_global(const EncodeParams& p, uint64_t base, uint32_t lane,
                                                   uint32_t (&w)[4][4], uint32_t (&cnt)[4], int* err) {
    const uint64_t n = p.L.n;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint64_t i0 = base + k * 256u + lane * 8u;
        cnt[k] = i0 >= n ? 0u : (n - i0 >= 8 ? 8u : (uint32_t)(n - i0));
        const uint8_t* g = p.in + (cnt[k] ? elem_offset<PAGED>(p.pm, i0, 2, err) : 2 * i0);
        if (p.vec && cnt[k] == 8) {
            const uint4 v = ld_stream_v4(g);
            w[k][0] = v.x, w[k][1] = v.y, w[k][2] = v.z, w[k][3] = v.w;
        } else {
#pragma unroll
            for (int q = 0; q < 4; q++) w[k][q] = 0;
#pragma unroll
            for (int jj = 0; jj < 8; jj++) {
                if ((uint32_t)jj < cnt[k]) {
                    const uint8_t* e = g + 2 * jj;
                    w[k][jj >> 1] |= ((uint32_t)e[0] | ((uint32_t)e[1] << 8)) << (16 * (jj & 1));
                }
            }
        }
    }
}

// Writes the records of lane's escapes among one warp's 1,024 elements
// starting at element `base`: record index first + off[k] + rank in group k,
// for indexes below cap.  One loop per group, so that each group's exponent
// words and offset are fixed registers: an iteration is a handful of
// instructions, and the warp iterates as often as the busiest lane of each
// group has escapes.
__device__ __forceinline__ void emit_records(uint64_t base, uint32_t lane, const uint32_t (&ex)[4][2],
                                             const uint32_t (&esc)[4], const uint32_t (&off)[4], uint32_t first,
                                             uint8_t* dst, uint32_t cap) {
    const uint32_t pos_base = (uint32_t)(base + lane * 8u) & 0xFFFFu;  // a warp never straddles a chunk
#pragma unroll
    for (uint32_t k = 0; k < 4; k++) {
        uint32_t m = esc[k], idx = first + off[k];
        while (m) {
            const uint32_t jj = __ffs(m) - 1;
            m &= m - 1;
            // Byte jj of the group's exponent bytes (the low byte is stored).
            const uint32_t e = __byte_perm(ex[k][0], ex[k][1], jj);
            const uint32_t pos = pos_base + k * 256u + jj;
            if (idx < cap) {
                dst[3 * idx] = (uint8_t)pos;
                dst[3 * idx + 1] = (uint8_t)(pos >> 8);
                dst[3 * idx + 2] = (uint8_t)e;
            }
            idx++;
        }
    }
}

// bad_codebook: the device codebook failed its check (SZ_ERR_INVALID_ARG).
// At its end the block writes its error code to ws_err[blockIdx.x].
template <bool CONTIG, bool PAGED>
__device__ __forceinline__ void encode_bf16_body(const EncodeParams& p, const uint8_t (&cb)[16], bool bad_codebook) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    EncodeSmem& S = *reinterpret_cast<EncodeSmem*>(smem_raw);
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint64_t n = p.L.n;
    const uint32_t G = p.grid;
    const uint32_t num_scan = p.num_tiles;                          // scan tiles
    const uint32_t num_subs = n == 0 ? 1u : (uint32_t)((n + kBf16Tile - 1) / kBf16Tile);
    const uint32_t my_scans = blockIdx.x >= num_scan ? 0u : (num_scan - 1 - blockIdx.x) / G + 1;
    auto scan_of = [&](uint32_t k) { return blockIdx.x + k * G; };
    auto subs_in = [&](uint32_t st) { return min(kSubsPerScan, num_subs - st * kSubsPerScan); };
    // Sub-tiles of this block, in order: index i -> scan tile i/4, part i%4.
    const uint32_t my_subs = my_scans == 0 ? 0u : (my_scans - 1) * kSubsPerScan + subs_in(scan_of(my_scans - 1));
    auto sub_of = [&](uint32_t i) { return scan_of(i / kSubsPerScan) * kSubsPerScan + i % kSubsPerScan; };
    // Paged input goes through the ring when a sub-tile is at most 8 page
    // pieces (pages of >= 1,024 elements); smaller pages are read directly.
    const uint32_t piece_lg = PAGED ? min(p.pm.lg, 13u) : 13u;  // 2^13 = one sub-tile
    auto full_sub = [&](uint32_t u) {
        return p.vec && (uint64_t)(u + 1) * kBf16Tile <= n && (!PAGED || p.pm.lg >= 10);
    };

    if (tid == 0) {
        for (uint32_t s = 0; s < kEncStages; s++) mbar_init(&S.full[s], 1);
        S.err = 0;  // reported to only after the barrier below
        fence_mbar_init();
    }
    {
        uint32_t code = 0x10u;
#pragma unroll
        for (int k = 0; k < kCodes; k++)
            if (cb[k] == tid) code = (uint32_t)k;
        S.code[tid] = (uint8_t)code;
    }
    if (blockIdx.x == 0 && tid == 0) {
#pragma unroll
        for (int k = 0; k < kCodes; k++) p.out[p.L.cb_off + k] = cb[k];
    }
    __syncthreads();

    const uint32_t lane_add = ((0x100u - cb[0]) & 0xFFu) * 0x01010101u;  // (256 - cb0) per byte
    auto issue = [&](uint32_t i) {  // thread 0 only: sub-tile i of this block into ring slot i % S
        const uint32_t u = sub_of(i), slot = i % kEncStages;
        if (p.skip_first && blockIdx.x == 0 && i == 0) return;  // test hook: this slot never fills
        if (full_sub(u)) {
            mbar_arrive_expect_tx(&S.full[slot], kTileBytes);
            if (PAGED) {
                const uint32_t piece = 1u << piece_lg;  // elements per copy
                for (uint32_t e = 0; e < kBf16Tile; e += piece)
                    bulk_g2s(S.in[slot] + 2 * e, p.in + elem_offset<true>(p.pm, (uint64_t)u * kBf16Tile + e, 2, &S.err),
                             2 * piece, &S.full[slot]);
            } else {
                bulk_g2s(S.in[slot], p.in + (uint64_t)u * kTileBytes, kTileBytes, &S.full[slot]);
            }
        } else {
            mbar_arrive(&S.full[slot]);  // read straight from global instead
        }
    };
    uint32_t issued = 0, waited = 0;
    if (tid == 0)
        for (; issued < my_subs && issued < kEncStages; issued++) issue(issued);

    bool aborted = false;
    uint32_t i = 0;  // sub-tiles processed by this block
    for (uint32_t ks = 0; ks < my_scans && !aborted; ks++) {
        const uint32_t st = scan_of(ks);
        const uint32_t subs = subs_in(st);
        uint32_t run = 0;  // escapes so far in this scan tile
        for (uint32_t part = 0; part < subs; part++, i++) {
            const uint32_t slot = i % kEncStages;
            const uint32_t u = st * kSubsPerScan + part;
            const uint64_t wbase = (uint64_t)u * kBf16Tile + warp * 1024u;
            // A failed wait is voted on at the block barrier below, so that all
            // threads leave the loop together.
            const bool failed_wait = !mbar_wait(&S.full[slot], (i / kEncStages) & 1u, p.wait_limit_ns);
            if (!failed_wait) waited = i + 1;
            uint32_t w[4][4], cnt[4], esc[4], ex[4][2];
            if (full_sub(u)) {
                // Whole sub-tile in range, buffers aligned: no bounds logic;
                // lane's group k sits at constant offsets from its group 0.
                const uint8_t* src = S.in[slot] + 2 * (warp * 1024u + lane * 8u);
                uint8_t* o_sm = p.out + wbase + lane * 8u;
                uint8_t* o_nib = p.out + p.L.nib_off + (wbase + lane * 8u) / 2;
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const uint4 v = *reinterpret_cast<const uint4*>(src + k * 512);
                    w[k][0] = v.x, w[k][1] = v.y, w[k][2] = v.z, w[k][3] = v.w;
                    const GroupOut o = code_group<CONTIG, true>(w[k], 8, lane_add, S.code);
                    esc[k] = o.esc;
                    ex[k][0] = o.ex0, ex[k][1] = o.ex1;
                    st_stream_v2(o_sm + k * 256, make_uint2(o.sm_lo, o.sm_hi));
                    st_stream_u32(o_nib + k * 128, o.nib);
                }
            } else {
                load_groups_global<PAGED>(p, wbase, lane, w, cnt, &S.err);
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const uint64_t i0 = wbase + k * 256u + lane * 8u;
                    const GroupOut o = code_group<CONTIG, false>(w[k], cnt[k], lane_add, S.code);
                    esc[k] = o.esc;
                    ex[k][0] = o.ex0, ex[k][1] = o.ex1;
                    if (p.vec && cnt[k] == 8) {
                        st_stream_v2(p.out + i0, make_uint2(o.sm_lo, o.sm_hi));
                        st_stream_u32(p.out + p.L.nib_off + i0 / 2, o.nib);
                    } else if (cnt[k] > 0) {
                        const uint64_t smv = (uint64_t)o.sm_lo | ((uint64_t)o.sm_hi << 32);
                        for (uint32_t jj = 0; jj < cnt[k]; jj++) p.out[i0 + jj] = (uint8_t)(smv >> (8 * jj));
                        for (uint32_t b = 0; b < (cnt[k] + 1) / 2; b++)
                            p.out[p.L.nib_off + i0 / 2 + b] = (uint8_t)(o.nib >> (8 * b));
                    }
                }
            }
            uint32_t off[4];
            const uint32_t warp_total = warp_escape_ranks(esc, lane, off);
            if (lane == 0) S.warp_esc[part][warp] = warp_total;
            // Block barrier: warp totals visible, the ring slot consumed by
            // every thread (its words were used by the stores above).
            if (__syncthreads_or(failed_wait)) {
                aborted = true;
                break;
            }
            if (tid == 0 && issued < my_subs) issue(issued++);
            uint32_t warp_off, sub_esc;
            {
                // Inclusive prefix sums of the 8 warp totals; this warp's
                // offset is the one before it, picked by the warp index bits
                // (fixed per thread, so the tests leave the loop).
                static_assert(kWarps == 8, "eight warp totals");
                const uint4 a = *reinterpret_cast<const uint4*>(&S.warp_esc[part][0]);
                const uint4 b = *reinterpret_cast<const uint4*>(&S.warp_esc[part][4]);
                const uint32_t p0 = a.x, p1 = p0 + a.y, p2 = p1 + a.z, p3 = p2 + a.w;
                const uint32_t p4 = p3 + b.x, p5 = p4 + b.y, p6 = p5 + b.z, p7 = p6 + b.w;
                const uint32_t lo = (warp & 2u) ? ((warp & 1u) ? p2 : p1) : ((warp & 1u) ? p0 : 0u);
                const uint32_t hi = (warp & 2u) ? ((warp & 1u) ? p6 : p5) : ((warp & 1u) ? p4 : p3);
                warp_off = (warp & 4u) ? hi : lo;
                sub_esc = p7;
            }
            // Records beyond ws_cap are not staged; the finish kernel re-derives
            // that scan tile's records from the input.  They are gathered in
            // shared memory and leave once per scan tile, in 16-byte stores.
            if (warp_total && run + warp_off < p.ws_cap)
                emit_records(wbase, lane, ex, esc, off, run + warp_off, S.rec, p.ws_cap);
            run += sub_esc;
        }
        if (aborted) break;  // block-uniform
        if (tid == 0) p.ws_count[st] = run;
        __syncthreads();  // every record of the scan tile is in S.rec
        // A scan tile with more escapes than it stages also leaves the escape
        // count of each unit (warp w of sub-tile part is unit part * 8 + w),
        // from which the finish kernel re-derives the rest; others need none.
        if (run > p.ws_cap && tid < subs * kWarps)
            p.ws_unit[(uint64_t)st * kUnitsPerScan + tid] = (uint16_t)S.warp_esc[tid / kWarps][tid % kWarps];
        {
            // The workspace region (3 ws_cap bytes, a multiple of 16) starts
            // 16-byte aligned, so whole 16-byte pieces stay inside it.
            const uint32_t nbytes = 3 * min(run, p.ws_cap);
            uint8_t* dst = p.ws_rec + (uint64_t)st * 3 * p.ws_cap;
            for (uint32_t b = 16 * tid; b < nbytes; b += 16 * kComputeThreads)
                *reinterpret_cast<uint4*>(dst + b) = *reinterpret_cast<const uint4*>(S.rec + b);
        }
        // The next scan tile writes S.rec only after its first sub-tile's
        // barrier, which every thread reaches after this copy.
    }
    if (aborted && tid == 0) {
        // Copies in flight must land before the block exits (bounded).
        for (uint32_t k = waited; k < issued; k++)
            if (!(p.skip_first && blockIdx.x == 0 && k == 0))
                mbar_wait(&S.full[k % kEncStages], (k / kEncStages) & 1u, p.wait_limit_ns);
    }
    // The block's error code for the finish kernel: a timed-out wait, a bad
    // device codebook, or (paged input, reported by any thread) a bad page id.
    if (PAGED) __syncthreads();
    if (tid == 0)
        p.ws_err[blockIdx.x] = aborted ? kStatusTimeout : (bad_codebook ? kStatusInvalid : (PAGED ? S.err : 0));
}

// MODE 0: codebook in the parameters, table coding; 1: in the parameters,
// contiguous; 2: in device memory, checked (a bad one is reported as
// SZ_ERR_INVALID_ARG) and the coding chosen on the device.
// PAGED: the input is a paged tensor (EncodeParams::pm).
template <int MODE, bool PAGED = false>
__global__ void __launch_bounds__(kComputeThreads, SZ_ENC_MIN_BLOCKS) encode_bf16_kernel(const EncodeParams p) {
    uint8_t cb[16];
    bool contig;
    const bool ok = load_codebook(p.cb, MODE == 2 ? p.cb_dev : nullptr, 256u, cb, contig);
    if (MODE == 2) {
        if (contig)
            encode_bf16_body<true, false>(p, cb, !ok);
        else
            encode_bf16_body<false, false>(p, cb, !ok);
    } else {
        encode_bf16_body<MODE == 1, PAGED>(p, cb, false);
    }
}

// ---------------------------------------------------------------------------
// Decode: a persistent kernel; block b owns the contiguous tile range
// [bT/G, (b+1)T/G).  Because escape records are stored in element order, a
// block's records also form one contiguous run of the stream: one block
// search finds where the run starts (only when the range starts inside a
// chunk), then a cursor walks the records through shared-memory windows
// that asynchronous copies fill ahead of the walk (RecordWindow).
// Dense input (sign|mantissa bytes and nibbles) arrives through a 2-stage ring
// of TMA bulk copies.  Per tile: nibble byte -> two exponents via a 256-entry
// LUT, joined with the sm bytes; the tile's escapes, gathered into a bitmap
// and an exponent table, are applied in registers, so every output byte is
// stored once.
//
// One block barrier per tile.  The escapes are gathered one tile ahead into
// the other of two bitmap/table buffers: while tile t is decoded from buffer
// t % 2, every thread takes up to four of the next 1,024 records (cursor +
// tid + 256 k) and, for each that lies below tile t+1's end, checks it and
// enters it into buffer (t+1) % 2.  The tile's closing barrier
// (count_prefix_sync) both publishes those entries and counts them, which
// advances the cursor; only a tile with more than 1,024 escapes takes further
// counted steps.  The record windows keep two windows of copies in flight
// ahead of the walk.  A bitmap word is read only by its owning thread, which
// clears it right after reading.  Chunk headers are read two tiles ahead,
// also ahead of a closing barrier.
//
// Validation: every record is consumed by exactly one tile and checked there
// (position inside the tile, above the previous one); a chunk's last tile
// checks that all of the chunk's records were consumed, and a block whose
// range ends inside a chunk checks that its cursor stops where the next
// block's search starts.  Headers are checked as running sums.
// ---------------------------------------------------------------------------
namespace {

constexpr uint32_t kDecStages = 2;
constexpr uint32_t kDecThreads = kBf16Threads;  // 256
constexpr uint32_t kDecR = 4;                   // records a thread takes per step
constexpr uint32_t kDecWindows = 4;             // record windows: two resident, two in flight
constexpr uint32_t kStepRecs = kDecR * kDecThreads;

struct DecodeSmem {
    alignas(128) uint8_t sm[kDecStages][kBf16Tile];
    alignas(128) uint8_t nib[kDecStages][kBf16Tile / 2];
    uint64_t full[kDecStages];
    uint32_t lut[256];
    uint32_t bits[2][kDecThreads];  // escape bitmaps: word tid belongs to thread tid
    uint8_t patch[2][kBf16Tile];    // escape exponents by position in the tile
    alignas(16) uint8_t win[kDecWindows][kWinBytes];  // record windows (RecordWindow)
    uint32_t hdr[2][2];             // {offset, count} of a chunk, by chunk parity
    uint32_t taken[2][kDecThreads / 32];  // per-warp step counts (count_prefix_sync)
    uint32_t scratch[8];
    int bad;
    int abort;
};

// Four blocks per SM: 4 x (this + 1 KB reserved) within 228 KB.
static_assert(sizeof(DecodeSmem) <= 56 * 1024, "decode shared memory");

}  // namespace

// PAGED: the output is a paged tensor (DecodeParams::pm).
// TOP8: the Top-8 layout of the codebook ablation (3-bit codes, 8 per 3
// bytes, an 8-entry codebook); everything else is shared.
// ADDS: for streams dense in escapes (the host picks it from the escape
// count): with a codebook of 16 consecutive exponents cb0 .. cb0 + 15, whole
// tiles take their exponents from code + cb0 instead of the 256-entry table.
// A table lookup per two elements reads shared memory at random banks, and
// where the escape tables are busy too that costs more than the adds; on
// sparse streams the table measured faster, so they keep it.
template <bool PAGED, bool TOP8 = false, bool ADDS = false>
__global__ void __launch_bounds__(kDecThreads, 4) decode_bf16_kernel(const DecodeParams p) {
    constexpr uint32_t kCodeBytes = TOP8 ? kBf16Tile / 8 * 3 : kBf16Tile / 2;  // code bytes per tile
    constexpr int kEntries = TOP8 ? 8 : kCodes;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // launched as a programmatic dependent
    extern __shared__ __align__(128) uint8_t smem_raw[];
    DecodeSmem& S = *reinterpret_cast<DecodeSmem*>(smem_raw);
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint64_t n = p.L.n;
    const uint32_t T = p.num_tiles, G = gridDim.x;
    const uint32_t t_begin = (uint32_t)((uint64_t)blockIdx.x * T / G);
    const uint32_t t_end = (uint32_t)((uint64_t)(blockIdx.x + 1) * T / G);
    const uint8_t* cb = p.in + p.L.cb_off;
    const uint8_t* rec = p.in + p.L.rec_off;
    // Bulk copies need both dense streams 16-byte aligned.
    const bool tma = p.vec && (reinterpret_cast<uintptr_t>(p.in) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(p.in + p.L.nib_off) % 16 == 0);

    if (tid == 0) {
        for (uint32_t s = 0; s < kDecStages; s++) mbar_init(&S.full[s], 1);
        S.bad = 0;
        S.abort = 0;
        fence_mbar_init();
    }
    // Two codes -> their two exponents, pre-shifted into both 16-bit halves:
    // a nibble byte (Top-16) or 6 bits (Top-8).
    if (TOP8)
        S.lut[tid] = tid < 64 ? ((uint32_t)cb[tid & 7u] << 7) | ((uint32_t)cb[tid >> 3] << 23) : 0u;
    else
        S.lut[tid] = ((uint32_t)cb[tid & 15u] << 7) | ((uint32_t)cb[tid >> 4] << 23);
    S.bits[0][tid] = 0;
    S.bits[1][tid] = 0;
    if (tid < (uint32_t)kEntries) {  // a codebook holds distinct exponents
        bool dup = false;
        for (int k = 0; k < kEntries; k++) dup |= (k != (int)tid) && cb[k] == cb[tid];
        if (dup) S.bad = 1;  // ordered before the reads by the barriers below
    }
    // Consecutive codebook (no wrap): exponent = code + cb0 (ADDS only).
    bool contig = false;
    if (ADDS && !TOP8) {
        const bool mine = tid >= (uint32_t)kCodes || ((uint32_t)cb[0] + 15u <= 255u && cb[tid] == cb[0] + tid);
        contig = __syncthreads_and(mine) != 0;
    } else {
        __syncthreads();
    }
    const uint32_t add7 = ((uint32_t)cb[0] * 0x10001u) << 7;  // cb0 at bits 7 and 23

    auto full_tile = [&](uint32_t t) { return tma && (uint64_t)(t + 1) * kBf16Tile <= n; };
    auto issue = [&](uint32_t slot, uint32_t t) {  // thread 0 only
        if (full_tile(t)) {
            mbar_arrive_expect_tx(&S.full[slot], kBf16Tile + kCodeBytes);
            bulk_g2s(S.sm[slot], p.in + (uint64_t)t * kBf16Tile, kBf16Tile, &S.full[slot]);
            bulk_g2s(S.nib[slot], p.in + p.L.nib_off + (uint64_t)t * kCodeBytes, kCodeBytes, &S.full[slot]);
        } else {
            mbar_arrive(&S.full[slot]);
        }
    };
    uint32_t issued = 0, waited = 0;
    if (tid == 0)
        for (uint32_t t = t_begin; t < t_end && t < t_begin + kDecStages; t++, issued++) issue((t - t_begin) % kDecStages, t);

    auto tile_p0 = [&](uint32_t t) { return (t % kTilesPerChunk) * kBf16Tile; };
    auto tile_len_of = [&](uint32_t t) {
        const uint64_t b = (uint64_t)t * kBf16Tile;
        return n - b >= kBf16Tile ? kBf16Tile : (uint32_t)(n - b);
    };
    auto last_of_chunk = [&](uint32_t t) { return t % kTilesPerChunk == kTilesPerChunk - 1 || t == T - 1; };

    // Record windows and the walk state (the chunk of the tile whose escapes
    // are gathered next).  All of it is block-uniform, so every thread
    // reaches the same barriers.
    RecordWindow<kDecThreads, kDecWindows> W(S.win, rec, p.n_esc);
    uint32_t parity = 0;  // count_prefix_sync's slot parity (block-uniform)
    auto count_step = [&](uint32_t took) { return count_prefix_sync<kDecThreads, kDecR>(took, &S.taken[0][0], parity); };
    uint32_t chunk_o = 0, chunk_end = 0, cursor = 0;
    // The next step's records [cursor, cursor + kStepRecs), and record
    // cursor - 1 when the step continues a tile, must be resident.
    auto cover = [&](bool with_prev) {
        const uint32_t nb = min(kStepRecs, chunk_end - cursor);
        if (nb > 0) W.cover(with_prev ? cursor - 1 : cursor, cursor + nb);
    };
    // Chunk header {o, m} of chunk c into S.hdr[c & 1], after its checks;
    // prev_end is o + m of chunk c - 1 (used only at a chunk's first tile).
    // Thread 0 only.
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
        return (uint64_t)o + (bad ? 0u : m);
    };
    // A tile at a chunk start takes the chunk's records from its header.
    auto begin_tile = [&](uint32_t tw) {
        if (p.L.num_chunks > 0 && tw % kTilesPerChunk == 0) {
            const uint32_t c = tw / kTilesPerChunk;
            chunk_o = S.hdr[c & 1][0];
            chunk_end = chunk_o + S.hdr[c & 1][1];
            cursor = chunk_o;
        }
    };
    // One gathering step for tile tw into buffer b: thread tid takes records
    // cursor + tid + 256 k (k < kDecR) while they lie below the tile's end.
    // Returns how many it took; each is checked, and a good one is entered.
    // prev: position of the tile's record before the cursor, or ~0 at the
    // tile's start.
    auto gather = [&](uint32_t tw, uint32_t b, uint32_t prev) {
        const uint32_t p0 = tile_p0(tw);
        uint32_t took = 0;
#pragma unroll
        for (uint32_t k = 0; k < kDecR; k++) {
            // 64-bit: cursor + 1023 may pass 2^32 near the end of 2^32 records.
            const uint64_t r64 = (uint64_t)cursor + tid + k * kDecThreads;
            if (r64 >= chunk_end) break;
            const uint32_t r = (uint32_t)r64;
            const uint8_t* rp = W.at(r);
            const uint32_t pos = (uint32_t)rp[0] | ((uint32_t)rp[1] << 8);
            if (pos >= p0 + kBf16Tile) break;
            took++;
            const uint32_t before = (tid == 0 && k == 0) ? prev : W.pos(r - 1);
            if (pos < p0 || pos - p0 >= tile_len_of(tw) || (before != 0xFFFFFFFFu && pos <= before)) {
                S.bad = 1;
                continue;
            }
            const uint32_t q = pos - p0;
            S.patch[b][q] = rp[2];
            atomicOr(&S.bits[b][(q >> 10) * 32u + ((q >> 3) & 31u)], 1u << (((q >> 8) & 3u) * 8u + (q & 7u)));
        }
        return took;
    };
    // After a counted step that took k records: further steps while a step
    // was full, then the chunk-end and hand-off checks of tile tw.
    auto end_tile = [&](uint32_t tw, uint32_t b, uint32_t k) {
        cursor += k;
        while (k == kStepRecs && cursor < chunk_end) {
            const uint32_t prev = W.pos(cursor - 1);  // still resident
            cover(true);
            k = count_step(gather(tw, b, prev));
            cursor += k;
        }
        if (last_of_chunk(tw) && cursor != chunk_end && tid == 0) S.bad = 1;
        if (tw == t_end - 1 && !last_of_chunk(tw) && chunk_end > chunk_o) {
            // Hand-off: the next block starts its walk where its search says.
            const uint32_t e = tile_p0(tw) + kBf16Tile;
            uint32_t a, bb;
            block_lower_bounds<kDecThreads>(rec, chunk_o, chunk_end - chunk_o, e, e, S.scratch, &a, &bb);
            if (tid == 0 && a != cursor) S.bad = 1;
        }
    };

    // Prologue: the first chunk's header (and the next one's when tile
    // t_begin + 1 starts a chunk), where the range's records start, and the
    // escapes of tile t_begin.
    if (t_begin < t_end) {
        if (p.L.num_chunks > 0) {
            const uint32_t c = t_begin / kTilesPerChunk;
            const bool at_start = t_begin % kTilesPerChunk == 0;
            if (tid == 0) {
                const uint8_t* h = p.in + p.L.hdr_off + 8ull * c;
                const uint64_t prev_end =
                    (c > 0 && at_start) ? (uint64_t)load_u32_le(h - 8) + load_u32_le(h - 4) : 0ull;
                const uint64_t end = store_header(c, load_u32_le(h), load_u32_le(h + 4), at_start, prev_end);
                if (t_begin + 1 < t_end && (t_begin + 1) % kTilesPerChunk == 0)
                    store_header(c + 1, load_u32_le(h + 8), load_u32_le(h + 12), true, end);
            }
            __syncthreads();
            chunk_o = S.hdr[c & 1][0];
            chunk_end = chunk_o + S.hdr[c & 1][1];
            cursor = chunk_o;
            if (!at_start && chunk_end > chunk_o) {
                uint32_t a, b;
                const uint32_t p0 = tile_p0(t_begin);
                block_lower_bounds<kDecThreads>(rec, chunk_o, chunk_end - chunk_o, p0, p0, S.scratch, &a, &b);
                cursor = a;
            }
        }
        cover(false);
        end_tile(t_begin, 0, count_step(gather(t_begin, 0, 0xFFFFFFFFu)));
    }

    bool aborted = false;
    uint32_t i = 0;
    for (uint32_t t = t_begin; t < t_end; t++, i++) {
        const uint32_t slot = i % kDecStages, buf = i & 1u;
        const uint64_t base = (uint64_t)t * kBf16Tile;

        // The header of the chunk that starts at tile t + 2: loaded now,
        // checked and stored before this tile's closing barrier.  Its
        // predecessor is the chunk of tiles t and t + 1.
        const bool prefetch = tid == 0 && p.L.num_chunks > 0 && t + 2 < t_end && (t + 2) % kTilesPerChunk == 0;
        uint32_t next_o = 0, next_m = 0;
        if (prefetch) {
            const uint8_t* h = p.in + p.L.hdr_off + 8ull * ((t + 2) / kTilesPerChunk);
            next_o = load_u32_le(h);
            next_m = load_u32_le(h + 4);
        }

        // Tile t: dense input, with the escapes gathered into buffer buf.
        const bool failed_wait = !mbar_wait(&S.full[slot], (i / kDecStages) & 1u, p.wait_limit_ns);
        if (!failed_wait) {
            waited = i + 1;
            const uint32_t bits = S.bits[buf][tid];
            S.bits[buf][tid] = 0;  // only this thread reads this word
            const uint32_t qt = warp * 1024u + lane * 8u;  // the thread's first element in the tile
            // Group k of the thread: sm bytes (2 words), nibbles (1 word) -> 4 output words.
            // CONTIG (a std::bool_constant): exponents by byte adds, else by
            // the table.
            auto decode_group = [&](auto CONTIG, int k, uint2 smv, uint32_t nibv, uint32_t (&y)[4]) {
                // The low and the high code of every nibble byte, one per byte.
                const uint32_t c_lo = nibv & 0x0F0F0F0Fu, c_hi = (nibv >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    // Each sm byte twice per 16-bit half: the high copy keeps the
                    // sign (bit 15), the low copy the mantissa (bits 0..6).
                    const uint32_t smw = q < 2 ? smv.x : smv.y;
                    const uint32_t tt = __byte_perm(smw, 0, (q & 1) ? 0x3322 : 0x1100);
                    uint32_t e;
                    if (decltype(CONTIG)::value) {
                        // Byte q of c_lo and of c_hi into bytes 0 and 2; bytes 1
                        // and 3 are the (zero) sign of a code byte.
                        e = prmt(c_lo, c_hi, 0xC480u + 0x1111u * q) * 128u + add7;
                    } else {
                        e = S.lut[TOP8 ? (nibv >> (6 * q)) & 63u : (nibv >> (8 * q)) & 0xFFu];
                    }
                    y[q] = (tt & 0x807F807Fu) | e;
                }
                const uint32_t gb = (bits >> (8 * k)) & 0xFFu;
                if (gb) {
                    const uint8_t* pt = S.patch[buf] + qt + k * 256u;
#pragma unroll
                    for (int jj = 0; jj < 8; jj++) {
                        if ((gb >> jj) & 1u) {
                            const uint32_t sh = 7 + 16 * (jj & 1);
                            y[jj >> 1] = (y[jj >> 1] & ~(0xFFu << sh)) | ((uint32_t)pt[jj] << sh);
                        }
                    }
                }
            };
            // Whole tile in the stage slot: no bounds to check.
            auto whole_tile = [&](auto CONTIG) {
                const RunOffset<PAGED> tile_off(p.pm, base, 13, 2, p.status);  // 8,192-element tile
                const uint8_t* ssm = S.sm[slot] + qt;
                const uint8_t* snb = S.nib[slot] + qt / 2;
                const uint32_t* scw = reinterpret_cast<const uint32_t*>(S.nib[slot]);
                uint8_t* o = p.out + 2 * (base + qt);
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    uint32_t y[4], codes;
                    if (TOP8) {
                        // 24 code bits at byte 3g of the tile's codes (g = the
                        // group's index in the tile); two aligned words hold them.
                        const uint32_t at = 3 * (qt / 8 + 32 * k);
                        codes = __funnelshift_r(scw[at >> 2], scw[(at >> 2) + 1], 8 * (at & 3)) & 0xFFFFFFu;
                    } else {
                        codes = *reinterpret_cast<const uint32_t*>(snb + k * 128);
                    }
                    decode_group(CONTIG, k, *reinterpret_cast<const uint2*>(ssm + k * 256), codes, y);
                    // A group of 8 never straddles a page; a tile in one page
                    // takes one lookup.
                    uint8_t* dst = PAGED ? p.out + tile_off.at(p.pm, base, qt + k * 256u, 2, p.status) : o + k * 512;
                    st_v4(dst, make_uint4(y[0], y[1], y[2], y[3]));
                }
            };
            if (full_tile(t)) {
                if (ADDS && contig)
                    whole_tile(std::true_type{});
                else
                    whole_tile(std::false_type{});
            } else {
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const uint64_t i0 = base + qt + k * 256u;
                    const uint32_t cnt = i0 >= n ? 0u : (n - i0 >= 8 ? 8u : (uint32_t)(n - i0));
                    uint2 smv;
                    uint32_t nibv;
                    if (p.vec && cnt == 8 && !TOP8) {
                        smv = ld_stream_v2(p.in + i0);
                        nibv = ld_stream_u32(p.in + p.L.nib_off + i0 / 2);
                    } else {
                        uint64_t sv = 0;
                        uint32_t nb = 0;
                        for (uint32_t jj = 0; jj < cnt; jj++) sv |= (uint64_t)p.in[i0 + jj] << (8 * jj);
                        if (TOP8) {  // a started group has all 3 of its code bytes
                            if (cnt)
                                for (uint32_t b = 0; b < 3; b++) nb |= (uint32_t)p.in[p.L.nib_off + 3 * (i0 / 8) + b] << (8 * b);
                        } else {
                            for (uint32_t b = 0; b < (cnt + 1) / 2; b++)
                                nb |= (uint32_t)p.in[p.L.nib_off + i0 / 2 + b] << (8 * b);
                        }
                        smv = make_uint2((uint32_t)sv, (uint32_t)(sv >> 32));
                        nibv = nb;
                    }
                    uint32_t y[4];
                    decode_group(std::false_type{}, k, smv, nibv, y);
                    uint8_t* dst = p.out + (cnt ? elem_offset<PAGED>(p.pm, i0, 2, p.status) : 2 * i0);
                    if (p.vec && cnt == 8) {
                        st_v4(dst, make_uint4(y[0], y[1], y[2], y[3]));
                    } else {
#pragma unroll
                        for (uint32_t jj = 0; jj < 8; jj++) {
                            if (jj < cnt) {
                                const uint32_t v = y[jj >> 1] >> (16 * (jj & 1));
                                dst[2 * jj] = (uint8_t)v;
                                dst[2 * jj + 1] = (uint8_t)(v >> 8);
                            }
                        }
                    }
                }
            }
        }

        // Tile t + 1: its first gathering step, into the other buffer.
        uint32_t mine = 0;
        if (t + 1 < t_end) {
            begin_tile(t + 1);
            cover(false);
            mine = gather(t + 1, buf ^ 1u, 0xFFFFFFFFu);
        }
        if (prefetch) store_header((t + 2) / kTilesPerChunk, next_o, next_m, true, chunk_end);
        if (failed_wait) S.abort = 1;
        // Closing barrier: stage slot and buffer buf free, buffer buf ^ 1 and
        // the next header published, the step counted.
        const uint32_t k = count_step(mine);
        if (S.abort) {
            aborted = true;
            break;
        }
        if (t + 1 < t_end) end_tile(t + 1, buf ^ 1u, k);
        if (tid == 0 && t + kDecStages < t_end) issue(slot, t + kDecStages), issued++;
    }
    if (tid == 0 && aborted) {
        for (uint32_t k = waited; k < issued; k++)
            mbar_wait(&S.full[k % kDecStages], (k / kDecStages) & 1u, p.wait_limit_ns);
        if (p.status) atomicMax(p.status, kStatusTimeout);
    }
    W.drain();
    __syncthreads();
    if (tid == 0 && S.bad && p.status) atomicMax(p.status, kStatusCorrupt);
}

cudaError_t launch_encode_bf16(const EncodeParams& p, cudaStream_t s) {
    const size_t smem = sizeof(EncodeSmem);
    const bool paged = p.pm.ids != nullptr;  // host codebooks only
    const void* kern = p.cb_dev   ? (const void*)encode_bf16_kernel<2>
                       : p.contig ? (paged ? (const void*)encode_bf16_kernel<1, true> : (const void*)encode_bf16_kernel<1>)
                                  : (paged ? (const void*)encode_bf16_kernel<0, true> : (const void*)encode_bf16_kernel<0>);
    int sms = 0, per_sm = 0;
    cudaError_t err = kernel_fit(kern, kComputeThreads, smem, &sms, &per_sm);
    if (err != cudaSuccess) return err;
    EncodeParams q = p;
    q.grid = (uint32_t)std::min<uint64_t>(p.num_tiles, (uint64_t)std::max(per_sm, 1) * sms);
    void* args[] = {&q};
    err = cudaLaunchKernel(kern, q.grid, kComputeThreads, args, smem, s);
    if (err != cudaSuccess) return err;
    return launch_finish(q, true, s);
}

cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t s, bool top8, bool adds) {
    const size_t smem = sizeof(DecodeSmem);
    auto kern = top8      ? decode_bf16_kernel<false, true>
                : p.pm.ids ? decode_bf16_kernel<true>
                : adds     ? decode_bf16_kernel<false, false, true>
                           : decode_bf16_kernel<false>;
    int sms = 0, per_sm = 0;
    cudaError_t err = kernel_fit((const void*)kern, kDecThreads, smem, &sms, &per_sm);
    if (err != cudaSuccess) return err;
    const uint32_t grid = (uint32_t)std::min<uint64_t>(p.num_tiles, (uint64_t)std::max(per_sm, 1) * sms);
    // A programmatic dependent of whatever kernel precedes it (the stream's
    // producer): only the launch overlaps, the kernel waits first thing.
    return launch_dependent(kern, dim3(grid), dim3(kDecThreads), smem, s, p);
}

}  // namespace sz
