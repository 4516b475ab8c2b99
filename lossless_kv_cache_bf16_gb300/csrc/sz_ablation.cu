// sz_ablation.cu -- the two alternative designs of the codebook ablation as
// working BF16 codecs, so that their decoding can be measured against the
// Top-16 format (SplitZip technical summary, gist.science/es, "Resultados" >
// "Estudios de Ablacion": Top-8 loses coverage and decodes slower; storing
// escape positions beats a Top-15 sentinel on decode speed; "Metodologia:
// SplitZip" > "Decision de Diseno").  Layouts (the pages give none):
//   Top-8     [sm N][codes 3 ceil(N/8)][cb 8][hdr 8C][records 3E]: code j of
//             group g at bits 3j..3j+2 of the 24-bit little-endian word at
//             byte 3g; an escape gets code 0 and a (u16 position, u8
//             exponent) record, exactly as in the Top-16 format.
//   Sentinel  [sm N][nibbles ceil(N/2)][cb 15][hdr 8C][exponent bytes E]:
//             code 15 marks an escape, whose exponent is the next byte of its
//             chunk's run; headers {offset, count} per 65,536-element chunk.
//
// The encoders here are plain (one block per chunk: count, scan, write);
// only decode speed is compared.  Top-8 decodes with the Top-16 decoder's
// TOP8 variant (sz_bf16.cu).  The sentinel decoder below has the same
// persistent TMA structure as the Top-16 decoder, but must rank every
// sentinel of a tile in element order (a block scan per tile) before it can
// fetch the escape bytes, and chunks cannot be split between blocks.
#include <algorithm>

#include "sz_device.cuh"
#include "sz_params.h"
#include "sz_pipeline.cuh"

namespace sz {

namespace {

constexpr uint32_t kAblThreads = 256;
constexpr uint32_t kAblStep = 8 * kAblThreads;  // elements per write step: a group of 8 per thread

// Exponent of the BF16 element in the two bytes at e.
__device__ __forceinline__ uint32_t bf16_exponent(const uint8_t* e) {
    return (((uint32_t)e[0] | ((uint32_t)e[1] << 8)) >> 7) & 0xFFu;
}

// s_code[e] = code of exponent e, or 0xFF for an escape.
__device__ __forceinline__ void build_codes(const AblationParams& p, uint8_t* s_code) {
    const uint32_t tid = threadIdx.x;
    uint32_t code = 0xFFu;
    for (uint32_t k = 0; k < p.k; k++)
        if (p.cb[k] == tid) code = k;
    s_code[tid] = (uint8_t)code;
}

// Block-wide exclusive prefix of v in thread order; *total gets the sum.
__device__ __forceinline__ uint32_t block_exclusive(uint32_t v, uint32_t* s_warp, uint32_t* total) {
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= (uint32_t)d) incl += a;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    uint32_t before = 0, sum = 0;
    for (uint32_t w = 0; w < kAblThreads / 32; w++) {
        before += w < warp ? s_warp[w] : 0u;
        sum += s_warp[w];
    }
    __syncthreads();  // s_warp is reused by the next call
    *total = sum;
    return before + incl - v;
}

}  // namespace

// Escapes per chunk (one block per chunk).
__global__ void __launch_bounds__(kAblThreads) abl_count_kernel(const AblationParams p) {
    __shared__ uint8_t s_code[256];
    __shared__ uint32_t s_warp[kAblThreads / 32];
    build_codes(p, s_code);
    __syncthreads();
    const uint64_t lo = (uint64_t)blockIdx.x * kChunk;
    const uint64_t hi = min(lo + kChunk, p.n);
    uint32_t cnt = 0;
    for (uint64_t i = lo + threadIdx.x; i < hi; i += kAblThreads) cnt += s_code[bf16_exponent(p.in + 2 * i)] == 0xFFu;
    uint32_t total;
    block_exclusive(cnt, s_warp, &total);
    if (threadIdx.x == 0) p.counts[blockIdx.x] = total;
}

// One block: chunk offsets (exclusive scan of the counts), the headers, the
// codebook and the stream size.
__global__ void __launch_bounds__(kAblThreads) abl_scan_kernel(const AblationParams p) {
    __shared__ uint32_t s_warp[kAblThreads / 32];
    const uint32_t tid = threadIdx.x, C = p.chunks;
    const uint32_t per = (C + kAblThreads - 1) / kAblThreads;  // consecutive chunks per thread
    const uint32_t c0 = min(C, tid * per), c1 = min(C, c0 + per);
    uint32_t mine = 0;
    for (uint32_t c = c0; c < c1; c++) mine += p.counts[c];
    uint32_t total;
    uint32_t run = block_exclusive(mine, s_warp, &total);
    for (uint32_t c = c0; c < c1; c++) {
        const uint32_t cnt = p.counts[c];
        p.offsets[c] = run;
        store_u32_le(p.out + p.hdr_off + 8ull * c, run);
        store_u32_le(p.out + p.hdr_off + 8ull * c + 4, cnt);
        run += cnt;
    }
    if (tid < p.k) p.out[p.cb_off + tid] = p.cb[tid];
    if (tid == 0) *p.out_bytes = p.rec_off + (unsigned long long)(p.top8 ? 3u : 1u) * total;
}

// Dense bytes and escapes of one chunk, 2,048 elements per step: thread t
// owns group t of the step, so thread order is element order.
__global__ void __launch_bounds__(kAblThreads) abl_write_kernel(const AblationParams p) {
    __shared__ uint8_t s_code[256];
    __shared__ uint32_t s_warp[kAblThreads / 32];
    build_codes(p, s_code);
    __syncthreads();
    const uint64_t lo = (uint64_t)blockIdx.x * kChunk;
    const uint64_t hi = min(lo + kChunk, p.n);
    uint32_t run = p.offsets[blockIdx.x];  // escapes before this step
    for (uint64_t s0 = lo; s0 < hi; s0 += kAblStep) {
        const uint64_t i0 = s0 + 8ull * threadIdx.x;
        const uint32_t cnt = i0 >= hi ? 0u : (hi - i0 >= 8 ? 8u : (uint32_t)(hi - i0));
        uint32_t codes = 0, esc = 0;
        for (uint32_t j = 0; j < cnt; j++) {
            const uint8_t* e = p.in + 2 * (i0 + j);
            const uint32_t v = (uint32_t)e[0] | ((uint32_t)e[1] << 8);
            p.out[i0 + j] = (uint8_t)(((v >> 8) & 0x80u) | (v & 0x7Fu));  // sign | mantissa
            uint32_t c = s_code[(v >> 7) & 0xFFu];
            if (c == 0xFFu) {
                esc |= 1u << j;
                c = p.top8 ? 0u : 15u;
            }
            codes |= c << (p.top8 ? 3 * j : 4 * j);
        }
        if (cnt) {
            if (p.top8) {
                for (uint32_t b = 0; b < 3; b++) p.out[p.n + 3 * (i0 / 8) + b] = (uint8_t)(codes >> (8 * b));
            } else {
                for (uint32_t b = 0; b < (cnt + 1) / 2; b++) p.out[p.n + i0 / 2 + b] = (uint8_t)(codes >> (8 * b));
            }
        }
        uint32_t total;
        uint32_t at = run + block_exclusive(__popc(esc), s_warp, &total);
        while (esc) {
            const uint32_t j = __ffs(esc) - 1;
            esc &= esc - 1;
            const uint32_t ex = bf16_exponent(p.in + 2 * (i0 + j));
            if (p.top8) {
                const uint32_t pos = (uint32_t)(i0 + j - lo);
                p.out[p.rec_off + 3ull * at] = (uint8_t)pos;
                p.out[p.rec_off + 3ull * at + 1] = (uint8_t)(pos >> 8);
                p.out[p.rec_off + 3ull * at + 2] = (uint8_t)ex;
            } else {
                p.out[p.rec_off + at] = (uint8_t)ex;
            }
            at++;
        }
        run += total;
    }
}

// ---------------------------------------------------------------------------
// Sentinel decode.  Block b owns chunks [bC/G, (b+1)C/G) (a chunk cannot be
// split: a sentinel's exponent is found by counting every sentinel before it
// in its chunk), i.e. the tiles [8 c_begin, 8 c_end), which stream through a
// 2-stage TMA ring as in the Top-16 decoder.  Per tile: the dense pass into
// registers (nibble byte -> two exponents by table; code 15 decodes to a
// placeholder), the tile's sentinels ranked in element order (per warp in
// (group, lane, element) order, then across warps at one block barrier), the
// sentinels' exponent bytes fetched from the escape run and patched in, one
// 16-byte store per group.  Checks: 15 distinct codebook entries, headers as
// running sums ending at E, each chunk's sentinels equal to its count, every
// escape index inside its chunk's run.
// ---------------------------------------------------------------------------
namespace {

constexpr uint32_t kSenStages = 2;
constexpr uint32_t kSenWarps = kAblThreads / 32;
constexpr uint32_t kSenTilesPerChunk = kChunk / kBf16Tile;  // 8

struct SentinelSmem {
    alignas(128) uint8_t sm[kSenStages][kBf16Tile];
    alignas(128) uint8_t nib[kSenStages][kBf16Tile / 2];
    uint64_t full[kSenStages];
    uint32_t lut[256];
    uint32_t warp_cnt[2][kSenWarps];
    int bad;
    int abort;
};

// Sentinel ranks inside one warp's 1,024 elements in (k, lane, j) order:
// off[k] = sentinels of this warp before lane's group k; returns the total.
__device__ __forceinline__ uint32_t warp_sentinel_ranks(const uint32_t (&c)[4], uint32_t lane, uint32_t (&off)[4]) {
    const uint32_t c01 = c[0] | (c[1] << 16), c23 = c[2] | (c[3] << 16);
    uint32_t s01 = c01, s23 = c23;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, s01, d);
        const uint32_t b = __shfl_up_sync(0xFFFFFFFFu, s23, d);
        if (lane >= (uint32_t)d) s01 += a, s23 += b;
    }
    const uint32_t t01 = __shfl_sync(0xFFFFFFFFu, s01, 31), t23 = __shfl_sync(0xFFFFFFFFu, s23, 31);
    const uint32_t x01 = s01 - c01, x23 = s23 - c23;
    const uint32_t tot0 = t01 & 0xFFFFu, tot1 = t01 >> 16, tot2 = t23 & 0xFFFFu, tot3 = t23 >> 16;
    off[0] = x01 & 0xFFFFu;
    off[1] = tot0 + (x01 >> 16);
    off[2] = tot0 + tot1 + (x23 & 0xFFFFu);
    off[3] = tot0 + tot1 + tot2 + (x23 >> 16);
    return tot0 + tot1 + tot2 + tot3;
}

}  // namespace

__global__ void __launch_bounds__(kAblThreads, 4) decode_sentinel_kernel(const DecodeParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    SentinelSmem& S = *reinterpret_cast<SentinelSmem*>(smem_raw);
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint64_t n = p.L.n;
    const uint32_t C = p.L.num_chunks, G = gridDim.x, T = p.num_tiles;
    const uint32_t c_begin = (uint32_t)((uint64_t)blockIdx.x * C / G);
    const uint32_t c_end = (uint32_t)((uint64_t)(blockIdx.x + 1) * C / G);
    const uint32_t t_begin = c_begin * kSenTilesPerChunk, t_end = min(c_end * kSenTilesPerChunk, T);
    const uint8_t* cb = p.in + p.L.cb_off;
    const uint8_t* esc = p.in + p.L.rec_off;
    const bool tma = p.vec && (reinterpret_cast<uintptr_t>(p.in) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(p.in + p.L.nib_off) % 16 == 0);

    if (tid == 0) {
        for (uint32_t s = 0; s < kSenStages; s++) mbar_init(&S.full[s], 1);
        S.bad = 0;
        S.abort = 0;
        fence_mbar_init();
    }
    {
        // Code 15 is the sentinel: its table entry is a placeholder, patched later.
        const uint32_t lo = tid & 15u, hi = tid >> 4;
        S.lut[tid] = (lo < 15 ? (uint32_t)cb[lo] << 7 : 0u) | (hi < 15 ? (uint32_t)cb[hi] << 23 : 0u);
    }
    if (tid < 15) {
        bool dup = false;
        for (uint32_t k = 0; k < 15; k++) dup |= k != tid && cb[k] == cb[tid];
        if (dup) S.bad = 1;
    }
    __syncthreads();

    auto full_tile = [&](uint32_t t) { return tma && (uint64_t)(t + 1) * kBf16Tile <= n; };
    auto issue = [&](uint32_t slot, uint32_t t) {  // thread 0 only
        if (full_tile(t)) {
            mbar_arrive_expect_tx(&S.full[slot], kBf16Tile + kBf16Tile / 2);
            bulk_g2s(S.sm[slot], p.in + (uint64_t)t * kBf16Tile, kBf16Tile, &S.full[slot]);
            bulk_g2s(S.nib[slot], p.in + p.L.nib_off + (uint64_t)t * (kBf16Tile / 2), kBf16Tile / 2, &S.full[slot]);
        } else {
            mbar_arrive(&S.full[slot]);
        }
    };
    uint32_t issued = 0, waited = 0;
    if (tid == 0)
        for (uint32_t t = t_begin; t < t_end && t < t_begin + kSenStages; t++, issued++) issue(t - t_begin, t);

    uint32_t o = 0, m = 0, seen = 0;  // the current chunk's run and sentinels so far
    uint64_t prev_end = 0;            // o + m of the chunk before
    bool aborted = false;
    uint32_t i = 0;
    for (uint32_t t = t_begin; t < t_end; t++, i++) {
        const uint32_t slot = i % kSenStages, buf = i & 1u;
        const uint64_t base = (uint64_t)t * kBf16Tile;
        const uint32_t chunk = t / kSenTilesPerChunk;
        if (t % kSenTilesPerChunk == 0) {  // a new chunk: its header (every thread reads it)
            const uint8_t* h = p.in + p.L.hdr_off + 8ull * chunk;
            if (t == t_begin && chunk > 0) prev_end = (uint64_t)load_u32_le(h - 8) + load_u32_le(h - 4);
            o = load_u32_le(h);
            m = load_u32_le(h + 4);
            const uint64_t rest = n - (uint64_t)chunk * kChunk;
            const uint64_t len = rest < kChunk ? rest : kChunk;
            bool bad = m > len || (uint64_t)o + m > p.n_esc || (uint64_t)o != (chunk == 0 ? 0ull : prev_end);
            if (chunk == C - 1) bad |= (uint64_t)o + m != p.n_esc;
            if (bad) {
                if (tid == 0) S.bad = 1;
                m = 0;
            }
            prev_end = (uint64_t)o + m;
            seen = 0;
        }

        const bool failed_wait = !mbar_wait(&S.full[slot], (i / kSenStages) & 1u, p.wait_limit_ns);
        uint32_t y[4][4], sent[4], cnt[4], n_in[4];
        const uint32_t qt = warp * 1024u + lane * 8u;
        if (!failed_wait) waited = i + 1;
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const uint64_t i0 = base + qt + k * 256u;
            n_in[k] = i0 >= n ? 0u : (n - i0 >= 8 ? 8u : (uint32_t)(n - i0));
            uint2 smv = make_uint2(0, 0);
            uint32_t nibv = 0;
            if (!failed_wait) {
                if (full_tile(t)) {
                    smv = *reinterpret_cast<const uint2*>(S.sm[slot] + qt + k * 256);
                    nibv = *reinterpret_cast<const uint32_t*>(S.nib[slot] + qt / 2 + k * 128);
                } else {
                    uint64_t sv = 0;
                    for (uint32_t jj = 0; jj < n_in[k]; jj++) sv |= (uint64_t)p.in[i0 + jj] << (8 * jj);
                    for (uint32_t b = 0; b < (n_in[k] + 1) / 2; b++)
                        nibv |= (uint32_t)p.in[p.L.nib_off + i0 / 2 + b] << (8 * b);
                    smv = make_uint2((uint32_t)sv, (uint32_t)(sv >> 32));
                }
            }
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const uint32_t smw = q < 2 ? smv.x : smv.y;
                const uint32_t tt = __byte_perm(smw, 0, (q & 1) ? 0x3322 : 0x1100);
                y[k][q] = (tt & 0x807F807Fu) | S.lut[(nibv >> (8 * q)) & 0xFFu];
            }
            // Nibble j == 15: bit 4j of the AND of the word's four shifts.
            const uint32_t f = nibv & (nibv >> 1) & (nibv >> 2) & (nibv >> 3) & 0x11111111u;
            uint32_t s8 = 0;
#pragma unroll
            for (int jj = 0; jj < 8; jj++) s8 |= ((f >> (4 * jj)) & 1u) << jj;
            sent[k] = s8 & ((1u << n_in[k]) - 1u);
            cnt[k] = __popc(sent[k]);
        }
        uint32_t off[4];
        const uint32_t wtotal = warp_sentinel_ranks(cnt, lane, off);
        if (lane == 0) S.warp_cnt[buf][warp] = wtotal;
        if (failed_wait) S.abort = 1;
        __syncthreads();  // warp totals published; the ring slot consumed
        if (S.abort) {
            aborted = true;
            break;
        }
        if (tid == 0 && t + kSenStages < t_end) issue(slot, t + kSenStages), issued++;
        uint32_t wpre = 0, total = 0;
#pragma unroll
        for (uint32_t w = 0; w < kSenWarps; w++) {
            const uint32_t c = S.warp_cnt[buf][w];
            wpre += w < warp ? c : 0u;
            total += c;
        }
#pragma unroll
        for (int k = 0; k < 4; k++) {
            if (sent[k]) {
                const uint32_t first = o + seen + wpre + off[k];  // index of the group's first sentinel
#pragma unroll
                for (uint32_t jj = 0; jj < 8; jj++) {
                    if ((sent[k] >> jj) & 1u) {
                        const uint32_t idx = first + __popc(sent[k] & ((1u << jj) - 1u));
                        uint32_t e = 0;
                        if (idx < o + m && idx < p.n_esc)
                            e = esc[idx];
                        else
                            S.bad = 1;  // more sentinels than the chunk's run holds
                        const uint32_t sh = 7 + 16 * (jj & 1);
                        y[k][jj >> 1] = (y[k][jj >> 1] & ~(0xFFu << sh)) | (e << sh);
                    }
                }
            }
            const uint64_t i0 = base + qt + k * 256u;
            if (p.vec && n_in[k] == 8) {
                st_stream_v4(p.out + 2 * i0, make_uint4(y[k][0], y[k][1], y[k][2], y[k][3]));
            } else {
#pragma unroll
                for (uint32_t jj = 0; jj < 8; jj++) {
                    if (jj < n_in[k]) {
                        const uint32_t v = y[k][jj >> 1] >> (16 * (jj & 1));
                        p.out[2 * (i0 + jj)] = (uint8_t)v;
                        p.out[2 * (i0 + jj) + 1] = (uint8_t)(v >> 8);
                    }
                }
            }
        }
        seen += total;
        const bool last_of_chunk = t % kSenTilesPerChunk == kSenTilesPerChunk - 1 || t == T - 1;
        if (last_of_chunk && seen != m && tid == 0) S.bad = 1;
    }
    if (tid == 0 && aborted) {
        for (uint32_t k = waited; k < issued; k++)
            mbar_wait(&S.full[k % kSenStages], (k / kSenStages) & 1u, p.wait_limit_ns);
        if (p.status) atomicMax(p.status, kStatusTimeout);
    }
    __syncthreads();
    if (tid == 0 && S.bad && p.status) atomicMax(p.status, kStatusCorrupt);
}

cudaError_t launch_decode_sentinel(const DecodeParams& p, cudaStream_t s) {
    if (p.L.num_chunks == 0) return cudaSuccess;
    const size_t smem = sizeof(SentinelSmem);
    int sms = 0, per_sm = 0;
    const cudaError_t err = kernel_fit((const void*)decode_sentinel_kernel, kAblThreads, smem, &sms, &per_sm);
    if (err != cudaSuccess) return err;
    const uint32_t grid = (uint32_t)std::min<uint64_t>(p.L.num_chunks, (uint64_t)std::max(per_sm, 1) * sms);
    decode_sentinel_kernel<<<grid, kAblThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_ablation_encode(const AblationParams& p, cudaStream_t s) {
    const uint32_t C = std::max<uint32_t>(p.chunks, 1u);
    if (p.chunks > 0) abl_count_kernel<<<C, kAblThreads, 0, s>>>(p);
    abl_scan_kernel<<<1, kAblThreads, 0, s>>>(p);
    if (p.chunks > 0) abl_write_kernel<<<C, kAblThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sz
