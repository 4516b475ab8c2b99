// sz_device.cuh -- device-side building blocks shared by the SplitZip kernels:
// streaming loads/stores, the global timer for bounded waits, little-endian
// helpers, the decoders' block search for where a range's escape records
// start, the encoders' codebook loader, and paged-tensor addressing.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "sz_params.h"

namespace sz {

constexpr uint32_t kChunk = 65536;  // elements per escape chunk (u16 positions)
constexpr int kCodes = 16;          // top-16 codebook

// Device status codes (same values as sz_status in splitzip.h).
constexpr int kStatusInvalid = 1;  // a codebook read from device memory is not valid
constexpr int kStatusCapacity = 3;
constexpr int kStatusCorrupt = 4;
constexpr int kStatusTimeout = 5;

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Streaming (read-once) global loads that skip L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Plain (write-back) 16-byte store.  On the decoders' output and on the
// E5M2 encoder's packed bytes it measures 0.7-1.4% faster than evict-first.
__device__ __forceinline__ void st_v4(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// Byte permute with the sign mode of PTX prmt: a selector nibble with bit 3
// set gives the selected byte's top bit replicated over the byte.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Evict-first stores for output that is not read again by this kernel.
__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_stream_v2(void* p, uint2 v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_stream_u32(void* p, uint32_t v) {
    asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Little-endian byte stores for the few unaligned header fields.
__device__ __forceinline__ void store_u32_le(uint8_t* p, uint32_t v) {
    p[0] = (uint8_t)v;
    p[1] = (uint8_t)(v >> 8);
    p[2] = (uint8_t)(v >> 16);
    p[3] = (uint8_t)(v >> 24);
}
__device__ __forceinline__ uint32_t load_u32_le(const uint8_t* p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

}  // namespace sz

namespace sz {

// Position (u16, little-endian) of escape record j; records are 3 bytes.
__device__ __forceinline__ uint32_t rec_pos(const uint8_t* rec, uint32_t j) {
    return (uint32_t)rec[3ull * j] | ((uint32_t)rec[3ull * j + 1] << 8);
}

// Block-wide lower bounds in one chunk's escape positions.
//
// For key a and key b, returns the index of the first record in [o, o + m)
// whose position is >= key, assuming positions ascend (m in 1..65536).  Two
// rounds: 1024 evenly spaced probes bracket each answer to at most
// ceil(65536 / 1024) = 64 records; a second round counts inside the bracket.
// The result depends only on the data, so two blocks asking for the same key
// get the same index even for a corrupt stream; the decoders rely on that to
// give every record to exactly one tile.  Must be called by all THREADS
// threads of the block; s_cnt is 4 words of shared scratch.
template <uint32_t THREADS>
__device__ void block_lower_bounds(const uint8_t* rec, uint32_t o, uint32_t m, uint32_t key_a, uint32_t key_b,
                                   uint32_t* s_cnt, uint32_t* out_a, uint32_t* out_b) {
    constexpr uint32_t kProbes = 1024;
    constexpr uint32_t kPer = kProbes / THREADS;
    static_assert(kProbes % THREADS == 0 && THREADS >= 128, "two 64-record brackets need 128 threads");
    const uint32_t tid = threadIdx.x, lane = tid & 31u;
    auto probe = [&](uint32_t i) { return o + (uint32_t)(((uint64_t)i * m) / kProbes); };
    if (tid < 4) s_cnt[tid] = 0;
    __syncthreads();
    uint32_t ca = 0, cb = 0;
#pragma unroll
    for (uint32_t u = 0; u < kPer; u++) {
        const uint32_t pos = rec_pos(rec, probe(tid * kPer + u));
        ca += pos < key_a;
        cb += pos < key_b;
    }
    ca = __reduce_add_sync(0xFFFFFFFFu, ca);
    cb = __reduce_add_sync(0xFFFFFFFFu, cb);
    if (lane == 0) atomicAdd(&s_cnt[0], ca), atomicAdd(&s_cnt[1], cb);
    __syncthreads();
    uint32_t lo[2], hi[2];
#pragma unroll
    for (int s = 0; s < 2; s++) {
        const uint32_t c = s_cnt[s];
        lo[s] = c == 0 ? o : probe(c - 1) + 1;
        hi[s] = c == kProbes ? o + m : probe(c);
        if (lo[s] > hi[s]) lo[s] = hi[s];  // only for corrupt (unsorted) data
    }
    // Second round: threads [0, T/2) bracket a, [T/2, T) bracket b.
    const uint32_t half = THREADS / 2;
    const uint32_t s = tid / half, t = tid % half;
    uint32_t below = 0;
    for (uint32_t u = t; u < hi[s] - lo[s]; u += half) below += rec_pos(rec, lo[s] + u) < (s == 0 ? key_a : key_b);
    below = __reduce_add_sync(0xFFFFFFFFu, below);
    if (lane == 0 && below) atomicAdd(&s_cnt[2 + s], below);
    __syncthreads();
    *out_a = lo[0] + s_cnt[2];
    *out_b = lo[1] + s_cnt[3];
    __syncthreads();
}

}  // namespace sz

namespace sz {

// The codebook of an encode in registers: the 16 bytes of the parameters, or,
// when cb_dev is set, 16 bytes of device memory (16-byte aligned) that are
// checked here.  Returns whether they are 16 strictly ascending exponents
// below `limit`; contig: cb[k] = cb[0] + k for every k.
__device__ __forceinline__ bool load_codebook(const uint8_t (&param_cb)[16], const uint8_t* cb_dev, uint32_t limit,
                                              uint8_t (&cb)[16], bool& contig) {
    if (cb_dev) {
        const uint4 v = *reinterpret_cast<const uint4*>(cb_dev);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 16; k++) cb[k] = (uint8_t)(w[k >> 2] >> (8 * (k & 3)));
    } else {
#pragma unroll
        for (int k = 0; k < 16; k++) cb[k] = param_cb[k];
    }
    bool ok = true;
    contig = true;
#pragma unroll
    for (int k = 0; k < 16; k++) {
        ok &= cb[k] < limit;
        if (k > 0) ok &= cb[k] > cb[k - 1];
        contig &= (uint32_t)cb[k] == (uint32_t)cb[0] + k;
    }
    return ok;
}

// Byte offset of element e in a paged tensor (see PageMap), elements of
// `esize` bytes.  An id outside the pool maps to page 0 (so that nothing
// outside the pool is touched) and clears ok.
__device__ __forceinline__ uint64_t paged_offset(const PageMap& m, uint64_t e, uint32_t esize, bool& ok) {
    const int32_t id = m.ids[e >> m.lg];
    ok = (uint32_t)id < m.pool_pages;
    const uint64_t page = ok ? (uint64_t)(uint32_t)id : 0ull;
    return ((page << m.lg) + (e & ((1ull << m.lg) - 1ull))) * esize;
}

// Byte offset of element e: linear, or through the page map.  A bad page id
// raises SZ_ERR_INVALID_ARG in *status.
template <bool PAGED>
__device__ __forceinline__ uint64_t elem_offset(const PageMap& m, uint64_t e, uint32_t esize, int* status) {
    if (!PAGED) return e * esize;
    bool ok;
    const uint64_t off = paged_offset(m, e, esize, ok);
    if (!ok && status) atomicMax(status, kStatusInvalid);
    return off;
}

// Byte offset of element first + i (0 <= i < 2^lg_run) of a run that starts
// at `first`, aligned to 2^lg_run elements: when the run lies in one page
// (pages of at least 2^lg_run elements) one page lookup serves the whole run.
template <bool PAGED>
struct RunOffset {
    uint64_t base;
    bool one_page;
    __device__ __forceinline__ RunOffset(const PageMap& m, uint64_t first, uint32_t lg_run, uint32_t esize, int* status) {
        one_page = !PAGED || m.lg >= lg_run;
        base = one_page ? elem_offset<PAGED>(m, first, esize, status) : 0ull;
    }
    __device__ __forceinline__ uint64_t at(const PageMap& m, uint64_t first, uint32_t i, uint32_t esize,
                                           int* status) const {
        return one_page ? base + (uint64_t)i * esize : elem_offset<PAGED>(m, first + i, esize, status);
    }
};

// Integer multiply-adds with a constant multiplier (IMAD, on the FMA pipe).
// A right shift by k of a word whose low k bits are masked off is a high
// multiply by 2^(32-k), and adding disjoint bit fields equals OR-ing them, so
// bit packing can be split between the integer ALU and FMA pipes.
template <uint32_t B>
__device__ __forceinline__ uint32_t mad_lo(uint32_t a, uint32_t c) {  // a * B + c
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "n"(B), "r"(c));
    return d;
}
template <uint32_t B>
__device__ __forceinline__ uint32_t mad_hi(uint32_t a, uint32_t c) {  // (a * B >> 32) + c
    uint32_t d;
    asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "n"(B), "r"(c));
    return d;
}
template <uint32_t B>
__device__ __forceinline__ uint32_t mul_hi(uint32_t a) {  // a * B >> 32
    uint32_t d;
    asm("mul.hi.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "n"(B));
    return d;
}

}  // namespace sz
