// sz_records.cuh -- the decoders' walk over escape records.
//
// Escape records are 3-byte (u16 position in the chunk, u8 exponent) pairs in
// element order (SplitZip technical summary, gist.science/es, "Metodologia:
// SplitZip" > "Flujo de Escape").  A decoder block consumes its records as
// one contiguous run, a step of up to R records per thread at a time.  They
// are read from shared memory: NB buffers of kWinRecs records each, two
// resident (the records a step reads) and the NB - 2 after them already in
// flight as asynchronous copies (cp.async, 16 bytes each, zero-filled past
// the end of the stream; one commit group per window).  When a step no
// longer needs the older resident window, the oldest in-flight one is waited
// for and joins, and the freed buffer starts loading the window after the
// last one in flight; a long run of records then costs one barrier per
// kWinRecs records instead of a full memory round trip, with NB - 2 windows
// of copies under way.  Only a jump outside the resident windows (the first
// step of a block, or a corrupt header) reloads them synchronously.
#pragma once

#include <cstdint>

#include "sz_pipeline.cuh"

namespace sz {

constexpr uint32_t kWinRecs = 1024;                // records per window
constexpr uint32_t kWinBytes = 3 * kWinRecs + 32;  // + the 16-byte alignment offset, rounded up

// Block-uniform state: every thread holds the same values and calls the
// members in the same order (their barriers are block-wide).
template <uint32_t THREADS, uint32_t NB = 3>
struct RecordWindow {
    static_assert(NB >= 3, "two resident windows and at least one in flight");
    uint8_t (*buf)[kWinBytes];  // NB buffers in shared memory, 16-byte aligned
    const uint8_t* rec;         // the stream's first record (global memory)
    uint32_t n_esc;             // records in the stream
    uint32_t lo = 0;            // first record of the older resident window
    uint32_t slot = 0;          // its buffer; the newer one is in slot + 1
    bool valid = false;
    const uint8_t* base0 = nullptr;  // record lo in shared memory
    const uint8_t* base1 = nullptr;  // record lo + kWinRecs

    __device__ __forceinline__ RecordWindow(uint8_t (*b)[kWinBytes], const uint8_t* r, uint32_t n)
        : buf(b), rec(r), n_esc(n) {}

    __device__ __forceinline__ static uint32_t next(uint32_t s) { return s + 1 == NB ? 0u : s + 1; }
    // Where record `first` lands in buffer b: the copies start at the 16-byte
    // boundary below it.
    __device__ __forceinline__ const uint8_t* start(uint64_t first, uint32_t b) const {
        return buf[b] + (reinterpret_cast<uintptr_t>(rec + 3ull * first) & 15u);
    }
    // Issues the copies of records [first, first + kWinRecs) (clipped to the
    // stream) into buffer b; at most 194 pieces, one per thread.
    __device__ __forceinline__ void issue(uint64_t first, uint32_t b) const {
        if (first >= n_esc) return;
        const uint32_t len = n_esc - first < kWinRecs ? (uint32_t)(n_esc - first) : kWinRecs;
        const uintptr_t s = reinterpret_cast<uintptr_t>(rec + 3ull * first), e = s + 3ull * len;
        const uintptr_t as = s & ~(uintptr_t)15;
        const uint32_t pieces = (uint32_t)((e - as + 15) / 16);
        for (uint32_t i = threadIdx.x; i < pieces; i += THREADS) {
            const uintptr_t src = as + 16ull * i;
            cp_async16(buf[b] + 16 * i, reinterpret_cast<const void*>(src), e - src >= 16 ? 16u : (uint32_t)(e - src));
        }
    }
    __device__ __forceinline__ void set_bases() {
        base0 = start(lo, slot);
        base1 = start((uint64_t)lo + kWinRecs, next(slot));
    }
    // Record j (resident): its 3 bytes.
    __device__ __forceinline__ const uint8_t* at(uint32_t j) const {
        const uint32_t d = j - lo;
        return d < kWinRecs ? base0 + 3 * d : base1 + 3 * (d - kWinRecs);
    }
    __device__ __forceinline__ uint32_t pos(uint32_t j) const {
        const uint8_t* r = at(j);
        return (uint32_t)r[0] | ((uint32_t)r[1] << 8);
    }
    // Makes records [need_lo, need_hi) resident (need_hi - need_lo <=
    // kWinRecs + 1; nothing when empty).  Block-wide.  Window bounds are
    // 64-bit: lo + NB kWinRecs may pass 2^32 near the end of 2^32 records.
    __device__ __forceinline__ void cover(uint32_t need_lo, uint32_t need_hi) {
        if (need_hi <= need_lo) return;
        const uint64_t lo64 = lo;
        if (valid && need_lo >= lo64 + kWinRecs && need_hi <= lo64 + 3 * kWinRecs) {
            // The older window is done with: the oldest in-flight one joins
            // (the NB - 3 younger ones may still be landing), and the freed
            // buffer loads the window after the last one in flight.
            cp_async_wait_group<NB - 3>();
            __syncthreads();
            const uint32_t freed = slot;
            lo += kWinRecs;
            slot = next(slot);
            issue((uint64_t)lo + (NB - 1) * (uint64_t)kWinRecs, freed);
            cp_async_commit();
            set_bases();
        }
        if (!valid || need_lo < lo || need_hi > (uint64_t)lo + 2 * kWinRecs) {
            cp_async_wait_all();  // no copy may land in a buffer after this reload
            __syncthreads();
            lo = need_lo;
            slot = 0;
            valid = true;
            issue(lo, 0);
            issue((uint64_t)lo + kWinRecs, 1);
            cp_async_wait_all();
            __syncthreads();
#pragma unroll
            for (uint32_t b = 2; b < NB; b++) {
                issue((uint64_t)lo + b * (uint64_t)kWinRecs, b);
                cp_async_commit();
            }
            set_bases();
        }
    }
    // Before the block exits: no copy may still be writing its shared memory.
    __device__ __forceinline__ void drain() const { cp_async_wait_all(); }
};

// Block-wide barrier that also counts the records a step took, when thread
// t took records cursor + t + THREADS k for k < took (k = 0, 1; a second one
// only after the first).  Records in order make the taken ones a prefix of
// the step, so the count is the number of threads that took one, plus, when
// all of them did, the number that took two (a second barrier, only in
// steps that take more than THREADS records).  For records out of order
// (a corrupt stream, which the checks report) the result still never
// exceeds the records taken.
template <uint32_t THREADS>
__device__ __forceinline__ uint32_t count_taken_sync(uint32_t took) {
    uint32_t k = (uint32_t)__syncthreads_count(took >= 1);
    if (k == THREADS) k += (uint32_t)__syncthreads_count(took >= 2);
    return k;
}

// Block-wide barrier that also counts the records a step took, when thread
// t took records cursor + t + THREADS k for k < took (took <= R, a prefix of
// its own records).  The count is the length of the prefix of the step that
// was taken: the first record not taken is cursor + t + THREADS took for some
// thread t with took < R, and the smallest such index ends the prefix (all R
// THREADS records when every thread took R).  Records in order make every
// taken record part of that prefix; for records out of order (a corrupt
// stream, which the checks report) the walk never passes a record it did
// not take.  slots: 2 x (THREADS / 32) words of shared memory, used
// alternately (parity flips on every call, the same in every thread).
template <uint32_t THREADS, uint32_t R>
__device__ __forceinline__ uint32_t count_prefix_sync(uint32_t took, uint32_t* slots, uint32_t& parity) {
    constexpr uint32_t kW = THREADS / 32;
    const uint32_t first_gap = took < R ? threadIdx.x + THREADS * took : R * THREADS;
    const uint32_t m = __reduce_min_sync(0xFFFFFFFFu, first_gap);
    uint32_t* s = slots + parity * kW;
    if ((threadIdx.x & 31u) == 0) s[threadIdx.x >> 5] = m;
    __syncthreads();
    uint32_t k = s[0];
#pragma unroll
    for (uint32_t v = 1; v < kW; v++) k = min(k, s[v]);
    parity ^= 1u;
    return k;
}

}  // namespace sz
