// sz_concat.cu -- joining shard streams into the stream of the whole tensor.
//
// A stream's escapes are grouped per 65,536-element chunk behind
// {offset, count} headers (SplitZip technical summary, gist.science/es,
// "Metodologia: SplitZip" > "Flujo de Escape": 16-bit positions), so shards
// of whole chunks encode independently.  Joining them needs, per shard, the
// number of elements and escapes before it (host arithmetic on the stream
// sizes); the dense bytes and the records then move with device-to-device
// copies, and concat_headers_kernel writes the codebook once and every
// shard's headers with their offsets shifted.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "splitzip.h"
#include "sz_device.cuh"

namespace {

constexpr uint32_t kConcatShards = 64;  // shards per header launch
constexpr uint32_t kConcatThreads = 256;

struct ConcatShard {
    const uint8_t* in;       // the shard's stream
    uint64_t cb_in;          // byte offset of its codebook
    uint64_t first_chunk;    // chunks before it in the whole tensor
    uint32_t chunks;         // its chunk count
    uint32_t esc_before;     // escapes before it in the whole tensor
};

struct ConcatParams {
    const uint8_t* cb0;      // the first shard's codebook
    uint8_t* out;
    uint64_t cb_out;         // byte offsets in the joined stream
    uint64_t hdr_out;
    int* status;             // nullable
    uint32_t count;          // shards in this launch
    ConcatShard s[kConcatShards];
};

__device__ __forceinline__ uint32_t load_u32_bytes(const uint8_t* p) {
    return (uint32_t)p[0] | (uint32_t)p[1] << 8 | (uint32_t)p[2] << 16 | (uint32_t)p[3] << 24;
}
__device__ __forceinline__ void store_u32_bytes(uint8_t* p, uint32_t v) {
    p[0] = (uint8_t)v;
    p[1] = (uint8_t)(v >> 8);
    p[2] = (uint8_t)(v >> 16);
    p[3] = (uint8_t)(v >> 24);
}

// blockIdx.y = shard of this launch.  Headers sit at any byte offset (their
// place depends on n), so they move as bytes; there are N / 65,536 of them.
__global__ void __launch_bounds__(kConcatThreads) concat_headers_kernel(const ConcatParams p) {
    const ConcatShard& s = p.s[blockIdx.y];
    const uint32_t t = threadIdx.x;
    if (blockIdx.x == 0 && t < sz::kCodes) {
        const uint8_t want = p.cb0[t];
        if (s.in[s.cb_in + t] != want && p.status) atomicMax(p.status, sz::kStatusInvalid);
        if (blockIdx.y == 0) p.out[p.cb_out + t] = want;
    }
    const uint8_t* hdr_in = s.in + s.cb_in + sz::kCodes;
    uint8_t* hdr_out = p.out + p.hdr_out + 8 * s.first_chunk;
    for (uint32_t c = blockIdx.x * kConcatThreads + t; c < s.chunks; c += gridDim.x * kConcatThreads) {
        // offsets stay below 2^32: the joined tensor has fewer than 2^32 elements
        store_u32_bytes(hdr_out + 8ull * c, load_u32_bytes(hdr_in + 8ull * c) + s.esc_before);
        store_u32_bytes(hdr_out + 8ull * c + 4, load_u32_bytes(hdr_in + 8ull * c + 4));
    }
}

uint64_t cdiv(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
uint64_t dense_of(sz_dtype dt, uint64_t n) { return dt == SZ_BF16 ? n + cdiv(n, 2) : 7 * cdiv(n, 8); }

sz_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SZ_OK : SZ_ERR_CUDA; }

}  // namespace

extern "C" sz_status sz_concat(sz_dtype dt, size_t count, const void* const* h_streams, const size_t* h_bytes,
                               const size_t* h_n, void* d_out, size_t out_capacity, size_t* h_out_bytes,
                               int* d_status, cudaStream_t stream) {
    if ((dt != SZ_BF16 && dt != SZ_FP8_E5M2) || count == 0 || !h_streams || !h_bytes || !h_n || !d_out)
        return SZ_ERR_INVALID_ARG;
    if (d_status && reinterpret_cast<uintptr_t>(d_status) % 4 != 0) return SZ_ERR_INVALID_ARG;
    // Shard sizes -> escape counts; totals.  Only the last non-empty shard
    // may end inside a chunk.
    std::vector<uint64_t> esc(count);
    uint64_t n_all = 0, e_all = 0;
    bool partial = false;
    for (size_t k = 0; k < count; k++) {
        if (!h_streams[k]) return SZ_ERR_INVALID_ARG;
        if (partial && h_n[k] > 0) return SZ_ERR_INVALID_ARG;
        partial = partial || h_n[k] % SZ_CHUNK_ELEMS != 0;
        if ((uint64_t)h_n[k] >= (1ull << 32)) return SZ_ERR_INVALID_ARG;
        const uint64_t fixed = sz_encoded_size(dt, h_n[k], 0);
        if (h_bytes[k] < fixed || (h_bytes[k] - fixed) % 3 != 0) return SZ_ERR_CORRUPT;
        esc[k] = (h_bytes[k] - fixed) / 3;
        if (esc[k] > h_n[k]) return SZ_ERR_CORRUPT;
        n_all += h_n[k];
        e_all += esc[k];
    }
    if (n_all >= (1ull << 32)) return SZ_ERR_INVALID_ARG;
    const uint64_t total = sz_encoded_size(dt, n_all, e_all);
    if (out_capacity < total) return SZ_ERR_CAPACITY;
    if (h_out_bytes) *h_out_bytes = total;

    uint8_t* out = static_cast<uint8_t*>(d_out);
    const uint64_t dense_all = dense_of(dt, n_all);
    const uint64_t hdr_out = dense_all + SZ_CODEBOOK_SIZE;
    const uint64_t rec_out = hdr_out + 8 * cdiv(n_all, SZ_CHUNK_ELEMS);
    cudaError_t err = d_status ? cudaMemsetAsync(d_status, 0, sizeof(int), stream) : cudaSuccess;
    // Dense bytes and records: one copy per part.  Earlier shards hold whole
    // chunks, so every part of shard k starts on a byte (nibble pairs and
    // 8-element E5M2 groups never straddle two shards).
    uint64_t n_before = 0, e_before = 0;
    for (size_t k = 0; k < count && err == cudaSuccess; k++) {
        const uint8_t* in = static_cast<const uint8_t*>(h_streams[k]);
        const uint64_t n = h_n[k], dense = dense_of(dt, n);
        const uint64_t rec_in = dense + SZ_CODEBOOK_SIZE + 8 * cdiv(n, SZ_CHUNK_ELEMS);
        if (dt == SZ_BF16) {
            if (n) err = cudaMemcpyAsync(out + n_before, in, n, cudaMemcpyDeviceToDevice, stream);
            if (n && err == cudaSuccess)
                err = cudaMemcpyAsync(out + n_all + n_before / 2, in + n, cdiv(n, 2), cudaMemcpyDeviceToDevice, stream);
        } else if (n) {
            err = cudaMemcpyAsync(out + n_before / 8 * 7, in, dense, cudaMemcpyDeviceToDevice, stream);
        }
        if (esc[k] && err == cudaSuccess)
            err = cudaMemcpyAsync(out + rec_out + 3 * e_before, in + rec_in, 3 * esc[k], cudaMemcpyDeviceToDevice,
                                  stream);
        n_before += n;
        e_before += esc[k];
    }
    // Codebook and headers, up to kConcatShards shards per launch.
    ConcatParams p{};
    p.cb0 = static_cast<const uint8_t*>(h_streams[0]) + dense_of(dt, h_n[0]);
    p.out = out;
    p.cb_out = dense_all;
    p.hdr_out = hdr_out;
    p.status = d_status;
    n_before = 0;
    e_before = 0;
    for (size_t k0 = 0; k0 < count && err == cudaSuccess; k0 += kConcatShards) {
        p.count = (uint32_t)std::min<size_t>(kConcatShards, count - k0);
        uint32_t most = 0;
        for (uint32_t j = 0; j < p.count; j++) {
            const size_t k = k0 + j;
            ConcatShard& s = p.s[j];
            s.in = static_cast<const uint8_t*>(h_streams[k]);
            s.cb_in = dense_of(dt, h_n[k]);
            s.first_chunk = n_before / SZ_CHUNK_ELEMS;
            s.chunks = (uint32_t)cdiv(h_n[k], SZ_CHUNK_ELEMS);
            s.esc_before = (uint32_t)e_before;
            most = std::max(most, s.chunks);
            n_before += h_n[k];
            e_before += esc[k];
        }
        const uint32_t gx = (uint32_t)std::min<uint64_t>(std::max<uint64_t>(1, cdiv(most, kConcatThreads)), 64);
        concat_headers_kernel<<<dim3(gx, p.count), kConcatThreads, 0, stream>>>(p);
        err = cudaGetLastError();
    }
    return from_cuda(err);
}
