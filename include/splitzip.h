/*
 * splitzip.h -- C ABI of the SplitZip lossless KV-cache codec for GB300 (sm_103a).
 *
 * Method: "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
 * Serving" (arXiv 2605.01708v2).  Citations below name the page and section:
 *   [ABS] authors' abstract (fugumt.com page for arXiv 2605.01708v2);
 *   [MET] technical summary (gist.science/es), "Metodologia: SplitZip",
 *         items "Estrategia de Codificacion" / "Estrategia de Decodificacion";
 *   [EXT] same summary, "Contribuciones Clave", item 4 "Extensibilidad";
 *   [CAL] same summary, "Resultados" > "Estudios de Ablacion" > "Calibracion".
 *
 * What the codec does ([ABS], [MET]): each element is split into its sign and
 * mantissa bits, stored raw, and its exponent.  An offline-calibrated top-16
 * codebook maps the exponent to a 4-bit code.  An exponent outside the
 * codebook is an escape: its element gets code 0 in the dense stream and a
 * (position, raw exponent) record in a sparse escape stream.  Decode rebuilds
 * every element from the dense stream, then overwrites the escaped exponents,
 * which restores the input bit for bit.  FP8 E5M2 works the same way with a
 * 3-bit sign|mantissa field ([EXT]).
 *
 * Encoded stream (all multi-byte integers little-endian, no padding):
 *   BF16 : [sm u8 x N][nib u8 x ceil(N/2)][cb u8 x 16][hdr x C][esc x E]
 *   E5M2 : [packed u8 x 7*ceil(N/8)]      [cb u8 x 16][hdr x C][esc x E]
 *   sm   = sign << 7 | 7-bit mantissa (BF16)
 *   nib  = code(2k) | code(2k+1) << 4; the unused high nibble of an odd N is 0
 *   E5M2 = per element a 7-bit field code | (sign << 2 | mantissa) << 4; field j
 *          of each group of 8 sits at bits 7j..7j+6 of a 56-bit little-endian
 *          word written as 7 bytes; a short last group is padded with zeros
 *   cb   = the 16 codebook exponents in ascending order; code k = cb[k]
 *   C    = ceil(N / 65536) chunks; hdr = { u32 offset, u32 count }: offset =
 *          escapes in earlier chunks, count = escapes in this chunk
 *   esc  = 3 bytes per escape, in element order: u16 position inside the
 *          65,536-element chunk, then the raw exponent (u8)
 *   size = N + ceil(N/2) + 3E + 16 + 8C (BF16);  7*ceil(N/8) + 3E + 16 + 8C (E5M2)
 *
 * Conventions for every call:
 *  - Pointers named d_* are device pointers, h_* host pointers.  The caller
 *    owns every buffer; the library allocates no memory and keeps no state
 *    between calls other than a per-device cache of kernel launch shapes
 *    (filled under a lock on first use), so calls on different streams with
 *    different buffers, from any host threads, may run concurrently.  The one
 *    exception is sz_encode_noalloc's static scratch, below.
 *  - Element data needs only its natural alignment (2 bytes for BF16); the
 *    kernels take a vectorised path when the buffers are 16-byte aligned and
 *    N is a multiple of 32, and a byte-exact slower path otherwise.
 *  - Calls are asynchronous on `stream` unless stated otherwise.  Argument
 *    errors that the host can see are returned at once and nothing is
 *    launched.  Errors that depend on device data are written to *d_status
 *    (a device int, nullable) when the kernels finish; no kernel traps.
 *  - N must be below 2^32 (headers hold u32 escape offsets).
 */
#ifndef SPLITZIP_H
#define SPLITZIP_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SZ_CHUNK_ELEMS 65536u /* elements addressed by a u16 escape position */
#define SZ_CODEBOOK_SIZE 16   /* top-16 exponent codebook, 4-bit codes */

typedef enum sz_status {
    SZ_OK = 0,
    SZ_ERR_INVALID_ARG = 1, /* null pointer, bad dtype, N >= 2^32, bad codebook, misaligned element data */
    SZ_ERR_UNSUPPORTED = 2, /* no usable CUDA device for this build (needs sm_103) */
    SZ_ERR_CAPACITY = 3,    /* output or workspace too small */
    SZ_ERR_CORRUPT = 4,     /* encoded stream fails validation */
    SZ_ERR_TIMEOUT = 5,     /* a bounded in-kernel wait for an asynchronous copy gave up (about 1 s) */
    SZ_ERR_CUDA = 6         /* a CUDA runtime call failed */
} sz_status;

typedef enum sz_dtype {
    SZ_BF16 = 0,     /* bfloat16: 1 sign, 8 exponent, 7 mantissa bits [MET] */
    SZ_FP8_E5M2 = 1  /* float8 E5M2: 1 sign, 5 exponent, 2 mantissa bits [EXT] */
} sz_dtype;

/* The top-16 exponent codebook ([ABS], [MET] "Codificacion de Longitud
 * Fija"): exp[k] is the exponent that code k stands for.  Entries must be
 * distinct and below 256 (BF16) or 32 (E5M2).  Encode accepts them in any
 * order and writes them to the stream in ascending order, so code k is the
 * k-th smallest exponent. */
typedef struct sz_codebook {
    uint8_t exp[SZ_CODEBOOK_SIZE];
} sz_codebook;

/* Size in bytes of the stream for n elements with n_escapes escapes (the
 * closed form above; [MET] "Codificacion de Longitud Fija", "Flujo de
 * Escape").  sz_encoded_size(dt, n, n) bounds every stream of n elements.
 * Host only; returns 0 for an unknown dtype. */
size_t sz_encoded_size(sz_dtype dt, size_t n, size_t n_escapes);

/* Bytes of device workspace that sz_encode needs for n elements: for every
 * 32,768-element scan tile its escape count, an error word, the escape
 * counts of its units, and up to 2,048 (BF16) or 1,024 (E5M2) staged escape
 * records of 3 bytes -- about 9.6% of the input bytes for either dtype.  A
 * scan tile with more escapes than it stages has the rest of its records
 * re-derived from the input (same stream, more time).  The
 * workspace is scratch: its contents on entry do not matter (every count is
 * written before it is read), and it must not be shared by encodes that can
 * run at the same time.  Host only; returns 0 for an unknown dtype. */
size_t sz_workspace_size(sz_dtype dt, size_t n);

/* Number of exponent bins: 256 (BF16) or 32 (E5M2); 0 for an unknown dtype. */
size_t sz_histogram_bins(sz_dtype dt);

/* Exponent histogram of a calibration sample ([ABS]: offline calibration;
 * [CAL]).  d_sample: n elements of dtype dt.  d_hist: caller-owned device
 * array of sz_histogram_bins(dt) uint64 counts, overwritten (the call clears
 * it first).  Asynchronous. */
sz_status sz_histogram(sz_dtype dt, const void* d_sample, size_t n,
                       unsigned long long* d_hist, cudaStream_t stream);

/* Top-16 selection on the host ([ABS], [MET]): the 16 exponents with the
 * largest counts; equal counts go to the smaller exponent; when fewer than 16
 * exponents occur, the smallest unseen exponents fill the rest.  Writes them in
 * ascending order.  h_hist holds sz_histogram_bins(dt) counts. */
sz_status sz_codebook_from_histogram(sz_dtype dt, const unsigned long long* h_hist,
                                     sz_codebook* h_cb);

/* Top-16 selection on the device: the same rule as
 * sz_codebook_from_histogram, from sz_histogram_bins(dt) counts in device
 * memory (d_hist, 8-byte aligned) to 16 ascending exponents in device memory
 * (d_cb, 16 bytes, 16-byte aligned).  One block; asynchronous, no host
 * synchronisation.  The pages calibrate offline; this is the device
 * counterpart for per-tensor (online) calibration, whose cost the pages'
 * calibration ablation ([RES] "Calibracion") weighs. */
sz_status sz_codebook_from_histogram_device(sz_dtype dt, const unsigned long long* d_hist,
                                            uint8_t* d_cb, cudaStream_t stream);

/* Online calibration, all on the device: the exponent histogram of a sample
 * of d_x, then sz_codebook_from_histogram_device into d_cb.  The sample is
 * made of 128-byte lines (line k = elements [64k, 64k + 64) for BF16,
 * [128k, 128k + 128) for E5M2, clipped to n).  With S = sample_stride, the
 * lines form runs w = 0, 1, ... of S lines (the last run may be shorter, L
 * lines); run w contributes line wS + floor(lowbias32(w) * L / 2^32), where
 * lowbias32 is C. Wellons' 32-bit integer hash (x ^= x >> 16; x *= 0x7feb352d;
 * x ^= x >> 15; x *= 0x846ca68b; x ^= x >> 16).  S = 1 takes every element.
 * One line in S costs about 1/S of a full read and does not alias with a
 * periodic KV layout.  d_hist as for sz_histogram.
 * Asynchronous, no host synchronisation: an sz_encode_dcb can follow on the
 * same stream (and both can be captured in a CUDA graph). */
sz_status sz_calibrate_device(sz_dtype dt, const void* d_x, size_t n, uint32_t sample_stride,
                              unsigned long long* d_hist, uint8_t* d_cb, cudaStream_t stream);

/* Codebook ablation ([RES] "Estudios de Ablacion": Top-16 vs Top-8, and
 * explicit escape positions vs a Top-15 sentinel).  From the exponent
 * histogram h_hist (sz_histogram_bins(dt) counts) of n elements, the stream
 * sizes in bytes of (h_sizes[0]) this format with its top-16 codebook,
 * (h_sizes[1]) 3-bit Top-8 codes (BF16: sm bytes + 8 codes in 3 bytes; E5M2:
 * 6-bit code|sm3 fields, 4 in 3 bytes) with the same 3-byte escape records,
 * an 8-byte codebook and the same headers, and (h_sizes[2]) Top-15 codes
 * with code 15 as an escape sentinel, each escape storing only its exponent
 * byte, a 15-byte codebook and the same headers.  The pages name these
 * designs but not their layouts; these are the plainest ones that keep the
 * rest of the format.  Host only. */
sz_status sz_ablation_sizes(sz_dtype dt, const unsigned long long* h_hist, size_t n,
                            unsigned long long* h_sizes);

/* Offline calibration = sz_histogram, a device-to-host copy of the counts,
 * and sz_codebook_from_histogram.  Synchronises `stream` (the only call that
 * does).  d_hist is the same caller-owned scratch as for sz_histogram. */
sz_status sz_calibrate(sz_dtype dt, const void* d_sample, size_t n,
                       unsigned long long* d_hist, sz_codebook* h_cb,
                       cudaStream_t stream);

/* Encode ([MET] "Estrategia de Codificacion"; [EXT] for E5M2).
 *  h_cb          codebook (host), read during the call only
 *  d_in          n elements of dtype dt (device)
 *  d_out         stream buffer (device) of out_capacity bytes; must hold at
 *                least sz_encoded_size(dt, n, 0) bytes.  When the escapes do
 *                not fit, *d_status becomes SZ_ERR_CAPACITY and the stream is
 *                incomplete; sz_encoded_size(dt, n, n) always suffices
 *  d_out_bytes   u64 the device can write, receives the stream size (also
 *                on SZ_ERR_CAPACITY, where it is the size that was needed):
 *                device memory, or pinned host memory (mapped into the
 *                device's address space under unified addressing), which a
 *                host thread can read once the stream has passed the call
 *                without a copy
 *  d_status      device int or NULL: SZ_OK, SZ_ERR_CAPACITY or SZ_ERR_TIMEOUT
 *                (sz_encode_dcb also SZ_ERR_INVALID_ARG for a bad codebook).
 *                Written once, by the call's last kernel; what it held before
 *                the call does not matter
 *  d_ws          device workspace of ws_bytes >= sz_workspace_size(dt, n)
 * Asynchronous; the stream is byte-for-byte the layout above. */
sz_status sz_encode(sz_dtype dt, const sz_codebook* h_cb, const void* d_in, size_t n,
                    void* d_out, size_t out_capacity, unsigned long long* d_out_bytes,
                    int* d_status, void* d_ws, size_t ws_bytes, cudaStream_t stream);

/* sz_encode with the codebook in device memory (d_cb: 16 bytes, 16-byte
 * aligned, read on the device when the kernels run), e.g. as written by
 * sz_calibrate_device.  The stream is the one sz_encode gives for the same
 * 16 exponents.  The codebook must be 16 strictly ascending exponents (below
 * 32 for E5M2); otherwise *d_status becomes SZ_ERR_INVALID_ARG and the stream
 * is meaningless.  The pages calibrate offline; this entry point serves
 * per-tensor calibration without a host round trip. */
sz_status sz_encode_dcb(sz_dtype dt, const uint8_t* d_cb, const void* d_in, size_t n,
                        void* d_out, size_t out_capacity, unsigned long long* d_out_bytes,
                        int* d_status, void* d_ws, size_t ws_bytes, cudaStream_t stream);

/* Decode ([MET] "Estrategia de Decodificacion"): dense LUT pass, then the
 * escape overwrite.
 *  d_in, in_bytes  the stream (device); in_bytes must match the closed form
 *                  for n and some escape count, else SZ_ERR_CORRUPT is
 *                  returned at once
 *  n               element count (the decoder knows the tensor's shape)
 *  d_out           n elements of dtype dt (device)
 *  d_status        device int or NULL: SZ_OK or SZ_ERR_CORRUPT (bad codebook,
 *                  headers that are not a running sum, a position outside its
 *                  chunk or out of order, an E5M2 exponent above 31), or
 *                  SZ_ERR_TIMEOUT if an in-kernel copy did not land within
 *                  the bounded wait (about 1 s).  On an error the contents of
 *                  d_out are unspecified, but nothing outside d_out[0, n) is
 *                  written.
 * Asynchronous. */
sz_status sz_decode(sz_dtype dt, const void* d_in, size_t in_bytes, size_t n,
                    void* d_out, int* d_status, cudaStream_t stream);

/* Paged KV tensors.  Serving engines keep a KV cache as a pool of equal
 * pages and each sequence as a block table of page ids; these two calls
 * encode such a tensor straight from its pages and decode straight into
 * them, with no contiguous copy.  The pages describe the codec for a
 * contiguous tensor; this is the gather/scatter step around it.
 *  d_pool        the pool (device, 16-byte aligned): pool_pages pages of
 *                page_elems elements each, page q at d_pool + q * page_elems
 *                * element size
 *  page_elems    a power of two, 16 <= page_elems <= 2^30
 *  d_block_ids   device int32[ceil(n / page_elems)]: element e of the logical
 *                tensor is element e % page_elems of page d_block_ids[e /
 *                page_elems].  The kernels read the first ceil(n /
 *                page_elems) entries without a bound, so the table must hold
 *                at least that many (the library cannot see its length; the
 *                Python binding checks it).  An id outside [0, pool_pages)
 *                is never dereferenced: *d_status becomes SZ_ERR_INVALID_ARG
 *                and the result is meaningless.  Decode writes only the
 *                pages the table names (ids must not repeat for decode).
 * The stream is byte for byte the sz_encode stream of the logical tensor;
 * other arguments and errors as for sz_encode / sz_decode. */
sz_status sz_encode_paged(sz_dtype dt, const sz_codebook* h_cb, const void* d_pool, size_t pool_pages,
                          size_t page_elems, const int32_t* d_block_ids, size_t n,
                          void* d_out, size_t out_capacity, unsigned long long* d_out_bytes,
                          int* d_status, void* d_ws, size_t ws_bytes, cudaStream_t stream);
sz_status sz_decode_paged(sz_dtype dt, const void* d_in, size_t in_bytes, size_t n,
                          void* d_pool, size_t pool_pages, size_t page_elems,
                          const int32_t* d_block_ids, int* d_status, cudaStream_t stream);

/* Concatenation of shard streams into the stream of the whole tensor.  The
 * chunk headers make every 65,536-element chunk addressable on its own
 * ([MET] "Flujo de Escape": positions are 16-bit, so escapes are grouped per
 * chunk), so a tensor cut into shards of whole chunks can be encoded shard by
 * shard (on one GPU each, or as pipeline segments) and joined afterwards:
 * the dense parts and the escape records are copied to their places, the
 * codebook once, and each shard's header offsets are shifted by the escapes
 * of the shards before it (an exclusive scan of the shard escape counts, on
 * the host from the stream sizes).  The result is byte-for-byte the stream
 * sz_encode gives for the whole tensor with the same codebook.
 *  count           number of shards (>= 1), in tensor order
 *  h_streams       host array of count device pointers to the shard streams
 *  h_bytes, h_n    host arrays: each shard's stream size and element count;
 *                  only the last non-empty shard may end inside a chunk
 *                  (h_n[k] % 65536 != 0; empty shards are allowed anywhere),
 *                  and each size must be the closed form for h_n[k] and some
 *                  escape count, else SZ_ERR_INVALID_ARG / SZ_ERR_CORRUPT is
 *                  returned at once
 *  d_out           device buffer of out_capacity bytes, not overlapping any
 *                  shard stream; receives sz_encoded_size(dt, sum n, sum E)
 *                  bytes, the size also written to *h_out_bytes (nullable)
 *  d_status        device int or NULL: SZ_OK, or SZ_ERR_INVALID_ARG when a
 *                  shard's codebook differs from the first shard's
 * Asynchronous (device-to-device copies and one header kernel per 64
 * shards).  The shards' own headers are not checked here; a decode of the
 * result checks them all. */
sz_status sz_concat(sz_dtype dt, size_t count, const void* const* h_streams, const size_t* h_bytes,
                    const size_t* h_n, void* d_out, size_t out_capacity, size_t* h_out_bytes,
                    int* d_status, cudaStream_t stream);

/* The codebook ablation's two alternative designs as working BF16 codecs,
 * for measuring their decode speed against this format ([RES] "Estudios de
 * Ablacion": Top-8 is reported to decode 3x slower, a Top-15 sentinel 3.5x
 * slower; [MET] "Decision de Diseno").  Not part of the SplitZip format; the
 * pages give no layouts, so these are readings:
 *  SZ_ABL_TOP8      [sm N][codes 3 ceil(N/8)][codebook 8][headers 8C]
 *                   [records 3E]: code j of group g at bits 3j..3j+2 of the
 *                   24-bit little-endian word at byte 3g; escapes as in the
 *                   SplitZip stream (code 0 + a position/exponent record).
 *  SZ_ABL_SENTINEL  [sm N][nibbles ceil(N/2)][codebook 15][headers 8C]
 *                   [exponent bytes E]: code 15 marks an escape, whose
 *                   exponent is the next byte of its chunk's run.
 * h_cb: 8 or 15 distinct exponents, code c = h_cb[c].  out_capacity must be
 * at least sz_ablation_encoded_size(variant, n, n); d_ws at least
 * sz_ablation_workspace_size(n) bytes, 4-byte aligned.  Decode reports
 * SZ_ERR_CORRUPT in *d_status for headers that are not running sums, a
 * sentinel count that disagrees with its chunk's header, or (Top-8) record
 * positions out of order; it writes nothing outside d_out[0, 2n).
 * Asynchronous; encode writes the stream size to *d_out_bytes. */
enum sz_ablation { SZ_ABL_TOP8 = 1, SZ_ABL_SENTINEL = 2 };
size_t sz_ablation_encoded_size(int variant, size_t n, size_t n_escapes);
/* The 8 (Top-8) or 15 (sentinel) most frequent exponents of a BF16 histogram
 * (256 counts), chosen as for sz_codebook_from_histogram, ascending.  Host. */
sz_status sz_ablation_codebook(int variant, const unsigned long long* h_hist, uint8_t* h_cb);
size_t sz_ablation_workspace_size(size_t n);
sz_status sz_ablation_encode(int variant, const uint8_t* h_cb, const void* d_in, size_t n,
                             void* d_out, size_t out_capacity, unsigned long long* d_out_bytes,
                             void* d_ws, size_t ws_bytes, cudaStream_t stream);
sz_status sz_ablation_decode(int variant, const void* d_in, size_t in_bytes, size_t n,
                             void* d_out, int* d_status, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* sz_status_string(int status);

/* sz_encode for callers that cannot allocate device memory.  The paper has
 * no counterpart: this entry point exists for integration only.  Some callers
 * cannot call cudaMalloc -- for instance a serving engine that has handed
 * almost all device memory to its KV-cache pool and forbids further
 * allocations, or a latency-critical path that must not take cudaMalloc's
 * implicit device synchronisation -- and so cannot provide the workspace
 * that sz_encode takes.  This call uses a workspace of 6,881,280 bytes
 * (6.56 MiB) held in a static device array inside the library instead, and
 * otherwise behaves exactly like sz_encode (same arguments, stream bytes,
 * d_out_bytes and d_status semantics).  It allocates nothing and calls no
 * allocating routine.
 *  - Limit: n up to 2^28 elements of either dtype; larger n returns
 *    SZ_ERR_CAPACITY at once and launches nothing.  Its smaller staging area
 *    (256 escape records per scan tile, of either dtype) makes scan tiles
 *    with more escapes re-derive the rest of their records from the input;
 *    the output is the same.
 *  - Every GPU that loads the library holds the array until the process
 *    exits.
 *  - The first call on each device looks up the array's device address with
 *    that device current and keeps it; make that first call before any
 *    stream capture.  The address belongs to the device's primary context:
 *    do not use this call after a cudaDeviceReset in the same process.
 *  - Nothing in the array is cleared: each call writes every count it later
 *    reads, so what an earlier call left there does not matter.  The output
 *    of a call that reported an error is undefined.
 *  - All calls on a device share the one array, so calls that can overlap
 *    on the GPU -- on different streams without ordering between them --
 *    race and corrupt each other's output.  Serialise them, e.g. by issuing
 *    them on one stream. */
sz_status sz_encode_noalloc(sz_dtype dt, const sz_codebook* h_cb, const void* d_in, size_t n,
                            void* d_out, size_t out_capacity, unsigned long long* d_out_bytes,
                            int* d_status, cudaStream_t stream);

/* Testing hook, not for production use: sz_encode, except that one wait
 * inside the encode never completes: the first input copy of block 0 is never
 * issued, so that block's wait for it gives up after wait_limit_ns.  Lets a
 * test check that the wait ends with SZ_ERR_TIMEOUT in *d_status instead of
 * hanging.  BF16 only (the E5M2 encoder has no in-kernel wait; E5M2 returns
 * SZ_ERR_UNSUPPORTED).  d_status must not be NULL. */
sz_status sz_debug_encode_stalled(sz_dtype dt, const sz_codebook* h_cb, const void* d_in,
                                  size_t n, void* d_out, size_t out_capacity,
                                  unsigned long long* d_out_bytes, int* d_status,
                                  void* d_ws, size_t ws_bytes,
                                  unsigned long long wait_limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPLITZIP_H */
