/*
 * splitzip_oracle.c -- plain, slow, single-threaded CPU oracle of the SplitZip
 * lossless KV-cache format (BF16 and FP8 E5M2).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity reference that the CUDA
 * path is checked against.  Only the test suite, the smoke check and the
 * bench's CPU-baseline and reference legs may load it.  It shares no code,
 * header, table or constant generator with the CUDA library; it includes
 * only the C standard library.
 *
 * Sources (the method is described in prose only; no listing is followed):
 *  [ABS]  SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
 *         Serving -- authors' abstract (arXiv 2605.01708v2, fugumt.com page).
 *  [MET]  same paper, technical summary (gist.science/es), section
 *         "Metodologia: SplitZip", items "Estrategia de Codificacion" and
 *         "Estrategia de Decodificacion".
 *  [EXT]  same summary, "Contribuciones Clave", item 4 "Extensibilidad"
 *         (FP8 E5M2 variant).
 *  [CAL]  same summary, "Resultados" > "Estudios de Ablacion" > "Calibracion"
 *         (one offline codebook).
 *
 * Readings of points the pages leave open:
 *  R1  sign|mantissa byte = sign << 7 | mantissa (BF16); 3-bit field
 *      sign << 2 | mantissa (E5M2).
 *  R2  two 4-bit codes per byte, the even element in the low nibble.
 *  R3  codes are given in ascending exponent order (code k = k-th smallest
 *      codebook exponent).
 *  R4  top-16 ties break toward the smaller exponent; fewer than 16 seen
 *      exponents are padded with the smallest unseen ones.
 *  R5  an escaped element gets code 0 in the dense stream.
 *  R6  escapes are (position, value) pairs stored in element order, 3 bytes
 *      each: position as a little-endian u16 within its 65,536-element chunk,
 *      then the raw exponent as a u8.
 *  R7  one 8-byte header per chunk: u32 offset (escapes in earlier chunks),
 *      u32 count (escapes in this chunk), little-endian.
 *  R8  E5M2: 7-bit field = code | sm3 << 4; element j of a group of 8 sits at
 *      bits 7j..7j+6 of a 56-bit little-endian word written as 7 bytes; a
 *      short last group is padded with zero fields.
 *  R9  stream = [dense][codebook 16 B][headers 8 B x C][escapes 3 B x E];
 *      BF16 dense = [sign|mantissa byte x N][nibble byte x ceil(N/2)];
 *      E5M2 dense = [7 bytes x ceil(N/8)].  No global header, no padding.
 *  R10 zero, subnormal, Inf and NaN need no special case: an exponent field
 *      is just a value.
 *
 * The codebook ablation ([RES] "Estudios de Ablacion": Top-16 vs Top-8, and
 * explicit positions vs a Top-15 sentinel) names the alternative designs but
 * not their layouts; orc_ablation_sizes counts them under the plainest
 * layouts that keep everything else of this format:
 *  A1  Top-8: 3-bit codes; BF16 keeps the sm bytes and packs 8 codes in 3
 *      bytes; E5M2 packs 6-bit code|sm3 fields, 4 in 3 bytes; escapes as R6;
 *      the codebook takes 8 bytes.
 *  A2  Top-15 + sentinel: 4-bit codes with 15 marking an escape; an escape
 *      stores only its exponent byte, in element order; the codebook takes
 *      15 bytes; the chunk headers stay (they give each chunk's first escape).
 *  A3  top-k selection follows R4 with k in place of 16.
 *  A4  as full codecs (orc_abl_*): Top-8 puts element j of group g at bits
 *      3j..3j+2 of the 24-bit little-endian word at byte 3g; the sentinel's
 *      escape exponent is the next byte of its chunk's run; both decoders
 *      check what keeps them in bounds (closed-form size, running-sum
 *      headers, Top-8 record positions as R11, sentinel counts per chunk).
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORC_OK 0
#define ORC_INVALID_ARG 1
#define ORC_CAPACITY 3
#define ORC_CORRUPT 4

#define ORC_BF16 0
#define ORC_E5M2 1

#define ORC_CHUNK 65536u   /* a u16 position addresses 65,536 elements [MET] */
#define ORC_CB 16          /* top-16 codebook, 4-bit codes [MET] */
#define ORC_NO_CODE 0xFFu
#define ORC_ABL_TOP8 1
#define ORC_ABL_SENTINEL 2

static uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

static int exponent_bins(int dt) { return dt == ORC_BF16 ? 256 : 32; }

/* ---- element fields ([MET] field split; [EXT] for E5M2) ---------------- */

/* BF16 element i as a 16-bit pattern (little-endian storage). */
static unsigned bf16_at(const uint8_t *x, uint64_t i) {
    return (unsigned)x[2 * i] | ((unsigned)x[2 * i + 1] << 8);
}

/* Exponent field of element i: bits 14..7 for BF16, bits 6..2 for E5M2. */
static unsigned exponent_at(int dt, const uint8_t *x, uint64_t i) {
    if (dt == ORC_BF16) return (bf16_at(x, i) >> 7) & 0xFFu;
    return ((unsigned)x[i] >> 2) & 0x1Fu;
}

/* ---- sizes (closed form; [MET] + R9) ----------------------------------- */

uint64_t orc_dense_bytes(int dt, uint64_t n) {
    if (dt == ORC_BF16) return n + ceil_div(n, 2);
    return 7 * ceil_div(n, 8);
}

uint64_t orc_num_chunks(uint64_t n) { return ceil_div(n, ORC_CHUNK); }

uint64_t orc_encoded_size(int dt, uint64_t n, uint64_t n_escapes) {
    return orc_dense_bytes(dt, n) + ORC_CB + 8 * orc_num_chunks(n) + 3 * n_escapes;
}

/* ---- calibration ([ABS]: offline top-16; [CAL]) ------------------------ */

/* hist[e] = number of elements whose exponent field equals e. */
void orc_histogram(int dt, const uint8_t *x, uint64_t n, uint64_t *hist) {
    for (int e = 0; e < exponent_bins(dt); e++) hist[e] = 0;
    for (uint64_t i = 0; i < n; i++) hist[exponent_at(dt, x, i)]++;
}

/* Pick the 16 most frequent exponents (R4: ties toward the smaller exponent,
 * unseen exponents fill up from the smallest), then list them ascending (R3). */
/* taken[e] = 1 for the k most frequent exponents (R4 for any k <= bins). */
static void pick_most_frequent(int dt, const uint64_t *hist, int k, int *taken) {
    int bins = exponent_bins(dt);
    for (int e = 0; e < 256; e++) taken[e] = 0;
    for (int r = 0; r < k; r++) {
        int best = -1;
        for (int e = 0; e < bins; e++) {
            if (taken[e]) continue;
            if (best < 0 || hist[e] > hist[best]) best = e;
        }
        taken[best] = 1;
    }
}

int orc_codebook_from_histogram(int dt, const uint64_t *hist, uint8_t *cb) {
    int taken[256];
    int bins = exponent_bins(dt);
    pick_most_frequent(dt, hist, ORC_CB, taken);
    int k = 0;
    for (int e = 0; e < bins; e++)
        if (taken[e]) cb[k++] = (uint8_t)e;
    return ORC_OK;
}

/* A codebook is 16 distinct exponents that the dtype can hold. */
int orc_codebook_valid(int dt, const uint8_t *cb) {
    for (int a = 0; a < ORC_CB; a++) {
        if ((int)cb[a] >= exponent_bins(dt)) return 0;
        for (int b = a + 1; b < ORC_CB; b++)
            if (cb[a] == cb[b]) return 0;
    }
    return 1;
}

/* inv[e] = code of exponent e, or ORC_NO_CODE when e is outside the codebook. */
static void inverse_codebook(const uint8_t *cb, uint8_t *inv) {
    for (int e = 0; e < 256; e++) inv[e] = ORC_NO_CODE;
    for (int k = 0; k < ORC_CB; k++) inv[cb[k]] = (uint8_t)k;
}

/* Number of elements whose exponent is outside the codebook. */
uint64_t orc_count_escapes(int dt, const uint8_t *cb, const uint8_t *x, uint64_t n) {
    uint8_t inv[256];
    uint64_t count = 0;
    inverse_codebook(cb, inv);
    for (uint64_t i = 0; i < n; i++)
        if (inv[exponent_at(dt, x, i)] == ORC_NO_CODE) count++;
    return count;
}

/* ---- little-endian helpers --------------------------------------------- */

static void put_u16(uint8_t *p, unsigned v) {
    p[0] = (uint8_t)(v & 0xFFu);
    p[1] = (uint8_t)((v >> 8) & 0xFFu);
}

static void put_u32(uint8_t *p, uint64_t v) {
    for (int b = 0; b < 4; b++) p[b] = (uint8_t)((v >> (8 * b)) & 0xFFu);
}

static unsigned get_u16(const uint8_t *p) { return (unsigned)p[0] | ((unsigned)p[1] << 8); }

static uint64_t get_u32(const uint8_t *p) {
    uint64_t v = 0;
    for (int b = 0; b < 4; b++) v |= (uint64_t)p[b] << (8 * b);
    return v;
}

/* ---- encode ([MET] Estrategia de Codificacion; [EXT]) ------------------ */

/*
 * Encode n elements of x (2n bytes for BF16, n bytes for E5M2) with codebook
 * cb into out (capacity bytes).  On success writes the stream size to
 * *out_bytes.  If the stream does not fit, nothing is written except
 * *out_bytes (the size needed) and ORC_CAPACITY is returned.
 */
int orc_encode(int dt, const uint8_t *cb, const uint8_t *x, uint64_t n,
               uint8_t *out, uint64_t capacity, uint64_t *out_bytes) {
    if (dt != ORC_BF16 && dt != ORC_E5M2) return ORC_INVALID_ARG;
    if (n >= ((uint64_t)1 << 32)) return ORC_INVALID_ARG;
    if (!orc_codebook_valid(dt, cb)) return ORC_INVALID_ARG;

    uint8_t inv[256];
    inverse_codebook(cb, inv);

    uint64_t n_esc = orc_count_escapes(dt, cb, x, n);
    uint64_t size = orc_encoded_size(dt, n, n_esc);
    *out_bytes = size;
    if (size > capacity) return ORC_CAPACITY;

    uint64_t dense = orc_dense_bytes(dt, n);
    uint64_t chunks = orc_num_chunks(n);
    uint8_t *cb_out = out + dense;
    uint8_t *hdr = cb_out + ORC_CB;
    uint8_t *rec = hdr + 8 * chunks;
    memset(out, 0, dense);

    /* Step 1: dense stream, element by element, collecting escapes in order. */
    uint64_t j = 0; /* escapes written so far */
    for (uint64_t i = 0; i < n; i++) {
        unsigned e = exponent_at(dt, x, i);
        unsigned code = inv[e];
        if (code == ORC_NO_CODE) {
            /* Escape: keep position within the chunk and the raw exponent (R6);
             * the dense stream gets code 0 (R5). */
            put_u16(rec + 3 * j, (unsigned)(i % ORC_CHUNK));
            rec[3 * j + 2] = (uint8_t)e;
            j++;
            code = 0;
        }
        if (dt == ORC_BF16) {
            unsigned v = bf16_at(x, i);
            unsigned sign = (v >> 15) & 1u;
            unsigned mant = v & 0x7Fu;
            out[i] = (uint8_t)((sign << 7) | mant);          /* R1 */
            out[n + i / 2] |= (uint8_t)(code << (4 * (i % 2))); /* R2 */
        } else {
            unsigned v = x[i];
            unsigned sign = (v >> 7) & 1u;
            unsigned mant = v & 0x3u;
            unsigned field = code | (((sign << 2) | mant) << 4); /* R1, R8 */
            uint64_t g = i / 8;
            unsigned bit = 7 * (unsigned)(i % 8);
            /* Field j of the group occupies bits 7j..7j+6 of the group's
             * 56-bit little-endian word: spread it over the bytes it touches. */
            for (unsigned b = 0; b < 7; b++) {
                unsigned lo = 8 * b;
                if (bit + 7 <= lo || bit >= lo + 8) continue;
                if (bit >= lo)
                    out[7 * g + b] |= (uint8_t)((field << (bit - lo)) & 0xFFu);
                else
                    out[7 * g + b] |= (uint8_t)((field >> (lo - bit)) & 0xFFu);
            }
        }
    }

    /* Step 2: codebook, then per-chunk headers (R7). */
    memcpy(cb_out, cb, ORC_CB);
    uint64_t offset = 0;
    for (uint64_t c = 0; c < chunks; c++) {
        uint64_t lo = c * ORC_CHUNK;
        uint64_t hi = lo + ORC_CHUNK < n ? lo + ORC_CHUNK : n;
        uint64_t count = 0;
        for (uint64_t i = lo; i < hi; i++)
            if (inv[exponent_at(dt, x, i)] == ORC_NO_CODE) count++;
        put_u32(hdr + 8 * c, offset);
        put_u32(hdr + 8 * c + 4, count);
        offset += count;
    }
    return ORC_OK;
}

/* ---- validation --------------------------------------------------------- */

/*
 * Check that `in` (in_bytes) is a well-formed stream for n elements: the size
 * matches the closed form for some escape count E, the codebook is valid, the
 * header offsets are the running sum of the counts and end at E, every chunk
 * count fits its chunk, and positions are strictly increasing inside a chunk
 * and below the chunk's length; E5M2 escape exponents must fit 5 bits.
 * Returns ORC_OK (and E in *n_escapes) or ORC_CORRUPT.
 */
int orc_validate(int dt, const uint8_t *in, uint64_t in_bytes, uint64_t n, uint64_t *n_escapes) {
    if (dt != ORC_BF16 && dt != ORC_E5M2) return ORC_INVALID_ARG;
    if (n >= ((uint64_t)1 << 32)) return ORC_INVALID_ARG;
    uint64_t fixed = orc_encoded_size(dt, n, 0);
    if (in_bytes < fixed || (in_bytes - fixed) % 3 != 0) return ORC_CORRUPT;
    uint64_t n_esc = (in_bytes - fixed) / 3;

    uint64_t dense = orc_dense_bytes(dt, n);
    uint64_t chunks = orc_num_chunks(n);
    const uint8_t *cb = in + dense;
    const uint8_t *hdr = cb + ORC_CB;
    const uint8_t *rec = hdr + 8 * chunks;
    if (!orc_codebook_valid(dt, cb)) return ORC_CORRUPT;

    uint64_t running = 0;
    for (uint64_t c = 0; c < chunks; c++) {
        uint64_t offset = get_u32(hdr + 8 * c);
        uint64_t count = get_u32(hdr + 8 * c + 4);
        uint64_t lo = c * ORC_CHUNK;
        uint64_t len = (lo + ORC_CHUNK < n ? lo + ORC_CHUNK : n) - lo;
        if (offset != running || count > len || running + count > n_esc) return ORC_CORRUPT;
        for (uint64_t k = 0; k < count; k++) {
            unsigned pos = get_u16(rec + 3 * (offset + k));
            if (pos >= len) return ORC_CORRUPT;
            if (k > 0 && pos <= get_u16(rec + 3 * (offset + k - 1))) return ORC_CORRUPT;
            if (dt == ORC_E5M2 && rec[3 * (offset + k) + 2] >= 32) return ORC_CORRUPT;
        }
        running += count;
    }
    if (running != n_esc) return ORC_CORRUPT;
    *n_escapes = n_esc;
    return ORC_OK;
}

/* ---- decode ([MET] Estrategia de Decodificacion) ------------------------ */

/*
 * Decode a stream into y (2n bytes for BF16, n bytes for E5M2): validate,
 * then the dense pass (code -> exponent through the codebook, joined with
 * the stored sign and mantissa), then overwrite every escaped element's
 * exponent with its raw value.
 */
int orc_decode(int dt, const uint8_t *in, uint64_t in_bytes, uint64_t n, uint8_t *y) {
    uint64_t n_esc = 0;
    int st = orc_validate(dt, in, in_bytes, n, &n_esc);
    if (st != ORC_OK) return st;

    uint64_t dense = orc_dense_bytes(dt, n);
    uint64_t chunks = orc_num_chunks(n);
    const uint8_t *cb = in + dense;
    const uint8_t *hdr = cb + ORC_CB;
    const uint8_t *rec = hdr + 8 * chunks;

    /* Dense pass. */
    for (uint64_t i = 0; i < n; i++) {
        if (dt == ORC_BF16) {
            unsigned sm = in[i];
            unsigned code = (in[n + i / 2] >> (4 * (i % 2))) & 0xFu;
            unsigned v = ((sm >> 7) << 15) | ((unsigned)cb[code] << 7) | (sm & 0x7Fu);
            y[2 * i] = (uint8_t)(v & 0xFFu);
            y[2 * i + 1] = (uint8_t)(v >> 8);
        } else {
            uint64_t g = i / 8;
            unsigned bit = 7 * (unsigned)(i % 8);
            uint64_t word = 0;
            for (unsigned b = 0; b < 7; b++) word |= (uint64_t)in[7 * g + b] << (8 * b);
            unsigned field = (unsigned)((word >> bit) & 0x7Fu);
            unsigned code = field & 0xFu;
            unsigned sm3 = field >> 4;
            y[i] = (uint8_t)(((sm3 >> 2) << 7) | ((unsigned)cb[code] << 2) | (sm3 & 0x3u));
        }
    }

    /* Escape overwrite: put back the raw exponent of every escaped element. */
    for (uint64_t c = 0; c < chunks; c++) {
        uint64_t offset = get_u32(hdr + 8 * c);
        uint64_t count = get_u32(hdr + 8 * c + 4);
        for (uint64_t k = 0; k < count; k++) {
            uint64_t i = c * ORC_CHUNK + get_u16(rec + 3 * (offset + k));
            unsigned e = rec[3 * (offset + k) + 2];
            if (dt == ORC_BF16) {
                unsigned v = (unsigned)y[2 * i] | ((unsigned)y[2 * i + 1] << 8);
                v = (v & 0x807Fu) | (e << 7);
                y[2 * i] = (uint8_t)(v & 0xFFu);
                y[2 * i + 1] = (uint8_t)(v >> 8);
            } else {
                y[i] = (uint8_t)((y[i] & 0x83u) | (e << 2));
            }
        }
    }
    return ORC_OK;
}

/* ---- codebook ablation sizes ([RES] "Estudios de Ablacion") -------------- */

/* Elements whose exponent is outside the k most frequent ones (the same
 * selection rule as the codebook: repeated arg-max, ties toward the smaller
 * exponent, unseen exponents eligible). */
static uint64_t outside_top_k(int dt, const uint64_t *hist, uint64_t n, int k) {
    int taken[256];
    uint64_t covered = 0;
    pick_most_frequent(dt, hist, k, taken);
    for (int e = 0; e < exponent_bins(dt); e++)
        if (taken[e]) covered += hist[e];
    return n - covered;
}

/* Stream sizes of n elements under the three codebook designs the ablation
 * compares (readings A1-A3):
 *   sizes[0]  Top-16, this format: 4-bit codes, escapes as (u16 position,
 *             u8 exponent) records; = orc_encoded_size with the top-16 set;
 *   sizes[1]  Top-8: 3-bit codes (BF16: 8 codes in 3 bytes next to the sm
 *             bytes; E5M2: 6-bit code|sm3 fields, 4 in 3 bytes), escapes as
 *             above, an 8-byte codebook and the same chunk headers;
 *   sizes[2]  Top-15 + sentinel: code 15 marks an escape, which stores only
 *             its exponent byte (positions are implied), a 15-byte codebook
 *             and the same chunk headers (escape offsets per chunk). */
int orc_ablation_sizes(int dt, const uint64_t *hist, uint64_t n, uint64_t *sizes) {
    uint64_t chunks = orc_num_chunks(n);
    uint64_t e16 = outside_top_k(dt, hist, n, 16);
    uint64_t e8 = outside_top_k(dt, hist, n, 8);
    uint64_t e15 = outside_top_k(dt, hist, n, 15);
    uint64_t dense8 = dt == ORC_BF16 ? n + 3 * ((n + 7) / 8) : 3 * ((n + 3) / 4);
    sizes[0] = orc_encoded_size(dt, n, e16);
    sizes[1] = dense8 + 3 * e8 + 8 + 8 * chunks;
    sizes[2] = orc_dense_bytes(dt, n) + e15 + 15 + 8 * chunks;
    return ORC_OK;
}

/* ---- ablation codecs (BF16; readings A1, A2, A4) -------------------------- */

/* The two alternative designs of the ablation as full codecs, so that their
 * decoding can be compared, not just their sizes.  Variant ORC_ABL_TOP8 (A1):
 * [sm N][codes 3 ceil(N/8)][codebook 8][headers 8C][records 3E]; element j of
 * group g has its 3-bit code at bits 3j..3j+2 of the 24-bit little-endian
 * word at byte 3g, an escape gets code 0 and an R6 record.  Variant
 * ORC_ABL_SENTINEL (A2): [sm N][nibbles ceil(N/2)][codebook 15][headers 8C]
 * [exponent bytes E]; code 15 marks an escape, whose exponent is the next
 * byte of its chunk's run (headers as R7).  Codes follow ascending exponent
 * order (R3).  A4: the decoders check the closed-form size, the headers as
 * running sums, and (Top-8) the record positions as R11 or (sentinel) that
 * each chunk holds as many sentinels as its header counts. */

static int abl_k(int variant) { return variant == ORC_ABL_TOP8 ? 8 : 15; }

uint64_t orc_abl_size(int variant, uint64_t n, uint64_t n_escapes) {
    uint64_t chunks = orc_num_chunks(n);
    if (variant == ORC_ABL_TOP8) return n + 3 * ceil_div(n, 8) + 8 + 8 * chunks + 3 * n_escapes;
    return n + ceil_div(n, 2) + 15 + 8 * chunks + n_escapes;
}

/* The k most frequent exponents (A3), ascending. */
int orc_abl_codebook(int variant, const uint64_t *hist, uint8_t *cb) {
    int taken[256];
    if (variant != ORC_ABL_TOP8 && variant != ORC_ABL_SENTINEL) return ORC_INVALID_ARG;
    pick_most_frequent(ORC_BF16, hist, abl_k(variant), taken);
    int k = 0;
    for (int e = 0; e < 256; e++)
        if (taken[e]) cb[k++] = (uint8_t)e;
    return ORC_OK;
}

int orc_abl_encode(int variant, const uint8_t *cb, const uint8_t *x, uint64_t n,
                   uint8_t *out, uint64_t capacity, uint64_t *out_bytes) {
    if (variant != ORC_ABL_TOP8 && variant != ORC_ABL_SENTINEL) return ORC_INVALID_ARG;
    if (n >= ((uint64_t)1 << 32)) return ORC_INVALID_ARG;
    int k = abl_k(variant);
    uint8_t inv[256];
    for (int e = 0; e < 256; e++) inv[e] = ORC_NO_CODE;
    for (int c = 0; c < k; c++) {
        if (inv[cb[c]] != ORC_NO_CODE) return ORC_INVALID_ARG;
        inv[cb[c]] = (uint8_t)c;
    }
    uint64_t n_esc = 0;
    for (uint64_t i = 0; i < n; i++)
        if (inv[exponent_at(ORC_BF16, x, i)] == ORC_NO_CODE) n_esc++;
    uint64_t size = orc_abl_size(variant, n, n_esc);
    *out_bytes = size;
    if (size > capacity) return ORC_CAPACITY;

    uint64_t chunks = orc_num_chunks(n);
    uint64_t dense = variant == ORC_ABL_TOP8 ? n + 3 * ceil_div(n, 8) : n + ceil_div(n, 2);
    uint8_t *codes = out + n;
    uint8_t *cb_out = out + dense;
    uint8_t *hdr = cb_out + k;
    uint8_t *esc = hdr + 8 * chunks;
    memset(out, 0, dense);

    uint64_t j = 0; /* escapes so far */
    for (uint64_t i = 0; i < n; i++) {
        unsigned v = bf16_at(x, i);
        unsigned e = (v >> 7) & 0xFFu;
        unsigned code = inv[e];
        out[i] = (uint8_t)((((v >> 15) & 1u) << 7) | (v & 0x7Fu)); /* R1 */
        if (variant == ORC_ABL_TOP8) {
            if (code == ORC_NO_CODE) {
                put_u16(esc + 3 * j, (unsigned)(i % ORC_CHUNK));
                esc[3 * j + 2] = (uint8_t)e;
                j++;
                code = 0u; /* A1: an escape keeps code 0 */
            }
            /* 3-bit code j of group g: bits 3j..3j+2 of the 24-bit word. */
            unsigned bit = 3 * (unsigned)(i % 8);
            uint64_t g = i / 8;
            for (unsigned b = 0; b < 3; b++) {
                unsigned lo = 8 * b;
                if (bit + 3 <= lo || bit >= lo + 8) continue;
                if (bit >= lo)
                    codes[3 * g + b] |= (uint8_t)((code << (bit - lo)) & 0xFFu);
                else
                    codes[3 * g + b] |= (uint8_t)((code >> (lo - bit)) & 0xFFu);
            }
        } else {
            if (code == ORC_NO_CODE) {
                esc[j++] = (uint8_t)e;
                code = 15;
            }
            codes[i / 2] |= (uint8_t)(code << (4 * (i % 2))); /* R2 */
        }
    }
    memcpy(cb_out, cb, (size_t)k);
    uint64_t before = 0; /* escapes in earlier chunks */
    for (uint64_t c = 0; c < chunks; c++) {
        uint64_t lo = c * ORC_CHUNK;
        uint64_t hi = lo + ORC_CHUNK < n ? lo + ORC_CHUNK : n;
        uint64_t in_chunk = 0;
        for (uint64_t i = lo; i < hi; i++)
            if (inv[exponent_at(ORC_BF16, x, i)] == ORC_NO_CODE) in_chunk++;
        put_u32(hdr + 8 * c, before);
        put_u32(hdr + 8 * c + 4, in_chunk);
        before += in_chunk;
    }
    return ORC_OK;
}

int orc_abl_decode(int variant, const uint8_t *in, uint64_t in_bytes, uint64_t n, uint8_t *y) {
    if (variant != ORC_ABL_TOP8 && variant != ORC_ABL_SENTINEL) return ORC_INVALID_ARG;
    if (n >= ((uint64_t)1 << 32)) return ORC_INVALID_ARG;
    int k = abl_k(variant);
    uint64_t fixed = orc_abl_size(variant, n, 0);
    unsigned per_escape = variant == ORC_ABL_TOP8 ? 3u : 1u;
    if (in_bytes < fixed || (in_bytes - fixed) % per_escape != 0) return ORC_CORRUPT;
    uint64_t n_esc = (in_bytes - fixed) / per_escape;
    uint64_t chunks = orc_num_chunks(n);
    uint64_t dense = variant == ORC_ABL_TOP8 ? n + 3 * ceil_div(n, 8) : n + ceil_div(n, 2);
    const uint8_t *codes = in + n;
    const uint8_t *cb = in + dense;
    const uint8_t *hdr = cb + k;
    const uint8_t *esc = hdr + 8 * chunks;

    /* Headers: a running sum that ends at E; each count fits its chunk. */
    uint64_t running = 0;
    for (uint64_t c = 0; c < chunks; c++) {
        uint64_t offset = get_u32(hdr + 8 * c), count = get_u32(hdr + 8 * c + 4);
        uint64_t lo = c * ORC_CHUNK;
        uint64_t len = (lo + ORC_CHUNK < n ? lo + ORC_CHUNK : n) - lo;
        if (offset != running || count > len || running + count > n_esc) return ORC_CORRUPT;
        if (variant == ORC_ABL_TOP8) {
            for (uint64_t q = 0; q < count; q++) {
                unsigned pos = get_u16(esc + 3 * (offset + q));
                if (pos >= len || (q > 0 && pos <= get_u16(esc + 3 * (offset + q - 1)))) return ORC_CORRUPT;
            }
        } else {
            uint64_t sentinels = 0;
            for (uint64_t i = lo; i < lo + len; i++)
                if (((codes[i / 2] >> (4 * (i % 2))) & 0xFu) == 15u) sentinels++;
            if (sentinels != count) return ORC_CORRUPT;
        }
        running += count;
    }
    if (running != n_esc) return ORC_CORRUPT;

    for (uint64_t c = 0; c < chunks; c++) {
        uint64_t offset = get_u32(hdr + 8 * c);
        uint64_t lo = c * ORC_CHUNK;
        uint64_t hi = lo + ORC_CHUNK < n ? lo + ORC_CHUNK : n;
        uint64_t seen = 0; /* sentinels so far in this chunk */
        for (uint64_t i = lo; i < hi; i++) {
            unsigned sm = in[i], e;
            if (variant == ORC_ABL_TOP8) {
                uint64_t g = i / 8;
                unsigned word = (unsigned)codes[3 * g] | ((unsigned)codes[3 * g + 1] << 8) |
                                ((unsigned)codes[3 * g + 2] << 16);
                e = cb[(word >> (3 * (unsigned)(i % 8))) & 7u];
            } else {
                unsigned code = (codes[i / 2] >> (4 * (i % 2))) & 0xFu;
                e = code == 15u ? esc[offset + seen++] : cb[code];
            }
            unsigned v = ((sm >> 7) << 15) | (e << 7) | (sm & 0x7Fu);
            y[2 * i] = (uint8_t)(v & 0xFFu);
            y[2 * i + 1] = (uint8_t)(v >> 8);
        }
        if (variant == ORC_ABL_TOP8) { /* escape overwrite */
            uint64_t count = get_u32(hdr + 8 * c + 4);
            for (uint64_t q = 0; q < count; q++) {
                uint64_t i = lo + get_u16(esc + 3 * (offset + q));
                unsigned v = (unsigned)y[2 * i] | ((unsigned)y[2 * i + 1] << 8);
                v = (v & 0x807Fu) | ((unsigned)esc[3 * (offset + q) + 2] << 7);
                y[2 * i] = (uint8_t)(v & 0xFFu);
                y[2 * i + 1] = (uint8_t)(v >> 8);
            }
        }
    }
    return ORC_OK;
}
