/*
 * k3huf_oracle.c -- plain, slow, obviously-correct CPU oracle of the k3_huf
 * bf16 weight codec.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file.  It shares no code,
 * header, table or constant with the CUDA library: every constant and
 * every container offset below is written out here again from the format
 * specification.
 *
 * Source of the method: the article "Kimi K3 纯 CPU 推理中的无损 Trunk 压缩：
 * 一次被解码速度判死刑的 Huffman 压缩实验" (lossless trunk compression in
 * Kimi K3 CPU inference), sections
 *   - 核心思想 (the idea): only the high byte of each bf16 value is entropy
 *     coded with Huffman; the low (mantissa) byte is stored raw;
 *   - 已实现的部分 (what was implemented): container = layer header with the
 *     canonical code lengths codelen[256], then 64 MiB stripes of
 *     [stripe header][odd-byte Huffman bit stream][even bytes raw];
 *     bf16 is little-endian, so the odd offset is the high byte; code
 *     lengths are capped at 12 bits (the encoder flattens deeper trees);
 *   - 规范码分配与 Kraft 校验 (canonical assignment and Kraft check): the
 *     Kraft sum over the 12-bit code space must be full or under-full,
 *     over-subscribed or empty tables are rejected; codes are assigned
 *     longest-first, first[l] = code, then code = (code + count[l]) / 2,
 *     and symbols of one length take consecutive codes in symbol order;
 *     the encoder's lengths come from the depths of a standard Huffman tree
 *     followed by a BZip2-style correction that keeps lengthening the
 *     lowest-frequency code while the Kraft sum is over-full;
 *   - the decode loop keeps the head of the stream at the top of the bit
 *     window, i.e. the stream is read most-significant bit first.
 *
 * Readings where the article is silent or garbled (each is listed in the
 * design notes):
 *   R1 Huffman tie-break: min-heap keyed (count, id), leaves id = symbol,
 *      internal nodes id = 256 + creation index.
 *   R2 a single used symbol gets length 1.
 *   R3 limiter: clamp lengths above maxlen to maxlen; while the Kraft sum
 *      exceeds 2^maxlen, lengthen by one the code of lowest count among the
 *      codes still shorter than maxlen, ties to the larger symbol value.
 *   R4 canonical recurrence with rounding up, code = ceil((code+count[l])/2):
 *      identical to the article's halving on every complete code and
 *      conflict-free on incomplete ones.
 *   R5 bit order: bit j of a stream is bit 7-(j%8) of byte j/8; the last
 *      byte is zero padded.
 *   R6 container, chunk index, sub-stream index and padding: this
 *      project's own layout, version 1 (the article names only
 *      codelen[256] and the stripe order).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- format constants (written again here on purpose) ----------------- */
#define ORC_ALPHABET      256
#define ORC_MAGIC_LAYER   0x4648334Bu   /* bytes 'K','3','H','F' */
#define ORC_MAGIC_STRIPE  0x5348334Bu   /* bytes 'K','3','H','S' */
#define ORC_VERSION       1u
#define ORC_FMT_MAXLEN    12u
#define ORC_STRIPE_VALUES 33554432u     /* 64 MiB of raw bf16 per stripe */
#define ORC_LAYER_HDR     64u
#define ORC_TENSOR_ENTRY  32u
#define ORC_STRIPE_ENTRY  32u
#define ORC_STRIPE_HDR    32u
#define ORC_BITS_SLACK    32u

/* error codes, same meaning as the library's */
#define ORC_OK        0
#define ORC_E_ARG    -1
#define ORC_E_EMPTY  -2
#define ORC_E_OVERSUB -3
#define ORC_E_BADLEN -4
#define ORC_E_FORMAT -5

static uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

static void put16(uint8_t *p, uint32_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void put32(uint8_t *p, uint32_t v) { for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static void put64(uint8_t *p, uint64_t v) { for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static uint32_t get16(const uint8_t *p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8); }
static uint32_t get32(const uint8_t *p) {
    uint32_t v = 0;
    for (int i = 3; i >= 0; i--) v = (v << 8) | p[i];
    return v;
}
static uint64_t get64(const uint8_t *p) {
    uint64_t v = 0;
    for (int i = 7; i >= 0; i--) v = (v << 8) | p[i];
    return v;
}

/* ---- step 1: histogram of the high bytes (odd offsets) ------------------ */
void orc_histogram(const uint8_t *bf16_bytes, uint64_t n_values, uint64_t cnt[256])
{
    for (int s = 0; s < ORC_ALPHABET; s++) cnt[s] = 0;
    for (uint64_t i = 0; i < n_values; i++) cnt[bf16_bytes[2 * i + 1]]++;
}

/* ---- step 2: unconstrained Huffman code lengths (reading R1, R2) -------- */
typedef struct { uint64_t w; uint32_t id; } orc_node;

static int node_less(orc_node a, orc_node b) { return a.w < b.w || (a.w == b.w && a.id < b.id); }

static void heap_push(orc_node *h, int *n, orc_node x)
{
    int i = (*n)++;
    h[i] = x;
    while (i > 0) {
        int p = (i - 1) / 2;
        if (!node_less(h[i], h[p])) break;
        orc_node t = h[i]; h[i] = h[p]; h[p] = t;
        i = p;
    }
}

static orc_node heap_pop(orc_node *h, int *n)
{
    orc_node top = h[0];
    h[0] = h[--(*n)];
    int i = 0;
    for (;;) {
        int l = 2 * i + 1, r = l + 1, m = i;
        if (l < *n && node_less(h[l], h[m])) m = l;
        if (r < *n && node_less(h[r], h[m])) m = r;
        if (m == i) break;
        orc_node t = h[i]; h[i] = h[m]; h[m] = t;
        i = m;
    }
    return top;
}

/* len[s] = depth of leaf s in the Huffman tree; 0 for unused symbols. */
void orc_huffman_lengths(const uint64_t cnt[256], int len[256])
{
    orc_node heap[2 * ORC_ALPHABET];
    int parent[2 * ORC_ALPHABET];
    int hn = 0, used = 0;
    for (int s = 0; s < ORC_ALPHABET; s++) {
        len[s] = 0;
        if (cnt[s] > 0) {
            orc_node x = { cnt[s], (uint32_t)s };
            heap_push(heap, &hn, x);
            used++;
        }
    }
    if (used == 0) return;
    if (used == 1) {                       /* reading R2 */
        for (int s = 0; s < ORC_ALPHABET; s++) if (cnt[s] > 0) len[s] = 1;
        return;
    }
    for (int i = 0; i < 2 * ORC_ALPHABET; i++) parent[i] = -1;
    uint32_t next_id = ORC_ALPHABET;
    while (hn > 1) {
        orc_node a = heap_pop(heap, &hn);
        orc_node b = heap_pop(heap, &hn);
        orc_node c = { a.w + b.w, next_id++ };
        parent[a.id] = (int)c.id;
        parent[b.id] = (int)c.id;
        heap_push(heap, &hn, c);
    }
    for (int s = 0; s < ORC_ALPHABET; s++) {
        if (cnt[s] == 0) continue;
        int d = 0;
        for (int v = s; parent[v] >= 0; v = parent[v]) d++;
        len[s] = d;
    }
}

/* Kraft sum in units of 2^-maxlen: sum over used symbols of 2^(maxlen-len).
 * Lengths above maxlen contribute 0 here; callers check them separately. */
uint64_t orc_kraft(const int len[256], int maxlen)
{
    uint64_t k = 0;
    for (int s = 0; s < ORC_ALPHABET; s++)
        if (len[s] > 0 && len[s] <= maxlen) k += (uint64_t)1 << (maxlen - len[s]);
    return k;
}

/* ---- step 3: length limit, BZip2-style correction (reading R3) --------- */
void orc_limit_lengths(const uint64_t cnt[256], int len[256], int maxlen)
{
    for (int s = 0; s < ORC_ALPHABET; s++)
        if (len[s] > maxlen) len[s] = maxlen;
    const uint64_t full = (uint64_t)1 << maxlen;
    while (orc_kraft(len, maxlen) > full) {
        int pick = -1;
        for (int s = 0; s < ORC_ALPHABET; s++) {
            if (len[s] == 0 || len[s] >= maxlen) continue;
            if (pick < 0 || cnt[s] < cnt[pick] || (cnt[s] == cnt[pick] && s > pick)) pick = s;
        }
        if (pick < 0) break;               /* cannot happen for <= 256 symbols */
        len[pick] += 1;
    }
}

/* The encoder's code lengths: Huffman depths, then the limiter. */
void orc_code_lengths(const uint64_t cnt[256], int maxlen, int len[256])
{
    orc_huffman_lengths(cnt, len);
    orc_limit_lengths(cnt, len, maxlen);
}

/* ---- step 4: the table check of the decoder's build function ----------- */
int orc_check_codelen(const uint8_t codelen[256], int maxlen)
{
    uint64_t k = 0;
    for (int s = 0; s < ORC_ALPHABET; s++) {
        if (codelen[s] > maxlen) return ORC_E_BADLEN;
        if (codelen[s] > 0) k += (uint64_t)1 << (maxlen - codelen[s]);
    }
    if (k == 0) return ORC_E_EMPTY;
    if (k > ((uint64_t)1 << maxlen)) return ORC_E_OVERSUB;
    return ORC_OK;
}

/* ---- step 5: canonical longest-first assignment (reading R4) ----------- */
/* count[l], first[l] for l = 1..maxlen, code[s] for every used symbol. */
void orc_canonical(const int len[256], int maxlen, uint32_t count[33], uint32_t first[33], uint32_t code[256])
{
    for (int l = 0; l < 33; l++) { count[l] = 0; first[l] = 0; }
    for (int s = 0; s < ORC_ALPHABET; s++) if (len[s] > 0) count[len[s]]++;
    uint32_t c = 0;
    for (int l = maxlen; l >= 1; l--) {
        first[l] = c;
        c = (c + count[l] + 1) >> 1;
    }
    uint32_t rank[33];
    for (int l = 0; l < 33; l++) rank[l] = 0;
    for (int s = 0; s < ORC_ALPHABET; s++) {
        code[s] = 0;
        if (len[s] > 0) code[s] = first[len[s]] + rank[len[s]]++;
    }
}

/* ---- bit-serial decoding of one symbol (no lookup table) --------------- */
typedef struct {
    int maxlen;
    uint32_t count[33], first[33];
    uint8_t sym_by_rank[33][256];          /* symbols of length l, ascending */
} orc_code;

static int orc_code_init(orc_code *c, const uint8_t codelen[256], int maxlen)
{
    int rc = orc_check_codelen(codelen, maxlen);
    if (rc) return rc;
    int len[256];
    uint32_t code[256];
    for (int s = 0; s < ORC_ALPHABET; s++) len[s] = codelen[s];
    c->maxlen = maxlen;
    orc_canonical(len, maxlen, c->count, c->first, code);
    uint32_t rank[33] = {0};
    for (int s = 0; s < ORC_ALPHABET; s++)
        if (len[s] > 0) c->sym_by_rank[len[s]][rank[len[s]]++] = (uint8_t)s;
    return ORC_OK;
}

/* Reads bits one at a time through get_bit(ctx, i) for i = 0, 1, ...;
 * returns the symbol (>= 0) and its length in *used, or -1 if no code of
 * length <= maxlen matches the bits read. */
typedef int (*orc_bit_fn)(const void *ctx, uint64_t i);

static int orc_decode_symbol(const orc_code *c, orc_bit_fn get_bit, const void *ctx, uint64_t pos, int *used)
{
    uint32_t v = 0;
    for (int l = 1; l <= c->maxlen; l++) {
        v = (v << 1) | (uint32_t)get_bit(ctx, pos + (uint64_t)(l - 1));
        if (c->count[l] > 0 && v >= c->first[l] && v < c->first[l] + c->count[l]) {
            *used = l;
            return c->sym_by_rank[l][v - c->first[l]];
        }
    }
    *used = 0;
    return -1;
}

typedef struct { const uint8_t *bytes; uint64_t nbits; } orc_stream;

static int stream_bit(const void *ctx, uint64_t i)     /* reading R5 */
{
    const orc_stream *s = (const orc_stream *)ctx;
    if (i >= s->nbits) return 0;
    return (s->bytes[i >> 3] >> (7 - (i & 7))) & 1;
}

static int window_bit(const void *ctx, uint64_t i)
{
    const uint32_t *w = (const uint32_t *)ctx;          /* w[0] = window, w[1] = width */
    if (i >= w[1]) return 0;
    return (w[0] >> (w[1] - 1 - i)) & 1;
}

/* Decode the symbol at the top of a maxlen-bit window (the meaning of one
 * entry of the decoder's lookup table).  Returns the symbol and *used, or
 * -1 for a window that starts with no valid code; table errors are
 * returned as the codes of orc_check_codelen (< -1). */
int orc_decode_window(const uint8_t codelen[256], int maxlen, uint32_t window, int *used)
{
    orc_code c;
    int rc = orc_code_init(&c, codelen, maxlen);
    if (rc) { *used = 0; return rc; }
    uint32_t ctx[2] = { window, (uint32_t)maxlen };
    return orc_decode_symbol(&c, window_bit, ctx, 0, used);
}

/* ---- bit writer (reading R5) ------------------------------------------- */
static void put_bits(uint8_t *bytes, uint64_t *pos, uint32_t code, int len)
{
    for (int b = len - 1; b >= 0; b--) {
        if ((code >> b) & 1) bytes[*pos >> 3] |= (uint8_t)(0x80u >> (*pos & 7));
        (*pos)++;
    }
}

/* ---- container layout (reading R6) -------------------------------------
 * layer header (64 B, little-endian):
 *   0 u32 magic 'K3HF' | 4 u16 version | 6 u16 maxlen | 8 u32 chunk_syms
 *  12 u32 n_tables | 16 u32 n_tensors | 20 u32 n_stripes | 24 u64 raw_bytes
 *  32 u64 blob_bytes | 40 u32 stripe_values | 44 u32 hdr_bytes
 *  48 u64 out_bytes | 56 u32 sub_syms | 60 zero
 * then codelen[256] per table, the tensor directory (32 B each:
 *   u32 table_id, u32 first_stripe, u32 n_stripes, u32 0, u64 n_values,
 *   u64 out_offset), the stripe directory (32 B each: u64 blob_offset,
 *   u64 stripe_bytes, u64 out_offset, u32 n_values, u32 table_id), zero
 *   padding to hdr_bytes (a multiple of 256).
 * each stripe starts 256-B aligned:
 *   0 u32 magic 'K3HS' | 4 u32 table_id | 8 u32 n_values | 12 u32 n_chunks
 *  16 u64 huff_bits | 24 u32 bits_offset | 28 u32 even_offset
 *  32 u32 chunk_bitoff[n_chunks]
 *  then u16 sub_bitoff[n_chunks][S-1], S = chunk_syms / sub_syms: entry
 *     k-1 of chunk c is the bit offset, relative to chunk c's first bit,
 *     of the code of value min(k sub_syms, len_c) of the chunk
 *  bits_offset = align16(32 + 4 n_chunks + 2 n_chunks (S-1)): the bit stream, padded with zero
 *     bytes to align16(ceil(huff_bits/8)) + 32 bytes
 *  even_offset = end of the padded bit stream: the n low bytes, then zero
 *     padding to a multiple of 16 (stripe_bytes = even_offset + align16(n))
 * tensor outputs start at 256-B aligned offsets of the layer output. */

typedef struct {
    uint64_t n_values;
    uint32_t table;
    uint32_t n_stripes;
    uint64_t out_offset;
} orc_tensor_plan;

static uint32_t n_chunks_of(uint64_t n, uint32_t chunk_syms) { return (uint32_t)((n + chunk_syms - 1) / chunk_syms); }

/* Sub-streams per chunk.  A requested sub_syms that is 0, does not divide
 * chunk_syms, or would let a relative offset exceed 16 bits (chunks longer
 * than 65535 / 12 values) means no sub-stream index (one sub-stream). */
static uint32_t effective_sub_syms(uint32_t chunk_syms, uint32_t sub_syms)
{
    if (sub_syms == 0 || chunk_syms % sub_syms != 0 || (uint64_t)chunk_syms * ORC_FMT_MAXLEN > 65535u)
        return chunk_syms;
    return sub_syms;
}

static uint64_t index_bytes(uint32_t nch, uint32_t chunk_syms, uint32_t sub_syms)
{
    uint64_t S = chunk_syms / sub_syms;
    return 4ull * nch + 2ull * nch * (S - 1);
}

/* Encode a layer.  tensors[t] points at n_values[t] little-endian bf16
 * values.  shared_table != 0 gives one code table for the whole layer
 * (histogram summed over all tensors), else one table per tensor.  With
 * out == NULL only *blob_bytes is computed. */
int orc_encode_layer(int n_tensors, const uint8_t *const *tensors, const uint64_t *n_values,
                     uint32_t chunk_syms, uint32_t sub_syms_req, int shared_table, int maxlen,
                     uint8_t *out, uint64_t cap, uint64_t *blob_bytes)
{
    if (n_tensors <= 0 || chunk_syms == 0 || maxlen < 1 || maxlen > 16) return ORC_E_ARG;
    uint32_t sub_syms = effective_sub_syms(chunk_syms, sub_syms_req);
    uint32_t S = chunk_syms / sub_syms;
    for (int t = 0; t < n_tensors; t++) if (n_values[t] == 0) return ORC_E_ARG;
    int n_tables = shared_table ? 1 : n_tensors;
    int (*lens)[256] = calloc((size_t)n_tables, sizeof *lens);
    orc_tensor_plan *tp = calloc((size_t)n_tensors, sizeof *tp);
    if (!lens || !tp) { free(lens); free(tp); return ORC_E_ARG; }

    /* code lengths */
    for (int tb = 0; tb < n_tables; tb++) {
        uint64_t cnt[256] = {0}, part[256];
        for (int t = 0; t < n_tensors; t++) {
            if (!shared_table && t != tb) continue;
            orc_histogram(tensors[t], n_values[t], part);
            for (int s = 0; s < 256; s++) cnt[s] += part[s];
        }
        orc_code_lengths(cnt, maxlen, lens[tb]);
    }

    /* sizes */
    uint64_t n_stripes = 0, raw = 0, outp = 0;
    for (int t = 0; t < n_tensors; t++) {
        tp[t].n_values = n_values[t];
        tp[t].table = shared_table ? 0u : (uint32_t)t;
        tp[t].n_stripes = (uint32_t)((n_values[t] + ORC_STRIPE_VALUES - 1) / ORC_STRIPE_VALUES);
        outp = align_up(outp, 256);
        tp[t].out_offset = outp;
        outp += 2 * n_values[t];
        raw += 2 * n_values[t];
        n_stripes += tp[t].n_stripes;
    }
    uint64_t hdr = align_up(ORC_LAYER_HDR + 256ull * n_tables + ORC_TENSOR_ENTRY * (uint64_t)n_tensors
                            + ORC_STRIPE_ENTRY * n_stripes, 256);
    uint64_t pos = hdr;
    for (int t = 0; t < n_tensors; t++) {
        for (uint32_t k = 0; k < tp[t].n_stripes; k++) {
            uint64_t v0 = (uint64_t)k * ORC_STRIPE_VALUES;
            uint64_t nv = n_values[t] - v0 < ORC_STRIPE_VALUES ? n_values[t] - v0 : ORC_STRIPE_VALUES;
            uint64_t bits = 0;
            for (uint64_t i = 0; i < nv; i++) bits += (uint64_t)lens[tp[t].table][tensors[t][2 * (v0 + i) + 1]];
            uint32_t nch = n_chunks_of(nv, chunk_syms);
            uint64_t bits_off = align_up(ORC_STRIPE_HDR + index_bytes(nch, chunk_syms, sub_syms), 16);
            uint64_t even_off = bits_off + align_up((bits + 7) / 8, 16) + ORC_BITS_SLACK;
            uint64_t sbytes = even_off + align_up(nv, 16);
            pos = align_up(pos, 256) + sbytes;
        }
    }
    *blob_bytes = pos;
    if (!out) { free(lens); free(tp); return ORC_OK; }
    if (cap < pos) { free(lens); free(tp); return ORC_E_ARG; }
    memset(out, 0, pos);

    /* header, tables, tensor directory */
    put32(out + 0, ORC_MAGIC_LAYER);
    put16(out + 4, ORC_VERSION);
    put16(out + 6, (uint32_t)maxlen);
    put32(out + 8, chunk_syms);
    put32(out + 12, (uint32_t)n_tables);
    put32(out + 16, (uint32_t)n_tensors);
    put32(out + 20, (uint32_t)n_stripes);
    put64(out + 24, raw);
    put64(out + 32, pos);
    put32(out + 40, ORC_STRIPE_VALUES);
    put32(out + 44, (uint32_t)hdr);
    put64(out + 48, outp);
    put32(out + 56, sub_syms);
    for (int tb = 0; tb < n_tables; tb++)
        for (int s = 0; s < 256; s++) out[ORC_LAYER_HDR + 256 * tb + s] = (uint8_t)lens[tb][s];
    uint8_t *tdir = out + ORC_LAYER_HDR + 256 * n_tables;
    uint8_t *sdir = tdir + ORC_TENSOR_ENTRY * n_tensors;
    uint32_t stripe_id = 0;
    for (int t = 0; t < n_tensors; t++) {
        uint8_t *e = tdir + ORC_TENSOR_ENTRY * t;
        put32(e + 0, tp[t].table);
        put32(e + 4, stripe_id);
        put32(e + 8, tp[t].n_stripes);
        put64(e + 16, n_values[t]);
        put64(e + 24, tp[t].out_offset);
        stripe_id += tp[t].n_stripes;
    }

    /* stripes */
    pos = hdr;
    stripe_id = 0;
    for (int t = 0; t < n_tensors; t++) {
        int *ln = lens[tp[t].table];
        uint32_t count[33], first[33], code[256];
        orc_canonical(ln, maxlen, count, first, code);
        for (uint32_t k = 0; k < tp[t].n_stripes; k++, stripe_id++) {
            uint64_t v0 = (uint64_t)k * ORC_STRIPE_VALUES;
            uint64_t nv = n_values[t] - v0 < ORC_STRIPE_VALUES ? n_values[t] - v0 : ORC_STRIPE_VALUES;
            uint32_t nch = n_chunks_of(nv, chunk_syms);
            uint64_t bits_off = align_up(ORC_STRIPE_HDR + index_bytes(nch, chunk_syms, sub_syms), 16);
            pos = align_up(pos, 256);
            uint8_t *st = out + pos;
            uint8_t *bytes = st + bits_off;
            uint8_t *sub = st + ORC_STRIPE_HDR + 4ull * nch;
            uint64_t bp = 0, chunk_start = 0;
            for (uint64_t i = 0; i <= nv; i++) {
                uint64_t c = i / chunk_syms, k = (i % chunk_syms) / sub_syms;
                if (i < nv && i % chunk_syms == 0) {
                    put32(st + ORC_STRIPE_HDR + 4 * c, (uint32_t)bp);
                    chunk_start = bp;
                }
                /* sub-stream k (k >= 1) of chunk c starts at value c*chunk_syms + k*sub_syms */
                if (i % sub_syms == 0 && k > 0 && i <= nv)
                    put16(sub + 2 * (c * (S - 1) + (k - 1)), (uint32_t)(bp - chunk_start));
                if (i == nv) {
                    /* a short last chunk: its missing sub-stream starts sit at its end */
                    uint64_t clast = (nv - 1) / chunk_syms;
                    uint64_t used = nv - clast * chunk_syms;             /* values in the last chunk */
                    for (uint64_t kk = 1; kk < S; kk++)
                        if (kk * sub_syms >= used)
                            put16(sub + 2 * (clast * (S - 1) + (kk - 1)), (uint32_t)(bp - chunk_start));
                    break;
                }
                uint8_t s = tensors[t][2 * (v0 + i) + 1];
                put_bits(bytes, &bp, code[s], ln[s]);
            }
            uint64_t even_off = bits_off + align_up((bp + 7) / 8, 16) + ORC_BITS_SLACK;
            for (uint64_t i = 0; i < nv; i++) st[even_off + i] = tensors[t][2 * (v0 + i)];
            uint64_t sbytes = even_off + align_up(nv, 16);
            put32(st + 0, ORC_MAGIC_STRIPE);
            put32(st + 4, tp[t].table);
            put32(st + 8, (uint32_t)nv);
            put32(st + 12, nch);
            put64(st + 16, bp);
            put32(st + 24, (uint32_t)bits_off);
            put32(st + 28, (uint32_t)even_off);
            uint8_t *e = sdir + ORC_STRIPE_ENTRY * stripe_id;
            put64(e + 0, pos);
            put64(e + 8, sbytes);
            put64(e + 16, tp[t].out_offset + 2 * v0);
            put32(e + 24, (uint32_t)nv);
            put32(e + 28, tp[t].table);
            pos += sbytes;
        }
    }
    free(lens);
    free(tp);
    return ORC_OK;
}

/* ---- container reading and bit-serial decoding ------------------------- */

/* Header fields the Python side wants: fills info[0..9] =
 * chunk_syms, n_tables, n_tensors, n_stripes, raw_bytes, blob_bytes,
 * hdr_bytes, out_bytes, maxlen, sub_syms. */
int orc_layer_info(const uint8_t *blob, uint64_t bytes, uint64_t info[10])
{
    if (bytes < ORC_LAYER_HDR) return ORC_E_FORMAT;
    if (get32(blob) != ORC_MAGIC_LAYER || get16(blob + 4) != ORC_VERSION) return ORC_E_FORMAT;
    info[0] = get32(blob + 8);
    info[1] = get32(blob + 12);
    info[2] = get32(blob + 16);
    info[3] = get32(blob + 20);
    info[4] = get64(blob + 24);
    info[5] = get64(blob + 32);
    info[6] = get32(blob + 44);
    info[7] = get64(blob + 48);
    info[8] = get16(blob + 6);
    info[9] = get32(blob + 56);
    if (info[0] == 0 || info[9] == 0 || info[0] % info[9] != 0) return ORC_E_FORMAT;
    return ORC_OK;
}

/* Decode stripe `s` of the layer into out (the layer output buffer).  The
 * bit stream is read one bit at a time.  Returns ORC_OK, a table error, or
 * ORC_E_FORMAT for a malformed stream (a bit pattern with no code, a chunk
 * whose end does not meet the next chunk's recorded offset, or bits read
 * past the stream end).  first_chunk / n_chunks select a range of chunks
 * (n_chunks = 0xFFFFFFFF for all). */
int orc_decode_stripe_range(const uint8_t *blob, uint64_t bytes, uint32_t s,
                            uint32_t first_chunk, uint32_t n_chunks_sel, uint8_t *out)
{
    uint64_t info[10];
    int rc = orc_layer_info(blob, bytes, info);
    if (rc) return rc;
    uint32_t chunk_syms = (uint32_t)info[0], n_tables = (uint32_t)info[1];
    uint32_t sub_syms = (uint32_t)info[9], S = chunk_syms / sub_syms;
    uint32_t n_tensors = (uint32_t)info[2], n_stripes = (uint32_t)info[3];
    int maxlen = (int)info[8];
    if (s >= n_stripes || chunk_syms == 0) return ORC_E_ARG;
    const uint8_t *sdir = blob + ORC_LAYER_HDR + 256ull * n_tables + ORC_TENSOR_ENTRY * (uint64_t)n_tensors
                          + ORC_STRIPE_ENTRY * (uint64_t)s;
    uint64_t off = get64(sdir), sbytes = get64(sdir + 8), out_off = get64(sdir + 16);
    uint32_t table = get32(sdir + 28);
    if (table >= n_tables || off + sbytes > bytes) return ORC_E_FORMAT;
    const uint8_t *st = blob + off;
    if (get32(st) != ORC_MAGIC_STRIPE) return ORC_E_FORMAT;
    uint32_t nv = get32(st + 8), nch = get32(st + 12);
    uint64_t huff_bits = get64(st + 16);
    uint32_t bits_off = get32(st + 24), even_off = get32(st + 28);
    if (nch != n_chunks_of(nv, chunk_syms) || (uint64_t)even_off + nv > sbytes) return ORC_E_FORMAT;
    if (bits_off < ORC_STRIPE_HDR + index_bytes(nch, chunk_syms, sub_syms)) return ORC_E_FORMAT;
    const uint8_t *sub = st + ORC_STRIPE_HDR + 4ull * nch;
    orc_code code;
    rc = orc_code_init(&code, blob + ORC_LAYER_HDR + 256ull * table, maxlen);
    if (rc) return rc;
    orc_stream stream = { st + bits_off, huff_bits };
    uint32_t last = n_chunks_sel == 0xFFFFFFFFu ? nch : first_chunk + n_chunks_sel;
    if (last > nch) last = nch;
    for (uint32_t c = first_chunk; c < last; c++) {
        uint64_t bp = get32(st + ORC_STRIPE_HDR + 4ull * c);
        uint64_t end = (c + 1 < nch) ? get32(st + ORC_STRIPE_HDR + 4ull * (c + 1)) : huff_bits;
        uint64_t i0 = (uint64_t)c * chunk_syms;
        uint64_t i1 = i0 + chunk_syms < nv ? i0 + chunk_syms : nv;
        uint64_t cstart = bp;
        for (uint64_t i = i0; i < i1; i++) {
            int used;
            uint64_t k = (i - i0) / sub_syms;
            if ((i - i0) % sub_syms == 0 && k > 0 && get16(sub + 2 * ((uint64_t)c * (S - 1) + (k - 1))) != bp - cstart)
                return ORC_E_FORMAT;
            if (bp >= huff_bits) return ORC_E_FORMAT;
            int sym = orc_decode_symbol(&code, stream_bit, &stream, bp, &used);
            if (sym < 0) return ORC_E_FORMAT;
            bp += (uint64_t)used;
            out[out_off + 2 * i] = st[even_off + i];
            out[out_off + 2 * i + 1] = (uint8_t)sym;
        }
        if (bp != end) return ORC_E_FORMAT;
        for (uint64_t k = 1; k < S; k++)           /* sub-streams starting at or past the chunk end */
            if (k * sub_syms >= i1 - i0 && get16(sub + 2 * ((uint64_t)c * (S - 1) + (k - 1))) != bp - cstart)
                return ORC_E_FORMAT;
    }
    return ORC_OK;
}

/* Decode the whole layer into out (info[7] bytes; gaps between tensors are
 * left as they are). */
int orc_decode_layer(const uint8_t *blob, uint64_t bytes, uint8_t *out)
{
    uint64_t info[10];
    int rc = orc_layer_info(blob, bytes, info);
    if (rc) return rc;
    for (uint32_t s = 0; s < (uint32_t)info[3]; s++) {
        rc = orc_decode_stripe_range(blob, bytes, s, 0, 0xFFFFFFFFu, out);
        if (rc) return rc;
    }
    return ORC_OK;
}
