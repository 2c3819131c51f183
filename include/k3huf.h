/*
 * k3huf.h -- C ABI of the k3_huf bf16 weight codec on GB300 (sm_103a).
 *
 * The codec: the high byte (sign and exponent) of every little-endian bf16
 * value -- the odd byte offset -- is coded with a canonical, longest-first
 * Huffman code whose lengths are capped at 12 bits; the low (mantissa) byte
 * -- the even offset -- is stored raw.  Decoding is exact: the output bytes
 * equal the original bytes.  Source: the article "Kimi K3 纯 CPU 推理中的无损
 * Trunk 压缩：一次被解码速度判死刑的 Huffman 压缩实验", sections 核心思想
 * (byte-plane split), 已实现的部分 (container, 64 MiB stripes, 12-bit cap,
 * 4096-entry symbol/length table) and 规范码分配与 Kraft 校验 (table check
 * and canonical assignment).
 *
 * Conventions for every call:
 *  - the return value is K3HUF_OK (0) or a negative K3HUF_E_* code; no call
 *    throws, aborts or prints;
 *  - the caller owns every buffer and every stream; the decode calls
 *    allocate nothing (only k3huf_ring_create allocates, once);
 *  - "d_" pointers are device pointers on the current CUDA device and must
 *    be 16-byte aligned; "h_" pointers are host pointers;
 *  - decode calls are asynchronous on the given cudaStream_t (passed as
 *    void*, NULL = the legacy default stream).  Faults that the host can
 *    see (bad header, bad table, sizes, alignment) are returned at once;
 *    faults inside the compressed streams are OR-ed into *d_status (a
 *    device uint32 the caller zeroes beforehand and reads after the stream
 *    is synchronised); the output bytes are unspecified when it is nonzero;
 *  - no kernel of this library traps, asserts or waits without bound.
 *
 * Container, format version 1 (little-endian; all offsets in bytes):
 *  layer header, 64 B: u32 magic 'K3HF' | u16 version | u16 maxlen (12) |
 *    u32 chunk_syms | u32 n_tables | u32 n_tensors | u32 n_stripes |
 *    u64 raw_bytes | u64 blob_bytes | u32 stripe_values (2^25) |
 *    u32 hdr_bytes | u64 out_bytes | u32 sub_syms | 4 B zero
 *  codelen[256] per table; tensor directory, 32 B per tensor:
 *    u32 table, u32 first_stripe, u32 n_stripes, u32 0, u64 n_values,
 *    u64 out_offset; stripe directory, 32 B per stripe: u64 blob_offset,
 *    u64 stripe_bytes, u64 out_offset, u32 n_values, u32 table; zero
 *    padding up to hdr_bytes (a multiple of 256).
 *  stripe (256-B aligned; <= 2^25 values of one tensor):
 *    u32 magic 'K3HS' | u32 table | u32 n_values | u32 n_chunks |
 *    u64 huff_bits | u32 bits_offset | u32 even_offset, then
 *    u32 chunk_bitoff[n_chunks] (bit offset of the first code of every run
 *    of chunk_syms values), u16 sub_bitoff[n_chunks][S-1] with
 *    S = chunk_syms / sub_syms (entry k-1 of chunk c: bit offset, relative
 *    to the chunk's first bit, of the code of value min(k sub_syms, len_c)
 *    of the chunk -- S independent sub-streams per chunk; S = 1 when
 *    chunk_syms * 12 > 65535), the bit stream at bits_offset =
 *    align16(32 + 4 n_chunks + 2 n_chunks (S-1)), read most-significant bit first, zero padded
 *    to align16(ceil(huff_bits/8)) + 32 bytes; the n raw low bytes at
 *    even_offset = bits_offset + that padded size, zero padded to a
 *    multiple of 16.  Tensor outputs start at 256-B aligned offsets of the
 *    layer output (out_offset).
 */
#ifndef K3HUF_H
#define K3HUF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define K3HUF_MAXLEN         12          /* longest code, bits */
#define K3HUF_TABLE_ENTRIES  4096        /* 1 << K3HUF_MAXLEN */
#define K3HUF_STRIPE_VALUES  33554432u   /* 64 MiB of bf16 per stripe */
#define K3HUF_FORMAT_VERSION 1
#define K3HUF_LAYER_HDR_BYTES 64
#define K3HUF_STRIPE_HDR_BYTES 32

/* return codes */
#define K3HUF_OK         0
#define K3HUF_E_ARG     -1   /* bad argument: null, size, alignment */
#define K3HUF_E_EMPTY   -2   /* code table with no symbol */
#define K3HUF_E_OVERSUB -3   /* code table over-subscribed (Kraft sum > 2^12) */
#define K3HUF_E_BADLEN  -4   /* a code length above 12 */
#define K3HUF_E_FORMAT  -5   /* container malformed: magic, version, sizes, offsets */
#define K3HUF_E_CUDA    -6   /* a CUDA runtime call failed; see k3huf_last_cuda_error */
#define K3HUF_E_NOMEM   -7   /* host allocation failed (encoder / ring only) */
#define K3HUF_E_IO      -8   /* file open or read failed (storage feed only) */

/* bits OR-ed into *d_status by the decode kernels */
#define K3HUF_ST_BADCODE  1u  /* a bit pattern that starts no code */
#define K3HUF_ST_OVERRUN  2u  /* a chunk read past the end of its stripe's stream */
#define K3HUF_ST_INDEX    4u  /* a chunk did not end at the next chunk's recorded offset */
#define K3HUF_ST_HEADER   8u  /* a device-side stripe header disagrees with the layer header */
#define K3HUF_ST_TIMEOUT 16u  /* a bounded wait for an asynchronous copy gave up (work skipped) */

typedef struct {
    uint32_t chunk_syms, n_tables, n_tensors, n_stripes;
    uint64_t raw_bytes;      /* sum of 2 * n_values over tensors */
    uint64_t blob_bytes;     /* container size */
    uint64_t out_bytes;      /* decoded layer size, including alignment gaps */
    uint32_t hdr_bytes;      /* bytes of header + tables + directories (padded) */
    uint32_t stripe_values;
    uint32_t sub_syms;       /* values per independently decodable sub-stream */
    uint32_t reserved;
} k3huf_layer_info_t;

typedef struct {
    uint32_t table, first_stripe, n_stripes, reserved;
    uint64_t n_values, out_offset;
} k3huf_tensor_info_t;

/* Build the decoder's 4096-entry table from code lengths (host, pure).
 * Article section 规范码分配与 Kraft 校验: the Kraft sum
 * sum_s 2^(12 - codelen[s]) over used symbols must be at most 4096 (full or
 * under-full) and nonzero; codes are assigned longest-first,
 * first[l] = code; code = ceil((code + count[l]) / 2) for l = 12 .. 1, and
 * symbols of one length take consecutive codes in symbol order.  Entry i of
 * sym_len is (s << 4) | codelen[s] for the symbol s whose code is a prefix
 * of the 12-bit value i, 0 where no code is (incomplete tables).
 * codelen: 256 bytes, 0 = unused symbol.  sym_len: 4096 uint16 written by
 * the call (may be NULL to only check the table).
 * Returns K3HUF_OK, K3HUF_E_BADLEN, K3HUF_E_EMPTY, K3HUF_E_OVERSUB or
 * K3HUF_E_ARG (codelen NULL). */
int k3huf_build(const uint8_t codelen[256], uint16_t sym_len[4096]);

/* Parse and validate a layer header (host copy of the first hdr_bytes of
 * the container, or more): magic, version, maxlen, every table
 * (k3huf_build), the directories (stripe ranges inside blob_bytes, 256-B
 * alignment, tensor/stripe consistency).  Returns K3HUF_E_FORMAT with
 * info untouched when bytes < hdr_bytes.  The call reads only h_layer. */
int k3huf_layer_info(const void *h_layer, size_t bytes, k3huf_layer_info_t *info);

/* Directory entry of tensor t of a validated header. */
int k3huf_tensor_info(const void *h_layer, size_t bytes, uint32_t t, k3huf_tensor_info_t *out);

/* Decode a whole layer on the GPU.
 *  h_layer_hdr / hdr_bytes: host copy of at least the header part of the
 *    container (the same bytes as the device copy's first hdr_bytes);
 *  d_layer / layer_bytes: the whole container in device memory;
 *  d_out / out_bytes: decoded output (>= info.out_bytes); tensor t's bf16
 *    values land at d_out + out_offset(t); alignment gaps are not written;
 *  d_status: device uint32, OR-ed with K3HUF_ST_* bits;
 *  stream: cudaStream_t.
 * One kernel launch per 64 stripes.  Returns K3HUF_OK once launched. */
int k3huf_decode_layer(const void *h_layer_hdr, size_t hdr_bytes,
                       const void *d_layer, size_t layer_bytes,
                       void *d_out, size_t out_bytes,
                       uint32_t *d_status, void *stream);

/* Bytes of the work area of k3huf_decode_layer_ws. */
#define K3HUF_WORK_BYTES 68

/* k3huf_decode_layer with a work area that spreads the end of each launch
 * over all CTAs.  Not from the article: its decoder is a scalar loop per
 * stripe.  With fixed item ranges the launch ends with the CTAs whose items
 * were heaviest; here the last sixteenth of every CTA's range goes to the
 * pool of the CTAs whose ranges end in the same code table.  CTAs draw from
 * their own pool once their own items are taken, then from any pool with
 * items left, rebuilding their tables for it.  Containers without the
 * default 4096 / 256 chunk and sub-stream sizes, and launches of more than
 * 160 CTAs or 16 pools, decode as k3huf_decode_layer does.
 *  d_work / work_bytes: device memory, 4-byte aligned, >= K3HUF_WORK_BYTES,
 *    all zero before the first call; every launch leaves it zero.  The
 *    caller owns it and must not give it to two launches that may run at
 *    the same time (on two streams, or in graphs that may run together).
 *  Other arguments as for k3huf_decode_layer; the output is the same bytes.
 * Errors: K3HUF_E_ARG for a null, unaligned or short work area, else as
 * k3huf_decode_layer. */
int k3huf_decode_layer_ws(const void *h_layer_hdr, size_t hdr_bytes,
                          const void *d_layer, size_t layer_bytes,
                          void *d_out, size_t out_bytes,
                          uint32_t *d_status, void *d_work, size_t work_bytes, void *stream);

/* Flag of k3huf_decode_layer_ex: the launch may start early. */
#define K3HUF_DECODE_EARLY_START 1u

/* k3huf_decode_layer_ws with options; not from the article (its decoder
 * runs one call at a time).
 *  d_work / work_bytes: as for k3huf_decode_layer_ws, or d_work NULL (and
 *    work_bytes ignored) to decode as k3huf_decode_layer does;
 *  flags: 0 or K3HUF_DECODE_EARLY_START.  With that flag the kernels are
 *    launched with programmatic stream serialisation: a kernel's CTAs may
 *    start while the kernel before it in the stream is still running, take
 *    the SMs it frees, read the container, build their code tables and
 *    decode their first values into shared memory there; their first write
 *    to global memory (status, output) and their first access to the work
 *    area wait until that kernel has completed.  The caller guarantees that the
 *    kernel before this call in the stream does not write the container
 *    (d_layer); copies, event waits and kernels of other streams order the
 *    call as usual.  Back-to-back layer decodes, or a decode after the
 *    kernels that consume the previous layer, meet this.
 *  Other arguments as for k3huf_decode_layer_ws; the output is the same
 *  bytes.
 * Errors: K3HUF_E_ARG for an unknown flag or, when d_work is not NULL, an
 * unaligned or short work area; else as k3huf_decode_layer. */
int k3huf_decode_layer_ex(const void *h_layer_hdr, size_t hdr_bytes,
                          const void *d_layer, size_t layer_bytes,
                          void *d_out, size_t out_bytes,
                          uint32_t *d_status, void *d_work, size_t work_bytes,
                          uint32_t flags, void *stream);

/* Decode one tensor of a layer: its stripes only, in one launch (per
 * launch of up to 64 stripes), for a caller that decodes each weight just
 * before it is used.
 *  tensor: index in the layer's tensor directory;
 *  d_out / out_bytes: device, 16-byte aligned, at least 2 x the tensor's
 *    values; receives the tensor's bf16 bytes from offset 0 (not at the
 *    tensor's offset in the layer's output);
 *  other arguments as for k3huf_decode_layer_ex (work area, flags, stream;
 *    d_layer is the whole layer's container, as parsed from h_layer_hdr).
 * Errors: K3HUF_E_ARG for a tensor index out of range or a short output,
 * else as k3huf_decode_layer_ex. */
int k3huf_decode_tensor(const void *h_layer_hdr, size_t hdr_bytes,
                        const void *d_layer, size_t layer_bytes, uint32_t tensor,
                        void *d_out, size_t out_bytes,
                        uint32_t *d_status, void *d_work, size_t work_bytes,
                        uint32_t flags, void *stream);

/* Decode one stripe on the GPU (the article's per-stripe decode).
 *  codelen: host copy of the stripe's table (validated with k3huf_build);
 *  chunk_syms, sub_syms: values per indexed chunk and per sub-stream, as
 *    in the layer header;
 *  d_stripe / stripe_bytes: the stripe in device memory, from its header;
 *  n_values: values in the stripe (<= 2^25); d_out receives 2 n_values
 *  bytes of bf16.  The kernel checks the device-side stripe header against
 *  n_values / chunk_syms / stripe_bytes and sets K3HUF_ST_HEADER if they
 *  disagree. */
int k3huf_decode_stripe(const uint8_t codelen[256], uint32_t chunk_syms, uint32_t sub_syms,
                        const void *d_stripe, size_t stripe_bytes,
                        uint32_t n_values, void *d_out,
                        uint32_t *d_status, void *stream);

/* Select the decode kernel variant for later decode calls in this process:
 * the number of codes every table lookup of the lockstep decoder emits.
 * 0 = default (2), 1 = one code per lookup (the article's shelved
 * decoder's scheme), 2 = the article's double-symbol table (section
 * 如果将来重启): two codes per lookup when both fit in the 12-bit window,
 * otherwise the two codes are read one at a time.  All give identical
 * output.  Returns K3HUF_E_ARG for any other value. */
int k3huf_set_decoder_variant(int variant);

/* Pack-time encoder (host, multi-threaded), producing the container above
 * byte for byte as specified: per table, the histogram of the high bytes,
 * Huffman code lengths from a min-heap keyed (count, id) with leaves
 * id = symbol and internal nodes 256 + creation order (one used symbol gets
 * length 1), the 12-bit limit (clamp, then while the Kraft sum exceeds 4096
 * lengthen the code of lowest count among those shorter than 12, ties to
 * the larger symbol), the canonical assignment of k3huf_build.
 *  h_tensors[t]: n_values[t] (>= 1) little-endian bf16 values;
 *  chunk_syms: values per indexed chunk (>= 1);
 *  sub_syms: values per sub-stream of a chunk (a divisor of chunk_syms;
 *    0, a non-divisor, or chunk_syms * 12 > 65535 give one sub-stream);
 *  shared_table: nonzero = one table for the whole layer, else one per tensor;
 *  n_threads: worker threads (0 = hardware concurrency);
 *  h_blob / blob_cap: output; with h_blob NULL only *blob_bytes is set. */
int k3huf_encode_layer(uint32_t n_tensors, const void *const *h_tensors, const uint64_t *n_values,
                       uint32_t chunk_syms, uint32_t sub_syms, int shared_table, int n_threads,
                       void *h_blob, size_t blob_cap, size_t *blob_bytes);

/* Decode fused into its consumer: y[r] += sum_c W[r][c] * x[c] for tensor
 * `tensor` of the layer read as a row-major matrix of `cols` columns, with
 * the weights decoded on chip and never written to device memory.  The
 * article "Kimi K3 纯 CPU 推理中的无损 Trunk 压缩" (section 背景) streams
 * the trunk to feed matrix-vector products; the ECF8 article ("1. 指数集中
 * 现象", its PyTorch hook) decodes into a bf16 buffer and then copies it into
 * the weight; here the decoded values go straight into fp32 dot products.
 *  d_layer: as for k3huf_decode_layer; d_x: device, 16-byte aligned, cols
 *    bf16 values; d_y: device, 4-byte aligned, n_values / cols floats,
 *    accumulated (zero it for y = W x); atomic fp32 additions, so the
 *    summation order, and the last bits, vary from run to run.
 *  Needs: cols divides the tensor's values and is a multiple of 32 x
 *    sub_syms (every work item lies in one row), sub_syms a multiple of 8
 *    with 32 / (chunk_syms / sub_syms) whole, and sub-streams short enough
 *    to stage (sub_syms x 12 / 8 + 64 <= 5056, so sub_syms <= 2048 for
 *    powers of two): K3HUF_E_ARG otherwise.
 * Asynchronous on `stream`; stream faults set bits in *d_status. */
int k3huf_gemv_layer(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer, size_t layer_bytes,
                     uint32_t tensor, uint64_t cols, const void *d_x, float *d_y, uint32_t *d_status, void *stream);

/* Flag of k3huf_gemv_layer_ex: y is set to zero first (y = W x). */
#define K3HUF_GEMV_ZERO_Y 2u

/* k3huf_gemv_layer with options; not from the articles.
 *  flags: any of
 *   K3HUF_GEMV_ZERO_Y: a kernel of the call sets the n_values / cols
 *     floats of d_y to zero first, so the call computes y = W x;
 *   K3HUF_DECODE_EARLY_START: the call's kernels are launched with
 *     programmatic stream serialisation, as k3huf_decode_layer_ex does: the
 *     GEMV's CTAs may start, read the container and build their tables on
 *     the SMs the kernel before them frees, and their first global write
 *     (y, status) waits until that kernel has completed.  With both flags
 *     the zeroing kernel waits for the kernel before it and the GEMV for the
 *     zeroing, so back-to-back calls overlap one call's table build with
 *     the previous call's end.  The caller guarantees that the kernel
 *     before the call in the stream does not write the container (x is
 *     read only after that kernel has completed).
 *  Other arguments, requirements and errors as for k3huf_gemv_layer;
 *  K3HUF_E_ARG for an unknown flag. */
int k3huf_gemv_layer_ex(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer, size_t layer_bytes,
                        uint32_t tensor, uint64_t cols, const void *d_x, float *d_y, uint32_t *d_status,
                        uint32_t flags, void *stream);

/* Y += W X for n_vec vectors at once, W decoded on chip once for all of
 * them; not from the articles (their consumer copies decoded weights into
 * a framework tensor).  d_x: n_vec bf16 vectors of cols values, back to back
 * (vector b at d_x + 2 * b * cols bytes, 16-byte aligned); d_y: n_vec fp32
 * vectors of rows = n_values / cols entries, back to back (vector b at
 * d_y + b * rows).  n_vec is 1, 2, 4 or 8; above 1 the layer must use the
 * default chunk and sub-stream sizes (4096 / 256) and the default decoder
 * (two codes per lookup).  Flags as for k3huf_gemv_layer_ex
 * (K3HUF_GEMV_ZERO_Y zeroes all n_vec vectors of Y first).  Other arguments,
 * requirements and errors as for k3huf_gemv_layer; K3HUF_E_ARG for another
 * n_vec or layout. */
int k3huf_gemv_layer_batch(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer, size_t layer_bytes,
                           uint32_t tensor, uint64_t cols, const void *d_x, uint32_t n_vec, float *d_y,
                           uint32_t *d_status, uint32_t flags, void *stream);

/* GPU encoder: the same container as k3huf_encode_layer (byte for byte),
 * built from bf16 tensors already in device memory.  The article "Kimi K3
 * 纯 CPU 推理中的无损 Trunk 压缩" (section 已实现的部分) packs offline:
 * high-byte histogram, 12-bit-capped Huffman lengths, canonical
 * longest-first codes, MSB-first bit packing per stripe, low bytes raw.
 * Here the passes over the values (histogram, bit counts, packing, low-byte
 * copy) run on the GPU.  With the default chunk and sub-stream sizes (4096
 * and 256) the code lengths, codes and layout are decided on the GPU too,
 * with the CPU encoder's choices (ties included); with any other sizes on
 * the host, between the passes, with the CPU encoder's own functions.
 *  d_tensors[t]: device, 16-byte aligned, n_values[t] (>= 1) bf16 values;
 *  chunk_syms, sub_syms, shared_table: as for k3huf_encode_layer;
 *  d_scratch: device, 256-byte aligned, scratch_bytes >=
 *    k3huf_encode_scratch_bytes(...) (contents need not be initialised);
 *  d_blob: device, 256-byte aligned, blob_cap bytes; with d_blob NULL only
 *    *blob_bytes is set (the histogram pass still runs).  A buffer of
 *    k3huf_encode_bound(...) bytes always suffices, so one call encodes;
 *    the container fills its first *blob_bytes bytes.
 * Synchronises `stream` once, at the end, with the default sizes (twice
 * with others: after the histograms too) and returns when the container is
 * complete.  With the default sizes the first call on a host thread
 * allocates a 256 KB page-locked host buffer that the thread keeps for its
 * later calls (the call's one upload and its outcome; like any page-locked
 * allocation, that first one may synchronise the device).  K3HUF_E_ARG on a bad argument or a short buffer (nothing is
 * written to d_blob then; *blob_bytes is still set), K3HUF_E_FORMAT if the
 * packed bits disagree with the planned layout (an internal check),
 * K3HUF_E_CUDA on a CUDA error. */
int k3huf_encode_scratch_bytes(uint32_t n_tensors, const uint64_t *n_values, uint32_t chunk_syms,
                               uint32_t sub_syms, int shared_table, size_t *scratch_bytes);
/* Upper bound of the container's size for any values of these sizes: the
 * layout when every code has the limit's 12 bits (host, pure; allocates
 * nothing on the device).  Arguments as for k3huf_encode_layer_gpu;
 * K3HUF_E_ARG for an empty layer, a zero size or a null output. */
int k3huf_encode_bound(uint32_t n_tensors, const uint64_t *n_values, uint32_t chunk_syms, uint32_t sub_syms,
                       int shared_table, size_t *blob_bytes);
int k3huf_encode_layer_gpu(uint32_t n_tensors, const void *const *d_tensors, const uint64_t *n_values,
                           uint32_t chunk_syms, uint32_t sub_syms, int shared_table, void *d_scratch,
                           size_t scratch_bytes, void *d_blob, size_t blob_cap, size_t *blob_bytes, void *stream);

/* The GPU encoder without a scratch argument, for callers that may not
 * allocate device memory themselves: for example a plugin or custom operator
 * whose host framework hands it its inputs and outputs and owns the rest of
 * the GPU's memory, where a cudaMalloc of its own could fail or synchronise
 * the device in the middle of the framework's work.  The pages have no
 * counterpart: they encode offline on the CPU.
 * Its scratch is a fixed 32 MiB array inside the library, held by every GPU
 * that loads the library until the process exits; a layer whose
 * k3huf_encode_scratch_bytes exceeds 32 MiB (about 8.6 x 10^9 values in
 * 4096-value chunks: 16 bytes of scratch per chunk) is refused with K3HUF_E_ARG.  Arguments, output and
 * errors otherwise as k3huf_encode_layer_gpu; nothing is allocated on the
 * device, and no page-locked host memory either.  The first call on a device looks up the array's address on that
 * device (make that first call before any stream capture).  The array used
 * is the current device's copy, so every tensor, the output and the stream
 * must belong to the current device: a host pointer, another device's
 * pointer or another device's stream is refused with K3HUF_E_ARG before
 * any work is issued.  All calls share the one array: calls whose work
 * overlaps on the GPU (other streams, other host threads) race and must be
 * serialised by the caller. */
int k3huf_encode_layer_gpu_noalloc(uint32_t n_tensors, const void *const *d_tensors, const uint64_t *n_values,
                                   uint32_t chunk_syms, uint32_t sub_syms, int shared_table, void *d_blob,
                                   size_t blob_cap, size_t *blob_bytes, void *stream);

/* Streaming ring: layers held in pinned host memory are copied to device
 * slots with cudaMemcpyAsync on a copy stream while the previous layer is
 * decoded on a compute stream, double buffered.  The kimi-k3-in-c tuning
 * article (section 2.2) gives its trunk ring a second slot so that reading
 * the next layer overlaps computing on the current one.
 * k3huf_ring_create allocates n_slots device slots of slot_bytes each and
 * the streams/events it needs. */
typedef struct k3huf_ring k3huf_ring;

typedef struct {
    float total_ms;      /* first copy issued -> last decode finished */
    float decode_ms;     /* sum of the decode kernels' event times */
    float copy_ms;       /* sum of the copies' event times */
    uint64_t h2d_bytes;  /* bytes copied host -> device */
    uint64_t out_bytes;  /* bytes decoded */
} k3huf_ring_stats_t;

int k3huf_ring_create(size_t slot_bytes, int n_slots, k3huf_ring **ring);
/* Decode n_layers containers h_layers[i] (pinned host memory, layer_bytes[i]
 * bytes each, <= slot_bytes) into d_outs[i] (out_bytes[i] each).  Blocks
 * until all work is done; fills *stats when non-NULL. */
int k3huf_ring_run(k3huf_ring *ring, int n_layers, const void *const *h_layers, const size_t *layer_bytes,
                   void *const *d_outs, const size_t *out_bytes, uint32_t *d_status,
                   k3huf_ring_stats_t *stats);
int k3huf_ring_destroy(k3huf_ring *ring);

/* Storage feed: containers read from a file straight into the ring's pinned
 * host slots, then copied and decoded as above.  The article "Kimi K3 纯
 * CPU 推理中的无损 Trunk 压缩" (section 让方案被搁置的测量) sets the
 * decoder against a 3 GB/s SSD that streams the trunk; the article
 * "AIBit-探索开源项目" (section 工作原理：架构, 读取检查点) reads the
 * checkpoint with O_DIRECT, bypassing the page cache; the article "Kimi K3
 * 极限部署技术解析：Deltafin 如何在 M1 Max 上运行 2.8T 参数模型" (section
 * 5.1) reads the next layer on a background thread and contiguous byte
 * spans with parallel pread calls.  This feed does both: one file descriptor opened with
 * O_DIRECT where the filesystem allows it (else buffered), each read split
 * into 8 MiB pieces read by n_threads threads with pread. */
typedef struct k3huf_feed k3huf_feed;

/* Open path read-only (O_DIRECT when the filesystem accepts it).
 * n_threads: reader threads per read call (1..64).  K3HUF_E_IO when the
 * file cannot be opened. */
int k3huf_feed_open(const char *path, int n_threads, k3huf_feed **feed);
/* 1 when reads bypass the page cache (O_DIRECT), 0 when buffered, or
 * K3HUF_E_ARG. */
int k3huf_feed_direct(const k3huf_feed *feed);
/* Read bytes [offset, offset + bytes) of the file into h_buf.  offset and
 * h_buf must be 4096-byte aligned and buf_bytes >= bytes rounded up to 4096
 * (the read covers whole 4 KiB blocks; bytes past the end of the file are
 * left as they were).  Blocks until done.  K3HUF_E_ARG on a bad argument,
 * K3HUF_E_IO when a read fails or the file ends before offset + bytes. */
int k3huf_feed_read(k3huf_feed *feed, uint64_t offset, size_t bytes, void *h_buf, size_t buf_bytes);
int k3huf_feed_close(k3huf_feed *feed);

/* A ring that also owns n_slots pinned host slots (slot_bytes rounded up to
 * 4096 each) for k3huf_ring_run_file. */
int k3huf_ring_create_staged(size_t slot_bytes, int n_slots, k3huf_ring **ring);

typedef struct {
    float total_ms;      /* host wall time, first read issued -> last decode finished */
    float read_ms;       /* host time spent in the file reads */
    float copy_ms;       /* sum of the host -> device copies' event times */
    float decode_ms;     /* sum of the decode kernels' event times */
    uint64_t read_bytes; /* container bytes read from the file */
    uint64_t out_bytes;  /* bytes decoded */
} k3huf_feed_stats_t;

/* Decode n_layers containers stored in the feed's file at file_offsets[i]
 * (4096-byte aligned), layer_bytes[i] bytes each (<= slot_bytes), into
 * d_outs[i].  Layer i+1 is read into the next host slot while layer i is
 * copied and decoded; a host slot is reused once its copy has finished and
 * a device slot once its decode has finished.  Needs a staged ring.
 * Blocks until done; fills *stats when non-NULL. */
int k3huf_ring_run_file(k3huf_ring *ring, k3huf_feed *feed, int n_layers, const uint64_t *file_offsets,
                        const size_t *layer_bytes, void *const *d_outs, const size_t *out_bytes, uint32_t *d_status,
                        k3huf_feed_stats_t *stats);

/* Last CUDA error code seen by this library on the calling thread. */
int k3huf_last_cuda_error(void);
/* Static description of a K3HUF_E_* code. */
const char *k3huf_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* K3HUF_H */
