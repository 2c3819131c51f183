// Internal declarations shared by the host library and the CUDA decode /
// ring translation units (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "k3huf.h"

namespace k3huf {

struct TensorEntry {
    uint32_t table, first_stripe, n_stripes;
    uint64_t n_values, out_offset;
};

struct StripeEntry {
    uint64_t blob_offset, stripe_bytes, out_offset;
    uint32_t n_values, table;
};

struct Layer {
    k3huf_layer_info_t info{};
    const uint8_t *tables = nullptr;   // host copy, n_tables x 256 code lengths
    std::vector<TensorEntry> tensors;
    std::vector<StripeEntry> stripes;
};

// Parse and validate a host copy of a layer header (see k3huf_layer_info).
int parse_layer(const void *h_layer, size_t bytes, Layer *out);

// Little-endian field access (both supported hosts are little-endian, but
// the container's byte order is fixed, so read it byte by byte).
inline uint32_t rd16(const uint8_t *p) { return uint32_t(p[0]) | (uint32_t(p[1]) << 8); }
inline uint32_t rd32(const uint8_t *p) {
    return uint32_t(p[0]) | (uint32_t(p[1]) << 8) | (uint32_t(p[2]) << 16) | (uint32_t(p[3]) << 24);
}
inline uint64_t rd64(const uint8_t *p) { return uint64_t(rd32(p)) | (uint64_t(rd32(p + 4)) << 32); }
inline void wr16(uint8_t *p, uint32_t v) { p[0] = uint8_t(v); p[1] = uint8_t(v >> 8); }
inline void wr32(uint8_t *p, uint32_t v) {
    p[0] = uint8_t(v); p[1] = uint8_t(v >> 8); p[2] = uint8_t(v >> 16); p[3] = uint8_t(v >> 24);
}
inline void wr64(uint8_t *p, uint64_t v) { wr32(p, uint32_t(v)); wr32(p + 4, uint32_t(v >> 32)); }

constexpr uint32_t kLayerMagic = 0x4648334Bu;   // "K3HF"
constexpr uint32_t kStripeMagic = 0x5348334Bu;  // "K3HS"
constexpr uint32_t kBitsSlack = 32;             // zero bytes after each padded bit stream

inline uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// Sub-streams per chunk actually used for a requested size (see k3huf.h).
inline uint32_t effective_sub_syms(uint32_t chunk_syms, uint32_t sub_syms) {
    if (sub_syms == 0 || chunk_syms % sub_syms != 0 || uint64_t(chunk_syms) * K3HUF_MAXLEN > 65535u)
        return chunk_syms;
    return sub_syms;
}

// Bytes of a stripe's chunk index plus sub-stream index.
inline uint64_t index_bytes(uint64_t n_chunks, uint32_t chunk_syms, uint32_t sub_syms) {
    return 4 * n_chunks + 2 * n_chunks * (chunk_syms / sub_syms - 1);
}

// Record a CUDA error code for k3huf_last_cuda_error (thread-local).
void set_cuda_error(int code);

// --- code construction (host) ---------------------------------------------
// Canonical longest-first codes of a length vector (0 = unused symbol).
void canonical_codes(const uint8_t len[256], uint32_t code[256], uint32_t first[K3HUF_MAXLEN + 1],
                     uint32_t count[K3HUF_MAXLEN + 1]);
// Huffman code lengths of symbol counts, ties on (count, id).
void huffman_depths(const uint64_t cnt[256], int depth[256]);
// Cap the lengths at 12 bits (clamp, then lengthen the rarest shorter code
// while the Kraft sum is over-full).
void limit_depths(const uint64_t cnt[256], int depth[256]);

// --- container layout, shared by the CPU and GPU encoders -------------------
struct PlanStripe {
    uint32_t tensor, table;
    uint64_t v0, n;                // first value within the tensor, values
    uint64_t blob_offset, stripe_bytes, out_offset, huff_bits;
    uint32_t n_chunks, bits_offset, even_offset;
};

struct LayerPlan {
    uint32_t n_tensors = 0, n_tables = 0, chunk_syms = 0, sub_syms = 0;
    bool shared_table = false;
    std::vector<uint64_t> n_values, tensor_out;
    std::vector<PlanStripe> stripes;
    std::vector<uint8_t> codelen;  // n_tables x 256
    uint64_t raw = 0, out = 0, hdr = 0, total = 0;
};

// The layer's stripes (64 MiB of values each, per tensor, in order).
void plan_stripes(uint32_t n_tensors, const uint64_t *n_values, uint32_t chunk_syms, uint32_t sub_syms,
                  bool shared_table, LayerPlan &L);
// Code lengths from per-stripe high-byte histograms (stripes x 256), then
// every stripe's bit count, offsets and size.
void plan_layout(const uint64_t *stripe_hist, LayerPlan &L);
// Header size, then every stripe's offsets and size from its huff_bits.
void place_stripes(LayerPlan &L);
// Container size when every code is K3HUF_MAXLEN bits: no values give more.
uint64_t layout_bound(LayerPlan L);
// Bytes [0, L.hdr): layer header, code tables, tensor and stripe directories.
void write_layer_header(const LayerPlan &L, uint8_t *blob);
// The 32-byte stripe header.
void write_stripe_header(const PlanStripe &p, uint8_t *dst);

}  // namespace k3huf
