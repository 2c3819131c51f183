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

}  // namespace k3huf
