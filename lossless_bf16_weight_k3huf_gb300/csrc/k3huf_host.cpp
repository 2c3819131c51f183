// Host side of the k3_huf codec: table build and Kraft check, container
// header validation, and the multi-threaded pack-time encoder.
//
// Method: article "Kimi K3 纯 CPU 推理中的无损 Trunk 压缩：一次被解码速度判死刑
// 的 Huffman 压缩实验" -- section 核心思想 (code only the high byte of each
// bf16 value, keep the low byte raw), section 已实现的部分 (layer header
// with codelen[256], 64 MiB stripes, lengths capped at 12 bits, a
// 4096-entry (symbol << 4) | length table), section 规范码分配与 Kraft 校验
// (Kraft check, longest-first canonical codes, Huffman depths with a
// BZip2-style length correction).
#include <algorithm>
#include <atomic>
#include <cstring>
#include <new>
#include <queue>
#include <thread>
#include <vector>

#include "k3huf_internal.h"

namespace k3huf {
namespace {

constexpr int kMaxLen = K3HUF_MAXLEN;
constexpr uint32_t kSpace = 1u << kMaxLen;   // Kraft units of a full 12-bit code space

// Run fn(i) for i in [0, n) on up to `threads` workers.
template <class F>
void parallel_for(size_t n, int threads, F fn) {
    if (n == 0) return;
    int t = std::max(1, std::min<int>(threads, int(n)));
    if (t == 1) {
        for (size_t i = 0; i < n; ++i) fn(i);
        return;
    }
    std::atomic<size_t> next{0};
    std::vector<std::thread> pool;
    pool.reserve(t);
    for (int k = 0; k < t; ++k)
        pool.emplace_back([&] {
            for (size_t i = next.fetch_add(1); i < n; i = next.fetch_add(1)) fn(i);
        });
    for (auto &th : pool) th.join();
}

}  // namespace

// Canonical longest-first code of a length vector (lengths 0 = unused).
// Returns the code of every used symbol in code[]; first[]/count[] per length.
void canonical_codes(const uint8_t len[256], uint32_t code[256], uint32_t first[kMaxLen + 1],
                     uint32_t count[kMaxLen + 1]) {
    for (int l = 0; l <= kMaxLen; ++l) count[l] = 0;
    for (int s = 0; s < 256; ++s) count[len[s]]++;
    uint32_t next = 0;
    for (int l = kMaxLen; l >= 1; --l) {
        first[l] = next;
        next = (next + count[l] + 1) >> 1;   // rounding up keeps incomplete codes prefix-free
    }
    uint32_t cursor[kMaxLen + 1];
    for (int l = 1; l <= kMaxLen; ++l) cursor[l] = first[l];
    for (int s = 0; s < 256; ++s) code[s] = len[s] ? cursor[len[s]]++ : 0;
}

// Kraft check of a code length table; the Kraft sum in 2^-12 units in *kraft.
int check_table(const uint8_t codelen[256], uint32_t *kraft) {
    uint32_t k = 0;
    for (int s = 0; s < 256; ++s) {
        if (codelen[s] > kMaxLen) return K3HUF_E_BADLEN;
        if (codelen[s]) k += kSpace >> codelen[s];
    }
    if (kraft) *kraft = k;
    if (k == 0) return K3HUF_E_EMPTY;
    if (k > kSpace) return K3HUF_E_OVERSUB;
    return K3HUF_OK;
}

// Huffman code lengths (leaf depths), ties resolved on (count, id) with
// leaves id = symbol and internal nodes 256 + creation order.
void huffman_depths(const uint64_t cnt[256], int depth[256]) {
    struct Node {
        uint64_t w;
        uint32_t id;
    };
    auto later = [](const Node &a, const Node &b) { return a.w > b.w || (a.w == b.w && a.id > b.id); };
    std::priority_queue<Node, std::vector<Node>, decltype(later)> heap(later);
    for (int s = 0; s < 256; ++s) {
        depth[s] = 0;
        if (cnt[s]) heap.push({cnt[s], uint32_t(s)});
    }
    if (heap.size() == 1) {            // a lone symbol still needs a 1-bit code
        depth[heap.top().id] = 1;
        return;
    }
    if (heap.empty()) return;
    // children of internal node 256 + k
    std::vector<uint32_t> kid0, kid1;
    while (heap.size() > 1) {
        Node a = heap.top(); heap.pop();
        Node b = heap.top(); heap.pop();
        uint32_t id = 256 + uint32_t(kid0.size());
        kid0.push_back(a.id);
        kid1.push_back(b.id);
        heap.push({a.w + b.w, id});
    }
    // walk from the root (the last node created) down
    std::vector<int> d(256 + kid0.size(), 0);
    for (size_t k = kid0.size(); k-- > 0;) {
        int dk = d[256 + k];
        d[kid0[k]] = dk + 1;
        d[kid1[k]] = dk + 1;
    }
    for (int s = 0; s < 256; ++s)
        if (cnt[s]) depth[s] = d[s];
}

// Cap at 12 bits: clamp, then lengthen the lowest-count code shorter than 12
// (ties to the larger symbol) while the Kraft sum is over-full.
void limit_depths(const uint64_t cnt[256], int depth[256]) {
    uint64_t k = 0;
    for (int s = 0; s < 256; ++s) {
        if (!cnt[s]) continue;
        depth[s] = std::min(depth[s], kMaxLen);
        k += uint64_t(kSpace) >> depth[s];
    }
    while (k > kSpace) {
        int pick = -1;
        for (int s = 255; s >= 0; --s) {
            if (!cnt[s] || depth[s] >= kMaxLen) continue;
            if (pick < 0 || cnt[s] < cnt[pick]) pick = s;   // scanning down keeps the larger symbol on ties
        }
        if (pick < 0) break;
        k -= uint64_t(kSpace) >> (depth[pick] + 1);          // 2^(12-l) -> 2^(11-l)
        depth[pick] += 1;
    }
}

// ---------------------------------------------------------------------------
// container layout, shared by the CPU and GPU encoders

void plan_stripes(uint32_t n_tensors, const uint64_t *n_values, uint32_t chunk_syms, uint32_t sub_syms,
                  bool shared_table, LayerPlan &L) {
    L.n_tensors = n_tensors;
    L.n_tables = shared_table ? 1u : n_tensors;
    L.chunk_syms = chunk_syms;
    L.sub_syms = sub_syms;
    L.shared_table = shared_table;
    L.n_values.assign(n_values, n_values + n_tensors);
    L.tensor_out.assign(n_tensors, 0);
    L.stripes.clear();
    L.out = L.raw = 0;
    for (uint32_t t = 0; t < n_tensors; ++t) {
        L.out = align_up(L.out, 256);
        L.tensor_out[t] = L.out;
        for (uint64_t v0 = 0; v0 < n_values[t]; v0 += K3HUF_STRIPE_VALUES) {
            PlanStripe p{};
            p.tensor = t;
            p.table = shared_table ? 0u : t;
            p.v0 = v0;
            p.n = std::min<uint64_t>(K3HUF_STRIPE_VALUES, n_values[t] - v0);
            p.out_offset = L.out + 2 * v0;
            p.n_chunks = uint32_t((p.n + chunk_syms - 1) / chunk_syms);
            L.stripes.push_back(p);
        }
        L.out += 2 * n_values[t];
        L.raw += 2 * n_values[t];
    }
}

void plan_layout(const uint64_t *stripe_hist, LayerPlan &L) {
    L.codelen.assign(256ull * L.n_tables, 0);
    for (uint32_t tb = 0; tb < L.n_tables; ++tb) {
        uint64_t cnt[256] = {};
        for (size_t i = 0; i < L.stripes.size(); ++i)
            if (L.stripes[i].table == tb)
                for (int s = 0; s < 256; ++s) cnt[s] += stripe_hist[256 * i + s];
        int depth[256];
        huffman_depths(cnt, depth);
        limit_depths(cnt, depth);
        for (int s = 0; s < 256; ++s) L.codelen[256ull * tb + s] = uint8_t(depth[s]);
    }
    for (size_t i = 0; i < L.stripes.size(); ++i) {
        PlanStripe &p = L.stripes[i];
        const uint8_t *cl = &L.codelen[256ull * p.table];
        uint64_t bits = 0;
        for (int s = 0; s < 256; ++s) bits += stripe_hist[256 * i + s] * cl[s];
        p.huff_bits = bits;
    }
    place_stripes(L);
}

void place_stripes(LayerPlan &L) {
    L.hdr = align_up(K3HUF_LAYER_HDR_BYTES + 256ull * L.n_tables + 32ull * L.n_tensors + 32ull * L.stripes.size(), 256);
    uint64_t pos = L.hdr;
    for (size_t i = 0; i < L.stripes.size(); ++i) {
        PlanStripe &p = L.stripes[i];
        p.bits_offset = uint32_t(align_up(K3HUF_STRIPE_HDR_BYTES + index_bytes(p.n_chunks, L.chunk_syms, L.sub_syms), 16));
        p.even_offset = uint32_t(p.bits_offset + align_up((p.huff_bits + 7) / 8, 16) + kBitsSlack);
        p.stripe_bytes = p.even_offset + align_up(p.n, 16);
        pos = align_up(pos, 256);
        p.blob_offset = pos;
        pos += p.stripe_bytes;
    }
    L.total = pos;
}

uint64_t layout_bound(LayerPlan L) {
    for (PlanStripe &p : L.stripes) p.huff_bits = uint64_t(K3HUF_MAXLEN) * p.n;
    place_stripes(L);
    return L.total;
}

void write_layer_header(const LayerPlan &L, uint8_t *blob) {
    std::memset(blob, 0, L.hdr);
    wr32(blob + 0, kLayerMagic);
    wr16(blob + 4, K3HUF_FORMAT_VERSION);
    wr16(blob + 6, K3HUF_MAXLEN);
    wr32(blob + 8, L.chunk_syms);
    wr32(blob + 12, L.n_tables);
    wr32(blob + 16, L.n_tensors);
    wr32(blob + 20, uint32_t(L.stripes.size()));
    wr64(blob + 24, L.raw);
    wr64(blob + 32, L.total);
    wr32(blob + 40, K3HUF_STRIPE_VALUES);
    wr32(blob + 44, uint32_t(L.hdr));
    wr64(blob + 48, L.out);
    wr32(blob + 56, L.sub_syms);
    std::memcpy(blob + K3HUF_LAYER_HDR_BYTES, L.codelen.data(), L.codelen.size());
    uint8_t *td = blob + K3HUF_LAYER_HDR_BYTES + 256ull * L.n_tables;
    uint8_t *sd = td + 32ull * L.n_tensors;
    uint32_t sid = 0;
    for (uint32_t t = 0; t < L.n_tensors; ++t) {
        const uint32_t ns = uint32_t((L.n_values[t] + K3HUF_STRIPE_VALUES - 1) / K3HUF_STRIPE_VALUES);
        uint8_t *e = td + 32ull * t;
        wr32(e + 0, L.shared_table ? 0u : t);
        wr32(e + 4, sid);
        wr32(e + 8, ns);
        wr32(e + 12, 0);
        wr64(e + 16, L.n_values[t]);
        wr64(e + 24, L.tensor_out[t]);
        sid += ns;
    }
    for (size_t i = 0; i < L.stripes.size(); ++i) {
        const PlanStripe &p = L.stripes[i];
        uint8_t *e = sd + 32 * i;
        wr64(e + 0, p.blob_offset);
        wr64(e + 8, p.stripe_bytes);
        wr64(e + 16, p.out_offset);
        wr32(e + 24, uint32_t(p.n));
        wr32(e + 28, p.table);
    }
}

void write_stripe_header(const PlanStripe &p, uint8_t *st) {
    std::memset(st, 0, K3HUF_STRIPE_HDR_BYTES);
    wr32(st + 0, kStripeMagic);
    wr32(st + 4, p.table);
    wr32(st + 8, uint32_t(p.n));
    wr32(st + 12, p.n_chunks);
    wr64(st + 16, p.huff_bits);
    wr32(st + 24, p.bits_offset);
    wr32(st + 28, p.even_offset);
}

// ---------------------------------------------------------------------------
// header validation

int parse_layer(const void *h_layer, size_t bytes, Layer *L) {
    const uint8_t *p = static_cast<const uint8_t *>(h_layer);
    if (!p || !L) return K3HUF_E_ARG;
    if (bytes < K3HUF_LAYER_HDR_BYTES) return K3HUF_E_FORMAT;
    if (rd32(p) != kLayerMagic || rd16(p + 4) != K3HUF_FORMAT_VERSION || rd16(p + 6) != K3HUF_MAXLEN)
        return K3HUF_E_FORMAT;
    k3huf_layer_info_t in{};
    in.chunk_syms = rd32(p + 8);
    in.n_tables = rd32(p + 12);
    in.n_tensors = rd32(p + 16);
    in.n_stripes = rd32(p + 20);
    in.raw_bytes = rd64(p + 24);
    in.blob_bytes = rd64(p + 32);
    in.stripe_values = rd32(p + 40);
    in.hdr_bytes = rd32(p + 44);
    in.out_bytes = rd64(p + 48);
    in.sub_syms = rd32(p + 56);
    if (in.chunk_syms == 0 || in.n_tables == 0 || in.n_tensors == 0 || in.n_stripes == 0 ||
        in.stripe_values != K3HUF_STRIPE_VALUES || in.hdr_bytes % 256 != 0 || in.sub_syms == 0 ||
        effective_sub_syms(in.chunk_syms, in.sub_syms) != in.sub_syms)
        return K3HUF_E_FORMAT;
    const uint64_t need = K3HUF_LAYER_HDR_BYTES + 256ull * in.n_tables + 32ull * in.n_tensors + 32ull * in.n_stripes;
    if (need > in.hdr_bytes || in.hdr_bytes > in.blob_bytes) return K3HUF_E_FORMAT;
    if (bytes < in.hdr_bytes) return K3HUF_E_FORMAT;
    const uint8_t *tables = p + K3HUF_LAYER_HDR_BYTES;
    for (uint32_t t = 0; t < in.n_tables; ++t) {
        int rc = check_table(tables + 256ull * t, nullptr);
        if (rc) return rc;
    }
    const uint8_t *td = tables + 256ull * in.n_tables;
    const uint8_t *sd = td + 32ull * in.n_tensors;
    std::vector<TensorEntry> tensors(in.n_tensors);
    std::vector<StripeEntry> stripes(in.n_stripes);
    uint64_t raw = 0, out_end = 0, blob_end = in.hdr_bytes;
    uint32_t sid = 0;
    for (uint32_t t = 0; t < in.n_tensors; ++t) {
        const uint8_t *e = td + 32ull * t;
        TensorEntry te{rd32(e), rd32(e + 4), rd32(e + 8), rd64(e + 16), rd64(e + 24)};
        if (te.table >= in.n_tables || te.first_stripe != sid || te.n_values == 0 ||
            te.n_stripes != (te.n_values + K3HUF_STRIPE_VALUES - 1) / K3HUF_STRIPE_VALUES ||
            te.out_offset % 256 != 0 || te.out_offset < out_end ||
            te.n_stripes > in.n_stripes - sid)
            return K3HUF_E_FORMAT;
        out_end = te.out_offset + 2 * te.n_values;
        if (out_end > in.out_bytes) return K3HUF_E_FORMAT;
        raw += 2 * te.n_values;
        for (uint32_t k = 0; k < te.n_stripes; ++k, ++sid) {
            const uint8_t *s = sd + 32ull * sid;
            StripeEntry se{rd64(s), rd64(s + 8), rd64(s + 16), rd32(s + 24), rd32(s + 28)};
            const uint64_t v0 = uint64_t(k) * K3HUF_STRIPE_VALUES;
            const uint64_t nv = std::min<uint64_t>(K3HUF_STRIPE_VALUES, te.n_values - v0);
            const uint64_t nch = (nv + in.chunk_syms - 1) / in.chunk_syms;
            const uint64_t min_bytes =
                align_up(K3HUF_STRIPE_HDR_BYTES + index_bytes(nch, in.chunk_syms, in.sub_syms), 16) + kBitsSlack + nv;
            if (se.n_values != nv || se.table != te.table || se.out_offset != te.out_offset + 2 * v0 ||
                se.blob_offset % 256 != 0 || se.blob_offset < blob_end || se.stripe_bytes % 16 != 0 ||
                se.stripe_bytes < min_bytes || se.stripe_bytes > in.blob_bytes - se.blob_offset ||
                se.blob_offset > in.blob_bytes)
                return K3HUF_E_FORMAT;
            blob_end = se.blob_offset + se.stripe_bytes;
            stripes[sid] = se;
        }
        tensors[t] = te;
    }
    if (sid != in.n_stripes || raw != in.raw_bytes) return K3HUF_E_FORMAT;
    L->info = in;
    L->tables = tables;
    L->tensors.swap(tensors);
    L->stripes.swap(stripes);
    return K3HUF_OK;
}

}  // namespace k3huf

using namespace k3huf;

extern "C" int k3huf_build(const uint8_t codelen[256], uint16_t sym_len[4096]) {
    if (!codelen) return K3HUF_E_ARG;
    int rc = check_table(codelen, nullptr);
    if (rc || !sym_len) return rc;
    uint32_t code[256], first[kMaxLen + 1], count[kMaxLen + 1];
    canonical_codes(codelen, code, first, count);
    std::memset(sym_len, 0, sizeof(uint16_t) * K3HUF_TABLE_ENTRIES);
    for (int s = 0; s < 256; ++s) {
        const int l = codelen[s];
        if (!l) continue;
        const uint32_t lo = code[s] << (kMaxLen - l), hi = (code[s] + 1) << (kMaxLen - l);
        for (uint32_t i = lo; i < hi; ++i) sym_len[i] = uint16_t((s << 4) | l);
    }
    return K3HUF_OK;
}

extern "C" int k3huf_layer_info(const void *h_layer, size_t bytes, k3huf_layer_info_t *info) {
    if (!info) return K3HUF_E_ARG;
    Layer L;
    int rc = parse_layer(h_layer, bytes, &L);
    if (rc) return rc;
    *info = L.info;
    return K3HUF_OK;
}

extern "C" int k3huf_tensor_info(const void *h_layer, size_t bytes, uint32_t t, k3huf_tensor_info_t *out) {
    if (!out) return K3HUF_E_ARG;
    Layer L;
    int rc = parse_layer(h_layer, bytes, &L);
    if (rc) return rc;
    if (t >= L.info.n_tensors) return K3HUF_E_ARG;
    const TensorEntry &e = L.tensors[t];
    *out = k3huf_tensor_info_t{e.table, e.first_stripe, e.n_stripes, 0, e.n_values, e.out_offset};
    return K3HUF_OK;
}

extern "C" const char *k3huf_strerror(int code) {
    switch (code) {
        case K3HUF_OK: return "ok";
        case K3HUF_E_ARG: return "bad argument (null pointer, size or alignment)";
        case K3HUF_E_EMPTY: return "code table has no symbol";
        case K3HUF_E_OVERSUB: return "code table over-subscribed (Kraft sum above 2^12)";
        case K3HUF_E_BADLEN: return "code length above 12 bits";
        case K3HUF_E_FORMAT: return "malformed container";
        case K3HUF_E_CUDA: return "CUDA runtime error";
        case K3HUF_E_NOMEM: return "host allocation failed";
        case K3HUF_E_IO: return "file open or read failed";
        default: return "unknown error";
    }
}

// ---------------------------------------------------------------------------
// encoder

namespace {

constexpr uint64_t kSegValues = 1u << 20;   // values per encoder work item (a multiple of 2^12)


// Append `len` code bits to a big-endian bit stream at bit offset `pos`.
// Bytes fully owned by this writer are stored; the two partial edge bytes
// are OR-ed atomically because a neighbouring segment shares them.
struct BitWriter {
    uint8_t *bytes;
    uint64_t pos;        // absolute bit position of the next bit
    uint64_t acc = 0;    // pending bits, right-aligned
    int nacc = 0;
    uint64_t start;      // first bit of this segment
    BitWriter(uint8_t *b, uint64_t p) : bytes(b), pos(p), start(p) {
        // align to a byte boundary: the leading partial byte is shared
        nacc = int(p & 7);
        acc = 0;
    }
    void put(uint32_t code, int len) {
        acc = (acc << len) | code;
        nacc += len;
        pos += len;
        while (nacc >= 8) {
            nacc -= 8;
            const uint64_t byte_index = (pos - uint64_t(nacc)) / 8 - 1;
            const uint8_t v = uint8_t(acc >> nacc);
            if (byte_index == start / 8 && (start & 7))
                __atomic_fetch_or(&bytes[byte_index], v, __ATOMIC_RELAXED);
            else
                bytes[byte_index] = v;
        }
    }
    void finish() {
        if (nacc > 0) {
            const uint64_t byte_index = pos / 8;
            __atomic_fetch_or(&bytes[byte_index], uint8_t(acc << (8 - nacc)), __ATOMIC_RELAXED);
        }
    }
};

}  // namespace

extern "C" int k3huf_encode_layer(uint32_t n_tensors, const void *const *h_tensors, const uint64_t *n_values,
                                  uint32_t chunk_syms, uint32_t sub_syms_req, int shared_table, int n_threads,
                                  void *h_blob, size_t blob_cap, size_t *blob_bytes) {
    if (n_tensors == 0 || !h_tensors || !n_values || chunk_syms == 0 || !blob_bytes) return K3HUF_E_ARG;
    const uint32_t sub_syms = effective_sub_syms(chunk_syms, sub_syms_req);
    const uint32_t S = chunk_syms / sub_syms;
    for (uint32_t t = 0; t < n_tensors; ++t)
        if (!h_tensors[t] || n_values[t] == 0) return K3HUF_E_ARG;
    const int threads = n_threads > 0 ? n_threads : int(std::max(1u, std::thread::hardware_concurrency()));
    try {
        LayerPlan L;
        plan_stripes(n_tensors, n_values, chunk_syms, sub_syms, shared_table != 0, L);
        std::vector<PlanStripe> &sp = L.stripes;
        // histograms, one work item per segment of a stripe
        struct Seg { uint32_t stripe; uint64_t a, b; };
        std::vector<Seg> segs;
        for (uint32_t s = 0; s < sp.size(); ++s)
            for (uint64_t a = 0; a < sp[s].n; a += kSegValues)
                segs.push_back({s, a, std::min(sp[s].n, a + kSegValues)});
        std::vector<uint64_t> seg_hist(segs.size() * 256, 0);
        parallel_for(segs.size(), threads, [&](size_t i) {
            const Seg &g = segs[i];
            const PlanStripe &p = sp[g.stripe];
            const uint8_t *x = static_cast<const uint8_t *>(h_tensors[p.tensor]) + 2 * p.v0;
            uint64_t h[4][256] = {};
            uint64_t k = g.a;
            for (; k + 4 <= g.b; k += 4) {
                h[0][x[2 * k + 1]]++;
                h[1][x[2 * k + 3]]++;
                h[2][x[2 * k + 5]]++;
                h[3][x[2 * k + 7]]++;
            }
            for (; k < g.b; ++k) h[0][x[2 * k + 1]]++;
            uint64_t *dst = &seg_hist[i * 256];
            for (int s = 0; s < 256; ++s) dst[s] = h[0][s] + h[1][s] + h[2][s] + h[3][s];
        });
        std::vector<uint64_t> stripe_hist(sp.size() * 256, 0);
        for (size_t i = 0; i < segs.size(); ++i)
            for (int s = 0; s < 256; ++s) stripe_hist[256ull * segs[i].stripe + s] += seg_hist[i * 256 + s];
        plan_layout(stripe_hist.data(), L);
        const uint64_t hdr = L.hdr, pos = L.total;
        const uint32_t n_tables = L.n_tables;
        std::vector<uint8_t> &codelen = L.codelen;
        *blob_bytes = size_t(pos);
        if (!h_blob) return K3HUF_OK;
        if (blob_cap < pos) return K3HUF_E_ARG;
        uint8_t *blob = static_cast<uint8_t *>(h_blob);

        // header, tables, directories; zeroed gaps and stripes
        write_layer_header(L, blob);
        for (size_t i = 0; i < sp.size(); ++i) {
            const uint64_t prev_end = i ? sp[i - 1].blob_offset + sp[i - 1].stripe_bytes : hdr;
            std::memset(blob + prev_end, 0, sp[i].blob_offset - prev_end);
        }
        parallel_for(sp.size(), threads, [&](size_t i) {
            const PlanStripe &p = sp[i];
            std::memset(blob + p.blob_offset, 0, p.stripe_bytes);
            write_stripe_header(p, blob + p.blob_offset);
        });

        // chunk bit offsets: bits per segment (segments hold whole chunks
        // because kSegValues is a multiple of every chunk size that divides
        // it; otherwise sum per chunk below)
        std::vector<uint32_t> code(256ull * n_tables);
        for (uint32_t tb = 0; tb < n_tables; ++tb) {
            uint32_t first[kMaxLen + 1], count[kMaxLen + 1];
            canonical_codes(&codelen[256ull * tb], &code[256ull * tb], first, count);
        }
        // per-chunk bit counts and sub-stream starts, in parallel over segments
        std::vector<std::vector<uint32_t>> chunk_bits(sp.size());
        for (size_t i = 0; i < sp.size(); ++i) chunk_bits[i].assign(sp[i].n_chunks, 0);
        parallel_for(segs.size(), threads, [&](size_t i) {
            const Seg &g = segs[i];
            const PlanStripe &p = sp[g.stripe];
            const uint8_t *cl = &codelen[256ull * p.table];
            const uint8_t *x = static_cast<const uint8_t *>(h_tensors[p.tensor]) + 2 * p.v0;
            uint8_t *sub = blob + p.blob_offset + K3HUF_STRIPE_HDR_BYTES + 4ull * p.n_chunks;
            // chunks that start inside this segment are summed whole here
            uint64_t c0 = (g.a + chunk_syms - 1) / chunk_syms;
            for (uint64_t c = c0; c * chunk_syms < g.b; ++c) {
                const uint64_t a = c * chunk_syms, b = std::min<uint64_t>(p.n, a + chunk_syms);
                uint32_t bits = 0;
                for (uint32_t k = 0; k < S; ++k) {
                    const uint64_t ka = std::min(b, a + uint64_t(k) * sub_syms);
                    const uint64_t kb = std::min(b, ka + sub_syms);
                    if (k > 0) wr16(sub + 2 * (c * (S - 1) + (k - 1)), bits);
                    for (uint64_t j = ka; j < kb; ++j) bits += cl[x[2 * j + 1]];
                }
                chunk_bits[g.stripe][c] = bits;
            }
        });
        std::vector<std::vector<uint64_t>> chunk_off(sp.size());
        for (size_t i = 0; i < sp.size(); ++i) {
            auto &o = chunk_off[i];
            o.resize(sp[i].n_chunks + 1);
            o[0] = 0;
            for (uint32_t c = 0; c < sp[i].n_chunks; ++c) o[c + 1] = o[c] + chunk_bits[i][c];
            if (o[sp[i].n_chunks] != sp[i].huff_bits) return K3HUF_E_FORMAT;   // internal consistency
            uint8_t *st = blob + sp[i].blob_offset;
            for (uint32_t c = 0; c < sp[i].n_chunks; ++c) wr32(st + K3HUF_STRIPE_HDR_BYTES + 4ull * c, uint32_t(o[c]));
        }
        // bit packing and the raw low bytes, in parallel over segments
        parallel_for(segs.size(), threads, [&](size_t i) {
            const Seg &g = segs[i];
            const PlanStripe &p = sp[g.stripe];
            const uint8_t *cl = &codelen[256ull * p.table];
            const uint32_t *cd = &code[256ull * p.table];
            const uint8_t *x = static_cast<const uint8_t *>(h_tensors[p.tensor]) + 2 * p.v0;
            uint8_t *st = blob + p.blob_offset;
            // the segment's first chunk boundary at or after g.a
            const uint64_t c0 = (g.a + chunk_syms - 1) / chunk_syms;
            const uint64_t a = std::min<uint64_t>(p.n, c0 * chunk_syms);
            uint64_t c1 = (g.b + chunk_syms - 1) / chunk_syms;
            const uint64_t b = std::min<uint64_t>(p.n, c1 * chunk_syms);
            if (a < b) {
                BitWriter w(st + p.bits_offset, chunk_off[g.stripe][c0]);
                for (uint64_t k = a; k < b; ++k) {
                    const uint8_t s = x[2 * k + 1];
                    w.put(cd[s], cl[s]);
                }
                w.finish();
            }
            uint8_t *even = st + p.even_offset;
            for (uint64_t k = g.a; k < g.b; ++k) even[k] = x[2 * k];
        });
        return K3HUF_OK;
    } catch (const std::bad_alloc &) {
        return K3HUF_E_NOMEM;
    }
}
