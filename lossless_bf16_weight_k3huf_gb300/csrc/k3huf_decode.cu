// GPU decode of k3_huf containers on GB300 (sm_103a).
//
// Method: article "Kimi K3 纯 CPU 推理中的无损 Trunk 压缩：一次被解码速度判死刑
// 的 Huffman 压缩实验".  Section 已实现的部分: each 64 MiB stripe is
// [stripe header][Huffman bit stream of the odd (high) bytes][even (low)
// bytes raw], decodable independently; a 4096-entry table indexed by the
// next 12 bits gives symbol and length in one load.  Section 规范码分配与
// Kraft 校验: the table comes from codelen[256] by the Kraft check and the
// longest-first canonical assignment.  The decode loop keeps the head of
// the stream at the top of a 64-bit window refilled about once per 8
// symbols.  Section 如果将来重启 names the two standard speed-ups kept
// here: many interleaved streams (generalised to one stream per indexed
// chunk, thousands per stripe) and a double-symbol table (two symbols per
// lookup when both codes fit in the 12-bit window).
//
// GPU mapping (no tensor cores: a bit-serial scan bound by HBM bandwidth):
//  - the sub-stream index splits every chunk into independently decodable
//    sub-streams; lane = sub-stream.  A work item is 32 consecutive
//    sub-streams (one warp); their bits are one contiguous range of the
//    stripe's stream, staged into the warp's shared-memory slot by one bulk
//    copy (cp.async.bulk + the warp's mbarrier, bounded wait).  An item too
//    long for the slot is decoded in passes over prefixes of its lanes;
//  - one persistent CTA per SM (18 warps; 16 for the fused GEMV) takes a contiguous item range and
//    rebuilds the code table only when it changes; inside a table phase the
//    warps take items from a shared counter, multi-pass items first (with a
//    work area, the last sixteenth of every range is pooled across CTAs);
//  - every lockstep lookup emits exactly two codes from a double-symbol
//    table indexed by the next 14 bits (the codes stay 12-bit limited; the
//    wider window halves the pairs that do not fit): a window that does not
//    hold two whole codes gives the first code and the second is the first
//    code of a second lookup at the bits after it, so all lanes of the warp
//    advance by the same number of values per step.  The 64-bit window is a funnel shift
//    of three stream words kept in registers from one group of four lookups
//    to the next, and each lookup's successor is issued before the
//    fallback test;
//  - a round's 64 high bytes per lane are built in registers and stored to a
//    per-lane row in shared memory; every 64 values the warp merges its 32
//    sub-streams' high bytes with their raw low bytes (loads issued one round
//    early) into coalesced 16-byte bf16 stores;
//  - launched with early start, a grid's CTAs take the SMs the grid before
//    it frees, build their tables, copy their first items' bits and decode
//    their first round there; each thread's first global write and first
//    access to the work area wait (griddepcontrol.wait) until that grid has
//    completed;
//  - a sub-stream that ends away from the next recorded bit offset, or an
//    undecodable window, sets a status bit; every loop is bounded by value
//    counts, every shared/global read index is clamped, and the one spin
//    wait (the bulk copy's mbarrier) has an iteration limit (the early-start
//    wait ends when the grid before, itself bounded, completes).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <vector>

#include "k3huf_internal.h"

namespace k3huf {

static thread_local int g_last_cuda_error = 0;
void set_cuda_error(int code) { g_last_cuda_error = code; }

namespace {

constexpr int kItem = 32;                     // sub-streams per work item (one warp)
constexpr int kRound = 64;                    // values per lane between merges
constexpr int kRowBytes = 64;                 // per-lane row: one round of high bytes (8-byte units, swizzled)
constexpr int kMaxTasks = 64;                 // stripes per launch (kernel parameter space)
constexpr int kMaxDevices = 64;
constexpr uint32_t kWaitLimit = 1u << 24;     // mbarrier polls before giving up
constexpr int kMaxHeavy = 64;                 // items listed for the first sweep of a table phase
constexpr int kMaxPoolCtas = 160;             // pooled launches: CTAs, and pools (runs of CTAs whose
constexpr int kMaxPools = 16;                 // ranges end in one code table)

// Lockstep table, indexed by the next lock_bits(kPer) bits (14 for two codes
// per lookup, 12 for one): exactly kPer whole codes.
//   [4:0] bits used by the kPer codes (the shift, taken straight from the
//   entry by a wrapping funnel shift) [23:16] first symbol [31:24] second
//   symbol, [11:8] the first code's length.  0 in [4:0] when the window
//   does not hold kPer whole codes: the second code is then the first code
//   of the entry at the bits after the first code.  Any single code is read
//   that way ([23:16] and [11:8] of the entry its window indexes); the
//   4096-entry (sym << 4) | length table the lockstep table is built from
//   lives in the warp slots only while the tables are built.
// A window where no code starts decodes as symbol 0 of length 1 with
// kBadCode set (bit 12): the decoder ORs the entries it falls back on into
// one word and tests that bit once per pass.
constexpr uint32_t kBadCode = 1u << 12;
template <int kPer> __host__ __device__ constexpr int lock_bits() { return kPer == 2 ? 14 : 12; }
constexpr size_t kSmemLut = (size_t(1) << 14) * sizeof(uint32_t);
// The CTA's shape (one CTA per SM): warps, and each warp's slot of staged
// bit stream per pass.  Shared memory stays just under the 196 KB carve-out
// step, which leaves 60 KB of L1 for the low-byte loads in flight.  The
// decode takes 18 warps, which the register file allows at 96 registers per
// thread, with 5024-byte slots (a smaller slot splits more items into two
// passes); the fused GEMV keeps 16 warps and 5056-byte slots, its
// per-vector accumulators needing the registers.
template <int kGemv> struct Shape {
    static constexpr int warps = kGemv ? 16 : 18;
    static constexpr int threads = 32 * warps;
    static constexpr uint32_t bitbuf = kGemv ? 5056 : 5024;
    static constexpr size_t slot = bitbuf + 16 + size_t(32) * kRowBytes;   // bits + rows of one warp
    static constexpr size_t smem = kSmemLut + size_t(warps) * slot;
};
static_assert(Shape<0>::bitbuf % 16 == 0 && Shape<1>::bitbuf % 16 == 0, "16-byte bulk copies");
static_assert(Shape<0>::smem + 6528 + 1024 <= 200704 && Shape<1>::smem + 6528 + 1024 <= 200704,
              "shared memory (with the static arrays and the reserved 1 KB) under the 196 KB carve-out step");

struct StripeTask {
    const uint8_t *stripe;      // device: stripe header
    uint8_t *out;               // device: first output byte of the stripe
    uint64_t stripe_bytes;
    uint32_t n_values;
    uint32_t table;
    uint32_t item_begin;        // first work item of this stripe in the launch
    uint32_t tensor_stripe;     // index of the stripe within its tensor (fused GEMV)
};

struct DecodeParams {
    const uint8_t *tables;      // device tables (n x 256), or null: use inline_table
    uint32_t *status;
    uint32_t n_tasks;
    uint32_t chunk_syms;
    uint32_t sub_syms;
    uint32_t n_items;
    uint8_t inline_table[256];
    const uint8_t *gemv_x;      // fused GEMV: device bf16 x[cols] (vector b at gemv_x + b * gemv_ldx), or null
    float *gemv_y;              // fused GEMV: device y[rows] (vector b at gemv_y + b * gemv_ldy), accumulated
    uint64_t gemv_cols;
    uint64_t gemv_ldx;          // bytes from one x vector to the next
    uint64_t gemv_ldy;          // floats from one y vector to the next
    uint32_t *work;             // work area: [0] CTAs finished, [1 + j] next slot of pool j
                                // (all left zero), or null
    uint32_t n_pools;
    uint32_t pool_table[kMaxPools];     // code table of pool j's items
    uint16_t pool_cta[kMaxPools + 1];   // pool j: CTAs pool_cta[j] .. pool_cta[j + 1] - 1
    uint16_t pool_tail[kMaxPools];      // most items in one CTA's share of pool j
    uint32_t tail_begin[kMaxPoolCtas];  // CTA b's pooled items: tail_begin[b] .. the end of its range
    StripeTask task[kMaxTasks];
};
static_assert(sizeof(DecodeParams) <= 4096, "kernel parameters");

__device__ __forceinline__ uint32_t bswap32(uint32_t x) { return __byte_perm(x, 0, 0x0123); }

// acc + the dot product of 8 bf16 weights and 8 bf16 inputs (bf16 -> fp32 is
// exact: the 16 bits become the top half of the float)
__device__ __forceinline__ float dot8(const uint4 w, const uint4 x, float acc) {
    const uint32_t a[4] = {w.x, w.y, w.z, w.w}, b[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        acc = fmaf(__uint_as_float(a[k] << 16), __uint_as_float(b[k] << 16), acc);
        acc = fmaf(__uint_as_float(a[k] & 0xFFFF0000u), __uint_as_float(b[k] & 0xFFFF0000u), acc);
    }
    return acc;
}

// Row swizzle: 8-byte unit u of lane l's row sits at unit u ^ row_swz(l).
// The 32 lanes' 8-byte stores of one unit, and the merge's 8-byte reads of
// unit (lane % 8) of rows 4i .. 4i+3, then each touch every bank exactly twice.
__device__ __forceinline__ uint32_t row_swz(uint32_t l) { return (l >> 1) & 7u; }
__device__ __forceinline__ uint32_t row_byte(uint32_t j, uint32_t swz) { return (((j >> 3) ^ swz) << 3) | (j & 7u); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 4-byte global -> shared copy that lands asynchronously (cp.async), and
// the wait for all of this thread's such copies
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Programmatic dependent launch: the next grid in the stream, if launched
// with early start, may be scheduled once every CTA of this one has passed
// grid_dep_launch (or exited); grid_dep_wait returns once the grid before
// this one has completed and its writes are visible.  Both are no-ops for a
// grid launched the ordinary way.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// 64-bit MSB-first bit window over one sub-stream read straight from
// global memory (16-byte read-only loads, one block ahead) -- used for
// sub-streams too long to stage in shared memory.
struct GlobalBits {
    uint64_t acc;            // valid bits at the top
    int cnt;                 // number of valid bits in acc
    uint4 q;                 // current block, front word in q.x
    int qn;                  // words left in q
    uint4 nxt;               // prefetched next block
    const uint4 *p;          // block after nxt
    const uint4 *last;       // last block inside the stripe's stream
    uint32_t nref;           // 32-bit refills done
    uint32_t start;          // first bit

    __device__ __forceinline__ uint4 load(const uint4 *b) const { return __ldg(b <= last ? b : last); }

    __device__ __forceinline__ uint32_t pop() {
        uint32_t w = q.x;
        q.x = q.y;
        q.y = q.z;
        q.z = q.w;
        if (--qn == 0) {
            q = nxt;
            qn = 4;
            nxt = load(p);
            ++p;
        }
        return bswap32(w);
    }

    __device__ __forceinline__ void init(const uint4 *blocks, const uint4 *last_block, uint32_t bitoff) {
        last = last_block;
        start = bitoff;
        const uint4 *b = blocks + (bitoff >> 7);
        q = load(b);
        nxt = load(b + 1);
        p = b + 2;
        qn = 4;
        for (uint32_t i = (bitoff >> 5) & 3; i > 0; --i) (void)pop();
        const uint64_t hi = pop();
        const uint64_t lo = pop();
        const int sh = int(bitoff & 31);
        acc = ((hi << 32) | lo) << sh;
        cnt = 64 - sh;
        nref = 0;
    }

    // top 32 bits of the window, with at least 32 valid bits
    __device__ __forceinline__ uint32_t window() {
        if (cnt <= 32) {
            acc |= uint64_t(pop()) << (32 - cnt);
            cnt += 32;
            ++nref;
        }
        return uint32_t(acc >> 32);
    }

    __device__ __forceinline__ void advance(uint32_t t) {
        acc <<= t;
        cnt -= int(t);
    }

    // absolute bit position of the next unread bit
    __device__ __forceinline__ uint32_t position() const {
        return start + 64u - (start & 31u) + 32u * nref - uint32_t(cnt);
    }
};

// Build the single-code and lockstep tables in shared memory from the code
// lengths (thread t < 256 passes the length of symbol t).  Returns false,
// uniformly across the CTA, when the table fails the Kraft check.  All
// threads of the CTA must call it.
//  - warps 0..7 each rank 32 symbols among equal lengths (ascending symbol
//    order) and count their lengths; warp 0 then walks the lengths from 12
//    down to 1 for the first codes (longest first, each first code the
//    previous one plus its count, halved and rounded up), the Kraft sum and
//    the offsets of each length in the sorted symbol list;
//  - the codes of length l take the 12-bit windows
//    [first[l] << (12 - l), (first[l] + count[l]) << (12 - l)), disjoint
//    across lengths, so every window finds its length by comparisons and its
//    symbol by one index into the sorted list;
//  - a lockstep entry reads the single-code table for each of its two codes
//    (a block of four entries shares the first read, and fills all four
//    from one pair of at most 12 bits).
template <int kPer, int kThreads>
__device__ bool build_tables(uint32_t my_len, uint16_t *lut1, uint32_t *lut) {
    constexpr int L = K3HUF_MAXLEN;
    __shared__ uint32_t s_wcnt[8][L + 1];          // per warp: symbols of each length
    __shared__ uint32_t s_wbase[8][L + 1];         // per warp: symbols of each length in earlier warps
    __shared__ uint32_t s_lo[L + 1], s_hi[L + 1];  // window range of each length
    __shared__ int32_t s_adj[L + 1];               // sorted-list offset minus first code
    __shared__ uint32_t s_off[L + 1];
    __shared__ uint8_t s_sorted[256];
    __shared__ uint32_t s_badlen;
    __shared__ int s_ok;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) s_badlen = 0;
    uint32_t ls = 0, rank_in = 0;
    __syncthreads();
    if (tid < 256) {
        ls = my_len <= uint32_t(L) ? my_len : 0u;
        if (my_len > uint32_t(L)) atomicOr(&s_badlen, 1u);
        const uint32_t same = __match_any_sync(0xffffffffu, ls);
        rank_in = __popc(same & ((1u << lane) - 1u));
        // (rolled loops in this code that runs once per table: fresh
        // instructions cost an instruction-cache fill each)
#pragma unroll 1
        for (int j = 1; j <= L; ++j) {
            const uint32_t bj = __ballot_sync(0xffffffffu, ls == uint32_t(j));
            if (lane == j) s_wcnt[warp][j] = __popc(bj);
        }
    }
    __syncthreads();
    if (warp == 0) {
        // lane l (1..12): counts of length l before each warp, and in total
        uint32_t c = 0;
        if (lane >= 1 && lane <= L) {
#pragma unroll 1
            for (int w = 0; w < 8; ++w) {
                s_wbase[w][lane] = c;
                c += s_wcnt[w][lane];
            }
        }
        uint32_t code = 0, kraft = 0, first_l = 0;
#pragma unroll 1
        for (int l = L; l >= 1; --l) {
            const uint32_t cnt = __shfl_sync(0xffffffffu, c, l);
            if (lane == l) first_l = code;
            code = (code + cnt + 1) >> 1;
            kraft += cnt << (L - l);
        }
        // offsets of each length in the sorted list (ascending length)
        uint32_t incl = c;                                      // inclusive scan over lanes 1..12
#pragma unroll 1
        for (int d = 1; d < 16; d <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        if (lane >= 1 && lane <= L) {
            const uint32_t off = incl - c;
            s_off[lane] = off;
            s_lo[lane] = first_l << (L - lane);
            s_hi[lane] = (first_l + c) << (L - lane);
            s_adj[lane] = int32_t(off) - int32_t(first_l);
        }
        if (lane == 0) s_ok = (!s_badlen && kraft > 0 && kraft <= (1u << L)) ? 1 : 0;
    }
    __syncthreads();
    if (!s_ok) return false;
    if (tid < 256 && ls) s_sorted[s_off[ls] + s_wbase[warp][ls] + rank_in] = uint8_t(tid);
    uint32_t lo[L + 1], hi[L + 1];
#pragma unroll
    for (int j = 1; j <= L; ++j) {
        lo[j] = s_lo[j];
        hi[j] = s_hi[j];
    }
    __syncthreads();
    // single-code 12-bit table: the shortest length whose range holds the
    // window.  Eight windows per thread and step, stored as one 16-byte word:
    // a code of 9 bits or fewer owns an aligned range of at least 8 windows,
    // so when the block's first window falls in one, the whole block does
    auto entry1 = [&](uint32_t e) -> uint32_t {
        uint32_t l = 0;
#pragma unroll
        for (int j = L; j >= 1; --j) l = (e >= lo[j] && e < hi[j]) ? uint32_t(j) : l;
        return l ? (uint32_t(s_sorted[s_adj[l] + int32_t(e >> (L - l))]) << 4) | l : (kBadCode | 1u);
    };
    for (uint32_t m = tid; m < 4096u / 8; m += kThreads) {
        const uint32_t v0 = entry1(8 * m);
        uint32_t w[4];
        if (!(v0 & kBadCode) && (v0 & 15u) <= uint32_t(L - 3)) {
#pragma unroll
            for (int i = 0; i < 4; ++i) w[i] = v0 | (v0 << 16);
        } else {
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo16 = i ? entry1(8 * m + 2 * i) : v0;
                w[i] = lo16 | (entry1(8 * m + 2 * i + 1) << 16);
            }
        }
        reinterpret_cast<uint4 *>(lut1)[m] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
    // lockstep table: exactly kPer codes inside the window.  The second code
    // is looked up on the window's bits after the first code with zeros
    // after the window's end; a code that fits in the window's bits is
    // found the same way whatever those bits are
    // Four consecutive entries per thread and step, stored as one 16-byte
    // word; with a 14-bit window they share their first code, and when the
    // first entry's pair uses 12 bits or fewer, all four are that entry.
    constexpr int W = lock_bits<kPer>();
    for (uint32_t m = tid; m < (1u << W) / 4; m += kThreads) {
        const uint32_t a0 = lut1[(4 * m) >> (W - L)];
        uint32_t v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (W - L >= 2 && i > 0 && (v[0] & 31u) != 0 && (v[0] & 31u) <= uint32_t(L)) {
                v[i] = v[0];
                continue;
            }
            const uint32_t e = 4 * m + uint32_t(i);
            const uint32_t a = W - L >= 2 ? a0 : lut1[e >> (W - L)];
            const uint32_t l1 = a & 15u;
            uint32_t ent;
            if (a & kBadCode) {
                ent = kBadCode | (1u << 8);                        // read by the fallback
            } else if (kPer == 1) {
                ent = ((a >> 4) << 16) | (l1 << 8) | l1;
            } else {
                const uint32_t b = lut1[((e << l1) & ((1u << W) - 1u)) >> (W - L)];
                const uint32_t l2 = b & 15u;
                if (!(b & kBadCode) && l1 + l2 <= uint32_t(W))
                    ent = ((a >> 4) << 16) | ((b >> 4) << 24) | (l1 << 8) | (l1 + l2);
                else
                    ent = ((a >> 4) << 16) | (l1 << 8);            // second code read separately
            }
            v[i] = ent;
        }
        reinterpret_cast<uint4 *>(lut)[m] = make_uint4(v[0], v[1], v[2], v[3]);
    }
    __syncthreads();
    return true;
}

// The stripe task holding work item `item` (tasks: the launch's table, in
// shared memory)
__device__ __forceinline__ uint32_t find_task(const StripeTask *task, uint32_t n_tasks, uint32_t item) {
    uint32_t lo = 0, hi = n_tasks - 1;
    while (lo < hi) {
        const uint32_t mid = (lo + hi + 1) >> 1;
        if (task[mid].item_begin <= item) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Whether a work item's bits (estimated at chunk granularity from the
// chunk offsets) overflow one staging pass.  Such items take two or more
// passes and are started first.  Deterministic in the container bytes, so
// every warp classifies an item the same way; reads stay inside the stripe.
template <uint32_t kBitBuf>
__device__ bool item_heavy(const DecodeParams &P, const StripeTask *task, uint32_t wi) {
    const StripeTask &T = task[find_task(task, P.n_tasks, wi)];
    const uint32_t cs = P.chunk_syms, S = cs / P.sub_syms;
    const uint32_t nch = (T.n_values + cs - 1) / cs;
    if (uint64_t(K3HUF_STRIPE_HDR_BYTES) + 4ull * nch > T.stripe_bytes) return false;
    const uint32_t *h = reinterpret_cast<const uint32_t *>(T.stripe);
    const uint32_t *chunk_off = h + K3HUF_STRIPE_HDR_BYTES / 4;
    const uint32_t g0 = (wi - T.item_begin) * kItem;
    const uint32_t c0 = g0 / S, c1 = min(nch, (g0 + kItem - 1) / S + 1);
    if (c0 >= nch) return false;
    const uint32_t lo = chunk_off[c0], hi = c1 < nch ? chunk_off[c1] : h[4];
    return hi > lo && (hi - lo) / 8 + 64 > kBitBuf;
}

__device__ __forceinline__ uint32_t interleave_lo(uint32_t even4, uint32_t hi4) { return __byte_perm(even4, hi4, 0x5140); }
__device__ __forceinline__ uint32_t interleave_hi(uint32_t even4, uint32_t hi4) { return __byte_perm(even4, hi4, 0x7362); }

// Validate the device copy of a stripe header (its eight words in hdr)
// against the launch's view of it.
__device__ bool stripe_header_ok(const DecodeParams &P, const StripeTask &T, const uint32_t hdr[8]) {
    const uint32_t n = T.n_values, cs = P.chunk_syms, ss = P.sub_syms;
    const uint32_t nch = (n + cs - 1) / cs;
    const uint64_t huff_bits = uint64_t(hdr[4]) | (uint64_t(hdr[5]) << 32);
    const uint32_t bits_off = hdr[6], even_off = hdr[7];
    const uint64_t bits_need = ((huff_bits + 7) / 8 + 15) / 16 * 16 + kBitsSlack;
    const uint64_t index = 4ull * nch + 2ull * nch * (cs / ss - 1);
    bool ok = hdr[0] == kStripeMagic && hdr[2] == n && hdr[3] == nch &&
              bits_off == (K3HUF_STRIPE_HDR_BYTES + index + 15) / 16 * 16 && even_off % 16 == 0 &&
              huff_bits <= uint64_t(K3HUF_MAXLEN) * n && huff_bits >= n &&
              uint64_t(even_off) >= bits_off + bits_need && uint64_t(even_off) + n <= T.stripe_bytes;
    if (P.tables) ok = ok && hdr[1] == T.table;
    return ok;
}

// kFixed: the container's default sizes (chunks of 4096 values, sub-streams
// of 256) as compile-time constants, so that sub-stream and piece offsets
// fold into immediates and divisions by them into shifts
template <int kPer, bool kVec, bool kStaged, int kGemv, bool kFixed = false, bool kPool = false>
__global__ void __launch_bounds__(Shape<kGemv>::threads, 1)
decode_kernel(const __grid_constant__ DecodeParams P) {
    constexpr int kWarps = Shape<kGemv>::warps, kThreads = Shape<kGemv>::threads;
    constexpr uint32_t kBitBuf = Shape<kGemv>::bitbuf;
    constexpr size_t kWarpSlot = Shape<kGemv>::slot;
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t *lut = reinterpret_cast<uint32_t *>(smem);
    uint16_t *lut1 = reinterpret_cast<uint16_t *>(smem + kSmemLut);   // (in the warp slots, during the builds)
    __shared__ __align__(8) uint64_t s_bar[kWarps];
    __shared__ uint32_t s_heavy[kMaxHeavy];
    __shared__ uint32_t s_nheavy, s_next;
    __shared__ int s_pick;
    __shared__ uint32_t s_dead;                  // some warp stopped (a timed-out copy)
    __shared__ uint32_t s_empty;                 // bit j: pool j found empty by a warp of this CTA
    __shared__ uint32_t s_hdr[kMaxTasks][8];     // stripe headers, validated once per CTA
    __shared__ uint8_t s_hok[kMaxTasks];
    __shared__ __align__(16) StripeTask s_task[kMaxTasks];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // (one CTA per SM: a next grid started early takes the SMs this one frees)
    grid_dep_launch();
    uint8_t *wslot = smem + kSmemLut + size_t(warp) * kWarpSlot;
    uint32_t *bitbuf = reinterpret_cast<uint32_t *>(wslot);
    uint8_t *wrows = wslot + kBitBuf + 16;

    const uint32_t cs = kFixed ? 4096u : P.chunk_syms, ss = kFixed ? 256u : P.sub_syms, S = cs / ss;
    // contiguous item ranges whose sizes differ by at most one
    const uint32_t it0 = uint32_t(uint64_t(blockIdx.x) * P.n_items / gridDim.x);
    const uint32_t it1 = uint32_t(uint64_t(blockIdx.x + 1) * P.n_items / gridDim.x);
    // kPool (a work area): the last sixteenth of every CTA's range (inside
    // its last table phase) goes to the pool of the CTAs whose ranges end in
    // the same code table.  CTAs draw from their own pool, round-robin over
    // its CTAs, once their own items are taken, then from any pool with items
    // left (rebuilding their tables for it): fixed ranges leave the CTAs
    // whose items happen to be heavier finishing last.  (A quarter or an
    // eighth pooled was slower: multi-pass items in the pool start late.)
    const bool pool = kPool && P.work != nullptr;
    const uint32_t it_own = pool ? P.tail_begin[blockIdx.x] : it1;
    uint32_t j_me = 0;
    if (pool)
        while (j_me + 1 < P.n_pools && P.pool_cta[j_me + 1] <= blockIdx.x) ++j_me;
    // everything before a thread's first write to global memory (the status
    // word, the output, the work area) reads only the container and the
    // parameters; that write waits for the grid before this one (a no-op
    // for a grid launched the ordinary way)
    bool dep_done = false;
    auto dep = [&]() {
        if (!dep_done) {
            grid_dep_wait();
            dep_done = true;
        }
    };
    // the next item of pool j for this warp, or ~0u once the pool is empty
    // (slot p: item p / n of CTA pool_cta[j] + p % n's share)
    auto pool_grab = [&](uint32_t j) -> uint32_t {
        const uint32_t c0 = P.pool_cta[j], nb = uint32_t(P.pool_cta[j + 1]) - c0, max_tail = P.pool_tail[j];
        dep();
        for (;;) {
            uint32_t p = 0;
            if (lane == 0) p = atomicAdd(P.work + 1 + j, 1u);
            p = __shfl_sync(0xffffffffu, p, 0);
            const uint32_t b = c0 + p % nb, k = p / nb;
            if (k >= max_tail) return ~0u;
            const uint32_t a1 = uint32_t(uint64_t(b + 1) * P.n_items / gridDim.x);
            if (P.tail_begin[b] + k < a1) return P.tail_begin[b] + k;
        }
    };
    int table_built = -1;
    bool table_bad = false, dead = false;
    uint32_t phase = 0;

    if (lane == 0) {
        mbar_init(&s_bar[warp]);
        fence_proxy_async();
    }
    if (tid == 0) {
        s_dead = 0;
        s_empty = 0;
    }
    // the task table in shared memory (the prologue indexes it differently
    // in every lane, which parameter space serialises): warp w copies tasks
    // w, w + kWarps, ... one word per lane
    {
        constexpr uint32_t kWords = sizeof(StripeTask) / 4;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(P.task);
        uint32_t *dst = reinterpret_cast<uint32_t *>(s_task);
        for (uint32_t u = uint32_t(warp); u < P.n_tasks; u += kWarps)
            if (uint32_t(lane) < kWords) dst[u * kWords + lane] = src[u * kWords + lane];
    }
    __syncthreads();
    // stripe headers: copied now (thread u: task u), checked once the first
    // table is built
    const bool hown = uint32_t(tid) < P.n_tasks;
    if (hown) {
        const uint32_t *h = reinterpret_cast<const uint32_t *>(s_task[tid].stripe);
#pragma unroll
        for (int i = 0; i < 8; ++i) cp_async4(&s_hdr[tid][i], h + i);
    }

    // the CTA's items in phases of one code table each
    uint32_t item = it0;
    int steal = -1;                                   // pool drained after the CTA's own range
    for (;;) {                                        // CTA-uniform
        int table;
        uint32_t pend;
        if (item < it1) {
            const uint32_t ti0 = find_task(s_task, P.n_tasks, item);
            table = P.tables ? int(s_task[ti0].table) : 0;
            pend = it1;
            for (uint32_t u = ti0 + 1; u < P.n_tasks && s_task[u].item_begin < it1; ++u)
                if (P.tables && int(s_task[u].table) != table) {
                    pend = s_task[u].item_begin;
                    break;
                }
        } else {
            if (!pool || P.n_pools == 1) break;       // (one pool: drained in the last phase)
            // a pool with items left, the CTA's own first; none once a warp of
            // the CTA has stopped
            if (dead && lane == 0) atomicOr(&s_dead, 1u);
            dep();
            __syncthreads();
            if (tid == 0) {
                int pick = -1;
                for (uint32_t q = 0; q < P.n_pools && pick < 0 && !s_dead; ++q) {
                    const uint32_t j = (j_me + q) % P.n_pools;
                    if ((s_empty >> j) & 1u) continue;       // (slots only grow)
                    const uint32_t size = (uint32_t(P.pool_cta[j + 1]) - P.pool_cta[j]) * uint32_t(P.pool_tail[j]);
                    if (atomicAdd(P.work + 1 + j, 0u) < size) pick = int(j);
                }
                s_pick = pick;
            }
            __syncthreads();
            steal = s_pick;
            if (steal < 0) break;
            table = P.tables ? int(P.pool_table[steal]) : 0;
            pend = item;                              // no own items in this phase
        }
        // the phase's global reads go out before the barrier: the code
        // lengths of a new table, and which of the phase's items take more
        // than one pass (bit k: item item + tid + k * kThreads)
        const uint32_t pend_own = steal >= 0 ? item : min(pend, it_own);
        const bool rebuild = table != table_built;
        uint32_t my_len = 0;
        if (rebuild && tid < 256) my_len = (P.tables ? P.tables + 256ull * table : P.inline_table)[tid];
        uint32_t hmask = 0;
        for (uint32_t k = 0; k < 32u; ++k) {
            const uint32_t i = item + uint32_t(tid) + k * kThreads;
            if (i >= pend_own) break;
            if (item_heavy<kBitBuf>(P, s_task, i)) hmask |= 1u << k;
        }
        __syncthreads();                              // every warp done with the previous table
        if (rebuild) {
            table_bad = !build_tables<kPer, kThreads>(my_len, lut1, lut);
            table_built = table;
        }
        if (steal >= 0 && table_bad) {                // (CTA-uniform) its items cannot be taken
            dep();
            if (tid == 0) atomicOr(P.status, K3HUF_ST_HEADER);
            break;
        }
        if (item == it0 && hown) {                    // published by the next barrier
            cp_async_wait_all();
            s_hok[tid] = stripe_header_ok(P, s_task[tid], s_hdr[tid]) ? 1 : 0;
        }
        if (tid == 0) {
            s_nheavy = 0;
            s_next = 0;
        }
        __syncthreads();
        // list the phase's multi-pass items; warps then take items from a
        // shared counter, listed items first, the rest in index order
        if (!table_bad) {
            for (; hmask; hmask &= hmask - 1u) {
                const uint32_t k = atomicAdd(&s_nheavy, 1u);
                if (k < kMaxHeavy) s_heavy[k] = item + uint32_t(tid) + uint32_t(__ffs(hmask) - 1) * kThreads;
            }
            for (uint32_t i = item + uint32_t(tid) + 32u * kThreads; i < pend_own; i += kThreads)
                if (item_heavy<kBitBuf>(P, s_task, i)) {
                    const uint32_t k = atomicAdd(&s_nheavy, 1u);
                    if (k < kMaxHeavy) s_heavy[k] = i;
                }
        }
        __syncthreads();
        const uint32_t nheavy = s_nheavy <= uint32_t(kMaxHeavy) ? s_nheavy : 0u;   // overflow: index order only
        if (steal < 0 && rebuild && table_bad) {
            dep();
            if (tid == 0) atomicOr(P.status, K3HUF_ST_HEADER);
        }

        while (!table_bad && !dead) {
            uint32_t v = 0;
            if (lane == 0) v = atomicAdd(&s_next, 1u);
            v = __shfl_sync(0xffffffffu, v, 0);
            uint32_t wi;
            if (v < nheavy) {
                wi = s_heavy[v];
            } else {
                if (v - nheavy >= pend_own - item) {
                    // own items taken: the pool being drained, or the CTA's own
                    // pool after its last phase
                    const int j = steal >= 0 ? steal : (pool && pend == it1 ? int(j_me) : -1);
                    if (j < 0) break;
                    wi = pool_grab(uint32_t(j));
                    if (wi == ~0u) {
                        if (lane == 0) atomicOr(&s_empty, 1u << j);
                        break;
                    }
                } else {
                    wi = item + (v - nheavy);
                    bool listed = false;
                    for (uint32_t k = uint32_t(lane); k < nheavy; k += 32) listed |= s_heavy[k] == wi;
                    if (__any_sync(0xffffffffu, listed)) continue;   // taken in the first sweep
                }
            }
            const uint32_t ti = find_task(P.task, P.n_tasks, wi);   // warp-uniform: parameter reads
            const StripeTask &T = P.task[ti];
            uint32_t hdr[8];
            for (int i = 0; i < 8; ++i) hdr[i] = s_hdr[ti][i];
            if (!s_hok[ti]) {
                dep();
                if (lane == 0 && wi == T.item_begin) atomicOr(P.status, K3HUF_ST_HEADER);
                continue;
            }
            const uint32_t n = T.n_values;
            const uint32_t nch = hdr[3];
            const uint32_t huff_bits = hdr[4];       // < 2^32 for a valid stripe (<= 12 * 2^25)
            const uint8_t *stripe = T.stripe;
            const uint8_t *bits = stripe + hdr[6];
            const uint8_t *even = stripe + hdr[7];
            const uint32_t *chunk_off = reinterpret_cast<const uint32_t *>(stripe + K3HUF_STRIPE_HDR_BYTES);
            const uint16_t *sub_off = reinterpret_cast<const uint16_t *>(stripe + K3HUF_STRIPE_HDR_BYTES + 4ull * nch);
            uint8_t *out = T.out;
            const uint32_t n_streams = nch * S;
            const uint32_t g0 = (wi - T.item_begin) * kItem;
            // fused GEMV: the item lies inside one row of the matrix (the row
            // length is a multiple of the item's span)
            float gacc[kGemv > 0 ? kGemv : 1] = {};
            uint64_t grow = 0, gcol0 = 0;
            if (kGemv) {
                const uint64_t f0 = uint64_t(T.tensor_stripe) * K3HUF_STRIPE_VALUES + uint64_t(g0) * ss;
                grow = f0 / P.gemv_cols;
                gcol0 = f0 - grow * P.gemv_cols;
            }

            // this lane's sub-stream g: values [g*ss, g*ss + len)
            const uint32_t g = g0 + uint32_t(lane);
            const bool active = g < n_streams && uint64_t(g) * ss < n;
            const uint32_t my_len = active ? min(ss, n - g * ss) : 0u;
            uint32_t my_off = 0, my_end = 0;
            if (active) {
                const uint32_t c = g / S, k = g - c * S;
                const uint32_t base = chunk_off[c];
                my_off = base + (k ? uint32_t(sub_off[size_t(c) * (S - 1) + k - 1]) : 0u);
                my_end = k + 1 < S ? base + sub_off[size_t(c) * (S - 1) + k]
                                   : (c + 1 < nch ? chunk_off[c + 1] : huff_bits);
            }
            // clamp so that a corrupt index cannot move a read outside the stream
            const uint32_t c_off = min(my_off, huff_bits), c_end = min(max(my_end, c_off), huff_bits);
            // active sub-streams are a prefix of the item
            const uint32_t nact = uint32_t(__popc(__ballot_sync(0xffffffffu, active)));

            uint32_t pa = 0;
            while (pa < nact) {                              // warp-uniform passes
                uint32_t pb = nact, byte_lo = 0, nbytes = 32;
                if (kStaged) {
                    byte_lo = (__shfl_sync(0xffffffffu, c_off, int(pa)) >> 7) << 4;
                    const uint32_t need = ((c_end + 7) / 8 + 15) / 16 * 16 + 16;
                    const unsigned nofit = __ballot_sync(0xffffffffu, uint32_t(lane) > pa &&
                                                         uint32_t(lane) < nact && need - byte_lo > kBitBuf);
                    if (nofit) pb = uint32_t(__ffs(nofit)) - 1;
                    const uint32_t byte_hi = __shfl_sync(0xffffffffu, need, int(pb - 1));
                    // a corrupt index may claim a range that is reversed or too long:
                    // the copy stays inside the buffer and inside the stripe's
                    // stream (which holds at least 32 bytes past byte_lo), and
                    // reads are clamped below
                    const uint32_t region = hdr[7] - hdr[6];
                    const uint32_t span = byte_hi > byte_lo ? byte_hi - byte_lo : 32u;
                    nbytes = max(32u, min(min(span, kBitBuf), region - byte_lo));
                    if (lane == 0) {
                        fence_proxy_async();                 // earlier generic reads of the slot come first
                        mbar_arrive_expect_tx(&s_bar[warp], nbytes);
                        bulk_g2s(bitbuf, bits + byte_lo, nbytes, &s_bar[warp]);
                    }
                }

                // merge-phase assignment (vector path): piece i of this lane is the
                // item's sub-stream (i * 4 + lane / 8), values [r*64 + (lane % 8) * 8, +8)
                const uint32_t sub = uint32_t(lane) & 7u;
                auto piece_len = [&](int i) -> uint32_t {
                    const uint32_t t = uint32_t(i) * 4u + uint32_t(lane >> 3);
                    return (t >= pa && t < pb) ? min(ss, n - (g0 + t) * ss) : 0u;
                };
                // low bytes of a round, loaded one round ahead (the first round's
                // loads are in flight while the bit copy lands)
                uint2 ev[8];
                auto load_even = [&](uint32_t round) {
                    const uint32_t v = round * kRound + sub * 8u;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t gi = g0 + uint32_t(i) * 4u + uint32_t(lane >> 3);
                        ev[i] = kVec && v < piece_len(i)
                                    ? __ldg(reinterpret_cast<const uint2 *>(even + size_t(gi) * ss + v))
                                    : make_uint2(0, 0);
                    }
                };
                load_even(0);

                if (kStaged) {
                    // bounded wait for the copy
                    uint32_t polls = 0;
                    bool landed = false;
                    while (!(landed = mbar_try_wait(&s_bar[warp], phase)) && ++polls < kWaitLimit) {
                    }
                    phase ^= 1u;
                    if (!__all_sync(0xffffffffu, landed)) {
                        dep();
                        if (lane == 0) atomicOr(P.status, K3HUF_ST_TIMEOUT);
                        // let the copy in flight land (again bounded), then stop this warp's work
                        polls = 0;
                        while (!landed && !(landed = mbar_try_wait(&s_bar[warp], phase ^ 1u)) && ++polls < kWaitLimit) {
                        }
                        dead = true;
                        break;
                    }
                    __syncwarp();
                }

                const bool in_pass = uint32_t(lane) >= pa && uint32_t(lane) < pb;
                const uint32_t len = in_pass ? my_len : 0u;
                uint32_t bp = in_pass ? c_off - byte_lo * 8u : 0u;
                const uint32_t max_word = nbytes / 4 - 3;
                GlobalBits gb;
                if (!kStaged)
                    gb.init(reinterpret_cast<const uint4 *>(bits), reinterpret_cast<const uint4 *>(even) - 1, c_off);
                uint32_t bad = 0;

                constexpr int kW = lock_bits<kPer>();
                // rounds: the same number for every lane of the warp
                const uint32_t wlen = __reduce_max_sync(0xffffffffu, len);
                const uint32_t n_rounds = (wlen + kRound - 1) / kRound;

                // 64-bit window at bit position `cur` of the staged stream.  The
                // slot keeps the stream's byte order; each word is put MSB-first
                // (one byte permute) as a window loads it, which costs fewer
                // instructions than a pass that swaps the whole slot in place
                auto window = [&](uint32_t cur, uint32_t &hi, uint32_t &lo) {
                    const uint32_t i = min(cur >> 5, max_word);
                    const uint32_t w0 = bswap32(bitbuf[i]), w1 = bswap32(bitbuf[i + 1]), w2 = bswap32(bitbuf[i + 2]);
                    hi = __funnelshift_l(w1, w0, cur);
                    lo = __funnelshift_l(w2, w1, cur);
                };
                // one code: the first code of the lockstep entry its window
                // indexes; an undecodable window gives symbol 0 and one bit,
                // and sets kBadCode in `bad`.  Callers keep the low byte
                auto single = [&](uint32_t win, uint32_t &len_out) -> uint32_t {
                    const uint32_t a = lut[win >> (32 - kW)];
                    bad |= a;
                    len_out = (a >> 8) & 15u;
                    return a >> 16;
                };

                // full rounds (every sub-stream of the item has 64 more values in
                // this pass): piece i sits 4 * i sub-streams after piece 0
                const uint32_t q = uint32_t(lane) >> 3;
                uint8_t *const out_p0 = out + 2 * (size_t(g0 + q) * ss + sub * 8u);
                const uint8_t *const x_p0 = kGemv ? P.gemv_x + 2 * (gcol0 + size_t(q) * ss + sub * 8u) : nullptr;
                const uint8_t *const even_p0 = even + size_t(g0 + q) * ss + sub * 8u;
                const size_t pstride = size_t(4) * ss;

                // staged words rw_i .. rw_i + 2 held in registers from one group to
                // the next: a lane moves on by 0-2 words per group, so most groups
                // load one word, and their first lookup starts from registers
                // (the fused GEMV, short of registers, reloads all three)
                uint32_t rw_i = 0u - 8u, rw0 = 0, rw1 = 0, rw2 = 0;
                for (uint32_t r = 0; r < n_rounds; ++r) {
                    const uint32_t rem = len > r * kRound ? len - r * kRound : 0u;
                    uint8_t *row = wrows + size_t(lane) * kRowBytes;
                    const uint32_t swz = row_swz(uint32_t(lane));
                    const bool full = __all_sync(0xffffffffu, rem >= uint32_t(kRound));
                    if (kStaged && full) {
                        // lockstep round: every lookup yields exactly kPer codes, so
                        // each group of 4 lookups fills 4 * kPer bytes at a fixed place
#pragma unroll(kGemv ? 4 : 2)                    // (4 or 8 for decode: more code, slower)
                        for (int grp = 0; grp < kRound / (4 * kPer); ++grp) {
                            uint32_t cur = bp, cur0 = bp, hi, lo;
                            if (kGemv) {
                                window(cur, hi, lo);           // (no registers to spare)
                            } else {
                                const uint32_t i = min(cur >> 5, max_word);
                                const uint32_t d = i - rw_i;        // words moved since the last group
                                const uint32_t n2 = bswap32(bitbuf[i + 2]);
                                uint32_t n1 = rw2, n0 = rw1;
                                if (d >= 2) n1 = bswap32(bitbuf[i + 1]);
                                if (d >= 3) n0 = bswap32(bitbuf[i]);
                                if (d == 2) n0 = rw2;
                                if (d == 0) {
                                    n0 = rw0;
                                    n1 = rw1;
                                }
                                rw0 = n0;
                                rw1 = n1;
                                rw2 = n2;
                                rw_i = i;
                                hi = __funnelshift_l(n1, n0, cur);
                                lo = __funnelshift_l(n2, n1, cur);
                            }
                            uint32_t ek[4];
                            uint32_t e_next = lut[hi >> (32 - kW)];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                uint32_t e = e_next;
                                uint32_t t = e & 31u;
                                // a whole-pair entry shifts the window by its low five bits
                                uint32_t nhi = __funnelshift_l(lo, hi, e), nlo = __funnelshift_l(0u, lo, e);
                                // the next lookup goes out before the fallback test (and is
                                // redone after a fallback), which keeps the test and its
                                // branch off the chain of dependent lookups
                                if (k < 3) e_next = lut[nhi >> (32 - kW)];
                                if (t == 0u) {
                                    // the window does not hold kPer whole codes: take the
                                    // first code from the entry, read the second one alone.
                                    // The 64-bit window must cover these codes (up to 12
                                    // bits each) ...
                                    if (cur - cur0 > 64u - 12u * kPer) {
                                        window(cur, hi, lo);
                                        cur0 = cur;
                                    }
                                    const uint32_t l = (e >> 8) & 15u;
                                    bad |= e;
                                    uint32_t syms = e & 0x00FF0000u;
                                    nhi = __funnelshift_l(lo, hi, l);
                                    nlo = lo << l;
                                    t = l;
                                    if (kPer == 2) {
                                        uint32_t l2;
                                        syms |= single(nhi, l2) << 24;
                                        t += l2;
                                        nhi = __funnelshift_l(nlo, nhi, l2);
                                        nlo <<= l2;
                                    }
                                    e = syms;
                                    // ... and afterwards the group's remaining lookups (kW
                                    // bits each): reload it when it might not
                                    if (k < 3 && cur + t - cur0 > 64u - uint32_t(kW) * uint32_t(3 - k)) {
                                        window(cur + t, nhi, nlo);
                                        cur0 = cur + t;
                                    }
                                    if (k < 3) e_next = lut[nhi >> (32 - kW)];
                                }
                                hi = nhi;
                                lo = nlo;
                                cur += t;
                                ek[k] = e;
                            }
                            uint32_t R0, R1 = 0;
                            if (kPer == 2) {
                                R0 = __byte_perm(ek[0], ek[1], 0x7632);
                                R1 = __byte_perm(ek[2], ek[3], 0x7632);
                            } else {
                                R0 = __byte_perm(__byte_perm(ek[0], ek[1], 0x0062), __byte_perm(ek[2], ek[3], 0x0062), 0x5410);
                            }
                            bp = cur;
                            if (kPer == 2)
                                reinterpret_cast<uint2 *>(row)[uint32_t(grp) ^ swz] = make_uint2(R0, R1);
                            else
                                reinterpret_cast<uint32_t *>(row)[((uint32_t(grp >> 1) ^ swz) << 1) | uint32_t(grp & 1)] = R0;
                        }
                    } else {
                        // partial round (a stream's end or a split pass): exact single codes
                        const uint32_t cnt = min(rem, uint32_t(kRound));
                        for (uint32_t j = 0; j < cnt; ++j) {
                            uint32_t win;
                            if (kStaged) {
                                const uint32_t i = min(bp >> 5, max_word);
                                win = __funnelshift_l(bswap32(bitbuf[i + 1]), bswap32(bitbuf[i]), bp);
                            } else {
                                win = gb.window();
                            }
                            uint32_t l;
                            row[row_byte(j, swz)] = uint8_t(single(win, l));
                            if (kStaged) bp += l; else gb.advance(l);
                        }
                    }
                    __syncwarp();
                    // decoding wrote only shared memory: a launch started early
                    // decodes its first round before the grid ahead of it ends;
                    // the output stores (the GEMV's reads of x) wait for it
                    dep();
                    if (kVec && full) {
                        const uint32_t rv = r * kRound;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t gw = uint32_t(i) * 4u + q;
                            const uint2 h = *reinterpret_cast<const uint2 *>(wrows + gw * kRowBytes + ((sub ^ row_swz(gw)) << 3));
                            uint4 o;
                            o.x = interleave_lo(ev[i].x, h.x);
                            o.y = interleave_hi(ev[i].x, h.x);
                            o.z = interleave_lo(ev[i].y, h.y);
                            o.w = interleave_hi(ev[i].y, h.y);
                            if (kGemv) {
#pragma unroll
                                for (int b = 0; b < kGemv; ++b)
                                    gacc[b] = dot8(o, __ldg(reinterpret_cast<const uint4 *>(x_p0 + b * P.gemv_ldx + 2 * (size_t(i) * pstride + rv))), gacc[b]);
                            } else
                                *reinterpret_cast<uint4 *>(out_p0 + 2 * (size_t(i) * pstride + rv)) = o;
                        }
                        if (__all_sync(0xffffffffu, rem >= uint32_t(2 * kRound))) {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                ev[i] = __ldg(reinterpret_cast<const uint2 *>(even_p0 + size_t(i) * pstride + rv + kRound));
                        } else if (r + 1 < n_rounds) {
                            load_even(r + 1);
                        }
                    } else if (kVec) {
                        const uint32_t v = r * kRound + sub * 8u;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t m_len = piece_len(i);
                            if (v >= m_len) continue;
                            const uint32_t gw = uint32_t(i) * 4u + uint32_t(lane >> 3);
                            const uint2 h = *reinterpret_cast<const uint2 *>(wrows + gw * kRowBytes + ((sub ^ row_swz(gw)) << 3));
                            const uint32_t hx = h.x, hy = h.y;
                            uint4 o;
                            o.x = interleave_lo(ev[i].x, hx);
                            o.y = interleave_hi(ev[i].x, hx);
                            o.z = interleave_lo(ev[i].y, hy);
                            o.w = interleave_hi(ev[i].y, hy);
                            if (kGemv) {
                                uint4 wv = o;
                                if (v + 8 > m_len) {          // weights past the sub-stream's end count zero
                                    const uint32_t kk = m_len - v;
                                    wv.x = kk >= 2 ? wv.x : kk == 1 ? (wv.x & 0xFFFFu) : 0u;
                                    wv.y = kk >= 4 ? wv.y : kk == 3 ? (wv.y & 0xFFFFu) : 0u;
                                    wv.z = kk >= 6 ? wv.z : kk == 5 ? (wv.z & 0xFFFFu) : 0u;
                                    wv.w = kk >= 8 ? wv.w : kk == 7 ? (wv.w & 0xFFFFu) : 0u;
                                }
#pragma unroll
                                for (int b = 0; b < kGemv; ++b)
                                    gacc[b] = dot8(wv, __ldg(reinterpret_cast<const uint4 *>(P.gemv_x + b * P.gemv_ldx + 2 * (gcol0 + size_t(gw) * ss + v))), gacc[b]);
                                continue;
                            }
                            uint8_t *dst = out + 2 * (size_t(g0 + gw) * ss + v);
                            if (v + 8 <= m_len) {
                                *reinterpret_cast<uint4 *>(dst) = o;
                            } else {
                                const uint32_t kk = m_len - v;   // 1..7 values left in the sub-stream
                                uint16_t *d16 = reinterpret_cast<uint16_t *>(dst);
#pragma unroll
                                for (uint32_t j = 0; j < 8; ++j) {
                                    const uint32_t w = j < 2 ? o.x : j < 4 ? o.y : j < 6 ? o.z : o.w;
                                    if (j < kk) d16[j] = uint16_t(w >> (16 * (j & 1)));
                                }
                            }
                        }
                        if (r + 1 < n_rounds) load_even(r + 1);   // in flight while the next round decodes
                    } else if (len) {
                        // scalar path for sub-stream sizes that break 8-value alignment
                        const uint32_t a0 = r * kRound, b0 = min(len, a0 + kRound);
                        const size_t v0 = size_t(g) * ss;
                        for (uint32_t vv = a0; vv < b0; ++vv) {
                            out[2 * (v0 + vv)] = even[v0 + vv];
                            out[2 * (v0 + vv) + 1] = row[row_byte(vv - a0, swz)];
                        }
                    }
                    __syncwarp();
                }

                uint32_t st = 0;
                if (len) {
                    if (bad & kBadCode) st |= K3HUF_ST_BADCODE;
                    const uint32_t pos = kStaged ? bp + byte_lo * 8u : gb.position();
                    if (my_off > huff_bits || my_end > huff_bits) st |= K3HUF_ST_OVERRUN;
                    if (pos != my_end) st |= K3HUF_ST_INDEX;
                }
                st = __reduce_or_sync(0xffffffffu, st);
                if (st) dep();
                if (lane == 0 && st) atomicOr(P.status, st);
                __syncwarp();                            // slot free for the next pass / item
                pa = pb;
            }
            if (kGemv) {
#pragma unroll
                for (int b = 0; b < kGemv; ++b)
#pragma unroll
                    for (int d = 16; d; d >>= 1) gacc[b] += __shfl_xor_sync(0xffffffffu, gacc[b], d);
                dep();
                if (lane == 0)
#pragma unroll
                    for (int b = 0; b < kGemv; ++b)
                        if (gacc[b] != 0.f) atomicAdd(P.gemv_y + b * P.gemv_ldy + grow, gacc[b]);
            }
        }
        item = pend;
    }
    // the last CTA to finish returns the work area to zero for the next launch
    dep();
    if (pool) {
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            if (atomicAdd(P.work, 1u) == gridDim.x - 1u) {
                for (uint32_t j = 0; j <= P.n_pools; ++j) atomicExch(P.work + j, 0u);
                __threadfence();
            }
        }
    }
}

// Pools of a launch of `grid` CTAs over P's items: CTA b's pooled items are
// the last sixteenth of its range, kept inside its last table phase (the
// run of same-table stripes holding its last item); consecutive CTAs whose
// last phases share a table form one pool.  False when the launch has more
// CTAs or pools than the parameters hold.
bool pool_setup(DecodeParams &P, uint32_t grid) {
    if (grid > uint32_t(kMaxPoolCtas)) return false;
    uint32_t n_pools = 0;
    for (uint32_t b = 0; b < grid; ++b) {
        const uint32_t a0 = uint32_t(uint64_t(b) * P.n_items / grid), a1 = uint32_t(uint64_t(b + 1) * P.n_items / grid);
        uint32_t t = 0;
        while (t + 1 < P.n_tasks && P.task[t + 1].item_begin <= a1 - 1) ++t;
        const uint32_t table = P.tables ? P.task[t].table : 0u;
        uint32_t run = t;
        while (run > 0 && P.tables && P.task[run - 1].table == table) --run;
        const uint32_t phase0 = std::max(a0, P.task[run].item_begin);
        const uint32_t tail = std::max(a1 - ((a1 - a0) >> 4), phase0);
        P.tail_begin[b] = tail;
        if (b == 0 || P.pool_table[n_pools - 1] != table) {
            if (n_pools == uint32_t(kMaxPools)) return false;
            P.pool_table[n_pools] = table;
            P.pool_cta[n_pools] = uint16_t(b);
            P.pool_tail[n_pools] = 0;
            ++n_pools;
        }
        P.pool_tail[n_pools - 1] = uint16_t(std::max<uint32_t>(P.pool_tail[n_pools - 1], a1 - tail));
    }
    P.pool_cta[n_pools] = uint16_t(grid);
    P.n_pools = n_pools;
    return true;
}

template <int kPer, bool kVec, bool kStaged, int kGemv = 0, bool kFixed = false, bool kPool = false>
int launch(DecodeParams &P, cudaStream_t stream, bool early = false) {
    // per device and instantiation: the grid size, 0 until the first launch
    // has set the shared-memory opt-in (two threads doing it at once both set
    // the same values, which is harmless)
    static std::atomic<int> grid_max[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        set_cuda_error(int(e));
        return K3HUF_E_CUDA;
    }
    int gmax = grid_max[dev].load(std::memory_order_acquire);
    if (gmax == 0) {
        e = cudaFuncSetAttribute(decode_kernel<kPer, kVec, kStaged, kGemv, kFixed, kPool>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(Shape<kGemv>::smem));
        int sms = 0, per_sm = 0;
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<kPer, kVec, kStaged, kGemv, kFixed, kPool>,
                                                              Shape<kGemv>::threads, Shape<kGemv>::smem);
        if (e != cudaSuccess) {
            set_cuda_error(int(e));
            return K3HUF_E_CUDA;
        }
        gmax = std::max(1, sms * std::max(1, per_sm));
        grid_max[dev].store(gmax, std::memory_order_release);
    }
    const uint32_t grid = std::min<uint32_t>(P.n_items, uint32_t(gmax));
    if constexpr (kPool) {
        if (!pool_setup(P, grid)) {
            P.work = nullptr;
            return launch<kPer, kVec, kStaged, kGemv, kFixed, false>(P, stream, early);
        }
    }
    if (early) {
        // programmatic stream serialisation: the grid may start, reading only
        // the container, while the previous kernel in the stream finishes
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(Shape<kGemv>::threads);
        cfg.dynamicSmemBytes = Shape<kGemv>::smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, decode_kernel<kPer, kVec, kStaged, kGemv, kFixed, kPool>, P);
        if (e != cudaSuccess) {
            set_cuda_error(int(e));
            return K3HUF_E_CUDA;
        }
    } else {
        decode_kernel<kPer, kVec, kStaged, kGemv, kFixed, kPool><<<grid, Shape<kGemv>::threads, Shape<kGemv>::smem, stream>>>(P);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_cuda_error(int(e));
        return K3HUF_E_CUDA;
    }
    return K3HUF_OK;
}

// Decoder variant: codes per lockstep lookup (1 or 2).
int g_per = 2;

template <int kPer>
int launch_syms(DecodeParams &P, cudaStream_t stream, bool early) {
    const bool vec = P.sub_syms % 8 == 0;
    // a sub-stream's bits (at most 12 per value) must fit the shared buffer
    const bool staged = uint64_t(P.sub_syms) * K3HUF_MAXLEN / 8 + 64 <= Shape<0>::bitbuf;
    if constexpr (kPer == 2)
        if (staged && P.chunk_syms == 4096 && P.sub_syms == 256)
            return P.work ? launch<2, true, true, false, true, true>(P, stream, early)
                          : launch<2, true, true, false, true>(P, stream, early);
    P.work = nullptr;                                    // (the pool has the default sizes only)
    if (staged) return vec ? launch<kPer, true, true>(P, stream, early) : launch<kPer, false, true>(P, stream, early);
    return vec ? launch<kPer, true, false>(P, stream, early) : launch<kPer, false, false>(P, stream, early);
}

// fused GEMV launches: staged bits and the vector merge only
int launch_gemv(DecodeParams &P, uint32_t n_vec, cudaStream_t stream, bool early = false) {
    const bool fixed = P.chunk_syms == 4096 && P.sub_syms == 256;
    if (n_vec > 1) {
        // several vectors: the default layout and two codes per lookup only
        if (!fixed || g_per == 1) return K3HUF_E_ARG;
        switch (n_vec) {
            case 2: return launch<2, true, true, 2, true>(P, stream, early);
            case 4: return launch<2, true, true, 4, true>(P, stream, early);
            case 8: return launch<2, true, true, 8, true>(P, stream, early);
            default: return K3HUF_E_ARG;
        }
    }
    switch (g_per) {
        case 1: return launch<1, true, true, 1>(P, stream, early);
        default:
            if (fixed) return launch<2, true, true, 1, true>(P, stream, early);
            return launch<2, true, true, 1>(P, stream, early);
    }
}

// y = 0 ahead of a GEMV that accumulates into it.  It lets the kernel behind
// it be scheduled at once and writes only once the kernel before it (which
// may still be adding into y) has completed.
__global__ void __launch_bounds__(256) zero_y_kernel(float *y, uint64_t n) {
    grid_dep_launch();
    grid_dep_wait();
    for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += uint64_t(gridDim.x) * blockDim.x)
        y[i] = 0.f;
}

int launch_zero_y(float *y, uint64_t n, cudaStream_t stream, bool early) {
    const uint32_t grid = uint32_t(std::min<uint64_t>(64, (n + 255) / 256));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, zero_y_kernel, y, n);
    if (e != cudaSuccess) {
        set_cuda_error(int(e));
        return K3HUF_E_CUDA;
    }
    return K3HUF_OK;
}

int launch_tasks(DecodeParams &P, cudaStream_t stream, bool early = false) {
    switch (g_per) {
        case 1: return launch_syms<1>(P, stream, early);
        default: return launch_syms<2>(P, stream, early);
    }
}

uint32_t items_of(uint32_t n_values, uint32_t cs, uint32_t ss) {
    const uint64_t nch = (uint64_t(n_values) + cs - 1) / cs;
    const uint64_t streams = nch * (cs / ss);
    return uint32_t((streams + kItem - 1) / kItem);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace k3huf

using namespace k3huf;

extern "C" int k3huf_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" int k3huf_set_decoder_variant(int variant) {
    if (variant < 0 || variant > 2) return K3HUF_E_ARG;
    g_per = variant == 0 ? 2 : variant;
    return K3HUF_OK;
}

namespace {
// The layer's stripes [0, n) into d_out at the layer's output offsets, or,
// with tensor >= 0, that tensor's stripes into d_out from its first value
int decode_layer_impl(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer, size_t layer_bytes, void *d_out,
                      size_t out_bytes, uint32_t *d_status, uint32_t *d_work, bool early, void *stream,
                      int64_t tensor = -1) {
    if (!h_layer_hdr || !d_layer || !d_out || !d_status) return K3HUF_E_ARG;
    if (!aligned16(d_layer) || !aligned16(d_out) || (reinterpret_cast<uintptr_t>(d_status) & 3u)) return K3HUF_E_ARG;
    Layer L;
    int rc = parse_layer(h_layer_hdr, hdr_bytes, &L);
    if (rc) return rc;
    size_t s_begin = 0, s_end = L.stripes.size();
    uint64_t out_shift = 0, need = L.info.out_bytes;
    if (tensor >= 0) {
        if (uint64_t(tensor) >= L.tensors.size()) return K3HUF_E_ARG;
        const TensorEntry &te = L.tensors[size_t(tensor)];
        s_begin = te.first_stripe;
        s_end = size_t(te.first_stripe) + te.n_stripes;
        out_shift = te.out_offset;
        need = 2 * te.n_values;
    }
    if (layer_bytes < L.info.blob_bytes || out_bytes < need) return K3HUF_E_ARG;
    const uint8_t *blob = static_cast<const uint8_t *>(d_layer);
    uint8_t *out = static_cast<uint8_t *>(d_out);
    DecodeParams P{};
    P.tables = blob + K3HUF_LAYER_HDR_BYTES;
    P.status = d_status;
    P.chunk_syms = L.info.chunk_syms;
    P.sub_syms = L.info.sub_syms;
    for (size_t s0 = s_begin; s0 < s_end; s0 += kMaxTasks) {
        const size_t s1 = std::min(s_end, s0 + kMaxTasks);
        uint32_t items = 0;
        P.n_tasks = uint32_t(s1 - s0);
        for (size_t s = s0; s < s1; ++s) {
            const StripeEntry &e = L.stripes[s];
            StripeTask &t = P.task[s - s0];
            t.stripe = blob + e.blob_offset;
            t.out = out + (e.out_offset - out_shift);
            t.stripe_bytes = e.stripe_bytes;
            t.n_values = e.n_values;
            t.table = e.table;
            t.item_begin = items;
            t.tensor_stripe = 0;
            items += items_of(e.n_values, P.chunk_syms, P.sub_syms);
        }
        P.n_items = items;
        P.work = d_work;
        rc = launch_tasks(P, static_cast<cudaStream_t>(stream), early);
        if (rc) return rc;
    }
    return K3HUF_OK;
}
}  // namespace

extern "C" int k3huf_decode_layer(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer, size_t layer_bytes,
                                  void *d_out, size_t out_bytes, uint32_t *d_status, void *stream) {
    return decode_layer_impl(h_layer_hdr, hdr_bytes, d_layer, layer_bytes, d_out, out_bytes, d_status, nullptr, false,
                             stream);
}

extern "C" int k3huf_decode_layer_ws(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer, size_t layer_bytes,
                                     void *d_out, size_t out_bytes, uint32_t *d_status, void *d_work, size_t work_bytes,
                                     void *stream) {
    if (!d_work || work_bytes < K3HUF_WORK_BYTES || (reinterpret_cast<uintptr_t>(d_work) & 3u)) return K3HUF_E_ARG;
    return decode_layer_impl(h_layer_hdr, hdr_bytes, d_layer, layer_bytes, d_out, out_bytes, d_status,
                             static_cast<uint32_t *>(d_work), false, stream);
}

extern "C" int k3huf_decode_layer_ex(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer, size_t layer_bytes,
                                     void *d_out, size_t out_bytes, uint32_t *d_status, void *d_work, size_t work_bytes,
                                     uint32_t flags, void *stream) {
    if (flags & ~uint32_t(K3HUF_DECODE_EARLY_START)) return K3HUF_E_ARG;
    if (d_work && (work_bytes < K3HUF_WORK_BYTES || (reinterpret_cast<uintptr_t>(d_work) & 3u))) return K3HUF_E_ARG;
    return decode_layer_impl(h_layer_hdr, hdr_bytes, d_layer, layer_bytes, d_out, out_bytes, d_status,
                             static_cast<uint32_t *>(d_work), (flags & K3HUF_DECODE_EARLY_START) != 0, stream);
}

extern "C" int k3huf_decode_tensor(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer, size_t layer_bytes,
                                   uint32_t tensor, void *d_out, size_t out_bytes, uint32_t *d_status, void *d_work,
                                   size_t work_bytes, uint32_t flags, void *stream) {
    if (flags & ~uint32_t(K3HUF_DECODE_EARLY_START)) return K3HUF_E_ARG;
    if (d_work && (work_bytes < K3HUF_WORK_BYTES || (reinterpret_cast<uintptr_t>(d_work) & 3u))) return K3HUF_E_ARG;
    return decode_layer_impl(h_layer_hdr, hdr_bytes, d_layer, layer_bytes, d_out, out_bytes, d_status,
                             static_cast<uint32_t *>(d_work), (flags & K3HUF_DECODE_EARLY_START) != 0, stream,
                             int64_t(tensor));
}

extern "C" int k3huf_decode_stripe(const uint8_t codelen[256], uint32_t chunk_syms, uint32_t sub_syms,
                                   const void *d_stripe, size_t stripe_bytes, uint32_t n_values, void *d_out,
                                   uint32_t *d_status, void *stream) {
    if (!codelen || !d_stripe || !d_out || !d_status || chunk_syms == 0 || n_values == 0 ||
        n_values > K3HUF_STRIPE_VALUES || sub_syms == 0 || effective_sub_syms(chunk_syms, sub_syms) != sub_syms)
        return K3HUF_E_ARG;
    if (!aligned16(d_stripe) || !aligned16(d_out) || (reinterpret_cast<uintptr_t>(d_status) & 3u)) return K3HUF_E_ARG;
    int rc = k3huf_build(codelen, nullptr);
    if (rc) return rc;
    const uint32_t nch = (n_values + chunk_syms - 1) / chunk_syms;
    if (stripe_bytes < align_up(K3HUF_STRIPE_HDR_BYTES + index_bytes(nch, chunk_syms, sub_syms), 16) + kBitsSlack +
                           n_values)
        return K3HUF_E_ARG;
    DecodeParams P{};
    P.tables = nullptr;
    P.status = d_status;
    P.chunk_syms = chunk_syms;
    P.sub_syms = sub_syms;
    P.n_tasks = 1;
    for (int i = 0; i < 256; ++i) P.inline_table[i] = codelen[i];
    StripeTask &t = P.task[0];
    t.stripe = static_cast<const uint8_t *>(d_stripe);
    t.out = static_cast<uint8_t *>(d_out);
    t.stripe_bytes = stripe_bytes;
    t.n_values = n_values;
    t.table = 0;
    t.item_begin = 0;
    t.tensor_stripe = 0;
    P.n_items = items_of(n_values, chunk_syms, sub_syms);
    return launch_tasks(P, static_cast<cudaStream_t>(stream));
}

namespace {
int gemv_layer_impl(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer, size_t layer_bytes, uint32_t tensor,
                    uint64_t cols, const void *d_x, uint32_t n_vec, float *d_y, uint32_t *d_status, uint32_t flags,
                    void *stream) {
    using namespace k3huf;
    if (!h_layer_hdr || !d_layer || !d_x || !d_y || !d_status || cols == 0) return K3HUF_E_ARG;
    if (n_vec != 1 && n_vec != 2 && n_vec != 4 && n_vec != 8) return K3HUF_E_ARG;
    if (!aligned16(d_layer) || !aligned16(d_x) || (reinterpret_cast<uintptr_t>(d_y) & 3u) ||
        (reinterpret_cast<uintptr_t>(d_status) & 3u))
        return K3HUF_E_ARG;
    Layer L;
    int rc = parse_layer(h_layer_hdr, hdr_bytes, &L);
    if (rc) return rc;
    if (layer_bytes < L.info.blob_bytes || tensor >= L.tensors.size()) return K3HUF_E_ARG;
    const TensorEntry &te = L.tensors[tensor];
    const uint32_t ss = L.info.sub_syms, cs = L.info.chunk_syms;
    // every work item (32 sub-streams of ss values, whole chunks) must lie in one row
    if (te.n_values % cols != 0 || cols % (uint64_t(kItem) * ss) != 0 || ss % 8 != 0 || kItem % (cs / ss) != 0 ||
        uint64_t(ss) * K3HUF_MAXLEN / 8 + 64 > Shape<1>::bitbuf)
        return K3HUF_E_ARG;
    const uint8_t *blob = static_cast<const uint8_t *>(d_layer);
    DecodeParams P{};
    P.tables = blob + K3HUF_LAYER_HDR_BYTES;
    P.status = d_status;
    P.chunk_syms = cs;
    P.sub_syms = ss;
    P.gemv_x = static_cast<const uint8_t *>(d_x);
    P.gemv_y = d_y;
    P.gemv_cols = cols;
    P.gemv_ldx = 2 * cols;                     // X: n_vec rows of cols bf16
    P.gemv_ldy = te.n_values / cols;           // Y: n_vec rows of `rows` floats
    for (uint32_t s0 = 0; s0 < te.n_stripes; s0 += kMaxTasks) {
        const uint32_t s1 = std::min<uint32_t>(te.n_stripes, s0 + kMaxTasks);
        uint32_t items = 0;
        P.n_tasks = s1 - s0;
        for (uint32_t s = s0; s < s1; ++s) {
            const StripeEntry &e = L.stripes[te.first_stripe + s];
            StripeTask &t = P.task[s - s0];
            t.stripe = blob + e.blob_offset;
            t.out = nullptr;
            t.stripe_bytes = e.stripe_bytes;
            t.n_values = e.n_values;
            t.table = e.table;
            t.item_begin = items;
            t.tensor_stripe = s;
            items += items_of(e.n_values, cs, ss);
        }
        P.n_items = items;
        if (s0 == 0 && (flags & K3HUF_GEMV_ZERO_Y)) {
            rc = launch_zero_y(d_y, uint64_t(n_vec) * (te.n_values / cols), static_cast<cudaStream_t>(stream),
                               (flags & K3HUF_DECODE_EARLY_START) != 0);
            if (rc) return rc;
        }
        rc = launch_gemv(P, n_vec, static_cast<cudaStream_t>(stream), (flags & K3HUF_DECODE_EARLY_START) != 0);
        if (rc) return rc;
    }
    return K3HUF_OK;
}
}  // namespace

extern "C" int k3huf_gemv_layer(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer, size_t layer_bytes,
                                uint32_t tensor, uint64_t cols, const void *d_x, float *d_y, uint32_t *d_status,
                                void *stream) {
    return gemv_layer_impl(h_layer_hdr, hdr_bytes, d_layer, layer_bytes, tensor, cols, d_x, 1u, d_y, d_status, 0u,
                           stream);
}

extern "C" int k3huf_gemv_layer_ex(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer, size_t layer_bytes,
                                   uint32_t tensor, uint64_t cols, const void *d_x, float *d_y, uint32_t *d_status,
                                   uint32_t flags, void *stream) {
    if (flags & ~uint32_t(K3HUF_DECODE_EARLY_START | K3HUF_GEMV_ZERO_Y)) return K3HUF_E_ARG;
    return gemv_layer_impl(h_layer_hdr, hdr_bytes, d_layer, layer_bytes, tensor, cols, d_x, 1u, d_y, d_status, flags,
                           stream);
}

extern "C" int k3huf_gemv_layer_batch(const void *h_layer_hdr, size_t hdr_bytes, const void *d_layer,
                                      size_t layer_bytes, uint32_t tensor, uint64_t cols, const void *d_x,
                                      uint32_t n_vec, float *d_y, uint32_t *d_status, uint32_t flags, void *stream) {
    if (flags & ~uint32_t(K3HUF_DECODE_EARLY_START | K3HUF_GEMV_ZERO_Y)) return K3HUF_E_ARG;
    return gemv_layer_impl(h_layer_hdr, hdr_bytes, d_layer, layer_bytes, tensor, cols, d_x, n_vec, d_y, d_status,
                           flags, stream);
}
