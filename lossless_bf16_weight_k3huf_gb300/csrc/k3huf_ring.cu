// Pinned-host -> HBM streaming ring for k3_huf layers.
//
// The article "Kimi K3 纯 CPU 推理中的无损 Trunk 压缩：一次被解码速度判死刑的
// Huffman 压缩实验" (sections 背景 and 让方案被搁置的测量) streams the trunk
// layer by layer and charges decode against the feed rate ("two ledgers":
// bytes moved x bandwidth, and decode throughput); the engine's trunk ring
// keeps a second slot so reads overlap compute.  Here the feed is
// cudaMemcpyAsync from pinned host memory on a copy stream, double (or
// n-) buffered against the decode kernels on a compute stream, ordered by
// events: copy i waits until slot (i mod n) was decoded, decode i waits
// for copy i.  A staged ring also owns pinned host slots, filled from a
// file by the storage feed (k3huf_feed.cpp) while the previous layer is
// copied and decoded.
#include <cuda_runtime.h>

#include <chrono>
#include <new>
#include <vector>

#include "k3huf_internal.h"

struct k3huf_ring {
    int device = -1;
    int n_slots = 0;
    size_t slot_bytes = 0;
    std::vector<void *> slots;
    size_t host_slot_bytes = 0;
    std::vector<void *> host_raw;               // pinned allocations, staged rings only
    std::vector<void *> host_slots;             // 4096-aligned slots inside them
    cudaStream_t copy = nullptr, compute = nullptr;
};

namespace {

int fail(cudaError_t e) {
    k3huf::set_cuda_error(int(e));
    return K3HUF_E_CUDA;
}

void release(k3huf_ring *r) {
    for (void *p : r->slots)
        if (p) cudaFree(p);
    for (void *p : r->host_raw)
        if (p) cudaFreeHost(p);
    if (r->copy) cudaStreamDestroy(r->copy);
    if (r->compute) cudaStreamDestroy(r->compute);
    delete r;
}

}  // namespace

extern "C" int k3huf_ring_create(size_t slot_bytes, int n_slots, k3huf_ring **ring) {
    if (!ring || slot_bytes == 0 || n_slots < 1 || n_slots > 16) return K3HUF_E_ARG;
    k3huf_ring *r = new (std::nothrow) k3huf_ring;
    if (!r) return K3HUF_E_NOMEM;
    cudaError_t e = cudaGetDevice(&r->device);
    if (e != cudaSuccess) {
        release(r);
        return fail(e);
    }
    r->n_slots = n_slots;
    r->slot_bytes = slot_bytes;
    r->slots.assign(n_slots, nullptr);
    for (int i = 0; i < n_slots; ++i) {
        e = cudaMalloc(&r->slots[i], slot_bytes);
        if (e != cudaSuccess) {
            release(r);
            return fail(e);
        }
    }
    if ((e = cudaStreamCreateWithFlags(&r->copy, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&r->compute, cudaStreamNonBlocking)) != cudaSuccess) {
        release(r);
        return fail(e);
    }
    *ring = r;
    return K3HUF_OK;
}

extern "C" int k3huf_ring_create_staged(size_t slot_bytes, int n_slots, k3huf_ring **ring) {
    k3huf_ring *r = nullptr;
    int rc = k3huf_ring_create(slot_bytes, n_slots, &r);
    if (rc != K3HUF_OK) return rc;
    // file reads bypassing the page cache need 4096-byte aligned buffers; a
    // small pinned allocation may be carved from a pool at a finer alignment
    r->host_slot_bytes = (slot_bytes + 4095) / 4096 * 4096;
    r->host_raw.assign(size_t(n_slots), nullptr);
    r->host_slots.assign(size_t(n_slots), nullptr);
    for (int i = 0; i < n_slots; ++i) {
        cudaError_t e = cudaHostAlloc(&r->host_raw[size_t(i)], r->host_slot_bytes + 4096, cudaHostAllocDefault);
        if (e != cudaSuccess) {
            release(r);
            return fail(e);
        }
        const uintptr_t a = reinterpret_cast<uintptr_t>(r->host_raw[size_t(i)]);
        r->host_slots[size_t(i)] = reinterpret_cast<void *>((a + 4095) / 4096 * 4096);
    }
    *ring = r;
    return K3HUF_OK;
}

extern "C" int k3huf_ring_destroy(k3huf_ring *ring) {
    if (!ring) return K3HUF_E_ARG;
    cudaStreamSynchronize(ring->copy);
    cudaStreamSynchronize(ring->compute);
    release(ring);
    return K3HUF_OK;
}

extern "C" int k3huf_ring_run(k3huf_ring *r, int n_layers, const void *const *h_layers, const size_t *layer_bytes,
                              void *const *d_outs, const size_t *out_bytes, uint32_t *d_status,
                              k3huf_ring_stats_t *stats) {
    if (!r || n_layers < 1 || !h_layers || !layer_bytes || !d_outs || !out_bytes || !d_status) return K3HUF_E_ARG;
    for (int i = 0; i < n_layers; ++i)
        if (!h_layers[i] || !d_outs[i] || layer_bytes[i] > r->slot_bytes) return K3HUF_E_ARG;
    // validate every header before issuing any work
    uint64_t h2d = 0, decoded = 0;
    for (int i = 0; i < n_layers; ++i) {
        k3huf_layer_info_t info;
        int rc = k3huf_layer_info(h_layers[i], layer_bytes[i], &info);
        if (rc) return rc;
        if (info.blob_bytes > layer_bytes[i] || info.out_bytes > out_bytes[i]) return K3HUF_E_ARG;
        h2d += info.blob_bytes;
        decoded += info.raw_bytes;
    }
    // timing / ordering events: per layer copy start/end and decode start/end
    std::vector<cudaEvent_t> ev;
    auto make = [&](cudaEvent_t *out) {
        cudaError_t e = cudaEventCreate(out);
        if (e == cudaSuccess) ev.push_back(*out);
        return e;
    };
    auto cleanup = [&] {
        for (cudaEvent_t x : ev) cudaEventDestroy(x);
    };
    std::vector<cudaEvent_t> c0(n_layers), c1(n_layers), d0(n_layers), d1(n_layers);
    cudaEvent_t start, end;
    cudaError_t e = make(&start);
    if (e == cudaSuccess) e = make(&end);
    for (int i = 0; i < n_layers && e == cudaSuccess; ++i) {
        if ((e = make(&c0[i])) != cudaSuccess) break;
        if ((e = make(&c1[i])) != cudaSuccess) break;
        if ((e = make(&d0[i])) != cudaSuccess) break;
        e = make(&d1[i]);
    }
    if (e != cudaSuccess) {
        cleanup();
        return fail(e);
    }
    int rc = K3HUF_OK;
    e = cudaEventRecord(start, r->copy);
    for (int i = 0; i < n_layers && e == cudaSuccess && rc == K3HUF_OK; ++i) {
        const int slot = i % r->n_slots;
        const auto bytes = layer_bytes[i];
        if (i >= r->n_slots) e = cudaStreamWaitEvent(r->copy, d1[i - r->n_slots], 0);
        if (e == cudaSuccess) e = cudaEventRecord(c0[i], r->copy);
        if (e == cudaSuccess) e = cudaMemcpyAsync(r->slots[slot], h_layers[i], bytes, cudaMemcpyHostToDevice, r->copy);
        if (e == cudaSuccess) e = cudaEventRecord(c1[i], r->copy);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(r->compute, c1[i], 0);
        if (e == cudaSuccess) e = cudaEventRecord(d0[i], r->compute);
        if (e != cudaSuccess) break;
        rc = k3huf_decode_layer(h_layers[i], bytes, r->slots[slot], bytes, d_outs[i], out_bytes[i], d_status,
                                r->compute);
        if (rc == K3HUF_OK) e = cudaEventRecord(d1[i], r->compute);
    }
    if (e == cudaSuccess && rc == K3HUF_OK) e = cudaEventRecord(end, r->compute);
    cudaError_t es = cudaStreamSynchronize(r->copy);
    cudaError_t ec = cudaStreamSynchronize(r->compute);
    if (e == cudaSuccess) e = es != cudaSuccess ? es : ec;
    if (rc == K3HUF_OK && e == cudaSuccess && stats) {
        float t = 0;
        stats->total_ms = 0;
        stats->decode_ms = 0;
        stats->copy_ms = 0;
        if ((e = cudaEventElapsedTime(&t, start, end)) == cudaSuccess) stats->total_ms = t;
        for (int i = 0; i < n_layers && e == cudaSuccess; ++i) {
            if ((e = cudaEventElapsedTime(&t, d0[i], d1[i])) != cudaSuccess) break;
            stats->decode_ms += t;
            if ((e = cudaEventElapsedTime(&t, c0[i], c1[i])) != cudaSuccess) break;
            stats->copy_ms += t;
        }
        stats->h2d_bytes = h2d;
        stats->out_bytes = decoded;
    }
    cleanup();
    if (rc != K3HUF_OK) return rc;
    if (e != cudaSuccess) return fail(e);
    return K3HUF_OK;
}

extern "C" int k3huf_ring_run_file(k3huf_ring *r, k3huf_feed *feed, int n_layers, const uint64_t *file_offsets,
                                   const size_t *layer_bytes, void *const *d_outs, const size_t *out_bytes,
                                   uint32_t *d_status, k3huf_feed_stats_t *stats) {
    if (!r || !feed || n_layers < 1 || !file_offsets || !layer_bytes || !d_outs || !out_bytes || !d_status)
        return K3HUF_E_ARG;
    if (r->host_slots.empty()) return K3HUF_E_ARG;                 // not a staged ring
    for (int i = 0; i < n_layers; ++i)
        if (!d_outs[i] || layer_bytes[i] == 0 || layer_bytes[i] > r->slot_bytes || file_offsets[i] % 4096 != 0)
            return K3HUF_E_ARG;
    std::vector<cudaEvent_t> ev;
    auto make = [&](cudaEvent_t *out) {
        cudaError_t e = cudaEventCreate(out);
        if (e == cudaSuccess) ev.push_back(*out);
        return e;
    };
    auto cleanup = [&] {
        for (cudaEvent_t x : ev) cudaEventDestroy(x);
    };
    std::vector<cudaEvent_t> c0(n_layers), c1(n_layers), d0(n_layers), d1(n_layers);
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < n_layers && e == cudaSuccess; ++i) {
        if ((e = make(&c0[i])) != cudaSuccess) break;
        if ((e = make(&c1[i])) != cudaSuccess) break;
        if ((e = make(&d0[i])) != cudaSuccess) break;
        e = make(&d1[i]);
    }
    if (e != cudaSuccess) {
        cleanup();
        return fail(e);
    }
    using clock = std::chrono::steady_clock;
    const auto t_start = clock::now();
    double read_ms = 0;
    uint64_t read_bytes = 0, decoded = 0;
    int rc = K3HUF_OK;
    for (int i = 0; i < n_layers && e == cudaSuccess && rc == K3HUF_OK; ++i) {
        const int slot = i % r->n_slots;
        void *h = r->host_slots[size_t(slot)];
        // the host slot is free once the copy that last used it has finished
        if (i >= r->n_slots && (e = cudaEventSynchronize(c1[i - r->n_slots])) != cudaSuccess) break;
        const auto t0 = clock::now();
        rc = k3huf_feed_read(feed, file_offsets[i], layer_bytes[i], h, r->host_slot_bytes);
        read_ms += std::chrono::duration<double, std::milli>(clock::now() - t0).count();
        if (rc != K3HUF_OK) break;
        k3huf_layer_info_t info;
        if ((rc = k3huf_layer_info(h, layer_bytes[i], &info)) != K3HUF_OK) break;
        if (info.blob_bytes > layer_bytes[i] || info.out_bytes > out_bytes[i]) {
            rc = K3HUF_E_ARG;
            break;
        }
        read_bytes += layer_bytes[i];
        decoded += info.raw_bytes;
        if (i >= r->n_slots) e = cudaStreamWaitEvent(r->copy, d1[i - r->n_slots], 0);   // device slot free
        if (e == cudaSuccess) e = cudaEventRecord(c0[i], r->copy);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(r->slots[size_t(slot)], h, layer_bytes[i], cudaMemcpyHostToDevice, r->copy);
        if (e == cudaSuccess) e = cudaEventRecord(c1[i], r->copy);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(r->compute, c1[i], 0);
        if (e == cudaSuccess) e = cudaEventRecord(d0[i], r->compute);
        if (e != cudaSuccess) break;
        // the header is parsed from the host slot before this call returns
        rc = k3huf_decode_layer(h, layer_bytes[i], r->slots[size_t(slot)], layer_bytes[i], d_outs[i], out_bytes[i],
                                d_status, r->compute);
        if (rc == K3HUF_OK) e = cudaEventRecord(d1[i], r->compute);
    }
    cudaError_t es = cudaStreamSynchronize(r->copy);
    cudaError_t ec = cudaStreamSynchronize(r->compute);
    if (e == cudaSuccess) e = es != cudaSuccess ? es : ec;
    const double total_ms = std::chrono::duration<double, std::milli>(clock::now() - t_start).count();
    if (rc == K3HUF_OK && e == cudaSuccess && stats) {
        float t = 0;
        stats->total_ms = float(total_ms);
        stats->read_ms = float(read_ms);
        stats->copy_ms = 0;
        stats->decode_ms = 0;
        for (int i = 0; i < n_layers && e == cudaSuccess; ++i) {
            if ((e = cudaEventElapsedTime(&t, d0[i], d1[i])) != cudaSuccess) break;
            stats->decode_ms += t;
            if ((e = cudaEventElapsedTime(&t, c0[i], c1[i])) != cudaSuccess) break;
            stats->copy_ms += t;
        }
        stats->read_bytes = read_bytes;
        stats->out_bytes = decoded;
    }
    cleanup();
    if (rc != K3HUF_OK) return rc;
    if (e != cudaSuccess) return fail(e);
    return K3HUF_OK;
}
