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
// for copy i.
#include <cuda_runtime.h>

#include <new>
#include <vector>

#include "k3huf_internal.h"

struct k3huf_ring {
    int device = -1;
    int n_slots = 0;
    size_t slot_bytes = 0;
    std::vector<void *> slots;
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
