// Storage feed: reads container bytes from a file into host memory with
// pread, split across threads, through a descriptor opened with O_DIRECT
// where the filesystem allows it (the page cache is bypassed, as the
// article "AIBit-探索开源项目" (section 工作原理：架构, 读取检查点) reads its
// checkpoint).  Host code only; the ring (k3huf_ring.cu) stages the reads
// in pinned slots and overlaps them with the copies and the decode.
#include <fcntl.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <cerrno>
#include <cstdint>
#include <new>
#include <thread>
#include <vector>

#include "k3huf_internal.h"

struct k3huf_feed {
    int fd = -1;
    int direct = 0;
    int n_threads = 1;
};

namespace {

constexpr uint64_t kBlock = 4096;                  // O_DIRECT alignment of offsets, sizes and buffers
constexpr uint64_t kPiece = uint64_t(8) << 20;     // bytes per pread task

// Read [off, off + len) into dst; returns the bytes read (less only at the
// end of the file) or -1 on an error.
int64_t read_span(int fd, uint8_t *dst, uint64_t off, uint64_t len) {
    uint64_t got = 0;
    while (got < len) {
        const ssize_t r = pread(fd, dst + got, size_t(len - got), off_t(off + got));
        if (r < 0) {
            if (errno == EINTR) continue;
            return -1;
        }
        if (r == 0) break;                          // end of file
        got += uint64_t(r);
    }
    return int64_t(got);
}

}  // namespace

extern "C" int k3huf_feed_open(const char *path, int n_threads, k3huf_feed **feed) {
    if (!path || !feed || n_threads < 1 || n_threads > 64) return K3HUF_E_ARG;
    k3huf_feed *f = new (std::nothrow) k3huf_feed;
    if (!f) return K3HUF_E_NOMEM;
    f->n_threads = n_threads;
#ifdef O_DIRECT
    f->fd = open(path, O_RDONLY | O_DIRECT | O_CLOEXEC);
    if (f->fd >= 0) f->direct = 1;
#endif
    if (f->fd < 0) f->fd = open(path, O_RDONLY | O_CLOEXEC);   // filesystem without O_DIRECT
    if (f->fd < 0) {
        delete f;
        return K3HUF_E_IO;
    }
    *feed = f;
    return K3HUF_OK;
}

extern "C" int k3huf_feed_direct(const k3huf_feed *feed) {
    if (!feed) return K3HUF_E_ARG;
    return feed->direct;
}

extern "C" int k3huf_feed_read(k3huf_feed *f, uint64_t offset, size_t bytes, void *h_buf, size_t buf_bytes) {
    if (!f || !h_buf || bytes == 0 || offset % kBlock != 0 || reinterpret_cast<uintptr_t>(h_buf) % kBlock != 0)
        return K3HUF_E_ARG;
    const uint64_t span = (uint64_t(bytes) + kBlock - 1) / kBlock * kBlock;
    if (buf_bytes < span) return K3HUF_E_ARG;
    uint8_t *dst = static_cast<uint8_t *>(h_buf);
    const uint64_t n_pieces = (span + kPiece - 1) / kPiece;
    std::atomic<uint64_t> next{0};
    std::atomic<int> status{K3HUF_OK};
    auto worker = [&] {
        for (uint64_t p = next.fetch_add(1); p < n_pieces && status.load() == K3HUF_OK; p = next.fetch_add(1)) {
            const uint64_t a = p * kPiece, len = std::min(kPiece, span - a);
            const int64_t got = read_span(f->fd, dst + a, offset + a, len);
            // every byte below offset + bytes must come from the file
            const uint64_t need = std::min(len, uint64_t(bytes) - std::min<uint64_t>(a, bytes));
            if (got < 0 || uint64_t(got) < need) status.store(K3HUF_E_IO);
        }
    };
    const int n = int(std::min<uint64_t>(uint64_t(f->n_threads), n_pieces));
    if (n <= 1) {
        worker();
    } else {
        std::vector<std::thread> pool;
        pool.reserve(size_t(n));
        try {
            for (int i = 0; i < n; ++i) pool.emplace_back(worker);
        } catch (...) {
            status.store(K3HUF_E_NOMEM);
        }
        for (auto &t : pool) t.join();
    }
    return status.load();
}

extern "C" int k3huf_feed_close(k3huf_feed *feed) {
    if (!feed) return K3HUF_E_ARG;
    if (feed->fd >= 0) close(feed->fd);
    delete feed;
    return K3HUF_OK;
}
