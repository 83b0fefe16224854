// qpack.cpp -- the on-disk expert container and its reader (host code).
//
// One file holds every routed expert of a stack as a fixed-stride blob, so that a miss costs one
// positioned read and no index lookup (paotong.dev commentary on Swiftlet, paragraph on the .qpack
// container: experts repacked into fixed-stride blocks, one read per expert; alphalab.site
// "Swiftlet 實測資料解讀", section on SSD reads: pread per expert, no mmap, no page-cache pressure).
// Layout (little-endian):
//   bytes 0..4095   header: magic "MOEQPCK1", header bytes, version, moe_shape, layers, experts,
//                   blob bytes, stride, data offset, file bytes (the rest zero)
//   data offset     blob (layer l, expert e) at data_offset + (l * experts + e) * stride
// The stride is moe_expert_stride (a multiple of 4096) and the data offset 4096, so every blob
// starts on a 4096-byte boundary and is read with O_DIRECT when the file system allows it (bypassing
// the page cache, as the pages' reader does by not mapping the file). Reads of several blobs run
// in parallel on a small pool of threads, one positioned read each.
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <cerrno>
#include <condition_variable>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

#include "moe.h"
#include "qpack.h"

namespace {

constexpr char kMagic[8] = {'M', 'O', 'E', 'Q', 'P', 'C', 'K', '1'};
constexpr uint32_t kHeaderBytes = 4096;
constexpr uint32_t kVersion = 1;

struct Header {
    char magic[8];
    uint32_t header_bytes, version;
    moe_shape shape;
    uint32_t n_layers, n_experts;
    uint64_t blob_bytes, stride, data_offset, file_bytes;
};
static_assert(sizeof(Header) <= kHeaderBytes, "header fits its block");

// A fixed pool of reader threads running queued jobs; run() enqueues a batch and waits for it.
class Readers {
public:
    explicit Readers(int n)
    {
        for (int i = 0; i < n; ++i)
            threads_.emplace_back([this] { loop(); });
    }
    ~Readers()
    {
        {
            std::lock_guard<std::mutex> g(m_);
            stop_ = true;
        }
        cv_.notify_all();
        for (auto& t : threads_)
            t.join();
    }
    // Runs every job (on the pool, or inline without threads) and returns when all are done.
    void run(std::vector<std::function<void()>>& jobs)
    {
        if (threads_.empty() || jobs.size() <= 1) {
            for (auto& j : jobs)
                j();
            return;
        }
        std::unique_lock<std::mutex> g(m_);
        pending_ += jobs.size();
        for (auto& j : jobs)
            q_.push_back(std::move(j));
        cv_.notify_all();
        done_.wait(g, [this] { return pending_ == 0; });
    }

private:
    void loop()
    {
        for (;;) {
            std::function<void()> job;
            {
                std::unique_lock<std::mutex> g(m_);
                cv_.wait(g, [this] { return stop_ || !q_.empty(); });
                if (stop_ && q_.empty())
                    return;
                job = std::move(q_.front());
                q_.pop_front();
            }
            job();
            std::lock_guard<std::mutex> g(m_);
            if (--pending_ == 0)
                done_.notify_all();
        }
    }
    std::vector<std::thread> threads_;
    std::deque<std::function<void()>> q_;
    std::mutex m_;
    std::condition_variable cv_, done_;
    size_t pending_ = 0;
    bool stop_ = false;
};

moe_status qp_fail(moe_status st, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    moe::set_last_error(buf);
    return st;
}

// Positioned read or write of exactly n bytes (retrying short transfers and interrupts).
int full_pread(int fd, void* dst, size_t n, uint64_t off)
{
    uint8_t* p = static_cast<uint8_t*>(dst);
    while (n) {
        const ssize_t r = pread(fd, p, n, (off_t)off);
        if (r < 0) {
            if (errno == EINTR)
                continue;
            return errno;
        }
        if (r == 0)
            return EIO;  // past the end of the file
        p += r;
        n -= (size_t)r;
        off += (uint64_t)r;
    }
    return 0;
}

int full_pwrite(int fd, const void* src, size_t n, uint64_t off)
{
    const uint8_t* p = static_cast<const uint8_t*>(src);
    while (n) {
        const ssize_t r = pwrite(fd, p, n, (off_t)off);
        if (r < 0) {
            if (errno == EINTR)
                continue;
            return errno;
        }
        p += r;
        n -= (size_t)r;
        off += (uint64_t)r;
    }
    return 0;
}

}  // namespace

struct moe_qpack {
    int fd = -1;
    bool writable = false, direct = false;
    Header h{};
    Readers* readers = nullptr;
};

namespace moe {
namespace qp {

int read_many(moe_qpack* q, int n, const int32_t* layer, const int32_t* expert, void* const* dst)
{
    std::vector<int> err(n, 0);
    std::vector<std::function<void()>> jobs;
    jobs.reserve(n);
    for (int i = 0; i < n; ++i) {
        const uint64_t off = q->h.data_offset + ((uint64_t)layer[i] * q->h.n_experts + (uint64_t)expert[i]) * q->h.stride;
        void* d = dst[i];
        int* e = &err[i];
        jobs.push_back([q, d, off, e] { *e = full_pread(q->fd, d, q->h.stride, off); });
    }
    q->readers->run(jobs);
    for (int i = 0; i < n; ++i)
        if (err[i])
            return err[i];
    return 0;
}

uint64_t stride(const moe_qpack* q) { return q->h.stride; }
int n_layers(const moe_qpack* q) { return (int)q->h.n_layers; }
const moe_shape& shape(const moe_qpack* q) { return q->h.shape; }

}  // namespace qp
}  // namespace moe

extern "C" {

moe_status moe_qpack_create(const char* path, const moe_shape* shape, int32_t n_layers, moe_qpack** out)
{
    if (!path || !shape || !out || n_layers <= 0)
        return qp_fail(MOE_E_INVALID, "qpack create: NULL argument or n_layers <= 0");
    *out = nullptr;
    const size_t blob = moe_expert_bytes(shape, 0), stride = moe_expert_stride(shape, 0);
    if (blob == 0 || stride == 0 || shape->n_experts <= 0)
        return qp_fail(MOE_E_SHAPE, "qpack create: shape has no blob size");
    const int fd = open(path, O_RDWR | O_CREAT | O_TRUNC | O_CLOEXEC, 0644);
    if (fd < 0)
        return qp_fail(MOE_E_INVALID, "qpack create: cannot open %s (%s)", path, strerror(errno));
    auto* q = new moe_qpack();
    q->fd = fd;
    q->writable = true;
    memcpy(q->h.magic, kMagic, 8);
    q->h.header_bytes = kHeaderBytes;
    q->h.version = kVersion;
    q->h.shape = *shape;
    q->h.n_layers = (uint32_t)n_layers;
    q->h.n_experts = (uint32_t)shape->n_experts;
    q->h.blob_bytes = blob;
    q->h.stride = stride;
    q->h.data_offset = kHeaderBytes;
    q->h.file_bytes = kHeaderBytes + (uint64_t)n_layers * shape->n_experts * stride;
    std::vector<uint8_t> block(kHeaderBytes, 0);
    memcpy(block.data(), &q->h, sizeof(Header));
    int e = full_pwrite(fd, block.data(), kHeaderBytes, 0);
    if (!e && ftruncate(fd, (off_t)q->h.file_bytes) != 0)
        e = errno;
    if (e) {
        close(fd);
        delete q;
        return qp_fail(MOE_E_INVALID, "qpack create: writing %s failed (%s)", path, strerror(e));
    }
    *out = q;
    return MOE_OK;
}

moe_status moe_qpack_open(const char* path, int32_t flags, int32_t n_threads, moe_qpack** out)
{
    if (!path || !out || n_threads < 0)
        return qp_fail(MOE_E_INVALID, "qpack open: NULL argument or negative thread count");
    *out = nullptr;
    bool direct = false;
    int fd = -1;
    if (flags & MOE_QPACK_DIRECT) {
        fd = open(path, O_RDONLY | O_DIRECT | O_CLOEXEC);
        direct = fd >= 0;
    }
    if (fd < 0)
        fd = open(path, O_RDONLY | O_CLOEXEC);
    if (fd < 0)
        return qp_fail(MOE_E_INVALID, "qpack open: cannot open %s (%s)", path, strerror(errno));
    // the header through an aligned buffer (O_DIRECT needs one)
    void* block = nullptr;
    if (posix_memalign(&block, kHeaderBytes, kHeaderBytes) != 0) {
        close(fd);
        return qp_fail(MOE_E_NOMEM, "qpack open: no host memory for the header");
    }
    Header h{};
    int e = full_pread(fd, block, kHeaderBytes, 0);
    if (!e)
        memcpy(&h, block, sizeof(Header));
    free(block);
    struct stat st {};
    const bool sized = fstat(fd, &st) == 0;
    const bool tagged = !e && memcmp(h.magic, kMagic, 8) == 0;
    const size_t stride = tagged ? moe_expert_stride(&h.shape, 0) : 0;  // 0 for a shape without a blob
    if (!tagged || stride == 0 || h.header_bytes != kHeaderBytes || h.version != kVersion ||
        h.data_offset != kHeaderBytes || h.n_layers == 0 || h.n_experts == 0 || (int32_t)h.n_experts != h.shape.n_experts ||
        h.stride != stride || h.blob_bytes != moe_expert_bytes(&h.shape, 0) ||
        h.file_bytes != kHeaderBytes + (uint64_t)h.n_layers * h.n_experts * h.stride || !sized ||
        (uint64_t)st.st_size < h.file_bytes) {
        close(fd);
        return qp_fail(MOE_E_INVALID, "qpack open: %s is not a complete expert container of this format", path);
    }
    auto* q = new moe_qpack();
    q->fd = fd;
    q->direct = direct;
    q->h = h;
    q->readers = new Readers(n_threads);
    *out = q;
    return MOE_OK;
}

moe_status moe_qpack_info(const moe_qpack* q, moe_shape* shape, int32_t* n_layers, uint64_t* stride, int32_t* direct)
{
    if (!q)
        return qp_fail(MOE_E_INVALID, "qpack info: NULL container");
    if (shape)
        *shape = q->h.shape;
    if (n_layers)
        *n_layers = (int32_t)q->h.n_layers;
    if (stride)
        *stride = q->h.stride;
    if (direct)
        *direct = q->direct ? 1 : 0;
    return MOE_OK;
}

moe_status moe_qpack_write(moe_qpack* q, int32_t layer, int32_t expert, const void* h_blob)
{
    if (!q || !h_blob || !q->writable)
        return qp_fail(MOE_E_INVALID, "qpack write: NULL argument or container not opened for writing");
    if (layer < 0 || (uint32_t)layer >= q->h.n_layers || expert < 0 || (uint32_t)expert >= q->h.n_experts)
        return qp_fail(MOE_E_INVALID, "qpack write: layer %d / expert %d out of range", layer, expert);
    const uint64_t off = q->h.data_offset + ((uint64_t)layer * q->h.n_experts + (uint64_t)expert) * q->h.stride;
    const int e = full_pwrite(q->fd, h_blob, q->h.stride, off);
    if (e)
        return qp_fail(MOE_E_INVALID, "qpack write: %s", strerror(e));
    return MOE_OK;
}

moe_status moe_qpack_read(moe_qpack* q, int32_t layer, int32_t expert, void* h_dst)
{
    if (!q || !h_dst || !q->readers)
        return qp_fail(MOE_E_INVALID, "qpack read: NULL argument or container not opened for reading");
    if (layer < 0 || (uint32_t)layer >= q->h.n_layers || expert < 0 || (uint32_t)expert >= q->h.n_experts)
        return qp_fail(MOE_E_INVALID, "qpack read: layer %d / expert %d out of range", layer, expert);
    if (q->direct && (reinterpret_cast<uintptr_t>(h_dst) & (kHeaderBytes - 1)))
        return qp_fail(MOE_E_INVALID, "qpack read: direct reads need a 4096-byte aligned destination");
    const int e = moe::qp::read_many(q, 1, &layer, &expert, &h_dst);
    if (e)
        return qp_fail(MOE_E_INVALID, "qpack read: %s", strerror(e));
    return MOE_OK;
}

moe_status moe_qpack_close(moe_qpack* q)
{
    if (!q)
        return MOE_OK;
    int e = 0;
    if (q->writable && fsync(q->fd) != 0)
        e = errno;
    close(q->fd);
    delete q->readers;
    delete q;
    if (e)
        return qp_fail(MOE_E_INVALID, "qpack close: %s", strerror(e));
    return MOE_OK;
}

}  // extern "C"
