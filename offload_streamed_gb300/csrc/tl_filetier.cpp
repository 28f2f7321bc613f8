// tl_filetier.cpp -- reader / writer threads of the file tier (see tl_filetier.h).
#include "tl_filetier.h"

#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <cerrno>
#include <chrono>
#include <condition_variable>
#include <cstring>
#include <deque>
#include <functional>
#include <memory>
#include <mutex>
#include <thread>
#include <utility>
#include <vector>

namespace tl {
namespace {

constexpr size_t kIoAlign = 4096;            // direct I/O: offsets, sizes and buffers
constexpr size_t kChunk = size_t(16) << 20;  // one pread / pwrite per chunk of a tile

double now_s() {
    return std::chrono::duration<double>(std::chrono::steady_clock::now().time_since_epoch()).count();
}

// All `n` bytes at `off`, retrying short transfers and EINTR.
bool pread_all(int fd, void* buf, size_t n, size_t off) {
    auto* p = static_cast<uint8_t*>(buf);
    while (n > 0) {
        const ssize_t r = ::pread(fd, p, n, off_t(off));
        if (r < 0 && errno == EINTR) continue;
        if (r <= 0) return false;
        p += r;
        off += size_t(r);
        n -= size_t(r);
    }
    return true;
}

bool pwrite_all(int fd, const void* buf, size_t n, size_t off) {
    const auto* p = static_cast<const uint8_t*>(buf);
    while (n > 0) {
        const ssize_t r = ::pwrite(fd, p, n, off_t(off));
        if (r < 0 && errno == EINTR) continue;
        if (r <= 0) return false;
        p += r;
        off += size_t(r);
        n -= size_t(r);
    }
    return true;
}

// A fixed set of threads running one parallel loop at a time: run(n, fn)
// calls fn(0) .. fn(n-1) spread over the threads and returns when all have
// returned (false if any did).
class ChunkPool {
public:
    explicit ChunkPool(int threads) {
        for (int t = 0; t < threads; ++t) th_.emplace_back([this] { work(); });
    }
    ~ChunkPool() {
        {
            std::lock_guard<std::mutex> g(m_);
            stop_ = true;
        }
        cv_.notify_all();
        for (auto& t : th_) t.join();
    }
    bool run(int n, const std::function<bool(int)>& fn) {
        std::unique_lock<std::mutex> lk(m_);
        job_ = &fn;
        n_ = n;
        next_.store(0);
        finished_ = 0;
        ok_ = true;
        ++gen_;
        cv_.notify_all();
        done_.wait(lk, [&] { return finished_ == int(th_.size()); });
        job_ = nullptr;
        return ok_;
    }

private:
    void work() {
        uint64_t seen = 0;
        for (;;) {
            const std::function<bool(int)>* job;
            int n;
            {
                std::unique_lock<std::mutex> lk(m_);
                cv_.wait(lk, [&] { return stop_ || gen_ != seen; });
                if (stop_) return;
                seen = gen_;
                job = job_;
                n = n_;
            }
            bool ok = true;
            for (int i = next_.fetch_add(1); i < n; i = next_.fetch_add(1)) ok = (*job)(i) && ok;
            std::lock_guard<std::mutex> g(m_);
            ok_ = ok_ && ok;
            if (++finished_ == int(th_.size())) done_.notify_all();
        }
    }
    std::vector<std::thread> th_;
    std::mutex m_;
    std::condition_variable cv_, done_;
    const std::function<bool(int)>* job_ = nullptr;
    int n_ = 0;
    std::atomic<int> next_{0};
    int finished_ = 0;
    bool ok_ = true;
    bool stop_ = false;
    uint64_t gen_ = 0;
};

}  // namespace

struct FileTier::Impl {
    int fd_w = -1, fd_dw = -1;
    int32_t n_tiles = 0;
    size_t tb = 0;
    int32_t S = 0, nio = 0;
    std::vector<void*> wbuf, dwbuf;      // 4096-aligned slots inside the allocations below
    std::vector<void*> wbase, dwbase;    // cudaHostAlloc pointers (not always page-aligned)
    std::vector<cudaEvent_t> wev, dwev;

    std::mutex m;
    std::condition_variable cv;
    bool failed = false, stop = false;
    std::string err;
    // read side: requested tiles not yet read, slots free to read into (in
    // release order; need_sync: the copy that last read it may still run),
    // and read tiles in request order
    std::deque<int32_t> pending;
    std::deque<int> free_w;
    std::vector<char> need_sync;
    std::deque<std::pair<int, int32_t>> ready;
    bool reading = false;
    // write side
    std::deque<int> free_dw;
    std::deque<std::pair<int, int32_t>> to_write;
    int writing = 0;
    FileTierStats st;

    std::unique_ptr<ChunkPool> rpool, wpool;
    std::thread reader, writer;

    int chunks() const { return int((tb + kChunk - 1) / kChunk); }
    size_t chunk_len(int c) const { return std::min(kChunk, tb - size_t(c) * kChunk); }

    void fail_locked(const std::string& what) {
        if (!failed) err = what;
        failed = true;
        cv.notify_all();
    }

    void read_loop() {
        for (;;) {
            int s;
            int32_t tile;
            bool sync_first;
            {
                std::unique_lock<std::mutex> lk(m);
                cv.wait(lk, [&] { return stop || (!failed && !pending.empty() && !free_w.empty()); });
                if (stop) return;
                tile = pending.front();
                pending.pop_front();
                s = free_w.front();
                free_w.pop_front();
                sync_first = need_sync[size_t(s)] != 0;
                reading = true;
            }
            bool ok = true;
            std::string what;
            if (sync_first && cudaEventSynchronize(wev[size_t(s)]) != cudaSuccess) {
                ok = false;
                what = std::string("waiting for a host->device copy: ") + cudaGetErrorString(cudaGetLastError());
            }
            const double t0 = now_s();
            if (ok) {
                uint8_t* dst = static_cast<uint8_t*>(wbuf[size_t(s)]);
                const size_t base = size_t(tile) * tb;
                ok = rpool->run(chunks(), [&](int c) {
                    return pread_all(fd_w, dst + size_t(c) * kChunk, chunk_len(c), base + size_t(c) * kChunk);
                });
                if (!ok) what = "reading W tile " + std::to_string(tile) + " from its file failed";
            }
            const double dt = now_s() - t0;
            std::lock_guard<std::mutex> g(m);
            reading = false;
            need_sync[size_t(s)] = 0;
            if (!ok) {
                free_w.push_front(s);
                fail_locked(what);
            } else {
                ready.emplace_back(s, tile);
                st.read_bytes += int64_t(tb);
                st.read_s += dt;
            }
            cv.notify_all();
        }
    }

    void write_loop() {
        for (;;) {
            int s;
            int32_t tile;
            {
                std::unique_lock<std::mutex> lk(m);
                cv.wait(lk, [&] { return stop || !to_write.empty(); });
                if (to_write.empty()) return;  // stop, nothing left to write
                s = to_write.front().first;
                tile = to_write.front().second;
                to_write.pop_front();
                ++writing;
            }
            bool ok = cudaEventSynchronize(dwev[size_t(s)]) == cudaSuccess;
            std::string what = ok ? std::string() : std::string("waiting for a device->host copy: ") +
                                                        cudaGetErrorString(cudaGetLastError());
            const double t0 = now_s();
            if (ok) {
                const uint8_t* src = static_cast<const uint8_t*>(dwbuf[size_t(s)]);
                const size_t base = size_t(tile) * tb;
                ok = wpool->run(chunks(), [&](int c) {
                    return pwrite_all(fd_dw, src + size_t(c) * kChunk, chunk_len(c), base + size_t(c) * kChunk);
                });
                if (!ok) what = "writing dW tile " + std::to_string(tile) + " to its file failed";
            }
            const double dt = now_s() - t0;
            std::lock_guard<std::mutex> g(m);
            --writing;
            free_dw.push_back(s);
            if (!ok) {
                fail_locked(what);
            } else {
                st.write_bytes += int64_t(tb);
                st.write_s += dt;
            }
            cv.notify_all();
        }
    }
};

FileTier* FileTier::open(const char* w_path, const char* dw_path, int32_t n_tiles, size_t tile_bytes,
                         int32_t host_slots, int32_t io_threads, std::string* why) {
    auto bad = [&](const std::string& w) -> FileTier* {
        if (why) *why = w;
        return nullptr;
    };
    if (!w_path || !dw_path) return bad("null file path");
    if (n_tiles < 1 || tile_bytes == 0) return bad("empty weight store");
    if (tile_bytes % kIoAlign) return bad("a tile (K * M/N * 2 bytes) must be a multiple of 4096 bytes for direct I/O");
    if (host_slots < 2 || host_slots > 64) return bad("host_slots must be in 2..64");
    if (io_threads < 1 || io_threads > 64) return bad("io_threads must be in 1..64");
    auto* p = new Impl();
    FileTier* t = new FileTier(p);
    p->n_tiles = n_tiles;
    p->tb = tile_bytes;
    p->S = host_slots;
    p->nio = io_threads;
    const size_t total = size_t(n_tiles) * tile_bytes;
    auto fail = [&](const std::string& w) -> FileTier* {
        delete t;
        return bad(w);
    };
    p->fd_w = ::open(w_path, O_RDONLY | O_DIRECT | O_CLOEXEC);
    if (p->fd_w < 0) return fail(std::string("opening the W file with direct I/O: ") + std::strerror(errno));
    struct stat sb;
    if (fstat(p->fd_w, &sb) != 0 || size_t(sb.st_size) < total)
        return fail("the W file is shorter than N tiles (" + std::to_string(total) + " bytes)");
    p->fd_dw = ::open(dw_path, O_WRONLY | O_CREAT | O_DIRECT | O_CLOEXEC, 0644);
    if (p->fd_dw < 0) return fail(std::string("opening the dW file with direct I/O: ") + std::strerror(errno));
    if (fstat(p->fd_dw, &sb) != 0) return fail("fstat of the dW file failed");
    if (size_t(sb.st_size) < total && ftruncate(p->fd_dw, off_t(total)) != 0)
        return fail(std::string("extending the dW file: ") + std::strerror(errno));
    auto align = [](void* q) {
        return reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(q) + kIoAlign - 1) & ~uintptr_t(kIoAlign - 1));
    };
    for (int s = 0; s < host_slots; ++s) {
        void* a = nullptr;
        void* b = nullptr;
        cudaEvent_t ea = nullptr, eb = nullptr;
        if (cudaHostAlloc(&a, tile_bytes + kIoAlign, cudaHostAllocPortable) != cudaSuccess ||
            cudaHostAlloc(&b, tile_bytes + kIoAlign, cudaHostAllocPortable) != cudaSuccess ||
            cudaEventCreateWithFlags(&ea, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&eb, cudaEventDisableTiming) != cudaSuccess) {
            if (a) cudaFreeHost(a);
            if (b) cudaFreeHost(b);
            if (ea) cudaEventDestroy(ea);
            if (eb) cudaEventDestroy(eb);
            const std::string e = cudaGetErrorString(cudaGetLastError());
            return fail("pinned host slots: " + e);
        }
        p->wbase.push_back(a);
        p->dwbase.push_back(b);
        p->wbuf.push_back(align(a));
        p->dwbuf.push_back(align(b));
        p->wev.push_back(ea);
        p->dwev.push_back(eb);
        p->free_w.push_back(s);
        p->free_dw.push_back(s);
    }
    p->need_sync.assign(size_t(host_slots), 0);
    p->rpool.reset(new ChunkPool(io_threads));
    p->wpool.reset(new ChunkPool(io_threads));
    p->reader = std::thread([p] { p->read_loop(); });
    p->writer = std::thread([p] { p->write_loop(); });
    return t;
}

FileTier::~FileTier() {
    Impl* p = p_;
    if (p->writer.joinable()) {
        std::string ignored;
        sync(&ignored);
    }
    {
        std::lock_guard<std::mutex> g(p->m);
        p->stop = true;
    }
    p->cv.notify_all();
    if (p->reader.joinable()) p->reader.join();
    if (p->writer.joinable()) p->writer.join();
    p->rpool.reset();
    p->wpool.reset();
    for (size_t s = 0; s < p->wbuf.size(); ++s) {
        cudaEventSynchronize(p->wev[s]);
        cudaEventSynchronize(p->dwev[s]);
        cudaFreeHost(p->wbase[s]);
        cudaFreeHost(p->dwbase[s]);
        cudaEventDestroy(p->wev[s]);
        cudaEventDestroy(p->dwev[s]);
    }
    if (p->fd_w >= 0) ::close(p->fd_w);
    if (p->fd_dw >= 0) ::close(p->fd_dw);
    delete p;
}

void FileTier::request(int32_t tile) {
    std::lock_guard<std::mutex> g(p_->m);
    p_->pending.push_back(tile);
    p_->cv.notify_all();
}

int FileTier::acquire_w(int32_t tile, std::string* why) {
    Impl* p = p_;
    std::unique_lock<std::mutex> lk(p->m);
    const double t0 = now_s();
    p->cv.wait(lk, [&] { return p->failed || !p->ready.empty() || (p->pending.empty() && !p->reading); });
    p->st.fetch_wait_s += now_s() - t0;
    if (p->failed) {
        if (why) *why = p->err;
        return -1;
    }
    if (p->ready.empty()) {
        if (why) *why = "internal: W tile " + std::to_string(tile) + " was not requested from the file tier";
        return -1;
    }
    const auto front = p->ready.front();
    if (front.second != tile) {
        if (why) *why = "internal: file tier read order does not match the fetch order";
        return -1;
    }
    p->ready.pop_front();
    return front.first;
}

const void* FileTier::w_slot(int s) const { return p_->wbuf[size_t(s)]; }
cudaEvent_t FileTier::w_event(int s) const { return p_->wev[size_t(s)]; }

void FileTier::release_w(int s) {
    std::lock_guard<std::mutex> g(p_->m);
    p_->need_sync[size_t(s)] = 1;
    p_->free_w.push_back(s);
    p_->cv.notify_all();
}

void FileTier::clear_requests() {
    Impl* p = p_;
    std::unique_lock<std::mutex> lk(p->m);
    p->pending.clear();
    p->cv.wait(lk, [&] { return !p->reading; });
    for (const auto& r : p->ready) p->free_w.push_back(r.first);
    p->ready.clear();
    p->cv.notify_all();
}

int FileTier::acquire_dw(std::string* why) {
    Impl* p = p_;
    std::unique_lock<std::mutex> lk(p->m);
    const double t0 = now_s();
    p->cv.wait(lk, [&] { return p->failed || !p->free_dw.empty(); });
    p->st.writeback_wait_s += now_s() - t0;
    if (p->failed) {
        if (why) *why = p->err;
        return -1;
    }
    const int s = p->free_dw.front();
    p->free_dw.pop_front();
    return s;
}

void* FileTier::dw_slot(int s) const { return p_->dwbuf[size_t(s)]; }
cudaEvent_t FileTier::dw_event(int s) const { return p_->dwev[size_t(s)]; }

void FileTier::commit_dw(int s, int32_t tile) {
    std::lock_guard<std::mutex> g(p_->m);
    p_->to_write.emplace_back(s, tile);
    p_->cv.notify_all();
}

bool FileTier::sync(std::string* why) {
    Impl* p = p_;
    std::unique_lock<std::mutex> lk(p->m);
    p->cv.wait(lk, [&] { return p->to_write.empty() && p->writing == 0; });
    if (p->failed) {
        if (why) *why = p->err;
        return false;
    }
    return true;
}

FileTierStats FileTier::stats() const {
    std::lock_guard<std::mutex> g(p_->m);
    return p_->st;
}

int32_t FileTier::host_slots() const { return p_->S; }
int32_t FileTier::io_threads() const { return p_->nio; }

}  // namespace tl
