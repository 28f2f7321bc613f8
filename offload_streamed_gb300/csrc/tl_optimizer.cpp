// tl_optimizer.cpp -- host worker for the optimizer step of a streamed layer.
//
// After a backward call, each weight tile's dW is written to pinned host
// memory on the d2h copy stream, tile after tile.  The worker thread takes
// the tiles in the same order: it waits for the tile's copy event, then
// accumulates the gradient or runs the Adam update over the tile, split into
// row ranges across a small pool of CPU threads.  The update of early tiles
// thus overlaps the GPU's backward of later ones, and the forward of the next
// step can fetch a tile as soon as its own update is done.  The worker only
// waits on CUDA events; it never runs inside a CUDA callback, so nothing the
// GPU waits for depends on it except through the engine's host-side waits.
#include "tl_optimizer.h"

#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <deque>
#include <functional>
#include <mutex>
#include <thread>

namespace tl {

namespace {

// A fixed pool that runs fn(part) for part = 0..parts-1 and returns when all
// are done; the caller's thread runs part 0.
class Pool {
public:
    explicit Pool(int n) : n_(std::max(1, n)) {
        for (int i = 1; i < n_; ++i) threads_.emplace_back([this, i] { loop(i); });
    }
    ~Pool() {
        {
            std::lock_guard<std::mutex> g(mu_);
            stop_ = true;
        }
        cv_.notify_all();
        for (auto& t : threads_) t.join();
    }
    int size() const { return n_; }
    void run(const std::function<void(int)>& fn) {
        {
            std::lock_guard<std::mutex> g(mu_);
            fn_ = &fn;
            pending_ = n_ - 1;
            ++gen_;
        }
        cv_.notify_all();
        fn(0);
        std::unique_lock<std::mutex> lk(mu_);
        done_cv_.wait(lk, [this] { return pending_ == 0; });
        fn_ = nullptr;
    }

private:
    void loop(int i) {
        uint64_t seen = 0;
        for (;;) {
            const std::function<void(int)>* fn;
            {
                std::unique_lock<std::mutex> lk(mu_);
                cv_.wait(lk, [&] { return stop_ || gen_ != seen; });
                if (stop_) return;
                seen = gen_;
                fn = fn_;
            }
            (*fn)(i);
            {
                std::lock_guard<std::mutex> g(mu_);
                if (--pending_ == 0) done_cv_.notify_all();
            }
        }
    }
    int n_;
    std::vector<std::thread> threads_;
    std::mutex mu_;
    std::condition_variable cv_, done_cv_;
    const std::function<void(int)>* fn_ = nullptr;
    int pending_ = 0;
    uint64_t gen_ = 0;
    bool stop_ = false;
};

struct Job {
    bool step = false;
    int64_t step_no = 0;   // Adam step number (>= 1) for a step
    bool use_acc = false;  // step: add the accumulator; accumulate: false = overwrite
    std::vector<int> order;
    std::vector<cudaEvent_t> ev_w, ev_dw;
    int64_t id = 0;        // 1-based submission number
};

}  // namespace

class Optimizer {
public:
    Optimizer(const std::vector<Block>& tiles, const AdamHyper& hp, int threads)
        : tiles_(tiles), hp_(hp), pool_(threads > 0 ? threads : int(std::max(1u, std::thread::hardware_concurrency()))),
          read_done_(tiles.size(), 0), upd_done_(tiles.size(), 0) {
        worker_ = std::thread([this] { loop(); });
    }
    ~Optimizer() {
        {
            std::lock_guard<std::mutex> g(mu_);
            stop_ = true;
        }
        cv_.notify_all();
        worker_.join();
    }

    bool submit(bool step, const std::vector<int>& order, const std::vector<cudaEvent_t>& ev_w,
                const std::vector<cudaEvent_t>& ev_dw) {
        std::lock_guard<std::mutex> g(mu_);
        if (!error_.empty()) return false;
        Job j;
        j.step = step;
        j.order = order;
        j.ev_w = ev_w;
        j.ev_dw = ev_dw;
        j.id = ++submitted_;
        if (step) {
            j.step_no = ++steps_;
            j.use_acc = acc_filled_;
            acc_filled_ = false;
            upd_target_ = j.id;
        } else {
            j.use_acc = acc_filled_;  // false: the first accumulation overwrites
            acc_filled_ = true;
        }
        jobs_.push_back(std::move(j));
        cv_.notify_all();
        return true;
    }

    bool wait_tile(int g, bool update, double timeout_s) {
        std::unique_lock<std::mutex> lk(mu_);
        const int64_t target = update ? upd_target_ : submitted_;
        const auto& done = update ? upd_done_ : read_done_;
        const bool ok = done_cv_.wait_for(lk, std::chrono::duration<double>(timeout_s),
                                          [&] { return !error_.empty() || done[size_t(g)] >= target; });
        if (!ok && error_.empty()) error_ = "timed out waiting for the host optimizer";
        return error_.empty();
    }

    bool wait_all(double timeout_s) {
        std::unique_lock<std::mutex> lk(mu_);
        const int64_t target = submitted_;
        const bool ok = done_cv_.wait_for(lk, std::chrono::duration<double>(timeout_s),
                                          [&] { return !error_.empty() || finished_ >= target; });
        if (!ok && error_.empty()) error_ = "timed out waiting for the host optimizer";
        return error_.empty();
    }

    int64_t steps() const {
        std::lock_guard<std::mutex> g(mu_);
        return steps_;
    }
    double busy() const {
        std::lock_guard<std::mutex> g(mu_);
        return busy_s_;
    }
    std::string error() const {
        std::lock_guard<std::mutex> g(mu_);
        return error_;
    }

private:
    void fail(const std::string& why) {
        std::lock_guard<std::mutex> g(mu_);
        if (error_.empty()) error_ = why;
        done_cv_.notify_all();
    }

    void run_tile(const Job& j, int g) {
        const Block& b = tiles_[size_t(g)];
        const int parts = std::min<int64_t>(pool_.size(), std::max<int64_t>(1, b.rows));
        pool_.run([&](int part) {
            if (part >= parts) return;
            const int64_t r0 = b.rows * part / parts, r1 = b.rows * (part + 1) / parts;
            if (j.step)
                adam_rows(b, hp_, j.step_no, j.use_acc, r0, r1);
            else
                accumulate_rows(b, !j.use_acc, r0, r1);
        });
    }

    void loop() {
        for (;;) {
            Job j;
            {
                std::unique_lock<std::mutex> lk(mu_);
                cv_.wait(lk, [this] { return stop_ || !jobs_.empty(); });
                if (jobs_.empty()) return;  // stop_ with nothing left
                j = std::move(jobs_.front());
                jobs_.pop_front();
            }
            bool failed;
            {
                std::lock_guard<std::mutex> g(mu_);
                failed = !error_.empty();
            }
            for (int g : j.order) {
                if (!failed) {
                    cudaError_t e = cudaEventSynchronize(j.ev_dw[size_t(g)]);
                    if (e == cudaSuccess && j.step) e = cudaEventSynchronize(j.ev_w[size_t(g)]);
                    if (e != cudaSuccess) {
                        fail(std::string("host optimizer: waiting for a tile's copies: ") + cudaGetErrorString(e));
                        failed = true;
                    }
                }
                if (!failed) {
                    const auto t0 = std::chrono::steady_clock::now();
                    run_tile(j, g);
                    const double s = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
                    std::lock_guard<std::mutex> lk(mu_);
                    busy_s_ += s;
                }
                // a failed job still releases its waiters (they see the error)
                std::lock_guard<std::mutex> lk(mu_);
                read_done_[size_t(g)] = j.id;
                if (j.step) upd_done_[size_t(g)] = j.id;
                done_cv_.notify_all();
            }
            std::lock_guard<std::mutex> lk(mu_);
            finished_ = j.id;
            done_cv_.notify_all();
        }
    }

    std::vector<Block> tiles_;
    AdamHyper hp_;
    Pool pool_;
    mutable std::mutex mu_;
    std::condition_variable cv_, done_cv_;
    std::deque<Job> jobs_;
    std::vector<int64_t> read_done_, upd_done_;
    int64_t submitted_ = 0, finished_ = 0, steps_ = 0, upd_target_ = 0;
    bool acc_filled_ = false;
    bool stop_ = false;
    double busy_s_ = 0;
    std::string error_;
    std::thread worker_;
};

Optimizer* optimizer_new(const std::vector<Block>& tiles, const AdamHyper& hp, int threads) {
    return new Optimizer(tiles, hp, threads);
}
void optimizer_delete(Optimizer* o) {
    if (!o) return;
    o->wait_all(600.0);
    delete o;
}
bool optimizer_submit(Optimizer* o, bool step, const std::vector<int>& order, const std::vector<cudaEvent_t>& ev_w,
                      const std::vector<cudaEvent_t>& ev_dw) {
    return o->submit(step, order, ev_w, ev_dw);
}
bool optimizer_wait_update(Optimizer* o, int g, double timeout_s) { return o->wait_tile(g, true, timeout_s); }
bool optimizer_wait_read(Optimizer* o, int g, double timeout_s) { return o->wait_tile(g, false, timeout_s); }
bool optimizer_wait_all(Optimizer* o, double timeout_s) { return o->wait_all(timeout_s); }
int64_t optimizer_steps(const Optimizer* o) { return o->steps(); }
double optimizer_busy_seconds(const Optimizer* o) { return o->busy(); }
std::string optimizer_error(const Optimizer* o) { return o->error(); }

}  // namespace tl
