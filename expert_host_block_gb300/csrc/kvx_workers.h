// A small pool of host worker threads for splitting descriptor packing.
//
// Packing a batch of one-chunk descriptors writes record i from descriptor i,
// so the work splits into independent index ranges. For large batches the
// calling thread and up to `workers` pool threads each take ranges. Workers
// spin briefly after a job (so the next call, such as the other direction of
// a burst, starts at once), then sleep on a condition variable. One job runs
// at a time: a caller that finds the pool busy does its job alone.
#pragma once

#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cstdlib>
#include <cstring>
#include <exception>
#include <mutex>
#include <thread>
#include <vector>

namespace kvx {

class Workers {
  public:
    // Worker threads (besides the caller): KVX_PACK_THREADS, else
    // min(3, hardware threads / 4); 0 disables the pool.
    static Workers &get()
    {
        static Workers w;
        return w;
    }

    int threads() const { return (int)pool_.size(); }

    // Run fn(part) for every part in [0, parts), spread over the caller and the
    // pool. Returns false without running anything when the pool is disabled
    // or busy with another caller's job.
    template <class Fn>
    bool run(int parts, Fn &&fn)
    {
        if (pool_.empty() || parts < 2)
            return false;
        std::unique_lock<std::mutex> busy(job_mu_, std::try_to_lock);
        if (!busy.owns_lock())
            return false;
        struct Thunk {
            static void call(void *f, int p) { (*static_cast<Fn *>(f))(p); }
        };
        uint64_t g;
        {
            std::lock_guard<std::mutex> lk(mu_);
            job_fn_ = &Thunk::call;
            job_arg_ = &fn;
            job_parts_ = parts;
            job_next_ = 0;
            left_.store(parts, std::memory_order_relaxed);
            g = gen_.load(std::memory_order_relaxed) + 1;
            job_gen_ = g;
            gen_.store(g, std::memory_order_release);
        }
        cv_.notify_all();
        work(g);
        while (left_.load(std::memory_order_acquire) != 0)
            std::this_thread::yield();
        return true;
    }

    ~Workers()
    {
        {
            std::lock_guard<std::mutex> g(mu_);
            stop_ = true;
            gen_.fetch_add(1, std::memory_order_release);
        }
        cv_.notify_all();
        for (std::thread &t : pool_)
            t.join();
    }

  private:
    Workers()
    {
        int n = (int)std::thread::hardware_concurrency() / 4;
        if (n > 3)
            n = 3;
        if (const char *v = std::getenv("KVX_PACK_THREADS")) {
            char *end = nullptr;
            const long x = std::strtol(v, &end, 10);
            if (end != v && !*end && x >= 0 && x <= 64)
                n = (int)x;
        }
        // A thread that cannot be started (resource limits) leaves the pool
        // smaller, down to none: packing then runs on the caller's thread.
        try {
            pool_.reserve(n);
            for (int i = 0; i < n; ++i)
                pool_.emplace_back([this] { loop(); });
        } catch (const std::exception &) {
        }
    }

    // Take parts of job `g` until none is left; a worker that wakes after its
    // job finished finds a newer generation (or no part) and takes nothing.
    void work(uint64_t g)
    {
        for (;;) {
            void (*fn)(void *, int);
            void *arg;
            int p;
            {
                std::lock_guard<std::mutex> lk(mu_);
                if (job_gen_ != g || job_next_ >= job_parts_)
                    return;
                p = job_next_++;
                fn = job_fn_;
                arg = job_arg_;
            }
            fn(arg, p);
            left_.fetch_sub(1, std::memory_order_acq_rel);
        }
    }

    void loop()
    {
        uint64_t seen = 0;
        for (;;) {
            // spin for a while, then sleep until the next job
            const auto until = std::chrono::steady_clock::now() + std::chrono::microseconds(300);
            uint64_t g = gen_.load(std::memory_order_acquire);
            while (g == seen && std::chrono::steady_clock::now() < until) {
                std::this_thread::yield();
                g = gen_.load(std::memory_order_acquire);
            }
            if (g == seen) {
                std::unique_lock<std::mutex> lk(mu_);
                cv_.wait(lk, [&] { return gen_.load(std::memory_order_acquire) != seen; });
                g = gen_.load(std::memory_order_acquire);
            }
            seen = g;
            {
                std::lock_guard<std::mutex> lk(mu_);
                if (stop_)
                    return;
            }
            work(g);
        }
    }

    std::vector<std::thread> pool_;
    std::mutex job_mu_;  // one job at a time
    std::mutex mu_;
    std::condition_variable cv_;
    std::atomic<uint64_t> gen_{0};
    std::atomic<int> left_{0};
    // the current job, guarded by mu_
    void (*job_fn_)(void *, int) = nullptr;
    void *job_arg_ = nullptr;
    int job_parts_ = 0, job_next_ = 0;
    uint64_t job_gen_ = 0;
    bool stop_ = false;
};

}  // namespace kvx
