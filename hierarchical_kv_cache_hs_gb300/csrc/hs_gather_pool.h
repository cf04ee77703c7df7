// A host thread pool for the copy-engine variant's gather (host code only).
#pragma once

#include <atomic>
#include <condition_variable>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

// A fixed set of host threads that run `fn(task)` for every task of a batch
// and return when all are done (used by the copy-engine variant's gather).
// Tasks are claimed from one word holding (batch number << 32 | next task),
// so a thread still finishing an earlier batch can never claim, or call the
// function of, a later one.
class GatherPool {
public:
    explicit GatherPool(int n)
    {
        for (int i = 0; i < n; ++i) threads_.emplace_back([this] { loop(); });
    }
    ~GatherPool()
    {
        {
            std::lock_guard<std::mutex> g(mu_);
            stop_ = true;
        }
        cv_.notify_all();
        for (auto& t : threads_) t.join();
    }
    void run(int ntasks, const std::function<void(int)>& fn)
    {
        if (ntasks <= 0) return;
        std::unique_lock<std::mutex> g(mu_);
        fn_ = &fn;
        ntasks_ = ntasks;
        left_ = ntasks;
        ++gen_;
        claim_.store((gen_ & 0xffffffffull) << 32);
        cv_.notify_all();
        done_.wait(g, [this] { return left_ == 0; });
        fn_ = nullptr;
    }

private:
    void loop()
    {
        unsigned long long seen = 0;
        for (;;) {
            const std::function<void(int)>* fn;
            int n;
            {
                std::unique_lock<std::mutex> g(mu_);
                cv_.wait(g, [&] { return stop_ || gen_ != seen; });
                if (stop_) return;
                seen = gen_;
                fn = fn_;
                n = ntasks_;
            }
            int done = 0;
            for (;;) {
                unsigned long long v = claim_.load();
                if ((v >> 32) != (seen & 0xffffffffull)) break;  // a later batch
                const unsigned t = (unsigned)(v & 0xffffffffull);
                if (t >= (unsigned)n) break;
                if (!claim_.compare_exchange_weak(v, v + 1)) continue;
                (*fn)((int)t);
                ++done;
            }
            if (done) {
                std::lock_guard<std::mutex> g(mu_);
                left_ -= done;
                if (left_ == 0) done_.notify_all();
            }
        }
    }
    std::vector<std::thread> threads_;
    std::mutex mu_;
    std::condition_variable cv_, done_;
    const std::function<void(int)>* fn_ = nullptr;
    int ntasks_ = 0;
    int left_ = 0;
    std::atomic<unsigned long long> claim_{0};
    unsigned long long gen_ = 0;
    bool stop_ = false;
};
