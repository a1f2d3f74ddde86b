// ZeRO-Offload's update on the host: Adam on one shard of fp32 master /
// momentum / variance in host memory, from the fp16 gradient that crossed
// from the GPU, writing the fp16 weights that cross back.
//
// Sources (page title, section):
//  ZeRO 技术原理：进阶与 Offload §2.2 Offload 策略: the data-flow graph is cut
//    along the fp16 gradient and fp16 parameter edges; the O(M) parameter
//    update and float2half nodes run on the CPU next to the Adam state.
//  §2.3 扩展性: with ZeRO-2 each GPU's 1/N shard of gradients and state is
//    offloaded and at least one CPU process updates it.
//  §1.6.6 算子融合: the offloaded Adam is sped up with multithreading + SIMD.
//  深度学习专题：模型训练的数据并行（三） §（一）Adam 优化器 (the update).
//
// The arithmetic is the fused GPU step's, operation for operation, in IEEE
// binary32 (this file is built with -ffp-contract=off, so no multiply-add is
// contracted); fp16 conversions use the compiler's _Float16 (hardware
// conversion on AArch64, round to nearest even).
//
// Work is split into chunks of kChunk elements that the threads take from an
// atomic counter, so a thread slowed by another busy thread on its core only
// takes fewer chunks (a static split waits for the slowest thread; inside a
// CUDA host function that cost a third of the time).  Each chunk runs in three
// passes: widen the fp16 gradient into a float buffer, the fp32 Adam loop
// (only float loads and stores, branch-free, so it vectorises), narrow the
// new weights to fp16.
//
// The threads are a pool created on the first call and kept for the life of
// the process, so a call (and each piece of a pipelined offload step) pays
// no thread creation.
#include <sched.h>

#include <atomic>
#include <cmath>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include "zero_step.h"

namespace {

constexpr int64_t kChunk = 16384; // 64 KB of each fp32 stream: stays in the core's L2

struct HostScalars {
    float lr, b1, b2, omb1, omb2, bc1, bc2, bp1, bp2, eps;
};

inline float widen(uint16_t code)
{
    _Float16 h;
    std::memcpy(&h, &code, sizeof(h));
    return static_cast<float>(h);
}

inline uint16_t narrow(float x)
{
    const _Float16 h = static_cast<_Float16>(x);
    uint16_t code;
    std::memcpy(&code, &h, sizeof(code));
    return code;
}

template <int MODE>
void adam_floats(const float* __restrict g, float* __restrict w, float* __restrict m, float* __restrict v,
                 int64_t n, const HostScalars s)
{
    for (int64_t i = 0; i < n; ++i) {
        const float gi = g[i];
        const float gg = gi * gi;
        float m_new, v_new, m_hat, v_hat;
        if constexpr (MODE == ZERO_MODE_STANDARD) {
            m_new = s.b1 * m[i] + s.omb1 * gi;
            v_new = s.b2 * v[i] + s.omb2 * gg;
            m_hat = m_new / s.bc1;
            v_hat = v_new / s.bc2;
        } else if constexpr (MODE == ZERO_MODE_FOLDED_LITERAL) {
            m_new = (s.b1 * m[i] + s.omb1 * gi) / s.bc1;
            v_new = (s.b2 * v[i] + s.omb2 * gg) / s.bc2;
            m_hat = m_new;
            v_hat = v_new;
        } else {
            m_new = (s.b1 * (m[i] * s.bp1) + s.omb1 * gi) / s.bc1;
            v_new = (s.b2 * (v[i] * s.bp2) + s.omb2 * gg) / s.bc2;
            m_hat = m_new;
            v_hat = v_new;
        }
        const float denom = std::sqrt(v_hat) + s.eps;
        w[i] = w[i] - s.lr * (m_hat / denom);
        m[i] = m_new;
        v[i] = v_new;
    }
}

void adam_chunk(int mode, const uint16_t* g16, float* w, float* m, float* v, uint16_t* p16, int64_t n,
                const HostScalars& s, float* gbuf)
{
    for (int64_t i = 0; i < n; ++i) gbuf[i] = widen(g16[i]);
    switch (mode) {
    case ZERO_MODE_STANDARD: adam_floats<ZERO_MODE_STANDARD>(gbuf, w, m, v, n, s); break;
    case ZERO_MODE_FOLDED_LITERAL: adam_floats<ZERO_MODE_FOLDED_LITERAL>(gbuf, w, m, v, n, s); break;
    default: adam_floats<ZERO_MODE_FOLDED_STORAGE>(gbuf, w, m, v, n, s); break;
    }
    for (int64_t i = 0; i < n; ++i) p16[i] = narrow(w[i]);
}

// Worker threads that sleep on a condition variable between jobs.  One job
// runs at a time (concurrent callers queue on job_mu_); the caller works on
// it too and returns once every helper has finished, so the job's data may
// live on the caller's stack.  The pool is never destroyed: its threads are
// parked in a wait when the process exits.
class HostPool {
public:
    static HostPool& get()
    {
        static HostPool* pool = new HostPool(); // leaked on purpose (see above)
        return *pool;
    }

    int size() const { return static_cast<int>(threads_.size()); }

    // body(ctx) on the calling thread and on `helpers` pool threads.
    void run(int helpers, void (*body)(void*), void* ctx)
    {
        std::lock_guard<std::mutex> job(job_mu_);
        if (helpers > size()) helpers = size();
        {
            std::lock_guard<std::mutex> lk(mu_);
            body_ = body;
            ctx_ = ctx;
            want_ = helpers;
            pending_ = helpers;
            ++gen_;
        }
        if (helpers > 0) cv_.notify_all();
        body(ctx);
        std::unique_lock<std::mutex> lk(mu_);
        done_cv_.wait(lk, [&] { return pending_ == 0; });
    }

private:
    // One thread per CPU this process may run on (its affinity mask, which a
    // container may set below the machine's count), the caller included.
    static int usable_cpus()
    {
        cpu_set_t set;
        if (sched_getaffinity(0, sizeof(set), &set) == 0) {
            const int n = CPU_COUNT(&set);
            if (n > 0) return n;
        }
        const int hc = static_cast<int>(std::thread::hardware_concurrency());
        return hc > 0 ? hc : 1;
    }

    HostPool()
    {
        int n = usable_cpus() - 1;
        if (n > 1023) n = 1023;
        for (int i = 0; i < n; ++i) {
            try {
                threads_.emplace_back(&HostPool::worker, this, i);
            } catch (...) {
                break; // fewer helpers: every job still completes
            }
        }
    }

    void worker(int idx)
    {
        uint64_t seen = 0;
        for (;;) {
            void (*body)(void*) = nullptr;
            void* ctx = nullptr;
            {
                std::unique_lock<std::mutex> lk(mu_);
                cv_.wait(lk, [&] { return gen_ != seen; });
                seen = gen_;
                if (idx >= want_) continue;
                body = body_;
                ctx = ctx_;
            }
            body(ctx);
            std::lock_guard<std::mutex> lk(mu_);
            if (--pending_ == 0) done_cv_.notify_all();
        }
    }

    std::mutex job_mu_;
    std::mutex mu_;
    std::condition_variable cv_, done_cv_;
    uint64_t gen_ = 0;
    int want_ = 0;
    int pending_ = 0;
    void (*body_)(void*) = nullptr;
    void* ctx_ = nullptr;
    std::vector<std::thread> threads_;
};

struct Job {
    int mode;
    const uint16_t* g16;
    float* w;
    float* m;
    float* v;
    uint16_t* p16;
    int64_t n;
    HostScalars s;
    std::atomic<int64_t> next{0};
};

void work(void* arg)
{
    Job* job = static_cast<Job*>(arg);
    float gbuf[kChunk]; // 64 KB on the thread's stack
    const int64_t nchunks = (job->n + kChunk - 1) / kChunk;
    for (int64_t c = job->next.fetch_add(1); c < nchunks; c = job->next.fetch_add(1)) {
        const int64_t lo = c * kChunk;
        const int64_t len = job->n - lo < kChunk ? job->n - lo : kChunk;
        adam_chunk(job->mode, job->g16 + lo, job->w + lo, job->m + lo, job->v + lo, job->p16 + lo, len, job->s,
                   gbuf);
    }
}

} // namespace

extern "C" int zero_cpu_adam(const void* grad_fp16, float* master, float* m, float* v, void* params_fp16,
                             int64_t n, int64_t t, float lr, float beta1, float beta2, float eps, int32_t mode,
                             int32_t threads)
{
    if (n < 0 || t < 1 || mode < 0 || mode > 2) return ZERO_EINVAL;
    if (!std::isfinite(lr) || !std::isfinite(beta1) || !std::isfinite(beta2) || !std::isfinite(eps)) return ZERO_EINVAL;
    if (!(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f) || !(eps >= 0.0f)) return ZERO_EINVAL;
    if (threads < 0 || threads > 1024) return ZERO_EINVAL;
    if (n == 0) return ZERO_OK;
    if (!grad_fp16 || !master || !m || !v || !params_fp16) return ZERO_EINVAL;

    Job job;
    job.mode = mode;
    job.g16 = static_cast<const uint16_t*>(grad_fp16);
    job.w = master;
    job.m = m;
    job.v = v;
    job.p16 = static_cast<uint16_t*>(params_fp16);
    job.n = n;
    job.s.lr = lr;
    job.s.b1 = beta1;
    job.s.b2 = beta2;
    job.s.eps = eps;
    job.s.omb1 = 1.0f - beta1;
    job.s.omb2 = 1.0f - beta2;
    job.s.bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta1), static_cast<double>(t)));
    job.s.bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta2), static_cast<double>(t)));
    job.s.bp1 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta1), static_cast<double>(t - 1)));
    job.s.bp2 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta2), static_cast<double>(t - 1)));

    HostPool& pool = HostPool::get();
    int nt = threads > 0 ? threads : pool.size() + 1;
    const int64_t nchunks = (n + kChunk - 1) / kChunk;
    if (nt > nchunks) nt = static_cast<int>(nchunks);
    if (nt <= 1)
        work(&job);
    else
        pool.run(nt - 1, work, &job); // the calling thread works too
    return ZERO_OK;
}
