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
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
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

void work(Job* job)
{
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

    int nt = threads > 0 ? threads : static_cast<int>(std::thread::hardware_concurrency());
    if (nt < 1) nt = 1;
    const int64_t nchunks = (n + kChunk - 1) / kChunk;
    if (nt > nchunks) nt = static_cast<int>(nchunks);
    std::vector<std::thread> pool;
    try {
        pool.reserve(static_cast<size_t>(nt - 1));
        for (int k = 1; k < nt; ++k) pool.emplace_back(work, &job);
    } catch (...) {
        // fewer helpers than asked: the chunks still all get done
    }
    work(&job); // the calling thread works too
    for (auto& th : pool) th.join();
    return ZERO_OK;
}
