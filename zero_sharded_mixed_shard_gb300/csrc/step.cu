// The fused ZeRO step for GB300 (sm_103a): reduce-scatter of the P simulated
// ranks' fp16 gradients, fp32 Adam on the shard, fp16 cast and the write into
// the gathered parameter vector -- one pass over HBM, no intermediate buffer.
//
// Sources (page title, section):
//  深度学习专题：模型训练的数据并行（三） §（一）Adam 优化器: w_{t+1} = w_t - lr *
//    m_{t+1} / (sqrt(v_{t+1}) + eps) with the bias correction divided into the
//    moments; §（四）ZeRO-2 优化原理 第二步..第五步: reduce-scatter of the
//    gradient mean over elements s_k..e_k, shard-local moment and weight
//    update, all-gather of the updated parameters.
//  ZeRO 技术原理：进阶与 Offload §1.1.5 Reduce-Scatter, §1.1.6 All-Gather,
//    §1.4 (fp16 parameters and gradients, fp32 master / momentum / variance),
//    reference [10] Kingma & Ba (the standard bias-corrected Adam).
//  ZeRO 原理：把模型状态切到多张 GPU 上: the owning GPU updates its fp32
//    master copy and writes it back as fp16.
//  高效AI 第19讲：分布式训练（第一部分） 通信原语: g = (1/N) Σ g_i.
//
// Also plain SGD and SGD with momentum (same pages, §（一） and §1.1.1), which
// skip the state streams they do not use.
//
// The path is elementwise and HBM-bound (2P + 26 bytes moved per element
// against about 15 fp32 operations), so there are no tensor cores here.  Two
// kernels: the bulk-copy pipeline (one CTA per SM, TMA bulk copies of whole
// 4 KB rows into four shared-memory stages, bounded mbarrier waits) when
// every stream shares one 16-byte phase and the problem has a few tiles per
// SM, and a vector kernel (V consecutive elements per thread per iteration of
// a grid-stride loop) for small or misaligned problems.  Every arithmetic
// operation is an explicitly rounded fp32 intrinsic, so no multiply-add
// contraction can change a result.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>
#include <utility>
#include <vector>

#include "zero_step.h"

namespace {

constexpr int kThreads = 256;
constexpr int kRankBatch = 8; // gradient loads issued together per thread

// Arguments of one launch over a contiguous element range [0, n) of a shard
// or of the whole vector; every pointer already points at element 0.
struct StepArgs {
    const __half* g;    // rank 0's gradient for element 0
    long long stride;   // elements between ranks
    float* w;           // fp32 master weights
    float* m;           // fp32 first moment
    float* v;           // fp32 second moment
    __half* p;          // fp16 output (gathered parameter vector)
    long long n;        // elements in the range
    long long head;     // leading elements processed one by one (alignment)
    int P;              // ranks
    int p_pow2;         // P is a power of two: g * (1/P) == g / P exactly
    float inv_p;        // RN(1/P), an IEEE division on the host (exact when p_pow2)
    float lr, b1, b2, omb1, omb2, bc1, bc2, bp1, bp2, eps;
    unsigned int poison_tx; // diagnostic only: extra bytes CTA 0's first barrier expects (0 otherwise)
};

// ---------------------------------------------------------------------------
// Per-element arithmetic
// ---------------------------------------------------------------------------

// s / p correctly rounded without a divide, for finite nonzero s: with
// r = RN(1/p), q = RN(s r) is within a few ulp of s / p, the remainder
// s - q p is formed exactly by one fused multiply-add, and one correction
// step q + (s - q p) r rounds to the quotient (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990).  That the last step rounds correctly is a property of p:
// zero_selftest_mean_division checks it against the correctly rounded
// divide for every fp32 significand and every p from 1 to 1024, which covers
// every nonzero sum of fp16 gradients (they lie in [2^-24, 2^27), where
// scaling s by a power of two scales every step exactly).
__device__ __forceinline__ float div_by_count(float s, float p, float r)
{
    const float q = __fmul_rn(s, r);
    const float e = __fmaf_rn(-q, p, s);
    return __fmaf_rn(e, r, q);
}

template <int PT>
__device__ __forceinline__ float finish_mean(float sum, const StepArgs& a)
{
    if constexpr (PT > 0 && (PT & (PT - 1)) == 0) {
        return __fmul_rn(sum, 1.0f / static_cast<float>(PT));
    } else {
        if (a.p_pow2) return __fmul_rn(sum, a.inv_p);
        // +-0 / P = +-0, +-inf / P = +-inf, NaN stays NaN
        return (sum == 0.0f || !isfinite(sum)) ? sum
                                               : div_by_count(sum, static_cast<float>(PT > 0 ? PT : a.P), a.inv_p);
    }
}

// IEEE quotients whose operands are infinite or zero are formed directly:
// CUDA's correctly rounded divide and square root are slow on such operands
// (measured: the step on all-zero gradients and moments ran 2.6x slower),
// and they are common -- once the literal folded reading overflows v every
// element is infinite, and a parameter whose gradient and moments are still
// exactly zero (an embedding row no batch has touched) has zero numerators.
// The results are the IEEE 754 ones.
//   x / d for d positive and finite (the bias corrections): inf stays inf,
//   a zero stays the same zero.
template <int G>
__device__ __forceinline__ float div_by_positive(float x, float d)
{
    if constexpr (G == 0) return __fdiv_rn(x, d);
    return (isinf(x) || x == 0.0f) ? x : __fdiv_rn(x, d); // inf / d = inf, +-0 / d = +-0
}

__device__ __forceinline__ bool is_pos_inf(float x) { return x == __int_as_float(0x7f800000); }

//   sqrt(+inf) = +inf, sqrt(+-0) = +-0 (every other input goes to the
//   rounded square root).
template <int G>
__device__ __forceinline__ float sqrt_rn(float x)
{
    if constexpr (G == 0) return __fsqrt_rn(x);
    return (is_pos_inf(x) || x == 0.0f) ? x : __fsqrt_rn(x); // sqrt(+-0) = +-0
}

//   x / +inf: a zero carrying x's sign for finite x, NaN for infinite or NaN x;
//   +-0 / d = +-0 for finite d > 0.
template <int G>
__device__ __forceinline__ float div_rn(float x, float d)
{
    if constexpr (G == 0) return __fdiv_rn(x, d);
    if (is_pos_inf(d)) return isfinite(x) ? copysignf(0.0f, x) : __int_as_float(0x7fffffff);
    if (x == 0.0f && d > 0.0f) return x; // +-0 / d = +-0 for d > 0 (finite here)
    return __fdiv_rn(x, d);
}

// The state streams a mode reads and writes: Adam all three, SGD with
// momentum master and m, plain SGD master only.
constexpr bool uses_m(int mode) { return mode != ZERO_MODE_SGD; }
constexpr bool uses_v(int mode) { return mode <= ZERO_MODE_FOLDED_STORAGE; }
constexpr int state_rows(int mode) { return 1 + (uses_m(mode) ? 1 : 0) + (uses_v(mode) ? 1 : 0); }

// Adam on one element; w, m, v updated in place.  G = 1 takes the shortcuts
// above for infinite operands, G = 0 calls the rounded intrinsics directly
// (same results; only the speed on infinite operands differs).
template <int MODE, int G = 1>
__device__ __forceinline__ void adam_elem(const StepArgs& a, float g, float& w, float& m, float& v)
{
    if constexpr (MODE == ZERO_MODE_SGD) {
        // w <- w - lr * g (深度学习专题：模型训练的数据并行（三） §（一）)
        w = __fsub_rn(w, __fmul_rn(a.lr, g));
        return;
    } else if constexpr (MODE == ZERO_MODE_MOMENTUM) {
        // m <- b1 * m + g, w <- w - lr * m
        const float mn = __fadd_rn(__fmul_rn(a.b1, m), g);
        w = __fsub_rn(w, __fmul_rn(a.lr, mn));
        m = mn;
        return;
    }
    const float gg = __fmul_rn(g, g);
    float m_new, v_new, m_hat, v_hat;
    if constexpr (MODE == ZERO_MODE_STANDARD) {
        m_new = __fadd_rn(__fmul_rn(a.b1, m), __fmul_rn(a.omb1, g));
        v_new = __fadd_rn(__fmul_rn(a.b2, v), __fmul_rn(a.omb2, gg));
        m_hat = div_by_positive<G>(m_new, a.bc1);
        v_hat = div_by_positive<G>(v_new, a.bc2);
    } else if constexpr (MODE == ZERO_MODE_FOLDED_LITERAL) {
        m_new = div_by_positive<G>(__fadd_rn(__fmul_rn(a.b1, m), __fmul_rn(a.omb1, g)), a.bc1);
        v_new = div_by_positive<G>(__fadd_rn(__fmul_rn(a.b2, v), __fmul_rn(a.omb2, gg)), a.bc2);
        m_hat = m_new;
        v_hat = v_new;
    } else {
        m_new = div_by_positive<G>(__fadd_rn(__fmul_rn(a.b1, __fmul_rn(m, a.bp1)), __fmul_rn(a.omb1, g)), a.bc1);
        v_new = div_by_positive<G>(__fadd_rn(__fmul_rn(a.b2, __fmul_rn(v, a.bp2)), __fmul_rn(a.omb2, gg)), a.bc2);
        m_hat = m_new;
        v_hat = v_new;
    }
    const float denom = __fadd_rn(sqrt_rn<G>(v_hat), a.eps);
    const float upd = div_rn<G>(m_hat, denom);
    w = __fsub_rn(w, __fmul_rn(a.lr, upd));
    m = m_new;
    v = v_new;
}

// ---------------------------------------------------------------------------
// Vector loads and stores of V consecutive elements (streaming cache hints:
// every byte is touched once per step)
// ---------------------------------------------------------------------------

template <int V> struct HalfRaw;
template <> struct HalfRaw<8> { uint4 u; };
template <> struct HalfRaw<4> { uint2 u; };
template <> struct HalfRaw<2> { unsigned int u; };
template <> struct HalfRaw<1> { unsigned short u; };

template <int V>
__device__ __forceinline__ HalfRaw<V> load_halves(const __half* p)
{
    HalfRaw<V> r;
    if constexpr (V == 8) r.u = __ldcs(reinterpret_cast<const uint4*>(p));
    else if constexpr (V == 4) r.u = __ldcs(reinterpret_cast<const uint2*>(p));
    else if constexpr (V == 2) r.u = __ldcs(reinterpret_cast<const unsigned int*>(p));
    else r.u = __ldcs(reinterpret_cast<const unsigned short*>(p));
    return r;
}

__device__ __forceinline__ float2 u32_to_float2(unsigned int x)
{
    __half2 h;
    static_assert(sizeof(h) == sizeof(x), "half2 is 4 bytes");
    memcpy(&h, &x, sizeof(x));
    return __half22float2(h); // exact widening
}

// acc[j] = acc[j] + fp32(halves[j]), one rounded add per element
template <int V>
__device__ __forceinline__ void accumulate(float (&acc)[V], const HalfRaw<V>& r)
{
    if constexpr (V == 1) {
        acc[0] = __fadd_rn(acc[0], __half2float(__ushort_as_half(r.u)));
    } else {
        unsigned int words[V / 2];
        if constexpr (V == 8) { words[0] = r.u.x; words[1] = r.u.y; words[2] = r.u.z; words[3] = r.u.w; }
        else if constexpr (V == 4) { words[0] = r.u.x; words[1] = r.u.y; }
        else { words[0] = r.u; }
#pragma unroll
        for (int q = 0; q < V / 2; ++q) {
            const float2 f = u32_to_float2(words[q]);
            acc[2 * q] = __fadd_rn(acc[2 * q], f.x);
            acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], f.y);
        }
    }
}

template <int V>
__device__ __forceinline__ void load_floats(const float* p, float (&x)[V])
{
    if constexpr (V == 8) {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
        const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else if constexpr (V == 4) {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    } else if constexpr (V == 2) {
        const float2 a = __ldcs(reinterpret_cast<const float2*>(p));
        x[0] = a.x; x[1] = a.y;
    } else {
        x[0] = __ldcs(p);
    }
}

template <int V>
__device__ __forceinline__ void store_floats(float* p, const float (&x)[V])
{
    if constexpr (V == 8) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
        __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(x[4], x[5], x[6], x[7]));
    } else if constexpr (V == 4) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
    } else if constexpr (V == 2) {
        __stcs(reinterpret_cast<float2*>(p), make_float2(x[0], x[1]));
    } else {
        __stcs(p, x[0]);
    }
}

__device__ __forceinline__ unsigned int pack_half2_rn(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi); // round to nearest even, each half
    unsigned int x;
    memcpy(&x, &h, sizeof(x));
    return x;
}

template <int V>
__device__ __forceinline__ void store_halves(__half* p, const float (&x)[V])
{
    if constexpr (V == 8) {
        __stcs(reinterpret_cast<uint4*>(p),
               make_uint4(pack_half2_rn(x[0], x[1]), pack_half2_rn(x[2], x[3]),
                          pack_half2_rn(x[4], x[5]), pack_half2_rn(x[6], x[7])));
    } else if constexpr (V == 4) {
        __stcs(reinterpret_cast<uint2*>(p), make_uint2(pack_half2_rn(x[0], x[1]), pack_half2_rn(x[2], x[3])));
    } else if constexpr (V == 2) {
        __stcs(reinterpret_cast<unsigned int*>(p), pack_half2_rn(x[0], x[1]));
    } else {
        __stcs(reinterpret_cast<unsigned short*>(p), __half_as_ushort(__float2half_rn(x[0])));
    }
}

// ---------------------------------------------------------------------------
// V consecutive elements starting at i: reduce over ranks, Adam, cast, store
// ---------------------------------------------------------------------------

template <int MODE, int V, int PT>
__device__ __forceinline__ void step_elems(const StepArgs& a, long long i)
{
    const int P = PT > 0 ? PT : a.P;
    // state loads first so they are in flight with the gradient loads
    float w[V], m[V] = {}, v[V] = {};
    load_floats<V>(a.w + i, w);
    if constexpr (uses_m(MODE)) load_floats<V>(a.m + i, m);
    if constexpr (uses_v(MODE)) load_floats<V>(a.v + i, v);

    // reduce-scatter (own slice): fp32 sum in rank order 0..P-1 from +0
    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.0f;
    const __half* gp = a.g + i;
    int r = 0;
    constexpr int kOuter = (PT / kRankBatch) > 0 ? (PT / kRankBatch) : 1;
#pragma unroll kOuter
    for (; r + kRankBatch <= P; r += kRankBatch) {
        HalfRaw<V> buf[kRankBatch];
#pragma unroll
        for (int u = 0; u < kRankBatch; ++u) buf[u] = load_halves<V>(gp + (long long)u * a.stride);
#pragma unroll
        for (int u = 0; u < kRankBatch; ++u) accumulate<V>(acc, buf[u]);
        gp += (long long)kRankBatch * a.stride;
    }
    if constexpr (PT > 0 || V == 8 || V == 1) {
        constexpr int kInner = PT > 0 ? kRankBatch : 1;
#pragma unroll kInner
        for (; r < P; ++r) {
            accumulate<V>(acc, load_halves<V>(gp));
            gp += a.stride;
        }
    } else {
        // the last P mod 8 ranks, a count known only at run time: their loads
        // issued together under predicates, then summed in rank order
        // (measured, rows off the 16-byte phase, width 4: P = 3 0.78 -> 0.98,
        // 5 0.73 -> 0.94, 12 0.84 -> 0.97 of the copy roofline; width 2
        // alike.  At width 8 the buffer spills, at width 1 it costs CTAs per
        // SM: both keep the one-rank loop)
        const int rem = P - r;
        HalfRaw<V> buf[kRankBatch];
#pragma unroll
        for (int u = 0; u < kRankBatch; ++u)
            if (u < rem) buf[u] = load_halves<V>(gp + (long long)u * a.stride);
#pragma unroll
        for (int u = 0; u < kRankBatch; ++u)
            if (u < rem) accumulate<V>(acc, buf[u]);
    }

#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = finish_mean<PT>(acc[j], a); // the gradient means
    // the shortcuts for infinite and zero operands only in warps that need
    // them (the same warp-uniform dispatch as the bulk pipeline)
    bool special = false;
    if constexpr (MODE <= ZERO_MODE_FOLDED_STORAGE) {
#pragma unroll
        for (int j = 0; j < V; ++j)
            special |= !(isfinite(acc[j]) && isfinite(m[j]) && isfinite(v[j])) || acc[j] == 0.0f;
    }
    if (__any_sync(__activemask(), special)) {
#pragma unroll
        for (int j = 0; j < V; ++j) adam_elem<MODE, 1>(a, acc[j], w[j], m[j], v[j]);
    } else {
#pragma unroll
        for (int j = 0; j < V; ++j) adam_elem<MODE, 0>(a, acc[j], w[j], m[j], v[j]);
    }
    store_floats<V>(a.w + i, w);
    if constexpr (uses_m(MODE)) store_floats<V>(a.m + i, m);
    if constexpr (uses_v(MODE)) store_floats<V>(a.v + i, v);
    store_halves<V>(a.p + i, w); // all-gather: element i of the full vector
}

// Resident CTAs per SM the vector kernel is compiled for (its registers
// then fit 4 CTAs of 256 threads).  Measured on GB300 with L2 flushed: for
// P = 4, 8 and the generic instance, problems that need more than one wave
// at the default 3 CTAs per SM gain 8-22 % (1 M elements: P = 4 13.9 ->
// 12.8 us, P = 13 23.0 -> 18.0 us) and smaller ones are unchanged; for
// P = 16 the register cap costs up to 18 %, so the wider instances keep
// their registers.
constexpr int vector_min_blocks(int PT) { return PT == 0 || PT <= 8 ? 4 : 1; }

template <int MODE, int V, int PT>
__global__ void __launch_bounds__(kThreads, vector_min_blocks(PT)) zero_fused_step_kernel(const StepArgs a)
{
    const long long tid = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
    const long long nthreads = static_cast<long long>(gridDim.x) * kThreads;
    const long long body = (a.n - a.head) / V; // full V-element vectors after the head
    const long long tail_start = a.head + body * V;
    // ragged ends: fewer than V elements each, one element per thread
    if (tid < a.head) step_elems<MODE, 1, PT>(a, tid);
    if (tid < a.n - tail_start) step_elems<MODE, 1, PT>(a, tail_start + tid);
    for (long long c = tid; c < body; c += nthreads) step_elems<MODE, V, PT>(a, a.head + c * V);
}

// ---------------------------------------------------------------------------
// TMA bulk-copy pipeline: the main path when every stream shares one 16-byte
// phase.  One CTA per SM walks its tiles of kTile elements.  A unit of work is
// (tile, chunk of kChunkRanks ranks): one bulk copy of kTile*2 bytes per rank
// of the chunk, plus the tile's master / m / v rows with the first chunk, all
// landing in one of kStages shared-memory stages and counted by that stage's
// mbarrier.  Warp 0 issues the copies (thread 0 alone when a tile is one
// chunk, one row per lane otherwise); every thread then reads its elements of
// each row from shared memory, accumulates the chunk's ranks in rank order,
// and after the last chunk runs Adam and stores the results with streaming
// stores.  With P known only at run time, the last chunk's rank count is a
// compile-time parameter and each tile's first and last chunks are peeled,
// so every chunk is summed by straight-line code.  Copies of whole 4 KB rows keep the copy engine's
// issue rate far from the limit and keep every DRAM stream long and sequential.
// ---------------------------------------------------------------------------

constexpr int kTile = 2048;
constexpr int kChunkRanks = 8;
constexpr int kStages = 4;
constexpr uint32_t kGradBytes = kChunkRanks * kTile * 2;          // 32 KB of gradient rows
constexpr uint32_t kStageBytes = kGradBytes + 3 * kTile * 4;      // + 24 KB of fp32 state
constexpr size_t kBulkSmem = size_t(kStages) * kStageBytes;       // 224 KB
constexpr unsigned long long kWaitLimitNs = 2000000000ull;        // a bounded wait gives up after 2 s

// Bounded waits that gave up (0 in every correct run); read by zero_device_timeouts.
__device__ unsigned int g_wait_timeouts;

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(smem_addr(bar)), "r"(parity)
                 : "memory");
    return done != 0;
}

// Wait for the phase of `bar` with the given parity; false once kWaitLimitNs
// have passed (and in any case after 2^20 rounds of 256 polls).
__device__ __noinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity)
{
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (int round = 0; round < (1 << 20); ++round) {
        for (int k = 0; k < 256; ++k)
            if (mbar_test(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
    return false;
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
                 : "memory");
}

// Smem reads of E consecutive halves / floats.
template <int E>
__device__ __forceinline__ HalfRaw<E> smem_halves(const unsigned char* p)
{
    HalfRaw<E> r;
    if constexpr (E == 8) r.u = *reinterpret_cast<const uint4*>(p);
    else if constexpr (E == 4) r.u = *reinterpret_cast<const uint2*>(p);
    else r.u = *reinterpret_cast<const unsigned int*>(p);
    return r;
}

template <int E>
__device__ __forceinline__ void smem_floats(const unsigned char* p, float (&x)[E])
{
    if constexpr (E == 8) {
        const float4 lo = reinterpret_cast<const float4*>(p)[0], hi = reinterpret_cast<const float4*>(p)[1];
        x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
        x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
    } else if constexpr (E == 4) {
        const float4 lo = *reinterpret_cast<const float4*>(p);
        x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
    } else {
        const float2 lo = *reinterpret_cast<const float2*>(p);
        x[0] = lo.x; x[1] = lo.y;
    }
}

// acc += ranks 0..R-1 of a stage's gradient rows, in rank order (row q of
// the stage holds rank c*8+q; `row` points at this thread's elements of
// row 0, rows are kTile halves apart).
template <int E, int R>
__device__ __forceinline__ void accumulate_rows(float (&acc)[E], const unsigned char* row)
{
#pragma unroll
    for (int q = 0; q < R; ++q) accumulate<E>(acc, smem_halves<E>(row + static_cast<size_t>(q) * kTile * 2));
}

// After a tile's last chunk of ranks: the gradient means, Adam and the
// stores of this thread's E elements starting at element i of the range.
template <int MODE, int PT, int E, int G>
__device__ __forceinline__ void finish_tile(const StepArgs& a, const float (&acc)[E], float (&w)[E], float (&m)[E],
                                            float (&v)[E], long long i, float* w0, float* m0, float* v0, __half* p0)
{
    float gm[E];
    bool special = false;
#pragma unroll
    for (int j = 0; j < E; ++j) {
        gm[j] = finish_mean<PT>(acc[j], a);
        if constexpr (MODE <= ZERO_MODE_FOLDED_STORAGE) // the only modes that divide
            special |= !(isfinite(gm[j]) && isfinite(m[j]) && isfinite(v[j])) || gm[j] == 0.0f;
    }
    // G = 2: the shortcuts for infinite and zero operands are taken only
    // by warps in which some lane holds a non-finite gradient mean or
    // moment, or a zero gradient mean (what makes the numerators zero);
    // one warp-uniform branch, and both branches give the same IEEE
    // results
    if (G == 1 || (G == 2 && __any_sync(__activemask(), special))) {
#pragma unroll
        for (int j = 0; j < E; ++j) adam_elem<MODE, 1>(a, gm[j], w[j], m[j], v[j]);
    } else {
#pragma unroll
        for (int j = 0; j < E; ++j) adam_elem<MODE, 0>(a, gm[j], w[j], m[j], v[j]);
    }
    store_floats<E>(w0 + i, w);
    if constexpr (uses_m(MODE)) store_floats<E>(m0 + i, m);
    if constexpr (uses_v(MODE)) store_floats<E>(v0 + i, v);
    store_halves<E>(p0 + i, w); // all-gather: element head + i of the full vector
}

// NT consumer threads, E = kTile / NT consecutive elements each per tile.
// PT > 0: P known at compile time.  PT = 0: P read at run time, with RL
// (1..8) the rank count of the last chunk known at compile time, so P =
// 8 (nch - 1) + RL for the run-time chunk count nch.
template <int MODE, int PT, int NT, int G, int RL = 0>
__global__ void __launch_bounds__(NT, 1) zero_fused_step_tma_kernel(const StepArgs a)
{
    static_assert((PT > 0) == (RL == 0) && RL >= 0 && RL <= kChunkRanks, "RL only with a run-time P");
    constexpr int E = kTile / NT;
    static_assert(E * NT == kTile && (E == 2 || E == 4 || E == 8), "tile split over the threads");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[kStages];

    const int P = PT > 0 ? PT : a.P;
    const int nch = (P + kChunkRanks - 1) / kChunkRanks;
    const int tid = threadIdx.x;

    // The bulk range is [head, head + nbulk), nbulk a multiple of 8 so every
    // row copy is a multiple of 16 bytes; CTA 0 does the < 8 + < 8 ragged
    // elements outside it one by one.
    const long long nbulk = ((a.n - a.head) / 8) * 8;
    const long long tail_start = a.head + nbulk;
    if (blockIdx.x == 0) {
        if (tid < a.head) step_elems<MODE, 1, PT>(a, tid);
        if (tid < a.n - tail_start) step_elems<MODE, 1, PT>(a, tail_start + tid);
    }
    const long long ntiles = (nbulk + kTile - 1) / kTile;
    const long long my_tiles = ntiles > blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const long long units = my_tiles * nch;
    if (units == 0) return; // uniform over the CTA, before any barrier

    uint64_t policy = 0;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < 32) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    __syncthreads();

    const __half* g0 = a.g + a.head;
    float* w0 = a.w + a.head;
    float* m0 = uses_m(MODE) ? a.m + a.head : nullptr;
    float* v0 = uses_v(MODE) ? a.v + a.head : nullptr;
    __half* p0 = a.p + a.head;

    // (chunk, tile) of unit u.  With P known at compile time the division
    // by the chunk count is a shift or a multiply; with P read at run time
    // it would be a 64-bit division per unit, so the generic instance keeps
    // counters instead (units are walked in order: the next chunk of the
    // same tile, else chunk 0 of this CTA's next tile).  Measured: counters
    // in the compile-time instances cost P = 16 and 64 20-25 %.
    auto tile_of = [&](long long u) { return blockIdx.x + (u / nch) * gridDim.x; };
    int issue_c = 0;                   // generic instance, warp 0: chunk of the next unit to issue
    long long issue_tile = blockIdx.x; // and its tile
    // Who issues a unit's copies.  With more than one chunk per tile, the 32
    // lanes of warp 0, one row each (measured: P = 12 0.887 -> 0.929, 24
    // 0.945 -> 1.025, 33 0.860 -> 0.972, 96 0.931 -> 1.007 of the copy
    // roofline; 16 and 32 unchanged).  With one chunk, thread 0 alone, in
    // the order below (lanes cost P = 8 0.984 -> 0.907 and P = 5 1 %):
    // warp 0 is also a consumer, and the serial issue delays it least there.
    const bool lane_issue = PT > 0 ? PT > kChunkRanks : nch > 1;
    auto issue = [&](long long u) {    // the lanes of warp 0, for u = 0, 1, 2, ... in turn
        const int s = static_cast<int>(u % kStages);
        int c;
        long long i0;
        if constexpr (PT > 0) {
            c = static_cast<int>(u % nch);
            i0 = tile_of(u) * kTile;
        } else {
            c = issue_c;
            i0 = issue_tile * kTile;
            if (++issue_c == nch) {
                issue_c = 0;
                issue_tile += gridDim.x;
            }
        }
        const long long len = nbulk - i0 < kTile ? nbulk - i0 : kTile;
        const int rc = P - c * kChunkRanks < kChunkRanks ? P - c * kChunkRanks : kChunkRanks;
        const uint32_t hb = static_cast<uint32_t>(len) * 2, fb = static_cast<uint32_t>(len) * 4;
        unsigned char* st = smem + static_cast<size_t>(s) * kStageBytes;
        const uint32_t poison = (u == 0 && blockIdx.x == 0) ? a.poison_tx : 0u;
        if (lane_issue) {
            // one row per lane: gradient rows on lanes 0..rc-1, the state rows
            // of a tile's first chunk on lanes 8, 9, 10, all issued at once
            if (tid == 0) mbar_arrive_expect_tx(&full[s], hb * rc + (c == 0 ? state_rows(MODE) * fb : 0) + poison);
            __syncwarp();
            if (tid < rc) {
                const __half* src = g0 + (static_cast<long long>(c) * kChunkRanks + tid) * a.stride + i0;
                bulk_load(st + static_cast<size_t>(tid) * kTile * 2, src, hb, &full[s], policy);
            } else if (c == 0) {
                if (tid == kChunkRanks) bulk_load(st + kGradBytes, w0 + i0, fb, &full[s], policy);
                if constexpr (uses_m(MODE))
                    if (tid == kChunkRanks + 1) bulk_load(st + kGradBytes + kTile * 4, m0 + i0, fb, &full[s], policy);
                if constexpr (uses_v(MODE))
                    if (tid == kChunkRanks + 2)
                        bulk_load(st + kGradBytes + 2 * kTile * 4, v0 + i0, fb, &full[s], policy);
            }
            return;
        }
        if (tid != 0) return;
        mbar_arrive_expect_tx(&full[s], hb * rc + (c == 0 ? state_rows(MODE) * fb : 0) + poison);
        const __half* src = g0 + static_cast<long long>(c) * kChunkRanks * a.stride + i0;
        // the larger group of rows first (measured: with few ranks the state
        // rows first, P = 4 +2.5 %; with more, the gradient rows first).  Only
        // where P is known at compile time: decided at run time, the generic
        // instance lost 3-6 % (P = 3, 5)
        const bool state_first = PT > 0 && c == 0 && state_rows(MODE) * 2 > rc;
        auto load_state = [&]() {
            bulk_load(st + kGradBytes, w0 + i0, fb, &full[s], policy);
            if constexpr (uses_m(MODE)) bulk_load(st + kGradBytes + kTile * 4, m0 + i0, fb, &full[s], policy);
            if constexpr (uses_v(MODE)) bulk_load(st + kGradBytes + 2 * kTile * 4, v0 + i0, fb, &full[s], policy);
        };
        if (state_first) load_state();
        for (int q = 0; q < rc; ++q)
            bulk_load(st + static_cast<size_t>(q) * kTile * 2, src + q * a.stride, hb, &full[s], policy);
        if (c == 0 && !state_first) load_state();
    };

    if (tid < 32)
        for (long long u = 0; u < kStages && u < units; ++u) issue(u);

    float acc[E], w[E], m[E] = {}, v[E] = {};
    long long u = 0;
    bool failed = false;
    const int e0 = tid * E;
    // When a stage is refilled.  Late (one or two chunks per tile): once
    // every thread has passed the wait for unit uu, the stage of unit uu-1
    // (whose last reader was the Adam of that unit).  Early (three chunks or
    // more): once every thread has read unit uu's rows into registers, that
    // unit's own stage, so four units are in flight during the arithmetic
    // instead of three.  Measured, fraction of the copy roofline: early P =
    // 32 1.018 -> 1.063, 64 0.997 -> 1.036, 24 1.005 -> 0.988; P = 16 even;
    // and worse with fewer chunks (P = 8 0.977 -> 0.888, 12 0.913 -> 0.885).
    // Either way one barrier per unit, which also makes a wait that gave up
    // one decision for the whole CTA (before_read / after_read return false).
    // The consumer loop below is instantiated for each choice (early_tag), so
    // the choice costs nothing inside it; read there as a run-time flag it
    // cost P = 8 5 %.
    const bool early = PT > 0 ? PT > 2 * kChunkRanks : nch > 2;
    auto wait_full = [&](long long uu) -> bool {
        const int s = static_cast<int>(uu % kStages);
        return mbar_wait_bounded(&full[s], static_cast<uint32_t>((uu / kStages) & 1));
    };
    auto before_read = [&](auto early_tag, long long uu, bool ok) -> bool { // late refill
        if constexpr (decltype(early_tag)::value) {
            return true;
        } else {
            if (__syncthreads_or(!ok)) return false;
            if (tid < 32 && uu >= 1 && uu - 1 + kStages < units) issue(uu - 1 + kStages);
            return true;
        }
    };
    auto after_read = [&](auto early_tag, long long uu, bool ok) -> bool { // early refill
        if constexpr (!decltype(early_tag)::value) {
            return true;
        } else {
            if (__syncthreads_or(!ok)) return false;
            if (tid < 32 && uu + kStages < units) issue(uu + kStages);
            return true;
        }
    };
    auto stage_of = [&](long long uu) { return smem + static_cast<size_t>(uu % kStages) * kStageBytes; };
    auto load_state = [&](const unsigned char* st) {
#pragma unroll
        for (int j = 0; j < E; ++j) acc[j] = 0.0f;
        smem_floats<E>(st + kGradBytes + e0 * 4, w);
        if constexpr (uses_m(MODE)) smem_floats<E>(st + kGradBytes + kTile * 4 + e0 * 4, m);
        if constexpr (uses_v(MODE)) smem_floats<E>(st + kGradBytes + 2 * kTile * 4 + e0 * 4, v);
    };

    auto consume = [&](auto early_tag) {
        if constexpr (PT > 0) {
            for (; u < units; ++u) {
                const bool ok = wait_full(u);
                if (!before_read(early_tag, u, ok)) {
                    failed = true;
                    break;
                }
                const int c = static_cast<int>(u % nch);
                const long long i0 = tile_of(u) * kTile;
                const long long len = nbulk - i0 < kTile ? nbulk - i0 : kTile;
                const unsigned char* st = stage_of(u);
                constexpr bool kEarly = decltype(early_tag)::value;
                if (e0 < len) {
                    if (c == 0) load_state(st);
                    // ranks c*8 .. c*8+rc-1 of this tile, in rank order
                    const int rc = P - c * kChunkRanks < kChunkRanks ? P - c * kChunkRanks : kChunkRanks;
#pragma unroll
                    for (int q = 0; q < kChunkRanks; ++q)
                        if (q < rc) accumulate<E>(acc, smem_halves<E>(st + static_cast<size_t>(q) * kTile * 2 + e0 * 2));
                    if constexpr (!kEarly)
                        if (c == nch - 1) finish_tile<MODE, PT, E, G>(a, acc, w, m, v, i0 + e0, w0, m0, v0, p0);
                }
                if constexpr (kEarly) {
                    if (!after_read(early_tag, u, ok)) {
                        failed = true;
                        break;
                    }
                    if (e0 < len && c == nch - 1) finish_tile<MODE, PT, E, G>(a, acc, w, m, v, i0 + e0, w0, m0, v0, p0);
                }
            }
        } else {
            // Run-time P: each tile's units walked as its first chunk (with the
            // state rows), the full middle chunks and the last chunk of RL
            // ranks, so every chunk's rank count is known where it is summed.
            for (long long tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
                const long long i0 = tile * kTile;
                const long long len = nbulk - i0 < kTile ? nbulk - i0 : kTile;
                const bool mine = e0 < len;
                bool ok = wait_full(u);
                if (!before_read(early_tag, u, ok)) {
                    failed = true;
                    break;
                }
                const unsigned char* st = stage_of(u);
                if (nch == 1) { // P = RL: one unit per tile (the late refill)
                    if (mine) {
                        load_state(st);
                        accumulate_rows<E, RL>(acc, st + static_cast<size_t>(e0) * 2);
                        finish_tile<MODE, PT, E, G>(a, acc, w, m, v, i0 + e0, w0, m0, v0, p0);
                    }
                    ++u;
                    continue;
                }
                if (mine) {
                    load_state(st);
                    accumulate_rows<E, kChunkRanks>(acc, st + static_cast<size_t>(e0) * 2);
                }
                if (!after_read(early_tag, u, ok)) {
                    failed = true;
                    break;
                }
                ++u;
                for (int c = 1; c < nch - 1; ++c, ++u) {
                    ok = wait_full(u);
                    if (!before_read(early_tag, u, ok)) {
                        failed = true;
                        break;
                    }
                    if (mine) accumulate_rows<E, kChunkRanks>(acc, stage_of(u) + static_cast<size_t>(e0) * 2);
                    if (!after_read(early_tag, u, ok)) {
                        failed = true;
                        break;
                    }
                }
                if (failed) break;
                ok = wait_full(u);
                if (!before_read(early_tag, u, ok)) {
                    failed = true;
                    break;
                }
                if constexpr (decltype(early_tag)::value) {
                    if (mine) accumulate_rows<E, RL>(acc, stage_of(u) + static_cast<size_t>(e0) * 2);
                    if (!after_read(early_tag, u, ok)) {
                        failed = true;
                        break;
                    }
                    if (mine) finish_tile<MODE, PT, E, G>(a, acc, w, m, v, i0 + e0, w0, m0, v0, p0);
                } else if (mine) {
                    accumulate_rows<E, RL>(acc, stage_of(u) + static_cast<size_t>(e0) * 2);
                    finish_tile<MODE, PT, E, G>(a, acc, w, m, v, i0 + e0, w0, m0, v0, p0);
                }
                ++u;
            }
        }
    };
    if constexpr (PT > 0) {
        consume(std::integral_constant<bool, (PT > 2 * kChunkRanks)>{});
    } else {
        if (early)
            consume(std::true_type{});
        else
            consume(std::false_type{});
    }

    if (failed && tid == 0) {
        // let the copies already issued land before the CTA's shared memory goes away
        // units issued so far: up to u - 2 + kStages with the late refill (unit
        // j's wait refilled the stage of j - 1), up to u - 1 + kStages with the
        // early one (unit j's reads refilled its own stage)
        const long long next = (early ? u : (u >= 1 ? u - 1 : 0)) + kStages;
        const long long issued_end = next < units ? next : units;
        for (long long k = u; k < issued_end; ++k)
            (void)mbar_wait_bounded(&full[k % kStages], static_cast<uint32_t>((k / kStages) & 1));
        atomicAdd(&g_wait_timeouts, 1u);
    }
}

// ---------------------------------------------------------------------------
// Host side: validation, alignment analysis, launch
// ---------------------------------------------------------------------------

thread_local int g_last_cuda_error = 0;

bool finite(float x) { return std::isfinite(x); }

bool overlaps(uintptr_t a, uintptr_t a_bytes, uintptr_t b, uintptr_t b_bytes)
{
    return a < b + b_bytes && b < a + a_bytes;
}

using KernelFn = void (*)(const StepArgs);

template <int MODE, int V>
KernelFn pick_p(int P)
{
    if constexpr (V == 8) {
        switch (P) {
        case 4: return zero_fused_step_kernel<MODE, 8, 4>;
        case 8: return zero_fused_step_kernel<MODE, 8, 8>;
        case 16: return zero_fused_step_kernel<MODE, 8, 16>;
        case 32: return zero_fused_step_kernel<MODE, 8, 32>;
        case 64: return zero_fused_step_kernel<MODE, 8, 64>;
        default: return zero_fused_step_kernel<MODE, 8, 0>;
        }
    } else if constexpr (V == 4) {
        (void)P;
        return zero_fused_step_kernel<MODE, V, 0>;
    } else {
        // P = 4 compiled in at widths 2 and 1 (rows off the 16-byte phase):
        // 0.67 -> 1.00 and 0.47 -> 0.84 of the copy roofline
        return P == 4 ? zero_fused_step_kernel<MODE, V, 4> : zero_fused_step_kernel<MODE, V, 0>;
    }
}

template <int MODE>
KernelFn pick_v(int V, int P)
{
    switch (V) {
    case 8: return pick_p<MODE, 8>(P);
    case 4: return pick_p<MODE, 4>(P);
    case 2: return pick_p<MODE, 2>(P);
    default: return pick_p<MODE, 1>(P);
    }
}

KernelFn pick_kernel(int mode, int V, int P)
{
    switch (mode) {
    case ZERO_MODE_STANDARD: return pick_v<ZERO_MODE_STANDARD>(V, P);
    case ZERO_MODE_FOLDED_LITERAL: return pick_v<ZERO_MODE_FOLDED_LITERAL>(V, P);
    case ZERO_MODE_SGD: return pick_v<ZERO_MODE_SGD>(V, P);
    case ZERO_MODE_MOMENTUM: return pick_v<ZERO_MODE_MOMENTUM>(V, P);
    default: return pick_v<ZERO_MODE_FOLDED_STORAGE>(V, P);
    }
}

// Consumer width of the bulk-copy kernel by P (measured on GB300): with few
// ranks per tile the Adam arithmetic dominates and wants more warps; with
// 8 ranks one 16-byte shared-memory read per rank per thread is best; with
// 5-7 (256 consumers cost them 20 %) and with more ranks the rank reduction
// wants more warps again.
constexpr int tma_threads(int P)
{
    return P <= 4 ? 1024 : (P == 8 ? 256 : 512);
}

struct TmaKernel {
    KernelFn fn;
    int threads;
};

template <int MODE, int PT>
TmaKernel tma_instance()
{
    constexpr int NT = tma_threads(PT > 0 ? PT : 64);
    return TmaKernel{zero_fused_step_tma_kernel<MODE, PT, NT, 2>, NT};
}

// Rank counts above 8 without an instance of their own: P read at run time,
// the last chunk's rank count RL = P - 8 (nch - 1) at compile time, 512
// consumers.
template <int MODE, int RL>
TmaKernel tma_generic_rl()
{
    return TmaKernel{zero_fused_step_tma_kernel<MODE, 0, tma_threads(64), 2, RL>, tma_threads(64)};
}

template <int MODE>
TmaKernel tma_generic(int P)
{
    switch (P - ((P - 1) / kChunkRanks) * kChunkRanks) {
    case 1: return tma_generic_rl<MODE, 1>();
    case 2: return tma_generic_rl<MODE, 2>();
    case 3: return tma_generic_rl<MODE, 3>();
    case 4: return tma_generic_rl<MODE, 4>();
    case 5: return tma_generic_rl<MODE, 5>();
    case 6: return tma_generic_rl<MODE, 6>();
    case 7: return tma_generic_rl<MODE, 7>();
    default: return tma_generic_rl<MODE, 8>();
    }
}

template <int MODE>
TmaKernel pick_tma_p(int P)
{
    switch (P) {
    case 1: return tma_instance<MODE, 1>(); // every P up to one chunk of 8 ranks
    case 2: return tma_instance<MODE, 2>();
    case 3: return tma_instance<MODE, 3>();
    case 4: return tma_instance<MODE, 4>();
    case 5: return tma_instance<MODE, 5>();
    case 6: return tma_instance<MODE, 6>();
    case 7: return tma_instance<MODE, 7>();
    case 8: return tma_instance<MODE, 8>();
    case 16: return tma_instance<MODE, 16>();
    case 32: return tma_instance<MODE, 32>();
    case 64: return tma_instance<MODE, 64>();
    case 72: return tma_instance<MODE, 72>();   // one NVL72 rack of GB300s
    case 128: return tma_instance<MODE, 128>();
    case 144: return tma_instance<MODE, 144>(); // two racks
    case 256: return tma_instance<MODE, 256>();
    default: // P > 8
        return tma_generic<MODE>(P);
    }
}

// P = 8 with 512 consumers, for a step capped to fewer SMs than the device
// has: measured per SM, 55.6 GB/s against 44.8 with the 256 consumers the
// uncapped step takes (which is faster on all SMs: 0.785 against 0.869 ms
// on the gpt2s vector), whatever the cap from 16 to 48 SMs.
TmaKernel pick_tma_p8_wide(int mode)
{
    switch (mode) {
    case ZERO_MODE_STANDARD: return TmaKernel{zero_fused_step_tma_kernel<ZERO_MODE_STANDARD, 8, 512, 2>, 512};
    case ZERO_MODE_FOLDED_LITERAL: return TmaKernel{zero_fused_step_tma_kernel<ZERO_MODE_FOLDED_LITERAL, 8, 512, 2>, 512};
    case ZERO_MODE_SGD: return TmaKernel{zero_fused_step_tma_kernel<ZERO_MODE_SGD, 8, 512, 2>, 512};
    case ZERO_MODE_MOMENTUM: return TmaKernel{zero_fused_step_tma_kernel<ZERO_MODE_MOMENTUM, 8, 512, 2>, 512};
    default: return TmaKernel{zero_fused_step_tma_kernel<ZERO_MODE_FOLDED_STORAGE, 8, 512, 2>, 512};
    }
}

TmaKernel pick_tma_kernel(int mode, int P)
{
    switch (mode) {
    case ZERO_MODE_STANDARD: return pick_tma_p<ZERO_MODE_STANDARD>(P);
    case ZERO_MODE_FOLDED_LITERAL: return pick_tma_p<ZERO_MODE_FOLDED_LITERAL>(P);
    case ZERO_MODE_SGD: return pick_tma_p<ZERO_MODE_SGD>(P);
    case ZERO_MODE_MOMENTUM: return pick_tma_p<ZERO_MODE_MOMENTUM>(P);
    default: return pick_tma_p<ZERO_MODE_FOLDED_STORAGE>(P);
    }
}

// Widest vector V in {8,4,2,1} for which one head length h makes every
// stream's element h start on a V-element boundary (at most 16 bytes per
// access, so fp32 streams need min(V,4)-element alignment).
int pick_vector(const StepArgs& a, int mode, long long* head)
{
    const uintptr_t g = reinterpret_cast<uintptr_t>(a.g) / 2;
    const uintptr_t p = reinterpret_cast<uintptr_t>(a.p) / 2;
    const uintptr_t w = reinterpret_cast<uintptr_t>(a.w) / 4;
    const uintptr_t m = reinterpret_cast<uintptr_t>(a.m) / 4;
    const uintptr_t v = reinterpret_cast<uintptr_t>(a.v) / 4;
    for (int V = 8; V > 1; V /= 2) {
        if (a.P > 1 && a.stride % V != 0) continue;
        const uintptr_t ph = g % V;
        if (p % V != ph) continue;
        const int fv = V < 4 ? V : 4;
        if (w % fv != ph % fv) continue;
        if (uses_m(mode) && m % fv != ph % fv) continue;
        if (uses_v(mode) && v % fv != ph % fv) continue;
        long long h = static_cast<long long>((V - ph) % V);
        *head = h < a.n ? h : a.n;
        return V;
    }
    *head = 0;
    return 1;
}

int sm_count_of_current_device()
{
    static std::atomic<int> cache[64]; // devices 0..63; any other is asked every time
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const bool cached = dev >= 0 && dev < 64;
    int c = cached ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (c == 0) {
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        if (cached) cache[dev].store(c, std::memory_order_relaxed);
    }
    return c;
}

int record_cuda(cudaError_t e)
{
    g_last_cuda_error = static_cast<int>(e);
    return ZERO_ECUDA;
}

// Launch set-up done once per (kernel, device): the resident CTAs per SM of
// a vector-path kernel, or the dynamic shared-memory opt-in of a bulk-path
// kernel.  Returns the value (>= 1) or ZERO_ECUDA.  The table has room for
// every kernel of the library (about 120) on 8 devices; past that a kernel
// is set up again on each launch, which is slower but gives the same result.
struct SetupEntry {
    KernelFn fn;
    int dev;
    int value;
};
constexpr int kSetupEntries = 1024;
std::mutex g_setup_mu;
SetupEntry g_setup[kSetupEntries];
int g_setup_n = 0;

int kernel_setup(KernelFn fn, bool bulk)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda(e);
    std::lock_guard<std::mutex> lock(g_setup_mu);
    for (int i = 0; i < g_setup_n; ++i)
        if (g_setup[i].fn == fn && g_setup[i].dev == dev) return g_setup[i].value;
    int value = 1;
    if (bulk) {
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kBulkSmem));
    } else {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&value, fn, kThreads, 0);
        if (value < 1) value = 1;
    }
    if (e != cudaSuccess) return record_cuda(e);
    if (g_setup_n < kSetupEntries) g_setup[g_setup_n++] = SetupEntry{fn, dev, value};
    return value;
}

// Common validation of the hyper-parameters and sizes.
int check_scalars(int64_t N, int32_t P, int32_t stage, int64_t t, float lr, float b1, float b2,
                  float eps, int32_t mode)
{
    if (N < 1 || P < 1 || P > ZERO_MAX_RANKS) return ZERO_EINVAL;
    if (stage < 0 || stage > 3) return ZERO_EINVAL;
    if (mode < 0 || mode > ZERO_MODE_MOMENTUM) return ZERO_EINVAL;
    if (t < 1) return ZERO_EINVAL;
    if (!finite(lr) || !finite(b1) || !finite(b2) || !finite(eps)) return ZERO_EINVAL;
    if (!(b1 >= 0.0f && b1 < 1.0f) || !(b2 >= 0.0f && b2 < 1.0f) || !(eps >= 0.0f)) return ZERO_EINVAL;
    return ZERO_OK;
}

// Validate the buffers of the range described by `a` (n >= 1) and fill in
// the step scalars; *V and the head are chosen from the buffers' alignment.
int prepare_range(StepArgs& a, int64_t t, float lr, float b1, float b2, float eps, int mode, int* V)
{
    const bool um = uses_m(mode), uv = uses_v(mode);
    if (!a.g || !a.w || !a.p || (um && !a.m) || (uv && !a.v)) return ZERO_EINVAL;
    if (!um) a.m = nullptr; // a stream the mode does not use is never touched
    if (!uv) a.v = nullptr;
    if (a.P > 1 && a.stride < a.n) return ZERO_EINVAL; // rank slices must not overlap
    const uintptr_t gg = reinterpret_cast<uintptr_t>(a.g);
    if (reinterpret_cast<uintptr_t>(a.w) % 4 || reinterpret_cast<uintptr_t>(a.p) % 2 || gg % 2 ||
        reinterpret_cast<uintptr_t>(a.m) % 4 || reinterpret_cast<uintptr_t>(a.v) % 4)
        return ZERO_EALIGN;
    // the outputs the mode writes must not overlap each other or the gradients
    const uintptr_t fb = static_cast<uintptr_t>(a.n) * 4, hb = static_cast<uintptr_t>(a.n) * 2;
    const uintptr_t g_span = (static_cast<uintptr_t>(a.P - 1) * static_cast<uintptr_t>(a.stride) +
                              static_cast<uintptr_t>(a.n)) * 2;
    uintptr_t out[4][2];
    int n_out = 0;
    out[n_out][0] = reinterpret_cast<uintptr_t>(a.w), out[n_out++][1] = fb;
    out[n_out][0] = reinterpret_cast<uintptr_t>(a.p), out[n_out++][1] = hb;
    if (um) out[n_out][0] = reinterpret_cast<uintptr_t>(a.m), out[n_out++][1] = fb;
    if (uv) out[n_out][0] = reinterpret_cast<uintptr_t>(a.v), out[n_out++][1] = fb;
    for (int i = 0; i < n_out; ++i) {
        if (overlaps(gg, g_span, out[i][0], out[i][1])) return ZERO_EOVERLAP;
        for (int j = i + 1; j < n_out; ++j)
            if (overlaps(out[i][0], out[i][1], out[j][0], out[j][1])) return ZERO_EOVERLAP;
    }

    // step scalars: bias corrections in double from the fp32 betas, rounded once
    a.lr = lr;
    a.b1 = b1;
    a.b2 = b2;
    a.eps = eps;
    a.omb1 = 1.0f - b1;
    a.omb2 = 1.0f - b2;
    a.bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(b1), static_cast<double>(t)));
    a.bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(b2), static_cast<double>(t)));
    a.bp1 = static_cast<float>(1.0 - std::pow(static_cast<double>(b1), static_cast<double>(t - 1)));
    a.bp2 = static_cast<float>(1.0 - std::pow(static_cast<double>(b2), static_cast<double>(t - 1)));
    a.p_pow2 = (a.P & (a.P - 1)) == 0;
    a.inv_p = 1.0f / static_cast<float>(a.P);
    a.poison_tx = 0;

    long long head = 0;
    *V = pick_vector(a, mode, &head);
    a.head = head;
    return ZERO_OK;
}

// Tiles of the bulk range (elements [head, head + a multiple of 8)).
long long bulk_tiles(const StepArgs& a)
{
    return ((a.n - a.head) / 8 * 8 + kTile - 1) / kTile;
}

// What a step of the range will launch: the kernel, its vector width and
// its grid.  Decided once, by plan_range, for both the launch and the
// zero_step_plan diagnostic.
struct LaunchPlan {
    bool bulk = false; // the bulk-copy pipeline, else the vector kernel
    int V = 1;         // elements per vector access (8 on the pipeline)
    long long ctas = 0;
    int threads = 0;
    KernelFn fn = nullptr;
};

// The bulk-copy pipeline needs every stream on one 16-byte phase (V = 8) and
// pays off once every SM has a few tiles; smaller or misaligned problems take
// the vector path, whose many CTAs start and finish sooner.
constexpr int kMinTilesPerSm = 4;

// The SMs a fused step may occupy (0 = all of them); read when a step is
// enqueued.  Below the SM count it leaves SMs free for work on other streams.
std::atomic<int> g_step_max_sms{0};

int plan_range(StepArgs& a, int64_t t, float lr, float b1, float b2, float eps, int mode, LaunchPlan* plan)
{
    int V = 1;
    int rc = prepare_range(a, t, lr, b1, b2, eps, mode, &V);
    if (rc) return rc;
    int sms = sm_count_of_current_device();
    if (sms <= 0) return record_cuda(cudaGetLastError());
    const int cap = g_step_max_sms.load(std::memory_order_relaxed);
    if (cap > 0 && cap < sms) sms = cap;
    plan->V = V;
    if (V == 8 && bulk_tiles(a) >= static_cast<long long>(kMinTilesPerSm) * sms) {
        const bool capped = sms < sm_count_of_current_device();
        const TmaKernel k = (capped && a.P == 8) ? pick_tma_p8_wide(mode) : pick_tma_kernel(mode, a.P);
        rc = kernel_setup(k.fn, true);
        if (rc < 0) return rc;
        plan->bulk = true;
        plan->fn = k.fn;
        plan->threads = k.threads;
        plan->ctas = sms;
        return ZERO_OK;
    }
    KernelFn fn = pick_kernel(mode, V, a.P);
    const int per_sm = kernel_setup(fn, false);
    if (per_sm < 0) return per_sm;
    const long long body = (a.n - a.head) / V;
    long long blocks = (body + kThreads - 1) / kThreads;
    const long long limit = static_cast<long long>(sms) * per_sm;
    if (blocks > limit) blocks = limit;
    if (blocks < 1) blocks = 1;
    plan->bulk = false;
    plan->fn = fn;
    plan->threads = kThreads;
    plan->ctas = blocks;
    return ZERO_OK;
}

int launch_plan(const StepArgs& a, const LaunchPlan& plan, cudaStream_t stream)
{
    plan.fn<<<static_cast<unsigned int>(plan.ctas), plan.threads, plan.bulk ? kBulkSmem : 0, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ZERO_OK : record_cuda(e);
}

// The bulk-copy pipeline on one CTA per SM, whatever the problem size (the
// bounded-wait diagnostic).
int launch_tma(const StepArgs& a, int mode, int sms, cudaStream_t stream)
{
    const TmaKernel k = pick_tma_kernel(mode, a.P);
    const int rc = kernel_setup(k.fn, true);
    if (rc < 0) return rc;
    k.fn<<<static_cast<unsigned int>(sms), k.threads, kBulkSmem, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ZERO_OK : record_cuda(e);
}

int launch_range(StepArgs a, int64_t t, float lr, float b1, float b2, float eps, int mode,
                 cudaStream_t stream)
{
    LaunchPlan plan;
    const int rc = plan_range(a, t, lr, b1, b2, eps, mode, &plan);
    if (rc) return rc;
    return launch_plan(a, plan, stream);
}

} // namespace

extern "C" int zero_set_step_max_sms(int32_t max_sms, int32_t* previous)
{
    if (max_sms < 0) return ZERO_EINVAL;
    const int old = g_step_max_sms.exchange(max_sms, std::memory_order_relaxed);
    if (previous) *previous = old;
    return ZERO_OK;
}

extern "C" int zero_step_plan(const void* grads_fp16, int64_t rank_stride, float* master, float* m, float* v,
                              void* params_fp16, int64_t N, int32_t P, int32_t stage, int32_t mode,
                              int32_t* kernel, int32_t* vector_width, int64_t* ctas)
{
    if (!kernel || !vector_width || !ctas) return ZERO_EINVAL;
    // the hyper-parameters do not enter the choice: any valid ones will do
    const float lr = 1e-3f, b1 = 0.9f, b2 = 0.999f, eps = 1e-8f;
    int rc = check_scalars(N, P, stage, 1, lr, b1, b2, eps, mode);
    if (rc) return rc;
    if (rank_stride < N) return ZERO_EINVAL;
    StepArgs a{};
    a.g = static_cast<const __half*>(grads_fp16);
    a.stride = rank_stride;
    a.w = master;
    a.m = m;
    a.v = v;
    a.p = static_cast<__half*>(params_fp16);
    a.n = N;
    a.P = P;
    LaunchPlan plan;
    rc = plan_range(a, 1, lr, b1, b2, eps, mode, &plan);
    if (rc) return rc;
    *kernel = plan.bulk ? ZERO_KERNEL_BULK : ZERO_KERNEL_VECTOR;
    *vector_width = plan.V;
    *ctas = plan.ctas;
    return ZERO_OK;
}

extern "C" int zero_adam_step(const void* grads_fp16, int64_t rank_stride, float* master, float* m,
                              float* v, void* params_fp16, int64_t N, int32_t P, int32_t stage,
                              int64_t t, float lr, float beta1, float beta2, float eps, int32_t mode,
                              void* cuda_stream)
{
    int rc = check_scalars(N, P, stage, t, lr, beta1, beta2, eps, mode);
    if (rc) return rc;
    if (rank_stride < N) return ZERO_EINVAL;
    StepArgs a{};
    a.g = static_cast<const __half*>(grads_fp16);
    a.stride = rank_stride;
    a.w = master;
    a.m = m;
    a.v = v;
    a.p = static_cast<__half*>(params_fp16);
    a.n = N;
    a.P = P;
    return launch_range(a, t, lr, beta1, beta2, eps, mode, static_cast<cudaStream_t>(cuda_stream));
}

extern "C" int zero_adam_step_shard(const void* grads_fp16, int64_t rank_stride, int64_t grad_offset,
                                    int32_t k, float* master_s, float* m_s, float* v_s,
                                    void* params_out, int64_t N, int32_t P, int32_t stage, int64_t t,
                                    float lr, float beta1, float beta2, float eps, int32_t mode,
                                    void* cuda_stream)
{
    int rc = check_scalars(N, P, stage, t, lr, beta1, beta2, eps, mode);
    if (rc) return rc;
    if (k < 0 || k >= P || grad_offset < 0 || rank_stride < 1) return ZERO_EINVAL;
    const int64_t M = N / P + (N % P != 0);
    const int64_t b = static_cast<int64_t>(k) * M < N ? static_cast<int64_t>(k) * M : N;
    const int64_t e = b + M < N ? b + M : N;
    const int64_t len = e - b;
    // a trailing rank that owns nothing: no buffer is touched, so none is
    // examined (zero-length allocations are often NULL)
    if (len == 0) return ZERO_OK;
    if (!grads_fp16 || !master_s || !params_out) return ZERO_EINVAL; // m_s, v_s: checked by mode
    StepArgs a{};
    a.g = static_cast<const __half*>(grads_fp16) + grad_offset;
    a.stride = rank_stride;
    a.w = master_s;
    a.m = m_s;
    a.v = v_s;
    a.p = static_cast<__half*>(params_out);
    a.n = len;
    a.P = P;
    return launch_range(a, t, lr, beta1, beta2, eps, mode, static_cast<cudaStream_t>(cuda_stream));
}

namespace {

// The range [begin, end) of the whole-vector layout as a StepArgs.
StepArgs range_args(const void* grads_fp16, int64_t rank_stride, int64_t begin, int64_t end, float* master,
                    float* m, float* v, void* params_fp16, int32_t P)
{
    StepArgs a{};
    a.g = static_cast<const __half*>(grads_fp16) + begin;
    a.stride = rank_stride;
    a.w = master + begin;
    a.m = m ? m + begin : nullptr;
    a.v = v ? v + begin : nullptr;
    a.p = static_cast<__half*>(params_fp16) + begin;
    a.n = end - begin;
    a.P = P;
    return a;
}

} // namespace

extern "C" int zero_adam_step_range(const void* grads_fp16, int64_t rank_stride, int64_t begin, int64_t end,
                                    float* master, float* m, float* v, void* params_fp16, int64_t N,
                                    int32_t P, int32_t stage, int64_t t, float lr, float beta1, float beta2,
                                    float eps, int32_t mode, void* cuda_stream)
{
    int rc = check_scalars(N, P, stage, t, lr, beta1, beta2, eps, mode);
    if (rc) return rc;
    if (rank_stride < N || begin < 0 || begin >= end || end > N) return ZERO_EINVAL;
    if (!grads_fp16 || !master || !params_fp16) return ZERO_EINVAL; // m, v: checked by mode
    return launch_range(range_args(grads_fp16, rank_stride, begin, end, master, m, v, params_fp16, P), t, lr,
                        beta1, beta2, eps, mode, static_cast<cudaStream_t>(cuda_stream));
}

extern "C" int zero_adam_step_bucketed(const void* grads_fp16, int64_t rank_stride, float* master, float* m,
                                       float* v, void* params_fp16, int64_t N, int32_t P, int32_t stage,
                                       int64_t t, float lr, float beta1, float beta2, float eps, int32_t mode,
                                       const zero_bucket_t* buckets, int32_t n_buckets,
                                       void* const* ready_events, void* step_stream)
{
    int rc = check_scalars(N, P, stage, t, lr, beta1, beta2, eps, mode);
    if (rc) return rc;
    if (rank_stride < N || !buckets || n_buckets < 1) return ZERO_EINVAL;
    if (!grads_fp16 || !master || !params_fp16) return ZERO_EINVAL; // m, v: checked by mode
    // every bucket in range and no two overlapping, before anything is enqueued
    std::vector<std::pair<int64_t, int64_t>> sorted;
    sorted.reserve(static_cast<size_t>(n_buckets));
    for (int32_t b = 0; b < n_buckets; ++b) {
        if (buckets[b].begin < 0 || buckets[b].begin >= buckets[b].end || buckets[b].end > N) return ZERO_EINVAL;
        sorted.emplace_back(buckets[b].begin, buckets[b].end);
    }
    std::sort(sorted.begin(), sorted.end());
    for (size_t i = 1; i < sorted.size(); ++i)
        if (sorted[i].first < sorted[i - 1].second) return ZERO_EINVAL;
    // the buffers are validated once, for the whole vector
    StepArgs whole = range_args(grads_fp16, rank_stride, 0, N, master, m, v, params_fp16, P);
    int V = 1;
    rc = prepare_range(whole, t, lr, beta1, beta2, eps, mode, &V);
    if (rc) return rc;

    cudaStream_t stream = static_cast<cudaStream_t>(step_stream);
    for (int32_t b = 0; b < n_buckets; ++b) {
        if (ready_events && ready_events[b]) {
            const cudaError_t e = cudaStreamWaitEvent(stream, static_cast<cudaEvent_t>(ready_events[b]), 0);
            if (e != cudaSuccess) return record_cuda(e);
        }
        rc = launch_range(range_args(grads_fp16, rank_stride, buckets[b].begin, buckets[b].end, master, m, v,
                                     params_fp16, P),
                          t, lr, beta1, beta2, eps, mode, stream);
        if (rc) return rc;
    }
    return ZERO_OK;
}

// ---------------------------------------------------------------------------
// ZeRO-Offload's GPU side: the gradient mean of the ranks, rounded to fp16,
// written to device or page-locked host memory (the host side and the
// pipelined step are in offload.cu)
// ---------------------------------------------------------------------------

namespace {

// Mean of the P ranks' gradients to fp16, V elements per thread per
// iteration; uses StepArgs' g, stride, p (the fp16 output), n, head, P,
// p_pow2 and inv_p.
template <int V, int PT>
__global__ void __launch_bounds__(kThreads) zero_reduce_fp16_kernel(const StepArgs a)
{
    const int P = PT > 0 ? PT : a.P;
    const long long tid = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
    const long long nthreads = static_cast<long long>(gridDim.x) * kThreads;
    const long long body = (a.n - a.head) / V;
    const long long tail_start = a.head + body * V;
    auto one = [&](long long i, auto vtag) {
        constexpr int W = decltype(vtag)::value;
        float acc[W];
#pragma unroll
        for (int j = 0; j < W; ++j) acc[j] = 0.0f;
        const __half* gp = a.g + i;
#pragma unroll 8
        for (int r = 0; r < P; ++r) accumulate<W>(acc, load_halves<W>(gp + static_cast<long long>(r) * a.stride));
#pragma unroll
        for (int j = 0; j < W; ++j) acc[j] = finish_mean<PT>(acc[j], a);
        store_halves<W>(a.p + i, acc);
    };
    if (tid < a.head) one(tid, std::integral_constant<int, 1>{});
    if (tid < a.n - tail_start) one(tail_start + tid, std::integral_constant<int, 1>{});
    for (long long c = tid; c < body; c += nthreads) one(a.head + c * V, std::integral_constant<int, V>{});
}

KernelFn pick_reduce_kernel(int V, int P)
{
    if (V != 8) return zero_reduce_fp16_kernel<1, 0>;
    switch (P) {
    case 4: return zero_reduce_fp16_kernel<8, 4>;
    case 8: return zero_reduce_fp16_kernel<8, 8>;
    case 16: return zero_reduce_fp16_kernel<8, 16>;
    case 32: return zero_reduce_fp16_kernel<8, 32>;
    case 64: return zero_reduce_fp16_kernel<8, 64>;
    default: return zero_reduce_fp16_kernel<8, 0>;
    }
}

} // namespace

extern "C" int zero_reduce_scatter_fp16(const void* grads_fp16, int64_t rank_stride, int64_t grad_offset,
                                        int32_t P, int64_t n, void* out_fp16, void* cuda_stream)
{
    if (!grads_fp16 || !out_fp16 || n < 1 || P < 1 || P > ZERO_MAX_RANKS || grad_offset < 0) return ZERO_EINVAL;
    if (P > 1 && rank_stride < n) return ZERO_EINVAL;
    const uintptr_t gg = reinterpret_cast<uintptr_t>(grads_fp16), go = reinterpret_cast<uintptr_t>(out_fp16);
    if (gg % 2 || go % 2) return ZERO_EALIGN;
    const uintptr_t g_span = (static_cast<uintptr_t>(P - 1) * static_cast<uintptr_t>(rank_stride) +
                              static_cast<uintptr_t>(grad_offset) + static_cast<uintptr_t>(n)) * 2;
    if (overlaps(gg, g_span, go, static_cast<uintptr_t>(n) * 2)) return ZERO_EOVERLAP;
    StepArgs a{};
    a.g = static_cast<const __half*>(grads_fp16) + grad_offset;
    a.stride = rank_stride;
    a.p = static_cast<__half*>(out_fp16);
    a.n = n;
    a.P = P;
    a.p_pow2 = (P & (P - 1)) == 0;
    a.inv_p = 1.0f / static_cast<float>(P);
    // 16-byte vectors when every rank's slice and the output share one phase
    const uintptr_t ph = (reinterpret_cast<uintptr_t>(a.g) / 2) % 8;
    const bool v8 = (P == 1 || rank_stride % 8 == 0) && (go / 2) % 8 == ph;
    a.head = v8 ? static_cast<long long>((8 - ph) % 8) : 0;
    if (a.head > n) a.head = n;
    const int V = v8 ? 8 : 1;
    KernelFn fn = pick_reduce_kernel(V, P);
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return record_cuda(cudaGetLastError());
    const int per_sm = kernel_setup(fn, false);
    if (per_sm < 0) return per_sm;
    long long blocks = ((n - a.head) / V + kThreads - 1) / kThreads;
    const long long cap = static_cast<long long>(sms) * per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    fn<<<static_cast<unsigned int>(blocks), kThreads, 0, static_cast<cudaStream_t>(cuda_stream)>>>(a);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ZERO_OK : record_cuda(e);
}

extern "C" int zero_selftest_wait_timeout(const void* grads_fp16, int64_t rank_stride, float* master,
                                          float* m, float* v, void* params_fp16, int64_t N, int32_t P,
                                          int32_t stage, int64_t t, float lr, float beta1, float beta2,
                                          float eps, int32_t mode, void* cuda_stream)
{
    int rc = check_scalars(N, P, stage, t, lr, beta1, beta2, eps, mode);
    if (rc) return rc;
    if (rank_stride < N) return ZERO_EINVAL;
    StepArgs a{};
    a.g = static_cast<const __half*>(grads_fp16);
    a.stride = rank_stride;
    a.w = master;
    a.m = m;
    a.v = v;
    a.p = static_cast<__half*>(params_fp16);
    a.n = N;
    a.P = P;
    int V = 1;
    rc = prepare_range(a, t, lr, beta1, beta2, eps, mode, &V);
    if (rc) return rc;
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return record_cuda(cudaGetLastError());
    if (V != 8 || bulk_tiles(a) < sms) return ZERO_EINVAL; // CTA 0 must own a bulk tile
    a.poison_tx = 16; // 16 bytes that no copy will ever deliver
    return launch_tma(a, mode, sms, static_cast<cudaStream_t>(cuda_stream));
}

extern "C" const char* zero_strerror(int code)
{
    switch (code) {
    case ZERO_OK: return "success";
    case ZERO_EINVAL: return "invalid argument (null pointer, size, stage, mode, t or hyper-parameter)";
    case ZERO_EALIGN: return "pointer not aligned to its element size";
    case ZERO_EOVERLAP: return "output buffers overlap each other or the gradients";
    case ZERO_ECUDA: return "CUDA runtime error (see zero_last_cuda_error)";
    case ZERO_ENOMEM: return "host allocation failed";
    default: return "unknown status code";
    }
}

extern "C" int zero_device_timeouts(int64_t* count, int32_t reset)
{
    if (!count) return ZERO_EINVAL;
    unsigned int n = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&n, g_wait_timeouts, sizeof(n));
    if (e != cudaSuccess) return record_cuda(e);
    if (reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(zero));
        if (e != cudaSuccess) return record_cuda(e);
    }
    *count = n;
    return ZERO_OK;
}

namespace {

// Mismatches found by the mean-division check, and the first one's (p, s).
__device__ unsigned long long g_div_mismatches;
__device__ unsigned int g_div_first_p;
__device__ float g_div_first_s;

// div_by_count against the correctly rounded divide for every p in
// [p_lo, p_hi] and every fp32 significand s in [1, 2); r is formed the way
// the host forms StepArgs::inv_p, a correctly rounded 1/p.
__global__ void zero_mean_division_check_kernel(int p_lo, int p_hi)
{
    const long long total = static_cast<long long>(p_hi - p_lo + 1) << 23;
    const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long k = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; k < total; k += step) {
        const int p = p_lo + static_cast<int>(k >> 23);
        const float s = __uint_as_float(0x3f800000u | static_cast<unsigned int>(k & 0x7fffff));
        const float pf = static_cast<float>(p);
        const float want = __fdiv_rn(s, pf);
        const float got = div_by_count(s, pf, __frcp_rn(pf));
        if (__float_as_uint(want) != __float_as_uint(got) && atomicAdd(&g_div_mismatches, 1ull) == 0ull) {
            g_div_first_p = static_cast<unsigned int>(p);
            g_div_first_s = s;
        }
    }
}

} // namespace

extern "C" int zero_selftest_mean_division(int32_t p_lo, int32_t p_hi, int64_t* mismatches, int32_t* first_p,
                                           float* first_sum)
{
    if (!mismatches || p_lo < 1 || p_hi < p_lo || p_hi > ZERO_MAX_RANKS) return ZERO_EINVAL;
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return record_cuda(cudaGetLastError());
    const unsigned long long zero = 0;
    cudaError_t e = cudaMemcpyToSymbol(g_div_mismatches, &zero, sizeof(zero));
    if (e != cudaSuccess) return record_cuda(e);
    zero_mean_division_check_kernel<<<static_cast<unsigned int>(sms) * 8, kThreads>>>(p_lo, p_hi);
    e = cudaGetLastError();
    if (e != cudaSuccess) return record_cuda(e);
    unsigned long long n = 0;
    unsigned int fp = 0;
    float fs = 0.0f;
    e = cudaMemcpyFromSymbol(&n, g_div_mismatches, sizeof(n)); // waits for the kernel
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&fp, g_div_first_p, sizeof(fp));
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&fs, g_div_first_s, sizeof(fs));
    if (e != cudaSuccess) return record_cuda(e);
    *mismatches = static_cast<int64_t>(n);
    if (first_p) *first_p = n ? static_cast<int32_t>(fp) : 0;
    if (first_sum) *first_sum = n ? fs : 0.0f;
    return ZERO_OK;
}

// Used by the other translation units of the library (not exported).
__attribute__((visibility("hidden"))) int zero_record_cuda_error(int err)
{
    return record_cuda(static_cast<cudaError_t>(err));
}

__attribute__((visibility("hidden"))) int zero_check_step_scalars(int64_t N, int32_t P, int32_t stage, int64_t t,
                                                                  float lr, float b1, float b2, float eps,
                                                                  int32_t mode)
{
    return check_scalars(N, P, stage, t, lr, b1, b2, eps, mode);
}

extern "C" int zero_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" const char* zero_last_cuda_error_string(void)
{
    return cudaGetErrorName(static_cast<cudaError_t>(g_last_cuda_error));
}
