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
// The path is elementwise and HBM-bound (2P + 26 bytes moved per element
// against about 15 fp32 operations), so there are no tensor cores here.  Each
// thread owns V consecutive elements per iteration of a grid-stride loop:
// one 16-byte load per rank for V = 8, two 16-byte loads per fp32 stream,
// 16-byte stores.  Every arithmetic operation is an explicitly rounded fp32
// intrinsic, so no multiply-add contraction can change a result.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

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
    float inv_p;        // 1/P (exact when p_pow2)
    float lr, b1, b2, omb1, omb2, bc1, bc2, bp1, bp2, eps;
};

// ---------------------------------------------------------------------------
// Per-element arithmetic
// ---------------------------------------------------------------------------

template <int PT>
__device__ __forceinline__ float finish_mean(float sum, const StepArgs& a)
{
    if constexpr (PT > 0 && (PT & (PT - 1)) == 0) {
        return __fmul_rn(sum, 1.0f / static_cast<float>(PT));
    } else {
        return a.p_pow2 ? __fmul_rn(sum, a.inv_p) : __fdiv_rn(sum, static_cast<float>(a.P));
    }
}

// Adam on one element; w, m, v updated in place, returns the new master.
template <int MODE>
__device__ __forceinline__ void adam_elem(const StepArgs& a, float g, float& w, float& m, float& v)
{
    const float gg = __fmul_rn(g, g);
    float m_new, v_new, m_hat, v_hat;
    if constexpr (MODE == ZERO_MODE_STANDARD) {
        m_new = __fadd_rn(__fmul_rn(a.b1, m), __fmul_rn(a.omb1, g));
        v_new = __fadd_rn(__fmul_rn(a.b2, v), __fmul_rn(a.omb2, gg));
        m_hat = __fdiv_rn(m_new, a.bc1);
        v_hat = __fdiv_rn(v_new, a.bc2);
    } else if constexpr (MODE == ZERO_MODE_FOLDED_LITERAL) {
        m_new = __fdiv_rn(__fadd_rn(__fmul_rn(a.b1, m), __fmul_rn(a.omb1, g)), a.bc1);
        v_new = __fdiv_rn(__fadd_rn(__fmul_rn(a.b2, v), __fmul_rn(a.omb2, gg)), a.bc2);
        m_hat = m_new;
        v_hat = v_new;
    } else {
        m_new = __fdiv_rn(__fadd_rn(__fmul_rn(a.b1, __fmul_rn(m, a.bp1)), __fmul_rn(a.omb1, g)), a.bc1);
        v_new = __fdiv_rn(__fadd_rn(__fmul_rn(a.b2, __fmul_rn(v, a.bp2)), __fmul_rn(a.omb2, gg)), a.bc2);
        m_hat = m_new;
        v_hat = v_new;
    }
    const float denom = __fadd_rn(__fsqrt_rn(v_hat), a.eps);
    const float upd = __fdiv_rn(m_hat, denom);
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
    float w[V], m[V], v[V];
    load_floats<V>(a.w + i, w);
    load_floats<V>(a.m + i, m);
    load_floats<V>(a.v + i, v);

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
    constexpr int kInner = PT > 0 ? kRankBatch : 1;
#pragma unroll kInner
    for (; r < P; ++r) {
        accumulate<V>(acc, load_halves<V>(gp));
        gp += a.stride;
    }

#pragma unroll
    for (int j = 0; j < V; ++j) {
        const float g = finish_mean<PT>(acc[j], a);
        adam_elem<MODE>(a, g, w[j], m[j], v[j]);
    }
    store_floats<V>(a.w + i, w);
    store_floats<V>(a.m + i, m);
    store_floats<V>(a.v + i, v);
    store_halves<V>(a.p + i, w); // all-gather: element i of the full vector
}

template <int MODE, int V, int PT>
__global__ void __launch_bounds__(kThreads) zero_fused_step_kernel(const StepArgs a)
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
    } else {
        (void)P;
        return zero_fused_step_kernel<MODE, V, 0>;
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
    default: return pick_v<ZERO_MODE_FOLDED_STORAGE>(V, P);
    }
}

// Widest vector V in {8,4,2,1} for which one head length h makes every
// stream's element h start on a V-element boundary (at most 16 bytes per
// access, so fp32 streams need min(V,4)-element alignment).
int pick_vector(const StepArgs& a, long long* head)
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
        if (w % fv != ph % fv || m % fv != ph % fv || v % fv != ph % fv) continue;
        long long h = static_cast<long long>((V - ph) % V);
        *head = h < a.n ? h : a.n;
        return V;
    }
    *head = 0;
    return 1;
}

int sm_count_of_current_device()
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) dev = 63;
    int c = cache[dev].load(std::memory_order_relaxed);
    if (c == 0) {
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(c, std::memory_order_relaxed);
    }
    return c;
}

int record_cuda(cudaError_t e)
{
    g_last_cuda_error = static_cast<int>(e);
    return ZERO_ECUDA;
}

// Common validation of the hyper-parameters and sizes.
int check_scalars(int64_t N, int32_t P, int32_t stage, int64_t t, float lr, float b1, float b2,
                  float eps, int32_t mode)
{
    if (N < 1 || P < 1 || P > ZERO_MAX_RANKS) return ZERO_EINVAL;
    if (stage < 0 || stage > 3) return ZERO_EINVAL;
    if (mode < 0 || mode > 2) return ZERO_EINVAL;
    if (t < 1) return ZERO_EINVAL;
    if (!finite(lr) || !finite(b1) || !finite(b2) || !finite(eps)) return ZERO_EINVAL;
    if (!(b1 >= 0.0f && b1 < 1.0f) || !(b2 >= 0.0f && b2 < 1.0f) || !(eps >= 0.0f)) return ZERO_EINVAL;
    return ZERO_OK;
}

// Validate buffers and launch over the range described by `a` (n >= 1).
int launch_range(StepArgs a, int64_t t, float lr, float b1, float b2, float eps, int mode,
                 cudaStream_t stream)
{
    if (!a.g || !a.w || !a.m || !a.v || !a.p) return ZERO_EINVAL;
    if (a.P > 1 && a.stride < a.n) return ZERO_EINVAL; // rank slices must not overlap
    const uintptr_t gw = reinterpret_cast<uintptr_t>(a.w), gm = reinterpret_cast<uintptr_t>(a.m),
                    gv = reinterpret_cast<uintptr_t>(a.v), gp = reinterpret_cast<uintptr_t>(a.p),
                    gg = reinterpret_cast<uintptr_t>(a.g);
    if (gw % 4 || gm % 4 || gv % 4 || gp % 2 || gg % 2) return ZERO_EALIGN;
    const uintptr_t fb = static_cast<uintptr_t>(a.n) * 4, hb = static_cast<uintptr_t>(a.n) * 2;
    const uintptr_t g_span = (static_cast<uintptr_t>(a.P - 1) * static_cast<uintptr_t>(a.stride) +
                              static_cast<uintptr_t>(a.n)) * 2;
    if (overlaps(gw, fb, gm, fb) || overlaps(gw, fb, gv, fb) || overlaps(gm, fb, gv, fb) ||
        overlaps(gw, fb, gp, hb) || overlaps(gm, fb, gp, hb) || overlaps(gv, fb, gp, hb) ||
        overlaps(gg, g_span, gw, fb) || overlaps(gg, g_span, gm, fb) || overlaps(gg, g_span, gv, fb) ||
        overlaps(gg, g_span, gp, hb))
        return ZERO_EOVERLAP;

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

    long long head = 0;
    const int V = pick_vector(a, &head);
    a.head = head;
    KernelFn fn = pick_kernel(mode, V, a.P);

    const int sms = sm_count_of_current_device();
    if (sms <= 0) return record_cuda(cudaGetLastError());
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, 0);
    if (e != cudaSuccess) return record_cuda(e);
    if (per_sm < 1) per_sm = 1;
    const long long body = (a.n - a.head) / V;
    long long blocks = (body + kThreads - 1) / kThreads;
    const long long cap = static_cast<long long>(sms) * per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    fn<<<static_cast<unsigned int>(blocks), kThreads, 0, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return record_cuda(e);
    return ZERO_OK;
}

} // namespace

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
    if (!grads_fp16 || !master_s || !m_s || !v_s || !params_out) return ZERO_EINVAL;
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

extern "C" int zero_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" const char* zero_last_cuda_error_string(void)
{
    return cudaGetErrorName(static_cast<cudaError_t>(g_last_cuda_error));
}
