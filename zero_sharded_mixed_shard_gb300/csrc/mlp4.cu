// The layer-pipelined ZeRO-3 training step of the 4-layer scalar MLP.
//
// Source: 深度学习专题：模型训练的数据并行（三） §（四）ZeRO-3 层间流水线优化:
//  1. the model: scalar x and y, h_k = ReLU(w_k h_{k-1} + b_k) for k = 1..3
//     (h_0 = x), y = w_4 h_3 + b_4, L = (y - x)^2 / 2, and its backward pass
//     layer by layer (dL/dy = y - x, dL/dw_4 = (y - x) h_3, dL/dh_3 = (y - x)
//     w_4, and for k = 3..1 dL/dw_k = dL/dh_k h_{k-1} I(h_k > 0), dL/db_k =
//     dL/dh_k I(h_k > 0), dL/dh_{k-1} = dL/dh_k w_k I(h_k > 0));
//  2. the schedule: 4 GPUs, each storing one layer's 2 parameters and
//     training on 1/4 of the batch; the parameters of a layer are
//     all-gathered before they are used, and while layer k-1's backward runs,
//     layer k's gradients are reduce-scattered to its owner, which updates its
//     optimizer state and parameters.
//
// Each rank's local gradient is the mean over its own samples, summed in
// sample order from +0 and rounded to fp16; every operation is an explicitly
// rounded fp32 intrinsic.  The gradient kernel of layer k recomputes the
// forward pass of its samples instead of keeping activations (the
// recomputation the ZeRO pages discuss for activations), so it reads only the
// all-gathered fp16 parameters; the owners' updates write their own fp16
// shards, and the next step's all-gather copies them into the gathered
// vector.  One thread per rank: the model has 8 parameters and the point is
// the schedule, not the arithmetic.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "zero_step.h"

// Shared with step.cu (not exported): keeps zero_last_cuda_error current.
__attribute__((visibility("hidden"))) int zero_record_cuda_error(int err);

namespace {

constexpr int kMaxRanks = 8;
constexpr int kParams = 8;

struct Params {
    float w[4], b[4];
};

__device__ __forceinline__ Params load_params(const __half* p16)
{
    Params q;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        q.w[k] = __half2float(p16[2 * k]);
        q.b[k] = __half2float(p16[2 * k + 1]);
    }
    return q;
}

__device__ __forceinline__ float relu(float z) { return z > 0.0f ? z : 0.0f; }

struct Forward {
    float z[3], h[3], y;
};

__device__ __forceinline__ Forward forward(const Params& q, float x)
{
    Forward f;
    float hin = x;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        f.z[k] = __fadd_rn(__fmul_rn(q.w[k], hin), q.b[k]);
        f.h[k] = relu(f.z[k]);
        hin = f.h[k];
    }
    f.y = __fadd_rn(__fmul_rn(q.w[3], hin), q.b[3]);
    return f;
}

// Rank r = thread r: mean loss over its samples.
__global__ void mlp4_loss_kernel(const __half* p16, const float* x, int P, int n, float* loss)
{
    const int r = threadIdx.x;
    if (r >= P) return;
    const Params q = load_params(p16);
    float acc = 0.0f;
    for (int s = 0; s < n; ++s) {
        const float xs = x[static_cast<long long>(r) * n + s];
        const Forward f = forward(q, xs);
        const float d = __fsub_rn(f.y, xs);
        acc = __fadd_rn(acc, __fmul_rn(0.5f, __fmul_rn(d, d)));
    }
    loss[r] = __fdiv_rn(acc, static_cast<float>(n));
}

// Rank r = thread r: its mean gradient of w_k, b_k (layer = k, 1..4) as fp16.
__global__ void mlp4_layer_grads_kernel(int layer, const __half* p16, const float* x, int P, int n,
                                        __half* grads, long long rank_stride)
{
    const int r = threadIdx.x;
    if (r >= P) return;
    const Params q = load_params(p16);
    float acc_w = 0.0f, acc_b = 0.0f;
    for (int s = 0; s < n; ++s) {
        const float xs = x[static_cast<long long>(r) * n + s];
        const Forward f = forward(q, xs);
        const float dy = __fsub_rn(f.y, xs);
        float gw, gb;
        if (layer == 4) {
            gw = __fmul_rn(dy, f.h[2]);
            gb = dy;
        } else {
            float dh = __fmul_rn(dy, q.w[3]); // dL/dh_3
            gw = gb = 0.0f;
            for (int k = 3; k >= layer; --k) {
                const float gz = f.z[k - 1] > 0.0f ? dh : 0.0f; // dL/dh_k I(h_k > 0)
                if (k == layer) {
                    gw = __fmul_rn(gz, k > 1 ? f.h[k - 2] : xs);
                    gb = gz;
                } else {
                    dh = __fmul_rn(gz, q.w[k - 1]); // dL/dh_{k-1}
                }
            }
        }
        acc_w = __fadd_rn(acc_w, gw);
        acc_b = __fadd_rn(acc_b, gb);
    }
    const float count = static_cast<float>(n);
    __half* gr = grads + static_cast<long long>(r) * rank_stride + 2 * (layer - 1);
    gr[0] = __float2half_rn(__fdiv_rn(acc_w, count));
    gr[1] = __float2half_rn(__fdiv_rn(acc_b, count));
}

int last_error(cudaError_t e) { return e == cudaSuccess ? ZERO_OK : zero_record_cuda_error(static_cast<int>(e)); }

} // namespace

extern "C" int zero_mlp4_loss(const void* params_fp16, const float* x, int32_t P, int32_t n, float* loss,
                              void* cuda_stream)
{
    if (!params_fp16 || !x || !loss || P < 1 || P > kMaxRanks || n < 1) return ZERO_EINVAL;
    mlp4_loss_kernel<<<1, 32, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        static_cast<const __half*>(params_fp16), x, P, n, loss);
    return last_error(cudaGetLastError());
}

extern "C" int zero_mlp4_layer_grads(int32_t layer, const void* params_fp16, const float* x, int32_t P,
                                     int32_t n, void* grads_fp16, int64_t rank_stride, void* cuda_stream)
{
    if (layer < 1 || layer > 4 || !params_fp16 || !x || !grads_fp16 || P < 1 || P > kMaxRanks || n < 1 ||
        rank_stride < kParams)
        return ZERO_EINVAL;
    mlp4_layer_grads_kernel<<<1, 32, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        layer, static_cast<const __half*>(params_fp16), x, P, n, static_cast<__half*>(grads_fp16), rank_stride);
    return last_error(cudaGetLastError());
}

extern "C" int zero_mlp4_zero3_step(const float* x, int32_t P, int32_t n, void* gathered_fp16, float* master,
                                    float* m, float* v, void* shard_fp16, void* grads_fp16, int64_t rank_stride,
                                    float* loss, int64_t t, float lr, float beta1, float beta2, float eps,
                                    int32_t mode, int32_t pipelined, void* main_stream, void* step_stream)
{
    if (!x || !gathered_fp16 || !master || !m || !v || !shard_fp16 || !grads_fp16 || !loss) return ZERO_EINVAL;
    if (P < 1 || P > kMaxRanks || n < 1 || rank_stride < kParams || t < 1) return ZERO_EINVAL;
    cudaStream_t ms = static_cast<cudaStream_t>(main_stream);
    cudaStream_t ss = pipelined ? static_cast<cudaStream_t>(step_stream) : ms;
    const int64_t M = (kParams + P - 1) / P;
    __half* gathered = static_cast<__half*>(gathered_fp16);
    __half* shards = static_cast<__half*>(shard_fp16);
    const __half* grads = static_cast<const __half*>(grads_fp16);

    cudaEvent_t layer_done[5] = {}, step_done = nullptr, start = nullptr;
    auto cleanup = [&]() {
        for (auto& e : layer_done)
            if (e) cudaEventDestroy(e);
        if (step_done) cudaEventDestroy(step_done);
        if (start) cudaEventDestroy(start);
    };
    auto fail = [&](cudaError_t e) {
        cleanup();
        return zero_record_cuda_error(static_cast<int>(e == cudaSuccess ? cudaErrorUnknown : e));
    };
    cudaError_t e = cudaSuccess;
    for (int k = 1; k <= 4; ++k)
        if ((e = cudaEventCreateWithFlags(&layer_done[k], cudaEventDisableTiming)) != cudaSuccess) return fail(e);
    if ((e = cudaEventCreateWithFlags(&step_done, cudaEventDisableTiming)) != cudaSuccess) return fail(e);
    if ((e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming)) != cudaSuccess) return fail(e);

    // the step stream starts after everything already on the main stream
    if ((e = cudaEventRecord(start, ms)) != cudaSuccess) return fail(e);
    if (ss != ms && (e = cudaStreamWaitEvent(ss, start, 0)) != cudaSuccess) return fail(e);
    // all-gather: every owner's fp16 shard into the gathered vector the pass reads
    if ((e = cudaMemcpyAsync(gathered, shards, kParams * sizeof(__half), cudaMemcpyDeviceToDevice, ms)) !=
        cudaSuccess)
        return fail(e);
    int rc = zero_mlp4_loss(gathered, x, P, n, loss, ms);
    if (rc) {
        cleanup();
        return rc;
    }
    // backward, last layer first; shard k is complete once its lowest layer is
    for (int layer = 4; layer >= 1; --layer) {
        rc = zero_mlp4_layer_grads(layer, gathered, x, P, n, grads_fp16, rank_stride, ms);
        if (rc) {
            cleanup();
            return rc;
        }
        if ((e = cudaEventRecord(layer_done[layer], ms)) != cudaSuccess) return fail(e);
        for (int32_t k = P - 1; k >= 0; --k) {
            const int64_t b = k * M < kParams ? k * M : kParams;
            const int64_t end = b + M < kParams ? b + M : kParams;
            if (b >= end || static_cast<int>(b / 2) + 1 != layer) continue; // shard k's lowest layer
            if (ss != ms && (e = cudaStreamWaitEvent(ss, layer_done[layer], 0)) != cudaSuccess) return fail(e);
            // reduce-scatter of the shard's gradients to its owner, its Adam
            // update, its fp16 shard written (ZeRO-3 keeps only its own shard)
            rc = zero_adam_step_shard(grads, rank_stride, b, k, master + b, m + b, v + b, shards + b, kParams, P,
                                      3, t, lr, beta1, beta2, eps, mode, ss);
            if (rc) {
                cleanup();
                return rc;
            }
        }
    }
    // the main stream continues only once every shard has been updated
    if (ss != ms) {
        if ((e = cudaEventRecord(step_done, ss)) != cudaSuccess) return fail(e);
        if ((e = cudaStreamWaitEvent(ms, step_done, 0)) != cudaSuccess) return fail(e);
    }
    cleanup();
    return ZERO_OK;
}

// ---------------------------------------------------------------------------
// A variant of zero_mlp4_zero3_step for callers that cannot allocate device
// memory: its scratch -- the all-gathered fp16 parameters and every rank's
// fp16 gradients -- lives in one file-scope device array instead of buffers
// the caller provides.
// ---------------------------------------------------------------------------

namespace {

// Scratch layout (fp16): [0, 8) the all-gathered parameters, then 8 ranks x
// 8 gradients at rank stride 8.  144 bytes used, 256 reserved.
constexpr int kScratchHalves = 128;
constexpr int kScratchGrads = kParams;          // offset of rank 0's gradients
constexpr int kScratchRankStride = kParams;
static_assert(kScratchGrads + kMaxRanks * kScratchRankStride <= kScratchHalves, "scratch too small");

static __device__ __align__(256) __half g_mlp4_scratch[kScratchHalves];

// Device address of g_mlp4_scratch, looked up once per device with that
// device current.  Host code may not use the symbol's name as an address.
std::atomic<void*> g_scratch_addr[64];

int scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return zero_record_cuda_error(static_cast<int>(e));
    if (dev < 0 || dev >= 64) return ZERO_EINVAL;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_mlp4_scratch);
        if (e != cudaSuccess) return zero_record_cuda_error(static_cast<int>(e));
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return ZERO_OK;
}

} // namespace

extern "C" int zero_mlp4_zero3_step_noalloc(const float* x, int32_t P, int32_t n, float* master, float* m,
                                            float* v, void* shard_fp16, float* loss, int64_t t, float lr,
                                            float beta1, float beta2, float eps, int32_t mode, void* cuda_stream)
{
    // the scratch holds at most kMaxRanks ranks' gradients
    if (P < 1 || P > kMaxRanks) return ZERO_EINVAL;
    if (!x || !master || !m || !v || !shard_fp16 || !loss || n < 1 || t < 1) return ZERO_EINVAL;
    if (mode < 0 || mode > ZERO_MODE_MOMENTUM || !isfinite(lr) || !isfinite(beta1) || !isfinite(beta2) ||
        !isfinite(eps) || !(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f) || !(eps >= 0.0f))
        return ZERO_EINVAL; // refused before anything is enqueued
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc) return rc;
    __half* gathered = static_cast<__half*>(scratch);
    __half* grads = gathered + kScratchGrads;
    // the serial schedule of zero_mlp4_zero3_step on one stream: it creates
    // no events and allocates nothing; every scratch entry read below is
    // written earlier in the same call, so nothing has to be cleared
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    const cudaError_t e = cudaMemcpyAsync(gathered, shard_fp16, kParams * sizeof(__half), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return zero_record_cuda_error(static_cast<int>(e));
    rc = zero_mlp4_loss(gathered, x, P, n, loss, st);
    if (rc) return rc;
    const int64_t M = (kParams + P - 1) / P;
    __half* shards = static_cast<__half*>(shard_fp16);
    for (int layer = 4; layer >= 1; --layer) {
        rc = zero_mlp4_layer_grads(layer, gathered, x, P, n, grads, kScratchRankStride, st);
        if (rc) return rc;
        for (int32_t k = P - 1; k >= 0; --k) {
            const int64_t b = k * M < kParams ? k * M : kParams;
            const int64_t end = b + M < kParams ? b + M : kParams;
            if (b >= end || static_cast<int>(b / 2) + 1 != layer) continue; // shard k's lowest layer
            rc = zero_adam_step_shard(grads, kScratchRankStride, b, k, master + b, m + b, v + b, shards + b,
                                      kParams, P, 3, t, lr, beta1, beta2, eps, mode, st);
            if (rc) return rc;
        }
    }
    return ZERO_OK;
}
