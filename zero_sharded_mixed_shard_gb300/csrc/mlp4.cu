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
#include <cuda.h> // driver types only: the two driver calls are found through the runtime
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "zero_step.h"

// Shared with step.cu (not exported): keeps zero_last_cuda_error current,
// and the step's own validation of its sizes and hyper-parameters.
__attribute__((visibility("hidden"))) int zero_record_cuda_error(int err);
__attribute__((visibility("hidden"))) int zero_check_step_scalars(int64_t N, int32_t P, int32_t stage, int64_t t,
                                                                  float lr, float b1, float b2, float eps,
                                                                  int32_t mode);

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

// One device buffer of a training step: its address and its size in bytes.
struct Span {
    uintptr_t at;
    uintptr_t bytes;
};

// Every check of a training step's arguments, made before anything is
// enqueued so that a rejected call leaves every buffer as it was: sizes,
// hyper-parameters (as zero_adam_step_shard checks them), the alignment of
// every buffer to its element size, and that no two buffers share a byte
// (x is only read, but the kernels that read it run between writes of the
// others).  gathered and grads are absent (NULL) for the no-allocation step,
// whose scratch is inside the library.
int check_mlp4_step(const float* x, int32_t P, int32_t n, const void* gathered, const float* master,
                    const float* m, const float* v, const void* shard, const void* grads, int64_t rank_stride,
                    const float* loss, int64_t t, float lr, float beta1, float beta2, float eps, int32_t mode,
                    bool caller_scratch)
{
    if (P < 1 || P > kMaxRanks || n < 1) return ZERO_EINVAL;
    int rc = zero_check_step_scalars(kParams, P, 3, t, lr, beta1, beta2, eps, mode);
    if (rc) return rc;
    if (!x || !master || !m || !v || !shard || !loss) return ZERO_EINVAL;
    if (caller_scratch && (!gathered || !grads || rank_stride < kParams || rank_stride > (INT64_MAX >> 4)))
        return ZERO_EINVAL;
    const uintptr_t f4[] = {reinterpret_cast<uintptr_t>(x), reinterpret_cast<uintptr_t>(master),
                            reinterpret_cast<uintptr_t>(m), reinterpret_cast<uintptr_t>(v),
                            reinterpret_cast<uintptr_t>(loss)};
    for (uintptr_t a : f4)
        if (a % 4) return ZERO_EALIGN;
    if (reinterpret_cast<uintptr_t>(shard) % 2) return ZERO_EALIGN;
    if (caller_scratch && (reinterpret_cast<uintptr_t>(gathered) % 2 || reinterpret_cast<uintptr_t>(grads) % 2))
        return ZERO_EALIGN;
    Span spans[8];
    int ns = 0;
    spans[ns++] = Span{reinterpret_cast<uintptr_t>(x), static_cast<uintptr_t>(P) * static_cast<uintptr_t>(n) * 4};
    spans[ns++] = Span{reinterpret_cast<uintptr_t>(master), kParams * 4};
    spans[ns++] = Span{reinterpret_cast<uintptr_t>(m), kParams * 4};
    spans[ns++] = Span{reinterpret_cast<uintptr_t>(v), kParams * 4};
    spans[ns++] = Span{reinterpret_cast<uintptr_t>(shard), kParams * 2};
    spans[ns++] = Span{reinterpret_cast<uintptr_t>(loss), static_cast<uintptr_t>(P) * 4};
    if (caller_scratch) {
        spans[ns++] = Span{reinterpret_cast<uintptr_t>(gathered), kParams * 2};
        spans[ns++] = Span{reinterpret_cast<uintptr_t>(grads),
                           (static_cast<uintptr_t>(P - 1) * static_cast<uintptr_t>(rank_stride) + kParams) * 2};
    }
    for (int i = 0; i < ns; ++i)
        for (int j = i + 1; j < ns; ++j)
            if (spans[i].at < spans[j].at + spans[j].bytes && spans[j].at < spans[i].at + spans[i].bytes)
                return ZERO_EOVERLAP;
    return ZERO_OK;
}

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
    int rc = check_mlp4_step(x, P, n, gathered_fp16, master, m, v, shard_fp16, grads_fp16, rank_stride, loss, t,
                             lr, beta1, beta2, eps, mode, true);
    if (rc) return rc;
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
    rc = zero_mlp4_loss(gathered, x, P, n, loss, ms);
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

// Identity of the context current on this host thread, 0 when none is
// current or the driver cannot say.  The driver's cuCtxGetCurrent and
// cuCtxGetId are reached through the runtime's entry-point lookup, so the
// library needs no link against the driver library.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

unsigned long long current_context_id()
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult found = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &found) ==
                cudaSuccess &&
            found == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        found = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &found) == cudaSuccess &&
            found == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_mlp4_scratch per device, looked up with that device
// current and kept together with the identity of the context it belongs to.
// Host code may not use the symbol's name as an address.  A device reset
// (cudaDeviceReset, or the primary context torn down and created again) can
// load the library's module at another address; the new context has a new
// identity, so the address is looked up again instead of used stale.
struct ScratchSlot {
    unsigned long long ctx;
    void* addr;
};
constexpr int kScratchDevices = 64;
std::mutex g_scratch_mu;
ScratchSlot g_scratch_slot[kScratchDevices];

int scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return zero_record_cuda_error(static_cast<int>(e));
    if (dev < 0 || dev >= kScratchDevices) return ZERO_EINVAL;
    const unsigned long long ctx = current_context_id();
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        const ScratchSlot& s = g_scratch_slot[dev];
        if (ctx != 0 && s.ctx == ctx && s.addr) {
            *out = s.addr;
            return ZERO_OK;
        }
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_mlp4_scratch);
    if (e != cudaSuccess) return zero_record_cuda_error(static_cast<int>(e));
    // the lookup makes the device's primary context current if it was not
    const unsigned long long now = ctx != 0 ? ctx : current_context_id();
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        g_scratch_slot[dev] = ScratchSlot{now, p};
    }
    *out = p;
    return ZERO_OK;
}

} // namespace

extern "C" int zero_mlp4_zero3_step_noalloc(const float* x, int32_t P, int32_t n, float* master, float* m,
                                            float* v, void* shard_fp16, float* loss, int64_t t, float lr,
                                            float beta1, float beta2, float eps, int32_t mode, void* cuda_stream)
{
    // every argument is checked before anything is enqueued (P above
    // kMaxRanks: more ranks' gradients than the scratch holds)
    int rc = check_mlp4_step(x, P, n, nullptr, master, m, v, shard_fp16, nullptr, 0, loss, t, lr, beta1, beta2, eps,
                             mode, false);
    if (rc) return rc;
    void* scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc) return rc;
    // no caller buffer may lie inside the scratch
    const uintptr_t sb = reinterpret_cast<uintptr_t>(scratch), se = sb + sizeof(g_mlp4_scratch);
    const uintptr_t ends[][2] = {
        {reinterpret_cast<uintptr_t>(x), static_cast<uintptr_t>(P) * static_cast<uintptr_t>(n) * 4},
        {reinterpret_cast<uintptr_t>(master), kParams * 4},
        {reinterpret_cast<uintptr_t>(m), kParams * 4},
        {reinterpret_cast<uintptr_t>(v), kParams * 4},
        {reinterpret_cast<uintptr_t>(shard_fp16), kParams * 2},
        {reinterpret_cast<uintptr_t>(loss), static_cast<uintptr_t>(P) * 4}};
    for (const auto& b : ends)
        if (b[0] < se && sb < b[0] + b[1]) return ZERO_EOVERLAP;
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
