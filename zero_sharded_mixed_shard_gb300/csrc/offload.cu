// ZeRO-Offload's pipelined step: the GPU forms each piece's gradient mean and
// sends it to page-locked host memory as fp16 (zero_reduce_scatter_fp16),
// host threads run Adam on the piece beside the fp32 state in host memory
// (zero_cpu_adam), and the piece's fp16 weights are copied back into the
// gathered device vector, while the neighbouring pieces are reduced and
// copied.
//
// Sources (page title, section):
//  ZeRO 技术原理：进阶与 Offload §2.2 Offload 策略: the data-flow graph is cut
//    along the fp16 gradient and fp16 parameter edges; the parameter update
//    and float2half run on the CPU next to the Adam state.
//  §2.3 扩展性: each GPU's 1/N shard is updated by CPU workers.
//  §1.6.7 (CUDA streams): transfers and computation on separate streams run
//    at the same time.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <new>

#include "zero_step.h"

__attribute__((visibility("hidden"))) int zero_record_cuda_error(int err);
__attribute__((visibility("hidden"))) int zero_check_step_scalars(int64_t N, int32_t P, int32_t stage, int64_t t,
                                                                  float lr, float b1, float b2, float eps,
                                                                  int32_t mode);

namespace {

// The CPU update of one piece of the vector (whole shards, contiguous), run
// by the CUDA driver as a host function; one dynamically scheduled pass of
// the host threads over the piece updates every rank's shard in it (the
// offload strategy gives each GPU's shard to CPU workers); chunks go to
// whichever thread is free.
struct OffloadUpdate {
    const void* g16;
    float* w;
    float* m;
    float* v;
    void* p16;
    int64_t N;
    int64_t t;
    float lr, b1, b2, eps;
    int32_t mode;
    int32_t threads;
};

void CUDART_CB offload_update(void* arg)
{
    OffloadUpdate* u = static_cast<OffloadUpdate*>(arg);
    // the arguments were validated when the step was enqueued
    (void)zero_cpu_adam(u->g16, u->w, u->m, u->v, u->p16, u->N, u->t, u->lr, u->b1, u->b2, u->eps, u->mode,
                        u->threads);
    delete u;
}

// The offload step runs as a pipeline over pieces of the vector (groups of
// whole shards): the GPU reduces piece j+1 while the host updates piece j
// and piece j-1's weights cross back.  Host functions run on one internal
// stream and the weight copies on another, one pair per device, created on
// first use and kept; events order the three streams.
constexpr int kOffloadPieces = 16;
constexpr int64_t kOffloadMinPiece = int64_t(1) << 20; // elements

struct OffloadStreams {
    cudaStream_t host = nullptr;
    cudaStream_t copy = nullptr;
};

int offload_streams(OffloadStreams* out)
{
    static std::mutex mu;
    static OffloadStreams table[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return zero_record_cuda_error(static_cast<int>(e));
    if (dev < 0 || dev >= 64) return ZERO_EINVAL;
    std::lock_guard<std::mutex> lk(mu);
    OffloadStreams& s = table[dev];
    if (!s.host) {
        cudaStream_t h = nullptr, c = nullptr;
        e = cudaStreamCreateWithFlags(&h, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c, cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            if (h) cudaStreamDestroy(h);
            return zero_record_cuda_error(static_cast<int>(e));
        }
        s.host = h;
        s.copy = c;
    }
    *out = s;
    return ZERO_OK;
}

// `waiter` waits for the work enqueued so far on `src` (a fresh event each
// time; destroying it at once is allowed, the wait stays enqueued).
cudaError_t stream_after(cudaStream_t waiter, cudaStream_t src)
{
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    e = cudaEventRecord(ev, src);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(waiter, ev, 0);
    cudaEventDestroy(ev);
    return e;
}

} // namespace

extern "C" int zero_offload_step(const void* grads_fp16, int64_t rank_stride, float* master_host, float* m_host,
                                 float* v_host, void* grad16_host, void* params16_host, void* params_fp16,
                                 int64_t N, int32_t P, int32_t stage, int64_t t, float lr, float beta1,
                                 float beta2, float eps, int32_t mode, int32_t cpu_threads, void* cuda_stream)
{
    int rc = zero_check_step_scalars(N, P, stage, t, lr, beta1, beta2, eps, mode);
    if (rc) return rc;
    if (rank_stride < N || cpu_threads < 0 || cpu_threads > 1024) return ZERO_EINVAL;
    if (mode > ZERO_MODE_FOLDED_STORAGE) return ZERO_EINVAL; // the host update is Adam
    if (!grads_fp16 || !master_host || !m_host || !v_host || !grad16_host || !params16_host || !params_fp16)
        return ZERO_EINVAL;
    // every check the pieces' calls below would make, before anything is
    // enqueued: a refused call writes nothing
    if (reinterpret_cast<uintptr_t>(master_host) % 4 || reinterpret_cast<uintptr_t>(m_host) % 4 ||
        reinterpret_cast<uintptr_t>(v_host) % 4 || reinterpret_cast<uintptr_t>(params16_host) % 2 ||
        reinterpret_cast<uintptr_t>(params_fp16) % 2 || reinterpret_cast<uintptr_t>(grads_fp16) % 2 ||
        reinterpret_cast<uintptr_t>(grad16_host) % 2)
        return ZERO_EALIGN;
    {
        const uintptr_t gg = reinterpret_cast<uintptr_t>(grads_fp16);
        const uintptr_t g_span = (static_cast<uintptr_t>(P - 1) * static_cast<uintptr_t>(rank_stride) +
                                  static_cast<uintptr_t>(N)) * 2;
        const uintptr_t h = reinterpret_cast<uintptr_t>(grad16_host), hb = static_cast<uintptr_t>(N) * 2;
        if (gg < h + hb && h < gg + g_span) return ZERO_EOVERLAP;
    }
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    OffloadStreams side;
    rc = offload_streams(&side);
    if (rc) return rc;
    const int64_t M = N / P + (N % P != 0);
    const auto shard_begin = [&](int64_t k) { return k * M < N ? k * M : N; };
    int64_t pieces = P < kOffloadPieces ? P : kOffloadPieces;
    const int64_t by_size = (N + kOffloadMinPiece - 1) / kOffloadMinPiece;
    if (pieces > by_size) pieces = by_size;
    const uint16_t* g16 = static_cast<const uint16_t*>(grad16_host);
    uint16_t* p16 = static_cast<uint16_t*>(params16_host);
    uint16_t* params = static_cast<uint16_t*>(params_fp16);

    cudaError_t ce = cudaSuccess;
    for (int64_t j = 0; j < pieces && ce == cudaSuccess && rc == ZERO_OK; ++j) {
        const int64_t k0 = j * P / pieces, k1 = (j + 1) * P / pieces;
        const int64_t b = shard_begin(k0), e = shard_begin(k1);
        if (b >= e) continue;
        // 1. the GPU side of every rank: the fp16 gradient mean of the piece
        //    lands in host memory
        rc = zero_reduce_scatter_fp16(grads_fp16, rank_stride, b, P, e - b, const_cast<uint16_t*>(g16) + b,
                                      cuda_stream);
        if (rc) break;
        // 2. the host update of the piece, once its gradients have arrived
        ce = stream_after(side.host, stream);
        if (ce != cudaSuccess) break;
        OffloadUpdate* u = new (std::nothrow) OffloadUpdate{g16 + b, master_host + b, m_host + b, v_host + b,
                                                            p16 + b, e - b, t, lr, beta1, beta2, eps, mode,
                                                            cpu_threads};
        if (!u) {
            rc = ZERO_ENOMEM;
            break;
        }
        ce = cudaLaunchHostFunc(side.host, offload_update, u);
        if (ce != cudaSuccess) {
            delete u;
            break;
        }
        // 3. the all-gather: shard k's fp16 weights at offset kM of the device vector
        ce = stream_after(side.copy, side.host);
        for (int64_t k = k0; k < k1 && ce == cudaSuccess; ++k) {
            const int64_t sb = shard_begin(k), se = shard_begin(k + 1);
            if (sb < se)
                ce = cudaMemcpyAsync(params + sb, p16 + sb, static_cast<size_t>(se - sb) * 2,
                                     cudaMemcpyHostToDevice, side.copy);
        }
    }
    // the caller's stream passes this step only when all of it is done (also
    // after a failure part-way, for what was enqueued)
    const cudaError_t j1 = stream_after(stream, side.host);
    const cudaError_t j2 = stream_after(stream, side.copy);
    if (rc) return rc;
    if (ce != cudaSuccess) return zero_record_cuda_error(static_cast<int>(ce));
    if (j1 != cudaSuccess) return zero_record_cuda_error(static_cast<int>(j1));
    if (j2 != cudaSuccess) return zero_record_cuda_error(static_cast<int>(j2));
    return ZERO_OK;
}
