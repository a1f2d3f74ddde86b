/*
 * zero_step.h -- C ABI of the fused ZeRO partitioned mixed-precision Adam step
 * for NVIDIA GB300 (sm_103a).
 *
 * P data-parallel ranks are simulated on one GPU: each holds an fp16 local
 * gradient in device memory.  For every shard k of the flat parameter vector
 * (M = ceil(N/P) elements, the last one shorter or empty) one pass
 *   1. reduce-scatters: averages the P gradient slices of the shard in fp32,
 *      rank order 0..P-1;
 *   2. runs Adam on the fp32 master / momentum / variance shard;
 *   3. casts the new weights to fp16 (round to nearest, ties to even);
 *   4. writes them into the fp16 parameter vector at the shard's offset,
 *      which is the all-gather's output.
 * No intermediate gradient buffer is written: the mean lives in registers.
 *
 * Sources (page title, section):
 *  [P1] 深度学习专题：模型训练的数据并行（三） §（一）Adam 优化器 (update and
 *       moment equations, beta defaults, m0 = v0 = 0); §（二） (storage per
 *       GPU for plain data parallel); §（三）-（五） ZeRO-1/2/3 优化原理
 *       (ceil partition M = ceil(N/P), s_k = 1+(k-1)M .. e_k = kM, the
 *       reduce-scatter / update / all-gather steps, float counts per GPU).
 *  [P2] ZeRO 原理：把模型状态切到多张 GPU 上 (7.5B parameters on 64 GPUs:
 *       120 / 31.4 / 16.6 / 1.9 GB; fp32 master cast back to fp16 on the
 *       owning GPU).
 *  [P3] ZeRO 技术原理：进阶与 Offload §1.1.5 Reduce-Scatter, §1.1.6
 *       All-Gather, §1.4 显存分析 (16Φ bytes; P_os, P_os+g, P_os+g+p),
 *       §1.5 通信数据量分析 (2Φ / 3Φ per card), reference [10] Kingma & Ba.
 *  [P4] 高效AI 第19讲：分布式训练（第一部分） 通信原语 All-Reduce
 *       (g = (1/N) Σ g_i), ZeRO 和 FSDP (bytes per parameter).
 *
 * General rules for every function below:
 *  - Return 0 (ZERO_OK) on success or a negative ZERO_E* code; the code's
 *    text is zero_strerror(code).  A rejected call has no side effects.
 *  - Device pointers are caller-owned (for example torch tensors).  The
 *    library never allocates or frees device memory; kernels are enqueued
 *    on the caller's stream and the call returns immediately.  The only
 *    calls that wait for the device are the two diagnostics that read a
 *    device counter back (zero_device_timeouts, zero_selftest_mean_division);
 *    zero_cpu_adam runs on the calling host thread.  The offload step
 *    keeps two internal streams per device and the host Adam a pool of
 *    host threads, both created on first use and kept.
 *  - Element counts and strides are in elements, not bytes.
 *  - fp16 buffers are passed as void* holding IEEE binary16 codes.
 *  - zero_adam_step, zero_adam_step_shard and zero_adam_step_range enqueue
 *    one kernel launch on the stream and nothing else.  The first call for a
 *    kernel on a device also sets that kernel up (function attributes,
 *    occupancy); after it, calls on a capturing stream are recorded into a
 *    CUDA graph like any launch, and replaying the graph repeats the steps
 *    with the arguments they were captured with (t included).
 */
#ifndef ZERO_STEP_H
#define ZERO_STEP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------ */
/* Status codes                                                             */
/* ------------------------------------------------------------------------ */
#define ZERO_OK 0
#define ZERO_EINVAL (-1)   /* bad argument: null pointer, size, stage, mode, t, hyper-parameter */
#define ZERO_EALIGN (-2)   /* a pointer is not aligned to its element size (4 B fp32, 2 B fp16) */
#define ZERO_EOVERLAP (-3) /* output buffers overlap each other or the gradients */
#define ZERO_ECUDA (-4)    /* the CUDA runtime rejected the launch (see zero_last_cuda_error) */
#define ZERO_ENOMEM (-5)   /* host allocation for a layout table failed */

#define ZERO_MAX_RANKS 1024 /* largest P accepted */

/* Adam readings (see zero_adam_step). */
#define ZERO_MODE_STANDARD 0       /* m, v are raw moving averages; bias-corrected in the update */
#define ZERO_MODE_FOLDED_LITERAL 1 /* [P1] §（一） as printed: recursion on the divided m, v */
#define ZERO_MODE_FOLDED_STORAGE 2 /* stored m, v are bias-corrected; recursion on the raw average */
#define ZERO_MODE_SGD 3            /* [P1] §（一）: w <- w - lr g; m and v unused (may be NULL) */
#define ZERO_MODE_MOMENTUM 4       /* [P3] §1.1.1 SGD with momentum: m <- beta1 m + g, w <- w - lr m;
                                      v unused (may be NULL) */

/* ------------------------------------------------------------------------ */
/* Layout table (host only, no CUDA)                                        */
/* ------------------------------------------------------------------------ */

/* One piece of a flattened tensor that lies inside one shard. */
typedef struct {
    int64_t tensor_id;     /* index into the tensor list given to zero_init_layout */
    int64_t tensor_offset; /* first element of the piece within the tensor */
    int64_t shard_offset;  /* first element of the piece within the shard */
    int64_t len;           /* elements in the piece (> 0) */
} zero_segment_t;

/* The ceil partition of a flat vector built from a list of tensors, the
 * pieces of tensors each shard holds, and the per-rank accounting of the
 * pages.  Filled by zero_init_layout; every array is host memory owned by
 * the table and released by zero_free_layout. */
typedef struct {
    int64_t N;              /* total elements (sum of tensor sizes) */
    int64_t M;              /* ceil(N / P): the size of every shard but the trailing ones */
    int32_t P;              /* ranks */
    int32_t stage;          /* 0 = plain data parallel, 1/2/3 = ZeRO-1/2/3 */
    int32_t n_tensors;
    int32_t reserved;
    int64_t* shard_begin;   /* [P] first element of shard k: min(k*M, N) */
    int64_t* shard_end;     /* [P] one past the last: min((k+1)*M, N); begin == end when empty */
    int64_t* seg_offsets;   /* [P+1] shard k's pieces are segs[seg_offsets[k] .. seg_offsets[k+1]) */
    zero_segment_t* segs;   /* pieces in flat order */
    int64_t n_segs;
    double bytes_per_rank_mixed; /* model-state bytes per rank, K = 12 ([P3] §1.4) */
    double floats_per_rank_p1;   /* float count per rank ([P1] §（二）-（五）) */
    double comm_elems_per_rank;  /* elements sent + received per rank per step ([P3] §1.5) */
} zero_layout_t;

/* Build the layout table of the flat vector formed by concatenating
 * n_tensors tensors of tensor_numel[i] elements (each >= 0, total >= 1),
 * partitioned over P ranks ([P1] §（三） 准备步骤, 0-based: shard k is
 * [min(kM,N), min((k+1)M,N)); a shard past the end is empty).
 * stage selects the accounting only.  On success *out owns heap memory that
 * must be released with zero_free_layout.  Errors: ZERO_EINVAL (null
 * pointer, n_tensors < 1, a negative size, N < 1, P outside
 * [1, ZERO_MAX_RANKS], stage outside [0, 3]); ZERO_ENOMEM. */
int zero_init_layout(const int64_t* tensor_numel, int32_t n_tensors, int32_t P,
                     int32_t stage, zero_layout_t* out);

/* Release the arrays of a table filled by zero_init_layout and zero its
 * fields.  Accepts NULL and an already-freed table. */
void zero_free_layout(zero_layout_t* layout);

/* Shard bounds without a table: *begin = min(k*M, N), *end = min((k+1)*M, N)
 * with M = ceil(N/P).  Errors: ZERO_EINVAL (null output, N < 1, P outside
 * [1, ZERO_MAX_RANKS], k outside [0, P)). */
int zero_shard_range(int64_t N, int32_t P, int32_t k, int64_t* begin, int64_t* end);

/* Per-rank accounting for N parameters over P ranks at a ZeRO stage:
 *  *bytes_mixed  fp16 parameters + fp16 gradients + 12 bytes of fp32 Adam
 *                state per parameter, divided by stage: 16N, 4N + 12N/P,
 *                2N + 14N/P, 16N/P ([P3] §1.4; [P4] ZeRO 和 FSDP);
 *  *floats_p1    untyped float count: 4N, 2M + 2N, 3M + N, 4M ([P1]);
 *  *comm_elems   elements moved per rank per step: 2N for stages 0-2, 3N
 *                for stage 3 ([P3] §1.5).
 * Any output pointer may be NULL.  Errors: ZERO_EINVAL (N < 1, P outside
 * [1, ZERO_MAX_RANKS], stage outside [0, 3]). */
int zero_memory_bytes(int64_t N, int32_t P, int32_t stage, double* bytes_mixed,
                      double* floats_p1, double* comm_elems);

/* ------------------------------------------------------------------------ */
/* The fused step (device)                                                  */
/* ------------------------------------------------------------------------ */

/* One ZeRO optimizer step over the whole flat vector: all P shards' updates
 * in one launch on `cuda_stream` (a cudaStream_t; NULL = legacy default).
 *
 *  grads_fp16   device, fp16 [P][rank_stride]: rank r's local gradient of the
 *               N parameters starts at element r * rank_stride (read only).
 *  rank_stride  elements between ranks, >= N.  A multiple of 8 lets every
 *               rank's slice share one 16-byte phase (the fast path); any
 *               value is accepted.
 *  master, m, v device fp32 [N], read and written in place.
 *  params_fp16  device fp16 [N], written (never read): element i receives
 *               fp16(new master[i]) -- shard k's values land at [kM, ...),
 *               i.e. this buffer is the all-gather's output.
 *  N            parameters (>= 1);  P  ranks, 1 <= P <= ZERO_MAX_RANKS.
 *  stage        0..3; documents the buffer roles and does not change any
 *               result (every stage computes the same bytes).
 *  t            1-based index of the update being produced (first step: 1).
 *  lr, beta1, beta2, eps   Adam hyper-parameters; finite, 0 <= beta < 1,
 *               eps >= 0 ([P1] §（一）: eps is added outside the sqrt).
 *  mode         ZERO_MODE_STANDARD, ZERO_MODE_FOLDED_LITERAL,
 *               ZERO_MODE_FOLDED_STORAGE (Adam: master, m, v), ZERO_MODE_SGD
 *               (master only: m and v are neither read nor written and may
 *               be NULL) or ZERO_MODE_MOMENTUM (master and m; v may be NULL;
 *               beta1 is the momentum coefficient, beta2 and eps are only
 *               validated).  Bytes moved per element: 2P + 26 for Adam,
 *               2P + 18 with momentum, 2P + 10 for plain SGD.
 *
 * Per element i, every operation a separately rounded fp32 operation
 * (no contraction), in this order:
 *   g  = ((0 + g_0[i]) + g_1[i]) + ... + g_{P-1}[i];   g = g / P
 *   bc1 = fp32(1 - beta1^t), bc2 = fp32(1 - beta2^t)   (host, in double)
 *   mode 0: m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*(g*g);  mh = m/bc1;  vh = v/bc2
 *   mode 1: m = (b1*m + (1-b1)*g)/bc1;  v = (b2*v + (1-b2)*(g*g))/bc2;  mh = m;  vh = v
 *   mode 2: with bp = fp32(1 - beta^(t-1)):
 *           m = (b1*(m*bp1) + (1-b1)*g)/bc1;  v = (b2*(v*bp2) + (1-b2)*(g*g))/bc2
 *   master = master - lr * (mh / (sqrt(vh) + eps));  params[i] = fp16_rne(master)
 *   mode 3: master = master - lr * g
 *   mode 4: m = b1*m + g;  master = master - lr * m
 *
 * Errors: ZERO_EINVAL, ZERO_EALIGN, ZERO_EOVERLAP (any two of master, m, v,
 * params overlap, or one of them overlaps the gradient span), ZERO_ECUDA.
 * The grids never wait on anything: the call cannot hang the GPU. */
int zero_adam_step(const void* grads_fp16, int64_t rank_stride, float* master, float* m,
                   float* v, void* params_fp16, int64_t N, int32_t P, int32_t stage,
                   int64_t t, float lr, float beta1, float beta2, float eps, int32_t mode,
                   void* cuda_stream);

/* One rank's part of the step: shard k = [min(kM,N), min((k+1)M,N)) of
 * length len_k, M = ceil(N/P) ([P1] §（四） 第二步..第五步).
 *
 *  grads_fp16   device fp16: rank r's gradient for the shard's first element
 *               is at element grad_offset + r * rank_stride.  Full per-rank
 *               gradients: grad_offset = k*M, rank_stride >= N.  A packed
 *               receive buffer [P][stride] of the shard only: grad_offset = 0,
 *               rank_stride >= len_k.
 *  master_s, m_s, v_s   device fp32 [len_k], the shard's state (for full
 *               vectors pass master + k*M etc.).
 *  params_out   device fp16 [len_k]: where shard k's new fp16 weights go --
 *               params + k*M for the all-gathered vector (stages 0-2), or a
 *               shard-local buffer (stage 3 keeps only its own shard).
 *  The other arguments are as for zero_adam_step.  An empty shard
 *  (len_k == 0) returns ZERO_OK without launching anything and without
 *  examining the buffer pointers (they may be NULL); the scalar arguments
 *  are still validated.
 * The concatenation over k = 0..P-1 of the shard calls equals
 * zero_adam_step bit for bit. */
int zero_adam_step_shard(const void* grads_fp16, int64_t rank_stride, int64_t grad_offset,
                         int32_t k, float* master_s, float* m_s, float* v_s,
                         void* params_out, int64_t N, int32_t P, int32_t stage, int64_t t,
                         float lr, float beta1, float beta2, float eps, int32_t mode,
                         void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* Buckets: the step of one part of the vector as soon as its gradients are  */
/* ready ([P3] §1.5 通信数据量分析: gradients are bucketed so every 1/N is    */
/* sent once, and sending overlaps the backward pass of earlier layers;       */
/* [P3] §1.4: small tensors are bucketed and moved together; [P3] §1.6.7:    */
/* separate CUDA streams let communication and computation run together).    */
/* ------------------------------------------------------------------------ */

/* One bucket: the flat range [begin, end) covering tensors first..last. */
typedef struct {
    int64_t begin;
    int64_t end;
    int32_t first_tensor;
    int32_t last_tensor;
} zero_bucket_t;

/* Group consecutive tensors of the flat vector (tensor_numel[0..n_tensors))
 * into buckets of at least bucket_elems elements each (the last bucket may be
 * smaller); a tensor is never split, so a tensor larger than bucket_elems is a
 * bucket of its own.  backward_order != 0 walks the tensors from the last to
 * the first (the order a backward pass produces their gradients) and lists
 * the buckets in that order; 0 walks them front to back.
 * Two-call pattern: with buckets_out == NULL only *n_buckets is set;
 * otherwise max_buckets is the capacity of buckets_out.  Host only.
 * Errors: ZERO_EINVAL (null tensor_numel / n_buckets, n_tensors < 1, a
 * negative size, total < 1, bucket_elems < 1, capacity too small). */
int zero_plan_buckets(const int64_t* tensor_numel, int32_t n_tensors, int64_t bucket_elems,
                      int32_t backward_order, zero_bucket_t* buckets_out, int32_t max_buckets,
                      int32_t* n_buckets);

/* The step of zero_adam_step restricted to flat elements [begin, end) of the
 * whole-vector layout (all pointers are the full-vector bases; rank r's
 * gradient of element i is at grads_fp16 + r * rank_stride + i).  The bytes
 * written equal those zero_adam_step writes for these elements.
 * Errors: as zero_adam_step, and ZERO_EINVAL unless 0 <= begin < end <= N. */
int zero_adam_step_range(const void* grads_fp16, int64_t rank_stride, int64_t begin, int64_t end,
                         float* master, float* m, float* v, void* params_fp16, int64_t N,
                         int32_t P, int32_t stage, int64_t t, float lr, float beta1, float beta2,
                         float eps, int32_t mode, void* cuda_stream);

/* The whole step as n_buckets range steps enqueued on step_stream in list
 * order; before bucket b the stream waits for ready_events[b] (a cudaEvent_t
 * recorded by the producer of that bucket's gradients, e.g. on the stream of
 * the backward pass; NULL = no wait).  The buckets must be disjoint
 * sub-ranges of [0, N); together with any elements left out they give the
 * same bytes as zero_adam_step.  The call only enqueues work: it returns
 * before any bucket runs.
 * Errors: as zero_adam_step; ZERO_EINVAL for a null bucket array, an empty
 * or out-of-range bucket, or overlapping buckets (checked before anything is
 * enqueued); ZERO_ECUDA if a wait or launch is refused (buckets enqueued
 * before it stay enqueued). */
int zero_adam_step_bucketed(const void* grads_fp16, int64_t rank_stride, float* master, float* m,
                            float* v, void* params_fp16, int64_t N, int32_t P, int32_t stage,
                            int64_t t, float lr, float beta1, float beta2, float eps, int32_t mode,
                            const zero_bucket_t* buckets, int32_t n_buckets,
                            void* const* ready_events, void* step_stream);

/* How many SMs a fused step may occupy (no counterpart on the pages; the
 * counterpart of cuBLAS's SM-count target).  [P3] §1.6.7 runs communication
 * and computation on separate CUDA streams at the same time; on one GPU they
 * can only run side by side when each leaves SMs to the other.  A step
 * enqueued while max_sms > 0 launches at most max_sms SMs' worth of CTAs
 * (the bulk-copy kernel: max_sms CTAs of one per SM), so a producer kernel
 * held below (SM count - max_sms) SMs keeps the rest; 0 (the default) = every
 * SM; a value above the SM count acts as 0.  Process-wide, read when a step
 * is enqueued (zero_adam_step, _shard, _range, each bucket of _bucketed, the
 * ZeRO-3 example's steps), so a caller can enqueue some buckets capped and
 * the rest uncapped.  The results do not depend on it: tiles are dealt to the
 * CTAs in a fixed round-robin order and each element's arithmetic is the
 * same.  *previous (if not NULL) receives the value it replaces.  Host only,
 * thread-safe (atomic).  Errors: ZERO_EINVAL (max_sms < 0). */
int zero_set_step_max_sms(int32_t max_sms, int32_t* previous);

/* Which kernel zero_adam_step would launch for these arguments (a
 * diagnostic with no counterpart on the pages; nothing is launched).
 * *kernel = ZERO_KERNEL_BULK for the bulk-copy pipeline (one CTA per SM,
 * used when every buffer shares one 16-byte phase and there are at least 4
 * tiles of 2048 elements per SM) or ZERO_KERNEL_VECTOR for the vector
 * kernel; *vector_width = the elements of one access (8 on the pipeline,
 * else 8, 4, 2 or 1 by alignment); *ctas = the CTAs of the launch.  Depends
 * on the current device's SM count and on zero_set_step_max_sms.
 * Errors: as zero_adam_step (the hyper-parameters are not taken), and
 * ZERO_EINVAL for a null output pointer. */
#define ZERO_KERNEL_BULK 1
#define ZERO_KERNEL_VECTOR 2
int zero_step_plan(const void* grads_fp16, int64_t rank_stride, float* master, float* m, float* v,
                   void* params_fp16, int64_t N, int32_t P, int32_t stage, int32_t mode,
                   int32_t* kernel, int32_t* vector_width, int64_t* ctas);

/* ------------------------------------------------------------------------ */
/* ZeRO-Offload ([P3] §2.2 Offload 策略: the data-flow graph is cut along    */
/* the fp16 gradient and fp16 parameter edges, so the parameter update and   */
/* float2half run on the CPU beside the Adam state in host memory; §2.3: each */
/* GPU's 1/N shard is updated by a CPU process; §1.6.6: that CPU Adam uses    */
/* multithreading and SIMD).  These are explicit entry points of their own: */
/* the fused GPU step never falls back to them.                              */
/* ------------------------------------------------------------------------ */

/* GPU side of the offloaded step: out_fp16[i] = fp16_rne((sum over ranks
 * r = 0..P-1, in order, of grads_fp16[grad_offset + r * rank_stride + i]) / P)
 * for i in [0, n), the mean formed exactly as zero_adam_step forms it.
 * out_fp16 may be device memory or page-locked host memory (the kernel then
 * writes across the host link itself).  Enqueued on cuda_stream.
 * Errors: ZERO_EINVAL (null pointer, n < 1, P outside [1, ZERO_MAX_RANKS],
 * grad_offset < 0, rank_stride < n when P > 1), ZERO_EALIGN (a pointer not
 * 2-byte aligned), ZERO_EOVERLAP (out_fp16 inside the gradients),
 * ZERO_ECUDA. */
int zero_reduce_scatter_fp16(const void* grads_fp16, int64_t rank_stride, int64_t grad_offset,
                             int32_t P, int64_t n, void* out_fp16, void* cuda_stream);

/* CPU side of the offloaded step, on host memory: Adam on n elements of
 * fp32 master / m / v from the fp16 gradient grad_fp16, and the fp16 cast of
 * the new weights into params_fp16 -- the same operations, in the same order
 * and precision, as zero_adam_step (given the gradient).  `threads` host
 * threads take chunks of 16 Ki elements as they are free (0 = one per CPU
 * in the process's affinity mask, which is also the most used; the calling
 * thread is one of them, the others come from a pool created on the first
 * call and kept for the life of the process).  One call runs at a time:
 * concurrent calls wait for each other.  Runs synchronously on the calling
 * thread.
 * Errors: ZERO_EINVAL (null pointer with n > 0, n < 0, t < 1, bad mode or
 * hyper-parameter, threads outside [0, 1024]). */
int zero_cpu_adam(const void* grad_fp16, float* master, float* m, float* v, void* params_fp16,
                  int64_t n, int64_t t, float lr, float beta1, float beta2, float eps,
                  int32_t mode, int32_t threads);

/* One ZeRO-Offload step of the whole vector.  The shards k = 0..P-1
 * ([min(kM,N), min((k+1)M,N))) are grouped into at most 16 pieces of whole
 * shards (fewer when N is small: at least 2^20 elements a piece), and for
 * each piece, in order:
 *   1. zero_reduce_scatter_fp16 of the piece into grad16_host, on
 *      cuda_stream;
 *   2. a host function (cudaLaunchHostFunc) that runs zero_cpu_adam on the
 *      piece with cpu_threads host threads (0 = all), writing params16_host,
 *      on an internal stream that waits for step 1 of the piece;
 *   3. one async copy per shard of the piece of its fp16 weights into
 *      params_fp16 at offset kM (the all-gather's output), on a second
 *      internal stream that waits for step 2 of the piece.
 * So the GPU reduces piece j+1 and piece j-1's weights cross back while the
 * host updates piece j.  cuda_stream then waits for both internal streams
 * (one pair per device, created on the first call and kept), so everything
 * after the call on cuda_stream sees the whole step, as if it had run in
 * stream order.  The results do not depend on the pieces.
 * grads_fp16 and params_fp16 are device memory; master_host, m_host, v_host
 * (fp32 [N]) and grad16_host, params16_host (fp16 [N]) are page-locked host
 * memory that the caller keeps alive, and leaves alone, until the stream has
 * passed this step.  The call returns at once.  Numerically the step differs
 * from zero_adam_step only in that the gradient mean is rounded to fp16 on
 * its way to the host.  Sizes, hyper-parameters, alignment and the
 * gradients' overlap with grad16_host are checked before anything is
 * enqueued.  Errors: ZERO_EINVAL (also for a current device numbered 64 or
 * above, which has no slot for the internal streams), ZERO_EALIGN,
 * ZERO_EOVERLAP, ZERO_ENOMEM (host bookkeeping), ZERO_ECUDA (pieces
 * enqueued before the failure stay enqueued, and cuda_stream still waits for
 * them when that is possible). */
int zero_offload_step(const void* grads_fp16, int64_t rank_stride, float* master_host, float* m_host,
                      float* v_host, void* grad16_host, void* params16_host, void* params_fp16,
                      int64_t N, int32_t P, int32_t stage, int64_t t, float lr, float beta1,
                      float beta2, float eps, int32_t mode, int32_t cpu_threads, void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* The layer-pipelined ZeRO-3 example: a 4-layer scalar MLP on P ranks      */
/* ([P1] §（四）ZeRO-3 层间流水线优化).  Parameters in flat order            */
/* (w1, b1, w2, b2, w3, b3, w4, b4); h_k = ReLU(w_k h_{k-1} + b_k), h_0 = x; */
/* y = w4 h3 + b4; L = (y - x)^2 / 2.  x is device fp32 [P][n]: rank r's n  */
/* samples; 1 <= P <= 8.                                                     */
/* ------------------------------------------------------------------------ */

/* loss[r] = mean over rank r's samples of (y - x)^2 / 2, with the fp16
 * parameters params_fp16 [8] (device).  Errors: ZERO_EINVAL, ZERO_ECUDA. */
int zero_mlp4_loss(const void* params_fp16, const float* x, int32_t P, int32_t n, float* loss,
                   void* cuda_stream);

/* Rank r's mean gradient over its samples of layer `layer`'s (w, b)
 * (1 <= layer <= 4), written as fp16 to grads_fp16[r * rank_stride +
 * 2 (layer - 1) + {0, 1}] -- the backward formulas of [P1] §（四） 1., with
 * the forward pass recomputed from x (no activations are kept).
 * Errors: ZERO_EINVAL (rank_stride < 8, bad sizes), ZERO_ECUDA. */
int zero_mlp4_layer_grads(int32_t layer, const void* params_fp16, const float* x, int32_t P,
                          int32_t n, void* grads_fp16, int64_t rank_stride, void* cuda_stream);

/* One ZeRO-3 training step with the page's layer pipeline
 * ([P1] §（四） 2. 前向传播和反向传播的层间流水线并行执行):
 *  - all-gather: the owners' fp16 shards shard_fp16 [8] are copied into the
 *    gathered vector gathered_fp16 [8] that the pass reads;
 *  - forward: loss[r] as zero_mlp4_loss;
 *  - backward, layer 4 down to 1, on main_stream (zero_mlp4_layer_grads into
 *    grads_fp16 [P][rank_stride]); as soon as the lowest layer of shard k
 *    (M = ceil(8/P) parameters, ceil partition) is done, step_stream waits
 *    for it and runs zero_adam_step_shard(k) (stage 3): reduce-scatter of the
 *    shard's gradients to its owner, Adam on master / m / v [8] (the owners'
 *    fp32 shards, concatenated) and the owner's fp16 shard written into
 *    shard_fp16 -- while main_stream goes on with the lower layers.
 *  pipelined = 0 puts everything on main_stream in the same order.  Before
 *  returning, main_stream is made to wait for every update, so the next
 *  step's all-gather sees them.  All buffers are device memory.
 *  Every argument is checked before anything is enqueued: sizes and
 *  hyper-parameters as for zero_adam_step_shard (ZERO_EINVAL), each buffer
 *  aligned to its element size (ZERO_EALIGN), and no two of x [P][n],
 *  gathered_fp16, master, m, v, shard_fp16, loss [P] and the gradients'
 *  span ((P-1) rank_stride + 8 elements) sharing a byte (ZERO_EOVERLAP);
 *  such a rejected call writes nothing.  A ZERO_ECUDA from the runtime part
 *  way through may leave the work enqueued before it in place.
 * Errors: ZERO_EINVAL, ZERO_EALIGN, ZERO_EOVERLAP, ZERO_ECUDA. */
int zero_mlp4_zero3_step(const float* x, int32_t P, int32_t n, void* gathered_fp16, float* master,
                         float* m, float* v, void* shard_fp16, void* grads_fp16,
                         int64_t rank_stride, float* loss, int64_t t, float lr, float beta1,
                         float beta2, float eps, int32_t mode, int32_t pipelined,
                         void* main_stream, void* step_stream);

/* zero_mlp4_zero3_step for callers that cannot allocate device memory (no
 * counterpart in the pages).  Some host programs reserve all of a GPU's
 * memory for their own allocator when they start and allow no allocation
 * afterwards -- any buffer a library asked them for would have to come out
 * of a budget they have already handed out -- and some services may not
 * allocate once they are running.  Such a caller cannot provide the scratch
 * zero_mlp4_zero3_step needs between its kernels (the all-gathered fp16
 * parameters and every rank's fp16 gradients).  Here that scratch is a
 * 256-byte array inside the library, fixed for the life of the process on
 * every GPU that loads it; the caller passes only the inputs and outputs:
 * x, master / m / v, the owners' fp16 shards and loss, as for
 * zero_mlp4_zero3_step.
 *  - Limit: the array holds at most 8 ranks' gradients; P outside [1, 8]
 *    returns ZERO_EINVAL.  Every argument is checked, as for
 *    zero_mlp4_zero3_step (no two of x, master, m, v, shard_fp16 and loss
 *    may share a byte, nor any of them a byte of the array), before
 *    anything is enqueued: a rejected call writes nothing.
 *  - Schedule: the serial one (pipelined = 0) on cuda_stream; the call
 *    neither allocates nor creates events.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and keeps it together
 *    with the identity of the device's context; a call that finds another
 *    context current (after cudaDeviceReset, or once the primary context
 *    was destroyed and created again, which can move the array) looks the
 *    address up again.  Make the first call on a device, and the first after
 *    a reset, before any stream capture.
 *  - Every call on a device uses the same array, which keeps the contents
 *    of the last call (each call writes every entry before reading it, so
 *    nothing needs clearing).  Calls whose work overlaps on the GPU -- on
 *    two streams, or from two host threads -- race on it: order them.
 * Errors: ZERO_EINVAL (also for a current device numbered 64 or above),
 * ZERO_EALIGN, ZERO_EOVERLAP, ZERO_ECUDA. */
int zero_mlp4_zero3_step_noalloc(const float* x, int32_t P, int32_t n, float* master, float* m,
                                 float* v, void* shard_fp16, float* loss, int64_t t, float lr,
                                 float beta1, float beta2, float eps, int32_t mode,
                                 void* cuda_stream);

/* Bounded waits that gave up, over every step launched on the current
 * device since the last reset.  The fused kernels wait on shared-memory
 * barriers for their own bulk copies; each wait gives up after 2 seconds,
 * lets the copies already issued land, counts itself here and returns, so
 * a stuck copy can never hang the GPU.  The count is 0 in every correct run;
 * a non-zero count means the outputs of some step are incomplete.
 * Reading it synchronises with the current device (cudaMemcpyFromSymbol);
 * reset != 0 sets it back to 0.  Errors: ZERO_EINVAL (count NULL),
 * ZERO_ECUDA. */
int zero_device_timeouts(int64_t* count, int32_t reset);

/* Diagnostic of the gradient mean for rank counts that are not powers of
 * two (no counterpart on the pages).  The fused kernels form sum / P without
 * a divide: with r = RN(1/P), q = RN(sum r), then q + RN(sum - q P) r by two
 * fused multiply-adds (Markstein's correction step).  Whether that rounds to
 * the correctly rounded quotient depends on P, so this call checks it on the
 * current device against the correctly rounded divide for every P in
 * [p_lo, p_hi] and every fp32 significand in [1, 2) -- 2^23 values per P,
 * which covers every nonzero sum of P fp16 gradients, since those lie in
 * [2^-24, 2^26] where scaling by a power of two scales each step exactly.
 * *mismatches receives the number of (P, significand) pairs that differ
 * (0 means the fast mean is the IEEE mean for those P); *first_p and
 * *first_sum (each may be NULL) the first one found, or 0.  Synchronous
 * (waits for its kernel on the legacy default stream); ~10 ms for all
 * 1024 rank counts.  Errors: ZERO_EINVAL (mismatches NULL, p_lo < 1,
 * p_hi < p_lo, p_hi > ZERO_MAX_RANKS), ZERO_ECUDA. */
int zero_selftest_mean_division(int32_t p_lo, int32_t p_hi, int64_t* mismatches, int32_t* first_p,
                                float* first_sum);

/* Diagnostic of the bounded waits (no counterpart on the pages): enqueues
 * the step of zero_adam_step (same arguments) through the bulk-copy kernel
 * with one shared-memory barrier of its first CTA told to expect 16 bytes
 * that no copy delivers.  That CTA's wait runs out after 2 seconds, it lets
 * its other copies land (the poisoned wait runs out once more), adds 1 to
 * the count of zero_device_timeouts and returns; every other CTA finishes
 * normally and the context stays usable.  The first CTA's tiles are left
 * partly updated, so the buffers hold no valid step afterwards.  Takes
 * about 4 s of GPU time.  Errors: as zero_adam_step, and ZERO_EINVAL when
 * the problem does not take the bulk-copy path (buffers on different 16-byte
 * phases, or fewer 2048-element tiles than SMs). */
int zero_selftest_wait_timeout(const void* grads_fp16, int64_t rank_stride, float* master, float* m,
                               float* v, void* params_fp16, int64_t N, int32_t P, int32_t stage,
                               int64_t t, float lr, float beta1, float beta2, float eps,
                               int32_t mode, void* cuda_stream);

/* Text of a status code (static storage; never NULL). */
const char* zero_strerror(int code);

/* The cudaError_t of the most recent ZERO_ECUDA on this thread (0 if none),
 * and its name from the CUDA runtime. */
int zero_last_cuda_error(void);
const char* zero_last_cuda_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_STEP_H */
