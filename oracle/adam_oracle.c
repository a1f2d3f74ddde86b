/*
 * CPU oracle for the ZeRO partitioned mixed-precision Adam step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * include this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no source, header or constant with the
 * CUDA library.
 *
 * It is deliberately plain and slow: every arithmetic operation is one IEEE
 * binary32 operation, rounded to nearest-even, in the order written below.
 * Build with -ffp-contract=off (no fused multiply-add) and without
 * -ffast-math; FLT_EVAL_METHOD must be 0 (true for x86-64 SSE and AArch64).
 *
 * Sources (page title, section):
 *  [P1] 深度学习专题：模型训练的数据并行（三） ("data parallelism in model
 *       training, part III"), §（一）Adam 优化器: the update
 *       w_{t+1} = w_t - lr * m_{t+1} / (sqrt(v_{t+1}) + eps), the moment
 *       equations with the bias correction divided into m and v, beta
 *       defaults 0.9 / 0.999 and m_0 = v_0 = 0.
 *  [P1] §（三）ZeRO-1 / §（四）ZeRO-2 优化原理, 准备步骤 and 第一步..第五步:
 *       the ceil partition M = ceil(N/P), the reduce-scatter of the gradient
 *       mean for elements s_k..e_k, the shard-local moment and parameter
 *       update, and the all-gather of the updated parameter vector.
 *  [P3] ZeRO 技术原理：进阶与 Offload, §1.1.1 (Adam keeps exponential moving
 *       averages of the gradient and its square), §1.1.5 Reduce-Scatter,
 *       §1.1.6 All-Gather, §1.4 (fp16 parameters and gradients, fp32 master
 *       copy, momentum and variance), reference [10] Kingma & Ba (the
 *       standard bias-corrected form).
 *  [P4] 高效AI 第19讲：分布式训练（第一部分）, 通信原语 / All-Reduce: the
 *       synchronised gradient is the mean g = (1/N) sum_i g_i over workers.
 *
 * Readings of points the pages leave open (each is also listed in the design
 * notes of the repository):
 *  - The gradient mean is an fp32 sum in rank order 0..P-1 starting from
 *    +0.0f, then one division by P.
 *  - t >= 1 is the index of the update being produced ([P1]'s t+1 with t
 *    counted from 0).  The bias-correction scalars are 1 - beta^t evaluated
 *    in double from the fp32 beta and rounded once to fp32.
 *  - mode 0: standard Adam ([P3] ref. [10]): m, v are raw moving averages;
 *    m_hat = m / (1 - b1^t), v_hat = v / (1 - b2^t).
 *    mode 1: [P1]'s folded equations read literally: the stored m, v are the
 *    already-divided values and the recursion runs on them.
 *    mode 2: folded *storage*: the stored m, v are the bias-corrected values,
 *    the recursion runs on the raw average recovered by multiplying back
 *    (1 - b^(t-1)).  Equal to mode 0 in exact arithmetic.
 *  - eps is added outside the square root ([P1]'s update equation).
 *  - fp32 -> fp16 rounds to nearest, ties to even; overflow gives +-inf;
 *    subnormal halves are kept.
 *  - No weight decay, clipping or loss scaling (the pages mention none).
 *  - mode 3: plain SGD, w <- w - lr * g ([P1] §（一）; m and v untouched).
 *    mode 4: SGD with momentum; [P3] §1.1.1 names it and its extra buffer
 *    but prints no formula, so the plainest form: m <- b1 * m + g,
 *    w <- w - lr * m (b1 plays the momentum coefficient; v untouched).
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if defined(FLT_EVAL_METHOD) && FLT_EVAL_METHOD != 0
#error "the oracle needs FLT_EVAL_METHOD == 0 (each float op rounded to binary32)"
#endif

/* ---------------------------------------------------------------------- */
/* IEEE 754 binary16 <-> binary32, written from the format's definition:   */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.                */
/* ---------------------------------------------------------------------- */

float oracle_half_to_float(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    float mag;
    if (expo == 0) {
        /* zero or subnormal: frac * 2^-24 (exact in binary32) */
        mag = ldexpf((float)frac, -24);
    } else if (expo == 31) {
        if (frac == 0) {
            mag = INFINITY;
        } else {
            /* NaN: keep the payload in the top fraction bits */
            uint32_t bits = ((uint32_t)sign << 31) | 0x7f800000u | ((uint32_t)frac << 13);
            float out;
            memcpy(&out, &bits, sizeof out);
            return out;
        }
    } else {
        /* normal: (1024 + frac) * 2^(expo - 15 - 10) (exact in binary32) */
        mag = ldexpf((float)(1024 + frac), expo - 25);
    }
    return sign ? -mag : mag;
}

uint16_t oracle_float_to_half(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    const uint16_t sign = (uint16_t)((bits >> 31) << 15);
    if (isnan(f)) {
        /* quiet NaN; keep the top fraction bits when they are non-zero */
        uint16_t payload = (uint16_t)((bits >> 13) & 0x3ff);
        return (uint16_t)(sign | 0x7c00 | 0x200 | payload);
    }
    const double a = fabs((double)f); /* exact */
    /* The largest finite half is 65504 = (2 - 2^-10) * 2^15.  The midpoint to
     * the next step (2^16) is 65520; a tie there goes to the even neighbour,
     * which is 2^16, i.e. infinity. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);          /* a = mant * 2^e2, mant in [0.5, 1) */
    int e = e2 - 1;               /* 2^e <= a < 2^(e+1) */
    if (e < -14) e = -14;         /* subnormal range shares the quantum 2^-24 */
    const double quantum = ldexp(1.0, e - 10);
    const double k = a / quantum; /* exact: division by a power of two */
    const double r = nearbyint(k); /* default rounding mode: nearest, ties to even */
    /* For e == -14 the encoding of r * 2^-24 is r itself (this covers both
     * subnormals and the smallest binade, including r == 1024).  For larger
     * e, r is in [1024, 2048] and r == 2048 carries into the exponent field. */
    uint32_t enc;
    if (e == -14) {
        enc = (uint32_t)r;
    } else {
        enc = ((uint32_t)(e + 15) << 10) + ((uint32_t)r - 1024u);
    }
    return (uint16_t)(sign | enc);
}

void oracle_half_to_float_array(const uint16_t* in, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_half_to_float(in[i]);
}

void oracle_float_to_half_array(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_float_to_half(in[i]);
}

/* ---------------------------------------------------------------------- */
/* Step scalars                                                            */
/* ---------------------------------------------------------------------- */

/* 1 - beta^t, evaluated in double from the fp32 beta, rounded once. */
static float one_minus_pow(float beta, int64_t t)
{
    return (float)(1.0 - pow((double)beta, (double)t));
}

typedef struct {
    float lr, b1, b2, eps;
    float omb1, omb2;     /* 1 - b1, 1 - b2 in fp32 */
    float bc1, bc2;       /* 1 - b^t */
    float bp1, bp2;       /* 1 - b^(t-1) (mode 2 only) */
    int mode;
} step_scalars;

static step_scalars make_scalars(int64_t t, float lr, float b1, float b2, float eps, int mode)
{
    step_scalars s;
    s.lr = lr;
    s.b1 = b1;
    s.b2 = b2;
    s.eps = eps;
    s.omb1 = 1.0f - b1;
    s.omb2 = 1.0f - b2;
    s.bc1 = one_minus_pow(b1, t);
    s.bc2 = one_minus_pow(b2, t);
    s.bp1 = one_minus_pow(b1, t - 1);
    s.bp2 = one_minus_pow(b2, t - 1);
    s.mode = mode;
    return s;
}

/* ---------------------------------------------------------------------- */
/* The three steps of one shard's update, over elements [0, n) of a range. */
/* ---------------------------------------------------------------------- */

/* Reduce-scatter, own part: g[j] = (sum over ranks r = 0..P-1 of the fp16
 * gradient of rank r at element j, widened to fp32) / P.  Rank r's slice
 * starts at grads + r * rank_stride. */
static void reduce_mean(const uint16_t* grads, int64_t rank_stride, int32_t P,
                        int64_t n, float* g)
{
    for (int64_t j = 0; j < n; ++j) {
        float acc = 0.0f;
        for (int32_t r = 0; r < P; ++r) {
            acc = acc + oracle_half_to_float(grads[(int64_t)r * rank_stride + j]);
        }
        g[j] = acc / (float)P;
    }
}

/* Adam on the fp32 shard state (master w, momentum m, variance v) given the
 * averaged gradient g. */
static void adam_update(const step_scalars* s, const float* g, float* w, float* m,
                        float* v, int64_t n)
{
    for (int64_t j = 0; j < n; ++j) {
        const float gj = g[j];
        const float gg = gj * gj;
        float m_new, v_new, m_hat, v_hat;
        if (s->mode == 0) {
            /* standard: raw exponential moving averages, corrected in the update */
            m_new = s->b1 * m[j] + s->omb1 * gj;
            v_new = s->b2 * v[j] + s->omb2 * gg;
            m_hat = m_new / s->bc1;
            v_hat = v_new / s->bc2;
        } else if (s->mode == 1) {
            /* the folded equations as printed: recursion on the divided values */
            m_new = (s->b1 * m[j] + s->omb1 * gj) / s->bc1;
            v_new = (s->b2 * v[j] + s->omb2 * gg) / s->bc2;
            m_hat = m_new;
            v_hat = v_new;
        } else if (s->mode == 3) {
            /* plain SGD ([P1] §（一）): w <- w - lr * g; no moments */
            w[j] = w[j] - s->lr * gj;
            continue;
        } else if (s->mode == 4) {
            /* SGD with momentum ([P3] §1.1.1 names it and its extra buffer, no
             * formula): m <- beta1 * m + g, w <- w - lr * m */
            m_new = s->b1 * m[j] + gj;
            w[j] = w[j] - s->lr * m_new;
            m[j] = m_new;
            continue;
        } else {
            /* folded storage: undo the previous step's correction, advance the
             * raw average, store the corrected value */
            m_new = (s->b1 * (m[j] * s->bp1) + s->omb1 * gj) / s->bc1;
            v_new = (s->b2 * (v[j] * s->bp2) + s->omb2 * gg) / s->bc2;
            m_hat = m_new;
            v_hat = v_new;
        }
        const float denom = sqrtf(v_hat) + s->eps;
        const float step = m_hat / denom;
        w[j] = w[j] - s->lr * step;
        m[j] = m_new;
        v[j] = v_new;
    }
}

/* fp32 -> fp16 of the updated master weights. */
static void cast_half(const float* w, uint16_t* p, int64_t n)
{
    for (int64_t j = 0; j < n; ++j) p[j] = oracle_float_to_half(w[j]);
}

/* The three steps over one contiguous element range, with its own gradient
 * scratch. Returns 0, or -1 when the scratch cannot be allocated. */
static int range_step(const uint16_t* grads, int64_t rank_stride, int32_t P,
                      float* w, float* m, float* v, uint16_t* p_out, int64_t n,
                      const step_scalars* s)
{
    if (n <= 0) return 0;
    float* g = (float*)malloc((size_t)n * sizeof(float));
    if (!g) return -1;
    reduce_mean(grads, rank_stride, P, n, g);
    adam_update(s, g, w, m, v, n);
    cast_half(w, p_out, n);
    free(g);
    return 0;
}

typedef struct {
    const uint16_t* grads;
    int64_t rank_stride;
    int32_t P;
    float *w, *m, *v;
    uint16_t* p_out;
    int64_t n;
    const step_scalars* s;
    int status;
} range_job;

static void* range_job_run(void* arg)
{
    range_job* j = (range_job*)arg;
    j->status = range_step(j->grads, j->rank_stride, j->P, j->w, j->m, j->v, j->p_out, j->n, j->s);
    return NULL;
}

/* Elements are independent, so a split into contiguous sub-ranges computed by
 * separate threads gives the same bytes as one thread. */
static int threaded_range_step(const uint16_t* grads, int64_t rank_stride, int32_t P,
                               float* w, float* m, float* v, uint16_t* p_out, int64_t n,
                               const step_scalars* s, int32_t threads)
{
    if (threads <= 1 || n < 4096) return range_step(grads, rank_stride, P, w, m, v, p_out, n, s);
    if (threads > 256) threads = 256;
    pthread_t tid[256];
    range_job jobs[256];
    int started[256];
    const int64_t chunk = (n + threads - 1) / threads;
    int rc = 0;
    for (int32_t i = 0; i < threads; ++i) {
        const int64_t lo = (int64_t)i * chunk;
        const int64_t hi = lo + chunk < n ? lo + chunk : n;
        jobs[i] = (range_job){grads + lo, rank_stride, P, w + lo, m + lo, v + lo,
                              p_out + lo, hi > lo ? hi - lo : 0, s, 0};
        started[i] = pthread_create(&tid[i], NULL, range_job_run, &jobs[i]) == 0;
        if (!started[i]) range_job_run(&jobs[i]);
    }
    for (int32_t i = 0; i < threads; ++i) {
        if (started[i]) pthread_join(tid[i], NULL);
        if (jobs[i].status) rc = jobs[i].status;
    }
    return rc;
}

static int check_common(int32_t P, int64_t t, int mode)
{
    if (P < 1 || t < 1 || mode < 0 || mode > 4) return -2;
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Public oracle entry points                                              */
/* ---------------------------------------------------------------------- */

/* The elementwise step over n elements of any contiguous range (a window of a
 * larger problem, or a whole shard): rank r's gradient for element j is at
 * grads[r * rank_stride + j]; w, m, v, params_out are the range's own n
 * entries.  Elements never interact, so a window gives exactly the values
 * the full problem gives at those elements. */
int oracle_adam_elems(const uint16_t* grads, int64_t rank_stride, int32_t P,
                      float* w, float* m, float* v, uint16_t* params_out, int64_t n,
                      int64_t t, float lr, float b1, float b2, float eps, int32_t mode,
                      int32_t threads)
{
    int rc = check_common(P, t, mode);
    if (rc) return rc;
    if (n < 0) return -2;
    const step_scalars s = make_scalars(t, lr, b1, b2, eps, mode);
    return threaded_range_step(grads, rank_stride, P, w, m, v, params_out, n, &s, threads);
}

/* The ZeRO step over the whole flat vector of N parameters, written as the
 * pages order it:  M = ceil(N/P); for each rank k (0-based) owning
 * [k*M, min((k+1)*M, N)):  reduce-scatter its slice of the gradient mean,
 * update its fp32 master / momentum / variance shard, cast the new weights to
 * fp16 into its own shard buffer, then all-gather every shard's fp16 buffer
 * into the full parameter vector at offset k*M.
 * grads: rank r's full local gradient at grads + r * rank_stride
 * (rank_stride >= N).  master, m, v, params: N entries each. */
int oracle_zero_step(const uint16_t* grads, int64_t rank_stride, int32_t P, int64_t N,
                     float* master, float* m, float* v, uint16_t* params,
                     int64_t t, float lr, float b1, float b2, float eps, int32_t mode,
                     int32_t threads)
{
    int rc = check_common(P, t, mode);
    if (rc) return rc;
    if (N < 1 || rank_stride < N) return -2;
    const step_scalars s = make_scalars(t, lr, b1, b2, eps, mode);
    const int64_t M = (N + P - 1) / P;
    uint16_t* shard_half = (uint16_t*)malloc((size_t)M * sizeof(uint16_t));
    if (!shard_half) return -1;
    for (int32_t k = 0; k < P; ++k) {
        const int64_t begin = (int64_t)k * M;
        const int64_t end = begin + M < N ? begin + M : N;
        if (begin >= end) continue; /* trailing ranks can own nothing */
        const int64_t len = end - begin;
        rc = threaded_range_step(grads + begin, rank_stride, P, master + begin, m + begin,
                                 v + begin, shard_half, len, &s, threads);
        if (rc) break;
        /* all-gather: shard k's fp16 values land at offset k*M */
        memcpy(params + begin, shard_half, (size_t)len * sizeof(uint16_t));
    }
    free(shard_half);
    return rc;
}

/* ZeRO-Offload's update ([P3] ZeRO 技术原理：进阶与 Offload §2.2 Offload 策略:
 * the data-flow graph is cut along the fp16 gradient and fp16 parameter
 * edges, so the optimizer update and the float2half node run on the CPU;
 * §2.3: each GPU hands its 1/N shard of fp16 gradients to a CPU process).
 * The gradient mean is formed as in reduce_mean, then crosses to the CPU as
 * fp16 (rounded to nearest even) and is widened back before Adam; the rest
 * is the same update and cast.  g16_out (optional, n codes) receives the
 * fp16 gradient that crossed. */
int oracle_offload_elems(const uint16_t* grads, int64_t rank_stride, int32_t P,
                         float* w, float* m, float* v, uint16_t* params_out, uint16_t* g16_out,
                         int64_t n, int64_t t, float lr, float b1, float b2, float eps,
                         int32_t mode)
{
    int rc = check_common(P, t, mode);
    if (rc) return rc;
    if (n < 0) return -2;
    if (n == 0) return 0;
    const step_scalars s = make_scalars(t, lr, b1, b2, eps, mode);
    float* g = (float*)malloc((size_t)n * sizeof(float));
    if (!g) return -1;
    reduce_mean(grads, rank_stride, P, n, g);                 /* on the GPU */
    for (int64_t j = 0; j < n; ++j) {                          /* the fp16 gradient edge */
        const uint16_t h = oracle_float_to_half(g[j]);
        if (g16_out) g16_out[j] = h;
        g[j] = oracle_half_to_float(h);
    }
    adam_update(&s, g, w, m, v, n);                            /* on the CPU */
    cast_half(w, params_out, n);                               /* float2half on the CPU */
    free(g);
    return 0;
}

/* Double-precision evaluation of the same formulas, for error-bound checks of
 * the fp32 path on small inputs (not a parity reference: the fp32 oracle is).
 * State in double, gradients given as fp16 codes, output weights in double. */
int oracle_adam_elems_f64(const uint16_t* grads, int64_t rank_stride, int32_t P,
                          double* w, double* m, double* v, int64_t n, int64_t t,
                          double lr, double b1, double b2, double eps, int32_t mode)
{
    int rc = check_common(P, t, mode);
    if (rc) return rc;
    const double bc1 = 1.0 - pow(b1, (double)t), bc2 = 1.0 - pow(b2, (double)t);
    const double bp1 = 1.0 - pow(b1, (double)(t - 1)), bp2 = 1.0 - pow(b2, (double)(t - 1));
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int32_t r = 0; r < P; ++r)
            acc += (double)oracle_half_to_float(grads[(int64_t)r * rank_stride + j]);
        const double g = acc / (double)P;
        double m_new, v_new, m_hat, v_hat;
        if (mode == 3) {
            w[j] = w[j] - lr * g;
            continue;
        }
        if (mode == 4) {
            m[j] = b1 * m[j] + g;
            w[j] = w[j] - lr * m[j];
            continue;
        }
        if (mode == 0) {
            m_new = b1 * m[j] + (1.0 - b1) * g;
            v_new = b2 * v[j] + (1.0 - b2) * g * g;
            m_hat = m_new / bc1;
            v_hat = v_new / bc2;
        } else if (mode == 1) {
            m_new = (b1 * m[j] + (1.0 - b1) * g) / bc1;
            v_new = (b2 * v[j] + (1.0 - b2) * g * g) / bc2;
            m_hat = m_new;
            v_hat = v_new;
        } else {
            m_new = (b1 * (m[j] * bp1) + (1.0 - b1) * g) / bc1;
            v_new = (b2 * (v[j] * bp2) + (1.0 - b2) * g * g) / bc2;
            m_hat = m_new;
            v_hat = v_new;
        }
        w[j] = w[j] - lr * (m_hat / (sqrt(v_hat) + eps));
        m[j] = m_new;
        v[j] = v_new;
    }
    return 0;
}
