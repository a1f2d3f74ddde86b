// Host side of the ZeRO step library: the ceil partition, the shard/tensor
// layout table and the per-rank accounting.  No CUDA in this file.
//
// Sources (page title, section):
//  深度学习专题：模型训练的数据并行（三） §（三）ZeRO-1 优化原理 准备步骤: each of
//    P GPUs manages M = ceil(N/P) parameters, GPU k (1-based) owns s_k =
//    1+(k-1)M .. e_k = kM; float counts per GPU 4N (§（二）), 2M+2N (§（三）),
//    3M+N (§（四）), 4M (§（五）).
//  ZeRO 技术原理：进阶与 Offload §1.4 显存分析: 16Φ bytes of model states,
//    P_os 4Φ+12Φ/N, P_os+g 2Φ+(2Φ+12Φ)/N, P_os+g+p 16Φ/N;  §1.5
//    通信数据量分析: about 2Φ per card for data parallel, ZeRO-1 and ZeRO-2,
//    3Φ (+50 %) for ZeRO-3.
// The page's e_k = kM can run past N for the trailing GPUs: shard bounds are
// clamped to N and a shard that starts at or past N is empty.
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "zero_step.h"

namespace {

inline bool bad_np(int64_t N, int32_t P) { return N < 1 || P < 1 || P > ZERO_MAX_RANKS; }

inline int64_t ceil_div(int64_t a, int64_t b) { return a / b + (a % b != 0); }

inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

void accounting(int64_t N, int32_t P, int32_t stage, double* bytes_mixed, double* floats_p1,
                double* comm_elems)
{
    const double phi = static_cast<double>(N);
    const double np = static_cast<double>(P);
    const double M = static_cast<double>(ceil_div(N, P));
    const double K = 12.0; // fp32 master + momentum + variance
    double b = 0.0, f = 0.0, c = 0.0;
    switch (stage) {
    case 0: b = (2.0 + 2.0 + K) * phi;          f = 4.0 * phi;           c = 2.0 * phi; break;
    case 1: b = 4.0 * phi + K * phi / np;        f = 2.0 * M + 2.0 * phi; c = 2.0 * phi; break;
    case 2: b = 2.0 * phi + (2.0 + K) * phi / np; f = 3.0 * M + phi;      c = 2.0 * phi; break;
    default: b = (2.0 + 2.0 + K) * phi / np;     f = 4.0 * M;             c = 3.0 * phi; break;
    }
    if (bytes_mixed) *bytes_mixed = b;
    if (floats_p1) *floats_p1 = f;
    if (comm_elems) *comm_elems = c;
}

} // namespace

extern "C" int zero_shard_range(int64_t N, int32_t P, int32_t k, int64_t* begin, int64_t* end)
{
    if (!begin || !end || bad_np(N, P) || k < 0 || k >= P) return ZERO_EINVAL;
    const int64_t M = ceil_div(N, P);
    *begin = min64(static_cast<int64_t>(k) * M, N);
    *end = min64(static_cast<int64_t>(k + 1) * M, N);
    return ZERO_OK;
}

extern "C" int zero_memory_bytes(int64_t N, int32_t P, int32_t stage, double* bytes_mixed,
                                 double* floats_p1, double* comm_elems)
{
    if (bad_np(N, P) || stage < 0 || stage > 3) return ZERO_EINVAL;
    accounting(N, P, stage, bytes_mixed, floats_p1, comm_elems);
    return ZERO_OK;
}

extern "C" void zero_free_layout(zero_layout_t* layout)
{
    if (!layout) return;
    std::free(layout->shard_begin);
    std::free(layout->shard_end);
    std::free(layout->seg_offsets);
    std::free(layout->segs);
    std::memset(layout, 0, sizeof(*layout));
}

extern "C" int zero_init_layout(const int64_t* tensor_numel, int32_t n_tensors, int32_t P,
                                int32_t stage, zero_layout_t* out)
{
    if (!tensor_numel || !out || n_tensors < 1 || stage < 0 || stage > 3) return ZERO_EINVAL;
    int64_t N = 0;
    for (int32_t i = 0; i < n_tensors; ++i) {
        if (tensor_numel[i] < 0) return ZERO_EINVAL;
        if (tensor_numel[i] > INT64_MAX - N) return ZERO_EINVAL;
        N += tensor_numel[i];
    }
    if (bad_np(N, P)) return ZERO_EINVAL;
    const int64_t M = ceil_div(N, P);

    // Walk shards and tensors together in flat order: each step emits the
    // overlap of the current shard and the current tensor, then advances
    // whichever of the two ends first.  O(P + n_tensors) pieces.
    std::vector<zero_segment_t> segs;
    std::vector<int64_t> offs(static_cast<size_t>(P) + 1, 0);
    try {
        segs.reserve(static_cast<size_t>(P) + static_cast<size_t>(n_tensors));
        int32_t tid = 0;
        int64_t tensor_start = 0; // flat index of tensor tid's first element
        for (int32_t k = 0; k < P; ++k) {
            offs[k] = static_cast<int64_t>(segs.size());
            const int64_t b = min64(static_cast<int64_t>(k) * M, N);
            const int64_t e = min64(b + M, N);
            int64_t pos = b;
            while (pos < e) {
                // skip tensors that end at or before pos (including empty ones)
                while (tid < n_tensors && tensor_start + tensor_numel[tid] <= pos) {
                    tensor_start += tensor_numel[tid];
                    ++tid;
                }
                const int64_t tensor_end = tensor_start + tensor_numel[tid];
                const int64_t piece_end = min64(e, tensor_end);
                segs.push_back(zero_segment_t{tid, pos - tensor_start, pos - b, piece_end - pos});
                pos = piece_end;
            }
        }
        offs[P] = static_cast<int64_t>(segs.size());
    } catch (const std::bad_alloc&) {
        return ZERO_ENOMEM;
    }

    zero_layout_t t;
    std::memset(&t, 0, sizeof(t));
    t.N = N;
    t.M = M;
    t.P = P;
    t.stage = stage;
    t.n_tensors = n_tensors;
    t.n_segs = static_cast<int64_t>(segs.size());
    t.shard_begin = static_cast<int64_t*>(std::malloc(sizeof(int64_t) * P));
    t.shard_end = static_cast<int64_t*>(std::malloc(sizeof(int64_t) * P));
    t.seg_offsets = static_cast<int64_t*>(std::malloc(sizeof(int64_t) * (P + 1)));
    t.segs = static_cast<zero_segment_t*>(std::malloc(sizeof(zero_segment_t) * (segs.size() + 1)));
    if (!t.shard_begin || !t.shard_end || !t.seg_offsets || !t.segs) {
        zero_free_layout(&t);
        return ZERO_ENOMEM;
    }
    for (int32_t k = 0; k < P; ++k) {
        t.shard_begin[k] = min64(static_cast<int64_t>(k) * M, N);
        t.shard_end[k] = min64(static_cast<int64_t>(k + 1) * M, N);
    }
    std::memcpy(t.seg_offsets, offs.data(), sizeof(int64_t) * (P + 1));
    if (!segs.empty()) std::memcpy(t.segs, segs.data(), sizeof(zero_segment_t) * segs.size());
    accounting(N, P, stage, &t.bytes_per_rank_mixed, &t.floats_per_rank_p1, &t.comm_elems_per_rank);
    *out = t;
    return ZERO_OK;
}

// Buckets of consecutive tensors, each at least bucket_elems long (the last
// one may be shorter); tensors are never split.  In backward order the walk
// starts from the last tensor, the order in which a backward pass finishes
// the gradients ([P3] §1.5: bucketed gradients, sent while earlier layers'
// gradients are still being computed).
extern "C" int zero_plan_buckets(const int64_t* tensor_numel, int32_t n_tensors, int64_t bucket_elems,
                                 int32_t backward_order, zero_bucket_t* buckets_out, int32_t max_buckets,
                                 int32_t* n_buckets)
{
    if (!tensor_numel || !n_buckets || n_tensors < 1 || bucket_elems < 1) return ZERO_EINVAL;
    std::vector<int64_t> start(static_cast<size_t>(n_tensors) + 1, 0);
    for (int32_t i = 0; i < n_tensors; ++i) {
        if (tensor_numel[i] < 0 || tensor_numel[i] > INT64_MAX - start[i]) return ZERO_EINVAL;
        start[i + 1] = start[i] + tensor_numel[i];
    }
    if (start[n_tensors] < 1) return ZERO_EINVAL;

    int32_t count = 0;
    int64_t acc = 0;
    int32_t first = -1; // tensor that opened the current bucket (in walk order)
    auto emit = [&](int32_t lo, int32_t hi) -> bool {
        // tensors lo..hi in flat order
        if (buckets_out) {
            if (count >= max_buckets) return false;
            buckets_out[count] = zero_bucket_t{start[lo], start[hi + 1], lo, hi};
        }
        ++count;
        return true;
    };
    for (int32_t step = 0; step < n_tensors; ++step) {
        const int32_t i = backward_order ? n_tensors - 1 - step : step;
        if (first < 0) first = i;
        acc += tensor_numel[i];
        if (acc >= bucket_elems) {
            const int32_t lo = first < i ? first : i, hi = first < i ? i : first;
            if (!emit(lo, hi)) return ZERO_EINVAL;
            first = -1;
            acc = 0;
        }
    }
    if (first >= 0) {
        const int32_t last = backward_order ? 0 : n_tensors - 1;
        const int32_t lo = first < last ? first : last, hi = first < last ? last : first;
        if (acc > 0 || count == 0) {
            if (!emit(lo, hi)) return ZERO_EINVAL;
        } else if (count > 0 && buckets_out) {
            // only empty tensors are left: fold them into the previous bucket
            zero_bucket_t& b = buckets_out[count - 1];
            if (lo < b.first_tensor) b.first_tensor = lo;
            if (hi > b.last_tensor) b.last_tensor = hi;
        }
    }
    *n_buckets = count;
    return ZERO_OK;
}
