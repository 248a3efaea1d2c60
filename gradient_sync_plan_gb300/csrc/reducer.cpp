// reducer.cpp -- DDP's reducer: launch each bucket's allreduce as soon as its
// gradients are ready, in bucket order, overlapped with the rest of backward.
//
// "DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事", section 03
// "Overlap" and section 05 step 2, and "Day 17 · 梯度的集体行动" "梯度同步时机"
// and the Reducer pseudo-code: a hook fires when a parameter's gradient is
// ready; when the last gradient of a bucket is ready, the bucket's
// asynchronous allreduce starts; buckets are launched in bucket order (bucket
// i+1 never before bucket i); before the optimizer reads the gradients every
// bucket must have finished.
//
// Here "a gradient is ready" means its producer has been enqueued on the
// caller's compute stream; the reducer records an event there when a bucket
// completes and makes its comm stream wait on that event before the bucket's
// sync (pack -> ring -> / N -> unpack, or the fused view kernel).
#include <cuda_runtime.h>

#include <algorithm>
#include <memory>
#include <mutex>
#include <new>
#include <vector>

#include "ddp_abi_guard.h"
#include "ddp.h"
#include "ddp_trace.h"

namespace ddpk {
// ddp_api.cpp: one bucket's pack -> fused ring -> unpack, in L2-sized pieces when large
int32_t pack_ring_unpack(int32_t world, int32_t n, const void* const* g, const int64_t* ne, const int64_t* off,
                         void* const* bk, int64_t bucket_numel, int32_t dtype, int32_t divisor, void* stream);
// ddp_api.cpp: the calling thread's CTA cap (-1: none), returns the previous one
int set_thread_cta_cap(int cap);
// ddp_api.cpp: one bucket's bf16-hook pack -> bf16 ring -> unpack, in L2-sized pieces when large
int32_t hook_pack_ring_unpack(int32_t world, int32_t n, const void* const* g, const int64_t* ne, const int64_t* off,
                              void* const* bk, int64_t bucket_numel, int32_t divisor, void* stream);
}  // namespace ddpk

struct ddp_reducer {
    int32_t world = 0, n_params = 0, n_buckets = 0, dtype = 0, divisor = 0, algo = 0;
    int32_t max_ctas = -1;            // CTA budget of this reducer's syncs (-1: the process-wide one)
    cudaStream_t comm = nullptr;
    std::vector<int32_t> bucket_of;
    std::vector<int64_t> bucket_numel;
    // per bucket: member tables laid out for ddp_bucket_* calls
    std::vector<std::vector<void*>> member_grads;     // [world * n_members]
    std::vector<std::vector<int64_t>> member_numel, member_offset;
    std::vector<std::vector<void*>> bucket_bufs;      // [world]
    std::vector<int32_t> n_members;
    std::vector<cudaEvent_t> ready_ev;                // per bucket, recorded on the compute stream
    std::vector<cudaEvent_t> t0_ev, t1_ev;            // per bucket, timing events around its sync (comm stream)
    std::vector<char> timed;                          // bucket k's timing events were recorded this pass
    cudaEvent_t done_ev = nullptr;
    // per-backward state
    std::vector<int32_t> pending;
    std::vector<char> param_ready, bucket_ready;
    int32_t next_launch = 0;
    std::vector<int32_t> launch_log;
    int32_t first_error = DDP_OK;
    std::mutex mu;
};

namespace {

bool dry(const ddp_reducer* r) { return r->algo == DDP_ALGO_DRYRUN; }

// Sets the calling thread's CTA cap for a scope and restores the previous
// one on every exit, exceptions included.
struct CtaCapGuard {
    int prev;
    explicit CtaCapGuard(int cap) : prev(ddpk::set_thread_cta_cap(cap)) {}
    ~CtaCapGuard() { ddpk::set_thread_cta_cap(prev); }
};

int32_t sync_bucket(ddp_reducer* r, int32_t k) {
    const int32_t n = r->n_members[k];
    void* const* g = r->member_grads[k].data();
    const int64_t* ne = r->member_numel[k].data();
    const int64_t* off = r->member_offset[k].data();
    if (r->algo == DDP_ALGO_VIEW)
        return ddp_bucket_allreduce_view(r->world, n, g, ne, off, r->bucket_numel[k], r->dtype, r->divisor, r->comm);
    if (r->algo == DDP_ALGO_BF16_HOOK_VIEW)
        return ddp_bucket_allreduce_view_bf16(r->world, n, g, ne, off, r->bucket_numel[k], r->divisor, r->comm);
    if (r->algo == DDP_ALGO_FP16_HOOK_VIEW)
        return ddp_bucket_allreduce_view_fp16(r->world, n, g, ne, off, r->bucket_numel[k], r->divisor, r->comm);
    void* const* b = r->bucket_bufs[k].data();
    if (r->algo == DDP_ALGO_BF16_HOOK)
        return ddpk::hook_pack_ring_unpack(r->world, n, (const void* const*)g, ne, off, b, r->bucket_numel[k],
                                           r->divisor, r->comm);
    if (r->algo == DDP_ALGO_FUSED)
        return ddpk::pack_ring_unpack(r->world, n, (const void* const*)g, ne, off, b, r->bucket_numel[k], r->dtype,
                                      r->divisor, r->comm);
    int32_t st = ddp_bucket_pack(r->world, n, (const void* const*)g, ne, off, b, r->bucket_numel[k], r->dtype, r->comm);
    if (st) return st;
    st = ring_allreduce_staged(r->world, b, r->bucket_numel[k], r->dtype, r->divisor, r->comm);
    if (st) return st;
    return ddp_bucket_unpack(r->world, n, g, ne, off, (const void* const*)b, r->bucket_numel[k], r->dtype, r->comm);
}

// Launch every bucket from next_launch on that is ready, in order.
int32_t launch_ready_prefix(ddp_reducer* r) {
    while (r->next_launch < r->n_buckets && r->bucket_ready[r->next_launch]) {
        const int32_t k = r->next_launch;
        if (!dry(r)) {
            if (cudaStreamWaitEvent(r->comm, r->ready_ev[k], 0) != cudaSuccess) return DDP_ERR_CUDA;
            // timing events cannot be recorded into a graph being captured
            cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
            if (cudaStreamIsCapturing(r->comm, &cap) != cudaSuccess) return DDP_ERR_CUDA;
            const bool time_it = cap == cudaStreamCaptureStatusNone;
            if (time_it && cudaEventRecord(r->t0_ev[k], r->comm) != cudaSuccess) return DDP_ERR_CUDA;
            int32_t st;
            {
                CtaCapGuard cap_guard(r->max_ctas);      // this reducer's budget for its own launches only
                st = sync_bucket(r, k);
            }
            if (st) return st;
            if (time_it && cudaEventRecord(r->t1_ev[k], r->comm) != cudaSuccess) return DDP_ERR_CUDA;
            r->timed[k] = time_it ? 1 : 0;
        }
        r->launch_log.push_back(k);
        ++r->next_launch;
    }
    return DDP_OK;
}

void reset_step(ddp_reducer* r) {
    for (int32_t k = 0; k < r->n_buckets; ++k) r->pending[k] = r->n_members[k];
    std::fill(r->param_ready.begin(), r->param_ready.end(), 0);
    std::fill(r->bucket_ready.begin(), r->bucket_ready.end(), 0);
    std::fill(r->timed.begin(), r->timed.end(), 0);
    r->next_launch = 0;
    r->launch_log.clear();
    r->first_error = DDP_OK;
}

void destroy_events(ddp_reducer* r) {
    for (auto* v : {&r->ready_ev, &r->t0_ev, &r->t1_ev}) {
        for (cudaEvent_t e : *v)
            if (e) cudaEventDestroy(e);
        v->clear();
    }
    if (r->done_ev) cudaEventDestroy(r->done_ev);
    r->done_ev = nullptr;
}

}  // namespace

extern "C" {

int32_t ddp_reducer_create(int32_t world, int32_t n_params, void* const* grads, const int64_t* numel, int32_t dtype,
                           const int32_t* bucket_of_param, const int64_t* offset_of_param, int32_t n_buckets,
                           const int64_t* bucket_numel, void* const* buckets, int32_t algo, int32_t divisor,
                           void* comm_stream, ddp_reducer** out) try {
    DDP_TRACE_CALL();
    if (!out) return DDP_ERR_INVALID;
    *out = nullptr;
    if (world < 1 || world > DDP_MAX_WORLD || n_params < 0 || n_buckets < 0 || divisor < 0) return DDP_ERR_INVALID;
    if (dtype != DDP_F32 && dtype != DDP_BF16) return DDP_ERR_INVALID;
    if (algo != DDP_ALGO_FUSED && algo != DDP_ALGO_STAGED && algo != DDP_ALGO_VIEW && algo != DDP_ALGO_DRYRUN &&
        algo != DDP_ALGO_BF16_HOOK && algo != DDP_ALGO_BF16_HOOK_VIEW && algo != DDP_ALGO_FP16_HOOK_VIEW)
        return DDP_ERR_INVALID;
    if ((algo == DDP_ALGO_BF16_HOOK || algo == DDP_ALGO_BF16_HOOK_VIEW || algo == DDP_ALGO_FP16_HOOK_VIEW) &&
        dtype != DDP_F32)
        return DDP_ERR_INVALID;
    if (n_params > 0 && (!numel || !bucket_of_param || !offset_of_param)) return DDP_ERR_INVALID;
    if (n_buckets > 0 && !bucket_numel) return DDP_ERR_INVALID;
    if (algo != DDP_ALGO_DRYRUN && n_params > 0 && !grads) return DDP_ERR_INVALID;
    const bool needs_buckets = algo == DDP_ALGO_FUSED || algo == DDP_ALGO_STAGED || algo == DDP_ALGO_BF16_HOOK;
    if (needs_buckets && n_buckets > 0 && !buckets) return DDP_ERR_INVALID;

    // owned by `holder` until the reducer is complete: an early return or a
    // failed host allocation below frees it
    std::unique_ptr<ddp_reducer> holder(new ddp_reducer());
    ddp_reducer* r = holder.get();
    r->world = world;
    r->n_params = n_params;
    r->n_buckets = n_buckets;
    r->dtype = dtype;
    r->divisor = divisor;
    r->algo = algo;
    r->comm = static_cast<cudaStream_t>(comm_stream);
    r->bucket_of.assign(bucket_of_param, bucket_of_param + n_params);
    r->bucket_numel.assign(bucket_numel, bucket_numel + n_buckets);
    std::vector<std::vector<int32_t>> members(n_buckets);
    for (int32_t p = 0; p < n_params; ++p) {
        const int32_t k = bucket_of_param[p];
        if (k < 0 || k >= n_buckets) {
            return DDP_ERR_INVALID;
        }
        members[k].push_back(p);
    }
    r->n_members.resize(n_buckets);
    r->member_grads.resize(n_buckets);
    r->member_numel.resize(n_buckets);
    r->member_offset.resize(n_buckets);
    r->bucket_bufs.resize(n_buckets);
    for (int32_t k = 0; k < n_buckets; ++k) {
        auto& m = members[k];
        std::sort(m.begin(), m.end(),
                  [&](int32_t a, int32_t b) { return offset_of_param[a] < offset_of_param[b]; });
        const int32_t n = (int32_t)m.size();
        r->n_members[k] = n;
        // members inside the bucket and disjoint (sorted by offset): a bad
        // plan is refused here, not in the middle of a backward pass
        int64_t end = 0;
        for (int32_t i = 0; i < n; ++i) {
            const int64_t o = offset_of_param[m[i]], e = numel[m[i]];
            if (e < 0 || o < 0 || o > r->bucket_numel[k] - e || (e > 0 && o < end)) {
                return DDP_ERR_INVALID;
            }
            if (e > 0) end = o + e;
            r->member_numel[k].push_back(e);
            r->member_offset[k].push_back(o);
        }
        if (algo != DDP_ALGO_DRYRUN) {
            r->member_grads[k].resize((size_t)world * n);
            for (int32_t w = 0; w < world; ++w)
                for (int32_t i = 0; i < n; ++i) r->member_grads[k][(size_t)w * n + i] = grads[(size_t)w * n_params + m[i]];
        }
        if (needs_buckets) {
            r->bucket_bufs[k].resize(world);
            for (int32_t w = 0; w < world; ++w) r->bucket_bufs[k][w] = buckets[(size_t)w * n_buckets + k];
        }
    }
    r->pending.resize(n_buckets);
    r->param_ready.resize(n_params);
    r->bucket_ready.resize(n_buckets);
    r->timed.resize(n_buckets);
    if (algo != DDP_ALGO_DRYRUN) {
        r->ready_ev.assign(n_buckets, nullptr);
        r->t0_ev.assign(n_buckets, nullptr);
        r->t1_ev.assign(n_buckets, nullptr);
        for (int32_t k = 0; k < n_buckets; ++k)
            if (cudaEventCreateWithFlags(&r->ready_ev[k], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreate(&r->t0_ev[k]) != cudaSuccess || cudaEventCreate(&r->t1_ev[k]) != cudaSuccess) {
                destroy_events(r);
                return DDP_ERR_CUDA;
            }
        if (cudaEventCreateWithFlags(&r->done_ev, cudaEventDisableTiming) != cudaSuccess) {
            destroy_events(r);
            return DDP_ERR_CUDA;
        }
    }
    reset_step(r);
    *out = holder.release();
    return DDP_OK;
} DDP_ABI_CATCH

int32_t ddp_reducer_set_max_ctas(ddp_reducer* r, int32_t max_ctas) try {
    DDP_TRACE_CALL();
    if (!r || max_ctas < -1) return DDP_ERR_INVALID;
    std::lock_guard<std::mutex> lk(r->mu);
    r->max_ctas = max_ctas;
    return DDP_OK;
} DDP_ABI_CATCH

int32_t ddp_reducer_prepare(ddp_reducer* r) try {
    DDP_TRACE_CALL();
    if (!r) return DDP_ERR_INVALID;
    std::lock_guard<std::mutex> lk(r->mu);
    reset_step(r);
    return DDP_OK;
} DDP_ABI_CATCH

int32_t ddp_reducer_mark_ready(ddp_reducer* r, int32_t param, void* compute_stream) try {
    DDP_TRACE_CALL();
    if (!r) return DDP_ERR_INVALID;
    std::lock_guard<std::mutex> lk(r->mu);
    if (param < 0 || param >= r->n_params || r->param_ready[param]) return DDP_ERR_INVALID;
    r->param_ready[param] = 1;
    const int32_t k = r->bucket_of[param];
    if (--r->pending[k] > 0) return DDP_OK;
    if (!dry(r) && cudaEventRecord(r->ready_ev[k], static_cast<cudaStream_t>(compute_stream)) != cudaSuccess)
        return DDP_ERR_CUDA;
    r->bucket_ready[k] = 1;
    const int32_t st = launch_ready_prefix(r);
    if (st && r->first_error == DDP_OK) r->first_error = st;
    return st;
} DDP_ABI_CATCH

int32_t ddp_reducer_finalize(ddp_reducer* r, void* stream) try {
    DDP_TRACE_CALL();
    if (!r) return DDP_ERR_INVALID;
    std::lock_guard<std::mutex> lk(r->mu);
    if (r->first_error != DDP_OK) return r->first_error;
    // buckets with no member are ready from the start
    for (int32_t k = 0; k < r->n_buckets; ++k)
        if (r->n_members[k] == 0 && !r->bucket_ready[k]) {
            if (!dry(r) && cudaEventRecord(r->ready_ev[k], static_cast<cudaStream_t>(stream)) != cudaSuccess)
                return DDP_ERR_CUDA;
            r->bucket_ready[k] = 1;
        }
    const int32_t st = launch_ready_prefix(r);
    if (st) return st;
    if (r->next_launch < r->n_buckets) return DDP_ERR_INVALID;   // a bucket never became ready
    if (dry(r)) return DDP_OK;
    if (cudaEventRecord(r->done_ev, r->comm) != cudaSuccess) return DDP_ERR_CUDA;
    if (cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), r->done_ev, 0) != cudaSuccess) return DDP_ERR_CUDA;
    return DDP_OK;
} DDP_ABI_CATCH

int32_t ddp_reducer_launch_order(ddp_reducer* r, int32_t* order, int32_t capacity, int32_t* n) try {
    DDP_TRACE_CALL();
    if (!r || !n || capacity < 0 || (capacity > 0 && !order)) return DDP_ERR_INVALID;
    std::lock_guard<std::mutex> lk(r->mu);
    *n = (int32_t)r->launch_log.size();
    for (int32_t i = 0; i < std::min(*n, capacity); ++i) order[i] = r->launch_log[i];
    return DDP_OK;
} DDP_ABI_CATCH

int32_t ddp_reducer_bucket_times(ddp_reducer* r, float* ms, int32_t capacity, int32_t* n) try {
    DDP_TRACE_CALL();
    if (!r || !n || capacity < 0 || (capacity > 0 && !ms)) return DDP_ERR_INVALID;
    std::lock_guard<std::mutex> lk(r->mu);
    *n = r->next_launch;
    for (int32_t k = 0; k < std::min(r->next_launch, capacity); ++k) {
        ms[k] = -1.0f;
        if (dry(r) || !r->timed[k]) continue;
        if (cudaEventSynchronize(r->t1_ev[k]) != cudaSuccess) return DDP_ERR_CUDA;
        if (cudaEventElapsedTime(&ms[k], r->t0_ev[k], r->t1_ev[k]) != cudaSuccess) return DDP_ERR_CUDA;
    }
    return DDP_OK;
} DDP_ABI_CATCH

int32_t ddp_reducer_destroy(ddp_reducer* r) try {
    DDP_TRACE_CALL();
    if (!r) return DDP_OK;
    destroy_events(r);
    delete r;
    return DDP_OK;
} DDP_ABI_CATCH

}  // extern "C"
