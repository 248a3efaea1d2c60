// ddp_planner.cpp -- bucket assignment (host only).
//
// Rule ("DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事", section 03
// "Bucket" and "Overlap", section 05 step 2; "Day 17 · 梯度的集体行动"
// "bucket 与 overlap"): gradients become ready roughly in reverse
// registration order during backward, so buckets are filled walking the
// parameters from the last registered to the first.  The first bucket has
// its own, small cap (1 MiB by default) so that its allreduce can start
// early; the others use the bucket cap (25 MiB by default).  A bucket is
// closed as soon as its size reaches the cap; the trailing bucket is closed
// at the end.
#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include "ddp_abi_guard.h"
#include "ddp.h"
#include "ddp_trace.h"

extern "C" int32_t ddp_plan_buckets(int32_t n_params, const int64_t* numel, int32_t dtype,
                                    int64_t first_bucket_bytes, int64_t bucket_cap_bytes,
                                    int32_t* bucket_of_param, int64_t* offset_of_param, int64_t* bucket_numel,
                                    int32_t* n_buckets) try {
    DDP_TRACE_CALL();
    if (!n_buckets || n_params < 0) return DDP_ERR_INVALID;
    if (dtype != DDP_F32 && dtype != DDP_BF16) return DDP_ERR_INVALID;
    if (first_bucket_bytes <= 0 || bucket_cap_bytes <= 0) return DDP_ERR_INVALID;
    if (n_params > 0 && (!numel || !bucket_of_param || !offset_of_param || !bucket_numel)) return DDP_ERR_INVALID;
    const int64_t esize = (dtype == DDP_F32) ? 4 : 2;
    for (int32_t p = 0; p < n_params; ++p)
        if (numel[p] < 0 || numel[p] > (INT64_MAX / 4) / esize) return DDP_ERR_INVALID;

    int32_t bucket = 0;
    int64_t fill = 0;            // elements in the open bucket
    bool open = false;           // the open bucket holds at least one parameter
    int64_t cap = first_bucket_bytes;
    for (int32_t p = n_params - 1; p >= 0; --p) {
        if (fill > INT64_MAX / esize - numel[p]) return DDP_ERR_CAPACITY;   // bucket bytes would overflow
        bucket_of_param[p] = bucket;
        offset_of_param[p] = fill;
        fill += numel[p];
        open = true;
        if (fill * esize >= cap) {           // reached the cap: close it
            bucket_numel[bucket++] = fill;
            fill = 0;
            open = false;
            cap = bucket_cap_bytes;
        }
    }
    if (open) bucket_numel[bucket++] = fill;
    *n_buckets = bucket;
    const char* dbg = std::getenv("DDP_DEBUG");
    if (dbg && *dbg && *dbg != '0') {
        std::fprintf(stderr, "[ddp] plan: %d parameters -> %d buckets (first cap %lld B, cap %lld B)\n", n_params,
                     bucket, (long long)first_bucket_bytes, (long long)bucket_cap_bytes);
        for (int32_t k = 0; k < bucket; ++k)
            std::fprintf(stderr, "[ddp]   bucket %d: %lld elements (%lld B)\n", k, (long long)bucket_numel[k],
                         (long long)(bucket_numel[k] * esize));
    }
    return DDP_OK;
} DDP_ABI_CATCH

// 64-bit FNV-1a over the plan's integers, each fed as 8 little-endian bytes
// (the byte order is fixed here, so hosts of either endianness agree).
namespace {
struct Fnv64 {
    uint64_t h = 0xcbf29ce484222325ull;
    void add(int64_t v) {
        uint64_t u = (uint64_t)v;
        for (int b = 0; b < 8; ++b) {
            h ^= (u >> (8 * b)) & 0xffu;
            h *= 0x100000001b3ull;
        }
    }
};
}  // namespace

extern "C" int32_t ddp_plan_fingerprint(int32_t n_params, const int64_t* numel, int32_t dtype,
                                        const int32_t* bucket_of_param, const int64_t* offset_of_param,
                                        int32_t n_buckets, const int64_t* bucket_numel, uint64_t* fingerprint) try {
    DDP_TRACE_CALL();
    if (!fingerprint || n_params < 0 || n_buckets < 0) return DDP_ERR_INVALID;
    if (dtype != DDP_F32 && dtype != DDP_BF16) return DDP_ERR_INVALID;
    if (n_params > 0 && (!numel || !bucket_of_param || !offset_of_param)) return DDP_ERR_INVALID;
    if (n_buckets > 0 && !bucket_numel) return DDP_ERR_INVALID;
    Fnv64 f;
    f.add(n_params);
    f.add(dtype);
    for (int32_t p = 0; p < n_params; ++p) {
        f.add(numel[p]);
        f.add(bucket_of_param[p]);
        f.add(offset_of_param[p]);
    }
    f.add(n_buckets);
    for (int32_t k = 0; k < n_buckets; ++k) f.add(bucket_numel[k]);
    *fingerprint = f.h;
    return DDP_OK;
} DDP_ABI_CATCH
