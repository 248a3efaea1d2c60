// ddp_api.cpp -- the C ABI: argument checks, launch geometry, the reducer loop.
//
// Every entry point validates on the host and returns a ddp_status before it
// enqueues anything; the kernels themselves live in ring_kernels.cu and
// bucket_kernels.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <iterator>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>

#include "ddp_abi_guard.h"
#include "ddp.h"
#include "ddp_trace.h"
#include "ddp_internal.h"

namespace ddpk {

DivSpec make_div(int32_t divisor) {
    DivSpec d{kDivNone, 1.0f};
    if (divisor <= 1) return d;
    if ((divisor & (divisor - 1)) == 0) {
        d.mode = kDivPow2;
        d.operand = std::ldexp(1.0f, -(int)std::log2((double)divisor));   // exact 2^-k
    } else {
        d.mode = kDivIeee;
        d.operand = (float)divisor;   // exact: divisor < 2^24
    }
    return d;
}

bool debug_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("DDP_DEBUG");
        return v && *v && *v != '0';
    }();
    return on;
}

namespace {
std::atomic<int> g_max_ctas{0};                              // 0 = no cap (ddp_set_max_ctas)
std::atomic<int> g_fused_kernel{DDP_FUSED_AUTO};             // ddp_set_fused_kernel
}  // namespace

int fused_kernel_override() { return g_fused_kernel.load(std::memory_order_relaxed); }

namespace {
thread_local int t_cta_cap = -1;      // a reducer's own budget while it launches (-1: none set)
}  // namespace

int set_thread_cta_cap(int cap) {
    const int prev = t_cta_cap;
    t_cta_cap = cap;
    return prev;
}

int cta_cap() { return t_cta_cap >= 0 ? t_cta_cap : g_max_ctas.load(std::memory_order_relaxed); }

int cap_ctas(int64_t grid) {
    const int cap = cta_cap();
    if (cap > 0 && grid > cap) grid = cap;
    return (int)std::max<int64_t>(1, grid);
}

namespace {
std::mutex g_mu;
std::map<int, int> g_sms;                                    // device -> SM count
std::map<std::tuple<int, const void*, int>, int> g_occ;      // (device, kernel, threads) -> blocks per SM
}  // namespace

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_sms.find(dev);
    if (it != g_sms.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    g_sms[dev] = n;
    return n;
}

bool cta_cap_is_tight() {
    const int cap = cta_cap();
    return cap > 0 && cap < 4 * sm_count();
}

// Grid of a grid-stride kernel: four waves of resident blocks (SMs x blocks
// per SM x 4), but no more blocks than the work needs.  Four waves measured
// 2-8 % faster than one on GB300 for the copy, accumulate, vector-ring and
// staged-hop kernels (8 x 128 MiB, CUDA events); launches that stream 128 MiB
// or more now run one block per tile instead (rows_grid_x and the launchers).
int grid_for(const void* kernel, int64_t work_items, int threads) {
    const int sms = sm_count();
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, kernel, threads);
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) per_sm = it->second;
    }
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess || per_sm <= 0)
            per_sm = 1;
        std::lock_guard<std::mutex> lk(g_mu);
        g_occ[key] = per_sm;
    }
    const int64_t need = std::max<int64_t>(1, (work_items + threads - 1) / threads);
    return cap_ctas(std::min<int64_t>((int64_t)sms * per_sm * 4, need));
}

int rows_grid_x(const void* kernel, int64_t per_row, int rows, int64_t bytes) {
    const int64_t tiles = (per_row + kThreads - 1) / kThreads;
    if (bytes >= ((int64_t)128 << 20) && tiles * rows <= INT32_MAX && cap_ctas(tiles * rows) == tiles * rows)
        return (int)std::max<int64_t>(1, tiles);
    const int g = bytes >= ((int64_t)128 << 20) ? cap_ctas(std::min<int64_t>(tiles * rows, INT32_MAX))
                                                 : grid_for(kernel, per_row * rows);
    return std::max(1, (g + rows - 1) / rows);
}

// Host buffers of a host-memory allreduce: non-null and element-aligned;
// inputs pairwise disjoint; each output either is its own rank's input (in
// place) or overlaps no input and no other output.
int32_t check_host_in_out(int32_t world, const void* const* host_in, void* const* host_out, int64_t numel,
                          int32_t dtype) {
    const uintptr_t es = (uintptr_t)elem_bytes(dtype);
    const uintptr_t bytes = (uintptr_t)numel * es;
    std::vector<std::pair<uintptr_t, uintptr_t>> iv;
    for (int32_t r = 0; r < world; ++r) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(host_in[r]), b = reinterpret_cast<uintptr_t>(host_out[r]);
        if (!a || !b) return DDP_ERR_INVALID;
        if (a % es || b % es) return DDP_ERR_ALIGN;
        iv.emplace_back(a, a + bytes);
        if (b != a) iv.emplace_back(b, b + bytes);
    }
    std::sort(iv.begin(), iv.end());
    for (size_t i = 1; i < iv.size(); ++i)
        if (iv[i].first < iv[i - 1].second) return DDP_ERR_INVALID;
    return DDP_OK;
}

int32_t common_checks(int32_t world, int64_t numel, int32_t dtype) {
    if (world < 1 || world > DDP_MAX_WORLD) return world < 1 ? DDP_ERR_INVALID : DDP_ERR_CAPACITY;
    if (numel < 0 || (dtype != DDP_F32 && dtype != DDP_BF16)) return DDP_ERR_INVALID;
    if (numel > DDP_MAX_NUMEL) return DDP_ERR_CAPACITY;
    return DDP_OK;
}

namespace {
thread_local const char* t_last_cuda_error = "no error";
}  // namespace

int32_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return DDP_OK;
    t_last_cuda_error = cudaGetErrorString(e);
    if (debug_enabled()) fprintf(stderr, "[ddp] CUDA error: %s\n", t_last_cuda_error);
    return DDP_ERR_CUDA;
}

const char* last_cuda_error() { return t_last_cuda_error; }

}  // namespace ddpk

using namespace ddpk;

namespace {

// Rank buffers: non-null, element-aligned, pairwise disjoint.  Sets *vec_ok
// when every buffer is 16-byte aligned.
int32_t check_rank_buffers(int32_t world, const void* const* bufs, int64_t numel, int32_t dtype, bool* vec_ok) {
    if (!bufs) return DDP_ERR_INVALID;
    const uintptr_t es = (uintptr_t)elem_bytes(dtype);
    bool v = true;
    std::vector<std::pair<uintptr_t, uintptr_t>> iv;
    iv.reserve(world);
    for (int32_t r = 0; r < world; ++r) {
        const uintptr_t p = reinterpret_cast<uintptr_t>(bufs[r]);
        if (!p) return DDP_ERR_INVALID;
        if (p % es) return DDP_ERR_ALIGN;
        if (p % 16) v = false;
        iv.emplace_back(p, p + (uintptr_t)numel * es);
    }
    std::sort(iv.begin(), iv.end());
    for (size_t i = 1; i < iv.size(); ++i)
        if (iv[i].first < iv[i - 1].second) return DDP_ERR_INVALID;
    *vec_ok = v;
    return DDP_OK;
}

using Span = std::pair<uintptr_t, uintptr_t>;      // [first, second) in bytes

// True if two of the spans share a byte (sorts `v`).
bool any_overlap(std::vector<Span>* v) {
    std::sort(v->begin(), v->end());
    for (size_t i = 1; i < v->size(); ++i)
        if ((*v)[i].first < (*v)[i - 1].second) return true;
    return false;
}

// True if [a, b) shares a byte with one of the sorted, pairwise disjoint spans.
bool hits_any(const std::vector<Span>& sorted, uintptr_t a, uintptr_t b) {
    auto it = std::lower_bound(sorted.begin(), sorted.end(), Span{b, 0});   // first span starting at or after b
    return it != sorted.begin() && std::prev(it)->second > a;
}

// The memory a pack or unpack touches: the ranks' buckets must be disjoint,
// no gradient may share a byte with any bucket, and gradients that are
// written (unpack) must be disjoint too.
int32_t check_pack_memory(int32_t world, int32_t n, const void* const* grads, const int64_t* numel,
                          int64_t grad_es, const void* const* buckets, int64_t bucket_bytes, bool grads_written) {
    std::vector<Span> bk, gs;
    for (int32_t r = 0; r < world && bucket_bytes > 0; ++r) {
        const uintptr_t b = reinterpret_cast<uintptr_t>(buckets[r]);
        bk.emplace_back(b, b + (uintptr_t)bucket_bytes);
    }
    if (any_overlap(&bk)) return DDP_ERR_INVALID;
    for (int32_t r = 0; r < world; ++r)
        for (int32_t i = 0; i < n; ++i) {
            if (numel[i] == 0) continue;
            const uintptr_t g = reinterpret_cast<uintptr_t>(grads[(int64_t)r * n + i]);
            const uintptr_t e = g + (uintptr_t)(numel[i] * grad_es);
            if (hits_any(bk, g, e)) return DDP_ERR_INVALID;
            gs.emplace_back(g, e);
        }
    if (grads_written && any_overlap(&gs)) return DDP_ERR_INVALID;
    return DDP_OK;
}

// Large host buckets: pieces of kHostPieceBytes per rank flow through three
// streams -- host-to-device copies, the reduction, device-to-host copies --
// so that piece p+1 comes in while piece p is reduced and piece p-1 goes
// out, and the CPU-GPU link carries both directions at once.  A piece is
// reduced by the view kernel as one member per rank at its bucket offset,
// so every element is still folded in the ring order of its chunk of the
// whole bucket.  The caller's stream waits for the last copy out.
constexpr int64_t kHostPieceBytes = (int64_t)32 << 20;

cudaError_t from_host_pipelined(int32_t world, const void* const* host_in, void* const* host_out,
                                void* const* dev_bufs, int64_t numel, int32_t dtype, int32_t divisor, bool vec,
                                int64_t piece, cudaStream_t caller) {
    struct Streams {
        cudaStream_t in = nullptr, red = nullptr, out = nullptr;
        std::vector<cudaEvent_t> ev;
        ~Streams() {                     // released once their queued work is done
            for (cudaEvent_t e : ev) cudaEventDestroy(e);
            if (in) cudaStreamDestroy(in);
            if (red) cudaStreamDestroy(red);
            if (out) cudaStreamDestroy(out);
        }
        cudaError_t event(cudaEvent_t* e) {
            cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
            if (r == cudaSuccess) ev.push_back(*e);
            return r;
        }
    } S;
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&S.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&S.red, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&S.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    cudaEvent_t start, done;
    if ((e = S.event(&start)) != cudaSuccess || (e = S.event(&done)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(start, caller)) != cudaSuccess) return e;
    for (cudaStream_t t : {S.in, S.red, S.out})
        if ((e = cudaStreamWaitEvent(t, start, 0)) != cudaSuccess) return e;
    const int64_t es = elem_bytes(dtype);
    const DivSpec div = make_div(divisor);
    std::vector<void*> ptrs(world);
    for (int64_t a = 0; a < numel; a += piece) {
        const int64_t len = std::min(piece, numel - a);
        const size_t nb = (size_t)(len * es);
        cudaEvent_t in_done, red_done;
        if ((e = S.event(&in_done)) != cudaSuccess || (e = S.event(&red_done)) != cudaSuccess) return e;
        for (int32_t r = 0; r < world; ++r) {
            char* d = static_cast<char*>(dev_bufs[r]) + a * es;
            const char* h = static_cast<const char*>(host_in[r]) + a * es;
            if ((e = cudaMemcpyAsync(d, h, nb, cudaMemcpyHostToDevice, S.in)) != cudaSuccess) return e;
        }
        if ((e = cudaEventRecord(in_done, S.in)) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(S.red, in_done, 0)) != cudaSuccess) return e;
        for (int32_t r = 0; r < world; ++r) ptrs[r] = static_cast<char*>(dev_bufs[r]) + a * es;
        ViewMember m{len, a, ptrs.data(), vec && (a * es) % 16 == 0};
        if ((e = launch_bucket_view(world, &m, 1, numel, dtype, div, S.red)) != cudaSuccess) return e;
        if ((e = cudaEventRecord(red_done, S.red)) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(S.out, red_done, 0)) != cudaSuccess) return e;
        for (int32_t r = 0; r < world; ++r) {
            char* h = static_cast<char*>(host_out[r]) + a * es;
            const char* d = static_cast<const char*>(dev_bufs[r]) + a * es;
            if ((e = cudaMemcpyAsync(h, d, nb, cudaMemcpyDeviceToHost, S.out)) != cudaSuccess) return e;
        }
    }
    if ((e = cudaEventRecord(done, S.out)) != cudaSuccess) return e;
    return cudaStreamWaitEvent(caller, done, 0);
}

// Check one bucket's member table and build the copy items of pack/unpack.
int32_t bucket_items(int32_t world, int32_t n, const void* const* grads, const int64_t* numel,
                     const int64_t* offset, const void* const* buckets, int64_t bucket_numel, int32_t dtype,
                     bool to_bucket, std::vector<CopyItem>* items) {
    int32_t st = common_checks(world, bucket_numel, dtype);     // also caps bucket_numel, so byte sizes fit
    if (st) return st;
    if (n < 0) return DDP_ERR_INVALID;
    if (n > 0 && (!grads || !numel || !offset || !buckets)) return DDP_ERR_INVALID;
    const int64_t es = elem_bytes(dtype);
    // members must lie inside the bucket and not overlap each other
    std::vector<std::pair<int64_t, int64_t>> ranges;
    ranges.reserve(n);
    for (int32_t i = 0; i < n; ++i) {
        if (numel[i] < 0 || offset[i] < 0 || offset[i] > bucket_numel - numel[i]) return DDP_ERR_INVALID;
        if (numel[i] > 0) ranges.emplace_back(offset[i], offset[i] + numel[i]);
    }
    std::sort(ranges.begin(), ranges.end());
    for (size_t i = 1; i < ranges.size(); ++i)
        if (ranges[i].first < ranges[i - 1].second) return DDP_ERR_INVALID;
    items->clear();
    items->reserve((size_t)world * n);
    for (int32_t r = 0; r < world; ++r) {
        char* b = static_cast<char*>(const_cast<void*>(buckets[r]));
        if (!b && bucket_numel > 0) return DDP_ERR_INVALID;
        if (reinterpret_cast<uintptr_t>(b) % es) return DDP_ERR_ALIGN;
        for (int32_t i = 0; i < n; ++i) {
            if (numel[i] == 0) continue;
            char* g = static_cast<char*>(const_cast<void*>(grads[(int64_t)r * n + i]));
            if (!g) return DDP_ERR_INVALID;
            if (reinterpret_cast<uintptr_t>(g) % es) return DDP_ERR_ALIGN;
            char* slot = b + offset[i] * es;
            const int64_t bytes = numel[i] * es;
            if (to_bucket) items->push_back(CopyItem{g, slot, bytes});
            else items->push_back(CopyItem{slot, g, bytes});
        }
    }
    return check_pack_memory(world, n, grads, numel, es, buckets, bucket_numel * es, !to_bucket);
}

// Members of one bucket for the bf16 hook: float32 gradients, bf16 bucket.
int32_t hook_items(int32_t world, int32_t n, const void* const* grads, const int64_t* numel, const int64_t* offset,
                   const void* const* buckets, int64_t bucket_numel, bool to_bucket, std::vector<ConvItem>* items) {
    int32_t st = common_checks(world, bucket_numel, DDP_F32);   // also caps bucket_numel, so byte sizes fit
    if (st) return st;
    if (n < 0) return DDP_ERR_INVALID;
    if (n > 0 && (!grads || !numel || !offset || !buckets)) return DDP_ERR_INVALID;
    std::vector<std::pair<int64_t, int64_t>> ranges;
    for (int32_t i = 0; i < n; ++i) {
        if (numel[i] < 0 || offset[i] < 0 || offset[i] > bucket_numel - numel[i]) return DDP_ERR_INVALID;
        if (numel[i] > 0) ranges.emplace_back(offset[i], offset[i] + numel[i]);
    }
    std::sort(ranges.begin(), ranges.end());
    for (size_t i = 1; i < ranges.size(); ++i)
        if (ranges[i].first < ranges[i - 1].second) return DDP_ERR_INVALID;
    items->clear();
    for (int32_t r = 0; r < world; ++r) {
        char* b = static_cast<char*>(const_cast<void*>(buckets[r]));
        if (!b && bucket_numel > 0) return DDP_ERR_INVALID;
        if (reinterpret_cast<uintptr_t>(b) % 2) return DDP_ERR_ALIGN;
        for (int32_t i = 0; i < n; ++i) {
            if (numel[i] == 0) continue;
            char* g = static_cast<char*>(const_cast<void*>(grads[(int64_t)r * n + i]));
            if (!g) return DDP_ERR_INVALID;
            if (reinterpret_cast<uintptr_t>(g) % 4) return DDP_ERR_ALIGN;
            char* slot = b + offset[i] * 2;
            if (to_bucket) items->push_back(ConvItem{g, slot, numel[i]});
            else items->push_back(ConvItem{slot, g, numel[i]});
        }
    }
    return check_pack_memory(world, n, grads, numel, 4, buckets, bucket_numel * 2, !to_bucket);
}

int32_t view_members(int32_t world, int32_t n, void* const* grads, const int64_t* numel, const int64_t* offset,
                     int64_t bucket_numel, int32_t dtype, std::vector<ViewMember>* out) {
    int32_t st = common_checks(world, bucket_numel, dtype);
    if (st) return st;
    if (n < 0) return DDP_ERR_INVALID;
    if (n > 0 && (!grads || !numel || !offset)) return DDP_ERR_INVALID;
    const int64_t es = elem_bytes(dtype);
    std::vector<std::pair<int64_t, int64_t>> ranges;
    for (int32_t i = 0; i < n; ++i) {
        if (numel[i] < 0 || offset[i] < 0 || offset[i] > bucket_numel - numel[i]) return DDP_ERR_INVALID;
        if (numel[i] > 0) ranges.emplace_back(offset[i], offset[i] + numel[i]);
    }
    std::sort(ranges.begin(), ranges.end());
    for (size_t i = 1; i < ranges.size(); ++i)
        if (ranges[i].first < ranges[i - 1].second) return DDP_ERR_INVALID;
    // every (rank, member) gradient must be distinct memory
    std::vector<std::pair<uintptr_t, uintptr_t>> iv;
    out->clear();
    for (int32_t i = 0; i < n; ++i) {
        if (numel[i] == 0) continue;
        bool v = true;
        for (int32_t r = 0; r < world; ++r) {
            const uintptr_t p = reinterpret_cast<uintptr_t>(grads[(int64_t)r * n + i]);
            if (!p) return DDP_ERR_INVALID;
            if (p % (uintptr_t)es) return DDP_ERR_ALIGN;
            if (p % 16) v = false;
            iv.emplace_back(p, p + (uintptr_t)(numel[i] * es));
        }
        out->push_back(ViewMember{numel[i], offset[i], nullptr, v});   // ptrs set by the caller
    }
    std::sort(iv.begin(), iv.end());
    for (size_t i = 1; i < iv.size(); ++i)
        if (iv[i].first < iv[i - 1].second) return DDP_ERR_INVALID;
    return DDP_OK;
}

}  // namespace

namespace {

// One bucket of the unfused pipeline (pack -> fused ring -> unpack) run in
// pieces that fit in L2: for each piece [a, b) of the bucket, the members'
// parts that fall in it are packed, the piece is reduced by the view kernel
// with its bucket offset (so every element is folded in the ring order of its
// chunk of the whole bucket -- the same bits as the ring over the whole
// bucket), and unpacked, before the next piece is packed.  The ring and the
// unpack then read the piece from L2 instead of HBM.  Arguments are checked by
// the caller.  Buckets no larger than one and a half pieces run whole.
constexpr int64_t kPieceBytesAllRanks = (int64_t)96 << 20;   // bucket bytes over all ranks per piece

int64_t bucket_piece_elems(int32_t world, int32_t dtype) {
    const int64_t es = elem_bytes(dtype);
    int64_t piece = kPieceBytesAllRanks / world / es;
    piece = piece / 1024 * 1024;                                 // pieces start 16-byte aligned
    return std::max<int64_t>(piece, 64 * 1024);
}

cudaError_t sync_bucket_pieces(int32_t world, int32_t n, const void* const* g, const int64_t* ne, const int64_t* off,
                               void* const* bk, int64_t bucket_numel, int32_t dtype, int32_t divisor, bool vec,
                               cudaStream_t s) {
    const int64_t es = elem_bytes(dtype);
    const int64_t piece = bucket_piece_elems(world, dtype);
    const DivSpec div = make_div(divisor);
    std::vector<CopyItem> in, out;
    std::vector<void*> ptrs(world);
    for (int64_t a = 0; a < bucket_numel; a += piece) {
        const int64_t b = std::min(bucket_numel, a + piece);
        in.clear();
        out.clear();
        for (int32_t r = 0; r < world; ++r)
            for (int32_t i = 0; i < n; ++i) {
                const int64_t s0 = std::max(off[i], a), s1 = std::min(off[i] + ne[i], b);
                if (s1 <= s0) continue;
                const char* gp = static_cast<const char*>(g[(int64_t)r * n + i]) + (s0 - off[i]) * es;
                char* bp = static_cast<char*>(bk[r]) + s0 * es;
                in.push_back(CopyItem{gp, bp, (s1 - s0) * es});
                out.push_back(CopyItem{bp, const_cast<char*>(gp), (s1 - s0) * es});
            }
        cudaError_t e = launch_copy_items(in.data(), (int64_t)in.size(), s);
        if (e != cudaSuccess) return e;
        for (int32_t r = 0; r < world; ++r) ptrs[r] = static_cast<char*>(bk[r]) + a * es;
        ViewMember m{b - a, a, ptrs.data(), vec};
        if ((e = launch_bucket_view(world, &m, 1, bucket_numel, dtype, div, s)) != cudaSuccess) return e;
        if ((e = launch_copy_items(out.data(), (int64_t)out.size(), s)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// The bf16 compression hook's three passes over one bucket, in the same
// L2-sized pieces: for each piece the members' parts are rounded into the
// bf16 bucket, the piece is reduced in bf16 by the view kernel at its bucket
// offset (each element folded in the ring order of its chunk of the whole
// bucket, one bf16 rounding per hop), and widened back into the gradients --
// the bits of the whole-bucket pack, ring and unpack.  Arguments are checked
// by the caller.
cudaError_t hook_bucket_pieces(int32_t world, int32_t n, const void* const* g, const int64_t* ne, const int64_t* off,
                               void* const* bk, int64_t bucket_numel, int32_t divisor, bool vec, cudaStream_t s) {
    const int64_t piece = bucket_piece_elems(world, DDP_BF16);
    const DivSpec div = make_div(divisor);
    std::vector<ConvItem> in, out;
    std::vector<void*> ptrs(world);
    for (int64_t a = 0; a < bucket_numel; a += piece) {
        const int64_t b = std::min(bucket_numel, a + piece);
        in.clear();
        out.clear();
        for (int32_t r = 0; r < world; ++r)
            for (int32_t i = 0; i < n; ++i) {
                const int64_t s0 = std::max(off[i], a), s1 = std::min(off[i] + ne[i], b);
                if (s1 <= s0) continue;
                const char* gp = static_cast<const char*>(g[(int64_t)r * n + i]) + (s0 - off[i]) * 4;
                char* bp = static_cast<char*>(bk[r]) + s0 * 2;
                in.push_back(ConvItem{gp, bp, s1 - s0});
                out.push_back(ConvItem{bp, const_cast<char*>(gp), s1 - s0});
            }
        cudaError_t e = launch_convert_items(in.data(), (int64_t)in.size(), 1, s);
        if (e != cudaSuccess) return e;
        for (int32_t r = 0; r < world; ++r) ptrs[r] = static_cast<char*>(bk[r]) + a * 2;
        ViewMember m{b - a, a, ptrs.data(), vec};
        if ((e = launch_bucket_view(world, &m, 1, bucket_numel, DDP_BF16, div, s)) != cudaSuccess) return e;
        if ((e = launch_convert_items(out.data(), (int64_t)out.size(), 0, s)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

namespace ddpk {

// ddp_sync_buckets' and the reducer's bf16-hook path for one bucket:
// validated, then whole or in L2-sized pieces.
int32_t hook_pack_ring_unpack(int32_t world, int32_t n, const void* const* g, const int64_t* ne, const int64_t* off,
                              void* const* bk, int64_t bucket_numel, int32_t divisor, void* stream) {
    std::vector<ConvItem> items, back;
    int32_t st = hook_items(world, n, g, ne, off, (const void* const*)bk, bucket_numel, true, &items);
    if (st) return st;
    // the unpack writes the gradients: they must not overlap each other either
    if ((st = hook_items(world, n, g, ne, off, (const void* const*)bk, bucket_numel, false, &back))) return st;
    if (divisor < 0) return DDP_ERR_INVALID;
    if (bucket_numel == 0) return DDP_OK;
    bool vec = false;
    if ((st = check_rank_buffers(world, bk, bucket_numel, DDP_BF16, &vec))) return st;
    const int64_t piece = bucket_piece_elems(world, DDP_BF16);
    if (bucket_numel <= piece + piece / 2) {
        if ((st = cuda_status(launch_convert_items(items.data(), (int64_t)items.size(), 1, (cudaStream_t)stream))))
            return st;
        if ((st = ring_allreduce_fused(world, bk, bucket_numel, DDP_BF16, divisor, stream))) return st;
        return ddp_bucket_unpack_bf16(world, n, const_cast<void* const*>(g), ne, off, (const void* const*)bk,
                                      bucket_numel, stream);
    }
    return cuda_status(hook_bucket_pieces(world, n, g, ne, off, bk, bucket_numel, divisor, vec, (cudaStream_t)stream));
}

// ddp_sync_buckets' and the reducer's unfused fused-ring path for one bucket:
// validated, then whole or in pieces.
int32_t pack_ring_unpack(int32_t world, int32_t n, const void* const* g, const int64_t* ne, const int64_t* off,
                         void* const* bk, int64_t bucket_numel, int32_t dtype, int32_t divisor, void* stream) {
    std::vector<CopyItem> items, back;
    int32_t st = bucket_items(world, n, g, ne, off, (const void* const*)bk, bucket_numel, dtype, true, &items);
    if (st) return st;
    // the unpack writes the gradients: they must not overlap each other either
    if ((st = bucket_items(world, n, g, ne, off, (const void* const*)bk, bucket_numel, dtype, false, &back)))
        return st;
    if (divisor < 0) return DDP_ERR_INVALID;
    if (bucket_numel == 0) return DDP_OK;
    bool vec = false;
    if ((st = check_rank_buffers(world, bk, bucket_numel, dtype, &vec))) return st;
    const int64_t piece = bucket_piece_elems(world, dtype);
    if (bucket_numel <= piece + piece / 2) {
        if ((st = cuda_status(launch_copy_items(items.data(), (int64_t)items.size(), (cudaStream_t)stream))))
            return st;
        if ((st = ring_allreduce_fused(world, bk, bucket_numel, dtype, divisor, stream))) return st;
        return ddp_bucket_unpack(world, n, const_cast<void* const*>(g), ne, off, (const void* const*)bk, bucket_numel,
                                 dtype, stream);
    }
    return cuda_status(
        sync_bucket_pieces(world, n, g, ne, off, bk, bucket_numel, dtype, divisor, vec, (cudaStream_t)stream));
}

}  // namespace ddpk

extern "C" {

const char* ddp_status_string(int32_t status) {
    DDP_TRACE_CALL();
    switch (status) {
        case DDP_OK: return "DDP_OK";
        case DDP_ERR_INVALID: return "DDP_ERR_INVALID: invalid argument";
        case DDP_ERR_ALIGN: return "DDP_ERR_ALIGN: pointer not aligned to its element size";
        case DDP_ERR_CUDA: return "DDP_ERR_CUDA: a CUDA call or kernel launch failed";
        case DDP_ERR_TIMEOUT: return "DDP_ERR_TIMEOUT: a bounded device-side wait gave up";
        case DDP_ERR_CAPACITY: return "DDP_ERR_CAPACITY: size beyond a documented limit";
        case DDP_ERR_HOST: return "DDP_ERR_HOST: host memory allocation failed inside the library";
        default: return "unknown ddp_status";
    }
}

int32_t ddp_abi_version(void) { return DDP_ABI_VERSION; }

const char* ddp_last_cuda_error(void) { return last_cuda_error(); }

int32_t ddp_set_max_ctas(int32_t max_ctas, int32_t* previous) try {
    DDP_TRACE_CALL();
    if (max_ctas < 0) return DDP_ERR_INVALID;
    const int prev = g_max_ctas.exchange(max_ctas);
    if (previous) *previous = prev;
    return DDP_OK;
} DDP_ABI_CATCH

int32_t ddp_set_fused_kernel(int32_t kind, int32_t* previous) try {
    DDP_TRACE_CALL();
    if (kind < DDP_FUSED_AUTO || kind > DDP_FUSED_TMA) return DDP_ERR_INVALID;
    const int prev = g_fused_kernel.exchange(kind);
    if (previous) *previous = prev;
    return DDP_OK;
} DDP_ABI_CATCH

int32_t ddp_set_wait_limit_ms(int32_t limit_ms, int32_t* previous_ms) try {
    DDP_TRACE_CALL();
    if (limit_ms < 0 || limit_ms > 600000) return DDP_ERR_INVALID;
    const unsigned long long ns = (unsigned long long)(limit_ms ? limit_ms : 2000) * 1000000ull;
    unsigned long long prev = 0;
    set_wait_limit_ns(ns, &prev);
    if (previous_ms) *previous_ms = (int32_t)(prev / 1000000ull);
    return DDP_OK;
} DDP_ABI_CATCH

int32_t ddp_plant_stall(int64_t tile) try {
    DDP_TRACE_CALL();
    if (tile < -1) return DDP_ERR_INVALID;
    plant_stall((long long)tile);
    return DDP_OK;
} DDP_ABI_CATCH

int32_t ddp_device_status(int32_t* status, int32_t clear) try {
    DDP_TRACE_CALL();
    if (!status) return DDP_ERR_INVALID;
    return cuda_status(read_device_status(status, clear != 0));
} DDP_ABI_CATCH

int32_t ring_allreduce_fused(int32_t world, void* const* bufs, int64_t numel, int32_t dtype, int32_t divisor,
                             void* stream) try {
    DDP_TRACE_CALL();
    int32_t st = common_checks(world, numel, dtype);
    if (st) return st;
    if (divisor < 0) return DDP_ERR_INVALID;
    if (numel == 0) return DDP_OK;
    bool vec = false;
    if ((st = check_rank_buffers(world, bufs, numel, dtype, &vec))) return st;
    return cuda_status(launch_ring_fused(world, bufs, numel, dtype, make_div(divisor), vec, (cudaStream_t)stream));
} DDP_ABI_CATCH

int32_t ring_allreduce_staged(int32_t world, void* const* bufs, int64_t numel, int32_t dtype, int32_t divisor,
                              void* stream) try {
    DDP_TRACE_CALL();
    int32_t st = common_checks(world, numel, dtype);
    if (st) return st;
    if (divisor < 0) return DDP_ERR_INVALID;
    if (numel == 0) return DDP_OK;
    bool vec = false;
    if ((st = check_rank_buffers(world, bufs, numel, dtype, &vec))) return st;
    return cuda_status(launch_ring_staged(world, bufs, numel, dtype, make_div(divisor), vec, (cudaStream_t)stream));
} DDP_ABI_CATCH

static int32_t tree_common(bool staged, int32_t world, void* const* bufs, int64_t numel, int32_t dtype,
                           int32_t divisor, void* stream) {
    int32_t st = common_checks(world, numel, dtype);
    if (st) return st;
    if (!staged && world > 64) return DDP_ERR_CAPACITY;
    if (divisor < 0) return DDP_ERR_INVALID;
    if (numel == 0) return DDP_OK;
    bool vec = false;
    if ((st = check_rank_buffers(world, bufs, numel, dtype, &vec))) return st;
    return cuda_status(launch_tree_allreduce(staged, world, bufs, numel, dtype, make_div(divisor), vec,
                                             (cudaStream_t)stream));
}

int32_t tree_allreduce_fused(int32_t world, void* const* bufs, int64_t numel, int32_t dtype, int32_t divisor,
                             void* stream) try {
    DDP_TRACE_CALL();
    return tree_common(false, world, bufs, numel, dtype, divisor, stream);
} DDP_ABI_CATCH

int32_t tree_allreduce_staged(int32_t world, void* const* bufs, int64_t numel, int32_t dtype, int32_t divisor,
                              void* stream) try {
    DDP_TRACE_CALL();
    return tree_common(true, world, bufs, numel, dtype, divisor, stream);
} DDP_ABI_CATCH

int32_t ring_allreduce_persistent(int32_t world, void* const* bufs, int64_t numel, int32_t dtype, int32_t divisor,
                                  int32_t* dev_status, int32_t fail_at_step, int32_t wait_limit_ms, void* stream) try {
    DDP_TRACE_CALL();
    int32_t st = common_checks(world, numel, dtype);
    if (st) return st;
    if (divisor < 0 || !dev_status || wait_limit_ms < 0) return DDP_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(dev_status) % 8) return DDP_ERR_ALIGN;
    if (fail_at_step < -1 || (fail_at_step >= 0 && fail_at_step > 2 * (world - 1) - 2)) return DDP_ERR_INVALID;
    cudaStream_t s = (cudaStream_t)stream;
    bool vec = false;
    if (numel > 0 && (st = check_rank_buffers(world, bufs, numel, dtype, &vec))) return st;
    if (numel == 0 || world == 1) {
        // no ring step to wait on: clear the status word, and for one rank divide
        cudaError_t e = cudaMemsetAsync(dev_status, 0, 2 * sizeof(int32_t), s);
        if (e != cudaSuccess) return cuda_status(e);
        if (numel == 0) return DDP_OK;
        return cuda_status(launch_ring_fused(world, bufs, numel, dtype, make_div(divisor), vec, s));
    }
    const unsigned long long limit = (unsigned long long)(wait_limit_ms ? wait_limit_ms : 2000) * 1000000ull;
    return cuda_status(launch_ring_persistent(world, bufs, numel, dtype, make_div(divisor), vec, dev_status,
                                              fail_at_step, limit, s));
} DDP_ABI_CATCH

int32_t ring_allreduce_fused_from_host(int32_t world, const void* const* host_in, void* const* host_out,
                                       void* const* dev_bufs, int64_t numel, int32_t dtype, int32_t divisor,
                                       void* stream) try {
    DDP_TRACE_CALL();
    int32_t st = common_checks(world, numel, dtype);
    if (st) return st;
    if (divisor < 0 || !host_in || !host_out) return DDP_ERR_INVALID;
    if (numel == 0) return DDP_OK;
    bool vec = false;
    if ((st = check_rank_buffers(world, dev_bufs, numel, dtype, &vec))) return st;
    if ((st = check_host_in_out(world, host_in, host_out, numel, dtype))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t es = elem_bytes(dtype);
    const size_t bytes = (size_t)numel * es;
    const int64_t piece = kHostPieceBytes / es;                 // elements per rank and piece
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &capturing) != cudaSuccess) return cuda_status(cudaGetLastError());
    if (numel <= 2 * piece || capturing != cudaStreamCaptureStatusNone) {
        // small, or being captured into a graph: in, reduce, out on the caller's stream
        for (int32_t r = 0; r < world; ++r) {
            cudaError_t e = cudaMemcpyAsync(dev_bufs[r], host_in[r], bytes, cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess) return cuda_status(e);
        }
        if ((st = cuda_status(launch_ring_fused(world, dev_bufs, numel, dtype, make_div(divisor), vec, s))))
            return st;
        for (int32_t r = 0; r < world; ++r) {
            cudaError_t e = cudaMemcpyAsync(host_out[r], dev_bufs[r], bytes, cudaMemcpyDeviceToHost, s);
            if (e != cudaSuccess) return cuda_status(e);
        }
        return DDP_OK;
    }
    return cuda_status(from_host_pipelined(world, host_in, host_out, dev_bufs, numel, dtype, divisor, vec, piece, s));
} DDP_ABI_CATCH

// Device address through which the GPU reaches host buffer p, or nullptr
// if it cannot reach it: pinned (page-locked, mapped) memory, managed or
// device memory, and plain pageable memory on systems where the GPU reads
// pageable memory through the host page tables (coherent CPU-GPU nodes).
static void* device_view_of(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return const_cast<void*>(p);
    int dev = 0, pageable = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess) return nullptr;
    return pageable ? const_cast<void*>(p) : nullptr;
}

int32_t ring_allreduce_fused_host_direct(int32_t world, const void* const* host_in, void* const* host_out,
                                         int64_t numel, int32_t dtype, int32_t divisor, void* stream) try {
    DDP_TRACE_CALL();
    int32_t st = common_checks(world, numel, dtype);
    if (st) return st;
    if (divisor < 0 || !host_in || !host_out) return DDP_ERR_INVALID;
    if (numel == 0) return DDP_OK;
    if ((st = ddpk::check_host_in_out(world, host_in, host_out, numel, dtype))) return st;
    std::vector<void*> din(world), dout(world);
    bool vec = true;
    for (int32_t r = 0; r < world; ++r) {
        din[r] = device_view_of(host_in[r]);
        dout[r] = (host_out[r] == host_in[r]) ? din[r] : device_view_of(host_out[r]);
        if (!din[r] || !dout[r]) return DDP_ERR_INVALID;
        if (reinterpret_cast<uintptr_t>(din[r]) % 16 || reinterpret_cast<uintptr_t>(dout[r]) % 16) vec = false;
    }
    return cuda_status(launch_ring_fused_io(world, din.data(), dout.data(), numel, dtype, make_div(divisor), vec,
                                            (cudaStream_t)stream));
} DDP_ABI_CATCH

int32_t ddp_grad_accumulate(int32_t world, void* const* acc, const void* const* grads, int64_t numel,
                            int32_t dtype, void* stream) try {
    DDP_TRACE_CALL();
    int32_t st = common_checks(world, numel, dtype);
    if (st) return st;
    if (numel == 0) return DDP_OK;
    bool va = false, vg = false;
    if ((st = check_rank_buffers(world, acc, numel, dtype, &va))) return st;
    if ((st = check_rank_buffers(world, grads, numel, dtype, &vg))) return st;
    return cuda_status(launch_accumulate(world, acc, grads, numel, dtype, va && vg, (cudaStream_t)stream));
} DDP_ABI_CATCH

int32_t ddp_bucket_pack(int32_t world, int32_t n_in_bucket, const void* const* grads, const int64_t* numel,
                        const int64_t* offset, void* const* buckets, int64_t bucket_numel, int32_t dtype,
                        void* stream) try {
    DDP_TRACE_CALL();
    std::vector<CopyItem> items;
    int32_t st = bucket_items(world, n_in_bucket, grads, numel, offset, (const void* const*)buckets, bucket_numel,
                              dtype, true, &items);
    if (st) return st;
    return cuda_status(launch_copy_items(items.data(), (int64_t)items.size(), (cudaStream_t)stream));
} DDP_ABI_CATCH

int32_t ddp_bucket_unpack(int32_t world, int32_t n_in_bucket, void* const* grads, const int64_t* numel,
                          const int64_t* offset, const void* const* buckets, int64_t bucket_numel, int32_t dtype,
                          void* stream) try {
    DDP_TRACE_CALL();
    std::vector<CopyItem> items;
    int32_t st = bucket_items(world, n_in_bucket, (const void* const*)grads, numel, offset, buckets, bucket_numel,
                              dtype, false, &items);
    if (st) return st;
    return cuda_status(launch_copy_items(items.data(), (int64_t)items.size(), (cudaStream_t)stream));
} DDP_ABI_CATCH

int32_t ddp_bucket_pack_bf16(int32_t world, int32_t n_in_bucket, const void* const* grads, const int64_t* numel,
                             const int64_t* offset, void* const* buckets, int64_t bucket_numel, void* stream) try {
    DDP_TRACE_CALL();
    std::vector<ConvItem> items;
    int32_t st = hook_items(world, n_in_bucket, grads, numel, offset, (const void* const*)buckets, bucket_numel, true,
                            &items);
    if (st) return st;
    return cuda_status(launch_convert_items(items.data(), (int64_t)items.size(), 1, (cudaStream_t)stream));
} DDP_ABI_CATCH

int32_t ddp_bucket_unpack_bf16(int32_t world, int32_t n_in_bucket, void* const* grads, const int64_t* numel,
                               const int64_t* offset, const void* const* buckets, int64_t bucket_numel, void* stream) try {
    DDP_TRACE_CALL();
    std::vector<ConvItem> items;
    int32_t st = hook_items(world, n_in_bucket, (const void* const*)grads, numel, offset, buckets, bucket_numel, false,
                            &items);
    if (st) return st;
    return cuda_status(launch_convert_items(items.data(), (int64_t)items.size(), 0, (cudaStream_t)stream));
} DDP_ABI_CATCH

static int32_t view_one(int32_t world, int32_t n_in_bucket, void* const* grads, const int64_t* numel,
                        const int64_t* offset, int64_t bucket_numel, int32_t dtype, int32_t launch_dtype,
                        int32_t divisor, void* stream) {
    if (divisor < 0) return DDP_ERR_INVALID;
    std::vector<ViewMember> members;
    int32_t st = view_members(world, n_in_bucket, grads, numel, offset, bucket_numel, dtype, &members);
    if (st) return st;
    // per-member rank pointer tables (rank order)
    std::vector<std::vector<void*>> tables;
    tables.reserve(members.size());
    size_t k = 0;
    for (int32_t i = 0; i < n_in_bucket; ++i) {
        if (numel[i] == 0) continue;
        tables.emplace_back(world);
        for (int32_t r = 0; r < world; ++r) tables.back()[r] = grads[(int64_t)r * n_in_bucket + i];
        members[k++].ptrs = tables.back().data();
    }
    return cuda_status(launch_bucket_view(world, members.data(), (int)members.size(), bucket_numel, launch_dtype,
                                          make_div(divisor), (cudaStream_t)stream));
}

int32_t ddp_bucket_allreduce_view(int32_t world, int32_t n_in_bucket, void* const* grads, const int64_t* numel,
                                  const int64_t* offset, int64_t bucket_numel, int32_t dtype, int32_t divisor,
                                  void* stream) try {
    DDP_TRACE_CALL();
    return view_one(world, n_in_bucket, grads, numel, offset, bucket_numel, dtype, dtype, divisor, stream);
} DDP_ABI_CATCH

int32_t ddp_bucket_allreduce_view_bf16(int32_t world, int32_t n_in_bucket, void* const* grads, const int64_t* numel,
                                       const int64_t* offset, int64_t bucket_numel, int32_t divisor, void* stream) try {
    DDP_TRACE_CALL();
    return view_one(world, n_in_bucket, grads, numel, offset, bucket_numel, DDP_F32, kDtypeHook, divisor, stream);
} DDP_ABI_CATCH

int32_t ddp_bucket_allreduce_view_fp16(int32_t world, int32_t n_in_bucket, void* const* grads, const int64_t* numel,
                                       const int64_t* offset, int64_t bucket_numel, int32_t divisor, void* stream) try {
    DDP_TRACE_CALL();
    return view_one(world, n_in_bucket, grads, numel, offset, bucket_numel, DDP_F32, kDtypeHook16, divisor, stream);
} DDP_ABI_CATCH

int32_t ddp_sync_buckets(int32_t world, int32_t n_params, void* const* grads, const int64_t* numel,
                         const int32_t* bucket_of_param, const int64_t* offset_of_param, int32_t n_buckets,
                         const int64_t* bucket_numel, void* const* buckets, int32_t dtype, int32_t divisor,
                         int32_t algo, void* stream) try {
    DDP_TRACE_CALL();
    int32_t st = common_checks(world, 0, dtype);
    if (st) return st;
    if (n_params < 0 || n_buckets < 0 || divisor < 0) return DDP_ERR_INVALID;
    if (algo != DDP_ALGO_FUSED && algo != DDP_ALGO_STAGED && algo != DDP_ALGO_VIEW && algo != DDP_ALGO_BF16_HOOK &&
        algo != DDP_ALGO_BF16_HOOK_VIEW && algo != DDP_ALGO_FP16_HOOK_VIEW)
        return DDP_ERR_INVALID;
    if ((algo == DDP_ALGO_BF16_HOOK || algo == DDP_ALGO_BF16_HOOK_VIEW || algo == DDP_ALGO_FP16_HOOK_VIEW) &&
        dtype != DDP_F32)
        return DDP_ERR_INVALID;
    const bool view = algo == DDP_ALGO_VIEW || algo == DDP_ALGO_BF16_HOOK_VIEW || algo == DDP_ALGO_FP16_HOOK_VIEW;
    if (n_params > 0 && (!grads || !numel || !bucket_of_param || !offset_of_param)) return DDP_ERR_INVALID;
    if (n_buckets > 0 && !bucket_numel) return DDP_ERR_INVALID;
    if (!view && n_buckets > 0 && !buckets) return DDP_ERR_INVALID;
    // members of each bucket, in bucket order
    std::vector<std::vector<int32_t>> members(n_buckets);
    for (int32_t p = 0; p < n_params; ++p) {
        const int32_t k = bucket_of_param[p];
        if (k < 0 || k >= n_buckets) return DDP_ERR_INVALID;
        members[k].push_back(p);
    }
    if (view) {
        // validate every bucket, then sync all of them together
        std::vector<ViewMember> all;
        std::vector<std::vector<void*>> tables;
        std::vector<int> first(n_buckets), count(n_buckets);
        tables.reserve(n_params);
        for (int32_t k = 0; k < n_buckets; ++k) {
            auto& m = members[k];
            std::sort(m.begin(), m.end(),
                      [&](int32_t a, int32_t b) { return offset_of_param[a] < offset_of_param[b]; });
            const int32_t n = (int32_t)m.size();
            std::vector<void*> g((size_t)world * n);
            std::vector<int64_t> ne(n), off(n);
            for (int32_t i = 0; i < n; ++i) {
                ne[i] = numel[m[i]];
                off[i] = offset_of_param[m[i]];
                for (int32_t r = 0; r < world; ++r) g[(size_t)r * n + i] = grads[(size_t)r * n_params + m[i]];
            }
            std::vector<ViewMember> vm;
            st = view_members(world, n, g.data(), ne.data(), off.data(), bucket_numel[k], dtype, &vm);
            if (st) return st;
            first[k] = (int)all.size();
            size_t q = 0;
            for (int32_t i = 0; i < n; ++i) {
                if (ne[i] == 0) continue;
                tables.emplace_back(world);
                for (int32_t r = 0; r < world; ++r) tables.back()[r] = g[(size_t)r * n + i];
                vm[q].ptrs = tables.back().data();
                all.push_back(vm[q++]);
            }
            count[k] = (int)all.size() - first[k];
        }
        const int32_t launch_dtype = (algo == DDP_ALGO_BF16_HOOK_VIEW)   ? kDtypeHook
                                     : (algo == DDP_ALGO_FP16_HOOK_VIEW) ? kDtypeHook16
                                                                         : dtype;
        return cuda_status(launch_buckets_view(world, all.data(), first.data(), count.data(), bucket_numel, n_buckets,
                                               launch_dtype, make_div(divisor), (cudaStream_t)stream));
    }
    std::vector<const void*> g;
    std::vector<int64_t> ne, off;
    std::vector<void*> bk(world);
    for (int32_t k = 0; k < n_buckets; ++k) {
        auto& m = members[k];
        std::sort(m.begin(), m.end(), [&](int32_t a, int32_t b) { return offset_of_param[a] < offset_of_param[b]; });
        const int32_t n = (int32_t)m.size();
        g.assign((size_t)world * n, nullptr);
        ne.resize(n);
        off.resize(n);
        for (int32_t i = 0; i < n; ++i) {
            ne[i] = numel[m[i]];
            off[i] = offset_of_param[m[i]];
            for (int32_t r = 0; r < world; ++r) g[(size_t)r * n + i] = grads[(size_t)r * n_params + m[i]];
        }
        for (int32_t r = 0; r < world; ++r) bk[r] = buckets[(size_t)r * n_buckets + k];
        if (algo == DDP_ALGO_BF16_HOOK) {
            st = hook_pack_ring_unpack(world, n, g.data(), ne.data(), off.data(), bk.data(), bucket_numel[k], divisor,
                                       stream);
            if (st) return st;
            continue;
        }
        if (algo == DDP_ALGO_FUSED) {
            st = pack_ring_unpack(world, n, g.data(), ne.data(), off.data(), bk.data(), bucket_numel[k], dtype, divisor,
                                  stream);
            if (st) return st;
        } else {
            st = ddp_bucket_pack(world, n, g.data(), ne.data(), off.data(), bk.data(), bucket_numel[k], dtype, stream);
            if (st) return st;
            st = ring_allreduce_staged(world, bk.data(), bucket_numel[k], dtype, divisor, stream);
            if (st) return st;
            st = ddp_bucket_unpack(world, n, const_cast<void* const*>(g.data()), ne.data(), off.data(),
                                   (const void* const*)bk.data(), bucket_numel[k], dtype, stream);
            if (st) return st;
        }
        if (debug_enabled())
            fprintf(stderr, "[ddp] bucket %d: %d members, %lld elements\n", k, n, (long long)bucket_numel[k]);
    }
    return DDP_OK;
} DDP_ABI_CATCH

}  // extern "C"
