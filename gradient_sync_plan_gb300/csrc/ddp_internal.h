// ddp_internal.h -- declarations shared by the library's translation units.
// Not part of the C ABI (see include/ddp.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ddp.h"

namespace ddpk {

constexpr int kThreads = 256;            // threads per block of every kernel
constexpr size_t kMaxParamBytes = 32764;  // kernel parameter space per launch (CUDA 12.1+)

// Divide modes of the average y / divisor:
//   kDivNone  divisor 0 or 1, keep the sum
//   kDivPow2  divisor = 2^k: multiply by the exact reciprocal 2^-k, which is
//             the same correctly rounded value as an IEEE division
//   kDivIeee  any other divisor: one IEEE division (round to nearest even)
enum DivMode { kDivNone = 0, kDivPow2 = 1, kDivIeee = 2 };

struct DivSpec {
    int mode;
    float operand;   // 2^-k for kDivPow2, (float)divisor for kDivIeee
};
DivSpec make_div(int32_t divisor);

// Internal element type of the fused bf16 hook: float32 storage, bf16 arithmetic.
constexpr int kDtypeHook = 100;
constexpr int kDtypeHook16 = 101;         // the same with IEEE binary16 (fp16 compression hook)

inline int64_t chunk_len(int64_t numel, int world) { return (numel + world - 1) / world; }
inline int elem_bytes(int dtype) { return dtype == DDP_BF16 ? 2 : 4; }

// Host-side checks shared by the entry points: world in 1..DDP_MAX_WORLD,
// numel in 0..DDP_MAX_NUMEL, a known dtype.  Entry points call it before any
// byte arithmetic, so numel * element size cannot overflow afterwards.
int32_t common_checks(int32_t world, int64_t numel, int32_t dtype);
// Host buffers of a host-memory allreduce: non-null, element-aligned, inputs
// pairwise disjoint, each output its own input or disjoint from every buffer.
// Call after common_checks.
int32_t check_host_in_out(int32_t world, const void* const* host_in, void* const* host_out, int64_t numel,
                          int32_t dtype);
// DDP_OK for cudaSuccess; otherwise records the error text (ddp_last_cuda_error)
// and returns DDP_ERR_CUDA.
int32_t cuda_status(cudaError_t e);
const char* last_cuda_error();

// Launch geometry helpers (cached per device).
int sm_count();
int grid_for(const void* kernel, int64_t work_items, int threads = kThreads);
// x-extent of an (x, rows) grid whose rows each take per_row items, one per
// thread: one block per kThreads items of a row when the launch moves at
// least 128 MiB and the CTA cap allows it (blocks then run row after row,
// each row's in address order), else four waves of resident blocks shared
// among the rows.
int rows_grid_x(const void* kernel, int64_t per_row, int rows, int64_t bytes);
// Fused-ring kernel chosen by ddp_set_fused_kernel (DDP_FUSED_AUTO = by size).
int fused_kernel_override();

// Kernel that runs one in-place fused ring call.
enum class FusedPath { kScalar, kVector, kGroup, kTma };
constexpr int kGroupMaxWorld = 128;
FusedPath choose_fused_path(int world, int64_t numel, int dtype, bool vec_ok);
// grid clamped to the CTA cap in force (0 = none), at least 1: the calling
// thread's cap if one is set (a reducer's own budget while it launches),
// else the process-wide cap of ddp_set_max_ctas
int cap_ctas(int64_t grid);
// The CTA cap in effect for launches from this thread (0: none).
int cta_cap();
// A cap below four blocks per SM: too few 256-thread register blocks to keep
// HBM busy, where the TMA-staged kernels move several times more bytes per CTA.
bool cta_cap_is_tight();
// Sets the calling thread's cap (-1: none, follow the process-wide cap);
// returns the previous one.
int set_thread_cta_cap(int cap);
bool debug_enabled();

// ---- ring kernels (ring_kernels.cu) -----------------------------------
// All pointers are device pointers; `ptrs` is a host array of `world` entries.
cudaError_t launch_ring_fused(int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div,
                              bool vec_ok, cudaStream_t stream);
// Register path only, out of place: reads in[r], writes the result to out[r]
// (out[r] == in[r] for in place).  Used for buffers the copy engine must not
// stage, e.g. host memory the GPU reads directly.
cudaError_t launch_ring_fused_io(int world, void* const* in, void* const* out, int64_t numel, int dtype, DivSpec div,
                                 bool vec_ok, cudaStream_t stream);
cudaError_t launch_ring_staged(int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div,
                               bool vec_ok, cudaStream_t stream);
// Staged ring in one cooperative launch with bounded grid barriers
// (ring_persistent.cu).  ws: device int32[2] = {status, arrivals}.
cudaError_t launch_ring_persistent(int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div, bool vec_ok,
                                   int32_t* ws, int skip_step, unsigned long long limit_ns, cudaStream_t stream);
// Binomial-tree allreduce (tree_kernels.cu): fused (world <= 64) or one launch per step.
cudaError_t launch_tree_allreduce(bool staged, int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div,
                                  bool vec_ok, cudaStream_t stream);
cudaError_t launch_accumulate(int world, void* const* acc, const void* const* g, int64_t numel, int dtype,
                              bool vec_ok, cudaStream_t stream);

// ---- TMA-staged fused ring (ring_tma.cu) --------------------------------
// The TMA fused kernel can run this call: every buffer 16-byte aligned,
// chunk and bucket byte sizes multiples of 16, world <= 128 (any size; the
// size decision is the caller's).
bool tma_usable(int world, int64_t numel, int dtype, bool vec_ok);
// Bytes of one rank's tile in a TMA kernel with `stages` shared-memory
// stages per CTA (the kernels run 2, the view kernel 3 under tight CTA caps).
int64_t tma_tile_bytes(int world, int stages = 2);
cudaError_t launch_ring_fused_tma(int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div,
                                  cudaStream_t stream);
// The binomial tree's fused allreduce with the same TMA staging (world <= 64,
// buffers 16-byte aligned, bucket bytes a multiple of 16).
bool tree_tma_usable(int world, int64_t numel, int dtype, bool vec_ok);
cudaError_t launch_tree_fused_tma(int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div,
                                  cudaStream_t stream);
cudaError_t read_device_status(int32_t* out, bool clear);
// Wait limit of the TMA kernels' mbarrier waits, and a planted stall taken by
// the next TMA kernel launch (ddp_set_wait_limit_ms, ddp_plant_stall).
void set_wait_limit_ns(unsigned long long ns, unsigned long long* previous);
void plant_stall(long long tile);

// ---- bucket kernels (bucket_kernels.cu) --------------------------------
struct CopyItem {
    const void* src;
    void* dst;
    int64_t bytes;
};
cudaError_t launch_copy_items(const CopyItem* items, int64_t n, cudaStream_t stream);

// Converting copies (bf16 compression hook): float32 -> bf16 (to_bf16 = 1,
// round to nearest even) or bf16 -> float32 (to_bf16 = 0, exact).
struct ConvItem {
    const void* src;
    void* dst;
    int64_t numel;
};
cudaError_t launch_convert_items(const ConvItem* items, int64_t n, int to_bf16, cudaStream_t stream);

// One bucket member for the fused view kernel: its numel, its element offset
// in the bucket and its `world` gradient pointers (rank order).
struct ViewMember {
    int64_t numel;
    int64_t offset;
    void* const* ptrs;   // host array of world device pointers
    bool vec_ok;         // every pointer 16-byte aligned
    int64_t clen = 0;    // chunk length of the member's bucket (0: the bucket passed with it)
};
cudaError_t launch_bucket_view(int world, const ViewMember* members, int n, int64_t bucket_numel, int dtype,
                               DivSpec div, cudaStream_t stream);

// Several buckets' view syncs at once: bucket k is members
// [bucket_first[k], bucket_first[k] + bucket_count[k]) of `members`.
cudaError_t launch_buckets_view(int world, const ViewMember* members, const int* bucket_first, const int* bucket_count,
                                const int64_t* bucket_numel, int n_buckets, int dtype, DivSpec div,
                                cudaStream_t stream);

// A piece of one member that lies inside one ring chunk of its bucket:
// elements [start, start + len) of member `member`, summed from rank j + 1.
struct ViewSegment {
    int32_t member;
    int32_t j;
    int64_t start;
    int64_t len;
};
// A short piece of one member that the TMA view kernel folds element by
// element: elements [start, start + len) of member `member`; each element's
// chunk is its bucket position divided by clen.
struct ViewEdge {
    int32_t member;
    int64_t start;
    int64_t len;
    int64_t clen;
};
// Longest edge the TMA view kernel takes (one element per consumer thread).
constexpr int64_t kTmaEdgeMax = 256;
// Longest segment in one TMA view table entry (its length is 32-bit there);
// longer segment bodies are cut into several entries.
constexpr int64_t kViewSegMax = (int64_t)1 << 30;
// TMA-staged view kernel (ring_tma.cu): the segments' members have 16-byte
// aligned pointers, and every segment's start and length are multiples of
// 16 bytes; edges (len <= kTmaEdgeMax) may belong to any member.
cudaError_t launch_bucket_view_tma(int world, const ViewMember* members, int n_members, const ViewSegment* segs,
                                   int n_segs, const ViewEdge* edges, int n_edges, int dtype, DivSpec div,
                                   cudaStream_t stream);

}  // namespace ddpk
