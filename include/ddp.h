/*
 * ddp.h -- C ABI of the GB300 DDP gradient-synchronisation library.
 *
 * DDP keeps one full model replica per data-parallel rank and, after every
 * backward pass, replaces each rank's gradients by their average over the
 * ranks.  Gradients are grouped into flat buckets, each bucket is summed by a
 * ring allreduce, divided by the world size and copied back to the
 * parameters' gradients.  Sources (web pages on DDP gradient sync):
 *   [P1] "DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事"
 *        (blog.vllbc.top): section 01 (gradient averaging), section 03
 *        (reduce-scatter / all-gather, buckets, reverse order, caps,
 *        gradient_as_bucket_view, no_sync), section 04 (ring traffic),
 *        section 05 (step timeline, divide by world size).
 *   [P2] "Day 17 · 梯度的集体行动" (blog.ans20xx.com): "bucket 与 overlap",
 *        "梯度累积:正确使用 no_sync", and the Reducer pseudo-code
 *        (allreduce -> wait -> div_(world_size) -> copy back).
 *   [P3] "DDP 与 Ring-AllReduce" (xuesongtap.github.io): §1.3.1 (2(N-1)
 *        steps), §1.3.2 (3-GPU, length-6 worked example), §1.3.3 (traffic).
 *
 * Model of the ranks.  The N data-parallel ranks are N logical replicas whose
 * buffers all live in one GPU's memory; "rank r" is simply the r-th pointer
 * of a table.  Nothing here crosses a process or a device boundary.
 *
 * Conventions shared by every entry point:
 *   - Ownership: the caller owns every host and device buffer.  The library
 *     allocates no device memory at run time (the no-alloc entry point's
 *     64 MiB array is a static device array) and keeps no pointer after a
 *     call returns (except a ddp_reducer, which keeps the tables it was
 *     created with).  State kept between calls: cached device attributes,
 *     the two process-wide settings (ddp_set_max_ctas, ddp_set_fused_kernel)
 *     and the device status word (ddp_device_status).
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream).  Device work is enqueued asynchronously on it; the
 *     host returns without waiting for the GPU.  Calls may be captured into a
 *     CUDA graph.
 *   - Errors: the return value is a ddp_status.  A negative status from
 *     argument checking means that nothing was enqueued.  DDP_ERR_CUDA means
 *     a CUDA call or launch failed; some of the call's work may have been
 *     enqueued before the failure.  DDP_ERR_HOST means the library could not
 *     allocate host memory for its tables; as with DDP_ERR_CUDA, work before
 *     that point may have been enqueued.
 *   - Dtypes: DDP_F32 (IEEE binary32) or DDP_BF16 (bfloat16).  Element
 *     pointers must be aligned to the element size (DDP_ERR_ALIGN otherwise);
 *     16-byte aligned buffers take the vectorised paths, others a slower
 *     element-wise path with the same results.
 *   - Rank tables: arrays of `world` device pointers, read on the host during
 *     the call only.
 */
#ifndef DDP_GB300_DDP_H
#define DDP_GB300_DDP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DDP_ABI_VERSION 1
#define DDP_MAX_WORLD 512          /* largest supported number of logical ranks */
#define DDP_MAX_NUMEL ((int64_t)1 << 40)  /* largest element count of one rank's buffer or
                                           bucket (DDP_ERR_CAPACITY above it), so that
                                           byte sizes never overflow */

typedef enum {
    DDP_OK = 0,
    DDP_ERR_INVALID = -1,    /* bad argument: null pointer, world < 1, numel < 0,
                                unknown dtype, overlapping buffers, bad plan     */
    DDP_ERR_ALIGN = -2,      /* a pointer is not aligned to its element size    */
    DDP_ERR_CUDA = -3,       /* a CUDA runtime call or a kernel launch failed    */
    DDP_ERR_TIMEOUT = -4,    /* a bounded device-side wait gave up (status word) */
    DDP_ERR_CAPACITY = -5,   /* a size exceeds a documented limit               */
    DDP_ERR_HOST = -6        /* the library's host code failed (out of host
                                memory); no C++ exception leaves the library   */
} ddp_status;

typedef enum { DDP_F32 = 0, DDP_BF16 = 1 } ddp_dtype;

/* Human-readable name of a ddp_status (static string, never NULL). */
const char* ddp_status_string(int32_t status);

/* DDP_ABI_VERSION of the loaded library. */
int32_t ddp_abi_version(void);

/* Text of the last CUDA error that made a call on this host thread return
 * DDP_ERR_CUDA ("no error" if none); a static string, never NULL. */
const char* ddp_last_cuda_error(void);

/*
 * ddp_set_max_ctas -- upper bound on the thread blocks (CTAs) of every kernel
 * this library launches in this process from now on; 0 removes the bound
 * (the default: every kernel fills the GPU).  A bound leaves SMs to compute
 * that runs at the same time, e.g. backward kernels overlapping the bucket
 * syncs of ddp_reducer, at the price of less bandwidth for the sync itself.
 * Results do not depend on it.  *previous (if not NULL) receives the old
 * value.  DDP_ERR_INVALID for a negative bound.
 */
int32_t ddp_set_max_ctas(int32_t max_ctas, int32_t* previous);

/*
 * ddp_set_fused_kernel -- which kernel ring_allreduce_fused (and every call
 * that runs it on one buffer per rank: ddp_sync_buckets with
 * DDP_ALGO_FUSED / DDP_ALGO_BF16_HOOK, the reducer) uses from now on in this
 * process, and which kernel folds the aligned segments of the fused view
 * path (ddp_bucket_allreduce_view*, DDP_ALGO_VIEW and the hook views, the
 * L2-sized pieces of DDP_ALGO_FUSED): DDP_FUSED_TMA the TMA-staged view
 * kernel, DDP_FUSED_VECTOR or DDP_FUSED_GROUP the register view kernel,
 * DDP_FUSED_AUTO the TMA kernel for 16 or more ranks whose segments move
 * less than 128 MiB and the register kernel otherwise.  All of them compute
 * the same fold in the same order, so results are bit-identical whichever
 * runs; the choice only changes speed.
 *   DDP_FUSED_AUTO   by size (the default): the group kernel up to 4 KiB
 *                    per rank, up to 256 KiB over 2 ranks, and up to 16 KiB
 *                    over 8 fp32 ranks or where fp32 chunk boundaries are
 *                    not 16-byte aligned; the TMA kernel for 16 or more
 *                    ranks with little data each (up to 16 KiB per rank; up
 *                    to 1 MiB at 32-63 ranks, 256 KiB at 64-127, 64 KiB from
 *                    128; fp32 at 16-31 ranks from 256 KiB to 4 MiB); the
 *                    vector kernel otherwise, which includes every large
 *                    bucket -- except under a CTA cap (ddp_set_max_ctas, a
 *                    reducer's budget) below four CTAs per SM, where buckets
 *                    from 1 MiB per rank, and the view path's segments, go
 *                    to the TMA kernels;
 *   DDP_FUSED_VECTOR one thread per 16-byte vector (two over 2 or 3 ranks),
 *                    folding all N ranks; a bucket of 128 MiB or more over
 *                    all ranks runs one block per tile of vectors;
 *   DDP_FUSED_GROUP  a group of lanes per vector, one rank (or a few) per
 *                    lane, the fold done on values passed by warp shuffles
 *                    (N <= 128);
 *   DDP_FUSED_TMA    tiles of every rank staged in shared memory by bulk
 *                    copies (N <= 128, 16-byte-aligned chunks).
 * A kernel that cannot run a call (alignment, world size) is replaced by
 * the vector kernel, or the element-wise one for unaligned buffers.
 * tree_allreduce_fused follows the same forced choice among its own group,
 * vector and TMA kernels (its TMA kernel folds the staged tiles in the
 * tree's order and takes buckets whose bytes per rank are a multiple of 16,
 * N <= 64).  By size it runs the group kernel for 8 or more ranks up to 64
 * KiB per rank, the TMA kernel for 32 or more fp32 ranks between 64 and 512
 * KiB per rank, and the vector kernel otherwise.
 * *previous (if not NULL) receives the old choice.  DDP_ERR_INVALID for an
 * unknown kind.
 */
typedef enum {
    DDP_FUSED_AUTO = 0,
    DDP_FUSED_VECTOR = 1,
    DDP_FUSED_GROUP = 2,
    DDP_FUSED_TMA = 3
} ddp_fused_kernel;

int32_t ddp_set_fused_kernel(int32_t kind, int32_t* previous);

/*
 * ddp_device_status -- the library's sticky device-side status word on the
 * current device: DDP_OK, or DDP_ERR_TIMEOUT if a kernel's bounded wait on an
 * asynchronous copy gave up (the kernel then stopped early, so the buffers
 * of that call hold partial results).  Synchronous: call it after the
 * stream of interest has been synchronised.  clear != 0 resets the word.
 * Returns DDP_OK, DDP_ERR_INVALID (status NULL) or DDP_ERR_CUDA.
 */
int32_t ddp_device_status(int32_t* status, int32_t clear);

/*
 * ddp_set_wait_limit_ms -- limit of every bounded device-side wait in the
 * TMA-staged kernels (the fused ring's, the fused tree's and the fused
 * view's), in
 * milliseconds, for launches from now on in this process; 0 restores the
 * default of 2000 ms.  A kernel whose wait runs out sets the device status
 * word to DDP_ERR_TIMEOUT (ddp_device_status) and stops early instead of
 * hanging.  The pages describe the hang this guards against: a collective
 * waits for every rank, so a rank that never joins stalls the others
 * without an error ([P2] "INVARIANT 2" and "常见疑问" Q2).  Results do not
 * depend on the limit.  *previous_ms (if not NULL) receives the old limit.
 * DDP_ERR_INVALID unless 0 <= limit_ms <= 600000.
 */
int32_t ddp_set_wait_limit_ms(int32_t limit_ms, int32_t* previous_ms);

/*
 * ddp_plant_stall -- a test hook that plants the hang of [P2] "常见疑问" Q2 on
 * the GPU.  The next launch of a TMA-staged kernel (see
 * ddp_set_wait_limit_ms) takes the plant: the producer warp of the CTA that
 * owns tile `tile` of that launch issues no bulk copy for that tile or any
 * later one, and waits for the copies it did issue to be consumed; the CTA's
 * consumers wait for the missing tile until the wait limit runs out, set
 * DDP_ERR_TIMEOUT and stop.  No copy is left in flight and no memory is
 * touched out of bounds; the call's buffers hold partial results.  A tile
 * number beyond the launch's tiles plants nothing (the launch still takes
 * the plant).  tile = -1 removes a plant that no launch has taken yet.
 * Returns DDP_OK, or DDP_ERR_INVALID for tile < -1.
 */
int32_t ddp_plant_stall(int64_t tile);

/*
 * ddp_plan_buckets -- assign parameters to buckets ([P1] section 03 "Bucket"
 * and "Overlap", section 05 step 2; [P2] "bucket 与 overlap").
 *
 * Parameters are visited in REVERSE registration order (p = n_params-1 .. 0),
 * the order in which backward produces their gradients.  Each one is appended
 * to the open bucket at the bucket's current element count (no padding, so
 * in-bucket order is reverse registration order).  After an append, a bucket
 * whose byte size is >= its cap is closed: bucket 0 uses first_bucket_bytes
 * (DDP's default 1 MiB), every later bucket bucket_cap_bytes (default 25 MiB;
 * the pages' "MB" is MiB).  A bucket may therefore exceed its cap by its last
 * parameter, and a parameter larger than the cap closes its bucket at once.
 * A bucket still open at the end is closed if it holds any parameter.
 *
 *   n_params                 number of parameters (>= 0)
 *   numel[n_params]          elements of each parameter, registration order (>= 0)
 *   dtype                    element type of every gradient (one dtype per plan)
 *   first_bucket_bytes       cap of bucket 0, bytes (> 0)
 *   bucket_cap_bytes         cap of the other buckets, bytes (> 0)
 *   bucket_of_param[n_params] out: bucket index of each parameter
 *   offset_of_param[n_params] out: element offset of each parameter in its bucket
 *   bucket_numel[n_params]   out: elements of each bucket (room for n_params)
 *   n_buckets                out: number of buckets
 * Host only; no CUDA call.  DDP_ERR_INVALID on a bad argument.
 */
int32_t ddp_plan_buckets(int32_t n_params, const int64_t* numel, int32_t dtype,
                         int64_t first_bucket_bytes, int64_t bucket_cap_bytes,
                         int32_t* bucket_of_param, int64_t* offset_of_param,
                         int64_t* bucket_numel, int32_t* n_buckets);

/*
 * ddp_plan_fingerprint -- a 64-bit digest of a bucket plan (FNV-1a over the
 * parameter count, dtype, every parameter's numel, bucket and offset, the
 * bucket count and every bucket's numel, each as 8 little-endian bytes).
 * Ranks whose plans differ would run different collective sequences, which
 * on a real ring hangs without an error ([P2] "常见疑问", why DDP can hang);
 * ranks exchange this value over their host process group before the first
 * sync and stop on a mismatch.  Host only; no CUDA call.  DDP_ERR_INVALID on
 * a bad argument.
 */
int32_t ddp_plan_fingerprint(int32_t n_params, const int64_t* numel, int32_t dtype,
                             const int32_t* bucket_of_param, const int64_t* offset_of_param,
                             int32_t n_buckets, const int64_t* bucket_numel, uint64_t* fingerprint);

/*
 * ddp_bucket_pack -- copy gradients into each rank's flat bucket, the
 * "gradient -> bucket" copy DDP makes when gradient_as_bucket_view is off
 * ([P1] section 03 and section 05 step 2).
 *
 * For every rank r and member i:
 *   buckets[r][offset[i] .. offset[i]+numel[i]) <- grads[r*n_in_bucket + i][0 .. numel[i])
 *
 *   world                 logical ranks, 1 .. DDP_MAX_WORLD
 *   n_in_bucket           members of this bucket (>= 0)
 *   grads[world*n_in_bucket] host table of device pointers, rank-major
 *   numel[n_in_bucket]    elements of each member
 *   offset[n_in_bucket]   element offset of each member inside the bucket
 *   buckets[world]        host table of device pointers to the rank buckets
 *   bucket_numel          elements of each rank's bucket; every member must
 *                         satisfy offset + numel <= bucket_numel
 * Member ranges must not overlap each other (a plan from ddp_plan_buckets
 * never does); source and destination must not overlap.
 */
int32_t ddp_bucket_pack(int32_t world, int32_t n_in_bucket, const void* const* grads,
                        const int64_t* numel, const int64_t* offset, void* const* buckets,
                        int64_t bucket_numel, int32_t dtype, void* stream);

/*
 * ddp_bucket_unpack -- the inverse copy, bucket -> .grad, after the bucket's
 * allreduce and average ([P1] section 05 step 3; [P2] Reducer pseudo-code,
 * "copy back to param grads").
 *
 *   grads[r*n_in_bucket + i][0 .. numel[i]) <- buckets[r][offset[i] .. offset[i]+numel[i])
 * Arguments as for ddp_bucket_pack.
 */
int32_t ddp_bucket_unpack(int32_t world, int32_t n_in_bucket, void* const* grads,
                          const int64_t* numel, const int64_t* offset, const void* const* buckets,
                          int64_t bucket_numel, int32_t dtype, void* stream);

/*
 * ddp_bucket_pack_bf16 / ddp_bucket_unpack_bf16 -- the copies of the bf16
 * compression communication hook ([P2] reading list, "PyTorch DDP
 * Communication Hooks": fp16/bf16 compression): float32 gradients are rounded
 * to bf16 (nearest even) as they are packed into a bf16 bucket, the bucket is
 * reduced in bf16 (per-hop rounding, see ring_allreduce_fused), and the
 * averaged bf16 values are widened exactly to float32 as they are unpacked.
 * The pages do not say where the hook divides; like every other path here,
 * the division by the world size happens once, after the reduction.
 * Arguments as for ddp_bucket_pack / ddp_bucket_unpack, with float32 `grads`,
 * bf16 `buckets` (bucket_numel elements each) and no dtype argument.
 */
int32_t ddp_bucket_pack_bf16(int32_t world, int32_t n_in_bucket, const void* const* grads, const int64_t* numel,
                             const int64_t* offset, void* const* buckets, int64_t bucket_numel, void* stream);
int32_t ddp_bucket_unpack_bf16(int32_t world, int32_t n_in_bucket, void* const* grads, const int64_t* numel,
                               const int64_t* offset, const void* const* buckets, int64_t bucket_numel, void* stream);

/*
 * ring_allreduce_fused -- the ring allreduce of one bucket, in one pass over
 * memory, with the ring's exact result ([P1] section 03 "两阶段"; [P3]
 * §1.3.1-§1.3.2).
 *
 * The bucket of S = numel elements is cut into N = world chunks of
 * c = ceil(S/N) elements (chunk j = [min(jc,S), min((j+1)c,S)); trailing
 * chunks may be short or empty).  On the ring, rank r sends to rank r+1;
 * reduce-scatter step s (1..N-1) sends chunk (r-s) mod N and the receiver adds
 * it into its copy, all-gather step t (1..N-1) sends chunk (r-t+1) mod N and
 * the receiver overwrites.  Chunk j is therefore summed starting at rank
 * (j+1) mod N and finishing at rank j:
 *     y[i] = (((x_{j+1}[i] + x_{j+2}[i]) + ...) + x_{j+N}[i])   (ranks mod N)
 * and then, if divisor > 1, y[i] / divisor (one IEEE division).  This kernel
 * reads each rank's element once, folds in exactly that order and writes y to
 * all N buffers, so its result is bit-identical to the hop-by-hop ring
 * (which of its kernels runs: ddp_set_fused_kernel).
 * fp32: binary32 adds, round to nearest even.  bf16: each add is done in
 * binary32 and rounded to bf16 (nearest even), once per hop; the divide
 * rounds once to bf16.
 *
 *   world      logical ranks N, 1 .. DDP_MAX_WORLD
 *   bufs[world] host table of device pointers; rank r's bucket, S elements,
 *              read and overwritten in place; buffers must not overlap
 *   numel      S (>= 0; 0 is a no-op)
 *   divisor    0 or 1: leave the sum; > 1: divide (DDP passes the world size)
 */
int32_t ring_allreduce_fused(int32_t world, void* const* bufs, int64_t numel, int32_t dtype,
                             int32_t divisor, void* stream);

/*
 * ring_allreduce_staged -- the same allreduce reproduced hop by hop: N-1
 * reduce-scatter kernels then N-1 all-gather kernels on `stream`, each one
 * moving, for every rank at once, exactly the chunk the ring moves in that
 * step ([P1] section 03; [P3] §1.3.2).  The average is folded into the last
 * reduce-scatter step (the owner of each chunk divides it before it is
 * circulated).  Same arguments and bit-identical results as
 * ring_allreduce_fused; 5(N-1)/N * S elements of traffic per rank instead of 2.
 */
int32_t ring_allreduce_staged(int32_t world, void* const* bufs, int64_t numel, int32_t dtype,
                              int32_t divisor, void* stream);

/*
 * tree_allreduce_fused / tree_allreduce_staged -- the latency-oriented
 * alternative to the ring for small buckets ([P1] section 02 and section 07:
 * a tree-based allreduce, NCCL's Tree algorithm below a message-size
 * threshold).  The pages do not define the tree; this library uses the
 * binomial tree over the whole vector: reduce steps d = 1, 2, 4, ... < N in
 * which rank r (r mod 2d == 0) adds rank r+d's buffer into its own, the root
 * divides, and broadcast steps in reverse order copy rank r's buffer to rank
 * r+d.  Every element is summed in the pairwise order ((x0+x1)+(x2+x3))+...,
 * which differs from the ring's, so tree and ring results differ in the last
 * bits; both are reproducible.  2*ceil(log2 N) steps instead of 2(N-1).
 *   tree_allreduce_fused   one pass over memory; world <= 64 (DDP_ERR_CAPACITY)
 *   tree_allreduce_staged  one launch per tree step; world <= DDP_MAX_WORLD
 * Arguments, dtypes, rounding (bf16: one rounding per addition) and the
 * divide as for ring_allreduce_fused.
 */
int32_t tree_allreduce_fused(int32_t world, void* const* bufs, int64_t numel, int32_t dtype, int32_t divisor,
                             void* stream);
int32_t tree_allreduce_staged(int32_t world, void* const* bufs, int64_t numel, int32_t dtype, int32_t divisor,
                              void* stream);

/*
 * ring_allreduce_persistent -- ring_allreduce_staged in ONE cooperative
 * launch: the same 2(N-1) steps and the same bit-identical result ([P1]
 * section 03; [P3] §1.3.2), with the steps separated by grid-wide barriers
 * instead of kernel launches, which removes the per-step launch latency on
 * small buckets.
 *
 * A real ring hangs when one rank never joins a step ([P2] "常见疑问", on why
 * DDP can hang without an error).  Here every barrier wait is bounded by
 * wait_limit_ms (0 = 2000 ms): a block that waits longer writes
 * DDP_ERR_TIMEOUT to dev_status[0] and returns, so the context stays usable
 * and the buffers hold a partial result.
 *
 *   dev_status   device int32[2], 8-byte aligned, caller-owned: [0] status
 *                (DDP_OK or DDP_ERR_TIMEOUT after the kernel), [1] barrier
 *                arrivals.  Both are zeroed on `stream` before the launch; read
 *                [0] after synchronising.  Concurrent calls need separate words.
 *   fail_at_step -1 for normal use.  k in [0, 2(N-1)-2] plants a failure for
 *                testing: one block never arrives at the barrier that ends
 *                step k, so every block times out there.
 * Other arguments as for ring_allreduce_fused.
 */
int32_t ring_allreduce_persistent(int32_t world, void* const* bufs, int64_t numel, int32_t dtype, int32_t divisor,
                                  int32_t* dev_status, int32_t fail_at_step, int32_t wait_limit_ms, void* stream);

/*
 * ring_allreduce_fused_from_host -- ring_allreduce_fused for callers whose
 * gradients are in host memory: per rank, host_in[r] is copied to dev_bufs[r],
 * the fused allreduce runs, and the result is copied to host_out[r]
 * (host_out[r] may equal host_in[r]).  Buckets of more than 64 MiB per
 * rank go through in 32 MiB pieces on three internal streams, so that copies
 * in, the reduction of each piece (folded in the ring order of the whole
 * bucket's chunks) and copies out overlap; `stream` waits for the last copy
 * out.  Smaller buckets, and calls on a stream that is being captured into a
 * graph, run in, reduce, out on `stream` itself.  The caller synchronises
 * `stream` before reading host_out.  Host buffers should be pinned for the
 * copies to be asynchronous.
 * dev_bufs[world] is caller-provided device scratch of numel elements per rank.
 */
int32_t ring_allreduce_fused_from_host(int32_t world, const void* const* host_in, void* const* host_out,
                                       void* const* dev_bufs, int64_t numel, int32_t dtype,
                                       int32_t divisor, void* stream);

/*
 * ring_allreduce_fused_host_direct -- the fused allreduce run directly on
 * host buffers, without device copies: the kernel reads every rank's
 * elements from host_in[r] over the CPU-GPU link and writes the averaged
 * result to host_out[r] (host_out[r] may equal host_in[r]).  Result and order
 * as ring_allreduce_fused ([P1] section 03; [P3] §1.3.2).  Host traffic per
 * call: world * numel elements read, the same written, in one pass -- both
 * directions of the link at once, where a copy-based path moves them one
 * after the other.
 *
 * Every buffer must be reachable by the GPU: page-locked host memory
 * (cudaHostAlloc / cudaHostRegister), managed or device memory, or pageable
 * memory on systems whose GPU reads pageable memory directly; otherwise
 * DDP_ERR_INVALID before any work.  Inputs must not overlap; an output must
 * either be its own input or overlap no input and no other output.
 * Asynchronous on `stream`: synchronise before reading host_out.
 */
int32_t ring_allreduce_fused_host_direct(int32_t world, const void* const* host_in, void* const* host_out,
                                         int64_t numel, int32_t dtype, int32_t divisor, void* stream);

/*
 * ring_allreduce_fused_from_host_noalloc -- ring_allreduce_fused_from_host for
 * callers that cannot allocate device memory.  The pages have no counterpart
 * to this entry point; it exists for callers whose gradients sit in host
 * memory and who have no device allocator of their own to hand over scratch
 * buffers (for example a host-side loop inside a framework that owns all of
 * the device's memory, or a tool that links only this library).
 *
 * Instead of caller-provided device buffers, the ranks' copies live in one
 * array of DDP_STATIC_SCRATCH_BYTES bytes that the library reserves in its own
 * module: every GPU that loads the library holds that memory until the
 * process exits.  The call allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine).  Each rank's copy starts on a 256-byte
 * boundary, so world * round_up(numel * element size, 256) must not exceed
 * DDP_STATIC_SCRATCH_BYTES; larger requests return DDP_ERR_CAPACITY before
 * any CUDA work.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with the device current) and caches it; make
 * that first call before any stream capture.  The cached address belongs to
 * the device's context and does not survive cudaDeviceReset: after a reset of
 * a device, do not call this entry point on it again in the same process.
 * Sizes are checked (world, numel <= DDP_MAX_NUMEL, dtype, then the array's
 * capacity) before any byte count is formed.  All calls on a device share
 * the array: calls that overlap on the GPU (different streams, or host
 * threads without ordering) race and corrupt each other's results.  The
 * array keeps the last call's contents; no clearing is needed, since a call
 * overwrites every byte it uses before reading it.
 *
 * Arguments, copies, results and synchronisation as for
 * ring_allreduce_fused_from_host, without dev_bufs.
 */
#define DDP_STATIC_SCRATCH_BYTES (64ll << 20)   /* 64 MiB per GPU */
int32_t ring_allreduce_fused_from_host_noalloc(int32_t world, const void* const* host_in, void* const* host_out,
                                               int64_t numel, int32_t dtype, int32_t divisor, void* stream);

/*
 * ddp_grad_accumulate -- one no_sync micro-batch folded into the local
 * gradients of every rank ([P1] section 03 and section 05 step 5; [P2]
 * "梯度累积:正确使用 no_sync"): acc[r][i] <- acc[r][i] + grads[r][i]
 * (binary32 add; bf16: binary32 add rounded to bf16).  No communication.
 *   acc[world], grads[world]  host tables of device pointers, numel elements each
 */
int32_t ddp_grad_accumulate(int32_t world, void* const* acc, const void* const* grads, int64_t numel,
                            int32_t dtype, void* stream);

/* Allreduce algorithm used by ddp_sync_buckets for each bucket. */
typedef enum {
    DDP_ALGO_FUSED = 0,   /* pack -> ring_allreduce_fused -> unpack             */
    DDP_ALGO_STAGED = 1,  /* pack -> ring_allreduce_staged -> unpack            */
    DDP_ALGO_VIEW = 2,    /* ddp_bucket_allreduce_view (no bucket copies)        */
    DDP_ALGO_DRYRUN = 3,  /* ddp_reducer only: track readiness and launch order,
                             make no CUDA call (for checking a plan's order)    */
    DDP_ALGO_BF16_HOOK = 4, /* float32 gradients, bf16 buckets: ddp_bucket_pack_bf16
                             -> ring_allreduce_fused in bf16 -> ddp_bucket_unpack_bf16 */
    DDP_ALGO_BF16_HOOK_VIEW = 5, /* the same result in one pass, no bucket buffers:
                             ddp_bucket_allreduce_view_bf16                         */
    DDP_ALGO_FP16_HOOK_VIEW = 6 /* the fp16 compression hook in one pass (float32
                             gradients, IEEE binary16 arithmetic):
                             ddp_bucket_allreduce_view_fp16                         */
} ddp_algo;

/*
 * ddp_sync_buckets -- DDP's reducer step for a whole model: for every bucket
 * k = 0 .. n_buckets-1 in order, pack the members' gradients into each rank's
 * bucket k, ring-allreduce the bucket and divide by `divisor`, and copy the
 * result back into the gradients ([P2] Reducer pseudo-code: allreduce, wait,
 * div_(world_size), copy back; [P1] section 05 steps 2-3).  Bucket i+1 is
 * never started before bucket i (same stream).
 *
 *   grads[world*n_params]      host table of device pointers, rank-major,
 *                              registration order
 *   numel[n_params], bucket_of_param[n_params], offset_of_param[n_params],
 *   bucket_numel[n_buckets]    a plan from ddp_plan_buckets
 *   buckets[world*n_buckets]   host table of device pointers: rank r's buffer
 *                              for bucket k at [r*n_buckets + k], at least
 *                              bucket_numel[k] elements (may alias across k;
 *                              unused by DDP_ALGO_VIEW and may then be NULL)
 *   algo                       a ddp_algo (DDP_ALGO_BF16_HOOK: float32 `grads` and
 *                              dtype, bf16 `buckets`)
 * The same plan must be used on every rank (one plan is shared here by
 * construction).  DDP_ERR_INVALID if the plan is inconsistent.
 *
 * With DDP_ALGO_FUSED, a bucket whose bytes over all ranks exceed 1.5 pieces
 * of 96 MiB (more than the GPU's L2) runs piece by piece: each piece's slice
 * of the members is packed, the slice is reduced by the view pass at its
 * bucket offset (so every element is folded in the ring order of its chunk
 * of the WHOLE bucket), and the slice is unpacked before the next piece is
 * packed.  The result, in the gradients and in the bucket buffers, is
 * bit-identical to the whole-bucket pack -> ring -> unpack; only the HBM
 * traffic falls, since each piece is read back from L2.
 */
int32_t ddp_sync_buckets(int32_t world, int32_t n_params, void* const* grads, const int64_t* numel,
                         const int32_t* bucket_of_param, const int64_t* offset_of_param,
                         int32_t n_buckets, const int64_t* bucket_numel, void* const* buckets,
                         int32_t dtype, int32_t divisor, int32_t algo, void* stream);

/*
 * ddp_bucket_allreduce_view -- pack, ring allreduce, average and unpack of one
 * bucket fused into a single pass, as if every gradient were a view into its
 * bucket (gradient_as_bucket_view=True, [P1] section 03 and section 05; [P2]
 * "bucket 与 overlap"): each member's elements are read once from every
 * rank's gradient, summed in the ring order of the chunk their BUCKET
 * position falls in (chunk size ceil(bucket_numel/N)), divided, and written
 * back to every rank's gradient.  Bit-identical to ddp_bucket_pack +
 * ring_allreduce_fused + ddp_bucket_unpack on the same bucket, with a third
 * of the memory traffic and no bucket buffer.
 * Arguments as for ddp_bucket_pack, without the bucket buffers.
 */
int32_t ddp_bucket_allreduce_view(int32_t world, int32_t n_in_bucket, void* const* grads,
                                  const int64_t* numel, const int64_t* offset, int64_t bucket_numel,
                                  int32_t dtype, int32_t divisor, void* stream);

/*
 * ddp_reducer -- DDP's reducer: each bucket's allreduce starts as soon as its
 * gradients are ready, in bucket order, overlapping the rest of backward
 * ([P1] section 03 "Overlap", section 05 steps 2 and 5; [P2] "梯度同步时机"
 * and the Reducer pseudo-code).
 *
 * A reducer is created once per model and plan.  For every backward pass:
 *   ddp_reducer_prepare   forget the previous pass's readiness;
 *   ddp_reducer_mark_ready(p, compute_stream)
 *                         call after the producer of parameter p's gradient
 *                         (on every rank) has been enqueued on compute_stream;
 *                         when p completes its bucket, an event is recorded on
 *                         compute_stream, and every bucket of the ready prefix
 *                         (bucket 0, 1, ... not launched yet and complete) is
 *                         launched on comm_stream after its event -- bucket i+1
 *                         never before bucket i;
 *   ddp_reducer_finalize(stream)
 *                         the point before the optimizer step: `stream` waits
 *                         for every bucket's sync.  DDP_ERR_INVALID if some
 *                         bucket never became ready (a parameter that got no
 *                         gradient, the case DDP needs find_unused_parameters
 *                         for).
 * Marking a parameter twice in one pass is DDP_ERR_INVALID.
 *
 *   grads[world*n_params], numel, bucket_of_param, offset_of_param,
 *   bucket_numel, buckets[world*n_buckets]  as for ddp_sync_buckets (buckets may
 *                         be NULL for DDP_ALGO_VIEW, the fused hooks and
 *                         DDP_ALGO_DRYRUN, grads for DDP_ALGO_DRYRUN); the
 *                         reducer keeps these pointers until it is destroyed,
 *                         the caller keeps the memory
 *   algo                  any ddp_algo; each bucket's sync is the one
 *                         ddp_sync_buckets runs for that algo (pieces
 *                         included), the hooks with a float32 dtype
 *   comm_stream           cudaStream_t on which the buckets' syncs run
 * The reducer owns host memory and three CUDA events per bucket (readiness
 * and two timing events; created here, destroyed by ddp_reducer_destroy); it
 * allocates no device memory.
 */
typedef struct ddp_reducer ddp_reducer;
int32_t ddp_reducer_create(int32_t world, int32_t n_params, void* const* grads, const int64_t* numel, int32_t dtype,
                           const int32_t* bucket_of_param, const int64_t* offset_of_param, int32_t n_buckets,
                           const int64_t* bucket_numel, void* const* buckets, int32_t algo, int32_t divisor,
                           void* comm_stream, ddp_reducer** out);
int32_t ddp_reducer_prepare(ddp_reducer* reducer);
/*
 * ddp_reducer_set_max_ctas -- CTA budget of this reducer's bucket syncs, like
 * ddp_set_max_ctas but for the kernels this reducer launches only: -1 (the
 * default) follows the process-wide setting, 0 removes any cap for them,
 * n > 0 caps them at n CTAs.  A small budget leaves SMs to the backward that
 * runs beside the syncs ([P1] section 03 "Overlap"); on one GB300 with a GEMM
 * backward, a quarter of the SMs hid the most.  Results do not depend on it.
 * DDP_ERR_INVALID for a NULL reducer or max_ctas < -1.
 */
int32_t ddp_reducer_set_max_ctas(ddp_reducer* reducer, int32_t max_ctas);
int32_t ddp_reducer_mark_ready(ddp_reducer* reducer, int32_t param, void* compute_stream);
int32_t ddp_reducer_finalize(ddp_reducer* reducer, void* stream);
/* Buckets launched in the current pass, in launch order (up to capacity). */
int32_t ddp_reducer_launch_order(ddp_reducer* reducer, int32_t* order, int32_t capacity, int32_t* n);
/* Per-bucket sync time of the current pass, in bucket order: ms[k] is the
 * comm-stream time from the start to the end of bucket k's sync (DDP's
 * per-bucket communication time, [P2] "bucket 与 overlap", "四组实验记录法"); -1 for a bucket
 * launched on a stream that was being captured into a graph, or under
 * DDP_ALGO_DRYRUN.  Waits for those buckets' syncs to finish.  *n receives
 * the number of buckets launched so far (up to capacity are written). */
int32_t ddp_reducer_bucket_times(ddp_reducer* reducer, float* ms, int32_t capacity, int32_t* n);
int32_t ddp_reducer_destroy(ddp_reducer* reducer);

/*
 * ddp_bucket_allreduce_view_bf16 -- the bf16 compression hook fused like
 * ddp_bucket_allreduce_view: float32 gradients are read once from every
 * rank, each value is rounded to bf16, the values are summed in the ring
 * order of their bucket chunk with one bf16 rounding per hop, divided
 * (rounded to bf16), and the bf16 result is written back widened to float32.
 * Bit-identical to ddp_bucket_pack_bf16 + ring_allreduce_fused (bf16) +
 * ddp_bucket_unpack_bf16 on the same bucket, without the bucket buffers.
 * Arguments as for ddp_bucket_allreduce_view, with float32 gradients and no
 * dtype argument.
 */
int32_t ddp_bucket_allreduce_view_bf16(int32_t world, int32_t n_in_bucket, void* const* grads,
                                       const int64_t* numel, const int64_t* offset, int64_t bucket_numel,
                                       int32_t divisor, void* stream);

/*
 * ddp_bucket_allreduce_view_fp16 -- the fp16 compression hook ([P2] reading
 * list: DDP communication hooks, fp16/bf16 compression), fused like
 * ddp_bucket_allreduce_view_bf16 with IEEE binary16 in place of bf16: every
 * float32 gradient value is rounded to binary16 (nearest even), the values
 * are summed in the ring order of their bucket chunk with a binary32 add of
 * the two widened values rounded to binary16 after every hop, divided
 * (rounded to binary16), and written back widened to float32.  Values that
 * round beyond 65504 become infinity, as in binary16.  Arguments as for
 * ddp_bucket_allreduce_view_bf16.
 */
int32_t ddp_bucket_allreduce_view_fp16(int32_t world, int32_t n_in_bucket, void* const* grads,
                                       const int64_t* numel, const int64_t* offset, int64_t bucket_numel,
                                       int32_t divisor, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DDP_GB300_DDP_H */
