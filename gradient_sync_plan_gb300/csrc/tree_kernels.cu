// tree_kernels.cu -- binomial-tree allreduce over N logical ranks.
//
// The pages name a tree-based allreduce as the alternative to the ring when
// messages are small ("DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事",
// section 02 and section 07: NCCL's Tree algorithm and its small-message
// threshold).  Reading taken (the pages give no definition): a binomial tree
// over the whole vector.  Reduce steps d = 1, 2, 4, ... < N: rank r with
// r mod 2d == 0 adds the buffer of rank r + d into its own; rank 0 then holds
// the sum and divides it; broadcast steps run the distances in reverse and
// copy rank r's buffer to rank r + d.  Every element is therefore summed in
// the binomial pairwise order ((x0 + x1) + (x2 + x3)) + ..., the same for all
// elements, in 2 ceil(log2 N) steps instead of the ring's 2(N-1).
//
//   k_tree_fused  one pass: every element folded in that order, divided,
//                 written to every rank (N <= 64)
//   k_tree_fused_group  the same for buckets of a few KiB per rank, the
//                 ranks spread over the lanes of a warp
//   k_tree_hop    one launch per tree step, moving exactly what the step moves
#include <algorithm>
#include <cstdio>

#include "ddp_device.cuh"
#include "ddp_internal.h"

namespace ddpk {

template <int CAP>
struct TreeTable {
    char* p[CAP];
};

constexpr int kTreeMaxWorld = 4 * kTreeGroup;   // 64

// One thread per 16-byte vector.  A large bucket is launched with one block
// per kThreads vectors (LOOP = false), so blocks stream the ranks in address
// order as SMs free up; otherwise (and for buffers that are not 16-byte
// aligned, done element-wise) a few waves of blocks loop over the bucket.
template <class E, int DIV, int CAP, int MINB, bool LOOP>
__global__ void __launch_bounds__(kThreads, MINB)
k_tree_fused(const __grid_constant__ TreeTable<CAP> t, int world, int64_t numel, int vec_ok, float dop) {
    using V = typename E::V;
    using S = typename E::S;
    constexpr int L = E::L;
    pdl_release();
    pdl_acquire();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t done = 0;
    if (vec_ok) {
        const int64_t nv = numel / L;
        for (int64_t v = tid; v < nv; v += stride) {
            const int64_t off = v * 16;
            // eight ranks' loads in flight at a time
            V y = tree_fold<V, CAP, (CAP < 8 ? CAP : 8)>(world, [](V a, V b) { return E::vadd(a, b); },
                                                         [&](int r) { return ld_stream<V>(t.p[r] + off); });
            y = E::template vdiv<DIV>(y, dop);
            for (int r = 0; r < world; ++r) st_stream<V>(t.p[r] + off, y);
            if constexpr (!LOOP) break;
        }
        done = nv * L;
    }
    for (int64_t e = done + tid; e < numel; e += stride) {
        S y = tree_fold<S, CAP>(world, [](S a, S b) { return E::sadd(a, b); },
                                [&](int r) { return reinterpret_cast<const S*>(t.p[r])[e]; });
        y = E::template sdiv<DIV>(y, dop);
        for (int r = 0; r < world; ++r) reinterpret_cast<S*>(t.p[r])[e] = y;
    }
}

// Group fused tree for small buckets: P lanes share one 16-byte vector, lane
// q holding ranks q, q + P, ... (R = ceil(N / P) of them).  Tree levels
// d < P are warp shuffles (lane q, q a multiple of 2d, adds lane q + d's
// value), levels d >= P add a lane's own registers -- the binomial tree's
// additions in its order, as in tree_fold.  Lane 0 of the group ends with
// the sum, which every lane then takes and stores to its ranks.  Vectors
// that run past the end are done element-wise by the group's lane 0.
template <class E, int DIV, int CAP, int P, int R>
__global__ void __launch_bounds__(kThreads)
k_tree_fused_group(const __grid_constant__ TreeTable<CAP> t, int world, int64_t numel, float dop) {
    using V = typename E::V;
    using S = typename E::S;
    constexpr int L = E::L;
    constexpr int kGroups = 32 / P;
    const int lane = threadIdx.x & 31;
    const int q = lane & (P - 1);
    const int64_t nvec = (numel + L - 1) / L;
    const int64_t full = numel / L;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t base = warp * kGroups; base < nvec; base += n_warps * kGroups) {    // warp-uniform bounds
        const int64_t v = base + lane / P;
        const bool valid = v < nvec;
        const bool whole = v < full;
        const int64_t off = v * 16;
        V x[R];
#pragma unroll
        for (int m = 0; m < R; ++m) {
            const int r = m * P + q;
            x[m] = (whole && r < world) ? ld_stream<V>(t.p[r] + off) : make_zero<V>();
        }
#pragma unroll
        for (int d = 1; d < P; d <<= 1) {
#pragma unroll
            for (int m = 0; m < R; ++m) {
                const V o = shfl_down_vec(x[m], d, P);
                if ((q & (2 * d - 1)) == 0 && m * P + q + d < world) x[m] = E::vadd(x[m], o);
            }
        }
#pragma unroll
        for (int dm = 1; dm < R; dm <<= 1) {               // d = dm * P
#pragma unroll
            for (int m = 0; m + dm < R; m += 2 * dm)
                if (m * P + dm * P < world) x[m] = E::vadd(x[m], x[m + dm]);
        }
        const V y = E::template vdiv<DIV>(shfl_vec(x[0], 0, P), dop);
        if (whole) {
#pragma unroll
            for (int m = 0; m < R; ++m) {
                const int r = m * P + q;
                if (r < world) st_stream<V>(t.p[r] + off, y);
            }
        } else if (valid && q == 0) {
            for (int64_t e = v * L; e < numel; ++e) {
                S z = tree_fold<S>(world, [](S a, S b) { return E::sadd(a, b); },
                                   [&](int r) { return reinterpret_cast<const S*>(t.p[r])[e]; });
                z = E::template sdiv<DIV>(z, dop);
                for (int r = 0; r < world; ++r) reinterpret_cast<S*>(t.p[r])[e] = z;
            }
        }
    }
}

// One tree step for every pair at once; blockIdx.y is the pair index, its
// lower rank is r = blockIdx.y * 2d and its upper rank r + d.
//   phase 0 (reduce):    buf[r]     = buf[r] (+) buf[r + d]   (divided if `divide`)
//   phase 1 (broadcast): buf[r + d] = buf[r]
// Within a step, the ranks written and the ranks read are disjoint sets.
template <class E, int DIV, int CAP>
__global__ void __launch_bounds__(kThreads)
k_tree_hop(const __grid_constant__ TreeTable<CAP> t, int64_t numel, int d, int phase, int divide, int vec_ok,
           float dop) {
    using V = typename E::V;
    using S = typename E::S;
    constexpr int L = E::L;
    const int r = blockIdx.y * 2 * d;
    // programmatic dependent launch: let the next step be scheduled, and touch
    // no buffer before the previous step has completed
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    char* lo_buf = t.p[r];
    char* hi_buf = t.p[r + d];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t done = 0;
    if (vec_ok) {
        const int64_t nv = numel / L;
        for (int64_t v = tid; v < nv; v += stride) {
            const int64_t off = v * 16;
            if (phase == 0) {
                V y = E::vadd(ld_stream<V>(lo_buf + off), ld_stream<V>(hi_buf + off));
                if (DIV != kDivNone && divide) y = E::template vdiv<DIV>(y, dop);
                st_stream<V>(lo_buf + off, y);
            } else {
                st_stream<V>(hi_buf + off, ld_stream<V>(lo_buf + off));
            }
        }
        done = nv * L;
    }
    for (int64_t e = done + tid; e < numel; e += stride) {
        S* a = reinterpret_cast<S*>(lo_buf);
        S* b = reinterpret_cast<S*>(hi_buf);
        if (phase == 0) {
            S y = E::sadd(a[e], b[e]);
            if (DIV != kDivNone && divide) y = E::template sdiv<DIV>(y, dop);
            a[e] = y;
        } else {
            b[e] = a[e];
        }
    }
}

template <int CAP>
static TreeTable<CAP> tree_table(int world, void* const* ptrs) {
    TreeTable<CAP> t{};
    for (int r = 0; r < world; ++r) t.p[r] = static_cast<char*>(ptrs[r]);
    return t;
}

// Buckets of at least this many bytes over all ranks run one block per tile.
constexpr int64_t kTreeTilePerBlockBytes = 128ll << 20;

template <class E, int DIV, int W, int MINB>
static cudaError_t tree_fused_launch(int world, void* const* ptrs, int64_t numel, float dop, bool vec_ok,
                                     cudaStream_t st) {
    const int64_t tiles = vec_ok ? (numel / E::L + kThreads - 1) / kThreads : 0;
    const bool streamed = vec_ok && (int64_t)world * numel * (int64_t)sizeof(typename E::S) >= kTreeTilePerBlockBytes;
    if (streamed && tiles <= INT32_MAX && cap_ctas(tiles) == tiles) {
        // the tail elements past the last whole vector (fewer than L) fall to
        // threads 0 .. L-2 of block 0, which the grid always holds
        return launch_dependent(k_tree_fused<E, DIV, W, MINB, false>, dim3((unsigned)tiles), dim3(kThreads), 0, st,
                                tree_table<W>(world, ptrs), world, numel, 1, dop);
    }
    auto k = k_tree_fused<E, DIV, W, (W <= 8 ? 4 : 3), true>;
    const int64_t work = vec_ok ? (numel + E::L - 1) / E::L : numel;
    const int grid = grid_for((const void*)k, work);
    return launch_dependent(k, dim3(grid), dim3(kThreads), 0, st, tree_table<W>(world, ptrs), world, numel,
                            vec_ok ? 1 : 0, dop);
}

// Instantiated for the smallest power of two that holds the world: the fold
// is unrolled up to it.
template <class E, int DIV>
static cudaError_t tree_fused_impl(int world, void* const* ptrs, int64_t numel, float dop, bool vec_ok,
                                   cudaStream_t st) {
    // one-tile form: 4 blocks per SM (64 registers) up to 8 ranks, 3 above
    if (world <= 2) return tree_fused_launch<E, DIV, 2, 4>(world, ptrs, numel, dop, vec_ok, st);
    if (world <= 4) return tree_fused_launch<E, DIV, 4, 4>(world, ptrs, numel, dop, vec_ok, st);
    if (world <= 8) return tree_fused_launch<E, DIV, 8, 4>(world, ptrs, numel, dop, vec_ok, st);
    if (world <= 16) return tree_fused_launch<E, DIV, 16, 3>(world, ptrs, numel, dop, vec_ok, st);
    if (world <= 32) return tree_fused_launch<E, DIV, 32, 3>(world, ptrs, numel, dop, vec_ok, st);
    return tree_fused_launch<E, DIV, 64, 3>(world, ptrs, numel, dop, vec_ok, st);
}

constexpr int kTreeGroupThreads = 128;

template <class E, int DIV, int P, int R>
static cudaError_t tree_group_launch(int world, void* const* ptrs, int64_t numel, float dop, cudaStream_t st) {
    auto k = k_tree_fused_group<E, DIV, kTreeMaxWorld, P, R>;
    const int64_t nvec = (numel + E::L - 1) / E::L;
    const int64_t lanes = (nvec + 32 / P - 1) / (32 / P) * 32;
    const int grid = grid_for((const void*)k, lanes, kTreeGroupThreads);
    k<<<grid, kTreeGroupThreads, 0, st>>>(tree_table<kTreeMaxWorld>(world, ptrs), world, numel, dop);
    return cudaGetLastError();
}

template <class E, int DIV>
static cudaError_t tree_group_impl(int world, void* const* ptrs, int64_t numel, float dop, cudaStream_t st) {
    if (world <= 2) return tree_group_launch<E, DIV, 2, 1>(world, ptrs, numel, dop, st);
    if (world <= 4) return tree_group_launch<E, DIV, 4, 1>(world, ptrs, numel, dop, st);
    if (world <= 8) return tree_group_launch<E, DIV, 8, 1>(world, ptrs, numel, dop, st);
    if (world <= 16) return tree_group_launch<E, DIV, 16, 1>(world, ptrs, numel, dop, st);
    if (world <= 32) return tree_group_launch<E, DIV, 32, 1>(world, ptrs, numel, dop, st);
    return tree_group_launch<E, DIV, 32, 2>(world, ptrs, numel, dop, st);
}

// Kernel choice, from a sweep with every kernel forced (fp32 and bf16,
// N = 2 .. 64, 4 KiB .. 256 MiB per rank, CUDA-graph replay):
//  * the group kernel (log2(P) shuffle levels per vector) for 8 or more ranks
//    up to 64 KiB per rank (N = 64 x 16 KiB: 3.3 us against 6.7 on TMA and
//    9.7 on the vector kernel);
//  * the TMA kernel for 32 or more fp32 ranks between 64 and 512 KiB per rank
//    (N = 32 x 256 KiB: 5.9 against 6.6 us);
//  * the vector kernel everywhere else; with one block per tile on large
//    buckets it beats TMA there (N = 8 x 256 MiB: 616 against 649 us,
//    N = 32 x 256 MiB: 2501 against 2654 us).
// ddp_set_fused_kernel can force any of them.
static bool tree_use_group(int world, int64_t numel, int dtype, bool vec_ok) {
    if (!vec_ok || world < 2) return false;
    switch (fused_kernel_override()) {
        case DDP_FUSED_GROUP: return true;
        case DDP_FUSED_VECTOR:
        case DDP_FUSED_TMA: return false;
        default: break;
    }
    const int64_t KiB = 1024;
    const int64_t per_rank = numel * elem_bytes(dtype);
    return world >= 8 && per_rank <= 64 * KiB;
}

template <class E, int DIV>
static cudaError_t tree_staged_impl(int world, void* const* ptrs, int64_t numel, float dop, bool vec_ok,
                                    cudaStream_t st) {
    int depth = 0;
    while ((1 << depth) < world) ++depth;
    const TreeTable<DDP_MAX_WORLD> t = tree_table<DDP_MAX_WORLD>(world, ptrs);
    auto launch = [&](int d, int phase, bool divide) -> cudaError_t {
        const int pairs = (world - d - 1) / (2 * d) + 1;       // r = 0, 2d, ... with r + d < world
        auto kd = k_tree_hop<E, DIV, DDP_MAX_WORLD>;
        const int64_t per_pair = vec_ok ? numel / E::L + E::L : numel;
        const int gx = rows_grid_x((const void*)kd, per_pair, pairs, 0);    // four waves, as the ring's hops
        // each step a programmatic dependent of the previous kernel on the stream
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(gx, pairs);
        cfg.blockDim = dim3(kThreads);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kd, t, numel, d, phase, divide ? 1 : 0, vec_ok ? 1 : 0, dop);
    };
    for (int k = 0; k < depth; ++k) {
        cudaError_t e = launch(1 << k, 0, k == depth - 1);
        if (e != cudaSuccess) return e;
    }
    for (int k = depth - 1; k >= 0; --k) {
        cudaError_t e = launch(1 << k, 1, false);
        if (e != cudaSuccess) return e;
    }
    if (debug_enabled())
        fprintf(stderr, "[ddp] tree_staged world=%d numel=%lld launches=%d\n", world, (long long)numel, 2 * depth);
    return cudaSuccess;
}

template <class E>
static cudaError_t tree_by_div(bool staged, int world, void* const* ptrs, int64_t numel, DivSpec d, bool vec_ok,
                               cudaStream_t st) {
    switch (d.mode) {
        case kDivNone:
            return staged ? tree_staged_impl<E, kDivNone>(world, ptrs, numel, d.operand, vec_ok, st)
                          : tree_fused_impl<E, kDivNone>(world, ptrs, numel, d.operand, vec_ok, st);
        case kDivPow2:
            return staged ? tree_staged_impl<E, kDivPow2>(world, ptrs, numel, d.operand, vec_ok, st)
                          : tree_fused_impl<E, kDivPow2>(world, ptrs, numel, d.operand, vec_ok, st);
        default:
            return staged ? tree_staged_impl<E, kDivIeee>(world, ptrs, numel, d.operand, vec_ok, st)
                          : tree_fused_impl<E, kDivIeee>(world, ptrs, numel, d.operand, vec_ok, st);
    }
}

template <class E>
static cudaError_t tree_group_by_div(int world, void* const* ptrs, int64_t numel, DivSpec d, cudaStream_t st) {
    switch (d.mode) {
        case kDivNone: return tree_group_impl<E, kDivNone>(world, ptrs, numel, d.operand, st);
        case kDivPow2: return tree_group_impl<E, kDivPow2>(world, ptrs, numel, d.operand, st);
        default: return tree_group_impl<E, kDivIeee>(world, ptrs, numel, d.operand, st);
    }
}

static bool tree_use_tma(int world, int64_t numel, int dtype, bool vec_ok) {
    if (!tree_tma_usable(world, numel, dtype, vec_ok)) return false;
    switch (fused_kernel_override()) {
        case DDP_FUSED_TMA: return true;
        case DDP_FUSED_GROUP:
        case DDP_FUSED_VECTOR: return false;
        default: break;
    }
    const int64_t per_rank = numel * elem_bytes(dtype);
    return world >= 32 && dtype == DDP_F32 && per_rank > (64 << 10) && per_rank <= (512 << 10);
}

cudaError_t launch_tree_allreduce(bool staged, int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div,
                                  bool vec_ok, cudaStream_t stream) {
    if (numel == 0) return cudaSuccess;
    if (staged && world == 1) staged = false;                 // no step: the divide only
    if (!staged && tree_use_group(world, numel, dtype, vec_ok)) {
        if (dtype == DDP_F32) return tree_group_by_div<EF32>(world, ptrs, numel, div, stream);
        return tree_group_by_div<EBF16>(world, ptrs, numel, div, stream);
    }
    if (!staged && tree_use_tma(world, numel, dtype, vec_ok))
        return launch_tree_fused_tma(world, ptrs, numel, dtype, div, stream);
    if (dtype == DDP_F32) return tree_by_div<EF32>(staged, world, ptrs, numel, div, vec_ok, stream);
    return tree_by_div<EBF16>(staged, world, ptrs, numel, div, vec_ok, stream);
}

}  // namespace ddpk
