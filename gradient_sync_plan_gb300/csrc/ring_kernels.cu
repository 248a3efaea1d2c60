// ring_kernels.cu -- ring allreduce over N logical ranks held in one GPU.
//
// The ring of "DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事"
// (section 03, "两阶段：先规约，再扩散") and "DDP 与 Ring-AllReduce" (§1.3.1,
// §1.3.2): a bucket of S elements is cut into N chunks of c = ceil(S/N);
// rank r sends to r+1; reduce-scatter step s sends chunk (r-s) mod N and the
// receiver adds it in, all-gather step t sends chunk (r-t+1) mod N and the
// receiver overwrites.  Chunk j is thus summed from rank j+1 round to rank j.
//
// Two kernels reach that result:
//   * k_ring_fused: one pass; every element is read once from each rank,
//     folded in exactly that order, divided, and stored to every rank.
//     Traffic 2*N*S elements, the minimum.
//   * k_ring_hop: one launch per ring step, moving for every rank the chunk
//     the ring moves in that step.  Traffic 5(N-1)*S elements.
#include <algorithm>
#include <cstdio>

#include "ddp_device.cuh"
#include "ddp_internal.h"

namespace ddpk {

// Rank pointer table passed by value in the kernel's parameter space.
template <int CAP>
struct RankTable {
    char* p[CAP];
};

// ---------------------------------------------------------------------------
// Fused ring allreduce
// ---------------------------------------------------------------------------

// The fused kernels read rank r from t.p[r] and write it to t.p[world + r]:
// an in-place call passes the same pointer twice, an out-of-place call (host
// buffers read and written directly) two.  The table holds 2 * world entries.

// One element, any alignment: fold in ring order, divide, store to all ranks.
template <class E, int DIV, int CAP>
__device__ __forceinline__ void ring_element(const RankTable<CAP>& t, int world, int64_t e, int64_t clen,
                                             float dop) {
    using S = typename E::S;
    const int j = (int)(e / clen);
    const int start = (j + 1 == world) ? 0 : j + 1;
    auto at = [&](int r) -> const char* { return t.p[r]; };
    S y = E::template sdiv<DIV>(fold_ring_scalar<E>(at, world, start, e), dop);
    for (int r = 0; r < world; ++r) reinterpret_cast<S*>(t.p[world + r])[e] = y;
}

// The elements the vector path leaves: those of every 16-byte vector that
// straddles a chunk boundary, and of the ragged last vector.  Entry q of
// world * L takes lane q % L of the vector holding boundary q / L + 1 (or,
// for the last L entries, of the last vector); a vector that holds several
// boundaries (chunks shorter than a vector) is taken by its first entry
// only.  Each element is folded by its own thread, so a straddling vector
// costs one element's latency instead of L of them.
template <class E, int DIV, int CAP>
__device__ __forceinline__ void ring_edge_element(const RankTable<CAP>& t, int world, int64_t numel, int64_t clen,
                                                  int64_t q, float dop) {
    constexpr int L = E::L;
    const int64_t k = q / L;                   // boundary k + 1, or the last vector for k = world - 1
    const int64_t lane = q - k * L;
    // boundary k + 1 (at (k + 1) * clen) needs its vector taken when it is
    // inside the bucket and off the vector grid
    auto needs = [&](int64_t kk) {
        const int64_t b = (kk + 1) * clen;
        return b < numel && b % L != 0;
    };
    int64_t v;
    if (k < world - 1) {
        if (!needs(k)) return;
        v = (k + 1) * clen / L;
        if (k > 0 && needs(k - 1) && k * clen / L == v) return;      // taken by boundary k
    } else {
        if (numel % L == 0) return;
        v = numel / L;
        const int64_t kl = (numel + clen - 1) / clen - 2;           // last boundary inside the bucket
        if (kl >= 0 && needs(kl) && (kl + 1) * clen / L == v) return;
    }
    const int64_t e = v * L + lane;
    if (e < numel) ring_element<E, DIV, CAP>(t, world, e, clen, dop);
}

// Vectorised fused kernel: all rank buffers are 16-byte aligned.  The 16-byte
// vectors are cut into tiles of kThreads * U; block b takes tiles b, b + B,
// ... (B: the blocks that are not edge blocks).  Thread x of a tile takes its
// vectors x, x + kThreads, ..., x + (U - 1) * kThreads: their loads, G ranks
// at a time, are all in flight before the fold.  A large bucket is launched with one block per tile,
// so the block scheduler hands out small tiles in address order as SMs free
// up and the blocks in flight stream one compact window of every rank; a
// bucket that fits in L2 gets a few waves of blocks that loop over the tiles.
// A vector whose lanes fall in two chunks (only possible when c is not a
// multiple of the lane count) or runs past the end is done lane by lane, one
// lane per thread (ring_edge_element), by the launch's last edge_blocks
// blocks, which run beside the tiles.
// LOOP = false: the grid is one block per tile, plus the edge blocks.
template <class E, int DIV, int CAP, int G, int U, int MINB, bool LOOP>
__global__ void __launch_bounds__(kThreads, MINB)
k_ring_fused(const __grid_constant__ RankTable<CAP> t, int world, int64_t numel, int64_t clen, float dop,
             int edge_blocks) {
    using V = typename E::V;
    constexpr int L = E::L;
    constexpr int64_t kTile = (int64_t)kThreads * U;
    pdl_release();
    pdl_acquire();
    const int64_t nvec = (numel + L - 1) / L;
    const int64_t full = numel / L;
    const int64_t tiles = (nvec + kTile - 1) / kTile;
    auto at = [&](int r) -> const char* { return t.p[r]; };
    // the straddling and ragged vectors, one element per thread: by the last
    // edge_blocks blocks beside the tiles, or (edge_blocks < 0, under a CTA
    // cap) by every block before its tiles; the tiles' threads skip them
    if (edge_blocks < 0)
        for (int64_t q = (int64_t)blockIdx.x * kThreads + threadIdx.x; q < (int64_t)world * L;
             q += (int64_t)gridDim.x * kThreads)
            ring_edge_element<E, DIV, CAP>(t, world, numel, clen, q, dop);
    const int main_blocks = (int)gridDim.x - (edge_blocks > 0 ? edge_blocks : 0);
    if ((int)blockIdx.x >= main_blocks) {
        for (int64_t q = (int64_t)(blockIdx.x - main_blocks) * kThreads + threadIdx.x; q < (int64_t)world * L;
             q += (int64_t)edge_blocks * kThreads)
            ring_edge_element<E, DIV, CAP>(t, world, numel, clen, q, dop);
        return;
    }
    int64_t tile = blockIdx.x;
    int64_t vb = tile * kTile + threadIdx.x;
    if (vb >= nvec) return;
    // the chunk of this thread's first vector, advanced as the block moves on
    // to later tiles (chunk j ends at chunk_end; at most numel for the last)
    int64_t j = (vb * L) / clen;
    int64_t chunk_end = (j + 1) * clen;
    for (;;) {
        while (vb * L >= chunk_end) {
            ++j;
            chunk_end += clen;
        }
        const int64_t vl = vb + (U - 1) * kThreads;
        if (vl < full && vl * L + L <= chunk_end) {
            const int start = (j + 1 == world) ? 0 : (int)j + 1;
            V y[U];
            fold_ring_vecs<E, G, U>(at, world, start, vb * 16, (int64_t)kThreads * 16, y);
#pragma unroll
            for (int u = 0; u < U; ++u) y[u] = E::template vdiv<DIV>(y[u], dop);
            for (int r = 0; r < world; ++r) {
#pragma unroll
                for (int u = 0; u < U; ++u) st_stream<V>(t.p[world + r] + (vb + u * kThreads) * 16, y[u]);
            }
        } else {
            for (int u = 0; u < U; ++u) {
                const int64_t v = vb + (int64_t)u * kThreads;
                if (v >= nvec) break;
                const int64_t i = v * L;
                int64_t jv = j, end_v = chunk_end;
                while (i >= end_v) {
                    ++jv;
                    end_v += clen;
                }
                // whole vectors of this chunk; the others went to ring_edge_element
                if (U > 1 && v < full && i + L <= end_v) {     // U = 1: the fast path's test
                    const int start = (jv + 1 == world) ? 0 : (int)jv + 1;
                    V y = E::template vdiv<DIV>(fold_ring_vec<E, G>(at, world, start, v * 16), dop);
                    for (int r = 0; r < world; ++r) st_stream<V>(t.p[world + r] + v * 16, y);
                }
            }
        }
        // one tile per block, or the block's next tile
        if constexpr (!LOOP) {
            return;
        } else {
            tile += main_blocks;
            vb = tile * kTile + threadIdx.x;
            if (tile >= tiles || vb >= nvec) return;
        }
    }
}

// Group fused kernel, for buckets too small to fill the GPU with one thread
// per vector.  P lanes of a warp (a group) share one 16-byte vector: lane q
// loads the ranks at ring positions q, q + P, ... (position k is rank
// (start + k) mod N), and every lane of the group folds the N values in
// ring order, taking each from its owner lane by a warp shuffle -- the adds
// of k_ring_fused in the same order, on P times as many threads, each with
// ceil(N / P) = R loads in flight instead of N.  Vectors that straddle a
// chunk boundary or the end are done element-wise, one element per thread
// (ring_edge_element), by the launch's last edge_blocks blocks.
template <class E, int DIV, int CAP, int P, int R>
__global__ void __launch_bounds__(kThreads)
k_ring_fused_group(const __grid_constant__ RankTable<CAP> t, int world, int64_t numel, int64_t clen, float dop,
                   int edge_blocks) {
    using V = typename E::V;
    constexpr int L = E::L;
    pdl_release();
    pdl_acquire();
    constexpr int kGroups = 32 / P;                     // vectors per warp and pass
    const int lane = threadIdx.x & 31;
    const int q = lane & (P - 1);
    const int64_t nvec = (numel + L - 1) / L;
    const int64_t full = numel / L;
    if (edge_blocks < 0)                          // the edge elements (see k_ring_fused)
        for (int64_t qe = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; qe < (int64_t)world * L;
             qe += (int64_t)gridDim.x * blockDim.x)
            ring_edge_element<E, DIV, CAP>(t, world, numel, clen, qe, dop);
    const int main_blocks = (int)gridDim.x - (edge_blocks > 0 ? edge_blocks : 0);
    if ((int)blockIdx.x >= main_blocks) {
        for (int64_t qe = (int64_t)(blockIdx.x - main_blocks) * blockDim.x + threadIdx.x; qe < (int64_t)world * L;
             qe += (int64_t)edge_blocks * blockDim.x)
            ring_edge_element<E, DIV, CAP>(t, world, numel, clen, qe, dop);
        return;
    }
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)main_blocks * blockDim.x) >> 5;
    // the loop bounds are the same for every lane of a warp, so every lane
    // reaches every shuffle
    for (int64_t base = warp * kGroups; base < nvec; base += n_warps * kGroups) {
        const int64_t v = base + lane / P;
        const int64_t i = v * L;
        const bool valid = v < nvec;
        const int64_t j = valid ? i / clen : 0;
        const bool clean = valid && v < full && (i + L - 1) / clen == j;
        const int start = (j + 1 == world) ? 0 : (int)j + 1;
        const int64_t off = v * 16;
        V x[R];
#pragma unroll
        for (int m = 0; m < R; ++m) {
            const int k = m * P + q;
            x[m] = make_zero<V>();
            if (clean && k < world) {
                const int r = (start + k >= world) ? start + k - world : start + k;
                x[m] = ld_stream<V>(t.p[r] + off);
            }
        }
        V acc = shfl_vec(x[0], 0, P);
#pragma unroll
        for (int m = 0; m < R; ++m) {
#pragma unroll
            for (int qq = 0; qq < P; ++qq) {
                const int k = m * P + qq;
                if (k > 0 && k < world) acc = E::vadd(acc, shfl_vec(x[m], qq, P));
            }
        }
        if (clean) {
            const V y = E::template vdiv<DIV>(acc, dop);
#pragma unroll
            for (int m = 0; m < R; ++m) {
                const int k = m * P + q;
                if (k < world) {
                    const int r = (start + k >= world) ? start + k - world : start + k;
                    st_stream<V>(t.p[world + r] + off, y);
                }
            }
        }       // vectors that straddle a chunk boundary or the end: ring_edge_element, above
    }
}

// Element-wise fused kernel for buffers that are not 16-byte aligned.
template <class E, int DIV, int CAP>
__global__ void __launch_bounds__(kThreads)
k_ring_fused_scalar(const __grid_constant__ RankTable<CAP> t, int world, int64_t numel, int64_t clen, float dop) {
    pdl_release();
    pdl_acquire();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < numel; e += stride)
        ring_element<E, DIV, CAP>(t, world, e, clen, dop);
}

// ---------------------------------------------------------------------------
// Staged ring: one launch per step
// ---------------------------------------------------------------------------

// Ring step `s` of phase `phase` (0 = reduce-scatter, 1 = all-gather) for all
// ranks at once; blockIdx.y is the receiving rank r, its left neighbour r-1
// is the sender.
//   reduce-scatter: chunk (r-s-1) mod N of rank r += the same chunk of rank r-1
//   all-gather:     chunk (r-s)   mod N of rank r  = the same chunk of rank r-1
// In one step rank r writes chunk q while its right neighbour reads chunk q+1
// of rank r, so no element is both read and written by different ranks within
// a step; consecutive steps are ordered by the stream.  DIV is applied only
// in the last reduce-scatter step, by the chunk's owner, before the chunk is
// circulated by the all-gather.
template <class E, int DIV, int CAP>
__global__ void __launch_bounds__(kThreads)
k_ring_hop(const __grid_constant__ RankTable<CAP> t, int world, int64_t numel, int64_t clen, int phase, int s,
           int vec_ok, float dop) {
    using V = typename E::V;
    using S = typename E::S;
    constexpr int L = E::L;
    const int r = blockIdx.y;
    const int left = (r == 0) ? world - 1 : r - 1;
    int c = (phase == 0) ? (r - s - 1) : (r - s);
    c %= world;
    if (c < 0) c += world;
    const int64_t lo = std::min((int64_t)c * clen, numel);
    const int64_t hi = std::min(lo + clen, numel);
    // programmatic dependent launch: the next hop may be scheduled now, and
    // no buffer is touched before the previous hop (or whatever preceded
    // this kernel on the stream) has completed and its writes are visible
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (lo >= hi) return;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    char* dst = t.p[r];
    const char* src = t.p[left];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (vec_ok) {
        for (int64_t q = lo / L + tid; q * L < hi; q += stride) {
            const int64_t i = q * L;
            if (i >= lo && i + L <= hi) {
                V m = ld_stream<V>(src + q * 16);
                if (phase == 0) {
                    V d = ld_stream<V>(dst + q * 16);
                    m = E::template vdiv<DIV>(E::vadd(d, m), dop);
                }
                st_stream<V>(dst + q * 16, m);
            } else {
                for (int l = 0; l < L; ++l) {
                    const int64_t e = i + l;
                    if (e < lo || e >= hi) continue;
                    S m = reinterpret_cast<const S*>(src)[e];
                    if (phase == 0) m = E::template sdiv<DIV>(E::sadd(reinterpret_cast<S*>(dst)[e], m), dop);
                    reinterpret_cast<S*>(dst)[e] = m;
                }
            }
        }
    } else {
        for (int64_t e = lo + tid; e < hi; e += stride) {
            S m = reinterpret_cast<const S*>(src)[e];
            if (phase == 0) m = E::template sdiv<DIV>(E::sadd(reinterpret_cast<S*>(dst)[e], m), dop);
            reinterpret_cast<S*>(dst)[e] = m;
        }
    }
}

// ---------------------------------------------------------------------------
// Local accumulation (no_sync micro-batches)
// ---------------------------------------------------------------------------

template <class E, int CAP>
__global__ void __launch_bounds__(kThreads)
k_accumulate(const __grid_constant__ RankTable<CAP> acc, const __grid_constant__ RankTable<CAP> g, int64_t numel,
             int vec_ok) {
    using V = typename E::V;
    using S = typename E::S;
    constexpr int L = E::L;
    pdl_release();
    pdl_acquire();
    const int r = blockIdx.y;
    char* a = acc.p[r];
    const char* b = g.p[r];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t done = 0;
    if (vec_ok) {
        const int64_t nv = numel / L;
        for (int64_t q = tid; q < nv; q += stride)
            st_stream<V>(a + q * 16, E::vadd(ld_stream<V>(a + q * 16), ld_stream<V>(b + q * 16)));
        done = nv * L;
    }
    for (int64_t e = done + tid; e < numel; e += stride)
        reinterpret_cast<S*>(a)[e] = E::sadd(reinterpret_cast<S*>(a)[e], reinterpret_cast<const S*>(b)[e]);
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------

template <int CAP>
static RankTable<CAP> make_table(int world, void* const* ptrs) {
    RankTable<CAP> t{};
    for (int r = 0; r < world; ++r) t.p[r] = static_cast<char*>(ptrs[r]);
    return t;
}

// in + out pointer table of 2 * world entries (see the fused kernels)
template <int CAP>
static RankTable<CAP> make_io_table(int world, void* const* in, void* const* out) {
    RankTable<CAP> t{};
    for (int r = 0; r < world; ++r) {
        t.p[r] = static_cast<char*>(in[r]);
        t.p[world + r] = static_cast<char*>(out[r]);
    }
    return t;
}

// Blocks for the elements of straddling and ragged vectors (ring_edge_element)
// added to a launch of `grid` blocks: none when every chunk boundary and the
// end fall on the 16-byte grid; -1 (every block takes its share first) when
// the extra blocks would exceed the CTA cap.
static int edge_blocks_for(int world, int64_t numel, int lanes, int threads, int64_t grid) {
    const bool edges = numel % lanes != 0 || (world > 1 && chunk_len(numel, world) % lanes != 0);
    if (!edges) return 0;
    const int eb = (int)(((int64_t)world * lanes + threads - 1) / threads);
    const int cap = cta_cap();
    if ((cap > 0 && grid + eb > cap) || grid + eb > INT32_MAX) return -1;
    return eb;
}

// Buckets that do not fit in L2 run one block per tile (see k_ring_fused).
constexpr int64_t kTilePerBlockBytes = 128ll << 20;

template <class E, int DIV, int CAP, int G, int U, int MINB, int LOOP_U = U>
static cudaError_t fused_vec(int world, void* const* in, void* const* out, int64_t numel, float dop,
                             cudaStream_t st) {
    const int64_t nvec = (numel + E::L - 1) / E::L;
    const int64_t tiles = (nvec + (int64_t)kThreads * U - 1) / ((int64_t)kThreads * U);
    const bool streamed = (int64_t)world * numel * (int64_t)sizeof(typename E::S) >= kTilePerBlockBytes;
    int grid = 0;
    cudaError_t e;
    if (streamed && tiles <= INT32_MAX - 64 && cap_ctas(tiles) == tiles) {
        const int eb = edge_blocks_for(world, numel, E::L, kThreads, tiles);
        grid = (int)tiles + std::max(eb, 0);
        e = launch_dependent(k_ring_fused<E, DIV, 2 * CAP, G, U, MINB, false>, dim3(grid), dim3(kThreads), 0, st,
                             make_io_table<2 * CAP>(world, in, out), world, numel, chunk_len(numel, world), dop, eb);
    } else {
        // the looping form at 4 blocks per SM too (64 registers), except the
        // IEEE-division fold of 8 ranks, which needs a few more
        constexpr int kLoopMinb = (DIV == kDivIeee && G == 8) ? 3 : 4;
        auto loop = k_ring_fused<E, DIV, 2 * CAP, G, LOOP_U, kLoopMinb, true>;
        const int64_t loop_tiles = (nvec + (int64_t)kThreads * LOOP_U - 1) / ((int64_t)kThreads * LOOP_U);
        grid = streamed ? cap_ctas(std::min<int64_t>(loop_tiles, INT32_MAX - 64))
                        : grid_for((const void*)loop, loop_tiles * kThreads);
        const int eb = edge_blocks_for(world, numel, E::L, kThreads, grid);
        grid += std::max(eb, 0);
        e = launch_dependent(loop, dim3(grid), dim3(kThreads), 0, st, make_io_table<2 * CAP>(world, in, out), world,
                             numel, chunk_len(numel, world), dop, eb);
    }
    if (debug_enabled())
        fprintf(stderr, "[ddp] ring_fused world=%d numel=%lld grid=%d tiles=%lld G=%d U=%d CAP=%d\n", world,
                (long long)numel, grid, (long long)tiles, G, U, CAP);
    return e;
}

constexpr int kGroupThreads = 128;     // small blocks spread a small bucket over more SMs

template <class E, int DIV, int CAP, int P, int R>
static cudaError_t fused_group(int world, void* const* in, void* const* out, int64_t numel, float dop,
                               cudaStream_t st) {
    auto k = k_ring_fused_group<E, DIV, 2 * CAP, P, R>;
    const int64_t nvec = (numel + E::L - 1) / E::L;
    const int64_t lanes = (nvec + 32 / P - 1) / (32 / P) * 32;
    int grid = grid_for((const void*)k, lanes, kGroupThreads);
    const int eb = edge_blocks_for(world, numel, E::L, kGroupThreads, grid);
    grid += std::max(eb, 0);
    const cudaError_t e = launch_dependent(k, dim3(grid), dim3(kGroupThreads), 0, st,
                                           make_io_table<2 * CAP>(world, in, out), world, numel,
                                           chunk_len(numel, world), dop, eb);
    if (debug_enabled())
        fprintf(stderr, "[ddp] ring_fused_group world=%d numel=%lld grid=%d P=%d R=%d\n", world, (long long)numel,
                grid, P, R);
    return e;
}

template <class E, int DIV>
static cudaError_t group_dispatch(int world, void* const* in, void* const* out, int64_t numel, float dop,
                                  cudaStream_t st) {
    if (world <= 2) return fused_group<E, DIV, 16, 2, 1>(world, in, out, numel, dop, st);
    if (world <= 4) return fused_group<E, DIV, 16, 4, 1>(world, in, out, numel, dop, st);
    if (world <= 8) return fused_group<E, DIV, 16, 8, 1>(world, in, out, numel, dop, st);
    if (world <= 16) return fused_group<E, DIV, 16, 16, 1>(world, in, out, numel, dop, st);
    if (world <= 32) return fused_group<E, DIV, 64, 32, 1>(world, in, out, numel, dop, st);
    if (world <= 64) return fused_group<E, DIV, 64, 32, 2>(world, in, out, numel, dop, st);
    return fused_group<E, DIV, kGroupMaxWorld, 32, 4>(world, in, out, numel, dop, st);
}

template <class E, int DIV, int CAP>
static cudaError_t fused_scalar(int world, void* const* in, void* const* out, int64_t numel, float dop,
                                cudaStream_t st) {
    auto k = k_ring_fused_scalar<E, DIV, 2 * CAP>;
    const int grid = grid_for((const void*)k, numel);
    return launch_dependent(k, dim3(grid), dim3(kThreads), 0, st, make_io_table<2 * CAP>(world, in, out), world,
                            numel, chunk_len(numel, world), dop);
}

template <class E, int DIV>
static cudaError_t fused_dispatch(FusedPath path, int world, void* const* in, void* const* out, int64_t numel,
                                  float dop, cudaStream_t st) {
    if (path == FusedPath::kScalar) {
        if (world <= 16) return fused_scalar<E, DIV, 16>(world, in, out, numel, dop, st);
        return fused_scalar<E, DIV, DDP_MAX_WORLD>(world, in, out, numel, dop, st);
    }
    if (path == FusedPath::kGroup) return group_dispatch<E, DIV>(world, in, out, numel, dop, st);
    // G ranks' loads at a time, U vectors per thread, at least MINB blocks
    // per SM in the one-tile form (64 registers a thread at 4), LOOP_U in the
    // looping form: 4 to 8 loads in flight per thread in the one-tile form
    // (3 ranks: two vectors there, one in the looping form)
    if (world <= 2) return fused_vec<E, DIV, 16, 2, 2, 4>(world, in, out, numel, dop, st);
    if (world == 3) return fused_vec<E, DIV, 16, 4, 2, 4, 1>(world, in, out, numel, dop, st);
    if (world <= 4) return fused_vec<E, DIV, 16, 4, 1, 4>(world, in, out, numel, dop, st);
    if (world <= 8) return fused_vec<E, DIV, 16, 8, 1, 4>(world, in, out, numel, dop, st);
    if (world <= 16) return fused_vec<E, DIV, 16, 8, 1, 3>(world, in, out, numel, dop, st);
    if (world <= 64) return fused_vec<E, DIV, 64, 8, 1, 3>(world, in, out, numel, dop, st);
    return fused_vec<E, DIV, DDP_MAX_WORLD, 8, 1, 3>(world, in, out, numel, dop, st);
}

template <class E>
static cudaError_t fused_by_div(FusedPath path, int world, void* const* in, void* const* out, int64_t numel,
                                DivSpec d, cudaStream_t st) {
    switch (d.mode) {
        case kDivNone: return fused_dispatch<E, kDivNone>(path, world, in, out, numel, d.operand, st);
        case kDivPow2: return fused_dispatch<E, kDivPow2>(path, world, in, out, numel, d.operand, st);
        default: return fused_dispatch<E, kDivIeee>(path, world, in, out, numel, d.operand, st);
    }
}

FusedPath choose_fused_path(int world, int64_t numel, int dtype, bool vec_ok) {
    if (!vec_ok) return FusedPath::kScalar;
    const bool tma_ok = tma_usable(world, numel, dtype, vec_ok);
    const bool group_ok = world >= 2 && world <= kGroupMaxWorld;
    switch (fused_kernel_override()) {
        case DDP_FUSED_VECTOR: return FusedPath::kVector;
        case DDP_FUSED_GROUP: return group_ok ? FusedPath::kGroup : FusedPath::kVector;
        case DDP_FUSED_TMA: return tma_ok ? FusedPath::kTma : FusedPath::kVector;
        default: break;
    }
    // Crossovers measured on GB300 with every kernel forced (CUDA-graph
    // replay of back-to-back calls, fp32 and bf16, N = 2 .. 128, 16 KiB ..
    // 256 MiB per rank):
    //  * a few KiB per rank: the group kernel spreads the ranks over lanes;
    //    it stays ahead up to 256 KiB at 2 ranks, and up to 16 KiB at 8 fp32
    //    ranks and wherever fp32 chunk boundaries are not 16-byte aligned
    //    (N = 3, 5, 6, 7, 12, 24 on these sizes);
    //  * many ranks with little data each: the TMA kernel's one CTA per
    //    tile reaches more SMs (N >= 16 up to 16 KiB, N >= 32 up to 1 MiB,
    //    N >= 64 up to 256 KiB, N >= 128 up to 64 KiB; fp32 at 16-31 ranks
    //    from 256 KiB to 4 MiB);
    //  * everything else, and every large bucket: the vector kernel, whose
    //    one block per tile streams at or above the measured copy rate --
    //    except under a CTA budget of less than four blocks per SM, where
    //    buckets from 1 MiB per rank go to the TMA kernel.
    constexpr int64_t KiB = 1024, MiB = 1024 * 1024;
    const int64_t per_rank = numel * elem_bytes(dtype);
    const bool chunks_aligned = (chunk_len(numel, world) * elem_bytes(dtype)) % 16 == 0;
    if (group_ok && (per_rank <= 4 * KiB || (world == 2 && per_rank <= 256 * KiB) ||
                     (dtype == DDP_F32 && per_rank <= 16 * KiB && (world == 8 || !chunks_aligned))))
        return FusedPath::kGroup;
    if (tma_ok) {
        // a CTA budget below four blocks per SM: the TMA kernel keeps more
        // bytes in flight per CTA than the vector kernel's 256-thread blocks
        if (cta_cap_is_tight() && per_rank >= 1 * MiB) return FusedPath::kTma;
        if (world >= 16 && per_rank <= 16 * KiB) return FusedPath::kTma;
        if (world >= 128) {
            if (per_rank <= 64 * KiB) return FusedPath::kTma;
        } else if (world >= 64) {
            if (per_rank <= 256 * KiB) return FusedPath::kTma;
        } else if (world >= 32) {
            if (per_rank <= 1 * MiB) return FusedPath::kTma;
        } else if (world >= 16) {
            if (dtype == DDP_F32 && per_rank >= 256 * KiB && per_rank <= 4 * MiB) return FusedPath::kTma;
        }
    }
    return FusedPath::kVector;
}

cudaError_t launch_ring_fused(int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div, bool vec_ok,
                              cudaStream_t stream) {
    if (numel == 0) return cudaSuccess;
    const FusedPath path = choose_fused_path(world, numel, dtype, vec_ok);
    if (path == FusedPath::kTma) return launch_ring_fused_tma(world, ptrs, numel, dtype, div, stream);
    if (dtype == DDP_F32) return fused_by_div<EF32>(path, world, ptrs, ptrs, numel, div, stream);
    return fused_by_div<EBF16>(path, world, ptrs, ptrs, numel, div, stream);
}

cudaError_t launch_ring_fused_io(int world, void* const* in, void* const* out, int64_t numel, int dtype, DivSpec div,
                                 bool vec_ok, cudaStream_t stream) {
    if (numel == 0) return cudaSuccess;
    const FusedPath path = vec_ok ? FusedPath::kVector : FusedPath::kScalar;
    if (dtype == DDP_F32) return fused_by_div<EF32>(path, world, in, out, numel, div, stream);
    return fused_by_div<EBF16>(path, world, in, out, numel, div, stream);
}

template <class E, int DIV, int CAP>
static cudaError_t hop(const RankTable<CAP>& t, int world, int64_t numel, int phase, int s, bool vec_ok, float dop,
                       cudaStream_t st) {
    auto k = k_ring_hop<E, DIV, CAP>;
    const int64_t clen = chunk_len(numel, world);
    const int64_t per_rank = vec_ok ? (clen + E::L - 1) / E::L + 1 : clen;
    // blocks in x per rank: enough to fill the GPU once all ranks are counted
    // (one block per tile measured no faster here: a hop's chunk is read
    // back from L2 by the next hop, and the all-gather copies got slower)
    const int gx = rows_grid_x((const void*)k, per_rank, world, 0);
    // hops are launched as programmatic dependents of the previous kernel on
    // the stream: each one's launch overlaps the previous hop's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, world);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, t, world, numel, clen, phase, s, vec_ok ? 1 : 0, dop);
}

template <class E, int DIV, int CAP>
static cudaError_t staged_impl(int world, void* const* ptrs, int64_t numel, float dop, bool vec_ok, cudaStream_t st) {
    const RankTable<CAP> t = make_table<CAP>(world, ptrs);
    for (int s = 1; s <= world - 1; ++s) {
        cudaError_t e = (s == world - 1) ? hop<E, DIV, CAP>(t, world, numel, 0, s, vec_ok, dop, st)
                                         : hop<E, kDivNone, CAP>(t, world, numel, 0, s, vec_ok, dop, st);
        if (e != cudaSuccess) return e;
    }
    for (int s = 1; s <= world - 1; ++s) {
        cudaError_t e = hop<E, kDivNone, CAP>(t, world, numel, 1, s, vec_ok, dop, st);
        if (e != cudaSuccess) return e;
    }
    if (debug_enabled())
        fprintf(stderr, "[ddp] ring_staged world=%d numel=%lld launches=%d\n", world, (long long)numel,
                2 * (world - 1));
    return cudaSuccess;
}

template <class E, int DIV>
static cudaError_t staged_cap(int world, void* const* ptrs, int64_t numel, float dop, bool vec_ok, cudaStream_t st) {
    if (world <= 16) return staged_impl<E, DIV, 16>(world, ptrs, numel, dop, vec_ok, st);
    return staged_impl<E, DIV, DDP_MAX_WORLD>(world, ptrs, numel, dop, vec_ok, st);
}

template <class E>
static cudaError_t staged_by_div(int world, void* const* ptrs, int64_t numel, DivSpec d, bool vec_ok,
                                 cudaStream_t st) {
    switch (d.mode) {
        case kDivNone: return staged_cap<E, kDivNone>(world, ptrs, numel, d.operand, vec_ok, st);
        case kDivPow2: return staged_cap<E, kDivPow2>(world, ptrs, numel, d.operand, vec_ok, st);
        default: return staged_cap<E, kDivIeee>(world, ptrs, numel, d.operand, vec_ok, st);
    }
}

cudaError_t launch_ring_staged(int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div, bool vec_ok,
                               cudaStream_t stream) {
    if (numel == 0) return cudaSuccess;
    // One rank: there is no ring step, only the average.
    if (world == 1) return launch_ring_fused(world, ptrs, numel, dtype, div, vec_ok, stream);
    if (dtype == DDP_F32) return staged_by_div<EF32>(world, ptrs, numel, div, vec_ok, stream);
    return staged_by_div<EBF16>(world, ptrs, numel, div, vec_ok, stream);
}

template <class E, int CAP>
static cudaError_t accumulate_impl(int world, void* const* acc, const void* const* g, int64_t numel, bool vec_ok,
                                   cudaStream_t st) {
    auto k = k_accumulate<E, CAP>;
    RankTable<CAP> ta{}, tg{};
    for (int r = 0; r < world; ++r) {
        ta.p[r] = static_cast<char*>(acc[r]);
        tg.p[r] = static_cast<char*>(const_cast<void*>(g[r]));
    }
    const int64_t per_rank = vec_ok ? numel / E::L + E::L : numel;
    // 128 MiB or more of accumulators (vectorised): one block per kThreads
    // vectors of a rank; else a few waves of blocks striding over each rank
    const int64_t bytes = vec_ok ? (int64_t)world * numel * (int64_t)sizeof(typename E::S) : 0;
    const int gx = rows_grid_x((const void*)k, per_rank, world, bytes);
    return launch_dependent(k, dim3(gx, world), dim3(kThreads), 0, st, ta, tg, numel, vec_ok ? 1 : 0);
}

cudaError_t launch_accumulate(int world, void* const* acc, const void* const* g, int64_t numel, int dtype,
                              bool vec_ok, cudaStream_t stream) {
    if (numel == 0) return cudaSuccess;
    if (dtype == DDP_F32) {
        if (world <= 16) return accumulate_impl<EF32, 16>(world, acc, g, numel, vec_ok, stream);
        return accumulate_impl<EF32, DDP_MAX_WORLD>(world, acc, g, numel, vec_ok, stream);
    }
    if (world <= 16) return accumulate_impl<EBF16, 16>(world, acc, g, numel, vec_ok, stream);
    return accumulate_impl<EBF16, DDP_MAX_WORLD>(world, acc, g, numel, vec_ok, stream);
}

}  // namespace ddpk
