// ring_tma.cu -- fused ring allreduce with TMA bulk copies into shared memory.
//
// Same result as k_ring_fused (ring_kernels.cu): element i of chunk j is
// folded over the ranks starting at rank j+1 ("DDP 与 Ring-AllReduce", §1.3.2;
// "DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事", section 03),
// divided by the divisor and written to every rank.  What differs is how the
// bytes move.  The bucket is cut into tiles that never cross a chunk
// boundary; one resident CTA per SM (four waves of them for launches that
// stream more than 512 MiB) walks its tiles through a ring of shared-memory
// stages, with its warps split by role:
//   * a producer warp: one thread issues, for every tile, N bulk copies
//     (cp.async.bulk, one per rank) that complete on the stage's "full"
//     mbarrier, as soon as the consumers have released that stage;
//   * eight consumer warps: wait for a full stage, fold the N staged copies
//     in ring order, release the stage on its "empty" mbarrier, and store the
//     result vector from registers to every rank.
// No CTA-wide barrier sits in the loop: the producer refills a stage the
// moment the last consumer warp has read it, which keeps the copy engine's
// queue full.
//
// Waits are bounded: an mbarrier wait that exceeds the wait limit (2 s
// unless ddp_set_wait_limit_ms says otherwise) sets the library's device
// status word to DDP_ERR_TIMEOUT and the thread stops; the producer then
// waits (again bounded) for the copies it issued before it returns.
//
// A planted stall (ddp_plant_stall) makes the producer of the CTA that owns
// one chosen tile stop before that tile: it issues no copy for it or for any
// later tile, and waits for the copies it did issue to be consumed.  The
// consumers then wait for a tile that never arrives -- what a ring step
// looks like when one rank never joins it -- until the limit runs out.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "ddp_device.cuh"
#include "ddp_internal.h"
#include "view_batch.cuh"

namespace ddpk {

__device__ int32_t g_device_status = 0;     // sticky DDP_ERR_TIMEOUT flag, read by ddp_device_status()

constexpr int kTmaStages = 2;
constexpr int kTmaConsumerWarps = 8;
constexpr int kTmaThreads = 32 * (kTmaConsumerWarps + 1);    // + one producer warp
constexpr int kTmaMaxVec = 4;        // 16-byte vectors per consumer thread per tile (tile <= 16 KB)

// Per-launch control: the wait limit, and the tile whose copies are never
// issued (-1: none).
struct TmaCtl {
    unsigned long long limit_ns;
    long long stall_tile;
};

template <int CAP>
struct TmaTable {
    char* p[CAP];
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t tx_bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(tx_bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until the barrier's phase with this parity has completed, at most
// limit_ns; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// Bulk copy global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Tiles never cross a chunk boundary: chunk j (length clen, the last one
// shorter) holds ceil(len / tile) tiles; empty trailing chunks hold none.
// Tile k is tile q = k mod per_chunk of chunk j = k / per_chunk (the last
// chunk's tiles are a prefix of that numbering).
struct TileMap {
    int64_t numel, clen, tile, per_chunk, last_chunk, total;
    __host__ __device__ void init(int64_t n, int64_t c, int64_t t) {
        numel = n;
        clen = c;
        tile = t;
        per_chunk = (c + t - 1) / t;
        last_chunk = (n - 1) / c;
        const int64_t last_len = n - last_chunk * c;
        total = last_chunk * per_chunk + (last_len + t - 1) / t;
    }
};

// A CTA visits tiles k, k + G, k + 2G, ... (G = gridDim.x).  The cursor keeps
// (j, q) for its current tile and advances by G with adds and one compare:
// integer division on this path measurably delayed the refills.
struct TileCursor {
    int64_t k, j, q;          // tile index, its chunk, its tile within the chunk
    int64_t step_j, step_q;   // G / per_chunk, G % per_chunk
    __device__ void start(const TileMap& m, int64_t k0, int64_t g) {
        k = k0;
        j = k0 / m.per_chunk;
        q = k0 - j * m.per_chunk;
        step_j = g / m.per_chunk;
        step_q = g - step_j * m.per_chunk;
    }
    __device__ void advance(const TileMap& m, int64_t g) {
        k += g;
        j += step_j;
        q += step_q;
        if (q >= m.per_chunk) {
            q -= m.per_chunk;
            ++j;
        }
    }
    // first element and length of the current tile
    __device__ void range(const TileMap& m, int64_t& e0, int64_t& n) const {
        const int64_t cs = j * m.clen;
        const int64_t ce = (cs + m.clen < m.numel) ? cs + m.clen : m.numel;
        e0 = cs + q * m.tile;
        n = (ce - e0 < m.tile) ? ce - e0 : m.tile;
    }
};

// The body of both TMA-staged fused allreduces.  TREE = false: the ring's
// fold, element i of chunk j summed from rank j + 1 round to rank j; TREE =
// true: the binomial tree's pairwise fold of ranks 0 .. N - 1, the same for
// every element (the bucket is then one "chunk", tiles cut anywhere).
template <class E, int DIV, int CAP, bool TREE>
__device__ __forceinline__ void fused_tma_body(const TmaTable<CAP>& t, int world, const TileMap& map, float dop,
                                               const TmaCtl& ctl) {
    using V = typename E::V;
    using S = typename E::S;
    constexpr int L = E::L;
    constexpr int kConsumers = 32 * kTmaConsumerWarps;
    extern __shared__ __align__(128) unsigned char smem[];
    const int64_t tile_bytes = map.tile * (int64_t)sizeof(S);
    unsigned char* stages = smem;                                                    // [stages][world][tile]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kTmaStages * world * tile_bytes);
    uint64_t* empty = full + kTmaStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    pdl_release();
    pdl_acquire();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTmaStages; ++s) {
            mbar_init(&full[s], 1);                     // the producer's expect_tx arrival + bytes
            mbar_init(&empty[s], kTmaConsumerWarps);    // one arrival per consumer warp
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kTmaConsumerWarps) {
        // ---- producer ----
        if (lane != 0) return;
        TileCursor ic;
        ic.start(map, blockIdx.x, G);
        int it = 0;
        for (; ic.k < map.total; ic.advance(map, G), ++it) {
            if (ic.k == ctl.stall_tile) break;          // planted stall: nothing more is issued
            const int s = it % kTmaStages;
            // the stage's previous tile (it - kTmaStages) must have been read
            if (it >= kTmaStages &&
                !mbar_wait_bounded(&empty[s], (uint32_t)(it / kTmaStages - 1) & 1u, ctl.limit_ns)) {
                atomicExch(&g_device_status, (int32_t)DDP_ERR_TIMEOUT);
                break;
            }
            int64_t e0, n;
            ic.range(map, e0, n);
            const uint32_t bytes = (uint32_t)(n * (int64_t)sizeof(S));
            mbar_arrive_expect_tx(&full[s], bytes * (uint32_t)world);
            unsigned char* dst = stages + (size_t)s * world * tile_bytes;
            for (int r = 0; r < world; ++r)
                bulk_load(dst + (size_t)r * tile_bytes, t.p[r] + e0 * (int64_t)sizeof(S), bytes, &full[s]);
        }
        // do not leave while copies into this CTA's shared memory may still
        // be landing: wait until the consumers have drained the last stages
        for (int q = 1; q <= kTmaStages && it - q >= 0; ++q) {
            const int i2 = it - q;
            mbar_wait_bounded(&empty[i2 % kTmaStages], (uint32_t)(i2 / kTmaStages) & 1u, ctl.limit_ns);
        }
        return;
    }

    // ---- consumers ----
    TileCursor cc;
    cc.start(map, blockIdx.x, G);
    for (int it = 0; cc.k < map.total; cc.advance(map, G), ++it) {
        const int s = it % kTmaStages;
        int64_t e0, n;
        cc.range(map, e0, n);
        const int j = (int)cc.j;
        if (!mbar_wait_bounded(&full[s], (uint32_t)(it / kTmaStages) & 1u, ctl.limit_ns)) {
            atomicExch(&g_device_status, (int32_t)DDP_ERR_TIMEOUT);
            break;
        }
        const int start = (j + 1 == world) ? 0 : j + 1;
        const int nv = (int)(n / L);
        const unsigned char* sb = stages + (size_t)s * world * tile_bytes;
        V y[kTmaMaxVec];
#pragma unroll
        for (int u = 0; u < kTmaMaxVec; ++u) {
            const int v = threadIdx.x + u * kConsumers;
            if (v < nv) {
                auto staged = [&](int r) { return reinterpret_cast<const V*>(sb + (size_t)r * tile_bytes)[v]; };
                V acc;
                if constexpr (TREE) {
                    acc = tree_fold<V, CAP>(world, [](V a, V b) { return E::vadd(a, b); }, staged);
                } else {
                    int r = start;
                    acc = staged(r);
                    for (int q = 1; q < world; ++q) {
                        r = (r + 1 == world) ? 0 : r + 1;
                        acc = E::vadd(acc, staged(r));
                    }
                }
                y[u] = E::template vdiv<DIV>(acc, dop);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);      // this warp has read stage s
#pragma unroll
        for (int u = 0; u < kTmaMaxVec; ++u) {
            const int v = threadIdx.x + u * kConsumers;
            if (v < nv)
                for (int r = 0; r < world; ++r)
                    st_stream<V>(t.p[r] + e0 * (int64_t)sizeof(S) + (int64_t)v * 16, y[u]);
        }
    }
}

template <class E, int DIV, int CAP>
__global__ void __launch_bounds__(kTmaThreads, 1)
k_ring_fused_tma(const __grid_constant__ TmaTable<CAP> t, int world, TileMap map, float dop, TmaCtl ctl) {
    fused_tma_body<E, DIV, CAP, false>(t, world, map, dop, ctl);
}

// The fused binomial-tree allreduce (tree_kernels.cu's k_tree_fused) staged
// the same way: same bytes moved, the tree's additions in the tree's order.
template <class E, int DIV, int CAP>
__global__ void __launch_bounds__(kTmaThreads, 1)
k_tree_fused_tma(const __grid_constant__ TmaTable<CAP> t, int world, TileMap map, float dop, TmaCtl ctl) {
    fused_tma_body<E, DIV, CAP, true>(t, world, map, dop, ctl);
}

// ---------------------------------------------------------------------------
// The fused view path (pack + ring + average + unpack of one bucket) with the
// same producer / consumer structure.  The host cuts every member of the
// bucket at the bucket's chunk boundaries into segments; a segment has one
// ring start rank, and tiles are cut inside segments, so a tile never crosses
// a chunk.  Tiles are numbered segment after segment; each CTA walks its
// tiles k, k + G, ... and finds their segment by scanning forward.
//
// What a segment's 16-byte-aligned body leaves at a chunk boundary that is
// not 16-byte aligned -- a few elements on each side, an "edge" -- is folded
// element by element by the consumer warps of the same launch before they
// start on their tiles (edge e by CTA e mod G, one element per thread), with
// plain loads and stores.  An edge's elements share no 16-byte word with any
// body, so the two kinds of store never touch the same bytes.  The table
// (ViewSegBatch) is in view_batch.cuh; bucket_kernels.cu's register view
// kernel reads the same one.
// ---------------------------------------------------------------------------

static_assert(kViewEdgeMax == 32 * kTmaConsumerWarps, "an edge has one element per consumer thread");

struct SegCursor {
    int seg;
    template <class B>
    __device__ void seek(const B& b, int64_t k) {
        while (b.tile_end[seg] <= k) ++seg;
    }
    template <class B>
    __device__ void range(const B& b, int64_t k, int64_t& e0, int64_t& n) const {
        const int64_t first = seg ? b.tile_end[seg - 1] : 0;
        const int64_t off = (k - first) * b.tile;
        e0 = b.start[seg] + off;
        const int64_t len = b.len[seg];
        n = (len - off < b.tile) ? len - off : b.tile;
    }
};

template <class E, int DIV, class B, int ST>
__global__ void __launch_bounds__(kTmaThreads, 1)
k_bucket_view_tma(const __grid_constant__ B b, float dop, TmaCtl ctl) {
    using V = typename E::V;
    using S = typename E::S;
    constexpr int L = E::L;
    constexpr int kConsumers = 32 * kTmaConsumerWarps;
    extern __shared__ __align__(128) unsigned char smem[];
    const int world = b.world;
    const int64_t tile_bytes = b.tile * (int64_t)sizeof(S);
    unsigned char* stages = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)ST * world * tile_bytes);
    uint64_t* empty = full + ST;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    const int64_t total = b.n_seg > 0 ? b.tile_end[b.n_seg - 1] : 0;
    pdl_release();
    pdl_acquire();

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kTmaConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kTmaConsumerWarps) {
        if (lane != 0) return;
        SegCursor sc{0};
        int it = 0;
        for (int64_t k = blockIdx.x; k < total; k += G, ++it) {
            if (k == ctl.stall_tile) break;             // planted stall: nothing more is issued
            const int s = it % ST;
            if (it >= ST &&
                !mbar_wait_bounded(&empty[s], (uint32_t)(it / ST - 1) & 1u, ctl.limit_ns)) {
                atomicExch(&g_device_status, (int32_t)DDP_ERR_TIMEOUT);
                break;
            }
            sc.seek(b, k);
            int64_t e0, n;
            sc.range(b, k, e0, n);
            const uint32_t bytes = (uint32_t)(n * (int64_t)sizeof(S));
            mbar_arrive_expect_tx(&full[s], bytes * (uint32_t)world);
            unsigned char* dst = stages + (size_t)s * world * tile_bytes;
            char* const* pp = b.ptr + (size_t)b.mem[sc.seg] * world;
            for (int r = 0; r < world; ++r)
                bulk_load(dst + (size_t)r * tile_bytes, pp[r] + e0 * (int64_t)sizeof(S), bytes, &full[s]);
        }
        for (int q = 1; q <= ST && it - q >= 0; ++q) {
            const int i2 = it - q;
            mbar_wait_bounded(&empty[i2 % ST], (uint32_t)(i2 / ST) & 1u, ctl.limit_ns);
        }
        return;
    }

    // edges first: the first stages are still landing meanwhile
    for (int e = blockIdx.x; e < b.n_edge; e += (int)G) {
        const int t = threadIdx.x;
        if (t < b.e_len[e]) {
            const int64_t jj = (b.e_pos[e] + t) / b.e_clen[e];
            const int start = (jj + 1 == world) ? 0 : (int)jj + 1;
            char* const* pp = b.ptr + (size_t)b.e_mem[e] * world;
            const int64_t el = b.e_start[e] + t;
            auto at = [&](int r) -> const char* { return pp[r]; };
            const S y = E::template sdiv<DIV>(fold_ring_scalar<E>(at, world, start, el), dop);
            for (int r = 0; r < world; ++r) reinterpret_cast<S*>(pp[r])[el] = y;
        }
    }

    SegCursor sc{0};
    int it = 0;
    for (int64_t k = blockIdx.x; k < total; k += G, ++it) {
        const int s = it % ST;
        sc.seek(b, k);
        int64_t e0, n;
        sc.range(b, k, e0, n);
        const int j = b.j[sc.seg];
        char* const* pp = b.ptr + (size_t)b.mem[sc.seg] * world;
        if (!mbar_wait_bounded(&full[s], (uint32_t)(it / ST) & 1u, ctl.limit_ns)) {
            atomicExch(&g_device_status, (int32_t)DDP_ERR_TIMEOUT);
            break;
        }
        const int start = (j + 1 == world) ? 0 : j + 1;
        const int nv = (int)(n / L);
        const unsigned char* sb = stages + (size_t)s * world * tile_bytes;
        V y[kTmaMaxVec];
#pragma unroll
        for (int u = 0; u < kTmaMaxVec; ++u) {
            const int v = threadIdx.x + u * kConsumers;
            if (v < nv) {
                int r = start;
                V acc = reinterpret_cast<const V*>(sb + (size_t)r * tile_bytes)[v];
                for (int q = 1; q < world; ++q) {
                    r = (r + 1 == world) ? 0 : r + 1;
                    acc = E::vadd(acc, reinterpret_cast<const V*>(sb + (size_t)r * tile_bytes)[v]);
                }
                y[u] = E::template vdiv<DIV>(acc, dop);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
        for (int u = 0; u < kTmaMaxVec; ++u) {
            const int v = threadIdx.x + u * kConsumers;
            if (v < nv)
                for (int r = 0; r < world; ++r)
                    st_stream<V>(pp[r] + e0 * (int64_t)sizeof(S) + (int64_t)v * 16, y[u]);
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};   // ddp_set_wait_limit_ms
std::atomic<long long> g_stall_tile{-1};                          // ddp_plant_stall (one launch)

// Control of one launch: the current limit, and a planted stall, which only
// this launch takes.
TmaCtl take_ctl() {
    TmaCtl c;
    c.limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    c.stall_tile = g_stall_tile.load(std::memory_order_relaxed) < 0 ? -1 : g_stall_tile.exchange(-1);
    return c;
}

// Per (device, kernel): the dynamic shared-memory limit set on the function so
// far (a function attribute: it is only ever raised, never lowered, so a
// launch with less shared memory stays valid) and the CTAs per SM measured
// for each shared-memory size.
struct FnState {
    size_t smem_attr = 0;
    std::map<size_t, int> per_sm;
};
std::mutex g_tma_mu;
std::map<std::pair<int, const void*>, FnState> g_tma_fn;
}  // namespace

// CTA waves of a TMA launch: launches that stream more than 512 MiB through
// HBM run four waves of resident CTAs (each walking a quarter of the tiles it
// would walk alone), which measured 1-3 % faster on GB300 (8 x 1 GiB: 2.621
// against 2.640 ms); smaller launches -- the L2-sized pieces of the unfused
// pipeline above all -- keep one wave, since every wave pays the pipeline's
// fill again and those launches got slower with four.
static int tma_waves(int64_t moved_bytes) { return moved_bytes > ((int64_t)512 << 20) ? 4 : 1; }

// Bytes of one rank's tile: one CTA per SM holds kTmaStages x world tiles
// in about 200 KB of shared memory.  Tiles are powers of two (8 KB for eight
// ranks, at most 16 KB): tiles that start on page-sized boundaries stream
// measurably faster than odd sizes.  0 = path not usable.
int64_t tma_tile_bytes(int world, int stages) {
    const int64_t budget = 200 * 1024;
    const int64_t fit = budget / ((int64_t)stages * world);
    int64_t tb = 16384;
    while (tb > fit) tb >>= 1;
    return tb >= 512 ? tb : 0;
}

bool tma_usable(int world, int64_t numel, int dtype, bool vec_ok) {
    if (!vec_ok || world > 128) return false;
    const int64_t es = elem_bytes(dtype);
    const int64_t clen = chunk_len(numel, world);
    if ((clen * es) % 16 != 0 || (numel * es) % 16 != 0) return false;
    return tma_tile_bytes(world, kTmaStages) > 0;
}

template <class E, int DIV, int CAP, bool TREE>
static cudaError_t tma_launch(int world, void* const* ptrs, int64_t numel, float dop, cudaStream_t st) {
    void (*k)(TmaTable<CAP>, int, TileMap, float, TmaCtl);
    if constexpr (TREE) k = k_tree_fused_tma<E, DIV, CAP>;
    else k = k_ring_fused_tma<E, DIV, CAP>;
    const int64_t tile_bytes = tma_tile_bytes(world, kTmaStages);
    const int64_t tile = tile_bytes / (int64_t)sizeof(typename E::S);
    const size_t smem = (size_t)kTmaStages * world * tile_bytes + 2 * kTmaStages * sizeof(uint64_t);
    int dev = 0;
    cudaGetDevice(&dev);
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lk(g_tma_mu);
        FnState& fs = g_tma_fn[std::make_pair(dev, (const void*)k)];
        if (smem > fs.smem_attr) {
            cudaError_t e =
                cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            fs.smem_attr = smem;
        }
        auto it = fs.per_sm.find(smem);
        if (it != fs.per_sm.end()) {
            per_sm = it->second;
        } else {
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kTmaThreads, smem);
            if (e != cudaSuccess) return e;
            if (per_sm <= 0) per_sm = 1;
            fs.per_sm[smem] = per_sm;
        }
    }
    TileMap map;
    map.init(numel, TREE ? numel : chunk_len(numel, world), tile);      // the tree: one chunk
    const int64_t moved = 2 * (int64_t)world * numel * (int64_t)sizeof(typename E::S);
    const int grid = cap_ctas(std::min<int64_t>((int64_t)sm_count() * per_sm * tma_waves(moved), map.total));
    TmaTable<CAP> tab{};
    for (int r = 0; r < world; ++r) tab.p[r] = static_cast<char*>(ptrs[r]);
    cudaError_t e = launch_dependent(k, dim3(std::max(grid, 1)), dim3(kTmaThreads), smem, st, tab, world, map, dop,
                                     take_ctl());
    if (debug_enabled())
        fprintf(stderr, "[ddp] %s_fused_tma world=%d numel=%lld tile=%lld B grid=%d smem=%zu tiles=%lld\n",
                TREE ? "tree" : "ring", world, (long long)numel, (long long)tile_bytes, grid, smem,
                (long long)map.total);
    return e;
}

template <class E, int DIV, bool TREE>
static cudaError_t tma_cap(int world, void* const* ptrs, int64_t numel, float dop, cudaStream_t st) {
    if constexpr (TREE) {
        // the tree's fold is unrolled up to the table size: keep it tight
        if (world <= 2) return tma_launch<E, DIV, 2, TREE>(world, ptrs, numel, dop, st);
        if (world <= 4) return tma_launch<E, DIV, 4, TREE>(world, ptrs, numel, dop, st);
        if (world <= 8) return tma_launch<E, DIV, 8, TREE>(world, ptrs, numel, dop, st);
        if (world <= 16) return tma_launch<E, DIV, 16, TREE>(world, ptrs, numel, dop, st);
        return tma_launch<E, DIV, 64, TREE>(world, ptrs, numel, dop, st);
    } else {
        if (world <= 16) return tma_launch<E, DIV, 16, TREE>(world, ptrs, numel, dop, st);
        return tma_launch<E, DIV, 128, TREE>(world, ptrs, numel, dop, st);
    }
}

template <class E, bool TREE>
static cudaError_t tma_div(int world, void* const* ptrs, int64_t numel, DivSpec d, cudaStream_t st) {
    switch (d.mode) {
        case kDivNone: return tma_cap<E, kDivNone, TREE>(world, ptrs, numel, d.operand, st);
        case kDivPow2: return tma_cap<E, kDivPow2, TREE>(world, ptrs, numel, d.operand, st);
        default: return tma_cap<E, kDivIeee, TREE>(world, ptrs, numel, d.operand, st);
    }
}

cudaError_t launch_ring_fused_tma(int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div,
                                  cudaStream_t stream) {
    if (dtype == DDP_F32) return tma_div<EF32, false>(world, ptrs, numel, div, stream);
    return tma_div<EBF16, false>(world, ptrs, numel, div, stream);
}

bool tree_tma_usable(int world, int64_t numel, int dtype, bool vec_ok) {
    if (!vec_ok || world > 64) return false;
    return (numel * elem_bytes(dtype)) % 16 == 0 && tma_tile_bytes(world, kTmaStages) > 0;
}

cudaError_t launch_tree_fused_tma(int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div,
                                  cudaStream_t stream) {
    if (dtype == DDP_F32) return tma_div<EF32, true>(world, ptrs, numel, div, stream);
    return tma_div<EBF16, true>(world, ptrs, numel, div, stream);
}

template <class E, int DIV, class BT, int ST>
static cudaError_t view_tma_launch(int world, const ViewMember* members, const ViewSegment* segs, int n_segs,
                                   const ViewEdge* edges, int n_edges, float dop, cudaStream_t st) {
    auto k = k_bucket_view_tma<E, DIV, BT, ST>;
    const int64_t tile_bytes = tma_tile_bytes(world, ST);
    const int64_t tile = tile_bytes / (int64_t)sizeof(typename E::S);
    const size_t smem = (size_t)ST * world * tile_bytes + 2 * ST * sizeof(uint64_t);
    int dev = 0;
    cudaGetDevice(&dev);
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lk(g_tma_mu);
        FnState& fs = g_tma_fn[std::make_pair(dev, (const void*)k)];
        if (smem > fs.smem_attr) {
            cudaError_t e =
                cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            fs.smem_attr = smem;
        }
        auto it = fs.per_sm.find(smem);
        if (it != fs.per_sm.end()) {
            per_sm = it->second;
        } else {
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kTmaThreads, smem);
            if (e != cudaSuccess) return e;
            if (per_sm <= 0) per_sm = 1;
            fs.per_sm[smem] = per_sm;
        }
    }
    return fill_view_batches<BT>(
        world, members, segs, n_segs, edges, n_edges, tile, (int64_t)sizeof(typename E::S),
        [&](const BT& b, int64_t tiles, int64_t moved) -> cudaError_t {
            const int64_t work = std::max<int64_t>(tiles, b.n_edge);
            const int grid = cap_ctas(std::min<int64_t>((int64_t)sm_count() * per_sm * tma_waves(moved), work));
            const cudaError_t e = launch_dependent(k, dim3(grid), dim3(kTmaThreads), smem, st, b, dop, take_ctl());
            if (debug_enabled())
                fprintf(stderr, "[ddp] bucket_view_tma world=%d segments=%d edges=%d tiles=%lld grid=%d\n", world,
                        b.n_seg, b.n_edge, (long long)tiles, grid);
            return e;
        });
}

// The small table when the whole call fits in it, else the large one.
template <class E, int DIV>
static cudaError_t view_tma_pick(int world, const ViewMember* members, const ViewSegment* segs, int n_segs,
                                 const ViewEdge* edges, int n_edges, float dop, cudaStream_t st) {
    // under a CTA budget below four blocks per SM each CTA keeps a third stage
    // in flight: with few CTAs the bytes each one has in flight set the rate
    const bool small = view_fits_small(world, segs, n_segs, n_edges);
    if (cta_cap_is_tight() && tma_tile_bytes(world, 3) > 0) {
        if (small) return view_tma_launch<E, DIV, ViewSegSmall, 3>(world, members, segs, n_segs, edges, n_edges, dop, st);
        return view_tma_launch<E, DIV, ViewSegLarge, 3>(world, members, segs, n_segs, edges, n_edges, dop, st);
    }
    if (small) return view_tma_launch<E, DIV, ViewSegSmall, kTmaStages>(world, members, segs, n_segs, edges, n_edges, dop, st);
    return view_tma_launch<E, DIV, ViewSegLarge, kTmaStages>(world, members, segs, n_segs, edges, n_edges, dop, st);
}

template <class E>
static cudaError_t view_tma_div(int world, const ViewMember* m, int nm, const ViewSegment* sg, int ns,
                                const ViewEdge* ed, int ne, DivSpec d, cudaStream_t st) {
    switch (d.mode) {
        case kDivNone: return view_tma_pick<E, kDivNone>(world, m, sg, ns, ed, ne, d.operand, st);
        case kDivPow2: return view_tma_pick<E, kDivPow2>(world, m, sg, ns, ed, ne, d.operand, st);
        default: return view_tma_pick<E, kDivIeee>(world, m, sg, ns, ed, ne, d.operand, st);
    }
}

cudaError_t launch_bucket_view_tma(int world, const ViewMember* members, int n_members, const ViewSegment* segs,
                                   int n_segs, const ViewEdge* edges, int n_edges, int dtype, DivSpec div,
                                   cudaStream_t stream) {
    if (n_segs == 0 && n_edges == 0) return cudaSuccess;
    if (dtype == DDP_F32) return view_tma_div<EF32>(world, members, n_members, segs, n_segs, edges, n_edges, div, stream);
    if (dtype == kDtypeHook)
        return view_tma_div<EHOOK>(world, members, n_members, segs, n_segs, edges, n_edges, div, stream);
    if (dtype == kDtypeHook16)
        return view_tma_div<EHOOK16>(world, members, n_members, segs, n_segs, edges, n_edges, div, stream);
    return view_tma_div<EBF16>(world, members, n_members, segs, n_segs, edges, n_edges, div, stream);
}

void set_wait_limit_ns(unsigned long long ns, unsigned long long* previous) {
    const unsigned long long p = g_wait_limit_ns.exchange(ns);
    if (previous) *previous = p;
}

void plant_stall(long long tile) { g_stall_tile.store(tile < 0 ? -1 : tile); }

cudaError_t read_device_status(int32_t* out, bool clear) {
    int32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v));
    if (e != cudaSuccess) return e;
    if (clear && v != 0) {
        const int32_t zero = 0;
        e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
        if (e != cudaSuccess) return e;
    }
    *out = v;
    return cudaSuccess;
}

}  // namespace ddpk
