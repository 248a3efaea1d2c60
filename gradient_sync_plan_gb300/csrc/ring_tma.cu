// ring_tma.cu -- fused ring allreduce with TMA bulk copies into shared memory.
//
// Same result as k_ring_fused (ring_kernels.cu): element i of chunk j is
// folded over the ranks starting at rank j+1 ("DDP 与 Ring-AllReduce", §1.3.2;
// "DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事", section 03),
// divided by the divisor and written to every rank.  What differs is how the
// bytes move.  The bucket is cut into tiles that never cross a chunk
// boundary; one persistent CTA per SM streams its tiles through a ring of
// shared-memory stages, with its warps split by role:
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
// Waits are bounded: an mbarrier wait that exceeds kWaitLimitNs sets the
// library's device status word to DDP_ERR_TIMEOUT and the thread stops; the
// producer then waits (again bounded) for the copies it issued before it
// returns.
#include <algorithm>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include "ddp_device.cuh"
#include "ddp_internal.h"

namespace ddpk {

__device__ int32_t g_device_status = 0;     // sticky DDP_ERR_TIMEOUT flag, read by ddp_device_status()

constexpr int kTmaStages = 2;
constexpr int kTmaConsumerWarps = 8;
constexpr int kTmaThreads = 32 * (kTmaConsumerWarps + 1);    // + one producer warp
constexpr int kTmaMaxVec = 4;        // 16-byte vectors per consumer thread per tile (tile <= 16 KB)
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s

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
// kWaitLimitNs; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
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

template <class E, int DIV, int CAP>
__global__ void __launch_bounds__(kTmaThreads, 1)
k_ring_fused_tma(const __grid_constant__ TmaTable<CAP> t, int world, TileMap map, float dop) {
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
            const int s = it % kTmaStages;
            // the stage's previous tile (it - kTmaStages) must have been read
            if (it >= kTmaStages && !mbar_wait_bounded(&empty[s], (uint32_t)(it / kTmaStages - 1) & 1u)) {
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
            mbar_wait_bounded(&empty[i2 % kTmaStages], (uint32_t)(i2 / kTmaStages) & 1u);
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
        if (!mbar_wait_bounded(&full[s], (uint32_t)(it / kTmaStages) & 1u)) {
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

// ---------------------------------------------------------------------------
// The fused view path (pack + ring + average + unpack of one bucket) with the
// same producer / consumer structure.  The host cuts every member of the
// bucket at the bucket's chunk boundaries into segments; a segment has one
// ring start rank, and tiles are cut inside segments, so a tile never crosses
// a chunk.  Tiles are numbered segment after segment; each CTA walks its
// tiles k, k + G, ... and finds their segment by scanning forward.
// ---------------------------------------------------------------------------

constexpr int kViewSegs = 224;
constexpr int kViewPtrCap = 2816;

struct ViewTmaBatch {
    int32_t n_seg;
    int32_t world;
    int64_t tile;                    // elements per tile
    int64_t tile_end[kViewSegs];     // inclusive prefix of tiles per segment
    int64_t start[kViewSegs];        // first element of the segment in its member
    int64_t len[kViewSegs];
    int32_t j[kViewSegs];            // ring chunk of the segment
    int32_t mem[kViewSegs];          // member slot: its rank pointers are ptr[mem * world ..]
    char* ptr[kViewPtrCap];
};
static_assert(sizeof(ViewTmaBatch) <= kMaxParamBytes, "view batch exceeds the kernel parameter limit");

struct SegCursor {
    int seg;
    __device__ void seek(const ViewTmaBatch& b, int64_t k) {
        while (b.tile_end[seg] <= k) ++seg;
    }
    __device__ void range(const ViewTmaBatch& b, int64_t k, int64_t& e0, int64_t& n) const {
        const int64_t first = seg ? b.tile_end[seg - 1] : 0;
        const int64_t off = (k - first) * b.tile;
        e0 = b.start[seg] + off;
        n = (b.len[seg] - off < b.tile) ? b.len[seg] - off : b.tile;
    }
};

template <class E, int DIV>
__global__ void __launch_bounds__(kTmaThreads, 1)
k_bucket_view_tma(const __grid_constant__ ViewTmaBatch b, float dop) {
    using V = typename E::V;
    using S = typename E::S;
    constexpr int L = E::L;
    constexpr int kConsumers = 32 * kTmaConsumerWarps;
    extern __shared__ __align__(128) unsigned char smem[];
    const int world = b.world;
    const int64_t tile_bytes = b.tile * (int64_t)sizeof(S);
    unsigned char* stages = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kTmaStages * world * tile_bytes);
    uint64_t* empty = full + kTmaStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    const int64_t total = b.tile_end[b.n_seg - 1];

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTmaStages; ++s) {
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
            const int s = it % kTmaStages;
            if (it >= kTmaStages && !mbar_wait_bounded(&empty[s], (uint32_t)(it / kTmaStages - 1) & 1u)) {
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
        for (int q = 1; q <= kTmaStages && it - q >= 0; ++q) {
            const int i2 = it - q;
            mbar_wait_bounded(&empty[i2 % kTmaStages], (uint32_t)(i2 / kTmaStages) & 1u);
        }
        return;
    }

    SegCursor sc{0};
    int it = 0;
    for (int64_t k = blockIdx.x; k < total; k += G, ++it) {
        const int s = it % kTmaStages;
        sc.seek(b, k);
        int64_t e0, n;
        sc.range(b, k, e0, n);
        const int j = b.j[sc.seg];
        char* const* pp = b.ptr + (size_t)b.mem[sc.seg] * world;
        if (!mbar_wait_bounded(&full[s], (uint32_t)(it / kTmaStages) & 1u)) {
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

// Bytes of one rank's tile: one CTA per SM holds kTmaStages x world tiles
// in about 200 KB of shared memory.  Tiles are powers of two (8 KB for eight
// ranks, at most 16 KB): tiles that start on page-sized boundaries stream
// measurably faster than odd sizes.  0 = path not usable.
int64_t tma_tile_bytes(int world) {
    const int64_t budget = 200 * 1024;
    const int64_t fit = budget / ((int64_t)kTmaStages * world);
    int64_t tb = 16384;
    while (tb > fit) tb >>= 1;
    return tb >= 512 ? tb : 0;
}

bool tma_usable(int world, int64_t numel, int dtype, bool vec_ok) {
    if (!vec_ok || world > 128) return false;
    const int64_t es = elem_bytes(dtype);
    const int64_t clen = chunk_len(numel, world);
    if ((clen * es) % 16 != 0 || (numel * es) % 16 != 0) return false;
    return tma_tile_bytes(world) > 0;
}

template <class E, int DIV, int CAP>
static cudaError_t tma_launch(int world, void* const* ptrs, int64_t numel, float dop, cudaStream_t st) {
    auto k = k_ring_fused_tma<E, DIV, CAP>;
    const int64_t tile_bytes = tma_tile_bytes(world);
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
    map.init(numel, chunk_len(numel, world), tile);
    const int grid = cap_ctas(std::min<int64_t>((int64_t)sm_count() * per_sm, map.total));
    TmaTable<CAP> tab{};
    for (int r = 0; r < world; ++r) tab.p[r] = static_cast<char*>(ptrs[r]);
    k<<<std::max(grid, 1), kTmaThreads, smem, st>>>(tab, world, map, dop);
    if (debug_enabled())
        fprintf(stderr, "[ddp] ring_fused_tma world=%d numel=%lld tile=%lld B grid=%d smem=%zu tiles=%lld\n", world,
                (long long)numel, (long long)tile_bytes, grid, smem, (long long)map.total);
    return cudaGetLastError();
}

template <class E, int DIV>
static cudaError_t tma_cap(int world, void* const* ptrs, int64_t numel, float dop, cudaStream_t st) {
    if (world <= 16) return tma_launch<E, DIV, 16>(world, ptrs, numel, dop, st);
    return tma_launch<E, DIV, 128>(world, ptrs, numel, dop, st);
}

template <class E>
static cudaError_t tma_div(int world, void* const* ptrs, int64_t numel, DivSpec d, cudaStream_t st) {
    switch (d.mode) {
        case kDivNone: return tma_cap<E, kDivNone>(world, ptrs, numel, d.operand, st);
        case kDivPow2: return tma_cap<E, kDivPow2>(world, ptrs, numel, d.operand, st);
        default: return tma_cap<E, kDivIeee>(world, ptrs, numel, d.operand, st);
    }
}

cudaError_t launch_ring_fused_tma(int world, void* const* ptrs, int64_t numel, int dtype, DivSpec div,
                                  cudaStream_t stream) {
    if (dtype == DDP_F32) return tma_div<EF32>(world, ptrs, numel, div, stream);
    return tma_div<EBF16>(world, ptrs, numel, div, stream);
}

template <class E, int DIV>
static cudaError_t view_tma_launch(int world, const ViewMember* members, int n_members, const ViewSegment* segs,
                                   int n_segs, float dop, cudaStream_t st) {
    auto k = k_bucket_view_tma<E, DIV>;
    const int64_t tile_bytes = tma_tile_bytes(world);
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
    // launches take consecutive members (and all their segments) while the
    // pointer and segment tables have room
    const int max_members = kViewPtrCap / world;
    ViewTmaBatch b;
    b.world = world;
    b.tile = tile;
    int si = 0;
    while (si < n_segs) {
        b.n_seg = 0;
        int64_t tiles = 0;
        int first_member = segs[si].member, slots = 0, last_member = -1;
        while (si < n_segs && b.n_seg < kViewSegs) {
            const ViewSegment& g = segs[si];
            if (g.member != last_member) {
                if (slots == max_members) break;
                const ViewMember& m = members[g.member];
                for (int r = 0; r < world; ++r) b.ptr[(size_t)slots * world + r] = static_cast<char*>(m.ptrs[r]);
                last_member = g.member;
                ++slots;
            }
            tiles += (g.len + tile - 1) / tile;
            b.tile_end[b.n_seg] = tiles;
            b.start[b.n_seg] = g.start;
            b.len[b.n_seg] = g.len;
            b.j[b.n_seg] = g.j;
            b.mem[b.n_seg] = slots - 1;
            ++b.n_seg;
            ++si;
        }
        (void)first_member;
        if (b.n_seg == 0) break;
        const int grid = cap_ctas(std::min<int64_t>((int64_t)sm_count() * per_sm, tiles));
        k<<<grid, kTmaThreads, smem, st>>>(b, dop);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (debug_enabled())
            fprintf(stderr, "[ddp] bucket_view_tma world=%d segments=%d members=%d tiles=%lld grid=%d\n", world,
                    b.n_seg, slots, (long long)tiles, grid);
    }
    return cudaSuccess;
}

template <class E>
static cudaError_t view_tma_div(int world, const ViewMember* m, int nm, const ViewSegment* sg, int ns, DivSpec d,
                                cudaStream_t st) {
    switch (d.mode) {
        case kDivNone: return view_tma_launch<E, kDivNone>(world, m, nm, sg, ns, d.operand, st);
        case kDivPow2: return view_tma_launch<E, kDivPow2>(world, m, nm, sg, ns, d.operand, st);
        default: return view_tma_launch<E, kDivIeee>(world, m, nm, sg, ns, d.operand, st);
    }
}

cudaError_t launch_bucket_view_tma(int world, const ViewMember* members, int n_members, const ViewSegment* segs,
                                   int n_segs, int dtype, DivSpec div, cudaStream_t stream) {
    if (n_segs == 0) return cudaSuccess;
    if (dtype == DDP_F32) return view_tma_div<EF32>(world, members, n_members, segs, n_segs, div, stream);
    if (dtype == kDtypeHook) return view_tma_div<EHOOK>(world, members, n_members, segs, n_segs, div, stream);
    if (dtype == kDtypeHook16) return view_tma_div<EHOOK16>(world, members, n_members, segs, n_segs, div, stream);
    return view_tma_div<EBF16>(world, members, n_members, segs, n_segs, div, stream);
}

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
