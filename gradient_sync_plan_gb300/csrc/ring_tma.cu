// ring_tma.cu -- fused ring allreduce with TMA bulk copies through shared memory.
//
// Same result as k_ring_fused (ring_kernels.cu): element i of chunk j is
// folded over the ranks starting at rank j+1 ("DDP 与 Ring-AllReduce", §1.3.2;
// "DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事", section 03),
// divided by the divisor and written to every rank.  What differs is how the
// bytes move: the bucket is cut into tiles that never cross a chunk boundary;
// a persistent CTA streams its tiles through a ring of shared-memory stages.
// For every tile one thread issues N bulk copies (cp.async.bulk, one per
// rank) that complete on the stage's mbarrier; the CTA folds the N staged
// copies into one result tile in shared memory; the same thread then issues N
// bulk stores of that single result tile, one to each rank.  Per tile the
// threads execute no global load or store instruction at all, which removes
// the memory-instruction queue pressure of the register path.
//
// Waits are bounded: an mbarrier wait that exceeds kWaitLimitNs sets the
// library's device status word to DDP_ERR_TIMEOUT, waits (again bounded) for
// the CTA's copies still in flight, and the CTA returns.
#include <algorithm>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include "ddp_device.cuh"
#include "ddp_internal.h"

namespace ddpk {

__device__ int32_t g_device_status = 0;     // sticky DDP_ERR_TIMEOUT flag, read by ddp_device_status()

constexpr int kTmaStages = 3;
constexpr int kTmaThreads = 256;
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

// Bulk copy shared -> global, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src_smem)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Shared-memory writes by the threads must be visible to the async proxy
// before a bulk store reads them.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Tiles never cross a chunk boundary: chunk j (length clen, the last one
// shorter) holds ceil(len / tile) tiles; empty trailing chunks hold none.
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
    __device__ void at(int64_t k, int64_t& e0, int64_t& n, int& j) const {
        j = (int)(k / per_chunk);
        const int64_t cs = (int64_t)j * clen;
        const int64_t ce = (cs + clen < numel) ? cs + clen : numel;
        e0 = cs + (k - (int64_t)j * per_chunk) * tile;
        n = (ce - e0 < tile) ? ce - e0 : tile;
    }
};

template <class E, int DIV, int CAP>
__global__ void __launch_bounds__(kTmaThreads)
k_ring_fused_tma(const __grid_constant__ TmaTable<CAP> t, int world, TileMap map, float dop) {
    using V = typename E::V;
    using S = typename E::S;
    constexpr int L = E::L;
    extern __shared__ __align__(128) unsigned char smem[];
    const int64_t tile_bytes = map.tile * (int64_t)sizeof(S);
    unsigned char* stages = smem;                                           // [stages][world][tile]
    unsigned char* results = smem + (size_t)kTmaStages * world * tile_bytes;  // [2][tile]
    uint64_t* bars = reinterpret_cast<uint64_t*>(results + 2 * tile_bytes);  // [stages]
    const bool leader = threadIdx.x == 0;

    if (leader) {
        for (int s = 0; s < kTmaStages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncthreads();

    auto issue = [&](int64_t tile_idx, int s) {
        int64_t e0, n;
        int j;
        map.at(tile_idx, e0, n, j);
        const uint32_t bytes = (uint32_t)(n * (int64_t)sizeof(S));
        mbar_arrive_expect_tx(&bars[s], bytes * (uint32_t)world);
        unsigned char* dst = stages + (size_t)s * world * tile_bytes;
        for (int r = 0; r < world; ++r)
            bulk_load(dst + (size_t)r * tile_bytes, t.p[r] + e0 * (int64_t)sizeof(S), bytes, &bars[s]);
    };

    if (leader)
        for (int s = 0; s < kTmaStages; ++s) {
            const int64_t k = blockIdx.x + (int64_t)s * gridDim.x;
            if (k < map.total) issue(k, s);
        }

    int it = 0;
    bool failed = false;
    for (int64_t k = blockIdx.x; k < map.total; k += gridDim.x, ++it) {
        const int s = it % kTmaStages;
        const uint32_t parity = (uint32_t)(it / kTmaStages) & 1u;
        int64_t e0, n;
        int j;
        map.at(k, e0, n, j);
        const bool ok = mbar_wait_bounded(&bars[s], parity);
        if (!__syncthreads_and(ok)) {
            failed = true;
            break;
        }
        const int rb = it & 1;
        if (leader) bulk_wait_read<1>();      // result buffer rb was last stored two tiles ago
        __syncthreads();
        const int start = (j + 1 == world) ? 0 : j + 1;
        const int nv = (int)(n / L);
        const unsigned char* sb = stages + (size_t)s * world * tile_bytes;
        V* res = reinterpret_cast<V*>(results + rb * tile_bytes);
        for (int v = threadIdx.x; v < nv; v += blockDim.x) {
            int r = start;
            V acc = reinterpret_cast<const V*>(sb + (size_t)r * tile_bytes)[v];
            for (int q = 1; q < world; ++q) {
                r = (r + 1 == world) ? 0 : r + 1;
                acc = E::vadd(acc, reinterpret_cast<const V*>(sb + (size_t)r * tile_bytes)[v]);
            }
            res[v] = E::template vdiv<DIV>(acc, dop);
        }
        fence_async_smem();
        __syncthreads();
        if (leader) {
            const uint32_t bytes = (uint32_t)(n * (int64_t)sizeof(S));
            for (int r = 0; r < world; ++r) bulk_store(t.p[r] + e0 * (int64_t)sizeof(S), res, bytes);
            bulk_commit();
            const int64_t next = k + (int64_t)kTmaStages * gridDim.x;
            if (next < map.total) issue(next, s);
        }
    }
    if (failed && leader) {
        atomicExch(&g_device_status, (int32_t)DDP_ERR_TIMEOUT);
        // let the loads already issued for this CTA land before it exits
        for (int q = 0; q < kTmaStages; ++q) {
            const int it2 = it + q;
            const int64_t k2 = blockIdx.x + (int64_t)it2 * gridDim.x;
            if (k2 < map.total) mbar_wait_bounded(&bars[it2 % kTmaStages], (uint32_t)(it2 / kTmaStages) & 1u);
        }
    }
    if (leader) bulk_wait_all<0>();
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

// Bytes of one rank's tile: two CTAs per SM share ~220 KB, each CTA holds
// kTmaStages x world input tiles and two result tiles.  Tiles are powers of
// two (4 KB for eight ranks): tiles that start on page-sized boundaries
// stream measurably faster than odd sizes.  0 = path not usable.
int64_t tma_tile_bytes(int world) {
    const int64_t budget = 110 * 1024 - 64;
    const int64_t fit = budget / ((int64_t)kTmaStages * world + 2);
    int64_t tb = 16384;
    while (tb > fit) tb >>= 1;
    return tb >= 512 ? tb : 0;
}

bool tma_usable(int world, int64_t numel, int dtype, bool vec_ok) {
    if (!vec_ok || world > 128) return false;
    const int64_t es = elem_bytes(dtype);
    const int64_t clen = chunk_len(numel, world);
    if ((clen * es) % 16 != 0 || (numel * es) % 16 != 0) return false;
    if (numel * es * world < (int64_t)4 << 20) return false;     // small buckets: register path
    return tma_tile_bytes(world) > 0;
}

template <class E, int DIV, int CAP>
static cudaError_t tma_launch(int world, void* const* ptrs, int64_t numel, float dop, cudaStream_t st) {
    auto k = k_ring_fused_tma<E, DIV, CAP>;
    const int64_t tile_bytes = tma_tile_bytes(world);
    const int64_t tile = tile_bytes / (int64_t)sizeof(typename E::S);
    const size_t smem = (size_t)kTmaStages * world * tile_bytes + 2 * tile_bytes + kTmaStages * sizeof(uint64_t);
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
    const int grid = (int)std::min<int64_t>((int64_t)sm_count() * per_sm, map.total);
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
