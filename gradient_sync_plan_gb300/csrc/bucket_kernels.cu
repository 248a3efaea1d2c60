// bucket_kernels.cu -- gradient <-> bucket copies and the fused view path.
//
// DDP copies every gradient into its bucket before the bucket's allreduce and
// copies the averaged bucket back afterwards when gradient_as_bucket_view is
// off ("DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事", section 03
// "Overlap" and section 05 steps 2-3; "Day 17 · 梯度的集体行动" Reducer
// pseudo-code).  k_copy_items does one launch's worth of those copies: a
// table of (src, dst, bytes) items, cut into 16 KB tiles, one block per tile
// on launches of 128 MiB or more, else a grid-stride loop over a few waves
// of blocks.  The table travels in the kernel's parameter space, so a call
// needs no device workspace and no host-to-device copy.
//
// With gradient_as_bucket_view on, a gradient *is* a slice of its bucket.
// The view kernels take that to its end: they read every member's elements
// from every rank's gradient, fold them in the ring order of the chunk their
// bucket position falls in, divide and write back -- the pack, the ring
// allreduce, the average and the unpack in one pass.  k_bucket_view_seg
// folds the aligned segment bodies of a step's buckets (the table in
// view_batch.cuh), one block per tile; k_bucket_view places every element
// itself and takes what has no aligned body (members whose pointers are not
// 16-byte aligned, tiny buckets).
#include <algorithm>
#include <climits>
#include <cstdio>
#include <vector>

#include "ddp_device.cuh"
#include "ddp_internal.h"
#include "view_batch.cuh"

namespace ddpk {

// ---------------------------------------------------------------------------
// Multi-tensor copy
// ---------------------------------------------------------------------------

// Item tables come in two capacities: a launch's parameters are copied for
// every eager launch, so a call with few items (one bucket piece, a small
// bucket) sends about 1 KB instead of the 24 KB that 768 items take.
constexpr int kCopyItemsSmall = 32;
constexpr int kCopyItems = 768;          // items per launch (24 KB of parameters)
constexpr int64_t kCopyTile = 16384;     // bytes per tile: four 16-byte vectors per thread

template <int CAP>
struct CopyBatch {
    int32_t n;
    int32_t pad_;
    int64_t tile_end[CAP];   // inclusive prefix sum of tiles per item
    const char* src[CAP];
    char* dst[CAP];
    int64_t bytes[CAP];
};
static_assert(sizeof(CopyBatch<kCopyItems>) <= kMaxParamBytes, "copy batch exceeds the kernel parameter limit");

// Copy [b0, b1) bytes from src to dst with the whole block.  Element pointers
// are at least 2-byte aligned; when src and dst agree modulo 16 the middle is
// copied in 16-byte vectors, four in flight per thread.
__device__ __forceinline__ void block_copy(const char* src, char* dst, int64_t b0, int64_t b1) {
    const uintptr_t sa = reinterpret_cast<uintptr_t>(src + b0), da = reinterpret_cast<uintptr_t>(dst + b0);
    const int64_t n = b1 - b0;
    if (((sa ^ da) & 15u) == 0) {
        const int64_t head = std::min<int64_t>((16 - (da & 15u)) & 15u, n);
        for (int64_t k = 2 * (int64_t)threadIdx.x; k < head; k += 2 * blockDim.x)
            *reinterpret_cast<uint16_t*>(dst + b0 + k) = *reinterpret_cast<const uint16_t*>(src + b0 + k);
        const int64_t a0 = b0 + head;
        const int64_t nv = (b1 - a0) >> 4;
        const uint4* s4 = reinterpret_cast<const uint4*>(src + a0);
        uint4* d4 = reinterpret_cast<uint4*>(dst + a0);
        int64_t k = threadIdx.x;
        for (; k + 3 * (int64_t)blockDim.x < nv; k += 4 * (int64_t)blockDim.x) {
            uint4 x0 = s4[k], x1 = s4[k + blockDim.x], x2 = s4[k + 2 * blockDim.x], x3 = s4[k + 3 * blockDim.x];
            d4[k] = x0;
            d4[k + blockDim.x] = x1;
            d4[k + 2 * blockDim.x] = x2;
            d4[k + 3 * blockDim.x] = x3;
        }
        for (; k < nv; k += blockDim.x) d4[k] = s4[k];
        const int64_t a1 = a0 + (nv << 4);
        for (int64_t q = a1 + 2 * (int64_t)threadIdx.x; q < b1; q += 2 * blockDim.x)
            *reinterpret_cast<uint16_t*>(dst + q) = *reinterpret_cast<const uint16_t*>(src + q);
    } else if (((sa | da | (uintptr_t)n) & 3u) == 0) {
        for (int64_t k = 4 * (int64_t)threadIdx.x; k < n; k += 4 * blockDim.x)
            *reinterpret_cast<uint32_t*>(dst + b0 + k) = *reinterpret_cast<const uint32_t*>(src + b0 + k);
    } else {
        for (int64_t k = 2 * (int64_t)threadIdx.x; k < n; k += 2 * blockDim.x)
            *reinterpret_cast<uint16_t*>(dst + b0 + k) = *reinterpret_cast<const uint16_t*>(src + b0 + k);
    }
}

template <int CAP>
__global__ void __launch_bounds__(kThreads) k_copy_items(const __grid_constant__ CopyBatch<CAP> b) {
    pdl_release();
    pdl_acquire();
    const int64_t tiles = b.tile_end[b.n - 1];
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        int lo = 0, hi = b.n - 1;            // first item whose tile_end > tile
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (b.tile_end[mid] > tile) hi = mid; else lo = mid + 1;
        }
        const int64_t first = lo ? b.tile_end[lo - 1] : 0;
        const int64_t b0 = (tile - first) * kCopyTile;
        const int64_t b1 = std::min(b0 + kCopyTile, b.bytes[lo]);
        block_copy(b.src[lo], b.dst[lo], b0, b1);
    }
}

template <int CAP>
static cudaError_t copy_items_cap(const CopyItem* items, int64_t n, cudaStream_t stream) {
    CopyBatch<CAP> b;
    int64_t i = 0;
    while (i < n) {
        b.n = 0;
        b.pad_ = 0;
        int64_t tiles = 0;
        for (; i < n && b.n < CAP; ++i) {
            if (items[i].bytes <= 0) continue;
            tiles += (items[i].bytes + kCopyTile - 1) / kCopyTile;
            b.tile_end[b.n] = tiles;
            b.src[b.n] = static_cast<const char*>(items[i].src);
            b.dst[b.n] = static_cast<char*>(items[i].dst);
            b.bytes[b.n] = items[i].bytes;
            ++b.n;
        }
        if (b.n == 0) continue;
        // a launch that copies 128 MiB or more runs one block per tile, so the
        // blocks take the tiles in address order as SMs free up; a smaller
        // one, a few waves of blocks looping over the tiles
        const int grid = tiles * kCopyTile >= ((int64_t)128 << 20)
                             ? cap_ctas(std::min<int64_t>(tiles, INT32_MAX))
                             : grid_for((const void*)k_copy_items<CAP>, tiles * kThreads);
        cudaError_t e = launch_dependent(k_copy_items<CAP>,
                                         dim3((unsigned)std::max<int64_t>(1, std::min<int64_t>(grid, tiles))),
                                         dim3(kThreads), 0, stream, b);
        if (e != cudaSuccess) return e;
        if (debug_enabled())
            fprintf(stderr, "[ddp] copy_items n=%d tiles=%lld\n", b.n, (long long)tiles);
    }
    return cudaSuccess;
}

cudaError_t launch_copy_items(const CopyItem* items, int64_t n, cudaStream_t stream) {
    if (n <= kCopyItemsSmall) return copy_items_cap<kCopyItemsSmall>(items, n, stream);
    return copy_items_cap<kCopyItems>(items, n, stream);
}

// ---------------------------------------------------------------------------
// Converting copies for the bf16 compression hook
// ---------------------------------------------------------------------------
//
// DDP's communication hooks ("Day 17 · 梯度的集体行动", reading list on DDP
// communication hooks: fp16/bf16 compression) let the bucket travel in a
// narrower type: fp32 gradients are rounded to bf16 (nearest even) on the way
// into the bucket and widened back (exactly) on the way out.

constexpr int kConvItemsSmall = 32;
constexpr int kConvItems = 704;
constexpr int64_t kConvTile = 8192;      // elements per tile

template <int CAP>
struct ConvBatch {
    int32_t n;
    int32_t pad_;
    int64_t tile_end[CAP];
    const char* src[CAP];
    char* dst[CAP];
    int64_t numel[CAP];
    int32_t vec[CAP];
};
static_assert(sizeof(ConvBatch<kConvItems>) <= kMaxParamBytes, "convert batch exceeds the kernel parameter limit");

// MODE 0: float32 -> bf16 (round to nearest even); MODE 1: bf16 -> float32 (exact).
// Aligned items move groups of 4 elements: lane t of a warp takes group t, so
// the 16-byte float32 side and the 8-byte bf16 side of one load or store
// instruction are both contiguous across the warp and every L2 sector is
// written whole (a layout with two 16-byte stores 32 bytes apart per lane
// half-filled each sector per instruction and nearly doubled the L2 write
// traffic of the widening pass).  Each thread has kConvUnroll groups in
// flight.
constexpr int kConvUnroll = 8;

template <int MODE>
__device__ __forceinline__ void convert_group(const char* src, char* dst, int64_t e) {
    if (MODE == 0) {
        const float4 a = *reinterpret_cast<const float4*>(src + e * 4);
        *reinterpret_cast<uint2*>(dst + e * 2) = make_uint2(bf16x2_rn(a.x, a.y), bf16x2_rn(a.z, a.w));
    } else {
        const uint2 w = *reinterpret_cast<const uint2*>(src + e * 2);
        *reinterpret_cast<float4*>(dst + e * 4) = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
    }
}

template <int MODE, int CAP>
__global__ void __launch_bounds__(kThreads) k_convert_items(const __grid_constant__ ConvBatch<CAP> b) {
    pdl_release();
    pdl_acquire();
    const int64_t tiles = b.tile_end[b.n - 1];
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        int lo = 0, hi = b.n - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (b.tile_end[mid] > tile) hi = mid; else lo = mid + 1;
        }
        const int64_t first = lo ? b.tile_end[lo - 1] : 0;
        const int64_t e0 = (tile - first) * kConvTile;
        const int64_t e1 = std::min(e0 + kConvTile, b.numel[lo]);
        const char* src = b.src[lo];
        char* dst = b.dst[lo];
        int64_t done = e0;
        if (b.vec[lo]) {
            const int64_t ng = (e1 - e0) / 4;
            const int64_t bd = blockDim.x;
            int64_t g = threadIdx.x;
            for (; g + (kConvUnroll - 1) * bd < ng; g += kConvUnroll * bd) {
                if (MODE == 0) {
                    float4 a[kConvUnroll];
#pragma unroll
                    for (int u = 0; u < kConvUnroll; ++u)
                        a[u] = *reinterpret_cast<const float4*>(src + (e0 + 4 * (g + u * bd)) * 4);
#pragma unroll
                    for (int u = 0; u < kConvUnroll; ++u)
                        *reinterpret_cast<uint2*>(dst + (e0 + 4 * (g + u * bd)) * 2) =
                            make_uint2(bf16x2_rn(a[u].x, a[u].y), bf16x2_rn(a[u].z, a[u].w));
                } else {
                    uint2 w[kConvUnroll];
#pragma unroll
                    for (int u = 0; u < kConvUnroll; ++u)
                        w[u] = *reinterpret_cast<const uint2*>(src + (e0 + 4 * (g + u * bd)) * 2);
#pragma unroll
                    for (int u = 0; u < kConvUnroll; ++u)
                        *reinterpret_cast<float4*>(dst + (e0 + 4 * (g + u * bd)) * 4) =
                            make_float4(bf16_lo(w[u].x), bf16_hi(w[u].x), bf16_lo(w[u].y), bf16_hi(w[u].y));
                }
            }
            for (; g < ng; g += bd) convert_group<MODE>(src, dst, e0 + 4 * g);
            done = e0 + ng * 4;
        }
        for (int64_t e = done + threadIdx.x; e < e1; e += blockDim.x) {
            if (MODE == 0)
                reinterpret_cast<uint16_t*>(dst)[e] = f32_to_bf16_rn(reinterpret_cast<const float*>(src)[e]);
            else
                reinterpret_cast<float*>(dst)[e] = bf16_to_f32(reinterpret_cast<const uint16_t*>(src)[e]);
        }
    }
}

// One CTA per tile rather than a grid of resident CTAs walking the tiles:
// on GB300 the widening pass ran at 6.92 TB/s that way against 6.21 TB/s on
// the resident grid (8 x 2^25 elements, CUDA events).
template <int CAP>
static cudaError_t convert_items_cap(const ConvItem* items, int64_t n, int to_bf16, cudaStream_t stream) {
    ConvBatch<CAP> b;
    int64_t i = 0;
    while (i < n) {
        b.n = 0;
        b.pad_ = 0;
        int64_t tiles = 0;
        for (; i < n && b.n < CAP; ++i) {
            if (items[i].numel <= 0) continue;
            tiles += (items[i].numel + kConvTile - 1) / kConvTile;
            b.tile_end[b.n] = tiles;
            b.src[b.n] = static_cast<const char*>(items[i].src);
            b.dst[b.n] = static_cast<char*>(items[i].dst);
            b.numel[b.n] = items[i].numel;
            b.vec[b.n] = ((reinterpret_cast<uintptr_t>(items[i].src) | reinterpret_cast<uintptr_t>(items[i].dst)) % 16) == 0;
            ++b.n;
        }
        if (b.n == 0) continue;
        const int grid = cap_ctas(std::min<int64_t>(tiles, INT32_MAX));
        cudaError_t e = to_bf16 ? launch_dependent(k_convert_items<0, CAP>, dim3(grid), dim3(kThreads), 0, stream, b)
                                : launch_dependent(k_convert_items<1, CAP>, dim3(grid), dim3(kThreads), 0, stream, b);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_convert_items(const ConvItem* items, int64_t n, int to_bf16, cudaStream_t stream) {
    if (n <= kConvItemsSmall) return convert_items_cap<kConvItemsSmall>(items, n, to_bf16, stream);
    return convert_items_cap<kConvItems>(items, n, to_bf16, stream);
}

// ---------------------------------------------------------------------------
// Fused view: pack + ring allreduce + average + unpack of one bucket
// ---------------------------------------------------------------------------

constexpr int kViewMembers = 192;
constexpr int kViewPtrs = 3072;          // member x rank pointers per launch

struct ViewBatch {
    int32_t n;            // members in this launch
    int32_t world;
    int64_t clen[kViewMembers];   // chunk length of the member's bucket, ceil(bucket_numel / N)
    int64_t tile_end[kViewMembers];
    int64_t numel[kViewMembers];
    int64_t offset[kViewMembers];
    int32_t vec[kViewMembers];
    char* ptr[kViewPtrs];  // ptr[m * world + r]: rank r's gradient of member m
};
static_assert(sizeof(ViewBatch) <= kMaxParamBytes, "view batch exceeds the kernel parameter limit");

template <class E>
constexpr int64_t view_tile_elems() { return (int64_t)kThreads * E::L * 4; }

template <class E, int DIV, int G>
__global__ void __launch_bounds__(kThreads) k_bucket_view(const __grid_constant__ ViewBatch b, float dop) {
    using V = typename E::V;
    using S = typename E::S;
    constexpr int L = E::L;
    constexpr int64_t TILE = view_tile_elems<E>();
    pdl_release();
    pdl_acquire();
    const int world = b.world;
    const int64_t tiles = b.tile_end[b.n - 1];
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        int lo = 0, hi = b.n - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (b.tile_end[mid] > tile) hi = mid; else lo = mid + 1;
        }
        const int m = lo;
        const int64_t first = m ? b.tile_end[m - 1] : 0;
        const int64_t e0 = (tile - first) * TILE;
        const int64_t e1 = std::min(e0 + TILE, b.numel[m]);
        const int64_t base = b.offset[m];          // bucket position of element 0
        const int64_t clen = b.clen[m];
        auto at = [&](int r) -> const char* { return b.ptr[m * world + r]; };
        if (b.vec[m]) {
            // chunk of the tile's first element and where (member-relative)
            // the next chunk starts: most vectors are placed by one compare
            const int64_t j_first = (base + e0) / clen;
            const int64_t next_start = (j_first + 1) * clen - base;
            for (int64_t e = e0 + (int64_t)threadIdx.x * L; e < e1; e += (int64_t)blockDim.x * L) {
                const int64_t q = base + e;
                int64_t j;
                bool whole;
                if (e + L <= next_start) {
                    j = j_first;
                    whole = e + L <= e1;
                } else if (e >= next_start && e + L <= next_start + clen) {
                    j = j_first + 1;
                    whole = e + L <= e1;
                } else {
                    j = q / clen;
                    whole = e + L <= e1 && (q + L - 1) / clen == j;
                }
                if (whole) {
                    const int start = (j + 1 == world) ? 0 : (int)j + 1;
                    V y = E::template vdiv<DIV>(fold_ring_vec<E, G>(at, world, start, e * (int64_t)sizeof(S)), dop);
                    for (int r = 0; r < world; ++r) st_stream<V>(b.ptr[m * world + r] + e * (int64_t)sizeof(S), y);
                } else {
                    for (int l = 0; l < L && e + l < e1; ++l) {
                        const int jj = (int)((q + l) / clen);
                        const int start = (jj + 1 == world) ? 0 : jj + 1;
                        S y = E::template sdiv<DIV>(fold_ring_scalar<E>(at, world, start, e + l), dop);
                        for (int r = 0; r < world; ++r) reinterpret_cast<S*>(b.ptr[m * world + r])[e + l] = y;
                    }
                }
            }
        } else {
            for (int64_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
                const int jj = (int)((base + e) / clen);
                const int start = (jj + 1 == world) ? 0 : jj + 1;
                S y = E::template sdiv<DIV>(fold_ring_scalar<E>(at, world, start, e), dop);
                for (int r = 0; r < world; ++r) reinterpret_cast<S*>(b.ptr[m * world + r])[e] = y;
            }
        }
    }
}

template <class E, int DIV, int G>
static cudaError_t view_impl(int world, const ViewMember* members, int n, int64_t bucket_numel, float dop,
                             cudaStream_t st) {
    auto k = k_bucket_view<E, DIV, G>;
    constexpr int64_t TILE = view_tile_elems<E>();
    const int per_launch = std::min(kViewMembers, kViewPtrs / world);
    const int64_t bucket_clen = chunk_len(bucket_numel, world);
    ViewBatch b;
    b.world = world;
    int i = 0;
    while (i < n) {
        b.n = 0;
        int64_t tiles = 0;
        for (; i < n && b.n < per_launch; ++i) {
            if (members[i].numel <= 0) continue;
            tiles += (members[i].numel + TILE - 1) / TILE;
            b.tile_end[b.n] = tiles;
            b.numel[b.n] = members[i].numel;
            b.offset[b.n] = members[i].offset;
            b.vec[b.n] = members[i].vec_ok ? 1 : 0;
            b.clen[b.n] = members[i].clen > 0 ? members[i].clen : bucket_clen;
            for (int r = 0; r < world; ++r) b.ptr[b.n * world + r] = static_cast<char*>(members[i].ptrs[r]);
            ++b.n;
        }
        if (b.n == 0) continue;
        const int grid = grid_for((const void*)k, tiles * kThreads);
        cudaError_t e = launch_dependent(k, dim3((unsigned)std::max<int64_t>(1, std::min<int64_t>(grid, tiles))),
                                         dim3(kThreads), 0, st, b, dop);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <class E, int DIV>
static cudaError_t view_g(int world, const ViewMember* m, int n, int64_t bn, float dop, cudaStream_t st) {
    if (world <= 4) return view_impl<E, DIV, 4>(world, m, n, bn, dop, st);
    if (world <= 8) return view_impl<E, DIV, 8>(world, m, n, bn, dop, st);
    return view_impl<E, DIV, 16>(world, m, n, bn, dop, st);
}

template <class E>
static cudaError_t view_div(int world, const ViewMember* m, int n, int64_t bn, DivSpec d, cudaStream_t st) {
    switch (d.mode) {
        case kDivNone: return view_g<E, kDivNone>(world, m, n, bn, d.operand, st);
        case kDivPow2: return view_g<E, kDivPow2>(world, m, n, bn, d.operand, st);
        default: return view_g<E, kDivIeee>(world, m, n, bn, d.operand, st);
    }
}

// Register view kernel over a segment table (view_batch.cuh): the same
// segments and edges as the TMA-staged view kernel, folded from 16-byte
// register loads.  A tile is one vector per thread of one segment, so its
// chunk, and the fold's first rank, is the segment's.  Block b folds edge b
// (one element per thread), then its tile; a launch that moves at least
// 256 MiB has one block per tile (LOOP = false) and the block scheduler
// hands the tiles out in address order, like k_ring_fused's; otherwise a
// few waves of blocks loop over the tiles.
template <class E, int DIV, int G, int MINB, bool LOOP, class B>
__global__ void __launch_bounds__(kThreads, MINB) k_bucket_view_seg(const __grid_constant__ B b, float dop) {
    using V = typename E::V;
    using S = typename E::S;
    constexpr int L = E::L;
    pdl_release();
    pdl_acquire();
    const int world = b.world;
    for (int e = blockIdx.x; e < b.n_edge; e += gridDim.x) {
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
    const int64_t total = b.n_seg > 0 ? b.tile_end[b.n_seg - 1] : 0;
    for (int64_t k = blockIdx.x; k < total; k += gridDim.x) {
        int lo = 0, hi = b.n_seg - 1;          // the tile's segment: first with tile_end > k
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (b.tile_end[mid] > k) hi = mid; else lo = mid + 1;
        }
        const int64_t first = lo ? b.tile_end[lo - 1] : 0;
        const int64_t off = (k - first) * b.tile + (int64_t)threadIdx.x * L;    // bodies are whole vectors
        if (off < (int64_t)b.len[lo]) {
            const int j = b.j[lo];
            const int start = (j + 1 == world) ? 0 : j + 1;
            char* const* pp = b.ptr + (size_t)b.mem[lo] * world;
            auto at = [&](int r) -> const char* { return pp[r]; };
            const int64_t byte = (b.start[lo] + off) * (int64_t)sizeof(S);
            const V y = E::template vdiv<DIV>(fold_ring_vec<E, G>(at, world, start, byte), dop);
            for (int r = 0; r < world; ++r) st_stream<V>(pp[r] + byte, y);
        }
        if constexpr (!LOOP) break;
    }
}

template <class E, int DIV, int G, class BT>
static cudaError_t view_seg_launch(int world, const ViewMember* members, const ViewSegment* segs, int n_segs,
                                   const ViewEdge* edges, int n_edges, float dop, cudaStream_t st) {
    auto once = k_bucket_view_seg<E, DIV, G, 4, false, BT>;
    auto loop = k_bucket_view_seg<E, DIV, G, 4, true, BT>;          // 64 registers in both forms
    const int64_t tile = (int64_t)kThreads * E::L;
    return fill_view_batches<BT>(
        world, members, segs, n_segs, edges, n_edges, tile, (int64_t)sizeof(typename E::S),
        [&](const BT& b, int64_t tiles, int64_t moved) -> cudaError_t {
            const int64_t work = std::max<int64_t>(tiles, b.n_edge);
            const bool streamed = moved >= ((int64_t)256 << 20);
            if (streamed && work <= INT32_MAX && cap_ctas(work) == work)
                return launch_dependent(once, dim3((unsigned)work), dim3(kThreads), 0, st, b, dop);
            const int grid = streamed ? cap_ctas(std::min<int64_t>(work, INT32_MAX))
                                      : grid_for((const void*)loop, work * kThreads);
            return launch_dependent(loop, dim3(grid), dim3(kThreads), 0, st, b, dop);
        });
}

template <class E, int DIV, int G>
static cudaError_t view_seg_pick(int world, const ViewMember* members, const ViewSegment* segs, int n_segs,
                                 const ViewEdge* edges, int n_edges, float dop, cudaStream_t st) {
    if (view_fits_small(world, segs, n_segs, n_edges))
        return view_seg_launch<E, DIV, G, ViewSegSmall>(world, members, segs, n_segs, edges, n_edges, dop, st);
    return view_seg_launch<E, DIV, G, ViewSegLarge>(world, members, segs, n_segs, edges, n_edges, dop, st);
}

template <class E, int DIV>
static cudaError_t view_seg_g(int world, const ViewMember* m, const ViewSegment* sg, int ns, const ViewEdge* ed,
                              int ne, float dop, cudaStream_t st) {
    if (world <= 4) return view_seg_pick<E, DIV, 4>(world, m, sg, ns, ed, ne, dop, st);
    return view_seg_pick<E, DIV, 8>(world, m, sg, ns, ed, ne, dop, st);
}

template <class E>
static cudaError_t view_seg_div(int world, const ViewMember* m, const ViewSegment* sg, int ns, const ViewEdge* ed,
                                int ne, DivSpec d, cudaStream_t st) {
    switch (d.mode) {
        case kDivNone: return view_seg_g<E, kDivNone>(world, m, sg, ns, ed, ne, d.operand, st);
        case kDivPow2: return view_seg_g<E, kDivPow2>(world, m, sg, ns, ed, ne, d.operand, st);
        default: return view_seg_g<E, kDivIeee>(world, m, sg, ns, ed, ne, d.operand, st);
    }
}

static cudaError_t launch_bucket_view_seg(int world, const ViewMember* members, const ViewSegment* segs, int n_segs,
                                          const ViewEdge* edges, int n_edges, int dtype, DivSpec div,
                                          cudaStream_t stream) {
    if (n_segs == 0 && n_edges == 0) return cudaSuccess;
    if (dtype == DDP_F32) return view_seg_div<EF32>(world, members, segs, n_segs, edges, n_edges, div, stream);
    if (dtype == kDtypeHook) return view_seg_div<EHOOK>(world, members, segs, n_segs, edges, n_edges, div, stream);
    if (dtype == kDtypeHook16)
        return view_seg_div<EHOOK16>(world, members, segs, n_segs, edges, n_edges, div, stream);
    return view_seg_div<EBF16>(world, members, segs, n_segs, edges, n_edges, div, stream);
}

// Elements of a member that the TMA view kernel cannot stage with bulk
// copies: the pieces before and after each segment's 16-byte-aligned body
// (fewer than 16 bytes each side of a chunk boundary that is not 16-byte
// aligned), or the whole member if its pointers are not 16-byte aligned.
// Short ones the TMA kernel folds element by element itself; the rest run on
// the register view kernel, one rank-pointer table per piece.
struct ViewEdges {
    std::vector<ViewMember> pieces;
    std::vector<std::vector<void*>> tables;
    void add(int world, const ViewMember& m, int64_t start, int64_t len, int64_t es, int64_t clen) {
        if (len <= 0) return;
        tables.emplace_back(world);
        for (int r = 0; r < world; ++r) tables.back()[r] = static_cast<char*>(m.ptrs[r]) + start * es;
        pieces.push_back(ViewMember{len, m.offset + start, nullptr, false, clen});
    }
    void bind() {       // the tables no longer move
        for (size_t i = 0; i < pieces.size(); ++i) pieces[i].ptrs = tables[i].data();
    }
};

// Cut members [first, first + n) of one bucket at the bucket's chunk
// boundaries into segments (member indices are global).  A segment's
// 16-byte-aligned body goes to `segs`; what is left of it, and every member
// whose pointers are not 16-byte aligned, goes to `edges` (in member order).
static void split_segments(int world, const ViewMember* members, int first, int n, int64_t bucket_numel, int dtype,
                           std::vector<ViewSegment>* segs, std::vector<ViewEdge>* edges) {
    const int64_t es = elem_bytes(dtype);
    const int64_t lanes = 16 / es;                       // elements per 16 bytes
    const int64_t clen = chunk_len(bucket_numel, world);
    for (int i = first; i < first + n; ++i) {
        const ViewMember& m = members[i];
        auto edge = [&](int64_t start, int64_t len) {
            if (len > 0) edges->push_back(ViewEdge{i, start, len, clen});
        };
        if (!m.vec_ok) {
            edge(0, m.numel);
            continue;
        }
        int64_t a = m.offset;
        const int64_t end = m.offset + m.numel;
        int64_t pending = 0, pending_len = 0;             // edge piece still open (member-relative)
        while (a < end) {
            const int64_t j = a / clen;
            const int64_t b = std::min(end, (j + 1) * clen);
            const int64_t s0 = a - m.offset, s1 = b - m.offset;
            const int64_t body0 = (s0 + lanes - 1) / lanes * lanes, body1 = s1 / lanes * lanes;
            if (body1 > body0) {
                // the head joins the piece left open at the previous boundary
                if (body0 > s0) {
                    if (pending_len == 0) pending = s0;
                    pending_len = body0 - pending;
                }
                edge(pending, pending_len);
                pending_len = 0;
                for (int64_t c = body0; c < body1; c += kViewSegMax)     // kViewSegMax: a multiple of 16 bytes
                    segs->push_back(ViewSegment{i, (int32_t)j, c, std::min(kViewSegMax, body1 - c)});
                if (s1 > body1) {
                    pending = body1;
                    pending_len = s1 - body1;
                }
            } else {
                if (pending_len == 0) pending = s0;
                pending_len = s1 - pending;
            }
            a = b;
        }
        edge(pending, pending_len);
    }
}

// The TMA-staged kernel takes a set of segments when the tiles fit the world
// size and the bytes moved are worth its set-up.
static bool view_tma_worth(int world, int64_t elems, int dtype) {
    return world <= 128 && tma_tile_bytes(world) > 0 && elems * elem_bytes(dtype) * world >= ((int64_t)4 << 20);
}

// Which kernel folds a segment table: ddp_set_fused_kernel's forced choice
// (TMA, or the register kernel for the vector and group choices), else by
// size, from a sweep with both forced (one bucket of three members, chunk
// boundaries off the 16-byte grid, N = 4 .. 64, 2 MiB .. 8 GiB moved): the
// TMA kernel for 16 or more ranks whose bodies move less than 128 MiB (its
// CTAs spread few vectors per rank over more SMs: N = 64, 32 MiB, 12.6
// against 16.6 us), the register kernel everywhere else (N = 8, 1 GiB: 157
// against 166 us; the 355M decoder's view step: 3.23 against 3.47 ms).
static bool view_use_seg(int world, int64_t body_elems, int dtype) {
    switch (fused_kernel_override()) {
        case DDP_FUSED_TMA: return false;
        case DDP_FUSED_VECTOR:
        case DDP_FUSED_GROUP: return true;
        default: break;
    }
    // under a CTA budget of less than four blocks per SM (a reducer leaving
    // SMs to the backward) the TMA kernel, which keeps a whole stage of every
    // rank in flight per CTA: the decoder's view step on 38 CTAs overlapped
    // with the backward took 11.5 ms on it against 19.3 ms on the register kernel
    if (cta_cap_is_tight()) return false;
    return world < 16 || 2 * body_elems * elem_bytes(dtype) * world >= ((int64_t)128 << 20);
}

static cudaError_t view_register(int world, const ViewMember* members, int n, int64_t bucket_numel, int dtype,
                                 DivSpec div, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    if (dtype == DDP_F32) return view_div<EF32>(world, members, n, bucket_numel, div, stream);
    if (dtype == kDtypeHook) return view_div<EHOOK>(world, members, n, bucket_numel, div, stream);
    if (dtype == kDtypeHook16) return view_div<EHOOK16>(world, members, n, bucket_numel, div, stream);
    return view_div<EBF16>(world, members, n, bucket_numel, div, stream);
}

cudaError_t launch_buckets_view(int world, const ViewMember* members, const int* bucket_first, const int* bucket_count,
                                const int64_t* bucket_numel, int n_buckets, int dtype, DivSpec div,
                                cudaStream_t stream) {
    // the aligned bodies of every bucket, and the short edges around them, in
    // one set of TMA launches; long edges (members whose pointers are not
    // 16-byte aligned, runs of tiny chunks) in one register launch; buckets
    // too small for the TMA kernel all go to the register kernel
    std::vector<ViewSegment> segs;
    std::vector<ViewEdge> all_edges;
    int64_t body = 0;
    for (int k = 0; k < n_buckets; ++k)
        split_segments(world, members, bucket_first[k], bucket_count[k], bucket_numel[k], dtype, &segs, &all_edges);
    for (const ViewSegment& g : segs) body += g.len;
    if (view_tma_worth(world, body, dtype)) {
        int n_members = 0;
        for (int k = 0; k < n_buckets; ++k) n_members = std::max(n_members, bucket_first[k] + bucket_count[k]);
        std::vector<ViewEdge> short_edges;
        ViewEdges long_edges;
        const int64_t es = elem_bytes(dtype);
        for (const ViewEdge& g : all_edges) {
            if (g.len <= kTmaEdgeMax) short_edges.push_back(g);
            else long_edges.add(world, members[g.member], g.start, g.len, es, g.clen);
        }
        cudaError_t e = view_use_seg(world, body, dtype)
                            ? launch_bucket_view_seg(world, members, segs.data(), (int)segs.size(),
                                                     short_edges.data(), (int)short_edges.size(), dtype, div, stream)
                            : launch_bucket_view_tma(world, members, n_members, segs.data(), (int)segs.size(),
                                                     short_edges.data(), (int)short_edges.size(), dtype, div, stream);
        if (e != cudaSuccess) return e;
        long_edges.bind();
        if (debug_enabled())
            fprintf(stderr, "[ddp] bucket_view edges: %zu in the TMA launch, %zu on the register kernel\n",
                    short_edges.size(), long_edges.pieces.size());
        // every long edge carries its own bucket's chunk length
        return view_register(world, long_edges.pieces.data(), (int)long_edges.pieces.size(), 1, dtype, div, stream);
    }
    for (int k = 0; k < n_buckets; ++k) {
        cudaError_t e = view_register(world, members + bucket_first[k], bucket_count[k], bucket_numel[k], dtype, div,
                                      stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_bucket_view(int world, const ViewMember* members, int n, int64_t bucket_numel, int dtype,
                               DivSpec div, cudaStream_t stream) {
    if (n == 0 || bucket_numel == 0) return cudaSuccess;
    const int first = 0;
    return launch_buckets_view(world, members, &first, &n, &bucket_numel, 1, dtype, div, stream);
}

}  // namespace ddpk
