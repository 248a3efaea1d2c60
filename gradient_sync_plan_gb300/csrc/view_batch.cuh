// view_batch.cuh -- the table one fused-view launch reads, shared by the two
// view kernels that take it: the TMA-staged one (ring_tma.cu) and the
// register one (bucket_kernels.cu).
//
// The host cuts every member of a step's buckets at its bucket's chunk
// boundaries into segments ("DDP 与 Ring All-Reduce：梯度同步不是一次
// AllReduce 就完事", section 05: the gradients are views into the bucket, so
// the bucket position of an element decides its ring chunk, and the chunk
// decides the fold's first rank).  A segment's 16-byte-aligned body has one
// chunk, hence one ring start rank; tiles are cut inside segments and
// numbered segment after segment.  What a body leaves at a chunk boundary
// that is not 16-byte aligned -- a few elements each side, an "edge" -- is
// folded element by element, one element per thread.
#pragma once

#include <algorithm>
#include <cstdint>
#include <vector>

#include "ddp_internal.h"

namespace ddpk {

constexpr int kViewEdgeMax = 256;       // elements of one edge: one per thread of a 256-thread block
static_assert(kViewEdgeMax == kTmaEdgeMax, "edge length limit differs between host and kernels");

// One launch's table.  Two capacities: a launch's parameters are copied for
// every eager launch, so a call with few segments (one bucket piece, one
// small bucket) sends about 4 KB instead of the 32 KB of the large table.
template <int SEGS, int PTRS, int EDGES>
struct ViewSegBatch {
    static constexpr int kSegs = SEGS, kPtrs = PTRS, kEdges = EDGES;
    int32_t n_seg;
    int32_t world;
    int64_t tile;               // elements per tile
    int64_t tile_end[SEGS];     // inclusive prefix of tiles per segment
    int64_t start[SEGS];        // first element of the segment in its member
    uint32_t len[SEGS];         // elements (segments are cut at kViewSegMax)
    uint16_t j[SEGS];           // ring chunk of the segment (world <= 128)
    uint16_t mem[SEGS];         // member slot: its rank pointers are ptr[mem * world ..]
    int32_t n_edge;
    int32_t e_mem[EDGES];       // member slot of the edge
    int32_t e_len[EDGES];       // elements, at most kViewEdgeMax
    int64_t e_start[EDGES];     // first element of the edge in its member
    int64_t e_pos[EDGES];       // bucket position of that element
    int64_t e_clen[EDGES];      // chunk length of the member's bucket
    char* ptr[PTRS];
};
using ViewSegSmall = ViewSegBatch<32, 256, 16>;
using ViewSegLarge = ViewSegBatch<320, 2816, 64>;
static_assert(2816 < 65536 && 128 < 65536, "member slots and chunk indices fit 16 bits");
static_assert(sizeof(ViewSegLarge) <= kMaxParamBytes, "view batch exceeds the kernel parameter limit");

// Fill tables from segments and edges (both in member order) and call
// launch(table, tiles, moved) for each full table and the last one: `tiles`
// is the table's tile count at `tile` elements per tile, `moved` the bytes
// its segments read and write.  A launch takes consecutive members, each with
// its segments and edges, while the pointer, segment and edge tables have
// room; a member whose work does not fit goes on in the next launch, its
// pointers repeated.
template <class BT, class Launch>
cudaError_t fill_view_batches(int world, const ViewMember* members, const ViewSegment* segs, int n_segs,
                              const ViewEdge* edges, int n_edges, int64_t tile, int64_t es, Launch launch) {
    const int max_members = BT::kPtrs / world;
    struct Item {
        int member;
        int kind;      // 0 segment, 1 edge
        int index;
    };
    std::vector<Item> items;
    items.reserve((size_t)n_segs + (size_t)n_edges);
    {
        int si = 0, ei = 0;
        while (si < n_segs || ei < n_edges) {
            const bool take_seg = ei >= n_edges || (si < n_segs && segs[si].member <= edges[ei].member);
            if (take_seg) {
                items.push_back(Item{segs[si].member, 0, si});
                ++si;
            } else {
                items.push_back(Item{edges[ei].member, 1, ei});
                ++ei;
            }
        }
    }
    BT b;
    b.world = world;
    b.tile = tile;
    b.n_seg = 0;
    b.n_edge = 0;
    int64_t tiles = 0, moved = 0;
    int slots = 0, last_member = -1;
    auto flush = [&]() -> cudaError_t {
        if (b.n_seg == 0 && b.n_edge == 0) return cudaSuccess;
        const cudaError_t e = launch(b, tiles, moved);
        b.n_seg = 0;
        b.n_edge = 0;
        tiles = 0;
        moved = 0;
        slots = 0;
        last_member = -1;
        return e;
    };
    for (const Item& it : items) {
        const bool full_tab = (it.member != last_member && slots == max_members) ||
                              (it.kind == 0 && b.n_seg == BT::kSegs) || (it.kind == 1 && b.n_edge == BT::kEdges);
        if (full_tab) {
            const cudaError_t e = flush();
            if (e != cudaSuccess) return e;
        }
        if (it.member != last_member) {
            const ViewMember& m = members[it.member];
            for (int r = 0; r < world; ++r) b.ptr[(size_t)slots * world + r] = static_cast<char*>(m.ptrs[r]);
            last_member = it.member;
            ++slots;
        }
        if (it.kind == 0) {
            const ViewSegment& g = segs[it.index];
            tiles += (g.len + tile - 1) / tile;
            moved += 2 * g.len * es * world;
            b.tile_end[b.n_seg] = tiles;
            b.start[b.n_seg] = g.start;
            b.len[b.n_seg] = (uint32_t)g.len;
            b.j[b.n_seg] = (uint16_t)g.j;
            b.mem[b.n_seg] = (uint16_t)(slots - 1);
            ++b.n_seg;
        } else {
            const ViewEdge& g = edges[it.index];
            b.e_mem[b.n_edge] = slots - 1;
            b.e_len[b.n_edge] = (int32_t)g.len;
            b.e_start[b.n_edge] = g.start;
            b.e_pos[b.n_edge] = members[it.member].offset + g.start;
            b.e_clen[b.n_edge] = g.clen;
            ++b.n_edge;
        }
    }
    return flush();
}

// Whether the whole call fits in the small table.
inline bool view_fits_small(int world, const ViewSegment* segs, int n_segs, int n_edges) {
    int n_members = 0, last = -1;
    for (int i = 0; i < n_segs; ++i)
        if (segs[i].member != last) last = segs[i].member, ++n_members;
    n_members += n_edges;                       // at most one more slot per edge
    return n_segs <= ViewSegSmall::kSegs && n_edges <= ViewSegSmall::kEdges &&
           (int64_t)n_members * world <= ViewSegSmall::kPtrs;
}

}  // namespace ddpk
