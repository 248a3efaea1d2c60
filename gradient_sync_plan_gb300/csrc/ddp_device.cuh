// ddp_device.cuh -- device-side element operations shared by the kernels.
//
// The reduction operator of the ring ("DDP 与 Ring-AllReduce", §1.3.2: the
// receiver adds the incoming chunk into its own copy):
//   fp32: one binary32 add, round to nearest even (__fadd_rn, never contracted);
//   bf16: both operands widened exactly to binary32, one binary32 add, the sum
//         rounded to bf16 to nearest even -- once per hop.
// The average ("DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事",
// section 05; "Day 17 · 梯度的集体行动" Reducer pseudo-code): y / divisor with
// one IEEE division (or the exact power-of-two reciprocal, which rounds the
// same way), bf16 results rounded once.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ddp_internal.h"

namespace ddpk {

// Programmatic dependent launch.  A kernel launched by launch_dependent may
// be scheduled while the previous kernel on its stream is still running, so
// its launch latency overlaps that kernel's tail.  Every such kernel calls
// pdl_release() (its own dependents may be scheduled from now on) and then
// pdl_acquire(), which returns only once the previous kernel has completed
// and its writes are visible -- before it touches any buffer.  Both are
// no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_acquire() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <class... KArgs, class... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
    const cudaError_t last = cudaGetLastError();      // read (and clear) as a <<<>>> launch would be
    return e != cudaSuccess ? e : last;
}

template <int DIV>
__device__ __forceinline__ float div_f32(float a, float operand) {
    if constexpr (DIV == kDivNone) return a;
    else if constexpr (DIV == kDivPow2) return __fmul_rn(a, operand);
    else return __fdiv_rn(a, operand);
}

// bf16 <-> binary32.  Widening is exact: the bf16 bits are the top half of
// the binary32 bits.  Narrowing rounds to nearest even (cvt.rn.bf16x2.f32).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    __nv_bfloat162 r = __float22bfloat162_rn(make_float2(lo, hi));
    return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    __nv_bfloat16 r = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&r);
}

// ---- fp32 ---------------------------------------------------------------
struct EF32 {
    using S = float;     // one element
    using V = float4;    // one 16-byte vector
    static constexpr int L = 4;
    __device__ static __forceinline__ S sadd(S a, S b) { return __fadd_rn(a, b); }
    __device__ static __forceinline__ V vadd(V a, V b) {
        return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
    }
    template <int DIV>
    __device__ static __forceinline__ S sdiv(S a, float op) { return div_f32<DIV>(a, op); }
    template <int DIV>
    __device__ static __forceinline__ V vdiv(V a, float op) {
        if constexpr (DIV == kDivNone) return a;
        return make_float4(div_f32<DIV>(a.x, op), div_f32<DIV>(a.y, op), div_f32<DIV>(a.z, op),
                           div_f32<DIV>(a.w, op));
    }
};

// ---- bf16 (stored as raw 16-bit patterns) -------------------------------
struct EBF16 {
    using S = uint16_t;
    using V = uint4;     // 8 bf16
    static constexpr int L = 8;
    __device__ static __forceinline__ S sadd(S a, S b) {
        return f32_to_bf16_rn(__fadd_rn(bf16_to_f32(a), bf16_to_f32(b)));
    }
    __device__ static __forceinline__ uint32_t add2(uint32_t a, uint32_t b) {
        return bf16x2_rn(__fadd_rn(bf16_lo(a), bf16_lo(b)), __fadd_rn(bf16_hi(a), bf16_hi(b)));
    }
    __device__ static __forceinline__ V vadd(V a, V b) {
        return make_uint4(add2(a.x, b.x), add2(a.y, b.y), add2(a.z, b.z), add2(a.w, b.w));
    }
    template <int DIV>
    __device__ static __forceinline__ S sdiv(S a, float op) {
        if constexpr (DIV == kDivNone) return a;
        return f32_to_bf16_rn(div_f32<DIV>(bf16_to_f32(a), op));
    }
    template <int DIV>
    __device__ static __forceinline__ uint32_t div2(uint32_t a, float op) {
        return bf16x2_rn(div_f32<DIV>(bf16_lo(a), op), div_f32<DIV>(bf16_hi(a), op));
    }
    template <int DIV>
    __device__ static __forceinline__ V vdiv(V a, float op) {
        if constexpr (DIV == kDivNone) return a;
        return make_uint4(div2<DIV>(a.x, op), div2<DIV>(a.y, op), div2<DIV>(a.z, op), div2<DIV>(a.w, op));
    }
};

// ---- float32 storage, bf16 arithmetic (the bf16 compression hook, fused) --
// Every input is rounded to bf16 before it is used, every sum and the
// quotient are rounded to bf16, and the result is stored widened back to
// float32 -- exactly what packing into a bf16 bucket, a bf16 ring and
// unpacking produce.  Rounding is idempotent, so re-rounding a running sum
// that is already a bf16 value changes nothing.
struct EHOOK {
    using S = float;
    using V = float4;
    static constexpr int L = 4;
    __device__ static __forceinline__ float rt(float x) { return bf16_to_f32(f32_to_bf16_rn(x)); }
    __device__ static __forceinline__ float4 rt4(float4 a) {
        const uint32_t lo = bf16x2_rn(a.x, a.y), hi = bf16x2_rn(a.z, a.w);
        return make_float4(bf16_lo(lo), bf16_hi(lo), bf16_lo(hi), bf16_hi(hi));
    }
    __device__ static __forceinline__ S sadd(S a, S b) { return rt(__fadd_rn(rt(a), rt(b))); }
    __device__ static __forceinline__ V vadd(V a, V b) {
        const float4 x = rt4(a), y = rt4(b);
        return rt4(make_float4(__fadd_rn(x.x, y.x), __fadd_rn(x.y, y.y), __fadd_rn(x.z, y.z), __fadd_rn(x.w, y.w)));
    }
    template <int DIV>
    __device__ static __forceinline__ S sdiv(S a, float op) { return rt(div_f32<DIV>(rt(a), op)); }
    template <int DIV>
    __device__ static __forceinline__ V vdiv(V a, float op) {
        const float4 x = rt4(a);
        return rt4(make_float4(div_f32<DIV>(x.x, op), div_f32<DIV>(x.y, op), div_f32<DIV>(x.z, op),
                               div_f32<DIV>(x.w, op)));
    }
};

// ---- float32 storage, IEEE binary16 arithmetic (the fp16 compression hook,
// fused): as EHOOK with binary16 in place of bf16 -- every input, every sum
// and the quotient rounded to binary16 (nearest even), stored widened.
struct EHOOK16 {
    using S = float;
    using V = float4;
    static constexpr int L = 4;
    __device__ static __forceinline__ float rt(float x) { return __half2float(__float2half_rn(x)); }
    __device__ static __forceinline__ float4 rt4(float4 a) {
        const float2 lo = __half22float2(__float22half2_rn(make_float2(a.x, a.y)));
        const float2 hi = __half22float2(__float22half2_rn(make_float2(a.z, a.w)));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    __device__ static __forceinline__ S sadd(S a, S b) { return rt(__fadd_rn(rt(a), rt(b))); }
    __device__ static __forceinline__ V vadd(V a, V b) {
        const float4 x = rt4(a), y = rt4(b);
        return rt4(make_float4(__fadd_rn(x.x, y.x), __fadd_rn(x.y, y.y), __fadd_rn(x.z, y.z), __fadd_rn(x.w, y.w)));
    }
    template <int DIV>
    __device__ static __forceinline__ S sdiv(S a, float op) { return rt(div_f32<DIV>(rt(a), op)); }
    template <int DIV>
    __device__ static __forceinline__ V vdiv(V a, float op) {
        const float4 x = rt4(a);
        return rt4(make_float4(div_f32<DIV>(x.x, op), div_f32<DIV>(x.y, op), div_f32<DIV>(x.z, op),
                               div_f32<DIV>(x.w, op)));
    }
};

// Streaming 16-byte accesses: the buffers are touched once per call, so
// loads and stores are marked evict-first.
template <class V>
__device__ __forceinline__ V ld_stream(const void* p) { return __ldcs(reinterpret_cast<const V*>(p)); }
template <class V>
__device__ __forceinline__ void st_stream(void* p, V v) { __stcs(reinterpret_cast<V*>(p), v); }

template <class V> __device__ __forceinline__ V make_zero();
template <> __device__ __forceinline__ float4 make_zero<float4>() { return make_float4(0.f, 0.f, 0.f, 0.f); }
template <> __device__ __forceinline__ uint4 make_zero<uint4>() { return make_uint4(0u, 0u, 0u, 0u); }

// Warp shuffle of a 16-byte vector from lane `src` of the caller's `width`-lane
// segment (all 32 lanes must call it).
__device__ __forceinline__ float4 shfl_vec(float4 a, int src, int width) {
    return make_float4(__shfl_sync(0xffffffffu, a.x, src, width), __shfl_sync(0xffffffffu, a.y, src, width),
                       __shfl_sync(0xffffffffu, a.z, src, width), __shfl_sync(0xffffffffu, a.w, src, width));
}
__device__ __forceinline__ uint4 shfl_vec(uint4 a, int src, int width) {
    return make_uint4(__shfl_sync(0xffffffffu, a.x, src, width), __shfl_sync(0xffffffffu, a.y, src, width),
                      __shfl_sync(0xffffffffu, a.z, src, width), __shfl_sync(0xffffffffu, a.w, src, width));
}
// The same, from lane (caller + delta) of the segment (the caller's own value
// where that lane is past the segment's end).
__device__ __forceinline__ float4 shfl_down_vec(float4 a, int delta, int width) {
    return make_float4(__shfl_down_sync(0xffffffffu, a.x, delta, width),
                       __shfl_down_sync(0xffffffffu, a.y, delta, width),
                       __shfl_down_sync(0xffffffffu, a.z, delta, width),
                       __shfl_down_sync(0xffffffffu, a.w, delta, width));
}
__device__ __forceinline__ uint4 shfl_down_vec(uint4 a, int delta, int width) {
    return make_uint4(__shfl_down_sync(0xffffffffu, a.x, delta, width),
                      __shfl_down_sync(0xffffffffu, a.y, delta, width),
                      __shfl_down_sync(0xffffffffu, a.z, delta, width),
                      __shfl_down_sync(0xffffffffu, a.w, delta, width));
}

// Fold the N ranks' vectors at byte offset `off` in ring order, starting at
// rank `start` (the rank right after the chunk's owner) and wrapping around:
// acc = x[start]; acc = acc (+) x[start+1]; ... ; acc = acc (+) x[start-1].
// U vectors of the same chunk, at offsets off, off + ustep, ..., are folded
// side by side into acc[0..U).  Loads are issued in groups of G ranks before
// they are folded, so G * U 16-byte requests per thread are in flight at once.
template <class E, int G, int U, class PtrAt>
__device__ __forceinline__ void fold_ring_vecs(PtrAt ptr_at, int world, int start, int64_t off, int64_t ustep,
                                               typename E::V (&acc)[U]) {
    using V = typename E::V;
    int r = start;
    for (int k0 = 0; k0 < world; k0 += G) {
        V x[G][U];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (k0 + g < world) {
                const char* p = ptr_at(r) + off;
#pragma unroll
                for (int u = 0; u < U; ++u) x[g][u] = ld_stream<V>(p + u * ustep);
                r = (r + 1 == world) ? 0 : r + 1;
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (k0 + g < world) {
#pragma unroll
                for (int u = 0; u < U; ++u) acc[u] = (k0 + g == 0) ? x[g][u] : E::vadd(acc[u], x[g][u]);
            }
        }
    }
}

template <class E, int G, class PtrAt>
__device__ __forceinline__ typename E::V fold_ring_vec(PtrAt ptr_at, int world, int start, int64_t off) {
    typename E::V acc[1];
    fold_ring_vecs<E, G, 1>(ptr_at, world, start, off, 0, acc);
    return acc[0];
}

// The binomial tree's fold (tree_kernels.cu, ring_tma.cu).
constexpr int kTreeGroup = 16;
// Binomial pairwise sum of load(0) .. load(world - 1), world <= W (W a power
// of two, at most 64).  Ranks are loaded and folded in groups of GS (levels
// 1, 2, .., GS/2 inside a group), then the group sums are folded at levels
// GS, 2 GS, .. -- exactly the tree's additions, in its order; GS bounds the
// loads in flight (and the registers they take).  W is a compile-time bound:
// the fold is unrolled with its bounds checked at run time, so a bound much
// larger than the world costs registers and, for bf16 adds, enough code to
// miss in the instruction cache (the TMA tree kernel compiled for 16 ranks
// ran 2 bf16 ranks at 0.4 of its fp32 speed, stalled on instruction fetch).
template <class T, int W = 64, int GS = (W < kTreeGroup ? W : kTreeGroup), class Add, class Load>
__device__ __forceinline__ T tree_fold(int world, Add add, Load load) {
    static_assert(W == 2 || W == 4 || W == 8 || W == 16 || W == 32 || W == 64, "W: a power of two up to 64");
    static_assert(GS >= 2 && GS <= W && (GS & (GS - 1)) == 0, "GS: a power of two up to W");
    constexpr int NG = W / GS;
    T gs[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        if (GS * g < world) {
            T v[GS];
#pragma unroll
            for (int i = 0; i < GS; ++i)
                if (GS * g + i < world) v[i] = load(GS * g + i);
#pragma unroll
            for (int d = 1; d < GS; d <<= 1)
#pragma unroll
                for (int i = 0; i < GS; i += 2 * d)
                    if (GS * g + i + d < world) v[i] = add(v[i], v[i + d]);
            gs[g] = v[0];
        }
    }
#pragma unroll
    for (int d = GS; d < W; d <<= 1)
#pragma unroll
        for (int g = 0; g < NG; g += 2 * d / GS)
            if (GS * g + d < world) gs[g] = add(gs[g], gs[g + d / GS]);
    return gs[0];
}

// Scalar version of the same fold for one element at element index `e`,
// its loads issued eight at a time.
template <class E, class PtrAt>
__device__ __forceinline__ typename E::S fold_ring_scalar(PtrAt ptr_at, int world, int start, int64_t e) {
    using S = typename E::S;
    constexpr int G = 8;
    S acc{};
    int r = start;
    for (int k0 = 0; k0 < world; k0 += G) {
        S x[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (k0 + g < world) {
                x[g] = reinterpret_cast<const S*>(ptr_at(r))[e];
                r = (r + 1 == world) ? 0 : r + 1;
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (k0 + g < world) acc = (k0 + g == 0) ? x[g] : E::sadd(acc, x[g]);
        }
    }
    return acc;
}

}  // namespace ddpk
