/*
 * ddp_oracle.c -- CPU oracle for DDP bucketed ring-allreduce gradient sync.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU library computes.  Only the test suite, the
 * package smoke check and the CPU-baseline leg of the benchmark may load it;
 * the product path never links, imports or calls it, and it shares no code,
 * header or table with the CUDA library.
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 * (no FMA contraction, no fast-math, so every float operation below is one
 * IEEE-754 binary32 operation rounded to nearest even, subnormals kept).
 * The same flags plus -fopenmp give the optional multi-core timing build.
 *
 * Sources (web pages on DDP gradient synchronisation):
 *   [P1] "DDP 与 Ring All-Reduce：梯度同步不是一次 AllReduce 就完事"
 *        (blog.vllbc.top), section 03 "两阶段：先规约，再扩散", "Bucket"
 *        and "Overlap" parts; section 04 (bandwidth accounting); section 05
 *        (DDP step timeline, divide by world size).
 *   [P2] "Day 17 · 梯度的集体行动" (blog.ans20xx.com), "bucket 与 overlap"
 *        and "源码心智伪代码" (wait -> div_(world_size) -> copy back).
 *   [P3] "DDP 与 Ring-AllReduce" (xuesongtap.github.io), §1.3.1 algorithm
 *        overview and §1.3.2 worked example (3 GPUs, length-6 vector).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - chunk size c = ceil(S/N); chunk j = [min(j*c,S), min((j+1)*c,S)),
 *     trailing chunks may be short or empty ([P1] §03 and [P3] §1.3.2 only
 *     show N | S);
 *   - rank r sends to rank r+1; reduce-scatter step s sends chunk
 *     (r-s) mod N, all-gather step t sends chunk (r-t+1) mod N -- the
 *     placement [P3] §1.3.2 prints for every step;
 *   - the receiver adds the incoming chunk into its own copy; bf16 adds are
 *     done in binary32 and rounded to bf16 after every hop;
 *   - after the last step every rank divides every element by the divisor
 *     (world size) with one IEEE division ([P1] §05, [P2] pseudo-code);
 *   - an fp16 ring (the fp16 compression hook of [P2]'s reading list on DDP
 *     communication hooks) works like the bf16 one: binary32 add of the two
 *     widened values, rounded to binary16 after every hop.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F16 2

/* Built with -fopenmp (the optional multi-core timing build only), the ranks
 * of one half-step run side by side: within a half-step every rank reads and
 * writes only its own buffer and message, so the per-element order of the
 * operations is the same as in the default single-threaded build. */
#ifdef _OPENMP
#define ORACLE_EACH_RANK _Pragma("omp parallel for schedule(static)")
#else
#define ORACLE_EACH_RANK
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

/* ------------------------------------------------------------------------ */
/* bfloat16 <-> binary32, written from the IEEE-754 definition.              */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bfloat16 keeps the top 16 bits of a binary32 value.  Widening is exact. */
float oracle_bf16_to_f32(uint16_t h) { return bits_f32(((uint32_t)h) << 16); }

/* Round a binary32 value to bfloat16, to nearest, ties to even.
 * The 16 discarded bits are compared against one half of the last kept
 * place (0x8000); above it rounds up, at exactly one half it rounds to the
 * kept value whose last bit is 0.  A carry out of the significand moves into
 * the exponent, which is what the IEEE definition asks for (largest finite
 * values round up to infinity).  NaN stays NaN and is made quiet. */
uint16_t oracle_bf16_rne(float f)
{
    uint32_t u = f32_bits(f);
    uint32_t exp = (u >> 23) & 0xFFu, man = u & 0x7FFFFFu;
    if (exp == 0xFFu && man != 0)                 /* NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

void oracle_bf16_rne_array(const float* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_bf16_rne(x[i]);
}

/* ------------------------------------------------------------------------ */
/* The reduction operator and the average.                                  */
/* ------------------------------------------------------------------------ */

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32, written from the IEEE-754 definition.         */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Widening to binary32 is exact (subnormals included). */
float oracle_fp16_to_f32(uint16_t h)
{
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t exp = ((uint32_t)h >> 10) & 0x1Fu, frac = (uint32_t)h & 0x3FFu;
    if (exp == 0x1Fu)                                  /* infinity or NaN */
        return bits_f32(sign | 0x7F800000u | (frac << 13));
    if (exp == 0) {                                    /* zero or subnormal: frac * 2^-24, exact */
        float v = (float)frac * (1.0f / 16777216.0f);
        return bits_f32(f32_bits(v) | sign);
    }
    return bits_f32(sign | ((exp - 15u + 127u) << 23) | (frac << 13));
}

/* Round a binary32 value to binary16, to nearest, ties to even.  The value is
 * sig * 2^(E-23) with a 24-bit significand sig; in the normal range of
 * binary16 (E >= -14) 11 significant bits are kept, below it the result is a
 * multiple of 2^-24 (subnormal).  The dropped bits are compared with half of
 * the last kept place; a carry out of the kept bits moves into the exponent,
 * and values at or beyond 65520 become infinity.  NaN stays NaN, quiet. */
uint16_t oracle_fp16_rne(float f)
{
    uint32_t u = f32_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t exp = (u >> 23) & 0xFFu, man = u & 0x7FFFFFu;
    if (exp == 0xFFu) return (uint16_t)(sign | 0x7C00u | (man ? 0x0200u | (man >> 13) : 0u));
    if (exp == 0 && man == 0) return sign;
    int32_t E = exp ? (int32_t)exp - 127 : -126;
    uint64_t sig = exp ? (man | 0x800000u) : man;
    uint32_t shift = E >= -14 ? 13u : (uint32_t)(13 + (-14 - E));     /* bits dropped from sig */
    if (shift > 40) return sign;                                      /* far below half the least subnormal */
    uint64_t kept = sig >> shift, rem = sig & ((1ull << shift) - 1u), half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (kept & 1u))) kept += 1u;
    if (E >= -14) {
        int32_t be = E + 15;                                          /* biased exponent */
        if (kept == 0x800u) { kept >>= 1; be += 1; }                  /* carry into the exponent */
        if (be >= 31) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | ((uint32_t)be << 10) | (uint32_t)(kept & 0x3FFu));
    }
    return (uint16_t)(sign | (uint32_t)kept);          /* subnormal; kept == 0x400 is the least normal */
}

void oracle_fp16_rne_array(const float* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_fp16_rne(x[i]);
}

void oracle_fp16_to_f32_array(const uint16_t* h, float* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_fp16_to_f32(h[i]);
}

static size_t elem_size(int dtype) { return dtype == ORACLE_F32 ? 4u : 2u; }

/* dst[i] <- dst[i] (+) src[i] : binary32 add, or for bf16 a binary32 add of
 * the two widened values rounded back to bf16 (one rounding per hop). */
static void add_into(int dtype, void* dst, const void* src, int64_t n)
{
    if (dtype == ORACLE_F32) {
        float* d = (float*)dst;
        const float* s = (const float*)src;
        for (int64_t i = 0; i < n; ++i) d[i] = d[i] + s[i];
    } else if (dtype == ORACLE_F16) {
        uint16_t* d = (uint16_t*)dst;
        const uint16_t* s = (const uint16_t*)src;
        for (int64_t i = 0; i < n; ++i)
            d[i] = oracle_fp16_rne(oracle_fp16_to_f32(d[i]) + oracle_fp16_to_f32(s[i]));
    } else {
        uint16_t* d = (uint16_t*)dst;
        const uint16_t* s = (const uint16_t*)src;
        for (int64_t i = 0; i < n; ++i)
            d[i] = oracle_bf16_rne(oracle_bf16_to_f32(d[i]) + oracle_bf16_to_f32(s[i]));
    }
}

/* x[i] <- x[i] / divisor, one IEEE division per element. */
static void divide_all(int dtype, void* x, int64_t n, int32_t divisor)
{
    float dv = (float)divisor;
    if (dtype == ORACLE_F32) {
        float* p = (float*)x;
        for (int64_t i = 0; i < n; ++i) p[i] = p[i] / dv;
    } else if (dtype == ORACLE_F16) {
        uint16_t* p = (uint16_t*)x;
        for (int64_t i = 0; i < n; ++i) p[i] = oracle_fp16_rne(oracle_fp16_to_f32(p[i]) / dv);
    } else {
        uint16_t* p = (uint16_t*)x;
        for (int64_t i = 0; i < n; ++i) p[i] = oracle_bf16_rne(oracle_bf16_to_f32(p[i]) / dv);
    }
}

/* ------------------------------------------------------------------------ */
/* Ring allreduce: N ranks, each with S elements, two phases of N-1 steps.   */
/* ------------------------------------------------------------------------ */

static int64_t chunk_len_of(int64_t S, int32_t N) { return N > 0 ? (S + N - 1) / N : 0; }

static void chunk_range(int64_t S, int32_t N, int32_t j, int64_t* lo, int64_t* hi)
{
    int64_t c = chunk_len_of(S, N);
    int64_t a = (int64_t)j * c, b = a + c;
    *lo = a < S ? a : S;
    *hi = b < S ? b : S;
}

static int32_t mod(int64_t a, int32_t n) { int64_t m = a % n; return (int32_t)(m < 0 ? m + n : m); }

/* Simulate the ring on `world` rank buffers of `numel` elements each.
 *
 * bufs[r]   : rank r's buffer (float32, or bf16 bit patterns), updated in place.
 * divisor   : 0 or 1 = leave the sum; otherwise divide by it after the last step.
 * n_steps   : -1 = run the whole allreduce (2(N-1) steps, then the divide);
 *             k in [0, 2(N-1)] = stop after the first k steps, no divide
 *             (used to inspect the intermediate states the worked example prints).
 * sent      : optional [world] array; sent[r] += elements rank r put on the ring.
 *
 * Every step has two halves, as on a real ring where all ranks send and
 * receive at once: first every rank copies the chunk it sends into its own
 * outgoing message, then every rank takes its left neighbour's message and
 * adds it in (reduce-scatter) or stores it (all-gather).
 */
int oracle_ring_allreduce(int32_t world, int64_t numel, int32_t dtype, void** bufs,
                          int32_t divisor, int32_t n_steps, int64_t* sent)
{
    if (world < 1 || numel < 0 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) ||
        divisor < 0 || !bufs)
        return ORACLE_EINVAL;
    for (int32_t r = 0; r < world; ++r)
        if (!bufs[r] && numel > 0) return ORACLE_EINVAL;
    const int32_t total_steps = 2 * (world - 1);
    if (n_steps < -1 || n_steps > total_steps) return ORACLE_EINVAL;
    const int32_t run = n_steps < 0 ? total_steps : n_steps;

    const size_t es = elem_size(dtype);
    const int64_t c = chunk_len_of(numel, world);
    char** msg = (char**)calloc((size_t)world, sizeof(char*));
    int64_t* msg_lo = (int64_t*)calloc((size_t)world, sizeof(int64_t));
    int64_t* msg_len = (int64_t*)calloc((size_t)world, sizeof(int64_t));
    if (!msg || !msg_lo || !msg_len) { free(msg); free(msg_lo); free(msg_len); return ORACLE_ENOMEM; }
    for (int32_t r = 0; r < world; ++r) {
        msg[r] = (char*)malloc(c > 0 ? (size_t)c * es : 1u);
        if (!msg[r]) {
            for (int32_t q = 0; q < r; ++q) free(msg[q]);
            free(msg); free(msg_lo); free(msg_len);
            return ORACLE_ENOMEM;
        }
    }

    for (int32_t step = 1; step <= run; ++step) {
        const int reduce = step <= world - 1;            /* phase 1: reduce-scatter */
        const int32_t s = reduce ? step : step - (world - 1);
        /* send half: rank r puts chunk (r-s) (reduce-scatter) or (r-s+1) (all-gather) */
        ORACLE_EACH_RANK
        for (int32_t r = 0; r < world; ++r) {
            int32_t j = reduce ? mod((int64_t)r - s, world) : mod((int64_t)r - s + 1, world);
            int64_t lo, hi;
            chunk_range(numel, world, j, &lo, &hi);
            msg_lo[r] = lo;
            msg_len[r] = hi - lo;
            if (hi > lo) memcpy(msg[r], (char*)bufs[r] + (size_t)lo * es, (size_t)(hi - lo) * es);
            if (sent) sent[r] += hi - lo;
        }
        /* receive half: rank r takes the message of rank r-1 */
        ORACLE_EACH_RANK
        for (int32_t r = 0; r < world; ++r) {
            int32_t left = mod((int64_t)r - 1, world);
            char* dst = (char*)bufs[r] + (size_t)msg_lo[left] * es;
            if (msg_len[left] == 0) continue;
            if (reduce) add_into(dtype, dst, msg[left], msg_len[left]);
            else memcpy(dst, msg[left], (size_t)msg_len[left] * es);
        }
    }

    if (n_steps < 0 && divisor > 1) {
        ORACLE_EACH_RANK
        for (int32_t r = 0; r < world; ++r) divide_all(dtype, bufs[r], numel, divisor);
    }

    for (int32_t r = 0; r < world; ++r) free(msg[r]);
    free(msg); free(msg_lo); free(msg_len);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Tree allreduce: binomial-tree reduce to rank 0, divide, broadcast back.    */
/* ------------------------------------------------------------------------ */

/* The pages name a tree-based allreduce as the alternative to the ring for
 * small messages ([P1] section 02 and section 07, NCCL's Tree algorithm and
 * its small-message threshold) without spelling it out.  Reading taken: a
 * binomial tree over the whole vector.  Reduce steps use distances
 * d = 1, 2, 4, ... < N: every rank r with r mod 2d == d sends its buffer to
 * rank r - d, which adds it into its own (receiver's value first).  After the
 * last reduce step rank 0 holds the sum and divides it.  Broadcast steps use
 * the same distances in reverse: every rank r with r mod 2d == 0 and
 * r + d < N sends its buffer to r + d, which stores it.  Each step is again
 * "all send, then all receive".
 *
 * n_steps: -1 = everything (reduce, divide, broadcast); k = stop after the
 * first k of the 2 * ceil(log2 N) steps, no divide. */
static int32_t tree_depth(int32_t N)
{
    int32_t L = 0;
    while ((1 << L) < N) ++L;
    return L;
}

int oracle_tree_allreduce(int32_t world, int64_t numel, int32_t dtype, void** bufs, int32_t divisor,
                          int32_t n_steps, int64_t* sent)
{
    if (world < 1 || numel < 0 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16) || divisor < 0 || !bufs)
        return ORACLE_EINVAL;
    for (int32_t r = 0; r < world; ++r)
        if (!bufs[r] && numel > 0) return ORACLE_EINVAL;
    const int32_t depth = tree_depth(world);
    const int32_t total_steps = 2 * depth;
    if (n_steps < -1 || n_steps > total_steps) return ORACLE_EINVAL;
    const int32_t run = n_steps < 0 ? total_steps : n_steps;
    const size_t es = elem_size(dtype);
    const size_t bytes = (size_t)numel * es;
    char** msg = (char**)calloc((size_t)world, sizeof(char*));
    if (!msg) return ORACLE_ENOMEM;
    for (int32_t r = 0; r < world; ++r) {
        msg[r] = (char*)malloc(bytes ? bytes : 1u);
        if (!msg[r]) {
            for (int32_t q = 0; q < r; ++q) free(msg[q]);
            free(msg);
            return ORACLE_ENOMEM;
        }
    }
    for (int32_t step = 0; step < run; ++step) {
        const int reduce = step < depth;
        const int32_t d = reduce ? (1 << step) : (1 << (total_steps - 1 - step));
        /* send half */
        for (int32_t r = 0; r < world; ++r) {
            const int sends = reduce ? (r % (2 * d) == d) : (r % (2 * d) == 0 && r + d < world);
            if (!sends) continue;
            memcpy(msg[r], bufs[r], bytes);
            if (sent) sent[r] += numel;
        }
        /* receive half */
        for (int32_t r = 0; r < world; ++r) {
            if (reduce) {
                if (r % (2 * d) == 0 && r + d < world) add_into(dtype, bufs[r], msg[r + d], numel);
            } else {
                if (r % (2 * d) == d) memcpy(bufs[r], msg[r - d], bytes);
            }
        }
        if (n_steps < 0 && reduce && step == depth - 1 && divisor > 1)
            divide_all(dtype, bufs[0], numel, divisor);
    }
    if (n_steps < 0 && depth == 0 && divisor > 1) divide_all(dtype, bufs[0], numel, divisor);
    for (int32_t r = 0; r < world; ++r) free(msg[r]);
    free(msg);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Bucket plan: reverse registration order, first-bucket cap then bucket cap. */
/* ------------------------------------------------------------------------ */

/* Parameters are visited from the last registered to the first, the order
 * in which backward produces their gradients ([P1] §03 "Overlap", §05 step 2).
 * Each is appended to the open bucket at the bucket's running element count
 * (no padding).  Once the open bucket's bytes reach its cap it is closed; the
 * first bucket's cap is first_cap_bytes (1 MiB by default) and every later
 * bucket's is cap_bytes (25 MiB by default) ([P1] §03 "Bucket").  A bucket
 * left open at the end is closed if it holds any parameter.
 *
 * Outputs: bucket_of[p], offset_of[p] (elements, inside its bucket),
 * bucket_numel[k] (room for n_params entries), *n_buckets. */
int oracle_plan_buckets(int32_t n_params, const int64_t* numel, int64_t elem_bytes,
                        int64_t first_cap_bytes, int64_t cap_bytes,
                        int32_t* bucket_of, int64_t* offset_of, int64_t* bucket_numel,
                        int32_t* n_buckets)
{
    if (n_params < 0 || elem_bytes <= 0 || first_cap_bytes <= 0 || cap_bytes <= 0 || !n_buckets)
        return ORACLE_EINVAL;
    if (n_params > 0 && (!numel || !bucket_of || !offset_of || !bucket_numel)) return ORACLE_EINVAL;
    int32_t k = 0;             /* index of the open bucket */
    int64_t elems = 0;         /* elements already in the open bucket */
    int32_t members = 0;       /* parameters already in the open bucket */
    for (int32_t p = n_params - 1; p >= 0; --p) {
        if (numel[p] < 0) return ORACLE_EINVAL;
        bucket_of[p] = k;
        offset_of[p] = elems;
        elems += numel[p];
        members += 1;
        int64_t cap = (k == 0) ? first_cap_bytes : cap_bytes;
        if (elems * elem_bytes >= cap) {
            bucket_numel[k] = elems;
            k += 1;
            elems = 0;
            members = 0;
        }
    }
    if (members > 0) {
        bucket_numel[k] = elems;
        k += 1;
    }
    *n_buckets = k;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Copies between gradients and one rank's bucket; local accumulation.       */
/* ------------------------------------------------------------------------ */

/* bucket[offset[i] : offset[i]+numel[i]] <- grads[i]  (one rank). */
void oracle_bucket_pack(int32_t n, void* const* grads, const int64_t* numel, const int64_t* offset,
                        void* bucket, int64_t elem_bytes)
{
    for (int32_t i = 0; i < n; ++i)
        if (numel[i] > 0)
            memcpy((char*)bucket + offset[i] * elem_bytes, grads[i], (size_t)(numel[i] * elem_bytes));
}

/* grads[i] <- bucket[offset[i] : offset[i]+numel[i]]  (one rank). */
void oracle_bucket_unpack(int32_t n, void* const* grads, const int64_t* numel, const int64_t* offset,
                          const void* bucket, int64_t elem_bytes)
{
    for (int32_t i = 0; i < n; ++i)
        if (numel[i] > 0)
            memcpy(grads[i], (const char*)bucket + offset[i] * elem_bytes, (size_t)(numel[i] * elem_bytes));
}

/* acc[i] <- acc[i] (+) g[i]: one no_sync micro-batch folded into the local
 * gradient ([P1] §03 and §05 step 5; [P2] "梯度累积:正确使用 no_sync"). */
int oracle_accumulate(int32_t dtype, void* acc, const void* g, int64_t n)
{
    if ((dtype != ORACLE_F32 && dtype != ORACLE_BF16) || n < 0) return ORACLE_EINVAL;
    if (n > 0) add_into(dtype, acc, g, n);
    return ORACLE_OK;
}
