// schedule.cu -- CSR block schedules on the GPU: the dense causal CSR and the topology
// schedule (sink blocks, local window, top-k blocks by elder-rule salience over key-block
// centroids).
//
// Method: "Add topology-derived sparse attention kernel" (triton-lang/kernels#22), Summary
// (schedule from sink blocks, local-window blocks and a 0D-persistence-style salience over
// key-block centroids; dense causal CSR layout); the PR's mirror page, port note (the
// salience is the elder rule, exactly one block scores zero, a size tie is broken by index)
// and the world-model commit's schedule.py bullet (the salience follows from MST edges alone).
//
// The result is bit-identical to the CPU oracle because every floating-point step is fixed:
//   C[b][d]  = (sum over lanes of (sum over the block's tokens, ascending)) / (block * lanes)
//   d2(u,v)  = sum of (C[u][d] - C[v][d])^2 in a fixed order: 32 partial sums over
//              d = j mod 32 (ascending, fused multiply-add), then halving
//   ordering = strict key (d2, min(u,v), max(u,v)), so the MST is unique and Boruvka here
//              selects the same tree as Kruskal in the oracle.
//
// Kernels, in stream order:
//   centroid_partial      per (lane, block, d): sum of the block's tokens   (HBM stream of K)
//   centroid_final        per (block, d): sum over lanes, divide; also the binary32 copy
//   pairwise_bounds       per pair: an interval [lo, hi] that provably holds the binary64
//                         d2, from binary32 arithmetic                       (FP32 ALU)
//   schedule_graph_kernel one cooperative launch: Boruvka MST (exact binary64 d2 only for
//                         the edges whose interval can still hold a minimum), elder-rule
//                         salience, top-k CSR (see the section comment below)
// This part runs binary64 at a small fraction of its binary32 rate, so the nb^2 x D binary64
// distance matrix would cost more than all other schedule work together; Boruvka needs the
// exact key only to decide between edges whose intervals overlap the smallest upper bound.
#include <climits>

#include "tsa_device.cuh"
#include "tsa_internal.h"

namespace tsa {
namespace {

constexpr uint64_t kInfBits = 0x7FF0000000000000ull;  // +inf as binary64 bits

__device__ __forceinline__ double widen(uint16_t bits, bool bf16) {
    if (bf16) return (double)__uint_as_float((uint32_t)bits << 16);
    return (double)__half2float(__ushort_as_half(bits));
}

// ---------------------------------------------------------------- centroids
// part[l][b][d] = sum_{t=0}^{block-1} K[l][b*block+t][d], added in ascending t in binary64.
//
// FP64 runs at a small fraction of the FP32 rate on this part, so the sum is formed exactly
// in int64 fixed point whenever that provably equals the sequential binary64 sum:
//  * f16 elements are integer multiples of 2^-24 below 2^16 in magnitude, so every partial
//    sum of up to 4096 of them is a multiple of 2^-24 below 2^40 * 2^12 = 2^52: exactly
//    representable, hence the sequential binary64 sum is exact and equals the integer sum.
//  * bf16 elements with biased exponent e hold (128 + frac) * 2^(e - 134).  If all non-zero
//    elements of a column have e in [94, 142] (ulp >= 2^-40, |x| < 2^16), the column fits an
//    int64 in units of 2^-40 (block <= 64: |sum| < 2^62).  If moreover e_max - e_min <=
//    45 - ceil(log2(block)), every partial sum is a multiple of 2^(e_min - 134) below
//    2^(e_max - 126) * block <= 2^(e_min - 134 + 53), so again the sequential binary64 sum is
//    exact and equals the integer sum.
// A column that meets neither condition (subnormal, huge or widely spread values, inf/nan)
// is summed again the plain way, in binary64 in ascending t.
struct ColumnSum {
    long long acc;
    int emin, emax;
    bool bad;
};

__device__ __forceinline__ void col_init(ColumnSum &c) {
    c.acc = 0;
    c.emin = 1 << 20;
    c.emax = -(1 << 20);
    c.bad = false;
}

__device__ __forceinline__ void col_add(ColumnSum &c, uint32_t h, bool bf16) {
    const bool neg = (h & 0x8000u) != 0;
    long long mag;
    if (bf16) {
        const int e = (int)((h >> 7) & 0xFFu);
        const bool nonzero = (h & 0x7FFFu) != 0;
        const bool in_window = e >= 94 && e <= 142;
        const int sh = in_window ? e - 94 : 0;
        mag = (long long)((h & 0x7Fu) | 0x80u) << sh;
        if (!nonzero) mag = 0;
        if (nonzero) {
            c.emin = min(c.emin, e);
            c.emax = max(c.emax, e);
            c.bad |= !in_window;
        }
    } else {
        const int e = (int)((h >> 10) & 0x1Fu);
        const uint32_t f = h & 0x3FFu;
        c.bad |= (e == 31);
        mag = e ? ((long long)(0x400u | f) << (e - 1)) : (long long)f;  // units of 2^-24, < 2^40
    }
    c.acc += neg ? -mag : mag;
}

// True when the integer sum equals the sequential binary64 sum (see above).
__device__ __forceinline__ bool col_exact(const ColumnSum &c, bool bf16, int64_t block,
                                          int spread_limit) {
    if (c.bad) return false;
    if (!bf16) return block <= 4096;
    if (block > 64) return false;
    return c.emax < c.emin || c.emax - c.emin <= spread_limit;  // emax < emin: all zero
}

__device__ __forceinline__ double col_value(const ColumnSum &c, bool bf16) {
    return bf16 ? ldexp((double)c.acc, -40) : ldexp((double)c.acc, -24);
}

// Sequential binary64 sum of one column (the reference order), used for columns that none
// of the exact fast paths covers.
__device__ double column_sum_exact_slow(const uint16_t *src, int64_t D, int64_t block, bool bf16,
                                        int spread_limit) {
    ColumnSum c;
    col_init(c);
    for (int64_t t = 0; t < block; ++t) col_add(c, __ldg(src + t * D), bf16);
    if (col_exact(c, bf16, block, spread_limit)) return col_value(c, bf16);
    double acc = 0.0;
    for (int64_t t = 0; t < block; ++t) acc += widen(__ldg(src + t * D), bf16);
    return acc;
}

// One thread per (lane, block, 8 consecutive d); 16-byte loads; the int64 path above.  Used
// for bf16 keys in blocks longer than 64 tokens (the TwoSum bound below covers 64 terms); the
// streamed kernel further down takes every other 16-byte-aligned case.
__global__ void __launch_bounds__(256, 2) centroid_partial_vec8(const uint16_t *__restrict__ K, bool bf16, int64_t lanes,
                                      int64_t S, int64_t D, int64_t block, int64_t nb,
                                      int spread_limit, double *__restrict__ part) {
    const int64_t groups = D / 8;
    const int64_t total = lanes * nb * groups;
    for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < total;
         w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = w % groups;
        const int64_t lb = w / groups;  // l * nb + b
        const int64_t l = lb / nb, b = lb % nb;
        const int64_t n = (b + 1) * block <= S ? block : S - b * block;  // tokens in the block
        const uint16_t *src = K + ((l * S + b * block) * D + g * 8);
        double *dst = part + lb * D + g * 8;
        ColumnSum c[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) col_init(c[i]);
        int64_t t = 0;
        for (; t + 8 <= n; t += 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldg(reinterpret_cast<const uint4 *>(src + (t + u) * D));
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    col_add(c[2 * i], w4[i] & 0xFFFFu, bf16);
                    col_add(c[2 * i + 1], w4[i] >> 16, bf16);
                }
            }
        }
        for (; t < n; ++t) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src + t * D));
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                col_add(c[2 * i], w4[i] & 0xFFFFu, bf16);
                col_add(c[2 * i + 1], w4[i] >> 16, bf16);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (col_exact(c[i], bf16, n, spread_limit)) {
                dst[i] = col_value(c[i], bf16);
            } else {
                double acc = 0.0;
                for (int64_t tt = 0; tt < n; ++tt) acc += widen(__ldg(src + tt * D + i), bf16);
                dst[i] = acc;
            }
        }
    }
}

// The same sums for small grids (a few hundred items or fewer, where one thread per item would
// leave most SMs idle and each thread a long chain of rows): one warp per (lane, block, 8
// consecutive d).  Lane t adds tokens t, t + 32, ... into the int64 column sums of the path
// above; the warp then combines them (integer addition is associative, and the exponent range
// and the out-of-window flag combine by min / max / or), so the sums, and the test of whether
// they equal the sequential binary64 sum, are those of a single thread walking the block.
// Columns that fail the test are summed the plain way.
__global__ void __launch_bounds__(256) centroid_partial_warp(const uint16_t *__restrict__ K, bool bf16, int64_t lanes,
                                                             int64_t S, int64_t D, int64_t block, int64_t nb,
                                                             int spread_limit, double *__restrict__ part) {
    const int lane = threadIdx.x & 31;
    const int64_t groups = D / 8;
    const int64_t total = lanes * nb * groups;
    const int64_t wpb = blockDim.x >> 5;
    for (int64_t w = blockIdx.x * wpb + (threadIdx.x >> 5); w < total; w += (int64_t)gridDim.x * wpb) {
        const int64_t g = w % groups;
        const int64_t lb = w / groups;  // l * nb + b
        const int64_t l = lb / nb, b = lb % nb;
        const int64_t n = (b + 1) * block <= S ? block : S - b * block;  // tokens in the block
        const uint16_t *src = K + ((l * S + b * block) * D + g * 8);
        double *dst = part + lb * D + g * 8;
        ColumnSum c[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) col_init(c[i]);
        for (int64_t t = lane; t < n; t += 32) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src + t * D));
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                col_add(c[2 * i], w4[i] & 0xFFFFu, bf16);
                col_add(c[2 * i + 1], w4[i] >> 16, bf16);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                c[i].acc += __shfl_xor_sync(0xffffffffu, c[i].acc, off);
                c[i].emin = min(c[i].emin, __shfl_xor_sync(0xffffffffu, c[i].emin, off));
                c[i].emax = max(c[i].emax, __shfl_xor_sync(0xffffffffu, c[i].emax, off));
                c[i].bad = __any_sync(0xffffffffu, c[i].bad);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (lane == i) {
                if (col_exact(c[i], bf16, n, spread_limit)) {
                    dst[i] = col_value(c[i], bf16);
                } else {
                    double acc = 0.0;
                    for (int64_t tt = 0; tt < n; ++tt) acc += widen(__ldg(src + tt * D + i), bf16);
                    dst[i] = acc;
                }
            }
        }
    }
}

// Block sums with 16-byte rows streamed: each thread copies its next rows into shared memory
// with cp.async while it sums earlier ones, so a thread always has loads in flight instead of
// alternating between loading and summing.  The staging area is [stage][row][thread]
// (16-byte words), so the 32 lanes of a warp touch consecutive words.  One thread per (lane,
// block, 8 consecutive d); tokens in ascending order.  f16 keys take the int64 path above.
//
// bf16 fast path: the column is summed as an unevaluated pair hi + lo of fp32 values (packed
// two columns at a time).  Each step is Knuth's TwoSum, which splits hi + x exactly into the
// rounded sum and its error; the errors collect in lo.  Every element and every error is an
// integer multiple of 2^(e_min - 134), each error is below 2^(e_max - 143) in magnitude, so
// lo's partial sums (64 of them) need at most e_max - e_min - 4 significant bits: with
// e_max - e_min <= 28 (biased exponents of the non-zero elements, from the packed 16-bit
// max/min of |bits|; subnormals count as exponent 1; no inf/nan) lo is exact, hence
// hi + lo is the exact column sum.  That sum has at most e_max - e_min + 14 <= 42 significant
// bits, so the sequential binary64 sum is exact too and both equal (double)hi + (double)lo.
// Other columns take the sequential binary64 loop (column_sum_exact_slow).
//
// f16 keys in blocks of at most 64 tokens take the same pair (the int64 path costs ~15 integer
// operations per element and left the pass ALU-bound).  With biased exponents E (subnormals
// counted as 1) every element and every error is a multiple of 2^(E_min - 25), each element is
// below 2^(E_max - 14) and hi below 2^(E_max - 8), so each error is below 2^(E_max - 33) and
// lo's partial sums below 2^(E_max - 27): E_max - E_min - 2 significant bits, exact in fp32
// for E_max - E_min <= 26 (25 is required, and E_max <= 30: no inf/nan).  The column sum then
// has at most E_max - E_min + 17 <= 42 significant bits, so as above the sequential binary64
// sum is exact and equals (double)hi + (double)lo.

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Two shapes: large problems keep three chunks of 8 rows in flight per thread (256 threads,
// 96 KB, two CTAs per SM); small ones (a few CTAs) put a whole 64-row block in flight at once
// (64 threads, 64 KB) so the pass costs one memory round trip instead of eight.
template <int kThreads, int kStages>
struct StreamShape {
    static constexpr int kSmem = kStages * 8 * kThreads * 16;
};

// kTwoSum: the hi + lo pair (bf16, or f16 in blocks of at most 64 tokens); otherwise the
// int64 column sums (f16 in longer blocks).
template <int kThreads, int kStages, bool kBF16, bool kTwoSum>
__global__ void __launch_bounds__(kThreads, kThreads == 256 ? 2 : 1)
centroid_partial_stream(const uint16_t *__restrict__ K, int64_t lanes, int64_t S, int64_t D, int64_t block,
                        int64_t nb, int spread_limit, double *__restrict__ part) {
    static_assert(kTwoSum || !kBF16, "bf16 keys take the pair");
    extern __shared__ __align__(16) uint4 stage[];
    const uint32_t stage0 = smem_u32(stage) + threadIdx.x * 16u;
    const int64_t groups = D / 8;
    const int64_t total = lanes * nb * groups;
    for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < total;
         w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = w % groups;
        const int64_t lb = w / groups;  // l * nb + b
        const int64_t l = lb / nb, b = lb % nb;
        const int64_t n = (b + 1) * block <= S ? block : S - b * block;  // tokens in the block
        const uint16_t *src = K + ((l * S + b * block) * D + g * 8);
        double *dst = part + lb * D + g * 8;
        // pair state: hi + lo pairs and packed |bits| max/min; otherwise int64 column sums
        uint64_t hi[4], lo[4];
        uint32_t mx[4], mn[4];
        ColumnSum cs[kTwoSum ? 1 : 8];
        if constexpr (kTwoSum) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                hi[i] = f2_pack(0.f, 0.f);
                lo[i] = hi[i];
                mx[i] = 0u;
                mn[i] = 0xFFFFFFFFu;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) col_init(cs[i]);
        }
        auto add_word = [&](int i, uint32_t x) {
            if constexpr (kTwoSum) {
                // hi + lo += x exactly (TwoSum), two columns per packed operation
                uint64_t v;
                if constexpr (kBF16) {
                    v = f2_pack(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
                } else {
                    const float2 xf = __half22float2(*reinterpret_cast<const __half2 *>(&x));
                    v = f2_pack(xf.x, xf.y);  // low half first, as for bf16
                }
                const uint64_t s = f2_add(hi[i], v);
                const uint64_t bv = f2_sub(s, hi[i]);
                const uint64_t err = f2_add(f2_sub(hi[i], f2_sub(s, bv)), f2_sub(v, bv));
                lo[i] = f2_add(lo[i], err);
                hi[i] = s;
                const uint32_t a = x & 0x7FFF7FFFu;
                mx[i] = __vmaxu2(mx[i], a);
                // minimum of |bits| - 1 per half: a zero wraps to 0xFFFF and never lowers it
                mn[i] = __vminu2(mn[i], __vsub2(a, 0x00010001u));
            } else {
                col_add(cs[2 * i], x & 0xFFFFu, false);
                col_add(cs[2 * i + 1], x >> 16, false);
            }
        };
        auto add_row = [&](const uint4 v) {
            add_word(0, v.x);
            add_word(1, v.y);
            add_word(2, v.z);
            add_word(3, v.w);
        };
        const int64_t chunks = n >> 3;  // whole chunks of 8 tokens
        const int64_t full = chunks << 3;
        // Ring of kStages chunks; one commit group per chunk slot (empty past the end), so
        // wait_group<kStages - 1> always means "chunk c has landed".
        auto issue = [&](int64_t c) {
            if (c < chunks) {
                const int buf = (int)(c % kStages);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    cp_async16(stage0 + (uint32_t)((buf * 8 + u) * kThreads * 16), src + (c * 8 + u) * D);
            }
            cp_async_commit();
        };
#pragma unroll
        for (int c = 0; c < kStages - 1; ++c) issue(c);
        for (int64_t c = 0; c < chunks; ++c) {
            issue(c + kStages - 1);
            cp_async_wait<kStages - 1>();
            const int buf = (int)(c % kStages);
#pragma unroll
            for (int u = 0; u < 8; ++u) add_row(stage[(buf * 8 + u) * kThreads + threadIdx.x]);
        }
        cp_async_wait<0>();
        for (int64_t t = full; t < n; ++t) add_row(__ldg(reinterpret_cast<const uint4 *>(src + t * D)));
        if constexpr (kTwoSum) {
            constexpr int kMantBits = kBF16 ? 7 : 10;     // explicit mantissa bits
            constexpr int kMaxExp = kBF16 ? 240 : 30;     // no fp32 overflow / no inf, nan
            constexpr int kMaxSpread = kBF16 ? 28 : 25;   // lo stays exact (see above)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float h0, h1, l0, l1;
                f2_unpack(hi[i], h0, h1);
                f2_unpack(lo[i], l0, l1);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t amax = (mx[i] >> (16 * h)) & 0xFFFFu;
                    const uint32_t amin_m1 = (mn[i] >> (16 * h)) & 0xFFFFu;
                    const uint32_t amin = amin_m1 == 0xFFFFu ? 0xFFFFu : amin_m1 + 1u;  // 0xFFFF: all zero
                    const int emax = (int)(amax >> kMantBits);
                    const int emin = max(1, (int)(amin >> kMantBits));
                    const bool all_zero = amin == 0xFFFFu;
                    const bool exact = all_zero || (emax <= kMaxExp && emax - emin <= kMaxSpread);
                    dst[2 * i + h] = exact ? (double)(h ? h1 : h0) + (double)(h ? l1 : l0)
                                           : column_sum_exact_slow(src + 2 * i + h, D, n, kBF16, spread_limit);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (col_exact(cs[i], false, n, spread_limit)) {
                    dst[i] = col_value(cs[i], false);
                } else {
                    double acc = 0.0;
                    for (int64_t tt = 0; tt < n; ++tt) acc += widen(__ldg(src + tt * D + i), false);
                    dst[i] = acc;
                }
            }
        }
    }
}

// Same sums, one d per thread (any D, any alignment).
__global__ void centroid_partial_scalar(const uint16_t *__restrict__ K, bool bf16, int64_t lanes,
                                        int64_t S, int64_t D, int64_t block, int64_t nb,
                                        int spread_limit, double *__restrict__ part) {
    const int64_t total = lanes * nb * D;
    for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < total;
         w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t d = w % D;
        const int64_t lb = w / D;
        const int64_t l = lb / nb, b = lb % nb;
        const int64_t n = (b + 1) * block <= S ? block : S - b * block;  // tokens in the block
        const uint16_t *src = K + (l * S + b * block) * D + d;
        ColumnSum c;
        col_init(c);
        for (int64_t t = 0; t < n; ++t) col_add(c, __ldg(src + t * D), bf16);
        if (col_exact(c, bf16, n, spread_limit)) {
            part[w] = col_value(c, bf16);
        } else {
            double acc = 0.0;
            for (int64_t t = 0; t < n; ++t) acc += widen(__ldg(src + t * D), bf16);
            part[w] = acc;
        }
    }
}

// C[b][d] = (sum_{l ascending} part[l][b][d]) / (n_b * lanes), n_b the tokens block b holds
// (block, or fewer for a partial last block).
// Pins eight loaded values in registers at this point: the loads that produced them are
// issued before it and the arithmetic that uses them comes after, so independent loads are in
// flight together instead of being interleaved with a dependent add chain.
__device__ __forceinline__ void hold8(double *v) {
    asm volatile("" : "+d"(v[0]), "+d"(v[1]), "+d"(v[2]), "+d"(v[3]), "+d"(v[4]), "+d"(v[5]), "+d"(v[6]), "+d"(v[7]));
}

// Binary32 copy of a centroid coordinate for the distance bounds.  Zero and magnitudes in
// [2^-60, 2^60] round to nearest as normal binary32 numbers (relative error <= 2^-24, and
// every difference of two of them is a normal number or zero); anything else becomes NaN,
// which makes every bound of that block's pairs the whole range [0, +inf].
__device__ __forceinline__ float bounds_copy(double x) {
    const double m = fabs(x);
    if (x == 0.0) return 0.0f;
    return (m >= 0x1p-60 && m <= 0x1p60) ? __double2float_rn(x) : __int_as_float(0x7fc00000);
}

__global__ void centroid_final(const double *__restrict__ part, int64_t lanes, int64_t nb,
                               int64_t D, int64_t S, int64_t block, double *__restrict__ C,
                               float *__restrict__ C32) {
    const int64_t n = nb * D;
    for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < n;
         w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = w / D;
        const int64_t n_b = (b + 1) * block <= S ? block : S - b * block;
        // lanes in ascending order; the loads of 16 lanes are issued before their adds
        double total = 0.0;
        int64_t l = 0;
        for (; l + 16 <= lanes; l += 16) {
            double v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __ldg(part + (l + i) * n + w);
            hold8(v);
            hold8(v + 8);
#pragma unroll
            for (int i = 0; i < 16; ++i) total += v[i];
        }
        for (; l < lanes; ++l) total += part[l * n + w];
        // A power-of-two divisor 2^k: multiplying by the exact 2^-k rounds the same exact
        // quotient as the division, without the binary64 divide's instruction sequence.
        const int64_t N = n_b * lanes;
        double c;
        if ((N & (N - 1)) == 0) {
            const int k = 63 - __clzll((long long)N);
            c = total * __longlong_as_double((long long)(1023 - k) << 52);
        } else {
            c = total / (double)N;
        }
        C[w] = c;
        C32[w] = bounds_copy(c);
    }
}

// ---------------------------------------------------------------- content order
// The content tie rule (the port note's fix for the index dependence of the elder rule) breaks
// every tie by centroid content: blocks compare lexicographically over d, each coordinate in
// IEEE 754 totalOrder, and only bit-identical centroids fall back to the index.  That order is
// strict and total, so it ranks the blocks 0..nb-1.  Running the index-rule pipeline on the
// centroids permuted into rank order applies exactly the content rule (every tie the index
// rule breaks by index is then broken by rank), and the salience is written back through the
// permutation.

// totalOrder of binary64 as an unsigned key: negative values reversed below the positives.
__device__ __forceinline__ unsigned long long total_order_key(double x) {
    const unsigned long long b = (unsigned long long)__double_as_longlong(x);
    return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

// One warp per block b: rank[b] = #{c : c before b}; perm[rank[b]] = b.
__global__ void content_rank(const double *__restrict__ C, int64_t nb, int64_t D, int *__restrict__ perm) {
    const int lane = threadIdx.x & 31;
    const int64_t b = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= nb) return;
    const double *cb = C + b * D;
    int count = 0;
    for (int64_t c = lane; c < nb; c += 32) {
        const double *cc = C + c * D;
        int64_t d = 0;
        unsigned long long kc = 0, kb = 0;
        for (; d < D; ++d) {
            kc = total_order_key(cc[d]);
            kb = total_order_key(cb[d]);
            if (kc != kb) break;
        }
        count += d < D ? (kc < kb) : (c < b);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) count += __shfl_xor_sync(0xffffffffu, count, off);
    if (lane == 0) perm[count] = (int)b;
}

// Cp[r][:] = C[perm[r]][:], and its binary32 copy
__global__ void permute_rows(const double *__restrict__ C, const int *__restrict__ perm, int64_t nb,
                             int64_t D, double *__restrict__ Cp, float *__restrict__ Cp32) {
    const int64_t n = nb * D;
    for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < n;
         w += (int64_t)gridDim.x * blockDim.x)
    {
        const int b = perm[w / D];
        const double c = (b >= 0 && b < nb) ? C[(int64_t)b * D + w % D] : 0.0;
        Cp[w] = c;
        Cp32[w] = bounds_copy(c);
    }
}

// ---------------------------------------------------------------- distance bounds
constexpr int kPbTile = 16;        // pairs per tile side
constexpr int kPbChunk = 32;       // d values staged per step
constexpr int kPbFlatBelow = 256;  // nb below which pairwise_bounds_flat runs instead

// An interval [lo, hi] that holds the binary64 squared distance the graph kernel (and the
// oracle) computes from (C_u[d] - C_v[d])^2 (exact_d2 below), given
//   s       the binary32 fma-chain sum of (a_d - b_d)^2, a and b the rows' binary32 copies;
//   na, nv  the binary32 fma-chain sums of a_d^2 and b_d^2;
//   rel     D * 2^-22 (D <= 1024).
// Error budget; every step below rounds outward, so the interval can only widen:
//   * |a_d - C_u[d]| <= 2^-24 |C_u[d]| (normal binary32 range, see bounds_copy) and the
//     binary32 subtraction adds at most 2^-24 |a_d - b_d|, so each computed difference
//     t_d = fl(a_d - b_d) is off from the exact C_u[d] - C_v[d] by e_d <= 2^-22 (|a_d| + |b_d|);
//   * hence s* = the exact sum of t_d^2 (the terms s accumulates) is off from the exact sum of
//     (C_u[d] - C_v[d])^2 by at most sum e_d (2 |t_d| + e_d) <= 2^-21 sqrt(N) sqrt(s*) + 2^-44 N,
//     with N = 2 (sum a^2 + sum b^2) >= sum (|a_d| + |b_d|)^2 (Cauchy-Schwarz);
//   * a binary32 recursive sum of D non-negative terms is within a factor 1 -+ D 2^-23 of its
//     exact value, plus at most D 2^-149 from terms that underflow (inside the 2^-120 slack);
//   * the binary64 sum rounds each term at most D / 32 + 8 times, so it is within a factor
//     1 -+ (D + 8) 2^-53 of the exact real sum, inside
//     the final factor 1 -+ 2^-20; no binary64 step under- or overflows for coordinates in
//     bounds_copy's range.
// NaN anywhere (a block outside that range) or a binary32 overflow gives [0, +inf].
__device__ __forceinline__ float2 d2_interval(float s, float na, float nv, float rel) {
    const float tiny = 0x1p-120f;
    const float up = 1.0f + rel, dn = 1.0f - rel;  // exact: rel is a multiple of 2^-22, <= 2^-12
    const float s_up = __fmul_ru(__fadd_ru(s, tiny), up);
    const float s_dn = __fmul_rd(__fsub_rd(s, tiny), dn);
    const float n_up = __fmul_ru(__fmul_ru(__fadd_ru(__fadd_ru(na, nv), tiny), up), 2.0f);
    const float e = __fmaf_ru(0x1p-21f, __fmul_ru(__fsqrt_ru(n_up), __fsqrt_ru(s_up)), __fmul_ru(0x1p-44f, n_up));
    float hi = __fmul_ru(__fadd_ru(s_up, e), 1.0f + 0x1p-20f);
    float lo = __fmul_rd(__fsub_rd(s_dn, e), 1.0f - 0x1p-20f);
    hi = hi <= 0x1.fffffep127f ? hi : __int_as_float(0x7f800000);  // NaN or overflow: +inf
    lo = lo > 0.0f ? lo : 0.0f;                                      // NaN or negative: 0
    return make_float2(lo, hi);
}

// B[u][v] = B[v][u] = the interval of d2(u, v).  One CTA per tile (tu <= tv) of the upper
// triangle, 256 threads, one pair each (many resident warps hide the staging loads); the
// tile's 32 rows get their squared norms from the same staged values (threads 0..31, one row
// each).  Chunks are zero-padded past D (a zero difference adds exactly nothing), and rows are
// 16-byte aligned in shared memory so that each thread reads four coordinates per load.  The
// binary32 arithmetic is symmetric in u and v, so the mirrored entry is the interval computed
// for (v, u).
constexpr int kPbThreads = kPbTile * kPbTile;
constexpr int kPbPitch = kPbChunk + 4;  // floats per staged row: 16-byte rows, no bank conflicts
__global__ void __launch_bounds__(kPbThreads) pairwise_bounds(const float *__restrict__ C, int64_t nb, int64_t D,
                                                              int tiles, float rel, float2 *__restrict__ B,
                                                              unsigned *__restrict__ gbar) {
    if (blockIdx.x == 0 && threadIdx.x < 4) gbar[threadIdx.x] = 0u;  // the graph kernel's barrier words
    __shared__ __align__(16) float cu[kPbTile][kPbPitch];
    __shared__ __align__(16) float cv[kPbTile][kPbPitch];
    __shared__ float nrm[2 * kPbTile];
    // linear tile index -> (tu, tv), tu <= tv, row-major over the upper triangle
    int k = blockIdx.x, tu = 0;
    while (k >= tiles - tu) { k -= tiles - tu; ++tu; }
    const int tv = tu + k;
    const int tid = threadIdx.x, tx = tid % kPbTile, ty = tid / kPbTile;
    const int64_t u0 = (int64_t)tu * kPbTile, v0 = (int64_t)tv * kPbTile;
    float acc = 0.0f, nacc = 0.0f;
    for (int64_t d0 = 0; d0 < D; d0 += kPbChunk) {
        for (int i = tid; i < kPbTile * kPbChunk; i += kPbThreads) {
            const int r = i / kPbChunk, c = i % kPbChunk;
            const int64_t d = d0 + c;
            cu[r][c] = (u0 + r < nb && d < D) ? C[(u0 + r) * D + d] : 0.0f;
            cv[r][c] = (v0 + r < nb && d < D) ? C[(v0 + r) * D + d] : 0.0f;
        }
        __syncthreads();
        if (tid < 2 * kPbTile) {
            const float *row = tid < kPbTile ? cu[tid] : cv[tid - kPbTile];
#pragma unroll
            for (int c = 0; c < kPbChunk; c += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(row + c);
                nacc = __fmaf_rn(x.x, x.x, nacc);
                nacc = __fmaf_rn(x.y, x.y, nacc);
                nacc = __fmaf_rn(x.z, x.z, nacc);
                nacc = __fmaf_rn(x.w, x.w, nacc);
            }
        }
#pragma unroll
        for (int c = 0; c < kPbChunk; c += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(&cu[ty][c]);
            const float4 b = *reinterpret_cast<const float4 *>(&cv[tx][c]);
            float t;
            t = __fsub_rn(a.x, b.x); acc = __fmaf_rn(t, t, acc);
            t = __fsub_rn(a.y, b.y); acc = __fmaf_rn(t, t, acc);
            t = __fsub_rn(a.z, b.z); acc = __fmaf_rn(t, t, acc);
            t = __fsub_rn(a.w, b.w); acc = __fmaf_rn(t, t, acc);
        }
        __syncthreads();
    }
    if (tid < 2 * kPbTile) nrm[tid] = nacc;
    __syncthreads();
    const int64_t u = u0 + ty, v = v0 + tx;
    if (u < nb && v < nb) {
        const float2 iv = d2_interval(acc, nrm[ty], nrm[kPbTile + tx], rel);
        B[u * nb + v] = iv;
        B[v * nb + u] = iv;
    }
}

// The same intervals for small nb, where the tiled kernel would run a handful of CTAs: one
// thread per pair u < v, 32 pairs per CTA.  The diagonal gets [0, 0] (a block is never an edge
// of its own component).
__global__ void __launch_bounds__(32) pairwise_bounds_flat(const float *__restrict__ C, int64_t nb, int64_t D,
                                                           float rel, float2 *__restrict__ B,
                                                           unsigned *__restrict__ gbar) {
    if (blockIdx.x == 0 && threadIdx.x < 4) gbar[threadIdx.x] = 0u;  // the graph kernel's barrier words
    const int64_t npairs = nb * (nb - 1) / 2;
    const int64_t p = (int64_t)blockIdx.x * 32 + threadIdx.x;
    if (p < nb) B[p * nb + p] = make_float2(0.0f, 0.0f);
    if (p >= npairs) return;
    // p -> (u, v), u < v, row-major over the strict upper triangle: row u starts at
    // u * (2 nb - u - 1) / 2.  Float estimate, then exact integer correction.
    const double fnb = (double)nb;
    int64_t u = (int64_t)floor(((2.0 * fnb - 1.0) - sqrt((2.0 * fnb - 1.0) * (2.0 * fnb - 1.0) - 8.0 * (double)p)) / 2.0);
    if (u < 0) u = 0;
    if (u > nb - 2) u = nb - 2;
    while (u > 0 && u * (2 * nb - u - 1) / 2 > p) --u;
    while ((u + 1) * (2 * nb - u - 2) / 2 <= p) ++u;
    const int64_t v = u + 1 + (p - u * (2 * nb - u - 1) / 2);
    const float *cu = C + u * D, *cv = C + v * D;
    float s = 0.0f, na = 0.0f, nv = 0.0f;
    int64_t d = 0;
    for (; d + 16 <= D; d += 16) {
        float a[16], b[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            a[i] = __ldg(cu + d + i);
            b[i] = __ldg(cv + d + i);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float t = __fsub_rn(a[i], b[i]);
            s = __fmaf_rn(t, t, s);
            na = __fmaf_rn(a[i], a[i], na);
            nv = __fmaf_rn(b[i], b[i], nv);
        }
    }
    for (; d < D; ++d) {
        const float a = __ldg(cu + d), b = __ldg(cv + d);
        const float t = __fsub_rn(a, b);
        s = __fmaf_rn(t, t, s);
        na = __fmaf_rn(a, a, na);
        nv = __fmaf_rn(b, b, nv);
    }
    const float2 iv = d2_interval(s, na, nv, rel);
    B[u * nb + v] = iv;
    B[v * nb + u] = iv;
}

// ---------------------------------------------------------------- MST, elder rule, CSR
// One cooperative launch runs everything after the distance intervals.  Its CTAs are all
// resident (cudaLaunchCooperativeKernel), so they can meet at grid-wide barriers; the barrier
// is bounded in time like every other wait here.
//   Boruvka rounds: all warps find each vertex's lightest edge to another component (strict
//     key (d2, min(u,v), max(u,v))): the smallest upper bound H over its edges to other
//     components, then the exact binary64 d2 of every such edge whose lower bound is <= H (the
//     lightest edge is among them); a vertex whose previous lightest edge still leaves its
//     component keeps it (its edge set only shrinks).  CTA 0 takes each component's lightest
//     edge, hooks along
//     it (a mutual pair keeps the smaller label as root), records each chosen edge once,
//     flattens by pointer jumping and relabels.  The rounds stop at one component.
//   Elder rule (CTA 0): bitonic sort of the nb-1 MST edges by the same key, then one warp
//     merges in that order with a union-find in shared memory, 32 edges at a time (a prefix
//     of merges whose components are disjoint is applied at once): the smaller component is
//     absorbed (size tie: the root with the larger index) and its root receives the edge's d2.
//   CSR: every CTA sorts the blocks by (salience desc, index asc); warps count each row's
//     blocks from a per-row bitmap (sink range, local window, first topk blocks <= i of the
//     order); CTA 0 scans the counts into row_ptr; warps fill col_idx in ascending order.
struct GraphArgs {
    const float2 *bnd;  // [nb][nb] intervals [lo, hi] holding the binary64 d2
    const double *cent; // [nb][D] centroids (in rank order under the content rule)
    int64_t D;
    int nb, pow2, sink, r, topk, rounds;
    size_t xs_offset;  // byte offset of the sort exchange buffer in dynamic shared memory
    int *comp;
    double *vb_d;
    int *vb_u;
    double *mst_d;
    int *mst_u, *mst_v;
    int *counters;   // [0] components, [1] MST edges recorded, [2] CSR overflow
    unsigned *gbar;  // [0] arrivals so far, [2] a CTA gave up waiting
    double *sal;
    const int *perm; // content rule: block of each rank (the graph runs on ranks); else null
    double *sal_rank; // content rule: salience by rank, before the scatter to blocks
    int *cnt;        // per-row counts, then row starts
    int32_t *row_ptr, *col_idx;
    int64_t col_cap;
    DeviceFlags flags;
};

// Grid-wide barrier (generation counter).  Returns false for the whole grid once any CTA has
// given up waiting.
__device__ bool grid_sync(unsigned *gbar, const DeviceFlags &f) {
    __shared__ int s_ok;
    __syncthreads();
    // A lone CTA needs nothing more: __syncthreads orders its threads' global accesses.
    if (gridDim.x == 1) return true;
    if (threadIdx.x == 0) {
        // gbar[0] counts arrivals over the whole launch (zeroed before it), so barrier k is
        // passed once the count reaches (k + 1) * gridDim.x: one atomic per CTA and no reset.
        int ok = 1;
        __threadfence();
        const unsigned arrived = atomicAdd(&gbar[0], 1u) + 1u;
        const unsigned target = (arrived + gridDim.x - 1u) / gridDim.x * gridDim.x;
        if (arrived != target) {
            volatile unsigned *vg = gbar;
            const unsigned long long t0 = globaltimer();
            while (vg[0] < target) {
                if (vg[2] != 0u) { ok = 0; break; }
                if (globaltimer() - t0 > kWaitTimeoutNs) {
                    atomicExch(&gbar[2], 1u);
                    raise_status(f, kDevTimeout);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// The strict edge order (d2, min(u,v), max(u,v)).  Squared distances are sums of squares from
// +0, never negative zero or NaN (or the +inf sentinel), so their bit patterns order like their
// values: the comparison runs on the integer pipe, not on this part's slow FP64 one.
__device__ __forceinline__ bool key_less(double d1, int a1, int b1, double d2, int a2, int b2) {
    const unsigned long long u1 = (unsigned long long)__double_as_longlong(d1);
    const unsigned long long u2 = (unsigned long long)__double_as_longlong(d2);
    if (u1 != u2) return u1 < u2;
    if (a1 != a2) return a1 < a2;
    return b1 < b2;
}

// The exact binary64 d2 of blocks x and y in the fixed order of summation: lane j accumulates
// the terms d = j, j + 32, ... (ascending, one fused multiply-add each, from +0) of
// t_d = C[x][d] - C[y][d] (the square of -t is the square of t, so the sign does not matter),
// then halving adds: after the step with offset w every lane holds P_(j mod w) + P_(j mod w + w)
// (the two lanes of a pair add the same two values, and binary64 addition is commutative).
// A dependent binary64 operation takes a few hundred cycles here, so this is ~4 chain steps and
// 5 additions for D = 128 instead of 128 steps.
__device__ __forceinline__ double exact_d2(const double *__restrict__ C, int64_t D, int x, int y, int lane) {
    const double *cx = C + (int64_t)x * D, *cy = C + (int64_t)y * D;
    double acc = 0.0;
    int64_t d = lane;
    for (; d + 96 < D; d += 128) {  // four terms per lane in flight
        const double a0 = __ldg(cx + d), b0 = __ldg(cy + d);
        const double a1 = __ldg(cx + d + 32), b1 = __ldg(cy + d + 32);
        const double a2 = __ldg(cx + d + 64), b2 = __ldg(cy + d + 64);
        const double a3 = __ldg(cx + d + 96), b3 = __ldg(cy + d + 96);
        double t;
        t = a0 - b0; acc = fma(t, t, acc);
        t = a1 - b1; acc = fma(t, t, acc);
        t = a2 - b2; acc = fma(t, t, acc);
        t = a3 - b3; acc = fma(t, t, acc);
    }
    for (; d < D; d += 32) {
        const double t = __ldg(cx + d) - __ldg(cy + d);
        acc = fma(t, t, acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc = acc + __shfl_xor_sync(0xffffffffu, acc, off);
    return acc;
}

// Each vertex's lightest edge to another component; one warp per vertex, grid-wide.  Every
// CTA keeps its own copy of the component labels in shared memory (`scomp`).  Round 0 and
// every vertex whose previous lightest edge now stays inside its component scan the row of
// intervals: H = the smallest upper bound over edges to other components, then the exact key
// of each such edge with lower bound <= H.  The edge of least exact d2 has lower bound <= its
// d2 <= H, so it is always among them.  Equal d2 go to the smaller (min, max) pair.
__device__ void vertex_min_phase(const GraphArgs &a, const int *scomp, int round) {
    const int nb = a.nb;
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const int total = gridDim.x * wpb;
    double *vb_d = a.vb_d + (round & 1) * nb;
    int *vb_u = a.vb_u + (round & 1) * nb;
    const double *pvb_d = a.vb_d + ((round + 1) & 1) * nb;
    const int *pvb_u = a.vb_u + ((round + 1) & 1) * nb;
    for (int v = blockIdx.x * wpb + (threadIdx.x >> 5); v < nb; v += total) {
        const int cv = scomp[v];
        if (round > 0) {
            // written by some warp of the previous round, before the grid barrier
            const int pu = __ldcg(pvb_u + v);
            if (pu >= 0 && scomp[pu] != cv) {
                if (lane == 0) {
                    vb_d[v] = __ldcg(pvb_d + v);
                    vb_u[v] = pu;
                }
                continue;
            }
        }
        const float2 *row = a.bnd + (int64_t)v * nb;
        // each lane reads 16 intervals per 512-block batch; a row of at most 512 blocks is read
        // once and its intervals stay in registers for the candidate pass
        float2 iv[16];
        float h = __int_as_float(0x7f800000);
        for (int base = 0; base < nb; base += 32 * 16) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int u = base + lane + 32 * k;
                iv[k] = u < nb ? __ldg(&row[u]) : make_float2(0.0f, 0.0f);
            }
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int u = base + lane + 32 * k;
                if (u < nb && scomp[u] != cv) h = fminf(h, iv[k].y);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) h = fminf(h, __shfl_xor_sync(0xffffffffu, h, off));
        // the exact keys of the candidates, warp-uniform
        double bd = __longlong_as_double((long long)kInfBits);
        int ba = INT_MAX, bb = INT_MAX, bu = -1;
        for (int base = 0; base < nb; base += 32 * 16) {
            if (nb > 32 * 16) {
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int u = base + lane + 32 * k;
                    iv[k] = u < nb ? __ldg(&row[u]) : make_float2(0.0f, 0.0f);
                }
            }
            // lane k keeps the candidate mask of batch slot k
            unsigned mine = 0u;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int u = base + lane + 32 * k;
                const unsigned m = __ballot_sync(0xffffffffu, u < nb && scomp[u] != cv && iv[k].x <= h);
                if (lane == k) mine = m;
            }
#pragma unroll 1
            for (int k = 0; k < 16; ++k) {
                unsigned m = __shfl_sync(0xffffffffu, mine, k);
                while (m != 0u) {
                    const int w = base + (__ffs((int)m) - 1) + 32 * k;
                    m &= m - 1u;
                    const double d = exact_d2(a.cent, a.D, v, w, lane);
                    const int x = w < v ? w : v, y = w < v ? v : w;
                    if (key_less(d, x, y, bd, ba, bb)) { bd = d; ba = x; bb = y; bu = w; }
                }
            }
        }
        if (lane == 0) {
            vb_d[v] = bd;
            vb_u[v] = bu;
        }
    }
}

// Every CTA, on its own shared-memory copy: per component the lightest outgoing edge (min
// over its vertices), hooking (a mutual pair keeps the smaller label as root), flattening by
// pointer jumping and relabelling.  All CTAs compute the same result; CTA 0 also records the
// chosen edges.  Returns the number of components left.
__device__ int merge_phase(const GraphArgs &a, uint8_t *sm, int *scomp, const double *vb_d,
                           const int *vb_u, int *n_edges) {
    const int nb = a.nb;
    unsigned long long *cb_d = reinterpret_cast<unsigned long long *>(sm);
    unsigned long long *cb_ab = cb_d + nb;
    volatile int *par = reinterpret_cast<volatile int *>(cb_ab + nb);
    __shared__ int s_roots, s_edges;
    const int tid = threadIdx.x, nt = blockDim.x;
    const bool record = blockIdx.x == 0;
    if (tid == 0) { s_roots = 0; s_edges = *n_edges; }
    for (int c = tid; c < nb; c += nt) {
        cb_d[c] = kInfBits;
        cb_ab[c] = ~0ull;
    }
    __syncthreads();
    for (int v = tid; v < nb; v += nt)
        atomicMin(&cb_d[scomp[v]], (unsigned long long)__double_as_longlong(__ldcg(vb_d + v)));
    __syncthreads();
    for (int v = tid; v < nb; v += nt) {
        const int c = scomp[v];
        const int u = __ldcg(vb_u + v);
        if ((unsigned long long)__double_as_longlong(__ldcg(vb_d + v)) == cb_d[c] && u >= 0) {
            const unsigned x = (unsigned)min(v, u), y = (unsigned)max(v, u);
            atomicMin(&cb_ab[c], ((unsigned long long)x << 32) | y);
        }
    }
    __syncthreads();
    for (int c = tid; c < nb; c += nt) {
        if (scomp[c] != c) continue;
        const unsigned long long ab = cb_ab[c];
        if (ab == ~0ull) { par[c] = c; continue; }
        const int x = (int)(ab >> 32), y = (int)(ab & 0xFFFFFFFFu);
        const int other = scomp[x] == c ? scomp[y] : scomp[x];
        const bool mutual = cb_ab[other] == ab;
        par[c] = (mutual && c < other) ? c : other;
        if (record && (!mutual || c < other)) {
            const int idx = atomicAdd(&s_edges, 1);
            if (idx < nb - 1) {
                a.mst_d[idx] = __longlong_as_double((long long)cb_d[c]);
                a.mst_u[idx] = x;
                a.mst_v[idx] = y;
            }
        }
    }
    __syncthreads();
    for (int iter = 0; iter < 64; ++iter) {
        int changed = 0;
        for (int c = tid; c < nb; c += nt) {
            if (scomp[c] != c) continue;
            const int p = par[c];
            const int pp = par[p];
            if (p != pp) { par[c] = pp; changed = 1; }
        }
        if (!__syncthreads_or(changed)) break;
    }
    for (int c = tid; c < nb; c += nt)
        if (scomp[c] == c && par[c] == c) atomicAdd(&s_roots, 1);
    __syncthreads();
    for (int v = tid; v < nb; v += nt) scomp[v] = par[scomp[v]];
    __syncthreads();
    const int roots = s_roots;
    if (tid == 0) *n_edges = s_edges;
    __syncthreads();
    return roots;
}

// Sort 64-bit key pairs ascending (lexicographic on (k1, k2)); n is a power of two.
__device__ void bitonic_sort_pairs(unsigned long long *k1, unsigned long long *k2, int n) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool up = (i & size) == 0;
                    const bool gt = k1[i] > k1[j] || (k1[i] == k1[j] && k2[i] > k2[j]);
                    if (gt == up) {
                        const unsigned long long t1 = k1[i], t2 = k2[i];
                        k1[i] = k1[j]; k2[i] = k2[j];
                        k1[j] = t1; k2[j] = t2;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Bitonic sort of (k1, k2) pairs ascending with one element per thread (n == blockDim.x, a
// power of two): strides below 32 exchange through shuffles, larger ones through `xs`
// (2 * n words of shared memory).  On return k1/k2 hold the element of rank threadIdx.x.
// Sorts the keys of threads [0, m) (m a power of two, m <= blockDim.x) ascending; threads at
// or past m exchange only among themselves (i ^ stride >= m there), so their keys are left in
// some order of their own.  Every thread must call it (the cross-warp stages synchronize).
__device__ void bitonic_sort_regs(unsigned long long &k1, unsigned long long &k2,
                                  unsigned long long *xs, int m) {
    const int i = threadIdx.x, n = blockDim.x;
    for (int size = 2; size <= m; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            unsigned long long p1, p2;
            if (stride < 32) {
                p1 = __shfl_xor_sync(0xffffffffu, k1, stride);
                p2 = __shfl_xor_sync(0xffffffffu, k2, stride);
            } else {
                xs[i] = k1;
                xs[n + i] = k2;
                __syncthreads();
                p1 = xs[i ^ stride];
                p2 = xs[n + (i ^ stride)];
                __syncthreads();
            }
            const bool ascending = (i & size) == 0;
            const bool lower = (i & stride) == 0;
            const bool mine_less = k1 < p1 || (k1 == p1 && k2 < p2);
            const bool take_partner = (ascending == lower) ? !mine_less : mine_less;
            if (take_partner) {
                k1 = p1;
                k2 = p2;
            }
        }
    }
}

// CTA 0: elder-rule salience from the MST edges.
__device__ void elder_phase(const GraphArgs &a, uint8_t *sm, int n_edges, unsigned long long *xs) {
    const int nb = a.nb, pow2 = a.pow2;
    unsigned long long *kd = reinterpret_cast<unsigned long long *>(sm);
    unsigned long long *kab = kd + pow2;
    volatile int *size = reinterpret_cast<volatile int *>(kab + pow2);
    volatile int *label = size + nb;  // union-find parents, then two claim arrays (nb each)
    const int ne = nb - 1;
    // under content ties the merges run on ranks: salience goes to a rank-indexed scratch and
    // is scattered to blocks at the end (one global write per merge, no dependent load)
    double *sal = a.perm ? a.sal_rank : a.sal;
    if (threadIdx.x == 0 && n_edges != ne) raise_status(a.flags, kDevCapacity);
    for (int i = threadIdx.x; i < pow2; i += blockDim.x) {
        if (i < ne) {
            kd[i] = (unsigned long long)__double_as_longlong(a.mst_d[i]);
            kab[i] = ((unsigned long long)(unsigned)a.mst_u[i] << 32) | (unsigned)a.mst_v[i];
        } else {
            kd[i] = ~0ull;
            kab[i] = ~0ull;
        }
    }
    for (int v = threadIdx.x; v < nb; v += blockDim.x) {
        label[v] = v;
        size[v] = 1;
        sal[v] = 0.0;
    }
    __syncthreads();
    const bool fast = pow2 <= (int)blockDim.x;
    if (fast) {
        // one element per thread (padding sorts last), sorted copy written back to kd/kab
        unsigned long long k1 = threadIdx.x < pow2 ? kd[threadIdx.x] : ~0ull;
        unsigned long long k2 = threadIdx.x < pow2 ? kab[threadIdx.x] : ~0ull;
        __syncthreads();
        bitonic_sort_regs(k1, k2, xs, pow2);
        __syncthreads();
        if (threadIdx.x < pow2) {
            kd[threadIdx.x] = k1;
            kab[threadIdx.x] = k2;
        }
        __syncthreads();
    } else {
        bitonic_sort_pairs(kd, kab, pow2);
    }
    // Merges in edge order with a union-find in shared memory.  The smaller component is
    // absorbed (on a size tie the root with the larger index), so linking the absorbed root
    // under the survivor is union by size: trees stay O(log nb) deep, path halving keeps them
    // flatter, and the root of a component is always its survivor -- the one block of it that
    // has received no merge distance yet.
    // One warp takes the edges 32 at a time: each lane finds its edge's two roots (finds only
    // read parents or halve paths, so they may run together) and decides its merge from the
    // component sizes before the group.  A prefix of the group merges at once: lane l joins it
    // when no earlier lane touches the root l absorbs, and no earlier lane absorbs the root l
    // keeps.  A root shared by several of those lanes is then the survivor of each of their
    // merges; it only grows, so every decision is the one taken edge by edge, and the
    // absorbed roots are distinct.  (This covers a large component taking singletons one
    // edge after another, as well as merges of disjoint components.)  The group resumes at
    // the first lane that had to wait, which is never lane 0.
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int *par = const_cast<int *>(label);
        int *siz = const_cast<int *>(size);
        int *used = par + nb;      // lowest lane of the group using a root (INT_MAX: none)
        int *taken = used + nb;    // lowest lane of the group absorbing a root
        for (int v = lane; v < nb; v += 32) {
            used[v] = INT_MAX;
            taken[v] = INT_MAX;
        }
        __syncwarp();
        for (int e0 = 0; e0 < ne;) {
            const int e = e0 + lane;
            const bool has = e < ne;
            int x = 0, y = 0;
            if (has) {
                const unsigned long long ab = kab[e];
                x = (int)(ab >> 32);
                y = (int)(ab & 0xFFFFFFFFu);
            }
            if (__any_sync(0xffffffffu, has && (x < 0 || x >= nb || y < 0 || y >= nb))) {
                if (lane == 0) raise_status(a.flags, kDevCapacity);
                break;
            }
            int rx = x, ry = y;
            if (has) {
                for (int it = 0; it < nb; ++it) {  // both finds at once; at most nb steps
                    const int px = par[rx], py = par[ry];
                    if (px == rx && py == ry) break;
                    if (px != rx) {
                        const int gx = par[px];
                        par[rx] = gx;
                        rx = gx;
                    }
                    if (py != ry) {
                        const int gy = par[py];
                        par[ry] = gy;
                        ry = gy;
                    }
                }
            }
            int absorbed = 0, survivor = 0, sa = 0;
            if (has && rx != ry) {  // rx == ry cannot happen for MST edges
                const int sx = siz[rx], sy = siz[ry];
                if (sx < sy) { absorbed = rx; survivor = ry; sa = sx; }
                else if (sy < sx) { absorbed = ry; survivor = rx; sa = sy; }
                else { absorbed = rx > ry ? rx : ry; survivor = rx > ry ? ry : rx; sa = sx; }
                atomicMin(&used[absorbed], lane);
                atomicMin(&used[survivor], lane);
                atomicMin(&taken[absorbed], lane);
            }
            __syncwarp();
            // lane 0 is always ready (it is the lowest lane on both of its roots), so every round
            // merges at least one edge; an edge inside one component (impossible for MST edges)
            // is a ready no-op
            const bool ready = has && (rx == ry || (used[absorbed] == lane && taken[survivor] > lane));
            const unsigned wmask = __ballot_sync(0xffffffffu, !ready && has);
            const int k = wmask ? __ffs(wmask) - 1 : 32;  // lanes [0, k) merge now; k >= 1
            __syncwarp();
            if (lane < k && has && rx != ry) {
                par[absorbed] = survivor;
                atomicAdd(&siz[survivor], sa);
                sal[absorbed] = __longlong_as_double((long long)kd[e]);
            }
            __syncwarp();
            if (has && rx != ry) {
                used[absorbed] = INT_MAX;
                used[survivor] = INT_MAX;
                taken[absorbed] = INT_MAX;
            }
            __syncwarp();
            e0 += k;
        }
    }
    __syncthreads();
    if (a.perm) {
        for (int r = threadIdx.x; r < nb; r += blockDim.x) {
            const int b = a.perm[r];
            if (b >= 0 && b < nb) a.sal[b] = sal[r];
        }
        __syncthreads();
    }
}

// Bitmap of row i in `bm` (one warp): sink range, local window, and the first topk blocks
// j <= i of `order` (salience descending, index ascending).
__device__ void row_bitmap(const int *order, unsigned *bm, int words, int nb, int i, int sink,
                           int r, int topk) {
    const int lane = threadIdx.x & 31;
    const int s_end = min(sink, i + 1);           // sink blocks [0, s_end)
    const int l_beg = max(0, i - r);              // local blocks [l_beg, i]
    for (int w = lane; w < words; w += 32) {
        const int lo = w * 32;
        unsigned m = 0;
        if (s_end > lo) m |= (s_end - lo >= 32) ? 0xFFFFFFFFu : ((1u << (s_end - lo)) - 1u);
        const int x = max(l_beg, lo), y = min(i, lo + 31);
        if (x <= y) {
            const int n = y - x + 1;
            const unsigned run = (n >= 32) ? 0xFFFFFFFFu : ((1u << n) - 1u);
            m |= run << (x - lo);
        }
        bm[w] = m;
    }
    __syncwarp();
    int need = min(topk, i + 1);
    for (int base = 0; need > 0 && base < nb; base += 32) {
        const int t = base + lane;
        const int j = t < nb ? order[t] : INT_MAX;
        const bool pred = j <= i;
        const unsigned bal = __ballot_sync(0xffffffffu, pred);
        const int rank = __popc(bal & ((1u << lane) - 1u));
        if (pred && rank < need) atomicOr(&bm[j >> 5], 1u << (j & 31));
        need -= __popc(bal);
    }
    __syncwarp();
}

__global__ void __launch_bounds__(512, 1) schedule_graph_kernel(GraphArgs a) {
    extern __shared__ __align__(16) uint8_t sm[];
    const int nb = a.nb;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
    const int gwarp = blockIdx.x * nwarps + warp, gwarps = gridDim.x * nwarps;
    // exchange buffer of the register sorts: 2 x blockDim 64-bit words after the phase areas
    unsigned long long *xs = reinterpret_cast<unsigned long long *>(sm + a.xs_offset);
    // ---- Boruvka: labels per CTA in shared memory, vertex bests double-buffered by round
    int *scomp = reinterpret_cast<int *>(sm + (size_t)nb * 20);
    for (int v = tid; v < nb; v += nt) scomp[v] = v;
    if (blockIdx.x == 0 && tid == 0) a.counters[2] = 0;
    __syncthreads();
    int ncomp = nb, n_edges = 0;
    for (int round = 0; round < a.rounds && ncomp > 1; ++round) {
        vertex_min_phase(a, scomp, round);
        if (!grid_sync(a.gbar, a.flags)) return;
        ncomp = merge_phase(a, sm, scomp, a.vb_d + (round & 1) * nb, a.vb_u + (round & 1) * nb, &n_edges);
    }
    // ---- elder rule (CTA 0 holds the MST edges it recorded)
    if (blockIdx.x == 0) elder_phase(a, sm, n_edges, xs);
    if (!grid_sync(a.gbar, a.flags)) return;
    // ---- top-k + CSR: every CTA sorts its own copy of the order
    const int pow2 = a.pow2;
    const int words = (nb + 31) / 32;
    unsigned long long *ok1 = reinterpret_cast<unsigned long long *>(sm);
    unsigned long long *ok2 = ok1 + pow2;
    int *order = reinterpret_cast<int *>(ok2 + pow2);
    unsigned *bm = reinterpret_cast<unsigned *>(order + pow2) + warp * words;
    for (int i = tid; i < pow2; i += nt) {
        if (i < nb) {
            ok1[i] = ~(unsigned long long)__double_as_longlong(
                *reinterpret_cast<volatile double *>(&a.sal[i]));  // salience >= 0
            ok2[i] = (unsigned long long)i;
        } else {
            ok1[i] = ~0ull;
            ok2[i] = ~0ull;
        }
    }
    __syncthreads();
    if (pow2 <= nt) {
        unsigned long long k1 = tid < pow2 ? ok1[tid] : ~0ull;
        unsigned long long k2 = tid < pow2 ? ok2[tid] : ~0ull;
        __syncthreads();
        bitonic_sort_regs(k1, k2, xs, pow2);
        if (tid < nb) order[tid] = (int)k2;
    } else {
        bitonic_sort_pairs(ok1, ok2, pow2);
        for (int i = tid; i < nb; i += nt) order[i] = (int)ok2[i];
    }
    __syncthreads();
    for (int i = gwarp; i < nb; i += gwarps) {
        row_bitmap(order, bm, words, nb, i, a.sink, a.r, a.topk);
        int c = 0;
        for (int w = lane; w < words; w += 32) c += __popc(bm[w]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
        if (lane == 0) a.cnt[i] = c;
        __syncwarp();
    }
    if (!grid_sync(a.gbar, a.flags)) return;
    if (blockIdx.x == 0) {
        // exclusive scan of the counts: each thread a contiguous run, then warp / CTA totals
        __shared__ int warp_tot[32];
        const int per = (nb + nt - 1) / nt;
        const int beg = min(nb, tid * per), end = min(nb, beg + per);
        int run = 0;
        for (int i = beg; i < end; ++i) run += a.cnt[i];
        int incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int t = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, t, off);
                if (lane >= off) t += o;
            }
            warp_tot[lane] = t;
        }
        __syncthreads();
        int start = (warp > 0 ? warp_tot[warp - 1] : 0) + incl - run;
        for (int i = beg; i < end; ++i) {
            const int c = a.cnt[i];
            a.cnt[i] = start;
            a.row_ptr[i] = start;
            start += c;
        }
        if (tid == 0) {
            const int total = warp_tot[nwarps - 1];
            a.row_ptr[nb] = total;
            if ((int64_t)total > a.col_cap) {
                a.counters[2] = 1;
                raise_status(a.flags, kDevCapacity);
            }
        }
    }
    if (!grid_sync(a.gbar, a.flags)) return;
    if (*reinterpret_cast<volatile int *>(&a.counters[2]) != 0) return;
    for (int i = gwarp; i < nb; i += gwarps) {
        row_bitmap(order, bm, words, nb, i, a.sink, a.r, a.topk);
        int off = *reinterpret_cast<volatile int *>(&a.cnt[i]);
        for (int w0 = 0; w0 < words; w0 += 32) {
            const int w = w0 + lane;
            unsigned bits = w < words ? bm[w] : 0u;
            const int c = __popc(bits);
            int inc = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += x;
            }
            int pos = off + inc - c;
            while (bits) {
                const int bit = __ffs(bits) - 1;
                a.col_idx[pos++] = w * 32 + bit;
                bits &= bits - 1u;
            }
            off += __shfl_sync(0xffffffffu, inc, 31);
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------- dense causal CSR
__global__ void dense_csr(int64_t nb, int32_t *__restrict__ row_ptr, int32_t *__restrict__ col_idx) {
    const int64_t nnz = nb * (nb + 1) / 2;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i <= nb; i += stride)
        row_ptr[i] = (int32_t)(i * (i + 1) / 2);
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < nnz; e += stride) {
        int64_t i = (int64_t)((sqrt(8.0 * (double)e + 1.0) - 1.0) * 0.5);
        while (i * (i + 1) / 2 > e) --i;
        while ((i + 1) * (i + 2) / 2 <= e) ++i;
        col_idx[e] = (int32_t)(e - i * (i + 1) / 2);
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int next_pow2(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

template <typename K>
bool set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
           cudaSuccess;
}

}  // namespace

ScheduleWorkspace schedule_workspace_layout(int64_t lanes, int64_t nb, int64_t D) {
    ScheduleWorkspace w{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    w.part = take(sizeof(double) * (size_t)(lanes * nb * D));
    w.cent = take(sizeof(double) * (size_t)(nb * D));
    w.cent32 = take(sizeof(float) * (size_t)(nb * D));
    w.bnd = take(sizeof(float2) * (size_t)(nb * nb));
    w.comp = take(sizeof(int) * (size_t)nb);
    w.vb_d = take(sizeof(double) * (size_t)(2 * nb));
    w.vb_u = take(sizeof(int) * (size_t)(2 * nb));
    w.mst_d = take(sizeof(double) * (size_t)nb);
    w.mst_u = take(sizeof(int) * (size_t)nb);
    w.mst_v = take(sizeof(int) * (size_t)nb);
    w.counters = take(sizeof(int) * 4);
    w.sal = take(sizeof(double) * (size_t)nb);
    w.cnt = take(sizeof(int) * (size_t)(nb + 1));
    w.perm = take(sizeof(int) * (size_t)nb);
    w.sal_rank = take(sizeof(double) * (size_t)nb);
    w.gbar = take(sizeof(unsigned) * 4);
    w.total = o;
    return w;
}

// Grids of at most this many (lane, block, 8 d) items sum with a warp per item.
constexpr int64_t kWarpSumItems = 4096;

// Per-lane block sums of K into part[lanes][nb][D].
tsa_status launch_block_sums(const ScheduleLaunch &a, double *part) {
    cudaStream_t st = a.stream;
    const bool vec = (a.D % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.K) & 15u) == 0);
    const int64_t items = vec ? a.lanes * a.nb * (a.D / 8) : a.lanes * a.nb * a.D;
    const int threads = 256;
    const int64_t blocks = (items + threads - 1) / threads;
    const unsigned grid = (unsigned)(blocks < 152 * 64 ? blocks : 152 * 64);
    int log2_block = 0;
    while ((int64_t(1) << log2_block) < a.block) ++log2_block;
    const int spread_limit = 45 - log2_block;
    if (vec && (!a.bf16 || a.block <= 64) && items <= kWarpSumItems) {
        // few items: a warp per item
        const int64_t nblk = (items + 7) / 8;
        centroid_partial_warp<<<(unsigned)nblk, 256, 0, st>>>(a.K, a.bf16, a.lanes, a.S, a.D, a.block, a.nb,
                                                             spread_limit, part);
    } else if (vec && (!a.bf16 || a.block <= 64)) {  // the TwoSum exactness bound holds for <= 64 terms
        // the small shape only while it fills at most one CTA per SM
        const bool large = items >= (int64_t)152 * 64;
        // the pair for bf16, and for f16 in blocks of at most 64 tokens (its exactness bound)
        const bool pair = a.bf16 || a.block <= 64;
        auto kern = large ? (a.bf16 ? centroid_partial_stream<256, 3, true, true>
                                    : pair ? centroid_partial_stream<256, 3, false, true>
                                           : centroid_partial_stream<256, 3, false, false>)
                          : (a.bf16 ? centroid_partial_stream<64, 8, true, true>
                                    : pair ? centroid_partial_stream<64, 8, false, true>
                                           : centroid_partial_stream<64, 8, false, false>);
        const int nthr = large ? 256 : 64;
        const int smem = large ? StreamShape<256, 3>::kSmem : StreamShape<64, 8>::kSmem;
        const int64_t nblk = (items + nthr - 1) / nthr;
        const unsigned sgrid = (unsigned)(nblk < 152 * 64 ? nblk : 152 * 64);
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return TSA_ERR_CUDA;
        kern<<<sgrid, nthr, smem, st>>>(a.K, a.lanes, a.S, a.D, a.block, a.nb, spread_limit, part);
    } else if (vec)
        centroid_partial_vec8<<<grid, threads, 0, st>>>(a.K, a.bf16, a.lanes, a.S, a.D, a.block, a.nb,
                                                        spread_limit, part);
    else
        centroid_partial_scalar<<<grid, threads, 0, st>>>(a.K, a.bf16, a.lanes, a.S, a.D, a.block, a.nb,
                                                          spread_limit, part);
    return cudaGetLastError() == cudaSuccess ? TSA_OK : TSA_ERR_CUDA;
}

tsa_status launch_build_schedule(const ScheduleLaunch &a) {
    const ScheduleWorkspace ws = schedule_workspace_layout(a.lanes, a.nb, a.D);
    double *part = reinterpret_cast<double *>(a.workspace + ws.part);
    const tsa_status st = launch_block_sums(a, part);
    return st != TSA_OK ? st : launch_schedule_from_sums(a, part);
}

// Everything after the block sums: lane-mean centroids (lanes in ascending order), the
// content ranking if asked, distances, and the graph kernel.  `sums` is read only; the
// content rule's permuted centroids go to the workspace's own block-sum area, which is `sums`
// itself when called from launch_build_schedule (the sums are no longer needed by then).
tsa_status launch_schedule_from_sums(const ScheduleLaunch &a, const double *sums) {
    const int nb = (int)a.nb;
    const ScheduleWorkspace ws = schedule_workspace_layout(a.lanes, a.nb, a.D);
    uint8_t *w = a.workspace;
    double *part = reinterpret_cast<double *>(w + ws.part);
    double *cent = reinterpret_cast<double *>(w + ws.cent);
    float *cent32 = reinterpret_cast<float *>(w + ws.cent32);
    float2 *bnd = reinterpret_cast<float2 *>(w + ws.bnd);
    int *comp = reinterpret_cast<int *>(w + ws.comp);
    double *vb_d = reinterpret_cast<double *>(w + ws.vb_d);
    int *vb_u = reinterpret_cast<int *>(w + ws.vb_u);
    double *mst_d = reinterpret_cast<double *>(w + ws.mst_d);
    int *mst_u = reinterpret_cast<int *>(w + ws.mst_u);
    int *mst_v = reinterpret_cast<int *>(w + ws.mst_v);
    int *counters = reinterpret_cast<int *>(w + ws.counters);
    double *sal = a.salience_sq ? a.salience_sq : reinterpret_cast<double *>(w + ws.sal);
    cudaStream_t st = a.stream;

    // centroids
    {
        const int64_t n = a.nb * a.D;
        const unsigned g = (unsigned)((n + 255) / 256);
        centroid_final<<<g, 256, 0, st>>>(sums, a.lanes, a.nb, a.D, a.S, a.block, cent, cent32);
    }
    // content rule: rank the blocks, run the graph on the centroids in rank order
    int *perm = nullptr;
    const double *graph_cent = cent;
    if (a.content_ties) {
        perm = reinterpret_cast<int *>(w + ws.perm);
        content_rank<<<(unsigned)((a.nb + 7) / 8), 256, 0, st>>>(cent, a.nb, a.D, perm);
        const int64_t n = a.nb * a.D;
        permute_rows<<<(unsigned)((n + 255) / 256 < 152 * 16 ? (n + 255) / 256 : 152 * 16), 256, 0, st>>>(
            cent, perm, a.nb, a.D, part, cent32);
        graph_cent = part;  // the workspace's block-sum area; centroid_final has read the sums
    }
    // distance intervals (D <= 1024, so rel = D * 2^-22 is exact and at most 2^-12); the kernel
    // also zeroes the graph kernel's barrier words, which run after it in stream order
    unsigned *gbar = reinterpret_cast<unsigned *>(w + ws.gbar);
    const float rel = ldexpf((float)a.D, -22);
    if (nb < kPbFlatBelow) {
        const int64_t npairs = a.nb * (a.nb - 1) / 2;
        const int64_t n = npairs > a.nb ? npairs : a.nb;
        pairwise_bounds_flat<<<(unsigned)((n + 31) / 32), 32, 0, st>>>(cent32, a.nb, a.D, rel, bnd, gbar);
    } else {
        const int t = (nb + kPbTile - 1) / kPbTile;
        pairwise_bounds<<<(unsigned)(t * (t + 1) / 2), kPbThreads, 0, st>>>(cent32, a.nb, a.D, t, rel, bnd, gbar);
    }
    // MST, elder rule and CSR in one cooperative launch
    int rounds = 0;
    while ((1 << rounds) < nb) ++rounds;
    const int pow2 = next_pow2(nb);
    const int words = (nb + 31) / 32;
    constexpr int kGraphThreads = 512;
    const size_t merge_smem = (size_t)nb * (8 + 8 + 4 + 4);
    const size_t elder_smem = (size_t)pow2 * 16 + (size_t)nb * 16;  // edges, sizes, parents, 2 claims
    const size_t topk_smem = (size_t)pow2 * 20 + (size_t)(kGraphThreads / 32) * words * 4;
    size_t smem = merge_smem > elder_smem ? merge_smem : elder_smem;
    if (topk_smem > smem) smem = topk_smem;
    const size_t xs_offset = (smem + 15) & ~(size_t)15;
    smem = xs_offset + (size_t)kGraphThreads * 16;
    if (!set_smem(schedule_graph_kernel, smem)) return TSA_ERR_CUDA;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, schedule_graph_kernel, kGraphThreads, smem) !=
            cudaSuccess ||
        per_sm < 1)
        return TSA_ERR_CUDA;
    // one warp per vertex in the parallel phases is plenty; fewer CTAs make cheaper barriers
    int ggrid = (nb + kGraphThreads / 32 - 1) / (kGraphThreads / 32);
    if (ggrid > sms * per_sm) ggrid = sms * per_sm;
    if (ggrid > sms) ggrid = sms;
    if (ggrid < 1) ggrid = 1;
    GraphArgs g;
    g.bnd = bnd;
    g.cent = graph_cent;
    g.D = a.D;
    g.nb = nb;
    g.pow2 = pow2;
    g.sink = (int)a.sink;
    g.r = (int)a.local_radius;
    g.topk = (int)a.topk;
    g.rounds = rounds;
    g.xs_offset = xs_offset;
    g.comp = comp;
    g.vb_d = vb_d;
    g.vb_u = vb_u;
    g.mst_d = mst_d;
    g.mst_u = mst_u;
    g.mst_v = mst_v;
    g.counters = counters;
    g.gbar = gbar;
    g.sal = sal;
    g.perm = perm;
    g.sal_rank = reinterpret_cast<double *>(w + ws.sal_rank);
    g.cnt = reinterpret_cast<int *>(w + ws.cnt);
    g.row_ptr = a.row_ptr;
    g.col_idx = a.col_idx;
    g.col_cap = a.col_cap;
    g.flags = a.flags;
    void *args[] = {&g};
    if (cudaLaunchCooperativeKernel((const void *)schedule_graph_kernel, dim3((unsigned)ggrid),
                                    dim3(kGraphThreads), args, smem, st) != cudaSuccess)
        return TSA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TSA_OK : TSA_ERR_CUDA;
}

tsa_status launch_dense_causal_csr(int64_t nb, int32_t *row_ptr, int32_t *col_idx,
                                   cudaStream_t stream) {
    const int64_t nnz = nb * (nb + 1) / 2;
    const int64_t n = nnz > nb + 1 ? nnz : nb + 1;
    const int64_t blocks = (n + 255) / 256;
    dense_csr<<<(unsigned)(blocks < 152 * 16 ? blocks : 152 * 16), 256, 0, stream>>>(nb, row_ptr, col_idx);
    return cudaGetLastError() == cudaSuccess ? TSA_OK : TSA_ERR_CUDA;
}

}  // namespace tsa
