// backward.cu -- gradients of the scheduled causal attention on tcgen05 tensor cores (sm_103a).
//
// The forward is the kernel of "Add topology-derived sparse attention kernel"
// (triton-lang/kernels#22, Summary); its mirror page's segment-boundary record notes that the
// merged kernel has no backward pass, which is the step this file adds.  With P the softmax of
// the scaled scores over each query's allowed keys (the CSR row's blocks, keys <= the query in
// the diagonal block) and dO the upstream gradient:
//   Delta_q = <dO_q, O_q>,  dP = dO V^T,  dS = P o (dP - Delta),
//   dV = P^T dO,  dQ = scale dS K,  dK = scale dS^T Q.
// P is recomputed from the forward's log-sum-exp (P = exp(scale s - lse)), so nothing of size
// S x S is stored.
//
// Launches:
//   bwd_rows, bwd_col_count, bwd_col_scan, bwd_col_fill -- the transposed schedule: for every
//     key block j the ascending list of query blocks whose row holds j (a column bitmap, so
//     the lists come out sorted without a sort); rows are checked on the way (a row is cut at
//     its first entry that is out of order or out of [0, i], and the status word reports it).
//   bwd_delta -- Delta per query row from the stored O and dO.
//   bwd_dq_kernel -- one CTA per pair of query blocks (M = 128), walking the union of the two
//     CSR rows like the forward: S = Q K^T and dP = dO V^T into TMEM, dS formed by the four
//     elementwise warps and written back over S in the input dtype, dQ += dS K with dS read
//     from TMEM.
//   bwd_dkv_kernel -- one CTA per pair of key blocks (M = 128), walking the union of the two
//     transposed columns: S^T = K Q^T and dP^T = V dO^T into TMEM, P^T and dS^T written back
//     over them, dV += P^T dO and dK += dS^T Q.
// Warp roles are those of the forward: warp 4 produces (TMA), warp 5 issues the MMAs from one
// thread (the next step's products before the current step's accumulation), warps 0-3 do the
// elementwise work, one TMEM lane (row) per thread.  Every wait is bounded; on a timeout a CTA
// records TSA_ERR_TIMEOUT, drains what it issued, frees its TMEM and returns.
#include <climits>

#include "tsa_device.cuh"
#include "tsa_internal.h"

namespace tsa {
namespace {

constexpr int kBlock = 64;
constexpr int kThreads = 192;
constexpr int kRows = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kStream = 3;     // depth of the ring of streamed blocks
constexpr int kMetaRing = 4;   // > kStream: a slot is rewritten only after its step is consumed
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- transposed schedule

// One warp per CSR row: the valid prefix length, and bit i of column j's bitmap words for each
// valid entry j of row i.
__global__ void bwd_rows(int nb, const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
                         int words, int *__restrict__ vlen, unsigned *__restrict__ bitmap, DeviceFlags flags) {
    const int lane = threadIdx.x & 31;
    const int nw = gridDim.x * (blockDim.x >> 5);
    for (int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < nb; i += nw) {
        const int b = row_ptr[i], len = row_ptr[i + 1] - b;
        int valid = 0;
        if (len >= 0 && len <= i + 1) {
            valid = len;
            for (int e0 = 0; e0 < len; e0 += 32) {
                const int e = e0 + lane;
                bool bad = false;
                if (e < len) {
                    const int j = col_idx[b + e];
                    const int prev = e > 0 ? col_idx[b + e - 1] : -1;
                    bad = j < 0 || j > i || j <= prev;
                }
                const unsigned m = __ballot_sync(0xffffffffu, bad);
                if (m) {
                    valid = e0 + __ffs(m) - 1;
                    break;
                }
            }
        }
        if (lane == 0 && valid != len) raise_status(flags, kDevBadSchedule);
        for (int e = lane; e < valid; e += 32) {
            const int j = col_idx[b + e];
            atomicOr(&bitmap[(size_t)j * words + (i >> 5)], 1u << (i & 31));
        }
        if (lane == 0) vlen[i] = valid;
    }
}

// A CSR of 128-token blocks as the CSR of 64-token blocks with the same allowed keys: query
// block a = 2p + h (64 tokens) of 128-block row p holds the 64-blocks 2j and 2j+1 of every
// j < p in row p, and of j = p the ones not after it (2p; 2p+1 when h = 1) -- the token mask
// of the 64-token diagonal block then cuts keys k > q exactly as the 128-token rule does.
// One warp per 128-block row: its valid prefix (the checks of bwd_rows), the two counts.
__global__ void bwd_expand128_count(int nb128, int nb64, const int32_t *__restrict__ row_ptr,
                                    const int32_t *__restrict__ col_idx, int *__restrict__ vlen128,
                                    int *__restrict__ cnt64, DeviceFlags flags) {
    const int lane = threadIdx.x & 31;
    const int nw = gridDim.x * (blockDim.x >> 5);
    for (int p = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < nb128; p += nw) {
        const int b = row_ptr[p], len = row_ptr[p + 1] - b;
        int valid = 0;
        if (len >= 0 && len <= p + 1) {
            valid = len;
            for (int e0 = 0; e0 < len; e0 += 32) {
                const int e = e0 + lane;
                bool bad = false;
                if (e < len) {
                    const int j = col_idx[b + e];
                    const int prev = e > 0 ? col_idx[b + e - 1] : -1;
                    bad = j < 0 || j > p || j <= prev;
                }
                const unsigned m = __ballot_sync(0xffffffffu, bad);
                if (m) {
                    valid = e0 + __ffs(m) - 1;
                    break;
                }
            }
        }
        if (lane == 0) {
            if (valid != len) raise_status(flags, kDevBadSchedule);
            const int diag = valid > 0 && col_idx[b + valid - 1] == p ? 1 : 0;
            const int below = valid - diag;
            vlen128[p] = valid;
            cnt64[2 * p] = 2 * below + diag;
            if (2 * p + 1 < nb64) cnt64[2 * p + 1] = 2 * below + 2 * diag;
        }
    }
}

// One warp per 128-block row: writes the two 64-token rows at the scanned offsets.
__global__ void bwd_expand128_fill(int nb128, int nb64, const int32_t *__restrict__ row_ptr,
                                   const int32_t *__restrict__ col_idx, const int *__restrict__ vlen128,
                                   const int *__restrict__ rp64, int32_t *__restrict__ ci64) {
    const int lane = threadIdx.x & 31;
    const int nw = gridDim.x * (blockDim.x >> 5);
    for (int p = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < nb128; p += nw) {
        const int b = row_ptr[p], valid = vlen128[p];
        const bool second = 2 * p + 1 < nb64;
        // an overflowing total leaves the offsets equal (every row empty): nothing to write
        const int o0 = rp64[2 * p], o1 = second ? rp64[2 * p + 1] : 0;
        const bool room0 = rp64[2 * p + 1] > o0 || valid == 0;
        const bool room1 = second && (rp64[2 * p + 2] > o1 || valid == 0);
        for (int e = lane; e < valid; e += 32) {
            const int j = col_idx[b + e];
            if (j < p) {
                if (room0) { ci64[o0 + 2 * e] = 2 * j; ci64[o0 + 2 * e + 1] = 2 * j + 1; }
                if (room1) { ci64[o1 + 2 * e] = 2 * j; ci64[o1 + 2 * e + 1] = 2 * j + 1; }
            } else {  // j == p, the last entry
                if (room0) ci64[o0 + 2 * e] = 2 * p;
                if (room1) { ci64[o1 + 2 * e] = 2 * p; ci64[o1 + 2 * e + 1] = 2 * p + 1; }
            }
        }
    }
}

// One warp per column: number of query blocks whose row holds it.
__global__ void bwd_col_count(int nb, int words, const unsigned *__restrict__ bitmap, int *__restrict__ cnt) {
    const int lane = threadIdx.x & 31;
    const int nw = gridDim.x * (blockDim.x >> 5);
    for (int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); j < nb; j += nw) {
        int c = 0;
        for (int w = lane; w < words; w += 32) c += __popc(bitmap[(size_t)j * words + w]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
        if (lane == 0) cnt[j] = c;
    }
}

// One CTA: col_ptr = exclusive scan of the counts.  If the total exceeds the capacity of the
// row list, every column is left empty and the status word reports it.
__global__ void __launch_bounds__(1024) bwd_col_scan(int nb, const int *__restrict__ cnt, int *__restrict__ col_ptr,
                                                     long long cap, DeviceFlags flags) {
    __shared__ long long warp_tot[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int per = (nb + blockDim.x - 1) / blockDim.x;
    const int beg = min(nb, tid * per), end = min(nb, beg + per);
    long long run = 0;
    for (int j = beg; j < end; ++j) run += cnt[j];
    long long incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        long long t = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long o = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += o;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    const long long total = warp_tot[nwarps - 1];
    const bool fits = total <= cap;
    long long at = (warp > 0 ? warp_tot[warp - 1] : 0) + incl - run;
    for (int j = beg; j < end; ++j) {
        col_ptr[j] = fits ? (int)at : 0;
        at += cnt[j];
    }
    if (tid == 0) {
        col_ptr[nb] = fits ? (int)total : 0;
        if (!fits) raise_status(flags, kDevCapacity);
    }
}

// One warp per column: its query blocks in ascending order.
__global__ void bwd_col_fill(int nb, int words, const unsigned *__restrict__ bitmap,
                             const int *__restrict__ col_ptr, int32_t *__restrict__ row_idx) {
    const int lane = threadIdx.x & 31;
    const int nw = gridDim.x * (blockDim.x >> 5);
    for (int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); j < nb; j += nw) {
        int off = col_ptr[j];
        const int end = col_ptr[j + 1];
        for (int w0 = 0; w0 < words; w0 += 32) {
            const int w = w0 + lane;
            unsigned bits = w < words ? bitmap[(size_t)j * words + w] : 0u;
            const int c = __popc(bits);
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += x;
            }
            int pos = off + incl - c;
            while (bits) {
                const int bit = __ffs(bits) - 1;
                if (pos < end) row_idx[pos] = w * 32 + bit;
                ++pos;
                bits &= bits - 1u;
            }
            off += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
}

// One CTA: the key blocks sorted by the length of their transposed column (descending, then
// by index) and paired in that order -- pairs[2p], pairs[2p+1] (-1 if nb is odd and p is the
// last pair).  A dK/dV CTA walks the union of its two columns, so pairing a long column (a
// sink or top-k block that nearly every query block holds) with a short one would leave half
// of its 128-row tile idle for the whole long walk; sorted pairs also put the longest walks
// first in launch order.  Bitonic sort of (~count << 32 | j) keys in shared memory.
__global__ void __launch_bounds__(1024) bwd_col_pairs(int nb, int pow2, const int *__restrict__ cnt,
                                                       int *__restrict__ pairs) {
    extern __shared__ unsigned long long keys[];
    for (int i = threadIdx.x; i < pow2; i += blockDim.x)
        keys[i] = i < nb ? ((unsigned long long)(0xFFFFFFFFu - (unsigned)cnt[i]) << 32) | (unsigned)i : ~0ull;
    __syncthreads();
    for (int k = 2; k <= pow2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < pow2; i += blockDim.x) {
                const int p = i ^ j;
                if (p > i) {
                    const unsigned long long a = keys[i], b = keys[p];
                    if ((a > b) == ((i & k) == 0)) {
                        keys[i] = b;
                        keys[p] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    const int npairs = (nb + 1) >> 1;
    for (int q = threadIdx.x; q < 2 * npairs; q += blockDim.x)
        pairs[q] = q < nb ? (int)(keys[q] & 0xFFFFFFFFull) : -1;
}

// ---------------------------------------------------------------- Delta = rowsum(dO * O)
template <bool kBF16>
__device__ __forceinline__ float to_f32(uint32_t h16) {
    if constexpr (kBF16) return __uint_as_float(h16 << 16);
    else return __half2float(__ushort_as_half((unsigned short)h16));
}

// Delta per row in fp32.  kG = D / 8 threads per row (8 or 16, so a row never straddles a warp),
// each reading 16 bytes of O and of dO; products summed in the thread, then across the group.
// Grid: y over lanes, x over a lane's (row, 16-byte chunk) items -- at most 8192 * 64 * 16, so
// 32-bit indices and shifts -- with four items per thread whose loads are all issued before
// their arithmetic.  Rows are laid out per lane over Sp = nb * 64 tokens; the tokens past S (a
// partial last block) get Delta 0 and log-sum-exp -inf, and the given log-sum-exp is copied
// into the same layout.
constexpr int kDeltaItems = 4;
template <bool kBF16, int kG>
__global__ void __launch_bounds__(256) bwd_delta(const uint16_t *__restrict__ O, const uint16_t *__restrict__ dO,
                                                 const float *__restrict__ lse, int S, int Sp,
                                                 float *__restrict__ delta, float *__restrict__ lse_pad) {
    constexpr int D = kG * 8;
    const long long lane = blockIdx.y;
    const int per_lane = Sp * kG;
    const int first = (int)blockIdx.x * (int)blockDim.x * kDeltaItems + (int)threadIdx.x;
    uint4 a[kDeltaItems], b[kDeltaItems];
#pragma unroll
    for (int k = 0; k < kDeltaItems; ++k) {
        const int x = first + k * (int)blockDim.x;
        const int t = x / kG;  // token within the lane
        if (x < per_lane && t < S) {
            const size_t off = (size_t)(lane * S + t) * D + (size_t)(x % kG) * 8;
            a[k] = __ldg(reinterpret_cast<const uint4 *>(O + off));
            b[k] = __ldg(reinterpret_cast<const uint4 *>(dO + off));
        } else {
            a[k] = b[k] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
#pragma unroll
    for (int k = 0; k < kDeltaItems; ++k) {
        const int x = first + k * (int)blockDim.x;
        const int t = x / kG;
        const uint32_t av[4] = {a[k].x, a[k].y, a[k].z, a[k].w}, bv[4] = {b[k].x, b[k].y, b[k].z, b[k].w};
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc = fmaf(to_f32<kBF16>(av[q] & 0xFFFFu), to_f32<kBF16>(bv[q] & 0xFFFFu), acc);
            acc = fmaf(to_f32<kBF16>(av[q] >> 16), to_f32<kBF16>(bv[q] >> 16), acc);
        }
#pragma unroll
        for (int off = kG >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (x < per_lane && x % kG == 0) {
            const long long pr = lane * Sp + t;  // padded row
            delta[pr] = acc;
            lse_pad[pr] = t < S ? __ldg(lse + lane * S + t) : -INFINITY;
        }
    }
}

// ---------------------------------------------------------------- shared helpers

// Two floats rounded to the 16-bit input dtype and packed (first in the low half).
template <bool kBF16>
__device__ __forceinline__ uint32_t pack16x2(float a, float b) {
    if constexpr (kBF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

// Union of two ascending index lists (already checked), with membership bits (1: first list,
// 2: second list); -1 at the end.
struct ListUnion {
    const int32_t *a, *b;
    int ia, ia_end, ib, ib_end;

    __device__ int next(int &flags) {
        const int ja = ia < ia_end ? __ldg(a + ia) : INT_MAX;
        const int jb = ib < ib_end ? __ldg(b + ib) : INT_MAX;
        if (ja == INT_MAX && jb == INT_MAX) {
            flags = 0;
            return -1;
        }
        const int j = ja < jb ? ja : jb;
        flags = (ja == j ? 1 : 0) | (jb == j ? 2 : 0);
        if (ja == j) ++ia;
        if (jb == j) ++ib;
        return j;
    }
};

// 128 rows of fp32 accumulator in TMEM (this warp's 32 lanes, D columns starting at `col`),
// times `mul`, rounded and written to a 128-row SW128 staging tile in the layout TMA stores.
template <int D, bool kBF16>
__device__ __forceinline__ void stage_rows(uint32_t tmem_row, uint32_t col, bool valid, float mul,
                                           uint32_t tile, int row) {
    const uint32_t sw = (uint32_t)(row & 7);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
        const uint32_t o_row = tile + c * 16384 + row * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t o[32];
            if (valid) {
                tmem_ld32(tmem_row + col + c * 64 + h * 32, o);
            } else {
#pragma unroll
                for (int t = 0; t < 32; ++t) o[t] = 0u;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    w[t] = pack16x2<kBF16>(__uint_as_float(o[q * 8 + 2 * t]) * mul,
                                           __uint_as_float(o[q * 8 + 2 * t + 1]) * mul);
                st_shared_v4(o_row + (((uint32_t)(h * 4 + q) ^ sw) << 4), w[0], w[1], w[2], w[3]);
            }
        }
    }
}

// Row `row` (0-127) of a 128-row SW128 staging tile (the layout stage_rows writes: 64-column
// chunks of 16 KB, 16-byte units of a row permuted by row & 7) copied to a global row of D
// 16-bit values.
template <int D>
__device__ __forceinline__ void copy_staged_row(const uint8_t *tile, int row, uint16_t *dst) {
    const uint32_t sw = (uint32_t)(row & 7);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
        const uint8_t *src = tile + c * 16384 + row * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4 *>(dst + c * 64 + u * 8) =
                *reinterpret_cast<const uint4 *>(src + (((uint32_t)u ^ sw) << 4));
    }
}

// Meta area (byte offsets from the meta base), common to both kernels.
constexpr int kBarTile = 0;                           // resident tile(s) loaded
constexpr int kBarFull = 8;                           // kStream x 8: streamed block landed
constexpr int kBarEmpty = kBarFull + 8 * kStream;     // kStream x 8: streamed block released
constexpr int kBarSFull = kBarEmpty + 8 * kStream;    // 2 x 8: products of a step in TMEM
constexpr int kBarPFull = kBarSFull + 16;             // 2 x 8: elementwise results of a step in TMEM
constexpr int kBarDone = kBarPFull + 16;              // accumulation MMA of a step completed
constexpr int kBarFin = kBarDone + 8;
constexpr int kBarVFull = kBarFin + 8;                // dQ kernel: kStream x 8, V of a step landed
constexpr int kBarVEmpty = kBarVFull + 8 * kStream;   // dQ kernel: kStream x 8
constexpr int kTmemSlot = kBarVEmpty + 8 * kStream;
constexpr int kAbortFlag = kTmemSlot + 4;
constexpr int kMetaJ = kAbortFlag + 4;                // kMetaRing x 4
constexpr int kMetaF = kMetaJ + 4 * kMetaRing;        // kMetaRing x 4
constexpr int kMetaBytes = 256;
static_assert(kMetaF + 4 * kMetaRing <= kMetaBytes, "meta area");

constexpr uint32_t kTmemCols = 512;  // S0 | S1 | dP0 | dP1 | accumulator(s)

// Each CTA takes all 512 TMEM columns, so a second CTA on the same SM would only wait in its
// allocation: ask for more than half of the SM's shared memory so that one CTA fits.
constexpr int smem_bytes_one_cta(int need) { return need > 116 * 1024 ? need : 116 * 1024; }
__device__ __forceinline__ uint32_t s_col(int b) { return b ? 64u : 0u; }
__device__ __forceinline__ uint32_t dp_col(int b) { return b ? 192u : 128u; }
constexpr uint32_t kAccCol = 256;

// ---------------------------------------------------------------- dQ
template <int D>
struct DqSmem {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kRows * D * 2;   // Q and dO tiles (128 rows)
    static constexpr int kKVBytes = kBlock * D * 2;    // one K or V block
    static constexpr int kOffQ = 0;
    static constexpr int kOffDO = kOffQ + kTileBytes;
    static constexpr int kOffK = kOffDO + kTileBytes;
    static constexpr int kOffV = kOffK + kStream * kKVBytes;
    static constexpr int kOffMeta = kOffV + kStream * kKVBytes;
    static constexpr int kBytes = smem_bytes_one_cta(kOffMeta + kMetaBytes + 1024);  // + alignment slack
};

template <int D, bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
              const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const __grid_constant__ CUtensorMap tmdQ, const int32_t *__restrict__ row_ptr,
              const int32_t *__restrict__ col_idx, const int *__restrict__ vlen,
              const float *__restrict__ lse, const float *__restrict__ delta, int nb, int S,
              float scale, float scale_log2, uint16_t *__restrict__ dQ, DeviceFlags flags) {
    using L = DqSmem<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    if (base - raw_base + L::kOffMeta + kMetaBytes > (uint32_t)L::kBytes) {
        if (threadIdx.x == 0) raise_status(flags, kDevSmemAlign);
        return;
    }
    uint8_t *smem = smem_raw + (base - raw_base);
    const uint32_t sQ = base + L::kOffQ, sdO = base + L::kOffDO, sK = base + L::kOffK, sV = base + L::kOffV;
    const uint32_t meta = base + L::kOffMeta;
    volatile int *meta_j = reinterpret_cast<volatile int *>(smem + L::kOffMeta + kMetaJ);
    volatile int *meta_f = reinterpret_cast<volatile int *>(smem + L::kOffMeta + kMetaF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMeta + kAbortFlag);
    const uint32_t bar_tile = meta + kBarTile, bar_done = meta + kBarDone, bar_fin = meta + kBarFin;
#define BAR_K_FULL(s) (meta + kBarFull + 8u * (uint32_t)(s))
#define BAR_K_EMPTY(s) (meta + kBarEmpty + 8u * (uint32_t)(s))
#define BAR_V_FULL(s) (meta + kBarVFull + 8u * (uint32_t)(s))
#define BAR_V_EMPTY(s) (meta + kBarVEmpty + 8u * (uint32_t)(s))
#define BAR_S_FULL(b) (meta + kBarSFull + 8u * (uint32_t)(b))
#define BAR_P_FULL(b) (meta + kBarPFull + 8u * (uint32_t)(b))

    const int tid = threadIdx.x, warp = tid >> 5;
    const int lane_id = blockIdx.x;
    const int npairs = (nb + 1) >> 1;
    const int qa = 2 * (npairs - 1 - (int)blockIdx.y);  // longest rows first
    const bool has_b = qa + 1 < nb;
    const int row0 = lane_id * S;

    // The first global reads are issued together and waited for at the barrier below: whether
    // the launch already gave up elsewhere (one thread, so the whole CTA takes the same branch),
    // and the producer's two CSR rows.
    const bool gave_up = tid == 0 && *reinterpret_cast<volatile unsigned *>(flags.abort_epoch) == flags.epoch;
    ListUnion lu;
    if (tid == kProducerWarp * 32) {
        lu.a = col_idx + row_ptr[qa];
        lu.ia = 0;
        lu.ia_end = vlen[qa];
        lu.b = has_b ? col_idx + row_ptr[qa + 1] : col_idx;
        lu.ib = 0;
        lu.ib_end = has_b ? vlen[qa + 1] : 0;
    }

    if (tid == 0) {
        mbar_init(bar_tile, 1);
        for (int s = 0; s < kStream; ++s) {
            mbar_init(BAR_K_FULL(s), 1);
            mbar_init(BAR_K_EMPTY(s), 1);
            mbar_init(BAR_V_FULL(s), 1);
            mbar_init(BAR_V_EMPTY(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(BAR_S_FULL(b), 1);
            mbar_init(BAR_P_FULL(b), kRows);
        }
        mbar_init(bar_done, 1);
        mbar_init(bar_fin, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(meta + kTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    const bool leave = __syncthreads_or(gave_up);
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kOffMeta + kTmemSlot);
    if (leave) {  // nothing was issued yet: give the columns back and go
        if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
        return;
    }

    if (warp == kProducerWarp) {
        if ((tid & 31) == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmdO);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmdQ);
            mbar_arrive_expect_tx(bar_tile, 2 * L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c) {
                tma_load_2d(sQ + c * 16384, &tmQ, c * 64, row0 + qa * kBlock, bar_tile);
                tma_load_2d(sdO + c * 16384, &tmdO, c * 64, row0 + qa * kBlock, bar_tile);
            }
            bool ok = true;
            int k_issued = 0, v_issued = 0;
            for (int v = 0;; ++v) {
                const int s = v % kStream;
                const uint32_t par = (uint32_t)((v / kStream) - 1) & 1u;
                if (v >= kStream && !mbar_wait(BAR_K_EMPTY(s), par, flags)) { ok = false; break; }
                int f = 0;
                const int j = lu.next(f);
                meta_j[v % kMetaRing] = j;
                meta_f[v % kMetaRing] = f;
                if (j < 0) {
                    mbar_arrive(BAR_K_FULL(s));
                    break;
                }
                const int y = row0 + j * kBlock;
                mbar_arrive_expect_tx(BAR_K_FULL(s), L::kKVBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_2d(sK + s * L::kKVBytes + c * 8192, &tmK, c * 64, y, BAR_K_FULL(s));
                k_issued = v + 1;
                if (v >= kStream && !mbar_wait(BAR_V_EMPTY(s), par, flags)) { ok = false; break; }
                mbar_arrive_expect_tx(BAR_V_FULL(s), L::kKVBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_2d(sV + s * L::kKVBytes + c * 8192, &tmV, c * 64, y, BAR_V_FULL(s));
                v_issued = v + 1;
            }
            if (!ok) {
                *abort_flag = 1;
                (void)mbar_wait_timed(bar_tile, 0);
                for (int w = k_issued - kStream; w < k_issued; ++w)
                    if (w >= 0) (void)mbar_wait_timed(BAR_K_FULL(w % kStream), (w / kStream) & 1);
                for (int w = v_issued - kStream; w < v_issued; ++w)
                    if (w >= 0) (void)mbar_wait_timed(BAR_V_FULL(w % kStream), (w / kStream) & 1);
            }
        }
    } else if (warp == kMmaWarp) {
        if ((tid & 31) == 0) {
            constexpr uint32_t kIdescS = idesc_f16(kBF16, 128, 64, false);
            constexpr uint32_t kIdescAcc = idesc_f16(kBF16, 128, D, true);
            bool ok = mbar_wait(bar_tile, 0, flags);
            int u = 0;
            bool have = false;
            // products of step uu: S = Q K^T and dP = dO V^T; V's stage is free afterwards
            auto issue_products = [&](int uu) -> bool {
                const int s_ = uu % kStream;
                if (!mbar_wait(BAR_V_FULL(s_), (uu / kStream) & 1, flags)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint32_t boff = s_ * L::kKVBytes + (kk >> 2) * 8192 + (kk & 3) * 32;
                    tc_mma_ss(tmem + s_col(uu & 1), sdesc_sw128(sQ + koff, 16, 1024),
                              sdesc_sw128(sK + boff, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint32_t boff = s_ * L::kKVBytes + (kk >> 2) * 8192 + (kk & 3) * 32;
                    tc_mma_ss(tmem + dp_col(uu & 1), sdesc_sw128(sdO + koff, 16, 1024),
                              sdesc_sw128(sV + boff, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
                }
                tc_commit(BAR_S_FULL(uu & 1));
                tc_commit(BAR_V_EMPTY(s_));
                return true;
            };
            if (ok) {
                ok = mbar_wait(BAR_K_FULL(0), 0, flags);
                if (ok) {
                    if (meta_j[0] >= 0) {
                        ok = issue_products(0);
                        have = ok;
                    } else {
                        mbar_arrive(BAR_S_FULL(0));
                    }
                }
            }
            while (ok && have) {
                bool next = false;
                const int s1 = (u + 1) % kStream;
                ok = mbar_wait(BAR_K_FULL(s1), ((u + 1) / kStream) & 1, flags);
                if (!ok) break;
                if (meta_j[(u + 1) % kMetaRing] >= 0) {
                    ok = issue_products(u + 1);
                    if (!ok) break;
                    next = true;
                } else {
                    mbar_arrive(BAR_S_FULL((u + 1) & 1));
                }
                // dQ += dS_u K_u once the elementwise warps have written dS_u
                ok = mbar_wait(BAR_P_FULL(u & 1), (u >> 1) & 1, flags);
                if (!ok) break;
                const int s = u % kStream;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_ts(tmem + kAccCol, tmem + s_col(u & 1) + kk * 8,
                              sdesc_sw128(sK + s * L::kKVBytes + kk * 2048, 8192, 1024), kIdescAcc,
                              (u > 0 || kk > 0) ? 1u : 0u);
                tc_commit(BAR_K_EMPTY(s));
                tc_commit(bar_done);
                have = next;
                ++u;
            }
            if (!ok) *abort_flag = 1;
            tc_commit(bar_fin);
            (void)mbar_wait_timed(bar_fin, 0);
        }
    } else {
        // ------------------------------------------------------------ elementwise (warps 0-3)
        const int half = tid >> 6;
        const int r_in = tid & 63;
        const int my_block = qa + half;
        const bool row_exists = half == 0 || has_b;
        const uint32_t t_lane = (uint32_t)(warp * 32) << 16;
        // the row in the per-lane padded Delta / log-sum-exp arrays (nb * 64 rows per lane)
        const long long grow = ((long long)lane_id * nb + qa) * kBlock + tid;
        const float lse2 = row_exists ? lse[grow] * kLog2e : -INFINITY;
        const float dlt = row_exists ? delta[grow] : 0.f;
        const bool live = lse2 > -INFINITY;  // a row with keys
        bool ok = true;
        int u = 0;
        for (;; ++u) {
            if (!mbar_wait(BAR_S_FULL(u & 1), (u >> 1) & 1, flags)) { ok = false; break; }
            const int j = meta_j[u % kMetaRing];
            const int fl = meta_f[u % kMetaRing];
            if (j < 0) break;
            tc_fence_after();
            const bool in_row = row_exists && ((fl >> half) & 1);  // warp-uniform
            uint32_t dsw[32];
            __syncwarp();
            if (in_row) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t sr[32], pr[32];
                    tmem_ld32_pair(tmem + t_lane + s_col(u & 1) + h * 32, sr,
                                   tmem + t_lane + dp_col(u & 1) + h * 32, pr);
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        float ds[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int c = h * 32 + 2 * t + e;
                            const bool masked = !live || (j == my_block && c > r_in);
                            const float p = masked ? 0.f
                                                   : ex2_approx(fmaf(__uint_as_float(sr[2 * t + e]), scale_log2, -lse2));
                            ds[e] = p * (__uint_as_float(pr[2 * t + e]) - dlt);
                        }
                        dsw[h * 16 + t] = pack16x2<kBF16>(ds[0], ds[1]);
                    }
                }
            } else {
#pragma unroll
                for (int t = 0; t < 32; ++t) dsw[t] = 0u;
            }
            __syncwarp();
            tmem_st32(tmem + t_lane + s_col(u & 1), dsw);  // dS_u over the first 32 columns of S_u
            tc_fence_before();
            mbar_arrive(BAR_P_FULL(u & 1));
        }
        if (!ok) *abort_flag = 1;
        bool acc_valid = false;
        if (ok && u > 0) {
            acc_valid = mbar_wait(bar_done, (u - 1) & 1, flags);
            if (!acc_valid) *abort_flag = 1;
        }
        // one decision for all elementwise warps (the section below has a barrier of its own)
        if (!named_barrier_or(1, kRows, *abort_flag != 0)) {
            tc_fence_after();
            __syncwarp();
            // every product that read Q has completed: Q's tile stages dQ
            stage_rows<D, kBF16>(tmem + t_lane, kAccCol, acc_valid, scale, sQ, tid);
            fence_proxy_async_smem();
            named_barrier(1, kRows);
            // A partial last block (S not a multiple of 64) is not TMA-stored -- its box would
            // run into the next lane's rows -- but copied row by row from the staging tile.
            const bool part_a = (qa + 1) * kBlock > S, part_b = has_b && (qa + 2) * kBlock > S;
            if (tid == 0) {
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c) {
                    if (!part_a) tma_store_2d(&tmdQ, c * 64, row0 + qa * kBlock, sQ + c * 16384);
                    if (has_b && !part_b)
                        tma_store_2d(&tmdQ, c * 64, row0 + (qa + 1) * kBlock, sQ + c * 16384 + 8192);
                }
                tma_store_commit();
                tma_store_wait_read();
            }
            if ((half ? part_b : part_a) && qa * kBlock + tid < S)
                copy_staged_row<D>(smem + (sQ - base), tid, dQ + ((size_t)row0 + qa * kBlock + tid) * D);
        }
    }
#undef BAR_K_FULL
#undef BAR_K_EMPTY
#undef BAR_V_FULL
#undef BAR_V_EMPTY
#undef BAR_S_FULL
#undef BAR_P_FULL
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        raise_status(flags, kDevTimeout);
        atomicExch(flags.abort_epoch, flags.epoch);
    }
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- dK, dV
template <int D>
struct DkvSmem {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kRows * D * 2;   // K and V tiles (128 keys)
    static constexpr int kQBytes = kBlock * D * 2;     // one Q or dO block
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffQ = kOffV + kTileBytes;
    static constexpr int kOffDO = kOffQ + kStream * kQBytes;
    static constexpr int kOffLse = kOffDO + kStream * kQBytes;     // kStream x 64 floats
    static constexpr int kOffDelta = kOffLse + kStream * 256;      // kStream x 64 floats
    static constexpr int kOffMeta = kOffDelta + kStream * 256;
    static constexpr int kBytes = smem_bytes_one_cta(kOffMeta + kMetaBytes + 1024);
};

template <int D, bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dkv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
               const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
               const int *__restrict__ col_ptr, const int32_t *__restrict__ row_idx,
               const int *__restrict__ pairs, const float *__restrict__ lse,
               const float *__restrict__ delta, int nb, int S, float scale, float scale_log2,
               uint16_t *__restrict__ dK, uint16_t *__restrict__ dV, DeviceFlags flags) {
    using L = DkvSmem<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    if (base - raw_base + L::kOffMeta + kMetaBytes > (uint32_t)L::kBytes) {
        if (threadIdx.x == 0) raise_status(flags, kDevSmemAlign);
        return;
    }
    uint8_t *smem = smem_raw + (base - raw_base);
    const uint32_t sK = base + L::kOffK, sV = base + L::kOffV, sQ = base + L::kOffQ, sdO = base + L::kOffDO;
    const uint32_t sLse = base + L::kOffLse, sDelta = base + L::kOffDelta;
    const float *lse_s = reinterpret_cast<const float *>(smem + L::kOffLse);
    const float *delta_s = reinterpret_cast<const float *>(smem + L::kOffDelta);
    const uint32_t meta = base + L::kOffMeta;
    volatile int *meta_j = reinterpret_cast<volatile int *>(smem + L::kOffMeta + kMetaJ);
    volatile int *meta_f = reinterpret_cast<volatile int *>(smem + L::kOffMeta + kMetaF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMeta + kAbortFlag);
    const uint32_t bar_tile = meta + kBarTile, bar_done = meta + kBarDone, bar_fin = meta + kBarFin;
#define BAR_FULL(s) (meta + kBarFull + 8u * (uint32_t)(s))
#define BAR_EMPTY(s) (meta + kBarEmpty + 8u * (uint32_t)(s))
#define BAR_S_FULL(b) (meta + kBarSFull + 8u * (uint32_t)(b))
#define BAR_P_FULL(b) (meta + kBarPFull + 8u * (uint32_t)(b))

    const int tid = threadIdx.x, warp = tid >> 5;
    const int lane_id = blockIdx.x;
    // key blocks ka and kb (-1: none) from the pair list, heaviest transposed columns first
    const int ka = __ldg(pairs + 2 * blockIdx.y), kb = __ldg(pairs + 2 * blockIdx.y + 1);
    const bool has_b = kb >= 0;
    const int row0 = lane_id * S;

    // As in the dQ kernel: the abort flag and the producer's two transposed columns are read
    // before the first barrier.
    const bool gave_up = tid == 0 && *reinterpret_cast<volatile unsigned *>(flags.abort_epoch) == flags.epoch;
    ListUnion lu;
    if (tid == kProducerWarp * 32) {
        lu.a = row_idx + col_ptr[ka];
        lu.ia = 0;
        lu.ia_end = col_ptr[ka + 1] - col_ptr[ka];
        lu.b = has_b ? row_idx + col_ptr[kb] : row_idx;
        lu.ib = 0;
        lu.ib_end = has_b ? col_ptr[kb + 1] - col_ptr[kb] : 0;
    }

    if (tid == 0) {
        mbar_init(bar_tile, 1);
        for (int s = 0; s < kStream; ++s) {
            mbar_init(BAR_FULL(s), 1);
            mbar_init(BAR_EMPTY(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(BAR_S_FULL(b), 1);
            mbar_init(BAR_P_FULL(b), kRows);
        }
        mbar_init(bar_done, 1);
        mbar_init(bar_fin, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(meta + kTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    const bool leave = __syncthreads_or(gave_up);
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kOffMeta + kTmemSlot);
    if (leave) {  // nothing was issued yet: give the columns back and go
        if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
        return;
    }
    constexpr uint32_t kDVCol = kAccCol, kDKCol = kAccCol + D;

    if (warp == kProducerWarp) {
        if ((tid & 31) == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmdO);
            tma_prefetch_desc(&tmdK);
            tma_prefetch_desc(&tmdV);
            mbar_arrive_expect_tx(bar_tile, 2 * L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c) {
                tma_load_2d(sK + c * 16384, &tmK, c * 64, row0 + ka * kBlock, bar_tile);
                tma_load_2d(sV + c * 16384, &tmV, c * 64, row0 + ka * kBlock, bar_tile);
                // the second block's rows, or the first block's again (masked) if there is none
                tma_load_2d(sK + c * 16384 + 8192, &tmK, c * 64, row0 + (has_b ? kb : ka) * kBlock, bar_tile);
                tma_load_2d(sV + c * 16384 + 8192, &tmV, c * 64, row0 + (has_b ? kb : ka) * kBlock, bar_tile);
            }
            bool ok = true;
            int issued = 0;
            for (int v = 0;; ++v) {
                const int s = v % kStream;
                const uint32_t par = (uint32_t)((v / kStream) - 1) & 1u;
                if (v >= kStream && !mbar_wait(BAR_EMPTY(s), par, flags)) { ok = false; break; }
                int f = 0;
                const int i = lu.next(f);
                meta_j[v % kMetaRing] = i;
                meta_f[v % kMetaRing] = f;
                if (i < 0) {
                    mbar_arrive(BAR_FULL(s));
                    break;
                }
                const int y = row0 + i * kBlock;
                mbar_arrive_expect_tx(BAR_FULL(s), 2 * L::kQBytes + 512);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c) {
                    tma_load_2d(sQ + s * L::kQBytes + c * 8192, &tmQ, c * 64, y, BAR_FULL(s));
                    tma_load_2d(sdO + s * L::kQBytes + c * 8192, &tmdO, c * 64, y, BAR_FULL(s));
                }
                const long long py = ((long long)lane_id * nb + i) * kBlock;  // padded row
                bulk_load(sLse + s * 256, lse + py, 256, BAR_FULL(s));
                bulk_load(sDelta + s * 256, delta + py, 256, BAR_FULL(s));
                issued = v + 1;
            }
            if (!ok) {
                *abort_flag = 1;
                (void)mbar_wait_timed(bar_tile, 0);
                for (int w = issued - kStream; w < issued; ++w)
                    if (w >= 0) (void)mbar_wait_timed(BAR_FULL(w % kStream), (w / kStream) & 1);
            }
        }
    } else if (warp == kMmaWarp) {
        if ((tid & 31) == 0) {
            constexpr uint32_t kIdescS = idesc_f16(kBF16, 128, 64, false);
            constexpr uint32_t kIdescAcc = idesc_f16(kBF16, 128, D, true);
            bool ok = mbar_wait(bar_tile, 0, flags);
            int u = 0;
            bool have = false;
            // products of step uu: S^T = K Q^T and dP^T = V dO^T
            auto issue_products = [&](int uu) {
                const int s_ = uu % kStream;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint32_t boff = s_ * L::kQBytes + (kk >> 2) * 8192 + (kk & 3) * 32;
                    tc_mma_ss(tmem + s_col(uu & 1), sdesc_sw128(sK + aoff, 16, 1024),
                              sdesc_sw128(sQ + boff, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint32_t boff = s_ * L::kQBytes + (kk >> 2) * 8192 + (kk & 3) * 32;
                    tc_mma_ss(tmem + dp_col(uu & 1), sdesc_sw128(sV + aoff, 16, 1024),
                              sdesc_sw128(sdO + boff, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
                }
                tc_commit(BAR_S_FULL(uu & 1));
            };
            if (ok) {
                ok = mbar_wait(BAR_FULL(0), 0, flags);
                if (ok) {
                    if (meta_j[0] >= 0) {
                        issue_products(0);
                        have = true;
                    } else {
                        mbar_arrive(BAR_S_FULL(0));
                    }
                }
            }
            while (ok && have) {
                bool next = false;
                const int s1 = (u + 1) % kStream;
                ok = mbar_wait(BAR_FULL(s1), ((u + 1) / kStream) & 1, flags);
                if (!ok) break;
                if (meta_j[(u + 1) % kMetaRing] >= 0) {
                    issue_products(u + 1);
                    next = true;
                } else {
                    mbar_arrive(BAR_S_FULL((u + 1) & 1));
                }
                // dV += P^T_u dO_u and dK += dS^T_u Q_u once the elementwise warps wrote them
                ok = mbar_wait(BAR_P_FULL(u & 1), (u >> 1) & 1, flags);
                if (!ok) break;
                const int s = u % kStream;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_ts(tmem + kDVCol, tmem + s_col(u & 1) + kk * 8,
                              sdesc_sw128(sdO + s * L::kQBytes + kk * 2048, 8192, 1024), kIdescAcc,
                              (u > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_ts(tmem + kDKCol, tmem + dp_col(u & 1) + kk * 8,
                              sdesc_sw128(sQ + s * L::kQBytes + kk * 2048, 8192, 1024), kIdescAcc,
                              (u > 0 || kk > 0) ? 1u : 0u);
                tc_commit(BAR_EMPTY(s));
                tc_commit(bar_done);
                have = next;
                ++u;
            }
            if (!ok) *abort_flag = 1;
            tc_commit(bar_fin);
            (void)mbar_wait_timed(bar_fin, 0);
        }
    } else {
        // ------------------------------------------------------------ elementwise (warps 0-3)
        const int half = tid >> 6;               // 0: key block ka, 1: key block kb
        const int k_in = tid & 63;               // key token within its block
        const int key_block = half ? kb : ka;
        const bool row_exists = half == 0 || has_b;
        const uint32_t t_lane = (uint32_t)(warp * 32) << 16;
        bool ok = true;
        int u = 0;
        for (;; ++u) {
            if (!mbar_wait(BAR_S_FULL(u & 1), (u >> 1) & 1, flags)) { ok = false; break; }
            const int i = meta_j[u % kMetaRing];
            const int fl = meta_f[u % kMetaRing];
            if (i < 0) break;
            const int s = u % kStream;
            // the step's log-sum-exp and Delta rows arrived with its Q and dO blocks
            if (!mbar_wait(BAR_FULL(s), (u / kStream) & 1, flags)) { ok = false; break; }
            tc_fence_after();
            const bool in_col = row_exists && ((fl >> half) & 1);  // warp-uniform
            uint32_t pw[32], dw[32];
            __syncwarp();
            if (in_col) {
                const float *ls = lse_s + s * 64;
                const float *dl = delta_s + s * 64;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t sr[32], pr[32];
                    tmem_ld32_pair(tmem + t_lane + s_col(u & 1) + h * 32, sr,
                                   tmem + t_lane + dp_col(u & 1) + h * 32, pr);
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        float p[2], ds[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int c = h * 32 + 2 * t + e;  // query token within block i
                            const float l2 = ls[c] * kLog2e;
                            const bool masked = l2 == -INFINITY || (i == key_block && k_in > c);
                            p[e] = masked ? 0.f : ex2_approx(fmaf(__uint_as_float(sr[2 * t + e]), scale_log2, -l2));
                            ds[e] = p[e] * (__uint_as_float(pr[2 * t + e]) - dl[c]);
                        }
                        pw[h * 16 + t] = pack16x2<kBF16>(p[0], p[1]);
                        dw[h * 16 + t] = pack16x2<kBF16>(ds[0], ds[1]);
                    }
                }
            } else {
#pragma unroll
                for (int t = 0; t < 32; ++t) pw[t] = dw[t] = 0u;
            }
            __syncwarp();
            tmem_st32(tmem + t_lane + s_col(u & 1), pw);   // P^T over the first 32 columns of S^T
            tmem_st32(tmem + t_lane + dp_col(u & 1), dw);  // dS^T over the first 32 of dP^T
            tc_fence_before();
            mbar_arrive(BAR_P_FULL(u & 1));
        }
        if (!ok) *abort_flag = 1;
        bool acc_valid = false;
        if (ok && u > 0) {
            acc_valid = mbar_wait(bar_done, (u - 1) & 1, flags);
            if (!acc_valid) *abort_flag = 1;
        }
        // one decision for all elementwise warps (the section below has a barrier of its own)
        if (!named_barrier_or(1, kRows, *abort_flag != 0)) {
            tc_fence_after();
            __syncwarp();
            // every product that read K and V has completed: their tiles stage dK and dV
            stage_rows<D, kBF16>(tmem + t_lane, kDVCol, acc_valid, 1.f, sV, tid);
            stage_rows<D, kBF16>(tmem + t_lane, kDKCol, acc_valid, scale, sK, tid);
            fence_proxy_async_smem();
            named_barrier(1, kRows);
            // a partial last key block is copied row by row (see the dQ kernel)
            const bool part_a = (ka + 1) * kBlock > S, part_b = has_b && (kb + 1) * kBlock > S;
            if (tid == 0) {
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c) {
                    if (!part_a) {
                        tma_store_2d(&tmdV, c * 64, row0 + ka * kBlock, sV + c * 16384);
                        tma_store_2d(&tmdK, c * 64, row0 + ka * kBlock, sK + c * 16384);
                    }
                    if (has_b && !part_b) {
                        tma_store_2d(&tmdV, c * 64, row0 + kb * kBlock, sV + c * 16384 + 8192);
                        tma_store_2d(&tmdK, c * 64, row0 + kb * kBlock, sK + c * 16384 + 8192);
                    }
                }
                tma_store_commit();
                tma_store_wait_read();
            }
            if ((half ? part_b : part_a) && key_block * kBlock + k_in < S) {
                const size_t grow_k = ((size_t)row0 + key_block * kBlock + k_in) * D;
                copy_staged_row<D>(smem + (sV - base), tid, dV + grow_k);
                copy_staged_row<D>(smem + (sK - base), tid, dK + grow_k);
            }
        }
    }
#undef BAR_FULL
#undef BAR_EMPTY
#undef BAR_S_FULL
#undef BAR_P_FULL
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        raise_status(flags, kDevTimeout);
        atomicExch(flags.abort_epoch, flags.epoch);
    }
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool kBF16>
tsa_status launch_grad_kernels(const BwdLaunch &a) {
    auto kq = bwd_dq_kernel<D, kBF16>;
    auto kkv = bwd_dkv_kernel<D, kBF16>;
    if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, DqSmem<D>::kBytes) != cudaSuccess ||
        cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, DkvSmem<D>::kBytes) != cudaSuccess)
        return TSA_ERR_CUDA;
    const unsigned npairs = (unsigned)((a.nb + 1) / 2);
    const dim3 grid((unsigned)a.lanes, npairs);
    const float scale_log2 = a.scale * kLog2e;
    kq<<<grid, kThreads, DqSmem<D>::kBytes, a.stream>>>(*a.tmQ128, *a.tmdO128, *a.tmK64, *a.tmV64, *a.tmdQ64,
                                                        a.row_ptr, a.col_idx, a.vlen, a.lse_pad, a.delta, a.nb,
                                                        a.S, a.scale, scale_log2, a.dQ, a.flags);
    kkv<<<grid, kThreads, DkvSmem<D>::kBytes, a.stream>>>(*a.tmK64, *a.tmV64, *a.tmQ64, *a.tmdO64, *a.tmdK64,
                                                          *a.tmdV64, a.col_ptr, a.row_idx, a.pairs, a.lse_pad, a.delta,
                                                          a.nb, a.S, a.scale, scale_log2, a.dK, a.dV, a.flags);
    return cudaGetLastError() == cudaSuccess ? TSA_OK : TSA_ERR_CUDA;
}

}  // namespace

BwdWorkspace backward_workspace_layout(int64_t lanes, int64_t S, int64_t nb, int64_t nnz_cap, int64_t nb_in) {
    BwdWorkspace w{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = (o + bytes + 255) & ~(size_t)255;
        return at;
    };
    const int64_t words = (nb + 31) / 32;
    w.delta = take(sizeof(float) * (size_t)(lanes * nb * 64));  // rows padded to whole blocks
    w.lse_pad = take(sizeof(float) * (size_t)(lanes * nb * 64));
    w.vlen = take(sizeof(int) * (size_t)nb);
    w.cnt = take(sizeof(int) * (size_t)nb);
    w.col_ptr = take(sizeof(int) * (size_t)(nb + 1));
    w.bitmap = take(sizeof(unsigned) * (size_t)(nb * words));
    w.bitmap_bytes = sizeof(unsigned) * (size_t)(nb * words);
    w.row_idx = take(sizeof(int32_t) * (size_t)(nnz_cap > 0 ? nnz_cap : 1));
    w.pairs = take(sizeof(int) * (size_t)(2 * ((nb + 1) / 2)));
    // a CSR of 128-token blocks (nb_in rows) expanded to 64-token blocks: nnz_cap is then the
    // expanded capacity
    w.vlen_in = take(sizeof(int) * (size_t)(nb_in > 0 ? nb_in : 1));
    w.rp64 = take(sizeof(int32_t) * (size_t)(nb + 1));
    w.ci64 = take(sizeof(int32_t) * (size_t)(nb_in > 0 ? nnz_cap : 1));
    w.total = o;
    return w;
}

tsa_status launch_attention_backward(const BwdLaunch &a_in) {
    BwdLaunch a = a_in;
    cudaStream_t st = a.stream;
    const int nb = a.nb;
    const int words = (nb + 31) / 32;
    const unsigned wgrid = (unsigned)((nb + 7) / 8 < 152 * 8 ? (nb + 7) / 8 : 152 * 8);
    if (a.nb_in > 0) {
        // 128-token CSR: the equivalent 64-token CSR first (cnt is free until the columns)
        const unsigned g = (unsigned)((a.nb_in + 7) / 8 < 152 * 8 ? (a.nb_in + 7) / 8 : 152 * 8);
        bwd_expand128_count<<<g, 256, 0, st>>>(a.nb_in, nb, a.row_ptr, a.col_idx, a.vlen_in, a.cnt, a.flags);
        bwd_col_scan<<<1, 1024, 0, st>>>(nb, a.cnt, a.rp64, (long long)a.nnz_cap, a.flags);
        bwd_expand128_fill<<<g, 256, 0, st>>>(a.nb_in, nb, a.row_ptr, a.col_idx, a.vlen_in, a.rp64, a.ci64);
        a.row_ptr = a.rp64;
        a.col_idx = a.ci64;
    }
    if (cudaMemsetAsync(a.bitmap, 0, a.bitmap_bytes, st) != cudaSuccess) return TSA_ERR_CUDA;
    bwd_rows<<<wgrid, 256, 0, st>>>(nb, a.row_ptr, a.col_idx, words, a.vlen, a.bitmap, a.flags);
    bwd_col_count<<<wgrid, 256, 0, st>>>(nb, words, a.bitmap, a.cnt);
    bwd_col_scan<<<1, 1024, 0, st>>>(nb, a.cnt, a.col_ptr, (long long)a.nnz_cap, a.flags);
    bwd_col_fill<<<wgrid, 256, 0, st>>>(nb, words, a.bitmap, a.col_ptr, a.row_idx);
    {
        int pow2 = 1;
        while (pow2 < nb) pow2 <<= 1;
        const size_t smem = sizeof(unsigned long long) * (size_t)pow2;  // <= 64 KB (nb <= 8192)
        if (cudaFuncSetAttribute(bwd_col_pairs, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return TSA_ERR_CUDA;
        bwd_col_pairs<<<1, 1024, smem, st>>>(nb, pow2, a.cnt, a.pairs);
    }
    {
        const int Sp = a.nb * kBlock;
        const int per_lane = Sp * (a.D / 8);
        const dim3 grid((unsigned)((per_lane + 256 * kDeltaItems - 1) / (256 * kDeltaItems)), (unsigned)a.lanes);
        if (a.D == 128) {
            if (a.bf16) bwd_delta<true, 16><<<grid, 256, 0, st>>>(a.O, a.dO, a.lse, a.S, Sp, a.delta, a.lse_pad);
            else bwd_delta<false, 16><<<grid, 256, 0, st>>>(a.O, a.dO, a.lse, a.S, Sp, a.delta, a.lse_pad);
        } else if (a.D == 64) {
            if (a.bf16) bwd_delta<true, 8><<<grid, 256, 0, st>>>(a.O, a.dO, a.lse, a.S, Sp, a.delta, a.lse_pad);
            else bwd_delta<false, 8><<<grid, 256, 0, st>>>(a.O, a.dO, a.lse, a.S, Sp, a.delta, a.lse_pad);
        } else {
            return TSA_ERR_UNSUPPORTED;
        }
    }
    if (cudaGetLastError() != cudaSuccess) return TSA_ERR_CUDA;
    if (a.D == 64) return a.bf16 ? launch_grad_kernels<64, true>(a) : launch_grad_kernels<64, false>(a);
    if (a.D == 128) return a.bf16 ? launch_grad_kernels<128, true>(a) : launch_grad_kernels<128, false>(a);
    return TSA_ERR_UNSUPPORTED;
}

}  // namespace tsa
