// segment.cu -- block schedules of segment masks ("Add topology-derived sparse attention
// kernel" mirror page, the later commit on a forget gate's exact zeros feeding the merged CSR
// kernel: segment boundaries as a zero-error CSR schedule; 288 and 160 visited blocks under
// fixed 512- and 256-token segments at S 4096, block 64).
//
// Segments begin at token 0 and at every listed start.  Query token q may attend to key k
// iff s(q) <= k <= q, s(q) the last start <= q.  Since s is non-decreasing, the first token
// of query block i has the earliest start, so row i is the contiguous run of key blocks
// [s(block * i) / block, i].  Two launches: one CTA validates the starts, counts every row
// and scans the counts into row_ptr; then one warp per row writes its run into col_idx.
#include "tsa_internal.h"

namespace tsa {
namespace {

constexpr int kSegThreads = 1024;

// Segment start of token t: fixed length, or the last of starts[0, n) that is <= t.
__device__ __forceinline__ int64_t segment_start(int64_t t, int64_t seg_tokens,
                                                 const int32_t *__restrict__ starts, int64_t n) {
    if (seg_tokens > 0) return (t / seg_tokens) * seg_tokens;
    int64_t lo = 0, hi = n;  // number of starts <= t
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)starts[mid] <= t) lo = mid + 1;
        else hi = mid;
    }
    return lo > 0 ? (int64_t)starts[lo - 1] : 0;
}

__device__ __forceinline__ int64_t row_len(int64_t i, int64_t block, int64_t seg_tokens,
                                           const int32_t *starts, int64_t n) {
    return i - segment_start(i * block, seg_tokens, starts, n) / block + 1;
}

__global__ void __launch_bounds__(kSegThreads)
segment_rows(int64_t S, int64_t block, int64_t seg_tokens, const int32_t *__restrict__ starts,
             int64_t n_starts, int32_t *__restrict__ row_ptr, int64_t col_cap, DeviceFlags flags) {
    __shared__ unsigned long long first_bad;
    __shared__ long long warp_tot[kSegThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int64_t nb = S / block;
    if (tid == 0) first_bad = (unsigned long long)n_starts;
    __syncthreads();
    // the usable starts are the longest prefix that is strictly ascending inside [0, S)
    for (int64_t k = tid; k < n_starts; k += blockDim.x) {
        const int32_t v = starts[k];
        if (v < 0 || (int64_t)v >= S || (k > 0 && v <= starts[k - 1]))
            atomicMin(&first_bad, (unsigned long long)k);
    }
    __syncthreads();
    const int64_t n = (int64_t)first_bad;
    if (tid == 0 && n < n_starts) raise_status(flags, kDevBadSchedule);
    // each thread a contiguous run of rows; block-wide exclusive scan of the run totals
    const int64_t per = (nb + blockDim.x - 1) / blockDim.x;
    const int64_t beg = min(nb, tid * per), end = min(nb, beg + per);
    long long run = 0;
    for (int64_t i = beg; i < end; ++i) run += row_len(i, block, seg_tokens, starts, n);
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
    // rows that do not fit in col_cap are cut (the status word reports it)
    long long at = (warp > 0 ? warp_tot[warp - 1] : 0) + incl - run;
    for (int64_t i = beg; i < end; ++i) {
        row_ptr[i] = (int32_t)min(at, (long long)col_cap);
        at += row_len(i, block, seg_tokens, starts, n);
    }
    if (tid == 0) {
        const long long total = warp_tot[nwarps - 1];
        row_ptr[nb] = (int32_t)min(total, (long long)col_cap);
        if (total > col_cap) raise_status(flags, kDevCapacity);
    }
}

// Row i holds the `len` blocks ending at the diagonal: i - len + 1, ..., i.
__global__ void segment_fill(int64_t nb, const int32_t *__restrict__ row_ptr,
                             int32_t *__restrict__ col_idx) {
    const int lane = threadIdx.x & 31;
    const int64_t gwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t i = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); i < nb; i += gwarps) {
        const int32_t b = row_ptr[i], len = row_ptr[i + 1] - b;
        const int32_t lo = (int32_t)i - len + 1;
        for (int32_t k = lane; k < len; k += 32) col_idx[b + k] = lo + k;
    }
}

}  // namespace

tsa_status launch_segment_csr(int64_t S, int64_t block, int64_t seg_tokens, const int32_t *starts,
                              int64_t n_starts, int32_t *row_ptr, int32_t *col_idx, int64_t col_cap,
                              const DeviceFlags &flags, cudaStream_t stream) {
    const int64_t nb = S / block;
    segment_rows<<<1, kSegThreads, 0, stream>>>(S, block, seg_tokens, starts, n_starts, row_ptr, col_cap,
                                                flags);
    const int64_t ctas = (nb + 7) / 8;
    segment_fill<<<(unsigned)(ctas < 152 * 8 ? ctas : 152 * 8), 256, 0, stream>>>(nb, row_ptr, col_idx);
    return cudaGetLastError() == cudaSuccess ? TSA_OK : TSA_ERR_CUDA;
}

}  // namespace tsa
