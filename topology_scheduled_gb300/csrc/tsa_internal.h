// tsa_internal.h -- declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "tsa.h"
#include "tsa_device.cuh"

namespace tsa {

// Dynamic shared memory of the attention kernel.  The D = 128 figure is the largest size at
// which two CTAs fit on one SM (2 x (115712 + 1024 reserved) = 228 KB); it covers the
// 114816 bytes of tiles and barriers plus 896 bytes of alignment slack.
template <int D>
__host__ __device__ constexpr int kAttnSmemBytes() {
    return D == 128 ? 115712 : 66688;
}

struct AttnLaunch {
    const CUtensorMap *tmQ, *tmK, *tmV, *tmO;
    const int32_t *row_ptr, *col_idx;
    uint16_t *O;  // the output (a partial last block is written with plain stores)
    float *lse;  // optional: natural-log log-sum-exp of the scaled scores per query row
    int nb, S, D, lanes;  // nb: 64-token blocks
    bool bf16;
    int gran;  // token block of the CSR: 0 for 64, 1 for 128, 2 for 32
    float scale_log2;
    DeviceFlags flags;
    cudaStream_t stream;
};

tsa_status launch_scheduled_attention(const AttnLaunch &a);

// Byte offsets of the backward pass's workspace regions (each 256-byte aligned).
struct BwdWorkspace {
    size_t delta, lse_pad, vlen, cnt, col_ptr, bitmap, bitmap_bytes, row_idx, pairs, vlen_in, rp64, ci64, total;
};
// nb: 64-token blocks; nb_in: rows of a 128-token CSR to expand first (0: the CSR is 64-token)
BwdWorkspace backward_workspace_layout(int64_t lanes, int64_t S, int64_t nb, int64_t nnz_cap, int64_t nb_in);

// Largest number of query blocks the backward pass accepts (its column bitmap is nb^2 bits).
constexpr int64_t kMaxBackwardBlocks = 8192;

struct BwdLaunch {
    // 128-row boxes (tiles resident in a CTA) and 64-row boxes (streamed blocks, stores)
    const CUtensorMap *tmQ128, *tmdO128;
    const CUtensorMap *tmQ64, *tmdO64, *tmK64, *tmV64, *tmdQ64, *tmdK64, *tmdV64;
    const uint16_t *O, *dO;
    uint16_t *dQ, *dK, *dV;  // for the row stores of a partial last block
    const float *lse;
    const int32_t *row_ptr, *col_idx;
    int64_t nnz_cap;
    // Delta and the log-sum-exp per lane over nb * 64 rows (rows past S: 0 and -inf), so a
    // partial last block is read like any other
    float *delta, *lse_pad;
    int *vlen, *cnt, *col_ptr;
    unsigned *bitmap;
    size_t bitmap_bytes;
    int32_t *row_idx;
    int *pairs;  // dK/dV key-block pairs, 2 per pair (-1: none)
    int nb_in;   // > 0: row_ptr/col_idx are a CSR of nb_in 128-token blocks, expanded into
    int *vlen_in;  // rp64/ci64 (64-token blocks, capacity nnz_cap) before anything else
    int32_t *rp64, *ci64;
    int nb, S, D, lanes;
    bool bf16;
    float scale;
    DeviceFlags flags;
    cudaStream_t stream;
};

tsa_status launch_attention_backward(const BwdLaunch &a);

// Largest number of blocks the schedule builder accepts.
constexpr int64_t kMaxScheduleBlocks = 4096;
constexpr int64_t kMaxScheduleDim = 1024;

// Byte offsets of the builder's workspace regions (each 256-byte aligned).
struct ScheduleWorkspace {
    size_t part, cent, cent32, bnd, comp, vb_d, vb_u, mst_d, mst_u, mst_v, counters, sal, cnt, perm, sal_rank, gbar, total;
};
ScheduleWorkspace schedule_workspace_layout(int64_t lanes, int64_t nb, int64_t D);

struct ScheduleLaunch {
    const uint16_t *K;
    bool bf16;
    int64_t lanes, S, D, block, nb;
    int64_t sink, local_radius, topk;
    bool content_ties;  // break ties by centroid content instead of block index
    int32_t *row_ptr, *col_idx;
    int64_t col_cap;
    double *salience_sq;  // may be null
    uint8_t *workspace;
    DeviceFlags flags;
    cudaStream_t stream;
};

tsa_status launch_build_schedule(const ScheduleLaunch &a);
// The two halves of launch_build_schedule, for a lane-sharded build: per-lane block sums of K
// (part: lanes x nb x D doubles), and the schedule from block sums of all lanes.
tsa_status launch_block_sums(const ScheduleLaunch &a, double *part);
tsa_status launch_schedule_from_sums(const ScheduleLaunch &a, const double *sums);
tsa_status launch_dense_causal_csr(int64_t nb, int32_t *row_ptr, int32_t *col_idx,
                                   cudaStream_t stream);
// Segment schedule: fixed segments of seg_tokens (> 0), or the listed starts (seg_tokens 0).
tsa_status launch_segment_csr(int64_t S, int64_t block, int64_t seg_tokens, const int32_t *starts,
                              int64_t n_starts, int32_t *row_ptr, int32_t *col_idx, int64_t col_cap,
                              const DeviceFlags &flags, cudaStream_t stream);

}  // namespace tsa
