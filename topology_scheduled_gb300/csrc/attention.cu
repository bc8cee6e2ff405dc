// attention.cu -- scheduled causal attention forward on tcgen05 tensor cores (sm_103a).
//
// Method ("Add topology-derived sparse attention kernel" (triton-lang/kernels#22), Summary,
// and the port note on the PR's mirror page): for every 64-token query block visit only the
// key blocks of its CSR row, keep a running row maximum and denominator, rescale by
// exp(m_prev - m_new), and mask keys after the query token inside the diagonal block.
//
// GB300 design (not the pages' Triton kernel):
//  * One CTA computes a 128-row tile made of the query blocks 2p and 2p+1 of one lane, because
//    tcgen05 reaches full rate at M = 128.  It walks the sorted union of the two CSR rows; a
//    key block that is in only one row is masked for the other half (both halves are
//    warp-uniform, so that half skips its softmax).
//  * TMA loads Q once and K/V tiles per visited block (128-byte swizzle, two stages).  One
//    thread issues S = Q K^T (M128 N64) into TMEM; 128 threads own one row each, read S with
//    tcgen05.ld, do the online softmax in fp32 (exp2 with the scale folded in), write P in the
//    input dtype to shared memory, and one thread issues O += P V (M128 N=D) into TMEM.
//  * Rescaling is lazy: O and the denominator are rescaled only when a row's maximum grows by
//    more than 2^8; the final O / l uses the same stale maximum, so the result is unchanged.
//  * Epilogue: O / l rounded to the input dtype, staged in shared memory, TMA-stored per
//    64-row block.
//  * Two CTAs share an SM (D = 128; three for D = 64), so one CTA's softmax overlaps the
//    other's MMAs.
#include <climits>

#include "tsa_device.cuh"
#include "tsa_internal.h"

namespace tsa {
namespace {

constexpr int kRows = 128;           // query rows per CTA (two 64-token query blocks)
constexpr int kBlock = 64;           // tokens per key / query block
constexpr float kRescaleLog2 = 8.0f; // lazy-rescale threshold (log2 units)

template <int D>
struct AttnSmem {
    static constexpr int kChunks = D / 64;                  // 64-element (128 B) column chunks
    static constexpr int kQBytes = kRows * D * 2;           // Q tile, later the O staging tile
    static constexpr int kKVBytes = kBlock * D * 2;         // one K or V tile
    static constexpr int kPBytes = kRows * kBlock * 2;      // P tile
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;           // 2 stages
    static constexpr int kOffV = kOffK + 2 * kKVBytes;      // 2 stages
    static constexpr int kOffP = kOffV + 2 * kKVBytes;
    static constexpr int kOffMeta = kOffP + kPBytes;
    static constexpr int kMetaBytes = 128;
    static constexpr int kTmemCols = D == 128 ? 256 : 128;  // S (64 cols) + O (D cols)
    static constexpr int kSCol = 0;
    static constexpr int kOCol = 64;
};

// Meta area (byte offsets from kOffMeta).
constexpr int kBarQ = 0, kBarKV = 8 /* 2 x 8 */, kBarMma = 24, kBarFin = 32;
constexpr int kTmemSlot = 40, kMetaJ = 48 /* 2 x 4 */, kMetaF = 56 /* 2 x 4 */;

// Walks the union of two sorted CSR rows (query blocks qa and qa+1), checking the row
// contract on the way.  Used by one thread.
struct RowUnion {
    const int32_t *col;
    int ia, ia_end, ib, ib_end;
    int last_a, last_b, qa, qb;
    bool bad;

    __device__ void init(const int32_t *row_ptr, const int32_t *col_idx, int qa_, bool has_b) {
        col = col_idx;
        qa = qa_;
        qb = qa_ + 1;
        bad = false;
        ia = row_ptr[qa];
        ia_end = row_ptr[qa + 1];
        if (ia_end - ia < 0 || ia_end - ia > qa + 1) { bad = true; ia_end = ia; }
        if (has_b) {
            ib = row_ptr[qb];
            ib_end = row_ptr[qb + 1];
            if (ib_end - ib < 0 || ib_end - ib > qb + 1) { bad = true; ib_end = ib; }
        } else {
            ib = ib_end = 0;
        }
        last_a = last_b = -1;
    }

    // Next key block of the union and its membership bits (1: row qa, 2: row qb); -1 at end.
    __device__ int next(int &flags) {
        int ja = INT_MAX, jb = INT_MAX;
        if (ia < ia_end) {
            ja = __ldg(col + ia);
            if (ja <= last_a || ja > qa) { bad = true; ia_end = ia; ja = INT_MAX; }
        }
        if (ib < ib_end) {
            jb = __ldg(col + ib);
            if (jb <= last_b || jb > qb) { bad = true; ib_end = ib; jb = INT_MAX; }
        }
        if (ja == INT_MAX && jb == INT_MAX) { flags = 0; return -1; }
        const int j = ja < jb ? ja : jb;
        flags = (ja == j ? 1 : 0) | (jb == j ? 2 : 0);
        if (ja == j) { last_a = ja; ++ia; }
        if (jb == j) { last_b = jb; ++ib; }
        return j;
    }
};

template <int D, bool kBF16>
__global__ void __launch_bounds__(kRows, 1)
scheduled_attention_kernel(const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmO,
                           const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
                           int nb, int S, float scale_log2, DeviceFlags flags) {
    using L = AttnSmem<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];

    // A launch that already gave up elsewhere: leave before taking any resource (one thread
    // reads the flag so that the whole CTA takes the same branch).
    if (__syncthreads_or(threadIdx.x == 0 &&
                         *reinterpret_cast<volatile unsigned *>(flags.abort_epoch) == flags.epoch))
        return;

    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    if (base - raw_base + L::kOffMeta + L::kMetaBytes > (uint32_t)kAttnSmemBytes<D>()) {
        if (threadIdx.x == 0) raise_status(flags, kDevSmemAlign);
        return;
    }
    uint8_t *smem = smem_raw + (base - raw_base);
    const uint32_t sQ = base + L::kOffQ;
    const uint32_t sK0 = base + L::kOffK;
    const uint32_t sV0 = base + L::kOffV;
    const uint32_t sP = base + L::kOffP;
    const uint32_t meta = base + L::kOffMeta;
    const uint32_t bar_q = meta + kBarQ, bar_mma = meta + kBarMma, bar_fin = meta + kBarFin;
    volatile int *meta_j = reinterpret_cast<volatile int *>(smem + L::kOffMeta + kMetaJ);
    volatile int *meta_f = reinterpret_cast<volatile int *>(smem + L::kOffMeta + kMetaF);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane_id = blockIdx.y;                  // attention lane (batch * head)
    const int npairs = (nb + 1) >> 1;
    const int pair = npairs - 1 - (int)blockIdx.x;   // longest rows first
    const int qa = 2 * pair;
    const bool has_b = qa + 1 < nb;
    const int half = tid >> 6;                       // 0: block qa, 1: block qa+1
    const int r_in = tid & 63;                       // token within the query block
    const int my_block = qa + half;
    const bool row_exists = half == 0 || has_b;
    const int row0 = lane_id * S;                    // first row of this lane in [L*S, D]

    if (tid == 0) {
        mbar_init(bar_q, 1);
        mbar_init(meta + kBarKV, 1);
        mbar_init(meta + kBarKV + 8, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_fin, 1);
        fence_barrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
    }
    if (warp == 0) {
        tmem_alloc(meta + kTmemSlot, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kOffMeta + kTmemSlot);
    const uint32_t t_lane = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lane quarter

    // ---- producer state (thread 0): CSR row union and TMA issue
    RowUnion ru;
    int produced = 0;
    auto produce = [&](int v) {
        const int s = v & 1;
        int f = 0;
        const int j = ru.next(f);
        meta_j[s] = j;
        meta_f[s] = f;
        const uint32_t bar = meta + kBarKV + 8 * s;
        if (j < 0) {
            mbar_arrive(bar);
        } else {
            mbar_arrive_expect_tx(bar, 2 * L::kKVBytes);
            const int y = row0 + j * kBlock;
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c) {
                tma_load_2d(sK0 + s * L::kKVBytes + c * 8192, &tmK, c * 64, y, bar);
                tma_load_2d(sV0 + s * L::kKVBytes + c * 8192, &tmV, c * 64, y, bar);
            }
        }
        produced = v + 1;
    };
    if (tid == 0) {
        ru.init(row_ptr, col_idx, qa, has_b);
        mbar_arrive_expect_tx(bar_q, L::kQBytes);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) tma_load_2d(sQ + c * 16384, &tmQ, c * 64, row0 + qa * kBlock, bar_q);
        produce(0);
        produce(1);
    }

    constexpr uint32_t kIdescQK = idesc_f16(kBF16, 128, 64, false);
    constexpr uint32_t kIdescPV = idesc_f16(kBF16, 128, D, true);

    float m_used = -INFINITY;  // maximum the accumulators are scaled to (log2 units)
    float l_sum = 0.f;         // running denominator
    bool o_valid = false;
    bool aborted = false;
    uint32_t mma_phase = 0;
    bool ok = mbar_wait(bar_q, 0, flags);
    int u = 0;
    for (;; ++u) {
        const int s = u & 1;
        ok = mbar_wait(meta + kBarKV + 8 * s, (u >> 1) & 1, flags) && ok;
        if (__syncthreads_or(!ok)) { aborted = true; break; }
        const int j = meta_j[s];
        const int fl = meta_f[s];
        if (j < 0) break;

        // S = Q K_j^T  (M 128, N 64, K D)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t a = sdesc_sw128(sQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                const uint64_t b = sdesc_sw128(sK0 + s * L::kKVBytes + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
                tc_mma_ss(tmem + L::kSCol, a, b, kIdescQK, kk > 0 ? 1u : 0u);
            }
            tc_commit(bar_mma);
        }
        ok = mbar_wait(bar_mma, mma_phase, flags) && ok;
        mma_phase ^= 1u;
        tc_fence_after();

        // ---- online softmax on this thread's row
        const bool in_row = row_exists && ((fl >> half) & 1);  // warp-uniform
        const uint32_t p_row = sP + tid * 128;
        const uint32_t sw = (uint32_t)(tid & 7);
        if (in_row) {
            uint32_t sr[2][32];
            __syncwarp();  // the waits above may leave the warp diverged; tcgen05.ld is collective
            tmem_ld32(tmem + t_lane + L::kSCol, sr[0]);
            tmem_ld32(tmem + t_lane + L::kSCol + 32, sr[1]);
            const bool diag = (j == my_block);
            float x[64];
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                float v = __uint_as_float(sr[c >> 5][c & 31]) * scale_log2;
                if (diag && c > r_in) v = -INFINITY;
                x[c] = v;
                mx = fmaxf(mx, v);
            }
            // The rescale decision is per row, but tcgen05.ld/st are warp-collective: the whole
            // warp rescales when any of its rows must, with factor 1 for the other rows.
            const bool grow = mx > m_used + kRescaleLog2;
            if (__any_sync(0xffffffffu, grow)) {
                const float alpha = !grow ? 1.f : (m_used == -INFINITY ? 0.f : ex2_approx(m_used - mx));
                if (o_valid) {
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(tmem + t_lane + L::kOCol + c, o);
#pragma unroll
                        for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
                        tmem_st32(tmem + t_lane + L::kOCol + c, o);
                    }
                }
                if (grow) {
                    l_sum *= alpha;
                    m_used = mx;
                }
            }
            float lsum_blk = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float p0 = ex2_approx(x[q * 8 + 2 * t] - m_used);
                    const float p1 = ex2_approx(x[q * 8 + 2 * t + 1] - m_used);
                    if constexpr (kBF16) {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                        lsum_blk += __low2float(h) + __high2float(h);
                        w[t] = *reinterpret_cast<const uint32_t *>(&h);
                    } else {
                        const __half2 h = __floats2half2_rn(p0, p1);
                        lsum_blk += __low2float(h) + __high2float(h);
                        w[t] = *reinterpret_cast<const uint32_t *>(&h);
                    }
                }
                st_shared_v4(p_row + (((uint32_t)q ^ sw) << 4), w[0], w[1], w[2], w[3]);
            }
            l_sum += lsum_blk;
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) st_shared_v4(p_row + (q << 4), 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) { aborted = true; break; }

        // O += P V_j  (M 128, N D, K 64); V is MN-major (d contiguous)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t a = sdesc_sw128(sP + kk * 32, 16, 1024);
                const uint64_t b = sdesc_sw128(sV0 + s * L::kKVBytes + kk * 2048, 8192, 1024);
                tc_mma_ss(tmem + L::kOCol, a, b, kIdescPV, (u > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(bar_mma);
        }
        ok = mbar_wait(bar_mma, mma_phase, flags) && ok;
        mma_phase ^= 1u;
        tc_fence_after();
        o_valid = true;
        if (tid == 0) produce(u + 2);
    }

    if (tid == 0 && ru.bad) raise_status(flags, kDevBadSchedule);

    if (!aborted) {
        // ---- epilogue: O / l in the input dtype, staged in the Q tile, TMA store per block
        const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
        const uint32_t sw = (uint32_t)(tid & 7);
        __syncwarp();
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
            const uint32_t o_row = sQ + c * 16384 + tid * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t o[32];
                if (o_valid) {
                    tmem_ld32(tmem + t_lane + L::kOCol + c * 64 + h * 32, o);
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) o[t] = 0u;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float a = __uint_as_float(o[q * 8 + 2 * t]) * inv;
                        const float b = __uint_as_float(o[q * 8 + 2 * t + 1]) * inv;
                        if constexpr (kBF16) {
                            const __nv_bfloat162 hv = __floats2bfloat162_rn(a, b);
                            w[t] = *reinterpret_cast<const uint32_t *>(&hv);
                        } else {
                            const __half2 hv = __floats2half2_rn(a, b);
                            w[t] = *reinterpret_cast<const uint32_t *>(&hv);
                        }
                    }
                    const uint32_t chunk16 = (uint32_t)(h * 4 + q);
                    st_shared_v4(o_row + ((chunk16 ^ sw) << 4), w[0], w[1], w[2], w[3]);
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c) {
                tma_store_2d(&tmO, c * 64, row0 + qa * kBlock, sQ + c * 16384);
                if (has_b) tma_store_2d(&tmO, c * 64, row0 + (qa + 1) * kBlock, sQ + c * 16384 + 8192);
            }
            tma_store_commit();
            tma_store_wait_all();
        }
    } else if (tid == 0) {
        // Gave up: record it, then let in-flight tensor-core work and TMA loads drain (bounded)
        // before the shared memory and TMEM are released.
        raise_status(flags, kDevTimeout);
        atomicExch(flags.abort_epoch, flags.epoch);
        tc_commit(bar_fin);
        (void)mbar_wait_timed(bar_fin, 0);
        (void)mbar_wait_timed(bar_q, 0);
        for (int v = u; v < produced; ++v) (void)mbar_wait_timed(meta + kBarKV + 8 * (v & 1), (v >> 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int D, bool kBF16>
tsa_status launch_one(const AttnLaunch &a) {
    auto kern = scheduled_attention_kernel<D, kBF16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmemBytes<D>()) !=
        cudaSuccess)
        return TSA_ERR_CUDA;
    const int npairs = (a.nb + 1) / 2;
    dim3 grid((unsigned)npairs, (unsigned)a.lanes);
    kern<<<grid, kRows, kAttnSmemBytes<D>(), a.stream>>>(*a.tmQ, *a.tmK, *a.tmV, *a.tmO, a.row_ptr,
                                                         a.col_idx, a.nb, a.S, a.scale_log2,
                                                         a.flags);
    return cudaGetLastError() == cudaSuccess ? TSA_OK : TSA_ERR_CUDA;
}

}  // namespace

tsa_status launch_scheduled_attention(const AttnLaunch &a) {
    if (a.D == 64) return a.bf16 ? launch_one<64, true>(a) : launch_one<64, false>(a);
    if (a.D == 128) return a.bf16 ? launch_one<128, true>(a) : launch_one<128, false>(a);
    return TSA_ERR_UNSUPPORTED;
}

}  // namespace tsa
