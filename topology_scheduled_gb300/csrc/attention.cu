// attention.cu -- scheduled causal attention forward on tcgen05 tensor cores (sm_103a).
//
// Method ("Add topology-derived sparse attention kernel" (triton-lang/kernels#22), Summary,
// and the port note on the PR's mirror page): for every 64-token query block visit only the
// key blocks of its CSR row, keep a running row maximum and denominator, rescale by
// exp(m_prev - m_new), and mask keys after the query token inside the diagonal block.
//
// GB300 design (not the pages' Triton kernel):
//  * Tile.  One CTA computes 128 query rows: query blocks 2p and 2p+1 of one lane, because
//    tcgen05 runs at full rate at M = 128.  It walks the sorted union of the two CSR rows; a
//    key block in only one row is masked for the other half (each half is two whole warps).
//  * Warp roles (192 threads).  Warp 4 produces: one thread TMA-loads Q once and the K and V
//    tiles of each visited block into two-stage rings of their own (128-byte swizzle), polling
//    both rings so that neither stream waits behind the other.  Warp 5 issues the MMAs from
//    one thread: S = Q K^T (M128 N64 K=D, both operands in shared memory) into one of two TMEM
//    S buffers, and O += P V (M128 N=D K64) with P read from TMEM.  Warps 0-3 run the online
//    softmax, one row per thread: tcgen05.ld of the S row, exp2 with the scale folded in, the
//    new P written back over the S buffer in the input dtype with tcgen05.st.
//  * Pipeline.  The MMA warp issues QK(u+1) before PV(u), so the tensor core computes the next
//    scores while the softmax warps work on the current ones.  K and V have rings of their
//    own: a K stage is refilled as soon as its QK is done, so the next key tile is already
//    resident when the MMA warp reaches it.  Hand-offs are mbarriers: k_full/k_empty and
//    v_full/v_empty (producer <-> MMA), s_full (MMA -> softmax, also carries the end of the
//    row union), p_full (softmax -> MMA), o_done (PV completion, for rescaling and the
//    epilogue).
//  * Lazy rescale.  O and the denominator are rescaled only when a row's maximum grows by more
//    than 2^30 (bf16) or 2^15 (f16); the final O / l uses the same stale maximum, so the result
//    is unchanged.  The decision is per row but TMEM loads/stores are warp-collective, so a
//    warp rescales when any of its rows must (factor 1 for the others).
//  * Epilogue.  O / l rounded to the input dtype, staged in the Q tile, TMA-stored per block;
//    optionally the row's log-sum-exp (m + log l), which the backward pass recomputes P from.
//  * Partial last block (S not a multiple of 64).  Its key rows past S are read but never
//    weigh: the block is visited only as the diagonal block of the last row, where the causal
//    mask already drops keys after the query token.  Its query rows past S are computed and
//    dropped: the block's output is written row by row for the rows that exist.
//  * Two CTAs share an SM, so one CTA's softmax also overlaps the other's MMAs.
// Every mbarrier wait is bounded; on a timeout the CTA records TSA_ERR_TIMEOUT, drains its
// in-flight copies and MMAs (bounded), frees TMEM and returns.
#include <climits>

#include "tsa_device.cuh"
#include "tsa_internal.h"

namespace tsa {
namespace {

constexpr int kRows = 128;            // query rows per CTA (two 64-token query blocks)
constexpr int kBlock = 64;            // tokens per key / query block
constexpr int kKStages = 2;           // K ring depth
constexpr int kVStages = 2;           // V ring depth
constexpr int kThreads = 192;         // 4 softmax warps + producer warp + MMA warp
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
// Lazy-rescale threshold (log2 units): O and the denominator are rescaled only when a row's
// maximum grows past the one they are scaled to by more than this, so p stays at most 2^30
// (bf16: far inside its range and the fp32 accumulators') or 2^15 (f16: below its largest
// finite value, 65504).  Rescales cost a wait for the running PV product and a pass over O in
// TMEM; keys drawn around distinct cluster means made a small threshold (2^8) rescale often.
template <bool kBF16>
__device__ __forceinline__ constexpr float rescale_log2() { return kBF16 ? 30.0f : 15.0f; }

template <int D>
struct AttnSmem {
    static constexpr int kD = D;
    static constexpr int kChunks = D / 64;            // 64-element (128 B) column chunks
    static constexpr int kQBytes = kRows * D * 2;     // Q tile, later the O staging tile
    static constexpr int kKVBytes = kBlock * D * 2;   // one K or V tile
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;                // kKStages tiles
    static constexpr int kOffV = kOffK + kKStages * kKVBytes;    // kVStages tiles
    static constexpr int kOffMeta = kOffV + kVStages * kKVBytes;
    static constexpr int kMetaBytes = 256;
    static constexpr int kTmemCols = 256;  // S0 | S1 | O (P_b aliases the first 32 of S_b)
    static constexpr int kOCol = 128;
};

__device__ __forceinline__ uint32_t s_col(int b) { return b ? 64u : 0u; }

// Meta area layout (byte offsets from kOffMeta).
// Union entries in flight: the producer writes entry v once QK(v - kKStages) is done, while the
// softmax warps may still be about to read entry v - kKStages - 1, so the ring holds more.
constexpr int kMetaRing = 8;
static_assert(kMetaRing >= kKStages + 2, "meta ring shorter than the K ring's lead");
constexpr int kBarQ = 0;
constexpr int kBarKFull = 8;                          // kKStages x 8
constexpr int kBarKEmpty = kBarKFull + 8 * kKStages;  // kKStages x 8
constexpr int kBarVFull = kBarKEmpty + 8 * kKStages;  // kVStages x 8
constexpr int kBarVEmpty = kBarVFull + 8 * kVStages;  // kVStages x 8
constexpr int kBarSFull = kBarVEmpty + 8 * kVStages;  // 2 x 8
constexpr int kBarPFull = kBarSFull + 16;             // 2 x 8
constexpr int kBarODone = kBarPFull + 16;
constexpr int kBarFin = kBarODone + 8;
constexpr int kTmemSlot = kBarFin + 8;
constexpr int kAbortFlag = kTmemSlot + 4;
constexpr int kMetaJ = kAbortFlag + 4;                // kMetaRing x 4
constexpr int kMetaF = kMetaJ + 4 * kMetaRing;        // kMetaRing x 4
static_assert(kMetaF + 4 * kMetaRing <= 256, "meta area");

// Walks the union of two sorted CSR rows (query blocks qa and qa+1), checking the row
// contract on the way.  Used by the producer thread.
//
// With 128-token blocks (coarse) the CTA's two 64-token query blocks are one CSR row p = qa/2,
// and each 128-token key block j of it is visited as the 64-token blocks 2j and 2j+1: both
// for both halves when j < p; on the diagonal (j == p) block 2p for both halves (the token
// mask then holds keys to k <= q in the first half, the second half sees all of it) and block
// 2p+1 for the second half only.  The allowed key set of every token is the 128-block one.
struct RowUnion {
    const int32_t *col;
    int ia, ia_end, ib, ib_end;
    int last_a, last_b, qa, qb;
    bool bad;
    bool coarse, has_b;
    int nb64, pend, pend_flags;

    __device__ void init(const int32_t *row_ptr, const int32_t *col_idx, int qa_, bool has_b_,
                         bool coarse_ = false, int nb64_ = 0) {
        col = col_idx;
        qa = qa_;
        qb = qa_ + 1;
        bad = false;
        coarse = coarse_;
        has_b = has_b_;
        nb64 = nb64_;
        pend = -1;
        pend_flags = 0;
        if (coarse) {
            const int p = qa >> 1;
            ia = row_ptr[p];
            ia_end = row_ptr[p + 1];
            if (ia_end - ia < 0 || ia_end - ia > p + 1) { bad = true; ia_end = ia; }
            ib = ib_end = 0;
            last_a = last_b = -1;
            return;
        }
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

    // 64-token entries of a 128-token CSR row (see above).
    __device__ int next_coarse(int &flags) {
        if (pend >= 0) {
            const int j = pend;
            flags = pend_flags;
            pend = -1;
            return j;
        }
        const int p = qa >> 1;
        if (ia >= ia_end) { flags = 0; return -1; }
        const int j = __ldg(col + ia);
        if (j <= last_a || j > p) { bad = true; ia_end = ia; flags = 0; return -1; }
        last_a = j;
        ++ia;
        const int rows = has_b ? 3 : 1;
        flags = rows;
        const int fb = j < p ? rows : (rows & 2);
        if (2 * j + 1 < nb64 && fb != 0) {
            pend = 2 * j + 1;
            pend_flags = fb;
        }
        return 2 * j;
    }
};

// 32-token blocks: the CTA's 128 rows are query blocks r0 .. r0+3 (r0 = 2 qa), and each 64-token
// key block k of the union of their CSR rows carries one bit per (query quarter r, key half h):
// bit 2r + h when row r0 + r holds 32-token key block 2k + h.  Rows are checked as above.
struct RowUnion32 {
    const int32_t *col;
    int pos[4], end[4], last[4];
    int r0;
    bool bad;

    __device__ void init(const int32_t *row_ptr, const int32_t *col_idx, int r0_, int nrows) {
        col = col_idx;
        r0 = r0_;
        bad = false;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            last[r] = -1;
            pos[r] = end[r] = 0;
            if (r < nrows) {
                pos[r] = row_ptr[r0 + r];
                end[r] = row_ptr[r0 + r + 1];
                if (end[r] - pos[r] < 0 || end[r] - pos[r] > r0 + r + 1) { bad = true; end[r] = pos[r]; }
            }
        }
    }

    __device__ int head(int r) {
        if (pos[r] >= end[r]) return INT_MAX;
        const int x = __ldg(col + pos[r]);
        if (x <= last[r] || x > r0 + r) { bad = true; end[r] = pos[r]; return INT_MAX; }
        return x;
    }

    __device__ int next(int &flags) {
        int h[4], j = INT_MAX;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            h[r] = head(r);
            j = h[r] < j ? h[r] : j;
        }
        flags = 0;
        if (j == INT_MAX) return -1;
        const int k = j >> 1;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (h[r] == 2 * k + hh) {
                    flags |= 1 << (2 * r + hh);
                    last[r] = h[r];
                    ++pos[r];
                    h[r] = head(r);
                }
            }
        }
        return k;
    }
};

// The producer's walk for the CSR's block size kGran (0: 64, 1: 128, 2: 32 tokens): entries are
// 64-token key blocks with their membership bits -- with 32-token blocks bit 2r + h per (query
// quarter r, key half h), otherwise bit h per 64-row query half h (the whole 64-key step).
template <int kGran>
struct EntryWalk {
    RowUnion u;
    RowUnion32 u32;

    __device__ void init(const int32_t *row_ptr, const int32_t *col_idx, int qa, bool has_b, int nb64, int S) {
        if constexpr (kGran == 2) {
            const int nb32 = (S + 31) / 32;
            const int r0 = 2 * qa;
            u32.init(row_ptr, col_idx, r0, nb32 - r0 < 4 ? nb32 - r0 : 4);
        } else {
            u.init(row_ptr, col_idx, qa, has_b, kGran == 1, nb64);
        }
    }

    __device__ int next(int &flags) {
        if constexpr (kGran == 2) return u32.next(flags);
        else if constexpr (kGran == 1) return u.next_coarse(flags);
        else return u.next(flags);
    }

    __device__ bool bad() const {
        if constexpr (kGran == 2) return u32.bad;
        else return u.bad;
    }
};

// Two floats rounded to the 16-bit input dtype, packed (first in the low half); `sum` gets
// the rounded values.
template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float a, float b, float &sum) {
    if constexpr (kBF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        sum += __low2float(h) + __high2float(h);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __half2 h = __floats2half2_rn(a, b);
        sum += __low2float(h) + __high2float(h);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

// The layout leaves at least 512 bytes for aligning the dynamic shared-memory base to 1024
// (the kernel checks the actual alignment and reports kDevSmemAlign if it does not fit).
static_assert(AttnSmem<128>::kOffMeta + AttnSmem<128>::kMetaBytes + 512 <= kAttnSmemBytes<128>(), "smem");
static_assert(AttnSmem<64>::kOffMeta + AttnSmem<64>::kMetaBytes + 512 <= kAttnSmemBytes<64>(), "smem");

template <int D, bool kBF16, int kGran>
__global__ void __launch_bounds__(kThreads, 2)
scheduled_attention_kernel(const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmO,
                           const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
                           uint16_t *__restrict__ O, float *__restrict__ lse_out, int nb, int S,
                           float scale_log2, DeviceFlags flags) {
    constexpr bool kFine = kGran == 2;  // 32-token blocks: masks per (query quarter, key half)
    using L = AttnSmem<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];

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
    const uint32_t meta = base + L::kOffMeta;
    volatile int *meta_j = reinterpret_cast<volatile int *>(smem + L::kOffMeta + kMetaJ);
    volatile int *meta_f = reinterpret_cast<volatile int *>(smem + L::kOffMeta + kMetaF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMeta + kAbortFlag);
    const uint32_t bar_q = meta + kBarQ, bar_o_done = meta + kBarODone, bar_fin = meta + kBarFin;
#define BAR_K_FULL(s) (meta + kBarKFull + 8u * (uint32_t)(s))
#define BAR_K_EMPTY(s) (meta + kBarKEmpty + 8u * (uint32_t)(s))
#define BAR_V_FULL(s) (meta + kBarVFull + 8u * (uint32_t)(s))
#define BAR_V_EMPTY(s) (meta + kBarVEmpty + 8u * (uint32_t)(s))
#define BAR_S_FULL(b) (meta + kBarSFull + 8u * (uint32_t)(b))
#define BAR_P_FULL(b) (meta + kBarPFull + 8u * (uint32_t)(b))

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane_id = blockIdx.y;                  // attention lane (batch * head)
    const int npairs = (nb + 1) >> 1;
    const int pair = npairs - 1 - (int)blockIdx.x;   // longest rows first
    const int qa = 2 * pair;
    const bool has_b = qa + 1 < nb;
    const int row0 = lane_id * S;                    // first row of this lane in [L*S, D]

    // The first global reads are issued together and waited for at the barrier below: whether
    // the launch already gave up elsewhere (one thread reads the flag, so the whole CTA takes
    // the same branch), and the producer's CSR rows.
    const bool gave_up = tid == 0 && *reinterpret_cast<volatile unsigned *>(flags.abort_epoch) == flags.epoch;
    EntryWalk<kGran> ruk, ruv;  // the producer's walks of the row union, one per stream
    if (tid == kProducerWarp * 32) {
        ruk.init(row_ptr, col_idx, qa, has_b, nb, S);
        ruv.init(row_ptr, col_idx, qa, has_b, nb, S);
    }

    if (tid == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(BAR_K_FULL(s), 1);
            mbar_init(BAR_K_EMPTY(s), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(BAR_V_FULL(s), 1);
            mbar_init(BAR_V_EMPTY(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(BAR_S_FULL(b), 1);
            mbar_init(BAR_P_FULL(b), kRows);
        }
        mbar_init(bar_o_done, 1);
        mbar_init(bar_fin, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(meta + kTmemSlot, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    const bool leave = __syncthreads_or(gave_up);
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kOffMeta + kTmemSlot);
    if (leave) {  // nothing was issued yet: give the columns back and go
        if (warp == kMmaWarp) tmem_dealloc(tmem, L::kTmemCols);
        return;
    }

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer (TMA)
        // One thread, two independent streams: the K tile of union entry v goes into K stage
        // v % kKStages as soon as QK(v - kKStages) has freed it, the V tile into V stage
        // v % kVStages as soon as PV(v - kVStages) has; the thread polls both rings, so a K
        // load never waits behind a V stage.
        if ((tid & 31) == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmO);
            mbar_arrive_expect_tx(bar_q, L::kQBytes);
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c)
                tma_load_2d(sQ + c * 16384, &tmQ, c * 64, row0 + qa * kBlock, bar_q);
            bool ok = true, k_done = false, v_done = false;
            int kv = 0, vv = 0;  // next union entry of each stream
            unsigned long long t_idle = 0;
            for (uint32_t it = 0; !(k_done && v_done); ++it) {
                bool progress = false;
                if (!k_done && (kv < kKStages ||
                                mbar_try_wait(BAR_K_EMPTY(kv % kKStages), (uint32_t)((kv / kKStages) - 1) & 1u))) {
                    const int s = kv % kKStages;
                    int f = 0;
                    const int j = ruk.next(f);
                    meta_j[kv % kMetaRing] = j;
                    meta_f[kv % kMetaRing] = f;
                    if (j < 0) {
                        mbar_arrive(BAR_K_FULL(s));  // the end marker travels with the K ring
                        k_done = true;
                    } else {
                        mbar_arrive_expect_tx(BAR_K_FULL(s), L::kKVBytes);
#pragma unroll
                        for (int c = 0; c < L::kChunks; ++c)
                            tma_load_2d(sK0 + s * L::kKVBytes + c * 8192, &tmK, c * 64, row0 + j * kBlock,
                                        BAR_K_FULL(s));
                        ++kv;
                    }
                    progress = true;
                }
                if (!v_done && (vv < kVStages ||
                                mbar_try_wait(BAR_V_EMPTY(vv % kVStages), (uint32_t)((vv / kVStages) - 1) & 1u))) {
                    const int s = vv % kVStages;
                    int f = 0;
                    const int j = ruv.next(f);
                    if (j < 0) {
                        v_done = true;
                    } else {
                        mbar_arrive_expect_tx(BAR_V_FULL(s), L::kKVBytes);
#pragma unroll
                        for (int c = 0; c < L::kChunks; ++c)
                            tma_load_2d(sV0 + s * L::kKVBytes + c * 8192, &tmV, c * 64, row0 + j * kBlock,
                                        BAR_V_FULL(s));
                        ++vv;
                    }
                    progress = true;
                }
                // bounded: give up after kWaitTimeoutNs without progress, or when the launch did
                if (progress) {
                    t_idle = 0;
                } else if ((it & 63u) == 0u) {
                    const unsigned long long now = globaltimer();
                    if (t_idle == 0) t_idle = now;
                    if (now - t_idle > kWaitTimeoutNs ||
                        *reinterpret_cast<volatile unsigned *>(flags.abort_epoch) == flags.epoch) {
                        ok = false;
                        break;
                    }
                }
            }
            if (ruk.bad()) raise_status(flags, kDevBadSchedule);
            if (!ok) {
                // Drain: wait (bounded) for every load issued into the rings.
                *abort_flag = 1;
                (void)mbar_wait_timed(bar_q, 0);
                for (int w = kv - kKStages; w < kv; ++w)
                    if (w >= 0) (void)mbar_wait_timed(BAR_K_FULL(w % kKStages), (w / kKStages) & 1);
                for (int w = vv - kVStages; w < vv; ++w)
                    if (w >= 0) (void)mbar_wait_timed(BAR_V_FULL(w % kVStages), (w / kVStages) & 1);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if ((tid & 31) == 0) {
            constexpr uint32_t kIdescQK = idesc_f16(kBF16, 128, 64, false);
            constexpr uint32_t kIdescPV = idesc_f16(kBF16, 128, D, true);
            bool ok = mbar_wait(bar_q, 0, flags);
            int u = 0;
            bool have = false;  // entry u exists and QK(u) was issued
            // QK(u): S_{u%2} = Q K_u^T; frees K stage u % kKStages when done
#define ISSUE_QK(uu)                                                                              \
    do {                                                                                          \
        const int s_ = (uu) % kKStages;                                                           \
        tc_fence_after();                                                                         \
        _Pragma("unroll") for (int kk = 0; kk < D / 16; ++kk) {                                   \
            const uint64_t a_ = sdesc_sw128(sQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);    \
            const uint64_t b_ =                                                                   \
                sdesc_sw128(sK0 + s_ * L::kKVBytes + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024); \
            tc_mma_ss(tmem + s_col((uu) & 1), a_, b_, kIdescQK, kk > 0 ? 1u : 0u);               \
        }                                                                                         \
        tc_commit(BAR_S_FULL((uu) & 1));                                                          \
        tc_commit(BAR_K_EMPTY(s_));                                                               \
    } while (0)
            // The end of the row union is passed to the softmax warps as an s_full arrival
            // without scores (they read the end marker from the meta ring).
            if (ok) {
                ok = mbar_wait(BAR_K_FULL(0), 0, flags);
                if (ok) {
                    // test hook: the launch's first CTA withholds its first scores (no product,
                    // no arrival), so its softmax warps' bounded wait runs out
                    const bool withhold = flags.inject == 1u && blockIdx.x == 0 && blockIdx.y == 0;
                    if (meta_j[0] >= 0 && !withhold) {
                        ISSUE_QK(0);
                        have = true;
                    } else if (meta_j[0] < 0) {
                        mbar_arrive(BAR_S_FULL(0));
                    }
                }
            }
            while (ok && have) {
                // next scores first, so they overlap the softmax of u
                bool next = false;
                const int s1 = (u + 1) % kKStages;
                ok = mbar_wait(BAR_K_FULL(s1), ((u + 1) / kKStages) & 1, flags);
                if (!ok) break;
                if (meta_j[(u + 1) % kMetaRing] >= 0) {
                    ISSUE_QK(u + 1);
                    next = true;
                } else {
                    mbar_arrive(BAR_S_FULL((u + 1) & 1));
                }
                // O += P_u V_u once the softmax has written P_u and V_u has landed
                ok = mbar_wait(BAR_P_FULL(u & 1), (u >> 1) & 1, flags);
                if (!ok) break;
                const int s = u % kVStages;
                ok = mbar_wait(BAR_V_FULL(s), (u / kVStages) & 1, flags);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t b = sdesc_sw128(sV0 + s * L::kKVBytes + kk * 2048, 8192, 1024);
                    tc_mma_ts(tmem + L::kOCol, tmem + s_col(u & 1) + kk * 8, b, kIdescPV,
                              (u > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(BAR_V_EMPTY(s));
                tc_commit(bar_o_done);
                have = next;
                ++u;
            }
#undef ISSUE_QK
            if (!ok) *abort_flag = 1;
            // all tensor-core work of this CTA has completed once this arrives
            tc_commit(bar_fin);
            (void)mbar_wait_timed(bar_fin, 0);
        }
    } else {
        // ------------------------------------------------------------ softmax (warps 0-3)
        const int half = tid >> 6;               // 0: block qa, 1: block qa+1
        const int my_block = qa + half;
        const bool row_exists = half == 0 || has_b;
        const uint32_t t_lane = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lane quarter
        float m_used = -INFINITY;                // maximum the accumulators are scaled to (log2)
        float l_sum = 0.f;                       // running denominator
        bool ok = true;
        int u = 0;
        for (;; ++u) {
            if (!mbar_wait(BAR_S_FULL(u & 1), (u >> 1) & 1, flags)) { ok = false; break; }
            const int j = meta_j[u % kMetaRing];
            const int fl = meta_f[u % kMetaRing];
            if (j < 0) break;
            tc_fence_after();
            // key halves this warp's 32 rows hold (both, with 64- or 128-token blocks)
            const int fq = kFine ? (fl >> (2 * warp)) & 3 : ((fl >> half) & 1) * 3;
            const bool in_row = row_exists && fq != 0;  // warp-uniform
            const uint32_t s_addr = tmem + t_lane + s_col(u & 1);
            uint32_t pw[32];
            __syncwarp();
            if (in_row) {
                uint32_t sr[2][32];
                tmem_ld32x2(s_addr, sr[0], sr[1]);
                float x[64];  // raw scores q.k
#pragma unroll
                for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(sr[c >> 5][c & 31]);
                if constexpr (kFine) {
                    if (fq != 3) {  // a 32-token key half this row does not hold
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            if (!((fq >> (c >> 5)) & 1)) x[c] = -INFINITY;
                    }
                    if (j >= qa) {  // near the diagonal: keys after the query token are masked
                        const int lim = (qa - j) * kBlock + tid;  // key 64j + c > query 64qa + tid
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            if (c > lim) x[c] = -INFINITY;
                    }
                } else if (j == my_block) {  // diagonal block: keys after the query token are masked
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (c > (tid & 63)) x[c] = -INFINITY;
                }
                float m21[22];
#pragma unroll
                for (int t = 0; t < 21; ++t) m21[t] = max3f(x[3 * t], x[3 * t + 1], x[3 * t + 2]);
                m21[21] = x[63];
                const float m7a = max3f(max3f(m21[0], m21[1], m21[2]), max3f(m21[3], m21[4], m21[5]),
                                        max3f(m21[6], m21[7], m21[8]));
                const float m7b = max3f(max3f(m21[9], m21[10], m21[11]), max3f(m21[12], m21[13], m21[14]),
                                        max3f(m21[15], m21[16], m21[17]));
                const float mx = max3f(m7a, m7b, max3f(m21[18], m21[19], fmaxf(m21[20], m21[21]))) * scale_log2;
                const bool grow = mx > m_used + rescale_log2<kBF16>();
                if (__any_sync(0xffffffffu, grow)) {
                    const float alpha = !grow ? 1.f : (m_used == -INFINITY ? 0.f : ex2_approx(m_used - mx));
                    if (u > 0) {
                        // O must be quiescent: PV(u-1) has completed
                        const bool done = mbar_wait(bar_o_done, (u - 1) & 1, flags);
                        if (__any_sync(0xffffffffu, !done)) { ok = false; break; }
                        tc_fence_after();
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
                // p = 2^(x * scale * log2(e) - m): one packed FMA per pair, exp2 on the MUFU
                const uint64_t cc = f2_pack(scale_log2, scale_log2);
                const uint64_t nm = f2_pack(-m_used, -m_used);
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    float e0, e1;
                    f2_unpack(f2_fma(f2_pack(x[2 * t], x[2 * t + 1]), cc, nm), e0, e1);
                    const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
                    if constexpr (kBF16) {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                        pw[t] = *reinterpret_cast<const uint32_t *>(&h);
                    } else {
                        const __half2 h = __floats2half2_rn(p0, p1);
                        pw[t] = *reinterpret_cast<const uint32_t *>(&h);
                    }
                    // The denominator sums the rounded P that the PV product uses, so a row
                    // dominated by one key normalizes exactly.
                    add_half<kBF16, false>(ls[(t & 1) * 2], pw[t]);
                    add_half<kBF16, true>(ls[(t & 1) * 2 + 1], pw[t]);
                }
                l_sum += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            } else {
#pragma unroll
                for (int t = 0; t < 32; ++t) pw[t] = 0u;
            }
            __syncwarp();
            tmem_st32(s_addr, pw);  // P_u over the first 32 columns of S_u
            tc_fence_before();
            mbar_arrive(BAR_P_FULL(u & 1));
        }
        if (!ok) *abort_flag = 1;
        // ---- epilogue: O / l in the input dtype, staged in the Q tile, TMA-stored per block
        bool o_valid = false;
        if (ok && u > 0) {
            o_valid = mbar_wait(bar_o_done, (u - 1) & 1, flags);
            if (!o_valid) *abort_flag = 1;
        }
        // one decision for all softmax warps (the section below has a barrier of its own)
        if (!named_barrier_or(1, kRows, *abort_flag != 0)) {
            tc_fence_after();
            const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
            // A partial last query block (S not a multiple of 64) is not TMA-stored -- its box
            // would run into the next lane's rows -- but written row by row from registers.
            const int tok = qa * kBlock + tid;  // this thread's token (rows of both halves)
            const bool partial = (my_block + 1) * kBlock > S;
            const bool tok_ok = row_exists && tok < S;
            // log-sum-exp of the scaled scores in natural-log units, for the backward pass
            if (lse_out && tok_ok)
                lse_out[row0 + tok] = l_sum > 0.f ? (m_used + log2f(l_sum)) * 0.6931471805599453f : -INFINITY;
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
                        float unused = 0.f;
                        uint32_t w[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            w[t] = pack2<kBF16>(__uint_as_float(o[q * 8 + 2 * t]) * inv,
                                                __uint_as_float(o[q * 8 + 2 * t + 1]) * inv, unused);
                        const uint32_t chunk16 = (uint32_t)(h * 4 + q);
                        st_shared_v4(o_row + ((chunk16 ^ sw) << 4), w[0], w[1], w[2], w[3]);
                        if (partial && tok_ok)
                            *reinterpret_cast<uint4 *>(O + ((size_t)row0 + tok) * L::kD + c * 64 + chunk16 * 8) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            fence_proxy_async_smem();
            named_barrier(1, kRows);
            if (tid == 0) {
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c) {
                    if ((qa + 1) * kBlock <= S) tma_store_2d(&tmO, c * 64, row0 + qa * kBlock, sQ + c * 16384);
                    if (has_b && (qa + 2) * kBlock <= S)
                        tma_store_2d(&tmO, c * 64, row0 + (qa + 1) * kBlock, sQ + c * 16384 + 8192);
                }
                tma_store_commit();
                tma_store_wait_read();
            }
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
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int D, bool kBF16, int kGran>
tsa_status launch_one(const AttnLaunch &a) {
    auto kern = scheduled_attention_kernel<D, kBF16, kGran>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmemBytes<D>()) !=
        cudaSuccess)
        return TSA_ERR_CUDA;
    const int npairs = (a.nb + 1) / 2;
    dim3 grid((unsigned)npairs, (unsigned)a.lanes);
    kern<<<grid, kThreads, kAttnSmemBytes<D>(), a.stream>>>(*a.tmQ, *a.tmK, *a.tmV, *a.tmO, a.row_ptr,
                                                            a.col_idx, a.O, a.lse, a.nb, a.S,
                                                            a.scale_log2, a.flags);
    return cudaGetLastError() == cudaSuccess ? TSA_OK : TSA_ERR_CUDA;
}

template <int kGran>
tsa_status launch_gran(const AttnLaunch &a) {
    if (a.D == 64) return a.bf16 ? launch_one<64, true, kGran>(a) : launch_one<64, false, kGran>(a);
    if (a.D == 128) return a.bf16 ? launch_one<128, true, kGran>(a) : launch_one<128, false, kGran>(a);
    return TSA_ERR_UNSUPPORTED;
}

}  // namespace

tsa_status launch_scheduled_attention(const AttnLaunch &a) {
    return a.gran == 2 ? launch_gran<2>(a) : a.gran == 1 ? launch_gran<1>(a) : launch_gran<0>(a);
}

}  // namespace tsa
