// api.cu -- the C ABI declared in include/tsa.h: host-side validation, tensor-map encoding
// and kernel launches.  No call allocates or frees memory.
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>
#include <vector>

#include "tsa_internal.h"

namespace tsa {
namespace {

__device__ unsigned g_status;       // sticky device-side error bits
__device__ unsigned g_abort_epoch;  // epoch of the last launch that gave up

constexpr int kMaxDevices = 64;
struct DeviceState {
    bool ready = false;
    unsigned *status = nullptr;
    unsigned *abort_epoch = nullptr;
};
DeviceState g_devices[kMaxDevices];
std::mutex g_mutex;
std::atomic<unsigned> g_epoch{0};

tsa_status current_device(int *dev) {
    // Launch errors are read back with cudaGetLastError after each launch; an error an earlier
    // call on this thread left pending (another library's, e.g. on an autograd worker thread)
    // is cleared first so that it is not reported as this call's.
    (void)cudaGetLastError();
    // cudaSetDevice binds the device's primary context to this thread: a thread that has not
    // touched the runtime yet (a worker thread) has no current context, and encoding a tensor
    // map needs one.
    if (cudaGetDevice(dev) != cudaSuccess || cudaSetDevice(*dev) != cudaSuccess) {
        cudaGetLastError();
        return TSA_ERR_CUDA;
    }
    return (*dev >= 0 && *dev < kMaxDevices) ? TSA_OK : TSA_ERR_UNSUPPORTED;
}

// Device addresses of the status words (looked up once per device) and a fresh epoch.
// Process-wide test hook for the failure path (tsa_debug_set_wait_injection).
std::atomic<unsigned> g_wait_injection{0u};

tsa_status device_flags(int dev, DeviceFlags *f) {
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        DeviceState &d = g_devices[dev];
        if (!d.ready) {
            if (cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_status) != cudaSuccess ||
                cudaGetSymbolAddress(reinterpret_cast<void **>(&d.abort_epoch), g_abort_epoch) !=
                    cudaSuccess) {
                cudaGetLastError();
                return TSA_ERR_CUDA;
            }
            d.ready = true;
        }
        f->status = d.status;
        f->abort_epoch = d.abort_epoch;
    }
    unsigned e;
    do {
        e = ++g_epoch;
    } while (e == 0u || e == ~0u);
    f->epoch = e;
    f->inject = g_wait_injection.load();
    return TSA_OK;
}

tsa_status check_device_ptr(const void *p, int dev) {
    if (p == nullptr) return TSA_ERR_INVALID_ARGUMENT;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return TSA_ERR_NOT_DEVICE_POINTER;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
        return TSA_ERR_NOT_DEVICE_POINTER;
    if (at.device != dev) return TSA_ERR_DEVICE_MISMATCH;
    return TSA_OK;
}

#define TSA_TRY(expr)                       \
    do {                                    \
        const tsa_status s_ = (expr);       \
        if (s_ != TSA_OK) return s_;        \
    } while (0)

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            p = nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// Row-major [rows, cols] 16-bit matrix; boxes of 64 columns (128 B, 128-byte swizzle) x box_rows.
bool encode_2d(CUtensorMap *map, const void *ptr, bool bf16, uint64_t rows, uint64_t cols,
               uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
              const_cast<void *>(ptr), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

tsa_status launch_attention_checked(const void *Q, const void *K, const void *V, const int32_t *row_ptr,
                                    const int32_t *col_idx, void *O, float *lse, bool bf16, int64_t lanes,
                                    int64_t S, int64_t D, int64_t block, float scale, cudaStream_t stream,
                                    int dev);

int64_t max_nnz_bound(int64_t nb, int64_t sink, int64_t r, int64_t topk) {
    // sum_{i < nb} min(i + 1, per), per = sink + r + 1 + topk (saturating at nb)
    int64_t per = nb;
    if (sink < nb && r < nb && topk < nb) per = sink + r + 1 + topk;
    if (per >= nb) return nb * (nb + 1) / 2;
    return per * (per + 1) / 2 + (nb - per) * per;
}

}  // namespace
}  // namespace tsa

using namespace tsa;

extern "C" {

const char *tsa_status_string(tsa_status s) {
    switch (s) {
        case TSA_OK: return "TSA_OK";
        case TSA_ERR_INVALID_ARGUMENT: return "TSA_ERR_INVALID_ARGUMENT";
        case TSA_ERR_UNSUPPORTED: return "TSA_ERR_UNSUPPORTED";
        case TSA_ERR_NOT_DEVICE_POINTER: return "TSA_ERR_NOT_DEVICE_POINTER";
        case TSA_ERR_DEVICE_MISMATCH: return "TSA_ERR_DEVICE_MISMATCH";
        case TSA_ERR_CAPACITY: return "TSA_ERR_CAPACITY";
        case TSA_ERR_CUDA: return "TSA_ERR_CUDA";
        case TSA_ERR_TIMEOUT: return "TSA_ERR_TIMEOUT";
        case TSA_ERR_BAD_SCHEDULE: return "TSA_ERR_BAD_SCHEDULE";
        case TSA_ERR_DEVICE: return "TSA_ERR_DEVICE";
    }
    return "TSA_ERR_UNKNOWN";
}

int64_t tsa_schedule_max_nnz(int64_t S, int64_t block, int64_t sink, int64_t local_radius,
                             int64_t topk) {
    if (S <= 0 || block <= 0 || sink < 0 || local_radius < 0 || topk < 0) return -1;
    return max_nnz_bound((S + block - 1) / block, sink, local_radius, topk);
}

size_t tsa_build_schedule_workspace_bytes(int64_t lanes, int64_t S, int64_t D, int64_t block) {
    if (lanes <= 0 || S <= 0 || D <= 0 || block <= 0) return 0;
    const int64_t nb = (S + block - 1) / block;
    if (nb > kMaxScheduleBlocks || D > kMaxScheduleDim) return 0;
    // the block sums alone are 8 * lanes * nb * D bytes: refuse sizes whose total would wrap
    if (lanes > INT64_MAX / S / D || lanes > INT64_MAX / 16 / nb / D) return 0;
    return schedule_workspace_layout(lanes, nb, D).total;
}

tsa_status tsa_build_schedule(const void *K, tsa_dtype dtype, int64_t lanes, int64_t S, int64_t D,
                              int64_t block, int64_t sink, int64_t local_radius, int64_t topk,
                              int32_t *row_ptr, int32_t *col_idx, int64_t col_cap,
                              double *salience_sq, void *workspace, size_t workspace_bytes,
                              tsa_stream_t stream) {
    return tsa_build_schedule_ex(K, dtype, lanes, S, D, block, sink, local_radius, topk, TSA_TIE_INDEX,
                                 row_ptr, col_idx, col_cap, salience_sq, workspace, workspace_bytes,
                                 stream);
}

tsa_status tsa_build_schedule_ex(const void *K, tsa_dtype dtype, int64_t lanes, int64_t S, int64_t D,
                                 int64_t block, int64_t sink, int64_t local_radius, int64_t topk,
                                 tsa_tie_break tie_break, int32_t *row_ptr, int32_t *col_idx,
                                 int64_t col_cap, double *salience_sq, void *workspace,
                                 size_t workspace_bytes, tsa_stream_t stream) {
    if (!K || !row_ptr || !col_idx || !workspace) return TSA_ERR_INVALID_ARGUMENT;
    if (tie_break != TSA_TIE_INDEX && tie_break != TSA_TIE_CONTENT) return TSA_ERR_INVALID_ARGUMENT;
    if (dtype != TSA_F16 && dtype != TSA_BF16) return TSA_ERR_INVALID_ARGUMENT;
    if (lanes <= 0 || S <= 0 || D <= 0 || block <= 0) return TSA_ERR_INVALID_ARGUMENT;
    if (sink < 0 || local_radius < 0 || topk < 0) return TSA_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(K) & 1u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return TSA_ERR_INVALID_ARGUMENT;
    const int64_t nb = (S + block - 1) / block;  // a partial last block counts
    if (nb > kMaxScheduleBlocks || D > kMaxScheduleDim) return TSA_ERR_UNSUPPORTED;
    if (lanes > INT64_MAX / S / D || lanes > INT64_MAX / 16 / nb / D) return TSA_ERR_INVALID_ARGUMENT;
    const int64_t need = max_nnz_bound(nb, sink, local_radius, topk);
    if (col_cap < need) return TSA_ERR_CAPACITY;
    const ScheduleWorkspace ws = schedule_workspace_layout(lanes, nb, D);
    if (workspace_bytes < ws.total) return TSA_ERR_CAPACITY;
    int dev;
    TSA_TRY(current_device(&dev));
    TSA_TRY(check_device_ptr(K, dev));
    TSA_TRY(check_device_ptr(row_ptr, dev));
    TSA_TRY(check_device_ptr(col_idx, dev));
    TSA_TRY(check_device_ptr(workspace, dev));
    if (salience_sq) TSA_TRY(check_device_ptr(salience_sq, dev));
    ScheduleLaunch a;
    a.K = static_cast<const uint16_t *>(K);
    a.bf16 = dtype == TSA_BF16;
    a.lanes = lanes;
    a.S = S;
    a.D = D;
    a.block = block;
    a.nb = nb;
    a.sink = sink < nb ? sink : nb;
    a.local_radius = local_radius < nb ? local_radius : nb;
    a.topk = topk < nb ? topk : nb;
    a.content_ties = tie_break == TSA_TIE_CONTENT;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.col_cap = col_cap;
    a.salience_sq = salience_sq;
    a.workspace = static_cast<uint8_t *>(workspace);
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    TSA_TRY(device_flags(dev, &a.flags));
    return launch_build_schedule(a);
}

tsa_status tsa_block_sums(const void *K, tsa_dtype dtype, int64_t lanes, int64_t S, int64_t D,
                          int64_t block, double *part, tsa_stream_t stream) {
    if (!K || !part) return TSA_ERR_INVALID_ARGUMENT;
    if (dtype != TSA_F16 && dtype != TSA_BF16) return TSA_ERR_INVALID_ARGUMENT;
    if (lanes <= 0 || S <= 0 || D <= 0 || block <= 0) return TSA_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(K) & 1u) || (reinterpret_cast<uintptr_t>(part) & 7u))
        return TSA_ERR_INVALID_ARGUMENT;
    const int64_t nb = (S + block - 1) / block;
    if (nb > kMaxScheduleBlocks || D > kMaxScheduleDim) return TSA_ERR_UNSUPPORTED;
    if (lanes > INT64_MAX / S / D) return TSA_ERR_INVALID_ARGUMENT;
    if (overlaps(part, (size_t)(lanes * nb * D) * 8, K, (size_t)(lanes * S * D) * 2)) return TSA_ERR_INVALID_ARGUMENT;
    int dev;
    TSA_TRY(current_device(&dev));
    TSA_TRY(check_device_ptr(K, dev));
    TSA_TRY(check_device_ptr(part, dev));
    ScheduleLaunch a{};
    a.K = static_cast<const uint16_t *>(K);
    a.bf16 = dtype == TSA_BF16;
    a.lanes = lanes;
    a.S = S;
    a.D = D;
    a.block = block;
    a.nb = nb;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    TSA_TRY(device_flags(dev, &a.flags));
    return launch_block_sums(a, part);
}

tsa_status tsa_build_schedule_from_sums(const double *part, int64_t lanes, int64_t S, int64_t D,
                                        int64_t block, int64_t sink, int64_t local_radius,
                                        int64_t topk, tsa_tie_break tie_break, int32_t *row_ptr,
                                        int32_t *col_idx, int64_t col_cap, double *salience_sq,
                                        void *workspace, size_t workspace_bytes,
                                        tsa_stream_t stream) {
    if (!part || !row_ptr || !col_idx || !workspace) return TSA_ERR_INVALID_ARGUMENT;
    if (tie_break != TSA_TIE_INDEX && tie_break != TSA_TIE_CONTENT) return TSA_ERR_INVALID_ARGUMENT;
    if (lanes <= 0 || S <= 0 || D <= 0 || block <= 0) return TSA_ERR_INVALID_ARGUMENT;
    if (sink < 0 || local_radius < 0 || topk < 0) return TSA_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(part) & 7u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return TSA_ERR_INVALID_ARGUMENT;
    const int64_t nb = (S + block - 1) / block;
    if (nb > kMaxScheduleBlocks || D > kMaxScheduleDim) return TSA_ERR_UNSUPPORTED;
    if (lanes > INT64_MAX / nb / D / 8) return TSA_ERR_INVALID_ARGUMENT;
    const int64_t need = max_nnz_bound(nb, sink, local_radius, topk);
    if (col_cap < need) return TSA_ERR_CAPACITY;
    const ScheduleWorkspace ws = schedule_workspace_layout(lanes, nb, D);
    if (workspace_bytes < ws.total) return TSA_ERR_CAPACITY;
    if (overlaps(part, (size_t)(lanes * nb * D) * 8, workspace, ws.total)) return TSA_ERR_INVALID_ARGUMENT;
    int dev;
    TSA_TRY(current_device(&dev));
    TSA_TRY(check_device_ptr(part, dev));
    TSA_TRY(check_device_ptr(row_ptr, dev));
    TSA_TRY(check_device_ptr(col_idx, dev));
    TSA_TRY(check_device_ptr(workspace, dev));
    if (salience_sq) TSA_TRY(check_device_ptr(salience_sq, dev));
    ScheduleLaunch a{};
    a.K = nullptr;
    a.lanes = lanes;
    a.S = S;
    a.D = D;
    a.block = block;
    a.nb = nb;
    a.sink = sink < nb ? sink : nb;
    a.local_radius = local_radius < nb ? local_radius : nb;
    a.topk = topk < nb ? topk : nb;
    a.content_ties = tie_break == TSA_TIE_CONTENT;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.col_cap = col_cap;
    a.salience_sq = salience_sq;
    a.workspace = static_cast<uint8_t *>(workspace);
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    TSA_TRY(device_flags(dev, &a.flags));
    return launch_schedule_from_sums(a, part);
}

tsa_status tsa_dense_causal_csr(int64_t S, int64_t block, int32_t *row_ptr, int32_t *col_idx,
                                int64_t col_cap, tsa_stream_t stream) {
    if (!row_ptr || !col_idx) return TSA_ERR_INVALID_ARGUMENT;
    if (S <= 0 || block <= 0) return TSA_ERR_INVALID_ARGUMENT;
    const int64_t nb = (S + block - 1) / block;
    if (nb > 65534) return TSA_ERR_INVALID_ARGUMENT;  // nb(nb+1)/2 must stay below 2^31
    if (col_cap < nb * (nb + 1) / 2) return TSA_ERR_CAPACITY;
    int dev;
    TSA_TRY(current_device(&dev));
    TSA_TRY(check_device_ptr(row_ptr, dev));
    TSA_TRY(check_device_ptr(col_idx, dev));
    return launch_dense_causal_csr(nb, row_ptr, col_idx, reinterpret_cast<cudaStream_t>(stream));
}

int64_t tsa_fixed_segment_nnz(int64_t S, int64_t block, int64_t segment_tokens) {
    if (S <= 0 || block <= 0 || S % block != 0 || segment_tokens <= 0) return -1;
    const int64_t nb = S / block;
    if (nb > 65534) return -1;
    int64_t total = 0;  // row i runs from the block of its segment start to i
    for (int64_t i = 0; i < nb; ++i) total += i - ((i * block) / segment_tokens) * segment_tokens / block + 1;
    return total;
}

tsa_status tsa_fixed_segment_csr(int64_t S, int64_t block, int64_t segment_tokens, int32_t *row_ptr,
                                 int32_t *col_idx, int64_t col_cap, tsa_stream_t stream) {
    if (!row_ptr || !col_idx) return TSA_ERR_INVALID_ARGUMENT;
    const int64_t need = tsa_fixed_segment_nnz(S, block, segment_tokens);
    if (need < 0) return TSA_ERR_INVALID_ARGUMENT;
    if (col_cap < need) return TSA_ERR_CAPACITY;
    int dev;
    TSA_TRY(current_device(&dev));
    TSA_TRY(check_device_ptr(row_ptr, dev));
    TSA_TRY(check_device_ptr(col_idx, dev));
    DeviceFlags flags;
    TSA_TRY(device_flags(dev, &flags));
    return launch_segment_csr(S, block, segment_tokens, nullptr, 0, row_ptr, col_idx, col_cap, flags,
                              reinterpret_cast<cudaStream_t>(stream));
}

tsa_status tsa_segment_csr(int64_t S, int64_t block, const int32_t *starts, int64_t n_starts,
                           int32_t *row_ptr, int32_t *col_idx, int64_t col_cap, tsa_stream_t stream) {
    if (!row_ptr || !col_idx || (n_starts > 0 && !starts) || n_starts < 0) return TSA_ERR_INVALID_ARGUMENT;
    if (S <= 0 || block <= 0 || S % block != 0 || col_cap < 1) return TSA_ERR_INVALID_ARGUMENT;
    const int64_t nb = S / block;
    if (nb > 65534 || S > INT_MAX) return TSA_ERR_INVALID_ARGUMENT;
    int dev;
    TSA_TRY(current_device(&dev));
    if (n_starts > 0) TSA_TRY(check_device_ptr(starts, dev));
    TSA_TRY(check_device_ptr(row_ptr, dev));
    TSA_TRY(check_device_ptr(col_idx, dev));
    DeviceFlags flags;
    TSA_TRY(device_flags(dev, &flags));
    return launch_segment_csr(S, block, 0, n_starts > 0 ? starts : nullptr, n_starts, row_ptr, col_idx,
                              col_cap, flags, reinterpret_cast<cudaStream_t>(stream));
}

tsa_status tsa_scheduled_attention(const void *Q, const void *K, const void *V,
                                   const int32_t *row_ptr, const int32_t *col_idx, void *O,
                                   tsa_dtype dtype, int64_t B, int64_t H, int64_t S, int64_t D,
                                   int64_t block, float scale, tsa_stream_t stream) {
    return tsa_scheduled_attention_fwd(Q, K, V, row_ptr, col_idx, O, nullptr, dtype, B, H, S, D, block,
                                       scale, stream);
}

tsa_status tsa_scheduled_attention_fwd(const void *Q, const void *K, const void *V,
                                       const int32_t *row_ptr, const int32_t *col_idx, void *O,
                                       float *lse, tsa_dtype dtype, int64_t B, int64_t H, int64_t S,
                                       int64_t D, int64_t block, float scale, tsa_stream_t stream) {
    if (!Q || !K || !V || !row_ptr || !col_idx || !O) return TSA_ERR_INVALID_ARGUMENT;
    if (dtype != TSA_F16 && dtype != TSA_BF16) return TSA_ERR_INVALID_ARGUMENT;
    if (B <= 0 || H <= 0 || S <= 0 || D <= 0 || block <= 0) return TSA_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(scale)) return TSA_ERR_INVALID_ARGUMENT;
    if ((block != 32 && block != 64 && block != 128) || (D != 64 && D != 128)) return TSA_ERR_UNSUPPORTED;
    // S need not be a multiple of the block: the last query / key block may be partial
    if (B > 65535 || H > 65535 || B * H > 65535) return TSA_ERR_UNSUPPORTED;
    const int64_t lanes = B * H;
    if (lanes * S >= (int64_t)INT_MAX) return TSA_ERR_UNSUPPORTED;
    for (const void *p : {Q, K, V, static_cast<const void *>(O)})
        if (reinterpret_cast<uintptr_t>(p) & 15u) return TSA_ERR_INVALID_ARGUMENT;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return TSA_ERR_INVALID_ARGUMENT;
    const size_t bytes = (size_t)(lanes * S * D) * 2;
    if (overlaps(O, bytes, Q, bytes) || overlaps(O, bytes, K, bytes) || overlaps(O, bytes, V, bytes))
        return TSA_ERR_INVALID_ARGUMENT;
    if (lse) {
        const size_t lb = (size_t)(lanes * S) * 4;
        if (overlaps(lse, lb, Q, bytes) || overlaps(lse, lb, K, bytes) || overlaps(lse, lb, V, bytes) ||
            overlaps(lse, lb, O, bytes))
            return TSA_ERR_INVALID_ARGUMENT;
    }
    int dev;
    TSA_TRY(current_device(&dev));
    for (const void *p : {Q, K, V, static_cast<const void *>(O), static_cast<const void *>(row_ptr),
                          static_cast<const void *>(col_idx)})
        TSA_TRY(check_device_ptr(p, dev));
    if (lse) TSA_TRY(check_device_ptr(lse, dev));
    return launch_attention_checked(Q, K, V, row_ptr, col_idx, O, lse, dtype == TSA_BF16, lanes, S, D, block,
                                    scale, reinterpret_cast<cudaStream_t>(stream), dev);
}

}  // extern "C"

namespace tsa {
namespace {

constexpr int kHostStepDevices = 64;
// The attention launch once the arguments have been checked.
tsa_status launch_attention_checked(const void *Q, const void *K, const void *V, const int32_t *row_ptr,
                                    const int32_t *col_idx, void *O, float *lse, bool bf16, int64_t lanes,
                                    int64_t S, int64_t D, int64_t block, float scale, cudaStream_t stream,
                                    int dev) {
    const uint64_t rows = (uint64_t)(lanes * S);
    CUtensorMap tmQ, tmK, tmV, tmO;
    if (!encode_2d(&tmQ, Q, bf16, rows, (uint64_t)D, 128) || !encode_2d(&tmK, K, bf16, rows, (uint64_t)D, 64) ||
        !encode_2d(&tmV, V, bf16, rows, (uint64_t)D, 64) || !encode_2d(&tmO, O, bf16, rows, (uint64_t)D, 64))
        return TSA_ERR_CUDA;
    AttnLaunch a;
    a.tmQ = &tmQ;
    a.tmK = &tmK;
    a.tmV = &tmV;
    a.tmO = &tmO;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.O = static_cast<uint16_t *>(O);
    a.lse = lse;
    a.nb = (int)((S + 63) / 64);  // the kernel works in 64-token blocks
    a.gran = block == 128 ? 1 : block == 32 ? 2 : 0;
    a.S = (int)S;
    a.D = (int)D;
    a.lanes = (int)lanes;
    a.bf16 = bf16;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);  // scale * log2(e)
    a.stream = stream;
    TSA_TRY(device_flags(dev, &a.flags));
    return launch_scheduled_attention(a);
}
// Copy streams and events of tsa_topology_attention_host, created on the first call on each
// device and kept for the life of the process.  A call holds its device's lock while it
// enqueues, so calls from several host threads take turns; an event recorded again by a later
// call is safe, because each stream wait binds to the event's most recent record at the time
// the wait is enqueued.
struct HostStepResources {
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    std::vector<cudaEvent_t> events;
};
HostStepResources g_host_step[kHostStepDevices];
std::mutex g_host_step_mutex[kHostStepDevices];

// The streams of device `dev` (current) and at least `n` events; false on a CUDA error.
bool host_step_resources(int dev, size_t n, HostStepResources **out) {
    HostStepResources &r = g_host_step[dev];
    if (!r.ready) {
        if (cudaStreamCreateWithFlags(&r.s_in, cudaStreamNonBlocking) != cudaSuccess) return false;
        if (cudaStreamCreateWithFlags(&r.s_out, cudaStreamNonBlocking) != cudaSuccess) {
            cudaStreamDestroy(r.s_in);
            r.s_in = nullptr;
            return false;
        }
        r.ready = true;
    }
    while (r.events.size() < n) {
        cudaEvent_t e;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
        r.events.push_back(e);
    }
    *out = &r;
    return true;
}

}  // namespace
}  // namespace tsa

extern "C" {

size_t tsa_attention_backward_workspace_bytes(int64_t lanes, int64_t S, int64_t block, int64_t nnz_cap) {
    if (lanes <= 0 || S <= 0 || (block != 64 && block != 128) || nnz_cap < 1) return 0;
    const int64_t nb = (S + 63) / 64;  // 64-token blocks; a partial last block counts
    if (nb > kMaxBackwardBlocks || lanes * S >= (int64_t)INT_MAX || nnz_cap > INT_MAX / 4) return 0;
    // a 128-token CSR is expanded to 64-token blocks first: up to 4 entries per entry
    const int64_t nb_in = block == 128 ? (S + 127) / 128 : 0;
    return backward_workspace_layout(lanes, S, nb, block == 128 ? 4 * nnz_cap : nnz_cap, nb_in).total;
}

tsa_status tsa_scheduled_attention_backward(const void *Q, const void *K, const void *V, const void *O,
                                            const void *dO, const float *lse, const int32_t *row_ptr,
                                            const int32_t *col_idx, int64_t nnz_cap, void *dQ, void *dK,
                                            void *dV, tsa_dtype dtype, int64_t B, int64_t H, int64_t S,
                                            int64_t D, int64_t block, float scale, void *workspace,
                                            size_t workspace_bytes, tsa_stream_t stream) {
    if (!Q || !K || !V || !O || !dO || !lse || !row_ptr || !col_idx || !dQ || !dK || !dV || !workspace)
        return TSA_ERR_INVALID_ARGUMENT;
    if (dtype != TSA_F16 && dtype != TSA_BF16) return TSA_ERR_INVALID_ARGUMENT;
    if (B <= 0 || H <= 0 || S <= 0 || D <= 0 || block <= 0 || nnz_cap < 1) return TSA_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(scale)) return TSA_ERR_INVALID_ARGUMENT;
    if ((block != 64 && block != 128) || (D != 64 && D != 128)) return TSA_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535 || B * H > 65535) return TSA_ERR_UNSUPPORTED;
    // 64-token blocks (a partial last block counts); a 128-token CSR is expanded to them
    const int64_t lanes = B * H, nb = (S + 63) / 64;
    const int64_t nb_in = block == 128 ? (S + 127) / 128 : 0;
    if (lanes * S >= (int64_t)INT_MAX || nb > kMaxBackwardBlocks || nnz_cap > INT_MAX / 4)
        return TSA_ERR_UNSUPPORTED;
    const int64_t cap = block == 128 ? 4 * nnz_cap : nnz_cap;
    const void *ins[] = {Q, K, V, O, dO};
    void *outs[] = {dQ, dK, dV};
    for (const void *p : ins)
        if (reinterpret_cast<uintptr_t>(p) & 15u) return TSA_ERR_INVALID_ARGUMENT;
    for (const void *p : outs)
        if (reinterpret_cast<uintptr_t>(p) & 15u) return TSA_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(lse) & 15u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return TSA_ERR_INVALID_ARGUMENT;
    const size_t bytes = (size_t)(lanes * S * D) * 2;
    for (int x = 0; x < 3; ++x) {
        for (const void *p : ins)
            if (overlaps(outs[x], bytes, p, bytes)) return TSA_ERR_INVALID_ARGUMENT;
        if (overlaps(outs[x], bytes, lse, (size_t)(lanes * S) * 4)) return TSA_ERR_INVALID_ARGUMENT;
        for (int y = x + 1; y < 3; ++y)
            if (overlaps(outs[x], bytes, outs[y], bytes)) return TSA_ERR_INVALID_ARGUMENT;
    }
    const BwdWorkspace ws = backward_workspace_layout(lanes, S, nb, cap, nb_in);
    if (workspace_bytes < ws.total) return TSA_ERR_CAPACITY;
    int dev;
    TSA_TRY(current_device(&dev));
    for (const void *p : ins) TSA_TRY(check_device_ptr(p, dev));
    for (const void *p : outs) TSA_TRY(check_device_ptr(p, dev));
    for (const void *p : {static_cast<const void *>(lse), static_cast<const void *>(row_ptr),
                          static_cast<const void *>(col_idx), static_cast<const void *>(workspace)})
        TSA_TRY(check_device_ptr(p, dev));
    const bool bf16 = dtype == TSA_BF16;
    const uint64_t rows = (uint64_t)(lanes * S), cols = (uint64_t)D;
    CUtensorMap tQ128, tdO128, tQ64, tdO64, tK64, tV64, tdQ64, tdK64, tdV64;
    if (!encode_2d(&tQ128, Q, bf16, rows, cols, 128) || !encode_2d(&tdO128, dO, bf16, rows, cols, 128) ||
        !encode_2d(&tQ64, Q, bf16, rows, cols, 64) || !encode_2d(&tdO64, dO, bf16, rows, cols, 64) ||
        !encode_2d(&tK64, K, bf16, rows, cols, 64) || !encode_2d(&tV64, V, bf16, rows, cols, 64) ||
        !encode_2d(&tdQ64, dQ, bf16, rows, cols, 64) || !encode_2d(&tdK64, dK, bf16, rows, cols, 64) ||
        !encode_2d(&tdV64, dV, bf16, rows, cols, 64))
        return TSA_ERR_CUDA;
    uint8_t *w = static_cast<uint8_t *>(workspace);
    BwdLaunch a;
    a.tmQ128 = &tQ128;
    a.tmdO128 = &tdO128;
    a.tmQ64 = &tQ64;
    a.tmdO64 = &tdO64;
    a.tmK64 = &tK64;
    a.tmV64 = &tV64;
    a.tmdQ64 = &tdQ64;
    a.tmdK64 = &tdK64;
    a.tmdV64 = &tdV64;
    a.O = static_cast<const uint16_t *>(O);
    a.dO = static_cast<const uint16_t *>(dO);
    a.dQ = static_cast<uint16_t *>(dQ);
    a.dK = static_cast<uint16_t *>(dK);
    a.dV = static_cast<uint16_t *>(dV);
    a.lse = lse;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.nnz_cap = cap;
    a.nb_in = (int)nb_in;
    a.vlen_in = reinterpret_cast<int *>(w + ws.vlen_in);
    a.rp64 = reinterpret_cast<int32_t *>(w + ws.rp64);
    a.ci64 = reinterpret_cast<int32_t *>(w + ws.ci64);
    a.delta = reinterpret_cast<float *>(w + ws.delta);
    a.lse_pad = reinterpret_cast<float *>(w + ws.lse_pad);
    a.vlen = reinterpret_cast<int *>(w + ws.vlen);
    a.cnt = reinterpret_cast<int *>(w + ws.cnt);
    a.col_ptr = reinterpret_cast<int *>(w + ws.col_ptr);
    a.bitmap = reinterpret_cast<unsigned *>(w + ws.bitmap);
    a.bitmap_bytes = ws.bitmap_bytes;
    a.row_idx = reinterpret_cast<int32_t *>(w + ws.row_idx);
    a.pairs = reinterpret_cast<int *>(w + ws.pairs);
    a.nb = (int)nb;
    a.S = (int)S;
    a.D = (int)D;
    a.lanes = (int)lanes;
    a.bf16 = bf16;
    a.scale = scale;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    TSA_TRY(device_flags(dev, &a.flags));
    return launch_attention_backward(a);
}

tsa_status tsa_last_device_status(tsa_stream_t stream) {
    int dev;
    TSA_TRY(current_device(&dev));
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return TSA_ERR_CUDA;
    }
    unsigned bits = 0;
    const unsigned zero = 0;
    if (cudaMemcpyFromSymbol(&bits, g_status, sizeof(bits)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) {
        cudaGetLastError();
        return TSA_ERR_CUDA;
    }
    if (bits & kDevTimeout) return TSA_ERR_TIMEOUT;
    if (bits & kDevBadSchedule) return TSA_ERR_BAD_SCHEDULE;
    if (bits) return TSA_ERR_DEVICE;
    return TSA_OK;
}

tsa_status tsa_debug_set_wait_injection(int on) {
    if (on != 0 && on != 1) return TSA_ERR_INVALID_ARGUMENT;
    g_wait_injection.store((unsigned)on);
    return TSA_OK;
}


// One forward step from host memory, copies overlapped with the work (see include/tsa.h).
tsa_status tsa_topology_attention_host(const void *hQ, const void *hK, const void *hV, void *hO,
                                       tsa_dtype dtype, int64_t B, int64_t H, int64_t S, int64_t D,
                                       int64_t block, int64_t sink, int64_t local_radius, int64_t topk,
                                       tsa_tie_break tie_break, float scale, void *dQ, void *dK, void *dV,
                                       void *dO, int32_t *row_ptr, int32_t *col_idx, int64_t col_cap,
                                       void *workspace, size_t workspace_bytes, int64_t lane_chunk,
                                       tsa_stream_t stream) {
    if (!hQ || !hK || !hV || !hO || !dQ || !dK || !dV || !dO || !row_ptr || !col_idx || !workspace)
        return TSA_ERR_INVALID_ARGUMENT;
    if (dtype != TSA_F16 && dtype != TSA_BF16) return TSA_ERR_INVALID_ARGUMENT;
    if (tie_break != TSA_TIE_INDEX && tie_break != TSA_TIE_CONTENT) return TSA_ERR_INVALID_ARGUMENT;
    if (B <= 0 || H <= 0 || S <= 0 || D <= 0 || block <= 0 || lane_chunk < 0) return TSA_ERR_INVALID_ARGUMENT;
    if (sink < 0 || local_radius < 0 || topk < 0 || !std::isfinite(scale)) return TSA_ERR_INVALID_ARGUMENT;
    if ((block != 32 && block != 64 && block != 128) || (D != 64 && D != 128)) return TSA_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535 || B * H > 65535) return TSA_ERR_UNSUPPORTED;
    const int64_t lanes = B * H;
    if (lanes * S >= (int64_t)INT_MAX) return TSA_ERR_UNSUPPORTED;
    const int64_t nb = (S + block - 1) / block;
    if (nb > kMaxScheduleBlocks || D > kMaxScheduleDim) return TSA_ERR_UNSUPPORTED;
    void *dev_bufs[] = {dQ, dK, dV, dO};
    for (void *p : dev_bufs)
        if (reinterpret_cast<uintptr_t>(p) & 15u) return TSA_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TSA_ERR_INVALID_ARGUMENT;
    const size_t bytes = (size_t)(lanes * S * D) * 2;
    for (int x = 0; x < 4; ++x)
        for (int y = x + 1; y < 4; ++y)
            if (overlaps(dev_bufs[x], bytes, dev_bufs[y], bytes)) return TSA_ERR_INVALID_ARGUMENT;
    if (col_cap < max_nnz_bound(nb, sink, local_radius, topk)) return TSA_ERR_CAPACITY;
    const ScheduleWorkspace ws = schedule_workspace_layout(lanes, nb, D);
    if (workspace_bytes < ws.total) return TSA_ERR_CAPACITY;
    int dev;
    TSA_TRY(current_device(&dev));
    for (void *p : dev_bufs) TSA_TRY(check_device_ptr(p, dev));
    for (const void *p : {static_cast<const void *>(row_ptr), static_cast<const void *>(col_idx),
                          static_cast<const void *>(workspace)})
        TSA_TRY(check_device_ptr(p, dev));
    // the host side must be host memory (pinned for the copies to overlap; pageable works too)
    for (const void *p : {hQ, hK, hV, static_cast<const void *>(hO)}) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
            cudaGetLastError();
            return TSA_ERR_INVALID_ARGUMENT;
        }
        if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return TSA_ERR_INVALID_ARGUMENT;
    }
    const bool bf16 = dtype == TSA_BF16;
    const int64_t lc = lane_chunk > 0 ? (lane_chunk < lanes ? lane_chunk : lanes) : (lanes + 15) / 16;
    const int64_t nchunks = (lanes + lc - 1) / lc;
    if (nchunks > 4096) return TSA_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    DeviceFlags flags;
    TSA_TRY(device_flags(dev, &flags));

    // Two copy streams beside the caller's, the library's own (created once per device):
    // host-to-device (K first, then Q and V) and device-to-host (O).  The work itself runs on
    // the caller's stream.
    if (dev >= kHostStepDevices) return TSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_host_step_mutex[dev]);
    HostStepResources *res = nullptr;
    const size_t n_events = (size_t)(3 * nchunks + 3);
    if (!host_step_resources(dev, n_events, &res)) {
        cudaGetLastError();
        return TSA_ERR_CUDA;
    }
    cudaStream_t s_in = res->s_in, s_out = res->s_out;
    size_t next_event = 0;
    auto event = [&](cudaEvent_t *e) {
        *e = res->events[next_event++];
        return true;
    };
    const size_t lane_bytes = (size_t)(S * D) * 2;
    auto chunk = [&](const void *base, int64_t c) {
        return static_cast<const uint8_t *>(base) + (size_t)(c * lc) * lane_bytes;
    };
    auto chunk_lanes = [&](int64_t c) { return (c + 1) * lc <= lanes ? lc : lanes - c * lc; };
    bool ok = true;
    cudaEvent_t e_start = nullptr, e_end = nullptr;
    ok = ok && event(&e_start) && event(&e_end) && cudaEventRecord(e_start, st) == cudaSuccess &&
         cudaStreamWaitEvent(s_in, e_start, 0) == cudaSuccess && cudaStreamWaitEvent(s_out, e_start, 0) == cudaSuccess;
    std::vector<cudaEvent_t> e_k(nchunks), e_qv(nchunks), e_o(nchunks);
    for (int64_t c = 0; ok && c < nchunks; ++c) {
        const size_t n = (size_t)chunk_lanes(c) * lane_bytes;
        ok = event(&e_k[c]) &&
             cudaMemcpyAsync((void *)chunk(dK, c), chunk(hK, c), n, cudaMemcpyHostToDevice, s_in) == cudaSuccess &&
             cudaEventRecord(e_k[c], s_in) == cudaSuccess;
    }
    for (int64_t c = 0; ok && c < nchunks; ++c) {
        const size_t n = (size_t)chunk_lanes(c) * lane_bytes;
        ok = event(&e_qv[c]) &&
             cudaMemcpyAsync((void *)chunk(dQ, c), chunk(hQ, c), n, cudaMemcpyHostToDevice, s_in) == cudaSuccess &&
             cudaMemcpyAsync((void *)chunk(dV, c), chunk(hV, c), n, cudaMemcpyHostToDevice, s_in) == cudaSuccess &&
             cudaEventRecord(e_qv[c], s_in) == cudaSuccess;
    }
    // the schedule: per-lane block sums as each K chunk lands, then the lane mean and the graph
    ScheduleLaunch a{};
    a.K = static_cast<const uint16_t *>(dK);
    a.bf16 = bf16;
    a.lanes = lanes;
    a.S = S;
    a.D = D;
    a.block = block;
    a.nb = nb;
    a.sink = sink < nb ? sink : nb;
    a.local_radius = local_radius < nb ? local_radius : nb;
    a.topk = topk < nb ? topk : nb;
    a.content_ties = tie_break == TSA_TIE_CONTENT;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.col_cap = col_cap;
    a.salience_sq = nullptr;
    a.workspace = static_cast<uint8_t *>(workspace);
    a.stream = st;
    a.flags = flags;
    double *part = reinterpret_cast<double *>(a.workspace + ws.part);
    tsa_status status = ok ? TSA_OK : TSA_ERR_CUDA;
    for (int64_t c = 0; status == TSA_OK && c < nchunks; ++c) {
        if (cudaStreamWaitEvent(st, e_k[c], 0) != cudaSuccess) { status = TSA_ERR_CUDA; break; }
        ScheduleLaunch ac = a;
        ac.K = reinterpret_cast<const uint16_t *>(chunk(dK, c));
        ac.lanes = chunk_lanes(c);
        status = launch_block_sums(ac, part + (size_t)(c * lc) * (size_t)(nb * D));
    }
    if (status == TSA_OK) status = launch_schedule_from_sums(a, part);
    // attention per lane chunk as its Q and V land; its O goes back while the next one runs
    for (int64_t c = 0; status == TSA_OK && c < nchunks; ++c) {
        if (cudaStreamWaitEvent(st, e_qv[c], 0) != cudaSuccess) { status = TSA_ERR_CUDA; break; }
        status = launch_attention_checked(chunk(dQ, c), chunk(dK, c), chunk(dV, c), row_ptr, col_idx,
                                          (void *)chunk(dO, c), nullptr, bf16, chunk_lanes(c), S, D, block,
                                          scale, st, dev);
        if (status != TSA_OK) break;
        const size_t n = (size_t)chunk_lanes(c) * lane_bytes;
        if (!event(&e_o[c]) || cudaEventRecord(e_o[c], st) != cudaSuccess ||
            cudaStreamWaitEvent(s_out, e_o[c], 0) != cudaSuccess ||
            cudaMemcpyAsync((void *)chunk(hO, c), chunk(dO, c), n, cudaMemcpyDeviceToHost, s_out) != cudaSuccess)
            status = TSA_ERR_CUDA;
    }
    // the caller's stream continues once every copy has been made
    if (e_end) {
        cudaEvent_t e_in = nullptr;
        if (!event(&e_in) || cudaEventRecord(e_in, s_in) != cudaSuccess ||
            cudaStreamWaitEvent(s_out, e_in, 0) != cudaSuccess || cudaEventRecord(e_end, s_out) != cudaSuccess ||
            cudaStreamWaitEvent(st, e_end, 0) != cudaSuccess)
            status = TSA_ERR_CUDA;
    }
    if (status != TSA_OK) cudaGetLastError();
    return status;
}

}  // extern "C"
