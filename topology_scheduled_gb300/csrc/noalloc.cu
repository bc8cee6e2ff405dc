// noalloc.cu -- tsa_build_schedule_noalloc: the topology schedule builder with its scratch in
// a fixed device array owned by this library, for callers that cannot allocate device memory.
//
// The scratch is one file-scope __device__ array of TSA_NOALLOC_SCRATCH_BYTES.  Every device
// that loads the library holds it until the process exits.  Host code cannot use the array's
// name as a device address (in host code it names a host-side stand-in), so the first call on
// each device looks the device address up with cudaGetSymbolAddress, with that device
// current, and caches it.
#include <climits>
#include <cstdint>
#include <mutex>

#include "tsa_internal.h"

namespace tsa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_address[kMaxScratchDevices] = {};

// Device address of g_noalloc_scratch on the current device `dev` (looked up once).
tsa_status scratch_address(int dev, void **out) {
    if (dev < 0 || dev >= kMaxScratchDevices) return TSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_address[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return TSA_ERR_CUDA;
        }
        g_scratch_address[dev] = p;
    }
    *out = g_scratch_address[dev];
    return TSA_OK;
}

}  // namespace
}  // namespace tsa

extern "C" tsa_status tsa_build_schedule_noalloc(const void *K, tsa_dtype dtype, int64_t lanes,
                                                 int64_t S, int64_t D, int64_t block,
                                                 int64_t sink, int64_t local_radius,
                                                 int64_t topk, int32_t *row_ptr,
                                                 int32_t *col_idx, int64_t col_cap,
                                                 double *salience_sq, tsa_stream_t stream) {
    if (!K || !row_ptr || !col_idx) return TSA_ERR_INVALID_ARGUMENT;
    // The callee's size checks, repeated before the scratch need is computed: the array is
    // shared by every call on the device, so a size that wrapped around must never pass the
    // capacity test below.
    if (lanes <= 0 || S <= 0 || D <= 0 || block <= 0) return TSA_ERR_INVALID_ARGUMENT;
    const int64_t nb = (S + block - 1) / block;
    if (nb > tsa::kMaxScheduleBlocks || D > tsa::kMaxScheduleDim) return TSA_ERR_UNSUPPORTED;
    if (lanes > INT64_MAX / S / D || lanes > INT64_MAX / 16 / nb / D) return TSA_ERR_INVALID_ARGUMENT;
    // Same scratch layout as the workspace of tsa_build_schedule.
    const size_t need = tsa_build_schedule_workspace_bytes(lanes, S, D, block);
    if (need == 0) return TSA_ERR_INVALID_ARGUMENT;
    if (need > (size_t)TSA_NOALLOC_SCRATCH_BYTES) return TSA_ERR_CAPACITY;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TSA_ERR_CUDA;
    }
    void *scratch = nullptr;
    const tsa_status st = tsa::scratch_address(dev, &scratch);
    if (st != TSA_OK) return st;
    // Nothing in the scratch has to start at zero: every region the builder reads is written
    // earlier in the same call, so the previous call's contents are never used.
    return tsa_build_schedule(K, dtype, lanes, S, D, block, sink, local_radius, topk, row_ptr,
                              col_idx, col_cap, salience_sq, scratch,
                              (size_t)TSA_NOALLOC_SCRATCH_BYTES, stream);
}
