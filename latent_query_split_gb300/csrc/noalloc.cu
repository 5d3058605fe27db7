// noalloc.cu -- the split-KV encoder for callers that cannot allocate device
// memory: flare_encoder_fwd_noalloc (include/flare.h).
//
// Its scratch memory (the ticket counters, the per-piece partial outputs and
// log-normalisers of the split-KV encoder) lives in one file-scope device
// array of kNoAllocScratchBytes. Every GPU that loads this library holds that
// array until the process exits, and every call on a device reuses it.
#include "flare_internal.cuh"

#include <cstdio>
#include <mutex>
#include <vector>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
std::vector<void *> g_scratch_ptr;   // device address of the array, per device ordinal

// Device address of the scratch array on the current device. In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current.
flare_status_t scratch_on_current_device(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return flare::report_error(FLARE_ERR_CUDA, cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(g_mutex);
    if ((int)g_scratch_ptr.size() <= dev) g_scratch_ptr.resize(dev + 1, nullptr);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char msg[160];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress(scratch) failed: %s", cudaGetErrorString(e));
            return flare::report_error(FLARE_ERR_CUDA, msg);
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return FLARE_OK;
}

}  // namespace

extern "C" FLARE_API flare_status_t flare_encoder_fwd_noalloc(
    const flare_dims_t *dims, const void *Q, const void *K, const void *V, const uint8_t *mask,
    const int64_t *shard_offsets, int R, float *O_r, float *L_r, float *Z, float *L, void *stream) {
    FLARE_TRACE();
    const size_t need = flare::encoder_workspace_size(dims, shard_offsets, R);
    if (need == (size_t)-1)
        return flare::encoder_fwd_with_workspace(dims, Q, K, V, mask, shard_offsets, R, O_r, L_r, Z,
                                                 L, nullptr, 0, (cudaStream_t)stream);
    if (need > kNoAllocScratchBytes) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "problem needs %zu bytes of scratch; the static scratch of "
                 "flare_encoder_fwd_noalloc holds %zu (use flare_encoder_fwd with a workspace)",
                 need, kNoAllocScratchBytes);
        return flare::report_error(FLARE_ERR_WORKSPACE, msg);
    }
    void *scratch = nullptr;
    flare_status_t s = scratch_on_current_device(&scratch);
    if (s != FLARE_OK) return s;
    return flare::encoder_fwd_with_workspace(dims, Q, K, V, mask, shard_offsets, R, O_r, L_r, Z, L,
                                             scratch, kNoAllocScratchBytes, (cudaStream_t)stream);
}
