// flare_internal.cuh -- declarations shared by the library's translation units.
//
// The work decomposition: the tokens of every shard are cut into chunks of at
// most `chunk_len` tokens that never cross a shard boundary. A chunk is the
// unit of work of one encoder CTA; it produces the same pair the pages' local
// primitive returns for a shard (a normalised partial output and its row
// log-normaliser), so chunks merge into shards, and shards into the global
// result, by the one log-sum-exp rule of eq. 23.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/flare.h"

#include <nvtx3/nvToolsExt.h>

namespace flare {

constexpr int kMaxShards = FLARE_MAX_SHARDS;

// An NVTX range over one entry point, named after it: Nsight tools show each
// library call with the kernels it launched (`ncu --nvtx --nvtx-include
// "flare_fwd/"` profiles only the launches of flare_fwd). Without an attached
// tool a push or pop costs one pointer test.
struct TraceRange {
    explicit TraceRange(const char *name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};
#define FLARE_TRACE() ::flare::TraceRange flare_trace_range_(__func__)

// Shard offsets and their chunking, passed to kernels by value (about 3 KB of
// kernel parameters at the maximum shard count).
struct ShardPlan {
    int R;
    int chunk_len;                      // tokens per chunk (a multiple of the tile)
    int total_chunks;                   // chunks over all shards
    int pad_;
    int64_t off[kMaxShards + 1];        // shard token offsets
    int chunk_start[kMaxShards + 1];    // first chunk of each shard (prefix sums)
};

// Shard that owns chunk `c` (binary search over chunk_start).
__host__ __device__ inline int shard_of_chunk(const ShardPlan &p, int c) {
    int lo = 0, hi = p.R - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (p.chunk_start[mid] <= c) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Token range [n0, n1) of chunk `c`.
__host__ __device__ inline void chunk_range(const ShardPlan &p, int c, int64_t &n0, int64_t &n1) {
    int r = shard_of_chunk(p, c);
    int64_t start = p.off[r] + (int64_t)(c - p.chunk_start[r]) * p.chunk_len;
    n0 = start;
    n1 = start + p.chunk_len < p.off[r + 1] ? start + p.chunk_len : p.off[r + 1];
}

// Common problem description handed to the launchers.
struct Problem {
    int B, H, M, N, D;
    float scale;
    int64_t q_bstride;                   // elements between batch elements of Q
    bool bf16;                           // token tensors and Q are bf16
};

// Encoder workspace carve-up (all offsets are 256-byte aligned).
struct EncoderWorkspace {
    unsigned *tickets;   // [B*H*mtiles]
    float *part_L;       // [B*H*total_chunks*M]
    float *part_O;       // [B*H*total_chunks*M*D]
    float *shard_L;      // [B*H*R*M]  (scratch for L_r when the caller wants none)
    size_t bytes;
};

// Outputs of the encoder; any of them may be null (see flare_encoder_fwd).
struct EncoderOut {
    float *O_r, *L_r, *Z, *L;
};

// Device status word set by kernels that abandon a bounded wait.
enum : unsigned { kDevOk = 0, kDevTimeout = 1 };

// ---- launchers (each returns the cudaGetLastError() of its launches) --------
cudaError_t launch_encoder_simt(const Problem &pr, const ShardPlan &plan, const void *Q,
                                bool q_is_f32, const void *K, const void *V, const uint8_t *mask,
                                const EncoderWorkspace &ws, const EncoderOut &out,
                                cudaStream_t st);
cudaError_t launch_lse_merge(const float *O_r, const float *L_r, int R, int B, int H, int M,
                             int D, float *Z, float *L, cudaStream_t st);
// after_encoder: the previous kernel in the stream is this library's encoder
// that writes Z (the decode is launched as its programmatic dependent).
cudaError_t launch_decode_simt(const Problem &pr, const void *Q, bool q_is_f32, const float *Z,
                               const void *K, void *Y, bool after_encoder, cudaStream_t st);
cudaError_t launch_encoder_bwd_simt(const Problem &pr, const void *Q, const void *K,
                                    const void *V, const uint8_t *mask, const float *Z,
                                    const float *L, const float *dZ, float *dQ, void *dK,
                                    void *dV, void *ws, size_t ws_bytes, cudaStream_t st,
                                    bool accumulate = false);   // dQ, dK += this share
size_t encoder_bwd_simt_workspace(const Problem &pr);
cudaError_t launch_decode_bwd_simt(const Problem &pr, const void *Q, const float *Z, const void *K,
                                   const void *dY, float *dQ, float *dZ, void *dK, void *ws,
                                   cudaStream_t st);
size_t decode_bwd_simt_workspace(const Problem &pr);

// Rows of latents one SIMT encoder CTA handles.
constexpr int kSimtRows = 32;
// Tokens one SIMT encoder tile covers.
constexpr int kSimtTile = 32;

// Shared with the allocation-free encoder entry point (noalloc.cu).
size_t encoder_workspace_size(const flare_dims_t *dims, const int64_t *off, int R);
flare_status_t encoder_fwd_with_workspace(const flare_dims_t *dims, const void *Q, const void *K,
                                          const void *V, const uint8_t *mask, const int64_t *off,
                                          int R, float *O_r, float *L_r, float *Z, float *L,
                                          void *ws, size_t ws_bytes, cudaStream_t st);
flare_status_t report_error(flare_status_t s, const char *msg);

// Counts kernel launches for flare_launch_count (call once per <<<...>>>).
void note_launch();

void reset_device_status();
unsigned read_and_clear_device_status(cudaStream_t st, cudaError_t *err);

}  // namespace flare
