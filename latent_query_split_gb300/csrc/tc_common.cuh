// tc_common.cuh -- host-side interface of the tensor-core (tcgen05 / TMEM,
// TMA) kernels: which shapes they cover, how the encoder splits its work, the
// workspace it needs, and the launchers.
#pragma once

#include "flare_internal.cuh"

namespace flare {

// bf16 token tensors with M in {64, 128, 256} latents and D in {64, 128}
// (M = 256 only with D = 64).
bool tc_supported(bool bf16, int M, int D);
// TMA needs 16-byte aligned bases and a token stride (H*D*2 bytes) that is a
// multiple of 16.
bool tc_pointers_ok(const void *a, const void *b, int H, int D);

// Split of the encoder's work. Every shard is cut into tiles of `tile` tokens
// (the last one ragged); all (b, h) share the shard layout, so tile t of the
// flattened order (b, h)-major, then shard, then tile sits at a computable
// place. `grid` persistent CTAs each take one contiguous, equally long span
// of that order; a span cut into (b, h, shard) pieces gives one partial
// (normalised output and log-normaliser) per piece, merged afterwards by a
// separate kernel.
struct TcTilePlan {
    int R;
    int tile;                       // tokens per tile
    int T_bh;                       // tiles per (b, h)
    int P_max;                      // partial slots per (b, h, shard)
    int grid;                       // persistent CTAs
    int64_t T_total;                // tiles over every (b, h)
    int64_t off[kMaxShards + 1];    // shard token offsets
    int tile_start[kMaxShards + 1]; // first tile of each shard within a (b, h)
};

// Byte offsets of the encoder workspace regions: per-piece partials (L, O)
// and a bf16 copy of an fp32 query.
struct TcEncLayout {
    size_t part_L, part_O, q_bf16, bytes;
};

bool tc_encoder_plan(const Problem &pr, const int64_t *off, int R, int sms, TcTilePlan &plan,
                     TcEncLayout &lay);

cudaError_t launch_encoder_tc(const Problem &pr, const TcTilePlan &plan, const TcEncLayout &lay,
                              const void *Q, bool q_is_f32, const void *K, const void *V,
                              const uint8_t *mask, void *ws, const EncoderOut &out,
                              unsigned *status, cudaStream_t st);
bool tc_decode_available();
// after_merge: the previous kernel in the stream is this library's encoder
// kernel that writes Z, and Q and K were written before it (the decode then
// overlaps that kernel's tail); callers whose previous kernel is unknown pass
// false.
cudaError_t launch_decode_tc(const Problem &pr, const void *Q, bool q_is_f32, const float *Z,
                             const void *K, void *Y, int sms, unsigned *status, bool after_merge,
                             cudaStream_t st);

// bf16 with D = 64 and M in {64, 128}.
bool tc_bwd_supported(bool bf16, int M, int D);
size_t tc_encoder_bwd_workspace(const Problem &pr, int sms);
cudaError_t launch_encoder_bwd_tc(const Problem &pr, const void *Q, const void *K, const void *V,
                                  const uint8_t *mask, const float *Z, const float *L,
                                  const float *dZ, float *dQ, void *dK, void *dV, void *ws,
                                  size_t ws_bytes, int sms, unsigned *status, cudaStream_t st,
                                  bool accumulate = false);   // dQ, dK += this share

// One small kernel that waits on an mbarrier nothing arrives on and gives the
// wait up after limit_ns (the library's bounded-wait path, with no other work).
cudaError_t launch_bounded_wait_probe(unsigned long long limit_ns, unsigned *status,
                                      cudaStream_t st);

// y[i] = x[i] rounded to bf16 (nearest even), n elements.
cudaError_t launch_f32_to_bf16(const float *x, void *y, int64_t n, cudaStream_t st);

// Decode backward on tensor cores: bf16 with D = 64 and M in {64, 128}.
bool tc_decode_bwd_supported(bool bf16, int M, int D);
size_t tc_decode_bwd_workspace(const Problem &pr, int sms);
cudaError_t launch_decode_bwd_tc(const Problem &pr, const void *Q, const float *Z, const void *K,
                                 const void *dY, float *dQ, float *dZ, void *dK, void *ws,
                                 size_t ws_bytes, int sms, unsigned *status, cudaStream_t st);

}  // namespace flare
