// tc_common.cuh -- host-side interface of the tensor-core (tcgen05 / TMEM,
// TMA) kernels: which shapes they cover, how the encoder is tiled, and the
// launchers.
#pragma once

#include "flare_internal.cuh"

namespace flare {

// bf16 token tensors with M in {64, 128, 256} latents and D in {64, 128}.
bool tc_supported(bool bf16, int M, int D);
// TMA needs 16-byte aligned bases and a token stride (H*D*2 bytes) that is a
// multiple of 16.
bool tc_pointers_ok(const void *a, const void *b, int H, int D);

int tc_encoder_tile();                      // tokens per pipeline stage
int tc_encoder_min_chunk(int M, int D);     // smallest chunk worth a partial
int tc_encoder_ctas_per_sm(int M, int D);   // resident encoder CTAs per SM
int tc_encoder_waves();                     // grid size target in waves

cudaError_t launch_encoder_tc(const Problem &pr, const ShardPlan &plan, const void *Q,
                              bool q_is_f32, const void *K, const void *V, const uint8_t *mask,
                              const EncoderWorkspace &ws, const EncoderOut &out,
                              unsigned *status, cudaStream_t st);
cudaError_t launch_decode_tc(const Problem &pr, const void *Q, bool q_is_f32, const float *Z,
                             const void *K, void *Y, int sms, unsigned *status, cudaStream_t st);

bool tc_bwd_available();
size_t tc_encoder_bwd_workspace(const Problem &pr, int sms);
cudaError_t launch_encoder_bwd_tc(const Problem &pr, const void *Q, const void *K, const void *V,
                                  const uint8_t *mask, const float *Z, const float *L,
                                  const float *dZ, float *dQ, void *dK, void *dV, void *ws,
                                  size_t ws_bytes, int sms, unsigned *status, cudaStream_t st);

}  // namespace flare
