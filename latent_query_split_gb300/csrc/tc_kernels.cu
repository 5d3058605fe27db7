// tc_kernels.cu -- tensor-core kernels (placeholder: no shape routed here yet).
#include "tc_common.cuh"

namespace flare {

bool tc_supported(bool, int, int) { return false; }
bool tc_pointers_ok(const void *, const void *, int, int) { return false; }
int tc_encoder_tile() { return 128; }
int tc_encoder_min_chunk(int, int) { return 1024; }
int tc_encoder_ctas_per_sm(int, int) { return 1; }
int tc_encoder_waves() { return 2; }
cudaError_t launch_encoder_tc(const Problem &, const ShardPlan &, const void *, bool, const void *,
                              const void *, const uint8_t *, const EncoderWorkspace &,
                              const EncoderOut &, unsigned *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_decode_tc(const Problem &, const void *, bool, const float *, const void *,
                             void *, int, unsigned *, cudaStream_t) {
    return cudaErrorNotSupported;
}
bool tc_bwd_available() { return false; }
size_t tc_encoder_bwd_workspace(const Problem &, int) { return 0; }
cudaError_t launch_encoder_bwd_tc(const Problem &, const void *, const void *, const void *,
                                  const uint8_t *, const float *, const float *, const float *,
                                  float *, void *, void *, void *, size_t, int, unsigned *,
                                  cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace flare
