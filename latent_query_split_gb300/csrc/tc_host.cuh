// tc_host.cuh -- host helpers shared by the tensor-core launchers: workspace
// alignment, the driver's tensor-map encoder and the 4-D bf16 tensor maps, and
// launches with programmatic dependent launch.
#pragma once

#include "tc_common.cuh"

#include <cudaTypedefs.h>

#include <mutex>

namespace flare {
namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 4-D bf16 tensor map, dims innermost first, 128-byte swizzle, box {64, b1, b2, 1}.
bool make_map(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t d3, uint32_t box1, uint32_t box2) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {d0, d1, d2, d3};
    const cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
    const cuuint32_t box[4] = {64, box1, box2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch with the programmatic-stream-serialization attribute when `pdl`: the
// kernel may start before the previous kernel in the stream has finished and
// must wait (griddepcontrol.wait) before touching that kernel's results.
template <typename Kernel, typename... Args>
cudaError_t launch_ex(Kernel k, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                      Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace
}  // namespace flare
