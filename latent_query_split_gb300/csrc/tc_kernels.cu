// tc_kernels.cu -- host side of the tensor-core forward kernels: shape
// coverage, the encoder's work split and workspace, TMA tensor maps, and the
// encoder, merge and decode launchers.
#include "tc_common.cuh"
#include "tc_encoder.cuh"
#include "tc_decode.cuh"
#include "tc_host.cuh"

#include <cstring>

namespace flare {
namespace {

__global__ void f32_to_bf16_kernel(const float *__restrict__ x, __nv_bfloat16 *__restrict__ y,
                                   int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        y[i] = __float2bfloat16_rn(x[i]);
}

// A CTA whose only work is a bounded wait on an mbarrier that nothing ever
// arrives on: the wait gives up after limit_ns exactly as the library's
// kernels do (abort flag, timeout in the device status word) and the kernel
// returns. No copy or MMA is in flight, so giving up leaves nothing behind.
__global__ void bounded_wait_probe_kernel(unsigned long long limit_ns, unsigned *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = tc::smem_u32(&bar);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        tc::mbar_init(b, 1);             // one arrival expected, none ever made
        tc::fence_mbar_init();
    }
    __syncthreads();
    const tc::Waiter wt{&abort_flag, status};
    if (threadIdx.x == 0) wt.wait_for(b, 0, limit_ns);
    __syncthreads();
}

}  // namespace

cudaError_t launch_bounded_wait_probe(unsigned long long limit_ns, unsigned *status,
                                      cudaStream_t st) {
    bounded_wait_probe_kernel<<<1, 32, 0, st>>>(limit_ns, status);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float *x, void *y, int64_t n, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
    f32_to_bf16_kernel<<<(unsigned)blocks, 256, 0, st>>>(x, (__nv_bfloat16 *)y, n);
    note_launch();
    return cudaGetLastError();
}

namespace {
template <class C, class Kernel>
cudaError_t launch_enc(Kernel k, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mq,
                       const tc::EncArgs &args, int grid, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::ALLOC);
    if (e != cudaSuccess) return e;
    k<<<grid, C::THREADS, C::ALLOC, st>>>(mk, mv, mq, args);
    note_launch();
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_merge(const Problem &pr, const tc::EncArgs &args, cudaStream_t st) {
    constexpr uint32_t smem = tc::merge_smem_bytes(D);
    auto k = tc::enc_merge_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int nrb = (pr.M + tc::merge_rows(D) - 1) / tc::merge_rows(D);
    e = launch_ex(k, dim3((unsigned)((int64_t)pr.B * pr.H * nrb)), dim3(256), smem, st, true, args);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool tc_supported(bool bf16, int M, int D) {
    if (!bf16) return false;
    if (D == 64) return M == 64 || M == 128 || M == 256;
    if (D == 128) return M == 64 || M == 128;
    return false;
}

bool tc_pointers_ok(const void *a, const void *b, int H, int D) {
    return ((uintptr_t)a % 16 == 0) && ((uintptr_t)b % 16 == 0) && ((size_t)H * D * 2) % 16 == 0;
}

bool tc_encoder_plan(const Problem &pr, const int64_t *off, int R, int sms, TcTilePlan &p,
                     TcEncLayout &lay) {
    std::memset(&p, 0, sizeof p);
    p.R = R;
    p.tile = pr.D == 128 ? 64 : 128;          // one K/V stage is 32 KB either way
    int ts = 0, max_nt = 0;
    for (int r = 0; r < R; ++r) {
        p.off[r] = off[r];
        p.tile_start[r] = ts;
        const int nt = (int)((off[r + 1] - off[r] + p.tile - 1) / p.tile);
        ts += nt;
        if (nt > max_nt) max_nt = nt;
    }
    p.off[R] = off[R];
    p.tile_start[R] = ts;
    p.T_bh = ts;
    p.T_total = (int64_t)pr.B * pr.H * ts;
    const int64_t want = (int64_t)sms;   // one persistent CTA per SM
    p.grid = (int)(p.T_total < want ? p.T_total : want);
    if (p.grid < 1) p.grid = 1;
    const int64_t span_min = p.T_total > 0 ? p.T_total / p.grid : 1;
    p.P_max = (int)((max_nt + span_min - 1) / (span_min > 0 ? span_min : 1)) + 1;
    // the merge keeps the pieces of one (b, h) in a table of kMergePieces
    if ((int64_t)R * p.P_max > tc::kMergePieces) return false;
    const size_t bh = (size_t)pr.B * pr.H;
    size_t o = 0;
    lay.part_L = o;
    o += align256(sizeof(float) * bh * R * p.P_max * pr.M);
    lay.part_O = o;
    o += align256(sizeof(float) * bh * R * p.P_max * pr.M * pr.D);
    lay.q_bf16 = o;
    o += align256(2 * bh * pr.M * pr.D);
    lay.bytes = o;
    return true;
}

cudaError_t launch_encoder_tc(const Problem &pr, const TcTilePlan &plan, const TcEncLayout &lay,
                              const void *Q, bool q_is_f32, const void *K, const void *V,
                              const uint8_t *mask, void *ws, const EncoderOut &out,
                              unsigned *status, cudaStream_t st) {
    char *w = (char *)ws;
    cudaError_t e;
    const void *Qbf = Q;
    int64_t qb = pr.q_bstride == 0 ? 1 : pr.B;
    if (q_is_f32) {
        // the dynamic FLARE++ queries are fp32: round them to bf16 once for TMA
        const int64_t n = qb * pr.H * pr.M * pr.D;
        f32_to_bf16_kernel<<<(unsigned)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024), 256, 0, st>>>(
            (const float *)Q, (__nv_bfloat16 *)(w + lay.q_bf16), n);
        note_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        Qbf = w + lay.q_bf16;
    }
    CUtensorMap mk, mv, mq;
    const uint32_t qrows = pr.M < 128 ? (uint32_t)pr.M : 128u;
    if (!make_map(&mk, K, pr.D, pr.H, pr.N, pr.B, 1, (uint32_t)plan.tile) ||
        !make_map(&mv, V, pr.D, pr.H, pr.N, pr.B, 1, (uint32_t)plan.tile) ||
        !make_map(&mq, Qbf, pr.D, pr.M, pr.H, qb, qrows, 1))
        return cudaErrorInvalidValue;
    tc::EncArgs a;
    a.B = pr.B;
    a.H = pr.H;
    a.M = pr.M;
    a.N = pr.N;
    a.sl2 = pr.scale * 1.4426950408889634f;
    a.q_per_batch = pr.q_bstride != 0;
    a.mask = mask;
    a.part_L = (float *)(w + lay.part_L);
    a.part_O = (float *)(w + lay.part_O);
    a.O_r = out.O_r;
    a.L_r = out.L_r;
    a.Z = out.Z;
    a.L = out.L;
    a.status = status;
    a.plan = plan;
    if (pr.D == 64 && pr.M <= 128)
        e = launch_enc<tc::CsCfg<64, 5>>(tc::enc_cs_kernel<64, 5>, mk, mv, mq, a, plan.grid, st);
    else if (pr.D == 128 && pr.M <= 128)
        e = launch_enc<tc::CsCfg<128, 4>>(tc::enc_cs_kernel<128, 4>, mk, mv, mq, a, plan.grid, st);
    else if (pr.D == 64 && pr.M == 256)
        e = launch_enc<tc::RingCfg<4>>(tc::enc_ring_kernel<4>, mk, mv, mq, a, plan.grid, st);
    else
        return cudaErrorNotSupported;
    if (e != cudaSuccess) return e;
    return pr.D == 64 ? launch_merge<64>(pr, a, st) : launch_merge<128>(pr, a, st);
}

bool tc_decode_available() { return true; }

namespace {
template <int M, int D, int STAGES, int QZB>
cudaError_t launch_dec(const CUtensorMap &mk, const CUtensorMap &my, const tc::DecArgs &args,
                       bool pdl, cudaStream_t st) {
    using C = tc::DecCfg<M, D, STAGES, QZB>;
    auto k = tc::dec_fwd_tc_kernel<M, D, STAGES, QZB>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::ALLOC);
    if (e != cudaSuccess) return e;
    e = launch_ex(k, dim3(args.grid), dim3(C::THREADS), C::ALLOC, st, pdl, mk, my, args);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}
}  // namespace

cudaError_t launch_decode_tc(const Problem &pr, const void *Q, bool q_is_f32, const float *Z,
                             const void *K, void *Y, int sms, unsigned *status, bool after_merge,
                             cudaStream_t st) {
    CUtensorMap mk, my;
    if (!make_map(&mk, K, pr.D, pr.H, pr.N, pr.B, 1, 128) ||
        !make_map(&my, Y, pr.D, pr.H, pr.N, pr.B, 1, 32))
        return cudaErrorInvalidValue;
    tc::DecArgs a;
    a.B = pr.B;
    a.H = pr.H;
    a.M = pr.M;
    a.N = pr.N;
    a.sl2 = pr.scale * 1.4426950408889634f;
    a.q_per_batch = pr.q_bstride != 0;
    a.q_f32 = q_is_f32;
    a.Q = Q;
    a.Z = Z;
    a.Y = (__nv_bfloat16 *)Y;
    a.T_bh = (pr.N + 127) / 128;
    a.T_total = (int64_t)pr.B * pr.H * a.T_bh;
    a.grid = (int)(a.T_total < sms ? a.T_total : sms);
    a.status = status;
    if (a.T_total == 0) return cudaSuccess;
    // <M, D, K stages, Q/Z buffers>, each within the shared-memory budget
    if (pr.M == 128 && pr.D == 64) return launch_dec<128, 64, 6, 2>(mk, my, a, after_merge, st);
    if (pr.M == 64 && pr.D == 64) return launch_dec<64, 64, 8, 2>(mk, my, a, after_merge, st);
    if (pr.M == 256 && pr.D == 64) return launch_dec<256, 64, 6, 1>(mk, my, a, after_merge, st);
    if (pr.M == 64 && pr.D == 128) return launch_dec<64, 128, 3, 1>(mk, my, a, after_merge, st);
    if (pr.M == 128 && pr.D == 128) return launch_dec<128, 128, 3, 1>(mk, my, a, after_merge, st);
    return cudaErrorNotSupported;
}

}  // namespace flare
