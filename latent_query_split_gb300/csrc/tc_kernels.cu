// tc_kernels.cu -- host side of the tensor-core kernels: shape coverage, the
// encoder's work split and workspace, TMA tensor maps, and the launchers.
#include "tc_common.cuh"
#include "tc_encoder.cuh"
#include "tc_decode.cuh"
#include "tc_backward.cuh"
#include "tc_decode_bwd.cuh"

#include <cudaTypedefs.h>

#include <cstring>
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

bool tc_bwd_supported(bool bf16, int M, int D) {
    return bf16 && ((D == 64 && (M == 64 || M == 128 || M == 256)) || (D == 128 && M == 64));
}

namespace {
// Backward workspace: dZ in bf16 [B*H*M*D], the row constants [B*H][2][M]
// and the dQ partials [B*H][P_max][M][64] of each 64-column half of D.
struct BwdLayout {
    int64_t T_bh, T_total;
    int grid, P_max;
    size_t dzb, lc, part, part_half, bytes;
};

void bwd_layout(const Problem &pr, int sms, BwdLayout &l) {
    l.T_bh = (pr.N + 127) / 128;
    l.T_total = (int64_t)pr.B * pr.H * l.T_bh;
    l.grid = (int)(l.T_total < sms ? l.T_total : sms);
    if (l.grid < 1) l.grid = 1;
    // a (b, h) spans at most ceil(T_bh / shortest span) + 1 CTAs
    const int64_t span_min = l.T_total > 0 ? l.T_total / l.grid : 1;
    l.P_max = l.T_bh > 0 ? (int)((l.T_bh + span_min - 1) / span_min) + 1 : 1;
    const size_t bhm = (size_t)pr.B * pr.H * pr.M;
    size_t o = 0;
    l.dzb = o;
    o += align256(2 * bhm * (size_t)pr.D);
    l.lc = o;
    o += align256(4 * bhm * 2);
    l.part = o;
    l.part_half = align256(4 * bhm * (size_t)l.P_max * 64);
    o += l.part_half * (size_t)(pr.D / 64);
    l.bytes = o;
}

template <int M, bool ACC, bool ACCV = false, int D = 64>
cudaError_t launch_bwd(const CUtensorMap *maps, const tc::BwdArgs &a, cudaStream_t st) {
    // the dV-accumulating pass keeps two K/V stages (its old-dV buffer takes
    // the third stage's shared memory), and so does D = 128 (stages of 64 KB)
    constexpr int STAGES = (ACCV || D == 128) ? 2 : 3;
    using C = tc::BwdCfg<M, STAGES, ACCV, D>;
    auto k = tc::bwd_tc_kernel<M, STAGES, ACC, ACCV, D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::ALLOC);
    if (e != cudaSuccess) return e;
    k<<<a.grid, C::THREADS, C::ALLOC, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], a);
    note_launch();
    return cudaGetLastError();
}
}  // namespace

size_t tc_encoder_bwd_workspace(const Problem &pr, int sms) {
    if (!tc_bwd_supported(pr.bf16, pr.M, pr.D)) return 0;
    BwdLayout l;
    bwd_layout(pr, sms, l);
    return l.bytes;
}

cudaError_t launch_encoder_bwd_tc(const Problem &pr, const void *Q, const void *K, const void *V,
                                  const uint8_t *mask, const float *Z, const float *L,
                                  const float *dZ, float *dQ, void *dK, void *dV, void *ws,
                                  size_t ws_bytes, int sms, unsigned *status, cudaStream_t st,
                                  bool accumulate) {
    if (!tc_bwd_supported(pr.bf16, pr.M, pr.D)) return cudaErrorNotSupported;
    BwdLayout l;
    bwd_layout(pr, sms, l);
    if (ws_bytes < l.bytes) return cudaErrorInvalidValue;
    const int64_t BH = (int64_t)pr.B * pr.H;
    if (BH == 0) return cudaSuccess;
    if (l.T_total == 0)            // no token: no share of dQ, no dK / dV
        return accumulate ? cudaSuccess : cudaMemsetAsync(dQ, 0, sizeof(float) * (size_t)BH * pr.M * pr.D, st);
    char *w = (char *)ws;
    __nv_bfloat16 *dzb = (__nv_bfloat16 *)(w + l.dzb);
    float *lc = (float *)(w + l.lc), *part = (float *)(w + l.part);
    const int64_t rows = BH * pr.M;
    tc::bwd_prep_kernel<<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(Z, L, dZ, dzb, lc, rows, pr.M,
                                                                            pr.scale, pr.D);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t qb = pr.q_bstride == 0 ? 1 : pr.B;
    // M = 256 runs as two passes over the tokens, one per half of the latent
    // rows (128 each, the TMEM columns of one pass); the second adds its
    // shares of dK and dV to the first's
    const int Mp = pr.M > 128 ? 128 : pr.M;
    CUtensorMap maps[6];
    if (!make_map(&maps[0], K, pr.D, pr.H, pr.N, pr.B, 1, 128) ||
        !make_map(&maps[1], V, pr.D, pr.H, pr.N, pr.B, 1, 128) ||
        !make_map(&maps[2], Q, pr.D, pr.M, pr.H, qb, (uint32_t)Mp, 1) ||
        !make_map(&maps[3], dzb, pr.D, pr.M, pr.H, pr.B, (uint32_t)Mp, 1) ||
        !make_map(&maps[4], dK, pr.D, pr.H, pr.N, pr.B, 1, 32) ||
        !make_map(&maps[5], dV, pr.D, pr.H, pr.N, pr.B, 1, 32))
        return cudaErrorInvalidValue;
    tc::BwdArgs a;
    a.B = pr.B;
    a.H = pr.H;
    a.M = Mp;
    a.N = pr.N;
    a.m0 = 0;
    a.M_all = pr.M;
    a.s = pr.scale;
    a.sl2 = pr.scale * 1.4426950408889634f;
    a.q_per_batch = pr.q_bstride != 0;
    a.mask = mask;
    a.lc = lc;
    a.part = part;
    a.dh = 0;
    a.dk_acc = accumulate ? (const __nv_bfloat16 *)dK : nullptr;
    a.dv_acc = nullptr;
    a.P_max = l.P_max;
    a.T_bh = l.T_bh;
    a.T_total = l.T_total;
    a.grid = l.grid;
    a.status = status;
    if (pr.D == 128) {
        // one pass per 64-column half of dK, dV and dQ (M = 64)
        for (int dh = 0; dh < 2 && e == cudaSuccess; ++dh) {
            a.dh = dh;
            a.part = (float *)(w + l.part + dh * l.part_half);
            e = accumulate ? launch_bwd<64, true, false, 128>(maps, a, st)
                           : launch_bwd<64, false, false, 128>(maps, a, st);
        }
    } else if (pr.M == 256) {
        // latent rows [0, 128): dK (+)= and dV = their shares
        e = accumulate ? launch_bwd<128, true>(maps, a, st) : launch_bwd<128, false>(maps, a, st);
        if (e != cudaSuccess) return e;
        // latent rows [128, 256): dK += and dV += their shares
        a.m0 = 128;
        a.dk_acc = (const __nv_bfloat16 *)dK;
        a.dv_acc = (const __nv_bfloat16 *)dV;
        e = launch_bwd<128, true, true>(maps, a, st);
    } else if (accumulate)
        e = pr.M == 128 ? launch_bwd<128, true>(maps, a, st) : launch_bwd<64, true>(maps, a, st);
    else
        e = pr.M == 128 ? launch_bwd<128, false>(maps, a, st) : launch_bwd<64, false>(maps, a, st);
    if (e != cudaSuccess) return e;
    const int64_t n4 = BH * pr.M * (pr.D / 4);
    tc::bwd_dq_reduce_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(
        part, dQ, BH, pr.M, l.P_max, l.T_bh, l.T_total, l.grid, accumulate ? 1 : 0, pr.D,
        (int64_t)(l.part_half / sizeof(float)));
    note_launch();
    return cudaGetLastError();
}

bool tc_decode_bwd_supported(bool bf16, int M, int D) {
    return bf16 && ((D == 64 && (M == 64 || M == 128 || M == 256)) || (D == 128 && M == 64));
}

namespace {
// Decode-backward workspace: Z in bf16 [B*H*M*D] and the dQ/dZ pieces
// [B*H][P_max][2][M][64] of each 64-column half of D; tiles and spans as for
// the encoder backward. M = 256 adds the per-token statistics [B*H][N]
// (lse2, r) and the second latent half's dK share [B][N][H][64] bf16.
struct DbwLayout {
    int64_t T_bh, T_total;
    int grid, P_max;
    size_t zb, part, part_half, stats, dk2, bytes;
};

void dbw_layout(const Problem &pr, int sms, DbwLayout &l) {
    l.T_bh = (pr.N + 127) / 128;
    l.T_total = (int64_t)pr.B * pr.H * l.T_bh;
    l.grid = (int)(l.T_total < sms ? l.T_total : sms);
    if (l.grid < 1) l.grid = 1;
    const int64_t span_min = l.T_total > 0 ? l.T_total / l.grid : 1;
    l.P_max = l.T_bh > 0 ? (int)((l.T_bh + span_min - 1) / span_min) + 1 : 1;
    const size_t bhm = (size_t)pr.B * pr.H * pr.M;
    size_t o = 0;
    l.zb = o;
    o += align256(2 * bhm * (size_t)pr.D);
    l.part = o;
    l.part_half = align256(4 * bhm * (size_t)l.P_max * 2 * 64);
    o += l.part_half * (size_t)(pr.D / 64);
    l.stats = l.dk2 = o;
    if (pr.M > 128) {
        const size_t bhn = (size_t)pr.B * pr.H * (size_t)pr.N;
        o += align256(8 * bhn);
        l.dk2 = o;
        o += align256(2 * bhn * 64);
    }
    l.bytes = o;
}

template <int M, bool ST = false, int D = 64>
cudaError_t launch_dbw(const CUtensorMap *maps, const tc::DbwArgs &a, cudaStream_t st) {
    constexpr int STAGES = D == 128 ? 2 : 3;     // K/dY stages of 64 KB at D = 128
    using C = tc::DbwCfg<M, STAGES, D>;
    auto k = tc::dbw_tc_kernel<M, STAGES, ST, D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::ALLOC);
    if (e != cudaSuccess) return e;
    k<<<a.grid, C::THREADS, C::ALLOC, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], a);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_dbs(const CUtensorMap *maps, const tc::DbsArgs &a, cudaStream_t st) {
    using C = tc::DbsCfg;
    cudaError_t e = cudaFuncSetAttribute(tc::dbs_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::ALLOC);
    if (e != cudaSuccess) return e;
    tc::dbs_stats_kernel<<<a.grid, C::THREADS, C::ALLOC, st>>>(maps[0], maps[1], maps[2], maps[3], a);
    note_launch();
    return cudaGetLastError();
}
}  // namespace

size_t tc_decode_bwd_workspace(const Problem &pr, int sms) {
    if (!tc_decode_bwd_supported(pr.bf16, pr.M, pr.D)) return 0;
    DbwLayout l;
    dbw_layout(pr, sms, l);
    return l.bytes;
}

cudaError_t launch_decode_bwd_tc(const Problem &pr, const void *Q, const float *Z, const void *K,
                                 const void *dY, float *dQ, float *dZ, void *dK, void *ws,
                                 size_t ws_bytes, int sms, unsigned *status, cudaStream_t st) {
    if (!tc_decode_bwd_supported(pr.bf16, pr.M, pr.D)) return cudaErrorNotSupported;
    DbwLayout l;
    dbw_layout(pr, sms, l);
    if (ws_bytes < l.bytes) return cudaErrorInvalidValue;
    const int64_t BH = (int64_t)pr.B * pr.H;
    if (BH == 0) return cudaSuccess;
    if (l.T_total == 0) {           // no token: dQ = dZ = 0, no dK
        cudaError_t e = cudaMemsetAsync(dQ, 0, sizeof(float) * (size_t)BH * pr.M * pr.D, st);
        return e != cudaSuccess ? e : cudaMemsetAsync(dZ, 0, sizeof(float) * (size_t)BH * pr.M * pr.D, st);
    }
    char *w = (char *)ws;
    __nv_bfloat16 *zb = (__nv_bfloat16 *)(w + l.zb);
    float *part = (float *)(w + l.part);
    const int64_t n2 = BH * pr.M * (pr.D / 2);
    tc::dbw_prep_kernel<<<(unsigned)((n2 + 255) / 256), 256, 0, st>>>(Z, zb, n2);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t qb = pr.q_bstride == 0 ? 1 : pr.B;
    // the tile kernel's latent rows per launch: all of them, or one half of 256
    const uint32_t Mp = pr.M > 128 ? 128 : (uint32_t)pr.M;
    CUtensorMap maps[5];
    if (!make_map(&maps[0], K, pr.D, pr.H, pr.N, pr.B, 1, 128) ||
        !make_map(&maps[1], dY, pr.D, pr.H, pr.N, pr.B, 1, 128) ||
        !make_map(&maps[2], Q, pr.D, pr.M, pr.H, qb, Mp, 1) ||
        !make_map(&maps[3], zb, pr.D, pr.M, pr.H, pr.B, Mp, 1) ||
        !make_map(&maps[4], dK, pr.D, pr.H, pr.N, pr.B, 1, 32))
        return cudaErrorInvalidValue;
    tc::DbwArgs a;
    a.B = pr.B;
    a.H = pr.H;
    a.M = (int)Mp;
    a.m0 = 0;
    a.M_all = pr.M;
    a.stats = nullptr;
    a.dh = 0;
    a.N = pr.N;
    a.s = pr.scale;
    a.sl2 = pr.scale * 1.4426950408889634f;
    a.q_per_batch = pr.q_bstride != 0;
    a.part = part;
    a.P_max = l.P_max;
    a.T_bh = l.T_bh;
    a.T_total = l.T_total;
    a.grid = l.grid;
    a.status = status;
    if (pr.D == 128) {
        // one pass per 64-column half of dK, dQ and dZ (M = 64)
        for (int dh = 0; dh < 2; ++dh) {
            a.dh = dh;
            a.part = (float *)(w + l.part + dh * l.part_half);
            if ((e = launch_dbw<64, false, 128>(maps, a, st)) != cudaSuccess) return e;
        }
    } else if (pr.M <= 128) {
        e = pr.M == 128 ? launch_dbw<128>(maps, a, st) : launch_dbw<64>(maps, a, st);
        if (e != cudaSuccess) return e;
    } else {
        // M = 256: the token statistics over all latents, then one pass per
        // half of the latents; the second half's dK share is added after
        float2 *stats = (float2 *)(w + l.stats);
        __nv_bfloat16 *dk2 = (__nv_bfloat16 *)(w + l.dk2);
        CUtensorMap smaps[4], dk2map;
        if (!make_map(&smaps[0], K, pr.D, pr.H, pr.N, pr.B, 1, 128) ||
            !make_map(&smaps[1], dY, pr.D, pr.H, pr.N, pr.B, 1, 128) ||
            !make_map(&smaps[2], Q, pr.D, pr.M, pr.H, qb, (uint32_t)pr.M, 1) ||
            !make_map(&smaps[3], zb, pr.D, pr.M, pr.H, pr.B, (uint32_t)pr.M, 1) ||
            !make_map(&dk2map, dk2, pr.D, pr.H, pr.N, pr.B, 1, 32))
            return cudaErrorInvalidValue;
        tc::DbsArgs sa;
        sa.B = pr.B;
        sa.H = pr.H;
        sa.N = pr.N;
        sa.sl2 = a.sl2;
        sa.q_per_batch = a.q_per_batch;
        sa.stats = stats;
        sa.T_bh = l.T_bh;
        sa.T_total = l.T_total;
        sa.grid = l.grid;
        sa.status = status;
        if ((e = launch_dbs(smaps, sa, st)) != cudaSuccess) return e;
        a.stats = stats;
        if ((e = launch_dbw<128, true>(maps, a, st)) != cudaSuccess) return e;
        a.m0 = 128;
        maps[4] = dk2map;
        if ((e = launch_dbw<128, true>(maps, a, st)) != cudaSuccess) return e;
        const int64_t n8 = (int64_t)pr.B * pr.N * pr.H * 8;     // uint4s of dK
        tc::dbw_add_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, st>>>(
            (uint4 *)dK, (const uint4 *)dk2, n8);
        note_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int64_t n4 = 2 * BH * pr.M * (pr.D / 4);
    tc::dbw_reduce_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(
        part, dQ, dZ, BH, pr.M, l.P_max, l.T_bh, l.T_total, l.grid, pr.D, (int64_t)(l.part_half / sizeof(float)));
    note_launch();
    return cudaGetLastError();
}

}  // namespace flare
