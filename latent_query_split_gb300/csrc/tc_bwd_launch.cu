// tc_bwd_launch.cu -- host side of the tensor-core backward kernels: shape
// coverage, workspace layouts, TMA tensor maps and the launchers of the
// encoder backward and the decode backward.
#include "tc_common.cuh"
#include "tc_backward.cuh"
#include "tc_decode_bwd.cuh"
#include "tc_host.cuh"

namespace flare {

bool tc_bwd_supported(bool bf16, int M, int D) {
    return bf16 && ((D == 64 && (M == 64 || M == 128 || M == 256)) || (D == 128 && (M == 64 || M == 128)));
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
    // the third stage's shared memory), and so does D = 128 (stages of 64 KB;
    // one beside M = 128's Q and dZ)
    constexpr int STAGES = D == 128 ? (M == 128 ? 1 : 2) : (ACCV ? 2 : 3);
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
        // one pass per 64-column half of dK, dV and dQ (M = 64 or 128)
        for (int dh = 0; dh < 2 && e == cudaSuccess; ++dh) {
            a.dh = dh;
            a.part = (float *)(w + l.part + dh * l.part_half);
            if (pr.M == 128)
                e = accumulate ? launch_bwd<128, true, false, 128>(maps, a, st)
                               : launch_bwd<128, false, false, 128>(maps, a, st);
            else
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
    return bf16 && ((D == 64 && (M == 64 || M == 128 || M == 256)) || (D == 128 && (M == 64 || M == 128)));
}

namespace {
// Decode-backward workspace: Z in bf16 [B*H*M*D] and the dQ/dZ pieces
// [B*H][P_max][2][M][64] of each 64-column half of D; tiles and spans as for
// the encoder backward. M = 256 adds the per-token statistics [B*H][N]
// (lse2, r).
struct DbwLayout {
    int64_t T_bh, T_total;
    int grid, P_max;
    size_t zb, part, part_half, stats, bytes;
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
    l.stats = o;
    if (pr.M > 128) o += align256(8 * (size_t)pr.B * pr.H * (size_t)pr.N);
    l.bytes = o;
}

template <int M, bool ST = false, int D = 64, bool ACCK = false>
cudaError_t launch_dbw(const CUtensorMap *maps, const tc::DbwArgs &a, cudaStream_t st) {
    // K/dY stages of 64 KB at D = 128: two at M = 64, one beside M = 128's Q and Z
    constexpr int STAGES = D == 128 ? (M == 128 ? 1 : 2) : 3;
    using C = tc::DbwCfg<M, STAGES, D>;
    auto k = tc::dbw_tc_kernel<M, STAGES, ST, D, ACCK>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::ALLOC);
    if (e != cudaSuccess) return e;
    // the warpgroups' register budgets (setmaxnreg) must add up to no more
    // than the block's registers at launch, or an increase would wait forever
    static_assert((C::REG_CTL + 2 * C::REG_SOFT + C::REG_EPI) * 128 <= 65536, "register budgets exceed the SM");
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, k)) != cudaSuccess) return e;
    // (four warpgroups: numRegs per thread at launch against their four budgets)
    if ((uint32_t)fa.numRegs * 4 < C::REG_CTL + 2 * C::REG_SOFT + C::REG_EPI) return cudaErrorInvalidConfiguration;
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
        // one pass per 64-column half of dK, dQ and dZ (M = 64 or 128)
        for (int dh = 0; dh < 2; ++dh) {
            a.dh = dh;
            a.part = (float *)(w + l.part + dh * l.part_half);
            e = pr.M == 128 ? launch_dbw<128, false, 128>(maps, a, st) : launch_dbw<64, false, 128>(maps, a, st);
            if (e != cudaSuccess) return e;
        }
    } else if (pr.M <= 128) {
        e = pr.M == 128 ? launch_dbw<128>(maps, a, st) : launch_dbw<64>(maps, a, st);
        if (e != cudaSuccess) return e;
    } else {
        // M = 256: the token statistics over all latents, then one pass per
        // half of the latents; the second adds its dK share to the first's
        float2 *stats = (float2 *)(w + l.stats);
        CUtensorMap smaps[4];
        if (!make_map(&smaps[0], K, pr.D, pr.H, pr.N, pr.B, 1, 128) ||
            !make_map(&smaps[1], dY, pr.D, pr.H, pr.N, pr.B, 1, 128) ||
            !make_map(&smaps[2], Q, pr.D, pr.M, pr.H, qb, (uint32_t)pr.M, 1) ||
            !make_map(&smaps[3], zb, pr.D, pr.M, pr.H, pr.B, (uint32_t)pr.M, 1))
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
        if ((e = launch_dbw<128, true, 64, true>(maps, a, st)) != cudaSuccess) return e;
    }
    const int64_t n4 = 2 * BH * pr.M * (pr.D / 4);
    tc::dbw_reduce_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(
        part, dQ, dZ, BH, pr.M, l.P_max, l.T_bh, l.T_total, l.grid, pr.D, (int64_t)(l.part_half / sizeof(float)));
    note_launch();
    return cudaGetLastError();
}

}  // namespace flare
