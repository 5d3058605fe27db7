// tc_decode_bwd.cuh -- FLARE decode backward on sm_103a tensor cores.
//
// The chain rule of the local decode (FLARE decode paragraph of "FLARE++:
// Low-rank attention with dynamic attention routing", appendix on context
// parallelism). For a (b, h), token n and latent m:
//   A_nm = softmax_m(s <K_n, Q_m>),  g_nm = <dY_n, Z_m>,  r_n = sum_m A_nm g_nm,
//   dT_nm = A_nm (g_nm - r_n),
//   dK_n = s sum_m dT_nm Q_m,  dQ_m = s sum_n dT_nm K_n,  dZ_m = sum_n A_nm dY_n.
//
// Kernels (D = 64, M in {64, 128}; the other shapes below):
//  * dbw_prep_kernel: Z rounded to bf16 (an MMA operand).
//  * dbw_tc_kernel: one persistent CTA per SM over a contiguous span of
//    128-token tiles in (b, h, tile) order. Per tile, token rows in the TMEM
//    lanes:
//        S^T = K Q^T,  G^T = dY Z^T                 (A, B from shared memory)
//        A, s dT from the row softmax (warps 4-11)  (fp32, bf16 operands out)
//        dK = (s dT) Q                              (A = s dT in its own TMEM columns)
//        dQ += (s dT)^T K,  dZ += A^T dY           (A from shared memory, MN-major)
//    Eight warps form two latent halves of every token row; the halves
//    exchange the row maximum, then their partial row sums and <A, g>.
//    Because s dT leaves S's columns, S/G of the next tile (same (b, h)) is
//    issued as soon as the halves have read this tile's, ahead of this tile's
//    gradient MMAs. dK leaves through shared memory (one TMA store per 32
//    rows, by the epilogue warps); dQ and dZ accumulate in TMEM over the
//    (b, h)'s tiles of the span and are written as one fp32 piece per (b, h)
//    of the span.
//  * dbw_reduce_kernel: dQ and dZ = the sums of the pieces in piece order.
// Warp roles (four warpgroups, each with its own register budget): warp 0
// TMA producer (K, dY ring; Q, Z on every (b, h) change), warp 1 TMEM
// allocator and MMA issuer (the converged warp; elect.sync picks the issuing
// lane), warps 4-11 the two latent halves, warps 12-15 the epilogue (dK of a
// lane quadrant's 32 token rows per tile, dQ and dZ pieces at a piece's end),
// so the halves never wait for a store.
//
// M = 256: S^T and G^T of one tile would fill all 512 TMEM columns, so the
// row statistics come first from dbs_stats_kernel (for every token, over all
// 256 latents: lse2_n = log2 sum_m 2^(s log2e <K_n, Q_m>) and r_n =
// sum_m A_nm g_nm), and dbw_tc_kernel<128, 3, true> then runs once per half
// of the latent rows with those statistics instead of its own (A_nm =
// 2^(s log2e <K_n, Q_m> - lse2_n), no exchange between the halves); the
// second pass (ACCK) adds its dK share to the first's: each epilogue warp
// loads the tile's old dK rows by TMA into its quadrant's staging slab
// before the tile's dK is ready, and adds them in fp32 before rounding once
// more.
//
// D = 128 (M = 64 or 128) runs as two passes over the tokens, one per
// 64-column half of dK, dQ and dZ: each pass contracts S and G over all 128 columns (K, dY,
// Q and Z tiles of two 64-column atoms) and computes its half's gradients in
// the TMEM columns of D = 64; each pass has its own dQ/dZ piece array. Two
// 64 KB K/dY stages leave no room for the dK staging slabs and the halves'
// exchange buffers, so at M = 64 these sit in the upper atoms of the A^T and
// s dT^T buffers: those atoms feed latent rows 64..127 of the dZ and dQ MMAs,
// whose output lanes are never read. At M = 128 there is room for one 64 KB
// stage only: S/G of the next tile is then issued after this tile's dQ and dZ
// have released the stage (no early issue).
#pragma once

#include "tc_backward.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace flare {
namespace tc {

struct DbwArgs {
    int B, H, M, N;
    // latent rows [m0, m0 + M) of M_all (Q and Z tiles, dQ and dZ pieces);
    // with precomputed statistics (M = 256), one (lse2, r) per token
    int m0, M_all;
    const float2 *stats;        // [B*H][N]
    float sl2;                  // s * log2(e)
    float s;                    // score scale
    int q_per_batch;            // Q has a batch dimension
    float *part;                // [B*H][P_max][2][M][64]: dQ, then dZ pieces (of this pass's half)
    int dh;                     // D = 128: the output column half [64 dh, 64 dh + 64)
    int P_max;
    int64_t T_bh, T_total;      // 128-token tiles per (b, h), and overall
    int grid;
    unsigned *status;
};

template <int M_, int STAGES_, int D_ = 64>
struct DbwCfg {
    static constexpr int M = M_, D = D_, TILE = 128, STAGES = STAGES_;
    static constexpr int DA = D / 64;                      // 64-column atoms of a row
    // four warpgroups: producer and MMA issuer (warps 0, 1; 2 and 3 idle),
    // the two latent halves (warps 4-11), the dK/dQ/dZ epilogue (warps 12-15)
    static constexpr int THREADS = 512;
    static constexpr int SOFT0 = 4, EPI0 = 12;
    // registers per thread of each warpgroup (setmaxnreg): 128 at launch,
    // 112 + 144 + 144 + 112 = 4 x 128
    static constexpr uint32_t REG_CTL = 112, REG_SOFT = 144, REG_EPI = 112;
    static constexpr uint32_t TILE_BYTES = TILE * 128;     // 128 rows x 64 bf16 (swizzled)
    static constexpr uint32_t QZA = M * 128;               // one [M][64] bf16 atom (swizzled)
    static constexpr uint32_t QZ_BYTES = DA * QZA;         // Q (or Z): its atoms in column order
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t ZB_OFF = Q_OFF + QZ_BYTES;
    static constexpr uint32_t STAGE_OFF = ZB_OFF + QZ_BYTES;
    static constexpr uint32_t STAGE_BYTES = 2 * DA * TILE_BYTES; // K atoms, then dY atoms
    // A^T and s dT^T in bf16: token rows of 64-latent atoms (atom a at a * TILE_BYTES)
    static constexpr uint32_t A_OFF = STAGE_OFF + STAGES * STAGE_BYTES;
    static constexpr uint32_t DT_OFF = A_OFF + 2 * TILE_BYTES;
    // D = 128 at M = 64: staging and exchange buffers in the upper atoms
    static constexpr bool IN_UPPER = DA == 2 && M <= 64;
    static constexpr uint32_t OUT_OFF = IN_UPPER ? A_OFF + TILE_BYTES : DT_OFF + 2 * TILE_BYTES;  // dK staging (4 slabs)
    // row statistics exchanged between the halves: [2 parity][2 half][128]
    static constexpr uint32_t XM_OFF = IN_UPPER ? DT_OFF + TILE_BYTES : OUT_OFF + TILE_BYTES;  // float: maxima
    static constexpr uint32_t XL_OFF = XM_OFF + 2 * 2 * 128 * 4;    // float2: (sum, <p, g>)
    static constexpr uint32_t BAR_OFF = IN_UPPER ? DT_OFF + 2 * TILE_BYTES : XL_OFF + 2 * 2 * 128 * 8;
    static_assert(!IN_UPPER || XL_OFF + 2 * 2 * 128 * 8 <= DT_OFF + 2 * TILE_BYTES, "exchange buffers overflow");
    // full[S], empty[S], qz_full, qz_free, s_full, p_full, at_free, dk_full,
    // dk_free, pz_full, pz_free, drain, sg_free, dkin[4] (ACCK: old dK rows)
    static constexpr int NBAR = 2 * STAGES + 15;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t BYTES = MISC_OFF + 64;
    static constexpr uint32_t ALLOC = BYTES + 1024;
    static_assert(ALLOC <= 232448, "shared memory budget of one CTA exceeded");
    static_assert(QZ_BYTES % 1024 == 0, "operand tiles must stay 1 KB aligned");
    // tensor memory columns
    // (s dT of a tile in bf16 pairs at DT_COL, so S/G of the next tile can
    // overwrite S_COL/G_COL while dK reads s dT)
    static constexpr uint32_t S_COL = 0, G_COL = 128, DK_COL = 256, DQ_COL = 320, DZ_COL = 384, DT_COL = 448;
    static constexpr uint32_t TMEM_COLS = 512;
};

// Z rounded to bf16, two elements per thread.
__global__ void __launch_bounds__(256) dbw_prep_kernel(const float *__restrict__ Z,
                                                       __nv_bfloat16 *__restrict__ Zb, int64_t n2) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n2) return;
    const float2 z = reinterpret_cast<const float2 *>(Z)[i];
    reinterpret_cast<uint32_t *>(Zb)[i] = pack_bf16(z.x, z.y);
}

// dQ (which = 0) and dZ (which = 1) = the sums of the pieces of each (b, h).
// The pieces of column half dh (D = 128: one piece array per pass) start at
// part + dh * half_stride floats; each holds [B*H][P_max][2][M][64].
__global__ void __launch_bounds__(256) dbw_reduce_kernel(const float *__restrict__ part,
                                                         float *__restrict__ dQ, float *__restrict__ dZ,
                                                         int64_t BH, int M, int P_max, int64_t T_bh,
                                                         int64_t T_total, int grid, int D,
                                                         int64_t half_stride) {
    const int64_t per = (int64_t)M * (D / 4);               // float4s of one (b, h) tensor
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= 2 * BH * per) return;
    const int which = (int)(i / (BH * per));
    const int64_t rest = i - which * BH * per;
    const int64_t bh = rest / per, rem = rest - bh * per;
    const int64_t m = rem / (D / 4);
    const int c4 = (int)(rem - m * (D / 4));
    const int c0 = bwd_cta_of(bh * T_bh, T_total, grid);
    const int np = bwd_cta_of(bh * T_bh + T_bh - 1, T_total, grid) - c0 + 1;
    const int64_t piece = (int64_t)M * 16;                  // float4s of one piece tensor
    const float4 *src = reinterpret_cast<const float4 *>(part + (c4 >> 4) * half_stride) +
                        (bh * P_max * 2 + which) * piece + m * 16 + (c4 & 15);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = 0; p < np; ++p) {
        const float4 v = __ldcg(src + p * 2 * piece);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    reinterpret_cast<float4 *>(which ? dZ : dQ)[bh * per + rem] = acc;
}

// ---- the row statistics of the M = 256 decode backward ----------------------
struct DbsArgs {
    int B, H, N;
    float sl2;                  // s * log2(e)
    int q_per_batch;
    float2 *stats;              // [B*H][N]: (lse2, r)
    int64_t T_bh, T_total;
    int grid;
    unsigned *status;
};

struct DbsCfg {
    static constexpr int M = 256, TILE = 128, STAGES = 3;
    static constexpr int THREADS = 320;                     // producer, MMA issuer, eight row warps
    static constexpr uint32_t TILE_BYTES = TILE * 128;      // 128 rows x 64 bf16 (swizzled)
    static constexpr uint32_t QZ_BYTES = M * 128;           // [256][64] bf16 (swizzled)
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t ZB_OFF = Q_OFF + QZ_BYTES;
    static constexpr uint32_t STAGE_OFF = ZB_OFF + QZ_BYTES;
    static constexpr uint32_t STAGE_BYTES = 2 * TILE_BYTES;   // K tile, then dY tile
    // the second latent half's (m, l, rg) per token row: [2][3][128] by tile parity
    static constexpr uint32_t XS_OFF = STAGE_OFF + STAGES * STAGE_BYTES;
    static constexpr uint32_t BAR_OFF = XS_OFF + 2 * 3 * 128 * 4;
    // full[S], empty[S], qz_full, qz_free, s_full, s_free, drain, x_full[4], x_free[4]
    static constexpr int NBAR = 2 * STAGES + 13;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t BYTES = MISC_OFF + 64;
    static constexpr uint32_t ALLOC = BYTES + 1024;
    static_assert(ALLOC <= 232448, "shared memory budget of one CTA exceeded");
    static constexpr uint32_t S_COL = 0, G_COL = 256, TMEM_COLS = 512;
};

// One persistent CTA per SM over a contiguous span of 128-token tiles in
// (b, h, tile) order. Per tile: S^T = K Q^T and G^T = dY Z^T (256 latents
// each, all of TMEM); two warps per lane quadrant take its 32 token rows,
// each folding 128 of the latents, 64 at a time, with a running maximum:
// l = sum 2^(t - m), rg = sum 2^(t - m) g. The second half's (m, l, rg) goes
// through shared memory (mbarrier hand-off per quadrant) to the first, which
// combines the two and writes lse2 = m + log2 l and r = rg / l.
__global__ void __launch_bounds__(DbsCfg::THREADS, 1)
dbs_stats_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmdY,
                 const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmZ,
                 const DbsArgs a) {
    using C = DbsCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::Q_OFF, sZ = sbase + C::ZB_OFF, sStage = sbase + C::STAGE_OFF;
    const uint32_t bar0 = sbase + C::BAR_OFF;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    const uint32_t qz_full = bar0 + 8u * (2 * C::STAGES), qz_free = qz_full + 8;
    const uint32_t s_full = qz_full + 16, s_free = qz_full + 24, drain = qz_full + 32;
    auto x_full = [&](int q) { return qz_full + 40 + 8u * q; };
    auto x_free = [&](int q) { return qz_full + 72 + 8u * q; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int64_t tb = ((int64_t)cta * a.T_total + a.grid - 1) / a.grid;
    const int64_t te = ((int64_t)(cta + 1) * a.T_total + a.grid - 1) / a.grid;
    const int64_t ntiles = te - tb;
    const int64_t bh0 = tb / a.T_bh, k0 = tb - bh0 * a.T_bh;
    Waiter wt{abort_flag, a.status};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(qz_full, 1);
        mbar_init(qz_free, 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, 8);          // one arrival per row warp
        mbar_init(drain, 1);
        for (int q = 0; q < 4; ++q) {
            mbar_init(x_full(q), 1);   // the quadrant's second-half warp has published
            mbar_init(x_free(q), 1);   // the quadrant's first-half warp has read
        }
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmdY);
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmZ);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- producer ----------------
        const uint64_t pol = policy_evict_first();
        int64_t bh = bh0, kt = k0, cur = -1;
        int b = (int)(bh0 / a.H), h = (int)(bh0 - (int64_t)b * a.H);
        int u = -1;
        int64_t j = 0;
        for (; j < ntiles && !wt.aborted(); ++j) {
            if (bh != cur) {
                ++u;
                cur = bh;
                // Q and Z of the previous (b, h) are no longer read
                if (u > 0 && !__all_sync(0xffffffffu, wt.wait_inline(qz_free, (uint32_t)(u - 1) & 1))) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(qz_full, 2 * C::QZ_BYTES);
                    if (dcheck(h >= 0 && h < a.H && b >= 0 && b < a.B, kChkDbwQ, a.status)) {
                        tma_load_4d(sQ, &tmQ, 0, 0, h, a.q_per_batch ? b : 0, qz_full);
                        tma_load_4d(sZ, &tmZ, 0, 0, h, b, qz_full);
                    }
                }
                __syncwarp();
            }
            const int s = (int)(j % C::STAGES);
            if (!__all_sync(0xffffffffu, wt.wait_inline(empty(s), ((uint32_t)(j / C::STAGES) & 1) ^ 1))) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(full(s), C::STAGE_BYTES);
                const uint32_t dst = sStage + s * C::STAGE_BYTES;
                if (dcheck(tile_in_tensor(0, h, kt * 128, b, a.H, a.N, a.B) && kt < a.T_bh, kChkDbwKV, a.status)) {
                    tma_load_4d_hint(dst, &tmK, 0, h, (int)(kt * 128), b, full(s), pol);
                    tma_load_4d_hint(dst + C::TILE_BYTES, &tmdY, 0, h, (int)(kt * 128), b, full(s), pol);
                }
            }
            __syncwarp();
            if (++kt == a.T_bh) {
                kt = 0;
                ++bh;
                if (++h == a.H) {
                    h = 0;
                    ++b;
                }
            }
        }
        if (wt.aborted() && lane == 0) {
            const uint64_t t0 = globaltimer();
            for (int64_t jj = (j > C::STAGES ? j - C::STAGES : 0); jj < j; ++jj)
                while (!mbar_try_wait(full((int)(jj % C::STAGES)), (uint32_t)(jj / C::STAGES) & 1) &&
                       globaltimer() - t0 < 500000000ull) {
                }
            if (u >= 0)
                while (!mbar_try_wait(qz_full, (uint32_t)u & 1) && globaltimer() - t0 < 500000000ull) {
                }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (converged warp, elect.sync issues) ----------------
        {
            constexpr uint32_t idS = idesc_bf16(128, 256, 0, 0);
            const uint64_t dQk = desc_sw128(sQ, 16, 1024);
            const uint64_t dZk = desc_sw128(sZ, 16, 1024);
            int64_t bh = bh0, kt = k0, cur = -1;
            int u = -1;
            bool ok = true;
            for (int64_t j = 0; j < ntiles && ok; ++j) {
                if (bh != cur) {
                    ++u;
                    cur = bh;
                    if (!(ok = __all_sync(0xffffffffu, wt.wait_inline(qz_full, (uint32_t)u & 1)))) break;
                }
                const int s = (int)(j % C::STAGES);
                if (!(ok = __all_sync(0xffffffffu, wt.wait_inline(full(s), (uint32_t)(j / C::STAGES) & 1)))) break;
                // the row warps have read the previous tile's S and G
                if (j > 0 && !(ok = __all_sync(0xffffffffu, wt.wait_inline(s_free, (uint32_t)(j - 1) & 1)))) break;
                tc_fence_after();
                const uint64_t dK = desc_sw128(sStage + s * C::STAGE_BYTES, 16, 1024);
                const uint64_t dY = desc_sw128(sStage + s * C::STAGE_BYTES + C::TILE_BYTES, 16, 1024);
#pragma unroll
                for (int kb = 0; kb < 4; ++kb)
                    umma_ss_elect(tmem + C::S_COL, dK + 2 * kb, dQk + 2 * kb, idS, kb > 0 ? 1u : 0u);
#pragma unroll
                for (int kb = 0; kb < 4; ++kb)
                    umma_ss_elect(tmem + C::G_COL, dY + 2 * kb, dZk + 2 * kb, idS, kb > 0 ? 1u : 0u);
                umma_commit_elect(s_full);
                umma_commit_elect(empty(s));
                if (++kt == a.T_bh) {
                    kt = 0;
                    ++bh;
                    umma_commit_elect(qz_free);   // the (b, h)'s last S and G read Q and Z
                }
            }
            if (wt.aborted()) {
                umma_commit_elect(drain);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < 500000000ull) {
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- row warps (warps 2-9, two per lane quadrant) ----------------
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;                 // latents [128 half, 128 half + 128)
        const int rig = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const float sl2 = a.sl2;
        float *xs = reinterpret_cast<float *>(smem + C::XS_OFF);
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait_inline(bar, par));
        };
        int64_t bh = bh0, kt = k0;
        for (int64_t j = 0; j < ntiles; ++j) {
            if (!wwait(s_full, (uint32_t)j & 1)) break;
            tc_fence_after();
            float m = -INFINITY, l0 = 0.f, l1 = 0.f, r0 = 0.f, r1 = 0.f;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                const uint32_t col = 128 * half + 64 * c;
                uint32_t sv[2][32], gv[2][32];
                tmem_ld32(tmem + C::S_COL + col + lane_off, sv[0]);
                tmem_ld32(tmem + C::S_COL + col + 32 + lane_off, sv[1]);
                tmem_ld32(tmem + C::G_COL + col + lane_off, gv[0]);
                tmem_ld32(tmem + C::G_COL + col + 32 + lane_off, gv[1]);
                tmem_wait_ld();
                if (c == 1) {
                    // S and G are in registers: the next tile's may be computed
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(s_free);
                }
                float c0 = -INFINITY, c1 = -INFINITY;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    c0 = max3(c0, __uint_as_float(sv[0][2 * i]), __uint_as_float(sv[0][2 * i + 1]));
                    c1 = max3(c1, __uint_as_float(sv[1][2 * i]), __uint_as_float(sv[1][2 * i + 1]));
                }
                const float cm = fmaxf(c0, c1) * sl2;
                if (cm > m) {
                    const float f = (m == -INFINITY) ? 0.f : ex2(m - cm);
                    l0 *= f;
                    l1 *= f;
                    r0 *= f;
                    r1 *= f;
                    m = cm;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float p0 = ex2(fmaf(__uint_as_float(sv[0][i]), sl2, -m));
                    const float p1 = ex2(fmaf(__uint_as_float(sv[1][i]), sl2, -m));
                    l0 += p0;
                    l1 += p1;
                    r0 = fmaf(p0, __uint_as_float(gv[0][i]), r0);
                    r1 = fmaf(p1, __uint_as_float(gv[1][i]), r1);
                }
            }
            const float l = l0 + l1, rg = r0 + r1;
            float *x = xs + (j & 1) * 384;
            if (half == 1) {
                // publish (m, l, rg) once the first half has read the previous
                // tile's: x_full then never runs two phases ahead of its
                // reader (a parity wait cannot tell phase j from phase j + 2)
                if (j >= 1 && !wwait(x_free(quad), (uint32_t)(j - 1) & 1)) break;
                x[rig] = m;
                x[128 + rig] = l;
                x[256 + rig] = rg;
                __syncwarp();
                if (lane == 0) mbar_arrive(x_full(quad));
            } else {
                if (!wwait(x_full(quad), (uint32_t)j & 1)) break;
                const float m1 = x[rig], l1v = x[128 + rig], r1v = x[256 + rig];
                __syncwarp();
                if (lane == 0) mbar_arrive(x_free(quad));
                const float mm = fmaxf(m, m1);
                const float f0 = ex2(m - mm), f1 = ex2(m1 - mm);   // maxima are finite
                const float lt = l * f0 + l1v * f1, rt = rg * f0 + r1v * f1;
                const int64_t n = kt * 128 + rig;
                if (n < a.N) a.stats[bh * a.N + n] = make_float2(mm + __log2f(lt), rt / lt);
            }
            if (++kt == a.T_bh) {
                kt = 0;
                ++bh;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// Per-warpgroup register budgets (every warp of a warpgroup executes the same one).
template <uint32_t R>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <uint32_t R>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

// Spin with test_wait and the bounded loop inline (no call: the warpgroups'
// register budgets differ).
__device__ __forceinline__ bool spin_inline(const Waiter &wt, uint32_t bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_test(bar, parity)) return true;
        if (*wt.abort) return false;
        if (globaltimer() - t0 > kWaitNs) {
            *wt.abort = 1;
            atomicCAS(wt.status, 0u, 1u);
            return false;
        }
    }
}

template <int M, int STAGES, bool ST = false, int D = 64, bool ACCK = false>
__global__ void __launch_bounds__(DbwCfg<M, STAGES, D>::THREADS, 1)
dbw_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmdY,
              const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmZ,
              const __grid_constant__ CUtensorMap tmdK, const DbwArgs a) {
    using C = DbwCfg<M, STAGES, D>;
    constexpr uint32_t TB = C::TILE_BYTES;
    constexpr int DA = C::DA;
    constexpr int W = M / 2;                                   // latents of each half
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::Q_OFF, sZ = sbase + C::ZB_OFF, sStage = sbase + C::STAGE_OFF;
    const uint32_t sA = sbase + C::A_OFF, sDT = sbase + C::DT_OFF;
    const uint32_t bar0 = sbase + C::BAR_OFF;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t qz_full = bar0 + 8u * (2 * STAGES), qz_free = qz_full + 8;
    const uint32_t s_full = qz_full + 16, p_full = qz_full + 24, at_free = qz_full + 32;
    const uint32_t dk_full = qz_full + 40, dk_free = qz_full + 48;
    const uint32_t pz_full = qz_full + 56, pz_free = qz_full + 64, drain = qz_full + 72;
    const uint32_t sg_free = qz_full + 80;
    auto dkin = [&](int q) { return qz_full + 88 + 8u * q; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int64_t tb = ((int64_t)cta * a.T_total + a.grid - 1) / a.grid;
    const int64_t te = ((int64_t)(cta + 1) * a.T_total + a.grid - 1) / a.grid;
    const int64_t ntiles = te - tb;
    const int64_t bh0 = tb / a.T_bh, k0 = tb - bh0 * a.T_bh;
    Waiter wt{abort_flag, a.status};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(qz_full, 1);
        mbar_init(qz_free, 1);
        mbar_init(s_full, 1);
        mbar_init(p_full, 8);          // one arrival per softmax warp
        mbar_init(at_free, 1);
        mbar_init(dk_full, 1);
        mbar_init(dk_free, 4);         // one arrival per epilogue warp
        mbar_init(pz_full, 1);
        mbar_init(pz_free, 4);
        mbar_init(drain, 1);
        mbar_init(sg_free, 8);         // every softmax warp has read S and G of the tile
        for (int q = 0; q < 4; ++q) mbar_init(dkin(q), 1);   // a quadrant's old dK rows are in
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmdY);
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmZ);
        prefetch_tmap(&tmdK);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (M < 128 && warp >= C::SOFT0 && warp < C::EPI0) {
        // latents M..127 of A^T and dT^T stay zero: the dQ and dZ MMAs span 128 rows
        for (int q = threadIdx.x - 32 * C::SOFT0; q < (int)TB / 16; q += 256) {
            reinterpret_cast<uint4 *>(smem + C::A_OFF + TB)[q] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4 *>(smem + C::DT_OFF + TB)[q] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < C::SOFT0) {
    regs_dec<C::REG_CTL>();
    if (warp == 0) {
        // ---------------- producer ----------------
        const uint64_t pol = policy_evict_first();
        int64_t bh = bh0, kt = k0, cur = -1;
        int b = (int)(bh0 / a.H), h = (int)(bh0 - (int64_t)b * a.H);   // (b, h) of tile j
        int u = -1;
        int64_t j = 0;
        for (; j < ntiles && !wt.aborted(); ++j) {
            if (bh != cur) {
                ++u;
                cur = bh;
                // Q and Z of the previous (b, h) are no longer read
                if (u > 0 && !__all_sync(0xffffffffu, wt.wait_inline(qz_free, (uint32_t)(u - 1) & 1))) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(qz_full, 2 * C::QZ_BYTES);
                    if (dcheck(h >= 0 && h < a.H && b >= 0 && b < a.B, kChkDbwQ, a.status)) {
#pragma unroll
                        for (int at = 0; at < DA; ++at) {
                            tma_load_4d(sQ + at * C::QZA, &tmQ, 64 * at, a.m0, h, a.q_per_batch ? b : 0, qz_full);
                            tma_load_4d(sZ + at * C::QZA, &tmZ, 64 * at, a.m0, h, b, qz_full);
                        }
                    }
                }
                __syncwarp();
            }
            const int s = (int)(j % STAGES);
            if (!__all_sync(0xffffffffu, wt.wait_inline(empty(s), ((uint32_t)(j / STAGES) & 1) ^ 1))) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(full(s), C::STAGE_BYTES);
                const uint32_t dst = sStage + s * C::STAGE_BYTES;
                if (dcheck(tile_in_tensor(0, h, kt * 128, b, a.H, a.N, a.B) && kt < a.T_bh, kChkDbwKV, a.status)) {
#pragma unroll
                    for (int at = 0; at < DA; ++at) {
                        tma_load_4d_hint(dst + at * TB, &tmK, 64 * at, h, (int)(kt * 128), b, full(s), pol);
                        tma_load_4d_hint(dst + (DA + at) * TB, &tmdY, 64 * at, h, (int)(kt * 128), b, full(s), pol);
                    }
                }
            }
            __syncwarp();
            if (++kt == a.T_bh) {
                kt = 0;
                ++bh;
                if (++h == a.H) {
                    h = 0;
                    ++b;
                }
            }
        }
        if (wt.aborted() && lane == 0) {
            // let every issued load land before the CTA exits
            const uint64_t t0 = globaltimer();
            for (int64_t jj = (j > STAGES ? j - STAGES : 0); jj < j; ++jj)
                while (!mbar_try_wait(full((int)(jj % STAGES)), (uint32_t)(jj / STAGES) & 1) &&
                       globaltimer() - t0 < 500000000ull) {
                }
            if (u >= 0)
                while (!mbar_try_wait(qz_full, (uint32_t)u & 1) && globaltimer() - t0 < 500000000ull) {
                }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (converged warp, elect.sync issues) ----------------
        {
            constexpr uint32_t idS = idesc_bf16(128, M, 0, 0);
            constexpr uint32_t idG = idesc_bf16(128, 64, 0, 1);    // dK: A in TMEM, B MN-major
            constexpr uint32_t idR = idesc_bf16(128, 64, 1, 1);    // dQ, dZ: A, B MN-major
            const uint64_t dQk = desc_sw128(sQ, 16, 1024);          // Q, K-major (B of S^T)
            const uint64_t dZk = desc_sw128(sZ, 16, 1024);          // Z, K-major (B of G^T)
            const uint64_t dQm = desc_sw128(sQ + a.dh * C::QZA, TB, 1024);   // Q, MN-major (B of dK)
            const uint64_t dAm = desc_sw128(sA, TB, 1024);          // A^T, MN-major (A of dZ)
            const uint64_t dDTm = desc_sw128(sDT, TB, 1024);        // s dT^T, MN-major (A of dQ)
            int64_t bhS = bh0, ktS = k0, curS = -1;
            int uS = -1;
            bool ok = true;
            auto issue_sg = [&](int64_t jj) -> bool {
                if (bhS != curS) {
                    ++uS;
                    curS = bhS;
                    if (!__all_sync(0xffffffffu, wt.wait_inline(qz_full, (uint32_t)uS & 1))) return false;
                }
                const int s = (int)(jj % STAGES);
                if (!__all_sync(0xffffffffu, wt.wait_inline(full(s), (uint32_t)(jj / STAGES) & 1))) return false;
                tc_fence_after();
                const uint64_t dK = desc_sw128(sStage + s * C::STAGE_BYTES, 16, 1024);
                const uint64_t dY = desc_sw128(sStage + s * C::STAGE_BYTES + DA * TB, 16, 1024);
                // over all D columns: 16 per MMA, four per atom
#pragma unroll
                for (int kb = 0; kb < 4 * DA; ++kb)
                    umma_ss_elect(tmem + C::S_COL, dK + (((kb >> 2) * TB) >> 4) + 2 * (kb & 3),
                                 dQk + (((kb >> 2) * C::QZA) >> 4) + 2 * (kb & 3), idS, kb > 0 ? 1u : 0u);
#pragma unroll
                for (int kb = 0; kb < 4 * DA; ++kb)
                    umma_ss_elect(tmem + C::G_COL, dY + (((kb >> 2) * TB) >> 4) + 2 * (kb & 3),
                                 dZk + (((kb >> 2) * C::QZA) >> 4) + 2 * (kb & 3), idS, kb > 0 ? 1u : 0u);
                umma_commit_elect(s_full);
                if (++ktS == a.T_bh) {
                    ktS = 0;
                    ++bhS;
                }
                return true;
            };
            // the waits on the halves' arrivals (sg_free, p_full, dk_free, pz_free)
            // spin with test_wait rather than suspend: this tile's products
            // start as soon as the slowest quadrant is done
            int64_t bhP = bh0, ktP = k0;
            int uP = 0;
            if (ntiles > 0) ok = issue_sg(0);
            for (int64_t j = 0; j < ntiles && ok; ++j) {
                const bool first = (j == 0) || ktP == 0;
                int64_t bhN = bhP, ktN = ktP + 1;
                if (ktN == a.T_bh) {
                    ktN = 0;
                    ++bhN;
                }
                const bool last = (j + 1 == ntiles) || bhN != bhP;
                // tile j + 1 of the same (b, h): its S/G as soon as S/G of tile j is read
                // (one K/dY stage: the next tile's load waits for this tile's dQ, dZ)
                const bool early = STAGES > 1 && j + 1 < ntiles && !last;
                if (early) {
                    if (!(ok = __all_sync(0xffffffffu, spin_inline(wt, sg_free, (uint32_t)j & 1)))) break;
                    if (!(ok = issue_sg(j + 1))) break;
                }
                if (!(ok = __all_sync(0xffffffffu, spin_inline(wt, p_full, (uint32_t)j & 1)))) break;
                tc_fence_after();
                if (j > 0 && !(ok = __all_sync(0xffffffffu, spin_inline(wt, dk_free, (uint32_t)(j - 1) & 1)))) break;
                tc_fence_after();
                // dK = (s dT) Q: K = M latents, 16 per MMA (A = s dT from its TMEM columns)
#pragma unroll
                for (int kb = 0; kb < M / 16; ++kb)
                    umma_ts_elect(tmem + C::DK_COL, tmem + C::DT_COL + 8 * kb, dQm + kb * (2048 >> 4), idG,
                                 kb > 0 ? 1u : 0u);
                umma_commit_elect(dk_full);
                if (last) umma_commit_elect(qz_free);
                // a tile of the next (b, h): its Q and Z arrive once qz_free fired
                if (STAGES > 1 && j + 1 < ntiles && !early && !(ok = issue_sg(j + 1))) break;
                // dQ += (s dT)^T K, dZ += A^T dY over the tile's 128 tokens
                if (first && uP > 0 && !(ok = __all_sync(0xffffffffu, spin_inline(wt, pz_free, (uint32_t)(uP - 1) & 1)))) break;
                tc_fence_after();
                const int s = (int)(j % STAGES);
                // the output column half's atoms of the K and dY tiles
                const uint64_t dKm = desc_sw128(sStage + s * C::STAGE_BYTES + a.dh * TB, TB, 1024);
                const uint64_t dYm = desc_sw128(sStage + s * C::STAGE_BYTES + (DA + a.dh) * TB, TB, 1024);
#pragma unroll
                for (int kb = 0; kb < 8; ++kb)
                    umma_ss_elect(tmem + C::DQ_COL, dDTm + kb * (2048 >> 4), dKm + kb * (2048 >> 4), idR,
                                 (kb > 0 || !first) ? 1u : 0u);
#pragma unroll
                for (int kb = 0; kb < 8; ++kb)
                    umma_ss_elect(tmem + C::DZ_COL, dAm + kb * (2048 >> 4), dYm + kb * (2048 >> 4), idR,
                                 (kb > 0 || !first) ? 1u : 0u);
                umma_commit_elect(at_free);
                umma_commit_elect(empty(s));
                if (last) {
                    umma_commit_elect(pz_full);
                    ++uP;
                }
                // one stage: S/G of the next tile once this tile's dQ, dZ have released it
                if (STAGES == 1 && j + 1 < ntiles && !(ok = issue_sg(j + 1))) break;
                bhP = bhN;
                ktP = ktN;
            }
            if (wt.aborted()) {
                umma_commit_elect(drain);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < 500000000ull) {
                }
            }
        }
        __syncwarp();
    }
    } else if (warp < C::EPI0) {
        regs_inc<C::REG_SOFT>();
        // ---------------- the two latent halves (warps 4-11) ----------------
        // Per tile j: S and G loaded (then sg_free, so S/G of tile j + 1 can be
        // computed), A and s dT formed, s dT into DT_COL once dK of tile j - 1
        // is done, A^T and s dT^T into shared memory once dQ, dZ of tile j - 1
        // are done, p_full.
        const int hf = (warp - C::SOFT0) >> 2;                // latent half
        const int quad = warp & 3;
        const int rig = quad * 32 + lane;                     // token row within the tile
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t s_tm = tmem + C::S_COL + W * hf + lane_off;
        const uint32_t g_tm = tmem + C::G_COL + W * hf + lane_off;
        const uint32_t t_tm = tmem + C::DT_COL + (W / 2) * hf + lane_off;   // this half's s dT (bf16 pairs)
        const float sl2 = a.sl2, sc = a.s;
        float *xm = reinterpret_cast<float *>(smem + C::XM_OFF);
        float2 *xl = reinterpret_cast<float2 *>(smem + C::XL_OFF);
        const int pair_bar = 1 + quad;                         // named barrier of the quadrant
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait_inline(bar, par));
        };
        int64_t bh = bh0, kt = k0;
        bool ok = true;
        for (int64_t j = 0; j < ntiles; ++j) {
            const int64_t n = kt * 128 + rig;
            const bool valid = n < a.N;
            // ST: the token's (lse2, r) over all latents, computed beforehand
            float2 stv = make_float2(0.f, 0.f);
            if constexpr (ST) {
                if (valid) stv = __ldg(a.stats + bh * a.N + n);
            }
            if (!(ok = wwait(s_full, (uint32_t)j & 1))) break;
            tc_fence_after();
            uint32_t sv[W / 32][32];
#pragma unroll
            for (int c = 0; c < W / 32; ++c) tmem_ld32(s_tm + 32 * c, sv[c]);
            tmem_wait_ld();
            const int par = (int)(j & 1);
            float m2;
            if constexpr (ST) {
                m2 = stv.x;                               // p = 2^(s log2e t - lse2) = A
            } else {
                // this half's scores: the maximum, exchanged with the other half
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < W / 32; ++c)
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        mx = max3(mx, __uint_as_float(sv[c][2 * i]), __uint_as_float(sv[c][2 * i + 1]));
                xm[(par * 2 + hf) * 128 + rig] = mx;
                named_bar_sync(pair_bar, 64);
                m2 = fmaxf(mx, xm[(par * 2 + (hf ^ 1)) * 128 + rig]) * sl2;
            }
            // p = 2^(s t log2 e - max), the half's partial sum and <p, g>
            uint32_t gv[W / 32][32];
#pragma unroll
            for (int c = 0; c < W / 32; ++c) tmem_ld32(g_tm + 32 * c, gv[c]);
            tmem_wait_ld();
            // S and G of this tile are in registers: the next tile's may be computed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sg_free);
            // two latents per packed instruction; two partial sums of each kind
            const uint64_t sl2x2 = f2pack(sl2, sl2), nm2x2 = f2pack(-m2, -m2);
            uint64_t ls2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
            uint64_t lr2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < W / 32; ++c)
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float t0, t1;
                    f2unpack(fma2(f2pack(__uint_as_float(sv[c][2 * i]), __uint_as_float(sv[c][2 * i + 1])), sl2x2,
                                  nm2x2),
                             t0, t1);
                    const float p0 = ex2(t0), p1 = ex2(t1);
                    sv[c][2 * i] = __float_as_uint(p0);
                    sv[c][2 * i + 1] = __float_as_uint(p1);
                    const uint64_t p2 = f2pack(p0, p1);
                    ls2[i & 1] = add2(ls2[i & 1], p2);
                    lr2[i & 1] = fma2(p2, f2pack(__uint_as_float(gv[c][2 * i]), __uint_as_float(gv[c][2 * i + 1])),
                                      lr2[i & 1]);
                }
            float inv, r;
            if constexpr (ST) {
                inv = valid ? 1.f : 0.f;                  // p is A already; tokens past N: A = 0
                r = stv.y;
            } else {
                float ls, lr;
                {
                    float x0, x1, x2, x3;
                    f2unpack(add2(ls2[0], ls2[1]), x0, x1);
                    f2unpack(add2(lr2[0], lr2[1]), x2, x3);
                    ls = x0 + x1;
                    lr = x2 + x3;
                }
                xl[(par * 2 + hf) * 128 + rig] = make_float2(ls, lr);
                named_bar_sync(pair_bar, 64);
                const float2 o = xl[(par * 2 + (hf ^ 1)) * 128 + rig];
                inv = valid ? 1.f / (ls + o.x) : 0.f;      // tokens past N: A = 0
                r = (lr + o.y) / (ls + o.x);
            }
            // s dT into DT_COL once dK of the previous tile (which read it) is
            // done; A^T and s dT^T into the MN-major operands of dZ and dQ once
            // the previous tile's products have read them
            if (j > 0 && !(ok = wwait(dk_full, (uint32_t)(j - 1) & 1))) break;
            if (j > 0 && !(ok = wwait(at_free, (uint32_t)(j - 1) & 1))) break;
            // A = p inv and s dT = A (s g - s r), two latents per instruction
            const uint64_t inv2 = f2pack(inv, inv), sc2 = f2pack(sc, sc), nsr2 = f2pack(-sc * r, -sc * r);
#pragma unroll
            for (int c = 0; c < W / 32; ++c) {
                uint32_t aw[16], tw[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint64_t a2 =
                        mul2(f2pack(__uint_as_float(sv[c][2 * i]), __uint_as_float(sv[c][2 * i + 1])), inv2);
                    const uint64_t t2 = mul2(
                        a2, fma2(f2pack(__uint_as_float(gv[c][2 * i]), __uint_as_float(gv[c][2 * i + 1])), sc2, nsr2));
                    float a0, a1, t0, t1;
                    f2unpack(a2, a0, a1);
                    f2unpack(t2, t0, t1);
                    aw[i] = pack_bf16(a0, a1);
                    tw[i] = pack_bf16(t0, t1);
                }
                tmem_st16(t_tm + 16 * c, tw);
                const int m0 = W * hf + 32 * c;
                uint8_t *arow = smem + C::A_OFF + (m0 >> 6) * TB + rig * 128;
                uint8_t *trow = smem + C::DT_OFF + (m0 >> 6) * TB + rig * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int pos = ((((m0 & 63) >> 3) + q) ^ (rig & 7)) << 4;
                    *reinterpret_cast<uint4 *>(arow + pos) = make_uint4(aw[4 * q], aw[4 * q + 1], aw[4 * q + 2], aw[4 * q + 3]);
                    *reinterpret_cast<uint4 *>(trow + pos) = make_uint4(tw[4 * q], tw[4 * q + 1], tw[4 * q + 2], tw[4 * q + 3]);
                }
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            if (++kt == a.T_bh) {
                kt = 0;
                ++bh;
            }
        }
        (void)ok;
    } else {
        regs_dec<C::REG_EPI>();
        // ---------------- epilogue (warps 12-15, one per lane quadrant) ----------------
        // Per tile j: dK of the quadrant's 32 token rows (all 64 columns) out
        // of TMEM once computed, through the quadrant's shared-memory slab by
        // one TMA store (ACCK: the old rows, loaded into the slab first, added
        // in fp32); at the end of a (b, h) piece, the span's dQ and dZ pieces
        // of the quadrant's 32 latent rows.
        const int quad = warp & 3;
        const int rig = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        uint8_t *slab = smem + C::OUT_OFF + quad * (32 * 128);
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait_inline(bar, par));
        };
        int64_t bh = bh0, kt = k0;
        int b = (int)(bh0 / a.H), h = (int)(bh0 - (int64_t)b * a.H);
        int pieces = 0;
        uint32_t stores = 0, dk_loads = 0, dk_issued = 0;
        for (int64_t j = 0; j < ntiles; ++j) {
            int64_t bhN = bh, ktN = kt + 1;
            int bN = b, hN = h;
            if (ktN == a.T_bh) {
                ktN = 0;
                ++bhN;
                if (++hN == a.H) {
                    hN = 0;
                    ++bN;
                }
            }
            const bool last = (j + 1 == ntiles) || bhN != bh;
            const int n0 = (int)(kt * 128) + quad * 32;
            const bool rows = n0 < a.N;
            // the slab is free once its last store has read it
            if (stores > 0 && lane == 0) bulk_wait_group_read0();
            __syncwarp();
            if (ACCK && rows) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(dkin(quad), 32 * 128);
                    if (dcheck(tile_in_tensor(64 * a.dh, h, n0, b, a.H, a.N, a.B), kChkDbwOut, a.status))
                        tma_load_4d(smem_u32(slab), &tmdK, 64 * a.dh, h, n0, b, dkin(quad));
                }
                ++dk_issued;
            }
            if (!wwait(dk_full, (uint32_t)j & 1)) break;
            tc_fence_after();
            uint32_t rk[2][32];
            tmem_ld32(tmem + C::DK_COL + lane_off, rk[0]);
            tmem_ld32(tmem + C::DK_COL + 32 + lane_off, rk[1]);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dk_free);
            if (ACCK && rows) {
                if (!wwait(dkin(quad), (uint32_t)dk_loads & 1)) break;
                ++dk_loads;
            }
            uint8_t *srow = slab + lane * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t *k8 = rk[q >> 2] + 8 * (q & 3);
                uint4 *dst = reinterpret_cast<uint4 *>(srow + ((q ^ (lane & 7)) << 4));
                if constexpr (ACCK) {
                    // bf16 pairs of the old row, the even column in the low half
                    const uint4 o = *dst;
                    const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        k8[2 * k] = __float_as_uint(__uint_as_float(k8[2 * k]) + __uint_as_float(ow[k] << 16));
                        k8[2 * k + 1] =
                            __float_as_uint(__uint_as_float(k8[2 * k + 1]) + __uint_as_float(ow[k] & 0xffff0000u));
                    }
                }
                *dst = make_uint4(pack_bf16(__uint_as_float(k8[0]), __uint_as_float(k8[1])),
                                  pack_bf16(__uint_as_float(k8[2]), __uint_as_float(k8[3])),
                                  pack_bf16(__uint_as_float(k8[4]), __uint_as_float(k8[5])),
                                  pack_bf16(__uint_as_float(k8[6]), __uint_as_float(k8[7])));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && rows && dcheck(tile_in_tensor(64 * a.dh, h, n0, b, a.H, a.N, a.B), kChkDbwOut, a.status)) {
                // rows past N are clipped by the tensor map
                tma_store_4d(&tmdK, smem_u32(slab), 64 * a.dh, h, n0, b);
                bulk_commit_group();
            }
            ++stores;
            if (last) {
                if (!wwait(pz_full, (uint32_t)pieces & 1)) break;
                tc_fence_after();
                const int piece = cta - bwd_cta_of(bh * a.T_bh, a.T_total, a.grid);
#pragma unroll 1
                for (int which = 0; which < 2; ++which) {     // dQ, then dZ
                    uint32_t rq[2][32];
                    tmem_ld32(tmem + (which ? C::DZ_COL : C::DQ_COL) + lane_off, rq[0]);
                    tmem_ld32(tmem + (which ? C::DZ_COL : C::DQ_COL) + 32 + lane_off, rq[1]);
                    tmem_wait_ld();
                    if (rig < M) {
                        float4 *dst = reinterpret_cast<float4 *>(
                            a.part + (((bh * a.P_max + piece) * 2 + which) * a.M_all + a.m0 + rig) * 64);
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                dst[8 * h2 + q] = make_float4(
                                    __uint_as_float(rq[h2][4 * q]), __uint_as_float(rq[h2][4 * q + 1]),
                                    __uint_as_float(rq[h2][4 * q + 2]), __uint_as_float(rq[h2][4 * q + 3]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pz_free);
                ++pieces;
            }
            bh = bhN;
            kt = ktN;
            b = bN;
            h = hN;
        }
        if constexpr (ACCK) {
            // an old-dK load still in flight (a wait given up) lands before the CTA exits
            if (lane == 0 && dk_issued > dk_loads) {
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(dkin(quad), (uint32_t)dk_loads & 1) && globaltimer() - t0 < 500000000ull) {
                }
            }
        }
        if (lane == 0) bulk_wait_group0();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace tc
}  // namespace flare
