// tc_backward.cuh -- global-normaliser FLARE encoder backward on sm_103a
// tensor cores.
//
// With the forward's global statistics (Z, L) every token's gradient is
// local ("FLARE++: Low-rank attention with dynamic attention routing",
// appendix on context parallelism, backward paragraphs: globally normalised
// local probabilities, the row scalar c, local key/value gradients, the query
// gradient summed over shards):
//   P_mn  = exp(s <Q_m, K_n> - L_m)       (0 for padding and for L_m = -inf)
//   dS_mn = P_mn (<dZ_m, V_n> - c_m),     c_m = <dZ_m, Z_m>
//   dV_n  = sum_m P_mn dZ_m,  dK_n = s sum_m dS_mn Q_m,  dQ_m = s sum_n dS_mn K_n.
//
// Three kernels:
//  * bwd_prep_kernel: per latent row, dZ rounded to bf16 (an MMA operand),
//    -L in log2 units (-inf for an empty row, so its P is 0) and -s c.
//  * bwd_tc_kernel: one persistent CTA per SM over a contiguous span of
//    128-token tiles in (b, h, tile) order (shards play no part: with the
//    global L and c each token is independent). Per tile, with the token rows
//    in the 128 TMEM lanes:
//        S^T = K Q^T,  dP^T = V dZ^T                    (A, B from shared memory)
//        P = exp2(S^T s log2e - L2), s dS = P (s dP - s c)  (softmax warps, fp32)
//        dV = P^T dZ                                    (A = bf16 P^T in its own TMEM columns)
//        dK = (s dS)^T Q,  dQ += (s dS) K               (A = bf16 dS^T in shared memory)
//    Because P and dS leave S/dP's columns, S/dP of the next tile (same
//    (b, h)) is issued as soon as the softmax warps have read this tile's,
//    ahead of this tile's gradient MMAs; the softmax warps store a tile's
//    dK/dV (its epilogue) after publishing the next tile's P and dS.
//    dK and dV leave through shared memory by TMA stores; dQ accumulates in
//    TMEM over the (b, h)'s tiles of the span and is written as one fp32
//    partial per (b, h) piece of the span.
//  * bwd_dq_reduce_kernel: dQ = sum of the pieces of each (b, h), in piece
//    order (deterministic).
// With accumulation on (the mixer backward, where the decode's shares of dK
// and dQ are already in the output buffers) dK = dK + the encoder's share and
// dQ = dQ + the encoder's share: the dK epilogue prefetches the tile's rows of
// the old dK with cp.async at the start of the tile and adds them in fp32
// before rounding once.
// D = 128 (M = 64 or 128) runs as two passes over the tokens, one per 64-column half
// of the outputs: each pass contracts S and dP over all 128 columns (K, V,
// Q and dZ tiles of two 64-column atoms each) and computes dV, dK and dQ for
// its half (the TMEM columns of D = 64); the dQ partials of each pass have
// their own piece array. The shared memory of two 64 KB K/V stages leaves
// no room for the old-dK rows beside the output staging, so at M = 64 those
// rows sit in the upper atom of the s dS^T buffer: that atom feeds latent
// rows 64..127 of the dQ MMA, whose output lanes are never read. At M = 128
// there is room for one 64 KB stage only: S/dP of the next tile is then
// issued after this tile's dQ has released the stage (no early issue).
// Warp roles of bwd_tc_kernel: warp 0 TMA producer (K, V ring; Q, dZ and the
// row statistics on every (b, h) change), warp 1 TMEM allocator and MMA
// issuer (the converged warp, elect.sync picking the issuing lane: about 9%
// faster than issuing from one lane in a divergent branch), warps 2-9 two
// halves of four warps, each half owning M/2 latents of every token row (one
// token row per thread): the half's P (bf16
// into its half of P's TMEM columns) and s dS (bf16 into shared memory), then
// the previous tile's epilogue (half 0 stores dV, half 1 dK, one TMA store
// per warp of 32 rows) and, at the end of a (b, h) piece, half of the dQ
// partial's columns.
#pragma once

#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace flare {
namespace tc {

struct BwdArgs {
    int B, H, M, N;
    // latent rows [m0, m0 + M) of M_all: M = 256 runs as two passes of 128
    // latent rows (row statistics, Q, dZ and the dQ partials are indexed
    // with M_all rows per (b, h))
    int m0, M_all;
    float sl2;                  // s * log2(e)
    float s;                    // score scale
    int q_per_batch;            // Q has a batch dimension
    const uint8_t *mask;        // [B, N] or null
    const float *lc;            // [B*H][2][M]: -L log2(e) (or -inf), then -s c
    float *part;                // [B*H][P_max][M][64] dQ partials (of this pass's column half)
    int dh;                     // D = 128: the output column half [64 dh, 64 dh + 64)
    const __nv_bfloat16 *dk_acc;  // with ACC: dK = dk_acc + this share (dk_acc may be dK)
    const __nv_bfloat16 *dv_acc;  // with ACCV: dV = dv_acc + this share (dv_acc may be dV)
    int P_max;
    int64_t T_bh, T_total;      // 128-token tiles per (b, h), and overall
    int grid;
    unsigned *status;
};

// CTA whose span holds tile t (spans: begin(c) = ceil(c T / grid)).
__host__ __device__ __forceinline__ int bwd_cta_of(int64_t t, int64_t T_total, int grid) {
    return (int)((t * grid) / T_total);
}

template <int M_, int STAGES_, bool ACCV_ = false, int D_ = 64>
struct BwdCfg {
    static constexpr int M = M_, D = D_, TILE = 128, STAGES = STAGES_;
    static constexpr int DA = D / 64;                      // 64-column atoms of a row
    static constexpr int THREADS = 320;
    static constexpr uint32_t TILE_BYTES = TILE * 128;     // 128 rows x 64 bf16 (swizzled)
    static constexpr uint32_t QZA = M * 128;               // one [M][64] bf16 atom (swizzled)
    static constexpr uint32_t QZ_BYTES = DA * QZA;         // Q (or dZ): its atoms in column order
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t DZ_OFF = Q_OFF + QZ_BYTES;
    static constexpr uint32_t STAGE_OFF = DZ_OFF + QZ_BYTES;
    static constexpr uint32_t STAGE_BYTES = 2 * DA * TILE_BYTES; // K atoms, then V atoms
    // s dS^T in bf16: token rows of 64-latent atoms (atom a at a * TILE_BYTES)
    static constexpr uint32_t DS_OFF = STAGE_OFF + STAGES * STAGE_BYTES;
    static constexpr uint32_t DS_BYTES = 2 * TILE_BYTES;
    static constexpr uint32_t OUT_OFF = DS_OFF + DS_BYTES;  // dK tile, then dV tile
    static constexpr uint32_t OUT_BYTES = 2 * TILE_BYTES;
    // rows of the old dK being accumulated into (one 128-byte row per thread
    // of the dK half, 16-byte chunks XOR-swizzled by the row)
    // (D = 128 at M = 64: the upper atom of the s dS^T buffer)
    static constexpr bool DKIN_IN_DS = DA == 2 && M <= 64;
    static constexpr uint32_t DKIN_OFF = DKIN_IN_DS ? DS_OFF + TILE_BYTES : OUT_OFF + OUT_BYTES;
    static constexpr uint32_t DKIN_BYTES = DKIN_IN_DS ? 0 : TILE_BYTES;
    // the same for the old dV rows (ACCV: the second latent pass of M = 256)
    static constexpr uint32_t DVIN_OFF = OUT_OFF + OUT_BYTES + DKIN_BYTES;
    static constexpr uint32_t DVIN_BYTES = ACCV_ ? TILE_BYTES : 0;
    // row statistics of two (b, h) generations: [2][-L2 (M), -s c (M)]
    static constexpr uint32_t LC_OFF = DVIN_OFF + DVIN_BYTES;
    static constexpr uint32_t LC_BYTES = 2 * 2 * M * 4;
    static constexpr uint32_t BAR_OFF = LC_OFF + LC_BYTES;
    // full[S], empty[S], qd_full, qd_free, lc_full[2], s_full, p_full,
    // ds_free, dvdk_full, dvdk_free, dq_full, dq_free, drain, sdp_free
    static constexpr int NBAR = 2 * STAGES + 14;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t BYTES = MISC_OFF + 64;
    static constexpr uint32_t ALLOC = BYTES + 1024;
    static_assert(ALLOC <= 232448, "shared memory budget of one CTA exceeded");
    static_assert(QZ_BYTES % 1024 == 0, "operand tiles must stay 1 KB aligned");
    // tensor memory columns
    // (P^T of a tile in bf16 pairs at P_COL, so S/dP of the next tile can
    // overwrite S_COL/DP_COL while dV reads P)
    static constexpr uint32_t S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 320, DQ_COL = 384, P_COL = 448;
    static constexpr uint32_t TMEM_COLS = 512;
};

// ---- prologue: dZ in bf16 and the per-row constants -----------------------------
// One warp per latent row of D (64 or 128) columns, two per lane at a time.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const float *__restrict__ Z,
                                                       const float *__restrict__ L,
                                                       const float *__restrict__ dZ,
                                                       __nv_bfloat16 *__restrict__ dZb,
                                                       float *__restrict__ lc, int64_t rows, int M,
                                                       float s, int D) {
    const int lane = threadIdx.x & 31;
    const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (r >= rows) return;
    float c = 0.f;
    for (int k = lane; k < D / 2; k += 32) {
        const float2 z = reinterpret_cast<const float2 *>(Z + r * D)[k];
        const float2 g = reinterpret_cast<const float2 *>(dZ + r * D)[k];
        c = fmaf(z.x, g.x, c);
        c = fmaf(z.y, g.y, c);
        reinterpret_cast<uint32_t *>(dZb + r * D)[k] = pack_bf16(g.x, g.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) {
        const int64_t bh = r / M;
        const int m = (int)(r - bh * M);
        const float Lv = L[r];
        lc[bh * 2 * M + m] = (Lv == -INFINITY) ? -INFINITY : -Lv * 1.4426950408889634f;
        lc[bh * 2 * M + M + m] = -s * c;
    }
}

// ---- dQ = sum over the pieces of each (b, h) ------------------------------------
// The pieces of column half dh (D = 128: one piece array per pass) start at
// part + dh * half_stride floats; each holds [B*H][P_max][M][64].
__global__ void __launch_bounds__(256) bwd_dq_reduce_kernel(const float *__restrict__ part,
                                                            float *__restrict__ dQ, int64_t BH, int M,
                                                            int P_max, int64_t T_bh, int64_t T_total,
                                                            int grid, int accumulate, int D,
                                                            int64_t half_stride) {
    const int64_t per_bh = (int64_t)M * (D / 4);            // float4s of one (b, h)
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BH * per_bh) return;
    const int64_t bh = i / per_bh, rem = i - bh * per_bh;
    const int64_t m = rem / (D / 4);
    const int c4 = (int)(rem - m * (D / 4));
    const int c0 = bwd_cta_of(bh * T_bh, T_total, grid);
    const int np = bwd_cta_of(bh * T_bh + T_bh - 1, T_total, grid) - c0 + 1;
    const float4 *src = reinterpret_cast<const float4 *>(part + (c4 >> 4) * half_stride) +
                        (bh * P_max * M + m) * 16 + (c4 & 15);
    float4 acc = accumulate ? reinterpret_cast<const float4 *>(dQ)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = 0; p < np; ++p) {
        const float4 v = __ldcg(src + (int64_t)p * M * 16);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    reinterpret_cast<float4 *>(dQ)[i] = acc;
}

// ---- the tile kernel -------------------------------------------------------------
template <int M, int STAGES, bool ACC, bool ACCV = false, int D = 64>
__global__ void __launch_bounds__(BwdCfg<M, STAGES, ACCV, D>::THREADS, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdZ,
              const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
              const BwdArgs a) {
    using C = BwdCfg<M, STAGES, ACCV, D>;
    constexpr uint32_t TB = C::TILE_BYTES;
    constexpr int DA = C::DA;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::Q_OFF, sdZ = sbase + C::DZ_OFF, sStage = sbase + C::STAGE_OFF;
    const uint32_t sDS = sbase + C::DS_OFF, sOut = sbase + C::OUT_OFF;
    const uint32_t bar0 = sbase + C::BAR_OFF;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t qd_full = bar0 + 8u * (2 * STAGES), qd_free = qd_full + 8;
    auto lc_full = [&](int p) { return bar0 + 8u * (2 * STAGES + 2 + p); };
    const uint32_t s_full = bar0 + 8u * (2 * STAGES + 4), p_full = s_full + 8, ds_free = s_full + 16;
    const uint32_t dvdk_full = s_full + 24, dvdk_free = s_full + 32;
    const uint32_t dq_full = s_full + 40, dq_free = s_full + 48, drain = s_full + 56;
    const uint32_t sdp_free = s_full + 64;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    float *lcs = reinterpret_cast<float *>(smem + C::LC_OFF);

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
        mbar_init(qd_full, 1);
        mbar_init(qd_free, 1);
        mbar_init(lc_full(0), 1);
        mbar_init(lc_full(1), 1);
        mbar_init(s_full, 1);
        mbar_init(p_full, 8);          // one arrival per softmax warp
        mbar_init(ds_free, 1);
        mbar_init(dvdk_full, 1);
        mbar_init(dvdk_free, 8);       // one arrival per softmax/epilogue warp
        mbar_init(dq_full, 1);
        mbar_init(dq_free, 8);
        mbar_init(drain, 1);
        mbar_init(sdp_free, 8);        // every softmax warp has read S and dP of the tile
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmdZ);
        prefetch_tmap(&tmdK);
        prefetch_tmap(&tmdV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (M < 128 && warp >= 2) {
        // latents M..127 of dS^T stay zero: the dQ MMA always spans 128 rows
        for (int q = threadIdx.x - 64; q < (int)TB / 16; q += 256)
            reinterpret_cast<uint4 *>(smem + C::DS_OFF + TB)[q] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

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
                // Q, dZ and the statistics of the previous (b, h) are no longer read
                if (u > 0 && !__all_sync(0xffffffffu, wt.wait_inline(qd_free, (uint32_t)(u - 1) & 1))) break;
                float *dst = lcs + (u & 1) * 2 * M;
                const float *src = a.lc + bh * 2 * a.M_all + a.m0;
                for (int i = lane; i < 2 * M; i += 32) dst[i] = src[(i / M) * a.M_all + (i % M)];
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(lc_full(u & 1));
                    mbar_arrive_expect_tx(qd_full, 2 * C::QZ_BYTES);
                    if (dcheck(h >= 0 && h < a.H && b >= 0 && b < a.B, kChkBwdQ, a.status)) {
#pragma unroll
                        for (int at = 0; at < DA; ++at) {
                            tma_load_4d(sQ + at * C::QZA, &tmQ, 64 * at, a.m0, h, a.q_per_batch ? b : 0, qd_full);
                            tma_load_4d(sdZ + at * C::QZA, &tmdZ, 64 * at, a.m0, h, b, qd_full);
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
                if (dcheck(tile_in_tensor(0, h, kt * 128, b, a.H, a.N, a.B) && kt < a.T_bh, kChkBwdKV, a.status)) {
#pragma unroll
                    for (int at = 0; at < DA; ++at) {
                        tma_load_4d_hint(dst + at * TB, &tmK, 64 * at, h, (int)(kt * 128), b, full(s), pol);
                        tma_load_4d_hint(dst + (DA + at) * TB, &tmV, 64 * at, h, (int)(kt * 128), b, full(s), pol);
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
                while (!mbar_try_wait(qd_full, (uint32_t)u & 1) && globaltimer() - t0 < 500000000ull) {
                }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (converged warp, elect.sync issues) ----------------
        {
            constexpr uint32_t idS = idesc_bf16(128, M, 0, 0);
            constexpr uint32_t idG = idesc_bf16(128, 64, 0, 1);    // dV, dK: A in TMEM, B MN-major
            constexpr uint32_t idQ = idesc_bf16(128, 64, 1, 1);    // dQ: A, B MN-major
            const uint64_t dQk = desc_sw128(sQ, 16, 1024);          // Q, K-major (B of S^T)
            const uint64_t dZk = desc_sw128(sdZ, 16, 1024);         // dZ, K-major (B of dP^T)
            // the output column half's atoms of Q and dZ
            const uint64_t dQm = desc_sw128(sQ + a.dh * C::QZA, TB, 1024);   // Q, MN-major (B of dK)
            const uint64_t dZm = desc_sw128(sdZ + a.dh * C::QZA, TB, 1024);  // dZ, MN-major (B of dV)
            const uint64_t dDS = desc_sw128(sDS, TB, 1024);         // s dS^T, MN-major (A of dQ)
            const uint64_t dDSk = desc_sw128(sDS, 16, 1024);        // s dS^T, K-major (A of dK)
            int64_t bhS = bh0, ktS = k0, curS = -1;                  // cursor of the S tiles
            int uS = -1;
            bool ok = true;
            auto issue_sdp = [&](int64_t jj) -> bool {
                if (bhS != curS) {
                    ++uS;
                    curS = bhS;
                    if (!__all_sync(0xffffffffu, wt.wait_inline(qd_full, (uint32_t)uS & 1))) return false;
                }
                const int s = (int)(jj % STAGES);
                if (!__all_sync(0xffffffffu, wt.wait_inline(full(s), (uint32_t)(jj / STAGES) & 1))) return false;
                tc_fence_after();
                const uint64_t dK = desc_sw128(sStage + s * C::STAGE_BYTES, 16, 1024);
                const uint64_t dV = desc_sw128(sStage + s * C::STAGE_BYTES + DA * TB, 16, 1024);
                // over all D columns: 16 per MMA, four per atom
#pragma unroll
                for (int kb = 0; kb < 4 * DA; ++kb) {
                    umma_ss_elect(tmem + C::S_COL, dK + (((kb >> 2) * TB) >> 4) + 2 * (kb & 3),
                                 dQk + (((kb >> 2) * C::QZA) >> 4) + 2 * (kb & 3), idS, kb > 0 ? 1u : 0u);
                    umma_ss_elect(tmem + C::DP_COL, dV + (((kb >> 2) * TB) >> 4) + 2 * (kb & 3),
                                 dZk + (((kb >> 2) * C::QZA) >> 4) + 2 * (kb & 3), idS, kb > 0 ? 1u : 0u);
                }
                umma_commit_elect(s_full);
                if (++ktS == a.T_bh) {
                    ktS = 0;
                    ++bhS;
                }
                return true;
            };
            int64_t bhP = bh0, ktP = k0;                             // cursor of the gradient tiles
            int uP = 0;                                              // piece of the current tile
            if (ntiles > 0) ok = issue_sdp(0);
            for (int64_t j = 0; j < ntiles && ok; ++j) {
                const bool first = (j == 0) || ktP == 0;
                int64_t bhN = bhP, ktN = ktP + 1;
                if (ktN == a.T_bh) {
                    ktN = 0;
                    ++bhN;
                }
                const bool last = (j + 1 == ntiles) || bhN != bhP;
                // tile j + 1 of the same (b, h): its S/dP as soon as S/dP of tile j is read
                // (one K/V stage: the next tile's load waits for this tile's dQ)
                const bool early = STAGES > 1 && j + 1 < ntiles && !last;
                if (early) {
                    if (!(ok = __all_sync(0xffffffffu, wt.wait_inline(sdp_free, (uint32_t)j & 1)))) break;
                    if (!(ok = issue_sdp(j + 1))) break;
                }
                if (!(ok = __all_sync(0xffffffffu, wt.wait_inline(p_full, (uint32_t)j & 1)))) break;
                tc_fence_after();
                if (j > 0 && !(ok = __all_sync(0xffffffffu, wt.wait_inline(dvdk_free, (uint32_t)(j - 1) & 1)))) break;
                tc_fence_after();
                // dV = P^T dZ (A = P^T from tensor memory), dK = (s dS)^T Q (A = dS^T
                // from shared memory): K = M latents, 16 per MMA
#pragma unroll
                for (int kb = 0; kb < M / 16; ++kb) {
                    umma_ts_elect(tmem + C::DV_COL, tmem + C::P_COL + 8 * kb, dZm + kb * (2048 >> 4), idG,
                                 kb > 0 ? 1u : 0u);
                    umma_ss_elect(tmem + C::DK_COL, dDSk + (uint64_t)(((kb >> 2) * TB + (kb & 3) * 32) >> 4),
                                 dQm + kb * (2048 >> 4), idG, kb > 0 ? 1u : 0u);
                }
                umma_commit_elect(dvdk_full);
                if (last) umma_commit_elect(qd_free);
                // a tile of the next (b, h): its Q and dZ arrive once qd_free fired
                if (STAGES > 1 && j + 1 < ntiles && !early && !(ok = issue_sdp(j + 1))) break;
                // dQ += (s dS) K over the tile's 128 tokens, 16 per MMA
                if (first && uP > 0 && !(ok = __all_sync(0xffffffffu, wt.wait_inline(dq_free, (uint32_t)(uP - 1) & 1)))) break;
                tc_fence_after();
                const int s = (int)(j % STAGES);
                const uint64_t dKm = desc_sw128(sStage + s * C::STAGE_BYTES + a.dh * TB, TB, 1024);
#pragma unroll
                for (int kb = 0; kb < 8; ++kb)
                    umma_ss_elect(tmem + C::DQ_COL, dDS + kb * (2048 >> 4), dKm + kb * (2048 >> 4), idQ,
                                 (kb > 0 || !first) ? 1u : 0u);
                umma_commit_elect(ds_free);
                umma_commit_elect(empty(s));
                if (last) {
                    umma_commit_elect(dq_full);
                    ++uP;
                }
                // one stage: S/dP of the next tile once this tile's dQ has released it
                if (STAGES == 1 && j + 1 < ntiles && !(ok = issue_sdp(j + 1))) break;
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
    } else {
        // ---------------- softmax halves + deferred epilogue (warps 2-9) ----------------
        // Per tile j: S and dP loaded (then sdp_free, so S/dP of tile j + 1 can
        // be computed), P into P_COL once dV of tile j - 1 is done, s dS^T into
        // shared memory once dK and dQ of tile j - 1 are done, p_full; then the
        // epilogue of tile j - 1, whose dV, dK were computed meanwhile.
        constexpr int W = M / 2;                              // latents of each half
        const int hf = (warp - 2) >> 2;                       // latent half
        const int quad = warp & 3;
        const int rig = quad * 32 + lane;                     // token row within the tile
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t s_tm = tmem + C::S_COL + W * hf + lane_off;
        const uint32_t dp_tm = tmem + C::DP_COL + W * hf + lane_off;
        const uint32_t p_tm = tmem + C::P_COL + (W / 2) * hf + lane_off;   // this half's P^T (bf16 pairs)
        const uint64_t c2 = f2pack(a.sl2, a.sl2), sc2 = f2pack(a.s, a.s);
        // this warp's 32-row slab of the dV (half 0) or dK (half 1) staging tile
        uint8_t *slab = smem + C::OUT_OFF + (hf * 4 + quad) * (32 * 128);
        const CUtensorMap *tmOut = hf ? &tmdK : &tmdV;
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait_inline(bar, par));
        };
        // The mask byte of this thread's token is loaded two tiles ahead and
        // only compared when its tile comes up, so the load's latency is never
        // waited for (0 stands for padding and for tokens past N).
        // a tile cursor: (b, h) index bh = b * H + h, token tile kt; no divisions per tile
        struct Cursor {
            int64_t bh, kt;
            int b, h;
        };
        auto advance = [&](Cursor &t) {
            if (++t.kt == a.T_bh) {
                t.kt = 0;
                ++t.bh;
                if (++t.h == a.H) {
                    t.h = 0;
                    ++t.b;
                }
            }
        };
        auto mask_byte = [&](const Cursor &t) -> uint32_t {
            const int64_t n = t.kt * 128 + rig;
            uint32_t v = n < a.N ? 1u : 0u;
            if (a.mask != nullptr && n < a.N) v = __ldg(a.mask + (int64_t)t.b * a.N + n);
            return v;
        };
        // Accumulation into this half's output (dK for half 1 with ACC, dV for
        // half 0 with ACCV): the old rows of tile t (this thread's row; read by
        // this thread only, in the tile's epilogue)
        constexpr bool kAccAny = ACC || ACCV;
        const bool acc_mine = hf == 1 ? ACC : ACCV;
        const __nv_bfloat16 *acc_src = hf == 1 ? a.dk_acc : a.dv_acc;
        const uint32_t acc_buf = hf == 1 ? C::DKIN_OFF : C::DVIN_OFF;
        auto prefetch_dk = [&](const Cursor &t) {
            const int64_t n = t.kt * 128 + rig;
            if (acc_mine && n < a.N) {
                const __nv_bfloat16 *src = acc_src + (((int64_t)t.b * a.N + n) * a.H + t.h) * D + 64 * a.dh;
                const uint32_t dst = sbase + acc_buf + (uint32_t)rig * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) cp_async16(dst + ((c ^ (rig & 7)) << 4), src + 8 * c);
                cp_async_commit();
            }
        };
        int pieces = 0;
        // Epilogue of tile jp (cursor t): half 0 stores dV, half 1 dK of the
        // warp's 32 token rows; at the end of a (b, h) piece, half hf writes
        // columns [32 hf, 32 hf + 32) of the piece's dQ partial. `nxt`: the tile
        // whose epilogue comes next (its old dK rows are prefetched), or null.
        auto epilogue = [&](int64_t jp, const Cursor &t, bool lastp, const Cursor *nxt) -> bool {
            if (!wwait(dvdk_full, (uint32_t)jp & 1)) return false;
            tc_fence_after();
            const uint32_t out_tm = tmem + (hf ? C::DK_COL : C::DV_COL) + lane_off;
            uint8_t *srow = slab + lane * 128;
            // 32 fp32 columns [32 h2, 32 h2 + 32) of the row into the slab as bf16;
            // with `old`, the old dK row's bf16 values are added first
            auto pack32 = [&](const uint32_t *g, int h2, bool old) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int chunk = 4 * h2 + q;
                    float f[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) f[k] = __uint_as_float(g[8 * q + k]);
                    if (old) {
                        // bf16 pairs, the even column in the low half
                        const uint4 o = *reinterpret_cast<const uint4 *>(smem + acc_buf + rig * 128 +
                                                                          ((chunk ^ (rig & 7)) << 4));
                        const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            f[2 * k] += __uint_as_float(ow[k] << 16);
                            f[2 * k + 1] += __uint_as_float(ow[k] & 0xffff0000u);
                        }
                    }
                    *reinterpret_cast<uint4 *>(srow + ((chunk ^ (lane & 7)) << 4)) =
                        make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                                   pack_bf16(f[6], f[7]));
                }
            };
            // the slab is free once the warp's previous store has read it
            if (jp > 0) {
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
            }
            if constexpr (!kAccAny) {
                uint32_t rg[2][32];
                tmem_ld32(out_tm, rg[0]);
                tmem_ld32(out_tm + 32, rg[1]);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dvdk_free);
                pack32(rg[0], 0, false);
                pack32(rg[1], 1, false);
            } else {
                // one 32-column half at a time (fewer live registers); TMEM is
                // released after the second half
                const bool acc_row = acc_mine && t.kt * 128 + rig < a.N;
                if (acc_row) cp_async_wait0();
#pragma unroll 1
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t rg[32];
                    tmem_ld32(out_tm + 32 * h2, rg);
                    tmem_wait_ld();
                    if (h2 == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(dvdk_free);
                    }
                    pack32(rg, h2, acc_row);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            const int n0 = (int)(t.kt * 128) + quad * 32;
            if (lane == 0 && n0 < a.N &&
                dcheck(tile_in_tensor(64 * a.dh, t.h, n0, t.b, a.H, a.N, a.B), kChkBwdOut, a.status)) {
                // rows past N are clipped by the tensor map
                tma_store_4d(tmOut, smem_u32(slab), 64 * a.dh, t.h, n0, t.b);
                bulk_commit_group();
            }
            if (nxt != nullptr) prefetch_dk(*nxt);
            if (lastp) {
                // the (b, h)'s dQ partial of this span: latent rows in the
                // lanes, half hf takes columns [32 hf, 32 hf + 32)
                if (!wwait(dq_full, (uint32_t)pieces & 1)) return false;
                tc_fence_after();
                uint32_t rq[32];
                tmem_ld32(tmem + C::DQ_COL + 32 * hf + lane_off, rq);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dq_free);
                if (rig < M) {
                    const int piece = cta - bwd_cta_of(t.bh * a.T_bh, a.T_total, a.grid);
                    float4 *dst = reinterpret_cast<float4 *>(
                        a.part + ((t.bh * a.P_max + piece) * a.M_all + a.m0 + rig) * 64 + 32 * hf);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_float4(__uint_as_float(rq[4 * q]), __uint_as_float(rq[4 * q + 1]),
                                             __uint_as_float(rq[4 * q + 2]), __uint_as_float(rq[4 * q + 3]));
                }
                ++pieces;
            }
            return true;
        };
        Cursor cu{bh0, k0, (int)(bh0 / a.H), (int)(bh0 - (bh0 / a.H) * a.H)};
        int64_t cur = -1;
        int u = -1;
        Cursor ca = cu;                                           // tile j + 2
        uint32_t mb0 = 0, mb1 = 0;                                // mask bytes of tiles j, j + 1
        if (ntiles > 0) {
            mb0 = mask_byte(ca);
            prefetch_dk(ca);
        }
        advance(ca);
        if (ntiles > 1) mb1 = mask_byte(ca);
        advance(ca);
        Cursor pv = cu;                                           // the previous tile
        bool pv_last = false;
        bool ok = true;
        for (int64_t j = 0; j < ntiles; ++j) {
            const int64_t bh = cu.bh;
            if (bh != cur) {
                ++u;
                cur = bh;
                if (!(ok = wwait(lc_full(u & 1), (uint32_t)(u >> 1) & 1))) break;
            }
            Cursor cn = cu;
            advance(cn);
            const bool last = (j + 1 == ntiles) || cn.bh != bh;
            const float *nl2 = lcs + (u & 1) * 2 * M, *ncs = nl2 + M;
            const bool valid = mb0 != 0;
            mb0 = mb1;
            mb1 = j + 2 < ntiles ? mask_byte(ca) : 0u;
            advance(ca);
            if (!(ok = wwait(s_full, (uint32_t)j & 1))) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < W / 32; ++c) {
                uint32_t rs[32], rp[32];
                tmem_ld32(s_tm + 32 * c, rs);
                tmem_ld32(dp_tm + 32 * c, rp);
                tmem_wait_ld();
                if (c == W / 32 - 1) {
                    // S and dP of this tile are in registers: the next tile's may be computed
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sdp_free);
                }
                uint32_t pw[16], dw[16];
                const int m0 = W * hf + 32 * c;                   // first latent of the chunk
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int m = m0 + 2 * i;
                        const uint64_t nl = *reinterpret_cast<const uint64_t *>(nl2 + m);
                        const uint64_t nc = *reinterpret_cast<const uint64_t *>(ncs + m);
                        float t0, t1;
                        f2unpack(fma2(f2pack(__uint_as_float(rs[2 * i]), __uint_as_float(rs[2 * i + 1])), c2, nl),
                                 t0, t1);
                        const uint64_t p2 = f2pack(ex2(t0), ex2(t1));
                        const uint64_t g2 =
                            fma2(f2pack(__uint_as_float(rp[2 * i]), __uint_as_float(rp[2 * i + 1])), sc2, nc);
                        float p0, p1, d0, d1;
                        f2unpack(p2, p0, p1);
                        f2unpack(mul2(p2, g2), d0, d1);
                        pw[i] = pack_bf16(p0, p1);
                        dw[i] = pack_bf16(d0, d1);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) pw[i] = dw[i] = 0u;
                }
                // P^T into P_COL once dV of the previous tile (which read it) is done
                if (c == 0 && j > 0 && !(ok = wwait(dvdk_full, (uint32_t)(j - 1) & 1))) break;
                tmem_st16(p_tm + 16 * c, pw);
                // the previous tile's dK and dQ MMAs have read the shared dS buffer
                if (c == 0 && j > 0 && !(ok = wwait(ds_free, (uint32_t)(j - 1) & 1))) break;
                // s dS^T row: the K-major A of dK and the MN-major A of dQ
                uint8_t *row = smem + C::DS_OFF + (m0 >> 6) * TB + rig * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int chunk = ((m0 & 63) >> 3) + q;
                    *reinterpret_cast<uint4 *>(row + ((chunk ^ (rig & 7)) << 4)) =
                        make_uint4(dw[4 * q], dw[4 * q + 1], dw[4 * q + 2], dw[4 * q + 3]);
                }
            }
            if (!ok) break;
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            // the previous tile's epilogue (its dV, dK were computed meanwhile)
            if (j > 0 && !(ok = epilogue(j - 1, pv, pv_last, &cu))) break;
            pv = cu;
            pv_last = last;
            cu = cn;
        }
        if (ok && ntiles > 0) epilogue(ntiles - 1, pv, pv_last, nullptr);
        if (lane == 0) bulk_wait_group0();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace tc
}  // namespace flare
