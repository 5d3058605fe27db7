// tc_encoder.cuh -- split-KV FLARE encoder on sm_103a tensor cores.
//
// Computes, for every (b, h) and shard r, the pages' local primitive: O_r =
// softmax(s Q K_r^T) V_r normalised over shard r and its row log-normaliser
// L_r, then merges shards by eq. 23 (cross-rank log-sum-exp) into Z and L
// ("FLARE++: Low-rank attention with dynamic attention routing", appendix on
// context parallelism: the per-shard encoder, eq. 23 and the cross-rank
// log-sum-exp paragraph). Scores are never written to memory.
//
// One persistent CTA per SM walks a contiguous span of 128-token tiles (see
// TcTilePlan). Warp roles:
//   warp 0     TMA producer: Q of the current (b, h) and K/V tiles into a
//              STAGES-deep ring (L2 evict-first); the tile's padding mask,
//              prefetched one tile ahead, becomes an additive bias (0 / -inf).
//   warp 1     TMEM allocator; lane 0 issues every tcgen05.mma from a polling
//              loop so score MMAs run ahead of the softmax:
//                S_g = Q K^T            (A, B from shared memory)
//                O_g += P_g V           (A = P from tensor memory, B = V smem)
//   warps 2-9  two softmax groups of four warps, one latent row per thread
//              (= TMEM lane). With M <= 128 the groups take alternate tiles
//              (two tiles in flight, each group with its own running max, sum
//              and output accumulator, combined when a piece ends); with
//              M = 256 each group owns 128 rows of every tile.
// Softmax: log2 domain, scale folded into one FFMA with the mask bias, lazy
// rescale (O and l are rescaled only when the row maximum grows by more than
// kTau), P rounded to bf16 and written over S in tensor memory.
// At the end of each (b, h, shard) piece of its span a CTA writes a partial
// (normalised output, log-normaliser); the CTA that completes the last piece
// of a (b, h) (atomic ticket, nobody waits) merges them: pieces into shards
// (O_r, L_r), shards into (Z, L), in fixed order.
#pragma once

#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace flare {
namespace tc {

constexpr float kTau = 8.0f;           // lazy-rescale threshold (log2 units)
constexpr int kMergePieces = 512;      // pieces of one (b, h) the fast merge handles
constexpr int kMergeRB = 8;            // shards per block of the row reduction
constexpr int kMergePB = 8;            // pieces per block of the output sum
constexpr uint32_t kAtom = 128 * 128;  // bytes of one 128-row x 128-byte swizzle column

struct EncArgs {
    int B, H, M, N;
    float sl2;                 // score scale * log2(e)
    int q_per_batch;           // Q has a batch dimension
    const uint8_t *mask;
    unsigned *tickets;
    float *part_L, *part_O, *shard_L;
    float *O_r, *L_r, *Z, *L;
    unsigned *status;
    TcTilePlan plan;
};

struct TileInfo {
    int bh, r, k, nt;
    int64_t n0, n1;
};

__device__ __forceinline__ TileInfo decompose(const TcTilePlan &p, int64_t t) {
    TileInfo ti;
    ti.bh = (int)(t / p.T_bh);
    const int w = (int)(t - (int64_t)ti.bh * p.T_bh);
    int lo = 0, hi = p.R - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.tile_start[mid] <= w) lo = mid; else hi = mid - 1;
    }
    ti.r = lo;
    ti.k = w - p.tile_start[lo];
    ti.nt = p.tile_start[lo + 1] - p.tile_start[lo];
    ti.n0 = p.off[lo] + (int64_t)ti.k * 128;
    ti.n1 = min(ti.n0 + 128, p.off[lo + 1]);
    return ti;
}

// CTA whose span holds tile t; first tile of CTA c's span.
__device__ __forceinline__ int cta_of(const TcTilePlan &p, int64_t t) {
    return (int)((t * p.grid) / p.T_total);
}
__device__ __forceinline__ int64_t span_begin(const TcTilePlan &p, int c) {
    return ((int64_t)c * p.T_total + p.grid - 1) / p.grid;
}

// Walks the tiles of a span in order without divisions: (b*H+h, shard, tile).
struct TileCursor {
    int bh, r, k, nt;
    int64_t n0, n1, shard_end;
    __device__ __forceinline__ void init(const TcTilePlan &p, int64_t t) {
        const TileInfo ti = decompose(p, t);
        bh = ti.bh;
        r = ti.r;
        k = ti.k;
        nt = ti.nt;
        n0 = ti.n0;
        n1 = ti.n1;
        shard_end = p.off[r + 1];
    }
    __device__ __forceinline__ void next(const TcTilePlan &p) {
        if (++k < nt) {
            n0 += 128;
            n1 = min(n0 + 128, shard_end);
            return;
        }
        do {
            if (++r == p.R) {
                r = 0;
                ++bh;
            }
        } while (p.tile_start[r + 1] == p.tile_start[r]);
        k = 0;
        nt = p.tile_start[r + 1] - p.tile_start[r];
        n0 = p.off[r];
        shard_end = p.off[r + 1];
        n1 = min(n0 + 128, shard_end);
    }
};

template <int D, bool HALVES, int STAGES>
struct EncCfg {
    static constexpr int KA = D / 64;                 // 64-element atoms along D
    static constexpr int NSOFT = 256;                 // two groups of 128 threads
    static constexpr int THREADS = 64 + NSOFT;
    static constexpr int QBLK = HALVES ? 2 : 1;       // 128-row blocks of Q
    static constexpr int PERIOD = HALVES ? 1 : 2;     // tiles between two uses of a group
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t STAGE_OFF = Q_OFF + QBLK * KA * kAtom;
    static constexpr uint32_t STAGE_BYTES = 2 * KA * kAtom;   // K atoms then V atoms
    static constexpr uint32_t BIAS_OFF = STAGE_OFF + STAGES * STAGE_BYTES;
    static constexpr uint32_t BAR_OFF = BIAS_OFF + STAGES * 128 * 4;
    // full[S], empty[S], q_full, q_free, s_full[2], p_chunk[2][4], o_done[2], soft
    static constexpr int NBAR = 2 * STAGES + 2 + 2 + 8 + 2 + 1;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t STAT_OFF = MISC_OFF + 64;       // [2 groups][128 rows] (m, l)
    // merge scratch: row max/sum [2][256], piece prefix [kMaxShards+2], piece
    // slot and shard [2][kMergePieces], shard block [kMergeRB][256], piece weights [kMergePB][256]
    static constexpr uint32_t MERGE_OFF = STAT_OFF + 2 * 128 * 8;
    static constexpr uint32_t MERGE_BYTES = 2 * 256 * 4 + (kMaxShards + 2) * 4 + 2 * kMergePieces * 4 +
                                            kMergeRB * 256 * 4 + kMergePB * 256 * 4;
    static constexpr uint32_t BYTES = MERGE_OFF + MERGE_BYTES;
    static constexpr uint32_t ALLOC = BYTES + 1024;           // room to align the base to 1 KB
    static_assert(ALLOC <= 232448, "shared memory budget of one CTA exceeded");
    static constexpr uint32_t TMEM_COLS = 512;                 // group g: S/P at 256g, O at 256g+128
};

template <int D, bool HALVES, int STAGES>
__global__ void __launch_bounds__(EncCfg<D, HALVES, STAGES>::THREADS, 1)
enc_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmQ, const EncArgs a) {
    using C = EncCfg<D, HALVES, STAGES>;
    constexpr int KA = C::KA;
    constexpr int NSOFT = C::NSOFT;
    constexpr int PERIOD = C::PERIOD;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::Q_OFF, sStage = sbase + C::STAGE_OFF;
    float *bias = reinterpret_cast<float *>(smem + C::BIAS_OFF);
    const uint32_t bar0 = sbase + C::BAR_OFF;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t q_full = bar0 + 8u * (2 * STAGES), q_free = q_full + 8;
    auto s_full = [&](int g) { return bar0 + 8u * (2 * STAGES + 2 + g); };
    // P of a tile is published in four chunks of 32 tokens (16 TMEM columns)
    auto p_chunk = [&](int g, int c) { return bar0 + 8u * (2 * STAGES + 4 + 4 * g + c); };
    auto o_done = [&](int g) { return bar0 + 8u * (2 * STAGES + 12 + g); };
    const uint32_t soft = bar0 + 8u * (2 * STAGES + 14);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    volatile int *last_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 8);
    float2 *stat = reinterpret_cast<float2 *>(smem + C::STAT_OFF);
    float *s_lmax = reinterpret_cast<float *>(smem + C::MERGE_OFF);
    float *s_asum = s_lmax + 256;
    int *s_pstart = reinterpret_cast<int *>(s_asum + 256);          // [R + 1] piece prefix
    int *s_pslot = s_pstart + kMaxShards + 2;                        // [P] slot of each piece
    int *s_pshard = s_pslot + kMergePieces;                          // [P] shard of each piece
    float *s_blk = reinterpret_cast<float *>(s_pshard + kMergePieces);   // [kMergeRB][M]
    float *s_w = s_blk + kMergeRB * 256;                             // [kMergePB][M]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TcTilePlan &pl = a.plan;
    const int cta = blockIdx.x;
    const int64_t tb = span_begin(pl, cta), te = span_begin(pl, cta + 1);
    const int64_t ntiles = te - tb;
    Waiter wt{abort_flag, a.status};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        *last_flag = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_free, 1);
        for (int g = 0; g < 2; ++g) {
            mbar_init(s_full(g), 1);
            for (int c = 0; c < 4; ++c) mbar_init(p_chunk(g, c), 128);
            mbar_init(o_done(g), 1);
        }
        mbar_init(soft, NSOFT);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmQ);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp >= 2 && a.M < 128) {
        // rows M..127 of the query tile stay zero (only M rows are loaded)
        for (int i = threadIdx.x - 64; i < KA * (int)kAtom / 16; i += NSOFT) {
            const int row = (i * 16 % (int)kAtom) / 128;
            if (row >= a.M) reinterpret_cast<uint4 *>(smem + C::Q_OFF)[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        const uint64_t pol = policy_evict_first();
        int cur_bh = -1;
        uint32_t q_uses = 0;
        // mask bytes of the next tile are loaded one iteration ahead
        auto load_mask = [&](const TileCursor &ti, uint8_t (&mb)[4]) {
            const int b = ti.bh / a.H;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t n = ti.n0 + lane + 32 * i;
                mb[i] = (n < ti.n1) ? (a.mask ? a.mask[(int64_t)b * a.N + n] : (uint8_t)1) : (uint8_t)0;
            }
        };
        uint8_t mb[4] = {0, 0, 0, 0}, mb_next[4] = {0, 0, 0, 0};
        TileCursor ti, tn;
        ti.init(pl, tb);
        tn = ti;
        load_mask(ti, mb);
        int64_t j = 0;
        for (; j < ntiles && !wt.aborted(); ++j) {
            if (j + 1 < ntiles) {
                tn.next(pl);
                load_mask(tn, mb_next);
            }
            const int b = ti.bh / a.H, h = ti.bh - b * a.H;
            if (ti.bh != cur_bh) {
                if (q_uses > 0 && !__all_sync(0xffffffffu, wt.wait(q_free, (q_uses - 1) & 1))) break;
                if (lane == 0) {
                    const int rows = a.M < 128 ? a.M : 128;
                    mbar_arrive_expect_tx(q_full, C::QBLK * KA * rows * 128);
                    const int qb = a.q_per_batch ? b : 0;
                    for (int blk = 0; blk < C::QBLK; ++blk)
                        for (int ka = 0; ka < KA; ++ka)
                            tma_load_4d(sQ + (blk * KA + ka) * kAtom, &tmQ, 64 * ka, 128 * blk, h, qb, q_full);
                }
                ++q_uses;
                cur_bh = ti.bh;
            }
            const int s = (int)(j % STAGES);
            if (!__all_sync(0xffffffffu, wt.wait(empty(s), ((uint32_t)(j / STAGES) & 1) ^ 1))) break;
            float *bs = bias + s * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i) bs[lane + 32 * i] = mb[i] ? 0.f : -INFINITY;
            __threadfence_block();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(full(s), C::STAGE_BYTES);
                const uint32_t dst = sStage + s * C::STAGE_BYTES;
                for (int ka = 0; ka < KA; ++ka) {
                    tma_load_4d_hint(dst + ka * kAtom, &tmK, 64 * ka, h, (int)ti.n0, b, full(s), pol);
                    tma_load_4d_hint(dst + (KA + ka) * kAtom, &tmV, 64 * ka, h, (int)ti.n0, b, full(s), pol);
                }
            }
            __syncwarp();
            ti = tn;
#pragma unroll
            for (int i = 0; i < 4; ++i) mb[i] = mb_next[i];
        }
        // after an abort: let every issued load land before the CTA exits
        if (wt.aborted() && lane == 0) {
            const uint64_t t0 = globaltimer();
            for (int64_t jj = (j > STAGES ? j - STAGES : 0); jj < j; ++jj)
                while (!mbar_try_wait(full((int)(jj % STAGES)), (uint32_t)(jj / STAGES) & 1) &&
                       globaltimer() - t0 < 500000000ull) {
                }
            if (q_uses > 0)
                while (!mbar_try_wait(q_full, (q_uses - 1) & 1) && globaltimer() - t0 < 500000000ull) {
                }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // Order: S_0 .. S_{PERIOD-1}, then for every tile j: PV_j as soon as its
        // P is written, then S_{j+PERIOD} (into the S/P columns PV_j has just
        // been queued to read: tcgen05 MMAs of one thread execute in order).
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_m128(128, 0);
            constexpr uint32_t idPV = idesc_bf16_m128(D, 1);
            constexpr int NG = HALVES ? 2 : 1;   // groups served per tile
            // descriptors at offset 0; k-blocks advance the start-address field
            const uint64_t dQ0 = desc_sw128(sQ, 16, 1024);
            const uint64_t dK0 = desc_sw128(sStage, 16, 1024);
            const uint64_t dV0 = desc_sw128(sStage + KA * kAtom, kAtom, 1024);
            constexpr uint64_t kStageDesc = C::STAGE_BYTES >> 4;
            int cur_bh = -1;
            uint32_t q_uses = 0;
            bool ok = true;
            TileCursor cs, cp;                    // cursors of the S and the PV tiles
            cs.init(pl, tb);
            cp = cs;
            auto issue_s = [&](int64_t jj) -> bool {
                const int s = (int)(jj % STAGES);
                if (cs.bh != cur_bh) {
                    if (!wt.wait(q_full, q_uses & 1)) return false;
                    ++q_uses;
                    cur_bh = cs.bh;
                }
                if (!wt.wait(full(s), (uint32_t)(jj / STAGES) & 1)) return false;
                tc_fence_after();
                const int g0 = HALVES ? 0 : (int)(jj & 1);
                const uint64_t dK = dK0 + kStageDesc * s;
#pragma unroll
                for (int gg = 0; gg < NG; ++gg) {
                    const int g = g0 + gg;
                    const uint64_t dQ = dQ0 + (HALVES ? (uint64_t)(gg * KA * kAtom) >> 4 : 0);
#pragma unroll
                    for (int kb = 0; kb < D / 16; ++kb) {
                        const uint64_t off = (uint64_t)((kb >> 2) * kAtom + (kb & 3) * 32) >> 4;
                        umma_bf16_ss(tmem + g * 256, dQ + off, dK + off, idS, kb > 0 ? 1u : 0u);
                    }
                    umma_commit(s_full(g));
                }
                const int bh_now = cs.bh;
                if (jj + 1 < ntiles) cs.next(pl);
                if (jj + 1 == ntiles || cs.bh != bh_now) umma_commit(q_free);
                return true;
            };
            for (int64_t jj = 0; jj < PERIOD && jj < ntiles && ok; ++jj) ok = issue_s(jj);
            int64_t seg_start = 0;
            for (int64_t jP = 0; jP < ntiles && ok; ++jP) {
                const int g0 = HALVES ? 0 : (int)(jP & 1);
                const int64_t kP = HALVES ? jP : (jP >> 1);
                if (jP == 0 || cp.k == 0) seg_start = jP;
                // the group's first tile of a piece starts a fresh accumulator
                const uint32_t acc0 = (jP - seg_start) < PERIOD ? 0u : 1u;
                const int sj = (int)(jP % STAGES);
                const uint64_t dV = dV0 + kStageDesc * sj;
                // PV in four 32-token chunks, each as soon as its P chunk is written
                for (int c = 0; c < 4 && ok; ++c) {
#pragma unroll
                    for (int gg = 0; gg < NG; ++gg)
                        if (ok) ok = wt.wait(p_chunk(g0 + gg, c), (uint32_t)kP & 1);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int gg = 0; gg < NG; ++gg) {
                        const int g = g0 + gg;
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const int kb = 2 * c + kk;
                            umma_bf16_ts(tmem + g * 256 + 128, tmem + g * 256 + kb * 8, dV + kb * (2048 >> 4),
                                         idPV, kb == 0 ? acc0 : 1u);
                        }
                    }
                }
                if (!ok) break;
#pragma unroll
                for (int gg = 0; gg < NG; ++gg) umma_commit(o_done(g0 + gg));
                umma_commit(empty(sj));
                if (jP + PERIOD < ntiles) ok = issue_s(jP + PERIOD);
                if (jP + 1 < ntiles) cp.next(pl);
            }
        }
        __syncwarp();
    } else {
        // ---------------- softmax warps ----------------
        const int g = (warp - 2) >> 2;            // group
        const int quad = warp & 3;                // TMEM lane quadrant of this warp
        const int rig = quad * 32 + lane;         // row within the group's 128 (TMEM lane)
        const int row = (HALVES ? g * 128 : 0) + rig;
        const int stid = threadIdx.x - 64;        // 0 .. NSOFT-1
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t s_tmem = tmem + g * 256 + lane_off;
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait(bar, par));
        };
        uint32_t soft_phase = 0;
        auto soft_sync = [&]() -> bool {        // bounded barrier of all softmax warps
            mbar_arrive(soft);
            return wwait(soft, soft_phase++ & 1);
        };
        float m_ref = -INFINITY, l = 0.f;
        bool has = false;                        // this group saw a tile of the current piece
        int64_t k_last = 0;                      // group-local index of that tile

        // End of a (b, h, shard) piece: write its partial; the last CTA to
        // finish a piece of the (b, h) merges all pieces (ticket, no waiting).
        auto finalize_piece = [&](const TileCursor &ti) -> bool {
            if (has && !wwait(o_done(g), (uint32_t)k_last & 1)) return false;
            tc_fence_after();
            const int bhh = ti.bh;
            const int64_t us = (int64_t)bhh * pl.T_bh + pl.tile_start[ti.r];
            const int64_t slot = ((int64_t)bhh * pl.R + ti.r) * pl.P_max + (cta - cta_of(pl, us));
            float *part_row = a.part_O + (slot * a.M + row) * D;
            if (HALVES) {
                const bool live = l > 0.f;
                const float inv = live ? 1.f / l : 0.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tmem + g * 256 + 128 + lane_off + c * 32, r);
                    tmem_wait_ld();
                    float4 *dst = reinterpret_cast<float4 *>(part_row + c * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                             __uint_as_float(r[4 * i + 2]) * inv,
                                             __uint_as_float(r[4 * i + 3]) * inv);
                }
                a.part_L[slot * a.M + row] = live ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            } else {
                // combine the two groups' running states of this row (same rows)
                stat[g * 128 + rig] = make_float2(has ? m_ref : -INFINITY, has ? l : 0.f);
                if (!soft_sync()) return false;
                const float2 s0 = stat[rig], s1 = stat[128 + rig];
                const float m = fmaxf(s0.x, s1.x);
                const float w0 = (s0.y > 0.f) ? ex2(s0.x - m) : 0.f;
                const float w1 = (s1.y > 0.f) ? ex2(s1.x - m) : 0.f;
                const float lt = w0 * s0.y + w1 * s1.y;
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                const float c0 = w0 * inv, c1 = w1 * inv;
                // group g writes columns [g*D/2, (g+1)*D/2)
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    const int col = g * (D / 2) + c * 32;
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tmem + 128 + lane_off + col, r0);
                    tmem_ld32(tmem + 256 + 128 + lane_off + col, r1);
                    tmem_wait_ld();
                    if (rig < a.M) {
                        float4 *dst = reinterpret_cast<float4 *>(part_row + col);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            float v[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float x0 = c0 > 0.f ? c0 * __uint_as_float(r0[4 * i + e]) : 0.f;
                                const float x1 = c1 > 0.f ? c1 * __uint_as_float(r1[4 * i + e]) : 0.f;
                                v[e] = x0 + x1;
                            }
                            dst[i] = make_float4(v[0], v[1], v[2], v[3]);
                        }
                    }
                }
                if (g == 0 && rig < a.M)
                    a.part_L[slot * a.M + row] = lt > 0.f ? (m + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
            }
            tc_fence_before();
            __threadfence();
            if (!soft_sync()) return false;
            if (stid == 0) {
                int expected = 0;
                for (int r = 0; r < pl.R; ++r) {
                    const int nt = pl.tile_start[r + 1] - pl.tile_start[r];
                    if (nt == 0) continue;
                    const int64_t u0 = (int64_t)bhh * pl.T_bh + pl.tile_start[r];
                    expected += cta_of(pl, u0 + nt - 1) - cta_of(pl, u0) + 1;
                }
                const unsigned prev = atomicAdd(&a.tickets[bhh], 1u);
                *last_flag = (prev == (unsigned)expected - 1u) ? 1 : 0;
            }
            if (!soft_sync()) return false;
            if (!*last_flag) return true;
            __threadfence();
            // ---- merge every piece of (b, h): eq. 23 over shards, pieces inside shards ----
            // L_r = log sum_p exp(L_p) over the pieces of shard r; then per row
            // L = L_max + log a with a = sum_r exp(L_r - L_max) (an online max/sum
            // over shard blocks), and Z = sum_r exp(L_r - L_max)/a * O_r
            //   = sum_pieces exp(L_p - L_max)/a * O_p  (the same sum, distributed).
            const int M = a.M;
            const int64_t BH = (int64_t)a.B * a.H;
            for (int r = stid; r < pl.R; r += NSOFT) {
                const int nt = pl.tile_start[r + 1] - pl.tile_start[r];
                int np = 0;
                if (nt > 0) {
                    const int64_t u0 = (int64_t)bhh * pl.T_bh + pl.tile_start[r];
                    np = cta_of(pl, u0 + nt - 1) - cta_of(pl, u0) + 1;
                }
                s_pstart[r + 1] = np;
            }
            if (!soft_sync()) return false;
            if (stid == 0) {
                s_pstart[0] = 0;
                int q = 0;
                for (int r = 0; r < pl.R; ++r) {
                    const int np = s_pstart[r + 1];
                    for (int p = 0; p < np; ++p, ++q)
                        if (q < kMergePieces) {
                            s_pslot[q] = (int)(((int64_t)bhh * pl.R + r) * pl.P_max + p);
                            s_pshard[q] = r;
                        }
                    s_pstart[r + 1] = q;
                }
            }
            if (!soft_sync()) return false;
            const int P = s_pstart[pl.R];
            if (P > kMergePieces) {                  // plans keep P within the table
                if (stid == 0) atomicExch(a.status, 2u);
                return false;
            }
            // 1. shard log-normalisers, in blocks of kMergeRB shards; online row max/sum
            float rm = -INFINITY, ra = 0.f;
            for (int rb0 = 0; rb0 < pl.R; rb0 += kMergeRB) {
                const int nb = min(kMergeRB, pl.R - rb0);
                for (int it = stid; it < nb * M; it += NSOFT) {
                    const int rr = it / M, i = it - rr * M, r = rb0 + rr;
                    const int q0 = s_pstart[r], q1 = s_pstart[r + 1];
                    float cm = -INFINITY;
                    for (int q = q0; q < q1; ++q) cm = fmaxf(cm, __ldcg(a.part_L + (int64_t)s_pslot[q] * M + i));
                    float Lr = -INFINITY;
                    if (cm != -INFINITY) {
                        float sum = 0.f;
                        for (int q = q0; q < q1; ++q) {
                            const float lp = __ldcg(a.part_L + (int64_t)s_pslot[q] * M + i);
                            if (lp != -INFINITY) sum += expf(lp - cm);
                        }
                        Lr = cm + logf(sum);
                    }
                    if (a.L_r) a.L_r[((int64_t)r * BH + bhh) * M + i] = Lr;
                    s_blk[rr * M + i] = Lr;
                }
                if (!soft_sync()) return false;
                if (stid < M) {
                    for (int rr = 0; rr < nb; ++rr) {
                        const float Lr = s_blk[rr * M + stid];
                        if (Lr == -INFINITY) continue;
                        if (rm == -INFINITY) {
                            rm = Lr;
                            ra = 1.f;
                        } else {
                            const float mn = fmaxf(rm, Lr);
                            ra = ra * expf(rm - mn) + expf(Lr - mn);
                            rm = mn;
                        }
                    }
                }
                if (!soft_sync()) return false;
            }
            if (stid < M) {
                s_lmax[stid] = rm;
                s_asum[stid] = ra;
                if (a.L) a.L[(int64_t)bhh * M + stid] = rm == -INFINITY ? -INFINITY : rm + logf(ra);
            }
            if (!soft_sync()) return false;
            // 2. Z = sum over pieces of exp(L_p - L_max)/a * O_p, kMergePB pieces at a time
            constexpr int Q4 = D / 4;
            constexpr int QPT = (HALVES ? 256 : 128) * Q4 / NSOFT;   // quads per thread
            float4 acc[QPT];
#pragma unroll
            for (int u = 0; u < QPT; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int qb0 = 0; qb0 < P; qb0 += kMergePB) {
                const int nb = min(kMergePB, P - qb0);
                for (int it = stid; it < nb * M; it += NSOFT) {
                    const int qq = it / M, i = it - qq * M;
                    const float lp = __ldcg(a.part_L + (int64_t)s_pslot[qb0 + qq] * M + i);
                    const float lm = s_lmax[i];
                    s_w[qq * M + i] = (lp == -INFINITY || lm == -INFINITY) ? 0.f : expf(lp - lm) / s_asum[i];
                }
                if (!soft_sync()) return false;
#pragma unroll
                for (int u = 0; u < QPT; ++u) {
                    const int qd = stid + u * NSOFT;
                    if (qd >= M * Q4) break;
                    const int i = qd / Q4, d4 = qd - i * Q4;
                    float4 v[kMergePB];
                    float w[kMergePB];
#pragma unroll
                    for (int qq = 0; qq < kMergePB; ++qq) {
                        w[qq] = qq < nb ? s_w[qq * M + i] : 0.f;
                        v[qq] = w[qq] != 0.f
                                    ? __ldcg(reinterpret_cast<const float4 *>(a.part_O + ((int64_t)s_pslot[qb0 + qq] * M + i) * D) + d4)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int qq = 0; qq < kMergePB; ++qq) {
                        acc[u].x = fmaf(w[qq], v[qq].x, acc[u].x);
                        acc[u].y = fmaf(w[qq], v[qq].y, acc[u].y);
                        acc[u].z = fmaf(w[qq], v[qq].z, acc[u].z);
                        acc[u].w = fmaf(w[qq], v[qq].w, acc[u].w);
                    }
                }
                if (!soft_sync()) return false;
            }
            if (a.Z) {
#pragma unroll
                for (int u = 0; u < QPT; ++u) {
                    const int qd = stid + u * NSOFT;
                    if (qd >= M * Q4) break;
                    const int i = qd / Q4, d4 = qd - i * Q4;
                    reinterpret_cast<float4 *>(a.Z + ((int64_t)bhh * M + i) * D)[d4] = acc[u];
                }
            }
            // 3. per-shard outputs O_r = sum_p exp(L_p - L_r) O_p (when requested)
            if (a.O_r) {
                for (int qd = stid; qd < M * Q4; qd += NSOFT) {
                    const int i = qd / Q4, d4 = qd - i * Q4;
                    for (int r = 0; r < pl.R; ++r) {
                        const float Lr = __ldcg(a.L_r + ((int64_t)r * BH + bhh) * M + i);
                        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (Lr != -INFINITY)
                            for (int q = s_pstart[r]; q < s_pstart[r + 1]; ++q) {
                                const float lp = __ldcg(a.part_L + (int64_t)s_pslot[q] * M + i);
                                if (lp == -INFINITY) continue;
                                const float wgt = expf(lp - Lr);
                                const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                                                            a.part_O + ((int64_t)s_pslot[q] * M + i) * D) + d4);
                                o.x = fmaf(wgt, v.x, o.x);
                                o.y = fmaf(wgt, v.y, o.y);
                                o.z = fmaf(wgt, v.z, o.z);
                                o.w = fmaf(wgt, v.w, o.w);
                            }
                        reinterpret_cast<float4 *>(a.O_r + (((int64_t)r * BH + bhh) * M + i) * D)[d4] = o;
                    }
                }
            }
            return soft_sync();
        };

        TileCursor ti;
        ti.init(pl, tb);
        const uint64_t c2 = f2pack(a.sl2, a.sl2);
        for (int64_t j = 0; j < ntiles; ++j) {
            const bool first = (j == 0) || ti.k == 0;
            const bool last = (j + 1 == ntiles) || ti.k == ti.nt - 1;
            if (first) {
                m_ref = -INFINITY;
                l = 0.f;
                has = false;
            }
            const bool mine = HALVES || ((int)(j & 1) == g);
            if (mine) {
                const int64_t k = HALVES ? j : (j >> 1);
                const int s = (int)(j % STAGES);
                if (!wwait(s_full(g), (uint32_t)k & 1)) break;
                // the stage's bias was published with the K/V load (complete by now)
                if (!wwait(full(s), (uint32_t)(j / STAGES) & 1)) break;
                tc_fence_after();
                // pass 1: row maximum of the scaled, masked scores (log2 units)
                const float4 *bs = reinterpret_cast<const float4 *>(bias + s * 128);
                float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tmem_ld32(s_tmem + c * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 bb = bs[c * 8 + i];
                        float t0, t1, t2, t3;
                        f2unpack(fma2(f2pack(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])), c2,
                                      f2pack(bb.x, bb.y)), t0, t1);
                        f2unpack(fma2(f2pack(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])), c2,
                                      f2pack(bb.z, bb.w)), t2, t3);
                        mx[0] = max3(mx[0], t0, t1);
                        mx[1] = max3(mx[1], t2, t3);
                    }
                }
                const float mt = fmaxf(mx[0], mx[1]);
                const bool need = mt > m_ref + kTau;
                if (__any_sync(0xffffffffu, need)) {
                    const float m_new = need ? mt : m_ref;
                    const float f = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
                    if (__any_sync(0xffffffffu, has)) {
                        // rescale the running output (its last PV finished before this S)
                        const uint32_t o_tmem = tmem + g * 256 + 128 + lane_off;
#pragma unroll
                        for (int c = 0; c < D / 16; ++c) {
                            uint32_t r[16];
                            tmem_ld16(o_tmem + c * 16, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
                            tmem_st16(o_tmem + c * 16, r);
                        }
                        tmem_wait_st();
                    }
                    l *= f;
                    m_ref = m_new;
                }
                // pass 2: P = exp2(t - m) in bf16, written over S's first 64 columns
                // (chunk c lands on columns 16c..16c+15, already read by then)
                // rows with no valid token yet (a per-token property, so the
                // same for every row of the warp) contribute P = 0
                const bool live = __all_sync(0xffffffffu, m_ref != -INFINITY);
                const uint64_t nm2 = live ? f2pack(-m_ref, -m_ref) : f2pack(0.f, 0.f);
                uint64_t ls2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pw[16];
                    if (live) {
                        uint32_t r[32];
                        tmem_ld32(s_tmem + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 bb = bs[c * 8 + i];
                            float t0, t1, t2, t3;
                            f2unpack(add2(fma2(f2pack(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])), c2, nm2),
                                          f2pack(bb.x, bb.y)), t0, t1);
                            f2unpack(add2(fma2(f2pack(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])), c2, nm2),
                                          f2pack(bb.z, bb.w)), t2, t3);
                            const float p0 = ex2(t0), p1 = ex2(t1), p2 = ex2(t2), p3 = ex2(t3);
                            ls2[0] = add2(ls2[0], f2pack(p0, p1));
                            ls2[1] = add2(ls2[1], f2pack(p2, p3));
                            pw[2 * i] = pack_bf16(p0, p1);
                            pw[2 * i + 1] = pack_bf16(p2, p3);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) pw[i] = 0u;
                    }
                    tmem_st16(s_tmem + c * 16, pw);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(p_chunk(g, c));
                }
                tmem_wait_st();
                {
                    float a0, a1, a2, a3;
                    f2unpack(ls2[0], a0, a1);
                    f2unpack(ls2[1], a2, a3);
                    l += (a0 + a1) + (a2 + a3);
                }
                has = true;
                k_last = k;

            }
            if (last && !finalize_piece(ti)) break;
            if (j + 1 < ntiles) ti.next(pl);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace tc
}  // namespace flare
