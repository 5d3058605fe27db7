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
//   warp 0       TMA producer: Q of the current (b, h) and K/V tiles into a
//                STAGES-deep ring; writes each tile's mask as an additive
//                bias (0 or -inf) next to it.
//   warp 1       TMEM allocator; lane 0 issues every tcgen05.mma:
//                S_g = Q_g K^T into TMEM, then O_g += P_g V.
//   warps 2..    ROWG groups of 4 softmax warps, one latent row per thread
//                (TMEM lane): online softmax in the log2 domain with a lazy
//                rescale (O and l are rescaled only when the row maximum grows
//                by more than kTau), P rounded to bf16 into shared memory.
// At the end of each (b, h, shard) piece of its span a CTA writes one partial
// (normalised output, log-normaliser); the CTA that completes the last piece
// of a (b, h) (atomic ticket, nobody waits) merges them: pieces into shards
// (O_r, L_r), shards into (Z, L), in fixed order.
#pragma once

#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace flare {
namespace tc {

constexpr float kTau = 8.0f;           // lazy-rescale threshold (log2 units)
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

// CTA whose span holds tile t.
__device__ __forceinline__ int cta_of(const TcTilePlan &p, int64_t t) {
    return (int)((t * p.grid) / p.T_total);
}
__device__ __forceinline__ int64_t span_begin(const TcTilePlan &p, int c) {
    return ((int64_t)c * p.T_total + p.grid - 1) / p.grid;
}

template <int D, int ROWG, int STAGES>
struct EncSmem {
    static constexpr int KA = D / 64;
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t P_OFF = Q_OFF + ROWG * KA * kAtom;
    static constexpr uint32_t STAGE_OFF = P_OFF + ROWG * 2 * kAtom;
    static constexpr uint32_t STAGE_BYTES = 2 * KA * kAtom;          // K then V
    static constexpr uint32_t BIAS_OFF = STAGE_OFF + STAGES * STAGE_BYTES;
    static constexpr uint32_t BAR_OFF = BIAS_OFF + STAGES * 128 * 4;
    // barriers: full[S], empty[S], q_full, q_free, s_full[G], s_free[G], p_full[G], o_done[G],
    // drain, soft (a bounded barrier among the softmax warps)
    static constexpr int NBAR = 2 * STAGES + 2 + 4 * ROWG + 2;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t MERGE_OFF = MISC_OFF + 64;             // 2 x 256 floats
    static constexpr uint32_t BYTES = MERGE_OFF + 2 * 256 * 4;
    static constexpr uint32_t ALLOC = BYTES + 1024;                   // room to align to 1 KB
    static constexpr uint32_t TMEM_COLS = ROWG == 1 ? 256 : 512;
};

template <int D, int ROWG, int STAGES>
__global__ void __launch_bounds__(64 + 128 * ROWG, 1)
enc_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmQ, const EncArgs a) {
    using L = EncSmem<D, ROWG, STAGES>;
    constexpr int KA = L::KA;
    constexpr int NSOFT = 128 * ROWG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + L::Q_OFF, sP = sbase + L::P_OFF, sStage = sbase + L::STAGE_OFF;
    float *bias = reinterpret_cast<float *>(smem + L::BIAS_OFF);
    const uint32_t bar0 = sbase + L::BAR_OFF;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t q_full = bar0 + 8u * (2 * STAGES), q_free = q_full + 8;
    auto s_full = [&](int g) { return bar0 + 8u * (2 * STAGES + 2 + g); };
    auto s_free = [&](int g) { return bar0 + 8u * (2 * STAGES + 2 + ROWG + g); };
    auto p_full = [&](int g) { return bar0 + 8u * (2 * STAGES + 2 + 2 * ROWG + g); };
    auto o_done = [&](int g) { return bar0 + 8u * (2 * STAGES + 2 + 3 * ROWG + g); };
    const uint32_t drain = bar0 + 8u * (2 * STAGES + 2 + 4 * ROWG);
    const uint32_t soft = drain + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);
    volatile int *last_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 8);
    float *s_lmax = reinterpret_cast<float *>(smem + L::MERGE_OFF);
    float *s_asum = s_lmax + 256;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TcTilePlan &pl = a.plan;
    const int cta = blockIdx.x;
    const int64_t tb = span_begin(pl, cta), te = span_begin(pl, cta + 1);
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
        for (int g = 0; g < ROWG; ++g) {
            mbar_init(s_full(g), 1);
            mbar_init(s_free(g), 128);
            mbar_init(p_full(g), 128);
            mbar_init(o_done(g), 1);
        }
        mbar_init(drain, 1);
        mbar_init(soft, NSOFT);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmQ);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp >= 2 && a.M < 128) {
        // rows M..127 of the query tile stay zero (only M rows are loaded)
        const int st = threadIdx.x - 64;
        for (int i = st; i < KA * kAtom / 16; i += NSOFT) {
            const int row = (i * 16 % kAtom) / 128;
            if (row >= a.M) reinterpret_cast<uint4 *>(smem + L::Q_OFF)[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        int cur_bh = -1;
        uint32_t q_uses = 0;
        int64_t j = 0;
        for (int64_t t = tb; t < te && !wt.aborted(); ++t, ++j) {
            const TileInfo ti = decompose(pl, t);
            const int b = ti.bh / a.H, h = ti.bh % a.H;
            if (ti.bh != cur_bh) {
                if (q_uses > 0 && !__all_sync(0xffffffffu, wt.wait(q_free, (q_uses - 1) & 1))) break;
                if (lane == 0) {
                    const int rows = a.M < 128 ? a.M : 128;
                    mbar_arrive_expect_tx(q_full, ROWG * KA * rows * 128);
                    const int qb = a.q_per_batch ? b : 0;
                    for (int g = 0; g < ROWG; ++g)
                        for (int ka = 0; ka < KA; ++ka)
                            tma_load_4d(sQ + (g * KA + ka) * kAtom, &tmQ, 64 * ka, 128 * g, h, qb, q_full);
                }
                ++q_uses;
                cur_bh = ti.bh;
            }
            const int s = (int)(j % STAGES);
            const uint32_t use = (uint32_t)(j / STAGES);
            if (!__all_sync(0xffffffffu, wt.wait(empty(s), (use & 1) ^ 1))) break;
            float *bs = bias + s * 128;
            for (int i = 0; i < 4; ++i) {
                const int tok = lane + 32 * i;
                const int64_t n = ti.n0 + tok;
                const bool ok = n < ti.n1 && (!a.mask || a.mask[(int64_t)b * a.N + n]);
                bs[tok] = ok ? 0.f : -INFINITY;
            }
            __threadfence_block();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(full(s), L::STAGE_BYTES);
                const uint32_t dst = sStage + s * L::STAGE_BYTES;
                for (int ka = 0; ka < KA; ++ka) {
                    tma_load_4d(dst + ka * kAtom, &tmK, 64 * ka, h, (int)ti.n0, b, full(s));
                    tma_load_4d(dst + (KA + ka) * kAtom, &tmV, 64 * ka, h, (int)ti.n0, b, full(s));
                }
            }
            __syncwarp();
        }
        // drain: wait for every load this CTA issued (needed only after an abort)
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
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_m128(128, 0);
            constexpr uint32_t idPV = idesc_bf16_m128(D, 1);
            int cur_bh = -1;
            uint32_t q_uses = 0;
            int64_t j = 0;
            bool ok = true;
            int64_t pending = -1;         // tile whose PV is still to issue
            bool pending_first = false;
            auto issue_pv = [&](int64_t jj, bool first) -> bool {
                const int sj = (int)(jj % STAGES);
                const uint32_t vbase = sStage + sj * L::STAGE_BYTES + KA * kAtom;
                for (int g = 0; g < ROWG; ++g) {
                    if (!wt.wait(p_full(g), (uint32_t)jj & 1)) return false;
                    tc_fence_after();
                    const uint32_t o_tmem = tmem + g * 256 + 128;
                    const uint32_t pbase = sP + g * 2 * kAtom;
#pragma unroll
                    for (int kb = 0; kb < 8; ++kb) {
                        const uint64_t da = desc_sw128(pbase + (kb >> 2) * kAtom + (kb & 3) * 32, 16, 1024);
                        const uint64_t db = desc_sw128(vbase + kb * 2048, kAtom, 1024);
                        umma_bf16_ss(o_tmem, da, db, idPV, (first && kb == 0) ? 0u : 1u);
                    }
                    umma_commit(o_done(g));
                }
                umma_commit(empty(sj));
                return true;
            };
            for (int64_t t = tb; t < te && ok; ++t, ++j) {
                const TileInfo ti = decompose(pl, t);
                const int s = (int)(j % STAGES);
                if (ti.bh != cur_bh) {
                    if (!wt.wait(q_full, q_uses & 1)) { ok = false; break; }
                    ++q_uses;
                    cur_bh = ti.bh;
                }
                if (!wt.wait(full(s), (uint32_t)(j / STAGES) & 1)) { ok = false; break; }
                const uint32_t kbase = sStage + s * L::STAGE_BYTES;
                for (int g = 0; g < ROWG && ok; ++g) {
                    if (j > 0 && !wt.wait(s_free(g), (uint32_t)(j - 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t qbase = sQ + g * KA * kAtom;
#pragma unroll
                    for (int kb = 0; kb < D / 16; ++kb) {
                        const uint32_t off = (kb >> 2) * kAtom + (kb & 3) * 32;
                        umma_bf16_ss(tmem + g * 256, desc_sw128(qbase + off, 16, 1024),
                                     desc_sw128(kbase + off, 16, 1024), idS, kb > 0 ? 1u : 0u);
                    }
                    umma_commit(s_full(g));
                }
                if (!ok) break;
                if (t + 1 == te || decompose(pl, t + 1).bh != ti.bh) umma_commit(q_free);
                if (pending >= 0 && !issue_pv(pending, pending_first)) { ok = false; break; }
                pending = j;
                pending_first = (t == tb) || ti.k == 0;
            }
            if (ok && pending >= 0) issue_pv(pending, pending_first);
            // make every issued MMA finish before TMEM is released
            umma_commit(drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < 2000000000ull) {
            }
        }
        __syncwarp();
    } else {
        // ---------------- softmax warps ----------------
        const int sw = warp - 2;
        const int g = sw >> 2;                  // row group
        const int quad = warp & 3;              // TMEM lane quadrant of this warp
        const int rig = quad * 32 + lane;       // row within the group (TMEM lane)
        const int row = g * 128 + rig;          // latent row
        const int stid = threadIdx.x - 64;      // 0 .. NSOFT-1
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t s_tmem = tmem + g * 256 + lane_off;
        const uint32_t o_tmem = tmem + g * 256 + 128 + lane_off;
        const uint32_t prow = sP + g * 2 * kAtom + rig * 128;
        const uint32_t swz = (uint32_t)(rig & 7);
        // every wait is taken by all lanes and its outcome made warp-uniform
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait(bar, par));
        };
        uint32_t soft_phase = 0;
        auto soft_sync = [&]() -> bool {     // bounded barrier of the softmax warps
            mbar_arrive(soft);
            return wwait(soft, soft_phase++ & 1);
        };
        float m_ref = -INFINITY, l = 0.f;
        // End of a (b, h, shard) piece of this CTA's span: write its partial
        // (normalised output and log-normaliser); the CTA that completes the
        // last piece of the (b, h) merges every piece (ticket, no waiting).
        auto finalize_piece = [&](const TileInfo &ti, int64_t jt) -> bool {
            if (!wwait(o_done(g), (uint32_t)jt & 1)) return false;
            tc_fence_after();
            const int bhh = ti.bh;
            const int64_t us = (int64_t)bhh * pl.T_bh + pl.tile_start[ti.r];
            const int piece = cta - cta_of(pl, us);
            const int64_t slot = ((int64_t)bhh * pl.R + ti.r) * pl.P_max + piece;
            const bool has = l > 0.f;
            const float inv = has ? 1.f / l : 0.f;
            const float Lp = has ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(o_tmem + c * 32, r);
                tmem_wait_ld();
                if (row < a.M) {
                    float4 *dst = reinterpret_cast<float4 *>(a.part_O + (slot * a.M + row) * D + c * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                             __uint_as_float(r[4 * i + 2]) * inv,
                                             __uint_as_float(r[4 * i + 3]) * inv);
                }
            }
            tc_fence_before();
            if (row < a.M) a.part_L[slot * a.M + row] = Lp;
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
            // ---- merge: pieces -> shards (O_r, L_r) -> global (Z, L), fixed order ----
            const int M = a.M;
            const int64_t BH = (int64_t)a.B * a.H;
            auto shard_L_at = [&](int r, int i) -> float * {
                return a.L_r ? a.L_r + ((int64_t)r * BH + bhh) * M + i
                             : a.shard_L + ((int64_t)bhh * pl.R + r) * M + i;
            };
            auto pieces = [&](int r, int64_t &s0) -> int {
                const int nt = pl.tile_start[r + 1] - pl.tile_start[r];
                if (nt == 0) return 0;
                const int64_t u0 = (int64_t)bhh * pl.T_bh + pl.tile_start[r];
                s0 = ((int64_t)bhh * pl.R + r) * pl.P_max;
                return cta_of(pl, u0 + nt - 1) - cta_of(pl, u0) + 1;
            };
            for (int i = stid; i < M; i += NSOFT) {
                float lmax = -INFINITY;
                for (int r = 0; r < pl.R; ++r) {
                    int64_t s0 = 0;
                    const int np = pieces(r, s0);
                    float cm = -INFINITY;
                    for (int p = 0; p < np; ++p) cm = fmaxf(cm, __ldcg(a.part_L + (s0 + p) * M + i));
                    float Lr = -INFINITY;
                    if (cm != -INFINITY) {
                        float sum = 0.f;
                        for (int p = 0; p < np; ++p) {
                            const float lp = __ldcg(a.part_L + (s0 + p) * M + i);
                            if (lp != -INFINITY) sum += expf(lp - cm);
                        }
                        Lr = cm + logf(sum);
                    }
                    *shard_L_at(r, i) = Lr;
                    lmax = fmaxf(lmax, Lr);
                }
                float asum = 0.f;
                if (lmax != -INFINITY)
                    for (int r = 0; r < pl.R; ++r) {
                        const float Lr = *shard_L_at(r, i);
                        if (Lr != -INFINITY) asum += expf(Lr - lmax);
                    }
                s_lmax[i] = lmax;
                s_asum[i] = asum;
                if (a.L) a.L[(int64_t)bhh * M + i] = lmax == -INFINITY ? -INFINITY : lmax + logf(asum);
            }
            if (!soft_sync()) return false;
            constexpr int Q4 = D / 4;
            for (int q = stid; q < M * Q4; q += NSOFT) {
                const int i = q / Q4, d4 = q % Q4;
                const float lmax = s_lmax[i];
                float4 U = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int r = 0; r < pl.R; ++r) {
                    const float Lr = *shard_L_at(r, i);
                    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (Lr != -INFINITY) {
                        int64_t s0 = 0;
                        const int np = pieces(r, s0);
                        for (int p = 0; p < np; ++p) {
                            const float lp = __ldcg(a.part_L + (s0 + p) * M + i);
                            if (lp == -INFINITY) continue;
                            const float wgt = expf(lp - Lr);
                            const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                                                        a.part_O + ((s0 + p) * M + i) * D) + d4);
                            o.x = fmaf(wgt, v.x, o.x);
                            o.y = fmaf(wgt, v.y, o.y);
                            o.z = fmaf(wgt, v.z, o.z);
                            o.w = fmaf(wgt, v.w, o.w);
                        }
                        const float wr = expf(Lr - lmax);
                        U.x = fmaf(wr, o.x, U.x);
                        U.y = fmaf(wr, o.y, U.y);
                        U.z = fmaf(wr, o.z, U.z);
                        U.w = fmaf(wr, o.w, U.w);
                    }
                    if (a.O_r)
                        reinterpret_cast<float4 *>(a.O_r + (((int64_t)r * BH + bhh) * M + i) * D)[d4] = o;
                }
                if (a.Z) {
                    const float inva = lmax == -INFINITY ? 0.f : 1.f / s_asum[i];
                    reinterpret_cast<float4 *>(a.Z + ((int64_t)bhh * M + i) * D)[d4] =
                        make_float4(U.x * inva, U.y * inva, U.z * inva, U.w * inva);
                }
            }
            return soft_sync();
        };
        int64_t j = 0;
        for (int64_t t = tb; t < te; ++t, ++j) {
            const TileInfo ti = decompose(pl, t);
            const bool first = (t == tb) || ti.k == 0;
            const bool last = (t + 1 == te) || ti.k == ti.nt - 1;
            const int s = (int)(j % STAGES);
            if (first) {
                m_ref = -INFINITY;
                l = 0.f;
            }
            if (!wwait(s_full(g), (uint32_t)j & 1)) break;
            // the stage's bias was published with the K/V load (already complete)
            if (!wwait(full(s), (uint32_t)(j / STAGES) & 1)) break;
            tc_fence_after();
            float sv[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(s_tmem + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(r[i]);
            }
            tc_fence_before();
            mbar_arrive(s_free(g));
            // scale to log2 units and mask (bias 0 or -inf); row maximum
            const float4 *bs = reinterpret_cast<const float4 *>(bias + s * 128);
            float mt = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float4 bb = bs[i];
                sv[4 * i + 0] = fmaf(sv[4 * i + 0], a.sl2, bb.x);
                sv[4 * i + 1] = fmaf(sv[4 * i + 1], a.sl2, bb.y);
                sv[4 * i + 2] = fmaf(sv[4 * i + 2], a.sl2, bb.z);
                sv[4 * i + 3] = fmaf(sv[4 * i + 3], a.sl2, bb.w);
                mt = fmaxf(mt, fmaxf(fmaxf(sv[4 * i], sv[4 * i + 1]), fmaxf(sv[4 * i + 2], sv[4 * i + 3])));
            }
            const bool need = mt > m_ref + kTau;
            bool o_ready = false;
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = need ? mt : m_ref;
                const float f = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
                if (!first) {
                    // rescale the running output: the previous PV must be done
                    if (!wwait(o_done(g), (uint32_t)(j - 1) & 1)) break;
                    tc_fence_after();
                    o_ready = true;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(o_tmem + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
                        tmem_st32(o_tmem + c * 32, r);
                    }
                    tmem_wait_st();
                }
                l *= f;
                m_ref = m_new;
            }
            // the P buffer is free once the previous PV has read it
            if (j > 0 && !o_ready && !wwait(o_done(g), (uint32_t)(j - 1) & 1)) break;
            const bool live = m_ref != -INFINITY;
#pragma unroll
            for (int c = 0; c < 16; ++c) {      // 16 chunks of 8 tokens
                uint32_t w4[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float p0 = live ? ex2(sv[8 * c + 2 * q] - m_ref) : 0.f;
                    const float p1 = live ? ex2(sv[8 * c + 2 * q + 1] - m_ref) : 0.f;
                    l += p0 + p1;
                    w4[q] = pack_bf16(p0, p1);
                }
                const uint32_t addr = prow + (c >> 3) * kAtom + ((((uint32_t)c & 7) ^ swz) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w4[0]),
                             "r"(w4[1]), "r"(w4[2]), "r"(w4[3])
                             : "memory");
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full(g));
            if (last && !finalize_piece(ti, j)) break;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace tc
}  // namespace flare
