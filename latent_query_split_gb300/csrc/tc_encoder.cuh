// tc_encoder.cuh -- split-KV FLARE encoder on sm_103a tensor cores.
//
// Computes, for every (b, h) and shard r, the pages' local primitive: O_r =
// softmax(s Q K_r^T) V_r normalised over shard r and its row log-normaliser
// L_r, then merges shards by eq. 23 (cross-rank log-sum-exp) into Z and L
// ("FLARE++: Low-rank attention with dynamic attention routing", appendix on
// context parallelism: the per-shard encoder, eq. 23 and the cross-rank
// log-sum-exp paragraph). Scores are never written to memory.
//
// One persistent CTA per SM walks a contiguous span of TILE-token tiles (see
// TcTilePlan; TILE = 128 for D = 64, 64 for D = 128). Eleven warps: warp 0 is
// the TMA producer, warp 1 allocates tensor memory and issues the PV MMAs,
// warp 2 issues the S MMAs (an MMA issue blocks until the tensor pipe accepts
// it, so two issuing warps overlap one's bookkeeping with the other's issue),
// warps 3-10 form two softmax groups of four warps (one per TMEM lane quadrant,
// one latent row per thread).
//
// Producer: K/V tiles into a STAGES-deep ring (L2 evict-first). The tile's
// padding mask (prefetched one tile ahead; tokens past the shard end count as
// padding) becomes a bf16 bias column (0 / -inf) beside the stage, which one
// extra K = 16 MMA adds to every row of S:
//     S = [1 0..0] [bias 0..0]^T + Q K^T,
// so padding arrives in tensor memory as -inf and the softmax never reads the
// mask.
//
// Two kernels share the producer and the merge:
//  * enc_cs_kernel (M <= 128): S is double-buffered in tensor memory, so S of
//    the next tile is computed while the softmax of this one runs; S_{j+2}
//    waits for PV_j, which read P from the same buffer (buf_free). The two
//    groups split each tile's tokens in halves; each keeps its own running
//    max, sum and output
//    accumulator (the PV MMAs of a tile accumulate the first half of its
//    tokens into O_0 and the second into O_1), so the groups never exchange
//    anything inside a piece and are combined once when a piece ends.
//  * enc_ring_kernel (M = 256): each group owns 128 latent rows; the two
//    groups' S tiles take turns in a ring of three tensor-memory buffers, so
//    each group's next S is computed while its softmax runs.
// A tile without padded tokens skips the bias MMA (the producer flags it).
// Softmax: the row maximum over S (already scaled into log2 units by one
// FFMA), lazy rescale (O and l are rescaled only when the row maximum grows by
// more than kTau), P = exp2(S - m) in bf16 written back into tensor memory
// for the PV MMA (A operand from tensor memory).
// At the end of each (b, h, shard) piece of its span a CTA writes a partial
// (normalised output, log-normaliser). enc_merge_kernel, launched right after,
// merges them in fixed order: pieces into shards (O_r, L_r), shards into
// (Z, L), by the one log-sum-exp rule.
#pragma once

#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace flare {
namespace tc {

constexpr float kTau = 8.0f;           // lazy-rescale threshold (log2 units)
constexpr int kMergePieces = 512;      // pieces of one (b, h) the merge handles
constexpr uint32_t kAtom = 128 * 128;  // bytes of one 128-row x 128-byte swizzle column

struct EncArgs {
    int B, H, M, N;
    float sl2;                 // score scale * log2(e)
    int q_per_batch;           // Q has a batch dimension
    const uint8_t *mask;
    float *part_L, *part_O;    // per-piece partials (workspace)
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
    ti.n0 = p.off[lo] + (int64_t)ti.k * p.tile;
    ti.n1 = min(ti.n0 + p.tile, p.off[lo + 1]);
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
            n0 += p.tile;
            n1 = min(n0 + p.tile, shard_end);
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
        n1 = min(n0 + p.tile, shard_end);
    }
};

// ---- shared-memory pieces common to both kernels ------------------------------
// Mask bias rows of one stage: TILE rows of 16 bytes (bf16 bias, then 7
// zeros): the first K-core-matrix of a K = 16 block, no swizzle. The constant
// A block of the bias MMA ("ones"): 128 rows [1, 0 x 7], then 128 rows of
// zeros (the second core matrix along K); the bias MMA's B takes its second
// core matrix from those zeros too.
constexpr uint32_t kOnesBytes = 2 * 128 * 16;

// S = bias (every row) via one K = 16 MMA, warp-collective; Q K^T accumulates on top.
__device__ __forceinline__ void umma_bias_elect(uint32_t d_tmem, uint32_t s_ones, uint32_t s_bias,
                                                uint32_t idesc) {
    umma_ss_elect(d_tmem, desc_noswz(s_ones, 128 * 16, 128),
                  desc_noswz(s_bias, s_ones + 128 * 16 - s_bias, 128), idesc, 0u);
}

// ---- producer (one warp): K/V tiles and their mask bias -----------------------
// full(s) = bar0 + 8 s, empty(s) = bar0 + 8 (STAGES + s). Beside the bias rows
// a per-stage word at PADF_OFF says whether the tile has any padded token.
template <class C>
__device__ __forceinline__ void produce_kv(const CUtensorMap *tmK, const CUtensorMap *tmV,
                                           const EncArgs &a, int64_t tb, int64_t ntiles,
                                           uint8_t *smem, uint32_t bar0, const Waiter &wt,
                                           int lane) {
    constexpr int TILE = C::TILE, KA = C::KA, STAGES = C::STAGES;
    const TcTilePlan &pl = a.plan;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t sStage = smem_u32(smem + C::STAGE_OFF);
    const uint64_t pol = policy_evict_first();
    // With a mask, its bytes are fetched AHEAD tiles before their tile is
    // issued, into one of AHEAD register sets taken in turn (the loop is
    // unrolled AHEAD times, so no set is read before its loads have had AHEAD
    // iterations to land): a load consumed in the next iteration put its
    // whole latency on every tile. Without a mask (only shard ends to mark,
    // no loads) the plain loop with one set is kept: the unrolled one was
    // measurably slower there.
    constexpr int MB = TILE / 32;
    constexpr int AHEAD = 4;
    auto load_mask = [&](const TileCursor &ti, uint8_t (&mb)[MB]) {
        const int b = ti.bh / a.H;
#pragma unroll
        for (int i = 0; i < MB; ++i) {
            const int64_t n = ti.n0 + lane + 32 * i;
            mb[i] = (n < ti.n1) ? (a.mask ? a.mask[(int64_t)b * a.N + n] : (uint8_t)1) : (uint8_t)0;
        }
    };
    uint8_t m0[MB], m1[MB], m2[MB], m3[MB];
    TileCursor ti, tl;                  // the tile being issued; the next tile whose mask is fetched
    ti.init(pl, tb);
    tl = ti;
    int64_t jl = 0;                     // index of tile tl
    auto fetch = [&](uint8_t (&mb)[MB]) {
        if (jl < ntiles) {
            load_mask(tl, mb);
            if (jl + 1 < ntiles) tl.next(pl);
        }
        ++jl;
    };
    fetch(m0);
    if (a.mask != nullptr) {
        fetch(m1);
        fetch(m2);
        fetch(m3);
    }
    int64_t j = 0;
    // issues tile j with its mask bytes mb, then fetches tile j + AHEAD's into mb
    auto step = [&](uint8_t (&mb)[MB]) -> bool {
        if (j >= ntiles || wt.aborted()) return false;
        const int b = ti.bh / a.H, h = ti.bh - b * a.H;
        const int s = (int)(j % STAGES);
        if (!__all_sync(0xffffffffu, wt.wait(empty(s), ((uint32_t)(j / STAGES) & 1) ^ 1))) return false;
        // bias rows of this stage: bf16 0 (valid) or -inf (padding), then zeros
        uint4 *bs = reinterpret_cast<uint4 *>(smem + C::BIAS_OFF + s * C::BIAS_BYTES);
        bool pad = false;
#pragma unroll
        for (int i = 0; i < MB; ++i) {
            bs[lane + 32 * i] = make_uint4(mb[i] ? 0u : 0xFF80u, 0u, 0u, 0u);
            pad |= mb[i] == 0;
        }
        // whether the tile has a padded token (else the MMA warp skips the bias MMA)
        pad = __any_sync(0xffffffffu, pad);
        if (lane == 0) reinterpret_cast<volatile uint32_t *>(smem + C::PADF_OFF)[s] = pad ? 1u : 0u;
        fence_proxy_async_smem();
        __syncwarp();
        const bool place_ok =
            dcheck(tile_in_tensor(64 * (KA - 1), h, ti.n0, b, a.H, a.N, a.B) && ti.n0 < ti.n1 && ti.n1 <= a.N,
                   kChkEncKV, a.status) &&
            dcheck(ti.r >= 0 && ti.r < pl.R && ti.n0 >= pl.off[ti.r] && ti.n1 <= pl.off[ti.r + 1],
                   kChkEncCursor, a.status);
        if (lane == 0) {
            mbar_arrive_expect_tx(full(s), C::STAGE_BYTES);
            const uint32_t dst = sStage + s * C::STAGE_BYTES;
            for (int ka = 0; ka < KA && place_ok; ++ka) {
                tma_load_4d_hint(dst + ka * C::KV_ATOM, tmK, 64 * ka, h, (int)ti.n0, b, full(s), pol);
                tma_load_4d_hint(dst + (KA + ka) * C::KV_ATOM, tmV, 64 * ka, h, (int)ti.n0, b, full(s), pol);
            }
        }
        __syncwarp();
        fetch(mb);
        if (j + 1 < ntiles) ti.next(pl);
        ++j;
        return true;
    };
    static_assert(AHEAD == 4, "the unrolled loop below takes the four register sets in turn");
    if (a.mask != nullptr) {
        while (step(m0) && step(m1) && step(m2) && step(m3)) {
        }
    } else {
        // no mask loads to hide: one register set (the masks only mark shard ends)
        while (step(m0)) {
        }
    }
    // after an abort: let every issued load land before the CTA exits
    if (wt.aborted() && lane == 0) {
        const uint64_t t0 = globaltimer();
        for (int64_t jj = (j > STAGES ? j - STAGES : 0); jj < j; ++jj)
            while (!mbar_try_wait(full((int)(jj % STAGES)), (uint32_t)(jj / STAGES) & 1) &&
                   globaltimer() - t0 < 500000000ull) {
            }
    }
}

// Slot of the partial of the piece that tile `ti` ends (this CTA's piece of
// its (b, h, shard)).
__device__ __forceinline__ int64_t piece_slot_of(const TcTilePlan &pl, const TileCursor &ti, int cta) {
    const int64_t us = (int64_t)ti.bh * pl.T_bh + pl.tile_start[ti.r];
    return ((int64_t)ti.bh * pl.R + ti.r) * pl.P_max + (cta - cta_of(pl, us));
}

// ===============================================================================
// enc_cs_kernel: M <= 128 (column split, double-buffered S, one MMA warp)
// ===============================================================================
template <int D, int STAGES_>
struct CsCfg {
    static constexpr int STAGES = STAGES_;
    static constexpr int TILE = D == 128 ? 64 : 128;    // tokens per tile (32 KB of K+V)
    static constexpr int HALF = TILE / 2;               // tokens of one group in a tile
    static constexpr int KA = D / 64;                   // 64-element atoms along D
    static constexpr int NSOFT = 256;
    static constexpr int THREADS = 96 + NSOFT;         // producer, PV issuer, S issuer, softmax
    // tensor memory: S buffers b = 0, 1 at b*TILE (P of group g written as
    // bf16 pairs over the first HALF/2 columns of its own half of S), then O_0, O_1
    static constexpr uint32_t O_COL = 2 * TILE;
    static_assert(O_COL + 2 * D <= 512, "tensor-memory columns exceeded");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t Q_ATOM = kAtom;           // 128 rows x 128 bytes
    static constexpr uint32_t KV_ATOM = TILE * 128;     // TILE rows x 128 bytes
    static constexpr uint32_t Q_OFF = 0;                // two Q buffers (consecutive (b, h))
    static constexpr uint32_t Q_BYTES = KA * Q_ATOM;
    static constexpr uint32_t STAGE_OFF = Q_OFF + 2 * Q_BYTES;
    static constexpr uint32_t STAGE_BYTES = 2 * KA * KV_ATOM;   // K atoms then V atoms
    static constexpr uint32_t BIAS_OFF = STAGE_OFF + STAGES * STAGE_BYTES;
    static constexpr uint32_t BIAS_BYTES = TILE * 16;
    static constexpr uint32_t ONES_OFF = BIAS_OFF + STAGES * BIAS_BYTES;
    static constexpr uint32_t PADF_OFF = ONES_OFF + kOnesBytes;   // per stage: tile has padding
    static constexpr uint32_t BAR_OFF = PADF_OFF + 16 * ((STAGES * 4 + 15) / 16);
    // full[S], empty[S], q_full[2], s_full[2], p_full[2], o_done[2], drain, soft, buf_free[2], drain2
    static constexpr int NBAR = 2 * STAGES + 13;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    // the two groups' (m, l) of each row at a piece end, double-buffered by
    // piece parity: [2][2 groups][128 rows]
    static constexpr uint32_t STAT_OFF = MISC_OFF + 64;
    static constexpr uint32_t BYTES = STAT_OFF + 2 * 2 * 128 * 8;
    static constexpr uint32_t ALLOC = BYTES + 1024;           // room to align the base to 1 KB
    static_assert(ALLOC <= 232448, "shared memory budget of one CTA exceeded");
};

template <int D, int STAGES>
__global__ void __launch_bounds__(CsCfg<D, STAGES>::THREADS, 1)
enc_cs_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const __grid_constant__ CUtensorMap tmQ, const EncArgs a) {
    using C = CsCfg<D, STAGES>;
    constexpr int KA = C::KA, TILE = C::TILE, HALF = C::HALF, NSOFT = C::NSOFT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::Q_OFF, sStage = sbase + C::STAGE_OFF;
    const uint32_t sBias = sbase + C::BIAS_OFF, sOnes = sbase + C::ONES_OFF;
    const uint32_t bar0 = sbase + C::BAR_OFF;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto q_full = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto s_full = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    auto p_full = [&](int b) { return bar0 + 8u * (2 * STAGES + 4 + b); };
    auto o_done = [&](int b) { return bar0 + 8u * (2 * STAGES + 6 + b); };
    const uint32_t drain = bar0 + 8u * (2 * STAGES + 8);
    const uint32_t soft = bar0 + 8u * (2 * STAGES + 9);
    auto buf_free = [&](int b) { return bar0 + 8u * (2 * STAGES + 10 + b); };
    const uint32_t drain2 = bar0 + 8u * (2 * STAGES + 12);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    float2 *stat = reinterpret_cast<float2 *>(smem + C::STAT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TcTilePlan &pl = a.plan;
    const int cta = blockIdx.x;
    const int64_t tb = span_begin(pl, cta), te = span_begin(pl, cta + 1);
    const int64_t ntiles = te - tb;
    Waiter wt{abort_flag, a.status};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(q_full(b), 1);
            mbar_init(s_full(b), 1);
            mbar_init(p_full(b), 8);          // one arrival per softmax warp
            mbar_init(o_done(b), 1);
            mbar_init(buf_free(b), 1);
        }
        mbar_init(drain, 1);
        mbar_init(drain2, 1);
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
    if (warp >= 3) {
        const int i = threadIdx.x - 96;           // 0 .. 255
        // rows M..127 of both query buffers stay zero (only M rows are loaded)
        if (a.M < 128)
            for (int q = i; q < 2 * (int)C::Q_BYTES / 16; q += NSOFT) {
                const int row = (q * 16 % (int)C::Q_ATOM) / 128;
                if (row >= a.M) reinterpret_cast<uint4 *>(smem + C::Q_OFF)[q] = make_uint4(0, 0, 0, 0);
            }
        // the bias MMA's constant A: row r = [1.0, 0, ...] then a zero core matrix
        reinterpret_cast<uint4 *>(smem + C::ONES_OFF)[i] = make_uint4(i < 128 ? 0x3F80u : 0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        produce_kv<C>(&tmK, &tmV, a, tb, ntiles, smem, bar0, wt, lane);
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA issue: warp 2 every S, warp 1 every PV ----------------
        // S_{j+2} goes into buffer j & 1 once PV_j (which read P there) has
        // completed (buf_free). Q of generation u sits in buffer u & 1;
        // generation u + 1 is fetched once S of generation u - 1 has completed.
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait(bar, par));
        };
        constexpr uint32_t idS = idesc_bf16_m128(TILE, 0);
        constexpr uint32_t idPV = idesc_bf16_m128(D, 1);
        const uint32_t my_drain = warp == 1 ? drain : drain2;
        bool ok = true;
        int q_req = -1;
        if (warp == 2) {
            const int bh0 = (int)(tb / pl.T_bh);
            const int last_gen = ntiles > 0 ? (int)((te - 1) / pl.T_bh) - bh0 : -1;
            auto request_q = [&](int u) {
                if (lane == 0) {
                    const int bh = bh0 + u, b = bh / a.H, h = bh - b * a.H;
                    const int rows = a.M < 128 ? a.M : 128;
                    mbar_arrive_expect_tx(q_full(u & 1), KA * rows * 128);
                    const bool q_ok = dcheck(bh < a.B * a.H && h >= 0 && b >= 0, kChkEncQ, a.status);
#pragma unroll
                    for (int ka = 0; ka < KA && q_ok; ++ka)
                        tma_load_4d(sQ + (u & 1) * C::Q_BYTES + ka * C::Q_ATOM, &tmQ, 64 * ka, 0, h,
                                    a.q_per_batch ? b : 0, q_full(u & 1));
                }
                __syncwarp();
                q_req = u;
            };
            TileCursor cs;
            cs.init(pl, tb);
            int s_bh = -1;
            if (ntiles > 0) {
                request_q(0);
                if (last_gen >= 1) request_q(1);
            }
            for (int64_t js = 0; js < ntiles && ok; ++js) {
                const int u = cs.bh - bh0;
                const bool gen_start = cs.bh != s_bh;
                const int b = (int)(js & 1);
                if (js >= 2 && !(ok = wwait(buf_free(b), (uint32_t)((js >> 1) - 1) & 1))) break;
                if (gen_start && !(ok = wwait(q_full(u & 1), (uint32_t)(u >> 1) & 1))) break;
                const int s = (int)(js % STAGES);
                if (!(ok = wwait(full(s), (uint32_t)(js / STAGES) & 1))) break;
                tc_fence_after();
                const uint32_t tS = tmem + (uint32_t)b * TILE;
                const bool pad = reinterpret_cast<const volatile uint32_t *>(smem + C::PADF_OFF)[s] != 0;
                if (pad) umma_bias_elect(tS, sOnes, sBias + s * C::BIAS_BYTES, idS);
                const uint64_t dQ = desc_sw128(sQ + (u & 1) * C::Q_BYTES, 16, 1024);
                const uint64_t dK = desc_sw128(sStage + s * C::STAGE_BYTES, 16, 1024);
#pragma unroll
                for (int kb = 0; kb < D / 16; ++kb) {
                    const uint64_t offQ = (uint64_t)((kb >> 2) * C::Q_ATOM + (kb & 3) * 32) >> 4;
                    const uint64_t offK = (uint64_t)((kb >> 2) * C::KV_ATOM + (kb & 3) * 32) >> 4;
                    umma_ss_elect(tS, dQ + offQ, dK + offK, idS, (pad || kb > 0) ? 1u : 0u);
                }
                umma_commit_elect(s_full(b));
                s_bh = cs.bh;
                if (gen_start && u + 1 <= last_gen && q_req < u + 1) {
                    if (u >= 1 && !(ok = wwait(s_full((int)((js - 1) & 1)), (uint32_t)((js - 1) >> 1) & 1))) break;
                    request_q(u + 1);
                }
                if (js + 1 < ntiles) cs.next(pl);
            }
        } else {
            TileCursor cp;
            cp.init(pl, tb);
            for (int64_t j = 0; j < ntiles && ok; ++j) {
                const int b = (int)(j & 1);
                if (!(ok = wwait(p_full(b), (uint32_t)(j >> 1) & 1))) break;
                tc_fence_after();
                // O_g += P_g V_g over the tile's two halves; a piece's first tile
                // starts both accumulators afresh
                const bool first = (j == 0) || cp.k == 0;
                const int s = (int)(j % STAGES);
                const uint64_t dV = desc_sw128(sStage + s * C::STAGE_BYTES + KA * C::KV_ATOM, C::KV_ATOM, 1024);
                const uint32_t tP = tmem + (uint32_t)b * TILE;
#pragma unroll
                for (int g = 0; g < 2; ++g)
#pragma unroll
                    for (int kb = 0; kb < HALF / 16; ++kb)
                        umma_ts_elect(tmem + C::O_COL + g * D, tP + g * HALF + kb * 8,
                                      dV + (uint64_t)((g * HALF + kb * 16) * 128 >> 4), idPV,
                                      (kb > 0 || !first) ? 1u : 0u);
                umma_commit_elect(o_done(b));
                umma_commit_elect(buf_free(b));
                umma_commit_elect(empty(s));
                if (j + 1 < ntiles) cp.next(pl);
            }
        }
        if (wt.aborted()) {
            umma_commit_elect(my_drain);
            if (lane == 0) {
                const uint64_t t0 = globaltimer();
                for (int u = (q_req > 0 ? q_req - 1 : 0); u <= q_req; ++u)
                    while (!mbar_try_wait(q_full(u & 1), (uint32_t)(u >> 1) & 1) &&
                           globaltimer() - t0 < 500000000ull) {
                    }
                while (!mbar_try_wait(my_drain, 0) && globaltimer() - t0 < 500000000ull) {
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- softmax groups (column halves) ----------------
        const int g = (warp - 3) >> 2;            // group: tokens [g*HALF, (g+1)*HALF) of a tile
        const int quad = warp & 3;                // TMEM lane quadrant of this warp
        const int rig = quad * 32 + lane;         // latent row (TMEM lane)
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t o_tmem = tmem + C::O_COL + g * D + lane_off;
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
        uint32_t pieces = 0;                     // pieces finished (parity selects the stat buffer)

        // End of a (b, h, shard) piece: the two groups' states of each row are
        // combined into the piece's partial (normalised output, log-normaliser).
        auto finalize_piece = [&](const TileCursor &ti, int64_t j) -> bool {
            // PV of the piece's last tile must be complete (o_done of its buffer)
            if (!wwait(o_done((int)(j & 1)), (uint32_t)(j >> 1) & 1)) return false;
            tc_fence_after();
            const int64_t slot = piece_slot_of(pl, ti, cta);
            const int64_t piece = slot - ((int64_t)ti.bh * pl.R + ti.r) * pl.P_max;
            const bool slot_ok = dcheck(ti.bh < a.B * a.H && piece >= 0 && piece < pl.P_max, kChkEncPiece, a.status);
            float *part_row = a.part_O + (slot * a.M + rig) * D;
            float2 *st = stat + (pieces++ & 1) * 256;
            st[g * 128 + rig] = make_float2(has ? m_ref : -INFINITY, has ? l : 0.f);
            if (!soft_sync()) return false;
            const float2 s0 = st[rig], s1 = st[128 + rig];
            const float m = fmaxf(s0.x, s1.x);
            const float w0 = (s0.y > 0.f) ? ex2(s0.x - m) : 0.f;
            const float w1 = (s1.y > 0.f) ? ex2(s1.x - m) : 0.f;
            const float lt = w0 * s0.y + w1 * s1.y;
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            const float c0 = w0 * inv, c1 = w1 * inv;
            // group g writes columns [g*D/2, (g+1)*D/2) of the row
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                const int col = g * (D / 2) + c * 32;
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + C::O_COL + lane_off + col, r0);
                tmem_ld32(tmem + C::O_COL + D + lane_off + col, r1);
                tmem_wait_ld();
                if (rig < a.M && slot_ok) {
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
            if (g == 0 && rig < a.M && slot_ok)
                a.part_L[slot * a.M + rig] = lt > 0.f ? (m + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
            return true;
        };

        TileCursor ti;
        ti.init(pl, tb);
        const uint64_t c2 = f2pack(a.sl2, a.sl2);
        constexpr int NC = HALF / 32;             // 32-column chunks of this group's half
        for (int64_t j = 0; j < ntiles; ++j) {
            const bool first = (j == 0) || ti.k == 0;
            const bool last = (j + 1 == ntiles) || ti.k == ti.nt - 1;
            if (first) {
                m_ref = -INFINITY;
                l = 0.f;
                has = false;
            }
            const int b = (int)(j & 1);
            const uint32_t s_tmem = tmem + (uint32_t)b * TILE + g * HALF + lane_off;
            if (!wwait(s_full(b), (uint32_t)(j >> 1) & 1)) break;
            tc_fence_after();
            // this group's half of the row, held in registers for both passes
            uint32_t r[NC][32];
#pragma unroll
            for (int c = 0; c < NC; ++c) tmem_ld32(s_tmem + c * 32, r[c]);
            tmem_wait_ld();
            // the row maximum of the masked scores (padding is -inf in S
            // already), in log2 units (the scale is positive)
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    mx[0] = max3(mx[0], __uint_as_float(r[c][4 * i]), __uint_as_float(r[c][4 * i + 1]));
                    mx[1] = max3(mx[1], __uint_as_float(r[c][4 * i + 2]), __uint_as_float(r[c][4 * i + 3]));
                }
            const float mt = fmaxf(mx[0], mx[1]) * a.sl2;
            const bool need = mt > m_ref + kTau;
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = need ? mt : m_ref;
                const float f = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
                if (__any_sync(0xffffffffu, has)) {
                    // O holds PV of the previous tile once its o_done has fired
                    if (!wwait(o_done((int)((j - 1) & 1)), (uint32_t)((j - 1) >> 1) & 1)) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 16; ++c) {
                        uint32_t o[16];
                        tmem_ld16(o_tmem + c * 16, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
                        tmem_st16(o_tmem + c * 16, o);
                    }
                }
                l *= f;
                m_ref = m_new;
            }
            // P = exp2(t - m) in bf16 over this group's own S columns (rows
            // with no valid token yet -- a per-token property, the same for
            // every row of the warp -- give P = 0)
            const bool live = __all_sync(0xffffffffu, m_ref != -INFINITY);
            const uint64_t nm2 = live ? f2pack(-m_ref, -m_ref) : f2pack(0.f, 0.f);
            uint64_t ls2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                uint32_t pw[16];
                if (live) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float t0, t1, t2, t3;
                        f2unpack(fma2(f2pack(__uint_as_float(r[c][4 * i]), __uint_as_float(r[c][4 * i + 1])), c2, nm2), t0, t1);
                        f2unpack(fma2(f2pack(__uint_as_float(r[c][4 * i + 2]), __uint_as_float(r[c][4 * i + 3])), c2, nm2), t2, t3);
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
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(b));    // one arrival per warp
            {
                float a0, a1, a2, a3;
                f2unpack(ls2[0], a0, a1);
                f2unpack(ls2[1], a2, a3);
                l += (a0 + a1) + (a2 + a3);
            }
            has = true;
            if (last && !finalize_piece(ti, j)) break;
            if (j + 1 < ntiles) ti.next(pl);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
    pdl_launch_dependents();   // the merge may be scheduled (it waits for this grid)
}

// ===============================================================================
// enc_ring_kernel: M = 256, D = 64 (two groups of 128 latent rows, three S buffers)
// ===============================================================================
// Group g owns latent rows [128 g, 128 g + 128) and its own accumulator O_g.
// S of (tile j, group g) is the q-th S computed, q = 2 j + g, and lives in
// tensor-memory buffer q mod 3; P is written as bf16 pairs over the first
// half of that buffer. Warp 2 issues S(0), S(1), ... (S(q + 3) once PV(q),
// which read the same buffer, has completed: buf_free); warp 1 issues PV(q)
// once P(q) is written. A group's next S is thus computed while its softmax
// of this tile runs.
template <int STAGES_>
struct RingCfg {
    static constexpr int STAGES = STAGES_;
    static constexpr int D = 64;
    static constexpr int TILE = 128;
    static constexpr int KA = 1;
    static constexpr int NCH = TILE / 32;
    static constexpr int NSOFT = 256;
    static constexpr int THREADS = 96 + NSOFT;         // producer, PV issuer, S issuer, softmax
    static constexpr uint32_t O_COL = 3 * TILE;         // O_0, O_1 after the three S buffers
    static_assert(O_COL + 2 * D <= 512, "tensor-memory columns exceeded");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t KV_ATOM = TILE * 128;
    static constexpr uint32_t Q_OFF = 0;                // two Q buffers (consecutive (b, h)) of 256 rows
    static constexpr uint32_t Q_BYTES = 2 * kAtom;
    static constexpr uint32_t STAGE_OFF = Q_OFF + 2 * Q_BYTES;
    static constexpr uint32_t STAGE_BYTES = 2 * KV_ATOM;   // K atom, then V atom
    static constexpr uint32_t BIAS_OFF = STAGE_OFF + STAGES * STAGE_BYTES;
    static constexpr uint32_t BIAS_BYTES = TILE * 16;
    static constexpr uint32_t ONES_OFF = BIAS_OFF + STAGES * BIAS_BYTES;
    static constexpr uint32_t PADF_OFF = ONES_OFF + kOnesBytes;   // per stage: tile has padding
    static constexpr uint32_t BAR_OFF = PADF_OFF + 16 * ((STAGES * 4 + 15) / 16);
    // full[S], empty[S], q_full[2], s_full[3], p_full[3], o_done[2], drain[2], buf_free[3],
    // p_half[3]
    static constexpr int NBAR = 2 * STAGES + 18;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t BYTES = MISC_OFF + 64;
    static constexpr uint32_t ALLOC = BYTES + 1024;
    static_assert(ALLOC <= 232448, "shared memory budget of one CTA exceeded");
};

template <int STAGES>
__global__ void __launch_bounds__(RingCfg<STAGES>::THREADS, 1)
enc_ring_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmQ, const EncArgs a) {
    using C = RingCfg<STAGES>;
    constexpr int D = C::D, TILE = C::TILE, NCH = C::NCH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::Q_OFF, sStage = sbase + C::STAGE_OFF;
    const uint32_t sBias = sbase + C::BIAS_OFF, sOnes = sbase + C::ONES_OFF;
    const uint32_t bar0 = sbase + C::BAR_OFF;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto q_full = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto s_full = [&](int u) { return bar0 + 8u * (2 * STAGES + 2 + u); };
    auto p_full = [&](int u) { return bar0 + 8u * (2 * STAGES + 5 + u); };
    auto o_done = [&](int g) { return bar0 + 8u * (2 * STAGES + 8 + g); };
    auto drain = [&](int w) { return bar0 + 8u * (2 * STAGES + 10 + w); };
    auto buf_free = [&](int u) { return bar0 + 8u * (2 * STAGES + 12 + u); };
    // the first half of P (tokens 0..63 of the tile) is in place
    auto p_half = [&](int u) { return bar0 + 8u * (2 * STAGES + 15 + u); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TcTilePlan &pl = a.plan;
    const int cta = blockIdx.x;
    const int64_t tb = span_begin(pl, cta), te = span_begin(pl, cta + 1);
    const int64_t ntiles = te - tb;
    Waiter wt{abort_flag, a.status};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);               // committed after the tile's second PV
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(q_full(b), 1);
            mbar_init(o_done(b), 1);
        }
        for (int u = 0; u < 3; ++u) {
            mbar_init(s_full(u), 1);
            mbar_init(p_full(u), 4);              // the owning group's four warps
            mbar_init(p_half(u), 4);
            mbar_init(buf_free(u), 1);            // PV of the buffer's P has completed
        }
        mbar_init(drain(0), 1);
        mbar_init(drain(1), 1);
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
    if (warp >= 3) {
        const int i = threadIdx.x - 96;
        reinterpret_cast<uint4 *>(smem + C::ONES_OFF)[i] = make_uint4(i < 128 ? 0x3F80u : 0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        produce_kv<C>(&tmK, &tmV, a, tb, ntiles, smem, bar0, wt, lane);
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA issue: warp 2 the S MMAs, warp 1 the PV MMAs ----------------
        // (whole warps, elect.sync). S(q + 3) goes into the buffer of PV(q)
        // once PV(q) has completed (buf_free); the two warps issue concurrently.
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait(bar, par));
        };
        constexpr uint32_t idS = idesc_bf16_m128(TILE, 0);
        constexpr uint32_t idPV = idesc_bf16_m128(D, 1);
        const int64_t nq = 2 * ntiles;
        const int me = warp - 1;                 // drain barrier of this warp
        bool ok = true;
        int q_req = -1;                          // newest Q generation requested (warp 2)
        if (warp == 2) {
            // Q of generation u (the u-th (b, h) of the span, both row halves)
            // sits in buffer u & 1; generation u + 1 is fetched once S of
            // generation u - 1 has completed.
            const int bh0 = (int)(tb / pl.T_bh);
            const int last_gen = ntiles > 0 ? (int)((te - 1) / pl.T_bh) - bh0 : -1;
            auto request_q = [&](int u) {
                if (lane == 0) {
                    const int bh = bh0 + u, b = bh / a.H, h = bh - b * a.H;
                    mbar_arrive_expect_tx(q_full(u & 1), 256 * 128);
                    const bool q_ok = dcheck(bh < a.B * a.H && h >= 0 && b >= 0, kChkEncQ, a.status);
                    for (int g = 0; g < 2 && q_ok; ++g)
                        tma_load_4d(sQ + (u & 1) * C::Q_BYTES + g * kAtom, &tmQ, 0, 128 * g, h,
                                    a.q_per_batch ? b : 0, q_full(u & 1));
                }
                __syncwarp();
                q_req = u;
            };
            const volatile uint32_t *padf = reinterpret_cast<const volatile uint32_t *>(smem + C::PADF_OFF);
            TileCursor cs;
            cs.init(pl, tb);
            int s_bh = -1;
            if (ntiles > 0) {
                request_q(0);
                if (last_gen >= 1) request_q(1);
            }
            for (int64_t qs = 0; qs < nq && ok; ++qs) {
                const int64_t j = qs >> 1;
                const int g = (int)(qs & 1);
                const int u = cs.bh - bh0;
                const int s = (int)(j % STAGES);
                const int buf = (int)(qs % 3);
                const bool gen_start = g == 0 && cs.bh != s_bh;
                if (qs >= 3 && !(ok = wwait(buf_free(buf), (uint32_t)(qs / 3 - 1) & 1))) break;
                if (gen_start && !(ok = wwait(q_full(u & 1), (uint32_t)(u >> 1) & 1))) break;
                if (g == 0 && !(ok = wwait(full(s), (uint32_t)(j / STAGES) & 1))) break;
                tc_fence_after();
                const uint32_t tS = tmem + (uint32_t)buf * TILE;
                const bool pad = padf[s] != 0;
                if (pad) umma_bias_elect(tS, sOnes, sBias + s * C::BIAS_BYTES, idS);
                const uint64_t dQ = desc_sw128(sQ + (u & 1) * C::Q_BYTES + g * kAtom, 16, 1024);
                const uint64_t dK = desc_sw128(sStage + s * C::STAGE_BYTES, 16, 1024);
#pragma unroll
                for (int kb = 0; kb < D / 16; ++kb)
                    umma_ss_elect(tS, dQ + (uint64_t)(kb * 32 >> 4), dK + (uint64_t)(kb * 32 >> 4), idS,
                                  (pad || kb > 0) ? 1u : 0u);
                umma_commit_elect(s_full(buf));
                s_bh = cs.bh;
                if (gen_start && u + 1 <= last_gen && q_req < u + 1) {
                    if (u >= 1 && !(ok = wwait(s_full((int)((qs - 1) % 3)), (uint32_t)((qs - 1) / 3) & 1))) break;
                    request_q(u + 1);
                }
                if (g == 1 && j + 1 < ntiles) cs.next(pl);
            }
        } else {
            TileCursor cp;
            cp.init(pl, tb);
            for (int64_t q = 0; q < nq && ok; ++q) {
                const int64_t j = q >> 1;
                const int g = (int)(q & 1);
                const int buf = (int)(q % 3);
                // the first half of P: its PV MMAs overlap the second half's
                // exponentials
                if (!(ok = wwait(p_half(buf), (uint32_t)(q / 3) & 1))) break;
                tc_fence_after();
                // O_g += P V; a piece's first tile starts the accumulator afresh
                const bool first = (j == 0) || cp.k == 0;
                const int s = (int)(j % STAGES);
                const uint64_t dV = desc_sw128(sStage + s * C::STAGE_BYTES + C::KV_ATOM, C::KV_ATOM, 1024);
                const uint32_t tP = tmem + (uint32_t)buf * TILE;
#pragma unroll
                for (int kb = 0; kb < TILE / 16; ++kb) {
                    if (kb == TILE / 32) {
                        if (!(ok = wwait(p_full(buf), (uint32_t)(q / 3) & 1))) break;
                        tc_fence_after();
                    }
                    umma_ts_elect(tmem + C::O_COL + g * D, tP + kb * 8, dV + (uint64_t)(kb * (2048 >> 4)), idPV,
                                  (kb > 0 || !first) ? 1u : 0u);
                }
                if (!ok) break;
                umma_commit_elect(o_done(g));
                umma_commit_elect(buf_free(buf));
                if (g == 1) {
                    umma_commit_elect(empty(s));
                    if (j + 1 < ntiles) cp.next(pl);
                }
            }
        }
        if (wt.aborted()) {
            umma_commit_elect(drain(me));
            if (lane == 0) {
                const uint64_t t0 = globaltimer();
                for (int u = (q_req > 0 ? q_req - 1 : 0); u <= q_req; ++u)
                    while (!mbar_try_wait(q_full(u & 1), (uint32_t)(u >> 1) & 1) &&
                           globaltimer() - t0 < 500000000ull) {
                    }
                while (!mbar_try_wait(drain(me), 0) && globaltimer() - t0 < 500000000ull) {
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- softmax groups (latent-row halves) ----------------
        const int g = (warp - 3) >> 2;            // group: latent rows [128 g, 128 g + 128)
        const int quad = warp & 3;
        const int rig = quad * 32 + lane;
        const int row = g * 128 + rig;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t o_tmem = tmem + C::O_COL + g * D + lane_off;
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait(bar, par));
        };
        float m_ref = -INFINITY, l = 0.f;
        bool has = false;

        auto finalize_piece = [&](const TileCursor &ti, int64_t j) -> bool {
            // the group's PV of the piece's last tile must be complete
            if (!wwait(o_done(g), (uint32_t)j & 1)) return false;
            tc_fence_after();
            const int64_t slot = piece_slot_of(pl, ti, cta);
            const int64_t piece = slot - ((int64_t)ti.bh * pl.R + ti.r) * pl.P_max;
            if (!dcheck(ti.bh < a.B * a.H && piece >= 0 && piece < pl.P_max, kChkEncPiece, a.status))
                return true;                     // FLARE_DEBUG: the write is skipped
            float *part_row = a.part_O + (slot * a.M + row) * D;
            const bool live = l > 0.f;
            const float inv = live ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(o_tmem + c * 32, r);
                tmem_wait_ld();
                float4 *dst = reinterpret_cast<float4 *>(part_row + c * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                         __uint_as_float(r[4 * i + 2]) * inv,
                                         __uint_as_float(r[4 * i + 3]) * inv);
            }
            a.part_L[slot * a.M + row] = live ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            return true;
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
            const int64_t q = 2 * j + g;
            const int buf = (int)(q % 3);
            const uint32_t s_tmem = tmem + (uint32_t)buf * TILE + lane_off;
            if (!wwait(s_full(buf), (uint32_t)(q / 3) & 1)) break;
            tc_fence_after();
            // pass 1: the row maximum (padding is -inf in S already)
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int c0 = 0; c0 < NCH; c0 += 2) {
                uint32_t r[2][32];
                tmem_ld32(s_tmem + c0 * 32, r[0]);
                tmem_ld32(s_tmem + c0 * 32 + 32, r[1]);
                tmem_wait_ld();
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        mx[0] = max3(mx[0], __uint_as_float(r[b][4 * i]), __uint_as_float(r[b][4 * i + 1]));
                        mx[1] = max3(mx[1], __uint_as_float(r[b][4 * i + 2]), __uint_as_float(r[b][4 * i + 3]));
                    }
            }
            const float mt = fmaxf(mx[0], mx[1]) * a.sl2;
            const bool need = mt > m_ref + kTau;
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = need ? mt : m_ref;
                const float f = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
                if (__any_sync(0xffffffffu, has)) {
                    // O holds the group's PV of the previous tile once it completed
                    if (!wwait(o_done(g), (uint32_t)(j - 1) & 1)) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 16; ++c) {
                        uint32_t r[16];
                        tmem_ld16(o_tmem + c * 16, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
                        tmem_st16(o_tmem + c * 16, r);
                    }
                }
                l *= f;
                m_ref = m_new;
            }
            // pass 2: P = exp2(t - m) in bf16 over the buffer's first 64 columns
            // (chunk c of S is loaded before P of chunk c is stored over S
            // columns [16 c, 16 c + 16), which belong to chunks <= c)
            const bool live = __all_sync(0xffffffffu, m_ref != -INFINITY);
            const uint64_t nm2 = live ? f2pack(-m_ref, -m_ref) : f2pack(0.f, 0.f);
            uint64_t ls2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
            for (int c0 = 0; c0 < NCH; c0 += 2) {
                uint32_t r[2][32];
                tmem_ld32(s_tmem + c0 * 32, r[0]);
                tmem_ld32(s_tmem + c0 * 32 + 32, r[1]);
                tmem_wait_ld();
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    uint32_t pw[16];
                    if (live) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            float t0, t1, t2, t3;
                            f2unpack(fma2(f2pack(__uint_as_float(r[b][4 * i]), __uint_as_float(r[b][4 * i + 1])), c2, nm2),
                                     t0, t1);
                            f2unpack(fma2(f2pack(__uint_as_float(r[b][4 * i + 2]), __uint_as_float(r[b][4 * i + 3])), c2, nm2),
                                     t2, t3);
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
                    tmem_st16(s_tmem + (c0 + b) * 16, pw);
                }
                if (c0 + 2 == NCH / 2) {
                    // the first half of P is in place: PV may start on it
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_half(buf));
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(buf));  // one arrival per warp
            {
                float a0, a1, a2, a3;
                f2unpack(ls2[0], a0, a1);
                f2unpack(ls2[1], a2, a3);
                l += (a0 + a1) + (a2 + a3);
            }
            has = true;
            if (last && !finalize_piece(ti, j)) break;
            if (j + 1 < ntiles) ti.next(pl);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
    pdl_launch_dependents();   // the merge may be scheduled (it waits for this grid)
}

// ===============================================================================
// enc_merge_kernel: the partials of every (b, h) into (Z, L) and (O_r, L_r)
// ===============================================================================
// eq. 23 over shards, and the same log-sum-exp rule over the pieces of one
// shard: L_r = log sum_p exp(L_p); L = log sum_r exp(L_r);
// Z = sum_p exp(L_p - L) O_p (= sum_r exp(L_r - L) O_r); O_r = sum_{p in r}
// exp(L_p - L_r) O_p. Rows with no valid token anywhere get L = -inf, Z = 0.
// One block per (b, h) and kMergeRows(D) latent rows; a thread per output quad.
__host__ __device__ constexpr int merge_rows(int D) { return 1024 / D; }
__host__ __device__ constexpr uint32_t merge_smem_bytes(int D) {
    return (uint32_t)((kMergePieces + kMaxShards + 1) * merge_rows(D) * 4);
}

template <int D>
__global__ void __launch_bounds__(256) enc_merge_kernel(const EncArgs a) {
    constexpr int RB = merge_rows(D);          // RB * D / 4 = 256 output quads per block
    constexpr int Q4 = D / 4;
    // launched as a programmatic dependent of the encoder: every global access
    // below comes after the encoder grid has completed
    pdl_wait();
    pdl_launch_dependents();
    const TcTilePlan &pl = a.plan;
    const int M = a.M;
    const int nrb = (M + RB - 1) / RB;
    const int bh = blockIdx.x / nrb, i0 = (blockIdx.x - bh * nrb) * RB;
    const int64_t BH = (int64_t)a.B * a.H;
    extern __shared__ float msm[];
    float *Lp = msm;                           // [kMergePieces][RB] piece log-normalisers
    float *Lr = Lp + kMergePieces * RB;        // [kMaxShards][RB]   shard log-normalisers
    float *Lrow = Lr + kMaxShards * RB;        // [RB]               row log-normalisers
    __shared__ int pstart[kMaxShards + 1];
    __shared__ uint32_t piece[kMergePieces];   // shard << 16 | index within the shard
    const int tid = threadIdx.x;
    for (int r = tid; r < pl.R; r += 256) {
        const int nt = pl.tile_start[r + 1] - pl.tile_start[r];
        int np = 0;
        if (nt > 0) {
            const int64_t u0 = (int64_t)bh * pl.T_bh + pl.tile_start[r];
            np = cta_of(pl, u0 + nt - 1) - cta_of(pl, u0) + 1;
        }
        pstart[r + 1] = np;
    }
    __syncthreads();
    if (tid == 0) {
        pstart[0] = 0;
        for (int r = 0; r < pl.R; ++r) pstart[r + 1] += pstart[r];
    }
    __syncthreads();
    const int P = pstart[pl.R];
    if (P > kMergePieces) {                    // plans keep P within the table
        if (tid == 0) atomicExch(a.status, 2u);
        return;
    }
    for (int r = tid; r < pl.R; r += 256)
        for (int q = pstart[r]; q < pstart[r + 1]; ++q) piece[q] = ((uint32_t)r << 16) | (uint32_t)(q - pstart[r]);
    __syncthreads();
    auto slot = [&](int q) -> int64_t {
        const uint32_t e = piece[q];
        return ((int64_t)bh * pl.R + (e >> 16)) * pl.P_max + (e & 0xffffu);
    };
    if (a.O_r == nullptr && a.L_r == nullptr) {
        // Only (Z, L): every piece of the (b, h) straight into the global rule
        // (the same log-sum-exp, without the per-shard level), one thread per
        // row quad; each batch issues the log-normalisers and outputs of 16
        // pieces together and is folded in with a running maximum, in piece
        // order (deterministic).
        const int i = tid / Q4, d4 = tid - i * Q4;
        if (i0 + i >= M) return;
        const int64_t orow = (int64_t)(i0 + i) * D;
        float m = -INFINITY, sum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int qb = 0; qb < P; qb += 16) {
            float lp[16];
            float4 v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int q = qb + u;
                lp[u] = -INFINITY;
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (q < P) {
                    const int64_t sl = slot(q);
                    lp[u] = __ldcg(a.part_L + sl * M + i0 + i);
                    v[u] = __ldcg(reinterpret_cast<const float4 *>(a.part_O + sl * M * D + orow) + d4);
                }
            }
            float mb = m;
#pragma unroll
            for (int u = 0; u < 16; ++u) mb = fmaxf(mb, lp[u]);
            if (mb == -INFINITY) continue;                 // no valid token so far
            if (mb > m) {
                const float f = m == -INFINITY ? 0.f : expf(m - mb);
                sum *= f;
                acc.x *= f;
                acc.y *= f;
                acc.z *= f;
                acc.w *= f;
                m = mb;
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float w = lp[u] == -INFINITY ? 0.f : expf(lp[u] - m);
                sum += w;
                acc.x = fmaf(w, v[u].x, acc.x);
                acc.y = fmaf(w, v[u].y, acc.y);
                acc.z = fmaf(w, v[u].z, acc.z);
                acc.w = fmaf(w, v[u].w, acc.w);
            }
        }
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
        if (a.Z)
            reinterpret_cast<float4 *>(a.Z + (int64_t)bh * M * D + orow)[d4] =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (a.L && d4 == 0) a.L[(int64_t)bh * M + i0 + i] = sum > 0.f ? m + logf(sum) : -INFINITY;
        return;
    }
    for (int x = tid; x < P * RB; x += 256) {
        const int q = x / RB, i = x - q * RB;
        Lp[x] = (i0 + i < M) ? __ldcg(a.part_L + slot(q) * M + i0 + i) : -INFINITY;
    }
    __syncthreads();
    for (int x = tid; x < pl.R * RB; x += 256) {
        const int r = x / RB, i = x - r * RB;
        float m = -INFINITY;
        for (int q = pstart[r]; q < pstart[r + 1]; ++q) m = fmaxf(m, Lp[q * RB + i]);
        float Lv = -INFINITY;
        if (m != -INFINITY) {
            float sum = 0.f;
            for (int q = pstart[r]; q < pstart[r + 1]; ++q) {
                const float v = Lp[q * RB + i];
                if (v != -INFINITY) sum += expf(v - m);
            }
            Lv = m + logf(sum);
        }
        Lr[x] = Lv;
        if (a.L_r && i0 + i < M) a.L_r[((int64_t)r * BH + bh) * M + i0 + i] = Lv;
    }
    __syncthreads();
    if (tid < RB) {
        float m = -INFINITY;
        for (int r = 0; r < pl.R; ++r) m = fmaxf(m, Lr[r * RB + tid]);
        float Lv = -INFINITY;
        if (m != -INFINITY) {
            float sum = 0.f;
            for (int r = 0; r < pl.R; ++r) {
                const float v = Lr[r * RB + tid];
                if (v != -INFINITY) sum += expf(v - m);
            }
            Lv = m + logf(sum);
        }
        Lrow[tid] = Lv;
        if (a.L && i0 + tid < M) a.L[(int64_t)bh * M + i0 + tid] = Lv;
    }
    __syncthreads();
    const int i = tid / Q4, d4 = tid - i * Q4;
    if (i0 + i >= M) return;
    const int64_t orow = (int64_t)(i0 + i) * D;
    // weighted sum of the pieces [q0, q1) with weights exp(L_p - Lv); the
    // loads of eight pieces are issued together (every piece slot was written
    // by the encoder, empty pieces with zeros, so each load is of defined data)
    auto wsum = [&](int q0, int q1, float Lv) -> float4 {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (Lv == -INFINITY) return acc;
        for (int qb = q0; qb < q1; qb += 8) {
            float4 v[8];
            float w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int q = qb + u;
                w[u] = 0.f;
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (q < q1) {
                    const float lp = Lp[q * RB + i];
                    w[u] = lp == -INFINITY ? 0.f : expf(lp - Lv);
                    v[u] = __ldcg(reinterpret_cast<const float4 *>(a.part_O + slot(q) * M * D + orow) + d4);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                acc.x = fmaf(w[u], v[u].x, acc.x);
                acc.y = fmaf(w[u], v[u].y, acc.y);
                acc.z = fmaf(w[u], v[u].z, acc.z);
                acc.w = fmaf(w[u], v[u].w, acc.w);
            }
        }
        return acc;
    };
    if (a.Z) reinterpret_cast<float4 *>(a.Z + (int64_t)bh * M * D + orow)[d4] = wsum(0, P, Lrow[i]);
    if (a.O_r)
        for (int r = 0; r < pl.R; ++r)
            reinterpret_cast<float4 *>(a.O_r + ((int64_t)r * BH + bh) * M * D + orow)[d4] =
                wsum(pstart[r], pstart[r + 1], Lr[r * RB + i]);
}

}  // namespace tc
}  // namespace flare
