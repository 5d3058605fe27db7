// tc_decode.cuh -- FLARE local decode on sm_103a tensor cores.
//
// Y[b,n,h] = sum_m softmax_m(s <K[b,n,h], Q_m>) Z[b,h,m]  ("FLARE++: Low-rank
// attention with dynamic attention routing", appendix on context parallelism,
// FLARE decode paragraph: each token's query is local, the latent tensors Q
// and Z are replicated). Each token row's softmax runs over the M latents, so
// it is exact in one tile (no running rescale).
//
// One persistent CTA per SM walks a contiguous span of 128-token tiles in
// (h, b, tile) order (head-major: the CTAs of different heads cover the same
// token positions at the same time, so the H head rows of a token, adjacent
// in memory, are fetched together). Warp roles:
//   warp 0     producer: K tiles by TMA into a STAGES-deep ring.
//   warp 1     TMEM allocator and MMA issuer (converged warp, elect.sync):
//                S_g = K Q^T   (A = K tile, B = Q, both shared memory)
//                Y_g = P_g Z   (A = P from tensor memory, B = Z shared memory)
//   warps 2..9 M <= 128: two groups of four warps take alternate tiles (one
//              token row per thread = TMEM lane): row max, exp2, P over S in
//              tensor memory; where 3 M + 2 D columns fit, S rotates through
//              three TMEM buffers so the MMA chain spans three tiles. The
//              epilogue of a tile (Y / l rounded to bf16, staged in shared
//              memory, one TMA store per warp of 32 token rows) runs in the
//              group's next iteration, once that tile's scores have arrived,
//              so the group never waits for its own P Z product.
//              M > 128: two warps per lane quadrant (latent halves, the row
//              maximum exchanged through shared memory); S is single-buffered
//              but free once its scores are read, P (fp16) and Y have columns
//              of their own, so S of tile j + 1 and P Z of tile j - 1 run on
//              the tensor pipe while the softmax of tile j takes its
//              exponentials.
//   warp 10    stager (below).
//   warps 11.. M > 128 only: warps 11..14 the epilogue, one warp per lane
//              quadrant, so the softmax warps never wait for a Y store; warp
//              15 issues the S MMAs (warp 1 then issues only P Z), so S of the
//              next tile never waits behind this tile's P Z issue.
//   stager     converts each (b, h)'s Q and Z into swizzled operand
//              tiles, into one of two buffers while the other is in use, so a
//              (b, h) change does not stall the tile stream.
#pragma once

#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace flare {
namespace tc {

struct DecArgs {
    int B, H, M, N;
    float sl2;                  // score scale * log2(e)
    int q_per_batch;            // Q has a batch dimension
    int q_f32;                  // Q is fp32 (else bf16)
    const void *Q;
    const float *Z;
    __nv_bfloat16 *Y;
    int64_t T_bh;               // tiles per (b, h)
    int64_t T_total;            // tiles over every (b, h)
    int grid;
    unsigned *status;
};

template <int M, int D, int STAGES_, int QZB_>
struct DecCfg {
    static constexpr int STAGES = STAGES_;
    static constexpr int QZB = QZB_;                    // Q/Z buffers (1 or 2)
    static constexpr int KA = D / 64;                   // 64-element atoms along D
    static constexpr int NG = M <= 128 ? 2 : 1;         // softmax groups (tiles in flight)
    // M > 128: one group of eight warps, two per TMEM lane quadrant, each
    // owning M/2 latents of its token rows (a row maximum is exchanged)
    static constexpr int GW = NG == 2 ? 4 : 8;          // warps per group
    static constexpr int STAGER = 2 + 8;                // warp index of the stager
    // M > 128: four more warps (11..14, one per TMEM lane quadrant) take the
    // epilogue, so the softmax warps never wait for a Y store
    static constexpr int EPI0 = STAGER + 1;
    static constexpr int NEPI = NG == 1 ? 4 : 0;
    // M > 128: warp 15 issues the S MMAs, warp 1 only the P Z MMAs (an MMA
    // issue blocks until the tensor pipe accepts it, so one warp issuing both
    // held each tile's S back behind the previous tile's P Z)
    static constexpr int SISS = NG == 1 ? EPI0 + NEPI : -1;
    static constexpr int THREADS = 32 * (STAGER + 1 + NEPI + (NG == 1 ? 1 : 0));
    static constexpr uint32_t QZ_ATOM = M * 128;        // bytes of one M-row x 64-col atom
    // F16P: P and Z enter Y = P Z as fp16, and Z gets one more 16-column block
    // holding the constant c (the power of two Z was scaled by, see
    // stage_z_f16), so the same MMA also returns c * l, the row sum of P,
    // next to c * Y. Needs D + 16 more tensor-memory columns per group.
    // RING (M <= 128): S tiles rotate through three TMEM buffers of M
    // columns (P over the first M/2), each group keeps one Y, when 3 M + 2 D
    // columns fit; fp16 P with the row-sum block when 3 M + 2 (D + 16) fit too.
    static constexpr bool RING = NG == 2 && 3 * M + 2 * D <= 512;
    static constexpr bool F16P = RING ? (3 * M + 2 * (D + 16) <= 512)
                                      : (NG == 2 ? (M + D + 16 <= 256) : (M + D + 16 <= 512));
    static constexpr int YN = F16P ? D + 16 : D;        // N of the P Z product
    static constexpr int ZA = F16P ? KA + 1 : KA;       // atoms of the staged Z
    static constexpr uint32_t QZ_BYTES = (KA + ZA) * QZ_ATOM;   // one Q + Z buffer
    static constexpr uint32_t STAGE_BYTES = KA * 128 * 128;     // one K tile
    static constexpr int NCH = M / 32;                  // P chunks of 32 latents
    // full[S], empty[S], qz_full[2], qz_free[2], s_full[2], p_chunk[2][8], o_done[2],
    // epi_done[2], s_free (M > 128: the single S buffer has been read)
    static constexpr int NBAR = 2 * STAGES + 4 + 2 + 16 + 2 + 2 + 1 + 1 + 1;   // + the third s_full, drain
    static constexpr uint32_t STAGE_OFF = QZB * QZ_BYTES;
    // Y staging of each group for the TMA stores: 128 token rows, KA atoms
    static constexpr uint32_t OUT_OFF = STAGE_OFF + STAGES * STAGE_BYTES;
    static constexpr uint32_t OUT_BYTES = KA * 128 * 128;
    // row maxima of the two latent halves (M > 128), double-buffered by tile parity
    static constexpr uint32_t XMAX_OFF = OUT_OFF + NG * OUT_BYTES;
    static constexpr uint32_t XMAX_BYTES = NG == 1 ? 2 * 2 * 128 * 4 : 0;
    static constexpr uint32_t BAR_OFF = XMAX_OFF + XMAX_BYTES;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t BYTES = MISC_OFF + 64;
    static constexpr uint32_t ALLOC = BYTES + 1024;
    static_assert(ALLOC <= 232448, "shared memory budget of one CTA exceeded");
    // M <= 128: two TMEM buffers b = tile parity, 256 columns each: S (and P
    // over its first M/2 columns) at 256 b, Y at 256 b + Y_COL.
    // M > 128: one S buffer (M columns) at 0, P (fp16 pairs, M/2 columns) at
    // P_COL and Y at Y_COL: S of the next tile is computed as soon as the
    // softmax has read this tile's scores, P waits only for the previous
    // tile's P Z and Y for the previous tile's epilogue.
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t P_COL = NG == 2 ? 0 : M;
    static constexpr uint32_t Y_COL = NG == 2 ? M : M + M / 2;
    static constexpr int NSB = RING ? 3 : (NG == 2 ? 2 : 1);   // S buffers
    // column of S buffer b, and of group g's Y
    static __host__ __device__ constexpr uint32_t s_col(int b) {
        return RING ? (uint32_t)(b * M) : (NG == 2 ? (uint32_t)(b * 256) : 0u);
    }
    static __host__ __device__ constexpr uint32_t y_col(int g) {
        return RING ? (uint32_t)(3 * M + g * YN) : (NG == 2 ? (uint32_t)(g * 256) + Y_COL : Y_COL);
    }
    static_assert(!RING || 3 * M + 2 * YN <= TMEM_COLS, "tensor-memory columns exceeded");
    static_assert(NG == 1 || Y_COL + YN <= 256, "tensor-memory columns of one buffer exceeded");
    static_assert(NG == 2 || Y_COL + YN <= TMEM_COLS, "tensor-memory columns exceeded");
};

// Writes rows [0, M) x D of a row-major matrix into the 128-byte-swizzled bf16
// operand layout (64-column atoms of M rows, 16-byte chunk j of row r at chunk
// position j ^ (r % 8)), by the 32 lanes of one warp. 16-byte loads.
__device__ __forceinline__ uint4 load_chunk8(const __nv_bfloat16 *src) {
    return __ldg(reinterpret_cast<const uint4 *>(src));
}
__device__ __forceinline__ uint4 load_chunk8(const float *src) {
    const float4 lo = __ldg(reinterpret_cast<const float4 *>(src));
    const float4 hi = __ldg(reinterpret_cast<const float4 *>(src) + 1);
    return make_uint4(pack_bf16(lo.x, lo.y), pack_bf16(lo.z, lo.w), pack_bf16(hi.x, hi.y),
                      pack_bf16(hi.z, hi.w));
}
// Threads t0, t0 + step, ... of the cooperating threads take the chunks.
template <int M, int D, typename T>
__device__ __forceinline__ void stage_rows_bf16(uint8_t *dst, const T *src, int t0, int step) {
    constexpr int CHUNKS = M * D / 8;                   // 16-byte output chunks
#pragma unroll 8
    for (int c = t0; c < CHUNKS; c += step) {
        const int row = c / (D / 8), j = c % (D / 8);    // chunk j covers cols 8j..8j+7
        const int atom = j >> 3, jj = j & 7;
        uint8_t *p = dst + atom * (M * 128) + row * 128 + ((jj ^ (row & 7)) << 4);
        *reinterpret_cast<uint4 *>(p) = load_chunk8(src + (int64_t)row * D + 8 * j);
    }
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x) {
    uint32_t y;
    asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Z [M, D] fp32 -> the fp16 operand layout of stage_rows_bf16, multiplied by
// c = 2^-e where 2^e <= max|Z| < 2^(e+1) (e clamped to [-14, 24], so c and
// every scaled element stay within fp16 range), plus atom D/64 whose first
// column is c in every row (the row-sum block). c cancels in Y = (c Y)/(c l).
// In two steps so that several warps can share them: z_absmax_part (this
// thread's share of max|Z|), then z_stage_f16 with c = z_scale(max|Z|).
template <int M, int D>
__device__ __forceinline__ float z_absmax_part(const float *src, int t0, int step) {
    constexpr int CHUNKS = M * D / 8;
    float mx = 0.f;
#pragma unroll 8
    for (int q = t0; q < CHUNKS; q += step) {
        const float4 lo = __ldg(reinterpret_cast<const float4 *>(src) + 2 * q);
        const float4 hi = __ldg(reinterpret_cast<const float4 *>(src) + 2 * q + 1);
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(lo.x), fabsf(lo.y)), fmaxf(fabsf(lo.z), fabsf(lo.w))));
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(hi.x), fabsf(hi.y)), fmaxf(fabsf(hi.z), fabsf(hi.w))));
    }
    return mx;
}
__device__ __forceinline__ float z_scale(float mx) {
    int e = mx > 0.f ? ((__float_as_int(mx) >> 23) & 0xff) - 127 : 0;   // floor(log2 max|Z|)
    e = e < -14 ? -14 : (e > 24 ? 24 : e);
    return __int_as_float((127 - e) << 23);                            // 2^-e, exact
}
template <int M, int D>
__device__ __forceinline__ void z_stage_f16(uint8_t *dst, const float *src, float c, int t0, int step) {
    constexpr int CHUNKS = M * D / 8;
#pragma unroll 8
    for (int q = t0; q < CHUNKS; q += step) {
        const int row = q / (D / 8), j = q % (D / 8);
        const int atom = j >> 3, jj = j & 7;
        const float4 lo = __ldg(reinterpret_cast<const float4 *>(src) + 2 * q);
        const float4 hi = __ldg(reinterpret_cast<const float4 *>(src) + 2 * q + 1);
        *reinterpret_cast<uint4 *>(dst + atom * (M * 128) + row * 128 + ((jj ^ (row & 7)) << 4)) =
            make_uint4(pack_f16(lo.x * c, lo.y * c), pack_f16(lo.z * c, lo.w * c),
                       pack_f16(hi.x * c, hi.y * c), pack_f16(hi.z * c, hi.w * c));
    }
    // the row-sum block: columns D..D+15 = [c, 0, ..., 0] (chunks 0 and 1 of the atom)
    uint8_t *ones = dst + (D / 64) * (M * 128);
    for (int row = t0; row < M; row += step) {
        *reinterpret_cast<uint4 *>(ones + row * 128 + ((0 ^ (row & 7)) << 4)) = make_uint4(pack_f16(c, 0.f), 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(ones + row * 128 + ((1 ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Q and Z of (b, h) index bh (head-major: bh = h * B + b) into Q/Z buffer q,
// by the 32 lanes of one warp (the stager, for every (b, h) after the first).
// Not inlined: it runs once per (b, h) and would otherwise add its registers
// to the tile loops'.
template <class C, int M, int D>
__device__ __noinline__ void dec_stage_qz(uint8_t *smem, const void *Q, const float *Z, int q_f32,
                                          int q_per_batch, int B, int H, int64_t bh, int q, int lane) {
    const int t0 = lane, step = 32;
    constexpr int KA = C::KA;
    const int h = (int)(bh / B), b = (int)(bh - (int64_t)h * B);
    uint8_t *qdst = smem + q * C::QZ_BYTES, *zdst = qdst + KA * C::QZ_ATOM;
    const int64_t qoff = ((int64_t)(q_per_batch ? b : 0) * H + h) * M * D;
    const float *zsrc = Z + ((int64_t)b * H + h) * M * D;
    if (q_f32)
        stage_rows_bf16<M, D>(qdst, reinterpret_cast<const float *>(Q) + qoff, t0, step);
    else
        stage_rows_bf16<M, D>(qdst, reinterpret_cast<const __nv_bfloat16 *>(Q) + qoff, t0, step);
    if constexpr (C::F16P) {
        float mx = z_absmax_part<M, D>(zsrc, t0, step);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        z_stage_f16<M, D>(zdst, zsrc, z_scale(mx), t0, step);
    } else {
        stage_rows_bf16<M, D>(zdst, zsrc, t0, step);
    }
}

// The first (b, h), staged by the cooperating warps 2..STAGER in one pass:
// every thread loads all of its Q and Z chunks before it stores any (one
// round trip to memory instead of one per matrix and pass), max|Z| (fp16 Z)
// is combined through shared memory, and the chunks go to shared memory from
// registers. Thread t0 takes chunks t0, t0 + STEP, ...
template <class C, int M, int D>
__device__ __noinline__ void dec_stage_qz_first(uint8_t *smem, const void *Q, const float *Z, int q_f32,
                                                int q_per_batch, int B, int H, int64_t bh, int t0, int wid,
                                                int lane) {
    constexpr int KA = C::KA, CHUNKS = M * D / 8, STEP = 32 * (C::STAGER - 1);
    constexpr int NC = (CHUNKS + STEP - 1) / STEP;
    const int h = (int)(bh / B), b = (int)(bh - (int64_t)h * B);
    uint8_t *qdst = smem, *zdst = smem + KA * C::QZ_ATOM;   // Q/Z buffer 0
    const int64_t qoff = ((int64_t)(q_per_batch ? b : 0) * H + h) * M * D;
    const float4 *zsrc = reinterpret_cast<const float4 *>(Z + ((int64_t)b * H + h) * M * D);
    uint4 qv[NC];
    float4 zv[NC][2];
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const int c = t0 + i * STEP;   // chunk c: elements 8c .. 8c + 7 of the row-major matrix
        if (c < CHUNKS) {
            qv[i] = q_f32 ? load_chunk8(reinterpret_cast<const float *>(Q) + qoff + 8 * c)
                          : load_chunk8(reinterpret_cast<const __nv_bfloat16 *>(Q) + qoff + 8 * c);
            zv[i][0] = __ldg(zsrc + 2 * c);
            zv[i][1] = __ldg(zsrc + 2 * c + 1);
        }
    }
    float cz = 1.f;
    if constexpr (C::F16P) {
        float mx = 0.f;
#pragma unroll
        for (int i = 0; i < NC; ++i)
            if (t0 + i * STEP < CHUNKS)
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(zv[i][k].x), fabsf(zv[i][k].y)),
                                         fmaxf(fabsf(zv[i][k].z), fabsf(zv[i][k].w))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float *xz = reinterpret_cast<float *>(smem + C::MISC_OFF + 16);   // one per warp
        if (lane == 0) xz[wid] = mx;
        named_bar_sync(5, STEP);
#pragma unroll
        for (int w = 0; w < C::STAGER - 1; ++w) mx = fmaxf(mx, xz[w]);
        cz = z_scale(mx);
    }
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const int c = t0 + i * STEP;
        if (c < CHUNKS) {
            const int row = c / (D / 8), j = c % (D / 8);
            const uint32_t o = (uint32_t)((j >> 3) * (M * 128) + row * 128 + (((j & 7) ^ (row & 7)) << 4));
            *reinterpret_cast<uint4 *>(qdst + o) = qv[i];
            const float4 lo = zv[i][0], hi = zv[i][1];
            *reinterpret_cast<uint4 *>(zdst + o) =
                C::F16P ? make_uint4(pack_f16(lo.x * cz, lo.y * cz), pack_f16(lo.z * cz, lo.w * cz),
                                     pack_f16(hi.x * cz, hi.y * cz), pack_f16(hi.z * cz, hi.w * cz))
                        : make_uint4(pack_bf16(lo.x, lo.y), pack_bf16(lo.z, lo.w), pack_bf16(hi.x, hi.y),
                                     pack_bf16(hi.z, hi.w));
        }
    }
    if constexpr (C::F16P) {
        // the row-sum block: columns D..D+15 = [c, 0, ..., 0]
        uint8_t *ones = zdst + KA * (M * 128);
        for (int row = t0; row < M; row += STEP) {
            *reinterpret_cast<uint4 *>(ones + row * 128 + ((0 ^ (row & 7)) << 4)) = make_uint4(pack_f16(cz, 0.f), 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(ones + row * 128 + ((1 ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

template <int M, int D, int STAGES, int QZB_>
__global__ void __launch_bounds__(DecCfg<M, D, STAGES, QZB_>::THREADS, 1)
dec_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmY,
                  const DecArgs a) {
    using C = DecCfg<M, D, STAGES, QZB_>;
    constexpr int KA = C::KA, NG = C::NG, NCH = C::NCH, QZB = C::QZB;
    static_assert(QZB == 1 || QZB == 2, "one or two Q/Z buffers");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem), sStage = sbase + C::STAGE_OFF;
    const uint32_t bar0 = sbase + C::BAR_OFF;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto qz_full = [&](int q) { return bar0 + 8u * (2 * STAGES + q); };
    auto qz_free = [&](int q) { return bar0 + 8u * (2 * STAGES + 2 + q); };
    auto s_full = [&](int g) { return bar0 + 8u * (2 * STAGES + (g < 2 ? 4 + g : 27)); };
    auto p_chunk = [&](int g, int c) { return bar0 + 8u * (2 * STAGES + 6 + 8 * g + c); };
    auto o_done = [&](int g) { return bar0 + 8u * (2 * STAGES + 22 + g); };
    auto epi_done = [&](int g) { return bar0 + 8u * (2 * STAGES + 24 + g); };
    const uint32_t s_free = bar0 + 8u * (2 * STAGES + 26);
    const uint32_t drain_s = bar0 + 8u * (2 * STAGES + 28);   // M > 128: the S issuer's MMAs
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int64_t tb = ((int64_t)cta * a.T_total + a.grid - 1) / a.grid;
    const int64_t te = ((int64_t)(cta + 1) * a.T_total + a.grid - 1) / a.grid;
    const int64_t ntiles = te - tb;
    Waiter wt{abort_flag, a.status};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(qz_full(q), 1);
            mbar_init(qz_free(q), 1);
        }
        for (int g = 0; g < 2; ++g) {
            // one arrival per warp that reads Y: the softmax warps (M <= 128),
            // the four epilogue warps (M > 128)
            mbar_init(epi_done(g), NG == 1 ? C::NEPI : C::GW);
            mbar_init(s_full(g), 1);
            for (int c = 0; c < 8; ++c) mbar_init(p_chunk(g, c), C::GW);   // one arrival per softmax warp
            mbar_init(o_done(g), 1);
        }
        mbar_init(s_full(2), 1);
        mbar_init(s_free, C::GW);            // M > 128: every softmax warp has read S
        mbar_init(drain_s, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmY);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // first tile: its (b, h) index (head-major: bh = h * B + b) and token tile
    const int64_t bh0 = tb / a.T_bh;
    const int64_t k0 = tb - bh0 * a.T_bh;
    const int64_t n_gen = ntiles > 0 ? (te - 1) / a.T_bh - bh0 + 1 : 0;   // (b, h) of the span
    // The first (b, h) is staged by warps 2..STAGER together (idle until its
    // first S anyway). Inside the library's forward the decode is launched as
    // a programmatic dependent of the merge that writes Z: only these warps
    // read Z or Q, so only they wait, and the K stream starts during the
    // merge's tail.
    if (warp >= 2 && warp <= C::STAGER && n_gen > 0) {
        pdl_wait();
        const int wid = warp - 2;
        dec_stage_qz_first<C, M, D>(smem, a.Q, a.Z, a.q_f32, a.q_per_batch, a.B, a.H, bh0, 32 * wid + lane, wid,
                                    lane);
        fence_proxy_async_smem();
        named_bar_sync(5, 32 * (C::STAGER - 1));
        if (warp == C::STAGER && lane == 0) mbar_arrive(qz_full(0));
    }

    if (warp == 0) {
        // ---------------- producer: K tiles ----------------
        const uint64_t pol = policy_evict_first();
        int64_t kt = k0;
        int h = (int)(bh0 / a.B), b = (int)(bh0 - (int64_t)h * a.B);   // tile j's head and batch
        int64_t j = 0;
        for (; j < ntiles && !wt.aborted(); ++j) {
            const int s = (int)(j % STAGES);
            if (!__all_sync(0xffffffffu, wt.wait(empty(s), ((uint32_t)(j / STAGES) & 1) ^ 1))) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(full(s), C::STAGE_BYTES);
                const uint32_t dst = sStage + s * C::STAGE_BYTES;
                const bool ok_k = dcheck(tile_in_tensor(64 * (KA - 1), h, kt * 128, b, a.H, a.N, a.B) && kt < a.T_bh,
                                         kChkDecK, a.status);
                for (int ka = 0; ka < KA && ok_k; ++ka)
                    tma_load_4d_hint(dst + ka * (128 * 128), &tmK, 64 * ka, h, (int)(kt * 128), b, full(s), pol);
            }
            __syncwarp();
            if (++kt == a.T_bh) {
                kt = 0;
                if (++b == a.B) {             // head-major: bh = h * B + b
                    b = 0;
                    ++h;
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
        }
    } else if (warp == C::STAGER) {
        // ---------------- stager: Q and Z of each later (b, h) ----------------
        for (int64_t u = 1; u < n_gen && !wt.aborted(); ++u) {
            const int q = (int)(u % QZB);
            // the buffer's previous (b, h) has had its last P Z issued and done
            if (u >= QZB && !__all_sync(0xffffffffu, wt.wait(qz_free(q), (uint32_t)(u / QZB - 1) & 1))) break;
            dec_stage_qz<C, M, D>(smem, a.Q, a.Z, a.q_f32, a.q_per_batch, a.B, a.H, bh0 + u, (int)(u % QZB),
                                  lane);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qz_full(q));
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (whole warp, elect.sync issues) ----------------
        // The warp stays converged so that its operands stay warp-uniform.
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait(bar, par));
        };
        // M > 128: the waits on the softmax warps' arrivals spin (test_wait)
        // instead of suspending in try_wait: a suspended issuer woke ~1000
        // cycles after the last arrival, and each tile's P Z waited on it
        auto wspin = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.spin(bar, par));
        };
        constexpr uint32_t idS = idesc_bf16_m128(M, 0);
        // P Z: bf16, or fp16 with the row-sum block (N = D + 16)
        constexpr uint32_t idPV = C::F16P ? idesc_f16(128, C::YN, 0, 1) : idesc_bf16_m128(D, 1);
        const uint64_t dK0 = desc_sw128(sStage, 16, 1024);
        constexpr uint64_t kStageDesc = C::STAGE_BYTES >> 4;
        int64_t bhS = bh0, ktS = k0;                 // cursor of the S tiles
        int64_t bhP = bh0, ktP = k0;                 // cursor of the PV tiles
        int64_t uS = -1, uP = 0;                     // (b, h) generation of each cursor
        bool ok = true;
        auto issue_s = [&](int64_t jj) -> bool {
            const int s = (int)(jj % STAGES);
            if (bhS - bh0 != uS) {
                uS = bhS - bh0;
                if (!wwait(qz_full((int)(uS % QZB)), (uint32_t)(uS / QZB) & 1)) return false;
            }
            if (!wwait(full(s), (uint32_t)(jj / STAGES) & 1)) return false;
            tc_fence_after();
            const int g = C::RING ? (int)(jj % 3) : (NG == 1 ? 0 : (int)(jj & 1));   // S buffer
            // M > 128: the single S buffer is free once the previous tile's scores are read
            if (NG == 1 && jj >= 1 && !wwait(s_free, (uint32_t)(jj - 1) & 1)) return false;
            tc_fence_after();
            const uint64_t dK = dK0 + kStageDesc * s;
            const uint64_t dQ0 = desc_sw128(sbase + (uint32_t)(uS % QZB) * C::QZ_BYTES, 16, 1024);
#pragma unroll
            for (int kb = 0; kb < D / 16; ++kb) {
                const uint64_t offK = (uint64_t)((kb >> 2) * (128 * 128) + (kb & 3) * 32) >> 4;
                const uint64_t offQ = (uint64_t)((kb >> 2) * C::QZ_ATOM + (kb & 3) * 32) >> 4;
                umma_ss_elect(tmem + C::s_col(g), dK + offK, dQ0 + offQ, idS, kb > 0 ? 1u : 0u);
            }
            umma_commit_elect(s_full(g));
            umma_commit_elect(empty(s));            // the K tile is only read by S
            if (++ktS == a.T_bh) {
                ktS = 0;
                ++bhS;
            }
            return true;
        };
        // S runs at most NG tiles ahead of PV; with a single Q/Z buffer the S of
        // a new (b, h) also waits until every older tile's P Z is issued
        int64_t jS = 0, nP = 0;
        auto pump_s = [&]() -> bool {
            if (NG == 1) return true;                // M > 128: the S issuer warp
            while (jS < ntiles && jS < nP + (C::RING ? 3 : 2) && (QZB == 2 || bhS - bh0 == uS || nP == jS))
                if (!issue_s(jS++)) return false;
            return true;
        };
        ok = pump_s();
        for (; nP < ntiles && ok;) {
            const int64_t jP = nP;
            const int g = NG == 1 ? 0 : (int)(jP & 1);
            const int64_t kP = NG == 1 ? jP : jP >> 1;
            const uint64_t dZ0 = desc_sw128(sbase + (uint32_t)(uP % QZB) * C::QZ_BYTES + KA * C::QZ_ATOM,
                                            C::QZ_ATOM, 1024);
            for (int c = 0; c < NCH && ok; ++c) {
                // P arrives whole, published by every softmax warp at once
                if (c == 0) {
                    ok = NG == 1 ? wspin(p_chunk(g, 0), (uint32_t)kP & 1) : wwait(p_chunk(g, 0), (uint32_t)kP & 1);
                    // M > 128: Y of the previous tile has been read by its epilogue
                    if (ok && NG == 1 && jP >= 1) ok = wspin(epi_done(0), (uint32_t)(jP - 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                }
                const uint32_t y_t = tmem + C::y_col(g);
                const uint32_t p_t = NG == 1 ? tmem + C::P_COL : tmem + C::s_col(C::RING ? (int)(jP % 3) : g);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int kb = 2 * c + kk;       // 16 latents per MMA
                    umma_ts_elect(y_t, p_t + kb * 8, dZ0 + kb * (2048 >> 4), idPV, kb > 0 ? 1u : 0u);
                }
            }
            if (!ok) break;
            umma_commit_elect(o_done(g));
            if (++ktP == a.T_bh) {
                ktP = 0;
                ++bhP;
            }
            ++nP;
            if (nP == ntiles || bhP - bh0 != uP) {
                umma_commit_elect(qz_free((int)(uP % QZB)));   // this (b, h)'s Q and Z are done
                ++uP;
            }
            ok = pump_s();
        }
        // make every issued MMA finish before TMEM is released
        if (ok && ntiles > 0) {
            const int gl = NG == 1 ? 0 : (int)((ntiles - 1) & 1);
            const int64_t kl = NG == 1 ? ntiles - 1 : (ntiles - 1) >> 1;
            wwait(o_done(gl), (uint32_t)kl & 1);
        }
        __syncwarp();
    } else if (NG == 1 && warp < C::STAGER) {
        // ---------------- softmax halves (M > 128) ----------------
        // Warps w and w + 4 share a TMEM lane quadrant (32 token rows); half h
        // owns latents [M/2 h, M/2 (h + 1)). Per tile j: a first pass over
        // the half's scores (32 columns at a time) gives its row maximum,
        // which the halves exchange; a second pass turns the scores into the
        // fp16 exponents t = s log2(e) S - m, packed in pairs; then S is
        // free (s_free: S of tile j + 1 may be computed) and the exponentials
        // are taken in registers while the tensor pipe still runs P Z of tile
        // j - 1. Once that product is done P's columns are free and P of tile
        // j is stored (which starts its P Z). Two passes over tensor memory
        // keep a thread's registers at one chunk of scores plus the packed
        // exponents; the epilogue warps take Y.
        constexpr int HM = M / 2;                     // latents of a half
        constexpr int NC = HM / 32;                   // 32-column chunks of a half
        const int half = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int rig = quad * 32 + lane;             // token row within the tile
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint64_t c2 = f2pack(a.sl2, a.sl2);
        float *xmax = reinterpret_cast<float *>(smem + C::XMAX_OFF);   // [2 parity][2 half][128 rows]
        const int pair_bar = 1 + quad;                // named barrier of the quadrant's two warps
        const uint32_t s_tmem = tmem + HM * half + lane_off;
        const uint32_t p_tmem = tmem + C::P_COL + (HM / 2) * half + lane_off;
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait(bar, par));
        };
        for (int64_t j = 0; j < ntiles; ++j) {
            if (!wwait(s_full(0), (uint32_t)j & 1)) break;
            tc_fence_after();
            // pass 1: the half's row maximum
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < NC; c += 2) {
                uint32_t r[2][32];
                tmem_ld32(s_tmem + c * 32, r[0]);
                tmem_ld32(s_tmem + c * 32 + 32, r[1]);
                tmem_wait_ld();
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        mx[(2 * b) & 3] = max3(mx[(2 * b) & 3], __uint_as_float(r[b][4 * i]), __uint_as_float(r[b][4 * i + 1]));
                        mx[(2 * b + 1) & 3] = max3(mx[(2 * b + 1) & 3], __uint_as_float(r[b][4 * i + 2]), __uint_as_float(r[b][4 * i + 3]));
                    }
            }
            float *xm = xmax + (j & 1) * 256;
            xm[half * 128 + rig] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            named_bar_sync(pair_bar, 64);                 // both halves' maxima are published
            const float m = fmaxf(xm[rig], xm[128 + rig]) * a.sl2;
            const uint64_t nm2 = f2pack(-m, -m);
            // pass 2: the exponents in fp16 pairs
            uint32_t pw[NC][16];
#pragma unroll
            for (int c = 0; c < NC; c += 2) {
                uint32_t r[2][32];
                tmem_ld32(s_tmem + c * 32, r[0]);
                tmem_ld32(s_tmem + c * 32 + 32, r[1]);
                tmem_wait_ld();
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float t0, t1;
                        f2unpack(fma2(f2pack(__uint_as_float(r[b][2 * i]), __uint_as_float(r[b][2 * i + 1])), c2, nm2), t0, t1);
                        pw[c + b][i] = pack_f16(t0, t1);
                    }
            }
            // the scores are read: S of the next tile may be computed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
                for (int i = 0; i < 16; ++i) pw[c][i] = ex2_f16x2(pw[c][i]);
            // P's columns are free once the previous tile's P Z is done (an
            // inline wait: P is live in registers, and registers live across
            // the out-of-line wait's call would be saved to memory)
            if (j > 0 && !__all_sync(0xffffffffu, wt.wait_inline(o_done(0), (uint32_t)(j - 1) & 1))) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < NC; ++c) tmem_st16(p_tmem + c * 16, pw[c]);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_chunk(0, 0));
        }
    } else if (NG == 1 && warp == C::SISS) {
        // ---------------- S issuer (M > 128; whole warp, elect.sync issues) ----------------
        // S of tile j once its K tile has landed, the single S buffer has been
        // read by the softmax (s_free of tile j - 1) and, at the first tile of
        // a (b, h), the stager has put that (b, h)'s Q in place.
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait(bar, par));
        };
        // the wait for the softmax warps' reads spins (see the P Z issuer)
        auto wspin = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.spin(bar, par));
        };
        constexpr uint32_t idS = idesc_bf16_m128(M, 0);
        const uint64_t dK0 = desc_sw128(sStage, 16, 1024);
        constexpr uint64_t kStageDesc = C::STAGE_BYTES >> 4;
        int64_t ktS = k0, u = 0;
        bool issued = false;
        for (int64_t jj = 0; jj < ntiles; ++jj) {
            const int s = (int)(jj % STAGES);
            if (jj == 0 || ktS == 0) {
                if (jj > 0) ++u;
                if (!wwait(qz_full((int)(u % QZB)), (uint32_t)(u / QZB) & 1)) break;
            }
            if (!wwait(full(s), (uint32_t)(jj / STAGES) & 1)) break;
            if (jj >= 1 && !wspin(s_free, (uint32_t)(jj - 1) & 1)) break;
            tc_fence_after();
            const uint64_t dK = dK0 + kStageDesc * s;
            const uint64_t dQ0 = desc_sw128(sbase + (uint32_t)(u % QZB) * C::QZ_BYTES, 16, 1024);
#pragma unroll
            for (int kb = 0; kb < D / 16; ++kb) {
                const uint64_t offK = (uint64_t)((kb >> 2) * (128 * 128) + (kb & 3) * 32) >> 4;
                const uint64_t offQ = (uint64_t)((kb >> 2) * C::QZ_ATOM + (kb & 3) * 32) >> 4;
                umma_ss_elect(tmem + C::s_col(0), dK + offK, dQ0 + offQ, idS, kb > 0 ? 1u : 0u);
            }
            umma_commit_elect(s_full(0));
            umma_commit_elect(empty(s));            // the K tile is only read by S
            issued = true;
            if (++ktS == a.T_bh) ktS = 0;
        }
        // every S this warp issued completes before TMEM is released
        if (issued) {
            umma_commit_elect(drain_s);
            wwait(drain_s, 0);
        }
        __syncwarp();
    } else if (NG == 1) {
        // ---------------- epilogue (M > 128) ----------------
        // One warp per TMEM lane quadrant: once P Z of tile j is done it reads
        // the quadrant's 32 rows of Y and c * l (then Y is free for the next
        // tile's P Z), divides, rounds to bf16 into its shared-memory slab and
        // stores the 32 token rows with one TMA store.
        const int quad = warp & 3;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t y_tmem = tmem + C::Y_COL + lane_off;
        uint8_t *slab = smem + C::OUT_OFF + quad * 32 * 128;         // the quadrant's 32 Y rows
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait(bar, par));
        };
        int64_t kt = k0;
        int ch = (int)(bh0 / a.B), cb = (int)(bh0 - (int64_t)ch * a.B);   // tile j's head and batch
        for (int64_t j = 0; j < ntiles; ++j) {
            if (!wwait(o_done(0), (uint32_t)j & 1)) break;
            tc_fence_after();
            uint32_t yr[2][32];
            tmem_ld32(y_tmem, yr[0]);
            tmem_ld32(y_tmem + 32, yr[1]);
            const uint32_t lw = tmem_ld1(y_tmem + D);             // c * l from the row-sum block
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(epi_done(0));               // Y may take the next tile's P Z
            // the slab is free once the warp's previous store has read it
            if (j > 0) {
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
            }
            const float inv = 1.f / __uint_as_float(lw);
            uint8_t *row = slab + lane * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int chunk = 4 * h + q;
                    const uint32_t *v = yr[h] + 8 * q;
                    *reinterpret_cast<uint4 *>(row + ((chunk ^ (lane & 7)) << 4)) = make_uint4(
                        pack_bf16(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                        pack_bf16(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                        pack_bf16(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                        pack_bf16(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
                }
            fence_proxy_async_smem();
            __syncwarp();
            const int n0 = (int)(kt * 128) + quad * 32;
            if (lane == 0 && n0 < a.N &&
                dcheck(tile_in_tensor(0, ch, n0, cb, a.H, a.N, a.B), kChkDecY, a.status)) {
                // token rows past N are clipped by the tensor map
                tma_store_4d(&tmY, smem_u32(slab), 0, ch, n0, cb);
                bulk_commit_group();
            }
            if (++kt == a.T_bh) {
                kt = 0;
                if (++cb == a.B) {
                    cb = 0;
                    ++ch;
                }
            }
        }
        if (lane == 0) bulk_wait_group0();
    } else {
        // ---------------- softmax + epilogue warps ----------------
        const int g = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int rig = quad * 32 + lane;            // token row within the tile (TMEM lane)
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t y_tmem = tmem + C::y_col(g) + lane_off;
        const uint64_t c2 = f2pack(a.sl2, a.sl2);
        // each warp stages and stores its own 32 token rows (a 4 KB slab per atom)
        uint8_t *stage_out = smem + C::OUT_OFF + g * C::OUT_BYTES + quad * 32 * 128;
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, wt.wait(bar, par));
        };
        // the group's previous tile, whose Y is still in tensor memory
        bool have_prev = false;
        int prev_b = 0, prev_h = 0, prev_n0 = 0;
        int64_t prev_k = 0;
        float prev_l = 1.f;
        uint32_t stores = 0;
        auto epilogue = [&]() -> bool {
            if (!wwait(o_done(g), (uint32_t)prev_k & 1)) return false;
            tc_fence_after();
            uint32_t r[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32(y_tmem + c * 32, r[c]);
            uint32_t lw = 0;
            if constexpr (C::F16P) lw = tmem_ld1(y_tmem + D);    // c * l from the row-sum block
            tmem_wait_ld();
            tc_fence_before();
            // the staging slab is free once the warp's previous store has read it
            if (stores > 0) {
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
            }
            const float inv = 1.f / (C::F16P ? __uint_as_float(lw) : prev_l);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint8_t *row = stage_out + (c >> 1) * (128 * 128) + lane * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int chunk = 4 * (c & 1) + q;
                    const uint32_t *v = r[c] + 8 * q;
                    *reinterpret_cast<uint4 *>(row + ((chunk ^ (rig & 7)) << 4)) = make_uint4(
                        pack_bf16(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                        pack_bf16(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                        pack_bf16(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                        pack_bf16(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            const int n0 = prev_n0 + quad * 32;
            if (lane == 0 && n0 < a.N &&
                dcheck(tile_in_tensor(64 * (KA - 1), prev_h, n0, prev_b, a.H, a.N, a.B), kChkDecY, a.status)) {
                // token rows past N are clipped by the tensor map
#pragma unroll
                for (int ka = 0; ka < KA; ++ka)
                    tma_store_4d(&tmY, smem_u32(stage_out) + ka * (128 * 128), 64 * ka, prev_h, n0, prev_b);
                bulk_commit_group();
            }
            ++stores;
            return true;
        };
        int64_t bh = bh0, kt = k0;
        int ch = (int)(bh0 / a.B), cb = (int)(bh0 - (int64_t)ch * a.B);   // tile j's head and batch
        bool ok = true;
        for (int64_t j = 0; j < ntiles && ok; ++j) {
            const bool mine = NG == 1 || (int)(j & 1) == g;
            if (mine) {
                const int64_t k = NG == 2 ? (j >> 1) : j;
                const int sb = C::RING ? (int)(j % 3) : g;        // S buffer of tile j
                const uint32_t s_tmem = tmem + C::s_col(sb) + lane_off;
                if (!wwait(s_full(sb), (uint32_t)(C::RING ? j / 3 : k) & 1)) break;
                tc_fence_after();
                if (have_prev && !(ok = epilogue())) break;
                float l;
                {
                    // every score of the row in registers: one load, max, exp
                    uint32_t r[NCH][32];
#pragma unroll
                    for (int c = 0; c < NCH; ++c) tmem_ld32(s_tmem + c * 32, r[c]);
                    tmem_wait_ld();
                    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            mx[i & 1] = max3(mx[i & 1], __uint_as_float(r[c][2 * i]), __uint_as_float(r[c][2 * i + 1]));
                    const float m = fmaxf(mx[0], mx[1]) * a.sl2;
                    const uint64_t nm2 = f2pack(-m, -m);
                    if constexpr (C::F16P) {
                        // P = exp2(t) two at a time in fp16; the row sum comes from the MMA
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            uint32_t pw[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                float t0, t1;
                                f2unpack(fma2(f2pack(__uint_as_float(r[c][2 * i]), __uint_as_float(r[c][2 * i + 1])), c2, nm2), t0, t1);
                                pw[i] = ex2_f16x2(pack_f16(t0, t1));
                            }
                            tmem_st16(s_tmem + c * 16, pw);
                        }
                        l = 1.f;
                    } else {
                        uint64_t ls2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            uint32_t pw[16];
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
                            tmem_st16(s_tmem + c * 16, pw);
                        }
                        float a0, a1, a2, a3;
                        f2unpack(ls2[0], a0, a1);
                        f2unpack(ls2[1], a2, a3);
                        l = (a0 + a1) + (a2 + a3);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_chunk(g, 0));
                }
                have_prev = true;
                prev_h = ch;
                prev_b = cb;
                prev_n0 = (int)(kt * 128);
                prev_k = k;
                prev_l = l;
            }
            if (++kt == a.T_bh) {
                kt = 0;
                ++bh;
                if (++cb == a.B) {
                    cb = 0;
                    ++ch;
                }
            }
        }
        if (ok && have_prev && !wt.aborted()) epilogue();
        if (lane == 0) bulk_wait_group0();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace tc
}  // namespace flare
