// simt_kernels.cu -- CUDA-core (FFMA) kernels of the FLARE token mixer.
//
// These serve the fp32 path (the tensor cores offer no fp32-exact product)
// and every shape the tensor-core kernels do not cover. They follow the same
// definitions as the tensor-core kernels:
//   encoder  -- per-shard local encoder and eq. 23 of the FLARE++
//               context-parallel appendix, computed per token chunk with an
//               online softmax (scores are never stored), then merged;
//   merge    -- the cross-rank log-sum-exp rule (L_max, a, U, Z = U/a);
//   decode   -- the local decode, each token's key querying the M latents;
//   backward -- the global-normaliser backward (P with the global L, the row
//               scalar c, dV, dS, dK, and dQ summed over all tokens).
// Warp-shuffle reductions carry the row max and row sum of every softmax.
#include "flare_internal.cuh"

#include <math.h>

namespace flare {
namespace {

constexpr int kThreads = 128;        // 4 warps (backward kernels)
// The encoder and decode spread a tile's 32 rows over 16 warps of 2 rows:
// each warp's chain of dependent steps (dot products, shuffle reductions,
// exponentials, broadcasts) is short, and a small problem, where each SM
// holds one CTA, still has four warps per sub-partition to interleave.
constexpr int kFwdThreads = 512;
constexpr int kRowsPerWarp = 2;      // 16 warps x 2 rows = kSimtRows
static_assert(kFwdThreads / 32 * kRowsPerWarp == 32, "a tile's 32 rows over the CTA's warps");
// The encoder and decode are compiled for a D capacity DC in {32, 64, 128}
// (the smallest that holds D): a lane accumulates DC / 32 output components,
// and a thread moves DC / 4 elements of a 32-row tile.
template <int DC> constexpr int per_lane() { return DC / 32; }
template <int DC> constexpr int tile_elems() { return 32 * DC / kFwdThreads; }

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One 32-key tile of the online softmax for the 8 rows a warp owns.
//   Rs  [32][D+1]  row vectors (already multiplied by the score scale)
//   Ks  [32][D+1]  key vectors of the tile (lane j reads key j)
//   Vs  [32][D]    value vectors of the tile
//   key_ok         this lane's key is valid
// State per row i: running max m[i], running sum l[i] (relative to m[i]) and
// the unnormalised accumulator acc[i][j] for value component d = lane + 32 j.
template <int DC>
__device__ __forceinline__ void online_tile(const float *Rs, const float *Ks, const float *Vs,
                                            bool key_ok, int D, int row0, float *m, float *l,
                                            float (*acc)[per_lane<DC>()]) {
    constexpr int kMaxDPerLane = per_lane<DC>();
    const int lane = threadIdx.x & 31;
    const int ld = D + 1;
    const float *k = Ks + lane * ld;
    // fully unrolled: the per-row state m, l, acc is indexed by constants and
    // stays in registers (a run-time row index put it in local memory)
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const float *r = Rs + (row0 + i) * ld;
        // four independent partial sums keep the FMA chain short
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        int d = 0;
        for (; d + 4 <= D; d += 4) {
            s0 = fmaf(r[d], k[d], s0);
            s1 = fmaf(r[d + 1], k[d + 1], s1);
            s2 = fmaf(r[d + 2], k[d + 2], s2);
            s3 = fmaf(r[d + 3], k[d + 3], s3);
        }
        for (; d < D; ++d) s0 = fmaf(r[d], k[d], s0);
        float s = (s0 + s1) + (s2 + s3);
        s = key_ok ? s : -INFINITY;
        const float mnew = fmaxf(m[i], warp_max(s));
        if (mnew == -INFINITY) continue;                 // nothing valid yet
        const float p = key_ok ? expf(s - mnew) : 0.f;
        const float corr = (m[i] == -INFINITY) ? 0.f : expf(m[i] - mnew);
        l[i] = l[i] * corr + warp_sum(p);
        m[i] = mnew;
#pragma unroll
        for (int j = 0; j < kMaxDPerLane; ++j) acc[i][j] *= corr;
        // unrolled so that several broadcasts are in flight at once
#pragma unroll 8
        for (int t = 0; t < 32; ++t) {
            const float pt = __shfl_sync(0xffffffffu, p, t);
            const float *v = Vs + t * D;
#pragma unroll
            for (int j = 0; j < kMaxDPerLane; ++j) {
                const int d = lane + 32 * j;
                if (d < D) acc[i][j] = fmaf(pt, v[d], acc[i][j]);
            }
        }
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Log-sum-exp merge of chunk partials into shards and shards into the global
// result, for rows [m0, m0 + rows) of one (b, h). Used by the last CTA of the
// encoder grid for that (b, h, row tile) and, with one chunk per shard, by the
// standalone merge kernel.
//   part_L [.., total_chunks, M] / part_O [.., total_chunks, M, D] at base
//   offsets for this (b, h); chunk_start describes which chunks form a shard.
// Per row:  L_r  = log sum_{c in r} exp(L_c)       (chunk -> shard)
//           O_r  = sum_{c in r} exp(L_c - L_r) O_c
//           L_max = max_r L_r, a = sum_r exp(L_r - L_max)
//           Z = sum_r exp(L_r - L_max) O_r / a,  L = L_max + log a.
// Shards are folded in index order (deterministic).
struct MergeArgs {
    const float *part_L;        // chunk log-normalisers, row stride 1, chunk stride M
    const float *part_O;        // chunk outputs, chunk stride M*D, row stride D
    int M, D, R;
    const int *chunk_start;     // R+1 prefix (in kernel parameter space)
    float *Lr_out;  int64_t Lr_shard_stride;   // L_r destination (never null)
    float *Or_out;  int64_t Or_shard_stride;   // O_r destination or null
    float *Z, *L;                              // global outputs (may be null)
};

__device__ void merge_rows(const MergeArgs &a, int m0, int rows, float *s_lmax, float *s_a) {
    // Every loop below issues the loads of up to kMergeBatch chunks together
    // and only then uses them (no load waits on another load's value, no
    // branch on a loaded value before the next load): the partials were
    // written by other CTAs a moment ago and sit in L2, so the merge's time
    // is a few round trips to L2 per shard instead of two per chunk.
    constexpr int kMergeBatch = 8;
    const int tid = threadIdx.x, nth = blockDim.x;
    for (int i = tid; i < rows; i += nth) {
        const int m = m0 + i;
        // every chunk of the row in batches (a batch may cross shard ends):
        // the running (maximum, rescaled sum) of the current shard, closed
        // into L_r at the shard's end and folded into the row's (L_max, a)
        const int total = a.chunk_start[a.R];
        float lmax = -INFINITY, asum = 0.f;
        float cmax = -INFINITY, sum = 0.f;
        int r = 0;
        auto close_shard = [&]() {
            const float Lr = (cmax == -INFINITY) ? -INFINITY : cmax + logf(sum);
            a.Lr_out[r * a.Lr_shard_stride + m] = Lr;
            if (Lr != -INFINITY) {
                if (Lr > lmax) {
                    asum = (lmax == -INFINITY) ? 0.f : asum * expf(lmax - Lr);
                    lmax = Lr;
                }
                asum += expf(Lr - lmax);
            }
            cmax = -INFINITY;
            sum = 0.f;
            ++r;
        };
        for (int cb = 0; cb < total; cb += kMergeBatch) {
            float lc[kMergeBatch];
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u)
                lc[u] = (cb + u < total) ? __ldcg(a.part_L + (int64_t)(cb + u) * a.M + m) : -INFINITY;
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                const int c = cb + u;
                if (c >= total) break;
                while (c >= a.chunk_start[r + 1]) close_shard();
                if (lc[u] != -INFINITY) {
                    if (lc[u] > cmax) {
                        sum = (cmax == -INFINITY) ? 0.f : sum * expf(cmax - lc[u]);
                        cmax = lc[u];
                    }
                    sum += expf(lc[u] - cmax);
                }
            }
        }
        while (r < a.R) close_shard();
        s_lmax[i] = lmax;
        s_a[i] = asum;
        if (a.L) a.L[m] = (lmax == -INFINITY) ? -INFINITY : lmax + logf(asum);
    }
    __syncthreads();
    if (a.Or_out == nullptr) {
        // Only (Z, L): Z = sum_c exp(L_c - L_max) O_c / a over every chunk of
        // the row, so no load waits on a shard-level value; each thread
        // takes kElems outputs at once and issues the loads of a batch of
        // chunks for all of them together.
        constexpr int kElems = 4;
        const int total = a.chunk_start[a.R];
        for (int e0 = tid; e0 < rows * a.D; e0 += kElems * nth) {
            int m[kElems], d[kElems];
            float lm[kElems], U[kElems];
#pragma unroll
            for (int k = 0; k < kElems; ++k) {
                const int e = e0 + k * nth, i = e / a.D;
                const bool in = e < rows * a.D;
                m[k] = m0 + (in ? i : 0);
                d[k] = in ? e - i * a.D : 0;
                lm[k] = in ? s_lmax[i] : -INFINITY;
                U[k] = 0.f;
            }
            for (int cb = 0; cb < total; cb += kMergeBatch) {
                float lc[kElems][kMergeBatch], oc[kElems][kMergeBatch];
#pragma unroll
                for (int k = 0; k < kElems; ++k)
#pragma unroll
                    for (int u = 0; u < kMergeBatch; ++u) {
                        const int64_t c = cb + u;
                        const bool in = cb + u < total && lm[k] != -INFINITY;
                        lc[k][u] = in ? __ldcg(a.part_L + c * a.M + m[k]) : -INFINITY;
                        oc[k][u] = in ? __ldcg(a.part_O + (c * a.M + m[k]) * a.D + d[k]) : 0.f;
                    }
#pragma unroll
                for (int k = 0; k < kElems; ++k)
#pragma unroll
                    for (int u = 0; u < kMergeBatch; ++u)
                        U[k] = fmaf(lc[k][u] == -INFINITY ? 0.f : expf(lc[k][u] - lm[k]), oc[k][u], U[k]);
            }
#pragma unroll
            for (int k = 0; k < kElems; ++k) {
                const int e = e0 + k * nth;
                if (e < rows * a.D && a.Z)
                    a.Z[(int64_t)m[k] * a.D + d[k]] = (lm[k] == -INFINITY) ? 0.f : U[k] / s_a[m[k] - m0];
            }
        }
        return;
    }
    for (int e = tid; e < rows * a.D; e += nth) {
        const int i = e / a.D, d = e % a.D, m = m0 + i;
        const float lmax = s_lmax[i];
        float U = 0.f;
        for (int r = 0; r < a.R; ++r) {
            const float Lr = a.Lr_out[r * a.Lr_shard_stride + m];
            const int c0 = a.chunk_start[r], c1 = a.chunk_start[r + 1];
            float o = 0.f;
            if (Lr != -INFINITY) {
                // every chunk's output slot was written (zeros for an empty
                // chunk), so it is loaded unconditionally and weighted
                for (int cb = c0; cb < c1; cb += kMergeBatch) {
                    float lc[kMergeBatch], oc[kMergeBatch];
#pragma unroll
                    for (int u = 0; u < kMergeBatch; ++u) {
                        const bool in = cb + u < c1;
                        const int64_t c = cb + u;
                        lc[u] = in ? __ldcg(a.part_L + c * a.M + m) : -INFINITY;
                        oc[u] = in ? __ldcg(a.part_O + (c * a.M + m) * a.D + d) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < kMergeBatch; ++u)
                        o = fmaf(lc[u] == -INFINITY ? 0.f : expf(lc[u] - Lr), oc[u], o);
                }
                U = fmaf(expf(Lr - lmax), o, U);
            }
            if (a.Or_out) a.Or_out[r * a.Or_shard_stride + (int64_t)m * a.D + d] = o;
        }
        if (a.Z) a.Z[(int64_t)m * a.D + d] = (lmax == -INFINITY) ? 0.f : U / s_a[i];
    }
}

namespace {

// ---------------------------------------------------------------------------
// Encoder: one CTA per (token chunk, head, batch x row tile of 32 latents).
template <typename TQ, typename TKV, int DC>
__global__ void __launch_bounds__(kFwdThreads)
enc_fwd_simt_kernel(Problem pr, ShardPlan plan, const TQ *__restrict__ Q,
                    const TKV *__restrict__ K, const TKV *__restrict__ V,
                    const uint8_t *__restrict__ mask, EncoderWorkspace ws, EncoderOut out,
                    int mtiles) {
    constexpr int kMaxDPerLane = per_lane<DC>(), kTileElems = tile_elems<DC>();
    extern __shared__ float smem[];
    const int D = pr.D, M = pr.M, H = pr.H, N = pr.N;
    const int ld = D + 1;
    float *Qs = smem;                 // [32][D+1]
    float *Ks = Qs + kSimtRows * ld;  // [32][D+1]
    float *Vs = Ks + kSimtTile * ld;  // [32][D]
    __shared__ unsigned char s_ok[kSimtTile];
    __shared__ int s_last;
    __shared__ float s_lmax[kSimtRows], s_a[kSimtRows];

    // a programmatic dependent (the decode) may be scheduled once every CTA
    // of this grid has started; it waits for this grid's results itself
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int c = blockIdx.x, h = blockIdx.y;
    const int b = blockIdx.z / mtiles, mt = blockIdx.z % mtiles;
    const int m0 = mt * kSimtRows;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int64_t n0, n1;
    chunk_range(plan, c, n0, n1);

    const TQ *Qb = Q + (int64_t)b * pr.q_bstride + (int64_t)h * M * D;
    // all of this thread's query loads first; the first tile's loads follow
    // before any store (one round trip to memory for both)
    float qv[kTileElems];
#pragma unroll
    for (int k = 0; k < kTileElems; ++k) {
        const int e = tid + k * kFwdThreads, i = e / D, d = e - i * D;
        qv[k] = (e < kSimtRows * D && m0 + i < M) ? to_f(Qb[(int64_t)(m0 + i) * D + d]) : 0.f;
    }
    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kMaxDPerLane];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxDPerLane; ++j) acc[i][j] = 0.f;
    }
    // The next tile's K, V and mask are loaded into registers while this one
    // is computed (its loads are in flight during the tile's arithmetic).
    float kr[kTileElems], vr[kTileElems];
    bool okr = false;
    auto fetch = [&](int64_t t0) {
#pragma unroll
        for (int k = 0; k < kTileElems; ++k) {
            const int e = tid + k * kFwdThreads, t = e / D, d = e - t * D;
            const int64_t n = t0 + t;
            kr[k] = vr[k] = 0.f;
            if (e < kSimtTile * D && n < n1) {
                const int64_t o = (((int64_t)b * N + n) * H + h) * D + d;
                kr[k] = to_f(K[o]);
                vr[k] = to_f(V[o]);
            }
        }
        const int64_t n = t0 + tid;
        okr = tid < kSimtTile && n < n1 && (!mask || mask[(int64_t)b * N + n]);
    };
    if (n0 < n1) fetch(n0);
#pragma unroll
    for (int k = 0; k < kTileElems; ++k) {
        const int e = tid + k * kFwdThreads, i = e / D, d = e - i * D;
        if (e < kSimtRows * D) Qs[i * ld + d] = pr.scale * qv[k];
    }
    for (int64_t t0 = n0; t0 < n1; t0 += kSimtTile) {
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kTileElems; ++k) {
            const int e = tid + k * kFwdThreads, t = e / D, d = e - t * D;
            if (e < kSimtTile * D) {
                Ks[t * ld + d] = kr[k];
                Vs[t * D + d] = vr[k];
            }
        }
        if (tid < kSimtTile) s_ok[tid] = okr;
        __syncthreads();
        if (t0 + kSimtTile < n1) fetch(t0 + kSimtTile);
        online_tile<DC>(Qs, Ks, Vs, s_ok[lane] != 0, D, warp * kRowsPerWarp, m, l, acc);
    }

    // chunk partial: normalised output and log-normaliser (empty row: -inf, 0)
    const int64_t pbase = ((int64_t)(b * H + h) * plan.total_chunks + c) * M;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int row = m0 + warp * kRowsPerWarp + i;
        if (row >= M) continue;
        const bool live = l[i] > 0.f;
        if (lane == 0) ws.part_L[pbase + row] = live ? m[i] + logf(l[i]) : -INFINITY;
        const float inv = live ? 1.f / l[i] : 0.f;
#pragma unroll
        for (int j = 0; j < kMaxDPerLane; ++j) {
            const int d = lane + 32 * j;
            if (d < D) ws.part_O[(pbase + row) * D + d] = acc[i][j] * inv;
        }
    }

    // last CTA of this (b, h, row tile) merges every chunk (no waiting)
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&ws.tickets[(b * H + h) * mtiles + mt], 1u);
        s_last = (prev == (unsigned)plan.total_chunks - 1u);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    MergeArgs ma;
    const int64_t bh = (int64_t)b * H + h;
    ma.part_L = ws.part_L + bh * plan.total_chunks * M;
    ma.part_O = ws.part_O + bh * plan.total_chunks * M * D;
    ma.M = M;
    ma.D = D;
    ma.R = plan.R;
    ma.chunk_start = plan.chunk_start;
    if (out.L_r) {
        ma.Lr_out = out.L_r + bh * M;
        ma.Lr_shard_stride = (int64_t)pr.B * H * M;
    } else {
        ma.Lr_out = ws.shard_L + bh * plan.R * M;
        ma.Lr_shard_stride = M;
    }
    ma.Or_out = out.O_r ? out.O_r + bh * M * D : nullptr;
    ma.Or_shard_stride = (int64_t)pr.B * H * M * D;
    ma.Z = out.Z ? out.Z + bh * M * D : nullptr;
    ma.L = out.L ? out.L + bh * M : nullptr;
    const int rows = min(kSimtRows, M - m0);
    merge_rows(ma, m0, rows, s_lmax, s_a);
}

// ---------------------------------------------------------------------------
// Standalone merge of R given shard results: one CTA per (b, h, 32 rows).
__global__ void __launch_bounds__(kFwdThreads)
lse_merge_kernel(const float *__restrict__ O_r, const float *__restrict__ L_r, int R, int B,
                 int H, int M, int D, float *Z, float *L) {
    __shared__ float s_lmax[kSimtRows], s_a[kSimtRows];
    const int mtiles = (M + kSimtRows - 1) / kSimtRows;
    const int64_t bh = blockIdx.x / mtiles;
    const int m0 = (blockIdx.x % mtiles) * kSimtRows;
    const int rows = min(kSimtRows, M - m0);
    const int64_t srow = (int64_t)B * H * M;     // shard stride of L_r
    const int tid = threadIdx.x;
    for (int i = tid; i < rows; i += blockDim.x) {
        const int64_t row = bh * M + m0 + i;
        float lmax = -INFINITY;
        for (int r = 0; r < R; ++r) lmax = fmaxf(lmax, L_r[r * srow + row]);
        float a = 0.f;
        if (lmax != -INFINITY)
            for (int r = 0; r < R; ++r) {
                const float lr = L_r[r * srow + row];
                if (lr != -INFINITY) a += expf(lr - lmax);
            }
        s_lmax[i] = lmax;
        s_a[i] = a;
        L[row] = (lmax == -INFINITY) ? -INFINITY : lmax + logf(a);
    }
    __syncthreads();
    for (int e = tid; e < rows * D; e += blockDim.x) {
        const int i = e / D, d = e % D;
        const int64_t row = bh * M + m0 + i;
        const float lmax = s_lmax[i];
        float U = 0.f;
        if (lmax != -INFINITY)
            for (int r = 0; r < R; ++r) {
                const float lr = L_r[r * srow + row];
                if (lr != -INFINITY) U = fmaf(expf(lr - lmax), O_r[(r * srow + row) * D + d], U);
            }
        Z[row * D + d] = (lmax == -INFINITY) ? 0.f : U / s_a[i];
    }
}

// ---------------------------------------------------------------------------
// Decode: rows are 32 tokens, keys are the M latents (tiles of 32), values Z.
template <typename TQ, typename TK, int DC>
__global__ void __launch_bounds__(kFwdThreads)
dec_fwd_simt_kernel(Problem pr, const TQ *__restrict__ Q, const float *__restrict__ Z,
                    const TK *__restrict__ K, TK *__restrict__ Y) {
    constexpr int kMaxDPerLane = per_lane<DC>(), kTileElems = tile_elems<DC>();
    extern __shared__ float smem[];
    const int D = pr.D, M = pr.M, H = pr.H, N = pr.N;
    const int ld = D + 1;
    float *Rs = smem;                 // [32 tokens][D+1]  (scaled keys)
    float *Ls = Rs + kSimtTile * ld;  // [32 latents][D+1]
    float *Zs = Ls + kSimtRows * ld;  // [32 latents][D]
    const int64_t t0 = (int64_t)blockIdx.x * kSimtTile;
    const int h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float kv[kTileElems];
#pragma unroll
    for (int k = 0; k < kTileElems; ++k) {
        const int e = tid + k * kFwdThreads, t = e / D, d = e - t * D;
        const int64_t n = t0 + t;
        kv[k] = (e < kSimtTile * D && n < N) ? pr.scale * to_f(K[(((int64_t)b * N + n) * H + h) * D + d]) : 0.f;
    }
    bool k_stored = false;   // the K tile goes to shared memory with the first latent tile's loads in flight
    // Launched as a programmatic dependent of the encoder that writes Z (in
    // flare_fwd / flare_pp_fwd), this CTA may start while that grid runs:
    // the K loads above go ahead, Q and Z are read only once it has completed
    // (a no-op for a launch without the attribute).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kMaxDPerLane];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxDPerLane; ++j) acc[i][j] = 0.f;
    }
    const TQ *Qb = Q + (int64_t)b * pr.q_bstride + (int64_t)h * M * D;
    const float *Zb = Z + ((int64_t)b * H + h) * M * D;
    for (int l0 = 0; l0 < M; l0 += kSimtRows) {
        float qv[kTileElems], zv[kTileElems];
#pragma unroll
        for (int k = 0; k < kTileElems; ++k) {
            const int e = tid + k * kFwdThreads, j = e / D, d = e - j * D;
            const bool ok = e < kSimtRows * D && l0 + j < M;
            qv[k] = ok ? to_f(Qb[(int64_t)(l0 + j) * D + d]) : 0.f;
            zv[k] = ok ? Zb[(int64_t)(l0 + j) * D + d] : 0.f;
        }
        if (!k_stored) {
#pragma unroll
            for (int k = 0; k < kTileElems; ++k) {
                const int e = tid + k * kFwdThreads, t = e / D, d = e - t * D;
                if (e < kSimtTile * D) Rs[t * ld + d] = kv[k];
            }
            k_stored = true;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kTileElems; ++k) {
            const int e = tid + k * kFwdThreads, j = e / D, d = e - j * D;
            if (e < kSimtRows * D) {
                Ls[j * ld + d] = qv[k];
                Zs[j * D + d] = zv[k];
            }
        }
        __syncthreads();
        online_tile<DC>(Rs, Ls, Zs, l0 + lane < M, D, warp * kRowsPerWarp, m, l, acc);
    }
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int64_t n = t0 + warp * kRowsPerWarp + i;
        if (n >= N) continue;
        const float inv = 1.f / l[i];
#pragma unroll
        for (int j = 0; j < kMaxDPerLane; ++j) {
            const int d = lane + 32 * j;
            if (d < D) Y[(((int64_t)b * N + n) * H + h) * D + d] = from_f<TK>(acc[i][j] * inv);
        }
    }
}

// ---------------------------------------------------------------------------
// Backward. Shared tile step: for 32 latent rows x 32 tokens compute
//   P  = exp(s <Q_m, K_n> - L_m)   (0 for masked tokens / empty rows)
//   dS = P (<dZ_m, V_n> - c_m)
struct BwdTile {
    float *Qt, *dZt, *Kt, *Vt;   // [32][D+1]
    float *Lt, *ct;              // [32]
    float *Pt, *dSt;             // [32 rows][33]
    unsigned char *tok_ok;       // [32]
};

__device__ void bwd_p_ds(const BwdTile &t, int D, float scale) {
    const int ld = D + 1;
    for (int p = threadIdx.x; p < 32 * 32; p += kThreads) {
        const int row = p >> 5, tok = p & 31;
        const float Lm = t.Lt[row];
        float P = 0.f, dS = 0.f;
        if (t.tok_ok[tok] && Lm != -INFINITY) {
            const float *q = t.Qt + row * ld, *k = t.Kt + tok * ld;
            const float *dz = t.dZt + row * ld, *v = t.Vt + tok * ld;
            float s = 0.f, dp = 0.f;
            for (int d = 0; d < D; ++d) {
                s = fmaf(q[d], k[d], s);
                dp = fmaf(dz[d], v[d], dp);
            }
            P = expf(scale * s - Lm);
            dS = P * (dp - t.ct[row]);
        }
        t.Pt[row * 33 + tok] = P;
        t.dSt[row * 33 + tok] = dS;
    }
}

// Loads latent rows [m0, m0+32) of (b, h): Q, dZ, L and c = <dZ, Z>.
template <typename TQ>
__device__ void bwd_load_rows(const BwdTile &t, const Problem &pr, const TQ *Qb, const float *Zb,
                              const float *dZb, const float *Lb, int m0) {
    const int D = pr.D, M = pr.M, ld = D + 1;
    for (int e = threadIdx.x; e < 32 * D; e += kThreads) {
        const int i = e / D, d = e % D;
        const bool ok = m0 + i < M;
        t.Qt[i * ld + d] = ok ? to_f(Qb[(int64_t)(m0 + i) * D + d]) : 0.f;
        t.dZt[i * ld + d] = ok ? dZb[(int64_t)(m0 + i) * D + d] : 0.f;
    }
    if (threadIdx.x < 32) {
        const int i = threadIdx.x;
        float cm = 0.f, Lm = -INFINITY;
        if (m0 + i < M) {
            for (int d = 0; d < D; ++d)
                cm = fmaf(dZb[(int64_t)(m0 + i) * D + d], Zb[(int64_t)(m0 + i) * D + d], cm);
            Lm = Lb[m0 + i];
        }
        t.ct[i] = cm;
        t.Lt[i] = Lm;
    }
}

template <typename TKV>
__device__ void bwd_load_tokens(const BwdTile &t, const Problem &pr, const TKV *K, const TKV *V,
                                const uint8_t *mask, int b, int h, int64_t t0, int64_t tend) {
    const int D = pr.D, ld = D + 1;
    for (int e = threadIdx.x; e < 32 * D; e += kThreads) {
        const int j = e / D, d = e % D;
        const int64_t n = t0 + j;
        float kv = 0.f, vv = 0.f;
        if (n < tend) {
            const int64_t o = (((int64_t)b * pr.N + n) * pr.H + h) * D + d;
            kv = to_f(K[o]);
            vv = to_f(V[o]);
        }
        t.Kt[j * ld + d] = kv;
        t.Vt[j * ld + d] = vv;
    }
    if (threadIdx.x < 32) {
        const int64_t n = t0 + threadIdx.x;
        t.tok_ok[threadIdx.x] = (n < tend) && (!mask || mask[(int64_t)b * pr.N + n]);
    }
}

__device__ BwdTile bwd_carve(float *smem, int D) {
    const int ld = D + 1;
    BwdTile t;
    t.Qt = smem;
    t.dZt = t.Qt + 32 * ld;
    t.Kt = t.dZt + 32 * ld;
    t.Vt = t.Kt + 32 * ld;
    t.Pt = t.Vt + 32 * ld;
    t.dSt = t.Pt + 32 * 33;
    t.Lt = t.dSt + 32 * 33;
    t.ct = t.Lt + 32;
    t.tok_ok = reinterpret_cast<unsigned char *>(t.ct + 32);
    return t;
}

__host__ __device__ inline size_t bwd_tile_floats(int D) {
    return 4 * 32 * (size_t)(D + 1) + 2 * 32 * 33 + 32 + 32 + 8;
}

// dK, dV of 32 tokens: loop over every latent row tile.
template <typename TQ, typename TKV>
__global__ void __launch_bounds__(kThreads)
bwd_dkdv_simt_kernel(Problem pr, const TQ *__restrict__ Q, const TKV *__restrict__ K,
                     const TKV *__restrict__ V, const uint8_t *__restrict__ mask,
                     const float *__restrict__ Z, const float *__restrict__ L,
                     const float *__restrict__ dZ, TKV *dK, TKV *__restrict__ dV, int accumulate) {
    extern __shared__ float smem[];
    const int D = pr.D, M = pr.M, H = pr.H, N = pr.N, ld = D + 1;
    BwdTile t = bwd_carve(smem, D);
    float *dKs = smem + bwd_tile_floats(D);   // [32][D+1]
    float *dVs = dKs + 32 * ld;               // [32][D+1]
    const int64_t t0 = (int64_t)blockIdx.x * 32;
    const int h = blockIdx.y, b = blockIdx.z;
    for (int e = threadIdx.x; e < 32 * ld; e += kThreads) dKs[e] = dVs[e] = 0.f;
    bwd_load_tokens(t, pr, K, V, mask, b, h, t0, (int64_t)N);
    const int64_t bh = (int64_t)b * H + h;
    const TQ *Qb = Q + (int64_t)b * pr.q_bstride + (int64_t)h * M * D;
    for (int m0 = 0; m0 < M; m0 += 32) {
        __syncthreads();
        bwd_load_rows(t, pr, Qb, Z + bh * M * D, dZ + bh * M * D, L + bh * M, m0);
        __syncthreads();
        bwd_p_ds(t, D, pr.scale);
        __syncthreads();
        for (int e = threadIdx.x; e < 32 * D; e += kThreads) {
            const int tok = e / D, d = e % D;
            float dv = dVs[tok * ld + d], dk = dKs[tok * ld + d];
            for (int row = 0; row < 32; ++row) {
                dv = fmaf(t.Pt[row * 33 + tok], t.dZt[row * ld + d], dv);
                dk = fmaf(t.dSt[row * 33 + tok], t.Qt[row * ld + d], dk);
            }
            dVs[tok * ld + d] = dv;
            dKs[tok * ld + d] = dk;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * D; e += kThreads) {
        const int tok = e / D, d = e % D;
        const int64_t n = t0 + tok;
        if (n >= N) continue;
        const int64_t o = (((int64_t)b * N + n) * H + h) * D + d;
        const float old = accumulate ? to_f(dK[o]) : 0.f;   // the decode's share
        dK[o] = from_f<TKV>(old + pr.scale * dKs[tok * ld + d]);
        dV[o] = from_f<TKV>(dVs[tok * ld + d]);
    }
}

// dQ partial of 32 latent rows over one token chunk; the last CTA of each
// (b, h, row tile) sums the chunk partials in chunk order.
template <typename TQ, typename TKV>
__global__ void __launch_bounds__(kThreads)
bwd_dq_simt_kernel(Problem pr, const TQ *__restrict__ Q, const TKV *__restrict__ K,
                   const TKV *__restrict__ V, const uint8_t *__restrict__ mask,
                   const float *__restrict__ Z, const float *__restrict__ L,
                   const float *__restrict__ dZ, float *__restrict__ dQ, unsigned *tickets,
                   float *part, int chunk_len, int nchunks, int mtiles, int accumulate) {
    extern __shared__ float smem[];
    __shared__ int s_last;
    const int D = pr.D, M = pr.M, H = pr.H, N = pr.N, ld = D + 1;
    BwdTile t = bwd_carve(smem, D);
    float *dQs = smem + bwd_tile_floats(D);   // [32][D+1]
    const int c = blockIdx.x, h = blockIdx.y;
    const int b = blockIdx.z / mtiles, mt = blockIdx.z % mtiles, m0 = mt * 32;
    const int64_t n0 = (int64_t)c * chunk_len;
    const int64_t n1 = min((int64_t)N, n0 + chunk_len);
    const int64_t bh = (int64_t)b * H + h;
    for (int e = threadIdx.x; e < 32 * ld; e += kThreads) dQs[e] = 0.f;
    const TQ *Qb = Q + (int64_t)b * pr.q_bstride + (int64_t)h * M * D;
    bwd_load_rows(t, pr, Qb, Z + bh * M * D, dZ + bh * M * D, L + bh * M, m0);
    for (int64_t t0 = n0; t0 < n1; t0 += 32) {
        __syncthreads();
        bwd_load_tokens(t, pr, K, V, mask, b, h, t0, n1);
        __syncthreads();
        bwd_p_ds(t, D, pr.scale);
        __syncthreads();
        for (int e = threadIdx.x; e < 32 * D; e += kThreads) {
            const int row = e / D, d = e % D;
            float q = dQs[row * ld + d];
            for (int tok = 0; tok < 32; ++tok) q = fmaf(t.dSt[row * 33 + tok], t.Kt[tok * ld + d], q);
            dQs[row * ld + d] = q;
        }
    }
    __syncthreads();
    const int rows = min(32, M - m0);
    float *pc = part + ((bh * nchunks + c) * M) * D;
    for (int e = threadIdx.x; e < rows * D; e += kThreads) {
        const int row = e / D, d = e % D;
        pc[(int64_t)(m0 + row) * D + d] = pr.scale * dQs[row * ld + d];
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(&tickets[bh * mtiles + mt], 1u);
        s_last = (prev == (unsigned)nchunks - 1u);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int e = threadIdx.x; e < rows * D; e += kThreads) {
        const int row = e / D, d = e % D;
        float *dst = dQ + (bh * M + m0 + row) * D + d;
        float acc = accumulate ? *dst : 0.f;
        for (int cc = 0; cc < nchunks; ++cc)
            acc += __ldcg(part + ((bh * nchunks + cc) * M + m0 + row) * D + d);
        *dst = acc;
    }
}

inline size_t enc_smem_bytes(int D) {
    return sizeof(float) * ((size_t)kSimtRows * (D + 1) + (size_t)kSimtTile * (D + 1) +
                            (size_t)kSimtTile * D);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

// ---- launchers -------------------------------------------------------------

namespace {
template <int DC>
cudaError_t launch_encoder_simt_dc(const Problem &pr, const ShardPlan &plan, const void *Q,
                                   bool q_is_f32, const void *K, const void *V, const uint8_t *mask,
                                   const EncoderWorkspace &ws, const EncoderOut &out, dim3 grid,
                                   int mtiles, cudaStream_t st) {
    const size_t smem = enc_smem_bytes(pr.D);
    cudaError_t e;
    if (!pr.bf16) {
        auto k = enc_fwd_simt_kernel<float, float, DC>;
        if ((e = set_smem(k, smem)) != cudaSuccess) return e;
        k<<<grid, kFwdThreads, smem, st>>>(pr, plan, (const float *)Q, (const float *)K,
                                        (const float *)V, mask, ws, out, mtiles);
    } else if (q_is_f32) {
        auto k = enc_fwd_simt_kernel<float, __nv_bfloat16, DC>;
        if ((e = set_smem(k, smem)) != cudaSuccess) return e;
        k<<<grid, kFwdThreads, smem, st>>>(pr, plan, (const float *)Q, (const __nv_bfloat16 *)K,
                                        (const __nv_bfloat16 *)V, mask, ws, out, mtiles);
    } else {
        auto k = enc_fwd_simt_kernel<__nv_bfloat16, __nv_bfloat16, DC>;
        if ((e = set_smem(k, smem)) != cudaSuccess) return e;
        k<<<grid, kFwdThreads, smem, st>>>(pr, plan, (const __nv_bfloat16 *)Q,
                                        (const __nv_bfloat16 *)K, (const __nv_bfloat16 *)V, mask,
                                        ws, out, mtiles);
    }
    note_launch();
    return cudaGetLastError();
}

// Launch with the programmatic-stream-serialization attribute when `pdl`.
template <typename Kernel, typename... Args>
cudaError_t launch_fwd(Kernel k, dim3 grid, size_t smem, cudaStream_t st, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kFwdThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

template <int DC>
cudaError_t launch_decode_simt_dc(const Problem &pr, const void *Q, bool q_is_f32, const float *Z,
                                  const void *K, void *Y, bool pdl, cudaStream_t st) {
    dim3 grid((pr.N + kSimtTile - 1) / kSimtTile, pr.H, pr.B);
    const size_t smem = sizeof(float) * ((size_t)kSimtTile * (pr.D + 1) +
                                         (size_t)kSimtRows * (pr.D + 1) + (size_t)kSimtRows * pr.D);
    cudaError_t e;
    if (!pr.bf16) {
        auto k = dec_fwd_simt_kernel<float, float, DC>;
        if ((e = set_smem(k, smem)) != cudaSuccess) return e;
        e = launch_fwd(k, grid, smem, st, pdl, pr, (const float *)Q, Z, (const float *)K, (float *)Y);
    } else if (q_is_f32) {
        auto k = dec_fwd_simt_kernel<float, __nv_bfloat16, DC>;
        if ((e = set_smem(k, smem)) != cudaSuccess) return e;
        e = launch_fwd(k, grid, smem, st, pdl, pr, (const float *)Q, Z, (const __nv_bfloat16 *)K,
                       (__nv_bfloat16 *)Y);
    } else {
        auto k = dec_fwd_simt_kernel<__nv_bfloat16, __nv_bfloat16, DC>;
        if ((e = set_smem(k, smem)) != cudaSuccess) return e;
        e = launch_fwd(k, grid, smem, st, pdl, pr, (const __nv_bfloat16 *)Q, Z,
                       (const __nv_bfloat16 *)K, (__nv_bfloat16 *)Y);
    }
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}
}  // namespace

cudaError_t launch_encoder_simt(const Problem &pr, const ShardPlan &plan, const void *Q,
                                bool q_is_f32, const void *K, const void *V, const uint8_t *mask,
                                const EncoderWorkspace &ws, const EncoderOut &out,
                                cudaStream_t st) {
    const int mtiles = (pr.M + kSimtRows - 1) / kSimtRows;
    if (plan.total_chunks == 0 || pr.B == 0) return cudaSuccess;
    dim3 grid(plan.total_chunks, pr.H, pr.B * mtiles);
    if (pr.D <= 32)
        return launch_encoder_simt_dc<32>(pr, plan, Q, q_is_f32, K, V, mask, ws, out, grid, mtiles, st);
    if (pr.D <= 64)
        return launch_encoder_simt_dc<64>(pr, plan, Q, q_is_f32, K, V, mask, ws, out, grid, mtiles, st);
    return launch_encoder_simt_dc<128>(pr, plan, Q, q_is_f32, K, V, mask, ws, out, grid, mtiles, st);
}

cudaError_t launch_lse_merge(const float *O_r, const float *L_r, int R, int B, int H, int M,
                             int D, float *Z, float *L, cudaStream_t st) {
    const int mtiles = (M + kSimtRows - 1) / kSimtRows;
    const int64_t blocks = (int64_t)B * H * mtiles;
    if (blocks == 0) return cudaSuccess;
    lse_merge_kernel<<<(unsigned)blocks, kThreads, 0, st>>>(O_r, L_r, R, B, H, M, D, Z, L);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_decode_simt(const Problem &pr, const void *Q, bool q_is_f32, const float *Z,
                               const void *K, void *Y, bool after_encoder, cudaStream_t st) {
    if (pr.B == 0 || pr.N == 0) return cudaSuccess;
    if (pr.D <= 32) return launch_decode_simt_dc<32>(pr, Q, q_is_f32, Z, K, Y, after_encoder, st);
    if (pr.D <= 64) return launch_decode_simt_dc<64>(pr, Q, q_is_f32, Z, K, Y, after_encoder, st);
    return launch_decode_simt_dc<128>(pr, Q, q_is_f32, Z, K, Y, after_encoder, st);
}

namespace {
constexpr int kBwdChunk = 2048;   // tokens per dQ partial
inline int bwd_nchunks(const Problem &pr) { return (pr.N + kBwdChunk - 1) / kBwdChunk; }
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
}  // namespace

size_t encoder_bwd_simt_workspace(const Problem &pr) {
    const int mtiles = (pr.M + 31) / 32;
    const size_t tickets = align256(sizeof(unsigned) * (size_t)pr.B * pr.H * mtiles);
    const size_t part = sizeof(float) * (size_t)pr.B * pr.H * bwd_nchunks(pr) * pr.M * pr.D;
    return tickets + align256(part);
}

cudaError_t launch_encoder_bwd_simt(const Problem &pr, const void *Q, const void *K,
                                    const void *V, const uint8_t *mask, const float *Z,
                                    const float *L, const float *dZ, float *dQ, void *dK,
                                    void *dV, void *ws, size_t ws_bytes, cudaStream_t st,
                                    bool accumulate) {
    if (pr.B == 0) return cudaSuccess;
    const int mtiles = (pr.M + 31) / 32;
    const int nchunks = bwd_nchunks(pr);
    const size_t tickets_bytes = align256(sizeof(unsigned) * (size_t)pr.B * pr.H * mtiles);
    unsigned *tickets = (unsigned *)ws;
    float *part = (float *)((char *)ws + tickets_bytes);
    const size_t tile = sizeof(float) * bwd_tile_floats(pr.D);
    const size_t smem_kv = tile + sizeof(float) * 2 * 32 * (pr.D + 1);
    const size_t smem_q = tile + sizeof(float) * 32 * (pr.D + 1);
    cudaError_t e;
    if (pr.N == 0) {   // no token: no share of dQ
        return accumulate ? cudaSuccess
                          : cudaMemsetAsync(dQ, 0, sizeof(float) * (size_t)pr.B * pr.H * pr.M * pr.D, st);
    }
    if ((e = cudaMemsetAsync(tickets, 0, tickets_bytes, st)) != cudaSuccess) return e;
    dim3 gkv((pr.N + 31) / 32, pr.H, pr.B), gq(nchunks, pr.H, pr.B * mtiles);
    const int acc = accumulate ? 1 : 0;
#define FLARE_BWD_LAUNCH(TQ, TKV)                                                             \
    {                                                                                         \
        auto k1 = bwd_dkdv_simt_kernel<TQ, TKV>;                                              \
        auto k2 = bwd_dq_simt_kernel<TQ, TKV>;                                                \
        if ((e = set_smem(k1, smem_kv)) != cudaSuccess) return e;                             \
        if ((e = set_smem(k2, smem_q)) != cudaSuccess) return e;                              \
        k1<<<gkv, kThreads, smem_kv, st>>>(pr, (const TQ *)Q, (const TKV *)K, (const TKV *)V, \
                                            mask, Z, L, dZ, (TKV *)dK, (TKV *)dV, acc);       \
        note_launch();                                                                        \
        k2<<<gq, kThreads, smem_q, st>>>(pr, (const TQ *)Q, (const TKV *)K, (const TKV *)V,   \
                                          mask, Z, L, dZ, dQ, tickets, part, kBwdChunk,       \
                                          nchunks, mtiles, acc);                              \
        note_launch();                                                                        \
    }
    if (!pr.bf16) FLARE_BWD_LAUNCH(float, float)
    else FLARE_BWD_LAUNCH(__nv_bfloat16, __nv_bfloat16)
#undef FLARE_BWD_LAUNCH
    (void)ws_bytes;
    return cudaGetLastError();
}

}  // namespace flare
