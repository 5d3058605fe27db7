// simt_decode_bwd.cu -- CUDA-core (FFMA) kernels of the FLARE decode backward.
//
// The chain rule of the local decode (FLARE decode paragraph of the FLARE++
// context-parallel appendix: each token's key queries the replicated
// latents). For a (b, h), token n and latent m:
//   A_nm = softmax_m(s <K_n, Q_m>),  g_nm = <dY_n, Z_m>,  r_n = sum_m A_nm g_nm,
//   dT_nm = A_nm (g_nm - r_n),
//   dK_n = s sum_m dT_nm Q_m,  dQ_m = s sum_n dT_nm K_n,  dZ_m = sum_n A_nm dY_n.
// Two kernels:
//   dec_bwd_dk_simt_kernel   one CTA per (32-token tile, h, b): every latent's
//                            score and g for the tile's tokens, the token's
//                            log-normaliser lse_n and r_n (saved), then dK;
//   dec_bwd_dqz_simt_kernel  one CTA per (token chunk, h, b x 32-latent tile):
//                            A and dT of its latents rebuilt from lse_n, r_n,
//                            dQ and dZ partials per chunk; the CTA taking the
//                            last ticket of a (b, h, latent tile) sums the
//                            chunks in chunk order.
// This path serves fp32 and every shape the tensor-core kernel leaves out.
#include "flare_internal.cuh"

#include <math.h>

namespace flare {
namespace {

constexpr int kT = 256;              // threads per CTA
constexpr int kTok = 32;             // tokens per tile
constexpr int kRows = 32;            // latents per dQ/dZ CTA
constexpr int kChunk = 2048;         // tokens per dQ/dZ partial

__device__ __forceinline__ float ld(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
template <typename T> __device__ __forceinline__ T cvt_out(float x);
template <> __device__ __forceinline__ float cvt_out<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 cvt_out<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// dK of 32 tokens and their (lse_n, r_n). Shared memory: K, dY tiles [32][D+1],
// scores / A and g / dT [32][M+1].
template <typename TQ, typename TK>
__global__ void __launch_bounds__(kT) dec_bwd_dk_simt_kernel(Problem pr, const TQ *__restrict__ Q,
                                                             const float *__restrict__ Z,
                                                             const TK *__restrict__ K,
                                                             const TK *__restrict__ dY,
                                                             TK *__restrict__ dK,
                                                             float2 *__restrict__ stats) {
    extern __shared__ float sm[];
    const int D = pr.D, M = pr.M, H = pr.H, N = pr.N;
    const int ldD = D + 1, ldM = M + 1;
    float *Ks = sm, *Ys = Ks + kTok * ldD, *T = Ys + kTok * ldD, *G = T + kTok * ldM;
    const int64_t t0 = (int64_t)blockIdx.x * kTok;
    const int h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const TQ *Qb = Q + (int64_t)b * pr.q_bstride + (int64_t)h * M * D;
    const float *Zb = Z + ((int64_t)b * H + h) * M * D;
    for (int e = tid; e < kTok * D; e += kT) {
        const int t = e / D, d = e % D;
        const int64_t n = t0 + t;
        float kv = 0.f, yv = 0.f;
        if (n < N) {
            const int64_t o = (((int64_t)b * N + n) * H + h) * D + d;
            kv = ld(K + o);
            yv = ld(dY + o);
        }
        Ks[t * ldD + d] = kv;
        Ys[t * ldD + d] = yv;
    }
    __syncthreads();
    // scores and g for every (token, latent)
    for (int e = tid; e < kTok * M; e += kT) {
        const int t = e % kTok, m = e / kTok;
        const TQ *q = Qb + (int64_t)m * D;
        const float *z = Zb + (int64_t)m * D;
        float sdot = 0.f, gdot = 0.f;
        for (int d = 0; d < D; ++d) {
            sdot = fmaf(Ks[t * ldD + d], ld(q + d), sdot);
            gdot = fmaf(Ys[t * ldD + d], ld(z + d), gdot);
        }
        T[t * ldM + m] = pr.scale * sdot;
        G[t * ldM + m] = gdot;
    }
    __syncthreads();
    // per token (one warp): max, sum, A, r, dT
    for (int t = warp; t < kTok; t += kT / 32) {
        float mx = -INFINITY;
        for (int m = lane; m < M; m += 32) mx = fmaxf(mx, T[t * ldM + m]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
        for (int m = lane; m < M; m += 32) sum += expf(T[t * ldM + m] - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float lse = mx + logf(sum);
        float r = 0.f;
        for (int m = lane; m < M; m += 32) {
            const float a = expf(T[t * ldM + m] - lse);
            T[t * ldM + m] = a;
            r = fmaf(a, G[t * ldM + m], r);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
        for (int m = lane; m < M; m += 32) G[t * ldM + m] = T[t * ldM + m] * (G[t * ldM + m] - r);
        const int64_t n = t0 + t;
        if (lane == 0 && n < N) stats[((int64_t)b * H + h) * N + n] = make_float2(lse, r);
    }
    __syncthreads();
    // dK_n = s sum_m dT_nm Q_m
    for (int e = tid; e < kTok * D; e += kT) {
        const int t = e / D, d = e % D;
        const int64_t n = t0 + t;
        if (n >= N) continue;
        float acc = 0.f;
        for (int m = 0; m < M; ++m) acc = fmaf(G[t * ldM + m], ld(Qb + (int64_t)m * D + d), acc);
        dK[(((int64_t)b * N + n) * H + h) * D + d] = cvt_out<TK>(pr.scale * acc);
    }
}

// dQ and dZ partials of 32 latents over one token chunk; the CTA taking the
// last ticket of its (b, h, latent tile) sums the chunk partials in order.
template <typename TQ, typename TK>
__global__ void __launch_bounds__(kT) dec_bwd_dqz_simt_kernel(
    Problem pr, const TQ *__restrict__ Q, const float *__restrict__ Z, const TK *__restrict__ K,
    const TK *__restrict__ dY, const float2 *__restrict__ stats, float *__restrict__ dQ,
    float *__restrict__ dZ, unsigned *tickets, float *part, int nchunks, int mtiles) {
    extern __shared__ float sm[];
    __shared__ int s_last;
    const int D = pr.D, M = pr.M, H = pr.H, N = pr.N, ldD = D + 1;
    float *Qs = sm, *Zs = Qs + kRows * ldD, *Ks = Zs + kRows * ldD, *Ys = Ks + kTok * ldD;
    float *A = Ys + kTok * ldD, *dT = A + kRows * (kTok + 1);
    const int c = blockIdx.x, h = blockIdx.y;
    const int b = blockIdx.z / mtiles, mt = blockIdx.z % mtiles, m0 = mt * kRows;
    const int rows = min(kRows, M - m0);
    const int tid = threadIdx.x;
    const int64_t bh = (int64_t)b * H + h;
    const int64_t n0 = (int64_t)c * kChunk, n1 = min((int64_t)N, n0 + kChunk);
    const TQ *Qb = Q + (int64_t)b * pr.q_bstride + (int64_t)h * M * D;
    for (int e = tid; e < kRows * D; e += kT) {
        const int i = e / D, d = e % D;
        const bool ok = i < rows;
        Qs[i * ldD + d] = ok ? ld(Qb + (int64_t)(m0 + i) * D + d) : 0.f;
        Zs[i * ldD + d] = ok ? Z[(bh * M + m0 + i) * D + d] : 0.f;
    }
    // accumulators: thread owns (row i, column d) pairs e = tid + kT * j
    constexpr int kAcc = kRows * 128 / kT;               // D <= 128
    float aq[kAcc], az[kAcc];
#pragma unroll
    for (int j = 0; j < kAcc; ++j) aq[j] = az[j] = 0.f;
    for (int64_t t0 = n0; t0 < n1; t0 += kTok) {
        __syncthreads();
        for (int e = tid; e < kTok * D; e += kT) {
            const int t = e / D, d = e % D;
            const int64_t n = t0 + t;
            float kv = 0.f, yv = 0.f;
            if (n < n1) {
                const int64_t o = (((int64_t)b * N + n) * H + h) * D + d;
                kv = ld(K + o);
                yv = ld(dY + o);
            }
            Ks[t * ldD + d] = kv;
            Ys[t * ldD + d] = yv;
        }
        __syncthreads();
        for (int e = tid; e < kRows * kTok; e += kT) {
            const int i = e / kTok, t = e % kTok;
            const int64_t n = t0 + t;
            float a = 0.f, g = 0.f;
            if (i < rows && n < n1) {
                float sdot = 0.f, gdot = 0.f;
                for (int d = 0; d < D; ++d) {
                    sdot = fmaf(Qs[i * ldD + d], Ks[t * ldD + d], sdot);
                    gdot = fmaf(Zs[i * ldD + d], Ys[t * ldD + d], gdot);
                }
                const float2 st = stats[bh * N + n];
                a = expf(pr.scale * sdot - st.x);
                g = a * (gdot - st.y);
            }
            A[i * (kTok + 1) + t] = a;
            dT[i * (kTok + 1) + t] = g;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kAcc; ++j) {
            const int e = tid + kT * j;
            const int i = e / D, d = e % D;
            if (e >= kRows * D) continue;
            float q = aq[j], z = az[j];
            for (int t = 0; t < kTok; ++t) {
                q = fmaf(dT[i * (kTok + 1) + t], Ks[t * ldD + d], q);
                z = fmaf(A[i * (kTok + 1) + t], Ys[t * ldD + d], z);
            }
            aq[j] = q;
            az[j] = z;
        }
    }
    // this chunk's partials: [bh][chunk][2][M][D]
    float *pc = part + ((bh * nchunks + c) * 2) * (int64_t)M * D;
#pragma unroll
    for (int j = 0; j < kAcc; ++j) {
        const int e = tid + kT * j;
        const int i = e / D, d = e % D;
        if (e >= kRows * D || i >= rows) continue;
        pc[(int64_t)(m0 + i) * D + d] = pr.scale * aq[j];
        pc[(int64_t)M * D + (int64_t)(m0 + i) * D + d] = az[j];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&tickets[bh * mtiles + mt], 1u);
        s_last = (prev == (unsigned)nchunks - 1u);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int e = tid; e < rows * D; e += kT) {
        const int i = e / D, d = e % D;
        float q = 0.f, z = 0.f;
        for (int cc = 0; cc < nchunks; ++cc) {
            const float *pcc = part + ((bh * nchunks + cc) * 2) * (int64_t)M * D;
            q += __ldcg(pcc + (int64_t)(m0 + i) * D + d);
            z += __ldcg(pcc + (int64_t)M * D + (int64_t)(m0 + i) * D + d);
        }
        dQ[(bh * M + m0 + i) * D + d] = q;
        dZ[(bh * M + m0 + i) * D + d] = z;
    }
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline int dq_nchunks(const Problem &pr) { return (pr.N + kChunk - 1) / kChunk; }

template <typename Kern>
cudaError_t smem_attr(Kern k, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

// Workspace: tickets [B*H*mtiles], token statistics [B*H*N] (float2), the
// chunk partials [B*H][nchunks][2][M][D].
size_t decode_bwd_simt_workspace(const Problem &pr) {
    const size_t bh = (size_t)pr.B * pr.H;
    const int mtiles = (pr.M + kRows - 1) / kRows;
    return align256(sizeof(unsigned) * bh * mtiles) + align256(sizeof(float) * 2 * bh * pr.N) +
           align256(sizeof(float) * bh * dq_nchunks(pr) * 2 * pr.M * pr.D);
}

cudaError_t launch_decode_bwd_simt(const Problem &pr, const void *Q, const float *Z, const void *K,
                                   const void *dY, float *dQ, float *dZ, void *dK, void *ws,
                                   cudaStream_t st) {
    const size_t bh = (size_t)pr.B * pr.H;
    if (bh == 0) return cudaSuccess;
    if (pr.N == 0) {
        cudaError_t e = cudaMemsetAsync(dQ, 0, sizeof(float) * bh * pr.M * pr.D, st);
        if (e != cudaSuccess) return e;
        return cudaMemsetAsync(dZ, 0, sizeof(float) * bh * pr.M * pr.D, st);
    }
    const int mtiles = (pr.M + kRows - 1) / kRows, nchunks = dq_nchunks(pr);
    char *w = (char *)ws;
    unsigned *tickets = (unsigned *)w;
    w += align256(sizeof(unsigned) * bh * mtiles);
    float2 *stats = (float2 *)w;
    w += align256(sizeof(float) * 2 * bh * pr.N);
    float *part = (float *)w;
    cudaError_t e = cudaMemsetAsync(tickets, 0, sizeof(unsigned) * bh * mtiles, st);
    if (e != cudaSuccess) return e;
    const size_t smem1 = sizeof(float) * (2 * kTok * (pr.D + 1) + 2 * kTok * (pr.M + 1));
    const size_t smem2 = sizeof(float) * (2 * kRows * (pr.D + 1) + 2 * kTok * (pr.D + 1) +
                                          2 * kRows * (kTok + 1));
    dim3 g1((pr.N + kTok - 1) / kTok, pr.H, pr.B), g2(nchunks, pr.H, pr.B * mtiles);
#define FLARE_DEC_BWD_LAUNCH(TQ, TK)                                                               \
    {                                                                                              \
        auto k1 = dec_bwd_dk_simt_kernel<TQ, TK>;                                                  \
        auto k2 = dec_bwd_dqz_simt_kernel<TQ, TK>;                                                 \
        if ((e = smem_attr(k1, smem1)) != cudaSuccess) return e;                                   \
        if ((e = smem_attr(k2, smem2)) != cudaSuccess) return e;                                   \
        k1<<<g1, kT, smem1, st>>>(pr, (const TQ *)Q, Z, (const TK *)K, (const TK *)dY, (TK *)dK,   \
                                  stats);                                                          \
        note_launch();                                                                             \
        k2<<<g2, kT, smem2, st>>>(pr, (const TQ *)Q, Z, (const TK *)K, (const TK *)dY, stats, dQ,  \
                                  dZ, tickets, part, nchunks, mtiles);                             \
        note_launch();                                                                             \
    }
    if (!pr.bf16) FLARE_DEC_BWD_LAUNCH(float, float)
    else FLARE_DEC_BWD_LAUNCH(__nv_bfloat16, __nv_bfloat16)
#undef FLARE_DEC_BWD_LAUNCH
    return cudaGetLastError();
}

}  // namespace flare
