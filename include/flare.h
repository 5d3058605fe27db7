/*
 * flare.h -- C ABI of the GB300 (sm_103a) FLARE / FLARE++ token-mixer library.
 *
 * The operations follow "FLARE++: Low-rank attention with dynamic attention
 * routing", appendix on context parallelism (arXiv 2608.11519, HTML). On that
 * page R context-parallel ranks each hold one token shard and exchange small
 * latent results with all-reduces; on one GPU the ranks become token shards of
 * one device buffer and the all-reduces become an in-device merge.
 *
 * Conventions shared by every entry point
 *  - Layouts are row-major. Token tensors (K, V, K~, V~, Y, dK, dV) are
 *    [B, N, H, D]: the per-token projection output with C = H*D channels.
 *    Latent tensors (Z, Q(X), dQ, dZ) are [B, H, M, D]. Row statistics (L)
 *    are [B, H, M]. A query Q (or FLARE++ seed tensor) is [H, M, D] shared by
 *    every batch element when dims->q_batch_stride == 0, else [B, H, M, D]
 *    with that many elements between batch elements.
 *  - Q, K, V, K~, V~, Y, dK, dV have the element type dims->dtype (fp32 or
 *    bf16). Z, L, O_r, L_r, Q(X), dZ, dQ are fp32. L values are natural-log
 *    log-normalisers that include the score scale.
 *  - mask is uint8 [B, N], 1 = valid token, 0 = padding (excluded from every
 *    softmax normalisation); NULL means every token is valid.
 *  - shard_offsets is a HOST array of R+1 int64 with offsets[0] = 0,
 *    offsets[R] = N and offsets nondecreasing; shard r owns tokens
 *    [offsets[r], offsets[r+1]) of every batch element. Shards may be empty.
 *    1 <= R <= FLARE_MAX_SHARDS.
 *  - Every other pointer is DEVICE memory owned by the caller. The library
 *    never allocates: a call that needs scratch memory takes a caller-owned
 *    workspace of at least flare_workspace_bytes() bytes. Workspaces and
 *    outputs must not overlap inputs. Concurrent calls need separate
 *    workspaces.
 *  - stream is a cudaStream_t (NULL = legacy default stream). Calls are
 *    stream-ordered and asynchronous: argument errors are reported
 *    synchronously before anything is launched (for the calls that chain
 *    several passes, the arguments of every pass are checked before the
 *    first launch); launch failures are returned
 *    as FLARE_ERR_CUDA; a kernel that abandoned a bounded wait records
 *    FLARE_ERR_TIMEOUT on the device, reported by flare_device_status().
 *  - On any error flare_last_error_string() describes it (thread-local).
 */
#ifndef FLARE_H_
#define FLARE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FLARE_API __attribute__((visibility("default")))
#else
#define FLARE_API
#endif

#define FLARE_MAX_SHARDS 256

typedef enum {
    FLARE_OK = 0,
    FLARE_ERR_INVALID_ARG = 1,  /* bad pointer, size, offsets or layout          */
    FLARE_ERR_UNSUPPORTED = 2,  /* valid, but no kernel for this shape or dtype  */
    FLARE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required    */
    FLARE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed          */
    FLARE_ERR_TIMEOUT = 5,      /* a kernel gave up a bounded wait (device flag) */
    FLARE_ERR_DEVICE_CHECK = 6  /* a device-side check of a FLARE_DEBUG build of
                                   the library failed (device flag); the access
                                   it guarded was skipped                        */
} flare_status_t;

typedef enum { FLARE_F32 = 0, FLARE_BF16 = 1 } flare_dtype_t;

/* Kernel family selection. AUTO picks the tensor-core (tcgen05/TMEM, TMA)
 * kernels for bf16 shapes they support and the CUDA-core kernels otherwise;
 * TENSOR returns FLARE_ERR_UNSUPPORTED where no tensor-core kernel applies.
 * Tensor-core shapes (bf16 only; fp32 always runs on CUDA cores):
 *   encoder, merge, decode:        D = 64 with M in {64, 128, 256},
 *                                  D = 128 with M in {64, 128};
 *   encoder and decode backward:   D = 64 with M in {64, 128, 256},
 *                                  D = 128 with M in {64, 128}.
 * The mixer entry points take, per step, the kernel family of that step. */
typedef enum { FLARE_KERNEL_AUTO = 0, FLARE_KERNEL_SIMT = 1, FLARE_KERNEL_TENSOR = 2 } flare_kernel_t;

typedef struct {
    int B;                  /* batch size                                      */
    int H;                  /* heads                                           */
    int M;                  /* latent queries per head (1..256)                */
    int N;                  /* tokens per batch element (all shards)           */
    int D;                  /* head dimension (1..128)                         */
    float scale;            /* score scale s; <= 0 selects s = D^-1/2          */
    flare_dtype_t dtype;    /* element type of the token tensors and of Q      */
    int64_t q_batch_stride; /* 0: Q is [H,M,D] replicated; H*M*D: [B,H,M,D]    */
    flare_kernel_t kernel;  /* kernel family (FLARE_KERNEL_AUTO by default)    */
} flare_dims_t;

typedef enum {
    FLARE_OP_ENCODER_FWD = 0,
    FLARE_OP_LSE_MERGE = 1,
    FLARE_OP_DECODE_FWD = 2,
    FLARE_OP_FWD = 3,
    FLARE_OP_PP_FWD = 4,
    FLARE_OP_ENCODER_BWD = 5,
    FLARE_OP_DECODE_BWD = 6,
    FLARE_OP_BWD = 7,
    FLARE_OP_PP_BWD = 8
} flare_op_t;

/* Workspace bytes `op` needs for these sizes and shard offsets (host array of
 * R+1 entries, may be NULL for ops that take none). Returns 0 when the op
 * needs no workspace, and (size_t)-1 when the arguments are invalid. */
FLARE_API size_t flare_workspace_bytes(flare_op_t op, const flare_dims_t *dims,
                             const int64_t *shard_offsets, int R);

/*
 * Split-KV encoder. Source: the per-shard local encoder and eq. 23 of the
 * appendix (the local primitive returns O_r normalised over shard r and the
 * row log-normaliser L_r; eq. 18 is the global result).
 * For every batch b, head h, latent m and shard r:
 *   S_mn = s <Q_m, K_n> over the valid tokens n of shard r,
 *   L_r  = log sum_n exp(S_mn),  O_r = sum_n exp(S_mn - L_r) V_n,
 * with L_r = -inf and O_r = 0 for a row that has no valid token on shard r.
 * When Z and L are given the shards are merged in the same call (eq. 23, see
 * flare_lse_merge) into the global Z [B,H,M,D] and L [B,H,M].
 *   Q       dims->dtype, [H,M,D] or [B,H,M,D] (dims->q_batch_stride)
 *   K, V    dims->dtype, [B,N,H,D]
 *   O_r     fp32 [R,B,H,M,D] or NULL;   L_r fp32 [R,B,H,M] or NULL
 *   Z       fp32 [B,H,M,D] or NULL;     L   fp32 [B,H,M] or NULL
 * At least one of the pairs (O_r, L_r) or (Z, L) must be given, each pair
 * complete. Scores are never stored: memory use does not grow with N*M.
 */
FLARE_API flare_status_t flare_encoder_fwd(const flare_dims_t *dims, const void *Q, const void *K,
                                 const void *V, const uint8_t *mask,
                                 const int64_t *shard_offsets, int R, float *O_r, float *L_r,
                                 float *Z, float *L, void *workspace, size_t workspace_bytes,
                                 void *stream);

/*
 * Exact log-sum-exp merge of R per-shard results. Source: eq. 23 and the
 * cross-rank log-sum-exp paragraph of the appendix (the all-reduce max and the
 * two all-reduce sums, done here in one kernel). Per row:
 *   L_max = max_r L_r,  a = sum_r exp(L_r - L_max),
 *   U = sum_r exp(L_r - L_max) O_r,  Z = U / a,  L = L_max + log a.
 * Rows where every L_r is -inf return L = -inf and Z = 0 (never NaN).
 *   O_r fp32 [R,B,H,M,D], L_r fp32 [R,B,H,M] -> Z fp32 [B,H,M,D], L fp32 [B,H,M].
 * No workspace. Shards are folded in index order, so results are
 * bit-reproducible run to run.
 */
FLARE_API flare_status_t flare_lse_merge(const float *O_r, const float *L_r, int R, int B, int H, int M,
                               int D, float *Z, float *L, void *stream);

/*
 * Local decode. Source: the FLARE decode paragraph of the appendix (the query
 * of each output token is local, both latent tensors replicated). Reading of
 * the stripped formula: each token's key is its decode query against the M
 * latent queries, with Z as values:
 *   Y[b,n,h] = sum_m softmax_m(s <K[b,n,h], Q_m>) Z[b,h,m].
 * Every token slot is decoded (there is no mask: the softmax runs over the M
 * latents, never empty).
 *   Q  dims->dtype [H,M,D] or [B,H,M,D];  Z fp32 [B,H,M,D];
 *   K  dims->dtype [B,N,H,D];  Y dims->dtype [B,N,H,D] (written).
 * No workspace.
 */
FLARE_API flare_status_t flare_decode_fwd(const flare_dims_t *dims, const void *Q, const float *Z,
                                const void *K, void *Y, void *stream);

/*
 * FLARE mixer forward: the split-KV encoder with the fused merge, then the
 * local decode. Source: the FLARE paragraph of the appendix (one globally
 * communicating encoder and one local decoder).
 *   Y dims->dtype [B,N,H,D]; Z fp32 [B,H,M,D]; L fp32 [B,H,M] (all written;
 *   Z and L are the saved forward statistics of the backward).
 */
FLARE_API flare_status_t flare_fwd(const flare_dims_t *dims, const void *Q, const void *K, const void *V,
                         const uint8_t *mask, const int64_t *shard_offsets, int R, void *Y,
                         float *Z, float *L, void *workspace, size_t workspace_bytes,
                         void *stream);

/*
 * FLARE++ mixer forward. Source: the FLARE++ paragraph of the appendix (the
 * same distributed encoder invoked twice, then the local decode):
 *   Q(X), L1 = encoder(seeds Q~, K~, V~)       (dynamic routing queries)
 *   Z, L2    = encoder(Q(X), K, V)             (physical latent values)
 *   Y        = decode(Q(X), Z, K)
 *   Qseed  dims->dtype, [H,M,D] or [B,H,M,D] (dims->q_batch_stride)
 *   Kt, Vt, K, V  dims->dtype [B,N,H,D] (projected tokens, same mask/shards)
 *   Y dims->dtype [B,N,H,D]; Qdyn fp32 [B,H,M,D]; L1, L2 fp32 [B,H,M];
 *   Z fp32 [B,H,M,D]. Both encoders' statistics are returned because their
 *   backward passes need their own saved outputs.
 * On the bf16 path Q(X) is rounded to bf16 (round-to-nearest-even) where it
 * feeds the tensor-core kernels; Qdyn itself is returned in fp32.
 */
FLARE_API flare_status_t flare_pp_fwd(const flare_dims_t *dims, const void *Qseed, const void *Kt,
                            const void *Vt, const void *K, const void *V, const uint8_t *mask,
                            const int64_t *shard_offsets, int R, void *Y, float *Qdyn,
                            float *L1, float *Z, float *L2, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * Encoder backward with the global forward statistics. Source: the backward
 * paragraphs of the appendix (globally normalised local probabilities, the
 * row scalar c, local gradients, query gradient summed over shards):
 *   P_mn = exp(s <Q_m, K_n> - L_m)   (global L; masked tokens and rows with
 *                                     L = -inf give P = 0)
 *   c_m  = <dZ_m, Z_m>
 *   dV_n = sum_m P_mn dZ_m
 *   dS_mn = P_mn (<dZ_m, V_n> - c_m)
 *   dK_n = s sum_m dS_mn Q_m,   dQ_m = s sum_n dS_mn K_n  (sum over all shards)
 *   Z, L  fp32 (from the forward), dZ fp32 [B,H,M,D] (summed over every
 *         consumer of Z by the caller)
 *   dQ fp32 [B,H,M,D] (one slice per batch element, also when Q is
 *         replicated: the caller sums over B); dK, dV dims->dtype [B,N,H,D].
 * With the global L and c every token's gradient is independent of the other
 * shards, so the shard offsets only need to be valid.
 */
FLARE_API flare_status_t flare_encoder_bwd(const flare_dims_t *dims, const void *Q, const void *K,
                                 const void *V, const uint8_t *mask,
                                 const int64_t *shard_offsets, int R, const float *Z,
                                 const float *L, const float *dZ, float *dQ, void *dK, void *dV,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * flare_encoder_bwd that adds its shares to gradients another consumer has
 * already written. Source: the backward paragraphs of the appendix (a
 * replicated tensor's gradient is the sum of its consumers' contributions;
 * dQ is summed over shards and ranks). Arguments, layouts and workspace are
 * those of flare_encoder_bwd, except:
 *   dQ  fp32 [B,H,M,D] is read and the encoder's share added to it;
 *   dK  dims->dtype [B,N,H,D] is read and the encoder's share added to it
 *       (the sum taken in fp32 and rounded once to dims->dtype);
 *   dV  dims->dtype [B,N,H,D] is written (V has no other consumer).
 * A context-parallel rank uses it after its decode backward: the decode's
 * shares of dQ and dK are in place, the all-reduced dZ is the input.
 */
FLARE_API flare_status_t flare_encoder_bwd_accumulate(const flare_dims_t *dims, const void *Q,
                                                      const void *K, const void *V,
                                                      const uint8_t *mask,
                                                      const int64_t *shard_offsets, int R,
                                                      const float *Z, const float *L,
                                                      const float *dZ, float *dQ, void *dK,
                                                      void *dV, void *workspace,
                                                      size_t workspace_bytes, void *stream);

/*
 * Decode backward: the chain rule of the local decode (the FLARE decode
 * paragraph of the appendix; the pages name the decoder's contribution to the
 * gradients of the latent tensors but print no formula). For the gradient dY
 * of the decode output, per batch b, head h, token n and latent m:
 *   A_nm  = softmax_m(s <K_n, Q_m>),  g_nm = <dY_n, Z_m>,  r_n = sum_m A_nm g_nm,
 *   dT_nm = A_nm (g_nm - r_n),
 *   dZ_m  = sum_n A_nm dY_n,  dK_n = s sum_m dT_nm Q_m,  dQ_m = s sum_n dT_nm K_n.
 *   Q   dims->dtype [H,M,D] or [B,H,M,D];  Z fp32 [B,H,M,D];
 *   K, dY  dims->dtype [B,N,H,D];
 *   dQ fp32 [B,H,M,D] (one slice per batch element, also when Q is
 *   replicated); dZ fp32 [B,H,M,D]; dK dims->dtype [B,N,H,D] (the decode's
 *   share of the key gradient; the encoder backward adds its own).
 * Every token slot contributes (the decode has no mask). Workspace:
 * flare_workspace_bytes(FLARE_OP_DECODE_BWD, dims, NULL, 0) bytes.
 */
FLARE_API flare_status_t flare_decode_bwd(const flare_dims_t *dims, const void *Q, const float *Z,
                                          const void *K, const void *dY, float *dQ, float *dZ,
                                          void *dK, void *workspace, size_t workspace_bytes,
                                          void *stream);

/*
 * FLARE mixer backward. Source: the backward paragraphs of the appendix (the
 * gradient of the replicated Z is first summed over its consumers, then the
 * encoder is differentiated with the forward's global Z and L). In the mixer
 * Z's only consumer is the decode; Q enters the encoder (latent queries) and
 * the decode (latent keys), K the encoder (keys) and the decode (token
 * queries). So: flare_decode_bwd gives dQ_dec, dZ, dK_dec; flare_encoder_bwd
 * with that dZ gives dQ_enc, dK_enc, dV; and
 *   dQ = dQ_dec + dQ_enc   fp32 [B,H,M,D] (one slice per batch element)
 *   dK = dK_dec + dK_enc   dims->dtype [B,N,H,D] (the decode's share is stored
 *                          in dims->dtype, then the encoder's fp32 share is
 *                          added and the sum rounded once more)
 *   dV = dV_enc            dims->dtype [B,N,H,D]
 *   Q, K, V, mask, shard_offsets: as for flare_fwd; Z, L: flare_fwd's outputs;
 *   dY dims->dtype [B,N,H,D].
 * Workspace: flare_workspace_bytes(FLARE_OP_BWD, dims, shard_offsets, R) bytes
 * (dZ, then the scratch of the two passes).
 */
FLARE_API flare_status_t flare_bwd(const flare_dims_t *dims, const void *Q, const void *K,
                                   const void *V, const uint8_t *mask,
                                   const int64_t *shard_offsets, int R, const float *Z,
                                   const float *L, const void *dY, float *dQ, void *dK, void *dV,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * FLARE++ mixer backward. Source: the FLARE++ backward paragraph of the
 * appendix. The decode with the dynamic queries Q(X) gives the decoder's
 * shares of dQ(X), dZ and dK; the physical-value encoder (its own Z, L2) adds
 * its shares of dQ(X) and dK and gives dV; the summed dQ(X) is the output
 * gradient of the query-synthesis encoder, whose backward with its own saved
 * output Q(X) and L1 gives the seeds' gradient and those of K~, V~:
 *   Qseed dims->dtype [H,M,D] or [B,H,M,D] (dims->q_batch_stride);
 *   Kt, Vt, K, V, dY dims->dtype [B,N,H,D]; Qdyn, L1, Z, L2: flare_pp_fwd's
 *   outputs (Qdyn 16-byte aligned);
 *   dQseed fp32 [B,H,M,D] (one slice per batch element); dKt, dVt, dK, dV
 *   dims->dtype [B,N,H,D]; dQdyn: optional fp32 [B,H,M,D] (16-byte aligned)
 *   receiving the summed gradient of Q(X), or NULL (kept in the workspace).
 * On the bf16 path Q(X) is rounded to bf16 (nearest even) as the operand of
 * the decode and physical-value encoder backward, as in the forward.
 * Workspace: flare_workspace_bytes(FLARE_OP_PP_BWD, dims, shard_offsets, R).
 */
FLARE_API flare_status_t flare_pp_bwd(const flare_dims_t *dims, const void *Qseed, const void *Kt,
                                      const void *Vt, const void *K, const void *V,
                                      const uint8_t *mask, const int64_t *shard_offsets, int R,
                                      const float *Qdyn, const float *L1, const float *Z,
                                      const float *L2, const void *dY, float *dQseed, void *dKt,
                                      void *dVt, void *dK, void *dV, float *dQdyn, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * Split-KV encoder without a workspace argument, for callers that cannot
 * allocate device memory: plugins inside host frameworks that own all device
 * memory and hand none to extensions, and code on paths where calling
 * cudaMalloc is not allowed. The pages have no counterpart; the arithmetic,
 * arguments and results are those of flare_encoder_fwd.
 * Its scratch memory is one static device array of 32 MiB (2^25 bytes) in
 * this library, held by every GPU that loads the library until the process
 * exits. Problems whose flare_workspace_bytes(FLARE_OP_ENCODER_FWD, ...)
 * exceeds it are rejected with FLARE_ERR_WORKSPACE. The first call on a
 * device looks the array's device address up (cudaGetSymbolAddress) and keeps
 * it for the life of the process, so make that first call before any stream
 * capture, and do not go on calling this entry point after cudaDeviceReset or
 * from another CUDA context of the same device (the module may then be loaded
 * at another address than the one kept). Every call on a device shares
 * the array: calls that may overlap on the GPU (other streams, other host
 * threads) race and give wrong results; serialise them. Nothing is allocated
 * or freed; the ticket counters are cleared with cudaMemsetAsync each call.
 */
FLARE_API flare_status_t flare_encoder_fwd_noalloc(const flare_dims_t *dims, const void *Q,
                                                   const void *K, const void *V, const uint8_t *mask,
                                                   const int64_t *shard_offsets, int R, float *O_r,
                                                   float *L_r, float *Z, float *L, void *stream);

/* Failure-path check of the bounded waits (no counterpart on the pages).
 * Launches, on `stream`, one small kernel whose only work is a wait on an
 * mbarrier that nothing arrives on; after limit_us microseconds (1..1000000)
 * it gives the wait up exactly as the library's kernels do when an expected
 * copy or MMA never completes: the CTA unwinds and FLARE_ERR_TIMEOUT is
 * recorded in the device status word, to be read (and cleared) by
 * flare_device_status. Nothing faults and the context stays usable, so a
 * caller can test its handling of FLARE_ERR_TIMEOUT. Returns
 * FLARE_ERR_INVALID_ARG for a limit out of range, FLARE_ERR_CUDA if the
 * launch fails. */
FLARE_API flare_status_t flare_check_bounded_wait(unsigned limit_us, void *stream);

/* Synchronises `stream`, then reads and clears the device status word that
 * kernels set when they abandon a bounded wait (or, in a FLARE_DEBUG build,
 * when a device-side check of a tile's place or a workspace index fails; the
 * first error recorded wins): FLARE_OK, FLARE_ERR_TIMEOUT,
 * FLARE_ERR_DEVICE_CHECK, or FLARE_ERR_CUDA if the synchronisation itself
 * failed. */
FLARE_API flare_status_t flare_device_status(void *stream);

/* Text of the calling thread's most recent error (empty if none). */
FLARE_API const char *flare_last_error_string(void);

/* Library version as major*10000 + minor*100 + patch. */
FLARE_API int flare_version(void);

/* Kernels this library has launched in this process so far (every device and
 * host thread; one count per kernel launch, memsets not included). A
 * diagnostic: the difference across a call is that call's launch count. */
FLARE_API unsigned long long flare_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FLARE_H_ */
