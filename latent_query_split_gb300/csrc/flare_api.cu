// flare_api.cu -- the C ABI (include/flare.h): argument validation, work
// planning, workspace carve-up and kernel selection. Every computation runs
// in the kernels of simt_kernels.cu and the tensor-core translation units.
#include "flare_internal.cuh"
#include "tc_common.cuh"

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

namespace flare {

// Status word of every kernel that waits with a bound (see flare_device_status).
__device__ unsigned g_device_status;

std::atomic<unsigned long long> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

thread_local std::string t_error;

flare_status_t fail(flare_status_t s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_error = buf;
    return s;
}

flare_status_t cuda_fail(cudaError_t e, const char *what) {
    return fail(FLARE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct DeviceInfo {
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    unsigned *status = nullptr;
};

std::mutex g_dev_mutex;
std::vector<DeviceInfo> g_devs;

// Per-device facts, looked up once per device (with that device current).
flare_status_t device_info(DeviceInfo &out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if ((int)g_devs.size() <= dev) g_devs.resize(dev + 1);
    DeviceInfo &d = g_devs[dev];
    if (d.sms == 0) {
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        void *p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_device_status)) != cudaSuccess) {
            d.sms = 0;
            return cuda_fail(e, "cudaGetSymbolAddress(status)");
        }
        d.status = (unsigned *)p;
    }
    out = d;
    return FLARE_OK;
}

// Streaming-multiprocessor count used for planning without a device query
// failing the workspace size function (the planner needs a number).
int planning_sms() {
    DeviceInfo d;
    if (device_info(d) == FLARE_OK && d.sms > 0) return d.sms;
    return 152;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

flare_status_t check_dims(const flare_dims_t *d) {
    if (!d) return fail(FLARE_ERR_INVALID_ARG, "dims is NULL");
    if (d->B < 0 || d->N < 0) return fail(FLARE_ERR_INVALID_ARG, "B and N must be >= 0");
    if (d->H < 1 || d->M < 1 || d->D < 1)
        return fail(FLARE_ERR_INVALID_ARG, "H, M and D must be >= 1 (H=%d M=%d D=%d)", d->H, d->M, d->D);
    if (d->dtype != FLARE_F32 && d->dtype != FLARE_BF16)
        return fail(FLARE_ERR_INVALID_ARG, "unknown dtype %d", (int)d->dtype);
    if (d->kernel != FLARE_KERNEL_AUTO && d->kernel != FLARE_KERNEL_SIMT &&
        d->kernel != FLARE_KERNEL_TENSOR)
        return fail(FLARE_ERR_INVALID_ARG, "unknown kernel family %d", (int)d->kernel);
    if (d->M > 256) return fail(FLARE_ERR_UNSUPPORTED, "M=%d > 256 latents", d->M);
    if (d->D > 128) return fail(FLARE_ERR_UNSUPPORTED, "D=%d > 128", d->D);
    const int64_t hmd = (int64_t)d->H * d->M * d->D;
    if (d->q_batch_stride != 0 && d->q_batch_stride != hmd)
        return fail(FLARE_ERR_INVALID_ARG, "q_batch_stride must be 0 or H*M*D (%lld)", (long long)hmd);
    if (!(std::isfinite(d->scale))) return fail(FLARE_ERR_INVALID_ARG, "scale is not finite");
    if ((int64_t)d->B * ((d->M + kSimtRows - 1) / kSimtRows) > 65535 || d->H > 65535)
        return fail(FLARE_ERR_UNSUPPORTED, "B*ceil(M/32) and H must stay within 65535");
    return FLARE_OK;
}

flare_status_t check_offsets(const int64_t *off, int R, int N) {
    if (R < 1 || R > kMaxShards)
        return fail(FLARE_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, kMaxShards);
    if (!off) return fail(FLARE_ERR_INVALID_ARG, "shard_offsets is NULL");
    if (off[0] != 0) return fail(FLARE_ERR_INVALID_ARG, "shard_offsets[0] must be 0");
    if (off[R] != N)
        return fail(FLARE_ERR_INVALID_ARG, "shard_offsets[R]=%lld must equal N=%d", (long long)off[R], N);
    for (int r = 0; r < R; ++r)
        if (off[r + 1] < off[r])
            return fail(FLARE_ERR_INVALID_ARG, "shard_offsets decrease at shard %d", r);
    return FLARE_OK;
}

Problem make_problem(const flare_dims_t *d) {
    Problem p;
    p.B = d->B;
    p.H = d->H;
    p.M = d->M;
    p.N = d->N;
    p.D = d->D;
    p.scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt((float)d->D);
    p.q_bstride = d->q_batch_stride;
    p.bf16 = d->dtype == FLARE_BF16;
    return p;
}

size_t elem_size(const flare_dims_t *d) { return d->dtype == FLARE_BF16 ? 2 : 4; }

// Chunking of the shards: chunks never cross a shard boundary and hold at most
// chunk_len tokens; chunk_len is sized so the grid covers the GPU several
// times over (B*H*mtiles CTAs per chunk index).
void make_plan(const int64_t *off, int R, int N, int tile, int min_chunk, int64_t ctas_per_chunk,
               int64_t target_ctas, ShardPlan &p) {
    std::memset(&p, 0, sizeof p);
    p.R = R;
    const int64_t work = ctas_per_chunk * (int64_t)N;              // CTA-token units
    int64_t ideal = (work + target_ctas - 1) / (target_ctas > 0 ? target_ctas : 1);
    ideal = ((ideal + tile - 1) / tile) * tile;
    int64_t chunk = ideal < min_chunk ? min_chunk : ideal;
    if (chunk > (1 << 30)) chunk = 1 << 30;
    p.chunk_len = (int)chunk;
    int total = 0;
    for (int r = 0; r < R; ++r) {
        p.off[r] = off[r];
        p.chunk_start[r] = total;
        const int64_t len = off[r + 1] - off[r];
        total += (int)((len + chunk - 1) / chunk);
    }
    p.off[R] = off[R];
    p.chunk_start[R] = total;
    p.total_chunks = total;
}

// Which kernel family runs an encoder / decode of these dims.
bool use_tensor_cores(const flare_dims_t *d) {
    if (d->kernel == FLARE_KERNEL_SIMT) return false;
    return tc_supported(d->dtype == FLARE_BF16, d->M, d->D);
}

struct EncoderLayout {
    ShardPlan plan;        // CUDA-core path
    int mtiles;
    bool tc;
    TcTilePlan tcplan;     // tensor-core path
    TcEncLayout tclay;
    EncoderWorkspace ws;   // pointers relative to a null base until bound
};

void encoder_layout(const flare_dims_t *d, const int64_t *off, int R, bool tc, EncoderLayout &lay) {
    const int sms = planning_sms();
    lay.tc = tc;
    const size_t bh = (size_t)d->B * d->H;
    EncoderWorkspace &w = lay.ws;
    if (tc) {
        lay.mtiles = 1;
        if (!tc_encoder_plan(make_problem(d), off, R, sms, lay.tcplan, lay.tclay)) {
            lay.tc = false;               // too many pieces per (b, h): CUDA-core path
            encoder_layout(d, off, R, false, lay);
            return;
        }
        w.tickets = nullptr;              // the tensor-core path merges in a separate kernel
        w.part_L = (float *)lay.tclay.part_L;
        w.part_O = (float *)lay.tclay.part_O;
        w.shard_L = nullptr;
        w.bytes = lay.tclay.bytes;
        return;
    }
    lay.mtiles = (d->M + kSimtRows - 1) / kSimtRows;
    // chunks of at least two tiles: small problems still spread over many CTAs
    make_plan(off, R, d->N, kSimtTile, 2 * kSimtTile, (int64_t)bh * lay.mtiles, (int64_t)sms * 8, lay.plan);
    size_t o = 0;
    w.tickets = (unsigned *)o;
    o += align256(sizeof(unsigned) * bh * lay.mtiles);
    w.part_L = (float *)o;
    o += align256(sizeof(float) * bh * lay.plan.total_chunks * d->M);
    w.part_O = (float *)o;
    o += align256(sizeof(float) * bh * lay.plan.total_chunks * d->M * d->D);
    w.shard_L = (float *)o;
    o += align256(sizeof(float) * bh * R * d->M);
    w.bytes = o;
}

EncoderWorkspace bind(const EncoderWorkspace &rel, void *base) {
    EncoderWorkspace w = rel;
    char *b = (char *)base;
    w.tickets = (unsigned *)(b + (size_t)rel.tickets);
    w.part_L = (float *)(b + (size_t)rel.part_L);
    w.part_O = (float *)(b + (size_t)rel.part_O);
    w.shard_L = (float *)(b + (size_t)rel.shard_L);
    return w;
}

size_t encoder_ws_bytes(const flare_dims_t *d, const int64_t *off, int R) {
    static thread_local EncoderLayout a;
    encoder_layout(d, off, R, false, a);
    size_t bytes = a.ws.bytes;
    if (use_tensor_cores(d)) {
        encoder_layout(d, off, R, true, a);
        if (a.ws.bytes > bytes) bytes = a.ws.bytes;
    }
    return bytes;
}

__global__ void fill_empty_kernel(float *O_r, int64_t nO, float *L_r, int64_t nLr, float *Z,
                                  int64_t nZ, float *L, int64_t nL) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = i; k < nO; k += stride) O_r[k] = 0.f;
    for (int64_t k = i; k < nLr; k += stride) L_r[k] = -INFINITY;
    for (int64_t k = i; k < nZ; k += stride) Z[k] = 0.f;
    for (int64_t k = i; k < nL; k += stride) L[k] = -INFINITY;
}

// Core of flare_encoder_fwd, also used by flare_fwd and flare_pp_fwd.
// q_is_f32: the query is fp32 even though the token tensors are bf16 (the
// FLARE++ dynamic queries). check_only: validate every argument and return
// before anything is launched (the composite calls check all of their
// stages before the first launch).
flare_status_t encoder_run(const flare_dims_t *d, const void *Q, bool q_is_f32, const void *K,
                           const void *V, const uint8_t *mask, const int64_t *off, int R,
                           float *O_r, float *L_r, float *Z, float *L, void *ws, size_t ws_bytes,
                           cudaStream_t st, bool check_only = false) {
    if ((O_r == nullptr) != (L_r == nullptr))
        return fail(FLARE_ERR_INVALID_ARG, "O_r and L_r must be given together");
    if ((Z == nullptr) != (L == nullptr))
        return fail(FLARE_ERR_INVALID_ARG, "Z and L must be given together");
    if (!O_r && !Z) return fail(FLARE_ERR_INVALID_ARG, "no output requested");
    const Problem pr = make_problem(d);
    if (pr.B == 0) return FLARE_OK;
    const size_t es = elem_size(d);
    if (!Q || (pr.N > 0 && (!K || !V))) return fail(FLARE_ERR_INVALID_ARG, "NULL input tensor");
    const size_t qes = q_is_f32 ? 4 : es;
    if (!aligned(Q, qes) || !aligned(K, es) || !aligned(V, es))
        return fail(FLARE_ERR_INVALID_ARG, "input tensors must be aligned to their element size");
    if (!aligned(O_r, 4) || !aligned(L_r, 4) || !aligned(Z, 4) || !aligned(L, 4))
        return fail(FLARE_ERR_INVALID_ARG, "fp32 outputs must be 4-byte aligned");
    const bool want_tc = use_tensor_cores(d);
    if (d->kernel == FLARE_KERNEL_TENSOR && !want_tc)
        return fail(FLARE_ERR_UNSUPPORTED, "no tensor-core encoder for dtype=%d M=%d D=%d",
                    (int)d->dtype, d->M, d->D);
    const bool tc = want_tc && tc_pointers_ok(K, V, d->H, d->D) && (q_is_f32 || aligned(Q, 16));
    if (d->kernel == FLARE_KERNEL_TENSOR && !tc)
        return fail(FLARE_ERR_INVALID_ARG, "tensor-core encoder needs 16-byte aligned Q, K and V");
    static thread_local EncoderLayout lay;     // ~7 KB: kept off the stack
    encoder_layout(d, off, R, tc, lay);
    const bool use_tc = lay.tc;
    const size_t need = encoder_ws_bytes(d, off, R);
    const int64_t bhm = (int64_t)pr.B * pr.H * pr.M;
    if (pr.N == 0) {                           // no token: every row is empty
        if (check_only) return FLARE_OK;
        fill_empty_kernel<<<64, 256, 0, st>>>(O_r, O_r ? R * bhm * pr.D : 0, L_r, L_r ? R * bhm : 0,
                                               Z, Z ? bhm * pr.D : 0, L, L ? bhm : 0);
        note_launch();
        cudaError_t e = cudaGetLastError();
        return e == cudaSuccess ? FLARE_OK : cuda_fail(e, "fill_empty_kernel launch");
    }
    if (!ws || ws_bytes < need)
        return fail(FLARE_ERR_WORKSPACE, "workspace of %zu bytes required, %zu given", need, ws_bytes);
    if (!aligned(ws, 256)) return fail(FLARE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (check_only) return FLARE_OK;
    EncoderWorkspace w = bind(lay.ws, ws);
    EncoderOut out{O_r, L_r, Z, L};
    cudaError_t e;
    if (use_tc) {
        DeviceInfo di;
        flare_status_t s = device_info(di);
        if (s != FLARE_OK) return s;
        e = launch_encoder_tc(pr, lay.tcplan, lay.tclay, Q, q_is_f32, K, V, mask, ws, out,
                              di.status, st);
    } else {
        e = cudaMemsetAsync(w.tickets, 0, sizeof(unsigned) * (size_t)pr.B * pr.H * lay.mtiles, st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(tickets)");
        e = launch_encoder_simt(pr, lay.plan, Q, q_is_f32, K, V, mask, w, out, st);
    }
    return e == cudaSuccess ? FLARE_OK : cuda_fail(e, "encoder launch");
}

flare_status_t decode_run(const flare_dims_t *d, const void *Q, bool q_is_f32, const float *Z,
                          const void *K, void *Y, bool after_merge, cudaStream_t st,
                          bool check_only = false) {
    const Problem pr = make_problem(d);
    if (pr.B == 0 || pr.N == 0) return FLARE_OK;
    if (!Q || !Z || !K || !Y) return fail(FLARE_ERR_INVALID_ARG, "NULL tensor");
    const size_t es = elem_size(d);
    if (!aligned(Q, q_is_f32 ? 4 : es) || !aligned(K, es) || !aligned(Y, es) || !aligned(Z, 4))
        return fail(FLARE_ERR_INVALID_ARG, "tensors must be aligned to their element size");
    const bool want_tc = use_tensor_cores(d) && tc_decode_available();
    if (d->kernel == FLARE_KERNEL_TENSOR && !want_tc)
        return fail(FLARE_ERR_UNSUPPORTED, "no tensor-core decode for dtype=%d M=%d D=%d",
                    (int)d->dtype, d->M, d->D);
    const bool tc = want_tc && tc_pointers_ok(K, Y, d->H, d->D) && aligned(Q, 16) && aligned(Z, 16);
    if (d->kernel == FLARE_KERNEL_TENSOR && !tc)
        return fail(FLARE_ERR_INVALID_ARG, "tensor-core decode needs 16-byte aligned Q, Z, K and Y");
    if (check_only) return FLARE_OK;
    cudaError_t e;
    if (tc) {
        DeviceInfo di;
        flare_status_t s = device_info(di);
        if (s != FLARE_OK) return s;
        e = launch_decode_tc(pr, Q, q_is_f32, Z, K, Y, di.sms, di.status, after_merge, st);
    } else {
        e = launch_decode_simt(pr, Q, q_is_f32, Z, K, Y, after_merge, st);
    }
    return e == cudaSuccess ? FLARE_OK : cuda_fail(e, "decode launch");
}


size_t encoder_bwd_ws(const flare_dims_t *d) {
    const Problem pr = make_problem(d);
    size_t b = encoder_bwd_simt_workspace(pr);
    if (d->kernel != FLARE_KERNEL_SIMT) {
        const size_t t = tc_encoder_bwd_workspace(pr, planning_sms());
        if (t > b) b = t;
    }
    return b;
}

size_t decode_bwd_ws(const flare_dims_t *d) {
    const Problem pr = make_problem(d);
    size_t b = decode_bwd_simt_workspace(pr);
    if (d->kernel != FLARE_KERNEL_SIMT) {
        const size_t t = tc_decode_bwd_workspace(pr, planning_sms());
        if (t > b) b = t;
    }
    return b;
}

// Core of flare_encoder_bwd (dims and offsets already checked). accumulate:
// dQ and dK already hold another consumer's share and this pass adds its own.
// check_only: as for encoder_run.
flare_status_t encoder_bwd_run(const flare_dims_t *dims, const void *Q, const void *K, const void *V,
                               const uint8_t *mask, const float *Z, const float *L, const float *dZ,
                               float *dQ, void *dK, void *dV, void *workspace, size_t workspace_bytes,
                               bool accumulate, cudaStream_t st, bool check_only = false) {
    const Problem pr = make_problem(dims);
    if (pr.B == 0) return FLARE_OK;
    if (!Q || !Z || !L || !dZ || !dQ || (pr.N > 0 && (!K || !V || !dK || !dV)))
        return fail(FLARE_ERR_INVALID_ARG, "NULL tensor");
    const size_t es = elem_size(dims);
    if (!aligned(Q, es) || !aligned(K, es) || !aligned(V, es) || !aligned(dK, es) ||
        !aligned(dV, es) || !aligned(Z, 4) || !aligned(L, 4) || !aligned(dZ, 4) || !aligned(dQ, 4))
        return fail(FLARE_ERR_INVALID_ARG, "tensors must be aligned to their element size");
    const bool want_tc = dims->kernel != FLARE_KERNEL_SIMT && tc_bwd_supported(pr.bf16, pr.M, pr.D);
    if (dims->kernel == FLARE_KERNEL_TENSOR && !want_tc)
        return fail(FLARE_ERR_UNSUPPORTED, "no tensor-core backward for dtype=%d M=%d D=%d",
                    (int)dims->dtype, dims->M, dims->D);
    const bool tc = want_tc && tc_pointers_ok(K, V, dims->H, dims->D) &&
                    tc_pointers_ok(dK, dV, dims->H, dims->D) && aligned(Q, 16) && aligned(Z, 16) &&
                    aligned(dZ, 16) && aligned(dQ, 16);
    if (dims->kernel == FLARE_KERNEL_TENSOR && !tc)
        return fail(FLARE_ERR_INVALID_ARG,
                    "tensor-core backward needs 16-byte aligned Q, K, V, Z, dZ, dQ, dK and dV");
    const size_t need = encoder_bwd_ws(dims);
    if (pr.N > 0 && (!workspace || workspace_bytes < need))
        return fail(FLARE_ERR_WORKSPACE, "workspace of %zu bytes required, %zu given", need,
                    workspace_bytes);
    if (workspace && !aligned(workspace, 256))
        return fail(FLARE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (check_only) return FLARE_OK;
    cudaError_t e;
    if (tc) {
        DeviceInfo di;
        flare_status_t s = device_info(di);
        if (s != FLARE_OK) return s;
        e = launch_encoder_bwd_tc(pr, Q, K, V, mask, Z, L, dZ, dQ, dK, dV, workspace,
                                  workspace_bytes, di.sms, di.status, st, accumulate);
    } else {
        e = launch_encoder_bwd_simt(pr, Q, K, V, mask, Z, L, dZ, dQ, dK, dV, workspace,
                                    workspace_bytes, st, accumulate);
    }
    return e == cudaSuccess ? FLARE_OK : cuda_fail(e, "encoder backward launch");
}

// Core of flare_decode_bwd (dims already checked). check_only: as for encoder_run.
flare_status_t decode_bwd_run(const flare_dims_t *dims, const void *Q, const float *Z, const void *K,
                              const void *dY, float *dQ, float *dZ, void *dK, void *workspace,
                              size_t workspace_bytes, cudaStream_t st, bool check_only = false) {
    const Problem pr = make_problem(dims);
    if (pr.B == 0) return FLARE_OK;
    if (!Q || !Z || !dQ || !dZ || (pr.N > 0 && (!K || !dY || !dK)))
        return fail(FLARE_ERR_INVALID_ARG, "NULL tensor");
    const size_t es = elem_size(dims);
    if (!aligned(Q, es) || !aligned(K, es) || !aligned(dY, es) || !aligned(dK, es) || !aligned(Z, 4) ||
        !aligned(dQ, 4) || !aligned(dZ, 4))
        return fail(FLARE_ERR_INVALID_ARG, "tensors must be aligned to their element size");
    const bool want_tc = dims->kernel != FLARE_KERNEL_SIMT && tc_decode_bwd_supported(pr.bf16, pr.M, pr.D);
    if (dims->kernel == FLARE_KERNEL_TENSOR && !want_tc)
        return fail(FLARE_ERR_UNSUPPORTED, "no tensor-core decode backward for dtype=%d M=%d D=%d",
                    (int)dims->dtype, dims->M, dims->D);
    const bool tc = want_tc && tc_pointers_ok(K, dY, dims->H, dims->D) &&
                    tc_pointers_ok(dK, dK, dims->H, dims->D) && aligned(Q, 16) && aligned(Z, 16) &&
                    aligned(dQ, 16) && aligned(dZ, 16);
    if (dims->kernel == FLARE_KERNEL_TENSOR && !tc)
        return fail(FLARE_ERR_INVALID_ARG,
                    "tensor-core decode backward needs 16-byte aligned Q, Z, K, dY, dQ, dZ and dK");
    const size_t need = decode_bwd_ws(dims);
    if (!workspace || workspace_bytes < need)
        return fail(FLARE_ERR_WORKSPACE, "workspace of %zu bytes required, %zu given", need,
                    workspace_bytes);
    if (!aligned(workspace, 256)) return fail(FLARE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (check_only) return FLARE_OK;
    cudaError_t e;
    if (tc) {
        DeviceInfo di;
        flare_status_t s = device_info(di);
        if (s != FLARE_OK) return s;
        e = launch_decode_bwd_tc(pr, Q, Z, K, dY, dQ, dZ, dK, workspace, workspace_bytes, di.sms,
                                 di.status, st);
    } else {
        e = launch_decode_bwd_simt(pr, Q, Z, K, dY, dQ, dZ, dK, workspace, st);
    }
    return e == cudaSuccess ? FLARE_OK : cuda_fail(e, "decode backward launch");
}

// Workspace of the mixer backward passes: the latent gradients that pass
// from one stage to the next, then scratch shared by the stages in turn.
struct MixerBwdLayout {
    size_t dz = 0, dqdyn = 0, qdyn_b = 0, scratch = 0, bytes = 0;
};

void mixer_bwd_layout(const flare_dims_t *d, bool pp, MixerBwdLayout &l) {
    const size_t lat = (size_t)d->B * d->H * d->M * d->D;
    size_t o = 0;
    l.dz = o;
    o += align256(sizeof(float) * lat);
    size_t scratch = decode_bwd_ws(d);
    const size_t enc = encoder_bwd_ws(d);
    if (enc > scratch) scratch = enc;
    if (pp) {
        l.dqdyn = o;
        o += align256(sizeof(float) * lat);
        l.qdyn_b = o;
        if (d->dtype == FLARE_BF16) o += align256(2 * lat);
    }
    l.scratch = o;
    l.bytes = o + scratch;
}

}  // namespace

// Entry points for the allocation-free encoder (noalloc.cu): the same
// validation, planning and launch as flare_encoder_fwd, with the workspace
// size and the error text exposed.
size_t encoder_workspace_size(const flare_dims_t *dims, const int64_t *off, int R) {
    if (check_dims(dims) != FLARE_OK || check_offsets(off, R, dims->N) != FLARE_OK) return (size_t)-1;
    return encoder_ws_bytes(dims, off, R);
}

flare_status_t encoder_fwd_with_workspace(const flare_dims_t *dims, const void *Q, const void *K,
                                          const void *V, const uint8_t *mask, const int64_t *off,
                                          int R, float *O_r, float *L_r, float *Z, float *L,
                                          void *ws, size_t ws_bytes, cudaStream_t st) {
    flare_status_t s = check_dims(dims);
    if (s != FLARE_OK) return s;
    if ((s = check_offsets(off, R, dims->N)) != FLARE_OK) return s;
    return encoder_run(dims, Q, false, K, V, mask, off, R, O_r, L_r, Z, L, ws, ws_bytes, st);
}

flare_status_t report_error(flare_status_t s, const char *msg) { return fail(s, "%s", msg); }

}  // namespace flare

using namespace flare;

extern "C" {

int flare_version(void) { return 1 * 10000 + 0 * 100 + 0; }

unsigned long long flare_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *flare_last_error_string(void) { return t_error.c_str(); }

size_t flare_workspace_bytes(flare_op_t op, const flare_dims_t *dims, const int64_t *off, int R) {
    const size_t bad = (size_t)-1;
    if (op == FLARE_OP_LSE_MERGE || op == FLARE_OP_DECODE_FWD) return 0;
    if (op == FLARE_OP_DECODE_BWD) {
        if (check_dims(dims) != FLARE_OK) return bad;
        return decode_bwd_ws(dims);
    }
    if (check_dims(dims) != FLARE_OK) return bad;
    if (check_offsets(off, R, dims->N) != FLARE_OK) return bad;
    switch (op) {
        case FLARE_OP_ENCODER_FWD:
        case FLARE_OP_FWD:
        case FLARE_OP_PP_FWD:
            return encoder_ws_bytes(dims, off, R);
        case FLARE_OP_ENCODER_BWD:
            return encoder_bwd_ws(dims);
        case FLARE_OP_BWD:
        case FLARE_OP_PP_BWD: {
            MixerBwdLayout l;
            mixer_bwd_layout(dims, op == FLARE_OP_PP_BWD, l);
            return l.bytes;
        }
        default:
            return bad;
    }
}

flare_status_t flare_encoder_fwd(const flare_dims_t *dims, const void *Q, const void *K,
                                 const void *V, const uint8_t *mask,
                                 const int64_t *shard_offsets, int R, float *O_r, float *L_r,
                                 float *Z, float *L, void *workspace, size_t workspace_bytes,
                                 void *stream) {
    FLARE_TRACE();
    flare_status_t s = check_dims(dims);
    if (s != FLARE_OK) return s;
    if ((s = check_offsets(shard_offsets, R, dims->N)) != FLARE_OK) return s;
    return encoder_run(dims, Q, false, K, V, mask, shard_offsets, R, O_r, L_r, Z, L, workspace,
                       workspace_bytes, (cudaStream_t)stream);
}

flare_status_t flare_lse_merge(const float *O_r, const float *L_r, int R, int B, int H, int M,
                               int D, float *Z, float *L, void *stream) {
    FLARE_TRACE();
    if (R < 1 || B < 0 || H < 1 || M < 1 || D < 1)
        return fail(FLARE_ERR_INVALID_ARG, "bad sizes R=%d B=%d H=%d M=%d D=%d", R, B, H, M, D);
    if (B == 0) return FLARE_OK;
    if (!O_r || !L_r || !Z || !L) return fail(FLARE_ERR_INVALID_ARG, "NULL tensor");
    if (!aligned(O_r, 4) || !aligned(L_r, 4) || !aligned(Z, 4) || !aligned(L, 4))
        return fail(FLARE_ERR_INVALID_ARG, "fp32 tensors must be 4-byte aligned");
    cudaError_t e = launch_lse_merge(O_r, L_r, R, B, H, M, D, Z, L, (cudaStream_t)stream);
    return e == cudaSuccess ? FLARE_OK : cuda_fail(e, "merge launch");
}

flare_status_t flare_decode_fwd(const flare_dims_t *dims, const void *Q, const float *Z,
                                const void *K, void *Y, void *stream) {
    FLARE_TRACE();
    flare_status_t s = check_dims(dims);
    if (s != FLARE_OK) return s;
    return decode_run(dims, Q, false, Z, K, Y, false, (cudaStream_t)stream);
}

flare_status_t flare_fwd(const flare_dims_t *dims, const void *Q, const void *K, const void *V,
                         const uint8_t *mask, const int64_t *shard_offsets, int R, void *Y,
                         float *Z, float *L, void *workspace, size_t workspace_bytes,
                         void *stream) {
    FLARE_TRACE();
    flare_status_t s = check_dims(dims);
    if (s != FLARE_OK) return s;
    if ((s = check_offsets(shard_offsets, R, dims->N)) != FLARE_OK) return s;
    if (!Z || !L) return fail(FLARE_ERR_INVALID_ARG, "flare_fwd needs Z and L");
    cudaStream_t st = (cudaStream_t)stream;
    // both stages' arguments are checked before the first launch
    for (const bool check : {true, false}) {
        if ((s = encoder_run(dims, Q, false, K, V, mask, shard_offsets, R, nullptr, nullptr, Z, L,
                             workspace, workspace_bytes, st, check)) != FLARE_OK)
            return s;
        if ((s = decode_run(dims, Q, false, Z, K, Y, true, st, check)) != FLARE_OK) return s;
    }
    return FLARE_OK;
}

flare_status_t flare_pp_fwd(const flare_dims_t *dims, const void *Qseed, const void *Kt,
                            const void *Vt, const void *K, const void *V, const uint8_t *mask,
                            const int64_t *shard_offsets, int R, void *Y, float *Qdyn,
                            float *L1, float *Z, float *L2, void *workspace,
                            size_t workspace_bytes, void *stream) {
    FLARE_TRACE();
    flare_status_t s = check_dims(dims);
    if (s != FLARE_OK) return s;
    if ((s = check_offsets(shard_offsets, R, dims->N)) != FLARE_OK) return s;
    if (!Qdyn || !L1 || !Z || !L2) return fail(FLARE_ERR_INVALID_ARG, "flare_pp_fwd outputs are required");
    cudaStream_t st = (cudaStream_t)stream;
    flare_dims_t d2 = *dims;                                   // Q(X) is per batch element
    d2.q_batch_stride = (int64_t)dims->H * dims->M * dims->D;
    // the three stages' arguments are checked before the first launch
    for (const bool check : {true, false}) {
        if ((s = encoder_run(dims, Qseed, false, Kt, Vt, mask, shard_offsets, R, nullptr, nullptr, Qdyn,
                             L1, workspace, workspace_bytes, st, check)) != FLARE_OK)
            return s;
        if ((s = encoder_run(&d2, Qdyn, true, K, V, mask, shard_offsets, R, nullptr, nullptr, Z, L2,
                             workspace, workspace_bytes, st, check)) != FLARE_OK)
            return s;
        if ((s = decode_run(&d2, Qdyn, true, Z, K, Y, true, st, check)) != FLARE_OK) return s;
    }
    return FLARE_OK;
}

flare_status_t flare_encoder_bwd(const flare_dims_t *dims, const void *Q, const void *K,
                                 const void *V, const uint8_t *mask,
                                 const int64_t *shard_offsets, int R, const float *Z,
                                 const float *L, const float *dZ, float *dQ, void *dK, void *dV,
                                 void *workspace, size_t workspace_bytes, void *stream) {
    FLARE_TRACE();
    flare_status_t s = check_dims(dims);
    if (s != FLARE_OK) return s;
    if ((s = check_offsets(shard_offsets, R, dims->N)) != FLARE_OK) return s;
    return encoder_bwd_run(dims, Q, K, V, mask, Z, L, dZ, dQ, dK, dV, workspace, workspace_bytes,
                           false, (cudaStream_t)stream);
}

flare_status_t flare_encoder_bwd_accumulate(const flare_dims_t *dims, const void *Q, const void *K,
                                            const void *V, const uint8_t *mask,
                                            const int64_t *shard_offsets, int R, const float *Z,
                                            const float *L, const float *dZ, float *dQ, void *dK,
                                            void *dV, void *workspace, size_t workspace_bytes,
                                            void *stream) {
    FLARE_TRACE();
    flare_status_t s = check_dims(dims);
    if (s != FLARE_OK) return s;
    if ((s = check_offsets(shard_offsets, R, dims->N)) != FLARE_OK) return s;
    return encoder_bwd_run(dims, Q, K, V, mask, Z, L, dZ, dQ, dK, dV, workspace, workspace_bytes,
                           true, (cudaStream_t)stream);
}

flare_status_t flare_decode_bwd(const flare_dims_t *dims, const void *Q, const float *Z,
                                const void *K, const void *dY, float *dQ, float *dZ, void *dK,
                                void *workspace, size_t workspace_bytes, void *stream) {
    FLARE_TRACE();
    flare_status_t s = check_dims(dims);
    if (s != FLARE_OK) return s;
    return decode_bwd_run(dims, Q, Z, K, dY, dQ, dZ, dK, workspace, workspace_bytes,
                          (cudaStream_t)stream);
}

flare_status_t flare_bwd(const flare_dims_t *dims, const void *Q, const void *K, const void *V,
                         const uint8_t *mask, const int64_t *shard_offsets, int R, const float *Z,
                         const float *L, const void *dY, float *dQ, void *dK, void *dV,
                         void *workspace, size_t workspace_bytes, void *stream) {
    FLARE_TRACE();
    flare_status_t s = check_dims(dims);
    if (s != FLARE_OK) return s;
    if ((s = check_offsets(shard_offsets, R, dims->N)) != FLARE_OK) return s;
    if (dims->B == 0) return FLARE_OK;
    MixerBwdLayout l;
    mixer_bwd_layout(dims, false, l);
    if (!workspace || workspace_bytes < l.bytes)
        return fail(FLARE_ERR_WORKSPACE, "workspace of %zu bytes required, %zu given", l.bytes,
                    workspace_bytes);
    if (!aligned(workspace, 256)) return fail(FLARE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    char *w = (char *)workspace;
    float *dZ = (float *)(w + l.dz);
    cudaStream_t st = (cudaStream_t)stream;
    // both stages' arguments are checked before the first launch
    for (const bool check : {true, false}) {
        // the decoder's shares of dQ and dK, and dZ (Z's only consumer in the mixer)
        if ((s = decode_bwd_run(dims, Q, Z, K, dY, dQ, dZ, dK, w + l.scratch,
                                workspace_bytes - l.scratch, st, check)) != FLARE_OK)
            return s;
        // the encoder with its global (Z, L) adds its shares and gives dV
        if ((s = encoder_bwd_run(dims, Q, K, V, mask, Z, L, dZ, dQ, dK, dV, w + l.scratch,
                                 workspace_bytes - l.scratch, true, st, check)) != FLARE_OK)
            return s;
    }
    return FLARE_OK;
}

flare_status_t flare_pp_bwd(const flare_dims_t *dims, const void *Qseed, const void *Kt,
                            const void *Vt, const void *K, const void *V, const uint8_t *mask,
                            const int64_t *shard_offsets, int R, const float *Qdyn,
                            const float *L1, const float *Z, const float *L2, const void *dY,
                            float *dQseed, void *dKt, void *dVt, void *dK, void *dV, float *dQdyn,
                            void *workspace, size_t workspace_bytes, void *stream) {
    FLARE_TRACE();
    flare_status_t s = check_dims(dims);
    if (s != FLARE_OK) return s;
    if ((s = check_offsets(shard_offsets, R, dims->N)) != FLARE_OK) return s;
    if (dims->B == 0) return FLARE_OK;
    if (!Qdyn || !L1 || !Z || !L2) return fail(FLARE_ERR_INVALID_ARG, "the forward's Qdyn, L1, Z, L2 are required");
    if (!aligned(Qdyn, 16) || !aligned(dQdyn, 16))
        return fail(FLARE_ERR_INVALID_ARG, "Qdyn and dQdyn must be 16-byte aligned");
    MixerBwdLayout l;
    mixer_bwd_layout(dims, true, l);
    if (!workspace || workspace_bytes < l.bytes)
        return fail(FLARE_ERR_WORKSPACE, "workspace of %zu bytes required, %zu given", l.bytes,
                    workspace_bytes);
    if (!aligned(workspace, 256)) return fail(FLARE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    char *w = (char *)workspace;
    float *dZ = (float *)(w + l.dz);
    float *dQX = dQdyn ? dQdyn : (float *)(w + l.dqdyn);
    void *scratch = w + l.scratch;
    const size_t scratch_bytes = workspace_bytes - l.scratch;
    cudaStream_t st = (cudaStream_t)stream;
    flare_dims_t d2 = *dims;                                   // Q(X) is per batch element
    d2.q_batch_stride = (int64_t)dims->H * dims->M * dims->D;
    // Q(X) as the operand of the decode and physical-value encoder: bf16 on the bf16 path
    const bool convert = dims->dtype == FLARE_BF16;
    const void *QX = convert ? (const void *)(w + l.qdyn_b) : (const void *)Qdyn;
    // the three stages' arguments are checked before the first launch
    for (const bool check : {true, false}) {
        if (!check && convert) {
            const cudaError_t e = launch_f32_to_bf16(Qdyn, w + l.qdyn_b,
                                                     (int64_t)dims->B * dims->H * dims->M * dims->D, st);
            if (e != cudaSuccess) return cuda_fail(e, "Q(X) conversion launch");
        }
        // decoder: its shares of dQ(X) and dK, and dZ
        if ((s = decode_bwd_run(&d2, QX, Z, K, dY, dQX, dZ, dK, scratch, scratch_bytes, st, check)) !=
            FLARE_OK)
            return s;
        // physical-value encoder (Z, L2): adds its shares of dQ(X) and dK, gives dV
        if ((s = encoder_bwd_run(&d2, QX, K, V, mask, Z, L2, dZ, dQX, dK, dV, scratch, scratch_bytes,
                                 true, st, check)) != FLARE_OK)
            return s;
        // query-synthesis encoder (its output Q(X), L1) with the summed dQ(X)
        if ((s = encoder_bwd_run(dims, Qseed, Kt, Vt, mask, Qdyn, L1, dQX, dQseed, dKt, dVt, scratch,
                                 scratch_bytes, false, st, check)) != FLARE_OK)
            return s;
    }
    return FLARE_OK;
}

flare_status_t flare_check_bounded_wait(unsigned limit_us, void *stream) {
    FLARE_TRACE();
    if (limit_us < 1 || limit_us > 1000000)
        return fail(FLARE_ERR_INVALID_ARG, "limit_us=%u outside [1, 1000000]", limit_us);
    DeviceInfo di;
    flare_status_t s = device_info(di);
    if (s != FLARE_OK) return s;
    cudaError_t e = launch_bounded_wait_probe(1000ull * limit_us, di.status, (cudaStream_t)stream);
    return e == cudaSuccess ? FLARE_OK : cuda_fail(e, "bounded-wait probe launch");
}

flare_status_t flare_device_status(void *stream) {
    FLARE_TRACE();
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned v = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpyFromSymbol(status)");
    if (v != kDevOk) {
        const unsigned zero = 0;
        cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
        if (v & 0x100u)
            return fail(FLARE_ERR_DEVICE_CHECK, "a device-side check failed (check %u); the access was skipped",
                        v & 0xffu);
        return fail(FLARE_ERR_TIMEOUT, "a kernel abandoned a bounded wait (code %u)", v);
    }
    return FLARE_OK;
}

}  // extern "C"
