// C-ABI front end of the SSD forward scan: argument validation, workspace
// accounting, algorithm selection and launch.  The operation itself is
// specified in include/ssd.h.
#include <cuda_runtime.h>
#include <string.h>

#include "ssd_device.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

__global__ void validate_cu_kernel(const int32_t *cu, int nseq, int64_t seqlen, int *status) {
    bool bad = false;
    for (int s = threadIdx.x; s < nseq; s += blockDim.x)
        if (cu[s + 1] < cu[s]) bad = true;
    if (threadIdx.x == 0 && (cu[0] != 0 || (int64_t)cu[nseq] != seqlen)) bad = true;
    if (bad) set_status(status, SSD_ERR_DEVICE_INPUT);
}

// Host-side checks that need no device access.  Fills `p` on success.
int resolve(const ssd_shape *s, Problem &p, int *algo_out) {
    if (!s) return SSD_ERR_INVALID_ARG;
    if (s->batch < 0 || s->seqlen < 0 || s->nheads < 1 || s->headdim < 1 || s->dstate < 1 ||
        s->ngroups < 1 || s->nheads % s->ngroups != 0 || s->nseq < 0)
        return SSD_ERR_INVALID_ARG;
    if (s->seqlen > (int64_t)INT32_MAX || shape_too_large(s)) return SSD_ERR_UNSUPPORTED;
    if (s->dtype != SSD_F32 && s->dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
    if (s->chunk_size != 64 && s->chunk_size != 128 && s->chunk_size != 256)
        return SSD_ERR_UNSUPPORTED;
    p.batch = s->batch; p.seqlen = s->seqlen;
    p.H = s->nheads; p.P = s->headdim; p.N = s->dstate; p.G = s->ngroups;
    p.Q = s->chunk_size; p.nseq = s->nseq; p.dtype = s->dtype;
    p.nc = (int)((s->seqlen + s->chunk_size - 1) / s->chunk_size);
    // SSD_ALGO_TC resolves to the fused kernel when it takes the shape and to
    // the two-pass kernels otherwise; AUTO prefers tensor cores over SIMT.
    int algo = s->algo;
    if (algo == SSD_ALGO_AUTO || algo == SSD_ALGO_TC) {
        if (fused_supported(p) == SSD_OK) algo = SSD_ALGO_TC;
        else if (tc_supported(p) == SSD_OK) algo = SSD_ALGO_TC_TWOPASS;
        else if (algo == SSD_ALGO_AUTO) algo = SSD_ALGO_SIMT;
        else return SSD_ERR_UNSUPPORTED;
    }
    int rc;
    if (algo == SSD_ALGO_SIMT) rc = simt_supported(p);
    else if (algo == SSD_ALGO_TC) rc = fused_supported(p);
    else if (algo == SSD_ALGO_TC_TWOPASS) rc = tc_supported(p);
    else return SSD_ERR_INVALID_ARG;
    if (rc != SSD_OK) return rc;
    *algo_out = algo;
    return SSD_OK;
}

size_t workspace_for(const Problem &p, int algo) {
    const size_t body = (algo == SSD_ALGO_TC)          ? fused_workspace_bytes(p)
                        : (algo == SSD_ALGO_TC_TWOPASS) ? tc_workspace_bytes(p)
                                                        : simt_workspace_bytes(p);
    return kStatusBytes + body;
}

// The two-pass kernels take no packed sequences.  A shape with one batch row
// may come with cu_seqlens, and AUTO then falls back to SIMT, so the
// workspace asked for covers both.  With a step-size transform, every path
// but the fused kernel reads the transformed dt from the end of the
// workspace.
size_t dt_prepass_bytes(const Problem &p) {
    return align_up((size_t)(p.batch * p.seqlen * p.H) * sizeof(float), 256);
}

size_t workspace_need(const ssd_shape *s, const Problem &p, int algo, bool dt_tf) {
    size_t need = workspace_for(p, algo);
    bool fallback = false;
    if (algo == SSD_ALGO_TC_TWOPASS && s->algo == SSD_ALGO_AUTO && p.batch == 1) {
        const size_t simt = workspace_for(p, SSD_ALGO_SIMT);
        if (simt > need) need = simt;
        fallback = true;
    }
    if (dt_tf && (algo != SSD_ALGO_TC || fallback)) need = align_up(need, 256) + dt_prepass_bytes(p);
    return need;
}

// Host check of a step-size transform; fills `t` (off for NULL).
int resolve_dtt(const ssd_dt_transform *d, DtTransform &t) {
    t = DtTransform();
    if (!d) return SSD_OK;
    if (!(d->dt_min <= d->dt_max)) return SSD_ERR_INVALID_ARG;   // also rejects NaN
    if (d->bias && ((uintptr_t)d->bias % 4) != 0) return SSD_ERR_UNSUPPORTED;
    t.bias = d->bias;
    t.softplus = d->softplus != 0;
    t.lo = d->dt_min;
    t.hi = d->dt_max;
    t.on = true;
    return SSD_OK;
}

bool aligned(const void *ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

}  // namespace

cudaError_t launch_validate_cu(const Problem &p) {
    validate_cu_kernel<<<1, 256, 0, p.stream>>>(p.cu, p.nseq, p.seqlen, p.status);
    return cudaGetLastError();
}

}  // namespace ssd

using namespace ssd;

extern "C" {

SSD_API const char *ssd_status_string(int status) {
    switch (status) {
        case SSD_OK: return "SSD_OK";
        case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG: null pointer or inconsistent shape";
        case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED: dtype/chunk/headdim/dstate/alignment not supported";
        case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE: workspace missing or too small";
        case SSD_ERR_CUDA: return "SSD_ERR_CUDA: CUDA runtime call or kernel launch failed";
        case SSD_ERR_DEVICE_TIMEOUT: return "SSD_ERR_DEVICE_TIMEOUT: a bounded device-side wait gave up";
        case SSD_ERR_DEVICE_INPUT: return "SSD_ERR_DEVICE_INPUT: malformed cu_seqlens";
        default: return "SSD_ERR_UNKNOWN";
    }
}

SSD_API int ssd_resolve_algo(const ssd_shape *shape) {
    Problem p;
    int algo = 0;
    const int rc = resolve(shape, p, &algo);
    return rc == SSD_OK ? algo : -rc;
}

SSD_API int ssd_scan_ex_workspace_size(const ssd_shape *shape,
                                       const ssd_dt_transform *dt_transform, size_t *bytes) {
    if (!bytes) return SSD_ERR_INVALID_ARG;
    Problem p;
    int algo = 0;
    int rc = resolve(shape, p, &algo);
    if (rc != SSD_OK) return rc;
    DtTransform tf;
    rc = resolve_dtt(dt_transform, tf);
    if (rc != SSD_OK) return rc;
    *bytes = workspace_need(shape, p, algo, tf.on);
    return SSD_OK;
}

SSD_API int ssd_scan_workspace_size(const ssd_shape *shape, size_t *bytes) {
    return ssd_scan_ex_workspace_size(shape, nullptr, bytes);
}

SSD_API int ssd_scan(const ssd_shape *shape, const void *x, const float *dt, const float *A,
                     const void *B, const void *C, const float *D,
                     const float *initial_states, const int32_t *cu_seqlens, void *y,
                     float *final_states, void *workspace, size_t workspace_bytes,
                     void *stream) {
    return ssd_scan_ex(shape, x, dt, nullptr, A, B, C, D, initial_states, cu_seqlens, y,
                       final_states, workspace, workspace_bytes, stream);
}

SSD_API int ssd_scan_ex(const ssd_shape *shape, const void *x, const float *dt,
                        const ssd_dt_transform *dt_transform, const float *A, const void *B,
                        const void *C, const float *D, const float *initial_states,
                        const int32_t *cu_seqlens, void *y, float *final_states, void *workspace,
                        size_t workspace_bytes, void *stream) {
    Problem p;
    int algo = 0;
    int rc = resolve(shape, p, &algo);
    if (rc != SSD_OK) return rc;
    rc = resolve_dtt(dt_transform, p.dtt);
    if (rc != SSD_OK) return rc;
    if (cu_seqlens) {
        if (p.batch != 1 || p.nseq < 1) return SSD_ERR_INVALID_ARG;
    } else if (p.nseq != p.batch) {
        return SSD_ERR_INVALID_ARG;
    }
    const size_t need = workspace_need(shape, p, algo, p.dtt.on);
    if (cu_seqlens && algo == SSD_ALGO_TC_TWOPASS) {
        if (shape->algo != SSD_ALGO_AUTO) return SSD_ERR_UNSUPPORTED;
        algo = SSD_ALGO_SIMT;
    }
    if (!workspace || workspace_bytes < need) return SSD_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return SSD_ERR_WORKSPACE;
    const int64_t tokens = p.batch * p.seqlen;
    if (tokens > 0 && (!x || !dt || !A || !B || !C || !y)) return SSD_ERR_INVALID_ARG;
    const size_t esz = p.dtype == SSD_F32 ? 4 : 2;
    if (!aligned(x, esz) || !aligned(B, esz) || !aligned(C, esz) || !aligned(y, esz) ||
        !aligned(dt, 4) || !aligned(A, 4) || !aligned(D, 4) || !aligned(initial_states, 4) ||
        !aligned(final_states, 4) || !aligned(cu_seqlens, 4))
        return SSD_ERR_UNSUPPORTED;
    if (algo != SSD_ALGO_SIMT &&
        (!aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(y, 16) ||
         !aligned(initial_states, 16) || !aligned(final_states, 16)))
        return SSD_ERR_UNSUPPORTED;

    p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D;
    p.init = initial_states; p.cu = cu_seqlens; p.y = y; p.final_states = final_states;
    p.status = (int *)workspace;
    p.ws = (char *)workspace + kStatusBytes;
    p.ws_bytes = workspace_bytes - kStatusBytes;
    p.stream = (cudaStream_t)stream;

    if (cudaMemsetAsync(p.status, 0, sizeof(int), p.stream) != cudaSuccess) return SSD_ERR_CUDA;
    if (p.cu && launch_validate_cu(p) != cudaSuccess) return SSD_ERR_CUDA;

    // Degenerate sizes: no tokens.  Final states are then the initial states.
    if (tokens == 0 || p.batch == 0) {
        if (final_states && p.nseq > 0) {
            const size_t bytes = (size_t)p.nseq * p.H * p.P * p.N * sizeof(float);
            cudaError_t e = initial_states
                ? cudaMemcpyAsync(final_states, initial_states, bytes, cudaMemcpyDeviceToDevice, p.stream)
                : cudaMemsetAsync(final_states, 0, bytes, p.stream);
            if (e != cudaSuccess) return SSD_ERR_CUDA;
        }
        return SSD_OK;
    }
    if (p.dtt.on && algo != SSD_ALGO_TC) {
        // the other paths read dt in several kernels: transform it once into
        // the end of the workspace
        float *dt_eff = (float *)((char *)workspace + (need - dt_prepass_bytes(p)));
        if (launch_dt_transform(p, dt_eff) != cudaSuccess) return SSD_ERR_CUDA;
        p.dt = dt_eff;
        p.dtt = DtTransform();
    }
    const cudaError_t e = (algo == SSD_ALGO_TC)          ? fused_launch(p)
                          : (algo == SSD_ALGO_TC_TWOPASS) ? tc_launch(p)
                                                          : simt_launch(p);
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

SSD_API int ssd_step(const ssd_step_shape *shape, const void *x, const float *dt,
                     const ssd_dt_transform *dt_transform, const float *A, const void *B,
                     const void *C, const float *D, float *state, void *y, void *stream) {
    if (!shape) return SSD_ERR_INVALID_ARG;
    const ssd_step_shape &s = *shape;
    if (s.batch < 0 || s.nheads < 1 || s.headdim < 1 || s.dstate < 1 || s.ngroups < 1 ||
        s.nheads % s.ngroups != 0 || s.reserved != 0)
        return SSD_ERR_INVALID_ARG;
    if (s.dtype != SSD_F32 && s.dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
    if (s.headdim > 1024 || s.dstate > 1024) return SSD_ERR_UNSUPPORTED;
    if (s.batch * s.nheads > (int64_t)INT32_MAX) return SSD_ERR_UNSUPPORTED;
    StepProblem p;
    int rc = resolve_dtt(dt_transform, p.dtt);
    if (rc != SSD_OK) return rc;
    p.batch = s.batch; p.H = s.nheads; p.P = s.headdim; p.N = s.dstate; p.G = s.ngroups;
    p.dtype = s.dtype;
    if (p.batch == 0) return SSD_OK;
    if (!x || !dt || !A || !B || !C || !state || !y) return SSD_ERR_INVALID_ARG;
    const size_t esz = p.dtype == SSD_F32 ? 4 : 2;
    if (!aligned(x, esz) || !aligned(B, esz) || !aligned(C, esz) || !aligned(y, esz) ||
        !aligned(dt, 4) || !aligned(A, 4) || !aligned(D, 4) || !aligned(state, 4))
        return SSD_ERR_UNSUPPORTED;
    p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.state = state; p.y = y;
    p.stream = (cudaStream_t)stream;
    return step_launch(p) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

SSD_API int ssd_scan_states(const ssd_shape *shape, const void *x, const float *dt,
                            const ssd_dt_transform *dt_transform, const float *A, const void *B,
                            const float *initial_states, const int32_t *cu_seqlens,
                            float *final_states, void *workspace, size_t workspace_bytes,
                            void *stream) {
    Problem p;
    int algo = 0;
    int rc = resolve(shape, p, &algo);
    if (rc != SSD_OK) return rc;
    if (algo != SSD_ALGO_TC) return SSD_ERR_UNSUPPORTED;   // the fused kernel's shapes only
    rc = resolve_dtt(dt_transform, p.dtt);
    if (rc != SSD_OK) return rc;
    if (cu_seqlens) {
        if (p.batch != 1 || p.nseq < 1) return SSD_ERR_INVALID_ARG;
    } else if (p.nseq != p.batch) {
        return SSD_ERR_INVALID_ARG;
    }
    const size_t need = workspace_need(shape, p, algo, p.dtt.on);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return SSD_ERR_WORKSPACE;
    const int64_t tokens = p.batch * p.seqlen;
    if (!final_states || (tokens > 0 && (!x || !dt || !A || !B))) return SSD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(B, 16) || !aligned(dt, 4) || !aligned(A, 4) ||
        !aligned(initial_states, 16) || !aligned(final_states, 16) || !aligned(cu_seqlens, 4))
        return SSD_ERR_UNSUPPORTED;

    p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = nullptr; p.D = nullptr;
    p.init = initial_states; p.cu = cu_seqlens; p.y = nullptr; p.final_states = final_states;
    p.states_only = true;
    p.status = (int *)workspace;
    p.ws = (char *)workspace + kStatusBytes;
    p.ws_bytes = workspace_bytes - kStatusBytes;
    p.stream = (cudaStream_t)stream;

    if (cudaMemsetAsync(p.status, 0, sizeof(int), p.stream) != cudaSuccess) return SSD_ERR_CUDA;
    if (p.cu && launch_validate_cu(p) != cudaSuccess) return SSD_ERR_CUDA;
    if (tokens == 0 || p.batch == 0) {
        if (p.nseq > 0) {
            const size_t bytes = (size_t)p.nseq * p.H * p.P * p.N * sizeof(float);
            cudaError_t e = initial_states
                ? cudaMemcpyAsync(final_states, initial_states, bytes, cudaMemcpyDeviceToDevice, p.stream)
                : cudaMemsetAsync(final_states, 0, bytes, p.stream);
            if (e != cudaSuccess) return SSD_ERR_CUDA;
        }
        return SSD_OK;
    }
    return fused_launch(p) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

SSD_API int ssd_check_device_status(const void *workspace, void *stream) {
    if (!workspace) return SSD_ERR_INVALID_ARG;
    int status = 0;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SSD_ERR_CUDA;
    if (cudaMemcpy(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SSD_ERR_CUDA;
    return status;
}

}  // extern "C"
