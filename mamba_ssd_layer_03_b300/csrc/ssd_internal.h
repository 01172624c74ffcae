// Internal declarations shared by the C-ABI front end and the kernels of
// the SSD forward scan.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/ssd.h"
#include "ssd_device.cuh"

namespace ssd {

// One call's arguments, resolved and validated on the host.
struct Problem {
    int64_t batch = 0, seqlen = 0;
    int H = 0, P = 0, N = 0, G = 0, Q = 0, nseq = 0;
    int nc = 0;          // chunks per batch row, ceil(seqlen / Q)
    int dtype = 0;       // ssd_dtype
    const void *x = nullptr;
    const float *dt = nullptr, *A = nullptr;
    const void *B = nullptr, *C = nullptr;
    const float *D = nullptr, *init = nullptr;
    DtTransform dtt;      // applied by the fused kernel as it reads dt
    const int32_t *cu = nullptr;
    void *y = nullptr;
    float *final_states = nullptr;
    int *status = nullptr;  // device status word (first bytes of workspace)
    char *ws = nullptr;     // workspace after the status block
    size_t ws_bytes = 0;
    cudaStream_t stream = nullptr;
    bool states_only = false;  // fused path only: final states, no y (ssd_scan_states)
};

// Bytes reserved at the start of every workspace for the status word.
constexpr size_t kStatusBytes = 256;

// ---- SIMT path (ssd_simt.cu) ----
size_t simt_workspace_bytes(const Problem &p);
int simt_supported(const Problem &p);          // SSD_OK or SSD_ERR_UNSUPPORTED
cudaError_t simt_launch(const Problem &p);

// ---- tensor-core path (ssd_tc.cu) ----
size_t tc_workspace_bytes(const Problem &p);
int tc_supported(const Problem &p);
cudaError_t tc_launch(const Problem &p);

// ---- fused single-pass tensor-core path (ssd_fused.cu) ----
size_t fused_workspace_bytes(const Problem &p);
int fused_supported(const Problem &p);
cudaError_t fused_launch(const Problem &p);

// ---- decode step (ssd_step.cu) ----
struct StepProblem {
    int64_t batch = 0;
    int H = 0, P = 0, N = 0, G = 0, dtype = 0;
    const void *x = nullptr, *B = nullptr, *C = nullptr;
    const float *dt = nullptr, *A = nullptr, *D = nullptr;
    DtTransform dtt;
    float *state = nullptr;
    void *y = nullptr;
    cudaStream_t stream = nullptr;
};
cudaError_t step_launch(const StepProblem &p);

// ---- step-size pre-pass (ssd_step.cu): dt' of every token into `out` ----
cudaError_t launch_dt_transform(const Problem &p, float *out);

// ---- shared helpers (ssd_api.cu) ----
// Device check of cu_seqlens: cu[0]==0, cu[nseq]==seqlen, non-decreasing.
// Sets *status = SSD_ERR_DEVICE_INPUT when malformed.
cudaError_t launch_validate_cu(const Problem &p);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Element counts of x/y, B/C and the states of a scan shape, in 128-bit
// arithmetic: a shape whose buffers could not exist (over 2^56 elements) is
// rejected before any size computed from it can wrap around.
inline bool shape_too_large(const ssd_shape *s) {
    const __int128 tokens = (__int128)s->batch * s->seqlen;
    const __int128 lim = (__int128)1 << 56;
    return tokens * s->nheads * s->headdim > lim || tokens * s->ngroups * s->dstate > lim ||
           (__int128)s->nseq * s->nheads * s->headdim * s->dstate > lim;
}

}  // namespace ssd
