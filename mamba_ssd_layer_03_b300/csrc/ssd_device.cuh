// Device helpers shared by the kernels of the SSD forward scan.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace ssd {

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ float ld_as_float(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld_as_float(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
__device__ __forceinline__ void st_from_float(float *p, float v) { *p = v; }
__device__ __forceinline__ void st_from_float(__nv_bfloat16 *p, float v) {
    *p = __float2bfloat16_rn(v);
}

// Index of the packed sequence that contains token t of the (single) row:
// the largest s in [0, nseq) with cu[s] <= t.  Always returns a value in
// [0, nseq) whatever cu holds, so a malformed cu_seqlens cannot send any
// index out of bounds (it is reported separately through the status word).
__device__ __forceinline__ int seg_of(const int32_t *cu, int nseq, int64_t t) {
    int lo = 0, hi = nseq - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if ((int64_t)__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Records the first error code in the status word (later codes are dropped).
__device__ __forceinline__ void set_status(int *status, int code) {
    atomicCAS(status, 0, code);
}

__device__ __forceinline__ bool status_bad(const int *status) {
    return *(volatile const int *)status != 0;
}

// The step-size transform of ssd_dt_transform (include/ssd.h): bias, then
// softplus log(1 + e^z) (z itself above 20, where the two agree to fp32
// precision), then the clamp.
struct DtTransform {
    const float *bias = nullptr;
    int softplus = 0;
    float lo = 0.f, hi = 0.f;
    bool on = false;
};

__device__ __forceinline__ float dt_apply(float raw, float bias, int softplus, float lo, float hi) {
    float z = raw + bias;
    if (softplus) z = z > 20.f ? z : log1pf(expf(z));
    return fminf(fmaxf(z, lo), hi);
}

}  // namespace ssd
