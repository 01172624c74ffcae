// Decode step of the SSD recurrence (one token per sequence, state updated in
// place) and the step-size pre-pass of the non-fused scan paths.
//
// The step is the recurrent form of the selective SSM -- the state cache that
// makes generation linear-time (Mamba-1 walkthrough "Mamba: Linear-Time
// Sequence Modeling with Selective State Spaces", sections 二(一) and
// 四(五)):
//     S <- exp(dt A_h) S + dt x (outer) B,   y = S C + D_h x.
// It is bound by HBM: each (sequence, head) reads and writes its P x N fp32
// state once, and everything else it touches is a few hundred bytes.
#include <cuda_runtime.h>

#include "ssd_device.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kStepThreads = 256;
constexpr int kStepWarps = kStepThreads / 32;
constexpr int kRowsPerWarp = 4;     // state rows a warp has in flight at once
constexpr int kMaxN = 1024;

struct StepArgs {
    int64_t batch;
    int H, P, N, G;
    const void *x, *B, *C;
    const float *dt, *A, *D;
    DtTransform dtt;
    float *state;
    void *y;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// One CTA per (sequence b, head h).  B and C of the token go to shared memory
// as fp32.  Warp w updates state rows p = 4w .. 4w + 3, then 4w + 32 ... (four
// rows' loads in flight; eight raise the registers to 128 and the lost
// occupancy costs more than the deeper queue gains); lane l holds columns
// n = 4 (l + 32 i) .. + 3 when N % 4 == 0 (16-byte accesses, coalesced along
// the row), else n = l + 32 i.
// The row's y is the warp's sum of S[p, n] C[n], plus D_h x[p].
template <typename T, bool VEC>
__global__ void __launch_bounds__(kStepThreads) k_ssd_step(StepArgs a) {
    __shared__ __align__(16) float sB[kMaxN];
    __shared__ __align__(16) float sC[kMaxN];
    const int64_t bh = blockIdx.x;
    const int h = (int)(bh % a.H);
    const int64_t b = bh / a.H;
    const int g = h / (a.H / a.G);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    float dt = __ldg(a.dt + bh);
    if (a.dtt.on)
        dt = dt_apply(dt, a.dtt.bias ? __ldg(a.dtt.bias + h) : 0.f, a.dtt.softplus, a.dtt.lo, a.dtt.hi);
    const float decay = expf(dt * __ldg(a.A + h));
    const float Dh = a.D ? __ldg(a.D + h) : 0.f;
    const T *xb = (const T *)a.x + bh * a.P;
    const T *Bb = (const T *)a.B + (b * a.G + g) * a.N;
    const T *Cb = (const T *)a.C + (b * a.G + g) * a.N;
    for (int n = tid; n < a.N; n += kStepThreads) {
        sB[n] = ld_as_float(Bb + n);
        sC[n] = ld_as_float(Cb + n);
    }
    __syncthreads();

    float *S = a.state + bh * (int64_t)a.P * a.N;
    T *yb = (T *)a.y + bh * a.P;
    for (int p0 = warp * kRowsPerWarp; p0 < a.P; p0 += kStepWarps * kRowsPerWarp) {
        float u[kRowsPerWarp], acc[kRowsPerWarp], xp[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            xp[r] = (p0 + r < a.P) ? ld_as_float(xb + p0 + r) : 0.f;
            u[r] = dt * xp[r];
            acc[r] = 0.f;
        }
        if (VEC) {
            const int n4 = a.N >> 2;
            for (int c = lane; c < n4; c += 32) {
                float4 s[kRowsPerWarp];
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r)
                    if (p0 + r < a.P) s[r] = *((const float4 *)(S + (int64_t)(p0 + r) * a.N) + c);
                const float4 bv = ((const float4 *)sB)[c], cv = ((const float4 *)sC)[c];
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r) {
                    if (p0 + r >= a.P) continue;
                    s[r].x = fmaf(decay, s[r].x, u[r] * bv.x);
                    s[r].y = fmaf(decay, s[r].y, u[r] * bv.y);
                    s[r].z = fmaf(decay, s[r].z, u[r] * bv.z);
                    s[r].w = fmaf(decay, s[r].w, u[r] * bv.w);
                    acc[r] += s[r].x * cv.x + s[r].y * cv.y + s[r].z * cv.z + s[r].w * cv.w;
                    *((float4 *)(S + (int64_t)(p0 + r) * a.N) + c) = s[r];
                }
            }
        } else {
            for (int n = lane; n < a.N; n += 32) {
                float s[kRowsPerWarp];
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r)
                    if (p0 + r < a.P) s[r] = S[(int64_t)(p0 + r) * a.N + n];
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r) {
                    if (p0 + r >= a.P) continue;
                    s[r] = fmaf(decay, s[r], u[r] * sB[n]);
                    acc[r] += s[r] * sC[n];
                    S[(int64_t)(p0 + r) * a.N + n] = s[r];
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const float v = warp_sum(acc[r]);
            if (lane == 0 && p0 + r < a.P) st_from_float(yb + p0 + r, v + Dh * xp[r]);
        }
    }
}

// dt' of every token (the transform of ssd_dt_transform), for the scan paths
// that read dt in several kernels.
__global__ void k_dt_transform(const float *dt, int64_t n, int H, DtTransform tf, float *out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int h = (int)(i % H);
        out[i] = dt_apply(__ldg(dt + i), tf.bias ? __ldg(tf.bias + h) : 0.f, tf.softplus, tf.lo, tf.hi);
    }
}

template <typename T>
cudaError_t launch_step_t(const StepArgs &a, int64_t nblocks, cudaStream_t st) {
    if (a.N % 4 == 0 && (uintptr_t)a.state % 16 == 0)
        k_ssd_step<T, true><<<(unsigned)nblocks, kStepThreads, 0, st>>>(a);
    else
        k_ssd_step<T, false><<<(unsigned)nblocks, kStepThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t step_launch(const StepProblem &p) {
    const int64_t nblocks = p.batch * p.H;
    if (nblocks == 0) return cudaSuccess;
    StepArgs a;
    a.batch = p.batch; a.H = p.H; a.P = p.P; a.N = p.N; a.G = p.G;
    a.x = p.x; a.B = p.B; a.C = p.C; a.dt = p.dt; a.A = p.A; a.D = p.D;
    a.dtt = p.dtt; a.state = p.state; a.y = p.y;
    return p.dtype == SSD_F32 ? launch_step_t<float>(a, nblocks, p.stream)
                              : launch_step_t<__nv_bfloat16>(a, nblocks, p.stream);
}

cudaError_t launch_dt_transform(const Problem &p, float *out) {
    const int64_t n = p.batch * p.seqlen * p.H;
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t want = (n + threads - 1) / threads;
    const unsigned blocks = (unsigned)(want < 148 * 16 ? want : 148 * 16);
    k_dt_transform<<<blocks, threads, 0, p.stream>>>(p.dt, n, p.H, p.dtt, out);
    return cudaGetLastError();
}

}  // namespace ssd
