// Sequence parallelism for the SSD forward scan: the carry exchange.
//
// QbitAI article "新架构Mamba更新二代！", section "Mamba-2：更强学习能力，更快训练推理":
// sequence parallelism lets the layer scale to longer sequences.  Cut every
// sequence into consecutive shards r = 0 .. R-1 (one per device).  The only
// quantity that crosses a shard boundary is the per-head state.  With S_r
// the state shard r reaches when scanned from a zero state, and
// logdec_r = sum over the shard's tokens of dt_t A_h (the log of its total
// decay), the state entering shard r is
//     H_in(0) = the sequence's initial state (or zero)
//     H_in(r + 1) = exp(logdec_r) H_in(r) + S_r
// and the sequence's final state is H_in(R): the same recurrence as the
// state passing between chunks, one step per shard.  Shard r's output is
// its scan started from H_in(r).  This file holds the two device steps of
// that exchange; the scans are ssd_scan().
#include <cuda_runtime.h>

#include <cooperative_groups.h>

#include "ssd_device.cuh"
#include "ssd_internal.h"

namespace cg = cooperative_groups;

namespace ssd {
namespace {

constexpr int kLogdecThreads = 256;
constexpr int kLogdecWarps = kLogdecThreads / 32;
constexpr int kLogdecCluster = 8;                    // CTAs per (sequence, head block)
constexpr int kLogdecStride = kLogdecWarps * kLogdecCluster;   // warps over one token range
constexpr int kLogdecRun = 16;                       // tokens summed in fp32 before fp64

// logdec[s][h] = A_h * sum_t dt'[s, t, h] over the L tokens of batch row s
// (sequence s's tokens on this shard; A_h is the same for every token, so
// it multiplies the sum once).  A cluster of kLogdecCluster CTAs takes one
// (sequence, 32-head block): warp w of CTA z takes tokens t = z * 8 + w,
// then every 64th token, lane = head, so that every load of a warp reads 32
// consecutive heads of one token.  Each thread sums runs of 16 tokens in
// fp32 and adds the runs in fp64; the CTA adds its warps in order, and CTA 0
// of the cluster adds the CTAs in order through distributed shared memory.
// The result does not depend on timing.
__global__ void __cluster_dims__(1, 1, kLogdecCluster) __launch_bounds__(kLogdecThreads)
    k_shard_logdec(const float *__restrict__ dt, const float *__restrict__ A, int64_t L, int H,
                   DtTransform tf, float *__restrict__ logdec) {
    __shared__ double part[kLogdecWarps][32];
    __shared__ double cta_sum[32];
    cg::cluster_group cluster = cg::this_cluster();
    const int s = blockIdx.x;
    const int z = (int)cluster.block_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * 32 + lane;
    double acc = 0.0;
    if (h < H) {
        const float bias = tf.bias ? __ldg(tf.bias + h) : 0.f;
        const float *row = dt + (int64_t)s * L * H + h;
        int64_t t = z * kLogdecWarps + warp;
        // full runs: all 16 loads in flight before the sum
        for (; t + (kLogdecRun - 1) * kLogdecStride < L; t += kLogdecRun * kLogdecStride) {
            float d[kLogdecRun];
#pragma unroll
            for (int k = 0; k < kLogdecRun; ++k) d[k] = __ldg(row + (t + k * kLogdecStride) * H);
            float run = 0.f;
#pragma unroll
            for (int k = 0; k < kLogdecRun; ++k) {
                if (tf.on) d[k] = dt_apply(d[k], bias, tf.softplus, tf.lo, tf.hi);
                run += d[k];
            }
            acc += (double)run;
        }
        float run = 0.f;   // the last, partial run
        for (; t < L; t += kLogdecStride) {
            float d = __ldg(row + t * H);
            if (tf.on) d = dt_apply(d, bias, tf.softplus, tf.lo, tf.hi);
            run += d;
        }
        acc += (double)run;
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        double sum = 0.0;
#pragma unroll
        for (int w = 0; w < kLogdecWarps; ++w) sum += part[w][lane];
        cta_sum[lane] = sum;
    }
    cluster.sync();   // every CTA's cta_sum is written
    if (z == 0 && warp == 0 && h < H) {
        double sum = 0.0;
#pragma unroll
        for (int q = 0; q < kLogdecCluster; ++q) sum += cluster.map_shared_rank(cta_sum, q)[lane];
        logdec[(int64_t)s * H + h] = (float)(sum * (double)__ldg(A + h));
    }
    cluster.sync();   // keep every CTA's shared memory alive until CTA 0 has read it
}

// The fold over shards, one state element per thread (four with float4 when
// the state rows and every pointer allow): e runs over (sequence, head, p,
// n), sh = e / PN is its (sequence, head).
//   H = init (or 0); for q = 0 .. nshards - 1:
//       (q == rank: h_in = H);  H = exp(logdec_q) H + S_q
//   total = H
// No load depends on the running H, so the S_q of the next shards are in
// flight while the multiply-adds run.
__global__ void k_carry_fold(const float *__restrict__ S_all, const float *__restrict__ logdec_all,
                             const float *__restrict__ init, int nshards, int rank, int64_t nsh,
                             int64_t PN, float *__restrict__ h_in, float *__restrict__ total) {
    const int64_t n = nsh * PN;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t sh = e / PN;
        float Hs = init ? __ldg(init + e) : 0.f;
#pragma unroll 4
        for (int q = 0; q < nshards; ++q) {
            if (q == rank && h_in) h_in[e] = Hs;
            const float dq = expf(__ldg(logdec_all + (int64_t)q * nsh + sh));
            Hs = fmaf(dq, Hs, __ldg(S_all + (int64_t)q * n + e));
        }
        if (total) total[e] = Hs;
    }
}

__global__ void k_carry_fold4(const float4 *__restrict__ S_all, const float *__restrict__ logdec_all,
                              const float4 *__restrict__ init, int nshards, int rank, int64_t nsh,
                              int64_t PN4, float4 *__restrict__ h_in, float4 *__restrict__ total) {
    const int64_t n4 = nsh * PN4;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n4;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t sh = e / PN4;
        float4 Hs = init ? __ldg(init + e) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int q = 0; q < nshards; ++q) {
            if (q == rank && h_in) h_in[e] = Hs;
            const float dq = expf(__ldg(logdec_all + (int64_t)q * nsh + sh));
            const float4 Sq = __ldg(S_all + (int64_t)q * n4 + e);
            Hs.x = fmaf(dq, Hs.x, Sq.x);
            Hs.y = fmaf(dq, Hs.y, Sq.y);
            Hs.z = fmaf(dq, Hs.z, Sq.z);
            Hs.w = fmaf(dq, Hs.w, Sq.w);
        }
        if (total) total[e] = Hs;
    }
}

bool aligned4(const void *p) { return ((uintptr_t)p % 4) == 0; }
bool aligned16(const void *p) { return ((uintptr_t)p % 16) == 0; }

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" SSD_API int ssd_seqpar_logdec(const ssd_shape *s, const float *dt,
                                         const ssd_dt_transform *dt_transform, const float *A,
                                         float *logdec, void *stream) {
    if (!s) return SSD_ERR_INVALID_ARG;
    if (s->batch < 0 || s->seqlen < 0 || s->nheads < 1 || s->nseq < 0) return SSD_ERR_INVALID_ARG;
    if (s->seqlen > (int64_t)INT32_MAX || shape_too_large(s)) return SSD_ERR_UNSUPPORTED;
    if (s->nseq != s->batch) return SSD_ERR_INVALID_ARG;
    if (s->nseq == 0) return SSD_OK;
    // dt is not read when the shard holds no tokens (an empty tensor may
    // have no storage)
    if ((s->seqlen > 0 && !dt) || !A || !logdec) return SSD_ERR_INVALID_ARG;
    if (!aligned4(dt) || !aligned4(A) || !aligned4(logdec)) return SSD_ERR_UNSUPPORTED;
    DtTransform tf;
    if (dt_transform) {
        if (!(dt_transform->dt_min <= dt_transform->dt_max)) return SSD_ERR_INVALID_ARG;
        if (!aligned4(dt_transform->bias)) return SSD_ERR_UNSUPPORTED;
        tf.bias = dt_transform->bias;
        tf.softplus = dt_transform->softplus != 0;
        tf.lo = dt_transform->dt_min;
        tf.hi = dt_transform->dt_max;
        tf.on = true;
    }
    if ((s->nheads + 31) / 32 > 65535) return SSD_ERR_UNSUPPORTED;   // grid.y limit
    const dim3 grid((unsigned)s->nseq, (unsigned)((s->nheads + 31) / 32), kLogdecCluster);
    k_shard_logdec<<<grid, kLogdecThreads, 0, (cudaStream_t)stream>>>(dt, A, s->seqlen,
                                                                      s->nheads, tf, logdec);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

extern "C" SSD_API int ssd_seqpar_fold(int32_t nshards, int32_t rank, int64_t nseq, int32_t nheads,
                                       int32_t headdim, int32_t dstate, const float *shard_states,
                                       const float *shard_logdec, const float *initial_states,
                                       float *shard_initial_states, float *final_states,
                                       void *stream) {
    if (nshards < 1 || rank < 0 || rank >= nshards || nseq < 0 || nheads < 1 || headdim < 1 ||
        dstate < 1)
        return SSD_ERR_INVALID_ARG;
    const __int128 elems = (__int128)nshards * nseq * nheads * headdim * dstate;
    if (elems > ((__int128)1 << 56)) return SSD_ERR_UNSUPPORTED;
    if (nseq == 0) return SSD_OK;
    if (!shard_states || !shard_logdec || (!shard_initial_states && !final_states))
        return SSD_ERR_INVALID_ARG;
    if (!aligned4(shard_states) || !aligned4(shard_logdec) || !aligned4(initial_states) ||
        !aligned4(shard_initial_states) || !aligned4(final_states))
        return SSD_ERR_UNSUPPORTED;
    const int64_t nsh = nseq * nheads, PN = (int64_t)headdim * dstate;
    const int threads = 256;
    const bool vec = PN % 4 == 0 && aligned16(shard_states) && aligned16(initial_states) &&
                     aligned16(shard_initial_states) && aligned16(final_states);
    const int64_t n = nsh * (vec ? PN / 4 : PN);
    const int64_t want = (n + threads - 1) / threads;
    const unsigned blocks = (unsigned)(want < 148 * 8 ? want : 148 * 8);
    if (vec)
        k_carry_fold4<<<blocks, threads, 0, (cudaStream_t)stream>>>(
            (const float4 *)shard_states, shard_logdec, (const float4 *)initial_states, nshards,
            rank, nsh, PN / 4, (float4 *)shard_initial_states, (float4 *)final_states);
    else
        k_carry_fold<<<blocks, threads, 0, (cudaStream_t)stream>>>(
            shard_states, shard_logdec, initial_states, nshards, rank, nsh, PN,
            shard_initial_states, final_states);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
