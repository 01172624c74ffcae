// Tensor-core (tcgen05 / TMEM / TMA) path of the SSD forward scan, bf16
// inputs with fp32 accumulation and fp32 decays/states.
//
// The scan is the block decomposition of the semiseparable matrix
// M = L o (C B^T) (QbitAI article "新架构Mamba更新二代！", sections
// "统一SSM和注意力机制" and "Mamba-2：更强学习能力，更快训练推理"): masked quadratic
// products inside a chunk plus a linear recurrence over per-chunk states.
// Two kernels:
//
// k_chunk_state (one CTA works on (row, chunk, head pair) tiles taken in
//   chunk-major order from an atomic counter):
//     cs_j  = sum of dt*A over the chunk up to j (warp scan, fp32)
//     Xw^T  = (exp(cs_last - cs_j) dt_j x_j)^T   -> TMEM, bf16, heads stacked
//                                                 on the 128 TMEM lanes
//     S^T   = Xw^T . B_chunk                     -> tcgen05.mma, TMEM fp32
//     chain: E_{c+1} = exp(cs_last) E_c + S_c, with E_c taken from the
//            previous chunk's tile through an L2-resident two-slot ring and
//            a release/acquire flag per (row, head pair); writes E_c in bf16
//            for the output kernel and the final state after the last chunk.
//
// k_chunk_output (one CTA per (row, chunk, head) tile).  The chunk of Q
//   tokens is split into 128-token blocks I; inside block I the masked
//   product runs on the tensor cores, and the earlier part of the chunk
//   reaches block 1 through the exact low-rank factorisation of the
//   off-diagonal block (the state after block 0):
//     CB_II = C_I B_I^T                          -> TMEM fp32 (128x128)
//     M_II  = CB_II o exp(cs_i - cs_j) dt_j [j<=i] -> bf16, in place in TMEM
//     acc_I = C_I H_I^T  (H_0 = E_c, H_1 = exp(cs_127) E_c + S_0)
//     acc_I = acc_I * exp(cs_i - r_I)  (r_0 = 0, r_1 = cs_127)
//     acc_I += M_II X_I                          (A operand read from TMEM)
//     y_I   = acc_I + D x_I                      -> TMA store
//   with S_0 = sum_{j<128} exp(cs_127 - cs_j) dt_j B_j x_j^T on the tensor
//   cores as well.  Every exponent is <= 0.
//
// Packed variable-length input and chunk sizes other than 128/256 take the
// SIMT path (tc_supported() rejects them).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include "ssd_device.cuh"
#include "ssd_internal.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;
typedef __nv_bfloat16 bf16;

constexpr int kThreads = 128;
constexpr int kBlk = 128;          // token block of the quadratic products
constexpr uint32_t kTile16 = 16384;  // one 128-row x 128-byte swizzled tile

struct TcArgs {
    int64_t L;
    int batch, H, P, N, G, Q, nc, hpg;
    int kh;            // heads per state tile (1 or 2)
    int npairs;        // state tiles per (row, chunk): ceil(H / kh)
    int state_tiles, out_tiles;
    const bf16 *x;
    const float *dt, *A, *D, *init;
    float *final_states;
    int *status;
    int *counter;      // tile counter of the state kernel
    int *flags;        // [batch][npairs] last chunk whose entry state is published
    float *ring;       // [batch][npairs][2][kh][P][N]
    bf16 *ebuf;        // [batch][nc][H][P][N] entry state of every chunk (bf16)
};

// ----------------------------------------------------------------------------
// small device helpers

__device__ __forceinline__ bool bail(const int *status) { return status_bad(status); }

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(int *p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded mbarrier wait that records a time-out in the status word.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, int *status) {
    if (mbar_wait(bar, parity)) return true;
    set_status(status, SSD_ERR_DEVICE_TIMEOUT);
    return false;
}

// Inclusive cumulative sum of a_j = dt_j * A over the chunk for one head,
// computed by one warp (lane l owns tokens [l*Q/32, (l+1)*Q/32)).  Tokens at
// or beyond `len` get dt = 0.  Writes cs[] and dtv[] in shared memory.
__device__ __forceinline__ void chunk_cumsum_warp(const float *dt_base, int64_t dt_stride,
                                                  float Ah, int Q, int len, float *cs,
                                                  float *dtv) {
    const int lane = threadIdx.x & 31;
    const int per = Q / 32;
    float local[8];
    float run = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        if (q < per) {
            const int j = lane * per + q;
            const float d = (j < len) ? __ldg(dt_base + (int64_t)j * dt_stride) : 0.f;
            dtv[j] = d;
            run += d * Ah;
            local[q] = run;
        }
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    const float excl = incl - run;
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (q < per) cs[lane * per + q] = local[q] + excl;
}

// ----------------------------------------------------------------------------
// k_chunk_state

struct StateSmem {
    float cs[2][256];
    float w[2][256];
    float dtv[2][256];
    uint64_t bar_load, bar_mma;
    uint32_t tmem;
    int tile;
};

__global__ void __launch_bounds__(kThreads, 1)
k_chunk_state(const __grid_constant__ CUtensorMap tmB, TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sB = base;                                   // Q x N bf16 (MN-major view)
    StateSmem *sm = (StateSmem *)(base + (size_t)a.Q * a.N * 2);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int nblk_n = a.N / 64, nblk_j = a.Q / kBlk;
    const uint32_t tmem_cols = (a.N <= 128) ? 256 : 512;

    if (tid == 0) {
        mbar_init(&sm->bar_load, 1);
        mbar_init(&sm->bar_mma, 1);
        fence_mbar_init();
        prefetch_tmap(&tmB);
    }
    if (warp == 0) { tmem_alloc(&sm->tmem, tmem_cols); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm->tmem;
    const uint32_t t_xw = tbase;            // Q/2 columns: Xw^T (bf16 pairs)
    const uint32_t t_s = tbase + 128;       // N columns: S^T (fp32)
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t ph_load = 0, ph_mma = 0;
    const int PN = a.P * a.N;

    while (true) {
        if (tid == 0) sm->tile = bail(a.status) ? a.state_tiles : atomicAdd(a.counter, 1);
        __syncthreads();
        const int tile = sm->tile;   // same value in every thread
        if (tile >= a.state_tiles) break;
        const int per_c = a.batch * a.npairs;
        const int c = tile / per_c;
        const int r = (tile % per_c) / a.npairs;
        const int pair = tile % a.npairs;
        const int h0 = pair * a.kh;
        const int g = h0 / a.hpg;
        const int64_t t0 = (int64_t)c * a.Q;
        const int len = (int)min64(a.Q, a.L - t0);

        if (tid == 0) {
            for (int jb = 0; jb < nblk_j; ++jb)
                for (int nb = 0; nb < nblk_n; ++nb)
                    tma_load_4d(sB + (size_t)(nb * nblk_j + jb) * kTile16, &tmB, &sm->bar_load,
                                nb * 64, g, (int)(t0 + jb * kBlk), r);
            mbar_arrive_expect_tx(&sm->bar_load, (uint32_t)(a.Q * a.N * 2));
        }
        // decay cumsum and weights per head (warp hh handles head h0 + hh)
        if (warp < a.kh && h0 + warp < a.H) {
            const int h = h0 + warp;
            chunk_cumsum_warp(a.dt + ((int64_t)r * a.L + t0) * a.H + h, a.H, __ldg(a.A + h), a.Q,
                              len, sm->cs[warp], sm->dtv[warp]);
            __syncwarp();
            const float cl = sm->cs[warp][len - 1];
            for (int j = (tid & 31); j < a.Q; j += 32)
                sm->w[warp][j] = (j < len) ? __expf(cl - sm->cs[warp][j]) * sm->dtv[warp][j] : 0.f;
        }
        __syncthreads();
        // Xw^T into TMEM: lane = (head slot, p), columns = token pairs
        {
            const int hh = tid / 64, p = tid % 64;
            const bool ok = (hh < a.kh) && (h0 + hh < a.H) && (p < a.P);
            const bf16 *xp = a.x + (((int64_t)r * a.L + t0) * a.H + (h0 + hh)) * a.P + p;
            const int64_t xs = (int64_t)a.H * a.P;
            for (int jc = 0; jc < a.Q / 2; jc += 16) {
                uint32_t pk[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int j = 2 * (jc + q);
                    float v0 = 0.f, v1 = 0.f;
                    if (ok) {
                        if (j < len) v0 = __bfloat162float(xp[(int64_t)j * xs]) * sm->w[hh][j];
                        if (j + 1 < len) v1 = __bfloat162float(xp[(int64_t)(j + 1) * xs]) * sm->w[hh][j + 1];
                    }
                    pk[q] = pack_bf16x2(v0, v1);
                }
                tmem_st16(t_xw + lane_off + jc, pk);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();
        const bool landed = !__syncthreads_or(!wait_bar(&sm->bar_load, ph_load, a.status));
        ph_load ^= 1;
        if (tid == 0 && landed) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16_f32(128, a.N, 0, 1);
            const uint32_t sb = smem_u32(sB);
            for (int kk = 0; kk < a.Q / 16; ++kk) {
                const uint32_t off = (uint32_t)(kk / 8) * kTile16 + (uint32_t)(kk % 8) * 2048;
                mma_ts(t_s, t_xw + kk * 8,
                       smem_desc(sb + off, (uint32_t)nblk_j * kTile16, 1024, kSwizzle128B), idesc,
                       kk > 0);
            }
            mma_commit(&sm->bar_mma);
        }
        if (!landed) break;
        if (__syncthreads_or(!wait_bar(&sm->bar_mma, ph_mma, a.status))) break;
        ph_mma ^= 1;
        tc_fence_after();

        // chain step: wait for the entry state E_c of this (row, head pair)
        int *flag = a.flags + (int64_t)r * a.npairs + pair;
        if (c > 0 && tid == 0) {
            const uint64_t tw = globaltimer_ns();
            while (ld_acquire(flag) < c) {
                if (bail(a.status)) break;
                if (globaltimer_ns() - tw > kWaitLimitNs) {
                    set_status(a.status, SSD_ERR_DEVICE_TIMEOUT);
                    break;
                }
                __nanosleep(64);
            }
        }
        if (__syncthreads_or(tid == 0 && bail(a.status))) break;
        {
            const int hh = tid / 64, p = tid % 64;
            const int h = h0 + hh;
            const bool ok = (hh < a.kh) && (h < a.H) && (p < a.P);
            float *ring_rp = a.ring + (((int64_t)r * a.npairs + pair) * 2) * a.kh * PN;
            const float *Ein = ring_rp + (int64_t)(c & 1) * a.kh * PN + (int64_t)hh * PN + (int64_t)p * a.N;
            float *Eout = ring_rp + (int64_t)((c + 1) & 1) * a.kh * PN + (int64_t)hh * PN + (int64_t)p * a.N;
            const float *Einit = a.init ? a.init + (((int64_t)r * a.H + h) * a.P + p) * a.N : nullptr;
            bf16 *eb = a.ebuf + ((((int64_t)r * a.nc + c) * a.H + h) * a.P + p) * a.N;
            float *fin = (a.final_states && c == a.nc - 1)
                             ? a.final_states + (((int64_t)r * a.H + h) * a.P + p) * a.N
                             : nullptr;
            const float decay = (hh < a.kh) ? __expf(sm->cs[hh < 2 ? hh : 0][len - 1]) : 0.f;
            for (int n0 = 0; n0 < a.N; n0 += 32) {
                uint32_t sv[32];
                tmem_ld32(t_s + lane_off + n0, sv);
                tmem_ld_wait();
                if (!ok) continue;
                float e[32];
#pragma unroll
                for (int q = 0; q < 32; q += 4) {
                    float4 v;
                    if (c == 0) v = Einit ? *(const float4 *)(Einit + n0 + q) : make_float4(0, 0, 0, 0);
                    else v = __ldcg((const float4 *)(Ein + n0 + q));
                    e[q] = v.x; e[q + 1] = v.y; e[q + 2] = v.z; e[q + 3] = v.w;
                }
                uint32_t pk[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) pk[q] = pack_bf16x2(e[2 * q], e[2 * q + 1]);
#pragma unroll
                for (int q = 0; q < 16; q += 4)
                    *(uint4 *)(eb + n0 + 2 * q) = make_uint4(pk[q], pk[q + 1], pk[q + 2], pk[q + 3]);
#pragma unroll
                for (int q = 0; q < 32; q += 4) {
                    float4 o;
                    o.x = decay * e[q] + __uint_as_float(sv[q]);
                    o.y = decay * e[q + 1] + __uint_as_float(sv[q + 1]);
                    o.z = decay * e[q + 2] + __uint_as_float(sv[q + 2]);
                    o.w = decay * e[q + 3] + __uint_as_float(sv[q + 3]);
                    __stcg((float4 *)(Eout + n0 + q), o);
                    if (fin) *(float4 *)(fin + n0 + q) = o;
                }
            }
        }
        __threadfence();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) st_release(flag, c + 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, tmem_cols);
}

// ----------------------------------------------------------------------------
// k_chunk_output

struct OutSmem {
    float cs[256];
    float dtv[256];
    uint64_t bar_load, bar_mma1, bar_mma2, bar_mma3;
    uint32_t tmem;
};

__global__ void __launch_bounds__(kThreads, 1)
k_chunk_output(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmE,
               const __grid_constant__ CUtensorMap tmY, TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int nblk_n = a.N / 64;
    uint8_t *sC = base;                                  // 128 x N (K-major), reused for Xw_0
    uint8_t *sB = sC + (size_t)nblk_n * kTile16;         // 128 x N
    uint8_t *sX = sB + (size_t)nblk_n * kTile16;         // 128 x 64, reused for the y tile
    uint8_t *sE = sX + kTile16;                          // 64 x N (K-major), E then H_1
    OutSmem *sm = (OutSmem *)(sE + (size_t)nblk_n * 8192);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t tmem_cols = (a.N <= 128) ? 256 : 512;

    if (tid == 0) {
        mbar_init(&sm->bar_load, 1);
        mbar_init(&sm->bar_mma1, 1);
        mbar_init(&sm->bar_mma2, 1);
        mbar_init(&sm->bar_mma3, 1);
        fence_mbar_init();
        prefetch_tmap(&tmX); prefetch_tmap(&tmB); prefetch_tmap(&tmC);
        prefetch_tmap(&tmE); prefetch_tmap(&tmY);
    }
    if (warp == 0) { tmem_alloc(&sm->tmem, tmem_cols); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm->tmem;
    const uint32_t t_cb = tbase;          // 128 cols: CB fp32, then M bf16 in cols 0..63
    const uint32_t t_acc = tbase + 128;   // 64 cols: y accumulator
    const uint32_t t_s0 = tbase + 192;    // 64 cols per 128 state rows: S_0 [n][p]
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t ph_load = 0, ph1 = 0, ph2 = 0, ph3 = 0;
    const uint32_t sc = smem_u32(sC), sbb = smem_u32(sB), sx = smem_u32(sX), se = smem_u32(sE);
    const uint32_t id_cb = idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t id_off = idesc_bf16_f32(128, 64, 0, 0);
    const uint32_t id_diag = idesc_bf16_f32(128, 64, 0, 1);
    const uint32_t id_s0 = idesc_bf16_f32(128, 64, 1, 1);
    bool alive = true;

    for (int tile = blockIdx.x; tile < a.out_tiles && alive; tile += gridDim.x) {
        if (__syncthreads_or(tid == 0 && bail(a.status))) break;
        const int per_c = a.batch * a.H;
        const int c = tile / per_c;
        const int r = (tile % per_c) / a.H;
        const int h = tile % a.H;
        const int g = h / a.hpg;
        const int64_t t0 = (int64_t)c * a.Q;
        const int len = (int)min64(a.Q, a.L - t0);
        const int nhalf = (len + kBlk - 1) / kBlk;
        const float Dh = a.D ? __ldg(a.D + h) : 0.f;

        if (warp == 0)
            chunk_cumsum_warp(a.dt + ((int64_t)r * a.L + t0) * a.H + h, a.H, __ldg(a.A + h), a.Q,
                              len, sm->cs, sm->dtv);
        __syncthreads();

        for (int I = 0; I < nhalf && alive; ++I) {
            const int tb = (int)t0 + I * kBlk;
            if (tid == 0) {
                tma_store_wait_read0();   // sX may still feed the previous y store
                for (int nb = 0; nb < nblk_n; ++nb) {
                    tma_load_4d(sC + nb * kTile16, &tmC, &sm->bar_load, nb * 64, g, tb, r);
                    tma_load_4d(sB + nb * kTile16, &tmB, &sm->bar_load, nb * 64, g, tb, r);
                }
                tma_load_4d(sX, &tmX, &sm->bar_load, 0, h, tb, r);
                uint32_t bytes = (uint32_t)(2 * nblk_n + 1) * kTile16;
                if (I == 0) {
                    const int erow = (int)((((int64_t)r * a.nc + c) * a.H + h) * a.P);
                    for (int nb = 0; nb < nblk_n; ++nb)
                        tma_load_2d(sE + nb * 8192, &tmE, &sm->bar_load, nb * 64, erow);
                    bytes += (uint32_t)nblk_n * 8192;
                }
                mbar_arrive_expect_tx(&sm->bar_load, bytes);
            }
            if (__syncthreads_or(!wait_bar(&sm->bar_load, ph_load, a.status))) { alive = false; break; }
            ph_load ^= 1;
            if (tid == 0) {
                tc_fence_after();
                // CB_II = C_I B_I^T and acc = C_I H_I^T
                for (int kk = 0; kk < a.N / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk / 4) * kTile16 + (uint32_t)(kk % 4) * 32;
                    mma_ss(t_cb, smem_desc(sc + off, 16, 1024, kSwizzle128B),
                           smem_desc(sbb + off, 16, 1024, kSwizzle128B), id_cb, kk > 0);
                }
                for (int kk = 0; kk < a.N / 16; ++kk) {
                    const uint32_t offa = (uint32_t)(kk / 4) * kTile16 + (uint32_t)(kk % 4) * 32;
                    const uint32_t offe = (uint32_t)(kk / 4) * 8192 + (uint32_t)(kk % 4) * 32;
                    mma_ss(t_acc, smem_desc(sc + offa, 16, 1024, kSwizzle128B),
                           smem_desc(se + offe, 16, 1024, kSwizzle128B), id_off, kk > 0);
                }
                mma_commit(&sm->bar_mma1);
            }
            if (__syncthreads_or(!wait_bar(&sm->bar_mma1, ph1, a.status))) { alive = false; break; }
            ph1 ^= 1;
            tc_fence_after();
            // mask CB in place into bf16 M_II, scale the state term of acc
            {
                const int i = tid;                 // row within the block
                const int gi = I * kBlk + i;       // row within the chunk
                const float csi = sm->cs[gi];
                const bool rowv = gi < len;
#pragma unroll 1
                for (int m = 0; m < 4; ++m) {
                    uint32_t v[32];
                    tmem_ld32(t_cb + lane_off + m * 32, v);
                    tmem_ld_wait();
                    uint32_t pk[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int j0 = m * 32 + 2 * q;
                        const int gj0 = I * kBlk + j0;
                        float f0 = 0.f, f1 = 0.f;
                        if (rowv && j0 <= i)
                            f0 = __uint_as_float(v[2 * q]) * __expf(csi - sm->cs[gj0]) * sm->dtv[gj0];
                        if (rowv && j0 + 1 <= i)
                            f1 = __uint_as_float(v[2 * q + 1]) * __expf(csi - sm->cs[gj0 + 1]) * sm->dtv[gj0 + 1];
                        pk[q] = pack_bf16x2(f0, f1);
                    }
                    tmem_st16(t_cb + lane_off + m * 16, pk);
                }
                const float sc_off = rowv ? __expf(csi - (I == 0 ? 0.f : sm->cs[kBlk - 1])) : 0.f;
#pragma unroll 1
                for (int m = 0; m < 2; ++m) {
                    uint32_t v[32];
                    tmem_ld32(t_acc + lane_off + m * 32, v);
                    tmem_ld_wait();
                    uint32_t o[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) o[q] = __float_as_uint(__uint_as_float(v[q]) * sc_off);
                    tmem_st16(t_acc + lane_off + m * 32, o);
#pragma unroll
                    for (int q = 0; q < 16; ++q) o[q] = __float_as_uint(__uint_as_float(v[16 + q]) * sc_off);
                    tmem_st16(t_acc + lane_off + m * 32 + 16, o);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            __syncthreads();
            // acc += M_II X_I  (A from TMEM, B = X tile, MN-major)
            if (tid == 0) {
                tc_fence_after();
                for (int kk = 0; kk < kBlk / 16; ++kk)
                    mma_ts(t_acc, t_cb + kk * 8,
                           smem_desc(sx + kk * 2048, kTile16, 1024, kSwizzle128B), id_diag, 1);
                mma_commit(&sm->bar_mma2);
            }
            const bool need_s0 = (I == 0) && (nhalf > 1);
            if (need_s0) {
                // Xw_0 = exp(cs_127 - cs_j) dt_j x_j into the (now free) C buffer,
                // same swizzled [j][p] layout as the X tile.
                const int j = tid;
                const float wj = (j < len) ? __expf(sm->cs[kBlk - 1] - sm->cs[j]) * sm->dtv[j] : 0.f;
                const uint8_t *src = sX + j * 128;
                uint8_t *dst = sC + j * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint4 u = *(const uint4 *)(src + ch * 16);
                    uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162 *>(&w4[q]);
                        float2 f = __bfloat1622float2(b2);
                        w4[q] = pack_bf16x2(f.x * wj, f.y * wj);
                    }
                    *(uint4 *)(dst + ch * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                fence_proxy_async_smem();
                __syncthreads();
                if (tid == 0) {
                    // S_0[n][p] = sum_j B_0[j][n] Xw_0[j][p]: A = B_0^T (MN-major), B = Xw_0 (MN-major)
                    for (int mt = 0; mt < a.N / 128; ++mt)
                        for (int kk = 0; kk < kBlk / 16; ++kk)
                            mma_ss(t_s0 + mt * 64,
                                   smem_desc(sbb + mt * 2 * kTile16 + kk * 2048, kTile16, 1024, kSwizzle128B),
                                   smem_desc(sc + kk * 2048, kTile16, 1024, kSwizzle128B), id_s0, kk > 0);
                    mma_commit(&sm->bar_mma3);
                }
            }
            // epilogue: y = acc + D x
            if (__syncthreads_or(!wait_bar(&sm->bar_mma2, ph2, a.status))) { alive = false; break; }
            ph2 ^= 1;
            tc_fence_after();
            {
                const int i = tid;
                uint8_t *row = sX + i * 128;
#pragma unroll 1
                for (int m = 0; m < 2; ++m) {
                    uint32_t v[32];
                    tmem_ld32(t_acc + lane_off + m * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        // logical 16-byte chunk (m*4 + ch) of the row lives at chunk ^ (i & 7)
                        const int lc = m * 4 + ch;
                        uint8_t *cp = row + ((lc ^ (i & 7)) * 16);
                        uint4 u = *(const uint4 *)cp;
                        uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162 *>(&w4[q]);
                            float2 f = __bfloat1622float2(b2);
                            const int e = ch * 8 + 2 * q;
                            w4[q] = pack_bf16x2(__uint_as_float(v[e]) + Dh * f.x,
                                                __uint_as_float(v[e + 1]) + Dh * f.y);
                        }
                        *(uint4 *)cp = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tma_store_4d(&tmY, sX, 0, h, tb, r);
                tma_store_commit();
            }
            if (need_s0) {
                if (__syncthreads_or(!wait_bar(&sm->bar_mma3, ph3, a.status))) { alive = false; break; }
                ph3 ^= 1;
                tc_fence_after();
                // H_1[p][n] = exp(cs_127) E[p][n] + S_0[n][p], written over E (bf16)
                const float d127 = __expf(sm->cs[kBlk - 1]);
                for (int mt = 0; mt < a.N / 128; ++mt) {
                    const int n = mt * 128 + tid;
                    const int nb = n / 64, nn = n % 64;
#pragma unroll 1
                    for (int m = 0; m < 2; ++m) {
                        uint32_t v[32];
                        tmem_ld32(t_s0 + mt * 64 + lane_off + m * 32, v);
                        tmem_ld_wait();
#pragma unroll 4
                        for (int q = 0; q < 32; ++q) {
                            const int p = m * 32 + q;
                            // element (row p, col nn) of the swizzled 64 x 64 tile nb
                            bf16 *ep = (bf16 *)(sE + nb * 8192 + p * 128 +
                                                ((((nn >> 3) ^ (p & 7)) << 4) | ((nn & 7) << 1)));
                            const float hv = d127 * __bfloat162float(*ep) + __uint_as_float(v[q]);
                            *ep = __float2bfloat16_rn(hv);
                        }
                    }
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            __syncthreads();
        }
    }
    if (tid == 0) tma_store_wait0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, tmem_cols);
}

// ----------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

// bf16 tensor map; dims[0] innermost, box inner 64 elements, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims,
              const uint32_t *box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    uint64_t stride = 2;
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i > 0) gs[i - 1] = stride;
        stride *= dims[i];
    }
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), gd, gs, bx, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

struct TcLayout {
    size_t hdr, ring, ebuf, total;
    int kh, npairs;
};

TcLayout tc_layout(const Problem &p) {
    TcLayout w{};
    w.kh = ((p.H / p.G) % 2 == 0) ? 2 : 1;
    w.npairs = (p.H + w.kh - 1) / w.kh;
    size_t off = 0;
    w.hdr = off;   // counter (4 B) + flags
    off = align_up(off + 256 + (size_t)p.batch * w.npairs * sizeof(int), 256);
    w.ring = off;
    off = align_up(off + (size_t)p.batch * w.npairs * 2 * w.kh * p.P * p.N * sizeof(float), 256);
    w.ebuf = off;
    off = align_up(off + (size_t)p.batch * p.nc * p.H * p.P * p.N * sizeof(bf16), 256);
    w.total = off;
    return w;
}

size_t state_smem_bytes(const Problem &p) {
    // at least 80 KB so that no more than two CTAs (2 x 256 TMEM columns) share an SM
    const size_t need = 1024 + (size_t)p.Q * p.N * 2 + sizeof(StateSmem);
    return need < 81920 ? 81920 : need;
}
size_t out_smem_bytes(const Problem &p) {
    const size_t nb = p.N / 64;
    return 1024 + nb * kTile16 * 2 + kTile16 + nb * 8192 + sizeof(OutSmem);
}

}  // namespace

size_t tc_workspace_bytes(const Problem &p) { return tc_layout(p).total; }

int tc_supported(const Problem &p) {
    if (p.dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
    if (p.P != 64) return SSD_ERR_UNSUPPORTED;
    if (p.N != 128 && p.N != 256) return SSD_ERR_UNSUPPORTED;
    if (p.Q != 128 && p.Q != 256) return SSD_ERR_UNSUPPORTED;
    if (p.cu != nullptr) return SSD_ERR_UNSUPPORTED;
    if (!encode_fn()) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

cudaError_t tc_launch(const Problem &p) {
    const TcLayout w = tc_layout(p);
    TcArgs a{};
    a.L = p.seqlen; a.batch = (int)p.batch; a.H = p.H; a.P = p.P; a.N = p.N; a.G = p.G;
    a.Q = p.Q; a.nc = p.nc; a.hpg = p.H / p.G; a.kh = w.kh; a.npairs = w.npairs;
    a.state_tiles = a.nc * a.batch * a.npairs;
    a.out_tiles = a.nc * a.batch * a.H;
    a.x = (const bf16 *)p.x; a.dt = p.dt; a.A = p.A; a.D = p.D; a.init = p.init;
    a.final_states = p.final_states; a.status = p.status;
    a.counter = (int *)(p.ws + w.hdr);
    a.flags = (int *)(p.ws + w.hdr + 256);
    a.ring = (float *)(p.ws + w.ring);
    a.ebuf = (bf16 *)(p.ws + w.ebuf);

    cudaError_t e = cudaMemsetAsync(p.ws + w.hdr, 0, w.ring - w.hdr, p.stream);
    if (e != cudaSuccess) return e;

    CUtensorMap tmX, tmY, tmB, tmC, tmE;
    const uint64_t L = (uint64_t)p.seqlen, b = (uint64_t)p.batch;
    const uint64_t dx[4] = {(uint64_t)p.P, (uint64_t)p.H, L, b};
    const uint32_t bx[4] = {64, 1, (uint32_t)kBlk, 1};
    const uint64_t dbc[4] = {(uint64_t)p.N, (uint64_t)p.G, L, b};
    const uint64_t de[2] = {(uint64_t)p.N, b * p.nc * p.H * p.P};
    const uint32_t be[2] = {64, (uint32_t)p.P};
    if (!make_map(&tmX, p.x, 4, dx, bx) || !make_map(&tmY, p.y, 4, dx, bx) ||
        !make_map(&tmB, p.B, 4, dbc, bx) || !make_map(&tmC, p.C, 4, dbc, bx) ||
        !make_map(&tmE, a.ebuf, 2, de, be))
        return cudaErrorInvalidValue;

    const size_t s_smem = state_smem_bytes(p), o_smem = out_smem_bytes(p);
    e = cudaFuncSetAttribute(k_chunk_state, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_chunk_output, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)o_smem);
    if (e != cudaSuccess) return e;
    const int sms = num_sms();
    const int per_sm_state = (p.N <= 128) ? 2 : 1;
    const int per_sm_out = (p.N <= 128) ? 2 : 1;
    const int g_state = (int)min64(a.state_tiles, (int64_t)sms * per_sm_state);
    const int g_out = (int)min64(a.out_tiles, (int64_t)sms * per_sm_out);
    k_chunk_state<<<g_state, kThreads, s_smem, p.stream>>>(tmB, a);
    k_chunk_output<<<g_out, kThreads, o_smem, p.stream>>>(tmX, tmB, tmC, tmE, tmY, a);
    return cudaGetLastError();
}

}  // namespace ssd
