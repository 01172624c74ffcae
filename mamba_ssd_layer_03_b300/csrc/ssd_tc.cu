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
    void *y_out;       // y (bf16), written directly by the two-head output kernel
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

constexpr int kStateThreads = 256;

// Inclusive cumulative sum cs[j] = sum_{k<=j} dtv[k] * Ah over a chunk of Q
// tokens held in shared memory, computed by one warp.
__device__ __forceinline__ void cumsum_warp_smem(const float *dtv, float Ah, int Q, float *cs) {
    const int lane = threadIdx.x & 31;
    const int per = Q / 32;
    float local[8];
    float run = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        if (q < per) {
            run += dtv[lane * per + q] * Ah;
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

struct StateSmem {
    float cs[2][256];
    float w[2][256];
    float dtv[2][256];
    uint64_t bar_load, bar_mma;
    uint32_t tmem;
    int tile;
};

struct StateTile {
    int c, r, pair, h0, g, len;
    int64_t t0;
};

__device__ __forceinline__ StateTile decode_state_tile(const TcArgs &a, int tile) {
    StateTile t;
    const int per_c = a.batch * a.npairs;
    t.c = tile / per_c;
    t.r = (tile % per_c) / a.npairs;
    t.pair = tile % a.npairs;
    t.h0 = t.pair * a.kh;
    t.g = t.h0 / a.hpg;
    t.t0 = (int64_t)t.c * a.Q;
    t.len = (int)min64(a.Q, a.L - t.t0);
    return t;
}

// TMA loads of one state tile: B (Q x N, tiles [nb][jb]) and x for the
// tile's heads (tiles [head slot][jb]).  Thread 0 only.
__device__ __forceinline__ void state_issue_loads(const TcArgs &a, const StateTile &t,
                                                  const CUtensorMap *tmB, const CUtensorMap *tmX,
                                                  uint8_t *sB, uint8_t *sX, uint64_t *bar) {
    const int nblk_n = a.N / 64, nblk_j = a.Q / kBlk;
    for (int jb = 0; jb < nblk_j; ++jb) {
        for (int nb = 0; nb < nblk_n; ++nb)
            tma_load_4d(sB + (size_t)(nb * nblk_j + jb) * kTile16, tmB, bar, nb * 64, t.g,
                        (int)(t.t0 + jb * kBlk), t.r);
        for (int hh = 0; hh < a.kh; ++hh)
            tma_load_4d(sX + (size_t)(hh * nblk_j + jb) * kTile16, tmX, bar, 0, t.h0 + hh,
                        (int)(t.t0 + jb * kBlk), t.r);
    }
    mbar_arrive_expect_tx(bar, (uint32_t)(nblk_j * (nblk_n + a.kh)) * kTile16);
}

// Per (row, chunk, head pair): S[n][(h,p)] = sum_j B[j][n] w_j x_j[(h,p)] on the
// tensor cores (A = B^T and B = scaled x, both MN-major views of TMA tiles),
// then the chain step E_{c+1} = exp(cs_last) E_c + S through the ring.
__global__ void __launch_bounds__(kStateThreads, 1)
k_chunk_state(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmX,
              TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int nblk_n = a.N / 64, nblk_j = a.Q / kBlk;
    uint8_t *sB = base;                                          // Q x N
    uint8_t *sX = sB + (size_t)nblk_n * nblk_j * kTile16;        // kh x Q x 64
    StateSmem *sm = (StateSmem *)(sX + (size_t)2 * nblk_j * kTile16);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t tmem_cols = 256;
    const int ncols = a.kh * 64;             // (h, p) columns of S per 128-row state tile

    if (tid == 0) {
        mbar_init(&sm->bar_load, 1);
        mbar_init(&sm->bar_mma, 1);
        fence_mbar_init();
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmX);
    }
    if (warp == 0) { tmem_alloc(&sm->tmem, tmem_cols); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t t_s = sm->tmem;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t ph_load = 0, ph_mma = 0;
    const int PN = a.P * a.N;

    if (tid == 0) {
        const int t = atomicAdd(a.counter, 1);
        sm->tile = t;
        if (t < a.state_tiles)
            state_issue_loads(a, decode_state_tile(a, t), &tmB, &tmX, sB, sX, &sm->bar_load);
    }
    __syncthreads();

    while (true) {
        const int tile = sm->tile;   // same value in every thread
        if (tile >= a.state_tiles) break;
        const StateTile T = decode_state_tile(a, tile);

        // dt of the tile's heads, then the per-head cumulative decay
        for (int idx = tid; idx < a.kh * a.Q; idx += kStateThreads) {
            const int hh = idx / a.Q, j = idx % a.Q;
            float d = 0.f;
            if (j < T.len && T.h0 + hh < a.H)
                d = __ldg(a.dt + ((int64_t)T.r * a.L + T.t0 + j) * a.H + T.h0 + hh);
            sm->dtv[hh][j] = d;
        }
        __syncthreads();
        if (warp < a.kh) cumsum_warp_smem(sm->dtv[warp], __ldg(a.A + min(T.h0 + warp, a.H - 1)),
                                          a.Q, sm->cs[warp]);
        __syncthreads();
        for (int idx = tid; idx < a.kh * a.Q; idx += kStateThreads) {
            const int hh = idx / a.Q, j = idx % a.Q;
            sm->w[hh][j] = __expf(sm->cs[hh][T.len - 1] - sm->cs[hh][j]) * sm->dtv[hh][j];
        }
        __syncthreads();
        if (__syncthreads_or(!wait_bar(&sm->bar_load, ph_load, a.status))) break;
        ph_load ^= 1;
        // scale x rows in place: row j of head slot hh times w_j
        for (int idx = tid; idx < a.kh * a.Q; idx += kStateThreads) {
            const int hh = idx / a.Q, j = idx % a.Q;
            uint4 *row = (uint4 *)(sX + (size_t)(hh * nblk_j + j / kBlk) * kTile16 + (j % kBlk) * 128);
            const float wj = sm->w[hh][j];
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint4 u = row[ch];
                uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = bf2_to_f2(w4[q]);
                    w4[q] = pack_bf16x2(f.x * wj, f.y * wj);
                }
                row[ch] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16_f32(128, ncols, 1, 1);
            const uint32_t sb = smem_u32(sB), sx = smem_u32(sX);
            for (int mt = 0; mt < a.N / 128; ++mt)
                for (int kk = 0; kk < a.Q / 16; ++kk) {
                    const uint32_t roff = (uint32_t)(kk / 8) * kTile16 + (uint32_t)(kk % 8) * 2048;
                    mma_ss(t_s + mt * ncols,
                           smem_desc(sb + (uint32_t)(2 * mt * nblk_j) * kTile16 + roff,
                                     (uint32_t)nblk_j * kTile16, 1024, kSwizzle128B),
                           smem_desc(sx + roff, (uint32_t)nblk_j * kTile16, 1024, kSwizzle128B),
                           idesc, kk > 0);
                }
            mma_commit(&sm->bar_mma);
        }
        if (__syncthreads_or(!wait_bar(&sm->bar_mma, ph_mma, a.status))) break;
        ph_mma ^= 1;
        tc_fence_after();
        // the shared buffers are free again: start the next tile's loads now
        if (tid == 0) {
            const int t = bail(a.status) ? a.state_tiles : atomicAdd(a.counter, 1);
            sm->tile = t;
            if (t < a.state_tiles)
                state_issue_loads(a, decode_state_tile(a, t), &tmB, &tmX, sB, sX, &sm->bar_load);
        }

        // chain step: wait until the previous chunk published this head pair's E_c
        int *flag = a.flags + (int64_t)T.r * a.npairs + T.pair;
        if (T.c > 0 && tid == 0) {
            const uint64_t tw = globaltimer_ns();
            while (ld_acquire(flag) < T.c) {
                if (bail(a.status)) break;
                if (globaltimer_ns() - tw > kWaitLimitNs) {
                    set_status(a.status, SSD_ERR_DEVICE_TIMEOUT);
                    break;
                }
                __nanosleep(32);
            }
        }
        if (__syncthreads_or(tid == 0 && bail(a.status))) break;
        const int hh = tid / 128;            // head slot of this thread
        const int h = T.h0 + hh;
        const bool hok = (hh < a.kh) && (h < a.H);
        float *ring_rp = a.ring + ((int64_t)T.r * a.npairs + T.pair) * 2 * a.kh * PN;
        const float *Ein = ring_rp + (int64_t)(T.c & 1) * a.kh * PN + (int64_t)hh * PN;
        float *Eout = ring_rp + (int64_t)((T.c + 1) & 1) * a.kh * PN + (int64_t)hh * PN;
        const float *Einit = (a.init && hok) ? a.init + ((int64_t)T.r * a.H + h) * PN : nullptr;
        const float decay = hok ? __expf(sm->cs[hh][T.len - 1]) : 0.f;
        // E_c (bf16, for the output kernel) and the final state are written
        // from registers here: once the flag below is released, the next
        // chunk's tile may overwrite this tile's input slot of the ring.
        bf16 *eb = hok ? a.ebuf + (((int64_t)T.r * a.nc + T.c) * a.H + h) * PN : nullptr;
        float *fin = (hok && a.final_states && T.c == a.nc - 1)
                         ? a.final_states + ((int64_t)T.r * a.H + h) * PN : nullptr;
        for (int mt = 0; mt < a.N / 128; ++mt) {
            const int n = mt * 128 + (tid & 127);
#pragma unroll
            for (int p0 = 0; p0 < 64; p0 += 32) {
                uint32_t sv[32];
                tmem_ld32(t_s + mt * ncols + (hh < a.kh ? hh : 0) * 64 + p0 + lane_off, sv);
                tmem_ld_wait();
                if (!hok) continue;
                // all 32 loads first: the ring slots are not known not to
                // alias, so interleaving them with the stores would serialise
                // one L2 round trip per element
                float ev[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int64_t idx = (int64_t)(p0 + q) * a.N + n;
                    if (T.c == 0) ev[q] = Einit ? __ldg(Einit + idx) : 0.f;
                    else ev[q] = __ldcg(Ein + idx);
                }
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int64_t idx = (int64_t)(p0 + q) * a.N + n;
                    const float e = ev[q];
                    const float en = decay * e + __uint_as_float(sv[q]);
                    __stcg(Eout + idx, en);
                    eb[idx] = __float2bfloat16_rn(e);
                    if (fin) fin[idx] = en;
                }
            }
        }
        __threadfence();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) st_release(flag, T.c + 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(t_s, tmem_cols);
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
                        const float2 f = bf2_to_f2(w4[q]);
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
                            const float2 f = bf2_to_f2(w4[q]);
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
#pragma unroll
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
// k_chunk_output_h2: a tile is HG heads of one (row, chunk) sharing one B/C
// group.  C B^T of the chunk's two 128-token diagonal blocks is computed once
// per tile and kept in TMEM (fp32); the tile's heads are then processed two
// at a time ("items"), the pair stacked along N in the state-term and state
// contractions.  Each head's masked block M = CB o (exp(cs_i - cs_j) dt_j)
// is written as bf16 into TMEM and fed to the MMA as the A operand.  The
// decay factor is split at 32-token sub-blocks: exp(cs_i - cs_j) =
// exp(cs_i - ref) exp(ref - cs_j) with ref the cs at the end of j's
// sub-block, so only the sub-block containing i needs pairwise exponentials;
// both factors are <= 1.

constexpr int kOutThreads = 256;

struct Out2Smem {
    float cs[2][256];
    float dtv[2][256];
    float vf[2][256];   // exp(cs[end of j's 32-block] - cs_j) dt_j
    uint64_t bar_cb, bar_cbm, bar_e, bar_x, bar_y, bar_d, bar_s;
    uint32_t tmem;
};

struct OutItem {
    int valid, c, r, h0, g, len, nhalf;
    int64_t t0;
};

__device__ __forceinline__ OutItem decode_item(const TcArgs &a, int tile, int k, int HG) {
    OutItem it{};
    const int nhg = a.H / HG;
    const int ntiles = a.nc * a.batch * nhg;
    it.valid = tile < ntiles && k < HG / 2;
    if (!it.valid) return it;
    const int per_c = a.batch * nhg;
    it.c = tile / per_c;
    it.r = (tile % per_c) / nhg;
    const int hg = tile % nhg;
    it.h0 = hg * HG + 2 * k;
    it.g = it.h0 / a.hpg;
    it.t0 = (int64_t)it.c * a.Q;
    it.len = (int)min64(a.Q, a.L - it.t0);
    it.nhalf = (it.len + kBlk - 1) / kBlk;
    return it;
}

__global__ void __launch_bounds__(kOutThreads, 1)
k_chunk_output_h2(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmE2,
                  TcArgs a, int HG) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int nhq = a.Q / kBlk;                           // 128-token blocks per chunk
    uint8_t *sC = base;                                   // [I][nb] 16 KB tiles, K-major
    uint8_t *sB = sC + (size_t)nhq * 2 * kTile16;         // [I][nb]; block 1 reused for Xw_0
    uint8_t *sX = sB + (size_t)nhq * 2 * kTile16;         // [head slot] 128 x 64
    uint8_t *sE = sX + 2 * kTile16;                       // [nb] 128 (h,p) rows x 64 n
    Out2Smem *sm = (Out2Smem *)(sE + 2 * kTile16);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int hh = tid >> 7;                              // head slot of this thread
    const int li = tid & 127;                             // TMEM lane / row of this thread
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;

    if (tid == 0) {
        mbar_init(&sm->bar_cb, 1); mbar_init(&sm->bar_cbm, 1); mbar_init(&sm->bar_e, 1);
        mbar_init(&sm->bar_x, 1); mbar_init(&sm->bar_y, 1); mbar_init(&sm->bar_d, 1);
        mbar_init(&sm->bar_s, 1);
        fence_mbar_init();
        prefetch_tmap(&tmX); prefetch_tmap(&tmB); prefetch_tmap(&tmC); prefetch_tmap(&tmE2);
    }
    if (warp == 0) { tmem_alloc(&sm->tmem, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t T_CB = sm->tmem, T_M = sm->tmem + 256, T_ACC = sm->tmem + 384;
    const uint32_t sc = smem_u32(sC), sbb = smem_u32(sB), sx = smem_u32(sX), se = smem_u32(sE);
    const uint32_t id_cb = idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t id_off = idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t id_diag = idesc_bf16_f32(128, 64, 0, 1);
    const uint32_t id_s0 = idesc_bf16_f32(128, 128, 1, 1);
    uint32_t ph_cb = 0, ph_cbm = 0, ph_e = 0, ph_x = 0, ph_y = 0, ph_d = 0, ph_s = 0;
    const int items = HG / 2;

    auto load_e = [&](const OutItem &it) {
        const int row = (int)((((int64_t)it.r * a.nc + it.c) * a.H + it.h0) * a.P);
        for (int nb = 0; nb < 2; ++nb)
            tma_load_2d(sE + nb * kTile16, &tmE2, &sm->bar_e, nb * 64, row);
        mbar_arrive_expect_tx(&sm->bar_e, 2 * kTile16);
    };
    auto load_x = [&](const OutItem &it, int I) {
        for (int s = 0; s < 2; ++s)
            tma_load_4d(sX + s * kTile16, &tmX, &sm->bar_x, 0, it.h0 + s, (int)(it.t0 + I * kBlk), it.r);
        mbar_arrive_expect_tx(&sm->bar_x, 2 * kTile16);
    };

    int tile = blockIdx.x;
    if (tid == 0) {
        const OutItem f = decode_item(a, tile, 0, HG);
        if (f.valid) { load_e(f); load_x(f, 0); }
    }
    for (; decode_item(a, tile, 0, HG).valid; tile += gridDim.x) {
        const OutItem first = decode_item(a, tile, 0, HG);
        // C and B of the chunk (both blocks), then C_I B_I^T for each block
        if (tid == 0) {
            for (int I = 0; I < first.nhalf; ++I)
                for (int nb = 0; nb < 2; ++nb) {
                    tma_load_4d(sC + (I * 2 + nb) * kTile16, &tmC, &sm->bar_cb, nb * 64, first.g,
                                (int)(first.t0 + I * kBlk), first.r);
                    tma_load_4d(sB + (I * 2 + nb) * kTile16, &tmB, &sm->bar_cb, nb * 64, first.g,
                                (int)(first.t0 + I * kBlk), first.r);
                }
            mbar_arrive_expect_tx(&sm->bar_cb, (uint32_t)first.nhalf * 4 * kTile16);
        }
        if (__syncthreads_or(!wait_bar(&sm->bar_cb, ph_cb, a.status))) goto done;
        ph_cb ^= 1;
        if (tid == 0) {
            tc_fence_after();
            for (int I = 0; I < first.nhalf; ++I)
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (uint32_t)(I * 2 + kk / 4) * kTile16 + (uint32_t)(kk % 4) * 32;
                    mma_ss(T_CB + I * 128, smem_desc(sc + off, 16, 1024, kSwizzle128B),
                           smem_desc(sbb + off, 16, 1024, kSwizzle128B), id_cb, kk > 0);
                }
            mma_commit(&sm->bar_cbm);
        }

        for (int k = 0; k < items; ++k) {
            const OutItem it = decode_item(a, tile, k, HG);
            const OutItem nx = (k + 1 < items) ? decode_item(a, tile, k + 1, HG)
                                               : decode_item(a, tile + gridDim.x, 0, HG);
            // per-head decay cumsum and column factors
            for (int idx = tid; idx < 2 * a.Q; idx += kOutThreads) {
                const int s = idx / a.Q, j = idx % a.Q;
                sm->dtv[s][j] = (j < it.len)
                    ? __ldg(a.dt + ((int64_t)it.r * a.L + it.t0 + j) * a.H + it.h0 + s) : 0.f;
            }
            __syncthreads();
            if (warp < 2) cumsum_warp_smem(sm->dtv[warp], __ldg(a.A + it.h0 + warp), a.Q, sm->cs[warp]);
            __syncthreads();
            for (int idx = tid; idx < 2 * a.Q; idx += kOutThreads) {
                const int s = idx / a.Q, j = idx % a.Q;
                sm->vf[s][j] = __expf(sm->cs[s][(j | 31)] - sm->cs[s][j]) * sm->dtv[s][j];
            }
            __syncthreads();
            const float Dh = a.D ? __ldg(a.D + it.h0 + hh) : 0.f;

            for (int I = 0; I < it.nhalf; ++I) {
                // state term: acc = C_I H_I^T for both heads (H_0 = E_c, H_1 written below)
                if (__syncthreads_or(I == 0 && !wait_bar(&sm->bar_e, ph_e, a.status))) goto done;
                if (I == 0) ph_e ^= 1;
                if (k == 0 && I == 0) {
                    if (__syncthreads_or(!wait_bar(&sm->bar_cbm, ph_cbm, a.status))) goto done;
                    ph_cbm ^= 1;
                }
                if (tid == 0) {
                    tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t offa = (uint32_t)(I * 2 + kk / 4) * kTile16 + (uint32_t)(kk % 4) * 32;
                        const uint32_t offe = (uint32_t)(kk / 4) * kTile16 + (uint32_t)(kk % 4) * 32;
                        mma_ss(T_ACC, smem_desc(sc + offa, 16, 1024, kSwizzle128B),
                               smem_desc(se + offe, 16, 1024, kSwizzle128B), id_off, kk > 0);
                    }
                    mma_commit(&sm->bar_y);
                }
                // masked diagonal block of this thread's head into TMEM (bf16)
                {
                    const int gi = I * kBlk + li;
                    const bool rowv = gi < it.len;
                    const float csi = sm->cs[hh][gi];
                    const int bi = li >> 5;
#pragma unroll 1
                    for (int m = 0; m < 4; ++m) {
                        uint32_t pk[16];
                        if (m > bi) {
#pragma unroll
                            for (int q = 0; q < 16; ++q) pk[q] = 0u;
                        } else {
                            uint32_t v[32];
                            tmem_ld32(T_CB + I * 128 + lane_off + m * 32, v);
                            tmem_ld_wait();
                            const int gj = I * kBlk + m * 32;
                            if (m < bi) {
                                const float u = rowv ? __expf(csi - sm->cs[hh][gj + 31]) : 0.f;
#pragma unroll
                                for (int q = 0; q < 16; ++q)
                                    pk[q] = pack_bf16x2(__uint_as_float(v[2 * q]) * u * sm->vf[hh][gj + 2 * q],
                                                        __uint_as_float(v[2 * q + 1]) * u * sm->vf[hh][gj + 2 * q + 1]);
                            } else {
                                const int lj = li & 31;
#pragma unroll
                                for (int q = 0; q < 16; ++q) {
                                    const int j0 = 2 * q, j1 = 2 * q + 1;
                                    const float f0 = (rowv && j0 <= lj)
                                        ? __uint_as_float(v[j0]) * __expf(csi - sm->cs[hh][gj + j0]) * sm->dtv[hh][gj + j0] : 0.f;
                                    const float f1 = (rowv && j1 <= lj)
                                        ? __uint_as_float(v[j1]) * __expf(csi - sm->cs[hh][gj + j1]) * sm->dtv[hh][gj + j1] : 0.f;
                                    pk[q] = pack_bf16x2(f0, f1);
                                }
                            }
                        }
                        tmem_st16(T_M + hh * 64 + lane_off + m * 16, pk);
                    }
                    // scale this head's state term: exp(cs_i - r_I)
                    if (__syncthreads_or(!wait_bar(&sm->bar_y, ph_y, a.status))) goto done;
                    ph_y ^= 1;
                    tc_fence_after();
                    // the item's last state-term MMA has read E/H: prefetch the next item's E
                    if (I + 1 == it.nhalf && tid == 0 && nx.valid) load_e(nx);
                    const float f = rowv ? __expf(csi - (I == 0 ? 0.f : sm->cs[hh][kBlk - 1])) : 0.f;
#pragma unroll 1
                    for (int m = 0; m < 2; ++m) {
                        uint32_t v[32];
                        tmem_ld32(T_ACC + hh * 64 + lane_off + m * 32, v);
                        tmem_ld_wait();
                        uint32_t o[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) o[q] = __float_as_uint(__uint_as_float(v[q]) * f);
                        tmem_st16(T_ACC + hh * 64 + lane_off + m * 32, o);
#pragma unroll
                        for (int q = 0; q < 16; ++q) o[q] = __float_as_uint(__uint_as_float(v[16 + q]) * f);
                        tmem_st16(T_ACC + hh * 64 + lane_off + m * 32 + 16, o);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                if (__syncthreads_or(!wait_bar(&sm->bar_x, ph_x, a.status))) goto done;
                ph_x ^= 1;
                // acc += M X for each head; then (block 0) S_0 for the block-1 state
                if (tid == 0) {
                    tc_fence_after();
                    for (int s = 0; s < 2; ++s)
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ts(T_ACC + s * 64, T_M + s * 64 + kk * 8,
                                   smem_desc(sx + s * kTile16 + kk * 2048, kTile16, 1024, kSwizzle128B),
                                   id_diag, 1);
                    mma_commit(&sm->bar_d);
                }
                const bool s0 = (I == 0) && (it.nhalf > 1);
                if (s0) {
                    // Xw_0 = exp(cs_127 - cs_j) dt_j x_j into block-1 B space (free after C_1 B_1^T)
                    const int j = li;
                    const float wj = __expf(sm->cs[hh][kBlk - 1] - sm->cs[hh][j]) * sm->dtv[hh][j];
                    const uint4 *src = (const uint4 *)(sX + hh * kTile16 + j * 128);
                    uint4 *dst = (uint4 *)(sB + 2 * kTile16 + hh * kTile16 + j * 128);
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint4 u = src[ch];
                        uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = bf2_to_f2(w4[q]);
                            w4[q] = pack_bf16x2(f.x * wj, f.y * wj);
                        }
                        dst[ch] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    fence_proxy_async_smem();
                    __syncthreads();
                    if (tid == 0) {
                        // S_0[n][(h,p)] = sum_j B_0[j][n] Xw_0[j][(h,p)] into the M columns
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(T_M, smem_desc(sbb + kk * 2048, kTile16, 1024, kSwizzle128B),
                                   smem_desc(sbb + 2 * kTile16 + kk * 2048, kTile16, 1024, kSwizzle128B),
                                   id_s0, kk > 0);
                        mma_commit(&sm->bar_s);
                    }
                }
                // epilogue: y = acc + D x for this thread's head, stored straight to global
                if (__syncthreads_or(!wait_bar(&sm->bar_d, ph_d, a.status))) goto done;
                ph_d ^= 1;
                tc_fence_after();
                {
                    const int i = li;
                    const int64_t tok = it.t0 + I * kBlk + i;
                    const uint8_t *row = sX + hh * kTile16 + i * 128;
                    bf16 *yrow = (bf16 *)a.y_out + (((int64_t)it.r * a.L + tok) * a.H + it.h0 + hh) * a.P;
#pragma unroll 1
                    for (int m = 0; m < 2; ++m) {
                        uint32_t v[32];
                        tmem_ld32(T_ACC + hh * 64 + lane_off + m * 32, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch) {
                            const int lc = m * 4 + ch;
                            const uint4 u = *(const uint4 *)(row + ((lc ^ (i & 7)) * 16));
                            uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float2 f = bf2_to_f2(w4[q]);
                                const int e = ch * 8 + 2 * q;
                                w4[q] = pack_bf16x2(__uint_as_float(v[e]) + Dh * f.x,
                                                    __uint_as_float(v[e + 1]) + Dh * f.y);
                            }
                            if (tok < a.L)
                                *(uint4 *)(yrow + lc * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                }
                tc_fence_before();
                __syncthreads();
                // x of the next block (or of the next item) into the now free X tiles
                if (tid == 0) {
                    if (I + 1 < it.nhalf) load_x(it, I + 1);
                    else if (nx.valid) load_x(nx, 0);
                }
                if (s0) {
                    // H_1[(h,p)][n] = exp(cs_127) E[(h,p)][n] + S_0[n][(h,p)], over E in place
                    if (__syncthreads_or(!wait_bar(&sm->bar_s, ph_s, a.status))) goto done;
                    ph_s ^= 1;
                    tc_fence_after();
                    const float d127 = __expf(sm->cs[hh][kBlk - 1]);
                    const int n = li, nb = n >> 6, nn = n & 63;
                    uint8_t *ebase = sE + nb * kTile16;
#pragma unroll 1
                    for (int m = 0; m < 2; ++m) {
                        uint32_t v[32];
                        tmem_ld32(T_M + hh * 64 + lane_off + m * 32, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            const int row = hh * 64 + m * 32 + q;
                            bf16 *ep = (bf16 *)(ebase + row * 128 + ((((nn >> 3) ^ (row & 7)) << 4) | ((nn & 7) << 1)));
                            *ep = __float2bfloat16_rn(d127 * __bfloat162float(*ep) + __uint_as_float(v[q]));
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncthreads();
                }
            }
        }
    }
done:
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(T_CB, 512);
}

// ----------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once.  A function-local static
// is initialised exactly once even when several host threads make their first
// call at the same time.
EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return (EncodeTiledFn)p;
        return nullptr;
    }();
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

// SM count of the current device (asked every time: calls may come from
// several devices).
int num_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
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
    const size_t nblk_j = p.Q / kBlk;
    return 1024 + (size_t)p.Q * p.N * 2 + 2 * nblk_j * kTile16 + sizeof(StateSmem);
}
size_t out2_smem_bytes(const Problem &p) {
    const size_t nhq = p.Q / kBlk;
    return 1024 + nhq * 4 * kTile16 + 4 * kTile16 + sizeof(Out2Smem);
}
// Heads per output tile of the two-head kernel: the largest of 8, 6, 4, 2
// that divides the heads of one B/C group.
int out2_heads_per_tile(const Problem &p) {
    const int hpg = p.H / p.G;
    for (int hg : {8, 6, 4, 2})
        if (hpg % hg == 0) return hg;
    return 0;
}
bool use_out2(const Problem &p) { return p.N == 128 && out2_heads_per_tile(p) > 0; }
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
    a.y_out = p.y;

    cudaError_t e = cudaMemsetAsync(p.ws + w.hdr, 0, w.ring - w.hdr, p.stream);
    if (e != cudaSuccess) return e;

    CUtensorMap tmX, tmY, tmB, tmC, tmE, tmE2;
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
    const uint32_t be2[2] = {64, 128};
    if (!make_map(&tmE2, a.ebuf, 2, de, be2)) return cudaErrorInvalidValue;

    const bool two = use_out2(p);
    const size_t s_smem = state_smem_bytes(p), o_smem = two ? out2_smem_bytes(p) : out_smem_bytes(p);
    e = cudaFuncSetAttribute(k_chunk_state, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_smem);
    if (e != cudaSuccess) return e;
    e = two ? cudaFuncSetAttribute(k_chunk_output_h2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)o_smem)
            : cudaFuncSetAttribute(k_chunk_output, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)o_smem);
    if (e != cudaSuccess) return e;
    const int sms = num_sms();
    const int per_sm_state = 1;
    const int per_sm_out = (p.N <= 128) ? 2 : 1;
    const int g_state = (int)min64(a.state_tiles, (int64_t)sms * per_sm_state);
    const int g_out = (int)min64(a.out_tiles, (int64_t)sms * per_sm_out);
    k_chunk_state<<<g_state, kStateThreads, s_smem, p.stream>>>(tmB, tmX, a);
    if (two) {
        const int HG = out2_heads_per_tile(p);
        const int tiles = a.nc * a.batch * (p.H / HG);
        k_chunk_output_h2<<<(int)min64(tiles, sms), kOutThreads, o_smem, p.stream>>>(tmX, tmB, tmC, tmE2, a, HG);
    } else {
        k_chunk_output<<<g_out, kThreads, o_smem, p.stream>>>(tmX, tmB, tmC, tmE, tmY, a);
    }
    return cudaGetLastError();
}

}  // namespace ssd
