// SIMT (CUDA-core) path of the SSD forward scan.
//
// This is the fp32 path (its 1e-5 tolerance rules out tf32 tensor cores) and
// the generic path for any headdim/dstate up to 256.  It follows the block
// decomposition of the semiseparable matrix M = L o (C B^T) described in the
// QbitAI article "新架构Mamba更新二代！" (section "统一SSM和注意力机制" for the
// semiseparable/masked-attention duality, section
// "Mamba-2：更强学习能力，更快训练推理" for the block-decomposition algorithm):
//
//   K1 chunk cumsum   cs_i = sum of a_k = dt_k A_h over the chunk, restarted
//                     at every packed-sequence start inside the chunk (fp64,
//                     a warp-wide segmented scan per head)
//   K2 chunk state    S_c = sum_j exp(cs_last - cs_j) dt_j x_j (outer) B_j over
//                     the chunk's last sequence piece, from a zero state
//   K3 state passing  E_c (state entering chunk c's first sequence piece):
//                     E_{c+1} = exp(cs_last) E'_c + S_c, or the next
//                     sequence's initial state when one starts at the chunk
//                     boundary; writes final states that end on a chunk end
//   K5 sequence final final states of packed sequences ending inside a chunk
//   K4 chunk output   y_i = sum_{j<=i, same seq} (C_i.B_j) exp(cs_i-cs_j) dt_j x_j
//                           + exp(cs_i) C_i . E(seq(i)) + D_h x_i
// Decay exponents are differences of fp64 partial sums so that long chunks
// of strongly decaying heads keep fp32-level relative accuracy.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ssd_device.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

struct KArgs {
    int64_t L;
    int H, P, N, G, Q, nc, nseq, hpg;
    bool varlen;
    const void *x;
    const float *dt, *A;
    const void *B, *C;
    const float *D, *init;
    const int32_t *cu;
    void *y;
    float *final_states;
    int *status;
    double *cs;   // [b][H][nc][Q]
    float *S;     // [b][nc][H][P][N]
    float *E;     // [b][nc][H][P][N]
};

__device__ __forceinline__ int64_t cs_index(const KArgs &a, int r, int h, int c) {
    return (((int64_t)r * a.H + h) * a.nc + c) * a.Q;
}
__device__ __forceinline__ int64_t st_index(const KArgs &a, int r, int c, int h) {
    return (((int64_t)r * a.nc + c) * a.H + h) * (int64_t)a.P * a.N;
}
// Sequence containing token t of row r, and that sequence's first token.
__device__ __forceinline__ int seq_of(const KArgs &a, int r, int64_t t) {
    return a.varlen ? seg_of(a.cu, a.nseq, t) : r;
}
__device__ __forceinline__ int64_t seq_start(const KArgs &a, int s) {
    return a.varlen ? (int64_t)__ldg(a.cu + s) : 0;
}

// K1: grid (nc, batch, ceil(H / 32)), block kK1Threads.  The chunk's dt for
// 32 heads is staged in shared memory with coalesced reads (32 consecutive
// heads of one token per warp load); then each warp takes whole heads, 32
// tokens per step: a warp-wide segmented inclusive scan in fp64 (a segment
// starts where a packed sequence starts), plus the running sum carried from
// the previous 32 tokens, written to cs as 32 consecutive doubles.
constexpr int kK1Threads = 256;
constexpr int kMaxQ = 256;

__global__ void __launch_bounds__(kK1Threads) k1_chunk_cumsum(KArgs a) {
    __shared__ float tile[kMaxQ][33];   // [token][head]; 33: no bank conflicts
    __shared__ int seg[kMaxQ];          // packed-sequence index of each token
    if (status_bad(a.status)) return;
    const int c = blockIdx.x, r = blockIdx.y, hb = blockIdx.z * 32;
    const int64_t t0 = (int64_t)c * a.Q;
    const int len = (int)min64(a.Q, a.L - t0);
    const int nh = min(32, a.H - hb);
    for (int idx = threadIdx.x; idx < len * 32; idx += kK1Threads) {
        const int i = idx >> 5, hl = idx & 31;
        if (hl < nh) tile[i][hl] = __ldg(a.dt + ((int64_t)r * a.L + t0 + i) * a.H + hb + hl);
    }
    if (a.varlen)
        for (int i = threadIdx.x; i < len; i += kK1Threads) seg[i] = seg_of(a.cu, a.nseq, t0 + i);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int hl = warp; hl < nh; hl += kK1Threads / 32) {
        const int h = hb + hl;
        const double Ah = (double)__ldg(a.A + h);
        double *out = a.cs + cs_index(a, r, h, c);
        double carry = 0.0;
        for (int i0 = 0; i0 < len; i0 += 32) {
            const int i = i0 + lane;
            const bool valid = i < len;
            double v = valid ? (double)tile[i][hl] * Ah : 0.0;
            // f: a segment starts at or before this lane within these 32 tokens
            int f = (a.varlen && valid && i > 0 && seg[i] != seg[i - 1]) ? 1 : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const double vv = __shfl_up_sync(0xffffffffu, v, d);
                const int ff = __shfl_up_sync(0xffffffffu, f, d);
                if (lane >= d) {
                    if (!f) v += vv;
                    f |= ff;
                }
            }
            const double run = f ? v : carry + v;
            if (valid) out[i] = run;
            carry = __shfl_sync(0xffffffffu, run, 31);
        }
    }
}

// K2: grid (nc, batch, H), block 256; threads over (p, n).  The chunk's
// weighted x (w_j x_j, head h) and B (group g) are staged in shared memory
// k2_tile() tokens at a time with coalesced loads, all in flight at once, so
// that the token loop reads shared memory instead of waiting on one cache
// line per token.
__host__ __device__ inline int k2_tile(int P, int N) { return P + N <= 256 ? 32 : 16; }

template <typename T>
__global__ void k2_chunk_state(KArgs a) {
    if (status_bad(a.status)) return;
    extern __shared__ float k2s[];   // w[Q], xs[tile][P], bs[tile][N]
    const int TJ = k2_tile(a.P, a.N);
    float *w_smem = k2s;
    float *xs = k2s + a.Q;
    float *bs = xs + TJ * a.P;
    const int c = blockIdx.x, r = blockIdx.y, h = blockIdx.z;
    const int g = h / a.hpg;
    const int64_t t0 = (int64_t)c * a.Q;
    const int len = (int)min64(a.Q, a.L - t0);
    const int ls = seq_of(a, r, t0 + len - 1);
    const int j0 = (int)max64(0, seq_start(a, ls) - t0);
    const double *cs = a.cs + cs_index(a, r, h, c);
    const double cl = cs[len - 1];
    for (int j = threadIdx.x; j < a.Q; j += blockDim.x) {
        float w = 0.f;
        if (j >= j0 && j < len)
            w = (float)exp(cl - cs[j]) * __ldg(a.dt + ((int64_t)r * a.L + t0 + j) * a.H + h);
        w_smem[j] = w;
    }
    const T *x = (const T *)a.x;
    const T *B = (const T *)a.B;
    const int PN = a.P * a.N;
    float *S = a.S + st_index(a, r, c, h);
    for (int e0 = 0; e0 < PN; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const int p = e / a.N, n = e % a.N;
        float acc = 0.f;
        for (int jt = j0; jt < len; jt += TJ) {
            const int nj = min(TJ, len - jt);
            __syncthreads();   // the weights are written; the previous tile is used up
            // unrolled: several loads in flight before their stores
#pragma unroll 4
            for (int idx = threadIdx.x; idx < nj * a.P; idx += blockDim.x) {
                const int jj = idx / a.P, pp = idx % a.P;
                const int64_t tok = (int64_t)r * a.L + t0 + jt + jj;
                xs[jj * a.P + pp] = w_smem[jt + jj] * ld_as_float(x + (tok * a.H + h) * a.P + pp);
            }
#pragma unroll 4
            for (int idx = threadIdx.x; idx < nj * a.N; idx += blockDim.x) {
                const int jj = idx / a.N, nn = idx % a.N;
                const int64_t tok = (int64_t)r * a.L + t0 + jt + jj;
                bs[jj * a.N + nn] = ld_as_float(B + (tok * a.G + g) * a.N + nn);
            }
            __syncthreads();
            if (e < PN)
                for (int jj = 0; jj < nj; ++jj) acc += xs[jj * a.P + p] * bs[jj * a.N + n];
        }
        if (e < PN) S[e] = acc;
    }
}

// K3: grid (ceil(P*N/256), H, batch), block 256; one thread per state
// element walks the chunks of its row in order.  The walk is a chain of one
// multiply-add per chunk; what feeds it does not depend on the chain, so it
// is computed ahead: per group of 32 chunks, lane j of every warp works out
// chunk c0 + j's decay exp(cs_last) (fp64 exp, once per chunk instead of
// once per element), its first/last sequence and whether a sequence starts
// or ends there, and shares them by shuffles; the chunk states S are loaded
// kK3Ahead chunks at a time before the chain consumes them.
constexpr int kK3Ahead = 8;

__global__ void __launch_bounds__(256) k3_state_passing(KArgs a) {
    if (status_bad(a.status)) return;
    const int h = blockIdx.y, r = blockIdx.z;
    const int PN = a.P * a.N;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = e < PN;            // dead lanes still take part in the shuffles
    const int lane = threadIdx.x & 31;
    const float *S = a.S + st_index(a, r, 0, h) + e;
    float *E = a.E + st_index(a, r, 0, h) + e;
    const int64_t cstride = (int64_t)a.H * PN;   // from chunk c to c + 1 in S and E
    const float *init = a.init ? a.init + (int64_t)h * PN + e : nullptr;   // + seq * H * PN
    float *fin = a.final_states ? a.final_states + (int64_t)h * PN + e : nullptr;
    float end_state = 0.f;
    for (int c0 = 0; c0 < a.nc; c0 += 32) {
        // per-chunk facts, chunk c0 + lane
        float dec_l = 0.f;
        int fs_l = 0, ls_l = 0, flags_l = 0;   // bit 0: sequence starts; bit 1: final here
        const int cl_ = c0 + lane;
        if (cl_ < a.nc) {
            const int64_t t0 = (int64_t)cl_ * a.Q;
            const int len = (int)min64(a.Q, a.L - t0);
            fs_l = seq_of(a, r, t0);
            ls_l = seq_of(a, r, t0 + len - 1);
            dec_l = (float)exp(a.cs[cs_index(a, r, h, cl_) + len - 1]);
            if (cl_ == 0 || seq_start(a, fs_l) == t0) flags_l |= 1;
            const int64_t seq_last = a.varlen ? (int64_t)__ldg(a.cu + ls_l + 1) - 1 : a.L - 1;
            if (seq_last == t0 + len - 1) flags_l |= 2;
        }
        const int ng = min(32, a.nc - c0);
        for (int j0 = 0; j0 < ng; j0 += kK3Ahead) {
            float Sv[kK3Ahead];
#pragma unroll
            for (int k = 0; k < kK3Ahead; ++k)
                Sv[k] = (live && j0 + k < ng) ? S[(int64_t)(c0 + j0 + k) * cstride] : 0.f;
#pragma unroll
            for (int k = 0; k < kK3Ahead; ++k) {
                const int j = j0 + k;
                const float dec = __shfl_sync(0xffffffffu, dec_l, j & 31);
                const int fs = __shfl_sync(0xffffffffu, fs_l, j & 31);
                const int ls = __shfl_sync(0xffffffffu, ls_l, j & 31);
                const int flags = __shfl_sync(0xffffffffu, flags_l, j & 31);
                if (j < ng && live) {
                    const int64_t c = c0 + j;
                    float Ec = end_state;   // carried across the boundary
                    if (flags & 1) Ec = init ? init[(int64_t)fs * a.H * PN] : 0.f;
                    E[c * cstride] = Ec;
                    const float El =
                        (ls == fs) ? Ec : (init ? init[(int64_t)ls * a.H * PN] : 0.f);
                    end_state = dec * El + Sv[k];
                    if (fin && (flags & 2)) fin[(int64_t)ls * a.H * PN] = end_state;
                }
            }
        }
    }
}

// K5: final states of packed sequences that end inside a chunk (or are
// empty).  grid (nseq, H), block 256; threads over (p, n).
template <typename T>
__global__ void k5_seq_final(KArgs a) {
    if (status_bad(a.status)) return;
    extern __shared__ float w_smem[];
    const int s = blockIdx.x, h = blockIdx.y, g = h / a.hpg;
    const int PN = a.P * a.N;
    const int64_t sa = __ldg(a.cu + s), sb = __ldg(a.cu + s + 1);
    float *fin = a.final_states + ((int64_t)s * a.H + h) * PN;
    if (sb <= sa) {   // empty sequence: final = initial
        for (int e = threadIdx.x; e < PN; e += blockDim.x)
            fin[e] = a.init ? a.init[((int64_t)s * a.H + h) * PN + e] : 0.f;
        return;
    }
    const int64_t T_last = min64(sb - 1, a.L - 1);
    if (T_last < 0) return;
    const int c = (int)(T_last / a.Q);
    const int64_t t0 = (int64_t)c * a.Q;
    const int len = (int)min64(a.Q, a.L - t0);
    if (T_last == t0 + len - 1) return;       // ends on a chunk end: K3 wrote it
    const int fs = seg_of(a.cu, a.nseq, t0);
    const int iT = (int)(T_last - t0);
    const int j0 = (int)max64(0, sa - t0);
    const double *cs = a.cs + cs_index(a, 0, h, c);
    const double cT = cs[iT];
    for (int j = threadIdx.x; j < a.Q; j += blockDim.x) {
        float w = 0.f;
        if (j >= j0 && j <= iT)
            w = (float)exp(cT - cs[j]) * __ldg(a.dt + (t0 + j) * a.H + h);
        w_smem[j] = w;
    }
    __syncthreads();
    const float dec = (float)exp(cT);
    const float *E = (s == fs) ? a.E + st_index(a, 0, c, h)
                               : (a.init ? a.init + ((int64_t)s * a.H + h) * PN : nullptr);
    const T *x = (const T *)a.x;
    const T *B = (const T *)a.B;
    for (int e = threadIdx.x; e < PN; e += blockDim.x) {
        const int p = e / a.N, n = e % a.N;
        float acc = E ? dec * E[e] : 0.f;
        for (int j = j0; j <= iT; ++j) {
            const int64_t tok = t0 + j;
            acc += w_smem[j] * ld_as_float(x + (tok * a.H + h) * a.P + p) *
                   ld_as_float(B + (tok * a.G + g) * a.N + n);
        }
        fin[e] = acc;
    }
}

constexpr int kPT = 16;  // output columns (p) per thread in K4

// K4: grid (nc, batch, H * ceil(P/16)), block Q; thread i owns token i of
// the chunk and 16 consecutive p columns.  B (group g), the 16 x columns,
// dt and cs of the chunk are staged in shared memory kK4Tile tokens at a
// time with coalesced loads, and the entry state's 16 rows after them, so
// that the token loop reads shared memory.
constexpr int kK4Tile = 32;
constexpr int kCiRegs = 32;   // dstate up to which C_i is held in registers

template <typename T>
__global__ void k4_chunk_output(KArgs a) {
    if (status_bad(a.status)) return;
    extern __shared__ float k4s[];   // bs[tile][N] (later E rows [16][N]), xs[tile][16], dts[tile], csj[tile] (double)
    float *bs = k4s;
    float *xs = bs + kK4Tile * a.N;   // (kK4Tile >= 16: the E rows fit where B was)
    float *dts = xs + kK4Tile * kPT;
    double *csj = (double *)(dts + kK4Tile);
    const int c = blockIdx.x, r = blockIdx.y;
    const int npt = (a.P + kPT - 1) / kPT;
    const int h = blockIdx.z / npt, p0 = (blockIdx.z % npt) * kPT;
    const int g = h / a.hpg;
    const int64_t t0 = (int64_t)c * a.Q;
    const int len = (int)min64(a.Q, a.L - t0);
    const int i = threadIdx.x;
    const bool active = i < len;
    const int64_t ti = t0 + min(i, len - 1);
    const int64_t tok_i = (int64_t)r * a.L + ti;
    const int si = seq_of(a, r, ti);
    const int fs = seq_of(a, r, t0);
    const int j0 = (int)max64(0, seq_start(a, si) - t0);
    const double *cs = a.cs + cs_index(a, r, h, c);
    const double csi = cs[min(i, len - 1)];
    const T *x = (const T *)a.x;
    const T *B = (const T *)a.B;
    const T *C = (const T *)a.C;
    const T *Ci = C + (tok_i * a.G + g) * a.N;
    float acc[kPT];
#pragma unroll
    for (int q = 0; q < kPT; ++q) acc[q] = 0.f;
    // C_i in registers when the state is small (the token loop's dot
    // products then wait on nothing but shared memory)
    float ci[kCiRegs];
#pragma unroll
    for (int n = 0; n < kCiRegs; ++n) ci[n] = (n < a.N) ? ld_as_float(Ci + n) : 0.f;
    for (int jt = 0; jt < len; jt += kK4Tile) {   // the same trip count in every thread
        const int nj = min(kK4Tile, len - jt);
        __syncthreads();
        // unrolled: several loads in flight before their stores
#pragma unroll 4
        for (int idx = threadIdx.x; idx < nj * a.N; idx += blockDim.x) {
            const int jj = idx / a.N, nn = idx % a.N;
            const int64_t tok = (int64_t)r * a.L + t0 + jt + jj;
            bs[jj * a.N + nn] = ld_as_float(B + (tok * a.G + g) * a.N + nn);
        }
#pragma unroll 4
        for (int idx = threadIdx.x; idx < nj * kPT; idx += blockDim.x) {
            const int jj = idx / kPT, q = idx % kPT;
            const int64_t tok = (int64_t)r * a.L + t0 + jt + jj;
            xs[jj * kPT + q] = (p0 + q < a.P) ? ld_as_float(x + (tok * a.H + h) * a.P + p0 + q) : 0.f;
        }
        for (int jj = threadIdx.x; jj < nj; jj += blockDim.x) {
            const int64_t tok = (int64_t)r * a.L + t0 + jt + jj;
            dts[jj] = __ldg(a.dt + tok * a.H + h);
            csj[jj] = cs[jt + jj];
        }
        __syncthreads();
        if (active) {
            const int jb = max(j0, jt), je = min(i, jt + nj - 1);
            for (int j = jb; j <= je; ++j) {
                const int jj = j - jt;
                const float *Bj = bs + jj * a.N;
                float cb = 0.f;
                if (a.N <= kCiRegs) {
#pragma unroll
                    for (int n = 0; n < kCiRegs; ++n)
                        if (n < a.N) cb += ci[n] * Bj[n];
                } else {
                    for (int n = 0; n < a.N; ++n) cb += ld_as_float(Ci + n) * Bj[n];
                }
                const float w = cb * expf((float)(csi - csj[jj])) * dts[jj];
#pragma unroll
                for (int q = 0; q < kPT; ++q) acc[q] += w * xs[jj * kPT + q];
            }
        }
    }
    const int PN = a.P * a.N;
    const float *E = (si == fs) ? a.E + st_index(a, r, c, h)
                                : (a.init ? a.init + ((int64_t)si * a.H + h) * PN : nullptr);
    // E rows p0 .. p0 + 15 (every thread of the chunk reads the same ones
    // unless a packed sequence starts inside the chunk): staged when shared
    const bool shared_E = (a.varlen == false);
    if (shared_E) {
        __syncthreads();
        if (E)
            for (int idx = threadIdx.x; idx < kPT * a.N; idx += blockDim.x) {
                const int q = idx / a.N;
                bs[idx] = (p0 + q < a.P) ? E[(int64_t)(p0 + q) * a.N + idx % a.N] : 0.f;
            }
        __syncthreads();
    }
    if (!active) return;
    if (E) {
        const float dec = expf((float)csi);
#pragma unroll
        for (int q = 0; q < kPT; ++q) {
            if (p0 + q >= a.P) continue;
            const float *Ep = shared_E ? bs + q * a.N : E + (int64_t)(p0 + q) * a.N;
            float s = 0.f;
            if (a.N <= kCiRegs) {
#pragma unroll
                for (int n = 0; n < kCiRegs; ++n)
                    if (n < a.N) s += ci[n] * Ep[n];
            } else {
                for (int n = 0; n < a.N; ++n) s += ld_as_float(Ci + n) * Ep[n];
            }
            acc[q] += dec * s;
        }
    }
    const float Dh = a.D ? __ldg(a.D + h) : 0.f;
    const T *xi = x + (tok_i * a.H + h) * a.P;
    T *y = (T *)a.y + (tok_i * a.H + h) * a.P;
#pragma unroll
    for (int q = 0; q < kPT; ++q)
        if (p0 + q < a.P) st_from_float(y + p0 + q, acc[q] + Dh * ld_as_float(xi + p0 + q));
}

static_assert(kK4Tile >= kPT, "the entry state's rows reuse the B tile");
size_t k4_smem_bytes(int N) {
    return (size_t)(kK4Tile * N + kK4Tile * kPT + kK4Tile) * sizeof(float) + kK4Tile * sizeof(double);
}

struct WsLayout {
    size_t cs, S, E, total;
};

WsLayout layout(const Problem &p) {
    WsLayout w{};
    const size_t units = (size_t)p.batch * p.nc * p.H;
    size_t off = 0;
    w.cs = off; off = align_up(off + units * p.Q * sizeof(double), 256);
    w.S = off;  off = align_up(off + units * (size_t)p.P * p.N * sizeof(float), 256);
    w.E = off;  off = align_up(off + units * (size_t)p.P * p.N * sizeof(float), 256);
    w.total = off;
    return w;
}

template <typename T>
cudaError_t launch_all(const Problem &p) {
    const WsLayout w = layout(p);
    KArgs a;
    a.L = p.seqlen; a.H = p.H; a.P = p.P; a.N = p.N; a.G = p.G; a.Q = p.Q;
    a.nc = p.nc; a.nseq = p.nseq; a.hpg = p.H / p.G; a.varlen = p.cu != nullptr;
    a.x = p.x; a.dt = p.dt; a.A = p.A; a.B = p.B; a.C = p.C; a.D = p.D;
    a.init = p.init; a.cu = p.cu; a.y = p.y; a.final_states = p.final_states;
    a.status = p.status;
    a.cs = (double *)(p.ws + w.cs);
    a.S = (float *)(p.ws + w.S);
    a.E = (float *)(p.ws + w.E);
    const unsigned b = (unsigned)p.batch;
    k1_chunk_cumsum<<<dim3(p.nc, b, (p.H + 31) / 32), kK1Threads, 0, p.stream>>>(a);
    const size_t k2_smem = (size_t)(p.Q + k2_tile(p.P, p.N) * (p.P + p.N)) * sizeof(float);
    k2_chunk_state<T><<<dim3(p.nc, b, p.H), 256, k2_smem, p.stream>>>(a);
    const int PN = p.P * p.N;
    k3_state_passing<<<dim3((PN + 255) / 256, p.H, b), 256, 0, p.stream>>>(a);
    if (a.varlen && p.final_states)
        k5_seq_final<T><<<dim3(p.nseq, p.H), 256, p.Q * sizeof(float), p.stream>>>(a);
    const int npt = (p.P + kPT - 1) / kPT;
    k4_chunk_output<T><<<dim3(p.nc, b, p.H * npt), p.Q, k4_smem_bytes(p.N), p.stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t simt_workspace_bytes(const Problem &p) { return layout(p).total; }

int simt_supported(const Problem &p) {
    if (p.P < 1 || p.P > 256 || p.N < 1 || p.N > 256) return SSD_ERR_UNSUPPORTED;
    if (p.Q != 64 && p.Q != 128 && p.Q != 256) return SSD_ERR_UNSUPPORTED;   // <= kMaxQ
    if (p.dtype != SSD_F32 && p.dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

cudaError_t simt_launch(const Problem &p) {
    if (p.dtype == SSD_F32) return launch_all<float>(p);
    return launch_all<__nv_bfloat16>(p);
}

}  // namespace ssd
