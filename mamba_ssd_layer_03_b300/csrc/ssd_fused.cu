// Fused single-pass tensor-core path of the SSD forward scan (bf16 x/B/C/y,
// fp32 dt/A/D/states, headdim 64, dstate 128 or 256).
//
// The scan is the block decomposition of the semiseparable matrix
// M = L o (C B^T) (QbitAI article "新架构Mamba更新二代！", sections
// "统一SSM和注意力机制" and "Mamba-2：更强学习能力，更快训练推理"): masked quadratic
// products inside a block of tokens plus a linear recurrence of the per-head
// state across blocks.  Here the recurrence never leaves the chip.
//
// Work decomposition.  A "lane" is one sequence and the heads it carries:
// two heads of the same B/C group with dstate 128 (narrow lanes), one head
// with dstate 256 (wide lanes).  Its blocks are consecutive 128-token pieces
// of the sequence.  All blocks of all lanes are numbered lane-major and every
// CTA takes a contiguous range of that numbering (its "ticket" decides which),
// so the load is balanced to within one block.  (Split wide lanes number sets
// of lanes of one B/C group instead, and a set of CTAs shares each range, one
// lane apiece: see set_blocks.)  A CTA walks its blocks in
// order and keeps the running state of its lane in TMEM.  When a lane is
// split between two CTAs, the earlier CTA hands the state at the split point
// to the later one through global memory; every CTA processes the lane it
// hands off first and the lane it receives last, so the receiver rarely
// waits.  With few long lanes (at most half as many as SMs) every lane is
// split several ways, and waiting would chain the CTAs of a lane.  Such a
// call runs the kernel twice: a state-only first run records each CTA's
// partial state and decay where its range splits a lane, and the second run
// starts every split from those records, folded by the state-passing
// recurrence at the split's start.
//
// Per block (tokens i, j in [0, 128), heads h of the lane, state H_h[p][n]
// at the block start, cs_h = within-block cumulative sum of dt*A_h):
//   CB   = C B^T                                   tensor cores -> TMEM
//   Ys_h = C H_h^T                                  tensor cores -> TMEM acc
//   Xw_h = exp(cs_h[127] - cs_h[j]) dt_h[j] x_h[j]   CUDA cores, shared memory
//   S_h  = B^T Xw_h                                 tensor cores -> TMEM
//   H_h <- exp(cs_h[127]) H_h + S_h                 decay by CUDA cores in TMEM,
//                                                   S accumulated by the MMA
//   M_h  = CB o exp(cs_h[i] - cs_h[j]) dt_h[j] [j <= i] + D_h [i == j]
//                                                   CUDA cores, TMEM (bf16)
//   acc_h = exp(cs_h[i]) Ys_h + M_h x_h            tensor cores (A from TMEM)
//   y_h  = acc_h                                    -> x tiles (smem) -> TMA store
// Every exponent is <= 0.  Adding D_h on the diagonal of M_h folds the skip
// term D_h x_h into the same product.  The masked block is factored at
// 32-token sub-blocks: for j in an earlier sub-block with last token e,
// exp(cs_i - cs_j) = exp(cs_i - cs_e) exp(cs_e - cs_j), so only the sub-block
// holding i needs one exponential per element.
//
// Roles (512 threads, one CTA per SM).  Warps 0-3 and 4-7 are two
// warpgroups that each cover all 128 TMEM lanes (thread index within the
// warpgroup = TMEM lane).  Narrow lanes: warpgroup h holds head h for the
// scan and the state, and columns [64 h, 64 h + 64) of C B^T for the mask.
// Wide lanes: both scan the one head; warpgroup h holds state rows
// [128 h, 128 h + 128), half of each row of Xw, and the same column half of
// C B^T.  Warp 8 issues the TMA loads and writes a descriptor of each block
// (lane, tokens, flags, A, D) into a small shared-memory ring; warp 9 issues
// the MMAs; warps 12-15 (a third warpgroup over the 128 TMEM lanes) take y
// of each finished block out of TMEM, stage it in the block's x tiles and
// store it with TMA, so that the compute warps go straight on to the next
// block.  Warps 10 and 11 only complete the warpgroup of warps 8 and 9.  The
// roles hand work to each other through mbarriers; every wait is bounded in
// time and, once the call's status word records an error, falls through so
// that the kernel always finishes.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ssd_device.cuh"
#include "ssd_internal.h"
#include "ssd_wait.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;
using namespace wait;
typedef __nv_bfloat16 bf16;

constexpr int kB = 128;                    // tokens per block
constexpr int kThreads = 512;              // 8 compute warps, TMA warp, MMA warp, 2 idle, 4 epilogue
// Register split (setmaxnreg).  The kernel is launched with kRegLaunch
// registers per thread (ptxas gives 128 to 512 threads on one SM); the TMA
// and MMA warpgroup (warps 8-11) gives registers back down to kRegProducer,
// the epilogue warpgroup (warps 12-15) down to kRegEpilogue, and the two
// compute warpgroups take them up to kRegCompute.  Each SM sub-partition
// holds one warp of each warpgroup: 2 x 168 + 88 + 88 = 512 registers per
// lane, exactly its share; the host launches the kernel only when ptxas gave
// it kRegLaunch, so that the increase is always granted.
constexpr int kRegLaunch = 128;
constexpr int kRegCompute = 168;
constexpr int kRegProducer = 88;    // TMA and MMA warpgroup (warps 8-11)
constexpr int kRegEpilogue = 88;    // epilogue warpgroup (warps 12-15)
static_assert(2 * 128 * kRegCompute + 128 * kRegProducer + 128 * kRegEpilogue <= kThreads * kRegLaunch,
              "register split");
static_assert(2 * kRegCompute + kRegProducer + kRegEpilogue <= 512, "register split per sub-partition");
constexpr uint32_t kT16 = 16384;           // one 128-row x 128-byte swizzled tile
constexpr int kP = 64;                     // headdim of this path
constexpr int kStateFloats = 2 * kP * 128; // state of one lane: 2 heads x 128 or 1 head x 256

// Lane geometry.  Narrow: dstate 128, two heads of a group per lane.  Wide:
// dstate 256, one head per lane; its state's two 128-row halves go to the two
// warpgroups, which for the narrow kernel hold the two heads.
template <bool kWide>
struct Geo {
    static constexpr int N = kWide ? 256 : 128;     // dstate
    static constexpr int HL = kWide ? 1 : 2;        // heads per lane
    static constexpr int NA = N / 64;               // 64-wide n atoms of a C or B tile
    static constexpr uint32_t ACC = kP * HL;        // TMEM columns of one accumulator
    // shared-memory tiles of 16 KB: C, B, X (2 slots), Xw, H_op
    static constexpr int TILES = 2 * NA + 2 * HL + HL + 2;
};

struct FArgs {
    int64_t L;                 // tokens per batch row
    int H, G, hpg, npg, ptot;  // heads, groups, heads per group, lanes per group, lanes per sequence
    int hpl;                   // heads per lane (2 narrow, 1 wide)
    int nseq, varlen, nb_fixed, grid;
    // CTAs per lane set: the qs CTAs with tickets qs v .. qs v + qs - 1
    // take the same block range of qs lanes of one B/C group, one lane each
    // (qs = 1: ranges of single lanes)
    int qs;
    const float *dt, *A, *D, *init;
    const int32_t *cu;
    bf16 *y;
    float *final_states;
    int *status;
    int *ticket;               // ticket counter
    int *hflag;                // [grid] handoff published by ticket i
    float *hslot;              // [grid][2][P][N] handoff states
    const int *seqblk;         // [nseq + 1] prefix of blocks per sequence (varlen)
    DtTransform dtt;           // step-size transform applied as dt is read
    // Few-lane workloads split lanes between CTAs and run twice (see the
    // kernel's kPre): per ticket, the log of the decay over its part of the
    // lane it hands off, [grid][2]; and the main run's flag to fold the state
    // at a split from those records instead of waiting for a handoff.
    float *logdec;
    float *hstart;             // unused (null): the kChain main run folds the records itself
    int chain;
    // State-only runs (kPre) serve two purposes: the first run of a split
    // call, which records each split's partial state and log-decay
    // (records), and a state-only scan (states_only), which takes splits
    // like a main run does and writes the final states.
    int records;
    int states_only;
};

// One block of a CTA's walk as the compute warps need it, written by the TMA
// thread ahead of the block's loads.  Holding it in shared memory rather than
// in every compute thread's registers keeps the compute warps' loop state
// small.
enum : int {
    kSegStart = 1,    // first block of this CTA's part of the lane
    kFromSlot = 2,    // ... and the lane began in an earlier CTA (state handed off)
    kSegEnd = 4,      // last block of this CTA's part of the lane
    kFin = 8,         // ... and the lane ends here (the sequence's final state)
    kHasNext = 16,    // the next block belongs to the same lane
    kTmaY = 32        // y of the block may leave as one TMA tile: the block lies
                      // inside the sequence, or its rows past the sequence are
                      // also past the batch row (TMA drops those)
};
struct BDesc {
    int row, tok, rem;   // batch row, first token of the block in it, tokens of
                         // the sequence from tok on (may exceed the block)
    int h0, nh, s;       // first head, heads in the lane (1 or 2), sequence
    int flags;
    float A[2], D[2];    // per head of the lane (0 for a missing second head)
    float bias[2];       // dt bias of the step-size transform (0 without one)
};
constexpr int kDescRing = 4;

struct Smem {
    // [block parity][head][token]: the other warpgroup may still read the
    // previous block's values while this one writes the next block's
    float cs[2][2][kB];
    float dtv[2][2][kB];
    float vf[2][2][kB];
    float part[2][4];
    float dtn[2][2][kB];   // [block parity][head][token]: dt prefetched one block ahead
    uint64_t c_full, b_full, x_full[2];
    uint64_t cb_done, s_done, mx_done[2], c_empty, b_empty, x_empty[2], mma_fin;
    uint64_t hop_ready, xw_ready, m_ready, acc_free[2];
    uint64_t desc_full[kDescRing], desc_free[kDescRing];
    BDesc desc[kDescRing];
    uint32_t tmem;
    int ticket;
};

template <bool kWide>
constexpr size_t smem_bytes() { return 1024 + (size_t)Geo<kWide>::TILES * kT16 + sizeof(Smem); }

// ----------------------------------------------------------------------------
// lanes and blocks

struct Lane {
    int s, row, h0, nh, g, len, nb;
    int64_t t0, start;   // first token in the row; first global block index
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int64_t total_blocks(const FArgs &a) {
    return a.varlen ? (int64_t)__ldg(a.seqblk + a.nseq) * a.ptot
                    : (int64_t)a.nseq * a.ptot * a.nb_fixed;
}

__device__ __forceinline__ Lane lane_info(const FArgs &a, int64_t l) {
    Lane n;
    n.s = (int)(l / a.ptot);
    const int pair = (int)(l % a.ptot);
    n.g = pair / a.npg;
    const int k = pair % a.npg;
    n.h0 = n.g * a.hpg + a.hpl * k;
    n.nh = min(a.hpl, a.hpg - a.hpl * k);
    if (a.varlen) {
        const int c0 = __ldg(a.cu + n.s), c1 = __ldg(a.cu + n.s + 1);
        n.row = 0;
        n.t0 = c0;
        n.len = max(0, c1 - c0);
        n.nb = cdiv(n.len, kB);
        n.start = (int64_t)__ldg(a.seqblk + n.s) * a.ptot + (int64_t)pair * n.nb;
    } else {
        n.row = n.s;
        n.t0 = 0;
        n.len = (int)a.L;
        n.nb = a.nb_fixed;
        n.start = l * a.nb_fixed;
    }
    return n;
}

// Lane sets: with qs > 1 (fixed-length sequences only) the ranges are cut
// in the numbering of sets of qs lanes of one B/C group, lane-set-major; set
// v is lanes qs v .. qs v + qs - 1, and a set's block b stands for block b
// of each of its lanes.  The qs CTAs of a ticket set take the same range, one
// lane of each set apiece, so they reach the same B and C tiles at about the
// same time.  The kernel passes qs as a constant 1 where it never differs
// (narrow lanes), which leaves their index arithmetic as it was.
__device__ __forceinline__ int64_t set_blocks(const FArgs &a, int qs) { return total_blocks(a) / qs; }

// First global block of lane set v (= lane v when qs = 1).
__device__ __forceinline__ int64_t set_start(const FArgs &a, int64_t v) {
    return a.varlen ? lane_info(a, v).start : v * a.nb_fixed;
}

// Lane set that holds set-numbered block g (0 <= g < set_blocks).
__device__ __forceinline__ int64_t find_lane(const FArgs &a, int64_t g) {
    if (!a.varlen) return g / a.nb_fixed;
    int lo = 0, hi = a.nseq - 1;
    while (lo < hi) {   // largest s with seqblk[s] * ptot <= g
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)__ldg(a.seqblk + mid) * a.ptot <= g) lo = mid; else hi = mid - 1;
    }
    const int64_t base = (int64_t)__ldg(a.seqblk + lo) * a.ptot;
    const int nb = max(1, __ldg(a.seqblk + lo + 1) - __ldg(a.seqblk + lo));
    const int64_t pair = min((int64_t)a.ptot - 1, (g - base) / nb);
    return (int64_t)lo * a.ptot + pair;
}

// The blocks of one CTA: range [g0, g1) of the lane-set numbering, visited
// lane by lane in the order last lane, middle lanes, first lane.  The
// state-only runs of a split call leave out the segments whose state nobody
// reads: the recording run needs only a segment that ends inside its lane
// (the partial state the main run folds; at most one per CTA, its last lane),
// and a state-only main run only the segments that end a lane (final
// states).
enum : int { kSegAll = 0, kSegSplit = 1, kSegFinal = 2 };
struct Walk {
    int64_t g0, g1, l0, l1, nl;   // l0, l1: lane sets
    int64_t k;      // segment index in visiting order
    int qs, member; // CTAs per set; which lane of each set
    int need;       // segments visited: kSegAll, kSegSplit, kSegFinal
    Lane ln;
    int b, b_begin, b_end;
    bool valid;
};

__device__ __forceinline__ int64_t seg_lane(const Walk &w, int64_t k) {
    if (w.l0 == w.l1 || k == 0) return w.l1;
    if (k == w.nl - 1) return w.l0;
    return w.l0 + k;
}

__device__ __forceinline__ void walk_load_seg(const FArgs &a, Walk &w) {
    while (w.k < w.nl) {
        const int64_t v = seg_lane(w, w.k);
        w.ln = lane_info(a, v * w.qs + w.member);
        const int64_t v0 = a.varlen ? w.ln.start : v * a.nb_fixed;   // set_start
        const int64_t lo = max64(w.g0, v0), hi = min64(w.g1, v0 + w.ln.nb);
        const bool fin = hi == v0 + w.ln.nb;
        if (lo < hi && (w.need == kSegAll || (w.need == kSegFinal) == fin)) {
            w.b_begin = (int)(lo - v0);
            w.b_end = (int)(hi - v0);
            w.b = w.b_begin;
            w.valid = true;
            return;
        }
        ++w.k;
    }
    w.valid = false;
}

// First block (lane-set numbering) of the range of ticket set u.
__device__ __forceinline__ int64_t range_begin(const FArgs &a, int64_t u, int qs) {
    return u * set_blocks(a, qs) / (a.grid / qs);
}

// Number of blocks in the range of CTA `ticket`.
__device__ __forceinline__ int cta_blocks(const FArgs &a, int ticket, int qs) {
    const int u = ticket / qs;
    return (int)(range_begin(a, u + 1, qs) - range_begin(a, u, qs));
}

__device__ __forceinline__ void walk_init(const FArgs &a, Walk &w, int ticket, int qs, int need) {
    const int u = ticket / qs;
    w.qs = qs;
    w.need = need;
    w.member = ticket % qs;
    w.g0 = range_begin(a, u, qs);
    w.g1 = range_begin(a, u + 1, qs);
    w.valid = false;
    if (w.g0 >= w.g1) return;
    w.l0 = find_lane(a, w.g0);
    w.l1 = find_lane(a, w.g1 - 1);
    w.nl = w.l1 - w.l0 + 1;
    w.k = 0;
    walk_load_seg(a, w);
}

__device__ __forceinline__ void walk_next(const FArgs &a, Walk &w) {
    if (++w.b < w.b_end) return;
    ++w.k;
    walk_load_seg(a, w);
}

// Blocks a run visits in the range of CTA `ticket`.
__device__ __forceinline__ int run_blocks(const FArgs &a, int ticket, int qs, int need) {
    if (need == kSegAll) return cta_blocks(a, ticket, qs);
    Walk w;
    walk_init(a, w, ticket, qs, need);
    int n = 0;
    while (w.valid) {
        n += w.b_end - w.b_begin;
        ++w.k;
        walk_load_seg(a, w);
    }
    return n;
}

// ----------------------------------------------------------------------------
// small helpers

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Warpgroup register reallocation; every warp of the warpgroup executes it.
template <uint32_t N>
__device__ __forceinline__ void regs_up() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_down() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Programmatic dependent launch.  A split call's three kernels are launched
// so that the next one may start while the previous one finishes:
// launch_dependents lets the next grid be scheduled once every CTA of this
// one has issued it, and wait blocks until every grid this one depends on
// has completed and its memory operations are visible (it returns at once
// for a grid launched the ordinary way).  The earlier grids always finish
// (every wait in them is bounded), so neither can wait forever.
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Plain bounded wait used only while draining at exit.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > 50000000ull) return;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}


// Two fp32 products in one packed instruction (mul.rn.f32x2, IEEE round to
// nearest in each half: the same results as two separate multiplies).
__device__ __forceinline__ void mul2(uint32_t &a0, uint32_t &a1, float s0, float s1) {
    asm("{\n .reg .b64 x, y;\n mov.b64 x, {%0, %1};\n mov.b64 y, {%2, %3};\n"
        " mul.rn.f32x2 x, x, y;\n mov.b64 {%0, %1}, x;\n}"
        : "+r"(a0), "+r"(a1)
        : "r"(__float_as_uint(s0)), "r"(__float_as_uint(s1)));
}
__device__ __forceinline__ float2 mul2f(float2 a, float2 b) {
    uint32_t x = __float_as_uint(a.x), y = __float_as_uint(a.y);
    mul2(x, y, b.x, b.y);
    return make_float2(__uint_as_float(x), __uint_as_float(y));
}

// TMEM column of k-step kk (tokens j in [16 kk, 16 kk + 16)) of the masked
// block of head hh: M is written over C B^T in place, each 32-column fp32
// chunk of C B^T (j in [32 m, 32 m + 32)) turning into the two heads'
// 16-column bf16 pieces of the same j range.
__device__ __forceinline__ uint32_t m_col(int kk, int hh) {
    return (uint32_t)(32 * (kk >> 1) + 16 * hh + 8 * (kk & 1));
}




// Masked block, one 32-column chunk holding the row's own token, with one
// exponential per element (taken only when the chunk's total decay is too
// large for the factored form).  Reads the C B^T chunk at `taddr` and writes
// both heads' bf16 pieces over it.  All 32 lanes of the warp call it.
__device__ __noinline__ void mask_chunk_exact(uint32_t taddr, float cs0, float cs1,
                                              const float *cj0, const float *cj1,
                                              const float *dj0, const float *dj1, int lim,
                                              float dd0, float dd1) {
    uint32_t v[32];
    tmem_ld32(taddr, v);
    tmem_ld_wait();
    uint32_t pk0[16], pk1[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const int j0 = 2 * q, j1 = 2 * q + 1;
        const float c0 = __uint_as_float(v[j0]), c1 = __uint_as_float(v[j1]);
        float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
        if (j0 <= lim) {
            a0 = c0 * __expf(cs0 - cj0[j0]) * dj0[j0];
            b0 = c0 * __expf(cs1 - cj1[j0]) * dj1[j0];
        }
        if (j1 <= lim) {
            a1 = c1 * __expf(cs0 - cj0[j1]) * dj0[j1];
            b1 = c1 * __expf(cs1 - cj1[j1]) * dj1[j1];
        }
        if (j0 == lim) { a0 += dd0; b0 += dd1; }
        if (j1 == lim) { a1 += dd0; b1 += dd1; }
        pk0[q] = pack_bf16x2(a0, a1);
        pk1[q] = pack_bf16x2(b0, b1);
    }
    tmem_st16(taddr, pk0);
    tmem_st16(taddr + 16, pk1);
}

// ----------------------------------------------------------------------------
// the kernel

// kDtTransform: the step-size transform is compiled in only where a call asks
// for it, so the plain scan carries no trace of it.
// kPre: a state-only run, which skips everything that only y needs (C,
// C B^T, C H^T, the mask, M x, the epilogue).  As the first run of a
// few-lane workload (records set), each CTA runs its range from a zero state
// where a lane began in an earlier CTA and records, where its range splits a
// lane, that partial state and the log of its decay; the second run (chain
// set) starts each split lane from those records instead of waiting for the
// previous CTA.  As a state-only scan (states_only set) it takes splits like
// a main run and writes the final states.  Either way it visits only the
// segments whose state is read (see Walk).
// kChain: the main run of a split call.  A CTA whose range begins inside a
// lane folds the pre run's records into its start state itself.  (Only the
// instances that split calls launch hold that code: the single-run kernel's
// loop is sensitive to its code size and layout.)
template <bool kDtTransform, bool kWide, bool kPre, bool kChain>
__global__ void __launch_bounds__(kThreads, 1)
k_ssd_fused(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmY,
            FArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    using Gm = Geo<kWide>;
    constexpr int HL = Gm::HL, NA = Gm::NA, NS = Gm::N;
    uint8_t *sC = base;                   // [n atom][128 rows][64]        NA x 16 KB
    uint8_t *sB = sC + NA * kT16;         // [n atom][128 rows][64]        NA x 16 KB
    uint8_t *sX = sB + NA * kT16;         // [slot][head][128 rows][64]    2 HL x 16 KB
    uint8_t *sXw = sX + 2 * HL * kT16;    // [head][128 rows][64]          HL x 16 KB
    uint8_t *sH = sXw + HL * kT16;        // narrow [head][128 n][64 p], wide [256 n][64 p]: 32 KB
    Smem *sm = (Smem *)(sH + 2 * kT16);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(&sm->c_full, 1); mbar_init(&sm->b_full, 1);
        mbar_init(&sm->x_full[0], 1); mbar_init(&sm->x_full[1], 1);
        mbar_init(&sm->cb_done, 1); mbar_init(&sm->s_done, 1);
        mbar_init(&sm->mx_done[0], 1); mbar_init(&sm->mx_done[1], 1);
        mbar_init(&sm->c_empty, 1); mbar_init(&sm->b_empty, 1);
        mbar_init(&sm->x_empty[0], 1); mbar_init(&sm->x_empty[1], 1);
        mbar_init(&sm->mma_fin, 1);
        mbar_init(&sm->hop_ready, 256); mbar_init(&sm->xw_ready, 256);
        mbar_init(&sm->m_ready, 256);
        mbar_init(&sm->acc_free[0], 128); mbar_init(&sm->acc_free[1], 128);
        for (int r = 0; r < kDescRing; ++r) {
            mbar_init(&sm->desc_full[r], 1);
            mbar_init(&sm->desc_free[r], 128);
        }
        fence_mbar_init();
        prefetch_tmap(&tmX); prefetch_tmap(&tmB); prefetch_tmap(&tmC); prefetch_tmap(&tmY);
        sm->ticket = atomicAdd(a.ticket, 1);
        grid_dep_launch();
    }
    if (warp == 0) { tmem_alloc(&sm->tmem, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm->tmem;
    const uint32_t R_cb = tbase, R_H = tbase + 128;
    const int ticket = sm->ticket;
    const int qs = kWide ? a.qs : 1;   // CTAs per lane set (only split wide lanes use sets)
    const int need = !kPre ? kSegAll
                   : a.records ? kSegSplit
                   : (a.states_only && a.chain) ? kSegFinal : kSegAll;
    // packed sequences: every role reads the lane table that
    // k_fused_varlen_setup, launched just before, writes
    if (a.varlen) grid_dep_wait();
    const bool run = !status_bad(a.status);

    // Roles.  Each role's code sits inside the branch that sets its register
    // count, so that it is compiled for that count.
    if (warp >= 8) {
    if (warp < 12) regs_down<kRegProducer>(); else regs_down<kRegEpilogue>();
    if (warp == 8) {
        // ------------------------------------------------------------ TMA
        if (lane == 0 && run) {
            Walk w;
            walk_init(a, w, ticket, qs, need);
            uint32_t k = 0;
            for (; w.valid; walk_next(a, w), ++k) {
                const int tok = (int)(w.ln.t0 + (int64_t)w.b * kB);
                const int slot = k & 1;
                {
                    // slot k % 4 last described block k - 4: the compute warps
                    // were done with it before they made block k - 2's H
                    // operand and Xw ready, which the c_empty and b_empty
                    // completions waited for in the previous iteration
                    // follow; the epilogue warps release it themselves
                    if (!kPre && k >= kDescRing)
                        fwait(&sm->desc_free[k % kDescRing], ((k / kDescRing) + 1) & 1, a.status);
                    BDesc &d = sm->desc[k % kDescRing];
                    const Lane &ln = w.ln;
                    const int i0 = w.b * kB;
                    d.row = ln.row;
                    d.tok = tok;
                    d.rem = ln.len - i0;
                    d.h0 = ln.h0;
                    d.nh = ln.nh;
                    d.s = ln.s;
                    d.flags = (w.b == w.b_begin ? kSegStart : 0) | (w.b_begin > 0 ? kFromSlot : 0) |
                              (w.b + 1 == w.b_end ? kSegEnd : 0) | (w.b_end == ln.nb ? kFin : 0) |
                              (w.b + 1 < w.b_end ? kHasNext : 0) |
                              ((i0 + kB <= ln.len || ln.t0 + ln.len >= a.L) ? kTmaY : 0);
                    d.A[0] = __ldg(a.A + ln.h0);
                    d.A[1] = ln.nh > 1 ? __ldg(a.A + ln.h0 + 1) : 0.f;
                    d.D[0] = a.D ? __ldg(a.D + ln.h0) : 0.f;
                    d.D[1] = (a.D && ln.nh > 1) ? __ldg(a.D + ln.h0 + 1) : 0.f;
                    d.bias[0] = a.dtt.bias ? __ldg(a.dtt.bias + ln.h0) : 0.f;
                    d.bias[1] = (a.dtt.bias && ln.nh > 1) ? __ldg(a.dtt.bias + ln.h0 + 1) : 0.f;
                    mbar_arrive(&sm->desc_full[k % kDescRing]);
                }
                if (k >= 2) fwait(&sm->x_empty[slot], ((k >> 1) + 1) & 1, a.status);
                for (int s = 0; s < HL; ++s)
                    tma_load_4d(sX + (size_t)(slot * HL + s) * kT16, &tmX, &sm->x_full[slot], 0,
                                w.ln.h0 + s, tok, w.ln.row);
                mbar_arrive_expect_tx(&sm->x_full[slot], HL * kT16);
                if (!kPre) {
                    if (k >= 1) fwait(&sm->c_empty, (k - 1) & 1, a.status);
                    for (int nb = 0; nb < NA; ++nb)
                        tma_load_4d(sC + nb * kT16, &tmC, &sm->c_full, nb * 64, w.ln.g, tok, w.ln.row);
                    mbar_arrive_expect_tx(&sm->c_full, NA * kT16);
                }
                if (kPre) {
                    // the pre run loads no C: B takes two slots, the second in
                    // C's tiles with C's barriers, and is fetched a block ahead
                    uint64_t *bf = slot ? &sm->c_full : &sm->b_full;
                    if (k >= 2) fwait(slot ? &sm->c_empty : &sm->b_empty, ((k >> 1) + 1) & 1, a.status);
                    for (int nb = 0; nb < NA; ++nb)
                        tma_load_4d((slot ? sC : sB) + nb * kT16, &tmB, bf, nb * 64, w.ln.g, tok, w.ln.row);
                    mbar_arrive_expect_tx(bf, NA * kT16);
                } else {
                    if (k >= 1) fwait(&sm->b_empty, (k - 1) & 1, a.status);
                    for (int nb = 0; nb < NA; ++nb)
                        tma_load_4d(sB + nb * kT16, &tmB, &sm->b_full, nb * 64, w.ln.g, tok, w.ln.row);
                    mbar_arrive_expect_tx(&sm->b_full, NA * kT16);
                }
            }
            // let every copy this thread started land before the CTA exits
            if (k >= 1) {
                if (kPre) {
                    drain_wait((k - 1) & 1 ? &sm->c_full : &sm->b_full, ((k - 1) >> 1) & 1);
                } else {
                    drain_wait(&sm->c_full, (k - 1) & 1);
                    drain_wait(&sm->b_full, (k - 1) & 1);
                }
                drain_wait(&sm->x_full[(k - 1) & 1], ((k - 1) >> 1) & 1);
            }
            if (k >= 2) {
                if (kPre) drain_wait(k & 1 ? &sm->c_full : &sm->b_full, ((k - 2) >> 1) & 1);
                drain_wait(&sm->x_full[k & 1], ((k - 2) >> 1) & 1);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && run) {
            // Ys and S have N = 64 per head: 128 with two heads, 64 with one
            const uint32_t id_cb = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t id_ys = idesc_bf16_f32(128, 64 * HL, 0, 1);
            const uint32_t id_s = idesc_bf16_f32(128, 64 * HL, 1, 1);
            const uint32_t id_mx = idesc_bf16_f32(128, 64, 0, 1);
            const uint32_t sc = smem_u32(sC), sbb = smem_u32(sB), sxw = smem_u32(sXw),
                           sh = smem_u32(sH), sx = smem_u32(sX);
            const uint32_t nblk = (uint32_t)run_blocks(a, ticket, qs, need);
            for (uint32_t k = 0; k < nblk; ++k) {
                const int slot = k & 1;
                const uint32_t R_acc = tbase + 256 + Gm::ACC * slot;
                if (kPre) {
                    // state only: H <- (decay H, in TMEM once hop_ready) + B^T Xw,
                    // B from its slot (the second one in C's tiles)
                    fwait(slot ? &sm->c_full : &sm->b_full, (k >> 1) & 1, a.status);
                    const uint32_t sbs = slot ? sc : sbb;
                    fwait(&sm->hop_ready, k & 1, a.status);
                    fwait(&sm->xw_ready, k & 1, a.status);
                    tc_fence_after();
#pragma unroll
                    for (int q = 0; q < (kWide ? 2 : 1); ++q)
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(R_H + 64 * q,
                                   smem_desc(sbs + 2 * q * kT16 + kk * 2048, kT16, 1024, kSwizzle128B),
                                   smem_desc(sxw + kk * 2048, kT16, 1024, kSwizzle128B), id_s, 1);
                    mma_commit(&sm->s_done);
                    mma_commit(slot ? &sm->c_empty : &sm->b_empty);
                    mma_commit(&sm->x_empty[slot]);   // x was read by Xw, before xw_ready
                    continue;
                }
                fwait(&sm->c_full, k & 1, a.status);
                fwait(&sm->b_full, k & 1, a.status);
                tc_fence_after();
                // CB = C B^T (over the previous block's M, read by its last product)
#pragma unroll
                for (int kk = 0; kk < 4 * NA; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * kT16 + (uint32_t)(kk & 3) * 32;
                    mma_ss(R_cb, smem_desc(sc + off, 16, 1024, kSwizzle128B),
                           smem_desc(sbb + off, 16, 1024, kSwizzle128B), id_cb, kk > 0);
                }
                // Ys = C H^T (narrow: both heads stacked along N; wide: K = 256
                // over H_op's 256 n rows)
                fwait(&sm->hop_ready, k & 1, a.status);
                if (k >= 2) fwait(&sm->acc_free[slot], ((k >> 1) + 1) & 1, a.status);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4 * NA; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * kT16 + (uint32_t)(kk & 3) * 32;
                    mma_ss(R_acc, smem_desc(sc + off, 16, 1024, kSwizzle128B),
                           smem_desc(sh + kk * 2048, kT16, 1024, kSwizzle128B), id_ys, kk > 0);
                }
                mma_commit(&sm->cb_done);
                mma_commit(&sm->c_empty);
                // S = B^T Xw (rows n, columns (head, p))
                fwait(&sm->xw_ready, k & 1, a.status);
                fwait(&sm->x_full[slot], (k >> 1) & 1, a.status);
                tc_fence_after();
                // H <- (decay H, already in TMEM) + B^T Xw; wide: one product
                // per 128-row half of n (B tile atoms 2q, 2q + 1)
#pragma unroll
                for (int q = 0; q < (kWide ? 2 : 1); ++q)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(R_H + 64 * q,
                               smem_desc(sbb + 2 * q * kT16 + kk * 2048, kT16, 1024, kSwizzle128B),
                               smem_desc(sxw + kk * 2048, kT16, 1024, kSwizzle128B), id_s, 1);
                mma_commit(&sm->s_done);
                mma_commit(&sm->b_empty);
                // acc_h += M_h x_h (M from TMEM)
                fwait(&sm->m_ready, k & 1, a.status);
                tc_fence_after();
#pragma unroll
                for (int hh = 0; hh < HL; ++hh)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(R_acc + hh * 64, R_cb + m_col(kk, hh),
                               smem_desc(sx + (uint32_t)(slot * HL + hh) * kT16 + kk * 2048, kT16,
                                         1024, kSwizzle128B),
                               id_mx, 1);
                mma_commit(&sm->mx_done[slot]);   // (the epilogue frees the x slot)
            }
            // every MMA this thread issued has completed before TMEM is freed
            mma_commit(&sm->mma_fin);
            drain_wait(&sm->mma_fin, 0);
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ epilogue
        // y of block k from the accumulator, off the compute warps' path.
        // Thread t is TMEM lane t, i.e. token row t of the block.  The rows
        // are staged, bf16 and swizzled, in the block's own x tiles: the M x
        // product was their last reader, so they are free once it has
        // landed, and they have y's shape and layout.  Thread 0 stores each
        // head's tile with TMA and, once the store has read them, hands the
        // x slot back to the TMA warp.  A block whose rows past the sequence
        // belong to another packed sequence writes its rows one by one
        // instead.
        if (!kPre && run) {
            const int t = tid & 127;
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t nblk = (uint32_t)run_blocks(a, ticket, qs, need);
            for (uint32_t k = 0; k < nblk; ++k) {
                const int slot = k & 1;
                fwait(&sm->desc_full[k % kDescRing], (k / kDescRing) & 1, a.status);
                const BDesc &dk = sm->desc[k % kDescRing];   // released after the store
                const bool tma_y = (dk.flags & kTmaY) != 0;
                fwait(&sm->mx_done[slot], (k >> 1) & 1, a.status);
                tc_fence_after();
                const uint32_t R_acc = tbase + 256 + Gm::ACC * slot;
#pragma unroll 1
                for (int hh = 0; hh < HL; ++hh) {
                    uint4 *dst = tma_y
                        ? (uint4 *)(sX + (size_t)(slot * HL + hh) * kT16 + t * 128)
                        : (t < dk.rem && hh < dk.nh)
                            ? (uint4 *)(a.y + (((int64_t)dk.row * a.L + dk.tok + t) * a.H + dk.h0 + hh) * kP)
                            : nullptr;
#pragma unroll 1
                    for (int q = 0; q < 4; ++q) {   // 16 columns (two 16-byte chunks) at a time
                        uint32_t v[16];
                        tmem_ld16(R_acc + lane_off + hh * 64 + q * 16, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const uint4 pk = make_uint4(
                                pack_bf16x2(__uint_as_float(v[8 * c]), __uint_as_float(v[8 * c + 1])),
                                pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3])),
                                pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5])),
                                pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7])));
                            // staged rows are swizzled like x (16-byte chunk j of
                            // row t at chunk j ^ (t & 7)); direct rows are plain
                            if (tma_y) dst[(2 * q + c) ^ (t & 7)] = pk;
                            else if (dst) dst[2 * q + c] = pk;
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&sm->acc_free[slot]);
                if (tma_y) fence_proxy_async_smem();
                named_bar(4, 128);   // every row of the staged tiles is written
                if (t == 0) {
                    if (tma_y) {
                        for (int hh = 0; hh < dk.nh; ++hh)
                            tma_store_4d(&tmY, sX + (size_t)(slot * HL + hh) * kT16, 0, dk.h0 + hh,
                                         dk.tok, dk.row);
                        tma_store_commit();
                    }
                }
                mbar_arrive(&sm->desc_free[k % kDescRing]);
                if (t == 0) {
                    if (tma_y) tma_store_wait_read0();
                    mbar_arrive(&sm->x_empty[slot]);
                }
            }
            if (t == 0) tma_store_wait0();
        }
    }
    } else {
    regs_up<kRegCompute>();
    if (run) {
        // ------------------------------------------------------------ compute
        // Warpgroup h: thread t is TMEM lane t, i.e. token row i = t of the
        // block for C B^T, M and the outputs, and state row n = t for H.  For
        // the state, the scan and the outputs the warpgroup works on head h of
        // the lane; for the masked block on C B^T columns [64 h, 64 h + 64)
        // for both heads.
        // Wide lanes (one head, dstate 256): both warpgroups scan the lane's
        // head; warpgroup h holds state rows n in [128 h, 128 h + 128), Xw and
        // y chunks [4 h, 4 h + 4) of each row, and acc columns [32 h, 32 h + 32).
        const int h = warp >> 2;
        const int hs = kWide ? 0 : h;     // head of the lane this warpgroup scans
        const int t = tid & 127;
        const int wq = warp & 3;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const int bar_wg = 1 + h;

        // dt of this thread's token and head in the block of `dk` starting
        // `off` tokens later, copied into dtn[par][h][t] asynchronously
        // (cp.async: barriers do not wait for it); zero outside the sequence
        // or the lane's heads
        auto prefetch_dt = [&](const BDesc &dk, int off, int par) {
            float *dst = &sm->dtn[par][h][t];
            if (hs < dk.nh && off + t < dk.rem) {
                const float *src = a.dt + ((int64_t)dk.row * a.L + dk.tok + off + t) * a.H + dk.h0 + hs;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)),
                             "l"(src) : "memory");
            } else {
                *dst = 0.f;
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        bool have_next = false;
        float ldsum = 0.f;         // pre run: sum of cs_last over the lane's blocks here
        const uint32_t nblk = (uint32_t)run_blocks(a, ticket, qs, need);
        // the main run of a split call starts splits from the pre run's
        // records: wait for the pre run to complete
        grid_dep_wait();

        for (uint32_t k = 0;; ++k) {
            const bool have = k < nblk;
            if (have) {
                fwait(&sm->desc_full[k % kDescRing], (k / kDescRing) & 1, a.status);
                const BDesc &dk = sm->desc[k % kDescRing];
                const int flags = dk.flags;
                const bool hv = hs < dk.nh;
                const int head = dk.h0 + (hv ? hs : 0);
                const int slot = k & 1;
                const uint32_t R_acc = tbase + 256 + Gm::ACC * slot;
                const bool seg_start = (flags & kSegStart) != 0;

                // (d) H_k -> H_op (bf16, operand of C H^T), then H <- decay H_k
                //     in TMEM (after the scan), ready for the S product to
                //     accumulate on.  A lane's first block takes H_k from the
                //     initial state (or the previous CTA's handoff) through TMEM.
                //     Narrow lanes do the first part before the scan, so that
                //     C H^T runs while the scan does; wide lanes after it (their
                //     S product of the previous block, which H_k waits for, and
                //     their larger C H^T are better left behind the scan:
                //     measured).
                auto state_in = [&]() {
                    if (seg_start) {
                        // A lane split at this CTA's range start begins from: zero
                        // (pre run); the fold of the earlier CTAs' pre-run records
                        // (main run of a few-lane workload); or the previous CTA's
                        // handoff.
                        const float *src = nullptr;
                        const int n_row = kWide ? 128 * h + t : t;   // this thread's state row
                        int uf = 0, ue = 0;   // later records to fold in: tickets uf, uf + qs, ... < ue
                        if (flags & kFromSlot) {
                            if (kPre && a.records) {
                            } else if (a.chain) {
                                if constexpr (kPre || kChain) {
                                    // The state-passing recurrence across the splits,
                                    // over the pre run's records (complete: the compute
                                    // warps waited for the pre run).  The lane's earlier
                                    // ranges are those of tickets qs apart; ticket set
                                    // u0's range holds the lane's first block, so its
                                    // record is the state up to its end, and each later
                                    // range's adds H <- exp(logdec_u) H + S_u.
                                    const int us = ticket / qs, mb = ticket % qs, vg = a.grid / qs;
                                    const int64_t TS = set_blocks(a, qs);
                                    const int64_t v0 = set_start(a, find_lane(a, (int64_t)us * TS / vg));
                                    // the last ticket set whose range begins at or before
                                    // the lane start: u TS / vg <= v0 (rounded down)
                                    // exactly when u <= ((v0 + 1) vg - 1) / TS
                                    const int u0 = (int)min64(us - 1, ((v0 + 1) * vg - 1) / TS);
                                    src = a.hslot + (size_t)(u0 * qs + mb) * kStateFloats + hs * kP * NS;
                                    uf = (u0 + 1) * qs + mb;
                                    ue = ticket;
                                } else {
                                    // not taken: split calls launch the kChain instance
                                    src = a.hstart + (size_t)ticket * kStateFloats + hs * kP * NS;
                                }
                            } else {
                                // the previous range of this lane: ticket - qs
                                wait_flag(a.hflag + (ticket - qs), a.status);
                                src = a.hslot + (size_t)(ticket - qs) * kStateFloats + hs * kP * NS;
                            }
                        } else if (a.init && hv) {
                            src = a.init + ((int64_t)dk.s * a.H + head) * kP * NS;
                        }
                        if (!hv) src = nullptr;
                        // 16 loads in flight per round: the state's 64 columns
                        // arrive in a few memory latencies, not sixteen
                        if (src) {
                            for (int c16 = 0; c16 < kP / 16; ++c16) {
                                uint32_t r[16];
#pragma unroll
                                for (int q = 0; q < 16; ++q)
                                    r[q] = __float_as_uint(__ldcg(src + (c16 * 16 + q) * NS + n_row));
                                if constexpr (kPre || kChain) {
#pragma unroll 1
                                    for (int u = uf; u < ue; u += qs) {
                                        const float d = __expf(__ldcg(a.logdec + 2 * u + hs));
                                        const float *su = a.hslot + (size_t)u * kStateFloats + hs * kP * NS;
#pragma unroll
                                        for (int q = 0; q < 16; ++q)
                                            r[q] = __float_as_uint(fmaf(d, __uint_as_float(r[q]),
                                                                        __ldcg(su + (c16 * 16 + q) * NS + n_row)));
                                    }
                                }
                                tmem_st16(R_H + lane_off + h * 64 + c16 * 16, r);
                            }
                        } else {
                            uint32_t r[16];
#pragma unroll
                            for (int q = 0; q < 16; ++q) r[q] = 0u;
#pragma unroll 1
                            for (int c16 = 0; c16 < kP / 16; ++c16) tmem_st16(R_H + lane_off + h * 64 + c16 * 16, r);
                        }
                        tmem_st_wait();
                    } else {
                        fwait(&sm->s_done, (k - 1) & 1, a.status);
                        tc_fence_after();
                    }
                };
                // H_k of this thread's state row -> H_op, then C H^T may
                // start.  Narrow lanes publish it before the scan and keep H_k
                // in registers over it; wide lanes, whose C H^T reads twice the
                // operands, after it (measured: the early product slows their
                // scan more than it gains).
                uint32_t hv2[2][32];
                auto publish_hop = [&]() {
                    tmem_ld32(R_H + lane_off + h * 64, hv2[0]);
                    tmem_ld32(R_H + lane_off + h * 64 + 32, hv2[1]);
                    tmem_ld_wait();
                    uint8_t *hrow = sH + h * kT16 + t * 128;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            if (!kPre) *(uint4 *)(hrow + (((half * 4 + c) ^ (t & 7)) << 4)) = make_uint4(
                                pack_bf16x2(__uint_as_float(hv2[half][8 * c]), __uint_as_float(hv2[half][8 * c + 1])),
                                pack_bf16x2(__uint_as_float(hv2[half][8 * c + 2]), __uint_as_float(hv2[half][8 * c + 3])),
                                pack_bf16x2(__uint_as_float(hv2[half][8 * c + 4]), __uint_as_float(hv2[half][8 * c + 5])),
                                pack_bf16x2(__uint_as_float(hv2[half][8 * c + 6]), __uint_as_float(hv2[half][8 * c + 7])));
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&sm->hop_ready);
                };
                if (!kWide) {
                    state_in();
                    publish_hop();
                }

                // (a) dt and the within-block cumulative decay cs of head h
                if (!have_next) prefetch_dt(dk, 0, slot);
                asm volatile("cp.async.wait_all;" ::: "memory");
                float d = sm->dtn[slot][h][t];
                if (kDtTransform && hv && t < dk.rem)
                    d = dt_apply(d, dk.bias[hs], a.dtt.softplus, a.dtt.lo, a.dtt.hi);
                have_next = (flags & kHasNext) != 0;
                if (have_next) prefetch_dt(dk, kB, slot ^ 1);
                float incl = d * dk.A[hs];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float v = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += v;
                }
                if (lane == 31) sm->part[h][wq] = incl;
                named_bar(bar_wg, 128);
                const float p0 = sm->part[h][0], p1 = sm->part[h][1], p2 = sm->part[h][2],
                            p3 = sm->part[h][3];
                incl += (wq > 0 ? p0 : 0.f) + (wq > 1 ? p1 : 0.f) + (wq > 2 ? p2 : 0.f);
                const float cs_last = ((p0 + p1) + p2) + p3;
                const float sub_end = __shfl_sync(0xffffffffu, incl, 31);
                if (!kPre) {   // for the mask
                    sm->cs[slot][h][t] = incl;
                    sm->dtv[slot][h][t] = d;
                    sm->vf[slot][h][t] = __expf(sub_end - incl) * d;
                }
                const float w_t = __expf(fminf(cs_last - incl, 0.f)) * d;
                const float decay = __expf(cs_last);
                if (kWide) {
                    state_in();
                    publish_hop();
                }

                if (kPre && seg_start) ldsum = 0.f;
                if (kPre) ldsum += cs_last;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
#pragma unroll
                    for (int q = 0; q < 32; q += 2) mul2(hv2[half][q], hv2[half][q + 1], decay, decay);
                    tmem_st32(R_H + lane_off + h * 64 + half * 32, hv2[half]);
                }

                // (b) Xw_h row t = w_t x_h row t, one packed bf16 x bf16 multiply
                //     per pair (w_t rounded to bf16 first: relative error 2^-8 on
                //     Xw, against 2^-9 for a product in fp32); visit the row's
                //     eight 16-byte chunks starting at a different one in each of
                //     8 lanes
                fwait(&sm->x_full[slot], (k >> 1) & 1, a.status);
                {
                    const uint4 *src = (const uint4 *)(sX + (size_t)(slot * HL + hs) * kT16 + t * 128);
                    uint4 *dst = (uint4 *)(sXw + hs * kT16 + t * 128);
                    const __nv_bfloat162 w2 = __floats2bfloat162_rn(w_t, w_t);
#pragma unroll
                    for (int c = kWide ? 4 * h : 0; c < (kWide ? 4 * h + 4 : 8); ++c) {
                        const int pc = c ^ (t & 7);
                        const uint4 u = src[pc];
                        uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162 *>(&ww[q]);
                            b2 = __hmul2(b2, w2);
                            ww[q] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        dst[pc] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
                    }
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&sm->xw_ready);

                if (!kPre) {   // everything below only serves y
                // (e) masked block, in place over C B^T: this warpgroup turns
                //     columns j in [64 h, 64 h + 64) into both heads' M pieces;
                //     then acc_h *= exp(cs_h[i]) for head h
                fwait(&sm->cb_done, k & 1, a.status);
                named_bar(3, 256);        // cs, dtv, vf of both heads are visible
                tc_fence_after();
                {
                    const int i = t;
                    const int ib = wq;
                    const float(*cs)[kB] = sm->cs[slot];
                    const float(*vfs)[kB] = sm->vf[slot];
                    const float(*dts)[kB] = sm->dtv[slot];
                    const float cs0 = cs[0][i], cs1 = cs[1][i];
#pragma unroll 1
                    for (int mm = 0; mm < 2; ++mm) {
                        const int m = 2 * h + mm;
                        uint32_t pk0[16], pk1[16];
                        if (m > ib) {
#pragma unroll
                            for (int q = 0; q < 16; ++q) { pk0[q] = 0u; pk1[q] = 0u; }
                        } else {
                            uint32_t v[32];
                            const float *cj0 = cs[0] + m * 32, *cj1 = cs[1] + m * 32;
                            const float end0 = cj0[31], end1 = cj1[31];
                            // Sub-blocks before i's: j <= i for all of them;
                            // exp(cs_i - cs_j) = exp(cs_i - cs_end) exp(cs_end - cs_j),
                            // both factors <= 1.  i's own sub-block: the same
                            // factors, the first in [1, e^R] and the second in
                            // [e^-R, 1] with R the sub-block's total decay, used
                            // while R < 80; otherwise one exponential per element.
                            const bool own = (m == ib);
                            const int lim = own ? (i & 31) : 31;
                            const float ref0 = (m == 0) ? 0.f : cs[0][m * 32 - 1];
                            const float ref1 = (m == 0) ? 0.f : cs[1][m * 32 - 1];
                            const bool fast = !own || ((ref0 - end0 < 80.f) && (ref1 - end1 < 80.f));
                            const float dd0 = own ? dk.D[0] : 0.f, dd1 = own ? dk.D[1] : 0.f;
                            if (fast) {
                                tmem_ld32(R_cb + lane_off + m * 32, v);
                                tmem_ld_wait();
                                const float u0 = __expf(cs0 - end0), u1 = __expf(cs1 - end1);
                                const float *vf0 = vfs[0] + m * 32, *vf1 = vfs[1] + m * 32;
                                if (!own) {
                                    // a chunk wholly below the diagonal: no causal
                                    // or diagonal test per element
#pragma unroll
                                    for (int q = 0; q < 16; ++q) {
                                        const float2 f0 = *(const float2 *)(vf0 + 2 * q);
                                        const float2 cc = make_float2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
                                        const float2 ca = mul2f(mul2f(cc, make_float2(u0, u0)), f0);
                                        pk0[q] = pack_bf16x2(ca.x, ca.y);
                                        if (!kWide) {
                                            const float2 f1 = *(const float2 *)(vf1 + 2 * q);
                                            const float2 cb = mul2f(mul2f(cc, make_float2(u1, u1)), f1);
                                            pk1[q] = pack_bf16x2(cb.x, cb.y);
                                        }
                                    }
                                } else
#pragma unroll
                                for (int q = 0; q < 16; ++q) {
                                    const int j0 = 2 * q, j1 = 2 * q + 1;
                                    const float c0 = (j0 <= lim) ? __uint_as_float(v[j0]) : 0.f;
                                    const float c1 = (j1 <= lim) ? __uint_as_float(v[j1]) : 0.f;
                                    const float2 f0 = *(const float2 *)(vf0 + j0);
                                    const float2 f1 = *(const float2 *)(vf1 + j0);
                                    const float2 ca = mul2f(mul2f(make_float2(c0, c1), make_float2(u0, u0)), f0);
                                    float a0 = ca.x, a1 = ca.y;
                                    if (j0 == lim && own) a0 += dd0;
                                    if (j1 == lim && own) a1 += dd0;
                                    pk0[q] = pack_bf16x2(a0, a1);
                                    if (!kWide) {   // wide lanes have one head
                                        const float2 cb = mul2f(mul2f(make_float2(c0, c1), make_float2(u1, u1)), f1);
                                        float b0 = cb.x, b1 = cb.y;
                                        if (j0 == lim && own) b0 += dd1;
                                        if (j1 == lim && own) b1 += dd1;
                                        pk1[q] = pack_bf16x2(b0, b1);
                                    }
                                }
                            } else {
                                mask_chunk_exact(R_cb + lane_off + m * 32, cs0, cs1, cj0, cj1,
                                                 dts[0] + m * 32, dts[1] + m * 32, lim, dd0, dd1);
                                continue;
                            }
                        }
                        tmem_st16(R_cb + lane_off + m * 32, pk0);
                        if (!kWide) tmem_st16(R_cb + lane_off + m * 32 + 16, pk1);
                    }
                    // acc_h *= exp(cs_h[i]): narrow, head h's 64 columns; wide,
                    // columns [32 h, 32 h + 32) of the one head
                    const float e = __expf(h == 0 || kWide ? cs0 : cs1);
                    {
                        // both halves' loads in flight before one wait
                        uint32_t v[2][32];
#pragma unroll
                        for (int half = 0; half < (kWide ? 1 : 2); ++half)
                            tmem_ld32(R_acc + lane_off + (kWide ? 32 * h : 64 * h + 32 * half), v[half]);
                        tmem_ld_wait();
#pragma unroll
                        for (int half = 0; half < (kWide ? 1 : 2); ++half) {
#pragma unroll
                            for (int q = 0; q < 32; q += 2) mul2(v[half][q], v[half][q + 1], e, e);
                            tmem_st32(R_acc + lane_off + (kWide ? 32 * h : 64 * h + 32 * half), v[half]);
                        }
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(&sm->m_ready);

                }
            }
            if (!have) break;

            // end of this CTA's part of the lane: the state after the block
            const BDesc &dk = sm->desc[k % kDescRing];
            const int flags = dk.flags;
            if (flags & kSegEnd) {
                const bool hv = hs < dk.nh;
                const int head = dk.h0 + (hv ? hs : 0);
                const bool fin = (flags & kFin) != 0;
                const int n_row = kWide ? 128 * h + t : t;   // this thread's state row
                // S of this block has landed in H.  (This wait also covers the
                // next block: a lane's first block here reloads H in TMEM and
                // rewrites Xw, which S of this block reads.)
                fwait(&sm->s_done, k & 1, a.status);
                tc_fence_after();
                float *dst = nullptr;
                if (fin) {
                    // the recording run leaves final states to the main run
                    if ((!kPre || a.states_only) && a.final_states && hv)
                        dst = a.final_states + ((int64_t)dk.s * a.H + head) * kP * NS;
                } else if (kPre && a.records) {
                    // the record the main run folds
                    dst = a.hslot + (size_t)ticket * kStateFloats + hs * kP * NS;
                    if (t == 0 && (!kWide || h == 0)) a.logdec[2 * ticket + hs] = ldsum;
                } else if (!a.chain) {
                    // handoff to the next CTA
                    dst = a.hslot + (size_t)ticket * kStateFloats + hs * kP * NS;
                }
#pragma unroll 1
                for (int c16 = 0; c16 < kP / 16; ++c16) {
                    uint32_t r[16];
                    tmem_ld16(R_H + lane_off + h * 64 + c16 * 16, r);
                    tmem_ld_wait();
                    if (dst) {
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            __stcg(dst + (c16 * 16 + q) * NS + n_row, __uint_as_float(r[q]));
                    }
                }
                tc_fence_before();
                if (!fin) {
                    __threadfence();
                    // all 256 compute threads have stored: publish
                    named_bar(3, 256);
                    if (tid == 0) st_release_i(a.hflag + ticket, 1);
                }
            }
        }
    }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// Varlen set-up: blocks per sequence (exclusive prefix) and the final states
// of empty sequences (their initial states).  One CTA.
__global__ void k_fused_varlen_setup(FArgs a, int P, int N) {
    if (threadIdx.x == 0) grid_dep_launch();   // the scan may be scheduled; it waits for this
    if (status_bad(a.status)) return;
    __shared__ int carry;
    __shared__ int warp_sum[32];
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    int *seqblk = const_cast<int *>(a.seqblk);
    for (int s0 = 0; s0 < a.nseq; s0 += blockDim.x) {
        const int s = s0 + threadIdx.x;
        int nb = 0;
        if (s < a.nseq) nb = cdiv(max(0, __ldg(a.cu + s + 1) - __ldg(a.cu + s)), kB);
        // block-wide exclusive scan of nb
        const int ln = threadIdx.x & 31, wp = threadIdx.x >> 5;
        int v = nb;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, v, off);
            if (ln >= off) v += o;
        }
        if (ln == 31) warp_sum[wp] = v;
        __syncthreads();
        int pre = carry;
        for (int q = 0; q < wp; ++q) pre += warp_sum[q];
        if (s < a.nseq) seqblk[s] = pre + v - nb;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = pre + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) seqblk[a.nseq] = carry;
    // empty sequences: final = initial (or zero)
    if (a.final_states) {
        const int PN = P * N;
        for (int s = 0; s < a.nseq; ++s) {
            if (__ldg(a.cu + s + 1) > __ldg(a.cu + s)) continue;
            for (int e = threadIdx.x; e < a.H * PN; e += blockDim.x) {
                const int64_t idx = (int64_t)s * a.H * PN + e;
                a.final_states[idx] = a.init ? a.init[idx] : 0.f;
            }
        }
    }
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

// bf16 map of a 4-d tensor, dims[0] innermost; 128-byte swizzle.
bool make_map4(CUtensorMap *m, const void *ptr, const uint64_t *dims, const uint32_t *box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gd[4], gs[3];
    cuuint32_t bx[4], es[4];
    uint64_t stride = 2;
    for (int i = 0; i < 4; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i > 0) gs[i - 1] = stride;
        stride *= dims[i];
    }
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), gd, gs, bx, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

// When splitting lanes between CTAs pays.  A split call runs three kernels,
// which costs a fixed ~15 us, and the state-only pre run adds about a third
// of a block's time per block.  Measured on 24 lanes of 16 blocks: 4 blocks
// per CTA 56 us against 70 us whole; on 24 lanes of 8 blocks every split was
// slower than the whole lanes.
constexpr int64_t kChainMinLaneBlocks = 16;   // blocks per lane
constexpr int64_t kChainMinCtaBlocks = 4;     // blocks per CTA

struct FLayout {
    size_t hdr, slots, logdec, seqblk, total;
    int grid;
    bool chain;   // few lanes: split them between CTAs, pre run + main run
    int qs;       // CTAs per lane set
};

// Heads per lane: two of a group with dstate 128, one with dstate 256.
int heads_per_lane(const Problem &p) { return p.N == 256 ? 1 : 2; }

int64_t lanes_per_seq(const Problem &p) {
    const int hpg = p.H / p.G, hpl = heads_per_lane(p);
    return (int64_t)p.G * ((hpg + hpl - 1) / hpl);
}

// Grid: at most one CTA per SM, and never more CTAs than blocks (so that no
// range is empty).  Without packing, lanes >= grid also keeps every range at
// least one lane long.  The workspace always has room for one handoff slot
// per SM, so its size does not depend on cu_seqlens.
FLayout fused_layout(const Problem &p) {
    FLayout w{};
    w.qs = 1;
    const int64_t ptot = lanes_per_seq(p);
    const int64_t sms = sm_count();
    const int64_t nb = (p.seqlen + kB - 1) / kB;
    int64_t grid;
    if (p.cu) {
        grid = min64(sms, ptot * nb);
    } else if ((int64_t)p.nseq * ptot * 2 <= sms && nb >= kChainMinLaneBlocks) {
        // At most half as many lanes as SMs, and long enough: lanes are split
        // between CTAs, which start from the pre run's records.
        grid = min64(sms, (int64_t)p.nseq * ptot * nb / kChainMinCtaBlocks);
        w.chain = true;
        // Wide lanes hold one head each, so the lanes of one B/C group read
        // the same B and C tiles, and a group's tiles over the whole
        // sequence outgrow L2 (64 KB per block).  Split ranges cut lane by
        // lane reach those tiles tens of blocks apart and re-read them from
        // DRAM; sets of CTAs that take the same range of a group's lanes
        // reach them together.  The set is the largest divisor of the lanes
        // per group up to 8, and the grid a multiple of it.
        const int npg = (int)(ptot / p.G);
        if (p.N == 256 && npg > 1) {
            int q = 1;
            for (int d = 2; d <= 8; ++d)
                if (npg % d == 0 && grid >= d) q = d;
            w.qs = q;
            grid = grid / q * q;
        }
    } else {
        grid = min64(sms, (int64_t)p.nseq * ptot);
    }
    w.grid = (int)max64(1, grid);
    size_t off = 0;
    w.hdr = off;     // ticket (4 B) + flags
    off = align_up(off + 256 + (size_t)sms * sizeof(int), 256);
    w.slots = off;
    off = align_up(off + (size_t)sms * kStateFloats * sizeof(float), 256);
    w.logdec = off;
    off = align_up(off + (size_t)sms * 2 * sizeof(float), 256);
    w.seqblk = off;
    off = align_up(off + (size_t)(p.nseq + 1) * sizeof(int), 256);
    w.total = off;
    return w;
}

}  // namespace

size_t fused_workspace_bytes(const Problem &p) { return fused_layout(p).total; }

int fused_supported(const Problem &p) {
    if (p.dtype != SSD_BF16 || p.P != kP || (p.N != 128 && p.N != 256)) return SSD_ERR_UNSUPPORTED;
    if (!encode_fn()) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

// The warpgroups trade registers (setmaxnreg); the trade adds up only with
// the launch allocation it was sized for.  Any other allocation could leave
// the increase waiting forever, so such a build is refused.
// A launch that may overlap the previous kernel on the stream (programmatic
// stream serialization); the kernel waits with griddepcontrol.wait before it
// reads what the previous kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, int threads, size_t smem,
                             cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename K>
cudaError_t check_regs(K kern) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    return fa.numRegs == kRegLaunch ? cudaSuccess : cudaErrorInvalidDeviceFunction;
}

cudaError_t fused_launch(const Problem &p) {
    const FLayout w = fused_layout(p);
    FArgs a{};
    a.L = p.seqlen;
    a.H = p.H; a.G = p.G; a.hpg = p.H / p.G; a.hpl = heads_per_lane(p);
    a.npg = (a.hpg + a.hpl - 1) / a.hpl; a.ptot = p.G * a.npg;
    a.nseq = p.nseq;
    a.varlen = p.cu != nullptr;
    a.nb_fixed = (int)((p.seqlen + kB - 1) / kB);
    a.grid = w.grid;
    a.qs = w.qs;
    a.dt = p.dt; a.A = p.A; a.D = p.D; a.init = p.init; a.cu = p.cu;
    a.dtt = p.dtt;
    a.y = (bf16 *)p.y;
    a.final_states = p.final_states;
    a.status = p.status;
    a.ticket = (int *)(p.ws + w.hdr);
    a.hflag = (int *)(p.ws + w.hdr + 256);
    a.hslot = (float *)(p.ws + w.slots);
    a.logdec = (float *)(p.ws + w.logdec);
    a.hstart = nullptr;   // split calls fold their start states in the main run
    a.seqblk = (const int *)(p.ws + w.seqblk);

    cudaError_t e = cudaMemsetAsync(p.ws + w.hdr, 0, w.slots - w.hdr, p.stream);
    if (e != cudaSuccess) return e;

    CUtensorMap tmX, tmB, tmC, tmY;
    const uint64_t L = (uint64_t)p.seqlen, b = (uint64_t)p.batch;
    const uint64_t dx[4] = {(uint64_t)p.P, (uint64_t)p.H, L, b};
    const uint64_t dbc[4] = {(uint64_t)p.N, (uint64_t)p.G, L, b};
    const uint32_t box[4] = {64, 1, (uint32_t)kB, 1};
    // a state-only scan reads no C and writes no y: its maps of them are
    // never used and point at B and x
    if (!make_map4(&tmX, p.x, dx, box) || !make_map4(&tmB, p.B, dbc, box) ||
        !make_map4(&tmC, p.states_only ? p.B : p.C, dbc, box) ||
        !make_map4(&tmY, p.states_only ? p.x : p.y, dx, box))
        return cudaErrorInvalidValue;

    if (a.varlen) {
        k_fused_varlen_setup<<<1, 1024, 0, p.stream>>>(a, p.P, p.N);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    a.states_only = p.states_only ? 1 : 0;
    const bool wide = p.N == 256;
    const size_t smem = wide ? smem_bytes<true>() : smem_bytes<false>();
    using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, FArgs);
    auto pick = [&](bool pre, bool chain) -> Kern {
        if (wide) {
            if (pre) return a.dtt.on ? k_ssd_fused<true, true, true, false> : k_ssd_fused<false, true, true, false>;
            if (chain) return a.dtt.on ? k_ssd_fused<true, true, false, true> : k_ssd_fused<false, true, false, true>;
            return a.dtt.on ? k_ssd_fused<true, true, false, false> : k_ssd_fused<false, true, false, false>;
        }
        if (pre) return a.dtt.on ? k_ssd_fused<true, false, true, false> : k_ssd_fused<false, false, true, false>;
        if (chain) return a.dtt.on ? k_ssd_fused<true, false, false, true> : k_ssd_fused<false, false, false, true>;
        return a.dtt.on ? k_ssd_fused<true, false, false, false> : k_ssd_fused<false, false, false, false>;
    };
    if (w.chain) {
        // pre run: the state records at every split; then the tickets start
        // again from zero for the main run
        Kern pre = pick(true, false);
        a.records = 1;
        e = check_regs(pre);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(pre, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (a.varlen) {
            e = launch_dependent(pre, dim3(w.grid), kThreads, smem, p.stream, tmX, tmB, tmC, tmY, a);
        } else {
            pre<<<w.grid, kThreads, smem, p.stream>>>(tmX, tmB, tmC, tmY, a);
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) return e;
        // the main run draws its tickets from a second counter (zeroed with
        // the first), so that no memset separates the kernels
        a.ticket += 1;
        a.chain = 1;
        a.records = 0;
    }
    // a state-only scan ends with a state-only run in place of the main run
    Kern kern = pick(p.states_only, w.chain);
    e = check_regs(kern);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (w.chain || a.varlen)
        return launch_dependent(kern, dim3(w.grid), kThreads, smem, p.stream, tmX, tmB, tmC, tmY, a);
    kern<<<w.grid, kThreads, smem, p.stream>>>(tmX, tmB, tmC, tmY, a);
    return cudaGetLastError();
}

}  // namespace ssd
