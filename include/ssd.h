/*
 * ssd.h -- C ABI of the SSD (structured state space duality) forward scan
 * for NVIDIA B300 (sm_103a).
 *
 * What it computes.  For every sequence s and head h (B/C group
 * g = h / (nheads / ngroups)), with a state h_t in R^{headdim x dstate}
 * starting at initial_states[s, h] (or zero):
 *
 *     h_t = exp(dt_t * A_h) * h_{t-1} + dt_t * (x_t (outer) B_t)
 *     y_t = h_t . C_t + D_h * x_t
 *
 * and final_states[s, h] = h after the sequence's last token.
 *   - The selective SSM (B, C, Delta functions of the input) and its
 *     recurrence: Mamba-1 walkthrough "Mamba: Linear-Time Sequence Modeling
 *     with Selective State Spaces", section 三(二) "引入选择机制到 SSM 中";
 *     Abar = exp(Delta * A): same page, section 三 3.
 *   - The same map is multiplication by the semiseparable matrix
 *     M = L o (C B^T); it is evaluated by block decomposition -- masked
 *     quadratic matmuls inside each chunk of chunk_size tokens plus a
 *     recurrence over per-chunk states: QbitAI article "新架构Mamba更新二代！",
 *     sections "统一SSM和注意力机制" (semiseparable matrices, structured masked
 *     attention, the two equivalent forms) and "Mamba-2：更强学习能力，更快训练推理"
 *     (block-decomposition matmul algorithm over the GPU memory hierarchy,
 *     multi-head SSM, variable sequence length).
 *   - Packed variable-length sequences reset the state at every cu_seqlens
 *     boundary: same section of the QbitAI article (variable sequence
 *     length) and the Mamba-1 walkthrough, section 三 2.3 "边界重置".
 *   dt is taken as given (already positive, e.g. after softplus): the scan
 *   applies no softplus, bias or clamp.  The chunk size changes only the
 *   rounding, never the result.
 *
 * Value domain.  As in the method, every decay exp(dt_t * A_h) lies in
 * (0, 1]: dt >= 0 and A_h <= 0.  The kernels rely on it (their exponents are
 * never positive).  These values live in device memory and are not checked;
 * outside this domain the results are unspecified.
 *
 * Layouts.  Row-major, contiguous, no padding:
 *   x, y            [batch][seqlen][nheads][headdim]   dtype (fp32 or bf16)
 *   dt              [batch][seqlen][nheads]            fp32
 *   A, D            [nheads]                           fp32
 *   B, C            [batch][seqlen][ngroups][dstate]   dtype
 *   initial_states,
 *   final_states    [nseq][nheads][headdim][dstate]    fp32
 *   cu_seqlens      [nseq + 1]                         int32
 * Without cu_seqlens, sequence s is batch row s and nseq must equal batch.
 * With cu_seqlens, batch must be 1 and sequence s is tokens
 * [cu_seqlens[s], cu_seqlens[s+1]) of that row; cu_seqlens[0] == 0,
 * cu_seqlens[nseq] == seqlen, non-decreasing (an empty sequence's final
 * state is its initial state).
 *
 * Ownership and execution.  Every pointer argument except `shape` and
 * `bytes` is a DEVICE pointer owned by the caller.  The library allocates
 * nothing, keeps no state between calls, never synchronises inside
 * ssd_scan(), and enqueues all its work on `stream` (a cudaStream_t, may be
 * NULL for the legacy default stream).  Calls on different streams with
 * different workspaces are independent; the workspace of a call must not be
 * reused until that call's work on its stream has finished.
 *
 * Errors.  Functions return an ssd_status.  Argument errors are detected on
 * the host before anything is enqueued.  Errors in DEVICE-resident inputs
 * (a malformed cu_seqlens) and device-side wait time-outs are recorded in
 * the workspace's status word; the kernels then skip their work and leave
 * y / final_states unspecified.  ssd_check_device_status() reads that word.
 * Nothing aborts, traps or throws across this ABI.
 */
#ifndef SSD_B300_SSD_H
#define SSD_B300_SSD_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ssd_dtype {
    SSD_F32 = 0,   /* x, B, C, y in fp32; all arithmetic fp32 SIMT */
    SSD_BF16 = 1   /* x, B, C, y in bf16; tensor-core contractions with
                      fp32 accumulation, fp32 decays and states */
} ssd_dtype;

typedef enum ssd_algo {
    SSD_ALGO_AUTO = 0,     /* tensor-core path when the shape allows, else SIMT */
    SSD_ALGO_SIMT = 1,     /* CUDA-core kernels, any supported shape/dtype */
    SSD_ALGO_TC = 2,       /* tcgen05/TMEM/TMA path (bf16 only): the fused
                              single-pass kernel for headdim 64 and dstate
                              128 or 256 (any chunk size, packed sequences
                              included), else the two-pass kernels;
                              UNSUPPORTED if the shape fits neither */
    SSD_ALGO_TC_TWOPASS = 3 /* the two-pass tensor-core kernels (chunk-state
                              scan, then chunk output): bf16, headdim 64,
                              dstate 128 or 256, chunk 128 or 256, no packed
                              sequences */
} ssd_algo;

typedef enum ssd_status {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,     /* null pointer, bad shape, nseq mismatch */
    SSD_ERR_UNSUPPORTED = 2,     /* dtype/chunk/headdim/dstate/alignment not
                                    supported by the requested algorithm */
    SSD_ERR_WORKSPACE = 3,       /* workspace missing or too small */
    SSD_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed */
    SSD_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait gave up */
    SSD_ERR_DEVICE_INPUT = 6     /* cu_seqlens (device memory) malformed */
} ssd_status;

typedef struct ssd_shape {
    int64_t batch;       /* >= 0 */
    int64_t seqlen;      /* >= 0, tokens per batch row (at most 2^31 - 1; every
                            buffer at most 2^56 elements) */
    int32_t nheads;      /* H >= 1 */
    int32_t headdim;     /* P, 1..256 (SIMT); 64 (TC) */
    int32_t dstate;      /* N, 1..256 (SIMT); 64, 128 or 256 (TC) */
    int32_t ngroups;     /* G >= 1, divides nheads */
    int32_t chunk_size;  /* Q in {64, 128, 256} */
    int32_t nseq;        /* number of sequences: batch, or len(cu_seqlens)-1 */
    int32_t dtype;       /* ssd_dtype */
    int32_t algo;        /* ssd_algo */
} ssd_shape;

/*
 * Optional transform of the raw step sizes, applied by the kernels as they
 * read dt (the selective SSM's Delta = softplus(parameter + s_Delta(x)):
 * Mamba-1 walkthrough "Mamba: Linear-Time Sequence Modeling with Selective
 * State Spaces", section 三(二) "引入选择机制到 SSM 中", where Delta passes
 * through tau_Delta = softplus).  For token t of head h:
 *     z  = dt[t, h] + (bias ? bias[h] : 0)
 *     dt' = softplus ? log(1 + exp(z)) : z
 *     dt' = min(max(dt', dt_min), dt_max)
 * and the scan uses dt' wherever the operation above has dt.  Tokens outside
 * every sequence are not transformed.  dt_min <= dt_max is required (use 0
 * and INFINITY for no clamp); a NULL transform means dt is used as given.
 */
typedef struct ssd_dt_transform {
    const float *bias;   /* [nheads] DEVICE pointer, nullable (0) */
    int32_t softplus;    /* nonzero: apply softplus after the bias */
    float dt_min;        /* clamp bounds, applied last */
    float dt_max;
} ssd_dt_transform;

/*
 * Bytes of device workspace ssd_scan() needs for `shape` (with the algorithm
 * the shape resolves to).  Writes *bytes; returns SSD_OK or the same
 * argument/support error ssd_scan() would return for this shape.
 */
SSD_API int ssd_scan_workspace_size(const ssd_shape *shape, size_t *bytes);

/*
 * Enqueue the SSD forward scan on `stream`.
 *   x, dt, A, B, C     required inputs (layouts above)
 *   D                  nullable: treated as all zeros
 *   initial_states     nullable: zero initial states
 *   cu_seqlens         nullable: no packing (nseq == batch)
 *   y                  required output, same dtype as x
 *   final_states       nullable: not written
 *   workspace          device buffer of >= ssd_scan_workspace_size() bytes,
 *                      256-byte aligned; contents need no initialisation
 * The tensor-core path additionally needs x, B, C, y 16-byte aligned.
 */
SSD_API int ssd_scan(const ssd_shape *shape, const void *x, const float *dt,
                     const float *A, const void *B, const void *C,
                     const float *D, const float *initial_states,
                     const int32_t *cu_seqlens, void *y, float *final_states,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * ssd_scan() with the step sizes first put through `dt_transform` (nullable:
 * then exactly ssd_scan()).  The fused tensor-core kernel applies the
 * transform as it loads dt; the other paths run a pre-pass that writes the
 * transformed dt into the workspace, which is why the workspace size depends
 * on the transform: ask ssd_scan_ex_workspace_size() with the same
 * arguments.  Errors as for ssd_scan(), plus SSD_ERR_INVALID_ARG when
 * dt_min > dt_max.
 */
SSD_API int ssd_scan_ex_workspace_size(const ssd_shape *shape,
                                       const ssd_dt_transform *dt_transform,
                                       size_t *bytes);
SSD_API int ssd_scan_ex(const ssd_shape *shape, const void *x, const float *dt,
                        const ssd_dt_transform *dt_transform, const float *A,
                        const void *B, const void *C, const float *D,
                        const float *initial_states, const int32_t *cu_seqlens,
                        void *y, float *final_states, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * Final states only: what ssd_scan_ex() writes to final_states, without y
 * (the state recurrence of the operation above, with no output read-out:
 * no C, no D, no y).  For callers that need only where a sequence ends, for
 * example the first pass of the sequence-parallel scan below, where each
 * shard's end state from a zero start is all the exchange needs.  It runs
 * the fused kernel's state-only mode, which skips C B^T, C H^T, the mask and
 * M x, so it reads x, B and dt once and writes only the states.
 *   shape          as for ssd_scan(); algo must be SSD_ALGO_AUTO or
 *                  SSD_ALGO_TC and the shape one the fused kernel takes (bf16,
 *                  headdim 64, dstate 128 or 256), else SSD_ERR_UNSUPPORTED
 *   x, dt, A, B    required (layouts above); dt_transform nullable
 *   initial_states nullable (zero); cu_seqlens nullable (as for ssd_scan())
 *   final_states   required output, [nseq][nheads][headdim][dstate] fp32
 *   workspace      >= ssd_scan_ex_workspace_size() of the same shape and
 *                  transform, 256-byte aligned
 * x, B, initial_states and final_states 16-byte aligned.  Errors and the
 * device status word as for ssd_scan(); asynchronous on `stream`.
 */
SSD_API int ssd_scan_states(const ssd_shape *shape, const void *x, const float *dt,
                            const ssd_dt_transform *dt_transform, const float *A,
                            const void *B, const float *initial_states,
                            const int32_t *cu_seqlens, float *final_states, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * One decode step of `batch` independent sequences: the recurrent form of the
 * same map, one token per sequence, with the state updated in place (the
 * selective SSM's state cache that makes generation linear-time: Mamba-1
 * walkthrough, sections 二(一) "从连续系统到离散建模" -- recurrent updates for
 * inference -- and 四(五) "计算效率评估").  For every sequence b and head h
 * (group g = h / (nheads / ngroups)):
 *     state[b, h] <- exp(dt' A_h) state[b, h] + dt' (x[b, h] (outer) B[b, g])
 *     y[b, h]      = state[b, h] . C[b, g] + D_h x[b, h]
 * with dt' = dt[b, h] put through dt_transform (nullable).  Equals ssd_scan()
 * of a one-token sequence with initial_states = final_states = state.
 *
 * Layouts (row-major, contiguous):
 *   x, y     [batch][nheads][headdim]           dtype (fp32 or bf16)
 *   dt       [batch][nheads]                    fp32
 *   A, D     [nheads]                           fp32 (D nullable: 0)
 *   B, C     [batch][ngroups][dstate]           dtype
 *   state    [batch][nheads][headdim][dstate]   fp32, read and written
 * All pointers are DEVICE pointers owned by the caller; x, B, C, dt, A, D
 * must not overlap state or y.  Any headdim and dstate in 1..1024.  No
 * workspace, no device-side waits: every error is found on the host and
 * returned before anything is enqueued.  Asynchronous on `stream`.
 */
typedef struct ssd_step_shape {
    int64_t batch;       /* >= 0 */
    int32_t nheads;      /* H >= 1 */
    int32_t headdim;     /* P, 1..1024 */
    int32_t dstate;      /* N, 1..1024 */
    int32_t ngroups;     /* G >= 1, divides nheads */
    int32_t dtype;       /* ssd_dtype */
    int32_t reserved;    /* must be 0 */
} ssd_step_shape;

SSD_API int ssd_step(const ssd_step_shape *shape, const void *x, const float *dt,
                     const ssd_dt_transform *dt_transform, const float *A,
                     const void *B, const void *C, const float *D, float *state,
                     void *y, void *stream);

/*
 * Synchronise `stream`, then read the status word that the last ssd_scan()
 * using `workspace` left there: SSD_OK, SSD_ERR_DEVICE_INPUT or
 * SSD_ERR_DEVICE_TIMEOUT (or SSD_ERR_CUDA if the sync/copy itself failed).
 */
SSD_API int ssd_check_device_status(const void *workspace, void *stream);

/*
 * Diagnostic of the failure path (not part of a scan).  Runs one of the fused
 * kernel's bounded device-side waits where nothing will ever satisfy it:
 * which = 0 waits on a shared-memory mbarrier that no thread or copy
 * completes, which = 1 on a handoff flag (global memory) that no CTA sets.
 * The wait gives up after its time limit (2 s), records the error in the
 * status word and returns, so the context stays usable.
 *   device_words  DEVICE pointer to 2 ints of scratch owned by the caller
 *                 (status word, flag); cleared by the call
 * Synchronises `stream`, then returns the status word the device recorded:
 * SSD_ERR_DEVICE_TIMEOUT when the path works.  SSD_ERR_INVALID_ARG for a bad
 * `which` or pointer, SSD_ERR_CUDA if a CUDA call failed.
 */
SSD_API int ssd_selftest_wait_timeout(int which, int *device_words, void *stream);

/* Static, human-readable name of a status code (never NULL). */
SSD_API const char *ssd_status_string(int status);

/* Which algorithm ssd_scan() would run for `shape` (SSD_ALGO_SIMT,
 * SSD_ALGO_TC for the fused kernel or SSD_ALGO_TC_TWOPASS), or a negative
 * ssd_status if the shape is rejected. */
SSD_API int ssd_resolve_algo(const ssd_shape *shape);

/*
 * Sequence parallelism: the carry exchange between shards of a sequence
 * (QbitAI article "新架构Mamba更新二代！", section "Mamba-2：更强学习能力，
 * 更快训练推理": sequence parallelism for longer sequences).  Every sequence
 * is cut into nshards consecutive pieces, shard r on device r.  The state is
 * the only thing that crosses a cut.  Each device scans its shard from a zero
 * state (ssd_scan(), final_states -> S_r) and computes its shard's log-decay
 *     logdec_r[s, h] = sum over the shard's tokens t of sequence s of dt'_t A_h
 * (ssd_seqpar_logdec).  The devices all-gather (S_r, logdec_r); each folds
 *     H_in(0)     = initial_states (or zero)
 *     H_in(q + 1) = exp(logdec_q) H_in(q) + S_q
 * (ssd_seqpar_fold) and re-scans its shard from H_in(r), which gives its part
 * of y exactly as the unsharded scan would; H_in(nshards) is the sequence's
 * final state.  This is the chunk-to-chunk state passing of the block
 * decomposition, one step per shard.
 */

/*
 * logdec[s][h] (fp32, DEVICE, [batch][nheads], caller-owned) for the shard
 * in `shape`'s layout: sequence s is batch row s (nseq == batch; packed
 * sequences are not sharded), and only batch, seqlen, nheads and nseq are
 * used (plus ssd_scan()'s size checks).  dt [batch][seqlen][nheads] and A
 * [nheads] are fp32 DEVICE pointers; dt_transform as for ssd_scan_ex()
 * (nullable).  seqlen 0 gives 0 (dt may then be NULL).  Sums in fp64, stores
 * fp32.  Errors on the host
 * before anything is enqueued: SSD_ERR_INVALID_ARG (null pointer, bad
 * shape), SSD_ERR_UNSUPPORTED (misaligned fp32 pointer, shape too large);
 * SSD_ERR_CUDA if the launch fails.  Asynchronous on `stream`; allocates
 * nothing.
 */
SSD_API int ssd_seqpar_logdec(const ssd_shape *shape, const float *dt,
                              const ssd_dt_transform *dt_transform, const float *A,
                              float *logdec, void *stream);

/*
 * The fold over shards, for shard `rank` of `nshards`.  All fp32 DEVICE
 * pointers owned by the caller:
 *   shard_states          [nshards][nseq][nheads][headdim][dstate]: S_q,
 *                         each shard's state scanned from zero (gathered)
 *   shard_logdec          [nshards][nseq][nheads]: logdec_q (gathered)
 *   initial_states        [nseq][nheads][headdim][dstate], nullable (zero)
 *   shard_initial_states  [nseq][nheads][headdim][dstate]: H_in(rank),
 *                         nullable (not written)
 *   final_states          [nseq][nheads][headdim][dstate]: H_in(nshards),
 *                         nullable (not written); at least one of the two
 *                         outputs is required
 * Outputs must not overlap inputs.  Errors on the host before anything is
 * enqueued: SSD_ERR_INVALID_ARG (rank outside [0, nshards), sizes < 1, nseq
 * < 0, missing pointer), SSD_ERR_UNSUPPORTED (misaligned pointer, over 2^56
 * elements); SSD_ERR_CUDA if the launch fails.  Asynchronous on `stream`;
 * allocates nothing.
 */
SSD_API int ssd_seqpar_fold(int32_t nshards, int32_t rank, int64_t nseq, int32_t nheads,
                            int32_t headdim, int32_t dstate, const float *shard_states,
                            const float *shard_logdec, const float *initial_states,
                            float *shard_initial_states, float *final_states,
                            void *stream);

/*
 * ssd_scan() without a workspace: for callers that cannot allocate device
 * memory when they run the scan -- code running inside another framework's
 * execution hook (an inference runtime's plugin enqueue, a custom-op
 * callback) where that framework owns all device allocations, or a
 * real-time loop that forbids allocation after start-up.  The pages
 * describing the method have no counterpart to this entry point; it exists
 * only for such callers.
 *
 * The call computes exactly what ssd_scan() computes on its two-pass
 * tensor-core path (SSD_ALGO_TC_TWOPASS), using a scratch array that belongs to the library: a static device
 * array of 32 MiB that every GPU loading the library holds until the
 * process exits.  The caller passes only inputs and outputs (same meaning,
 * layout and alignment as ssd_scan(); no cu_seqlens).
 *   device_status  nullable DEVICE pointer to one int; if given, the call's
 *                  device status word (SSD_OK or SSD_ERR_DEVICE_TIMEOUT) is
 *                  copied there on `stream` when the scan's work is done.
 * shape->algo may be SSD_ALGO_AUTO, SSD_ALGO_TC or SSD_ALGO_TC_TWOPASS (all
 * three run the two-pass kernels); any other value is SSD_ERR_UNSUPPORTED.
 * Returns SSD_ERR_WORKSPACE, before enqueuing anything, if the shape needs
 * more scratch than the 32 MiB array holds (the need is
 * ssd_scan_workspace_size() of the same shape with algo
 * SSD_ALGO_TC_TWOPASS), and SSD_ERR_UNSUPPORTED for shapes the two-pass
 * path does not take (dtype other than bf16, chunk_size other than 128 or
 * 256, headdim other than 64, dstate other than 128 or 256).
 * Allocates nothing: no cudaMalloc/cudaFree and no allocating library call.
 * All calls share the one array and it keeps the last call's contents (the
 * call clears what must start at zero), so calls whose GPU work overlaps --
 * on different streams or from different host threads -- race; order them,
 * for example by issuing them on one stream.  The first call on a device,
 * with that device current, looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture begins.
 */
SSD_API int ssd_scan_noalloc(const ssd_shape *shape, const void *x, const float *dt,
                             const float *A, const void *B, const void *C,
                             const float *D, const float *initial_states, void *y,
                             float *final_states, int *device_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_B300_SSD_H */
