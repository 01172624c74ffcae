// Allocation-free variant of the two-pass tensor-core SSD scan.
//
// Some callers cannot allocate device memory at the time they run the scan:
// code that executes inside another framework's execution hook (an inference
// runtime's plugin enqueue, a custom-op callback) where that framework owns
// every device allocation, or a real-time loop that forbids allocation after
// start-up.  Such callers also cannot hand ssd_scan() a workspace of the
// size it asks for.  ssd_scan_noalloc() therefore takes only the inputs and
// outputs and runs the two-pass tensor-core kernels on scratch memory that
// belongs to
// this library: a fixed-size static device array, set aside on every GPU
// that loads the library and kept until the process exits.
//
// Limits and rules (also stated in include/ssd.h):
//   * the scratch holds at most kNoAllocScratchBytes; shapes that need more
//     are rejected with SSD_ERR_WORKSPACE before anything is enqueued;
//   * only shapes the two-pass kernels take are accepted (bf16, headdim
//     64, dstate 128/256, chunk 128/256, no packed sequences);
//   * every call uses the same array, so calls whose GPU work overlaps
//     (different streams, or different host threads) race with each other;
//     callers must order them, e.g. by issuing them on one stream;
//   * the first call on a device looks up the array's device address with
//     cudaGetSymbolAddress() while that device is current and caches it;
//     make that first call before any stream capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;  // 32 MiB per GPU
constexpr int kMaxDevices = 64;

// The library-owned scratch.  In host code this name is only a stand-in for
// the symbol: its device address comes from cudaGetSymbolAddress().
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of the scratch on the current device (looked up once).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SSD_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SSD_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SSD_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SSD_OK;
}

bool is_aligned(const void *ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" SSD_API int ssd_scan_noalloc(const ssd_shape *s, const void *x, const float *dt,
                                        const float *A, const void *B, const void *C,
                                        const float *D, const float *initial_states, void *y,
                                        float *final_states, int *device_status, void *stream) {
    if (!s) return SSD_ERR_INVALID_ARG;
    if (s->batch < 1 || s->seqlen < 1 || s->nheads < 1 || s->headdim < 1 || s->dstate < 1 ||
        s->ngroups < 1 || s->nheads % s->ngroups != 0 || s->nseq != s->batch)
        return SSD_ERR_INVALID_ARG;
    if (s->seqlen > (int64_t)INT32_MAX || shape_too_large(s)) return SSD_ERR_UNSUPPORTED;
    if (s->algo != SSD_ALGO_AUTO && s->algo != SSD_ALGO_TC && s->algo != SSD_ALGO_TC_TWOPASS)
        return SSD_ERR_UNSUPPORTED;
    // the two-pass kernels' own limits, checked before anything is derived
    // from the chunk size (a chunk size of 0 must not reach the division below)
    if (s->dtype != SSD_BF16 || (s->chunk_size != 128 && s->chunk_size != 256))
        return SSD_ERR_UNSUPPORTED;
    if (!x || !dt || !A || !B || !C || !y) return SSD_ERR_INVALID_ARG;

    Problem p;
    p.batch = s->batch; p.seqlen = s->seqlen;
    p.H = s->nheads; p.P = s->headdim; p.N = s->dstate; p.G = s->ngroups;
    p.Q = s->chunk_size; p.nseq = s->nseq; p.dtype = s->dtype;
    p.nc = (int)((s->seqlen + s->chunk_size - 1) / s->chunk_size);
    if (tc_supported(p) != SSD_OK) return SSD_ERR_UNSUPPORTED;
    if (!is_aligned(x, 16) || !is_aligned(B, 16) || !is_aligned(C, 16) || !is_aligned(y, 16) ||
        !is_aligned(dt, 4) || !is_aligned(A, 4) || !is_aligned(D, 4) ||
        !is_aligned(initial_states, 16) || !is_aligned(final_states, 16) ||
        !is_aligned(device_status, 4))
        return SSD_ERR_UNSUPPORTED;

    const size_t need = kStatusBytes + tc_workspace_bytes(p);
    if (need > kNoAllocScratchBytes) return SSD_ERR_WORKSPACE;

    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != SSD_OK) return rc;

    p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D;
    p.init = initial_states; p.cu = nullptr; p.y = y; p.final_states = final_states;
    p.status = (int *)scratch;
    p.ws = (char *)scratch + kStatusBytes;
    p.ws_bytes = kNoAllocScratchBytes - kStatusBytes;
    p.stream = (cudaStream_t)stream;

    // The status word keeps the previous call's value: clear it first (the
    // tensor-core launch clears its own counters and flags).
    if (cudaMemsetAsync(p.status, 0, sizeof(int), p.stream) != cudaSuccess) return SSD_ERR_CUDA;
    if (tc_launch(p) != cudaSuccess) return SSD_ERR_CUDA;
    if (device_status &&
        cudaMemcpyAsync(device_status, p.status, sizeof(int), cudaMemcpyDeviceToDevice,
                        p.stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    return SSD_OK;
}
