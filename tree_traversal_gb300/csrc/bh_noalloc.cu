// bh_noalloc.cu -- orrery_bh_forces_noalloc: the whole force evaluation with
// its scratch in a fixed array that the library image itself carries, for
// callers that must not allocate device memory during a call.
//
// Who needs this: a host application or plugin that owns every device
// allocation itself (a pooled or arena allocator, a memory budget enforced
// from outside), code that runs while another thread may be capturing a CUDA
// graph on the device, and latency-sensitive loops that cannot afford the
// implicit device synchronisation of cudaMalloc / cudaFree. For them the
// ordinary entry point's grow-only workspace is the problem: its first call,
// and any call with a larger n than before, allocates.
//
// The scratch is one file-scope __device__ array of kScratchBytes. Every GPU
// on which this library's device code is loaded holds that memory until the
// process exits. Host code may not use the array's name as a device address
// (in host code it names a host-side shadow), so every call looks the
// address up with cudaGetSymbolAddress while the caller's device is current.
// The first call on a device may load the library's device code there (and
// sets the kernels' attributes): make it before any stream capture.
//
// All calls on a device share the array and it keeps the previous call's
// contents: every buffer that must start at zero is cleared by the call
// itself (the moments' arrival counters by the build, the status word by the
// cube kernel). Two calls whose GPU work overlapped would
// race on the array; this entry point serialises its calls with a lock and
// waits for its own work before returning, so its own calls never overlap.
// It does not share the array with orrery_bh_forces, whose workspace is
// separate.
#include <mutex>

#include "../../include/orrery_bh.h"
#include "bh_common.cuh"

namespace obh {
namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr int64_t kMaxN = int64_t(1) << 30;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_noalloc_mu;

// Device address of the current device's scratch. Looked up on every call
// (cheap once the library's module is loaded on the device), so a context
// that was torn down and created again (cudaDeviceReset) never gets a stale
// address.
int scratch_address(void **out)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return ORRERY_ECUDA;
    }
    *out = p;
    return ORRERY_OK;
}

}  // namespace
}  // namespace obh

using namespace obh;

extern "C" int orrery_bh_forces_noalloc(const float *pos_d, const float *mass_d, int64_t n,
                                        float theta, float eps, int32_t leaf_cap,
                                        int32_t traversal, float *acc_d, uint32_t *interactions_d,
                                        uint32_t *visits_d, void *stream)
{
    if (n < 0 || n > kMaxN || !(theta >= 0.0f) || !(eps >= 0.0f) || leaf_cap < 1 ||
        (traversal & ~(kTraversalMask | kFastTermFlag)) != 0 ||
        (traversal & kTraversalMask) > ORRERY_COHERENT_BALLOT)
        return ORRERY_EINVAL;
    if (n == 0) return ORRERY_OK;
    if (!pos_d || !mass_d || !acc_d) return ORRERY_EINVAL;
    Buffers b{};
    const int64_t nodes = node_bound(n, leaf_cap);
    if (nodes > (int64_t)INT32_MAX || carve(b, nullptr, n, nodes) > kScratchBytes)
        return ORRERY_ESCRATCH;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    void *base = nullptr;
    int rc = scratch_address(&base);
    if (rc != ORRERY_OK) return rc;
    carve(b, (char *)base, n, nodes);
    cudaStream_t st = (cudaStream_t)stream;
    uint64_t *keys_sorted = nullptr;
    uint32_t *perm = nullptr;
    launch_bbox(pos_d, mass_d, b, st);
    launch_morton(pos_d, b, st);
    launch_sort(b, st, &keys_sorted, &perm);
    launch_gather(pos_d, mass_d, perm, b, st);
    launch_build(keys_sorted, leaf_cap, b, st);
    launch_moments(keys_sorted, leaf_cap, b, st);
    launch_walk(traversal, theta, eps, perm, b, 0, n, acc_d, interactions_d, visits_d, st);
    int status = 0;
    cudaMemcpyAsync(&status, &b.params->status, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (cudaStreamSynchronize(st) != cudaSuccess || cudaGetLastError() != cudaSuccess)
        return ORRERY_ECUDA;
    if (status & kStatusNonFinite) return ORRERY_ENONFINITE;
    if (status & kStatusNodeBound) return ORRERY_ERANGE;
    if (status & kStatusWalkBound) return ORRERY_EWALK;
    if (status & kStatusInternal) return ORRERY_EINTERNAL;
    return ORRERY_OK;
}
