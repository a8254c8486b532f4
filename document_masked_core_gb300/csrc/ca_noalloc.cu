// ca_backward_noalloc: the backward pass for callers that cannot allocate
// device memory.
//
// ca_backward needs a workspace (an fp32 dQ accumulator and the D = dO.O
// vector) that the caller allocates.  Some callers cannot do that: code that
// runs inside a host framework which owns every device allocation (a fixed
// arena or a caching allocator it may not bypass), or plug-in code that is
// handed its input and output buffers and no way to ask for more memory.  For
// them this entry point takes its scratch from one file-scope device array of
// kNoAllocScratchBytes, reserved on every GPU that loads this library until
// the process exits.
#include <mutex>

#include "ca_internal.h"

namespace {

// 16 MiB: the backward's scratch is total_q * num_q_heads * (head_dim + 1)
// * 4 bytes (each part rounded up to 256) plus 256 bytes of counters: about
// 32 K (row, head) pairs at head_dim 128.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" ca_status_t ca_backward_noalloc(const ca_plan_t *p, const void *q, const void *k, const void *v,
                                           const void *o, const float *lse, const void *d_o, void *dq, void *dk,
                                           void *dv, void *stream) {
    using namespace ca;
    if (!p) return fail(CA_ERR_INVALID_ARG, "plan is NULL");
    // The backward touches the workspace up to the split-KV forward scratch:
    // the fp32 dQ accumulator, the D vector and the work-queue counters.
    const int64_t need = p->split_ws_off;
    if (need > static_cast<int64_t>(kNoAllocScratchBytes))
        return fail(CA_ERR_UNSUPPORTED, "this plan's backward needs " + std::to_string(need) +
                                            " bytes of scratch; ca_backward_noalloc has " +
                                            std::to_string(kNoAllocScratchBytes) +
                                            " (use ca_backward with a caller workspace)");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != p->device) return fail(CA_ERR_INVALID_ARG, "the plan was created on another device");
    if (dev < 0 || dev >= kMaxDevices) return fail(CA_ERR_UNSUPPORTED, "device ordinal out of range");
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    void *scratch = nullptr;
    {
        // Set-up per device, with that device current: the host-side name of
        // the array is not a device address, so look the address up.  Outside
        // a stream capture it is looked up on every call (a cudaDeviceReset
        // reloads the module and may move the array); inside a capture the
        // address of the last call outside one is used.
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (cap == cudaStreamCaptureStatusNone || !g_scratch_addr[dev]) {
            void *addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_bwd_scratch);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the backward scratch");
            g_scratch_addr[dev] = addr;
        }
        scratch = g_scratch_addr[dev];
    }
    const ca_status_t st = check_backward_args(p, q, k, v, o, lse, d_o, dq, dk, dv, scratch, need);
    if (st != CA_OK) return st;
    // the preprocess kernel of the backward zeroes the dQ accumulator and the
    // work-queue counter and rewrites D, so the array's previous contents
    // never leak into a result
    e = launch_backward(p, q, k, v, o, lse, d_o, dq, dk, dv, scratch, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "backward (no-allocation) launch");
    return CA_OK;
}
