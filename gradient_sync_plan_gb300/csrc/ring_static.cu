// ring_static.cu -- the host-buffer fused allreduce for callers that cannot
// allocate device memory.
//
// ring_allreduce_fused_from_host needs device buffers to hold every rank's
// bucket while the kernel runs, and its caller provides them.  Some callers
// have no way to get such buffers: code that runs where the device allocator
// belongs to someone else (a host-side training loop inside a framework that
// owns all device memory, a plug-in that must not grow a process's device
// footprint, tools that only link this library and no allocator).
// ring_allreduce_fused_from_host_noalloc serves them: its device buffers are
// carved out of one fixed array that this file reserves in the library's own
// module, so the call itself allocates nothing.
//
// The array, DDP_STATIC_SCRATCH_BYTES bytes, is reserved on every GPU that
// loads the library and stays reserved until the process exits.  Every call
// on a device uses the same array: two calls that run at the same time on
// the GPU (different streams, or different host threads) overwrite each
// other's data, so calls must be ordered (one stream, or synchronised).  The
// array keeps whatever the last call left in it; nothing needs to start at
// zero, because each call overwrites every byte it reads with its own
// host-to-device copy before the kernel runs.
//
// The array's device address is looked up once per device and cached.  The
// cache does not survive a device reset (cudaDeviceReset destroys the
// context the address belongs to): a process that resets a device must not
// call this entry point on that device afterwards.
#include <cuda_runtime.h>

#include <map>
#include <mutex>

#include "ddp_abi_guard.h"
#include "ddp.h"
#include "ddp_internal.h"
#include "ddp_trace.h"

// The scratch itself.  In host code this name is only a host-side stand-in
// for the symbol, never a device address: it is turned into one with
// cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) unsigned char ddp_static_scratch[DDP_STATIC_SCRATCH_BYTES];

namespace {

std::mutex g_scratch_mu;
std::map<int, unsigned char*> g_scratch_addr;     // device -> device address of ddp_static_scratch

// Device address of the scratch on the current device.  The first call on a
// device looks it up (with that device current) and caches it.
cudaError_t scratch_on_current_device(unsigned char** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    auto it = g_scratch_addr.find(dev);
    if (it != g_scratch_addr.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, ddp_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
    *out = static_cast<unsigned char*>(p);
    return cudaSuccess;
}

}  // namespace

extern "C" int32_t ring_allreduce_fused_from_host_noalloc(int32_t world, const void* const* host_in,
                                                          void* const* host_out, int64_t numel, int32_t dtype,
                                                          int32_t divisor, void* stream) try {
    DDP_TRACE_CALL();
    // sizes first: after common_checks numel <= DDP_MAX_NUMEL, so the byte
    // counts below cannot overflow
    if (int32_t st = ddpk::common_checks(world, numel, dtype)) return st;
    if (divisor < 0 || !host_in || !host_out) return DDP_ERR_INVALID;
    const int64_t es = ddpk::elem_bytes(dtype);
    if (numel > DDP_STATIC_SCRATCH_BYTES / es) return DDP_ERR_CAPACITY;
    // each rank's slice starts on a 256-byte boundary so the kernel's
    // vectorised paths apply
    const int64_t bytes = numel * es;
    const int64_t stride = (bytes + 255) & ~(int64_t)255;
    if (stride > DDP_STATIC_SCRATCH_BYTES / world) return DDP_ERR_CAPACITY;
    if (int32_t st = ddpk::check_host_in_out(world, host_in, host_out, numel, dtype)) return st;
    if (numel == 0) return DDP_OK;

    unsigned char* base = nullptr;
    if (int32_t st = ddpk::cuda_status(scratch_on_current_device(&base))) return st;
    void* dev[DDP_MAX_WORLD];
    for (int32_t r = 0; r < world; ++r) dev[r] = base + (int64_t)r * stride;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int32_t r = 0; r < world; ++r)
        if (int32_t st =
                ddpk::cuda_status(cudaMemcpyAsync(dev[r], host_in[r], (size_t)bytes, cudaMemcpyHostToDevice, s)))
            return st;
    if (int32_t st = ddpk::cuda_status(
            ddpk::launch_ring_fused(world, dev, numel, dtype, ddpk::make_div(divisor), true, s)))
        return st;
    for (int32_t r = 0; r < world; ++r)
        if (int32_t st =
                ddpk::cuda_status(cudaMemcpyAsync(host_out[r], dev[r], (size_t)bytes, cudaMemcpyDeviceToHost, s)))
            return st;
    return DDP_OK;
} DDP_ABI_CATCH
