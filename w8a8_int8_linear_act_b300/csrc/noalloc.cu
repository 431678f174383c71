// Entry points for callers that cannot allocate device memory (declared in
// include/w8a8.h): w8a8_linear_noalloc runs w8a8_linear with a workspace
// built into the library, and w8a8_noalloc_read_status reads that
// workspace's device status word.
//
// The workspace is the file-scope device array below.  It sits in this file
// alone so that it is part of a CUDA module that holds nothing else: with
// the runtime's lazy module loading (the default), a process that never
// calls these entry points never loads the module and never holds the
// array; one that does holds it on every device it used them on, until the
// process exits.
//
// In host code the array's name is a host-side stand-in, never a device
// address.  The device address is looked up with cudaGetSymbolAddress, with
// the device current, on the first call on each device, and cached together
// with the device's current context.  If the context changes (the device was
// reset with cudaDeviceReset and a new primary context created), the cached
// address belongs to the old context and is looked up again.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "../../include/w8a8.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[W8A8_NOALLOC_SCRATCH_BYTES];

struct ScratchAddr {
    CUcontext ctx = nullptr;   // context the address was looked up in
    void* ptr = nullptr;
};
ScratchAddr g_addr[kMaxDevices];
std::mutex g_mutex;

// cuCtxGetCurrent, through the runtime's driver entry-point query (the
// library does not link the driver library directly, so that it loads on
// machines without one).
PFN_cuCtxGetCurrent_v4000 g_ctx_get = nullptr;
std::once_flag g_ctx_get_once;

CUcontext current_context()
{
    std::call_once(g_ctx_get_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    if (g_ctx_get == nullptr || g_ctx_get(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}

// Device address of the built-in scratch on the current device, looked up
// once per device and context.  Returns nullptr (and the status in *st) when
// there is no usable device or the lookup fails.
void* scratch_address(w8a8_status* st)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        *st = W8A8_ERR_NO_DEVICE;
        return nullptr;
    }
    // The context current on this thread; none yet if the runtime has not
    // made its primary context current here (then the lookup below does).
    CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(g_mutex);
    ScratchAddr& a = g_addr[dev];
    if (a.ptr == nullptr || ctx == nullptr || a.ctx != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            *st = W8A8_ERR_CUDA;
            return nullptr;
        }
        ctx = current_context();
        a.ptr = p;
        a.ctx = ctx;
    }
    *st = W8A8_OK;
    return a.ptr;
}

}  // namespace

extern "C" {

w8a8_status w8a8_linear_noalloc(const void* X, int x_dtype, int64_t M, int64_t K, const uint16_t* Wp,
                                const float* sw, int64_t N, const void* bias, int bias_dtype, uint16_t* Y,
                                void* stream)
{
    if (M < 0 || K < 0) return W8A8_ERR_INVALID_ARG;
    // Refuse what does not fit before touching the device: nothing launched.
    const size_t need = w8a8_linear_workspace_min_bytes(M, K);
    if (need > W8A8_NOALLOC_SCRATCH_BYTES) return W8A8_ERR_WORKSPACE;
    w8a8_status st = W8A8_OK;
    void* scratch = scratch_address(&st);
    if (scratch == nullptr) return st;
    // w8a8_linear clears what must start at zero (the status word and the
    // split-tile counters) in its first kernel, so the previous call's
    // contents do not matter.
    return w8a8_linear(X, x_dtype, M, K, Wp, sw, N, bias, bias_dtype, Y, scratch, W8A8_NOALLOC_SCRATCH_BYTES,
                       stream);
}

w8a8_status w8a8_noalloc_read_status(void* stream, uint32_t* device_bits)
{
    if (!device_bits) return W8A8_ERR_INVALID_ARG;
    w8a8_status st = W8A8_OK;
    void* scratch = scratch_address(&st);
    if (scratch == nullptr) return st;
    return w8a8_read_status(scratch, stream, device_bits);
}

}  // extern "C"
