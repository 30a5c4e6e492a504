// pn_noalloc.cu -- pn_gemv_noalloc: the GEMV for callers that cannot allocate
// device memory.
//
// pn_gemv needs a small device workspace (a status word, one counter per
// thread-block boundary and two partial-sum slots per boundary) that the
// caller allocates.  Some callers cannot allocate: code running inside a host
// callback or a driver-managed stream where cudaMalloc is not allowed, plugins
// whose host framework owns every allocation, or code that must never touch
// the allocator once a model is loaded.  pn_gemv_noalloc gives them the same
// GEMV with the workspace taken from a fixed array in this library's device
// image instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits.  In host
// code its name is only a host-side stand-in, not a device address, so the
// device address is looked up with cudaGetSymbolAddress once per device, with
// that device current, and passed to the kernel like any other workspace.
#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/pn.h"
#include "pn_internal.h"

namespace {

// Room for the workspace of a device with up to 226 SMs (the workspace size
// depends only on the SM count: about 2.3 KiB per SM).
constexpr size_t kNoAllocScratchBytes = 512 * 1024;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};                 // device address per device, once looked up

// The scratch array's device address on the current device (looked up once).
pn_status scratch_address(void** out) {
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return pn::cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return PN_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return pn::cuda_error(e);
        if (!p) return PN_ECUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PN_OK;
}

}  // namespace

extern "C" pn_status pn_gemv_noalloc(int type, const void* W, int64_t N, int64_t K, const uint16_t* x,
                                     int M, float* y, pn_stream stream) {
    // Every argument check first, so a refused call enqueues nothing.
    bool uses_ws = false;
    pn_status st = pn::gemv_check(type, W, N, K, x, M, y, PN_ALGO_AUTO, &uses_ws);
    if (st != PN_OK) return st;
    if (N == 0) return PN_OK;
    // The workspace this call needs on the current device; beyond the fixed
    // array (a device with more SMs than it was sized for) the call is refused.
    int sms = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return pn::cuda_error(e);
    const pn::WorkspaceLayout L = pn::workspace_layout(sms);
    if (L.total > kNoAllocScratchBytes) return PN_EINVAL;
    void* ws = nullptr;
    if ((st = scratch_address(&ws)) != PN_OK) return st;
    // The array keeps the last call's contents.  The status word, the tagged
    // hand-off words and the counters must start at zero; a completed call
    // leaves them zero, an aborted one may not, so the workspace is cleared on
    // the stream before every call that launches a kernel using it (the
    // CUDA-core kernel does not).
    if (uses_ws && (e = cudaMemsetAsync(ws, 0, L.total, reinterpret_cast<cudaStream_t>(stream))) != cudaSuccess)
        return pn::cuda_error(e);
    return pn_gemv_ex(type, W, N, K, x, M, y, ws, kNoAllocScratchBytes, PN_ALGO_AUTO, stream);
}
