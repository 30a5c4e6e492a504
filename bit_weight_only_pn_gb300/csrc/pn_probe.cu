// pn_probe.cu -- pn_read_ranges: the plain read-bandwidth ceiling that the
// GEMV kernels are measured against.
//
// It reads every byte of up to kMaxLayer device ranges once, with 16-byte
// loads from a grid of a few blocks per SM, and folds what it read into one
// 32-bit XOR per range (so the loads cannot be dropped).  It is the same
// byte stream a GEMV launch reads from its weights, without the decode, so
// its time is the floor for a single pass over those weights on this GPU.
// Launched with programmatic dependent launch like the GEMV kernels, and
// releasing the next launch at once, so a stream of back-to-back launches
// measures the steady read rate.
#include <cstdint>

#include <cuda_runtime.h>

#include "pn_device.cuh"
#include "pn_internal.h"

namespace pn {
namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 4;

struct ReadRanges {
    const uint4* p[kMaxLayer];
    uint64_t n16[kMaxLayer];       // 16-byte words per range
    uint64_t start16[kMaxLayer + 1];   // prefix sums of n16
    int count;
};

// Folds a warp's words and adds them to sink[f] (one atomic per warp).
__device__ __forceinline__ void commit(uint32_t a, uint32_t* sink, int f) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a ^= __shfl_xor_sync(0xFFFFFFFFu, a, o);
    if ((threadIdx.x & 31) == 0 && a != 0u) atomicXor(sink + f, a);
}

// Block b reads 16-byte words [b * per, (b + 1) * per) of the ranges laid end
// to end: it finds its first range once, then streams each range segment with
// unrolled 16-byte loads.
__global__ void __launch_bounds__(kThreads) read_ranges_kernel(const __grid_constant__ ReadRanges R,
                                                               uint32_t* __restrict__ sink) {
    // nothing here depends on the previous launch (the sink takes atomics):
    // the next launch may start at once, so back-to-back launches stream
    // without a gap (programmatic dependent launch)
    griddep_launch_dependents();
    const uint64_t total = R.start16[R.count];
    const uint64_t per = (total + gridDim.x - 1) / gridDim.x;
    uint64_t b0 = static_cast<uint64_t>(blockIdx.x) * per;
    const uint64_t b1 = b0 + per < total ? b0 + per : total;
    int f = 0;
    while (f + 1 < R.count && b0 >= R.start16[f + 1]) ++f;
    while (b0 < b1) {
        const uint64_t end = b1 < R.start16[f + 1] ? b1 : R.start16[f + 1];
        const uint4* p = R.p[f] + (b0 - R.start16[f]);
        const uint64_t n = end - b0;
        uint32_t acc = 0u;
        for (uint64_t j = threadIdx.x; j < n; j += kThreads * kUnroll) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                v[u] = j + u * kThreads < n ? __ldcs(p + j + u * kThreads) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
        }
        commit(acc, sink, f);
        b0 = end;
        ++f;
    }
}

}  // namespace

cudaError_t launch_read_ranges(const void* const* ptrs, const size_t* bytes, int count, uint32_t* sink,
                               int num_sms, cudaStream_t s) {
    ReadRanges R{};
    R.count = count;
    for (int e = 0; e < count; ++e) {
        R.p[e] = static_cast<const uint4*>(ptrs[e]);
        R.n16[e] = bytes[e] / 16;
        R.start16[e + 1] = R.start16[e] + R.n16[e];
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(4 * (num_sms > 0 ? num_sms : 1));   // 4 blocks of 512 threads per SM
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, read_ranges_kernel, R, sink);
}

}  // namespace pn
