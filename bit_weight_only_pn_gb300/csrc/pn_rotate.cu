// pn_rotate.cu -- the runtime Hadamard rotation of the activations that reach
// the PN weights (tensorless docs, "Why a P100-native weight format", section
// "How Qwen3.8-27B-PN3 uses it": the model applies a Hadamard rotation to those
// activations and the engine performs it at run time).
//
// Every run of B consecutive activations of a row (B = 2^m, 2 <= B <= 4096)
// is multiplied by the orthonormal Sylvester Hadamard matrix H_B / sqrt(B)
// with a fixed arithmetic: fp16 -> fp32, fast Walsh-Hadamard butterflies in
// stages h = 1, 2, ..., B/2 in that order (pair (v[i], v[i+h]), (i & h) == 0,
// becomes (v[i] + v[i+h], v[i] - v[i+h]), each an IEEE fp32 add / subtract),
// one fp32 multiply by s, fp16 round-to-nearest-even.  Every output is the
// same sequence of roundings whatever the thread schedule, so results are
// reproducible bit for bit.
//
// One thread block per (row, run): the run sits in shared memory, each thread
// takes B / 2 / threads butterflies per stage, and a barrier separates stages.
// The activations are small (K * M * 2 bytes), so this is a short kernel.  It
// is launched with programmatic dependent launch, so the GEMV that follows can
// start and warm L2 with its first weights while the rotation runs.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pn_device.cuh"
#include "pn_internal.h"

namespace pn {
namespace {

__global__ void hadamard_kernel(const uint16_t* x, int64_t K, int block, int log2_block, float scale,
                                uint16_t* out) {
    extern __shared__ float v[];
    // programmatic dependent launch: the next kernel may start its own
    // preparation now; x is read only once the previous kernel has finished
    griddep_launch_dependents();
    griddep_wait();
    const int64_t off = static_cast<int64_t>(blockIdx.y) * K + static_cast<int64_t>(blockIdx.x) * block;
    for (int i = threadIdx.x; i < block; i += blockDim.x) v[i] = __half2float(__ushort_as_half(x[off + i]));
    __syncthreads();
    const int half = block >> 1;
    for (int lh = 0; lh < log2_block; ++lh) {
        const int h = 1 << lh;
        for (int j = threadIdx.x; j < half; j += blockDim.x) {
            const int i = ((j >> lh) << (lh + 1)) | (j & (h - 1));     // the j-th index with (i & h) == 0
            const float a = v[i], b = v[i + h];
            v[i] = __fadd_rn(a, b);
            v[i + h] = __fsub_rn(a, b);
        }
        __syncthreads();
    }
    for (int i = threadIdx.x; i < block; i += blockDim.x)
        out[off + i] = __half_as_ushort(__float2half_rn(__fmul_rn(v[i], scale)));
}

}  // namespace

cudaError_t launch_hadamard(const uint16_t* x, int M, int64_t K, int block, uint16_t* out, cudaStream_t s) {
    int m = 0;
    while ((1 << m) < block) ++m;
    // 2^(-m/2), or 2^(-(m+1)/2) times the fp32 nearest to sqrt(2) for odd m
    const float sqrt2 = 1.41421356237309504880f;
    const float scale = (m % 2) ? ldexpf(sqrt2, -(m + 1) / 2) : ldexpf(1.0f, -(m / 2));
    const int threads = block / 2 < 512 ? block / 2 : 512;
    const dim3 grid(static_cast<unsigned>(K / block), static_cast<unsigned>(M));
    const size_t smem = static_cast<size_t>(block) * sizeof(float);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, hadamard_kernel, x, K, block, m, scale, out);
}

}  // namespace pn
