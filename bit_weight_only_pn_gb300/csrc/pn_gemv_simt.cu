// pn_gemv_simt.cu -- CUDA-core PN GEMV (any alignment, any whole number of blocks).
//
// The page's own kernel design ("One lane, one word", tensorless docs, "Why a
// P100-native weight format"): each lane owns one packed 32-bit code word and
// the activations it multiplies, loads the word once as two 16-bit halves
// ("Codes never straddle the two halves of a word" makes that safe in every
// block) and decodes it in registers.  Here each lane multiplies its codes'
// (n - z) by x in fp32, scales the word's sum by d, and the warp reduces the
// row with shuffles.  It serves shapes the tensor-core kernel does not take
// (rows that are not 16-byte aligned) and is the CUDA-core side of the
// tensor-core / CUDA-core comparison.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pn_device.cuh"
#include "pn_internal.h"

namespace pn {
namespace {

constexpr int kWarps = 8;

// MAXM: accumulators per lane (8 or 16), at least M.
template <int TYPE, int MAXM>
__global__ void __launch_bounds__(kWarps * 32)
gemv_simt_kernel(const uint8_t* __restrict__ W, int N, int nb, const uint16_t* __restrict__ x,
                 int M, float* __restrict__ y) {
    using F = Format<TYPE>;
    const int lane = threadIdx.x & 31;
    const int K = nb * F::kPerBlock;
    const uint16_t* W16 = reinterpret_cast<const uint16_t*>(W);
    const int64_t halves_per_row = static_cast<int64_t>(nb) * (kBlockBytes / 2);
    const int words = nb * kWordsPerBlock;
    for (int row = blockIdx.x * kWarps + (threadIdx.x >> 5); row < N; row += gridDim.x * kWarps) {
        float acc[MAXM];
#pragma unroll
        for (int m = 0; m < MAXM; ++m) acc[m] = 0.0f;
        const uint16_t* rw = W16 + row * halves_per_row;
        for (int wi = lane; wi < words; wi += 32) {
            const int blk = wi >> 3, j = wi & 7;
            const uint16_t* bp = rw + blk * (kBlockBytes / 2);
            const float d = __half2float(__ushort_as_half(__ldg(bp)));
            const uint32_t word = static_cast<uint32_t>(__ldg(bp + 1 + 2 * j)) |
                                  (static_cast<uint32_t>(__ldg(bp + 2 + 2 * j)) << 16);
            const int k0 = blk * F::kPerBlock + j * F::kPerWord;
            float part[MAXM];
#pragma unroll
            for (int m = 0; m < MAXM; ++m) part[m] = 0.0f;
#pragma unroll
            for (int c = 0; c < F::kPerWord; ++c) {
                const int shift = 16 * (c & 1) + F::kBits * (c >> 1);
                const float v = static_cast<float>(
                    static_cast<int>((word >> shift) & ((1u << F::kBits) - 1u)) - F::kZero);
#pragma unroll
                for (int m = 0; m < MAXM; ++m) {
                    if (m < M) {
                        const float xv = __half2float(__ushort_as_half(__ldg(x + (int64_t)m * K + k0 + c)));
                        part[m] = fmaf(v, xv, part[m]);    // (n - z) * x is exact in fp32
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < MAXM; ++m) acc[m] = fmaf(d, part[m], acc[m]);
        }
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            if (m < M) {
                float v = acc[m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                if (lane == 0) y[(int64_t)m * N + row] = v;
            }
        }
    }
}

}  // namespace

cudaError_t launch_gemv_simt(const GemvTensor& t, int M, cudaStream_t s) {
    int64_t blocks = (static_cast<int64_t>(t.N) + kWarps - 1) / kWarps;
    const int grid = static_cast<int>(blocks > 65535 * 8 ? 65535 * 8 : (blocks < 1 ? 1 : blocks));
    if (t.type == kPn3t) {
        if (M <= 8) gemv_simt_kernel<kPn3t, 8><<<grid, kWarps * 32, 0, s>>>(t.W, t.N, t.nb, t.x, M, t.y);
        else gemv_simt_kernel<kPn3t, 16><<<grid, kWarps * 32, 0, s>>>(t.W, t.N, t.nb, t.x, M, t.y);
    } else {
        if (M <= 8) gemv_simt_kernel<kPn4t, 8><<<grid, kWarps * 32, 0, s>>>(t.W, t.N, t.nb, t.x, M, t.y);
        else gemv_simt_kernel<kPn4t, 16><<<grid, kWarps * 32, 0, s>>>(t.W, t.N, t.nb, t.x, M, t.y);
    }
    return cudaGetLastError();
}

}  // namespace pn
