// pn_codec.cu -- PN block quantiser (pn_pack) and exact decoder (pn_unpack).
//
// Decode follows "Exact decode in fp32" (tensorless docs, "Why a P100-native
// weight format"): w = d * (n - z) as one IEEE fp32 multiply, exact, so the
// device decoder and any correct CPU decoder agree bit for bit, including the
// sign of zero.  Pack follows "Zero is a code, and the scale has a sign": the
// signed scale puts step -z on the block's largest-magnitude weight.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pn_device.cuh"
#include "pn_internal.h"

namespace pn {
namespace {

// One thread per (row, code word): reads the word as two 16-bit halves (a
// word is only 2-byte aligned in every other block) and the block scale, and
// writes the word's cpw weights.
template <int TYPE>
__global__ void unpack_kernel(const uint8_t* __restrict__ W, int64_t N, int64_t nb,
                              float* __restrict__ w) {
    using F = Format<TYPE>;
    const int64_t words = N * nb * kWordsPerBlock;
    const uint16_t* W16 = reinterpret_cast<const uint16_t*>(W);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t blk = i / kWordsPerBlock;          // global block index (row-major)
        const int j = static_cast<int>(i % kWordsPerBlock);
        const int64_t h0 = blk * (kBlockBytes / 2);      // 17 halves per block
        const float d = __half2float(__ushort_as_half(W16[h0]));
        const uint32_t word = static_cast<uint32_t>(W16[h0 + 1 + 2 * j]) |
                              (static_cast<uint32_t>(W16[h0 + 2 + 2 * j]) << 16);
        float* out = w + blk * F::kPerBlock + j * F::kPerWord;
#pragma unroll
        for (int c = 0; c < F::kPerWord; ++c) {
            const int shift = 16 * (c & 1) + F::kBits * (c >> 1);
            const int n = static_cast<int>((word >> shift) & ((1u << F::kBits) - 1u));
            out[c] = __fmul_rn(d, static_cast<float>(n - F::kZero));
        }
    }
}

// One thread per block: argmax |v| (first index on ties), d = fp16(a / -z),
// codes n = clamp(rint(v / d), -z, z - 1) + z, all divides IEEE round-to-nearest.
template <int TYPE>
__global__ void pack_kernel(const float* __restrict__ w, int64_t N, int64_t nb,
                            uint8_t* __restrict__ W) {
    using F = Format<TYPE>;
    constexpr int Z = F::kZero;
    const int64_t blocks = N * nb;
    uint16_t* W16 = reinterpret_cast<uint16_t*>(W);
    for (int64_t blk = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; blk < blocks;
         blk += (int64_t)gridDim.x * blockDim.x) {
        const float* v = w + blk * F::kPerBlock;
        int jmax = 0;
        float amax = fabsf(v[0]);
        for (int j = 1; j < F::kPerBlock; ++j) {
            const float m = fabsf(v[j]);
            if (m > amax) { amax = m; jmax = j; }
        }
        const float a = v[jmax];
        uint32_t dbits = 0;
        bool zero_block = (a == 0.0f);
        if (!zero_block) {
            dbits = __half_as_ushort(__float2half_rn(__fdiv_rn(a, static_cast<float>(-Z))));
            if ((dbits & 0x7FFFu) == 0) zero_block = true;               // underflow
            else if ((dbits & 0x7FFFu) == 0x7C00u) dbits = (dbits & 0x8000u) | 0x7BFFu;  // saturate
        }
        uint32_t words[kWordsPerBlock];
#pragma unroll
        for (int j = 0; j < kWordsPerBlock; ++j) words[j] = 0;
        const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(dbits)));
        for (int k = 0; k < F::kPerBlock; ++k) {
            int n = Z;
            if (!zero_block) {
                float q = rintf(__fdiv_rn(v[k], d));
                q = fminf(fmaxf(q, static_cast<float>(-Z)), static_cast<float>(Z - 1));
                n = static_cast<int>(q) + Z;
            }
            const int j = k / F::kPerWord, c = k % F::kPerWord;
            words[j] |= static_cast<uint32_t>(n) << (16 * (c & 1) + F::kBits * (c >> 1));
        }
        uint16_t* out = W16 + blk * (kBlockBytes / 2);
        out[0] = static_cast<uint16_t>(zero_block ? 0u : dbits);
#pragma unroll
        for (int j = 0; j < kWordsPerBlock; ++j) {
            out[1 + 2 * j] = static_cast<uint16_t>(words[j] & 0xFFFFu);
            out[2 + 2 * j] = static_cast<uint16_t>(words[j] >> 16);
        }
    }
}

int grid_for(int64_t items, int threads) {
    int64_t g = (items + threads - 1) / threads;
    return static_cast<int>(g < 1 ? 1 : (g > 65535 * 16 ? 65535 * 16 : g));
}

}  // namespace

cudaError_t launch_unpack(int type, const void* W, int64_t N, int64_t nb, float* w,
                          cudaStream_t s) {
    const int threads = 256;
    const int grid = grid_for(N * nb * kWordsPerBlock, threads);
    const uint8_t* Wb = static_cast<const uint8_t*>(W);
    if (type == kPn3t) unpack_kernel<kPn3t><<<grid, threads, 0, s>>>(Wb, N, nb, w);
    else unpack_kernel<kPn4t><<<grid, threads, 0, s>>>(Wb, N, nb, w);
    return cudaGetLastError();
}

cudaError_t launch_pack(int type, const float* w, int64_t N, int64_t nb, void* W,
                        cudaStream_t s) {
    const int threads = 128;
    const int grid = grid_for(N * nb, threads);
    uint8_t* Wb = static_cast<uint8_t*>(W);
    if (type == kPn3t) pack_kernel<kPn3t><<<grid, threads, 0, s>>>(w, N, nb, Wb);
    else pack_kernel<kPn4t><<<grid, threads, 0, s>>>(w, N, nb, Wb);
    return cudaGetLastError();
}

}  // namespace pn
