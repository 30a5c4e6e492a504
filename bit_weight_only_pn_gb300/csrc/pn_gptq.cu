// pn_gptq.cu -- GPTQ-style quantiser on the device (pn_gptq).
//
// The tensorless docs ("How Qwen3.8-27B-PN3 uses it") say the model's weights
// were quantised "GPTQ-style".  This is the published GPTQ procedure (Frantar
// et al., "GPTQ: Accurate Post-Training Quantization for Generative
// Pre-trained Transformers", ICLR 2023, Algorithm 1) with the PN blocks as its
// groups:
//
//   H = 2 X^T X + lambda I,  lambda = damp * mean(diag(2 X^T X))
//   U = upper Cholesky factor of H^-1        (H^-1 = U^T U)
//   for every column k in order:
//     at the first column of a block, each row's scale comes from the block's
//     current weights (rounded to fp32) by the signed-scale rule
//       (largest-magnitude weight a, first index on ties; d = fp16(a / -z))
//     q = clamp(rint(w[k] / d), -z, z - 1); the code is q + z
//     err = (w[k] - d q) / U[k][k];  w[j] -= err * U[k][j] for every j > k
//
// in fp64 (fp32 for the scale and the rounding, as the format's own rule).
// Every floating-point step here is one IEEE operation with round-to-nearest
// (explicit _rn intrinsics, so nothing is fused), in the order above, so the
// result does not depend on how the work is spread over threads: products may
// be formed in parallel, but each sum adds its terms in index order.  Rows
// are independent given U, so the
// quantisation runs one thread block per group of rows; the factorisations
// run column by column, each column's entries in parallel.
//
// Not on the GEMV's path: an offline tool, so the call is synchronous and
// simple rather than fast.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/pn.h"
#include "pn_device.cuh"
#include "pn_internal.h"

namespace pn {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = 8;

// H[i][j] = 2 * sum_t x[t][i] x[t][j], the sum in t order.
__global__ void hessian_kernel(const float* __restrict__ X, int64_t n, int64_t K, double* __restrict__ H) {
    const int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (idx >= K * K) return;
    const int64_t i = idx / K, j = idx % K;
    double s = 0.0;
    for (int64_t t = 0; t < n; ++t)
        s = __dadd_rn(s, __dmul_rn(static_cast<double>(X[t * K + i]), static_cast<double>(X[t * K + j])));
    H[idx] = __dmul_rn(2.0, s);
}

// lambda = damp * (sum of the diagonal in order) / K, added to the diagonal.
__global__ void damp_kernel(double* __restrict__ H, int64_t K, double damp) {
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    double m = 0.0;
    for (int64_t i = 0; i < K; ++i) m = __dadd_rn(m, H[i * K + i]);
    m = __ddiv_rn(m, static_cast<double>(K));
    for (int64_t i = 0; i < K; ++i) H[i * K + i] = __dadd_rn(H[i * K + i], __dmul_rn(damp, m));
}

// Cholesky a = c c^T, column j.  The sums keep the sequential order (k =
// 0, 1, ...); what runs in parallel is the loading and the products.  fp64 is
// slow on this part, so each subtraction is done once, by the thread that
// owns the sum.  The pivot: one block; products in shared memory by tiles,
// one thread subtracts them ...
constexpr int kPivotTile = 2048;
constexpr int kUnroll = 8;

__global__ void chol_pivot_kernel(const double* __restrict__ a, double* __restrict__ c, int64_t K, int64_t j,
                                  uint32_t* __restrict__ failed) {
    __shared__ double prod[kPivotTile];
    double s = a[j * K + j];
    for (int64_t k0 = 0; k0 < j; k0 += kPivotTile) {
        const int n = static_cast<int>(j - k0 < kPivotTile ? j - k0 : kPivotTile);
        for (int q = threadIdx.x; q < n; q += blockDim.x) {
            const double v = c[j * K + k0 + q];
            prod[q] = __dmul_rn(v, v);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int q = 0;
            for (; q + kUnroll <= n; q += kUnroll) {
                double p[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) p[u] = prod[q + u];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) s = __dsub_rn(s, p[u]);
            }
            for (; q < n; ++q) s = __dsub_rn(s, prod[q]);
        }
        __syncthreads();
    }
    if (threadIdx.x != 0) return;
    if (!(s > 0.0)) {
        *failed = 1u;
        s = 1.0;                        // keeps the rest finite; the call reports the failure
    }
    c[j * K + j] = __dsqrt_rn(s);
}

// ... and the entries below it, one thread per row i > j; each block stages
// 32-column slices of its rows and of row j in shared memory (coalesced
// loads), and every thread subtracts its row's products in order.
constexpr int kColThreads = 32;

__global__ void __launch_bounds__(kColThreads) chol_column_kernel(const double* __restrict__ a,
                                                                  double* __restrict__ c, int64_t K, int64_t j) {
    __shared__ double tile[kColThreads][33];
    __shared__ double cj[32];
    const int64_t i0 = j + 1 + static_cast<int64_t>(blockIdx.x) * kColThreads;
    const int64_t i = i0 + threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    double t = i < K ? a[i * K + j] : 0.0;
    for (int64_t k0 = 0; k0 < j; k0 += 32) {
        const int n = static_cast<int>(j - k0 < 32 ? j - k0 : 32);
        // warp w loads rows i0 + w, w + 4, ...: lane = column within the slice
        for (int r = warp; r < kColThreads; r += kColThreads / 32) {
            const int64_t row = i0 + r;
            tile[r][lane] = (row < K && lane < n) ? c[row * K + k0 + lane] : 0.0;
        }
        if (threadIdx.x < 32) cj[threadIdx.x] = lane < n ? c[j * K + k0 + lane] : 0.0;
        __syncthreads();
        if (i < K)
            for (int q = 0; q < n; ++q) t = __dsub_rn(t, __dmul_rn(tile[threadIdx.x][q], cj[q]));
        __syncthreads();
    }
    if (i < K) c[i * K + j] = __ddiv_rn(t, c[j * K + j]);
}

// inv = a^-1 from a = c c^T, one thread per column: c y = e_col by forward
// substitution, then c^T x = y by back substitution.  y lives in tmp[i][col].
// The operands of kUnroll terms are loaded before they are subtracted in order.
__global__ void spd_inverse_kernel(const double* __restrict__ c, double* __restrict__ inv,
                                   double* __restrict__ tmp, int64_t K) {
    const int64_t col = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (col >= K) return;
    for (int64_t i = 0; i < K; ++i) {
        double s = (i == col) ? 1.0 : 0.0;
        int64_t k = 0;
        for (; k + kUnroll <= i; k += kUnroll) {
            double cv[kUnroll], tv[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                cv[u] = c[i * K + k + u];
                tv[u] = tmp[(k + u) * K + col];
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) s = __dsub_rn(s, __dmul_rn(cv[u], tv[u]));
        }
        for (; k < i; ++k) s = __dsub_rn(s, __dmul_rn(c[i * K + k], tmp[k * K + col]));
        tmp[i * K + col] = __ddiv_rn(s, c[i * K + i]);
    }
    for (int64_t i = K - 1; i >= 0; --i) {
        double s = tmp[i * K + col];
        int64_t k = i + 1;
        for (; k + kUnroll <= K; k += kUnroll) {
            double cv[kUnroll], iv[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                cv[u] = c[(k + u) * K + i];
                iv[u] = inv[(k + u) * K + col];
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) s = __dsub_rn(s, __dmul_rn(cv[u], iv[u]));
        }
        for (; k < K; ++k) s = __dsub_rn(s, __dmul_rn(c[k * K + i], inv[k * K + col]));
        inv[i * K + col] = __ddiv_rn(s, c[i * K + i]);
    }
}

// u[k][j] = c[j][k] for j >= k (the upper factor, rows contiguous).
__global__ void transpose_lower_kernel(const double* __restrict__ c, double* __restrict__ u, int64_t K) {
    const int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (idx >= K * K) return;
    const int64_t k = idx / K, j = idx % K;
    u[idx] = j >= k ? c[j * K + k] : 0.0;
}

// The signed-scale rule on one block's current weights: fp16 bits of d, or
// 0 for the zero block.
template <int TYPE>
__device__ uint16_t block_scale(const double* v) {
    using F = Format<TYPE>;
    int jmax = 0;
    float amax = fabsf(static_cast<float>(v[0]));
    for (int j = 1; j < F::kPerBlock; ++j) {
        const float m = fabsf(static_cast<float>(v[j]));
        if (m > amax) { amax = m; jmax = j; }
    }
    const float a = static_cast<float>(v[jmax]);
    if (a == 0.0f) return 0;
    uint16_t bits = __half_as_ushort(__float2half_rn(__fdiv_rn(a, static_cast<float>(-F::kZero))));
    if ((bits & 0x7FFFu) == 0) return 0;                                  // underflow: the zero block
    if ((bits & 0x7FFFu) == 0x7C00u) bits = static_cast<uint16_t>((bits & 0x8000u) | 0x7BFFu);   // saturate
    return bits;
}

// Rows r0 .. r0 + kRowsPerBlock - 1: W holds their fp64 working copy, u the
// upper factor; codes and scales go to the block's shared memory and each
// completed block is written as PN bytes.
template <int TYPE>
__global__ void __launch_bounds__(kThreads) gptq_rows_kernel(double* __restrict__ W, const double* __restrict__ u,
                                                             int64_t N, int64_t K, uint8_t* __restrict__ out) {
    using F = Format<TYPE>;
    constexpr int Z = F::kZero;
    __shared__ double err[kRowsPerBlock];
    __shared__ uint16_t dbits[kRowsPerBlock];
    __shared__ uint8_t codes[kRowsPerBlock][F::kPerBlock];
    const int64_t r0 = blockIdx.x * static_cast<int64_t>(kRowsPerBlock);
    const int rows = static_cast<int>(N - r0 < kRowsPerBlock ? N - r0 : kRowsPerBlock);
    const int64_t nb = K / F::kPerBlock;
    for (int64_t k = 0; k < K; ++k) {
        const int64_t b = k / F::kPerBlock;
        const int kk = static_cast<int>(k % F::kPerBlock);
        if (static_cast<int>(threadIdx.x) < rows) {
            double* w = W + (r0 + threadIdx.x) * K;
            if (kk == 0) dbits[threadIdx.x] = block_scale<TYPE>(w + b * F::kPerBlock);
            int code = Z;
            float wq = 0.0f;
            if (dbits[threadIdx.x] != 0) {
                const float d = __half2float(__ushort_as_half(dbits[threadIdx.x]));
                float q = rintf(__fdiv_rn(static_cast<float>(w[k]), d));
                q = fminf(fmaxf(q, static_cast<float>(-Z)), static_cast<float>(Z - 1));
                code = static_cast<int>(q) + Z;
                wq = __fmul_rn(d, q);
            }
            codes[threadIdx.x][kk] = static_cast<uint8_t>(code);
            err[threadIdx.x] = __ddiv_rn(__dsub_rn(w[k], static_cast<double>(wq)), u[k * K + k]);
        }
        __syncthreads();
        // every later column of every row: one subtraction per element and column k
        const int64_t span = K - k - 1;
        for (int64_t p = threadIdx.x; p < span * rows; p += kThreads) {
            const int r = static_cast<int>(p / span);
            const int64_t j = k + 1 + p % span;
            double* wj = W + (r0 + r) * K + j;
            *wj = __dsub_rn(*wj, __dmul_rn(err[r], u[k * K + j]));
        }
        if (kk == F::kPerBlock - 1 && static_cast<int>(threadIdx.x) < rows) {
            uint8_t* blk = out + ((r0 + threadIdx.x) * nb + b) * kBlockBytes;
            uint32_t words[kWordsPerBlock] = {};
            for (int j = 0; j < F::kPerBlock; ++j) {
                const int c = j % F::kPerWord;
                words[j / F::kPerWord] |= static_cast<uint32_t>(codes[threadIdx.x][j])
                                          << (16 * (c & 1) + F::kBits * (c >> 1));
            }
            const uint16_t d = dbits[threadIdx.x];
            blk[0] = static_cast<uint8_t>(d & 0xFFu);
            blk[1] = static_cast<uint8_t>(d >> 8);
            for (int wi = 0; wi < kWordsPerBlock; ++wi)
                for (int by = 0; by < 4; ++by) blk[2 + 4 * wi + by] = static_cast<uint8_t>(words[wi] >> (8 * by));
        }
        __syncthreads();
    }
}

__global__ void widen_kernel(const float* __restrict__ w, double* __restrict__ W, int64_t count) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        W[i] = static_cast<double>(w[i]);
}

struct GptqScratch {
    size_t h, c, inv, u, w, flag, total;
};

GptqScratch gptq_layout(int64_t N, int64_t K) {
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t kk = static_cast<size_t>(K) * static_cast<size_t>(K) * sizeof(double);
    GptqScratch L;
    L.h = 0;
    L.c = up(L.h + kk);
    L.inv = up(L.c + kk);
    L.u = up(L.inv + kk);                // also the substitution's tmp before it holds u
    L.w = up(L.u + kk);
    L.flag = up(L.w + static_cast<size_t>(N) * static_cast<size_t>(K) * sizeof(double));
    L.total = up(L.flag + sizeof(uint32_t));
    return L;
}

int blocks_for(int64_t count, int threads) {
    const int64_t b = (count + threads - 1) / threads;
    return static_cast<int>(b < 1 ? 1 : b);
}

}  // namespace
}  // namespace pn

extern "C" size_t pn_gptq_scratch_bytes(int64_t N, int64_t K) {
    if (N < 0 || K <= 0) return 0;
    return pn::gptq_layout(N, K).total;
}

extern "C" pn_status pn_gptq(int type, const float* w, int64_t N, int64_t K, const float* X, int64_t n, double damp,
                             void* W, void* scratch, size_t scratch_bytes, pn_stream stream) {
    if (type != PN_TYPE_PN3T && type != PN_TYPE_PN4T) return PN_EINVAL;
    const int bpb = pn::per_block(type);
    // (K x K work is launched as one thread per entry: K at most 65536)
    if (N < 0 || K <= 0 || K % bpb || n < 1 || !(damp > 0.0) || K > 65536 || N > (int64_t(1) << 34))
        return PN_EINVAL;
    if (N == 0) return PN_OK;
    if (!w || !X || !W || !scratch) return PN_EINVAL;
    if (reinterpret_cast<uintptr_t>(w) % 4 || reinterpret_cast<uintptr_t>(X) % 4 ||
        reinterpret_cast<uintptr_t>(scratch) % 256)
        return PN_EALIGN;
    const pn::GptqScratch L = pn::gptq_layout(N, K);
    if (scratch_bytes < L.total) return PN_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(scratch);
    double* H = reinterpret_cast<double*>(base + L.h);
    double* C = reinterpret_cast<double*>(base + L.c);
    double* Hi = reinterpret_cast<double*>(base + L.inv);
    double* U = reinterpret_cast<double*>(base + L.u);
    double* Wd = reinterpret_cast<double*>(base + L.w);
    uint32_t* failed = reinterpret_cast<uint32_t*>(base + L.flag);
    auto chol = [&](const double* a, double* c) {
        for (int64_t j = 0; j < K; ++j) {
            pn::chol_pivot_kernel<<<1, 256, 0, s>>>(a, c, K, j, failed);
            if (K - j - 1 > 0)
                pn::chol_column_kernel<<<pn::blocks_for(K - j - 1, pn::kColThreads), pn::kColThreads, 0, s>>>(a, c,
                                                                                                         K, j);
        }
    };
    cudaError_t e = cudaMemsetAsync(failed, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return pn::cuda_error(e);
    pn::hessian_kernel<<<pn::blocks_for(K * K, 256), 256, 0, s>>>(X, n, K, H);
    pn::damp_kernel<<<1, 1, 0, s>>>(H, K, damp);
    chol(H, C);
    pn::spd_inverse_kernel<<<pn::blocks_for(K, 32), 32, 0, s>>>(C, Hi, U, K);
    chol(Hi, C);
    pn::transpose_lower_kernel<<<pn::blocks_for(K * K, 256), 256, 0, s>>>(C, U, K);
    pn::widen_kernel<<<pn::blocks_for(N * K, 256) < 4096 ? pn::blocks_for(N * K, 256) : 4096, 256, 0, s>>>(
        w, Wd, N * K);
    const int grid = static_cast<int>((N + pn::kRowsPerBlock - 1) / pn::kRowsPerBlock);
    if (type == PN_TYPE_PN3T)
        pn::gptq_rows_kernel<pn::kPn3t><<<grid, pn::kThreads, 0, s>>>(Wd, U, N, K, static_cast<uint8_t*>(W));
    else
        pn::gptq_rows_kernel<pn::kPn4t><<<grid, pn::kThreads, 0, s>>>(Wd, U, N, K, static_cast<uint8_t*>(W));
    if ((e = cudaGetLastError()) != cudaSuccess) return pn::cuda_error(e);
    uint32_t bad = 0;
    if ((e = cudaMemcpyAsync(&bad, failed, sizeof(bad), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return pn::cuda_error(e);
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return pn::cuda_error(e);
    return bad ? PN_EINVAL : PN_OK;
}
