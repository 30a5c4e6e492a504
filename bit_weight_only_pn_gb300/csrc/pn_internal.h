// pn_internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pn {

constexpr int kMaxM = 8;
constexpr int kMaxLayer = 8;

// One tensor of a GEMV launch, as the host hands it to a kernel.
struct GemvTensor {
    const uint8_t* W;       // PN rows, row stride nb * 34 bytes
    const uint16_t* x;      // fp16 [M][K]
    float* y;               // fp32 [M][N]
    int type;               // 124 pn3t / 125 pn4t
    int N;                  // rows
    int nb;                 // blocks per row (K / weights per block)
};

cudaError_t launch_unpack(int type, const void* W, int64_t N, int64_t nb, float* w, cudaStream_t s);
cudaError_t launch_pack(int type, const float* w, int64_t N, int64_t nb, void* W, cudaStream_t s);

// CUDA-core GEMV: any nb, W and x 2-byte aligned, y 4-byte aligned.
cudaError_t launch_gemv_simt(const GemvTensor& t, int M, cudaStream_t s);

// Workspace layout of the tensor-core GEMV (all offsets in bytes).
struct WorkspaceLayout {
    size_t status = 0;        // uint32 status word (+ padding to 256)
    size_t partials = 256;    // float slots [boundary][side][16 rows x 8 tokens] (batch kernel)
    size_t counters = 0;      // uint32 per thread-block boundary (batch kernel)
    size_t tagged = 0;        // 64-bit {value, tag} words [boundary][16 rows x 2 tokens] (warp kernel)
    size_t total = 0;
};
WorkspaceLayout workspace_layout(int64_t total_tiles, int max_ctas);

// Tensor-core GEMV over `count` tensors (every one with nb % 8 == 0 and W, x
// 16-byte aligned).  `workspace` has the layout above, zeroed.
cudaError_t launch_gemv_tc(const GemvTensor* t, int count, int M, void* workspace,
                           size_t workspace_bytes, int num_sms, uint64_t timeout_ns, int stall,
                           cudaStream_t s, int* needs_bytes_out);

// Most thread blocks any tensor-core GEMV launch uses; the workspace holds a
// boundary slot pair for each.
int tc_max_ctas(int num_sms);

// Tensor-core GEMV for M <= 2 in which every warp streams its own units
// (same eligibility, same workspace layout as launch_gemv_tc).
cudaError_t launch_gemv_warp(const GemvTensor* t, int count, int M, void* workspace,
                             size_t workspace_bytes, int num_sms, uint64_t timeout_ns, int stall,
                             cudaStream_t s, int* needs_bytes_out);
int warp_max_ctas(int num_sms);

}  // namespace pn
