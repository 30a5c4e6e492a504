// pn_internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/pn.h"

namespace pn {

// Records e as the CUDA error behind this thread's latest PN_ECUDA (see
// pn_last_cuda_error), clears the runtime's last error and returns PN_ECUDA.
pn_status cuda_error(cudaError_t e);

constexpr int kMaxM = 16;
constexpr int kMaxLayer = 8;

// ---------------------------------------------------------- work split --
// The GEMV kernels number a call's work units (row tile x 8-block chunk)
// tensor by tensor and give every thread block one contiguous range.  Units
// of different tensors cost different decode work (a pn3t block-row holds 80
// codes, a pn4t one 64), so the ranges split the call's total cost, not its
// unit count, evenly: tensor e's units are [base[e], base[e+1]) at w[e] each,
// and block c's range starts at the first unit whose cumulative cost reaches
// total * c / grid.  With one weight for every tensor this is the plain even
// split of the units.  Computed on the host; the kernels read each block's
// first unit from a table in their parameters.
struct CostSplit {
    uint32_t base[kMaxLayer + 1];      // base[count] = all units
    uint64_t cbase[kMaxLayer + 1];     // cost of the units before tensor e; cbase[count] = total
    uint32_t w[kMaxLayer];             // cost of one unit of tensor e (>= 1)
    int count;
    int grid;

    // First unit of block c's range; start(grid) is the end of the last one.
    // Non-decreasing in c.
    uint32_t start(int c) const {
        if (c >= grid) return base[count];
        const uint64_t target = cbase[count] * static_cast<uint64_t>(c) / static_cast<uint64_t>(grid);
        int e = 0;
        while (e + 1 < count && cbase[e + 1] <= target) ++e;
        const uint64_t u = base[e] + (target - cbase[e] + w[e] - 1) / w[e];
        return u < base[e + 1] ? static_cast<uint32_t>(u) : base[e + 1];
    }

    // Tensor e has `units` units at cost `cost` each (in call order).
    void add(uint32_t units, uint32_t cost) {
        w[count] = cost;
        base[count + 1] = base[count] + units;
        cbase[count + 1] = cbase[count] + static_cast<uint64_t>(units) * cost;
        ++count;
    }

    // The largest grid <= max_grid whose ranges all hold at least
    // min_units units (so a tile of at most min_units units has at most two
    // owners); at least 1.
    int fit_grid(int max_grid, uint32_t min_units) {
        const uint32_t units = base[count];
        int g = static_cast<int>(units / (min_units > 0 ? min_units : 1));
        g = g < max_grid ? g : max_grid;
        for (grid = g < 1 ? 1 : g; grid > 1; --grid) {
            bool ok = true;
            uint32_t prev = 0;
            for (int c = 1; c <= grid && ok; ++c) {
                const uint32_t next = start(c);
                ok = next - prev >= min_units;
                prev = next;
            }
            if (ok) break;
        }
        return grid;
    }
};

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device (the attribute belongs to each device's copy of
// the kernel); `done` holds one bit per device already set.
template <typename Kernel>
cudaError_t set_smem_limit_once(Kernel* kernel, int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// One tensor of a GEMV launch, as the host hands it to a kernel.
struct GemvTensor {
    const uint8_t* W;       // PN rows, row stride nb * 34 bytes
    const uint16_t* x;      // fp16 [M][K]
    float* y;               // fp32 [M][N]
    int type;               // 124 pn3t / 125 pn4t
    int N;                  // rows
    int nb;                 // blocks per row (K / weights per block)
};

// Block Hadamard rotation of fp16 activations [M][K] (block = 2^m dividing K,
// 2 <= block <= 4096); out may equal x.
cudaError_t launch_hadamard(const uint16_t* x, int M, int64_t K, int block, uint16_t* out, cudaStream_t s);

cudaError_t launch_unpack(int type, const void* W, int64_t N, int64_t nb, float* w, cudaStream_t s);
cudaError_t launch_pack(int type, const float* w, int64_t N, int64_t nb, void* W, cudaStream_t s);

// Prefill: PN rows -> fp16 (exact decode rounded once), and the fp16 GEMM
// y[m * ldy + r] = sum_k w16[r][k] x[m][k] on the tcgen05 tensor cores (w16,
// x 16-byte aligned, K a multiple of 8; rows a multiple of
// gemm_f16_tile_rows() except the last chunk).
cudaError_t launch_unpack_f16(int type, const void* W, int64_t N, int64_t nb, uint16_t* w16, cudaStream_t s);
cudaError_t launch_gemm_f16(const uint16_t* w16, int64_t rows, int64_t K, const uint16_t* x, int64_t M,
                            float* y, int64_t ldy, uint32_t* status, int num_sms, uint64_t timeout_ns,
                            int stall, cudaStream_t s);
int gemm_f16_tile_rows();

// Read-bandwidth probe: every 16-byte word of `count` ranges read once, XORs into sink[e].
cudaError_t launch_read_ranges(const void* const* ptrs, const size_t* bytes, int count, uint32_t* sink,
                               int num_sms, cudaStream_t s);

// CUDA-core GEMV: any nb, W and x 2-byte aligned, y 4-byte aligned.
cudaError_t launch_gemv_simt(const GemvTensor& t, int M, cudaStream_t s);

// Workspace of the tensor-core GEMVs (offsets in bytes), every completed call
// leaves it zeroed:
//   status    uint32 status word (padded to 256 bytes);
//   tagged    one-/two-token kernel: per thread-block boundary, one
//             [16 rows][2 tokens] slot of 64-bit {tag, value} words through
//             which a block hands its part of a shared tile to its neighbour;
//   partials  batch kernel: per boundary, two [16 rows][8 tokens] fp32 slots;
//   counters  batch kernel: one uint32 per boundary.
struct WorkspaceLayout {
    size_t status = 0;
    size_t tagged = 0;
    size_t partials = 0;
    size_t counters = 0;
    size_t total = 0;
};
WorkspaceLayout workspace_layout(int num_sms);

// Tensor-core GEMV for M <= 2 over `count` tensors (every one with nb % 8 == 0
// and W, x 16-byte aligned): one block per SM streams a contiguous range of
// units through a TMA ring that its warps share.
// With rot_block (32 .. 1024, a power of two dividing every K) the kernel
// first rotates each tensor's activations as pn_hadamard would (fused) and
// multiplies the rotated values; 0 = no rotation.
cudaError_t launch_gemv_stream(const GemvTensor* t, int count, int M, uint32_t* status, uint64_t* tagged,
                               int num_sms, uint64_t timeout_ns, int stall, cudaStream_t s, int rot_block = 0);
// Whether a call on these tensors keeps their activations resident in the
// one-/two-token kernel's shared memory beside its full ring.
bool stream_resident_fits(const GemvTensor* t, int count, int M, int num_sms);
// Whether a fused-rotation call on these tensors fits the kernel's shared
// memory (the rotated activations of a block's tensors stay resident).
bool stream_rotation_fits(const GemvTensor* t, int count, int M, int num_sms, int rot_block);
int stream_max_ctas(int num_sms);
size_t stream_tagged_bytes(int num_sms);
// Longest row (in 8-block chunks) the one-/two-token kernel takes.
int stream_max_chunks();

// Tensor-core GEMV for 3 <= M <= 16 (same eligibility): thread blocks share
// each staged activation chunk among eight tiles.
cudaError_t launch_gemv_tc(const GemvTensor* t, int count, int M, uint32_t* status, float* partials,
                           uint32_t* counters, int num_sms, uint64_t timeout_ns, int stall, cudaStream_t s);
int tc_max_ctas(int num_sms);
// The tensor-core GEMV's split of the units of tensors t[0 .. count) over its
// thread blocks (host only): *grid blocks, block c taking units
// [starts[c], starts[c + 1]); false when the tensors are empty or too large.
bool tc_split(const GemvTensor* t, int count, int M, int num_sms, int* grid, uint32_t* starts);
size_t tc_partial_bytes(int num_sms);

// CUDA-core GEMV for 1 <= M <= 8 on the same TMA-staged rows (same
// eligibility, rows of at most ffma_max_chunks() chunks): the FMA-pipe side
// of the tensor-core comparison.  Uses only the workspace's status word.
cudaError_t launch_gemv_ffma(const GemvTensor* t, int count, int M, uint32_t* status, int num_sms,
                             uint64_t timeout_ns, cudaStream_t s);
int ffma_max_chunks();

// Host-side checks of a one-tensor GEMV, the same ones pn_gemv_ex makes before
// it launches anything.  On PN_OK, *uses_workspace tells whether the call
// would launch a tensor-core kernel (which reads and writes the workspace; the
// CUDA-core kernel does not, nor does a call with N = 0).
pn_status gemv_check(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int M, float* y,
                     int algo, bool* uses_workspace);

}  // namespace pn
