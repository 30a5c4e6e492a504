// pn_prefill.cu -- the large-M (prefill) path: PN rows rebuilt as fp16 in a
// transient buffer, then an fp16 GEMM on the fifth-generation tensor cores.
//
// What is computed (tensorless docs, "What the fork adds": for prefill the
// engine dequantizes the weights and runs a chunked GEMM; v100-skinny README,
// "How QPN works": above the skinny band the weights are rebuilt transiently
// from the packed codes and never kept): y[m][r] = sum_k w16[r][k] * x[m][k],
// where w16 is the exact decode d * (n - z) rounded once to fp16 (nearest,
// ties to even), accumulated in fp32.
//
// Design (GB300-first):
//  * unpack_f16_kernel: one thread per code word, exact fp32 product, one
//    rounding to fp16, half2 stores.  Memory-bound; it runs once per chunk of
//    rows, so at prefill sizes it is a small fraction of the GEMM.
//  * gemm_f16_kernel: persistent, one CTA per SM, output tiles of 128 rows x
//    256 tokens taken round-robin (token tile fastest, so the CTAs working at
//    one time share few weight tiles and the rebuilt weights cross HBM about
//    once).  Warp 0 lane 0 streams 64-wide K slices of the weight and
//    activation tiles into a 4-stage shared-memory ring with 2-D TMA
//    (128-byte swizzle, the layout the MMA reads directly); warp 1 lane 0
//    issues tcgen05.mma (kind::f16, M = 128, N = 256, K = 16) into one of two
//    fp32 accumulators of 256 TMEM columns each and hands every stage back
//    with tcgen05.commit; warps 2-5 read a finished accumulator (one weight
//    row per thread, tcgen05.ld) and store y while the MMAs fill the other.
//  * Every mbarrier wait is bounded in time; a CTA that gives up records
//    PN_ETIMEOUT, lets its copies and MMAs in flight finish (bounded), frees
//    its TMEM and returns.
#include <cstdint>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pn_device.cuh"
#include "pn_internal.h"

namespace pn {
namespace {

// The same copy with an L2 eviction policy (a createpolicy value) for the
// lines it reads.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* tmap, int x, int y, uint32_t bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(policy) : "memory");
}

// L2 policy: keep the lines this thread reads (evict them last).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}


// ------------------------------------------------------------- unpack f16 --

template <int TYPE>
__global__ void unpack_f16_kernel(const uint8_t* __restrict__ W, int64_t N, int64_t nb,
                                  __half2* __restrict__ w16) {
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
        // weights 2c (low half) and 2c + 1 (high half) are adjacent: one half2
        __half2* out = w16 + (blk * F::kPerBlock + j * F::kPerWord) / 2;
        constexpr uint32_t kMask = (1u << F::kBits) - 1u;
#pragma unroll
        for (int c = 0; c < F::kPerWord / 2; ++c) {
            const int lo = static_cast<int>((word >> (F::kBits * c)) & kMask);
            const int hi = static_cast<int>((word >> (16 + F::kBits * c)) & kMask);
            out[c] = __halves2half2(__float2half_rn(__fmul_rn(d, static_cast<float>(lo - F::kZero))),
                                    __float2half_rn(__fmul_rn(d, static_cast<float>(hi - F::kZero))));
        }
    }
}

// ------------------------------------------------------------------- GEMM --

constexpr int kTileRows = 128;                       // weight rows per tile (MMA M)
constexpr int kTileTokens = 256;                     // tokens per tile (MMA N)
constexpr int kKStep = 64;                           // K per stage: one 128-byte row of fp16
constexpr int kMmaK = 16;                            // K per tcgen05.mma, kind::f16
constexpr int kStages = 4;
constexpr int kThreads = 192;                        // producer, MMA issuer, 4 epilogue warps
constexpr int kAccBufs = 2;                          // TMEM accumulators (epilogue overlaps MMAs)
constexpr int kABytes = kTileRows * kKStep * 2;      // 16384
constexpr int kBBytes = kTileTokens * kKStep * 2;    // 32768
constexpr int kStageBytes = kABytes + kBBytes;       // 49152
constexpr int kBarOffset = kStages * kStageBytes;    // 196608
constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 1;   // ring full / empty, accumulator full / empty, drain
constexpr int kTmemSlot = kBarOffset + kNumBars * 8; // TMEM base address written by tcgen05.alloc
constexpr int kAbortSlot = kTmemSlot + 4;
constexpr int kSmemUsed = kAbortSlot + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;         // slack to align the ring to 1024 bytes
constexpr uint32_t kTmemCols = kAccBufs * kTileTokens;   // two fp32 accumulators of 128 lanes x 256 columns
constexpr uint32_t kStatusTimeout = 5;               // PN_ETIMEOUT
constexpr uint64_t kDrainLimitNs = 200ull * 1000 * 1000;

static_assert(kStageBytes % 1024 == 0 && kABytes % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
static_assert(kSmemBytes <= 227 * 1024, "fits one SM's shared memory");
static_assert(kTileRows == 128 && kTileTokens % 16 == 0 && kTileTokens <= 256, "a valid cta_group::1 MMA shape");

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits 4-5
// = 1), A and B fp16 (bits 7-9 and 10-12 = 0), both K-major (bits 15 and 16 =
// 0), N / 8 in bits 17-22, M / 16 in bits 24-28.
constexpr uint32_t kInstrDesc = (1u << 4) | (static_cast<uint32_t>(kTileTokens >> 3) << 17) |
                                (static_cast<uint32_t>(kTileRows >> 4) << 24);

// Shared-memory matrix descriptor of a K-major tile that TMA wrote with the
// 128-byte swizzle: 128-byte rows, 8-row atoms of 1024 bytes (stride byte
// offset 1024), leading byte offset unused by this layout (encoded 1),
// descriptor version 1 (bits 46-47), swizzle mode 2 = 128-byte (bits 61-63).
// Advancing the start address by 32 bytes selects the next 16 K values.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_slot), "r"(cols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (TMEM) = A B^T (+ D if accumulate): A, B from shared-memory descriptors.
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %3, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n\t}"
        :: "r"(tmem_d), "l"(da), "l"(db), "r"(accumulate), "r"(kInstrDesc) : "memory");
}

// One arrival on `bar` once every tcgen05.mma this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes
// 32 w .. 32 w + 31; taddr carries the warp's first lane in bits 16-31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct GemmParams {
    CUtensorMap amap;          // rebuilt weights, fp16 [rows][K]; box 64 x 128
    CUtensorMap bmap;          // activations, fp16 [M][K]; box 64 x 256
    float* y;                  // y[m * ldy + r] for r < rows, m < M
    int64_t ldy;
    int rows;
    int M;
    int K;
    int tiles_tok;             // ceil(M / 256)
    int tiles;                 // tiles_tok * ceil(rows / 128)
    uint32_t* status;
    uint64_t timeout_ns;
    int stall_first_step;      // testing aid: see pn_set_test_stall
};

// Waits for phase `parity` of an mbarrier; false after limit_ns, or at once
// when the CTA has aborted (abort may be null).  `nap` lets a thread that
// has nothing else to do leave its issue slots to the others.
__device__ bool wait_phase(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile uint32_t* abort,
                           bool nap) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (nap) __nanosleep(64);
        if (mbar_try_wait(bar, parity)) return true;
        if (abort && *abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ void raise_abort(const GemmParams& P, volatile uint32_t* abort) {
    *abort = 1u;
    atomicCAS(P.status, 0u, kStatusTimeout);
}

__global__ void __launch_bounds__(kThreads, 1) gemm_f16_kernel(const __grid_constant__ GemmParams P) {
    extern __shared__ uint8_t smem_raw[];
    // the swizzled ring wants 1024-byte alignment
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t bar0 = base + kBarOffset;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto acc_full = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
    auto acc_empty = [&](int a) { return bar0 + 8u * (2 * kStages + kAccBufs + a); };
    const uint32_t drain = bar0 + 8u * (2 * kStages + 2 * kAccBufs);
    volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(smem + kAbortSlot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = (P.K + kKStep - 1) / kKStep;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < kAccBufs; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), 4);       // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *abort = 0u;
        fence_mbar_init();
        prefetch_tensormap(&P.amap);
        prefetch_tensormap(&P.bmap);
    }
    if (warp == 0) {                          // the whole warp allocates the accumulators
        tmem_alloc(base + kTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTmemSlot);

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------ producer --
            int it = 0;                       // K slices issued, over all tiles
            bool stop = false;
            // the activations are read again for every weight-row tile: keep
            // them in L2 (the weight rows are read by the 16 token tiles of a
            // row tile at about the same time, and y is written streaming)
            const uint64_t keep = l2_policy_evict_last();
            for (int t = blockIdx.x; t < P.tiles && !stop; t += gridDim.x) {
                const int tok0 = (t % P.tiles_tok) * kTileTokens;
                const int row0 = (t / P.tiles_tok) * kTileRows;
                for (int kb = 0; kb < nk; ++kb) {
                    const int s = it % kStages;
                    if (it >= kStages &&
                        !wait_phase(empty(s), static_cast<uint32_t>((it / kStages) - 1) & 1u, P.timeout_ns, abort,
                                    false)) {
                        raise_abort(P, abort);
                        stop = true;
                        break;
                    }
                    if (*abort) { stop = true; break; }
                    const uint32_t a = base + s * kStageBytes;
                    mbar_arrive_expect_tx(full(s), kStageBytes);
                    // (testing aid: with stall_first_step the first slice's
                    // bytes are announced but never copied; its wait can only
                    // time out)
                    if (!(P.stall_first_step && it == 0)) {
                        tma_load_2d(a, &P.amap, kb * kKStep, row0, full(s));
                        tma_load_2d_hint(a + kABytes, &P.bmap, kb * kKStep, tok0, full(s), keep);
                    }
                    ++it;
                }
            }
            // every copy this thread started lands before the CTA can exit:
            // stage s was last filled by the largest issue i < it with i %
            // kStages == s (after a normal run the MMA thread waited for all)
            for (int s = 0; s < kStages; ++s) {
                if (it <= s) continue;
                const int last = s + kStages * ((it - 1 - s) / kStages);
                if (P.stall_first_step && last == 0) continue;   // never copied
                wait_phase(full(s), static_cast<uint32_t>(last / kStages) & 1u, kDrainLimitNs, nullptr, false);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ----------------------------------------------------- MMA issue --
            int it = 0, local = 0;
            bool stop = false;
            for (int t = blockIdx.x; t < P.tiles && !stop; t += gridDim.x, ++local) {
                const int acc = local & 1;
                // the epilogue has emptied this accumulator's previous tile
                if (local >= kAccBufs &&
                    !wait_phase(acc_empty(acc), static_cast<uint32_t>((local >> 1) + 1) & 1u, P.timeout_ns, abort,
                                false)) {
                    raise_abort(P, abort);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * kTileTokens);
                for (int kb = 0; kb < nk; ++kb) {
                    const int s = it % kStages;
                    if (!wait_phase(full(s), static_cast<uint32_t>(it / kStages) & 1u, P.timeout_ns, abort, false)) {
                        raise_abort(P, abort);
                        stop = true;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a = base + s * kStageBytes;
                    const uint32_t b = a + kABytes;
#pragma unroll
                    for (int kk = 0; kk < kKStep / kMmaK; ++kk)
                        mma_f16(d, smem_desc_sw128(a + kk * kMmaK * 2), smem_desc_sw128(b + kk * kMmaK * 2),
                                (kb | kk) != 0 ? 1u : 0u);
                    mma_commit(empty(s));     // the stage is free once these MMAs have read it
                    ++it;
                }
                if (!stop) mma_commit(acc_full(acc));
            }
            mma_commit(drain);                // every MMA of this CTA finished (also after an abort)
        }
    } else {
        // --------------------------------------------------------- epilogue --
        const int q = warp & 3;               // TMEM lane quadrant this warp may read
        int local = 0;
        for (int t = blockIdx.x; t < P.tiles; t += gridDim.x, ++local) {
            const int acc = local & 1;
            bool ok = true;
            if (lane == 0)
                ok = wait_phase(acc_full(acc), static_cast<uint32_t>(local >> 1) & 1u, P.timeout_ns, abort, true);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) {
                if (lane == 0) raise_abort(P, abort);
                break;
            }
            tc_fence_after_sync();
            const int tok0 = (t % P.tiles_tok) * kTileTokens;
            const int row = (t / P.tiles_tok) * kTileRows + q * 32 + lane;
            const uint32_t taddr = tmem + static_cast<uint32_t>(acc * kTileTokens) + (static_cast<uint32_t>(q * 32) << 16);
            for (int c = 0; c < kTileTokens; c += 32) {
                if (tok0 + c >= P.M) break;   // warp-uniform
                uint32_t v[32];
                tmem_ld32(taddr + static_cast<uint32_t>(c), v);
                tmem_wait_ld();
                if (row < P.rows) {
                    float* yc = P.y + static_cast<int64_t>(tok0 + c) * P.ldy + row;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (tok0 + c + j < P.M) __stcs(yc + static_cast<int64_t>(j) * P.ldy, __uint_as_float(v[j]));
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(acc));
        }
    }
    __syncwarp();
    // ------------------------------------------------------------ teardown --
    // no MMA may still write TMEM when it is freed
    if (threadIdx.x == 0) wait_phase(drain, 0u, kDrainLimitNs, nullptr, true);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// fp16 matrix [rows][K] (K-major), box = 64 K values (128 bytes) x box_rows,
// 128-byte swizzle; boxes past the edge are zero-filled.
bool encode_k_major(CUtensorMap* map, const void* p, int64_t rows, int64_t K, int box_rows) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKStep), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estride[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(p), dims, strides, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_unpack_f16(int type, const void* W, int64_t N, int64_t nb, uint16_t* w16, cudaStream_t s) {
    const int threads = 256;
    const int64_t words = N * nb * kWordsPerBlock;
    int64_t blocks = (words + threads - 1) / threads;
    if (blocks > 65535LL * 16) blocks = 65535LL * 16;
    if (blocks < 1) blocks = 1;
    const uint8_t* Wb = static_cast<const uint8_t*>(W);
    __half2* out = reinterpret_cast<__half2*>(w16);
    if (type == kPn3t) unpack_f16_kernel<kPn3t><<<static_cast<int>(blocks), threads, 0, s>>>(Wb, N, nb, out);
    else unpack_f16_kernel<kPn4t><<<static_cast<int>(blocks), threads, 0, s>>>(Wb, N, nb, out);
    return cudaGetLastError();
}

int gemm_f16_tile_rows() { return kTileRows; }

cudaError_t launch_gemm_f16(const uint16_t* w16, int64_t rows, int64_t K, const uint16_t* x, int64_t M,
                            float* y, int64_t ldy, uint32_t* status, int num_sms, uint64_t timeout_ns,
                            int stall, cudaStream_t s) {
    if (rows < 1 || M < 1 || K < 1 || K > INT32_MAX || M > INT32_MAX) return cudaErrorInvalidValue;
    const int64_t gy = (rows + kTileRows - 1) / kTileRows;
    const int64_t gx = (M + kTileTokens - 1) / kTileTokens;
    if (gx * gy > INT32_MAX) return cudaErrorInvalidValue;
    GemmParams P{};
    if (!encode_k_major(&P.amap, w16, rows, K, kTileRows) || !encode_k_major(&P.bmap, x, M, K, kTileTokens))
        return cudaErrorInvalidValue;
    P.y = y;
    P.ldy = ldy;
    P.rows = static_cast<int>(rows);
    P.M = static_cast<int>(M);
    P.K = static_cast<int>(K);
    P.tiles_tok = static_cast<int>(gx);
    P.tiles = static_cast<int>(gx * gy);
    P.status = status;
    P.timeout_ns = timeout_ns;
    P.stall_first_step = stall;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = set_smem_limit_once(gemm_f16_kernel, kSmemBytes, smem_set); e != cudaSuccess) return e;
    const int grid = P.tiles < num_sms ? P.tiles : (num_sms > 0 ? num_sms : 1);   // persistent: one CTA per SM
    gemm_f16_kernel<<<grid, kThreads, kSmemBytes, s>>>(P);
    return cudaGetLastError();
}

}  // namespace pn
