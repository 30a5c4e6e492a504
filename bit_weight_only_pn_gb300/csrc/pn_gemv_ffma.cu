// pn_gemv_ffma.cu -- PN decode GEMV on the CUDA cores for up to 8 tokens:
// the same TMA-staged rows as the tensor-core kernels, products on the FMA
// pipe instead of the tensor pipe.
//
// What is computed: y[m][r] = sum_k d_blk(r,k) * (n(r,k) - z) * x[m][k] (the
// decode GEMV of the tensorless docs, "Why a P100-native weight format", and
// its skinny verification batch, v100-skinny README, "How QPN works").  It
// exists to answer, by measurement, whether the tensor pipe beats the FMA
// pipe on this contraction at M = 8 tokens, so it is built to be a fair
// contender: weights stream through the same kind of TMA ring as the
// one-token kernel, every code pair is decoded once (LOP3 + HFMA2, the exact
// half2 (n - z, n' - z)) and feeds all M tokens, and each product goes
// through fma.rn.f32.f16 -- an fp16 x fp16 product (exact in fp32) added to an
// fp32 accumulator with one rounding, the same arithmetic as the tensor-core
// path, with no conversion instruction.  Each block's sum is scaled by its d
// in fp32 and added to the row's sum.
//
// Work: a unit is a 16-row tile x one 8-block chunk.  Each thread block (one
// per SM) takes a contiguous range of whole tiles (split on the host so that
// ranges hold the same number of units), so no tile is shared between
// blocks.  A producer warp's lanes copy units into a ring (weight box plus the
// chunk's activations of every token); eleven consumer warps take stages by
// ticket.  Lane (r, h) of a consumer computes row r of the tile over blocks
// 4h .. 4h+3 of the chunk for every token; the two halves are added with a
// shuffle, and a tile's chunk partials are added in chunk order in shared
// memory by the warp that finishes its last chunk.  Every wait is bounded.
#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pn_device.cuh"
#include "pn_internal.h"

namespace pn {
namespace {

constexpr int kConsumers = 11;
constexpr int kProducerWarp = kConsumers;
constexpr int kThreads = (kConsumers + 1) * 32;           // 384
constexpr int kStages = 12;                               // > kConsumers: see the consumer loop
constexpr int kIssueLanes = 12;                           // <= kStages
constexpr int kRows = 16;
constexpr int kChunkBlocks = 8;
constexpr int kChunkBytes = kChunkBlocks * kBlockBytes;   // 272
constexpr int kBoxWords = kChunkBytes / 4;                // 68
constexpr int kBoxBytes = kRows * kChunkBytes;            // 4352
constexpr int kMaxTok = 8;
constexpr int kXTokenBytes = kChunkBlocks * 80 * 2;       // 1280: one token's pn3t chunk (pn4t: 1024)
constexpr int kPartsLog2 = 6;
constexpr int kParts = 1 << kPartsLog2;                   // partial-sum slots (>= chunks of a row)
constexpr int kSlotFloats = kRows * kMaxTok;
constexpr int kMaxGrid = 512;
constexpr uint64_t kDrainLimitNs = 200ull * 1000 * 1000;
constexpr uint32_t kStatusTimeout = 5;
constexpr uint32_t kEnd = 0xFFFFFFFFu;
constexpr uint32_t kSuspendNs = 1000;
static_assert(kStages > kConsumers && kStages >= kIssueLanes, "ring depth");

__host__ __device__ constexpr int stage_bytes(int M) { return (kBoxBytes + M * kXTokenBytes + 127) / 128 * 128; }

struct Layout {
    int sbytes = 0, table = 0, full = 0, empty = 0, parts = 0, gens = 0, cnts = 0, misc = 0, total = 0;
    __host__ __device__ constexpr explicit Layout(int M) {
        sbytes = stage_bytes(M);
        table = kStages * sbytes;
        full = table + 16 * kStages;
        empty = full + 8 * kStages;
        parts = (empty + 8 * kStages + 15) / 16 * 16;
        gens = parts + kParts * kSlotFloats * 4;
        cnts = gens + 4 * kParts;
        misc = cnts + 4 * kParts;             // ticket (4), abort (4)
        total = misc + 16;
    }
};
static_assert(Layout(kMaxTok).total <= 227 * 1024, "fits one SM");

struct FTensor {
    const uint16_t* x;
    float* y;
    uint32_t unit_base;
    int N, K, type, chunks, tiles;
};

struct FParams {
    CUtensorMap wmap[kMaxLayer];
    FTensor t[kMaxLayer];
    int count, M, grid;
    uint32_t starts[kMaxGrid + 1];   // block c's units are [starts[c], starts[c + 1]) (whole tiles)
    uint32_t* status;
    uint64_t timeout_ns;
};

struct Rec {
    uint32_t tile, chunk_e, k_first, n_units;   // chunk_e: chunk | tensor << 24 | pn4t << 30
};

__device__ __forceinline__ void locate(const FParams& P, uint32_t u, int& e, int& tile, int& chunk) {
    e = 0;
    while (e + 1 < P.count && u >= P.t[e + 1].unit_base) ++e;
    const uint32_t rel = u - P.t[e].unit_base;
    const uint32_t ch = static_cast<uint32_t>(P.t[e].chunks);
    tile = static_cast<int>(rel / ch);
    chunk = static_cast<int>(rel - static_cast<uint32_t>(tile) * ch);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          const volatile uint32_t* abort_flag) {
    if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (__all_sync(0xFFFFFFFFu, mbar_wait_suspend(bar, parity, kSuspendNs))) return true;
        if (*abort_flag || globaltimer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                            const volatile uint32_t* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_wait_suspend(bar, parity, kSuspendNs)) return true;
        if ((abort_flag && *abort_flag) || globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// acc += (fp16 a) * (fp16 b) on the FMA pipe: the product is exact in fp32,
// the addition rounds once.
__device__ __forceinline__ void fma_h2(float& acc_lo_hi, uint32_t a, uint32_t b) {
    asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc_lo_hi) : "r"(a), "r"(b));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Code word j of block b of a staged row: blocks at even positions start 2
// bytes into an aligned word (realigned with a byte permute), odd ones are
// aligned.  EVEN is the parity of b.
template <bool EVEN>
__device__ __forceinline__ uint32_t code_word(const uint8_t* row, int b, int j) {
    const uint8_t* p = row + kBlockBytes * b + 2 + 4 * j;
    if constexpr (EVEN) {
        const uint8_t* a = p - 2;
        return prmt(lds_u32(a), lds_u32(a + 4), 0x5432u);
    } else {
        return lds_u32(p);
    }
}

// Lane (r, h): row r of the staged tile, blocks 4h .. 4h+3, tokens 0 .. M-1;
// acc[m] += the row's sum over those blocks for token m.
template <int TYPE>
__device__ __forceinline__ void unit_ffma(const uint8_t* stage, int M, int lane, float (&acc)[kMaxTok]) {
    using F = Format<TYPE>;
    constexpr int kP = F::kPairs;
    const int r = lane & 15, h = lane >> 4;
    const uint8_t* row = stage + r * kChunkBytes;
    const uint8_t* xs = stage + kBoxBytes;
    static_for<4>([&](auto ic) {
        constexpr int I = decltype(ic)::value;
        const int b = 4 * h + I;
        const float d = lds_half_as_float(row + kBlockBytes * b);
        float part[kMaxTok];
#pragma unroll
        for (int m = 0; m < kMaxTok; ++m) part[m] = 0.0f;
#pragma unroll
        for (int j = 0; j < kWordsPerBlock; ++j) {
            const uint32_t w = code_word<I % 2 == 0>(row, b, j);
            const uint32_t sh = w >> F::kHighShift;
            const int k0 = b * F::kPerBlock + j * F::kPerWord;      // the word's first activation
            static_for<kP>([&](auto pc) {
                constexpr int Pp = decltype(pc)::value;
                const uint32_t wv = decode_pair<TYPE, Pp>(w, sh);   // (n - z) of codes 2P, 2P + 1
#pragma unroll
                for (int m = 0; m < kMaxTok; ++m)
                    if (m < M) fma_h2(part[m], wv, lds_u32(xs + m * kXTokenBytes + 2 * (k0 + 2 * Pp)));
            });
        }
#pragma unroll
        for (int m = 0; m < kMaxTok; ++m) acc[m] = fmaf(d, part[m], acc[m]);
    });
}

__device__ __forceinline__ bool smem_wait_eq(const volatile uint32_t* p, uint32_t want, uint64_t limit_ns,
                                             const volatile uint32_t* abort_flag) {
    if (*p == want) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(32);
        if (*p == want) return true;
        if (*abort_flag || globaltimer_ns() - t0 > limit_ns) return false;
    }
}

__global__ void __launch_bounds__(kThreads, 1) gemv_ffma_kernel(const __grid_constant__ FParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    const Layout Lay(P.M);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t full0 = sbase + Lay.full, empty0 = sbase + Lay.empty;
    uint32_t* ticket = reinterpret_cast<uint32_t*>(smem + Lay.misc);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Lay.misc + 4);
    Rec* table = reinterpret_cast<Rec*>(smem + Lay.table);
    float* parts = reinterpret_cast<float*>(smem + Lay.parts);
    volatile uint32_t* gens = reinterpret_cast<volatile uint32_t*>(smem + Lay.gens);
    uint32_t* cnts = reinterpret_cast<uint32_t*>(smem + Lay.cnts);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_launch_dependents();
    for (int i = threadIdx.x; i < kParts; i += kThreads) {
        gens[i] = 0u;
        cnts[i] = 0u;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        *ticket = 0u;
        *abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t c0 = P.starts[blockIdx.x], c1 = P.starts[blockIdx.x + 1];
    const uint32_t n = c1 - c0;

    if (warp == kProducerWarp) {
        for (int e = lane; e < P.count; e += 32) prefetch_tensormap(&P.wmap[e]);
        const uint32_t total = n + kConsumers;
        bool ok = true, waited = false;
        uint32_t b0 = 0, filled_mask = 0;
        for (; b0 < total; b0 += kIssueLanes) {
            const uint32_t q = b0 + static_cast<uint32_t>(lane);
            bool mine_ok = true, filled = false;
            if (lane < kIssueLanes && q < total) {
                const uint32_t s = q % kStages;
                if (q >= static_cast<uint32_t>(kStages))
                    mine_ok = thread_wait(empty0 + 8 * s, ((q / kStages) - 1) & 1u, P.timeout_ns, abort_flag);
                if (mine_ok && q < n) {
                    int e, tile, chunk;
                    locate(P, c0 + q, e, tile, chunk);
                    const FTensor& T = P.t[e];
                    Rec rec;
                    rec.tile = static_cast<uint32_t>(tile);
                    rec.chunk_e = static_cast<uint32_t>(chunk) | (static_cast<uint32_t>(e) << 24) |
                                  (T.type == kPn3t ? 0u : 1u << 30);
                    rec.k_first = q - static_cast<uint32_t>(chunk);       // ranges hold whole tiles
                    rec.n_units = static_cast<uint32_t>(T.chunks);
                    table[s] = rec;
                    const int halves = kChunkBlocks * per_block(T.type);
                    mbar_arrive_expect_tx(full0 + 8 * s, kBoxBytes + P.M * halves * 2);
                    tma_load_2d(sbase + s * Lay.sbytes, &P.wmap[e], chunk * kBoxWords, tile * kRows, full0 + 8 * s);
                    if (!waited) griddep_wait();
                    waited = true;
                    const uint16_t* x = T.x + static_cast<int64_t>(chunk) * halves;
                    for (int m = 0; m < P.M; ++m)
                        bulk_g2s(sbase + s * Lay.sbytes + kBoxBytes + m * kXTokenBytes, x + static_cast<int64_t>(m) * T.K,
                                 halves * 2, full0 + 8 * s);
                    filled = true;
                } else if (mine_ok) {
                    table[s].tile = kEnd;
                    mbar_arrive(full0 + 8 * s);
                }
            }
            filled_mask = __ballot_sync(0xFFFFFFFFu, filled);
            ok = __all_sync(0xFFFFFFFFu, mine_ok);
            if (!ok) break;
        }
        if (!ok && lane == 0) {
            *abort_flag = 1u;
            atomicCAS(P.status, 0u, kStatusTimeout);
            const uint32_t end = b0 + kIssueLanes;
            for (uint32_t q = end > static_cast<uint32_t>(kStages) ? end - kStages : 0u; q < end && q < n; ++q) {
                const bool copied = q < b0 || ((filled_mask >> (q - b0)) & 1u) != 0u;
                if (copied) thread_wait(full0 + 8 * (q % kStages), (q / kStages) & 1u, kDrainLimitNs, nullptr);
            }
        }
        return;
    }

    griddep_wait();
    for (;;) {
        uint32_t k = 0;
        if (lane == 0) k = atomicAdd(ticket, 1u);
        k = __shfl_sync(0xFFFFFFFFu, k, 0);
        const uint32_t s = k % kStages, ph = k / kStages;
        // wait for ticket k - kStages to release the stage first, so its
        // parity-tested full barrier is at most one phase ahead
        if (k >= static_cast<uint32_t>(kStages) && !warp_wait(empty0 + 8 * s, (ph - 1) & 1u, P.timeout_ns, abort_flag)) {
            if (lane == 0) { *abort_flag = 1u; atomicCAS(P.status, 0u, kStatusTimeout); }
            return;
        }
        if (!warp_wait(full0 + 8 * s, ph & 1u, P.timeout_ns, abort_flag)) {
            if (lane == 0) {
                *abort_flag = 1u;
                atomicCAS(P.status, 0u, kStatusTimeout);
                thread_wait(full0 + 8 * s, ph & 1u, kDrainLimitNs, nullptr);
            }
            return;
        }
        const Rec rec = table[s];
        if (rec.tile == kEnd) return;
        float acc[kMaxTok];
#pragma unroll
        for (int m = 0; m < kMaxTok; ++m) acc[m] = 0.0f;
        const uint8_t* stage = smem + s * Lay.sbytes;
        if ((rec.chunk_e >> 30) == 0u) unit_ffma<kPn3t>(stage, P.M, lane, acc);
        else unit_ffma<kPn4t>(stage, P.M, lane, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        // blocks 0..3 (lanes 0..15) + blocks 4..7 (lanes 16..31)
#pragma unroll
        for (int m = 0; m < kMaxTok; ++m) acc[m] += __shfl_down_sync(0xFFFFFFFFu, acc[m], 16);
        const uint32_t slot = k & (kParts - 1), fslot = rec.k_first & (kParts - 1);
        bool ok = true;
        if (gens[slot] != (k >> kPartsLog2) || gens[fslot] != (rec.k_first >> kPartsLog2)) {
            if (lane == 0)
                ok = smem_wait_eq(gens + slot, k >> kPartsLog2, P.timeout_ns, abort_flag) &&
                     smem_wait_eq(gens + fslot, rec.k_first >> kPartsLog2, P.timeout_ns, abort_flag);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        }
        if (!ok) {
            if (lane == 0) { *abort_flag = 1u; atomicCAS(P.status, 0u, kStatusTimeout); }
            return;
        }
        if (lane < 16)
#pragma unroll
            for (int m = 0; m < kMaxTok; ++m) parts[slot * kSlotFloats + lane * kMaxTok + m] = acc[m];
        __syncwarp();
        uint32_t old = 0;
        if (lane == 0) old = atomicAdd(cnts + fslot, 1u);
        old = __shfl_sync(0xFFFFFFFFu, old, 0);
        if (old + 1 != rec.n_units) continue;
        // the tile's last chunk: add its chunks in order, lane (row, half of the tokens)
        const int e = static_cast<int>((rec.chunk_e >> 24) & 15u);
        const FTensor& T = P.t[e];
        const int row = lane & 15, m0 = (lane >> 4) * (kMaxTok / 2);
        float v[kMaxTok / 2];
#pragma unroll
        for (int i = 0; i < kMaxTok / 2; ++i) v[i] = 0.0f;
        for (uint32_t j = 0; j < rec.n_units; ++j) {
            const float* p = parts + ((rec.k_first + j) & (kParts - 1)) * kSlotFloats + row * kMaxTok + m0;
#pragma unroll
            for (int i = 0; i < kMaxTok / 2; ++i) v[i] += p[i];
        }
        __syncwarp();
        if (lane == 0) cnts[fslot] = 0u;
        for (uint32_t j = lane; j < rec.n_units; j += 32) {
            const uint32_t kk = rec.k_first + j;
            gens[kk & (kParts - 1)] = (kk >> kPartsLog2) + 1u;
        }
        const int r = static_cast<int>(rec.tile) * kRows + row;
        if (r < T.N)
#pragma unroll
            for (int i = 0; i < kMaxTok / 2; ++i)
                if (m0 + i < P.M) T.y[static_cast<int64_t>(m0 + i) * T.N + r] = v[i];
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

bool encode_rows(CUtensorMap* map, const GemvTensor& t) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(t.nb) * kBlockBytes;
    const cuuint64_t dims[2] = {row_bytes / 4, static_cast<cuuint64_t>(t.N)};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxWords), static_cast<cuuint32_t>(kRows)};
    const cuuint32_t estride[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(t.W), dims, strides, box,
              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int ffma_max_chunks() { return kParts; }

cudaError_t launch_gemv_ffma(const GemvTensor* t, int count, int M, uint32_t* status, int num_sms,
                             uint64_t timeout_ns, cudaStream_t s) {
    if (M < 1 || M > kMaxTok || count < 1 || count > kMaxLayer) return cudaErrorInvalidValue;
    FParams P{};
    uint64_t units = 0;
    CostSplit split{};
    for (int e = 0; e < count; ++e) {
        FTensor& T = P.t[e];
        T.x = t[e].x;
        T.y = t[e].y;
        T.N = t[e].N;
        T.type = t[e].type;
        T.K = t[e].nb * per_block(t[e].type);
        T.chunks = t[e].nb / kChunkBlocks;
        T.tiles = (t[e].N + kRows - 1) / kRows;
        T.unit_base = static_cast<uint32_t>(units);
        if (T.chunks > kParts || !encode_rows(&P.wmap[e], t[e])) return cudaErrorInvalidValue;
        units += static_cast<uint64_t>(T.chunks) * T.tiles;
        split.add(static_cast<uint32_t>(T.tiles), static_cast<uint32_t>(T.chunks));   // whole tiles, weighed by units
    }
    if (units == 0) return cudaSuccess;
    if (units >= (1ull << 31)) return cudaErrorInvalidValue;
    P.count = count;
    P.M = M;
    const int max_grid = num_sms < kMaxGrid ? num_sms : kMaxGrid;
    P.grid = split.fit_grid(max_grid, 1u);
    // tile boundaries -> unit boundaries
    for (int c = 0; c <= P.grid; ++c) {
        const uint32_t tb = split.start(c);
        int e = 0;
        while (e + 1 < count && tb >= split.base[e + 1]) ++e;
        const uint32_t rel = tb - split.base[e];
        P.starts[c] = c == P.grid ? static_cast<uint32_t>(units)
                                  : P.t[e].unit_base + rel * static_cast<uint32_t>(P.t[e].chunks);
    }
    P.status = status;
    P.timeout_ns = timeout_ns;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = set_smem_limit_once(gemv_ffma_kernel, Layout(kMaxTok).total, smem_set); e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(P.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Layout(M).total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_ffma_kernel, P);
}

}  // namespace pn
