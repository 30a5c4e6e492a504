// pn_gemv_tc.cu -- PN decode GEMV on GB300: TMA-staged rows, decode in registers,
// fp32 accumulation on the tensor cores (mma.sync m16n8k16).
//
// What is computed: y[m][r] = sum_k d_blk(r,k) * (n(r,k) - z) * x[m][k], the
// decode GEMV of the tensorless docs ("Why a P100-native weight format": "One
// lane, one word", "Exact decode in fp32") at M = 1 and its skinny M <= 8 form
// (speculative verification of k drafts in one batch, v100-skinny README, "How
// QPN works": packed weights stay compressed through HBM and are decoded at the
// point of consumption, straight into tensor-core register operands).
//
// Design (GB300-first; the pages' sm_60 and sm_70 kernels are prior art):
//  * Work unit = one 16-row tile x one 8-block chunk (8 x 34 = 272 bytes per
//    row, 16-byte aligned whenever the row is).  Units are numbered per group of
//    8 tiles, chunk-major, tile-minor, over every tensor of the call, and the
//    persistent grid (at most one CTA per SM) splits that sequence into equal
//    contiguous ranges, so every SM streams the same number of bytes.
//  * One producer warp per CTA issues cp.async.bulk copies (TMA engine, no
//    tensor map) of each step's rows and x chunk into a 4-stage shared-memory
//    ring, completing on mbarriers; 8 consumer warps (one per tile of the
//    group) decode and multiply.  Every wait is bounded in time.
//  * Decode: code words are read from shared memory as aligned 32-bit words
//    (blocks at even offsets are realigned with one byte-permute per word);
//    a LOP3 + HFMA2 per code pair turns two codes into the exact half2
//    (n - z, n' - z), which is exactly an A-fragment register of
//    m16n8k16 (rows g and g+8 of the tile, k pairs from code words 2t, 2t+1);
//    x is read as B fragments straight from the staged chunk; each block's
//    product sum starts from zero and is scaled by its d in fp32 (FFMA), so
//    every product is exact and every sum is an fp32 sum.
//  * Tiles split between CTAs are summed by their last contributor, in CTA
//    order, from partial slots in the workspace (a per-tile counter decides
//    who is last and is reset by it), so the result is deterministic.
#include <cstdint>
#include <type_traits>
#include <utility>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pn_device.cuh"
#include "pn_internal.h"

namespace pn {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTileRows = 16;
constexpr int kGroupTiles = kConsumerWarps;             // one tile per consumer warp
constexpr int kGroupRows = kGroupTiles * kTileRows;     // 128
constexpr int kChunkBlocks = 8;
constexpr int kChunkBytes = kChunkBlocks * kBlockBytes; // 272
constexpr int kRowPitch = 288;                          // staged row pitch (bank spread)
constexpr int kTileBytes = kTileRows * kRowPitch;
constexpr int kStageWBytes = kGroupTiles * kTileBytes;  // 36864
constexpr int kXPitchPn3t = kChunkBlocks * 80 * 2 + 16; // 1296
constexpr int kXPitchPn4t = kChunkBlocks * 64 * 2 + 16; // 1040
constexpr int kStageXBytes = kMaxM * kXPitchPn3t;       // 10368
constexpr int kStageBytes = kStageWBytes + kStageXBytes;
constexpr int kStages = 4;
constexpr int kBarrierOffset = kStages * kStageBytes;
constexpr int kSmemBytes = kBarrierOffset + 2 * kStages * 8 + 16;
constexpr uint64_t kDrainLimitNs = 200ull * 1000 * 1000;
constexpr uint32_t kStatusTimeout = 5;                  // PN_ETIMEOUT
constexpr int kSlotFloats = kTileRows * kMaxM;          // 128

static_assert(kStageWBytes % 16 == 0 && kStageBytes % 16 == 0, "TMA needs 16-byte alignment");

struct TcTensor {
    const uint8_t* W;
    const uint16_t* x;
    float* y;
    int64_t unit_base;      // first unit of this tensor in the launch's sequence
    int N;
    int nb;
    int type;
    int chunks;             // nb / 8
    int tiles;              // ceil(N / 16)
    int group_base;         // first global group index
    int tile_base;          // first global tile index (counter index)
};

struct TcParams {
    TcTensor t[kMaxLayer];
    int count;
    int M;
    int grid;
    int64_t units;
    uint32_t* status;
    uint32_t* counters;
    float* partials;
    uint64_t timeout_ns;
};

struct Step {
    int e;       // tensor
    int g;       // group within the tensor
    int c;       // chunk
    int jlo;     // first tile of the group in this step
    int jhi;     // one past the last
    int tg;      // tiles in the group
};

template <int N, typename Fn, int... I>
__device__ __forceinline__ void static_for_impl(Fn&& fn, std::integer_sequence<int, I...>) {
    (fn(std::integral_constant<int, I>{}), ...);
}
template <int N, typename Fn>
__device__ __forceinline__ void static_for(Fn&& fn) {
    static_for_impl<N>(fn, std::make_integer_sequence<int, N>{});
}

__device__ __forceinline__ int tensor_of(const TcParams& P, int64_t u) {
    int e = 0;
    while (e + 1 < P.count && u >= P.t[e + 1].unit_base) ++e;
    return e;
}

__device__ __forceinline__ int group_id_of(const TcParams& P, int64_t u) {
    const int e = tensor_of(P, u);
    const TcTensor& T = P.t[e];
    return T.group_base + static_cast<int>((u - T.unit_base) / (8LL * T.chunks));
}

// First unit of CTA c's range and the CTA whose range holds unit u.
__device__ __forceinline__ int64_t range_start(const TcParams& P, int c) {
    return P.units * c / P.grid;
}
__device__ __forceinline__ int cta_of(const TcParams& P, int64_t u) {
    return static_cast<int>(((u + 1) * P.grid - 1) / P.units);
}

// Walks a CTA's unit range one step (same tensor, group and chunk) at a time.
struct StepIter {
    int64_t u, end;
    __device__ bool next(const TcParams& P, Step& st) {
        if (u >= end) return false;
        const int e = tensor_of(P, u);
        const TcTensor& T = P.t[e];
        const int64_t rel = u - T.unit_base;
        const int64_t gsz = 8LL * T.chunks;
        const int g = static_cast<int>(rel / gsz);
        const int tg = min(kGroupTiles, T.tiles - g * kGroupTiles);
        const int64_t r2 = rel - g * gsz;
        const int c = static_cast<int>(r2 / tg);
        const int j = static_cast<int>(r2 - static_cast<int64_t>(c) * tg);
        const int64_t left = end - u;
        const int jhi = static_cast<int>(min(static_cast<int64_t>(tg), j + left));
        st.e = e; st.g = g; st.c = c; st.jlo = j; st.jhi = jhi; st.tg = tg;
        u += jhi - j;
        return true;
    }
};

__device__ __forceinline__ void raise_timeout(const TcParams& P, volatile uint32_t* abort_flag) {
    *abort_flag = 1u;
    atomicCAS(P.status, 0u, kStatusTimeout);
}

// Waits for phase `parity` of an mbarrier; gives up after limit_ns, or as soon
// as another warp of the CTA has aborted (abort_flag may be null).
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                             volatile uint32_t* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag && *abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ----------------------------------------------------------------- decode --

// Loads code words 2t and 2t+1 of block B of a staged row (8-byte aligned).
template <int B>
__device__ __forceinline__ void load_words(uint32_t row, int t, uint32_t& w0, uint32_t& w1) {
    constexpr int kOff = B * kBlockBytes;
    if constexpr (B % 2 == 0) {
        // block starts 4-byte aligned: its words start 2 bytes into aligned words
        const uint32_t a = row + kOff + 8 * t;
        uint32_t v0, v1, v2;
        if constexpr (kOff % 8 == 0) {
            const uint2 p = lds_u64(a);
            v0 = p.x; v1 = p.y; v2 = lds_u32(a + 8);
        } else {
            v0 = lds_u32(a);
            const uint2 p = lds_u64(a + 4);
            v1 = p.x; v2 = p.y;
        }
        w0 = realign16(v0, v1);
        w1 = realign16(v1, v2);
    } else {
        // block starts 2 bytes past a 4-byte boundary: its words are aligned
        const uint32_t a = row + kOff + 2 + 8 * t;
        if constexpr ((kOff + 2) % 8 == 0) {
            const uint2 p = lds_u64(a);
            w0 = p.x; w1 = p.y;
        } else {
            w0 = lds_u32(a);
            w1 = lds_u32(a + 4);
        }
    }
}

// x pairs for code words 2t (xb[0..P-1]) and 2t+1 (xb[P..2P-1]) of block B.
template <int TYPE, int B>
__device__ __forceinline__ void load_x(uint32_t xrow, int t, bool on, uint32_t (&xb)[2 * Format<TYPE>::kPairs]) {
    using F = Format<TYPE>;
    if (!on) {
#pragma unroll
        for (int i = 0; i < 2 * F::kPairs; ++i) xb[i] = 0u;
        return;
    }
    if constexpr (TYPE == kPn3t) {
        const uint32_t a = xrow + (B * F::kPerBlock + 2 * F::kPerWord * t) * 2;   // 8-byte aligned
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const uint2 p = lds_u64(a + 8 * i);
            xb[2 * i] = p.x; xb[2 * i + 1] = p.y;
        }
    } else {
        const uint32_t a = xrow + (B * F::kPerBlock + 2 * F::kPerWord * t) * 2;   // 16-byte aligned
        const uint4 p = lds_u128(a);
        const uint4 q = lds_u128(a + 16);
        xb[0] = p.x; xb[1] = p.y; xb[2] = p.z; xb[3] = p.w;
        xb[4] = q.x; xb[5] = q.y; xb[6] = q.z; xb[7] = q.w;
    }
}

// One consumer warp: the 16 rows of its tile times one 8-block chunk.  The
// chunk's eight scaled block sums are added up first and then added to the
// running sum, which keeps every fp32 summation chain short (at most 8 block
// terms + one term per chunk), whatever K is.
template <int TYPE>
__device__ __forceinline__ void mma_tile_chunk(uint32_t tile, uint32_t xbase, int xpitch, int M,
                                               int lane, float (&acc)[4]) {
    using F = Format<TYPE>;
    const int g = lane >> 2, t = lane & 3;
    const uint32_t r0 = tile + g * kRowPitch;
    const uint32_t r1 = r0 + 8 * kRowPitch;
    const bool xon = g < M;
    const uint32_t xrow = xbase + g * xpitch;
    float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    static_for<kChunkBlocks>([&](auto bc) {
        constexpr int B = decltype(bc)::value;
        const float d0 = half_bits_to_float(lds_u16(r0 + B * kBlockBytes));
        const float d1 = half_bits_to_float(lds_u16(r1 + B * kBlockBytes));
        uint32_t w00, w10, w01, w11;        // w<word><row>: words 2t / 2t+1 of rows g / g+8
        load_words<B>(r0, t, w00, w10);
        load_words<B>(r1, t, w01, w11);
        const uint32_t s00 = w00 >> F::kHighShift, s10 = w10 >> F::kHighShift;
        const uint32_t s01 = w01 >> F::kHighShift, s11 = w11 >> F::kHighShift;
        uint32_t xb[2 * F::kPairs];
        load_x<TYPE, B>(xrow, t, xon, xb);
        float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        static_for<F::kPairs>([&](auto pc) {
            constexpr int P = decltype(pc)::value;
            const uint32_t a[4] = {
                decode_pair<TYPE, P>(w00, s00),   // row g,   k = 2t, 2t+1   <- word 2t
                decode_pair<TYPE, P>(w01, s01),   // row g+8, k = 2t, 2t+1   <- word 2t
                decode_pair<TYPE, P>(w10, s10),   // row g,   k = 2t+8, 2t+9 <- word 2t+1
                decode_pair<TYPE, P>(w11, s11)};  // row g+8, k = 2t+8, 2t+9 <- word 2t+1
            mma_16816(c, a, xb[P], xb[F::kPairs + P], c);
        });
        part[0] = fmaf(d0, c[0], part[0]);
        part[1] = fmaf(d0, c[1], part[1]);
        part[2] = fmaf(d1, c[2], part[2]);
        part[3] = fmaf(d1, c[3], part[3]);
    });
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] += part[i];
}

// ------------------------------------------------------------------ flush --

__device__ __forceinline__ void store_tile(const TcTensor& T, int M, int g, int j, int lane,
                                           const float (&v)[4]) {
    const int row0 = g * kGroupRows + j * kTileRows + (lane >> 2);
    const int m0 = 2 * (lane & 3);
    const int rows[2] = {row0, row0 + 8};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (rows[h] < T.N) {
            if (m0 < M) T.y[static_cast<int64_t>(m0) * T.N + rows[h]] = v[2 * h];
            if (m0 + 1 < M) T.y[static_cast<int64_t>(m0 + 1) * T.N + rows[h]] = v[2 * h + 1];
        }
    }
}

__device__ __forceinline__ float* slot_ptr(const TcParams& P, int cta, int which, int j) {
    return P.partials + ((static_cast<int64_t>(cta) * 2 + which) * kGroupTiles + j) * kSlotFloats;
}

// Emits warp j's tile of group (e, g): stores it if this CTA covered all of
// its chunks, else deposits a partial and lets the last contributor sum them.
__device__ void flush_tile(const TcParams& P, const Step& st, int j, int lane, int64_t u0,
                           int64_t u1, const float (&acc)[4]) {
    const TcTensor& T = P.t[st.e];
    const int64_t first = T.unit_base + 8LL * T.chunks * st.g + j;
    const int64_t last = first + static_cast<int64_t>(T.chunks - 1) * st.tg;
    if (first >= u0 && last < u1) {
        store_tile(T, P.M, st.g, j, lane, acc);
        return;
    }
    const int gid = T.group_base + st.g;
    const int cta = blockIdx.x;
    const int ca = cta_of(P, first), cb = cta_of(P, last);
    const int own_which = (group_id_of(P, u0) == gid) ? 0 : 1;
    const int r = lane >> 2, m0 = 2 * (lane & 3);
    float* slot = slot_ptr(P, cta, own_which, j);
    __stcg(reinterpret_cast<float2*>(slot + r * kMaxM + m0), make_float2(acc[0], acc[1]));
    __stcg(reinterpret_cast<float2*>(slot + (r + 8) * kMaxM + m0), make_float2(acc[2], acc[3]));
    __threadfence();
    __syncwarp();
    uint32_t* counter = P.counters + T.tile_base + st.g * kGroupTiles + j;
    uint32_t old = 0;
    if (lane == 0) old = atomicAdd(counter, 1u);
    old = __shfl_sync(0xFFFFFFFFu, old, 0);
    if (old != static_cast<uint32_t>(cb - ca)) return;          // someone else finishes it
    __threadfence();
    float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int c = ca; c <= cb; ++c) {                            // fixed order: deterministic
        if (c == cta) {
#pragma unroll
            for (int i = 0; i < 4; ++i) sum[i] += acc[i];
        } else {
            const int which = (group_id_of(P, range_start(P, c)) == gid) ? 0 : 1;
            const float* s = slot_ptr(P, c, which, j);
            const float2 a = __ldcg(reinterpret_cast<const float2*>(s + r * kMaxM + m0));
            const float2 b = __ldcg(reinterpret_cast<const float2*>(s + (r + 8) * kMaxM + m0));
            sum[0] += a.x; sum[1] += a.y; sum[2] += b.x; sum[3] += b.y;
        }
    }
    store_tile(T, P.M, st.g, j, lane, sum);
    if (lane == 0) atomicExch(counter, 0u);
}

// ----------------------------------------------------------------- kernel --

__global__ void __launch_bounds__(kThreads, 1) gemv_tc_kernel(const __grid_constant__ TcParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    const uint32_t full0 = sbase + kBarrierOffset;
    const uint32_t empty0 = full0 + kStages * 8;
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kBarrierOffset + 2 * kStages * 8);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();

    const int64_t u0 = range_start(P, blockIdx.x);
    const int64_t u1 = range_start(P, blockIdx.x + 1);

    uint32_t issued[kStages];             // producer: copies issued per stage
#pragma unroll
    for (int s = 0; s < kStages; ++s) issued[s] = 0;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------- producer --
        StepIter it{u0, u1};
        Step st;
        int idx = 0;
        while (!*abort_flag && it.next(P, st)) {
            const int s = idx % kStages;
            const uint32_t round = static_cast<uint32_t>(idx / kStages);
            if (round > 0 && !wait_bounded(empty0 + 8 * s, (round - 1) & 1u, P.timeout_ns, abort_flag)) {
                raise_timeout(P, abort_flag);
                break;
            }
            const TcTensor& T = P.t[st.e];
            const int per_blk = per_block(T.type);
            const int xbytes = kChunkBlocks * per_blk * 2;
            const int xpitch = T.type == kPn3t ? kXPitchPn3t : kXPitchPn4t;
            const int row0 = st.g * kGroupRows + st.jlo * kTileRows;
            const int rows = min((st.jhi - st.jlo) * kTileRows, T.N - row0);
            const int64_t K = static_cast<int64_t>(T.nb) * per_blk;
            const int64_t rb = static_cast<int64_t>(T.nb) * kBlockBytes;
            const uint32_t full = full0 + 8 * s;
            const uint32_t stage = sbase + s * kStageBytes;
            if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(P.M * xbytes + rows * kChunkBytes));
            __syncwarp();
            const int total = P.M + rows;
            for (int i = lane; i < total; i += 32) {
                if (i < P.M) {
                    bulk_g2s(stage + kStageWBytes + i * xpitch,
                             T.x + i * K + static_cast<int64_t>(st.c) * kChunkBlocks * per_blk, xbytes, full);
                } else {
                    const int rr = i - P.M;
                    bulk_g2s(stage + (st.jlo * kTileRows + rr) * kRowPitch,
                             T.W + (row0 + rr) * rb + static_cast<int64_t>(st.c) * kChunkBytes,
                             kChunkBytes, full);
                }
            }
            issued[s] = round + 1;
            ++idx;
        }
    } else {
        // ------------------------------------------------------- consumers --
        StepIter it{u0, u1};
        Step st, cur{};
        int cur_gid = -1;
        bool active = false;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        int idx = 0;
        bool ok = true;
        while (it.next(P, st)) {
            const TcTensor& T = P.t[st.e];
            const int gid = T.group_base + st.g;
            if (gid != cur_gid) {
                if (active) flush_tile(P, cur, warp, lane, u0, u1, acc);
                active = false;
                acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
                cur_gid = gid;
                cur = st;
            }
            const int s = idx % kStages;
            const uint32_t parity = static_cast<uint32_t>(idx / kStages) & 1u;
            const bool got = wait_bounded(full0 + 8 * s, parity, P.timeout_ns, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) raise_timeout(P, abort_flag);
                ok = false;
                break;
            }
            if (st.jlo <= warp && warp < st.jhi) {
                const uint32_t stage = sbase + s * kStageBytes;
                const uint32_t tile = stage + warp * kTileBytes;
                const uint32_t xbase = stage + kStageWBytes;
                if (T.type == kPn3t) mma_tile_chunk<kPn3t>(tile, xbase, kXPitchPn3t, P.M, lane, acc);
                else mma_tile_chunk<kPn4t>(tile, xbase, kXPitchPn4t, P.M, lane, acc);
                active = true;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
            ++idx;
            if (*abort_flag) { ok = false; break; }
        }
        if (ok && active) flush_tile(P, cur, warp, lane, u0, u1, acc);
    }
    __syncthreads();
    // Every copy the producer started must land before the CTA exits.  After a
    // normal run each stage's last phase has completed and this returns at
    // once; after an abort it waits (bounded) for the copies still in flight.
    if (warp == kConsumerWarps) {
#pragma unroll
        for (int s = 0; s < kStages; ++s)
            if (issued[s]) wait_bounded(full0 + 8 * s, (issued[s] - 1) & 1u, kDrainLimitNs, nullptr);
    }
}

}  // namespace

// The counter array starts at an offset that depends only on the device (its
// SM count), so counters left at zero by one call are where the next call,
// of any shape, looks for them; partial slots never overlap counters.
WorkspaceLayout workspace_layout(int64_t total_tiles, int max_ctas) {
    WorkspaceLayout L;
    L.status = 0;
    L.partials = 256;
    L.counters = L.partials + static_cast<size_t>(max_ctas) * 2 * kGroupTiles * kSlotFloats * sizeof(float);
    L.total = L.counters + ((static_cast<size_t>(total_tiles) * 4 + 255) / 256) * 256;
    return L;
}

int tc_max_ctas(int num_sms) { return num_sms; }

cudaError_t launch_gemv_tc(const GemvTensor* t, int count, int M, void* workspace,
                           size_t workspace_bytes, int num_sms, uint64_t timeout_ns,
                           cudaStream_t s, int* needs_bytes_out) {
    TcParams P{};
    int64_t units = 0;
    int groups = 0, tiles = 0;
    for (int e = 0; e < count; ++e) {
        TcTensor& T = P.t[e];
        T.W = t[e].W; T.x = t[e].x; T.y = t[e].y;
        T.N = t[e].N; T.nb = t[e].nb; T.type = t[e].type;
        T.chunks = t[e].nb / kChunkBlocks;
        T.tiles = (t[e].N + kTileRows - 1) / kTileRows;
        T.unit_base = units;
        T.group_base = groups;
        T.tile_base = tiles;
        units += static_cast<int64_t>(T.chunks) * T.tiles;
        groups += (T.tiles + kGroupTiles - 1) / kGroupTiles;
        tiles += T.tiles;
    }
    P.count = count;
    P.M = M;
    P.units = units;
    int64_t grid = units / 8;
    if (grid > num_sms) grid = num_sms;
    if (grid < 1) grid = 1;
    P.grid = static_cast<int>(grid);
    const WorkspaceLayout L = workspace_layout(tiles, tc_max_ctas(num_sms));
    if (needs_bytes_out) *needs_bytes_out = 0;
    if (L.total > workspace_bytes) {
        if (needs_bytes_out) *needs_bytes_out = 1;
        return cudaSuccess;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    P.status = reinterpret_cast<uint32_t*>(ws + L.status);
    P.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
    P.partials = reinterpret_cast<float*>(ws + L.partials);
    P.timeout_ns = timeout_ns;

    static bool attr_set = false;   // per process; the attribute is per function
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    gemv_tc_kernel<<<P.grid, kThreads, kSmemBytes, s>>>(P);
    return cudaGetLastError();
}

}  // namespace pn
