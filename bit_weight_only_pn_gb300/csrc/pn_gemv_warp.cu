// pn_gemv_warp.cu -- PN decode GEMV for one or two tokens on GB300: every warp
// streams its own share of the weights through its own TMA ring.
//
// What is computed: y[m][r] = sum_k d_blk(r,k) * (n(r,k) - z) * x[m][k] for
// M <= 2, the decode GEMV of the tensorless docs ("Why a P100-native weight
// format": "One lane, one word", "Exact decode in fp32"), with the products on
// the tensor cores (mma.sync m16n8k16, fp16 inputs, fp32 sums) and every
// product exact.
//
// Design (GB300-first; the pages' sm_60 one-lane-per-word kernel is prior art):
//  * Work unit = one 16-row tile x one 8-block chunk (16 x 272 bytes).  Units
//    are numbered tile-major over every tensor of the call.  The grid (two
//    thread blocks per SM) splits them into equal contiguous ranges of at
//    least one tile each, so a tile is shared by at most two blocks.
//  * A block has seven compute warps and one epilogue warp.  The compute warps
//    split the block's units into equal contiguous shares of one sequence
//    that starts with the parts of the two tiles cut by the block's
//    boundaries, so those parts are finished first.  No compute warp ever
//    waits for another.
//  * Each compute warp owns a three-stage shared-memory ring: lane 0 issues
//    one 2-D TMA box (16 rows x 272 bytes) per unit, completing on the stage's
//    mbarrier, and the warp decodes one stage while the next two are in
//    flight.  x is read through L1, prefetched one unit ahead.
//  * A tile that one warp covers completely is stored at once.  The epilogue
//    warp adds the warps' parts of the other tiles in warp order; for a tile
//    cut by a block boundary it deposits the block's part in the workspace
//    while the compute warps are still busy, and the second of the two blocks
//    to get there adds left part + right part, so results do not depend on
//    timing and the slow global hand-off stays off the kernel's tail.
//  * Programmatic dependent launch: the kernel lets the next kernel on the
//    stream launch at once, prefetches its first units into L2, and only then
//    waits for the previous kernel to complete; W, x and the workspace are
//    read, and y written, after that wait.
//  * Every wait is bounded in time; a warp that gives up records PN_ETIMEOUT
//    in the workspace, lets its copies in flight land, and finishes.
#include <cstdint>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pn_device.cuh"
#include "pn_internal.h"

namespace pn {
namespace {

constexpr int kComputeWarps = 7;
constexpr int kEpilogueWarp = kComputeWarps;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr int kCtasPerSm = 2;
constexpr int kStages = 3;
constexpr int kTileRows = 16;
constexpr int kChunkBlocks = 8;
constexpr int kChunkBytes = kChunkBlocks * kBlockBytes;   // 272, one staged row
constexpr int kBoxWords = kChunkBytes / 4;                // TMA box inner extent, 32-bit elements
constexpr int kUnitBytes = kTileRows * kChunkBytes;       // 4352
constexpr int kWarpMaxM = 2;
constexpr int kRecFloats = kTileRows * kWarpMaxM;         // one part of a tile: [row][token]
// Tile parts a compute warp hands to the epilogue warp: its part of the
// left-cut tile, of the right-cut tile, and of the first and last tiles of its
// share of the middle when it does not cover them completely.
constexpr int kRecLeft = 0, kRecRight = 1, kRecMidFirst = 2, kRecMidLast = 3, kRecs = 4;
constexpr int kRingBytes = kComputeWarps * kStages * kUnitBytes;
constexpr int kRecOffset = kRingBytes;                                           // [warp][kRecs][kRecFloats]
constexpr int kKeyOffset = kRecOffset + kComputeWarps * kRecs * kRecFloats * 4;  // [warp][2] int64 (middle records)
constexpr int kBarOffset = kKeyOffset + kComputeWarps * 2 * 8;                  // [warp][stage], then left, right, done
constexpr int kSmemBytes = kBarOffset + (kComputeWarps * kStages + 3) * 8;
constexpr uint64_t kDrainLimitNs = 200ull * 1000 * 1000;
constexpr uint32_t kStatusTimeout = 5;                    // PN_ETIMEOUT
constexpr int kSlotFloats = kTileRows * kMaxM;            // one boundary slot (shared layout)

static_assert(kStagedRowBytes == kChunkBytes, "staged rows are one chunk wide");
static_assert(kUnitBytes % 128 == 0, "every stage starts 128-byte aligned");
static_assert(kSmemBytes <= 110 * 1024, "two thread blocks fit on one SM");

struct WTensor {
    const uint16_t* x;
    float* y;
    uint32_t unit_base;     // first unit of this tensor
    int N;
    int K;
    int type;
    int chunks;             // nb / 8
    int tiles;              // ceil(N / 16)
};

struct WarpParams {
    CUtensorMap wmap[kMaxLayer];   // PN rows as uint32 [N][row_bytes / 4]; box 68 words x 16 rows
    WTensor t[kMaxLayer];
    int count;
    int M;
    int grid;
    uint32_t units;                // units * grid < 2^32 and units * 8 < 2^32 (checked on the host)
    uint32_t* status;
    uint32_t* counters;            // one per thread-block boundary
    float* partials;               // [boundary][side][kSlotFloats]
    uint64_t timeout_ns;
    int stall_first_step;          // testing aid: see pn_set_test_stall
};

// Position of a unit: tensor, tile, chunk.
struct Cursor {
    int e, tile, chunk;
    __device__ void locate(const WarpParams& P, uint32_t u) {
        e = 0;
        while (e + 1 < P.count && u >= P.t[e + 1].unit_base) ++e;
        const uint32_t rel = u - P.t[e].unit_base;
        const uint32_t ch = static_cast<uint32_t>(P.t[e].chunks);
        tile = static_cast<int>(rel / ch);
        chunk = static_cast<int>(rel - static_cast<uint32_t>(tile) * ch);
    }
    __device__ void next(const WarpParams& P) {
        if (++chunk == P.t[e].chunks) {
            chunk = 0;
            if (++tile == P.t[e].tiles) { tile = 0; ++e; }
        }
    }
    __device__ int64_t key() const { return (static_cast<int64_t>(e) << 32) | static_cast<uint32_t>(tile); }
};

__device__ __forceinline__ uint32_t range_start(const WarpParams& P, int c) {
    return P.units * static_cast<uint32_t>(c) / static_cast<uint32_t>(P.grid);
}

// Waits for phase `parity` of an mbarrier for at most limit_ns.
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Warp-level wait: lane 0 polls; __syncwarp orders the other lanes' reads of
// the stage after lane 0's observation of the completed phase.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, int lane) {
    bool ok = true;
    if (lane == 0) ok = wait_bounded(bar, parity, limit_ns);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok;
}

// This lane's x pairs for one block: 2 * kPerWord halves from `p` on
// (pn3t: 40 bytes, 8-byte aligned; pn4t: 32 bytes, 16-byte aligned), read
// through L1.
template <int TYPE>
__device__ __forceinline__ void load_x_global(const uint16_t* p, uint32_t (&xb)[2 * Format<TYPE>::kPairs]) {
    if constexpr (TYPE == kPn3t) {
        const uint2* q = reinterpret_cast<const uint2*>(p);
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const uint2 v = __ldg(q + i);
            xb[2 * i] = v.x; xb[2 * i + 1] = v.y;
        }
    } else {
        const uint4* q = reinterpret_cast<const uint4*>(p);
        const uint4 v = __ldg(q), w = __ldg(q + 1);
        xb[0] = v.x; xb[1] = v.y; xb[2] = v.z; xb[3] = v.w;
        xb[4] = w.x; xb[5] = w.y; xb[6] = w.z; xb[7] = w.w;
    }
}

// One unit: the 16 staged rows of a chunk times the chunk of x of this lane's
// token (xc points at the chunk's first activation).  With M1 only the first
// token's column is scaled.  The eight scaled block
// sums are added up first and then added to the tile's running sum, so every
// fp32 summation chain stays short whatever K is.
template <int TYPE, bool M1>
__device__ __forceinline__ void unit_mma(const uint8_t* tile, const uint16_t* xc, int lane, float (&acc)[4]) {
    using F = Format<TYPE>;
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* r0 = tile + tile_row(g) * kChunkBytes;
    const uint8_t* r1 = r0 + 8 * kChunkBytes;
    const uint16_t* xl = xc + 2 * F::kPerWord * t;
    float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    static_for<kChunkBlocks>([&](auto bc) {
        constexpr int B = decltype(bc)::value;
        uint32_t xb[2 * F::kPairs];
        load_x_global<TYPE>(xl + B * F::kPerBlock, xb);
        block_mma<TYPE, B, !M1>(r0, r1, t, xb, part);
    });
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] += part[i];
}

// Stores a whole tile from the accumulator fragments (lanes t = 0 hold the
// columns of tokens 0 and 1).
__device__ __forceinline__ void store_tile(const WTensor& T, int M, int tile, int lane, const float (&v)[4]) {
    if ((lane & 3) != 0) return;
    const int row0 = tile * kTileRows + tile_row(lane >> 2);
    const int rows[2] = {row0, row0 + 8};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (rows[h] < T.N) {
            T.y[rows[h]] = v[2 * h];
            if (M > 1) T.y[static_cast<int64_t>(T.N) + rows[h]] = v[2 * h + 1];
        }
    }
}

// Writes a tile part into record r of this warp: [row][token].
__device__ __forceinline__ void put_record(float* rec, int lane, const float (&v)[4]) {
    if ((lane & 3) != 0) return;
    const int row = tile_row(lane >> 2);
    rec[row * kWarpMaxM + 0] = v[0];
    rec[row * kWarpMaxM + 1] = v[1];
    rec[(row + 8) * kWarpMaxM + 0] = v[2];
    rec[(row + 8) * kWarpMaxM + 1] = v[3];
}

__device__ __forceinline__ float* slot_ptr(const WarpParams& P, int boundary, int side) {
    return P.partials + (static_cast<int64_t>(boundary) * 2 + side) * kSlotFloats;
}

// A finished block-level sum of one tile, one value per lane: lane = row * 2 + token.
// `cut` is 0 for a tile wholly inside this block, 1 for the tile cut by the
// block's left boundary, 2 for the one cut by its right boundary.
__device__ void emit_tile(const WarpParams& P, int64_t key, float v, int cut, int lane) {
    const int e = static_cast<int>(key >> 32), tile = static_cast<int>(key & 0xFFFFFFFF);
    const WTensor& T = P.t[e];
    const int row = tile * kTileRows + (lane >> 1), m = lane & 1;
    if (cut != 0) {
        // our part is side 1 of boundary blockIdx.x (left cut) or side 0 of
        // boundary blockIdx.x + 1 (right cut); the second arriver adds both
        const int boundary = blockIdx.x + (cut == 2 ? 1 : 0);
        const int side = cut == 1 ? 1 : 0;
        __stcg(slot_ptr(P, boundary, side) + (lane >> 1) * kMaxM + m, v);
        __threadfence();
        __syncwarp();
        uint32_t old = 0;
        if (lane == 0) old = atomicAdd(P.counters + boundary, 1u);
        old = __shfl_sync(0xFFFFFFFFu, old, 0);
        if (old != 1u) return;
        __threadfence();
        const float o = __ldcg(slot_ptr(P, boundary, side ^ 1) + (lane >> 1) * kMaxM + m);
        v = side == 1 ? o + v : v + o;           // left part + right part
        if (lane == 0) atomicExch(P.counters + boundary, 0u);
    }
    if (row < T.N && m < P.M) T.y[static_cast<int64_t>(m) * T.N + row] = v;
}

// A compute warp's share of its block's units: up to three runs of
// consecutive units (left-cut part, right-cut part, middle), walked in order.
// The runs are kept in scalars (run 0 is the current one) so that nothing
// is indexed at run time.
struct Walk {
    uint32_t a0, b0, a1, b1, a2, b2;   // runs [a, b)
    int k0, k1, k2;                    // their kinds: kRecLeft, kRecRight, kRecMidFirst
    uint32_t u;                        // current unit, in run 0
    Cursor c;                          // its position
    __device__ void init() { a0 = b0 = a1 = b1 = a2 = b2 = 0; k0 = k1 = k2 = 0; }
    __device__ void add(uint32_t a, uint32_t b, int k) {
        if (a >= b) return;
        if (a0 == b0) { a0 = a; b0 = b; k0 = k; }
        else if (a1 == b1) { a1 = a; b1 = b; k1 = k; }
        else { a2 = a; b2 = b; k2 = k; }
    }
    __device__ bool valid() const { return a0 < b0; }
    __device__ void start(const WarpParams& P) {
        u = a0;
        if (valid()) c.locate(P, u);
    }
    __device__ void advance(const WarpParams& P) {
        if (++u < b0) {
            c.next(P);
            return;
        }
        a0 = a1; b0 = b1; k0 = k1;
        a1 = a2; b1 = b2; k1 = k2;
        a2 = b2 = 0;
        start(P);
    }
};

// Whether [p0, p1) and [lo, hi) share a position.
__device__ __forceinline__ bool meets(uint32_t p0, uint32_t p1, uint32_t lo, uint32_t hi) {
    return max(p0, lo) < min(p1, hi);
}

// Prefetches into L1 the chunk of x that unit `c` reads, one line per lane
// (pn3t chunks are 1280 bytes, pn4t chunks 1024 bytes, per token).
__device__ __forceinline__ void prefetch_x(const WarpParams& P, const Cursor& c, int lane) {
    const WTensor& T = P.t[c.e];
    const int per = T.type == kPn3t ? 10 : 8;          // 128-byte lines per token
    const int m = lane / per, l = lane - m * per;
    if (m < P.M)
        prefetch_l1(T.x + static_cast<int64_t>(m) * T.K + c.chunk * kChunkBlocks * per_block(T.type) + l * 64);
}

__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

template <bool M1>
__device__ __forceinline__ void compute_unit(const WTensor& T, const uint8_t* stage, const uint16_t* xc, int lane,
                                             float (&acc)[4]) {
    if (T.type == kPn3t) unit_mma<kPn3t, M1>(stage, xc, lane, acc);
    else unit_mma<kPn4t, M1>(stage, xc, lane, acc);
}

template <bool M1>
__device__ void compute_warp(const WarpParams& P, uint8_t* smem, int warp, int lane, uint32_t c0, uint32_t n,
                             uint32_t nl, uint32_t nr, uint32_t bar_left, uint32_t bar_right, uint32_t bar_done) {
    const uint32_t p0 = n * static_cast<uint32_t>(warp) / kComputeWarps;
    const uint32_t p1 = n * static_cast<uint32_t>(warp + 1) / kComputeWarps;
    // sequence position -> unit: [0, nl) left-cut part, [nl, nl + nr) right-cut
    // part (the block's last nr units), [nl + nr, n) the middle
    Walk w;
    w.init();
    w.add(c0 + min(p0, nl), c0 + min(p1, nl), kRecLeft);
    w.add(c0 + n - nr + (min(max(p0, nl), nl + nr) - nl), c0 + n - nr + (min(max(p1, nl), nl + nr) - nl), kRecRight);
    w.add(c0 + nl + (max(p0, nl + nr) - nl - nr), c0 + nl + (max(p1, nl + nr) - nl - nr), kRecMidFirst);
    const bool in_left = meets(p0, p1, 0, nl), in_right = meets(p0, p1, nl, nl + nr);

    const uint32_t ring = smem_addr(smem) + warp * kStages * kUnitBytes;
    const uint8_t* ring_p = smem + warp * kStages * kUnitBytes;
    const uint32_t bar0 = smem_addr(smem + kBarOffset) + warp * kStages * 8;
    float* recs = reinterpret_cast<float*>(smem + kRecOffset) + warp * kRecs * kRecFloats;
    int64_t* keys = reinterpret_cast<int64_t*>(smem + kKeyOffset) + warp * 2;

    Walk iss = w;
    iss.start(P);
    if (lane == 0) {
        // warm L2 with this warp's first units while the previous kernel finishes
        Walk p = iss;
        for (int k = 0; k < kStages && p.valid(); ++k) {
            tma_prefetch_l2_2d(&P.wmap[p.c.e], p.c.chunk * kBoxWords, p.c.tile * kTileRows);
            p.advance(P);
        }
    }
    griddep_wait();
    __syncwarp();

    // Lane 0 fills stage s with the unit at the issue cursor; the lanes
    // prefetch that unit's x.
    int issued = 0;
    auto issue = [&](int s) {
        if (lane == 0) {
            const uint32_t bar = bar0 + 8 * s;
            mbar_arrive_expect_tx(bar, kUnitBytes);
            // (testing aid: with stall_first_step a warp's first unit is
            // announced but never copied, so its wait can only time out)
            if (!(issued == 0 && P.stall_first_step))
                tma_load_2d(ring + s * kUnitBytes, &P.wmap[iss.c.e], iss.c.chunk * kBoxWords,
                            iss.c.tile * kTileRows, bar);
        }
        prefetch_x(P, iss.c, lane);
        iss.advance(P);
        ++issued;
    };
    for (int s = 0; s < kStages && iss.valid(); ++s) issue(s);

    Walk cur = w;
    cur.start(P);
    const int token = min(lane >> 2, P.M - 1);   // this lane's B column (columns past M repeat token M-1)
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    bool from_start = false;                      // the open middle tile began at chunk 0 in this warp
    bool mid_first = true;                        // no middle record written yet
    bool arrived_left = false, arrived_right = false;
    int done = 0;
    while (cur.valid()) {
        const int s = done % kStages;
        if (!warp_wait(bar0 + 8 * s, static_cast<uint32_t>(done / kStages) & 1u, P.timeout_ns, lane)) {
            if (lane == 0) atomicCAS(P.status, 0u, kStatusTimeout);
            break;
        }
        const WTensor& T = P.t[cur.c.e];
        const int kind = cur.k0;
        if (kind == kRecMidFirst && (cur.u == cur.a0 || cur.c.chunk == 0)) from_start = cur.c.chunk == 0;
        const uint16_t* xc = T.x + static_cast<int64_t>(token) * T.K + cur.c.chunk * kChunkBlocks * per_block(T.type);
        compute_unit<M1>(T, ring_p + s * kUnitBytes, xc, lane, acc);
        __syncwarp();
        if (iss.valid()) {                        // refill this stage
            if (lane == 0) fence_proxy_async_smem();
            issue(s);
        }
        ++done;
        const bool run_end = cur.u + 1 == cur.b0;
        const bool last_chunk = cur.c.chunk == T.chunks - 1;
        if (kind != kRecMidFirst) {
            if (run_end) {                        // this warp's part of a cut tile
                put_record(recs + kind * kRecFloats, lane, acc);
                if (kind == kRecLeft) { warp_arrive(bar_left, lane); arrived_left = true; }
                else { warp_arrive(bar_right, lane); arrived_right = true; }
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = 0.0f;
            }
        } else if (last_chunk || run_end) {
            if (from_start && last_chunk) {
                store_tile(T, P.M, cur.c.tile, lane, acc);
            } else {
                const int r = mid_first ? kRecMidFirst : kRecMidLast;
                put_record(recs + r * kRecFloats, lane, acc);
                if (lane == 0) keys[r - kRecMidFirst] = cur.c.key();
            }
            mid_first = false;
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = 0.0f;
        }
        cur.advance(P);
    }
    if (lane == 0) {
        // after a timeout: let every copy this warp started land before the block can exit
        for (int k = done; k < issued; ++k) {
            if (k == 0 && P.stall_first_step) continue;   // never copied
            wait_bounded(bar0 + 8 * (k % kStages), static_cast<uint32_t>(k / kStages) & 1u, kDrainLimitNs);
        }
    }
    if (in_left && !arrived_left) warp_arrive(bar_left, lane);
    if (in_right && !arrived_right) warp_arrive(bar_right, lane);
    warp_arrive(bar_done, lane);
}

// Number of compute warps whose share of an n-unit sequence meets [lo, hi).
__device__ __forceinline__ int warps_meeting(uint32_t n, uint32_t lo, uint32_t hi) {
    int k = 0;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w)
        k += meets(n * w / kComputeWarps, n * (w + 1) / kComputeWarps, lo, hi) ? 1 : 0;
    return k;
}

// The epilogue warp: finishes the block's two cut tiles as soon as the
// compute warps have their parts, then the tiles split between compute warps.
__device__ void epilogue_warp(const WarpParams& P, const uint8_t* smem, int lane, uint32_t c0, uint32_t n,
                              uint32_t nl, uint32_t nr, const Cursor& first, const Cursor& last,
                              uint32_t bar_left, uint32_t bar_right, uint32_t bar_done) {
    const float* recs = reinterpret_cast<const float*>(smem + kRecOffset);
    const int64_t* keys = reinterpret_cast<const int64_t*>(smem + kKeyOffset);
    for (int side = 0; side < 2; ++side) {
        const uint32_t lo = side == 0 ? 0 : nl, hi = side == 0 ? nl : nl + nr;
        if (lo == hi) continue;
        if (!warp_wait(side == 0 ? bar_left : bar_right, 0u, P.timeout_ns, lane)) {
            if (lane == 0) atomicCAS(P.status, 0u, kStatusTimeout);
            return;
        }
        float v = 0.0f;
        for (int w = 0; w < kComputeWarps; ++w) {
            if (meets(n * w / kComputeWarps, n * (w + 1) / kComputeWarps, lo, hi)) v += recs[(w * kRecs + (side == 0 ? kRecLeft : kRecRight)) * kRecFloats + lane];
        }
        emit_tile(P, side == 0 ? first.key() : last.key(), v, side == 0 ? 1 : 2, lane);
    }
    if (!warp_wait(bar_done, 0u, P.timeout_ns, lane)) {
        if (lane == 0) atomicCAS(P.status, 0u, kStatusTimeout);
        return;
    }
    int64_t run_key = -1;
    float run = 0.0f;
    for (int r = 0; r < 2 * kComputeWarps; ++r) {
        const int w = r >> 1, k = r & 1;
        const int64_t key = keys[w * 2 + k];
        if (key < 0) continue;
        const float v = recs[(w * kRecs + kRecMidFirst + k) * kRecFloats + lane];
        if (key == run_key) {
            run += v;
        } else {
            if (run_key >= 0) emit_tile(P, run_key, run, 0, lane);
            run_key = key;
            run = v;
        }
    }
    if (run_key >= 0) emit_tile(P, run_key, run, 0, lane);
    (void)c0;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) gemv_warp_kernel(const __grid_constant__ WarpParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t c0 = range_start(P, blockIdx.x), c1 = range_start(P, blockIdx.x + 1);
    const uint32_t n = c1 - c0;
    Cursor first{0, 0, 0}, last{0, 0, 0};
    if (n > 0) {
        first.locate(P, c0);
        last.locate(P, c1 - 1);
    }
    // the block's part of the tile it shares with the previous block, and of
    // the one it shares with the next block
    const uint32_t nl = (n > 0 && first.chunk != 0) ? static_cast<uint32_t>(P.t[first.e].chunks - first.chunk) : 0u;
    const uint32_t nr = (n > 0 && last.chunk != P.t[last.e].chunks - 1) ? static_cast<uint32_t>(last.chunk + 1) : 0u;
    const uint32_t bars = smem_addr(smem + kBarOffset) + kComputeWarps * kStages * 8;
    const uint32_t bar_left = bars, bar_right = bars + 8, bar_done = bars + 16;
    if (threadIdx.x == 0) {
        const int kl = warps_meeting(n, 0, nl), kr = warps_meeting(n, nl, nl + nr);
        mbar_init(bar_left, kl > 0 ? kl : 1);
        mbar_init(bar_right, kr > 0 ? kr : 1);
        mbar_init(bar_done, kComputeWarps);
    }
    if (warp < kComputeWarps && lane == 0) {
        const uint32_t bar0 = smem_addr(smem + kBarOffset) + warp * kStages * 8;
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
        int64_t* keys = reinterpret_cast<int64_t*>(smem + kKeyOffset) + warp * 2;
        keys[0] = -1;
        keys[1] = -1;
    }
    __syncthreads();
    if (warp != kEpilogueWarp) {
        if (P.M == 1) compute_warp<true>(P, smem, warp, lane, c0, n, nl, nr, bar_left, bar_right, bar_done);
        else compute_warp<false>(P, smem, warp, lane, c0, n, nl, nr, bar_left, bar_right, bar_done);
    } else {
        griddep_wait();
        epilogue_warp(P, smem, lane, c0, n, nl, nr, first, last, bar_left, bar_right, bar_done);
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

// Tensor map over a tensor's PN rows viewed as uint32 [N][row_bytes / 4],
// box = one 8-block chunk (68 words) x 16 rows; rows past N read as zero.
bool encode_rows(CUtensorMap* map, const GemvTensor& t) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(t.nb) * kBlockBytes;
    const cuuint64_t dims[2] = {row_bytes / 4, static_cast<cuuint64_t>(t.N)};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxWords), static_cast<cuuint32_t>(kTileRows)};
    const cuuint32_t estride[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(t.W), dims, strides, box,
              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int warp_max_ctas(int num_sms) { return kCtasPerSm * num_sms; }

cudaError_t launch_gemv_warp(const GemvTensor* t, int count, int M, void* workspace, size_t workspace_bytes,
                             int num_sms, uint64_t timeout_ns, int stall, cudaStream_t s, int* needs_bytes_out) {
    if (M < 1 || M > kWarpMaxM || count < 1 || count > kMaxLayer) return cudaErrorInvalidValue;
    WarpParams P{};
    uint64_t units = 0;
    int max_chunks = 1;
    for (int e = 0; e < count; ++e) {
        WTensor& T = P.t[e];
        T.x = t[e].x;
        T.y = t[e].y;
        T.N = t[e].N;
        T.type = t[e].type;
        T.K = t[e].nb * per_block(t[e].type);
        T.chunks = t[e].nb / kChunkBlocks;
        T.tiles = (t[e].N + kTileRows - 1) / kTileRows;
        T.unit_base = static_cast<uint32_t>(units);
        if (!encode_rows(&P.wmap[e], t[e])) return cudaErrorInvalidValue;
        units += static_cast<uint64_t>(T.chunks) * T.tiles;
        max_chunks = T.chunks > max_chunks ? T.chunks : max_chunks;
    }
    P.count = count;
    P.M = M;
    // every block range spans at least one whole tile, so a tile has at most two blocks
    uint64_t grid = units / static_cast<uint64_t>(max_chunks);
    if (grid > static_cast<uint64_t>(warp_max_ctas(num_sms))) grid = warp_max_ctas(num_sms);
    if (grid < 1) grid = 1;
    if (units * grid >= (1ull << 32) || units * kComputeWarps >= (1ull << 32)) return cudaErrorInvalidValue;
    P.grid = static_cast<int>(grid);
    P.units = static_cast<uint32_t>(units);
    const WorkspaceLayout L = workspace_layout(0, tc_max_ctas(num_sms));
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
    P.stall_first_step = stall;

    static bool attr_set = false;   // per process; the attribute is per function
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemv_warp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(P.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_warp_kernel, P);
}

}  // namespace pn
