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
//  * A block's eight warps split its units into equal contiguous shares of
//    one sequence that starts with the block's parts of the two tiles cut by
//    its boundaries, so those parts are finished first.  No warp ever waits
//    for another while it streams.
//  * Each warp owns a three-stage shared-memory ring: lane 0 issues one 2-D
//    TMA box (16 rows x 272 bytes) per unit, completing on the stage's
//    mbarrier, and the warp decodes one stage while the next two are in
//    flight.  x is read through L1, prefetched one unit ahead.
//  * A tile that one warp covers completely is stored at once.  The parts of
//    a tile split between warps go to shared memory; the last warp to finish
//    its part (a shared-memory counter) adds them in warp order.  A tile cut
//    by a block boundary is finished by the block holding its first chunks:
//    the other block stores its part as 64-bit {value, tag} words, which are
//    single-copy atomic and need no fence, and the first block picks them up
//    with loads it checks only after decoding its next unit, adds first part
//    + second part, stores, and clears the tags.  Results do not depend on
//    timing, and no fence, atomic or global round trip sits on the tail.
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

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kCtasPerSm = 2;
constexpr int kStages = 3;
constexpr int kTileRows = 16;
constexpr int kChunkBlocks = 8;
constexpr int kChunkBytes = kChunkBlocks * kBlockBytes;   // 272, one staged row
constexpr int kBoxWords = kChunkBytes / 4;                // TMA box inner extent, 32-bit elements
constexpr int kUnitBytes = kTileRows * kChunkBytes;       // 4352
constexpr int kWarpMaxM = 2;
constexpr int kRecFloats = kTileRows * kWarpMaxM;         // one part of a tile: [row][token]
// Segments of a block's sequence: its part of the tile cut by its left
// boundary, its part of the tile cut by its right boundary, the whole tiles
// in between.
constexpr int kSegLeft = 0, kSegRight = 1, kSegMid = 2;
// Per warp, two tile parts: [0] its part of a tile an earlier warp began,
// [1] its part of a tile it begins itself.
constexpr int kRingBytes = kWarps * kStages * kUnitBytes;
constexpr int kRecOffset = kRingBytes;                                  // [warp][2][kRecFloats] float
constexpr int kCntOffset = kRecOffset + kWarps * 2 * kRecFloats * 4;    // [warp] uint32: parts in, per begun tile
constexpr int kBarOffset = kCntOffset + kWarps * 4;                     // [warp][stage] mbarrier
constexpr int kSmemBytes = kBarOffset + kWarps * kStages * 8;
constexpr uint64_t kDrainLimitNs = 200ull * 1000 * 1000;
constexpr uint32_t kStatusTimeout = 5;                    // PN_ETIMEOUT
constexpr uint32_t kTagFull = 1u;                         // tag of a deposited part word

static_assert(kStagedRowBytes == kChunkBytes, "staged rows are one chunk wide");
static_assert(kUnitBytes % 128 == 0, "every stage starts 128-byte aligned");
static_assert(kSmemBytes <= 110 * 1024, "two thread blocks fit on one SM");
static_assert(kCntOffset % 8 == 0 && kBarOffset % 8 == 0, "aligned bookkeeping");

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
    uint32_t units;                // units * grid < 2^32 and units * 8 < 2^29 (checked on the host)
    uint32_t* status;
    uint64_t* tagged;              // [boundary][kRecFloats] {value bits, tag}
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

// Writes a tile part into record r of this warp: [row][token].
__device__ __forceinline__ void put_record(float* rec, int lane, const float (&v)[4]) {
    if ((lane & 3) != 0) return;
    const int row = tile_row(lane >> 2);
    rec[row * kWarpMaxM + 0] = v[0];
    rec[row * kWarpMaxM + 1] = v[1];
    rec[(row + 8) * kWarpMaxM + 0] = v[2];
    rec[(row + 8) * kWarpMaxM + 1] = v[3];
}

// Stores a finished tile sum held one value per lane: lane = row * 2 + token.
__device__ __forceinline__ void store_lanes(const WarpParams& P, const Cursor& c, float v, int lane) {
    const WTensor& T = P.t[c.e];
    const int row = c.tile * kTileRows + (lane >> 1), m = lane & 1;
    if (row < T.N && m < P.M) T.y[static_cast<int64_t>(m) * T.N + row] = v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// This block's part of the tile cut by its left boundary (the tile's later
// chunks), left for the previous block as {value bits, tag} words.
__device__ __forceinline__ void deposit(const WarpParams& P, float v, int lane) {
    st_relaxed_u64(P.tagged + static_cast<int64_t>(blockIdx.x) * kRecFloats + lane,
                   (static_cast<uint64_t>(kTagFull) << 32) | __float_as_uint(v));
}

// The tile cut by this block's right boundary: this block holds its first
// chunks and finishes it once the next block's part has arrived.  poll()
// checks the words loaded by the previous poll (issued at least one unit of
// decoding earlier) and loads them again while they are not all tagged.
struct Finisher {
    bool pending = false;
    float mine = 0.0f;         // this block's part (first chunks), lane = row * 2 + token
    uint64_t seen = 0;         // the word last loaded
    uint64_t t0 = 0;
    Cursor tile{0, 0, 0};
    __device__ uint64_t* word(const WarpParams& P, int lane) const {
        return P.tagged + static_cast<int64_t>(blockIdx.x + 1) * kRecFloats + lane;
    }
    __device__ void start(const WarpParams& P, const Cursor& c, float v, int lane) {
        pending = true;
        mine = v;
        tile = c;
        seen = ld_relaxed_u64(word(P, lane));
        t0 = globaltimer_ns();
    }
    __device__ void poll(const WarpParams& P, int lane) {
        if (!pending) return;
        if (__all_sync(0xFFFFFFFFu, static_cast<uint32_t>(seen >> 32) == kTagFull)) {
            store_lanes(P, tile, mine + __uint_as_float(static_cast<uint32_t>(seen)), lane);  // first + second part
            st_relaxed_u64(word(P, lane), 0ull);
            pending = false;
        } else if (globaltimer_ns() - t0 > P.timeout_ns) {
            if (lane == 0) atomicCAS(P.status, 0u, kStatusTimeout);
            pending = false;
        } else {
            seen = ld_relaxed_u64(word(P, lane));
        }
    }
};

// A warp's share of its block's units: up to three runs of consecutive units
// (left-cut part, right-cut part, middle), walked in order.  The runs are kept
// in scalars (run 0 is the current one) so that nothing is indexed at run time.
struct Walk {
    uint32_t a0, b0, a1, b1, a2, b2;   // runs [a, b) of units
    uint32_t q0, q1, q2;               // sequence position of each run's first unit
    int k0, k1, k2;                    // their segments: kSegLeft, kSegRight, kSegMid
    uint32_t u;                        // current unit, in run 0
    Cursor c;                          // its position
    __device__ void init() { a0 = b0 = a1 = b1 = a2 = b2 = 0; q0 = q1 = q2 = 0; k0 = k1 = k2 = 0; }
    __device__ void add(uint32_t a, uint32_t b, uint32_t q, int k) {
        if (a >= b) return;
        if (a0 == b0) { a0 = a; b0 = b; q0 = q; k0 = k; }
        else if (a1 == b1) { a1 = a; b1 = b; q1 = q; k1 = k; }
        else { a2 = a; b2 = b; q2 = q; k2 = k; }
    }
    __device__ bool valid() const { return a0 < b0; }
    __device__ uint32_t pos() const { return q0 + (u - a0); }
    __device__ void start(const WarpParams& P) {
        u = a0;
        if (valid()) c.locate(P, u);
    }
    __device__ void advance(const WarpParams& P) {
        if (++u < b0) {
            c.next(P);
            return;
        }
        a0 = a1; b0 = b1; q0 = q1; k0 = k1;
        a1 = a2; b1 = b2; q1 = q2; k1 = k2;
        a2 = b2 = 0;
        start(P);
    }
};

// The warp whose share [n w / 8, n (w + 1) / 8) holds sequence position pos.
__device__ __forceinline__ int warp_of(uint32_t pos, uint32_t n) {
    return min(static_cast<int>((pos * kWarps + kWarps - 1) / n), kWarps - 1);
}

// Accumulator fragments (lanes t = 0 hold rows tile_row(g), +8) as one value
// per lane, lane = row * 2 + token.
__device__ __forceinline__ float to_lanes(const float (&acc)[4], int lane) {
    const int row = lane >> 1, m = lane & 1, r = row & 7;
    const int src = (((r & 1) << 2) | (r >> 1)) << 2;      // lane g * 4 with tile_row(g) == r
    const float v0 = __shfl_sync(0xFFFFFFFFu, acc[0], src), v1 = __shfl_sync(0xFFFFFFFFu, acc[1], src);
    const float v2 = __shfl_sync(0xFFFFFFFFu, acc[2], src), v3 = __shfl_sync(0xFFFFFFFFu, acc[3], src);
    return row < 8 ? (m ? v1 : v0) : (m ? v3 : v2);
}

// This warp's part of a tile split between warps wa..wb (wa < wb).  The part goes to shared memory; the last warp
// to deliver its part gets true and the tile sum in warp order, one value per
// lane (lane = row * 2 + token).
__device__ bool hand_in(uint8_t* smem, int warp, int lane, int wa, int wb, uint32_t n, const float (&acc)[4],
                        float& sum) {
    float* recs = reinterpret_cast<float*>(smem + kRecOffset);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + kCntOffset);
    put_record(recs + (warp * 2 + (warp == wa ? 1 : 0)) * kRecFloats, lane, acc);
    // contributors: the warps of wa..wb whose share is not empty
    uint32_t parts = 0;
    for (int w = wa; w <= wb; ++w) parts += (n * (w + 1) / kWarps > n * w / kWarps) ? 1u : 0u;
    __threadfence_block();
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0) old = atomicAdd(cnt + wa, 1u);
    old = __shfl_sync(0xFFFFFFFFu, old, 0);
    if (old + 1 != parts) return false;
    __threadfence_block();
    sum = recs[(wa * 2 + 1) * kRecFloats + lane];
    for (int w = wa + 1; w <= wb; ++w)
        if (n * (w + 1) / kWarps > n * w / kWarps) sum += recs[(w * 2) * kRecFloats + lane];
    return true;
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

template <bool M1>
__device__ __forceinline__ void compute_unit(const WTensor& T, const uint8_t* stage, const uint16_t* xc, int lane,
                                             float (&acc)[4]) {
    if (T.type == kPn3t) unit_mma<kPn3t, M1>(stage, xc, lane, acc);
    else unit_mma<kPn4t, M1>(stage, xc, lane, acc);
}

template <bool M1>
__device__ void compute_warp(const WarpParams& P, uint8_t* smem, int warp, int lane, uint32_t c0, uint32_t n,
                             uint32_t nl, uint32_t nr, const Cursor& left_tile, const Cursor& right_tile) {
    const uint32_t p0 = n * static_cast<uint32_t>(warp) / kWarps;
    const uint32_t p1 = n * static_cast<uint32_t>(warp + 1) / kWarps;
    // sequence position -> unit: [0, nl) left-cut part, [nl, nl + nr) right-cut
    // part (the block's last nr units), [nl + nr, n) the middle
    Walk w;
    w.init();
    {
        const uint32_t l0 = min(p0, nl), l1 = min(p1, nl);
        const uint32_t r0 = min(max(p0, nl), nl + nr), r1 = min(max(p1, nl), nl + nr);
        const uint32_t m0 = max(p0, nl + nr), m1 = max(p1, nl + nr);
        w.add(c0 + l0, c0 + l1, l0, kSegLeft);
        w.add(c0 + n - nr + (r0 - nl), c0 + n - nr + (r1 - nl), r0, kSegRight);
        w.add(c0 + nl + (m0 - nl - nr), c0 + nl + (m1 - nl - nr), m0, kSegMid);
    }
    const uint32_t ring = smem_addr(smem) + warp * kStages * kUnitBytes;
    const uint8_t* ring_p = smem + warp * kStages * kUnitBytes;
    const uint32_t bar0 = smem_addr(smem + kBarOffset) + warp * kStages * 8;

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
    Finisher fin;
    int done = 0;
    while (cur.valid()) {
        const int s = done % kStages;
        if (!warp_wait(bar0 + 8 * s, static_cast<uint32_t>(done / kStages) & 1u, P.timeout_ns, lane)) {
            if (lane == 0) atomicCAS(P.status, 0u, kStatusTimeout);
            break;
        }
        const WTensor& T = P.t[cur.c.e];
        const uint16_t* xc = T.x + static_cast<int64_t>(token) * T.K + cur.c.chunk * kChunkBlocks * per_block(T.type);
        compute_unit<M1>(T, ring_p + s * kUnitBytes, xc, lane, acc);
        __syncwarp();
        if (iss.valid()) {                        // refill this stage
            if (lane == 0) fence_proxy_async_smem();
            issue(s);
        }
        ++done;
        fin.poll(P, lane);                        // words loaded one unit ago
        // the end of this warp's part of a tile?
        const int seg = cur.k0;
        const bool run_end = cur.u + 1 == cur.b0;
        const bool last_chunk = cur.c.chunk == T.chunks - 1;
        if (run_end || (seg == kSegMid && last_chunk)) {
            const uint32_t pos = cur.pos();
            const uint32_t ts = seg == kSegLeft ? 0u : seg == kSegRight ? nl : pos - cur.c.chunk;
            const uint32_t te = seg == kSegLeft ? nl : seg == kSegRight ? nl + nr : ts + T.chunks;
            const int wa = warp_of(ts, n), wb = warp_of(te - 1, n);
            float v = 0.0f;
            const bool whole = wa == wb;
            if (whole) v = to_lanes(acc, lane);
            if (whole || hand_in(smem, warp, lane, wa, wb, n, acc, v)) {
                if (seg == kSegLeft) deposit(P, v, lane);
                else if (seg == kSegRight) fin.start(P, right_tile, v, lane);
                else store_lanes(P, cur.c, v, lane);
            }
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
    while (fin.pending) {
        __nanosleep(64);
        fin.poll(P, lane);
    }
    (void)left_tile;
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
    if (lane == 0) {
        const uint32_t bar0 = smem_addr(smem + kBarOffset) + warp * kStages * 8;
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
        reinterpret_cast<uint32_t*>(smem + kCntOffset)[warp] = 0u;
    }
    __syncthreads();
    if (P.M == 1) compute_warp<true>(P, smem, warp, lane, c0, n, nl, nr, first, last);
    else compute_warp<false>(P, smem, warp, lane, c0, n, nl, nr, first, last);
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
    if (units * grid >= (1ull << 32) || units * kWarps >= (1ull << 32)) return cudaErrorInvalidValue;
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
    P.tagged = reinterpret_cast<uint64_t*>(ws + L.tagged);
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
