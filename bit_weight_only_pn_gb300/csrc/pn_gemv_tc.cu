// pn_gemv_tc.cu -- PN decode GEMV on GB300: TMA-staged rows, decode in registers,
// fp32 accumulation on the tensor cores (mma.sync m16n8k16).
//
// What is computed: y[m][r] = sum_k d_blk(r,k) * (n(r,k) - z) * x[m][k], the
// decode GEMV of the tensorless docs ("Why a P100-native weight format": "One
// lane, one word", "Exact decode in fp32") in its skinny M = 3 .. 16 form
// (speculative verification of k drafts in one batch, v100-skinny README, "How
// QPN works": packed weights stay compressed through HBM and are decoded at the
// point of consumption, straight into tensor-core register operands; M = 9 ..
// 16 is the band that README's "Where it stands" leaves to two 8-token tiles
// per weight pass).
//
// Design (GB300-first; the pages' sm_60 and sm_70 kernels are prior art):
//  * Work unit = one 16-row tile x one 8-block chunk (8 x 34 = 272 bytes per
//    row, 16-byte aligned whenever the row is).  Units are numbered tile-major
//    over every tensor of the call and the persistent grid (at most one CTA per
//    SM, each range at least one tile long) splits them into contiguous
//    ranges of equal modelled time (each unit's decode, a pn3t unit weighing
//    more than a pn4t one, plus a cost per batch step, since a step with few
//    tiles at work takes nearly as long as a full one), so every SM finishes
//    at about the same time and only a CTA's first and last tile can be
//    shared, each with one neighbour.  The split is searched on the host once
//    per call shape and cached.
//  * A CTA walks its tiles in batches of up to 8 consecutive tiles of one
//    tensor, chunk by chunk (one step = one chunk of the batch's tiles, so the
//    activation chunk is staged once for 8 tiles), last batch first so that
//    the shared tiles are settled early.
//  * One producer warp issues, per step, one tiled 2-D TMA copy per tile (a
//    tensor map over the PN rows, 16-row x 272-byte box) and one bulk copy per
//    activation row into a shared-memory ring (4 stages for M <= 8, 3 above)
//    completing on mbarriers.
//    Sixteen consumer warps, two per tile, each decode four of a chunk's eight
//    blocks.  An epilogue warp adds each tile's two halves (fixed order) and
//    stores it, or, for a shared tile, deposits its part and lets the last of
//    the two CTAs add both parts (fixed order), so results are deterministic.
//    Every wait is bounded in time.
//  * Decode: code words are read from shared memory as aligned 32-bit words
//    (blocks at even offsets are realigned with one byte-permute per word); a
//    LOP3 + HFMA2 per code pair turns two codes into the exact half2
//    (n - z, n' - z), which is exactly an A-fragment register of m16n8k16
//    (rows g and g+8 of the tile, k pairs from code words 2t, 2t+1); x is read
//    as B fragments straight from the staged chunk; each block's product sum
//    starts from zero and is scaled by its d in fp32, so every product is
//    exact and every sum is an fp32 sum.
//  * M = 9 .. 16 runs the same kernel with two 8-column tiles (NT = 2): each
//    decoded A fragment feeds two MMAs, one per 8 tokens, so the weights
//    still cross HBM once; the stage holds 16 activation rows and the ring
//    has three stages instead of four to stay within shared memory.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pn_device.cuh"
#include "pn_internal.h"

namespace pn {
namespace {

constexpr int kBatchTiles = 8;                          // tiles per batch (one per warp pair)
constexpr int kTileWarps = 2;                           // warps sharing a tile, 4 blocks each
constexpr int kConsumerWarps = kBatchTiles * kTileWarps;
constexpr int kProducerWarp = kConsumerWarps;           // warp 16
constexpr int kEpilogueWarp = kConsumerWarps + 1;       // warp 17
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kTileRows = 16;
constexpr int kChunkBlocks = 8;
constexpr int kWarpBlocks = kChunkBlocks / kTileWarps;  // blocks of a chunk per warp
constexpr int kChunkBytes = kChunkBlocks * kBlockBytes; // 272
constexpr int kRowPitch = kChunkBytes;                  // rows land densely (TMA box)
constexpr int kBoxWords = kChunkBytes / 4;              // box inner extent, 32-bit elements
constexpr int kTileBytes = kTileRows * kRowPitch;       // 4352
constexpr int kStageWBytes = kBatchTiles * kTileBytes;  // 34816
constexpr int kXPitchPn3t = kChunkBlocks * 80 * 2 + 16; // 1296
constexpr int kXPitchPn4t = kChunkBlocks * 64 * 2 + 16; // 1040
constexpr int kXRowBytes = (kXPitchPn3t + 127) / 128 * 128;   // 1408
constexpr int kOutBuffers = 2;
constexpr uint64_t kDrainLimitNs = 200ull * 1000 * 1000;
constexpr uint32_t kStatusTimeout = 5;                  // PN_ETIMEOUT
constexpr int kSlotFloats = kTileRows * kMaxM;          // 256: one tile's partial sums
// Weights of the work split (RangeModel): the cost of one batch step and of
// one pn3t / pn4t unit, for one and two column tiles.  A step costs several
// units because a batch step takes most of a full step's time even when few
// of its tiles have work.  The values were chosen by timing the kernel over a
// grid of weights (step 0 .. 180, pn3t 16 .. 28 against pn4t 15) on two
// mixed pn3t / pn4t layers (27B-class, hidden 5120; and hidden 2560) at 3, 8,
// 12 and 16 tokens: against an even split of the units at 16 / 15 they made
// the 27B-class layer 11 - 15 % faster with one column tile and 6 - 8 % with
// two, and the small layer 1 - 2 % faster.
struct SplitWeights {
    uint32_t step, pn3t, pn4t;
};
constexpr SplitWeights kSplitWeights[2] = {{126, 20, 15}, {90, 22, 15}};
constexpr int kMaxGrid = 256;                           // thread blocks per launch, at most

// Shared-memory layout of the kernel with NT 8-column tiles (M <= 8 NT).
template <int NT>
struct Smem {
    // Activations: one block of M rows per chunk lane, each block 128-byte
    // aligned (a tiled TMA destination); lanes * M <= 8 NT, so 8 NT rows of
    // the pn3t pitch rounded up to 128 bytes always fit.
    static constexpr int kXRows = 8 * NT;
    static constexpr int kStageXBytes = kXRows * kXRowBytes;       // 11264 / 22528
    static constexpr int kStageBytes = kStageWBytes + kStageXBytes;
    static constexpr int kStages = NT == 1 ? 4 : 3;
    // Finished tile sums handed to the epilogue warp:
    // [tile][buffer][half][column tile][lane] float4.
    static constexpr int kOutOffset = kStages * kStageBytes;
    static constexpr int kOutBytes = kBatchTiles * kOutBuffers * kTileWarps * NT * 32 * 16;
    static constexpr int kBarrierOffset = kOutOffset + kOutBytes;
    static constexpr int kNumBarriers = 2 * kStages + 2 * kBatchTiles * kOutBuffers;
    static constexpr int kBytes = kBarrierOffset + kNumBarriers * 8 + 16;
    static_assert(kStageBytes % 128 == 0, "TMA destinations stay aligned");
    static_assert(kXRows * kXPitchPn3t <= kStageXBytes, "one block of 8 NT activation rows fits");
    static_assert(kBytes <= 227 * 1024, "fits one SM's shared memory");
};

static_assert(kStageWBytes % 128 == 0, "TMA destinations stay aligned");
static_assert(2 * 8 <= kMaxM, "partial-sum slots hold 16 tokens");

// Bytes between the activation blocks of consecutive chunk lanes.
__host__ __device__ constexpr int x_block_bytes(int M, int pitch) { return (M * pitch + 127) / 128 * 128; }

struct TcTensor {
    const uint8_t* W;
    const uint16_t* x;
    float* y;
    uint32_t unit_base;     // first unit of this tensor (tile-major, chunk-minor)
    int N;
    int nb;
    int type;
    int chunks;             // nb / 8
    int tiles;              // ceil(N / 16)
};

constexpr int kBoxSizes = 4;       // row boxes of 1, 2, 4, 8 tiles

struct TcParams {
    // per tensor: PN rows as uint32 [N][row_bytes/4]; box 68 words x (16 << k) rows
    CUtensorMap wmap[kBoxSizes][kMaxLayer];
    // per tensor: activations as uint64 [M][K/4]; box = one chunk + 16 bytes x M rows,
    // so consecutive rows land at the padded pitch (the extra 16 bytes are unused)
    CUtensorMap xmap[kMaxLayer];
    TcTensor t[kMaxLayer];
    int count;
    int M;
    int x_rows;                    // activation rows a stage holds (8 per column tile)
    int grid;
    uint32_t starts[kMaxGrid + 1]; // block c's units are [starts[c], starts[c + 1])
    uint32_t* status;
    uint32_t* counters;            // one per CTA boundary
    float* partials;               // [boundary][side][kSlotFloats]
    uint64_t timeout_ns;
    int stall_first_step;          // testing aid: see pn_set_test_stall
};

// One batch: tiles [tb, tb + nt) of tensor e; its first tile starts at chunk
// cs0 and its last tile ends at chunk ce_last (a CTA boundary may cut them).
// A batch of fewer than 8 tiles gives each tile `lanes` warp pairs, which
// take consecutive chunks: warp pair p works on tile p / lanes, chunk
// c + p % lanes of each step.
struct Batch {
    int e, tb, nt, cs0, ce_last, lanes, lanes_log2, chunks;
};


// Whether warp pair p has work in the step of batch b starting at chunk c,
// and which tile (batch-relative) and chunk it takes.
__device__ __forceinline__ bool slot_work(const Batch& b, int c, int p, int& j, int& chunk) {
    j = p >> b.lanes_log2;
    chunk = c + (p & (b.lanes - 1));
    if (j >= b.nt) return false;
    const int cs = j == 0 ? b.cs0 : 0;
    const int ce = j == b.nt - 1 ? b.ce_last : b.chunks;
    return chunk >= cs && chunk < ce;
}

// First unit of CTA c's range.
__device__ __forceinline__ uint32_t range_start(const TcParams& P, int c) {
    return P.starts[c];
}

// Tensor, tile and chunk of unit u.
__device__ __forceinline__ void locate(const TcParams& P, uint32_t u, int& e, int& tile, int& c) {
    e = 0;
    while (e + 1 < P.count && u >= P.t[e + 1].unit_base) ++e;
    const uint32_t rel = u - P.t[e].unit_base;
    tile = static_cast<int>(rel / static_cast<uint32_t>(P.t[e].chunks));
    c = static_cast<int>(rel - static_cast<uint32_t>(tile) * P.t[e].chunks);
}

// Walks a CTA's unit range [u0, u1) batch by batch.  The batches are the
// windows of 8 tiles that start at the range's first tile (and at tile 0 of
// each later tensor); the last one is walked first, then the others in order.
// Within a batch the steps are c = cstart, cstart + lanes, ... < cend.
struct Walker {
    int e0, t0, c0, e1, t1, c1e;    // first unit; last unit's tensor, tile, chunk + 1
    Batch cur;
    int lastE, lastTb;              // the last batch
    int seq;                        // batches started so far
    int cstart, cend;               // step range of the current batch
    bool done;

    __device__ Batch make(const TcParams& P, int e, int tb) const {
        Batch b;
        b.e = e;
        b.tb = tb;
        int nt = min(kBatchTiles, P.t[e].tiles - tb);
        if (e == e1) nt = min(nt, t1 - tb + 1);
        b.nt = nt;
        b.cs0 = (e == e0 && tb == t0) ? c0 : 0;
        b.ce_last = (e == e1 && tb + nt - 1 == t1) ? c1e : P.t[e].chunks;
        // chunk lanes: a power of two, as many as the 8 warp pairs and the
        // staged activation rows allow, no more than the tile has chunks
        const int cap = min(min(kBatchTiles / nt, P.x_rows / P.M), P.t[e].chunks);
        b.lanes_log2 = cap >= 8 ? 3 : cap >= 4 ? 2 : cap >= 2 ? 1 : 0;
        b.lanes = 1 << b.lanes_log2;
        b.chunks = P.t[e].chunks;
        return b;
    }
    __device__ void start(const Batch& b) {
        cur = b;
        // only a batch of one tile can start late and end early at once
        cstart = b.nt == 1 ? b.cs0 : 0;
        cend = b.nt == 1 ? b.ce_last : b.chunks;
        ++seq;
    }
    __device__ void init(const TcParams& P, uint32_t u0, uint32_t u1) {
        seq = -1;
        done = u1 <= u0;
        if (done) return;
        locate(P, u0, e0, t0, c0);
        int c1;
        locate(P, u1 - 1, e1, t1, c1);
        c1e = c1 + 1;
        lastE = e1;
        lastTb = (e1 == e0) ? t0 + kBatchTiles * ((t1 - t0) / kBatchTiles)
                            : kBatchTiles * (t1 / kBatchTiles);
        start(make(P, lastE, lastTb));
    }
    // Moves to the batch after `cur` in processing order; done when none is left.
    __device__ void next_batch(const TcParams& P) {
        int e, tb;
        if (seq == 0) {                       // the last batch was first; now the first
            e = e0;
            tb = t0;
        } else {
            e = cur.e;
            tb = cur.tb + kBatchTiles;
            if (tb >= P.t[e].tiles) { ++e; tb = 0; }
        }
        if (e == lastE && tb == lastTb) { done = true; return; }
        start(make(P, e, tb));
    }
};

// Position in a ring of STAGES stages.
template <int STAGES>
struct Ring {
    int s = 0;
    uint32_t phase = 0;
    __device__ void advance() {
        if (++s == STAGES) { s = 0; phase ^= 1u; }
    }
};

__device__ __forceinline__ void raise_timeout(const TcParams& P, volatile uint32_t* abort_flag) {
    *abort_flag = 1u;
    atomicCAS(P.status, 0u, kStatusTimeout);
}

// Waits for phase `parity` of an mbarrier; gives up after limit_ns, or as soon
// as another warp of the CTA has aborted (abort_flag may be null).  Between
// probes the thread sleeps briefly, so waiting warps leave most issue slots
// to the warps that are decoding.
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                             volatile uint32_t* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(20);
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag && *abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Warp-level wait.  Fast path: every lane probes the barrier once and the
// warp votes; when the phase has already completed (the usual case) each lane
// has observed it itself, so its later shared-memory reads are ordered after
// it, and the warp goes on without a shuffle, a sync or a divergent branch
// (measured 4 to 5 % faster at 8 and 16 tokens).  Otherwise lane 0 polls
// (one poller per warp keeps the barrier traffic 32x below every-lane
// polling), the warp learns the outcome by shuffle, and __syncwarp orders the
// other lanes' later reads after lane 0's observation.  Every lane of the
// warp must call it.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          volatile uint32_t* abort_flag, int lane) {
    if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
    bool ok = true;
    if (lane == 0) ok = wait_bounded(bar, parity, limit_ns, abort_flag);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok;
}

// Warp-level arrive: after __syncwarp (all lanes' reads of the stage are done)
// lane 0 arrives once for the warp.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// ----------------------------------------------------------------- decode --

// x pairs for code words 2t (xb[0..P-1]) and 2t+1 (xb[P..2P-1]) of block B.
template <int TYPE, int B>
__device__ __forceinline__ void load_x(const uint8_t* xrow, int t, uint32_t (&xb)[2 * Format<TYPE>::kPairs]) {
    using F = Format<TYPE>;
    const uint8_t* a = xrow + (B * F::kPerBlock + 2 * F::kPerWord * t) * 2;
    if constexpr (TYPE == kPn3t) {                      // 8-byte aligned
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const uint2 p = lds_u64(a + 8 * i);
            xb[2 * i] = p.x; xb[2 * i + 1] = p.y;
        }
    } else {                                            // 16-byte aligned
        const uint4 p = lds_u128(a);
        const uint4 q = lds_u128(a + 16);
        xb[0] = p.x; xb[1] = p.y; xb[2] = p.z; xb[3] = p.w;
        xb[4] = q.x; xb[5] = q.y; xb[6] = q.z; xb[7] = q.w;
    }
}

// One consumer warp: the 16 rows of its tile times blocks 4H .. 4H+3 of a
// chunk (the other warp of the pair takes the other four), for NT column
// tiles of 8 tokens.  The scaled block sums are added up per call and then
// added to the running sum, which keeps every fp32 summation chain short (at
// most 4 block terms + one term per chunk) whatever K is.  xrow[n] is this
// lane's activation row in column tile n; lanes whose MMA column is past M
// read token 0 (a B column only feeds its own, unused, output column), so no
// lane takes a different path.
template <int TYPE, int H, int NT>
__device__ __forceinline__ void mma_tile_half(const uint8_t* tile, const uint8_t* const (&xrow)[NT], int lane,
                                              float (&acc)[NT][4]) {
    using F = Format<TYPE>;
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* r0 = tile + tile_row(g) * kRowPitch;
    const uint8_t* r1 = r0 + 8 * kRowPitch;
    float part[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) part[n][0] = part[n][1] = part[n][2] = part[n][3] = 0.0f;
    static_for<kWarpBlocks>([&](auto bc) {
        constexpr int B = H * kWarpBlocks + decltype(bc)::value;
        if constexpr (NT == 1) {
            // one column tile: the block's x pairs are loaded up front
            uint32_t xb[2 * F::kPairs];
            load_x<TYPE, B>(xrow[0], t, xb);
            block_mma<TYPE, B, 1>(r0, r1, t, [&](int, auto sc) {
                constexpr int S = decltype(sc)::value;
                return make_uint2(xb[2 * S], xb[2 * S + 1]);
            }, part);
        } else {
            // two: each MMA's pairs are loaded next to it (one 64-bit load per
            // MMA and tile), which keeps the operands within 96 registers
            const int xoff = (B * F::kPerBlock + 2 * F::kPerWord * t) * 2;
            block_mma<TYPE, B, NT>(r0, r1, t, [&](int n, auto sc) {
                constexpr int S = decltype(sc)::value;
                return lds_u64(xrow[n] + xoff + 8 * S);
            }, part);
        }
    });
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[n][i] += part[n][i];
}

// ------------------------------------------------------------------ flush --

// Row of a tile that fragment row g (and g + 8) reads, see tile_row.  v[n]
// holds tokens 8n + 2t, 8n + 2t + 1 of rows g and g + 8.
template <int NT>
__device__ __forceinline__ void store_tile(const TcTensor& T, int M, int tile, int lane,
                                           const float (&v)[NT][4]) {
    const int row0 = tile * kTileRows + tile_row(lane >> 2);
    const int rows[2] = {row0, row0 + 8};
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int m0 = 8 * n + 2 * (lane & 3);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (rows[h] < T.N) {
                if (m0 < M) T.y[static_cast<int64_t>(m0) * T.N + rows[h]] = v[n][2 * h];
                if (m0 + 1 < M) T.y[static_cast<int64_t>(m0 + 1) * T.N + rows[h]] = v[n][2 * h + 1];
            }
        }
    }
}

// Partial sums of the tile shared across CTA boundary b (between CTA b-1 and
// CTA b): side 0 holds CTA b-1's part (the tile's first chunks), side 1 CTA
// b's; [row][token], kMaxM tokens per row.
__device__ __forceinline__ float* slot_ptr(const TcParams& P, int boundary, int side) {
    return P.partials + (static_cast<int64_t>(boundary) * 2 + side) * kSlotFloats;
}

// Writes / reads this lane's values of a tile to / from a partial-sum slot.
template <int NT>
__device__ __forceinline__ void slot_store(float* s, int lane, const float (&v)[NT][4]) {
    const int r = lane >> 2;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int m0 = 8 * n + 2 * (lane & 3);
        __stcg(reinterpret_cast<float2*>(s + r * kMaxM + m0), make_float2(v[n][0], v[n][1]));
        __stcg(reinterpret_cast<float2*>(s + (r + 8) * kMaxM + m0), make_float2(v[n][2], v[n][3]));
    }
}
template <int NT>
__device__ __forceinline__ void slot_load(const float* s, int lane, float (&v)[NT][4]) {
    const int r = lane >> 2;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int m0 = 8 * n + 2 * (lane & 3);
        const float2 a = __ldcg(reinterpret_cast<const float2*>(s + r * kMaxM + m0));
        const float2 b = __ldcg(reinterpret_cast<const float2*>(s + (r + 8) * kMaxM + m0));
        v[n][0] = a.x; v[n][1] = a.y; v[n][2] = b.x; v[n][3] = b.y;
    }
}

template <int NT>
__device__ __forceinline__ uint32_t out_slot(uint32_t sbase, int tile, int buf, int half, int n, int lane) {
    return sbase + Smem<NT>::kOutOffset + ((((tile * kOutBuffers + buf) * kTileWarps + half) * NT + n) * 32 + lane) * 16;
}

// The finished sums of warp pair p (first half + second half, in that
// order), read from the hand-off slots in shared memory.
template <int NT>
__device__ __forceinline__ void tile_sum(uint32_t sbase, int j, int buf, int lane, float (&v)[NT][4]) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        float a[4], b[4];
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(a[0]), "=f"(a[1]), "=f"(a[2]), "=f"(a[3])
                     : "r"(out_slot<NT>(sbase, j, buf, 0, n, lane)) : "memory");
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(b[0]), "=f"(b[1]), "=f"(b[2]), "=f"(b[3])
                     : "r"(out_slot<NT>(sbase, j, buf, 1, n, lane)) : "memory");
#pragma unroll
        for (int i = 0; i < 4; ++i) v[n][i] = a[i] + b[i];
    }
}

// Emits the tiles of batch `b` from the epilogue warp.  Whole tiles are
// stored.  A tile cut by a CTA boundary deposits this CTA's part; after one
// fence the (at most two) boundary counters are bumped together; where this
// CTA arrived second it loads the neighbour's part and stores left + right.
// `bufs` holds each warp pair's hand-off buffer index in bit p.
template <int NT>
__device__ void flush_batch(const TcParams& P, const Batch& b, int lane, uint32_t sbase, uint32_t bufs) {
    const TcTensor& T = P.t[b.e];
    const int cta = blockIdx.x;
    const bool left_cut = b.cs0 > 0;                 // tile 0 began in CTA cta-1
    const bool right_cut = b.ce_last < T.chunks;     // tile nt-1 ends in CTA cta+1
    float vl[NT][4], vr[NT][4];
    // (the two-tile form keeps this loop rolled: unrolled, its sums do not
    // fit the 96 registers)
#pragma unroll (NT == 1 ? kBatchTiles : 1)
    for (int j = 0; j < kBatchTiles; ++j) {
        if (j >= b.nt) continue;
        float v[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) v[n][0] = v[n][1] = v[n][2] = v[n][3] = 0.0f;
        for (int q = 0; q < b.lanes; ++q) {          // the tile's chunk lanes, in order
            float w[NT][4];
            const int p = j * b.lanes + q;
            tile_sum<NT>(sbase, p, (bufs >> p) & 1u, lane, w);
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int i = 0; i < 4; ++i) v[n][i] += w[n][i];
        }
        const bool lc = left_cut && j == 0, rc = right_cut && j == b.nt - 1;
        if (lc) {
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int i = 0; i < 4; ++i) vl[n][i] = v[n][i];
        } else if (rc) {
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int i = 0; i < 4; ++i) vr[n][i] = v[n][i];
        } else {
            store_tile<NT>(T, P.M, b.tb + j, lane, v);
        }
    }
    if (!left_cut && !right_cut) return;
    // deposit: our part of the left-cut tile is side 1 of boundary cta; of the
    // right-cut tile, side 0 of boundary cta + 1
    if (left_cut) slot_store<NT>(slot_ptr(P, cta, 1), lane, vl);
    if (right_cut) slot_store<NT>(slot_ptr(P, cta + 1, 0), lane, vr);
    __threadfence();
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0 && left_cut) old = atomicAdd(P.counters + cta, 1u);
    if (lane == 1 && right_cut) old = atomicAdd(P.counters + cta + 1, 1u);
    const bool l_last = left_cut && __shfl_sync(0xFFFFFFFFu, old, 0) == 1u;
    const bool r_last = right_cut && __shfl_sync(0xFFFFFFFFu, old, 1) == 1u;
    if (!l_last && !r_last) return;
    __threadfence();
    if (l_last) {                                    // left part (cta-1) + right part (cta)
        float o[NT][4], v[NT][4];
        slot_load<NT>(slot_ptr(P, cta, 0), lane, o);
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) v[n][i] = o[n][i] + vl[n][i];
        store_tile<NT>(T, P.M, b.tb, lane, v);
        if (lane == 0) atomicExch(P.counters + cta, 0u);
    }
    if (r_last) {                                    // left part (cta) + right part (cta+1)
        float o[NT][4], v[NT][4];
        slot_load<NT>(slot_ptr(P, cta + 1, 1), lane, o);
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) v[n][i] = vr[n][i] + o[n][i];
        store_tile<NT>(T, P.M, b.tb + b.nt - 1, lane, v);
        if (lane == 0) atomicExch(P.counters + cta + 1, 0u);
    }
}

// ----------------------------------------------------------------- kernel --

struct Barriers {
    uint32_t full0, empty0, ofull0, ofree0;
    __device__ uint32_t full(int s) const { return full0 + 8 * s; }
    __device__ uint32_t empty(int s) const { return empty0 + 8 * s; }
    __device__ uint32_t out_full(int j, int b) const { return ofull0 + 8 * (j * kOutBuffers + b); }
    __device__ uint32_t out_free(int j, int b) const { return ofree0 + 8 * (j * kOutBuffers + b); }
};

// Consumer side of a tile hand-off: the k-th finished sum of `tile` goes to
// buffer k % 2 once the epilogue has emptied that buffer's previous use.
template <int NT>
__device__ bool handoff(const TcParams& P, const Barriers& B, uint32_t sbase, int tile, int half,
                        int lane, uint32_t k, const float (&acc)[NT][4], volatile uint32_t* abort_flag) {
    const int buf = k & 1u;
    const uint32_t use = k >> 1;
    if (use > 0 && !warp_wait(B.out_free(tile, buf), (use - 1) & 1u, P.timeout_ns, abort_flag, lane)) {
        if (lane == 0) raise_timeout(P, abort_flag);
        return false;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                     :: "r"(out_slot<NT>(sbase, tile, buf, half, n, lane)), "f"(acc[n][0]), "f"(acc[n][1]),
                        "f"(acc[n][2]), "f"(acc[n][3]) : "memory");
    warp_arrive(B.out_full(tile, buf), lane);
    return true;
}

// One consumer warp's steps of batch b: warp pair `slot` takes tile
// slot >> lanes_log2 at chunk c + (slot & (lanes - 1)) of every step.
// xtoken[n] is the activation row this lane reads for column tile n.
template <int TYPE, int H, int NT>
__device__ bool consume_batch(const TcParams& P, const Barriers& B, const Walker& it, const uint8_t* smem,
                              int slot, int lane, const int (&xtoken)[NT], Ring<Smem<NT>::kStages>& ring,
                              float (&acc)[NT][4], volatile uint32_t* abort_flag) {
    const Batch& b = it.cur;
    constexpr int kPitch = TYPE == kPn3t ? kXPitchPn3t : kXPitchPn4t;
    const int j = slot >> b.lanes_log2;
    const int q = slot & (b.lanes - 1);
    const bool in = j < b.nt;
    const int cs = (j == 0 ? b.cs0 : 0) - q;             // work when cs <= c < ce
    const int ce = (j == b.nt - 1 ? b.ce_last : b.chunks) - q;
    const int toff = slot * kTileBytes;
    const int xoff = kStageWBytes + q * x_block_bytes(P.M, kPitch);
    for (int c = it.cstart; c < it.cend; c += b.lanes) {
        if (!warp_wait(B.full(ring.s), ring.phase, P.timeout_ns, abort_flag, lane)) {
            if (lane == 0) raise_timeout(P, abort_flag);
            return false;
        }
        if (in && c >= cs && c < ce) {
            const uint8_t* stage = smem + ring.s * Smem<NT>::kStageBytes;
            const uint8_t* xrow[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) xrow[n] = stage + xoff + xtoken[n] * kPitch;
            mma_tile_half<TYPE, H, NT>(stage + toff, xrow, lane, acc);
        }
        warp_arrive(B.empty(ring.s), lane);
        ring.advance();
    }
    return !*abort_flag;
}

// One CTA per SM.  Its 18 warps sit on the SM's four schedulers as 5, 5, 4,
// 4, and a scheduler's 16,384 registers over 5 warps of 32 threads allow at
// most 96 registers per thread (what the launch bounds give).
template <int NT>
__global__ void __launch_bounds__(kThreads, 1) gemv_tc_kernel(const __grid_constant__ TcParams P) {
    using L = Smem<NT>;
    constexpr int kStages = L::kStages;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    Barriers B;
    B.full0 = sbase + L::kBarrierOffset;
    B.empty0 = B.full0 + kStages * 8;
    B.ofull0 = B.empty0 + kStages * 8;
    B.ofree0 = B.ofull0 + kBatchTiles * kOutBuffers * 8;
    volatile uint32_t* abort_flag =
        reinterpret_cast<volatile uint32_t*>(smem + L::kBarrierOffset + L::kNumBarriers * 8);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // programmatic dependent launch: the next kernel may start now; this one
    // touches activations, outputs and the workspace only after the previous
    // kernel has finished (griddep_wait below), warming L2 with its first
    // weights meanwhile
    griddep_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(B.full(s), 1);
            mbar_init(B.empty(s), kConsumerWarps);
        }
        for (int j = 0; j < kBatchTiles; ++j)
            for (int b = 0; b < kOutBuffers; ++b) {
                mbar_init(B.out_full(j, b), kTileWarps);
                mbar_init(B.out_free(j, b), 1);
            }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();

    const uint32_t u0 = range_start(P, blockIdx.x);
    const uint32_t u1 = range_start(P, blockIdx.x + 1);

    if (warp == kProducerWarp) {
        // ------------------------------------------------------- producer --
        // Per step: one barrier wait, one expect_tx, one copy per lane.  Every
        // per-batch quantity is computed when the batch starts, so the loop
        // that feeds the ring stays short (this warp shares its scheduler
        // with four decoding warps).
        if (lane < P.count) {
#pragma unroll
            for (int k = 0; k < kBoxSizes; ++k) prefetch_tensormap(&P.wmap[k][lane]);
            prefetch_tensormap(&P.xmap[lane]);
        }
        Walker it;
        it.init(P, u0, u1);
        if (!it.done && lane < kBatchTiles) {
            // the first two steps' weight rows of the first batch, into L2
            const Batch& b = it.cur;
            const int j = lane >> b.lanes_log2, q = lane & (b.lanes - 1);
            if (j < b.nt)
                for (int k = 0; k < 2; ++k) {
                    const int c = it.cstart + q + k * b.lanes;
                    if (c < it.cend) tma_prefetch_l2_2d(&P.wmap[0][b.e], c * kBoxWords, (b.tb + j) * kTileRows);
                }
        }
        griddep_wait();
        Ring<kStages> ring;
        int idx = 0;
        bool stop = false;
        while (!it.done && !stop) {
            const Batch b = it.cur;
            const bool p3 = P.t[b.e].type == kPn3t;
            const int xwords = p3 ? kChunkBlocks * 80 / 4 : kChunkBlocks * 64 / 4;   // u64 per chunk
            const int xrow_bytes = p3 ? kXPitchPn3t : kXPitchPn4t;
            const int xblock = x_block_bytes(P.M, xrow_bytes);
            const uint32_t xtx = static_cast<uint32_t>(P.M * xrow_bytes);
            const void* xmap = &P.xmap[b.e];
            const int row0 = b.tb * kTileRows;
            for (int c = it.cstart; c < it.cend; c += b.lanes) {
                if (*abort_flag) { stop = true; break; }
                if (idx >= kStages && !warp_wait(B.empty(ring.s), ring.phase ^ 1u, P.timeout_ns, abort_flag, lane)) {
                    if (lane == 0) raise_timeout(P, abort_flag);
                    stop = true;
                    break;
                }
                const int nq = min(b.lanes, b.chunks - c);
                // tiles with a box this step
                int jlo = 0, jhi = 0, nbox;
                uint32_t mask = 0;
                if (b.lanes == 1) {
                    jlo = c < b.cs0 ? 1 : 0;
                    jhi = c >= b.ce_last ? b.nt - 1 : b.nt;
                    nbox = jhi - jlo;
                } else {
#pragma unroll
                    for (int p = 0; p < kBatchTiles; ++p) {
                        int j, ch;
                        if (slot_work(b, c, p, j, ch)) mask |= 1u << p;
                    }
                    nbox = __popc(mask);
                }
                const uint32_t full = B.full(ring.s);
                const uint32_t stage = sbase + ring.s * L::kStageBytes;
                // a box past the last row or the end of x is zero-filled and still counts in full
                if (lane == 0) mbar_arrive_expect_tx(full, nq * xtx + static_cast<uint32_t>(nbox * kTileBytes));
                __syncwarp();
                if (!(P.stall_first_step && idx == 0)) {
                    if (lane < nq) {                // activation chunk c + lane, all M rows
                        tma_load_2d(stage + kStageWBytes + lane * xblock, xmap, (c + lane) * xwords, 0, full);
                    } else if (lane >= 8 && lane < 8 + kBatchTiles) {
                        const int i = lane - 8;
                        if (b.lanes == 1) {
                            // tiles [jlo, jhi) as boxes of 8, 4, 2, 1 tiles, largest
                            // first; this lane issues box number i
                            int j = jlo, k = 0;
                            for (int n = 0; j < jhi; ++n) {
                                const int left = jhi - j;
                                const int lg = left >= 8 ? 3 : left >= 4 ? 2 : left >= 2 ? 1 : 0;
                                if (n == i) { k = lg; break; }
                                j += 1 << lg;
                            }
                            if (j < jhi)
                                tma_load_2d(stage + j * kTileBytes, &P.wmap[k][b.e], c * kBoxWords,
                                            row0 + j * kTileRows, full);
                        } else if ((mask >> i) & 1u) {
                            tma_load_2d(stage + i * kTileBytes, &P.wmap[0][b.e],
                                        (c + (i & (b.lanes - 1))) * kBoxWords,
                                        row0 + (i >> b.lanes_log2) * kTileRows, full);
                        }
                    }
                }
                // (testing aid: with stall_first_step the first step's bytes
                // are announced but never copied; its wait can only time out)
                ring.advance();
                ++idx;
            }
            if (!stop) it.next_batch(P);
        }
        // Every copy this warp started must land before the CTA can exit.
        // Stage s was last filled by step s + kStages * r for the largest such
        // step below idx; after a normal run that phase has completed (the
        // consumers waited for it) and this returns at once; after an abort it
        // waits, bounded, for the copies still in flight.
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < kStages; ++s) {
                if (idx <= s) continue;
                const uint32_t last_round = static_cast<uint32_t>((idx - 1 - s) / kStages);
                if (P.stall_first_step && s == 0 && last_round == 0) continue;   // never copied
                wait_bounded(B.full(s), last_round & 1u, kDrainLimitNs, nullptr);
            }
        }
    } else if (warp == kEpilogueWarp) {
        // ------------------------------------------------------- epilogue --
        // Walks the same batches; when a batch's warp pairs have handed off
        // their sums it emits the batch.
        griddep_wait();
        Walker it;
        it.init(P, u0, u1);
        uint32_t kcount[kBatchTiles];
#pragma unroll
        for (int p = 0; p < kBatchTiles; ++p) kcount[p] = 0;
        while (!it.done) {
            const Batch& cur = it.cur;
            const int slots = cur.nt * cur.lanes;
            uint32_t bufs = 0;
            bool ok = true;
#pragma unroll
            for (int p = 0; p < kBatchTiles; ++p) {
                if (p >= slots || !ok) continue;
                const int buf = kcount[p] & 1u;
                bufs |= static_cast<uint32_t>(buf) << p;
                if (!warp_wait(B.out_full(p, buf), (kcount[p] >> 1) & 1u, P.timeout_ns, abort_flag, lane)) {
                    if (lane == 0) raise_timeout(P, abort_flag);
                    ok = false;
                }
            }
            if (!ok) break;
            flush_batch<NT>(P, cur, lane, sbase, bufs);
#pragma unroll
            for (int p = 0; p < kBatchTiles; ++p) {
                if (p >= slots) continue;
                warp_arrive(B.out_free(p, (bufs >> p) & 1u), lane);
                ++kcount[p];
            }
            if (*abort_flag) break;
            it.next_batch(P);
        }
    } else {
        // ------------------------------------------------------- consumers --
        griddep_wait();
        const int slot = warp >> 1, half = warp & 1;
        int xtoken[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) xtoken[n] = 8 * n + (lane >> 2) < P.M ? 8 * n + (lane >> 2) : 0;
        Walker it;
        it.init(P, u0, u1);
        Ring<kStages> ring;
        uint32_t handoffs = 0;
        while (!it.done) {
            float acc[NT][4];
#pragma unroll
            for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
            bool ok;
            if (P.t[it.cur.e].type == kPn3t)
                ok = half == 0
                    ? consume_batch<kPn3t, 0, NT>(P, B, it, smem, slot, lane, xtoken, ring, acc, abort_flag)
                    : consume_batch<kPn3t, 1, NT>(P, B, it, smem, slot, lane, xtoken, ring, acc, abort_flag);
            else
                ok = half == 0
                    ? consume_batch<kPn4t, 0, NT>(P, B, it, smem, slot, lane, xtoken, ring, acc, abort_flag)
                    : consume_batch<kPn4t, 1, NT>(P, B, it, smem, slot, lane, xtoken, ring, acc, abort_flag);
            if (!ok) break;
            if (slot < it.cur.nt * it.cur.lanes &&
                !handoff<NT>(P, B, sbase, slot, half, lane, handoffs++, acc, abort_flag))
                break;
            it.next_batch(P);
        }
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
// box = one 8-block chunk (68 words) x `rows` rows.
bool encode_rows(CUtensorMap* map, const GemvTensor& t, int rows) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(t.nb) * kBlockBytes;
    const cuuint64_t dims[2] = {row_bytes / 4, static_cast<cuuint64_t>(t.N)};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxWords), static_cast<cuuint32_t>(rows)};
    const cuuint32_t estride[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(t.W), dims, strides, box,
              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over a tensor's activations viewed as uint64 [M][K / 4]; box =
// one chunk plus 16 bytes (162 / 130 elements for pn3t / pn4t) x M rows.  A
// box reaching past the end of x is zero-filled.
bool encode_x(CUtensorMap* map, const GemvTensor& t, int M) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const int per_blk = t.type == kPn3t ? 80 : 64;
    const cuuint64_t K = static_cast<cuuint64_t>(t.nb) * per_blk;
    const cuuint64_t dims[2] = {K / 4, static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {K * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>((t.type == kPn3t ? kXPitchPn3t : kXPitchPn4t) / 8),
                               static_cast<cuuint32_t>(M)};
    const cuuint32_t estride[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint16_t*>(t.x), dims, strides, box,
              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------ work split --

// Host model of the time one CTA spends on the units [u0, u1): it walks them
// in the kernel's batches (Walker) and charges every batch step step_cost
// and every unit its decode cost.  A step takes about as long with one tile
// at work as with several (the other warp pairs idle), so ranges whose tiles
// fill few batches finish early and ranges that add a short batch finish
// late; the split below balances this modelled time, not the unit count.
struct RangeModel {
    uint32_t base[kMaxLayer + 1];   // first unit of each tensor; base[count] = all
    uint32_t unit_cost[kMaxLayer];
    uint32_t step_cost;
    int tiles[kMaxLayer], chunks[kMaxLayer];
    int count;
    int lane_rows;                  // staged activation rows / M (chunk lanes allowed)

    void locate(uint32_t u, int& e, int& tile, int& c) const {
        e = 0;
        while (e + 1 < count && u >= base[e + 1]) ++e;
        const uint32_t rel = u - base[e];
        tile = static_cast<int>(rel / static_cast<uint32_t>(chunks[e]));
        c = static_cast<int>(rel - static_cast<uint32_t>(tile) * chunks[e]);
    }

    uint64_t cost(uint32_t u0, uint32_t u1) const {
        if (u1 <= u0) return 0;
        int e0, t0, c0, e1, t1, c1;
        locate(u0, e0, t0, c0);
        locate(u1 - 1, e1, t1, c1);
        uint64_t steps = 0;
        // windows of 8 tiles from the first tile, then from tile 0 of each
        // later tensor, as the kernel walks them (order does not matter here)
        for (int e = e0, tb = t0;;) {
            int nt = tiles[e] - tb < kBatchTiles ? tiles[e] - tb : kBatchTiles;
            const bool last = e == e1 && t1 - tb < kBatchTiles;
            if (last) nt = t1 - tb + 1;
            const int cs0 = (e == e0 && tb == t0) ? c0 : 0;
            const int ce = last ? c1 + 1 : chunks[e];
            int cap = kBatchTiles / nt;
            cap = cap < lane_rows ? cap : lane_rows;
            cap = cap < chunks[e] ? cap : chunks[e];
            const int lanes = cap >= 8 ? 8 : cap >= 4 ? 4 : cap >= 2 ? 2 : 1;
            const int span = nt == 1 ? ce - cs0 : chunks[e];
            steps += static_cast<uint64_t>((span + lanes - 1) / lanes);
            if (last) break;
            tb += kBatchTiles;
            if (tb >= tiles[e]) { ++e; tb = 0; }
        }
        uint64_t c = steps * step_cost;
        for (int e = e0; e <= e1; ++e) {
            const uint32_t a = u0 > base[e] ? u0 : base[e];
            const uint32_t b = u1 < base[e + 1] ? u1 : base[e + 1];
            c += static_cast<uint64_t>(b - a) * unit_cost[e];
        }
        return c;
    }

    // The largest v in [u + min_units, units] with cost(u, v) <= limit that
    // leaves no remainder shorter than min_units; 0 when there is none.
    uint32_t extent(uint32_t u, uint64_t limit, uint32_t min_units) const {
        const uint32_t units = base[count];
        uint32_t ok = u + min_units;
        if (ok > units || cost(u, ok) > limit) return 0;
        uint32_t bad = units + 1;                        // first v known to fail
        for (uint32_t step = min_units; ok < units;) {   // gallop, then bisect
            const uint32_t v = units - ok > step ? ok + step : units;
            if (cost(u, v) <= limit) { ok = v; step *= 2; }
            else { bad = v; break; }
        }
        while (bad - ok > 1) {
            const uint32_t v = ok + (bad - ok) / 2;
            if (cost(u, v) <= limit) ok = v;
            else bad = v;
        }
        if (ok < units && units - ok < min_units) {      // the rest must be a range too
            ok = units - min_units;
            if (ok < u + min_units) return 0;
        }
        return ok;
    }

    // Packs the units greedily into ranges of modelled cost <= limit; the
    // number of ranges, or 0 when more than max_ranges would be needed.
    int pack(uint64_t limit, int max_ranges, uint32_t min_units, uint32_t* starts) const {
        const uint32_t units = base[count];
        uint32_t u = 0;
        int n = 0;
        starts[0] = 0;
        while (u < units) {
            if (n == max_ranges) return 0;
            const uint32_t v = extent(u, limit, min_units);
            if (v == 0) return 0;
            starts[++n] = v;
            u = v;
        }
        return n;
    }
};

// A split of the units over the thread blocks, kept per call shape: the
// search below costs some hundred microseconds of host time, a lookup none.
struct SplitKey {
    int count, M, max_grid;
    int type[kMaxLayer], nb[kMaxLayer], N[kMaxLayer];
};
struct SplitEntry {
    SplitKey key;
    int grid;
    uint32_t starts[kMaxGrid + 1];
};
constexpr int kSplitCacheEntries = 16;

// Fills grid and starts: the cost-weighted split (CostSplit) unless the
// greedy packing of RangeModel, searched over its cost limit, gives a lower
// largest range cost.  Both keep every range at least min_units long, so a
// tile has at most two owners.
void balanced_split(const RangeModel& m, int max_grid, uint32_t min_units, int& grid, uint32_t* starts) {
    CostSplit even{};
    for (int e = 0; e < m.count; ++e) even.add(m.base[e + 1] - m.base[e], m.unit_cost[e]);
    grid = even.fit_grid(max_grid, min_units);
    uint64_t hi = 0;
    for (int c = 0; c <= grid; ++c) starts[c] = even.start(c);
    for (int c = 0; c < grid; ++c) {
        const uint64_t v = m.cost(starts[c], starts[c + 1]);
        hi = v > hi ? v : hi;
    }
    uint64_t lo = (even.cbase[even.count] + static_cast<uint64_t>(max_grid) - 1) / static_cast<uint64_t>(max_grid);
    static thread_local uint32_t trial[kMaxGrid + 1];
    while (lo < hi) {                                  // smallest limit that packs
        const uint64_t mid = lo + (hi - lo) / 2;
        const int n = m.pack(mid, max_grid, min_units, trial);
        if (n > 0) {
            hi = mid;
            grid = n;
            for (int c = 0; c <= n; ++c) starts[c] = trial[c];
        } else {
            lo = mid + 1;
        }
    }
}

void cached_split(const SplitKey& key, const RangeModel& m, uint32_t min_units, int& grid, uint32_t* starts) {
    static std::mutex mu;
    static SplitEntry cache[kSplitCacheEntries];
    static int filled = 0, next = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < filled; ++i)
            if (std::memcmp(&cache[i].key, &key, sizeof key) == 0) {
                grid = cache[i].grid;
                std::memcpy(starts, cache[i].starts, sizeof(uint32_t) * (grid + 1));
                return;
            }
    }
    balanced_split(m, key.max_grid, min_units, grid, starts);
    std::lock_guard<std::mutex> lock(mu);
    SplitEntry& slot = cache[next];
    next = (next + 1) % kSplitCacheEntries;
    filled = filled < kSplitCacheEntries ? filled + 1 : filled;
    slot.key = key;
    slot.grid = grid;
    std::memcpy(slot.starts, starts, sizeof(uint32_t) * (grid + 1));
}

}  // namespace

int tc_max_ctas(int num_sms) { return num_sms < kMaxGrid ? num_sms : kMaxGrid; }

size_t tc_partial_bytes(int num_sms) {
    return static_cast<size_t>(tc_max_ctas(num_sms) + 1) * 2 * kSlotFloats * sizeof(float);
}

bool tc_split(const GemvTensor* t, int count, int M, int num_sms, int* grid, uint32_t* starts) {
    const int nt = M > 8 ? 2 : 1;                  // 8-column tiles
    const SplitWeights& wt = kSplitWeights[nt - 1];
    RangeModel model{};
    SplitKey key{};                                // zero-filled: compared bytewise
    model.count = key.count = count;
    model.lane_rows = 8 * nt / M;                  // staged activation rows / M
    model.step_cost = wt.step;
    key.M = M;
    key.max_grid = tc_max_ctas(num_sms);
    uint64_t units = 0;
    int max_chunks = 1;
    for (int e = 0; e < count; ++e) {
        const int chunks = t[e].nb / kChunkBlocks;
        const int tiles = (t[e].N + kTileRows - 1) / kTileRows;
        if (chunks < 1 || tiles < 1) return false;
        model.base[e] = static_cast<uint32_t>(units);
        model.unit_cost[e] = t[e].type == kPn3t ? wt.pn3t : wt.pn4t;
        model.tiles[e] = tiles;
        model.chunks[e] = chunks;
        key.type[e] = t[e].type;
        key.nb[e] = t[e].nb;
        key.N[e] = t[e].N;
        units += static_cast<uint64_t>(chunks) * tiles;
        max_chunks = chunks > max_chunks ? chunks : max_chunks;
    }
    if (units >= (1ull << 32)) return false;      // 32-bit unit numbers
    model.base[count] = static_cast<uint32_t>(units);
    // every range spans at least one whole tile, so a tile has at most two owners
    cached_split(key, model, static_cast<uint32_t>(max_chunks), *grid, starts);
    return true;
}

cudaError_t launch_gemv_tc(const GemvTensor* t, int count, int M, uint32_t* status, float* partials,
                           uint32_t* counters, int num_sms, uint64_t timeout_ns, int stall, cudaStream_t s) {
    TcParams P{};
    uint64_t units = 0;
    for (int e = 0; e < count; ++e) {
        TcTensor& T = P.t[e];
        T.W = t[e].W; T.x = t[e].x; T.y = t[e].y;
        T.N = t[e].N; T.nb = t[e].nb; T.type = t[e].type;
        T.chunks = t[e].nb / kChunkBlocks;
        T.tiles = (t[e].N + kTileRows - 1) / kTileRows;
        T.unit_base = static_cast<uint32_t>(units);
        for (int k = 0; k < kBoxSizes; ++k)
            if (!encode_rows(&P.wmap[k][e], t[e], kTileRows << k)) return cudaErrorInvalidValue;
        if (!encode_x(&P.xmap[e], t[e], M)) return cudaErrorInvalidValue;
        units += static_cast<uint64_t>(T.chunks) * T.tiles;
    }
    P.count = count;
    P.M = M;
    const int nt = M > 8 ? 2 : 1;                  // 8-column tiles
    P.x_rows = 8 * nt;
    if (!tc_split(t, count, M, num_sms, &P.grid, P.starts)) return cudaErrorInvalidValue;
    P.status = status;
    P.counters = counters;
    P.partials = partials;
    P.timeout_ns = timeout_ns;
    P.stall_first_step = stall;

    static std::atomic<uint64_t> smem_set[2] = {{0}, {0}};
    const int smem_bytes = nt == 1 ? Smem<1>::kBytes : Smem<2>::kBytes;
    if (cudaError_t e = nt == 1 ? set_smem_limit_once(gemv_tc_kernel<1>, smem_bytes, smem_set[0])
                                : set_smem_limit_once(gemv_tc_kernel<2>, smem_bytes, smem_set[1]);
        e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(P.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return nt == 1 ? cudaLaunchKernelEx(&cfg, gemv_tc_kernel<1>, P) : cudaLaunchKernelEx(&cfg, gemv_tc_kernel<2>, P);
}

}  // namespace pn
