// pn_gemv_stream.cu -- PN decode GEMV for one or two tokens on GB300: every
// warp streams its own share of the weights through a private TMA ring and
// decodes straight into tensor-core fragments.
//
// What is computed: y[m][r] = sum_k d_blk(r,k) * (n(r,k) - z) * x[m][k], the
// decode GEMV of the tensorless docs ("Why a P100-native weight format": "One
// lane, one word", "Exact decode in fp32") and its skinny verification batch
// (v100-skinny README, "How QPN works"), with exact products and fp32 sums.
//
// Decode.  A code pair (one code in each 16-bit half of a word, at the same
// offset, "Codes never straddle the two halves of a word") becomes the exact
// half2 (n - z, n' - z) with one LOP3 and one HFMA2 (decode_pair), which is
// an A-fragment register of mma.sync m16n8k16 (fp16 in, fp32 accumulate).
// The zero point is taken off every code before the multiply, so a weight on
// the zero code ("Zero is a code, and the scale has a sign") contributes an
// exact 0 and carries no rounding error, whatever its activation.
//
// Fragment mapping.  An MMA covers 8 blocks (M = 1) or 4 blocks (M = 2): its
// eight k-pairs are shared out between those blocks and its eight columns are
// (token, block) pairs, B holding a token's activations only where the k-pair
// belongs to the column's block.  So every MMA has a full 16 x 16 A tile
// although M is 1 or 2, and a 16-row x 8-block unit always takes 40 (pn3t) or
// 32 (pn4t) MMAs.  Each column's sum is scaled by its own block scale d and
// the columns of one token are then added.
//
// Staging.  Each warp streams its units through a private two-stage ring:
// per unit, one 2-D TMA box of weights (16 rows x 272 bytes) and one bulk
// copy per token of the chunk's fp16 activations land in the same stage on
// one mbarrier, so both the codes and x are read from shared memory.
//
// Work split.  A unit is a 16-row tile x one 8-block chunk (272 bytes per
// row).  Units are numbered tile-major over every tensor of the call; the grid
// splits them into equal contiguous ranges (see kCostPn3t), each at least one
// tile long, and the eight warps of a block split the block's range again.  A warp's whole tiles
// are stored directly; the parts of a tile split between warps are added in
// warp order by the last warp to deliver (a shared-memory counter); for a tile
// cut by a block boundary both blocks swap their tagged part into a shared
// slot with a 64-bit atomic exchange and the block that gets the other's part
// back adds first chunks + later chunks.  Results do not depend on timing.
//
// Every wait is bounded in time; a warp that gives up records PN_ETIMEOUT in
// the workspace, lets its copies in flight land, and finishes.
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
// Two stages per warp (68 KB of shared memory per block instead of 101 KB
// with three) measured 3 to 5 % faster than three.  Not through a larger L1:
// forcing the largest shared-memory carve-out measured the same.
constexpr int kStages = 2;
constexpr int kRows = 16;                                 // weight rows per tile
constexpr int kChunkBlocks = 8;
constexpr int kChunkBytes = kChunkBlocks * kBlockBytes;   // 272
constexpr int kBoxWords = kChunkBytes / 4;                // 68
constexpr int kBoxBytes = kRows * kChunkBytes;            // 4352
// Relative cost of one unit, pn3t / pn4t, for the split of the units over
// the thread blocks.  This kernel's time follows its memory stream more than
// its decode: on a mixed pn3t / pn4t layer an even split of the bytes measured
// fastest (weighting pn3t units 1.07 to 1.25 times a pn4t unit was 3 to 7 %
// slower), so both weigh the same.  Re-measured with x staged in shared
// memory on the 27B-class layer: 9 / 8 within 0.4 % of even at one token,
// 5 / 4 and every pn4t-heavier weight slower (up to 10 %); at two tokens 8 / 9
// was 2 % faster but 5 % slower at one token.
constexpr uint32_t kCostPn3t = 1, kCostPn4t = 1;
constexpr int kMaxGrid = 512;                             // thread blocks per launch, at most
constexpr int kStreamMaxM = 2;                            // tokens this kernel serves
// A stage holds one unit's weight box and its activation chunk for each
// token (token m at kXOffset + m * kXTokenBytes; a pn3t chunk is 640 fp16,
// a pn4t chunk 512), all copied on the stage's mbarrier, so the decode reads
// x from shared memory like the weights.
constexpr int kXOffset = kBoxBytes;
constexpr int kXTokenBytes = kChunkBlocks * 80 * 2;       // 1280
constexpr int kStageBytes = kXOffset + kStreamMaxM * kXTokenBytes;   // 6912
constexpr int kRingBytes = kWarps * kStages * kStageBytes;
constexpr int kZeroOffset = kRingBytes;
constexpr int kZeroBytes = 256;                           // zeros read by lanes with an empty B fragment
constexpr int kPartOffset = kZeroOffset + kZeroBytes;
constexpr int kSlotFloats = 16 * kStreamMaxM;             // [row][token]
constexpr int kPartBytes = kWarps * 2 * kSlotFloats * 4;
constexpr int kCntOffset = kPartOffset + kPartBytes;
constexpr int kBarOffset = kCntOffset + kWarps * 4;
constexpr int kSmemBytes = kBarOffset + kWarps * kStages * 8;
constexpr uint64_t kDrainLimitNs = 200ull * 1000 * 1000;
constexpr uint32_t kStatusTimeout = 5;                    // PN_ETIMEOUT

static_assert(kBoxBytes <= kXOffset && kXOffset % 16 == 0 && kStageBytes % 128 == 0, "stages stay TMA-aligned");
static_assert(kSmemBytes <= 113 * 1024, "two thread blocks fit on one SM");
static_assert(kXOffset % 128 == 0, "activation chunks stay 16-byte aligned");
static_assert(kBarOffset % 8 == 0, "aligned barriers");

struct STensor {
    const uint16_t* x;
    float* y;
    uint32_t unit_base;     // first unit of this tensor
    int N;
    int K;
    int type;
    int chunks;             // nb / 8
    int tiles;              // ceil(N / 15)
};

struct SParams {
    CUtensorMap wmap[kMaxLayer];   // PN rows as uint32 [N][row_bytes / 4]; box 68 words x 15 rows
    STensor t[kMaxLayer];
    int count;
    int M;
    int grid;
    uint32_t starts[kMaxGrid + 1]; // block c's units are [starts[c], starts[c + 1])
    uint32_t* status;
    uint64_t* tagged;              // [boundary][kSlotFloats] {tag, value bits}
    uint64_t timeout_ns;
    int stall_first_step;          // testing aid: see pn_set_test_stall
};

// Position of a unit: tensor, tile, chunk.
struct Cursor {
    int e, tile, chunk;
    __device__ void locate(const SParams& P, uint32_t u) {
        e = 0;
        while (e + 1 < P.count && u >= P.t[e + 1].unit_base) ++e;
        const uint32_t rel = u - P.t[e].unit_base;
        const uint32_t ch = static_cast<uint32_t>(P.t[e].chunks);
        tile = static_cast<int>(rel / ch);
        chunk = static_cast<int>(rel - static_cast<uint32_t>(tile) * ch);
    }
};

__device__ __forceinline__ uint32_t range_start(const SParams& P, int c) {
    return P.starts[c];
}

__device__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Fast path: every lane probes once and the warp votes; if the phase has
// completed, each lane has observed it itself and the warp goes on at once.
// Otherwise lane 0 polls and __syncwarp orders the other lanes' reads of the
// stage after lane 0's observation of the completed phase.  Every lane of the
// warp must call it.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, int lane) {
    if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
    bool ok = true;
    if (lane == 0) ok = wait_bounded(bar, parity, limit_ns);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ float half_lo(uint32_t v) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t v) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
}

// D += A * B, m16n8k16, fp16 inputs, fp32 accumulate, accumulator in place.
__device__ __forceinline__ void mma_acc(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four accumulators per lane: consecutive MMAs of a unit go to different
// ones, so a chain of dependent MMAs is a quarter of the unit long.
struct Acc4 {
    float c[4][4];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int i = 0; i < 4; ++i) c[k][i] = 0.0f;
    }
    // (c0 + c1) + (c2 + c3): a fixed tree
    __device__ __forceinline__ float sum(int i) const { return (c[0][i] + c[1][i]) + (c[2][i] + c[3][i]); }
};

// NP consecutive code-pair activations (fp16 pairs) from the staged chunk
// at p (shared memory, 16-byte aligned; NP a multiple of 4).
template <int NP>
__device__ __forceinline__ void load_pairs(const uint8_t* p, uint32_t (&v)[NP]) {
    static_assert(NP % 4 == 0, "16-byte loads");
#pragma unroll
    for (int i = 0; i < NP / 4; ++i) {
        const uint4 q = *reinterpret_cast<const uint4*>(p + 16 * i);
        v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
    }
}

// Words [w0, w0 + NW) of block b of a staged row (row = 272 bytes), realigned
// with a per-lane selector: blocks at even positions start 2 bytes into an
// aligned word (sel 0x5432), odd ones are aligned (sel 0x3210).
template <int NW>
__device__ __forceinline__ void load_words_rt(const uint8_t* row, int b, int w0, uint32_t sel, uint32_t (&w)[NW]) {
    const uint8_t* base = row + ((kBlockBytes * b + 2 + 4 * w0) & ~3);
    uint32_t v[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) v[i] = lds_u32(base + 4 * i);
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = prmt(v[i], v[i + 1], sel);
}

__device__ __forceinline__ float lds_half(const uint8_t* p) { return __half2float(*reinterpret_cast<const __half*>(p)); }

// Per-unit context of a lane.
struct Lane {
    int g, t;
    const uint8_t* r0;     // staged row g
    const uint8_t* r1;     // staged row g + 8
    const uint8_t* x;      // staged activations of token 0 (token m at + m * kXTokenBytes)
    const uint8_t* zeros;  // kZeroBytes of zeros
};

// ---------------------------------------------------------------------------
// One unit (16 rows, 8 blocks), Mp = 8 / BPM tokens.  Adds the lane's scaled
// sums to acc: acc[h] = row g + 8h of token tok(t).
// ---------------------------------------------------------------------------

template <int TYPE>
__device__ __forceinline__ void unit_b8(const Lane& L, int M, float (&acc)[4]) {
    using F = Format<TYPE>;
    constexpr int kP = F::kPairs;
    const int g = L.g, t = L.t;
    (void)M;
    // k-pair t <-> odd block 2t+1, k-pair t+4 <-> even block 2t; step s of
    // the unit takes code pair s % kP of word s / kP of both blocks.  The
    // B columns are the blocks: lane g == 2t+1 carries block 2t+1's
    // activations in b0, lane g == 2t block 2t's in b1, every other B
    // register is zero.
    const uint8_t* xo = (g == 2 * t + 1) ? L.x + (2 * t + 1) * F::kPerBlock * 2 : L.zeros;
    const uint8_t* xe = (g == 2 * t) ? L.x + 2 * t * F::kPerBlock * 2 : L.zeros;
    // block 2t starts 4-byte aligned in a staged row: aligned word v[i] at
    // byte 4i holds (previous half, next half); its words are realigned with
    // one byte permute, and v[0] / v[8] also hold the two blocks' scales
    const uint8_t* e0 = L.r0 + 68 * t;
    const uint8_t* e1 = L.r1 + 68 * t;
    float d_e0, d_e1;
    uint32_t we0[8], we1[8], wo0[8], wo1[8];
    uint32_t v0, v1;
    {
        uint32_t a0[9], a1[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) {
            a0[i] = lds_u32(e0 + 4 * i);
            a1[i] = lds_u32(e1 + 4 * i);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            we0[i] = prmt(a0[i], a0[i + 1], 0x5432u);
            we1[i] = prmt(a1[i], a1[i + 1], 0x5432u);
            wo0[i] = lds_u32(e0 + 36 + 4 * i);
            wo1[i] = lds_u32(e1 + 36 + 4 * i);
        }
        d_e0 = half_lo(a0[0]);
        d_e1 = half_lo(a1[0]);
        v0 = a0[8];
        v1 = a1[8];
    }
    Acc4 A;
    A.zero();
    static_for<2 * kP>([&](auto qc) {
        constexpr int Q = decltype(qc)::value;          // four steps per 16-byte activation load
        uint32_t bo[4], be[4];
        load_pairs<4>(xo + 16 * Q, bo);
        load_pairs<4>(xe + 16 * Q, be);
        static_for<4>([&](auto jc) {
            constexpr int S = 4 * Q + decltype(jc)::value;
            constexpr int W = S / kP, Pp = S % kP;
            const uint32_t so0 = wo0[W] >> F::kHighShift, so1 = wo1[W] >> F::kHighShift;
            const uint32_t se0 = we0[W] >> F::kHighShift, se1 = we1[W] >> F::kHighShift;
            mma_acc(A.c[S & 3],
                    decode_pair<TYPE, Pp>(wo0[W], so0), decode_pair<TYPE, Pp>(wo1[W], so1),
                    decode_pair<TYPE, Pp>(we0[W], se0), decode_pair<TYPE, Pp>(we1[W], se1), bo[S % 4], be[S % 4]);
        });
    });
    const float d_o0 = half_hi(v0), d_o1 = half_hi(v1);        // v[8]: the odd block's scale
    // column 2t <-> block 2t (even), 2t+1 <-> block 2t+1 (odd)
    float r0 = d_e0 * A.sum(0);
    r0 = fmaf(d_o0, A.sum(1), r0);
    float r1 = d_e1 * A.sum(2);
    r1 = fmaf(d_o1, A.sum(3), r1);
    r0 += __shfl_xor_sync(0xFFFFFFFFu, r0, 1);
    r1 += __shfl_xor_sync(0xFFFFFFFFu, r1, 1);
    r0 += __shfl_xor_sync(0xFFFFFFFFu, r0, 2);
    r1 += __shfl_xor_sync(0xFFFFFFFFu, r1, 2);
    acc[0] += r0;
    acc[1] += r1;
}

template <int TYPE>
__device__ __forceinline__ void unit_b4(const Lane& L, int M, float (&acc)[4]) {
    using F = Format<TYPE>;
    constexpr int kP = F::kPairs;
    constexpr int kSteps = 4 * kP;                 // per group of 4 blocks
    const int g = L.g, t = L.t;
    const uint32_t sel = (t & 1) ? 0x3210u : 0x5432u;
    // column c <-> token c >> 2, block c & 3 of the group; lane t decodes block t
    const bool has_b = (g & 3) == t && (g >> 2) < M;
    const uint8_t* xt = L.x + (g >> 2) * kXTokenBytes;
    static_for<2>([&](auto gc) {
        constexpr int G = decltype(gc)::value;
        const int blk = 4 * G + t;
        uint32_t w[2][8];
        load_words_rt<8>(L.r0, blk, 0, sel, w[0]);
        load_words_rt<8>(L.r1, blk, 0, sel, w[1]);
        const uint8_t* xb = has_b ? xt + blk * F::kPerBlock * 2 : L.zeros;
        uint32_t b0[kSteps], b1[kSteps];
        load_pairs<kSteps>(xb, b0);                                      // words 0..3
        load_pairs<kSteps>(has_b ? xb + 4 * kSteps : L.zeros, b1);       // words 4..7
        Acc4 A;
        A.zero();
        static_for<kSteps>([&](auto sc) {
            constexpr int S = decltype(sc)::value;
            constexpr int W = S / kP, P = S % kP;
            const uint32_t s00 = w[0][W] >> F::kHighShift, s10 = w[1][W] >> F::kHighShift;
            const uint32_t s01 = w[0][W + 4] >> F::kHighShift, s11 = w[1][W + 4] >> F::kHighShift;
            mma_acc(A.c[S & 3],
                    decode_pair<TYPE, P>(w[0][W], s00), decode_pair<TYPE, P>(w[1][W], s10),
                    decode_pair<TYPE, P>(w[0][W + 4], s01), decode_pair<TYPE, P>(w[1][W + 4], s11),
                    b0[S], b1[S]);
        });
        // lane columns 2t, 2t+1 <-> token t >> 1, blocks 4G + 2(t & 1) + {0, 1}
        const int bb = 4 * G + 2 * (t & 1);
        float v[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint8_t* r = h ? L.r1 : L.r0;
            const float d0 = lds_half(r + kBlockBytes * bb), d1 = lds_half(r + kBlockBytes * (bb + 1));
            v[h] = fmaf(d1, A.sum(2 * h + 1), d0 * A.sum(2 * h));
            v[h] += __shfl_xor_sync(0xFFFFFFFFu, v[h], 1);
            acc[h] += v[h];
        }
    });
}

template <int BPM, int TYPE>
__device__ __forceinline__ void unit(const Lane& L, int M, float (&acc)[4]) {
    if constexpr (BPM == 8) unit_b8<TYPE>(L, M, acc);
    else unit_b4<TYPE>(L, M, acc);
}

// ------------------------------------------------------------ tile results --

// The (row, token) a lane's acc[i] holds, and whether this lane is the one
// that stores / deposits it (several lanes hold the same sum for BPM 8 and 4).
template <int BPM>
__device__ __forceinline__ bool acc_slot(int g, int t, int i, int& row, int& tok) {
    row = g + 8 * i;
    if constexpr (BPM == 8) { tok = 0; return i < 2 && t == 0 && row < kRows; }
    else { tok = t >> 1; return i < 2 && (t & 1) == 0 && row < kRows; }
}

// Entries of acc a lane uses: rows g and g + 8.
template <int BPM>
__host__ __device__ constexpr int acc_entries() { return 2; }

// Index in a [row][token] slot of the lane's acc[i].
template <int BPM>
__device__ __forceinline__ int acc_index(int g, int t, int i) {
    int row, tok;
    acc_slot<BPM>(g, t, i, row, tok);
    return row * kStreamMaxM + tok;
}

template <int BPM>
__device__ __forceinline__ void store_tile(const SParams& P, const Cursor& c, int lane, const float (&acc)[4]) {
    const STensor& T = P.t[c.e];
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int row, tok;
        if (!acc_slot<BPM>(g, t, i, row, tok)) continue;
        const int r = c.tile * kRows + row;
        if (r < T.N && tok < P.M) T.y[static_cast<int64_t>(tok) * T.N + r] = acc[i];
    }
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

// Number of warps of the block with a non-empty share in [wa, wb].
__device__ __forceinline__ uint32_t contributors(uint32_t n, int wa, int wb) {
    uint32_t k = 0;
    for (int w = wa; w <= wb; ++w) k += (n * (w + 1) / kWarps > n * w / kWarps) ? 1u : 0u;
    return k;
}

// The warp whose share [n w / 8, n (w + 1) / 8) holds block-relative unit pos.
__device__ __forceinline__ int warp_of(uint32_t pos, uint32_t n) {
    int w = static_cast<int>(pos * kWarps / n);
    while (w > 0 && n * w / kWarps > pos) --w;
    while (w < kWarps - 1 && n * (w + 1) / kWarps <= pos) ++w;
    return w;
}

// Hands this warp's part of a tile split between warps wa..wb to shared
// memory; the last warp to deliver gets true and the sum in warp order.
template <int BPM>
__device__ bool hand_in(uint8_t* smem, int warp, int lane, int wa, int wb, uint32_t n, float (&acc)[4]) {
    float* parts = reinterpret_cast<float*>(smem + kPartOffset);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + kCntOffset);
    const int g = lane >> 2, t = lane & 3;
    float* mine = parts + (warp * 2 + (warp == wa ? 1 : 0)) * kSlotFloats;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int row, tok;
        if (acc_slot<BPM>(g, t, i, row, tok)) mine[row * kStreamMaxM + tok] = acc[i];
    }
    __threadfence_block();
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0) old = atomicAdd(cnt + wa, 1u);
    old = __shfl_sync(0xFFFFFFFFu, old, 0);
    if (old + 1 != contributors(n, wa, wb)) return false;
    __threadfence_block();
#pragma unroll
    for (int i = 0; i < acc_entries<BPM>(); ++i) {
        const int idx = acc_index<BPM>(g, t, i);
        float s = parts[(wa * 2 + 1) * kSlotFloats + idx];
        for (int w = wa + 1; w <= wb; ++w)
            if (n * (w + 1) / kWarps > n * w / kWarps) s += parts[(w * 2) * kSlotFloats + idx];
        acc[i] = s;
    }
    return true;
}

__device__ __forceinline__ uint64_t atom_exch_u64(uint64_t* p, uint64_t v) {
    return atomicExch(reinterpret_cast<unsigned long long*>(p), static_cast<unsigned long long>(v));
}

// A tile cut by a thread-block boundary has two parts, the first chunks
// (held by the block before the boundary) and the rest (held by the block
// after it).  Each side swaps its part, tagged with which part it is, into
// the boundary's slot with one 64-bit atomic exchange per output; exactly one
// side gets the other's part back, adds first + second in that order, stores
// the output and clears the slot.  Neither side waits for the other.
constexpr uint32_t kTagFirst = 1u, kTagSecond = 2u;

template <int BPM>
__device__ __forceinline__ void exchange(const SParams& P, const Cursor& c, int lane, bool first, int boundary,
                                         const float (&acc)[4]) {
    const int g = lane >> 2, t = lane & 3;
    uint64_t* slot = P.tagged + static_cast<int64_t>(boundary) * kSlotFloats;
    const uint64_t tag = static_cast<uint64_t>(first ? kTagFirst : kTagSecond) << 32;
    const STensor& T = P.t[c.e];
#pragma unroll
    for (int i = 0; i < acc_entries<BPM>(); ++i) {
        int row, tok;
        if (!(acc_slot<BPM>(g, t, i, row, tok) && tok < P.M)) continue;
        uint64_t* w = slot + acc_index<BPM>(g, t, i);
        const uint64_t got = atom_exch_u64(w, tag | __float_as_uint(acc[i]));
        if ((got >> 32) == 0) continue;                       // the other side finishes this output
        const float other = __uint_as_float(static_cast<uint32_t>(got));
        const float v = first ? acc[i] + other : other + acc[i];     // first chunks + later chunks
        const int r = c.tile * kRows + row;
        if (r < T.N) T.y[static_cast<int64_t>(tok) * T.N + r] = v;
        st_relaxed_u64(w, 0ull);
    }
}

// Issue cursor: the next unit to copy, following the block's processing
// order (see run_warp); the tensor's sizes are kept in registers.
struct Issuer {
    uint32_t q;            // sequence position
    Cursor c;
    int chunks, tiles;
    __device__ void set(const SParams& P, uint32_t u) {
        c.locate(P, u);
        chunks = P.t[c.e].chunks;
        tiles = P.t[c.e].tiles;
    }
    __device__ void advance(const SParams& P, uint32_t nr, uint32_t c0) {
        if (++q == nr) { set(P, c0); return; }
        if (++c.chunk == chunks) {
            c.chunk = 0;
            if (++c.tile == tiles) {
                c.tile = 0;
                ++c.e;
                if (c.e < P.count) { chunks = P.t[c.e].chunks; tiles = P.t[c.e].tiles; }
            }
        }
    }
};

// Ring position of a warp.
struct Ring {
    int s = 0;
    uint32_t phase = 0;
    uint32_t done = 0, issued = 0;
};

// Lane 0: the copies of unit c into stage `dst` (shared address), completing
// on `bar`: the weight box and the chunk's activations of every token.  With
// `copy` false the bytes are announced but nothing is copied (testing aid).
__device__ __forceinline__ void issue_unit(const SParams& P, uint32_t dst, uint32_t bar, const Cursor& c, bool copy) {
    const STensor& T = P.t[c.e];
    const int halves = kChunkBlocks * per_block(T.type);
    mbar_arrive_expect_tx(bar, kBoxBytes + P.M * halves * 2);
    if (!copy) return;
    tma_load_2d(dst, &P.wmap[c.e], c.chunk * kBoxWords, c.tile * kRows, bar);
    const uint16_t* x = T.x + static_cast<int64_t>(c.chunk) * halves;
    for (int m = 0; m < P.M; ++m)
        bulk_g2s(dst + kXOffset + m * kXTokenBytes, x + static_cast<int64_t>(m) * T.K, halves * 2, bar);
}

template <int BPM, int TYPE>
__device__ bool part_loop(const SParams& P, uint8_t* smem, int warp, int lane, Lane& L,
                          uint32_t len, uint32_t total, uint32_t nr, uint32_t c0, Ring& R, Issuer& I,
                          float (&acc)[4]) {
    const uint32_t ring = smem_addr(smem) + warp * kStages * kStageBytes;
    const uint8_t* ring_p = smem + warp * kStages * kStageBytes;
    const uint32_t bar0 = smem_addr(smem + kBarOffset) + warp * kStages * 8;
    for (uint32_t k = 0; k < len; ++k) {
        if (!warp_wait(bar0 + 8 * R.s, R.phase, P.timeout_ns, lane)) {
            if (lane == 0) atomicCAS(P.status, 0u, kStatusTimeout);
            return false;
        }
        const uint8_t* stage = ring_p + R.s * kStageBytes;
        L.r0 = stage + L.g * kChunkBytes;
        L.r1 = stage + (L.g + 8) * kChunkBytes;
        L.x = stage + kXOffset;
        unit<BPM, TYPE>(L, P.M, acc);
        __syncwarp();
        ++R.done;
        if (R.issued < total) {                   // refill this stage
            if (lane == 0) {
                fence_proxy_async_smem();
                issue_unit(P, ring + R.s * kStageBytes, bar0 + 8 * R.s, I.c, true);
            }
            I.advance(P, nr, c0);
            ++R.issued;
        }
        if (++R.s == kStages) { R.s = 0; R.phase ^= 1u; }
    }
    return true;
}

// A block's units are processed in this order: first its part of the tile
// that continues into the next block (nr units, the last of its range), then
// the rest of its range in order.  Its part of the tile begun by the previous
// block comes right after, so both tiles that cross a block boundary are
// exchanged early, away from the kernel's tail.  The eight warps split this
// sequence into equal contiguous shares.
template <int BPM>
__device__ void run_warp(const SParams& P, uint8_t* smem, int warp, int lane, uint32_t c0, uint32_t c1) {
    const uint32_t n = c1 - c0;
    Cursor lastc{0, 0, 0};
    lastc.locate(P, c1 - 1);
    const uint32_t nr = lastc.chunk != P.t[lastc.e].chunks - 1 ? static_cast<uint32_t>(lastc.chunk + 1) : 0u;
    const uint32_t p0 = n * static_cast<uint32_t>(warp) / kWarps;
    const uint32_t p1 = n * static_cast<uint32_t>(warp + 1) / kWarps;
    auto seq_unit = [&](uint32_t q) { return q < nr ? c1 - nr + q : c0 + (q - nr); };
    const uint32_t total = p1 - p0;
    const uint32_t bar0 = smem_addr(smem + kBarOffset) + warp * kStages * 8;
    const uint32_t ring = smem_addr(smem) + warp * kStages * kStageBytes;

    Issuer I;
    I.q = p0;
    if (total > 0) I.set(P, seq_unit(p0));
    if (lane == 0 && total > 0) {
        // warm L2 with this warp's first units while the previous kernel finishes
        Issuer J = I;
        for (uint32_t k = 0; k < kStages && k < total; ++k) {
            tma_prefetch_l2_2d(&P.wmap[J.c.e], J.c.chunk * kBoxWords, J.c.tile * kRows);
            J.advance(P, nr, c0);
        }
    }
    griddep_wait();
    __syncwarp();
    if (total == 0) return;

    Ring R;
    for (int s = 0; s < kStages && R.issued < total; ++s) {
        // (testing aid: with stall_first_step a warp's first unit is
        // announced but never copied, so its wait can only time out)
        if (lane == 0) issue_unit(P, ring + s * kStageBytes, bar0 + 8 * s, I.c, !(s == 0 && P.stall_first_step));
        I.advance(P, nr, c0);
        ++R.issued;
    }

    Lane L;
    L.g = lane >> 2;
    L.t = lane & 3;
    L.zeros = smem + kZeroOffset;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    uint32_t q = p0;
    Cursor cur{0, 0, 0};
    cur.locate(P, seq_unit(q));
    bool ok = true;
    while (q < p1) {
        const STensor& T = P.t[cur.e];
        const uint32_t run_end = q < nr ? (nr < p1 ? nr : p1) : p1;
        const uint32_t room = static_cast<uint32_t>(T.chunks - cur.chunk);
        const uint32_t len = run_end - q < room ? run_end - q : room;
        ok = T.type == kPn3t ? part_loop<BPM, kPn3t>(P, smem, warp, lane, L, len, total, nr, c0, R, I, acc)
                             : part_loop<BPM, kPn4t>(P, smem, warp, lane, L, len, total, nr, c0, R, I, acc);
        if (!ok) break;
        // this warp's part of tile cur.tile ends here
        const uint32_t tbeg = T.unit_base + static_cast<uint32_t>(cur.tile) * T.chunks;
        const uint32_t tend = tbeg + T.chunks;
        const bool right_cut = tend > c1, left_cut = tbeg < c0;
        const uint32_t ss = right_cut ? 0u : nr + (left_cut ? 0u : tbeg - c0);   // the tile's sequence range
        const uint32_t se = right_cut ? nr : nr + (tend - c0);
        const int wa = warp_of(ss, n), wb = warp_of(se - 1, n);
        if (wa == wb || hand_in<BPM>(smem, warp, lane, wa, wb, n, acc)) {
            if (right_cut || left_cut) {
                exchange<BPM>(P, cur, lane, right_cut, right_cut ? blockIdx.x + 1 : blockIdx.x, acc);
            } else {
                store_tile<BPM>(P, cur, lane, acc);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = 0.0f;
        q += len;
        if (q == nr && q < p1) {
            cur.locate(P, c0);
        } else {
            cur.chunk += static_cast<int>(len);
            if (cur.chunk == T.chunks) {
                cur.chunk = 0;
                if (++cur.tile == T.tiles) { cur.tile = 0; ++cur.e; }
            }
        }
    }
    if (!ok) {
        if (lane == 0) {
            // after a timeout: let every copy this warp started land before the block can exit
            for (uint32_t k = R.done; k < R.issued; ++k) {
                if (k == 0 && P.stall_first_step) continue;   // never copied
                wait_bounded(bar0 + 8 * (k % kStages), (k / kStages) & 1u, kDrainLimitNs);
            }
        }
        __syncwarp();
        return;
    }
}

template <int BPM>
__global__ void __launch_bounds__(kThreads, 2) gemv_stream_kernel(const __grid_constant__ SParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t c0 = range_start(P, blockIdx.x), c1 = range_start(P, blockIdx.x + 1);
    for (int i = threadIdx.x; i < kZeroBytes / 4; i += kThreads) reinterpret_cast<uint32_t*>(smem + kZeroOffset)[i] = 0u;
    if (lane == 0) {
        const uint32_t bar0 = smem_addr(smem + kBarOffset) + warp * kStages * 8;
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
        reinterpret_cast<uint32_t*>(smem + kCntOffset)[warp] = 0u;
    }
    __syncthreads();
    run_warp<BPM>(P, smem, warp, lane, c0, c1);
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
// box = one 8-block chunk (68 words) x 15 rows; rows past N read as zero.
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

template <int BPM>
cudaError_t launch_bpm(const SParams& P, cudaStream_t s) {
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = set_smem_limit_once(gemv_stream_kernel<BPM>, kSmemBytes, smem_set); e != cudaSuccess)
        return e;
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
    return cudaLaunchKernelEx(&cfg, gemv_stream_kernel<BPM>, P);
}

}  // namespace

int stream_max_ctas(int num_sms) { return 2 * num_sms < kMaxGrid ? 2 * num_sms : kMaxGrid; }

size_t stream_tagged_bytes(int num_sms) {
    return static_cast<size_t>(stream_max_ctas(num_sms) + 1) * kSlotFloats * sizeof(uint64_t);
}

cudaError_t launch_gemv_stream(const GemvTensor* t, int count, int M, uint32_t* status, uint64_t* tagged,
                               int num_sms, uint64_t timeout_ns, int stall, cudaStream_t s) {
    if (M < 1 || M > kStreamMaxM || count < 1 || count > kMaxLayer) return cudaErrorInvalidValue;
    SParams P{};
    uint64_t units = 0;
    int max_chunks = 1;
    for (int e = 0; e < count; ++e) {
        STensor& T = P.t[e];
        T.x = t[e].x;
        T.y = t[e].y;
        T.N = t[e].N;
        T.type = t[e].type;
        T.K = t[e].nb * per_block(t[e].type);
        T.chunks = t[e].nb / kChunkBlocks;
        T.tiles = (t[e].N + kRows - 1) / kRows;
        T.unit_base = static_cast<uint32_t>(units);
        if (!encode_rows(&P.wmap[e], t[e])) return cudaErrorInvalidValue;
        units += static_cast<uint64_t>(T.chunks) * T.tiles;
        max_chunks = T.chunks > max_chunks ? T.chunks : max_chunks;
    }
    P.count = count;
    P.M = M;
    if (units * kWarps >= (1ull << 32)) return cudaErrorInvalidValue;   // 32-bit unit arithmetic
    CostSplit split{};
    for (int e = 0; e < count; ++e)
        split.add(static_cast<uint32_t>(P.t[e].chunks) * P.t[e].tiles, P.t[e].type == kPn3t ? kCostPn3t : kCostPn4t);
    // every block range spans at least one whole tile, so a tile has at most two blocks
    P.grid = split.fit_grid(stream_max_ctas(num_sms), static_cast<uint32_t>(max_chunks));
    for (int c = 0; c <= P.grid; ++c) P.starts[c] = split.start(c);
    P.status = status;
    P.tagged = tagged;
    P.timeout_ns = timeout_ns;
    P.stall_first_step = stall;
    return M == 1 ? launch_bpm<8>(P, s) : launch_bpm<4>(P, s);
}

}  // namespace pn
