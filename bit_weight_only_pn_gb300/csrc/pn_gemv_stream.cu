// pn_gemv_stream.cu -- PN decode GEMV for one or two tokens on GB300: one
// thread block per SM streams its share of the weights through a deep TMA
// ring while fifteen warps decode it straight into tensor-core fragments.
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
// Work.  A unit is a 16-row tile x one 8-block chunk (272 bytes per row),
// numbered tile-major over every tensor of the call; each thread block (one
// per SM) takes one contiguous range of units, split on the host so that
// every range holds the same bytes and at least one whole tile.  In the block,
// lanes of a producer warp each copy one unit into the next stage of a ring
// (one 2-D TMA box of weights, 16 rows x 272 bytes, and one bulk copy per
// token of the chunk's fp16 activations, on the stage's mbarrier), and each of
// the fifteen consumer warps takes the next stage by ticket, decodes it and
// frees it, so the block's warps share its units as they become free.
//
// Activations.  Staged: each stage carries its unit's activations, as above.
// Resident (layers and two-token calls, where it fits beside the ring): the
// producer copies, once per block, the whole activation vectors of the
// tensors the block's range touches into shared memory, and the stages carry
// weights only.  Rotated (the fused runtime Hadamard rotation of the
// tensorless docs, "How Qwen3.8-27B-PN3 uses it"): the producer copies them
// in the same way, the consumer warps rotate them in place with
// pn_hadamard's arithmetic, then decode as in the resident case.
//
// Combining.  A unit's partial sums (16 rows x M tokens) go to a slot of a
// shared-memory ring; a counter per tile counts the units done, and the warp
// that finishes a tile's last unit adds the tile's partials in chunk order.
// A tile cut by a range boundary (at most the first and the last tile of a
// range) is settled between the two blocks without waiting: each swaps its
// tagged part into the boundary's slot with one 64-bit atomic exchange per
// output, and the side that gets the other's part back adds first chunks +
// later chunks and stores.  A block copies its last, cut tile first, so both
// exchanges happen early.  Results never depend on timing.
//
// Every wait is bounded in time; a warp that gives up records PN_ETIMEOUT in
// the workspace, and the thread block lets its copies in flight land and
// finishes.
#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pn_device.cuh"
#include "pn_internal.h"

namespace pn {
namespace {

constexpr int kConsumers = 15;                            // decoding warps
constexpr int kProducerWarp = kConsumers;
constexpr int kThreads = (kConsumers + 1) * 32;           // 512
constexpr int kIssueLanes = 16;                           // producer lanes issuing copies at once
constexpr int kResidentLead = 4;                          // stages requested before resident activations
constexpr int kRows = 16;                                 // weight rows per tile
constexpr int kChunkBlocks = 8;
constexpr int kChunkBytes = kChunkBlocks * kBlockBytes;   // 272
constexpr int kBoxWords = kChunkBytes / 4;                // 68
constexpr int kBoxBytes = kRows * kChunkBytes;            // 4352
constexpr int kStreamMaxM = 2;                            // tokens this kernel serves
constexpr int kXTokenBytes = kChunkBlocks * 80 * 2;       // 1280: a pn3t chunk of activations (pn4t: 1024)
constexpr int kStagesLog2 = 5;
constexpr int kStages = 1 << kStagesLog2;                 // ring stages (a power of two), at most
constexpr int kMinStagesLog2 = 4;                         // the ring's smallest size (> kConsumers)
constexpr int kPartsLog2 = 6;
constexpr int kParts = 1 << kPartsLog2;                   // partial-sum slots in shared memory
constexpr int kSlotFloats = kRows * kStreamMaxM;          // [row][token]
constexpr int kZeroBytes = 512;                           // zeros read by lanes with an empty B fragment
constexpr int kMaxGrid = 512;                             // thread blocks per launch, at most
constexpr uint64_t kDrainLimitNs = 200ull * 1000 * 1000;
constexpr uint32_t kStatusTimeout = 5;                    // PN_ETIMEOUT
constexpr uint32_t kEnd = 0xFFFFFFFFu;                    // tile field of a stage that ends a consumer
constexpr uint32_t kSuspendNs = 1000;                     // suspend hint of a barrier wait
static_assert((1 << kMinStagesLog2) > kConsumers, "a consumer never waits on a stage two phases ahead");
static_assert((1 << kMinStagesLog2) >= kIssueLanes, "one producer round fits the ring");

__host__ __device__ constexpr int stage_bytes(int M) { return (kBoxBytes + M * kXTokenBytes + 127) / 128 * 128; }

// Shared memory: the ring of S stages, one 16-byte unit record per stage, the
// full and empty barriers, the partial-sum slots with their generation words
// and tile counters, then either each consumer's copy of a one-token unit's
// activations (activations staged with the weights) or the activations the
// block keeps resident (resident_bytes > 0: then the stages hold weights
// only), the ticket counter, the abort flag, the resident offsets, the
// resident copy's barrier and zeros.
struct SmemLayout {
    int sbytes = 0, table = 0, full = 0, empty = 0, parts = 0, gens = 0, cnts = 0, xown = 0, resident = 0,
        misc = 0, xbar = 0, zeros = 0, total = 0;
    __host__ __device__ constexpr SmemLayout(int M, int S, uint32_t resident_bytes) {
        sbytes = resident_bytes ? kBoxBytes : stage_bytes(M);
        table = S * sbytes;
        full = table + 16 * S;
        empty = full + 8 * S;
        parts = empty + 8 * S;
        gens = parts + kParts * kSlotFloats * 4;
        cnts = gens + 4 * kParts;
        xown = cnts + 4 * kParts;
        resident = xown + (!resident_bytes && M == 1 ? kConsumers * kXTokenBytes : 0);
        misc = resident + static_cast<int>((resident_bytes + 15) / 16 * 16);   // ticket (4), abort (4), offsets (32)
        xbar = misc + 40;
        zeros = (xbar + 8 + 15) / 16 * 16;
        total = zeros + kZeroBytes;
    }
};
constexpr int kSmemLimit = 227 * 1024;

struct STensor {
    const uint16_t* x;
    float* y;
    uint32_t unit_base;     // first unit of this tensor
    int N;
    int K;
    int type;
    int chunks;             // nb / 8
    int tiles;              // ceil(N / 16)
};

struct SParams {
    CUtensorMap wmap[kMaxLayer];   // PN rows as uint32 [N][row_bytes / 4]; box 68 words x 16 rows
    STensor t[kMaxLayer];
    int count;
    int M;
    int grid;
    uint32_t starts[kMaxGrid + 1]; // block c's units are [starts[c], starts[c + 1])
    uint32_t* status;
    uint64_t* tagged;              // [boundary][kSlotFloats] {tag, value bits}
    uint64_t timeout_ns;
    int stall_first_step;          // testing aid: see pn_set_test_stall
    int stages_log2;               // the ring holds 1 << stages_log2 stages
    // rotation of the activations (0 = none): every run of rot_block
    // activations times H / sqrt(rot_block)
    int rot_block;
    float rot_scale;
    // > 0: every block keeps the activations of the tensors its range
    // touches in shared memory (rotated if rot_block), this many bytes at
    // most; 0: each stage carries its unit's activations with its weights
    uint32_t resident_bytes;
};

// Tensor, tile and chunk of unit u.
__device__ __forceinline__ void locate(const SParams& P, uint32_t u, int& e, int& tile, int& chunk) {
    e = 0;
    while (e + 1 < P.count && u >= P.t[e + 1].unit_base) ++e;
    const uint32_t rel = u - P.t[e].unit_base;
    const uint32_t ch = static_cast<uint32_t>(P.t[e].chunks);
    tile = static_cast<int>(rel / ch);
    chunk = static_cast<int>(rel - static_cast<uint32_t>(tile) * ch);
}

// Bounded wait on phase `parity` of an mbarrier by a whole warp (every lane
// calls it): each lane waits itself (suspending between probes), so its later
// reads of the stage are ordered after its own observation of the phase.
// Gives up after limit_ns or once the block has aborted.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          const volatile uint32_t* abort_flag) {
    if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (__all_sync(0xFFFFFFFFu, mbar_wait_suspend(bar, parity, kSuspendNs))) return true;
        if (*abort_flag || globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Single-thread bounded wait.
__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                            const volatile uint32_t* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_wait_suspend(bar, parity, kSuspendNs)) return true;
        if ((abort_flag && *abort_flag) || globaltimer_ns() - t0 > limit_ns) return false;
    }
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

__device__ __forceinline__ int lane_id() { return static_cast<int>(threadIdx.x & 31); }

// bar.sync on a named barrier among `threads` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float lds_half(const uint8_t* p) { return __half2float(*reinterpret_cast<const __half*>(p)); }

// Per-unit context of a lane.
struct Lane {
    int g, t;
    const uint8_t* r0;     // staged row g
    const uint8_t* r1;     // staged row g + 8
    const uint8_t* x;      // the chunk's activations of token 0 (token m at + m * xstride)
    int xstride;           // bytes between tokens' activations
    bool resident;         // x is in the block's resident activations (never overwritten)
    uint8_t* xown;         // this warp's own copy of one token's activations (one-token units)
    const uint8_t* zeros;  // kZeroBytes of zeros
};

// ---------------------------------------------------------------------------
// One unit (16 rows, 8 blocks), Mp = 8 / BPM tokens.  Adds the lane's scaled
// sums to acc: acc[h] = row g + 8h of token tok(t).
// ---------------------------------------------------------------------------

template <int TYPE, typename Release>
__device__ __forceinline__ void unit_b8(const Lane& L, int M, float (&acc)[4], Release&& release) {
    using F = Format<TYPE>;
    constexpr int kP = F::kPairs;
    const int g = L.g, t = L.t;
    (void)M;
    // k-pair t <-> odd block 2t+1, k-pair t+4 <-> even block 2t; step s of
    // the unit takes code pair s % kP of word s / kP of both blocks.  The
    // B columns are the blocks: lane g == 2t+1 carries block 2t+1's
    // activations in b0, lane g == 2t block 2t's in b1, every other B
    // register is zero.
    // block 2t starts 4-byte aligned in a staged row: aligned word i at byte
    // 4i holds (previous half, next half), so code word i is one byte permute
    // of aligned words i and i+1; word 0 also holds the even block's scale,
    // word 8 the odd block's.  The unit's code words (rows g and g+8 of blocks
    // 2t and 2t+1) go to registers and its activations to this warp's own
    // copy in shared memory first; then the stage is released, so the
    // producer can refill it while the MMAs run.
    const uint8_t* e0 = L.r0 + 68 * t;
    const uint8_t* e1 = L.r1 + 68 * t;
    uint32_t we0[8], we1[8], wo0[8], wo1[8];
    float d_e0, d_e1, d_o0, d_o1;
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
        d_o0 = half_hi(a0[8]);
        d_o1 = half_hi(a1[8]);
        // the chunk's activations (kXTokenBytes at most) to the private copy,
        // unless they sit in the block's resident rotated copy
        constexpr int kVec = kChunkBlocks * F::kPerBlock * 2 / 16;
        if (!L.resident) {
#pragma unroll
            for (int i = 0; i < (kVec + 31) / 32; ++i) {
                const int j = lane_id() + 32 * i;
                if (j < kVec) *reinterpret_cast<uint4*>(L.xown + 16 * j) = lds_u128(L.x + 16 * j);
            }
        }
    }
    release();                                          // (orders this warp's copy before its reads too)
    const uint8_t* xs = L.resident ? L.x : L.xown;
    const uint8_t* xo = (g == 2 * t + 1) ? xs + (2 * t + 1) * F::kPerBlock * 2 : L.zeros;
    const uint8_t* xe = (g == 2 * t) ? xs + 2 * t * F::kPerBlock * 2 : L.zeros;
    float c[2][4];
#pragma unroll
    for (int k = 0; k < 2; ++k) c[k][0] = c[k][1] = c[k][2] = c[k][3] = 0.0f;
    uint32_t bo[4], be[4];
    static_for<8>([&](auto wc) {
        constexpr int W = decltype(wc)::value;
        const uint32_t so0 = wo0[W] >> F::kHighShift, so1 = wo1[W] >> F::kHighShift;
        const uint32_t se0 = we0[W] >> F::kHighShift, se1 = we1[W] >> F::kHighShift;
        static_for<kP>([&](auto pc) {
            constexpr int Pp = decltype(pc)::value;
            constexpr int S = W * kP + Pp;
            if constexpr (S % 4 == 0) {                 // four steps per 16-byte activation load
                load_pairs<4>(xo + 4 * S, bo);
                load_pairs<4>(xe + 4 * S, be);
            }
            mma_acc(c[S & 1],
                    decode_pair<TYPE, Pp>(wo0[W], so0), decode_pair<TYPE, Pp>(wo1[W], so1),
                    decode_pair<TYPE, Pp>(we0[W], se0), decode_pair<TYPE, Pp>(we1[W], se1), bo[S % 4], be[S % 4]);
        });
    });
    // column 2t <-> block 2t (even), 2t+1 <-> block 2t+1 (odd)
    float r0 = d_e0 * (c[0][0] + c[1][0]);
    r0 = fmaf(d_o0, c[0][1] + c[1][1], r0);
    float r1 = d_e1 * (c[0][2] + c[1][2]);
    r1 = fmaf(d_o1, c[0][3] + c[1][3], r1);
    r0 += __shfl_xor_sync(0xFFFFFFFFu, r0, 1);
    r1 += __shfl_xor_sync(0xFFFFFFFFu, r1, 1);
    r0 += __shfl_xor_sync(0xFFFFFFFFu, r0, 2);
    r1 += __shfl_xor_sync(0xFFFFFFFFu, r1, 2);
    acc[0] += r0;
    acc[1] += r1;
}

template <int TYPE, typename Release>
__device__ __forceinline__ void unit_b4(const Lane& L, int M, float (&acc)[4], Release&& release) {
    using F = Format<TYPE>;
    constexpr int kP = F::kPairs;
    const int g = L.g, t = L.t;
    const uint32_t sel = (t & 1) ? 0x3210u : 0x5432u;
    // column c <-> token c >> 2, block c & 3 of the group; lane t decodes block t
    const bool has_b = (g & 3) == t && (g >> 2) < M;
    const uint8_t* xt = L.x + (g >> 2) * L.xstride;
    static_for<2>([&](auto gc) {
        constexpr int G = decltype(gc)::value;
        const int blk = 4 * G + t;
        // aligned words around the block's code words 0..3 (lo) and 4..7 (hi)
        // of rows g (r0) and g + 8 (r1), loaded word by word
        const uint8_t* b0p = L.r0 + ((kBlockBytes * blk + 2) & ~3);
        const uint8_t* b1p = L.r1 + ((kBlockBytes * blk + 2) & ~3);
        uint32_t l0 = lds_u32(b0p), l1 = lds_u32(b1p), h0 = lds_u32(b0p + 16), h1 = lds_u32(b1p + 16);
        const uint8_t* xb = has_b ? xt + blk * F::kPerBlock * 2 : L.zeros;
        const uint8_t* xb4 = has_b ? xb + 16 * kP : L.zeros;
        float c[2][4];
#pragma unroll
        for (int k = 0; k < 2; ++k) c[k][0] = c[k][1] = c[k][2] = c[k][3] = 0.0f;
        uint32_t xa[4], xh[4];
        static_for<4>([&](auto wc) {
            constexpr int W = decltype(wc)::value;
            const uint32_t nl0 = lds_u32(b0p + 4 * (W + 1)), nl1 = lds_u32(b1p + 4 * (W + 1));
            const uint32_t nh0 = lds_u32(b0p + 16 + 4 * (W + 1)), nh1 = lds_u32(b1p + 16 + 4 * (W + 1));
            const uint32_t w00 = prmt(l0, nl0, sel), w10 = prmt(l1, nl1, sel);     // word W, rows g / g+8
            const uint32_t w01 = prmt(h0, nh0, sel), w11 = prmt(h1, nh1, sel);     // word W+4
            l0 = nl0; l1 = nl1; h0 = nh0; h1 = nh1;
            const uint32_t s00 = w00 >> F::kHighShift, s10 = w10 >> F::kHighShift;
            const uint32_t s01 = w01 >> F::kHighShift, s11 = w11 >> F::kHighShift;
            static_for<kP>([&](auto pc) {
                constexpr int P = decltype(pc)::value;
                constexpr int S = W * kP + P;
                if constexpr (S % 4 == 0) {
                    load_pairs<4>(xb + 4 * S, xa);              // words 0..3
                    load_pairs<4>(xb4 + 4 * S, xh);             // words 4..7
                }
                mma_acc(c[S & 1],
                        decode_pair<TYPE, P>(w00, s00), decode_pair<TYPE, P>(w10, s10),
                        decode_pair<TYPE, P>(w01, s01), decode_pair<TYPE, P>(w11, s11),
                        xa[S % 4], xh[S % 4]);
            });
        });
        // lane columns 2t, 2t+1 <-> token t >> 1, blocks 4G + 2(t & 1) + {0, 1}
        const int bb = 4 * G + 2 * (t & 1);
        float v[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint8_t* r = h ? L.r1 : L.r0;
            const float d0 = lds_half(r + kBlockBytes * bb), d1 = lds_half(r + kBlockBytes * (bb + 1));
            v[h] = fmaf(d1, c[0][2 * h + 1] + c[1][2 * h + 1], d0 * (c[0][2 * h] + c[1][2 * h]));
            v[h] += __shfl_xor_sync(0xFFFFFFFFu, v[h], 1);
            acc[h] += v[h];
        }
    });
    release();
}

// One unit; release() is called once the unit no longer reads its stage.
template <int BPM, int TYPE, typename Release>
__device__ __forceinline__ void unit(const Lane& L, int M, float (&acc)[4], Release&& release) {
    if constexpr (BPM == 8) unit_b8<TYPE>(L, M, acc, release);
    else unit_b4<TYPE>(L, M, acc, release);
}

// ------------------------------------------------------------ tile results --

// The (row, token) a lane's acc[i] holds, and whether this lane is the one
// that deposits it (several lanes hold the same sum).
template <int BPM>
__device__ __forceinline__ bool acc_slot(int g, int t, int i, int& row, int& tok) {
    row = g + 8 * i;
    if constexpr (BPM == 8) { tok = 0; return i < 2 && t == 0; }
    else { tok = t >> 1; return i < 2 && (t & 1) == 0; }
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t atom_exch_u64(uint64_t* p, uint64_t v) {
    return atomicExch(reinterpret_cast<unsigned long long*>(p), static_cast<unsigned long long>(v));
}

constexpr uint32_t kTagFirst = 1u, kTagSecond = 2u;

// A tile cut by a thread-block boundary has two parts, the first chunks
// (held by the block before the boundary) and the rest (held by the block
// after it).  Each side swaps its part, tagged with which part it is, into
// the boundary's slot with one 64-bit atomic exchange per output; exactly one
// side gets the other's part back, adds first + second in that order, stores
// the output and clears the slot.  Neither side waits for the other.  Lane l
// holds output (row l & 15, token l >> 4).
__device__ __forceinline__ void exchange(const SParams& P, const STensor& T, int tile, int lane, bool first,
                                         int boundary, float v) {
    const int row = lane & 15, tok = lane >> 4;
    if (tok >= P.M) return;
    uint64_t* w = P.tagged + static_cast<int64_t>(boundary) * kSlotFloats + row * kStreamMaxM + tok;
    const uint64_t tag = static_cast<uint64_t>(first ? kTagFirst : kTagSecond) << 32;
    const uint64_t got = atom_exch_u64(w, tag | __float_as_uint(v));
    if ((got >> 32) == 0) return;                                 // the other side finishes this output
    const float other = __uint_as_float(static_cast<uint32_t>(got));
    const float s = first ? v + other : other + v;               // first chunks + later chunks
    const int r = tile * kRows + row;
    if (r < T.N) T.y[static_cast<int64_t>(tok) * T.N + r] = s;
    st_relaxed_u64(w, 0ull);
}

// Bounded wait (lane 0) until shared word *p equals want.
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

// --------------------------------------------------------------- rotation --
//
// The runtime Hadamard rotation (tensorless docs, "How Qwen3.8-27B-PN3 uses
// it"), fused: each block rotates the activations of the tensors its range
// touches once, into shared memory, before its warps decode.  The arithmetic
// is the one pn_hadamard fixes, so the rotated values are the same bits: fp16
// -> fp32, butterfly stages h = 1, 2, ..., B/2 in that order, each replacing
// (v[i], v[i+h]) for (i & h) == 0 by (v[i] + v[i+h], v[i] - v[i+h]) in fp32,
// one fp32 multiply by the scale, fp16 round-to-nearest-even.  A warp takes
// a job of 64 Q activations (one run of B = 64 Q, or two runs when B = 32):
// lane l holds the pairs 2l + 64i, 2l + 64i + 1 (i < Q), so stage h = 1 stays
// in the lane, the stages h = 2 .. 32 pair lane l with lane l ^ (h / 2) by
// shuffle, and the stages h >= 64 pair its i with i + h / 64.  Across lanes
// the lower lane keeps v + o and the upper one o - v, both as one
// fma(+-1, v, o): the product is exact, so the single rounding gives the
// same bits as the add or subtract.  Loads and stores are 32-bit (a pair).

template <int Q>
__device__ __forceinline__ void rotate_job(uint32_t* job, int B, float scale, int lane) {
    float v[2 * Q];
#pragma unroll
    for (int i = 0; i < Q; ++i) {
        const uint32_t w = job[lane + 32 * i];
        v[2 * i] = half_lo(w);
        v[2 * i + 1] = half_hi(w);
    }
#pragma unroll
    for (int i = 0; i < Q; ++i) {                       // h = 1
        const float a = v[2 * i], b = v[2 * i + 1];
        v[2 * i] = __fadd_rn(a, b);
        v[2 * i + 1] = __fsub_rn(a, b);
    }
#pragma unroll 1
    for (int d = 1; d <= 16 && 2 * d < B; d <<= 1) {   // h = 2d, while h < B
        const float sgn = (lane & d) ? -1.0f : 1.0f;
#pragma unroll
        for (int j = 0; j < 2 * Q; ++j) v[j] = __fmaf_rn(sgn, v[j], __shfl_xor_sync(0xFFFFFFFFu, v[j], d));
    }
#pragma unroll
    for (int g = 1; g < Q; g <<= 1) {                   // h = 64 g
#pragma unroll
        for (int i = 0; i < Q; ++i) {
            if (i & g) continue;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const float a = v[2 * i + c], b = v[2 * (i + g) + c];
                v[2 * i + c] = __fadd_rn(a, b);
                v[2 * (i + g) + c] = __fsub_rn(a, b);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < Q; ++i) {
        const uint32_t lo = __half_as_ushort(__float2half_rn(__fmul_rn(v[2 * i], scale)));
        const uint32_t hi = __half_as_ushort(__float2half_rn(__fmul_rn(v[2 * i + 1], scale)));
        job[lane + 32 * i] = lo | (hi << 16);
    }
}

// The consumer warps rotate, together and in place, every run of every token
// of tensors e_lo .. e_hi in the resident region (tensor e's token m at
// roff[e] + m * K_e * 2 bytes).  Lane e of every warp holds K_e in k_lane
// (read from the kernel parameters before the activations are waited for).
__device__ void rotate_resident(uint8_t* resident, const uint32_t* roff, int e_lo, int e_hi, int M, int B,
                                float scale, int k_lane, int warp, int lane) {
    const int q = B >= 64 ? B / 64 : 1;                 // pairs per lane
    const int job_elems = 64 * q;
    // jobs are numbered over (tensor, token, offset); this warp takes jobs
    // warp, warp + kConsumers, ... (e, base: the first job of tensor e)
    int e = e_lo, base = 0;
    int K = __shfl_sync(0xFFFFFFFFu, k_lane, e);
    for (int job = warp;; job += kConsumers) {
        while (job - base >= M * (K / job_elems)) {
            base += M * (K / job_elems);
            if (++e > e_hi) return;
            K = __shfl_sync(0xFFFFFFFFu, k_lane, e);
        }
        const int j = job - base;                         // token-major within the tensor
        uint32_t* p = reinterpret_cast<uint32_t*>(resident + roff[e]) + static_cast<size_t>(j) * job_elems / 2;
        switch (q) {
            case 1: rotate_job<1>(p, B, scale, lane); break;
            case 2: rotate_job<2>(p, B, scale, lane); break;
            case 4: rotate_job<4>(p, B, scale, lane); break;
            case 8: rotate_job<8>(p, B, scale, lane); break;
            default: rotate_job<16>(p, B, scale, lane); break;
        }
    }
}

// ----------------------------------------------------------------- kernel --

// Unit record of a stage, written by the producer: the unit's tile and chunk,
// its tensor and flags (this block's part of the tile starts / ends a cut),
// the ticket of the tile's first unit in this block and how many of the
// tile's units this block has.
struct Rec {
    uint32_t tile;
    uint32_t chunk_e_flags;        // chunk | tensor << 24 | left cut << 28 | right cut << 29 | pn4t << 30
    uint32_t k_first;
    uint32_t n_units;
};

// BPM: blocks per MMA (8: one token, 4: two tokens); SLOG: log2 of the ring's
// stages; RES: activations resident (P.resident_bytes > 0) or staged.
template <int BPM, int SLOG, bool RES>
__global__ void __launch_bounds__(kThreads, 1) gemv_stream_kernel(const __grid_constant__ SParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    const bool rot = RES && P.rot_block != 0;
    constexpr bool res = RES;
    const SmemLayout Lay(P.M, 1 << SLOG, RES ? P.resident_bytes : 0u);
    constexpr int slog = SLOG;
    constexpr uint32_t smask = (1u << slog) - 1u;
    const uint32_t sbase = smem_addr(smem);
    const uint32_t full0 = sbase + Lay.full, empty0 = sbase + Lay.empty;
    uint32_t* ticket = reinterpret_cast<uint32_t*>(smem + Lay.misc);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Lay.misc + 4);
    Rec* table = reinterpret_cast<Rec*>(smem + Lay.table);
    float* parts = reinterpret_cast<float*>(smem + Lay.parts);
    volatile uint32_t* gens = reinterpret_cast<volatile uint32_t*>(smem + Lay.gens);
    uint32_t* cnts = reinterpret_cast<uint32_t*>(smem + Lay.cnts);
    uint32_t* roff = reinterpret_cast<uint32_t*>(smem + Lay.misc + 8);    // resident offset per tensor
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // programmatic dependent launch: the next kernel may start now; this one
    // reads weights early but touches activations, outputs and the workspace
    // only after the previous kernel has finished (griddep_wait)
    griddep_launch_dependents();
    for (int i = threadIdx.x; i < kZeroBytes / 4; i += kThreads) reinterpret_cast<uint32_t*>(smem + Lay.zeros)[i] = 0u;
    for (int i = threadIdx.x; i < kParts; i += kThreads) {
        gens[i] = 0u;
        cnts[i] = 0u;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < (1 << slog); ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(sbase + Lay.xbar, 1);
        *ticket = 0u;
        *abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();

    const uint32_t c0 = P.starts[blockIdx.x], c1 = P.starts[blockIdx.x + 1];
    // This block's units in processing order: first its part of the tile that
    // continues into the next block (nr units, the end of its range), then the
    // rest of its range in order.
    int last_e, last_tile, last_chunk;
    locate(P, c1 - 1, last_e, last_tile, last_chunk);
    const uint32_t nr = last_chunk != P.t[last_e].chunks - 1 ? static_cast<uint32_t>(last_chunk + 1) : 0u;
    const uint32_t n = c1 - c0;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ producer --
        // Rounds of kIssueLanes tickets: lane i of a round fills ticket
        // b0 + i once that stage's previous unit has been consumed.  After
        // the units come one end record per consumer.
        for (int e = lane; e < P.count; e += 32) prefetch_tensormap(&P.wmap[e]);
        const uint32_t total = n + kConsumers;
        bool ok = true;
        bool waited = false, x_issued = false;
        uint32_t b0 = 0, filled_mask = 0;             // the last round and which of its lanes filled
        // (with resident activations the first round is short, so that the
        // activations are requested behind a few stages of weights only)
        uint32_t width = RES ? kResidentLead : kIssueLanes;
        for (; b0 < total; b0 += width, width = kIssueLanes) {
            const uint32_t q = b0 + static_cast<uint32_t>(lane);
            bool mine_ok = true, filled = false;
            if (lane < width && q < total) {
                const uint32_t s = q & smask;
                if (q > smask) mine_ok = thread_wait(empty0 + 8 * s, ((q >> slog) - 1) & 1u, P.timeout_ns, abort_flag);
                if (mine_ok && q < n) {
                    const uint32_t u = q < nr ? c1 - nr + q : c0 + (q - nr);
                    int e, tile, chunk;
                    locate(P, u, e, tile, chunk);
                    const STensor& T = P.t[e];
                    const uint32_t tbeg = T.unit_base + static_cast<uint32_t>(tile) * T.chunks;
                    const uint32_t tend = tbeg + T.chunks;
                    const bool left_cut = tbeg < c0, right_cut = tend > c1;
                    const uint32_t lo = left_cut ? c0 : tbeg, hi = right_cut ? c1 : tend;
                    Rec r;
                    r.tile = static_cast<uint32_t>(tile);
                    r.chunk_e_flags = static_cast<uint32_t>(chunk) | (static_cast<uint32_t>(e) << 24) |
                                      (left_cut ? 1u << 28 : 0u) | (right_cut ? 1u << 29 : 0u) |
                                      (T.type == kPn3t ? 0u : 1u << 30);
                    r.k_first = right_cut ? 0u : nr + (lo - c0);
                    r.n_units = hi - lo;
                    table[s] = r;
                    const int halves = kChunkBlocks * per_block(T.type);
                    // (with resident activations a stage holds weights only)
                    mbar_arrive_expect_tx(full0 + 8 * s, kBoxBytes + (res ? 0 : P.M * halves * 2));
                    // (testing aid: with stall_first_step the first unit's
                    // bytes are announced but never copied, so its wait can
                    // only time out)
                    if (!(q == 0 && P.stall_first_step)) {
                        tma_load_2d(sbase + s * Lay.sbytes, &P.wmap[e], chunk * kBoxWords, tile * kRows, full0 + 8 * s);
                        if (!res) {
                            if (!waited) griddep_wait();  // activations may come from the previous kernel
                            waited = true;
                            const uint16_t* x = T.x + static_cast<int64_t>(chunk) * halves;
                            for (int m = 0; m < P.M; ++m)
                                bulk_g2s(sbase + s * Lay.sbytes + kBoxBytes + m * kXTokenBytes,
                                         x + static_cast<int64_t>(m) * T.K, halves * 2, full0 + 8 * s);
                        }
                        filled = true;
                    }
                } else if (mine_ok) {
                    table[s].tile = kEnd;
                    mbar_arrive(full0 + 8 * s);
                }
            }
            filled_mask = __ballot_sync(0xFFFFFFFFu, filled);
            ok = __all_sync(0xFFFFFFFFu, mine_ok);
            if (!ok) break;
            if (RES && b0 == 0 && lane == 0) {
                // the resident activations, queued behind the first round's
                // weights only: their offsets, then one bulk copy per tensor
                // and token (the barrier's completion publishes the offsets)
                griddep_wait();
                int e_lo, dummy0, dummy1;
                locate(P, c0, e_lo, dummy0, dummy1);
                uint32_t off = 0;
                for (int e = e_lo; e <= last_e; ++e) {
                    roff[e] = off;
                    off += static_cast<uint32_t>(P.M * P.t[e].K * 2);
                }
                mbar_arrive_expect_tx(sbase + Lay.xbar, off);
                for (int e = e_lo; e <= last_e; ++e)
                    for (int m = 0; m < P.M; ++m)
                        bulk_g2s(sbase + Lay.resident + roff[e] + static_cast<uint32_t>(m * P.t[e].K * 2),
                                 P.t[e].x + static_cast<int64_t>(m) * P.t[e].K, static_cast<uint32_t>(P.t[e].K * 2),
                                 sbase + Lay.xbar);
                x_issued = true;
            }
        }
        if (!ok) {
            if (lane == 0) {
                *abort_flag = 1u;
                atomicCAS(P.status, 0u, kStatusTimeout);
                // let every copy this block started land before it can exit:
                // only the last S tickets can have copies in flight, one
                // per stage, each in its stage's latest phase
                const uint32_t end = b0 + width;
                for (uint32_t q = end > smask + 1 ? end - (smask + 1) : 0u; q < end && q < n; ++q) {
                    const bool copied = q < b0 ? !(q == 0 && P.stall_first_step) : ((filled_mask >> (q - b0)) & 1u) != 0u;
                    if (copied) thread_wait(full0 + 8 * (q & smask), (q >> slog) & 1u, kDrainLimitNs, nullptr);
                }
                if (x_issued) thread_wait(sbase + Lay.xbar, 0u, kDrainLimitNs, nullptr);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers --
    // (what the rotation reads of the parameters, loaded before the waits so
    // that their latency overlaps them: lane e holds tensor e's K and first
    // unit)
    int rot_k = 0, rot_b = 0;
    uint32_t rot_base = 0;
    float rot_scale = 0.0f;
    if (rot) {
        rot_b = P.rot_block;
        rot_scale = P.rot_scale;
        if (lane < P.count) {
            rot_k = P.t[lane].K;
            rot_base = P.t[lane].unit_base;
        }
    }
    griddep_wait();
    if (res && !warp_wait(sbase + Lay.xbar, 0u, P.timeout_ns, abort_flag)) {
        // (the producer's copies of the resident activations land before
        // the block can exit)
        if (lane == 0) {
            *abort_flag = 1u;
            atomicCAS(P.status, 0u, kStatusTimeout);
            if (warp == 0) thread_wait(sbase + Lay.xbar, 0u, kDrainLimitNs, nullptr);
        }
        return;
    }
    if (rot) {
        // rotate the resident activations in place (the producer streams
        // weights meanwhile), then every warp may read them
        // the first tensor of the range: the last whose first unit is <= c0
        const int e_lo = __popc(__ballot_sync(0xFFFFFFFFu, lane >= 1 && lane < P.count && c0 >= rot_base));
        rotate_resident(smem + Lay.resident, roff, e_lo, last_e, P.M, rot_b, rot_scale, rot_k, warp, lane);
        named_barrier_sync(1, kConsumers * 32);
    }
    Lane L;
    L.g = lane >> 2;
    L.t = lane & 3;
    L.zeros = smem + Lay.zeros;
    L.xown = smem + Lay.xown + warp * kXTokenBytes;
    L.resident = res;
    L.xstride = kXTokenBytes;
    for (;;) {
        uint32_t k = 0;
        if (lane == 0) k = atomicAdd(ticket, 1u);
        k = __shfl_sync(0xFFFFFFFFu, k, 0);
        const uint32_t s = k & smask;
        const uint32_t ph = k >> slog;
        // a stage's barriers are waited on by parity, which tells two
        // consecutive phases apart only: first wait until ticket k - S
        // has released the stage, so the full barrier is at most one phase ahead
        if (k > smask && !warp_wait(empty0 + 8 * s, (ph - 1) & 1u, P.timeout_ns, abort_flag)) {
            if (lane == 0) {
                *abort_flag = 1u;
                atomicCAS(P.status, 0u, kStatusTimeout);
            }
            return;
        }
        if (!warp_wait(full0 + 8 * s, ph & 1u, P.timeout_ns, abort_flag)) {
            if (lane == 0) {
                *abort_flag = 1u;
                atomicCAS(P.status, 0u, kStatusTimeout);
                // the stage's copies, if the producer issued them, land before this warp leaves
                if (!(k == 0 && P.stall_first_step)) thread_wait(full0 + 8 * s, ph & 1u, kDrainLimitNs, nullptr);
            }
            return;
        }
        const Rec rec = table[s];
        if (rec.tile == kEnd) return;
        const int e = static_cast<int>((rec.chunk_e_flags >> 24) & 15u);
        const uint8_t* stage = smem + s * Lay.sbytes;
        L.r0 = stage + L.g * kChunkBytes;
        L.r1 = stage + (L.g + 8) * kChunkBytes;
        if (res) {
            const int chunk = static_cast<int>(rec.chunk_e_flags & 0xFFFFFFu);
            const STensor& Tx = P.t[e];
            L.x = smem + Lay.resident + roff[e] + static_cast<size_t>(chunk) * kChunkBlocks * per_block(Tx.type) * 2;
            L.xstride = Tx.K * 2;
        } else {
            L.x = stage + kBoxBytes;
        }
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        auto release = [&] {                              // the stage may be refilled
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
        };
        if (((rec.chunk_e_flags >> 30) & 1u) == 0u) unit<BPM, kPn3t>(L, P.M, acc, release);
        else unit<BPM, kPn4t>(L, P.M, acc, release);
        // the unit's partials to slot k of the ring, once its previous user
        // (ticket k - kParts, a lower ticket) has been combined; the tile's
        // counter is in the slot of the tile's first ticket
        const uint32_t slot = k & (kParts - 1), fslot = rec.k_first & (kParts - 1);
        bool ok = true;
        // (every lane reads the same words, so the branch is uniform)
        if (gens[slot] != (k >> kPartsLog2) || gens[fslot] != (rec.k_first >> kPartsLog2)) {
            if (lane == 0)
                ok = smem_wait_eq(gens + slot, k >> kPartsLog2, P.timeout_ns, abort_flag) &&
                     smem_wait_eq(gens + fslot, rec.k_first >> kPartsLog2, P.timeout_ns, abort_flag);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        }
        if (!ok) {
            if (lane == 0) {
                *abort_flag = 1u;
                atomicCAS(P.status, 0u, kStatusTimeout);
            }
            return;
        }
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            int row, tok;
            if (acc_slot<BPM>(g, t, i, row, tok)) parts[slot * kSlotFloats + row * kStreamMaxM + tok] = acc[i];
        }
        __syncwarp();
        uint32_t old = 0;
        if (lane == 0) old = atomicAdd(cnts + fslot, 1u);
        old = __shfl_sync(0xFFFFFFFFu, old, 0);
        if (old + 1 != rec.n_units) continue;
        // this warp finished the tile's part in this block: its chunks in order
        const STensor& T = P.t[e];
        const int tile = static_cast<int>(rec.tile);
        const int row = lane & 15, tok = lane >> 4;
        float v = 0.0f;
        if (tok < P.M)
            for (uint32_t j = 0; j < rec.n_units; ++j)
                v += parts[((rec.k_first + j) & (kParts - 1)) * kSlotFloats + row * kStreamMaxM + tok];
        __syncwarp();
        // free the slots for their next users
        if (lane == 0) cnts[fslot] = 0u;
        for (uint32_t j = lane; j < rec.n_units; j += 32) {
            const uint32_t kk = rec.k_first + j;
            gens[kk & (kParts - 1)] = (kk >> kPartsLog2) + 1u;
        }
        const bool left_cut = (rec.chunk_e_flags >> 28) & 1u, right_cut = (rec.chunk_e_flags >> 29) & 1u;
        if (left_cut || right_cut) {
            exchange(P, T, tile, lane, right_cut, right_cut ? static_cast<int>(blockIdx.x) + 1 : static_cast<int>(blockIdx.x), v);
        } else if (tok < P.M) {
            const int r = tile * kRows + row;
            if (r < T.N) T.y[static_cast<int64_t>(tok) * T.N + r] = v;
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
// box = one 8-block chunk (68 words) x 16 rows; rows past N read as zero.
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

template <int BPM, int SLOG, bool RES>
cudaError_t launch_k(const SParams& P, int smem, cudaStream_t s) {
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = set_smem_limit_once(gemv_stream_kernel<BPM, SLOG, RES>, kSmemLimit, smem_set);
        e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(P.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_stream_kernel<BPM, SLOG, RES>, P);
}

// The ring has kStagesLog2 stages, or one power of two fewer where rotated
// activations need the room.
static_assert(kStagesLog2 == kMinStagesLog2 + 1, "two ring sizes");

template <int BPM>
cudaError_t launch_bpm(const SParams& P, int smem, cudaStream_t s) {
    if (!P.resident_bytes) return launch_k<BPM, kStagesLog2, false>(P, smem, s);
    return P.stages_log2 == kStagesLog2 ? launch_k<BPM, kStagesLog2, true>(P, smem, s)
                                        : launch_k<BPM, kMinStagesLog2, true>(P, smem, s);
}

static_assert(SmemLayout(kStreamMaxM, kStages, 0).total <= kSmemLimit, "the two-token layout fits one SM");

}  // namespace

int stream_max_chunks() { return kParts; }

int stream_max_ctas(int num_sms) { return num_sms < kMaxGrid ? num_sms : kMaxGrid; }

size_t stream_tagged_bytes(int num_sms) {
    return static_cast<size_t>(stream_max_ctas(num_sms) + 1) * kSlotFloats * sizeof(uint64_t);
}

// The resident activations a rotating call keeps in a block whose range is
// [u0, u1): every token's K of each tensor the range touches.
static uint32_t resident_need(const STensor* T, int count, int M, uint32_t u0, uint32_t u1) {
    uint32_t bytes = 0;
    for (int e = 0; e < count; ++e) {
        const uint32_t b = T[e].unit_base, end = b + static_cast<uint32_t>(T[e].chunks) * T[e].tiles;
        if (u0 < end && u1 > b) bytes += static_cast<uint32_t>(M) * T[e].K * 2;
    }
    return bytes;
}

cudaError_t launch_gemv_stream(const GemvTensor* t, int count, int M, uint32_t* status, uint64_t* tagged,
                               int num_sms, uint64_t timeout_ns, int stall, cudaStream_t s, int rot_block) {
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
        // a tile's chunk partials must all fit the shared-memory slot ring
        if (T.chunks > kParts) return cudaErrorInvalidValue;
        if (rot_block && T.K % rot_block) return cudaErrorInvalidValue;
        units += static_cast<uint64_t>(T.chunks) * T.tiles;
        max_chunks = T.chunks > max_chunks ? T.chunks : max_chunks;
    }
    if (units == 0) return cudaSuccess;
    if (units >= (1ull << 31)) return cudaErrorInvalidValue;    // 32-bit unit arithmetic
    P.count = count;
    P.M = M;
    // Every range spans at least one whole tile, so a tile has at most two
    // blocks, and holds the same number of units (pn3t and pn4t units move the
    // same bytes).
    CostSplit split{};
    for (int e = 0; e < count; ++e) split.add(static_cast<uint32_t>(P.t[e].chunks) * P.t[e].tiles, 1u);
    P.grid = split.fit_grid(stream_max_ctas(num_sms), static_cast<uint32_t>(max_chunks));
    for (int c = 0; c <= P.grid; ++c) P.starts[c] = split.start(c);
    P.status = status;
    P.tagged = tagged;
    P.timeout_ns = timeout_ns;
    P.stall_first_step = stall;
    P.stages_log2 = kStagesLog2;
    uint32_t need = 0;
    for (int c = 0; c < P.grid; ++c) {
        const uint32_t b = resident_need(P.t, count, M, P.starts[c], P.starts[c + 1]);
        need = b > need ? b : need;
    }
    if (rot_block) {
        int m = 0;
        while ((1 << m) < rot_block) ++m;
        if ((1 << m) != rot_block || rot_block < 32 || rot_block > 1024) return cudaErrorInvalidValue;
        const float sqrt2 = 1.41421356237309504880f;
        P.rot_block = rot_block;
        P.rot_scale = (m % 2) ? ldexpf(sqrt2, -(m + 1) / 2) : ldexpf(1.0f, -(m / 2));
        // a smaller ring leaves more room for the rotated activations
        P.resident_bytes = need;
        while (SmemLayout(M, 1 << P.stages_log2, need).total > kSmemLimit && P.stages_log2 > kMinStagesLog2)
            --P.stages_log2;
        if (SmemLayout(M, 1 << P.stages_log2, need).total > kSmemLimit) return cudaErrorInvalidValue;
    } else if ((count > 1 || M > 1) && SmemLayout(M, 1 << P.stages_log2, need).total <= kSmemLimit) {
        // the activations resident beside a full ring, copied in once per
        // block instead of once per unit.  Measured on GB300 (CUDA-event
        // timed graph replays): 2.3 us faster on the 27B-class layer at
        // M = 1, 0.2 us on single tensors at M = 2, but 1.2 to 1.6 us slower
        // on single tensors at M = 1, where every block copies the same
        // activations at the same moment; those stay staged.
        P.resident_bytes = need;
    }
    const int smem = SmemLayout(M, 1 << P.stages_log2, P.resident_bytes).total;
    return M == 1 ? launch_bpm<8>(P, smem, s) : launch_bpm<4>(P, smem, s);
}

namespace {

// The largest resident set of any block of a launch over these tensors (0 if
// the call has no units or does not suit the kernel).
uint32_t max_resident_need(const GemvTensor* t, int count, int M, int num_sms, int rot_block) {
    if (M < 1 || M > kStreamMaxM || count < 1 || count > kMaxLayer) return 0;
    STensor T[kMaxLayer] = {};
    uint64_t units = 0;
    int max_chunks = 1;
    CostSplit split{};
    for (int e = 0; e < count; ++e) {
        T[e].K = t[e].nb * per_block(t[e].type);
        T[e].chunks = t[e].nb / kChunkBlocks;
        T[e].tiles = (t[e].N + kRows - 1) / kRows;
        T[e].unit_base = static_cast<uint32_t>(units);
        if (t[e].nb % kChunkBlocks || T[e].chunks > kParts || (rot_block && T[e].K % rot_block)) return 0;
        units += static_cast<uint64_t>(T[e].chunks) * T[e].tiles;
        max_chunks = T[e].chunks > max_chunks ? T[e].chunks : max_chunks;
        split.add(static_cast<uint32_t>(T[e].chunks) * T[e].tiles, 1u);
    }
    if (units == 0) return 0;
    const int grid = split.fit_grid(stream_max_ctas(num_sms), static_cast<uint32_t>(max_chunks));
    uint32_t need = 0;
    for (int c = 0; c < grid; ++c) {
        const uint32_t b = resident_need(T, count, M, split.start(c), split.start(c + 1));
        need = b > need ? b : need;
    }
    return need;
}

}  // namespace

bool stream_rotation_fits(const GemvTensor* t, int count, int M, int num_sms, int rot_block) {
    if (rot_block < 32 || rot_block > 1024 || (rot_block & (rot_block - 1))) return false;
    const uint32_t need = max_resident_need(t, count, M, num_sms, rot_block);
    return need > 0 && SmemLayout(M, 1 << kMinStagesLog2, need).total <= kSmemLimit;
}

bool stream_resident_fits(const GemvTensor* t, int count, int M, int num_sms) {
    const uint32_t need = max_resident_need(t, count, M, num_sms, 0);
    return need > 0 && SmemLayout(M, 1 << kStagesLog2, need).total <= kSmemLimit;
}

}  // namespace pn
