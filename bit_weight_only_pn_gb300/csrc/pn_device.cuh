// pn_device.cuh -- PN format constants and the sm_103a PTX helpers used by the kernels.
//
// Format (tensorless docs, "Why a P100-native weight format"): a 34-byte block
// holds an fp16 scale d followed by eight 32-bit code words; pn3t packs ten
// 3-bit codes per word (80 weights per block), pn4t eight 4-bit codes (64).
// Even codes sit in bits 0..15 and odd codes in bits 16..31 at the same offsets
// ("Codes never straddle the two halves of a word"); a weight is d * (n - z)
// ("Exact decode in fp32") with mid-tread zero point z = 4 (pn3t) / 8 (pn4t).
// Layout readings: d in bytes 0..1, word j in bytes 2+4j..5+4j, weight k is code
// k % cpw of word k / cpw, code c at bit 16*(c&1) + bits*(c>>1).
#pragma once

#include <cstdint>
#include <type_traits>
#include <utility>

#include <cuda_fp16.h>

namespace pn {

constexpr int kBlockBytes = 34;
constexpr int kWordsPerBlock = 8;
constexpr int kPn3t = 124;
constexpr int kPn4t = 125;

template <int TYPE> struct Format;

template <> struct Format<kPn3t> {
    static constexpr int kPerBlock = 80;   // weights per block
    static constexpr int kPerWord = 10;    // codes per word
    static constexpr int kBits = 3;
    static constexpr int kZero = 4;
    static constexpr int kPairs = 5;       // half2 code pairs per word
    // Upper code pairs are shifted down by this much so that every pair's two
    // codes sit inside the 10-bit mantissa of an fp16 (see decode_pair).
    static constexpr int kHighShift = 9;
    static constexpr int kLowPairs = 3;    // pairs 0..2 decode from the unshifted word
};

template <> struct Format<kPn4t> {
    static constexpr int kPerBlock = 64;
    static constexpr int kPerWord = 8;
    static constexpr int kBits = 4;
    static constexpr int kZero = 8;
    static constexpr int kPairs = 4;
    static constexpr int kHighShift = 8;
    static constexpr int kLowPairs = 2;
};

__host__ __device__ constexpr int per_block(int type) { return type == kPn3t ? 80 : 64; }

// ------------------------------------------------------------- PTX helpers --

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}

// One non-blocking probe of phase `parity` of the barrier: true once that
// phase has completed.  (mbarrier.test_wait answers at once; a thread parked
// inside mbarrier.try_wait was measured to notice a completed phase late.)
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0;
}

// One probe of phase `parity` that may suspend the thread until the phase
// completes or about `hint_ns` nanoseconds pass (mbarrier.try_wait with a
// suspend-time hint); true once the phase has completed.  A suspended warp
// issues nothing, so waiting warps leave the issue slots to working ones.
__device__ __forceinline__ bool mbar_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
    return done != 0;
}

// Bulk copy (TMA engine, no tensor map) of `bytes` (multiple of 16, both
// addresses 16-byte aligned) from global to this CTA's shared memory; the
// byte count is credited to the transaction count of `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Tiled 2-D TMA load of one box of `tmap` at element coordinates (x, y) into
// this CTA's shared memory, credited to `bar`.  x * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar) : "memory");
}

// Prefetch of one box of `tmap` from global memory into L2 (no shared-memory
// destination, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 :: "l"(tmap), "r"(x), "r"(y) : "memory");
}

// Prefetch of the L1 line holding `p` (global memory).
__device__ __forceinline__ void prefetch_l1(const void* p) {
    asm volatile("prefetch.global.L1 [%0];" :: "l"(p));
}

// Brings a tensor map (a kernel parameter) into the TMA descriptor cache.
__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// its later async-proxy (TMA) accesses to shared memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: let the next kernel on the stream launch
// now / wait until the previous kernel has completed and its writes are visible.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Shared-memory loads as plain C++ loads through a pointer into the kernel's
// dynamic shared memory: the compiler may schedule them freely, but never
// across the mbarrier waits and arrives, which are asm with memory clobbers.

__device__ __forceinline__ uint32_t lds_u32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint2 lds_u64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint4 lds_u128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ float lds_half_as_float(const uint8_t* p) {
    return __half2float(*reinterpret_cast<const __half*>(p));
}

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Bytes {a.hi, b.lo}: the 32-bit word that starts two bytes into `a`.
__device__ __forceinline__ uint32_t realign16(uint32_t a, uint32_t b) {
    return __byte_perm(a, b, 0x5432);
}

// C += A * B, m16n8k16, fp16 inputs, fp32 accumulate, accumulator in place.
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float half_bits_to_float(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// ----------------------------------------------------------- code decoding --
//
// decode_pair<TYPE, P>(word, shifted) returns the half2 (n_{2P} - z, n_{2P+1} - z)
// of code pair P of a word, exactly.  A LOP3 keeps the pair's two codes (one
// per 16-bit half, same offset) and ORs in the fp16 bit pattern 0x6400 (1024.0),
// giving the halves 1024 + n * 2^off as long as the code lies in the 10-bit
// mantissa; one fma.rn.f16x2 by 2^-off minus (1024 * 2^-off + z) leaves n - z.
// Every intermediate value is an fp16 number, so the result is exact.  Pairs
// whose offset would reach the exponent bits use the word shifted right once.

template <int TYPE, int P>
__device__ __forceinline__ uint32_t decode_pair(uint32_t word, uint32_t shifted) {
    using F = Format<TYPE>;
    constexpr bool kHigh = P >= F::kLowPairs;
    constexpr int kOff = F::kBits * (kHigh ? P - F::kLowPairs : P);
    constexpr uint32_t kMask = ((1u << F::kBits) - 1u) << kOff;
    constexpr uint32_t kMask2 = kMask | (kMask << 16);
    // scale 2^-off as fp16 (exponent 15 - off), replicated into both halves
    constexpr uint32_t kScale = static_cast<uint32_t>(15 - kOff) << 10;
    constexpr uint32_t kScale2 = kScale | (kScale << 16);
    // bias -(1024 * 2^-off + z) as fp16
    constexpr uint32_t kBias = (TYPE == kPn3t)
        ? (kOff == 0 ? 0xE404u : kOff == 3 ? 0xD820u : 0xCD00u)   // -1028, -132, -20
        : (kOff == 0 ? 0xE408u : 0xD480u);                         // -1032, -72
    constexpr uint32_t kBias2 = kBias | (kBias << 16);
    return hfma2(and_or(kHigh ? shifted : word, kMask2, 0x64006400u), kScale2, kBias2);
}

// ------------------------------------------------- one block of a 16-row tile --
//
// A staged tile holds 16 rows of one 8-block chunk, 272 bytes apart.  Lane
// (g, t) of a warp (g = lane / 4, t = lane % 4) owns MMA rows g and g + 8 and
// code words 2t, 2t + 1 of every block: ten (pn3t) or eight (pn4t) code pairs
// q = 0, 1, ... (word 2t's pairs first), whose activations are the lane's
// consecutive x pairs 2 * kPerWord * t / 2 + q.  The block's s-th m16n8k16
// product takes pairs q = 2s (k-slots 2t, 2t+1) and q = 2s + 1 (k-slots
// 2t + 8, 2t + 9) of every lane, so its B fragment is two adjacent x pairs,
// one 64-bit load, and its 16 k-slots all lie in the block (one scale).

constexpr int kStagedRowBytes = 8 * kBlockBytes;    // 272: rows of a staged tile

template <int N, typename Fn, int... I>
__device__ __forceinline__ void static_for_impl(Fn&& fn, std::integer_sequence<int, I...>) {
    (fn(std::integral_constant<int, I>{}), ...);
}
template <int N, typename Fn>
__device__ __forceinline__ void static_for(Fn&& fn) {
    static_for_impl<N>(fn, std::make_integer_sequence<int, N>{});
}

// Fragment row g (and g + 8) of a tile reads staged row tile_row(g) (and +8).
// Rows are 272 bytes (68 banks, 4 mod 32) apart; taking the even rows for
// g = 0..3 and the odd rows for g = 4..7 makes every 64-bit load of a
// half-warp hit 32 distinct banks.
__device__ __forceinline__ int tile_row(int g) { return ((g & 3) << 1) | (g >> 2); }

// Loads code words 2t and 2t+1 of block B of a staged row (8-byte aligned).
template <int B>
__device__ __forceinline__ void load_words(const uint8_t* row, int t, uint32_t& w0, uint32_t& w1) {
    constexpr int kOff = B * kBlockBytes;
    if constexpr (B % 2 == 0) {
        // block starts 4-byte aligned: its words start 2 bytes into aligned words
        const uint8_t* a = row + kOff + 8 * t;
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
        const uint8_t* a = row + kOff + 2 + 8 * t;
        if constexpr ((kOff + 2) % 8 == 0) {
            const uint2 p = lds_u64(a);
            w0 = p.x; w1 = p.y;
        } else {
            w0 = lds_u32(a);
            w1 = lds_u32(a + 4);
        }
    }
}

// Code pair q of the lane's two words (q < kPairs: word 2t, else word 2t+1).
template <int TYPE, int Q>
__device__ __forceinline__ uint32_t lane_pair(uint32_t w0, uint32_t s0, uint32_t w1, uint32_t s1) {
    constexpr int kP = Format<TYPE>::kPairs;
    if constexpr (Q < kP) return decode_pair<TYPE, Q>(w0, s0);
    else return decode_pair<TYPE, Q - kP>(w1, s1);
}

// Block B of staged rows r0 (MMA row g) and r1 (row g + 8) times NT column
// tiles of x (tokens 8n .. 8n+7 in tile n).  xpair(n, S) gives the lane's two
// B-fragment registers of MMA S in tile n: the x pairs that go with code
// pairs 2S and 2S + 1 of lane_pair's numbering.  The A fragments are decoded
// once and feed one MMA per column tile.  Each block's products start from
// zero and are scaled by the rows' d in fp32: part[n][0..1] += d(r0) *
// (columns 2t, 2t+1 of tile n), part[n][2..3] += d(r1) * (same).
template <int TYPE, int B, int NT, typename XPair>
__device__ __forceinline__ void block_mma(const uint8_t* r0, const uint8_t* r1, int t, XPair&& xpair,
                                          float (&part)[NT][4]) {
    using F = Format<TYPE>;
    const float d0 = lds_half_as_float(r0 + B * kBlockBytes);
    const float d1 = lds_half_as_float(r1 + B * kBlockBytes);
    uint32_t w00, w10, w01, w11;        // w<word><row>: words 2t / 2t+1 of rows g / g+8
    load_words<B>(r0, t, w00, w10);
    load_words<B>(r1, t, w01, w11);
    const uint32_t s00 = w00 >> F::kHighShift, s10 = w10 >> F::kHighShift;
    const uint32_t s01 = w01 >> F::kHighShift, s11 = w11 >> F::kHighShift;
    float c[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) c[n][0] = c[n][1] = c[n][2] = c[n][3] = 0.0f;
    static_for<F::kPairs>([&](auto sc) {
        constexpr int S = decltype(sc)::value;
        const uint32_t a0 = lane_pair<TYPE, 2 * S>(w00, s00, w10, s10);       // row g,   k = 2t, 2t+1
        const uint32_t a1 = lane_pair<TYPE, 2 * S>(w01, s01, w11, s11);       // row g+8, k = 2t, 2t+1
        const uint32_t a2 = lane_pair<TYPE, 2 * S + 1>(w00, s00, w10, s10);   // row g,   k = 2t+8, 2t+9
        const uint32_t a3 = lane_pair<TYPE, 2 * S + 1>(w01, s01, w11, s11);   // row g+8, k = 2t+8, 2t+9
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const uint2 b = xpair(n, sc);
            mma_16816(c[n], a0, a1, a2, a3, b.x, b.y);
        }
    });
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        part[n][0] = fmaf(d0, c[n][0], part[n][0]);
        part[n][1] = fmaf(d0, c[n][1], part[n][1]);
        part[n][2] = fmaf(d1, c[n][2], part[n][2]);
        part[n][3] = fmaf(d1, c[n][3], part[n][3]);
    }
}

}  // namespace pn
