/*
 * pn.h -- C ABI of the PN weight-only decode GEMV library for GB300 (sm_103a).
 *
 * The PN formats come from the tensorless documentation, page "Why a P100-native
 * weight format":
 *   - "Every block is 34 bytes": a block is a 2-byte fp16 scale d and eight
 *     32-bit code words; pn3t holds 80 weights (ten 3-bit codes per word,
 *     3.40 bits/weight), pn4t holds 64 weights (eight 4-bit codes per word,
 *     4.25 bits/weight).  A row holds a whole number of blocks.
 *   - "Codes never straddle the two halves of a word": even codes fill bits
 *     0..15, odd codes bits 16..31, at the same offsets.
 *   - "Exact decode in fp32": weight = d * (n - z), exact in fp32.
 *   - "Zero is a code, and the scale has a sign": mid-tread codes, z = 4 for
 *     pn3t (steps -4..+3); the signed scale puts the extra step on the side of
 *     the block's largest weight.
 *
 * Where the page leaves the layout open this library reads it as follows (the
 * same readings as the CPU oracle used by the tests):
 *   - block bytes 0..1 = d (IEEE binary16, little-endian), bytes 2..33 = code
 *     words w0..w7 (little-endian);
 *   - weight k of a block is code c = k % cpw of word k / cpw (cpw = 10 pn3t,
 *     8 pn4t); code c sits in half (c & 1) at bit offset bits * (c >> 1);
 *     pn3t bits 15 and 31 are written as 0 and ignored on decode;
 *   - z = 4 (pn3t) and z = 8 (pn4t, steps -8..+7);
 *   - the packer rounds to nearest with d = fp16(a / -z), a = the block's
 *     largest-magnitude weight (first on ties); codes n = clamp(rint(v / d),
 *     -z, z-1) + z (fp32 divides, ties to even); a block whose scale is 0 or
 *     underflows fp16 is the zero block (d = +0, all codes z); a scale above
 *     the fp16 range saturates to +-65504.
 *
 * Layouts.  W: N rows of pn_row_bytes(type, K) bytes, row-major, no padding.
 * Dense weights w: fp32 [N][K] row-major.  Activations x: IEEE binary16 bit
 * patterns [M][K] row-major.  Outputs y: fp32 [M][N] row-major.
 *
 * Conventions.  Every pointer except descriptor arrays is device memory owned
 * by the caller; the library allocates nothing.  Every call is asynchronous on
 * the given CUDA stream (NULL = the legacy default stream) and returns after
 * the launch.  Arguments are checked on the host before anything is launched;
 * a failed check returns an error status and launches nothing.  A CUDA launch
 * error is returned as PN_ECUDA.  No call aborts, throws or prints.
 *
 * Thread safety: calls may be made from several host threads; calls that share
 * a workspace must be ordered on one stream.
 */
#ifndef PN_H
#define PN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                      /* == cudaStream_t / CUstream */
typedef struct CUstream_st* pn_stream;

/* Weight types; the values are the GGUF type ids the page gives for PN
 * ("Why the format is specific to this engine": 124 and 125). */
typedef enum { PN_TYPE_PN3T = 124, PN_TYPE_PN4T = 125 } pn_type;

typedef enum {
    PN_OK = 0,
    PN_EINVAL = 1,        /* bad type, size, count, null pointer, small workspace */
    PN_EALIGN = 2,        /* a pointer is not aligned as documented */
    PN_EUNSUPPORTED = 3,  /* valid request this build cannot serve (e.g. not sm_10x) */
    PN_ECUDA = 4,         /* a CUDA runtime call or launch failed */
    PN_ETIMEOUT = 5       /* a device-side wait gave up (reported by pn_workspace_status) */
} pn_status;

/* GEMV algorithm selection for pn_gemv_ex / pn_gemv_layer_ex. */
typedef enum {
    PN_ALGO_AUTO = 0,         /* tensor-core kernel where eligible, else CUDA cores */
    PN_ALGO_TENSOR_CORE = 1,  /* TMA-staged rows, decode into mma.sync fragments   */
    PN_ALGO_CUDA_CORE = 2,    /* one lane per code word, fp32 FMAs                 */
    PN_ALGO_CUDA_CORE_STAGED = 3  /* TMA-staged rows as for the tensor cores; each
                                     decoded fp16 (n - z) times fp16 x added in fp32
                                     on the FMA pipe (fma.rn.f32.f16) for every
                                     token; 1 <= M <= 8, rows of at most 64 chunks
                                     of 8 blocks, tensor-core alignment rules
                                     (PN_EUNSUPPORTED / PN_EALIGN otherwise) */
} pn_algo;

#define PN_BLOCK_BYTES 34
#define PN_MAX_M 16           /* largest activation count M per GEMV */
#define PN_MAX_LAYER 8        /* most tensors per pn_gemv_layer call */

/* Version of this ABI (incremented on any incompatible change). */
int pn_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* pn_status_string(pn_status s);

/* Name of the CUDA runtime error (as cudaGetErrorName gives it) behind the
 * latest PN_ECUDA that a failing CUDA call caused on the calling host thread;
 * "cudaSuccess" if there was none.  Static string. */
const char* pn_last_cuda_error(void);

/* Weights per block (80 / 64) or 0 for an unknown type. */
int pn_weights_per_block(int type);

/* Bytes per PN row: (K / weights_per_block) * 34, or 0 if the type is unknown
 * or K is not a positive multiple of the block size ("A row must hold a whole
 * number of blocks"). */
size_t pn_row_bytes(int type, int64_t K);

/*
 * pn_pack: quantise fp32 weights w [N][K] into PN rows W [N][row_bytes] with
 * the signed-scale round-to-nearest rule above.  w must be 4-byte aligned, W
 * 2-byte aligned; inputs must be finite (the result for non-finite inputs is
 * unspecified).  Deterministic and byte-identical to the CPU oracle.
 */
pn_status pn_pack(int type, const float* w, int64_t N, int64_t K, void* W, pn_stream stream);

/*
 * pn_unpack: decode PN rows W [N][row_bytes] into fp32 w [N][K]; each weight is
 * the single IEEE fp32 product d * (n - z), exact ("Exact decode in fp32"),
 * including the sign of zero.  W 2-byte aligned, w 4-byte aligned.
 */
pn_status pn_unpack(int type, const void* W, int64_t N, int64_t K, float* w, pn_stream stream);

/*
 * Workspace for the GEMV calls.  The tensor-core kernels split the rows and K
 * blocks of all tensors of a call evenly over their thread blocks; a tile of
 * rows whose K range is split between two thread blocks is finished by one of
 * them, which adds the other block's part in a fixed order, so results are
 * deterministic.  That needs device scratch: a status word and, per
 * thread-block boundary, hand-off slots and a counter.  The size depends only
 * on the device's SM count (about 2.3 KiB per SM), so calls of any shape can
 * share one workspace.
 *
 * pn_workspace_bytes(total_rows): bytes needed by one call whose tensors have
 * total_rows rows in all (sum of N), on the current device.
 * pn_workspace_init: zero a workspace (required once before first use; every
 * call that completes leaves it zeroed again).
 * pn_workspace_status: synchronise `stream`, read and clear the device status
 * word of the workspace; returns PN_OK or the device-side error (PN_ETIMEOUT),
 * and re-zeroes the whole workspace after an error.
 * Workspace pointers must be 256-byte aligned.
 */
size_t pn_workspace_bytes(int64_t total_rows);
pn_status pn_workspace_init(void* workspace, size_t workspace_bytes, pn_stream stream);
pn_status pn_workspace_status(void* workspace, size_t workspace_bytes, pn_stream stream);

/*
 * pn_gemv: y[m][r] = sum_k w[r][k] * x[m][k] for m < M (1 <= M <= 16), r < N,
 * where w is W decoded as in pn_unpack.  This is the decode GEMV of token
 * generation (M = 1) and its skinny verification batch (M <= 16, one token
 * plus up to 15 drafts); the weights cross memory once whatever M is.  Products are exact in fp32 and sums are kept in fp32; every output
 * is within 1e-5 * sum_k |w[r][k] x[m][k]| + 1e-6 of the exact value.
 * Alignment: W and x 16-byte aligned for the tensor-core kernel (otherwise
 * PN_ALGO_AUTO uses the CUDA-core kernel, which needs W and x 2-byte and y
 * 4-byte aligned).  y must not overlap W or x.
 */
pn_status pn_gemv(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int M,
                  float* y, void* workspace, size_t workspace_bytes, pn_stream stream);

pn_status pn_gemv_ex(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int M,
                     float* y, void* workspace, size_t workspace_bytes, int algo,
                     pn_stream stream);

/*
 * pn_gemv_layer: the GEMVs of several independent tensors (one decoder layer's
 * projections) in one launch, all with the same M.  The thread blocks share
 * out the rows and K blocks of every tensor in proportion to their bytes.
 * Descriptors are read on the host during the call.  No entry's y may overlap
 * any entry's W, x or y.  At most PN_MAX_LAYER entries.
 */
typedef struct {
    int type;               /* PN_TYPE_PN3T or PN_TYPE_PN4T            */
    const void* W;          /* device, [N][pn_row_bytes(type, K)]      */
    int64_t N;              /* rows                                    */
    int64_t K;              /* input width                             */
    const uint16_t* x;      /* device, fp16 [M][K]                     */
    float* y;               /* device, fp32 [M][N]                     */
} pn_gemv_desc;

pn_status pn_gemv_layer(const pn_gemv_desc* descs, int count, int M, void* workspace,
                        size_t workspace_bytes, pn_stream stream);

pn_status pn_gemv_layer_ex(const pn_gemv_desc* descs, int count, int M, void* workspace,
                           size_t workspace_bytes, int algo, pn_stream stream);

/*
 * pn_gemv_layer_host: pn_gemv_layer with the activations taken from and the
 * outputs returned to host memory, end to end in one call.  x_host holds every
 * entry's x fp16 [M][K] one after the other in entry order, y_host every
 * entry's y fp32 [M][N] the same way.  The call copies x_host into the
 * entries' device x buffers, runs the GEMVs (PN_ALGO_AUTO) on `stream`, copies
 * the entries' device y into y_host and waits for the stream: it returns when
 * y_host is written.  Entries whose device buffers follow each other are
 * copied in one transfer.  Page-locked (pinned) host memory keeps the copies
 * at full speed.  Every check (the descriptors as for pn_gemv_layer, null host
 * pointers, the workspace, which is required) runs before anything is
 * enqueued.
 */
pn_status pn_gemv_layer_host(const pn_gemv_desc* descs, int count, int M, const uint16_t* x_host, float* y_host,
                             void* workspace, size_t workspace_bytes, pn_stream stream);

/*
 * pn_gemv_noalloc: pn_gemv for callers that cannot allocate device memory --
 * code running where cudaMalloc is not allowed (a host callback, a stream
 * owned by another runtime), a plugin whose host framework owns every
 * allocation, or a serving loop that must not touch the allocator once the
 * model is loaded.  (The pages have no counterpart: this entry point only
 * changes where the scratch memory comes from.)  Same arguments, layouts,
 * results and alignment rules as pn_gemv; no workspace argument.
 *
 * Scratch: a fixed 512 KiB array in the library's device image, which every
 * GPU that loads the library holds until the process exits.  A device whose
 * workspace (pn_workspace_bytes) would not fit (more than 226 SMs) gets
 * PN_EINVAL and nothing is launched.  The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress, which may load the
 * library's device module); make that first call before capturing a stream
 * into a CUDA graph.  The address is kept for the life of the process: after
 * cudaDeviceReset on a device, do not call pn_gemv_noalloc on that device
 * again (the array may have moved).  Arguments are checked first, exactly as
 * pn_gemv checks them; a refused call enqueues nothing.  Every call shares the
 * array and it keeps the last call's contents: each call that launches a
 * tensor-core kernel first clears, on `stream`, the parts that must start at
 * zero.  Calls whose executions overlap on the GPU (other streams, other host
 * threads) race on the array and give wrong results; order them on one
 * stream.  A device-side wait that gives up (see pn_set_wait_timeout_ns)
 * leaves the outputs undefined and, unlike pn_gemv, cannot be read back.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
pn_status pn_gemv_noalloc(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int M,
                          float* y, pn_stream stream);

/*
 * pn_hadamard: the runtime Hadamard rotation of the activations that reach the
 * PN weights (tensorless docs, "Why a P100-native weight format", section "How
 * Qwen3.8-27B-PN3 uses it"; the page gives no size or normalisation, read
 * here as follows).  Every run of `block` consecutive activations of each of
 * the M rows of x (fp16 [M][K]) is multiplied by the orthonormal Sylvester
 * Hadamard matrix H_block / sqrt(block) (H_1 = [1], H_2n = [[H, H], [H, -H]]),
 * written to out (fp16 [M][K]; out may equal x, otherwise the two must not
 * overlap).  block is a power of two, 2 <= block <= 4096, dividing K;
 * 1 <= M <= 65535.  Arithmetic, fixed so results are reproducible bit for
 * bit: fp16 -> fp32; butterfly stages h = 1, 2, ..., block/2 in that order,
 * each replacing (v[i], v[i+h]) for (i & h) == 0 by (v[i] + v[i+h],
 * v[i] - v[i+h]) in fp32; one fp32 multiply by 2^(-m/2) (block = 2^m, m even)
 * or 2^(-(m+1)/2) * fp32(sqrt 2) (m odd); fp16 round-to-nearest-even.  x and
 * out 2-byte aligned.  Asynchronous on `stream`; a following pn_gemv on the
 * same stream reads the rotated activations.
 */
pn_status pn_hadamard(const uint16_t* x, int M, int64_t K, int block, uint16_t* out, pn_stream stream);

/*
 * pn_gemv_hadamard / pn_gemv_layer_hadamard: pn_gemv / pn_gemv_layer on the
 * activations rotated as pn_hadamard rotates them (runs of `block`, same
 * arithmetic, so the multiplied fp16 values are exactly pn_hadamard's
 * output), in one launch: the rotation is fused into the GEMV (tensorless
 * docs, "How Qwen3.8-27B-PN3 uses it": the engine applies the rotation at
 * run time).  x is read, not modified.  Limits of the fused path: 1 <= M <= 2;
 * block a power of two from 32 to 1024 dividing every K (else PN_EINVAL);
 * the tensor-core alignment rules and rows of at most 64 chunks of 8 blocks
 * (else PN_EALIGN / PN_EUNSUPPORTED); the rotated activations of the tensors
 * one SM works on must fit its shared memory (about 70 K activations per
 * token pair; else PN_EUNSUPPORTED).  Outside these limits, call pn_hadamard
 * and then pn_gemv.  Same workspace, result and tolerance as pn_gemv.
 */
pn_status pn_gemv_hadamard(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int M, int block,
                           float* y, void* workspace, size_t workspace_bytes, pn_stream stream);
pn_status pn_gemv_layer_hadamard(const pn_gemv_desc* descs, int count, int M, int block, void* workspace,
                                 size_t workspace_bytes, pn_stream stream);

/*
 * pn_gptq: GPTQ-style quantisation of fp32 weights w [N][K] into PN rows
 * W [N][pn_row_bytes(type, K)] (tensorless docs, "How Qwen3.8-27B-PN3 uses
 * it": the weights were quantised "GPTQ-style").  The published GPTQ
 * (Frantar et al., ICLR 2023, Algorithm 1) with the PN blocks as its groups:
 * H = 2 X^T X + lambda I over calibration inputs X fp32 [n][K] (lambda = damp
 * times the mean of diag(2 X^T X), damp > 0, typically 0.01); U the upper
 * Cholesky factor of H^-1; columns in order, each row's block scale taken by
 * the signed-scale rule from the block's current weights when the block
 * starts, each column rounded with that scale and its error / U[k][k] fed to
 * the later columns through U's row k.  fp64 throughout (fp32 for the scale
 * and the rounding), each sum in index order, so the bytes equal the CPU
 * oracle's.  Synchronous (returns when W is written).  scratch: device,
 * 256-byte aligned, pn_gptq_scratch_bytes(N, K) bytes (4 K^2 + N K doubles).
 * w and X 4-byte aligned, W any alignment.  K at most 65536.  PN_EINVAL for
 * bad sizes, a small scratch, or a Hessian that is not positive definite;
 * N = 0 does nothing.
 * Not part of the GEMV's path: an offline tool, quadratic in K.
 */
size_t pn_gptq_scratch_bytes(int64_t N, int64_t K);
pn_status pn_gptq(int type, const float* w, int64_t N, int64_t K, const float* X, int64_t n, double damp,
                  void* W, void* scratch, size_t scratch_bytes, pn_stream stream);

/*
 * Prefill (large M).  The pages' engine dequantizes the weights for prefill
 * and runs a chunked GEMM, rebuilding weights transiently from the packed
 * codes without keeping them (tensorless docs, "What the fork adds";
 * v100-skinny README, "How QPN works").  Reading taken here: each rebuilt
 * weight is the exact decode d * (n - z) rounded once to fp16 (nearest, ties
 * to even; beyond the fp16 range +-inf), and the GEMM multiplies fp16 by fp16
 * exactly and accumulates in fp32 (on the tcgen05 tensor cores).
 *
 * pn_unpack_f16: PN rows W [N][row_bytes] -> fp16 w16 [N][K] as above.  W
 * 2-byte and w16 4-byte aligned; they must not overlap.
 *
 * pn_gemm_f16: y[m * ldy + r] = sum_k w16[r][k] * x[m][k] for r < N, m < M
 * (w16 fp16 [N][K], x fp16 [M][K], y fp32 rows of ldy >= N floats).  w16 and
 * x 16-byte aligned, K a positive multiple of 8, y 4-byte aligned and not
 * overlapping w16 or x; 1 <= M < 2^31, N <= 8,388,480.  The workspace is the
 * GEMV's (pn_workspace_bytes); only its status word is used, which records
 * PN_ETIMEOUT if a device-side wait gives up (read with pn_workspace_status).
 * Each output sums its K products in fp32 in K order, 16 at a time; it is
 * within (K/16 + 16) * 2^-24 * sum_k |w16 x| + 1e-6 of the exact sum.
 *
 * pn_prefill: the whole path, y[m][r] = sum_k w16[r][k] x[m][k] for the PN
 * tensor W [N][row_bytes]: the rows are rebuilt chunk by chunk into `scratch`
 * (fp16, caller-owned, 16-byte aligned; a chunk is the largest multiple of
 * 128 rows that fits, at least 128 rows = 256 K bytes) and multiplied by x;
 * y is fp32 [M][N].  Same alignment rules as pn_gemm_f16; all launches are
 * asynchronous on `stream`, in order, so scratch is reused safely.
 */
pn_status pn_unpack_f16(int type, const void* W, int64_t N, int64_t K, uint16_t* w16, pn_stream stream);
pn_status pn_gemm_f16(const uint16_t* w16, int64_t N, int64_t K, const uint16_t* x, int64_t M, float* y,
                      int64_t ldy, void* workspace, size_t workspace_bytes, pn_stream stream);
pn_status pn_prefill(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int64_t M, float* y,
                     void* scratch, size_t scratch_bytes, void* workspace, size_t workspace_bytes,
                     pn_stream stream);

/*
 * pn_read_ranges (diagnostic): the plain read-bandwidth ceiling a GEMV is
 * measured against.  Reads the first floor(bytes[i] / 16) * 16 bytes of each
 * of `count` (1 .. PN_MAX_LAYER) device ranges ptrs[i] once, with 16-byte
 * loads, and XORs the 32-bit words read into sink[i] (device, `count` words;
 * zero them first if the value matters).  ptrs and bytes are host arrays
 * read during the call; every ptrs[i] 16-byte aligned, sink 4-byte aligned.
 */
pn_status pn_read_ranges(const void* const* ptrs, const size_t* bytes, int count, uint32_t* sink,
                         pn_stream stream);

/*
 * Testing aid: the time limit, in nanoseconds, of every device-side wait in
 * the tensor-core GEMV kernels and the prefill GEMM (default 1e9).  A wait that runs out stops its thread
 * block, which records PN_ETIMEOUT in the workspace status word and returns
 * after its outstanding copies land.  Process-wide; not for concurrent use.
 */
void pn_set_wait_timeout_ns(uint64_t ns);

/*
 * Testing aid for the failure path: while on (non-zero), every thread block of
 * the tensor-core GEMV kernels and of the prefill GEMM announces the bytes of
 * its first step but never copies them, so its consumers' wait can only end
 * by timing out; the call then reports PN_ETIMEOUT through
 * pn_workspace_status and its outputs are undefined.  Off by default.
 * Process-wide; not for concurrent use.
 */
void pn_set_test_stall(int on);

/*
 * Testing aid (host only; needs no device): the work split the tensor-core
 * GEMV kernel for 3 <= M <= 16 would use for a pn_gemv_layer call on
 * tensors of these types and shapes on a GPU with num_sms SMs.  types, N
 * and K are host arrays of `count` (1 .. PN_MAX_LAYER) entries; every N >= 1
 * and every K a positive multiple of 8 blocks (640 for pn3t, 512 for pn4t),
 * else PN_EINVAL.  Units are numbered over the tensors in order, each
 * tensor's 16-row tiles in turn and each tile's 8-block chunks within it.
 * On PN_OK, *grid is the number of thread blocks and block c takes units
 * [starts[c], starts[c + 1]) (starts: host array of at least num_sms + 1
 * entries; starts[0] = 0, starts[*grid] = all units).  Every range holds at
 * least one whole tile's units, so a tile has at most two owners; the split
 * depends only on the arguments.
 */
pn_status pn_tc_split(const int* types, const int64_t* N, const int64_t* K, int count, int M, int num_sms,
                      uint32_t* starts, int* grid);

#ifdef __cplusplus
}
#endif

#endif /* PN_H */
