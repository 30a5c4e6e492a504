// pn_capi.cu -- the C ABI declared in include/pn.h: argument checks, kernel choice, launches.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/pn.h"
#include "pn_internal.h"

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_cc_major[kMaxDevices];
std::atomic<uint64_t> g_timeout_ns{1000000000ull};
std::atomic<int> g_test_stall{0};
thread_local cudaError_t g_last_cuda_error = cudaSuccess;   // behind this thread's last PN_ECUDA

int per_block(int type) { return type == PN_TYPE_PN3T ? 80 : (type == PN_TYPE_PN4T ? 64 : 0); }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

}  // namespace

namespace pn {
pn_status cuda_error(cudaError_t e) {
    g_last_cuda_error = e;
    cudaGetLastError();             // clear it (a sticky error stays regardless)
    return PN_ECUDA;
}

WorkspaceLayout workspace_layout(int num_sms) {
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    WorkspaceLayout L;
    L.status = 0;
    L.tagged = 256;
    L.partials = up(L.tagged + stream_tagged_bytes(num_sms));
    L.counters = up(L.partials + tc_partial_bytes(num_sms));
    L.total = up(L.counters + static_cast<size_t>(tc_max_ctas(num_sms) + 1) * sizeof(uint32_t));
    return L;
}
}  // namespace pn

namespace {

// SM count and compute-capability major of the current device (cached).
pn_status device_info(int* sms, int* major) {
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return pn::cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return PN_EUNSUPPORTED;
    int s = g_sm_count[dev].load(std::memory_order_relaxed);
    int m = g_cc_major[dev].load(std::memory_order_relaxed);
    if (s <= 0) {
        cudaError_t e = cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m, cudaDevAttrComputeCapabilityMajor, dev);
        if (e != cudaSuccess) return pn::cuda_error(e);
        g_cc_major[dev].store(m, std::memory_order_relaxed);
        g_sm_count[dev].store(s, std::memory_order_relaxed);
    }
    *sms = s;
    *major = m;
    return PN_OK;
}

// Shared checks of one GEMV operand set; fills `t`.
pn_status check_tensor(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int M,
                       float* y, pn::GemvTensor* t) {
    const int bpb = per_block(type);
    if (bpb == 0 || K <= 0 || K % bpb != 0 || N < 0) return PN_EINVAL;
    if (M < 1 || M > PN_MAX_M) return PN_EINVAL;
    const int64_t nb = K / bpb;
    if (N > INT32_MAX / 2 || nb > INT32_MAX / 8 || K > INT32_MAX / PN_MAX_M) return PN_EINVAL;
    if (N > 0 && (!W || !x || !y)) return PN_EINVAL;
    if (!aligned(W, 2) || !aligned(x, 2) || !aligned(y, 4)) return PN_EALIGN;
    const size_t wbytes = static_cast<size_t>(N) * nb * PN_BLOCK_BYTES;
    const size_t xbytes = static_cast<size_t>(M) * K * 2, ybytes = static_cast<size_t>(M) * N * 4;
    if (N > 0 && (overlaps(y, ybytes, W, wbytes) || overlaps(y, ybytes, x, xbytes))) return PN_EINVAL;
    t->W = static_cast<const uint8_t*>(W);
    t->x = x;
    t->y = y;
    t->type = type;
    t->N = static_cast<int>(N);
    t->nb = static_cast<int>(nb);
    return PN_OK;
}

bool tc_eligible(const pn::GemvTensor& t) {
    return t.nb % 8 == 0 && aligned(t.W, 16) && aligned(t.x, 16);
}

// Sorts the tensors of a call into the tensor-core and CUDA-core kernels.
pn_status route(const pn::GemvTensor* ts, int count, int algo, int major, pn::GemvTensor* tc, int* ntc,
                pn::GemvTensor* simt, int* nsimt) {
    if (algo != PN_ALGO_AUTO && algo != PN_ALGO_TENSOR_CORE && algo != PN_ALGO_CUDA_CORE &&
        algo != PN_ALGO_CUDA_CORE_STAGED)
        return PN_EINVAL;
    *ntc = *nsimt = 0;
    for (int e = 0; e < count; ++e) {
        if (ts[e].N == 0) continue;
        const bool ok_tc = tc_eligible(ts[e]) && major >= 10;
        if ((algo == PN_ALGO_TENSOR_CORE || algo == PN_ALGO_CUDA_CORE_STAGED) && !ok_tc)
            return major >= 10 ? PN_EALIGN : PN_EUNSUPPORTED;
        if (algo == PN_ALGO_CUDA_CORE_STAGED && ts[e].nb / 8 > pn::ffma_max_chunks()) return PN_EUNSUPPORTED;
        if (algo != PN_ALGO_CUDA_CORE && ok_tc) tc[(*ntc)++] = ts[e];
        else simt[(*nsimt)++] = ts[e];
    }
    return PN_OK;
}

pn_status run_layer(const pn::GemvTensor* ts, int count, int M, void* ws, size_t ws_bytes, int algo,
                    cudaStream_t s) {
    int sms = 0, major = 0;
    pn_status st = device_info(&sms, &major);
    if (st != PN_OK) return st;
    pn::GemvTensor tc[pn::kMaxLayer];
    pn::GemvTensor simt[pn::kMaxLayer];
    int ntc = 0, nsimt = 0;
    if ((st = route(ts, count, algo, major, tc, &ntc, simt, &nsimt)) != PN_OK) return st;
    if (algo == PN_ALGO_CUDA_CORE_STAGED) {
        if (M > 8) return PN_EUNSUPPORTED;
        if (ntc == 0) return PN_OK;
        if (!ws || !aligned(ws, 256)) return PN_EINVAL;
        if (pn::workspace_layout(sms).total > ws_bytes) return PN_EINVAL;
        uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws));
        const cudaError_t e = pn::launch_gemv_ffma(tc, ntc, M, status, sms, g_timeout_ns.load(), s);
        return e == cudaSuccess ? PN_OK : pn::cuda_error(e);
    }
    if (ntc > 0) {
        if (!ws || !aligned(ws, 256)) return PN_EINVAL;
        const pn::WorkspaceLayout L = pn::workspace_layout(sms);
        if (L.total > ws_bytes) return PN_EINVAL;
        uint8_t* base = static_cast<uint8_t*>(ws);
        uint32_t* status = reinterpret_cast<uint32_t*>(base + L.status);
        // one or two tokens: one block per SM streams a range of units (rows of
        // at most stream_max_chunks() chunks); more tokens or longer rows:
        // thread blocks share each staged activation chunk among eight tiles
        bool stream = M <= 2;
        for (int i = 0; i < ntc; ++i) stream = stream && tc[i].nb / 8 <= pn::stream_max_chunks();
        // two tokens over several tensors: the one-token kernel only where it
        // keeps their activations resident (measured on GB300: 16.3 against
        // 20.5 us on two pn3t tensors whose activations fit; 37.9 against
        // 38.0 and 48.9 against 41.8 us on sets that do not fit, the
        // 27B-class layer the latter)
        if (stream && M == 2 && ntc > 1 && !pn::stream_resident_fits(tc, ntc, M, sms)) stream = false;
        cudaError_t e = stream
            ? pn::launch_gemv_stream(tc, ntc, M, status, reinterpret_cast<uint64_t*>(base + L.tagged), sms,
                                     g_timeout_ns.load(), g_test_stall.load(), s)
            : pn::launch_gemv_tc(tc, ntc, M, status, reinterpret_cast<float*>(base + L.partials),
                                 reinterpret_cast<uint32_t*>(base + L.counters), sms, g_timeout_ns.load(),
                                 g_test_stall.load(), s);
        if (e != cudaSuccess) return pn::cuda_error(e);
    }
    for (int i = 0; i < nsimt; ++i)
        if (cudaError_t e = pn::launch_gemv_simt(simt[i], M, s); e != cudaSuccess) return pn::cuda_error(e);
    return PN_OK;
}

// No output of a layer call may overlap another entry's operands or output.
pn_status check_layer_overlaps(const pn_gemv_desc* descs, int count, int M) {
    for (int a = 0; a < count; ++a) {
        if (descs[a].N == 0) continue;
        const size_t ya = static_cast<size_t>(M) * descs[a].N * 4;
        for (int b = 0; b < count; ++b) {
            if (b == a || descs[b].N == 0) continue;
            const int bpb = per_block(descs[b].type);
            const size_t wb = static_cast<size_t>(descs[b].N) * (descs[b].K / bpb) * PN_BLOCK_BYTES;
            const size_t xb = static_cast<size_t>(M) * descs[b].K * 2;
            const size_t yb = static_cast<size_t>(M) * descs[b].N * 4;
            if (overlaps(descs[a].y, ya, descs[b].W, wb) || overlaps(descs[a].y, ya, descs[b].x, xb) ||
                overlaps(descs[a].y, ya, descs[b].y, yb))
                return PN_EINVAL;
        }
    }
    return PN_OK;
}

// Checks shared by pn_gemm_f16 and pn_prefill (w16 is the fp16 operand: the
// caller's matrix or the scratch chunk).
pn_status check_gemm(int64_t N, int64_t K, const void* x, int64_t M, const float* y, int64_t ldy,
                     void* workspace, size_t workspace_bytes, int* sms, int* major) {
    if (N < 0 || K <= 0 || K % 8 != 0 || K > INT32_MAX || M < 1 || M > INT32_MAX || ldy < N) return PN_EINVAL;
    if (N > 65535LL * 128) return PN_EINVAL;
    if (N == 0) return PN_OK;
    if (!x || !y || !workspace) return PN_EINVAL;
    if (!aligned(x, 16) || !aligned(y, 4)) return PN_EALIGN;
    if (!aligned(workspace, 256)) return PN_EINVAL;
    pn_status st = device_info(sms, major);
    if (st != PN_OK) return st;
    if (*major < 10) return PN_EUNSUPPORTED;
    if (pn::workspace_layout(*sms).total > workspace_bytes) return PN_EINVAL;
    const size_t ybytes = (static_cast<size_t>(M - 1) * ldy + N) * 4;
    if (overlaps(y, ybytes, x, static_cast<size_t>(M) * K * 2)) return PN_EINVAL;
    return PN_OK;
}

}  // namespace

extern "C" {

int pn_abi_version(void) { return 1; }

const char* pn_status_string(pn_status s) {
    switch (s) {
        case PN_OK: return "ok";
        case PN_EINVAL: return "invalid argument";
        case PN_EALIGN: return "misaligned pointer";
        case PN_EUNSUPPORTED: return "unsupported on this device or build";
        case PN_ECUDA: return "CUDA error";
        case PN_ETIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

int pn_weights_per_block(int type) { return per_block(type); }

size_t pn_row_bytes(int type, int64_t K) {
    const int bpb = per_block(type);
    if (bpb == 0 || K <= 0 || K % bpb != 0) return 0;
    return static_cast<size_t>(K / bpb) * PN_BLOCK_BYTES;
}

pn_status pn_pack(int type, const float* w, int64_t N, int64_t K, void* W, pn_stream stream) {
    const int bpb = per_block(type);
    if (bpb == 0 || K <= 0 || K % bpb != 0 || N < 0) return PN_EINVAL;
    if (N == 0) return PN_OK;
    if (!w || !W) return PN_EINVAL;
    if (!aligned(w, 4) || !aligned(W, 2)) return PN_EALIGN;
    if (overlaps(w, static_cast<size_t>(N) * K * 4, W, static_cast<size_t>(N) * (K / bpb) * PN_BLOCK_BYTES))
        return PN_EINVAL;
    const cudaError_t e = pn::launch_pack(type, w, N, K / bpb, W, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PN_OK : pn::cuda_error(e);
}

pn_status pn_unpack(int type, const void* W, int64_t N, int64_t K, float* w, pn_stream stream) {
    const int bpb = per_block(type);
    if (bpb == 0 || K <= 0 || K % bpb != 0 || N < 0) return PN_EINVAL;
    if (N == 0) return PN_OK;
    if (!w || !W) return PN_EINVAL;
    if (!aligned(w, 4) || !aligned(W, 2)) return PN_EALIGN;
    if (overlaps(w, static_cast<size_t>(N) * K * 4, W, static_cast<size_t>(N) * (K / bpb) * PN_BLOCK_BYTES))
        return PN_EINVAL;
    const cudaError_t e = pn::launch_unpack(type, W, N, K / bpb, w, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PN_OK : pn::cuda_error(e);
}

size_t pn_workspace_bytes(int64_t total_rows) {
    int sms = 0, major = 0;
    if (total_rows < 0 || device_info(&sms, &major) != PN_OK) return 0;
    return pn::workspace_layout(sms).total;
}

pn_status pn_workspace_init(void* workspace, size_t workspace_bytes, pn_stream stream) {
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < 256) return PN_EINVAL;
    const cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PN_OK : pn::cuda_error(e);
}

pn_status pn_workspace_status(void* workspace, size_t workspace_bytes, pn_stream stream) {
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < 256) return PN_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return pn::cuda_error(e);
    if (word == 0) return PN_OK;
    if (cudaError_t e2 = cudaMemset(workspace, 0, workspace_bytes); e2 != cudaSuccess) return pn::cuda_error(e2);
    return word == PN_ETIMEOUT ? PN_ETIMEOUT : PN_ECUDA;
}

}  // extern "C"

namespace pn {
pn_status gemv_check(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int M, float* y,
                     int algo, bool* uses_workspace) {
    *uses_workspace = false;
    pn::GemvTensor t{};
    pn_status st = check_tensor(type, W, N, K, x, M, y, &t);
    if (st != PN_OK || N == 0) return st;
    int sms = 0, major = 0;
    if ((st = device_info(&sms, &major)) != PN_OK) return st;
    pn::GemvTensor tc[1], simt[1];
    int ntc = 0, nsimt = 0;
    if ((st = route(&t, 1, algo, major, tc, &ntc, simt, &nsimt)) != PN_OK) return st;
    *uses_workspace = ntc > 0;
    return PN_OK;
}
}  // namespace pn

extern "C" {

pn_status pn_gemv_ex(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int M,
                     float* y, void* workspace, size_t workspace_bytes, int algo, pn_stream stream) {
    pn::GemvTensor t{};
    pn_status st = check_tensor(type, W, N, K, x, M, y, &t);
    if (st != PN_OK) return st;
    if (N == 0) return PN_OK;
    return run_layer(&t, 1, M, workspace, workspace_bytes, algo, reinterpret_cast<cudaStream_t>(stream));
}

pn_status pn_gemv(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int M,
                  float* y, void* workspace, size_t workspace_bytes, pn_stream stream) {
    return pn_gemv_ex(type, W, N, K, x, M, y, workspace, workspace_bytes, PN_ALGO_AUTO, stream);
}

pn_status pn_gemv_layer_ex(const pn_gemv_desc* descs, int count, int M, void* workspace,
                           size_t workspace_bytes, int algo, pn_stream stream) {
    if (!descs || count < 1 || count > PN_MAX_LAYER) return PN_EINVAL;
    pn::GemvTensor ts[pn::kMaxLayer];
    for (int e = 0; e < count; ++e) {
        const pn_gemv_desc& d = descs[e];
        pn_status st = check_tensor(d.type, d.W, d.N, d.K, d.x, M, d.y, &ts[e]);
        if (st != PN_OK) return st;
    }
    if (pn_status st = check_layer_overlaps(descs, count, M); st != PN_OK) return st;
    return run_layer(ts, count, M, workspace, workspace_bytes, algo, reinterpret_cast<cudaStream_t>(stream));
}

pn_status pn_gemv_layer(const pn_gemv_desc* descs, int count, int M, void* workspace,
                        size_t workspace_bytes, pn_stream stream) {
    return pn_gemv_layer_ex(descs, count, M, workspace, workspace_bytes, PN_ALGO_AUTO, stream);
}

pn_status pn_gemv_layer_host(const pn_gemv_desc* descs, int count, int M, const uint16_t* x_host, float* y_host,
                             void* workspace, size_t workspace_bytes, pn_stream stream) {
    if (!descs || count < 1 || count > PN_MAX_LAYER || !x_host || !y_host) return PN_EINVAL;
    pn::GemvTensor ts[pn::kMaxLayer];
    for (int e = 0; e < count; ++e) {
        const pn_gemv_desc& d = descs[e];
        pn_status st = check_tensor(d.type, d.W, d.N, d.K, d.x, M, d.y, &ts[e]);
        if (st != PN_OK) return st;
    }
    if (pn_status st = check_layer_overlaps(descs, count, M); st != PN_OK) return st;
    int sms = 0, major = 0;
    if (pn_status st = device_info(&sms, &major); st != PN_OK) return st;
    if (!workspace || !aligned(workspace, 256) || pn::workspace_layout(sms).total > workspace_bytes)
        return PN_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // one copy per run of entries whose device buffers follow each other (the
    // host buffers always do)
    auto copy_runs = [&](bool in) -> cudaError_t {
        size_t host_off = 0, run_host = 0, run_bytes = 0;
        uint8_t* run_dev = nullptr;
        auto flush = [&]() -> cudaError_t {
            if (!run_bytes) return cudaSuccess;
            return in ? cudaMemcpyAsync(run_dev, reinterpret_cast<const uint8_t*>(x_host) + run_host, run_bytes,
                                        cudaMemcpyHostToDevice, s)
                      : cudaMemcpyAsync(reinterpret_cast<uint8_t*>(y_host) + run_host, run_dev, run_bytes,
                                        cudaMemcpyDeviceToHost, s);
        };
        for (int e = 0; e < count; ++e) {
            const pn_gemv_desc& d = descs[e];
            const size_t bytes = in ? static_cast<size_t>(M) * d.K * 2 : static_cast<size_t>(M) * d.N * 4;
            uint8_t* dev = in ? reinterpret_cast<uint8_t*>(const_cast<uint16_t*>(d.x)) : reinterpret_cast<uint8_t*>(d.y);
            if (d.N > 0 && bytes > 0) {
                if (run_bytes && dev == run_dev + run_bytes && host_off == run_host + run_bytes) {
                    run_bytes += bytes;
                } else {
                    if (cudaError_t e2 = flush(); e2 != cudaSuccess) return e2;
                    run_dev = dev;
                    run_host = host_off;
                    run_bytes = bytes;
                }
            }
            host_off += bytes;
        }
        return flush();
    };
    if (cudaError_t e = copy_runs(true); e != cudaSuccess) return pn::cuda_error(e);
    if (pn_status st = run_layer(ts, count, M, workspace, workspace_bytes, PN_ALGO_AUTO, s); st != PN_OK) return st;
    if (cudaError_t e = copy_runs(false); e != cudaSuccess) return pn::cuda_error(e);
    if (cudaError_t e = cudaStreamSynchronize(s); e != cudaSuccess) return pn::cuda_error(e);
    return PN_OK;
}

}  // extern "C"

namespace {

// GEMVs of `count` checked tensors on their activations rotated by blocks of
// `block` (pn_hadamard's arithmetic), in one launch of the one-/two-token
// kernel, which keeps the rotated activations in shared memory.
pn_status run_rotated(const pn::GemvTensor* ts, int count, int M, int block, void* ws, size_t ws_bytes,
                      cudaStream_t s) {
    if (block < 32 || block > 1024 || (block & (block - 1))) return PN_EINVAL;
    for (int e = 0; e < count; ++e)
        if ((static_cast<int64_t>(ts[e].nb) * per_block(ts[e].type)) % block) return PN_EINVAL;
    int sms = 0, major = 0;
    pn_status st = device_info(&sms, &major);
    if (st != PN_OK) return st;
    pn::GemvTensor live[pn::kMaxLayer];
    int n = 0;
    for (int e = 0; e < count; ++e) {
        if (ts[e].N == 0) continue;
        if (major < 10) return PN_EUNSUPPORTED;
        if (!tc_eligible(ts[e])) return PN_EALIGN;
        if (ts[e].nb / 8 > pn::stream_max_chunks()) return PN_EUNSUPPORTED;
        live[n++] = ts[e];
    }
    if (M > 2) return PN_EUNSUPPORTED;
    if (n == 0) return PN_OK;
    if (!pn::stream_rotation_fits(live, n, M, sms, block)) return PN_EUNSUPPORTED;
    if (!ws || !aligned(ws, 256)) return PN_EINVAL;
    const pn::WorkspaceLayout L = pn::workspace_layout(sms);
    if (L.total > ws_bytes) return PN_EINVAL;
    uint8_t* base = static_cast<uint8_t*>(ws);
    const cudaError_t e = pn::launch_gemv_stream(live, n, M, reinterpret_cast<uint32_t*>(base + L.status),
                                                 reinterpret_cast<uint64_t*>(base + L.tagged), sms,
                                                 g_timeout_ns.load(), g_test_stall.load(), s, block);
    return e == cudaSuccess ? PN_OK : pn::cuda_error(e);
}

}  // namespace

extern "C" {

pn_status pn_gemv_hadamard(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int M, int block,
                           float* y, void* workspace, size_t workspace_bytes, pn_stream stream) {
    pn::GemvTensor t{};
    pn_status st = check_tensor(type, W, N, K, x, M, y, &t);
    if (st != PN_OK) return st;
    return run_rotated(&t, 1, M, block, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

pn_status pn_gemv_layer_hadamard(const pn_gemv_desc* descs, int count, int M, int block, void* workspace,
                                 size_t workspace_bytes, pn_stream stream) {
    if (!descs || count < 1 || count > PN_MAX_LAYER) return PN_EINVAL;
    pn::GemvTensor ts[pn::kMaxLayer];
    for (int e = 0; e < count; ++e) {
        const pn_gemv_desc& d = descs[e];
        pn_status st = check_tensor(d.type, d.W, d.N, d.K, d.x, M, d.y, &ts[e]);
        if (st != PN_OK) return st;
    }
    if (pn_status st = check_layer_overlaps(descs, count, M); st != PN_OK) return st;
    return run_rotated(ts, count, M, block, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

pn_status pn_hadamard(const uint16_t* x, int M, int64_t K, int block, uint16_t* out, pn_stream stream) {
    if (M < 1 || M > 65535 || K <= 0 || block < 2 || block > 4096 || (block & (block - 1)) || K % block)
        return PN_EINVAL;
    if (!x || !out) return PN_EINVAL;
    if (!aligned(x, 2) || !aligned(out, 2)) return PN_EALIGN;
    const size_t bytes = static_cast<size_t>(M) * static_cast<size_t>(K) * 2;
    if (x != out && overlaps(x, bytes, out, bytes)) return PN_EINVAL;
    if (K / block > INT32_MAX) return PN_EINVAL;
    const cudaError_t e = pn::launch_hadamard(x, M, K, block, out, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PN_OK : pn::cuda_error(e);
}

pn_status pn_unpack_f16(int type, const void* W, int64_t N, int64_t K, uint16_t* w16, pn_stream stream) {
    const int bpb = per_block(type);
    if (bpb == 0 || K <= 0 || K % bpb != 0 || N < 0) return PN_EINVAL;
    if (N == 0) return PN_OK;
    if (!W || !w16) return PN_EINVAL;
    if (!aligned(W, 2) || !aligned(w16, 4)) return PN_EALIGN;
    if (overlaps(w16, static_cast<size_t>(N) * K * 2, W, static_cast<size_t>(N) * (K / bpb) * PN_BLOCK_BYTES))
        return PN_EINVAL;
    const cudaError_t e = pn::launch_unpack_f16(type, W, N, K / bpb, w16, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PN_OK : pn::cuda_error(e);
}

pn_status pn_gemm_f16(const uint16_t* w16, int64_t N, int64_t K, const uint16_t* x, int64_t M, float* y,
                      int64_t ldy, void* workspace, size_t workspace_bytes, pn_stream stream) {
    int sms = 0, major = 0;
    pn_status st = check_gemm(N, K, x, M, y, ldy, workspace, workspace_bytes, &sms, &major);
    if (st != PN_OK || N == 0) return st;
    if (!w16) return PN_EINVAL;
    if (!aligned(w16, 16)) return PN_EALIGN;
    const size_t ybytes = (static_cast<size_t>(M - 1) * ldy + N) * 4;
    if (overlaps(y, ybytes, w16, static_cast<size_t>(N) * K * 2)) return PN_EINVAL;
    uint32_t* status = static_cast<uint32_t*>(workspace);
    const cudaError_t e = pn::launch_gemm_f16(w16, N, K, x, M, y, ldy, status, sms, g_timeout_ns.load(),
                                              g_test_stall.load(), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PN_OK : pn::cuda_error(e);
}

pn_status pn_prefill(int type, const void* W, int64_t N, int64_t K, const uint16_t* x, int64_t M, float* y,
                     void* scratch, size_t scratch_bytes, void* workspace, size_t workspace_bytes,
                     pn_stream stream) {
    const int bpb = per_block(type);
    if (bpb == 0 || K <= 0 || K % bpb != 0) return PN_EINVAL;
    int sms = 0, major = 0;
    pn_status st = check_gemm(N, K, x, M, y, N, workspace, workspace_bytes, &sms, &major);
    if (st != PN_OK || N == 0) return st;
    if (!W || !scratch) return PN_EINVAL;
    if (!aligned(W, 2) || !aligned(scratch, 16)) return PN_EALIGN;
    const int tile = pn::gemm_f16_tile_rows();
    int64_t chunk = static_cast<int64_t>(scratch_bytes / (static_cast<size_t>(K) * 2)) / tile * tile;
    if (chunk < tile) return PN_EINVAL;
    if (chunk > N) chunk = N;
    const size_t wbytes = static_cast<size_t>(N) * (K / bpb) * PN_BLOCK_BYTES;
    const size_t ybytes = static_cast<size_t>(M) * N * 4;
    const size_t sbytes = static_cast<size_t>(chunk) * K * 2;
    if (overlaps(y, ybytes, W, wbytes) || overlaps(scratch, sbytes, W, wbytes) ||
        overlaps(scratch, sbytes, x, static_cast<size_t>(M) * K * 2) || overlaps(scratch, sbytes, y, ybytes))
        return PN_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint16_t* w16 = static_cast<uint16_t*>(scratch);
    uint32_t* status = static_cast<uint32_t*>(workspace);
    const int64_t nb = K / bpb;
    const size_t row_bytes = static_cast<size_t>(nb) * PN_BLOCK_BYTES;
    for (int64_t r0 = 0; r0 < N; r0 += chunk) {
        const int64_t rows = N - r0 < chunk ? N - r0 : chunk;
        cudaError_t e = pn::launch_unpack_f16(type, static_cast<const uint8_t*>(W) + r0 * row_bytes, rows, nb, w16, s);
        if (e == cudaSuccess)
            e = pn::launch_gemm_f16(w16, rows, K, x, M, y + r0, N, status, sms, g_timeout_ns.load(),
                                    g_test_stall.load(), s);
        if (e != cudaSuccess) return pn::cuda_error(e);
    }
    return PN_OK;
}

pn_status pn_read_ranges(const void* const* ptrs, const size_t* bytes, int count, uint32_t* sink,
                         pn_stream stream) {
    if (!ptrs || !bytes || !sink || count < 1 || count > PN_MAX_LAYER) return PN_EINVAL;
    for (int e = 0; e < count; ++e) {
        if (!ptrs[e] && bytes[e] >= 16) return PN_EINVAL;
        if (!aligned(ptrs[e], 16)) return PN_EALIGN;
    }
    if (!aligned(sink, 4)) return PN_EALIGN;
    int sms = 0, major = 0;
    pn_status st = device_info(&sms, &major);
    if (st != PN_OK) return st;
    const cudaError_t e = pn::launch_read_ranges(ptrs, bytes, count, sink, sms, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PN_OK : pn::cuda_error(e);
}

const char* pn_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda_error); }

void pn_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns); }

void pn_set_test_stall(int on) { g_test_stall.store(on ? 1 : 0); }

pn_status pn_tc_split(const int* types, const int64_t* N, const int64_t* K, int count, int M, int num_sms,
                      uint32_t* starts, int* grid) {
    if (!types || !N || !K || !starts || !grid) return PN_EINVAL;
    if (count < 1 || count > PN_MAX_LAYER || M < 3 || M > PN_MAX_M || num_sms < 1) return PN_EINVAL;
    pn::GemvTensor ts[pn::kMaxLayer] = {};
    for (int e = 0; e < count; ++e) {
        const int bpb = per_block(types[e]);
        if (bpb == 0 || K[e] <= 0 || K[e] % (8 * bpb) != 0 || N[e] < 1) return PN_EINVAL;
        const int64_t nb = K[e] / bpb;
        if (N[e] > INT32_MAX / 2 || nb > INT32_MAX / 8) return PN_EINVAL;
        ts[e].type = types[e];
        ts[e].N = static_cast<int>(N[e]);
        ts[e].nb = static_cast<int>(nb);
    }
    return pn::tc_split(ts, count, M, num_sms, grid, starts) ? PN_OK : PN_EINVAL;
}

}  // extern "C"
