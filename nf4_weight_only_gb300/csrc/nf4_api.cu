// C ABI of libnf4.so: argument checks, the per-device capability check and the M-based dispatch.
#include <atomic>
#include <cstdint>

#include <cuda_runtime_api.h>

#include "../../include/nf4.h"
#include "nf4_internal.h"

namespace nf4 {
int64_t gemv_max_k(int64_t M);
}

namespace {

constexpr int kMaxDevices = 64;

// The last CUDA error this host thread saw inside the library (read by nf4_last_cuda_error).
thread_local cudaError_t g_last_cuda_error = cudaSuccess;
constexpr int64_t kMaxDim = 0x7FFFFFFF;

// Per-device cache: 0 = unknown, -1 = unsupported, otherwise the SM count of a 10.3 device.
std::atomic<int> g_device_sms[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a_bytes > 0 && b_bytes > 0 && a0 < b0 + static_cast<uintptr_t>(b_bytes) &&
           b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

nf4_status check_k(int64_t K) {
    if (K <= 0 || K % NF4_GROUP_SIZE != 0 || K > kMaxDim) return NF4_ERR_SHAPE;
    return NF4_OK;
}

// Current device must be compute capability 10.3; returns its SM count through `sms`.
nf4_status current_device(int* device, int* sms) {
    if (cudaGetDevice(device) != cudaSuccess) {
        g_last_cuda_error = cudaGetLastError();
        return NF4_ERR_CUDA;
    }
    if (*device < 0 || *device >= kMaxDevices) return NF4_ERR_UNSUPPORTED_DEVICE;
    int cached = g_device_sms[*device].load(std::memory_order_relaxed);
    if (cached == 0) {
        int major = 0, minor = 0, count = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *device) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *device) != cudaSuccess ||
            cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, *device) != cudaSuccess) {
            g_last_cuda_error = cudaGetLastError();
            return NF4_ERR_CUDA;
        }
        cached = (major == 10 && minor == 3 && count > 0) ? count : -1;
        g_device_sms[*device].store(cached, std::memory_order_relaxed);
    }
    if (cached < 0) return NF4_ERR_UNSUPPORTED_DEVICE;
    *sms = cached;
    return NF4_OK;
}

nf4_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return NF4_OK;
    g_last_cuda_error = e;
    cudaGetLastError();
    return NF4_ERR_CUDA;
}

}  // namespace

namespace nf4 {
int abi_current_device(int* device, int* sms) { return current_device(device, sms); }
void note_cuda_error(cudaError_t e) {
    if (e != cudaSuccess) g_last_cuda_error = e;
}
}  // namespace nf4

extern "C" {

const char* nf4_status_str(nf4_status status) {
    switch (status) {
        case NF4_OK: return "NF4_OK";
        case NF4_ERR_NULL: return "NF4_ERR_NULL: a required pointer is NULL";
        case NF4_ERR_SHAPE: return "NF4_ERR_SHAPE: bad size (K must be a positive multiple of 64; sizes <= 2^31-1)";
        case NF4_ERR_ALIGN: return "NF4_ERR_ALIGN: a pointer is not 16-byte aligned";
        case NF4_ERR_ALIAS: return "NF4_ERR_ALIAS: an output overlaps an input";
        case NF4_ERR_UNSUPPORTED_DEVICE: return "NF4_ERR_UNSUPPORTED_DEVICE: current device is not sm_103";
        case NF4_ERR_CUDA: return "NF4_ERR_CUDA: a CUDA call or launch failed";
        case NF4_ERR_MEMORY: return "NF4_ERR_MEMORY: host memory not page-locked, or a ring used on another device";
        case NF4_ERR_CAPTURE:
            return "NF4_ERR_CAPTURE: first nf4_linear_host_noalloc call on this device made under stream capture (make one call outside capture first)";
    }
    return "NF4 status: unknown code";
}

int nf4_abi_version(void) { return NF4_ABI_VERSION; }

const char* nf4_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda_error); }

nf4_status nf4_linear_grouped(const uint16_t* x, int64_t M, int64_t K, int count, const uint8_t* const* codes,
                              const uint16_t* const* scales, uint16_t* const* ys, const int64_t* Ns,
                              cudaStream_t stream) {
    if (count < 1 || count > nf4::kMaxGroupedLinears) return NF4_ERR_SHAPE;
    if (!codes || !scales || !ys || !Ns) return NF4_ERR_NULL;
    if (M < 0 || M > kMaxDim) return NF4_ERR_SHAPE;
    nf4_status st = check_k(K);
    if (st != NF4_OK) return st;
    int64_t rows = 0;
    for (int i = 0; i < count; i++) {
        if (Ns[i] < 0 || Ns[i] > kMaxDim) return NF4_ERR_SHAPE;
        rows += Ns[i];
    }
    if (rows > kMaxDim) return NF4_ERR_SHAPE;
    if (M == 0 || rows == 0) return NF4_OK;
    if (!x) return NF4_ERR_NULL;
    if (!aligned16(x)) return NF4_ERR_ALIGN;
    const int64_t xb = M * K * 2;
    for (int i = 0; i < count; i++) {
        if (Ns[i] == 0) continue;
        if (!codes[i] || !scales[i] || !ys[i]) return NF4_ERR_NULL;
        if (!aligned16(codes[i]) || !aligned16(scales[i]) || !aligned16(ys[i])) return NF4_ERR_ALIGN;
    }
    for (int i = 0; i < count; i++) {
        if (Ns[i] == 0) continue;
        const int64_t yb = M * Ns[i] * 2;
        if (overlap(ys[i], yb, x, xb)) return NF4_ERR_ALIAS;
        for (int j = 0; j < count; j++) {
            if (Ns[j] == 0) continue;
            const int64_t cb = Ns[j] * K / 2, sb = Ns[j] * (K / NF4_GROUP_SIZE) * 2;
            if (overlap(ys[i], yb, codes[j], cb) || overlap(ys[i], yb, scales[j], sb)) return NF4_ERR_ALIAS;
            if (j != i && overlap(ys[i], yb, ys[j], M * Ns[j] * 2)) return NF4_ERR_ALIAS;
        }
    }
    int dev = 0, sms = 0;
    if ((st = current_device(&dev, &sms)) != NF4_OK) return st;
    // drop empty problems, keep the order
    const uint8_t* c[nf4::kMaxGroupedLinears];
    const uint16_t* sc[nf4::kMaxGroupedLinears];
    uint16_t* yy[nf4::kMaxGroupedLinears];
    int64_t nn[nf4::kMaxGroupedLinears];
    int k = 0;
    for (int i = 0; i < count; i++)
        if (Ns[i] > 0) {
            c[k] = codes[i];
            sc[k] = scales[i];
            yy[k] = ys[i];
            nn[k] = Ns[i];
            k++;
        }
    if (M <= nf4::kGemvMaxTokens && K <= nf4::gemv_max_k(M))
        return from_cuda(nf4::launch_gemv_grouped(x, k, c, sc, yy, nn, M, K, sms, stream));
    return from_cuda(nf4::launch_stream(x, k, c, sc, yy, nn, M, K, sms, stream));
}

nf4_status nf4_check_device_error(int* code) {
    if (!code) return NF4_ERR_NULL;
    *code = 0;
    int dev = 0, sms = 0;
    nf4_status st = current_device(&dev, &sms);
    if (st != NF4_OK) return st;
    int linear = 0, embed = 0;
    if ((st = from_cuda(nf4::read_and_clear_error(&linear))) != NF4_OK) return st;
    if ((st = from_cuda(nf4::read_and_clear_embed_error(&embed))) != NF4_OK) return st;
    *code = linear ? linear : embed;
    return NF4_OK;
}

nf4_status nf4_diag_bounded_wait(int64_t ns, cudaStream_t stream) {
    if (ns <= 0 || ns > (int64_t{1} << 31)) return NF4_ERR_SHAPE;
    int dev = 0, sms = 0;
    nf4_status st = current_device(&dev, &sms);
    if (st != NF4_OK) return st;
    return from_cuda(nf4::launch_diag_wait(ns, stream));
}

nf4_status nf4_diag_set_wait_limit(int64_t ns, cudaStream_t stream) {
    if (ns < 0 || ns > (int64_t{1} << 36)) return NF4_ERR_SHAPE;
    int dev = 0, sms = 0;
    nf4_status st = current_device(&dev, &sms);
    if (st != NF4_OK) return st;
    return from_cuda(nf4::set_wait_limit(ns, stream));
}

nf4_status nf4_embed(const int32_t* ids, int64_t n_ids, const uint8_t* codes, const uint16_t* scales, int64_t V,
                     int64_t K, uint16_t* out, cudaStream_t stream) {
    if (n_ids < 0 || V < 0 || n_ids > kMaxDim || V > kMaxDim) return NF4_ERR_SHAPE;
    nf4_status st = check_k(K);
    if (st != NF4_OK) return st;
    if (n_ids == 0) return NF4_OK;
    if (!ids || !out || (V > 0 && (!codes || !scales))) return NF4_ERR_NULL;
    if (!aligned16(ids) || !aligned16(out) || (V > 0 && (!aligned16(codes) || !aligned16(scales))))
        return NF4_ERR_ALIGN;
    const int64_t ob = n_ids * K * 2, ib = n_ids * 4, cb = V * K / 2, sb = V * (K / NF4_GROUP_SIZE) * 2;
    if (overlap(out, ob, ids, ib) || overlap(out, ob, codes, cb) || overlap(out, ob, scales, sb)) return NF4_ERR_ALIAS;
    int dev = 0, sms = 0;
    if ((st = current_device(&dev, &sms)) != NF4_OK) return st;
    return from_cuda(nf4::launch_embed(ids, n_ids, codes, scales, V, K, out, sms, stream));
}

nf4_status nf4_quantize(const float* w, int64_t N, int64_t K, uint8_t* codes, uint16_t* scales,
                        cudaStream_t stream) {
    if (N < 0 || N > kMaxDim) return NF4_ERR_SHAPE;
    nf4_status st = check_k(K);
    if (st != NF4_OK) return st;
    if (N == 0) return NF4_OK;
    if (!w || !codes || !scales) return NF4_ERR_NULL;
    if (!aligned16(w) || !aligned16(codes) || !aligned16(scales)) return NF4_ERR_ALIGN;
    const int64_t wb = N * K * 4, cb = N * K / 2, sb = N * (K / NF4_GROUP_SIZE) * 2;
    if (overlap(codes, cb, w, wb) || overlap(scales, sb, w, wb) || overlap(codes, cb, scales, sb))
        return NF4_ERR_ALIAS;
    int dev = 0, sms = 0;
    if ((st = current_device(&dev, &sms)) != NF4_OK) return st;
    return from_cuda(nf4::launch_quantize(w, N, K, codes, scales, sms, stream));
}

nf4_status nf4_dequant(const uint8_t* codes, const uint16_t* scales, int64_t N, int64_t K, uint16_t* w_hat,
                       cudaStream_t stream) {
    if (N < 0 || N > kMaxDim) return NF4_ERR_SHAPE;
    nf4_status st = check_k(K);
    if (st != NF4_OK) return st;
    if (N == 0) return NF4_OK;
    if (!codes || !scales || !w_hat) return NF4_ERR_NULL;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(w_hat)) return NF4_ERR_ALIGN;
    const int64_t ob = N * K * 2, cb = N * K / 2, sb = N * (K / NF4_GROUP_SIZE) * 2;
    if (overlap(w_hat, ob, codes, cb) || overlap(w_hat, ob, scales, sb)) return NF4_ERR_ALIAS;
    int dev = 0, sms = 0;
    if ((st = current_device(&dev, &sms)) != NF4_OK) return st;
    return from_cuda(nf4::launch_dequant(codes, scales, N, K, w_hat, sms, stream));
}

nf4_status nf4_linear(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, uint16_t* y, int64_t M,
                      int64_t N, int64_t K, cudaStream_t stream) {
    if (M < 0 || N < 0 || M > kMaxDim || N > kMaxDim) return NF4_ERR_SHAPE;
    nf4_status st = check_k(K);
    if (st != NF4_OK) return st;
    if (M == 0 || N == 0) return NF4_OK;
    if (!x || !codes || !scales || !y) return NF4_ERR_NULL;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(y)) return NF4_ERR_ALIGN;
    const int64_t yb = M * N * 2, xb = M * K * 2, cb = N * K / 2, sb = N * (K / NF4_GROUP_SIZE) * 2;
    if (overlap(y, yb, x, xb) || overlap(y, yb, codes, cb) || overlap(y, yb, scales, sb)) return NF4_ERR_ALIAS;
    int dev = 0, sms = 0;
    if ((st = current_device(&dev, &sms)) != NF4_OK) return st;
    if (M <= nf4::kGemvMaxTokens && K <= nf4::gemv_max_k(M))
        return from_cuda(nf4::launch_gemv(x, codes, scales, y, M, N, K, sms, stream));
    return from_cuda(nf4::launch_stream(x, 1, &codes, &scales, &y, &N, M, K, sms, stream));
}

}  // extern "C"
