// Overflow streaming: packed weights in page-locked host memory pass through two reusable device
// slots on their way to the linear kernels (deep-fold README, overview and execution-path table:
// a model that does not fit the card keeps part of its weights on the host and copies them into
// two reusable GPU slots, overlapped with the same GEMV / GEMM).
//
// Ordering per linear i, slot s = i mod 2 (host enqueue order; every wait snapshots the event's
// latest record, so two events per role suffice):
//   copy stream:    wait consumed[s]  ->  codes, scales host -> slot s  ->  record filled[s]
//   compute stream: wait filled[s]    ->  linear on slot s             ->  record consumed[s]
// The copy stream runs ahead of the compute stream by at most one slot, so the transfer of linear
// i + 1 overlaps the kernel of linear i.  On a GB300 the host link is NVLink-C2C; one copy engine
// carries the transfers and the kernels read the slot from HBM.
#include <mutex>
#include <new>

#include <cuda_runtime_api.h>

#include "../../include/nf4.h"
#include "nf4_internal.h"

struct nf4_ring {
    int device = -1;
    int64_t slot_bytes = 0;
    uint8_t* slot[2] = {nullptr, nullptr};
    cudaStream_t copy = nullptr;
    cudaEvent_t filled[2] = {nullptr, nullptr};
    cudaEvent_t consumed[2] = {nullptr, nullptr};
    cudaEvent_t fork = nullptr;
    // consumed[s] was last recorded outside a stream capture (an eager run may wait on it)
    bool eager_consumed[2] = {false, false};
    bool captured = false;  // some run was captured into a graph
    int next = 0;
    std::mutex mu;
};

namespace {

constexpr int64_t kMaxDim = 0x7FFFFFFF;
constexpr int64_t kScaleAlign = 256;  // scales start at this alignment inside a slot

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t codes_bytes(const nf4_host_linear& op) { return op.N * op.K / 2; }
int64_t scales_bytes(const nf4_host_linear& op) { return op.N * (op.K / NF4_GROUP_SIZE) * 2; }
int64_t scales_offset(const nf4_host_linear& op) {
    return (codes_bytes(op) + kScaleAlign - 1) / kScaleAlign * kScaleAlign;
}

// First and last byte of [p, p + bytes) are page-locked host memory.
bool pinned_host(const void* p, int64_t bytes) {
    const void* ends[2] = {p, static_cast<const uint8_t*>(p) + bytes - 1};
    for (const void* q : ends) {
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, q) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        if (a.type != cudaMemoryTypeHost) return false;
    }
    return true;
}

nf4_status check_op(const nf4_host_linear& op, int64_t slot_bytes) {
    if (op.M < 0 || op.N < 0 || op.M > kMaxDim || op.N > kMaxDim) return NF4_ERR_SHAPE;
    if (op.K <= 0 || op.K % NF4_GROUP_SIZE != 0 || op.K > kMaxDim) return NF4_ERR_SHAPE;
    if (op.M == 0 || op.N == 0) return NF4_OK;
    if (!op.x || !op.codes || !op.scales || !op.y) return NF4_ERR_NULL;
    if (!aligned16(op.x) || !aligned16(op.codes) || !aligned16(op.scales) || !aligned16(op.y))
        return NF4_ERR_ALIGN;
    if (scales_offset(op) + scales_bytes(op) > slot_bytes) return NF4_ERR_SHAPE;
    const uintptr_t y0 = reinterpret_cast<uintptr_t>(op.y), x0 = reinterpret_cast<uintptr_t>(op.x);
    const uintptr_t yb = static_cast<uintptr_t>(op.M * op.N * 2), xb = static_cast<uintptr_t>(op.M * op.K * 2);
    if (y0 < x0 + xb && x0 < y0 + yb) return NF4_ERR_ALIAS;
    if (!pinned_host(op.codes, codes_bytes(op)) || !pinned_host(op.scales, scales_bytes(op))) return NF4_ERR_MEMORY;
    return NF4_OK;
}

void release(nf4_ring* r) {
    for (int s = 0; s < 2; s++) {
        if (r->slot[s]) cudaFree(r->slot[s]);
        if (r->filled[s]) cudaEventDestroy(r->filled[s]);
        if (r->consumed[s]) cudaEventDestroy(r->consumed[s]);
    }
    if (r->fork) cudaEventDestroy(r->fork);
    if (r->copy) cudaStreamDestroy(r->copy);
    cudaGetLastError();
    delete r;
}

// Restores the caller's current device on scope exit.
struct DeviceScope {
    int saved = -1;
    explicit DeviceScope(int device) {
        if (cudaGetDevice(&saved) != cudaSuccess) {
            cudaGetLastError();
            saved = -1;
        }
        if (saved != device) cudaSetDevice(device);
    }
    ~DeviceScope() {
        if (saved >= 0) cudaSetDevice(saved);
    }
};

}  // namespace

extern "C" {

nf4_status nf4_ring_create(int64_t slot_bytes, nf4_ring** ring) {
    if (!ring) return NF4_ERR_NULL;
    *ring = nullptr;
    if (slot_bytes <= 0) return NF4_ERR_SHAPE;
    int dev = 0, sms = 0;
    nf4_status st = static_cast<nf4_status>(nf4::abi_current_device(&dev, &sms));
    if (st != NF4_OK) return st;
    nf4_ring* r = new (std::nothrow) nf4_ring;
    if (!r) return NF4_ERR_CUDA;
    r->device = dev;
    r->slot_bytes = slot_bytes;
    bool ok = cudaStreamCreateWithFlags(&r->copy, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&r->fork, cudaEventDisableTiming) == cudaSuccess;
    for (int s = 0; s < 2 && ok; s++) {
        ok = cudaMalloc(reinterpret_cast<void**>(&r->slot[s]), static_cast<size_t>(slot_bytes)) == cudaSuccess &&
             cudaEventCreateWithFlags(&r->filled[s], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&r->consumed[s], cudaEventDisableTiming) == cudaSuccess;
    }
    if (!ok) {
        release(r);
        return NF4_ERR_CUDA;
    }
    *ring = r;
    return NF4_OK;
}

nf4_status nf4_ring_run(nf4_ring* r, const nf4_host_linear* ops, int64_t count, cudaStream_t stream) {
    if (!r) return NF4_ERR_NULL;
    if (count < 0) return NF4_ERR_SHAPE;
    if (count == 0) return NF4_OK;
    if (!ops) return NF4_ERR_NULL;
    int dev = 0, sms = 0;
    nf4_status st = static_cast<nf4_status>(nf4::abi_current_device(&dev, &sms));
    if (st != NF4_OK) return st;
    if (dev != r->device) return NF4_ERR_MEMORY;
    for (int64_t i = 0; i < count; i++)
        if ((st = check_op(ops[i], r->slot_bytes)) != NF4_OK) return st;

    std::lock_guard<std::mutex> lock(r->mu);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        nf4::note_cuda_error(cudaGetLastError());
        return NF4_ERR_CUDA;
    }
    const bool capturing = cap == cudaStreamCaptureStatusActive;
    // Under capture the copy stream joins through an event recorded on `stream`; the graph then
    // orders this run's copies after the work captured before it (slots of an earlier run included).
    // Once a run has been captured, eager runs fork the same way, so that their copies follow a
    // replay of that graph on `stream`.
    r->captured = r->captured || capturing;
    if (r->captured && (cudaEventRecord(r->fork, stream) != cudaSuccess ||
                      cudaStreamWaitEvent(r->copy, r->fork, 0) != cudaSuccess)) {
        nf4::note_cuda_error(cudaGetLastError());
        return NF4_ERR_CUDA;
    }
    bool recorded_here[2] = {false, false};
    for (int64_t i = 0; i < count; i++) {
        const nf4_host_linear& op = ops[i];
        if (op.M == 0 || op.N == 0) continue;
        const int s = r->next;
        r->next ^= 1;
        uint8_t* codes = r->slot[s];
        uint16_t* scales = reinterpret_cast<uint16_t*>(r->slot[s] + scales_offset(op));
        const bool wait = capturing ? recorded_here[s] : r->eager_consumed[s];
        bool ok = (!wait || cudaStreamWaitEvent(r->copy, r->consumed[s], 0) == cudaSuccess) &&
                  cudaMemcpyAsync(codes, op.codes, static_cast<size_t>(codes_bytes(op)), cudaMemcpyHostToDevice,
                                  r->copy) == cudaSuccess &&
                  cudaMemcpyAsync(scales, op.scales, static_cast<size_t>(scales_bytes(op)), cudaMemcpyHostToDevice,
                                  r->copy) == cudaSuccess &&
                  cudaEventRecord(r->filled[s], r->copy) == cudaSuccess &&
                  cudaStreamWaitEvent(stream, r->filled[s], 0) == cudaSuccess;
        if (!ok) {
            nf4::note_cuda_error(cudaGetLastError());
            return NF4_ERR_CUDA;
        }
        if ((st = nf4_linear(op.x, codes, scales, op.y, op.M, op.N, op.K, stream)) != NF4_OK) return st;
        if (cudaEventRecord(r->consumed[s], stream) != cudaSuccess) {
            nf4::note_cuda_error(cudaGetLastError());
            return NF4_ERR_CUDA;
        }
        recorded_here[s] = true;
        r->eager_consumed[s] = !capturing;
    }
    return NF4_OK;
}

nf4_status nf4_ring_destroy(nf4_ring* r) {
    if (!r) return NF4_OK;
    DeviceScope scope(r->device);
    nf4_status st = NF4_OK;
    {
        std::lock_guard<std::mutex> lock(r->mu);
        if (cudaStreamSynchronize(r->copy) != cudaSuccess) st = NF4_ERR_CUDA;
        for (int s = 0; s < 2; s++)
            if (r->eager_consumed[s] && cudaEventSynchronize(r->consumed[s]) != cudaSuccess) st = NF4_ERR_CUDA;
    }
    release(r);
    return st;
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// One streamed linear without any allocation: the weights pass through a device array that is part
// of the library image instead of a slot from cudaMalloc.  The array's device address is looked up
// once per device (cudaGetSymbolAddress in host code gives the address for the current device; the
// name alone is a host-side stand-in that no kernel may be given).
// ---------------------------------------------------------------------------------------------
namespace {

static __device__ __align__(256) uint8_t g_noalloc_slot[NF4_NOALLOC_SLOT_BYTES];

constexpr int kMaxSlotDevices = 64;
std::mutex g_noalloc_mu;
uint8_t* g_noalloc_ptr[kMaxSlotDevices] = {};

// Device address of g_noalloc_slot on `device` (the current device), looked up on the first call;
// nullptr on failure.  With `lookup` false it only returns an address found before (or nullptr).
uint8_t* noalloc_slot(int device, bool lookup) {
    if (device < 0 || device >= kMaxSlotDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[device] && lookup) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_slot) != cudaSuccess || !p) {
            cudaGetLastError();
            return nullptr;
        }
        g_noalloc_ptr[device] = static_cast<uint8_t*>(p);
    }
    return g_noalloc_ptr[device];
}

}  // namespace

extern "C" nf4_status nf4_linear_host_noalloc(const uint16_t* x, const uint8_t* codes, const uint16_t* scales,
                                              uint16_t* y, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    const nf4_host_linear op = {x, codes, scales, y, M, N, K};
    nf4_status st = check_op(op, NF4_NOALLOC_SLOT_BYTES);
    if (st != NF4_OK || M == 0 || N == 0) return st;
    int dev = 0, sms = 0;
    if ((st = static_cast<nf4_status>(nf4::abi_current_device(&dev, &sms))) != NF4_OK) return st;
    uint8_t* slot = noalloc_slot(dev, false);
    if (!slot) {
        // First call on this device: the address lookup may load the library's device code, which a
        // capture forbids, so refuse under capture before touching anything.
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
            cudaGetLastError();
            return NF4_ERR_CAPTURE;
        }
        if (cs != cudaStreamCaptureStatusNone) return NF4_ERR_CAPTURE;
        slot = noalloc_slot(dev, true);
        if (!slot) return NF4_ERR_CUDA;
    }
    uint16_t* slot_scales = reinterpret_cast<uint16_t*>(slot + scales_offset(op));
    if (cudaMemcpyAsync(slot, codes, static_cast<size_t>(codes_bytes(op)), cudaMemcpyHostToDevice, stream) !=
            cudaSuccess ||
        cudaMemcpyAsync(slot_scales, scales, static_cast<size_t>(scales_bytes(op)), cudaMemcpyHostToDevice, stream) !=
            cudaSuccess) {
        nf4::note_cuda_error(cudaGetLastError());
        return NF4_ERR_CUDA;
    }
    return nf4_linear(x, slot, slot_scales, y, M, N, K, stream);
}

extern "C" int64_t nf4_noalloc_slot_bytes(void) { return NF4_NOALLOC_SLOT_BYTES; }
