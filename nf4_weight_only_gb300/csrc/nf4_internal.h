// Launchers shared between the C-ABI layer and the kernel translation units (host side).
#pragma once

#include <cstdint>
#include <cuda_runtime_api.h>

namespace nf4 {

// Each launcher enqueues its kernels on `stream` and returns the result of cudaGetLastError()
// (cudaSuccess when nothing was launched).  Arguments are validated by the caller.
cudaError_t launch_quantize(const float* w, int64_t N, int64_t K, uint8_t* codes, uint16_t* scales,
                            int num_sms, cudaStream_t stream);
cudaError_t launch_dequant(const uint8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                           uint16_t* w_hat, int num_sms, cudaStream_t stream);
// CUDA-core GEMV family: y[M, N] for 1 <= M <= kGemvMaxTokens (measured on the 14B-shaped decode
// pass: at M = 4 the tensor-core small-M kernel is faster, 1354 against 1204 GB/s).
constexpr int kGemvMaxTokens = 3;
cudaError_t launch_gemv(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, uint16_t* y,
                        int64_t M, int64_t N, int64_t K, int num_sms, cudaStream_t stream);

// The same for up to kMaxGroupedLinears linears sharing x and K (concatenated rows, one launch).
constexpr int kMaxGroupedLinears = 8;
cudaError_t launch_gemv_grouped(const uint16_t* x, int count, const uint8_t* const* codes,
                                const uint16_t* const* scales, uint16_t* const* ys, const int64_t* Ns, int64_t M,
                                int64_t K, int num_sms, cudaStream_t stream);

// tcgen05 weight streaming (dequantized tiles in tensor memory) for every M the GEMV does not take:
// y_i[M, N_i] for up to kMaxGroupedLinears linears that share x and K, one launch.
cudaError_t launch_stream(const uint16_t* x, int count, const uint8_t* const* codes, const uint16_t* const* scales,
                          uint16_t* const* ys, const int64_t* Ns, int64_t M, int64_t K, int num_sms,
                          cudaStream_t stream);
// Device error word of the linear kernels (nonzero after a bounded pipeline wait timed out).
cudaError_t read_and_clear_error(int* code);
cudaError_t launch_diag_wait(int64_t ns, cudaStream_t stream);
// Per-wait wall-clock limit of the pipeline waits on the current device (0 = the default, 1 s).
cudaError_t set_wait_limit(int64_t ns, cudaStream_t stream);

// Packed embedding rows (out-of-range ids write zeros and set the embed error word to 41).
cudaError_t launch_embed(const int32_t* ids, int64_t n_ids, const uint8_t* codes, const uint16_t* scales, int64_t V,
                         int64_t K, uint16_t* out, int num_sms, cudaStream_t stream);
cudaError_t read_and_clear_embed_error(int* code);

// The C-ABI layer's device check (an nf4_status value): the current device and its SM count.
int abi_current_device(int* device, int* sms);
// Records a CUDA error for nf4_last_cuda_error (no-op for cudaSuccess).
void note_cuda_error(cudaError_t e);

}  // namespace nf4
