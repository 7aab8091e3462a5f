/*
 * nf4.h - C ABI of the NF4 weight-only linear layer library (libnf4.so, NVIDIA GB300 / sm_103a).
 *
 * Format (deep-fold README, wertick01/deep-fold, format paragraph): weights are stored in groups of
 * 64 consecutive in-features of one output row; each group holds 64 four-bit NF4 codes and one
 * FP16 scale.  NF4 is the 16-value NormalFloat table introduced with QLoRA (deep-fold README,
 * method paragraph; values published by Dettmers et al., 2023).  The library fixes what the pages
 * leave open:
 *   - codes[N][K/2] (uint8): weight (n, 2j) in the low nibble of byte (n, j), weight (n, 2j+1) in
 *     the high nibble;
 *   - scales[N][K/64] (IEEE binary16 bits): scale of group g of row n = fp16 round-to-nearest-even
 *     of s = max |w[n][64g .. 64g+63]| computed in fp32;
 *   - code of w = the index i minimising the fp32 distance |fp32(w / s) - T[i]|, ties to the lower
 *     index; an all-zero group (s = 0) gets code 7 (T[7] = 0);
 *   - dequantized weight w_hat = bf16_rn(fp32(T[code] * float(scale)));
 *   - y[m][n] = bf16_rn(sum_k x[m][k] * w_hat[n][k]) with at least fp32 accumulation.  Accepted
 *     results satisfy |y - y64| <= 2^-8 |y64| + 2^-12 sum_k |x[m][k] w_hat[n][k]|, y64 being the
 *     same sum in exact products and double-precision addition.
 *
 * Common rules for every entry point:
 *   - Pointers are device pointers owned by the caller, row-major and contiguous, each aligned to
 *     16 bytes.  bf16 and fp16 values travel as their 16-bit patterns (uint16_t).
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream).  No call synchronises
 *     the device, allocates memory or keeps state beyond a per-device capability check, except the
 *     ring calls of the overflow-streaming section, which own explicitly created state.
 *   - Arguments are checked on the host before anything is launched; on an error nothing is
 *     launched and no output is written.  A failed launch returns NF4_ERR_CUDA and leaves the CUDA
 *     error state cleared.
 *   - Shapes: N and M may be 0 (nothing is launched, NF4_OK); K must be a positive multiple of 64;
 *     M, N and K must each be at most 2^31 - 1.
 *   - Non-finite inputs are outside the contract: results are unspecified, but no call faults.
 *   - The same inputs give the same output bytes on every call (no atomics, fixed reduction order).
 *   - Every call may be captured into a CUDA graph (the kernels build their constant tables in
 *     shared memory at launch; no call needs one-time device work), except the first call of
 *     nf4_linear_host_noalloc on a device (see there).
 *   - Every pipeline wait inside the kernels is bounded (one second of wall-clock time per wait by
 *     default).  A wait that runs out records a code in the device error word, and the kernel
 *     drains and exits instead of hanging; the call itself has already returned NF4_OK and the
 *     outputs of that launch are then unspecified.  Callers that need to know read the word with
 *     nf4_check_device_error (the tests and the benchmark do after every timed region).
 *   - Every entry point except the ring calls (see their section) may be called from several host
 *     threads at once, on the same or different streams: the only shared state is the per-device
 *     capability cache (atomic) and one-time kernel attributes (std::call_once).
 */
#ifndef NF4_H
#define NF4_H

#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

#define NF4_GROUP_SIZE 64
#define NF4_ABI_VERSION 3

typedef enum nf4_status {
    NF4_OK = 0,
    NF4_ERR_NULL = 1,               /* a required pointer is NULL */
    NF4_ERR_SHAPE = 2,              /* negative size, K not a positive multiple of 64, or > 2^31-1 */
    NF4_ERR_ALIGN = 3,              /* a pointer is not 16-byte aligned */
    NF4_ERR_ALIAS = 4,              /* an output range overlaps an input range */
    NF4_ERR_UNSUPPORTED_DEVICE = 5, /* the current device is not compute capability 10.3 (sm_103) */
    NF4_ERR_CUDA = 6,               /* a CUDA runtime call or kernel launch failed */
    NF4_ERR_MEMORY = 7,             /* memory of the wrong kind: a host pointer that is not page-locked,
                                       or a ring used on a device other than its own */
    NF4_ERR_CAPTURE = 8             /* the first nf4_linear_host_noalloc call on a device was made while
                                       `stream` is being captured into a CUDA graph: its one-time set-up
                                       cannot run inside a capture */
} nf4_status;

/*
 * nf4_quantize - pack fp32 weights into NF4 codes and fp16 group scales.
 * Defines: the format paragraph of the deep-fold README (64-weight groups, 4-bit NF4 codes, one
 * FP16 scale); the pages do this offline in their compressor, here it is a device kernel.
 *   w       in   float [N][K]
 *   codes   out  uint8 [N][K/2]   low nibble first
 *   scales  out  fp16 bits [N][K/64]
 * codes and scales must not overlap w or each other.
 */
nf4_status nf4_quantize(const float* w, int64_t N, int64_t K, uint8_t* codes, uint16_t* scales,
                        cudaStream_t stream);

/*
 * nf4_dequant - expand packed weights to a dense bf16 matrix (a test and inspection entry point:
 * the linear layer below never writes this matrix, as the execution-path table of the deep-fold
 * README requires).
 *   codes   in   uint8 [N][K/2]
 *   scales  in   fp16 bits [N][K/64]
 *   w_hat   out  bf16 bits [N][K], w_hat = bf16_rn(fp32(T[code] * float(scale)))
 */
nf4_status nf4_dequant(const uint8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                       uint16_t* w_hat, cudaStream_t stream);

/*
 * nf4_linear - y = x * w_hat^T with the weights streamed in packed form and dequantized tile by
 * tile on chip (deep-fold README, execution-path table: N=1 decode GEMV, prefill GEMM of up to 32
 * positions; larger M is this library's extension).  M <= 3 runs a CUDA-core GEMV (K up to 32768
 * for M = 1, 16384 for M = 2..3); M <= 32, and M <= 3 with a longer K, run a weight-streaming
 * kernel that dequantizes on the CUDA cores into tensor memory and multiplies on the tcgen05 tensor
 * cores (one CTA per SM, K split into slices when a CTA has few rows); larger M runs a tcgen05 GEMM
 * over 128-row weight tiles.  The kernel depends on M and K; the K split on M, N and the SM count.
 *   x       in   bf16 bits [M][K]
 *   codes   in   uint8 [N][K/2]
 *   scales  in   fp16 bits [N][K/64]
 *   y       out  bf16 bits [M][N]; must not overlap x, codes or scales
 */
nf4_status nf4_linear(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, uint16_t* y,
                      int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * nf4_linear_grouped - several linears that read the same x, y_i = x * w_hat_i^T for i < count
 * (for instance the q, k and v projections, or the gate and up projections, of one decoder layer;
 * the deep-fold README's execution-path table runs decode as GEMVs over such linears).  For M <= 32
 * the linears share one launch over their rows; for larger M they run one GEMM after another on
 * `stream`.  Each y_i meets the nf4_linear bound and repeated calls give the
 * same bytes; the K split can differ from a separate nf4_linear call, so low-order bits may too.
 *   x        in   bf16 bits [M][K], shared by all linears
 *   count    1 .. 8
 *   codes    host array of count device pointers; codes[i]: uint8 [Ns[i]][K/2]
 *   scales   host array of count device pointers; scales[i]: fp16 bits [Ns[i]][K/64]
 *   ys       host array of count device pointers; ys[i]: bf16 bits [M][Ns[i]]; no y may overlap x,
 *            any codes or scales, or another y
 *   Ns       host array of count row counts (each >= 0, sum <= 2^31 - 1); empty linears are skipped
 * The host arrays are read before the call returns.  Errors as for nf4_linear (count outside
 * 1..8 gives NF4_ERR_SHAPE).
 */
nf4_status nf4_linear_grouped(const uint16_t* x, int64_t M, int64_t K, int count, const uint8_t* const* codes,
                              const uint16_t* const* scales, uint16_t* const* ys, const int64_t* Ns,
                              cudaStream_t stream);

/*
 * nf4_embed - rows of a packed embedding table, dequantized on request (deep-fold README, overview
 * paragraph: embeddings reconstruct only the rows that are asked for; the 20B run of its results
 * uses these packed embedding rows).  The table has the same format as a linear's weights: V rows
 * of K dimensions, groups of 64 along K with one FP16 scale each.
 *   ids     in   int32 [n_ids]; each should be in [0, V)
 *   codes   in   uint8 [V][K/2]
 *   scales  in   fp16 bits [V][K/64]
 *   out     out  bf16 bits [n_ids][K], out[i][k] = bf16_rn(fp32(T[code] * float(scale))) of row ids[i]
 *            (bit for bit the rows nf4_dequant would write); must not overlap ids, codes or scales
 * An id outside [0, V) gives a row of zeros and records code 41 in the device error word (see
 * nf4_check_device_error); nothing is read for it.  n_ids = 0 is a no-op.  Other errors as for
 * nf4_dequant.
 */
nf4_status nf4_embed(const int32_t* ids, int64_t n_ids, const uint8_t* codes, const uint16_t* scales, int64_t V,
                     int64_t K, uint16_t* out, cudaStream_t stream);

/*
 * Overflow streaming (deep-fold README, overview and execution-path table: a model larger than the
 * card keeps part of its packed weights in pinned host memory and copies them through two reusable
 * device slots, overlapped with the same GEMV / GEMM; the 32B row of its results runs this way).
 *
 * A ring is the one stateful object of the library: two device slots, a copy stream and events,
 * created on the current device.  nf4_ring_run walks a list of linears whose packed weights live in
 * page-locked host memory.  Linear i is copied into slot i mod 2 on the ring's copy stream (after
 * the linear that last read that slot has finished) and then runs as nf4_linear on `stream`, so
 * the copy of linear i + 1 overlaps the compute of linear i.  The linears run in list order on
 * `stream`, so the y of one may be the x of a later one.  Results are bit for bit those of
 * nf4_linear on device-resident copies of the same weights.
 */
typedef struct nf4_ring nf4_ring;

/* One linear of a streamed list. */
typedef struct nf4_host_linear {
    const uint16_t* x;      /* device, bf16 bits [M][K] */
    const uint8_t* codes;   /* page-locked host, uint8 [N][K/2] */
    const uint16_t* scales; /* page-locked host, fp16 bits [N][K/64] */
    uint16_t* y;            /* device, bf16 bits [M][N]; must not overlap x */
    int64_t M, N, K;        /* as for nf4_linear; M = 0 or N = 0 skips the entry */
} nf4_host_linear;

/*
 * nf4_ring_create - allocate a ring whose two slots hold up to `slot_bytes` of packed weights each:
 * a linear fits when N*K/2 rounded up to 256, plus N*(K/64)*2, is at most slot_bytes.
 *   slot_bytes  > 0
 *   ring        out: the new ring (NULL on error)
 * Errors: NF4_ERR_NULL, NF4_ERR_SHAPE (slot_bytes <= 0), NF4_ERR_UNSUPPORTED_DEVICE, NF4_ERR_CUDA
 * (allocation failed; nothing is left allocated).
 */
nf4_status nf4_ring_create(int64_t slot_bytes, nf4_ring** ring);

/*
 * nf4_ring_run - stream `count` linears through the ring, asynchronously on `stream`.
 *   ring    from nf4_ring_create, used on its own device
 *   ops     host array of count entries (read before the call returns)
 *   count   >= 0 (0 is a no-op)
 * Every entry is checked before anything is enqueued: shapes and alignment as for nf4_linear,
 * NF4_ERR_SHAPE when an entry does not fit a slot, NF4_ERR_MEMORY when codes or scales are not
 * page-locked host memory (first and last byte checked) or the current device is not the ring's.
 * The host buffers must stay unchanged until the work enqueued by the call has finished.  A ring
 * may be captured into a CUDA graph: a captured run orders its copies after the work already on
 * `stream`, and so do the ring's eager runs from then on; a graph and eager runs that share a ring
 * must therefore be issued on one stream (or be ordered by the caller).  Calls on one ring must not run concurrently from several host threads; runs on
 * different streams are ordered through the ring's events.  A CUDA failure part way returns
 * NF4_ERR_CUDA with the earlier entries enqueued.
 */
nf4_status nf4_ring_run(nf4_ring* ring, const nf4_host_linear* ops, int64_t count, cudaStream_t stream);

/* nf4_ring_destroy - wait for the ring's outstanding work and free it.  NULL is a no-op. */
nf4_status nf4_ring_destroy(nf4_ring* ring);

/*
 * nf4_linear_host_noalloc - one linear whose packed weights live in page-locked host memory, staged
 * through a device buffer that is part of the library itself, so that nothing is allocated.  The
 * pages have no counterpart: it is an addition of this library.
 *
 * Who needs it: a caller that cannot allocate device memory when it runs the layer.  Examples: a
 * host application whose own pool allocator has already reserved the GPU's memory (a cudaMalloc
 * from the library would fail or fragment that pool), or a decode loop that cannot afford
 * cudaMalloc / cudaFree, which may synchronise the whole device.  nf4_ring_create allocates its
 * slots with cudaMalloc; this call uses one static device array of NF4_NOALLOC_SLOT_BYTES instead.
 * Every device on which the library runs holds that array until the process exits.
 *
 *   x       in   device, bf16 bits [M][K]
 *   codes   in   page-locked host, uint8 [N][K/2]
 *   scales  in   page-locked host, fp16 bits [N][K/64]
 *   y       out  device, bf16 bits [M][N]; must not overlap x
 *
 * On `stream` the call copies codes and scales into the array and then runs nf4_linear on that copy;
 * y is bit for bit what nf4_linear gives on device-resident weights.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 * Limit: N*K/2 rounded up to 256, plus N*(K/64)*2, must not exceed NF4_NOALLOC_SLOT_BYTES (16 MiB,
 * e.g. 11008 x 2048 fits); a larger linear returns NF4_ERR_SHAPE and nothing is enqueued.  Host
 * buffers that are not page-locked give NF4_ERR_MEMORY.  Other errors as for nf4_linear.  The host
 * buffers must stay unchanged until the call's work on `stream` has finished.
 * Sharing: all calls on a device use the same array, which keeps the weights of the last call (each
 * call rewrites every byte the kernels read, so nothing needs clearing).  Calls on one stream are
 * ordered and safe; calls whose work may overlap on the GPU (different streams with no ordering
 * between them) race on the array and give wrong results.
 * Set-up: the first call on a device looks up the array's device address; make that first call
 * before any stream capture.
 * A first call made while `stream` is capturing returns NF4_ERR_CAPTURE and leaves the capture
 * untouched.
 */
#define NF4_NOALLOC_SLOT_BYTES (16 * 1024 * 1024)
nf4_status nf4_linear_host_noalloc(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, uint16_t* y,
                                   int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * nf4_check_device_error - diagnostics: read and clear the device-side error words of the current
 * device.  The linear kernels bound every pipeline wait (one second of wall-clock time per wait,
 * see nf4_diag_set_wait_limit); a wait that runs out records a nonzero code (1..39; 39 is
 * nf4_diag_bounded_wait's), and the kernel drains and exits instead of hanging, leaving its outputs
 * unspecified.  nf4_embed records 41 for an id outside the table.  *code receives the first
 * recorded code (0 = none).  This call waits for the device (it is not meant for the hot path).
 */
nf4_status nf4_check_device_error(int* code);

/*
 * nf4_diag_bounded_wait - diagnostics, no counterpart in the pages: checks that a pipeline wait
 * which runs out reports instead of hanging.  Launches one thread on `stream` that waits on an
 * mbarrier nothing ever arrives on, through the same bounded wait and error word as the linear
 * kernels; after `ns` nanoseconds of wall-clock time it gives up and records code 39, which
 * nf4_check_device_error then returns.  The device stays usable.  ns must be in [1, 2^31] (about
 * 2.1 s), else NF4_ERR_SHAPE.
 */
nf4_status nf4_diag_bounded_wait(int64_t ns, cudaStream_t stream);

/*
 * nf4_diag_set_wait_limit - diagnostics, no counterpart in the pages: sets the wall-clock limit of
 * each pipeline wait of the linear kernels on the current device to `ns` nanoseconds, or restores
 * the default of one second when ns = 0.  The limit applies to every wait separately (it restarts
 * at each wait), so a kernel that runs far longer than the limit is unaffected as long as each of
 * its waits is shorter.  Stream-ordered on `stream`.  ns must be in [0, 2^36] (about 69 s), else
 * NF4_ERR_SHAPE.
 */
nf4_status nf4_diag_set_wait_limit(int64_t ns, cudaStream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char* nf4_status_str(nf4_status status);

/* NF4_ABI_VERSION of the built library. */
int nf4_abi_version(void);

/* NF4_NOALLOC_SLOT_BYTES of the built library (the size of nf4_linear_host_noalloc's array). */
int64_t nf4_noalloc_slot_bytes(void);

/* Name of the last CUDA error (for instance "cudaErrorInvalidValue") behind an NF4_ERR_CUDA returned
 * to the calling host thread, or "cudaSuccess" if there was none.  Static string, never NULL. */
const char* nf4_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* NF4_H */
