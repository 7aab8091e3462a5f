// NF4 GEMV family on CUDA cores (sm_103a): y[M, N] = x[M, K] * w_hat[N, K]^T for 1 <= M <= 4.
//
// Decode is weight streaming (deep-fold README, execution-path table: the N=1 decode step runs a
// GEMV on CUDA cores and dequantizes only the current tile).  The kernel's job is to consume the
// packed codes at HBM speed, which leaves about three to four issue slots per weight on a GB300.
//
// Scale factorisation.  A nonzero fp16 scale is 2^E * (1 + m/1024) with m its top ten fraction
// bits (fp16 subnormals included, read as binary32).  Rounding commutes with multiplication by a
// power of two, so w_hat = bf16(fp32(T[c] * scale)) = 2^E * V[m][c] with V[m][c] =
// bf16(fp32(T[c] * (1 + m/1024))).  V is a 1024 x 16 bf16 table built once per device.  A lane sums
// x_k * V[m][c_k] over its group in fp32 (each bf16 x bf16 product is exact) and scales the group
// sum by 2^E, which is exact too: the result equals the sum of x_k * w_hat_k in that order.
//
// Lookup.  Per (row, group) a lane holds its V row as eight registers: the low bytes and the high
// bytes of the 16 bf16 entries, each split into codes 0-7 and 8-15.  `prmt` reads a 4-bit code
// nibble as a byte selector, so one instruction looks up one byte plane for four codes; a
// sign-replicating `prmt` turns bit 3 of each code into a byte mask that picks the 0-7 or the 8-15
// half.  Eight weights cost 22 integer instructions before the multiply-adds.
//
// Work layout.  A warp owns a K-slice (32 groups at one lane per group, or 16 groups at two lanes
// per group) and keeps that slice of x in registers as bf16 pairs; it streams four rows at a time
// (128-bit loads), reduces the four row partial sums across lanes with a transposed butterfly and
// hands them to the CTA, whose warps cover all slices of the same rows; slice sums are added in a
// fixed order, so results are deterministic.  The grid is persistent over row blocks.
#include <mutex>

#include <cudaTypedefs.h>

#include "nf4_device.cuh"
#include "nf4_internal.h"

namespace nf4 {
namespace {

constexpr int kMaxWarps = 16;  // warps per CTA (slices x row lanes)
constexpr int kVtabBytes = 1024 * 32;  // V table copy in shared memory

// V table: row m holds the low bytes {L(0..3), L(4..7), L(15..12), L(11..8)} and the high bytes in
// the same order, L / H being the low / high byte of the bf16 entry V[m][c].  Codes 8..15 are stored
// in reverse so that the complemented nibble 15 - c (one IMAD) indexes them directly.  Rows are laid
// out in blocks of eight: the eight low-byte chunks, then the eight high-byte chunks, so the chunk
// of row m sits at index m + (m & ~7) (+ 8 for the high bytes) and eight lanes reading random rows
// spread over all eight 16-byte bank groups of a 128-byte line.
// Rows 1024..2047 repeat the table at twice the value (V[m][c] * 2, exact), which the tensor-core
// path uses to fold an odd scale exponent into the table.
__device__ uint4 g_vtab[2048 * 2];

__global__ void build_vtab_kernel() {
    const int m = blockIdx.x * blockDim.x + threadIdx.x;  // table row: 1024 * p + mantissa class
    if (m >= 2048) return;
    // (1 + (m mod 1024)/1024) * 2^(m / 1024), exactly
    const float s1 = __uint_as_float((0x3F800000u + (static_cast<uint32_t>(m >> 10) << 23)) |
                                     (static_cast<uint32_t>(m & 1023) << 13));
    uint32_t lo[4] = {0, 0, 0, 0}, hi[4] = {0, 0, 0, 0};
#pragma unroll
    for (int c = 0; c < 16; c++) {
        const uint32_t b = bf16_bits(__fmul_rn(kNF4[c], s1));
        const int slot = c < 8 ? c : 8 + (15 - c);  // byte position inside the 16-byte plane
        lo[slot >> 2] |= (b & 0xFFu) << (8 * (slot & 3));
        hi[slot >> 2] |= (b >> 8) << (8 * (slot & 3));
    }
    g_vtab[m + (m & ~7)] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    g_vtab[m + (m & ~7) + 8] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
}

// Eight codes (weight 2i in the low nibble of byte i) -> four bf16 pairs, weights in order.
// 18 ALU-pipe instructions (PRMT / LOP3) and 4 FMA-pipe ones (selector preparation).
__device__ __forceinline__ void lookup8(uint32_t w, const uint4& tl, const uint4& th, uint32_t m1, uint32_t p16,
                                        uint32_t out[4]) {
    const uint32_t nw = not_fma(w, m1);  // nibble 15 - c: codes 8..15 index the reversed second half
    const uint32_t w4 = shl4_fma(w);
    const uint32_t wh = shr16_fma(w, p16), nwh = shr16_fma(nw, p16);
    uint32_t msk = prmt(w4, w, 0xD9C8u);  // byte i = 0xFF iff code i >= 8 (i = 0..3)
    uint32_t lo = select_bits(prmt(tl.x, tl.y, w), prmt(tl.z, tl.w, nw), msk);
    uint32_t hi = select_bits(prmt(th.x, th.y, w), prmt(th.z, th.w, nw), msk);
    out[0] = prmt(lo, hi, 0x5140u);
    out[1] = prmt(lo, hi, 0x7362u);
    msk = prmt(w4, w, 0xFBEAu);  // codes 4..7
    lo = select_bits(prmt(tl.x, tl.y, wh), prmt(tl.z, tl.w, nwh), msk);
    hi = select_bits(prmt(th.x, th.y, wh), prmt(th.z, th.w, nwh), msk);
    out[2] = prmt(lo, hi, 0x5140u);
    out[3] = prmt(lo, hi, 0x7362u);
}

// Sum each of V values over the 32 lanes.  Recursive halving: at each of the first log2(V) steps a
// lane keeps the half of its values selected by one lane bit and adds its partner's copy of that
// half; the remaining steps are a plain butterfly.  Afterwards lane l holds value l >> (5 - log2 V).
template <int V>
__device__ __forceinline__ float reduce_transposed(float (&v)[V], int lane) {
    int n = V;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (n > 1) {
            const int half = n / 2;
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < half; i++) {
                const float send = upper ? v[i] : v[i + half];
                const float keep = upper ? v[i + half] : v[i];
                v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
            }
            n = half;
        } else {
            v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], off);
        }
    }
    return v[0];
}

__host__ __device__ constexpr int pow2_ceil(int v) { return v <= 1 ? 1 : 2 * pow2_ceil((v + 1) / 2); }

// Up to kMaxGroup linears that share x and K, run as one launch over their concatenated rows.
constexpr int kMaxGroup = 8;
struct GemvProblems {
    const uint8_t* codes[kMaxGroup];
    const uint16_t* scales[kMaxGroup];
    uint16_t* y[kMaxGroup];
    int row0[kMaxGroup + 1];  // first concatenated row of each problem; row0[count] = total rows
    int count;
};

// Problem holding concatenated row r (rows are sorted, count is small).
__device__ __forceinline__ int problem_of(const GemvProblems& P, int64_t r) {
    int p = 0;
    for (int i = 1; i < P.count; i++)
        if (r >= P.row0[i]) p = i;
    return p;
}

// MT tokens, LPG lanes per group, R rows per warp iteration, ST ring stages per warp.
template <int MT, int LPG, int R, int ST>
struct GemvShape {
    static constexpr int WPL = kGroup / LPG;   // weights per lane per row
    static constexpr int CB = WPL / 2;         // code bytes per lane per row
    static constexpr int CHUNKS = CB / 16;     // 16-byte copies per lane per row
    static constexpr int GPW = 32 / LPG;       // groups per warp slice
    static constexpr int SWIN = 2 * GPW + 16;  // bytes of a row's 16-byte-aligned scale window
    static constexpr int STAGE_CODES = R * 32 * CB;
    static constexpr int STAGE = STAGE_CODES + R * SWIN;
    static constexpr int WARP_SMEM = ST * STAGE;
};

// MT tokens; LPG lanes per 64-weight group (1 or 2); R rows per warp iteration (4 for large
// matrices, 1 for small ones so that more warps share the work); ST stages in each warp's ring.
// Shared memory: the V table (32 KB), then one private ring of ST row batches per warp (codes and
// scale windows, filled with cp.async), then two [S][Q*R][MT] slice-partial buffers when S > 1.
template <int MT, int LPG, int R, int ST>
__global__ void __launch_bounds__(kMaxWarps * 32, 1)
    gemv_kernel(const uint16_t* __restrict__ x, const __grid_constant__ GemvProblems P, int K, int S, int Q,
                uint32_t m1, uint32_t p16) {
    using SH = GemvShape<MT, LPG, R, ST>;
    constexpr int kRows = R;
    constexpr int kStages = ST;
    constexpr int V = pow2_ceil(kRows * MT);
    extern __shared__ __align__(16) uint8_t smem[];

    const int N = P.row0[P.count];  // concatenated rows
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int s = warp % S, q = warp / S;
    const int G = K / kGroup;
    const int g = s * SH::GPW + lane / LPG;
    const bool active = g < G;
    const int k0 = s * SH::GPW * kGroup + lane * SH::WPL;
    const int g_hi = min(G, (s + 1) * SH::GPW);        // one past the slice's last group
    const int sw = LPG == 1 ? ((lane >> 2) & 1) : 0;  // 16-byte chunk swizzle: conflict-free reads
    const uint4* vtab = reinterpret_cast<const uint4*>(smem);
    uint8_t* ring = smem + kVtabBytes + warp * SH::WARP_SMEM;
    float* red = reinterpret_cast<float*>(smem + kVtabBytes + nwarps * SH::WARP_SMEM);
    const int rows_per_block = Q * kRows;
    const int64_t nblocks = (static_cast<int64_t>(N) + rows_per_block - 1) / rows_per_block;
    const int64_t my_blocks =
        blockIdx.x < nblocks ? (nblocks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const uint32_t row_bytes = static_cast<uint32_t>(K / 2);
    const uint32_t row_sbytes = static_cast<uint32_t>(G * 2);
    const int64_t rstep = static_cast<int64_t>(gridDim.x) * rows_per_block;

    // Let the next kernel in the stream launch, warm L2 with this warp's first rows (a prefetch
    // never returns stale data: L2 is coherent), copy the constant table, then wait for the
    // previous kernel's results.
    pdl_launch_dependents();
    const int64_t r_first = static_cast<int64_t>(blockIdx.x) * rows_per_block + q * kRows;
    if (my_blocks > 0 && active) {
#pragma unroll
        for (int j = 0; j < kRows; j++)
            if (r_first + j < N) {
                const int pp = problem_of(P, r_first + j);
                prefetch_l2(P.codes[pp] + (r_first + j - P.row0[pp]) * row_bytes + k0 / 2);
            }
    }
    for (int i = threadIdx.x; i < kVtabBytes / 16; i += blockDim.x)  // all copies in flight at once
        cp_async16(smem + 16 * i, &g_vtab[i]);
    cp_async_commit();
    pdl_wait();

    uint32_t xr[MT][SH::WPL / 2];
#pragma unroll
    for (int t = 0; t < MT; t++) {
#pragma unroll
        for (int i = 0; i < SH::WPL / 8; i++) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (active) v = *reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * K + k0 + 8 * i);
            xr[t][4 * i + 0] = v.x;
            xr[t][4 * i + 1] = v.y;
            xr[t][4 * i + 2] = v.z;
            xr[t][4 * i + 3] = v.w;
        }
    }

    // Enqueue the copies of this warp's t-th row quad into ring stage t % kStages (one commit group
    // per quad, empty past the end so that group counting stays uniform).
    auto issue = [&](int64_t t) {
        if (t < my_blocks) {
            uint8_t* st = ring + static_cast<int>(t % kStages) * SH::STAGE;
            const int64_t r0 = r_first + t * rstep;
#pragma unroll
            for (int j = 0; j < kRows; j++) {
                const int64_t r = r0 + j;
                if (r < N) {
                    const int pp = problem_of(P, r);
                    const int64_t lr = r - P.row0[pp];  // row inside problem pp
                    // Consecutive lanes copy consecutive 16-byte chunks of the slice's row (full
                    // sectors per instruction); chunk q belongs to compute lane q / CHUNKS and lands
                    // in that lane's (swizzled) slot.
                    const uint8_t* src = P.codes[pp] + lr * row_bytes + s * SH::GPW * (kGroup / 2);
#pragma unroll
                    for (int c = 0; c < SH::CHUNKS; c++) {
                        const int q = lane + 32 * c;
                        const int lq = q / SH::CHUNKS, hq = q % SH::CHUNKS;
                        const int swq = LPG == 1 ? ((lq >> 2) & 1) : 0;
                        if (s * SH::GPW + lq / LPG < G)
                            cp_async16(st + ((j * 32 + lq) * SH::CHUNKS + (hq ^ swq)) * 16, src + 16 * q);
                    }
                    // scale window of this row's slice: [first byte rounded down to 16, last byte]
                    const int64_t sfirst = (lr * G + s * SH::GPW) * 2;
                    const int64_t chunk = (sfirst & ~static_cast<int64_t>(15)) + 16 * lane;
                    if (chunk < sfirst + 2 * (g_hi - s * SH::GPW)) {
                        const int64_t left =
                            static_cast<int64_t>(P.row0[pp + 1] - P.row0[pp]) * row_sbytes - chunk;
                        cp_async16(st + SH::STAGE_CODES + j * SH::SWIN + 16 * lane,
                                   reinterpret_cast<const uint8_t*>(P.scales[pp]) + chunk,
                                   static_cast<uint32_t>(left < 16 ? left : 16));
                    }
                }
            }
        }
        cp_async_commit();
    };

#pragma unroll
    for (int t = 0; t < kStages - 1; t++) issue(t);
    cp_async_wait<kStages - 1>();  // the V table group (the oldest) has landed
    __syncthreads();

    for (int64_t t = 0; t < my_blocks; t++) {
        issue(t + kStages - 1);
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const uint8_t* st = ring + static_cast<int>(t % kStages) * SH::STAGE;
        const int64_t r0 = r_first + t * rstep;
        // Row j's scale window starts at its first scale byte rounded down to 16; the lane's scale
        // sits (first byte mod 16) + 2 * (g - first group) bytes into it.
        const int goff = 2 * (g - s * SH::GPW);
        float part[V];
#pragma unroll
        for (int i = 0; i < V; i++) part[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < kRows; j++) {
            if (r0 + j >= N) continue;  // warp-uniform
            uint32_t sc = 0;
            if (active) {
                const int pp = problem_of(P, r0 + j);
                const uint32_t lr = static_cast<uint32_t>(r0 + j - P.row0[pp]);
                const int off = static_cast<int>(((lr * static_cast<uint32_t>(G) + s * SH::GPW) * 2u) & 15u) + goff;
                sc = *reinterpret_cast<const uint16_t*>(st + SH::STAGE_CODES + j * SH::SWIN + off);
            }
            const uint32_t sb = __float_as_uint(__half2float(__ushort_as_half(static_cast<uint16_t>(sc))));
            const uint32_t m = (sb >> 13) & 0x3FFu;
            const float pow2 = __uint_as_float(sb & 0xFF800000u);  // +-2^E, or 0 for a zero scale
            const uint4 tl = vtab[m + (m & ~7u)];
            const uint4 th = vtab[m + (m & ~7u) + 8];
            float a0[MT], a1[MT];
#pragma unroll
            for (int tt = 0; tt < MT; tt++) a0[tt] = a1[tt] = 0.0f;
#pragma unroll
            for (int c = 0; c < SH::CHUNKS; c++) {
                const uint4 cw = lds128(st + ((j * 32 + lane) * SH::CHUNKS + (c ^ sw)) * 16);
                const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                for (int wi = 0; wi < 4; wi++) {
                    uint32_t wp[4];
                    lookup8(words[wi], tl, th, m1, p16, wp);
#pragma unroll
                    for (int tt = 0; tt < MT; tt++) {
#pragma unroll
                        for (int p = 0; p < 4; p++)
                            fma_bf16x2(a0[tt], a1[tt], wp[p], xr[tt][4 * (4 * c + wi) + p]);
                    }
                }
            }
#pragma unroll
            for (int tt = 0; tt < MT; tt++) part[j * MT + tt] = (a0[tt] + a1[tt]) * pow2;
        }
        __syncwarp();  // every lane is done with this stage before it is refilled
        const float total = reduce_transposed<V>(part, lane);
        constexpr int lanes_per_value = 32 / V;
        const int idx = lane / lanes_per_value;
        const bool writer = (lane % lanes_per_value) == 0 && idx < kRows * MT;
        const int j = idx / MT, tt = idx % MT;
        if (S == 1) {
            if (writer && r0 + j < N) {
                const int pp = problem_of(P, r0 + j);
                const int np = P.row0[pp + 1] - P.row0[pp];
                P.y[pp][static_cast<int64_t>(tt) * np + (r0 + j - P.row0[pp])] = bf16_bits(total);
            }
        } else {
            const int64_t rb = blockIdx.x + t * gridDim.x;
            float* buf = red + (t & 1) * S * rows_per_block * MT;
            if (writer) buf[(s * rows_per_block + q * kRows + j) * MT + tt] = total;
            __syncthreads();
            for (int i = threadIdx.x; i < rows_per_block * MT; i += blockDim.x) {
                const int64_t r = rb * rows_per_block + i / MT;
                float acc = 0.0f;
                for (int ss = 0; ss < S; ss++) acc += buf[ss * rows_per_block * MT + i];
                if (r < N) {
                    const int pp = problem_of(P, r);
                    const int np = P.row0[pp + 1] - P.row0[pp];
                    P.y[pp][static_cast<int64_t>(i % MT) * np + (r - P.row0[pp])] = bf16_bits(acc);
                }
            }
        }
    }
    cp_async_wait<0>();
}

struct TableState {
    std::mutex mu;
    bool ready[64] = {};
};
TableState g_tables;

template <int MT, int LPG, int R, int ST>
cudaError_t launch_gemv_t(const uint16_t* x, const GemvProblems& P, int64_t K, int num_sms, cudaStream_t stream) {
    const int64_t N = P.row0[P.count];
    using SH = GemvShape<MT, LPG, R, ST>;
    constexpr int kRows = R;
    const int G = static_cast<int>(K / kGroup);
    const int S = (G + SH::GPW - 1) / SH::GPW;
    // Row lanes per slice: enough CTAs to cover the SMs when N is small, at most kMaxWarps warps.
    const int64_t quads = (N + kRows - 1) / kRows;
    int Q = static_cast<int>((quads + num_sms - 1) / num_sms);
    const int qmax = S >= kMaxWarps ? 1 : kMaxWarps / S;
    if (Q > qmax) Q = qmax;
    if (Q < 1) Q = 1;
    const int warps = S * Q;
    const int rows_per_block = Q * kRows;
    const int64_t blocks_needed = (N + rows_per_block - 1) / rows_per_block;
    const int grid = static_cast<int>(blocks_needed < num_sms ? blocks_needed : num_sms);
    const size_t smem = kVtabBytes + static_cast<size_t>(warps) * SH::WARP_SMEM +
                        (S > 1 ? 2 * static_cast<size_t>(S) * rows_per_block * MT * sizeof(float) : 0);
    static std::once_flag attr_once[64];  // the largest request, set once per device
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once[dev & 63], [&] {
        const size_t max_smem = kVtabBytes + static_cast<size_t>(kMaxWarps) * SH::WARP_SMEM +
                                2 * static_cast<size_t>(kMaxWarps) * kRows * MT * sizeof(float);
        attr_err = cudaFuncSetAttribute(gemv_kernel<MT, LPG, R, ST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(max_smem));
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * warps);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<MT, LPG, R, ST>, x, P, static_cast<int>(K), S, Q, 0xFFFFFFFFu,
                              0x10000u);
}

}  // namespace
}  // namespace nf4

#include "nf4_tc.cuh"

namespace nf4 {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

template <int T>
cudaError_t launch_tc_t(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, uint16_t* y, int64_t M,
                        int64_t N, int64_t K, cudaStream_t stream) {
    using L = tc::Layout<T>;
    auto encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap tx, tcodes;
    {   // x: bf16 [M][K], boxes of 64 (K) x T (tokens), 128-byte swizzle; rows past M read as zero
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(T)};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {   // codes: u8 [N][K/2], boxes of 32 bytes (one group) x 128 rows; rows past N read as zero
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
        const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(tc::kTileN)};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tcodes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const size_t smem = L::kBytes + 1024;  // + slack to align the base to 1024 bytes
    static std::once_flag attr_once[64];
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once[dev & 63], [&] {
        attr_err = cudaFuncSetAttribute(tc::gemm_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((N + tc::kTileN - 1) / tc::kTileN),
                       static_cast<unsigned>((M + T - 1) / T));
    cfg.blockDim = dim3(tc::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc::gemm_kernel<T>, tx, tcodes, scales, y, static_cast<int>(M),
                              static_cast<int>(N), static_cast<int>(K), 0xFFFFFFFFu, 0x10000u);
}

}  // namespace

cudaError_t launch_tc(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, uint16_t* y, int64_t M,
                      int64_t N, int64_t K, cudaStream_t stream) {
    if (M <= 16) return launch_tc_t<16>(x, codes, scales, y, M, N, K, stream);
    if (M <= 32) return launch_tc_t<32>(x, codes, scales, y, M, N, K, stream);
    if (M <= 64) return launch_tc_t<64>(x, codes, scales, y, M, N, K, stream);
    if (M <= 128) return launch_tc_t<128>(x, codes, scales, y, M, N, K, stream);
    return launch_tc_t<256>(x, codes, scales, y, M, N, K, stream);
}

cudaError_t read_and_clear_error(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
    *code = v;
    return e;
}

// Largest K the register-resident layout covers: kMaxWarps slices of 32 (one lane per group) or 16
// groups (two lanes per group).
int64_t gemv_max_k(int64_t M) { return static_cast<int64_t>(kMaxWarps) * (M == 1 ? 32 : 16) * kGroup; }

cudaError_t ensure_tables(int device, cudaStream_t stream) {
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_tables.mu);
    if (g_tables.ready[device]) return cudaSuccess;
    build_vtab_kernel<<<8, 256, 0, stream>>>();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // One-time wait so that later calls on any stream see the table.
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    g_tables.ready[device] = true;
    return cudaSuccess;
}

cudaError_t launch_gemv_grouped(const uint16_t* x, int count, const uint8_t* const* codes,
                                const uint16_t* const* scales, uint16_t* const* ys, const int64_t* Ns, int64_t M,
                                int64_t K, int num_sms, cudaStream_t stream) {
    if (count < 1 || count > kMaxGroup) return cudaErrorInvalidValue;
    GemvProblems P = {};
    P.count = count;
    int64_t rows = 0;
    for (int i = 0; i < count; i++) {
        P.codes[i] = codes[i];
        P.scales[i] = scales[i];
        P.y[i] = ys[i];
        P.row0[i] = static_cast<int>(rows);
        rows += Ns[i];
    }
    if (rows > 0x7FFFFFFF) return cudaErrorInvalidValue;
    P.row0[count] = static_cast<int>(rows);
    for (int i = count + 1; i <= kMaxGroup; i++) P.row0[i] = P.row0[count];
    // HBM latency under load is a few microseconds, so each SM needs on the order of 100 KB of
    // copies in flight: large matrices use 2 rows per warp iteration and a 5-deep ring (4 batches
    // in flight per warp), smaller ones 1 row and an 8-deep ring so that many warps share the rows.
    const bool large = rows >= static_cast<int64_t>(2) * kMaxWarps * num_sms;
    switch (M) {
        case 1: return large ? launch_gemv_t<1, 1, 2, 5>(x, P, K, num_sms, stream)
                             : launch_gemv_t<1, 1, 1, 8>(x, P, K, num_sms, stream);
        case 2: return large ? launch_gemv_t<2, 2, 4, 2>(x, P, K, num_sms, stream)
                             : launch_gemv_t<2, 2, 1, 4>(x, P, K, num_sms, stream);
        case 3: return large ? launch_gemv_t<3, 2, 4, 2>(x, P, K, num_sms, stream)
                             : launch_gemv_t<3, 2, 1, 4>(x, P, K, num_sms, stream);
        case 4: return large ? launch_gemv_t<4, 2, 4, 2>(x, P, K, num_sms, stream)
                             : launch_gemv_t<4, 2, 1, 4>(x, P, K, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, uint16_t* y,
                        int64_t M, int64_t N, int64_t K, int num_sms, cudaStream_t stream) {
    return launch_gemv_grouped(x, 1, &codes, &scales, &y, &N, M, K, num_sms, stream);
}

}  // namespace nf4
