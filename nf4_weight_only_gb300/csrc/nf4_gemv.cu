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

#include "nf4_device.cuh"
#include "nf4_internal.h"

namespace nf4 {
namespace {

constexpr int kRows = 4;       // rows per warp iteration
constexpr int kMaxWarps = 16;  // warps per CTA (slices x row lanes)

// V table: row m holds {L(0..3), L(4..7), L(8..11), L(12..15)} and {H(0..3), ..., H(12..15)},
// L / H being the low / high byte of the bf16 entry V[m][c].
__device__ uint4 g_vtab[1024 * 2];

__global__ void build_vtab_kernel() {
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= 1024) return;
    const float s1 = __uint_as_float(0x3F800000u | (static_cast<uint32_t>(m) << 13));  // 1 + m/1024
    uint32_t lo[4] = {0, 0, 0, 0}, hi[4] = {0, 0, 0, 0};
#pragma unroll
    for (int c = 0; c < 16; c++) {
        const uint32_t b = bf16_bits(__fmul_rn(kNF4[c], s1));
        lo[c >> 2] |= (b & 0xFFu) << (8 * (c & 3));
        hi[c >> 2] |= (b >> 8) << (8 * (c & 3));
    }
    g_vtab[2 * m] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    g_vtab[2 * m + 1] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
}

// Eight codes (weight 2i in the low nibble of byte i) -> four bf16 pairs, weights in order.
__device__ __forceinline__ void lookup8(uint32_t w, const uint4& tl, const uint4& th, uint32_t out[4]) {
    const uint32_t wb = w ^ 0x88888888u;  // bit 3 flipped: codes 8-15 index the second half
    const uint32_t w4 = w << 4;
    uint32_t msk = prmt(w4, w, 0xD9C8u);  // byte i = 0xFF iff code i >= 8 (i = 0..3)
    uint32_t lo = select_bits(prmt(tl.x, tl.y, w), prmt(tl.z, tl.w, wb), msk);
    uint32_t hi = select_bits(prmt(th.x, th.y, w), prmt(th.z, th.w, wb), msk);
    out[0] = prmt(lo, hi, 0x5140u);
    out[1] = prmt(lo, hi, 0x7362u);
    const uint32_t wh = w >> 16, wbh = wb >> 16;
    msk = prmt(w4, w, 0xFBEAu);  // codes 4..7
    lo = select_bits(prmt(tl.x, tl.y, wh), prmt(tl.z, tl.w, wbh), msk);
    hi = select_bits(prmt(th.x, th.y, wh), prmt(th.z, th.w, wbh), msk);
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

// MT tokens; LPG lanes per 64-weight group (1 or 2).
template <int MT, int LPG>
__global__ void __launch_bounds__(kMaxWarps * 32, 1)
    gemv_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ codes,
                const uint16_t* __restrict__ scales, uint16_t* __restrict__ y, int N, int K, int S, int Q) {
    constexpr int WPL = kGroup / LPG;  // weights per lane
    constexpr int WORDS = WPL / 8;     // code words per lane per row
    constexpr int GPW = 32 / LPG;      // groups per warp slice
    constexpr int V = pow2_ceil(kRows * MT);
    extern __shared__ float red[];  // [S][Q * kRows][MT] slice partials

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int s = warp % S, q = warp / S;
    const int G = K / kGroup;
    const int g = s * GPW + lane / LPG;
    const bool active = g < G;
    const int k0 = s * GPW * kGroup + lane * WPL;

    uint32_t xr[MT][WPL / 2];
#pragma unroll
    for (int t = 0; t < MT; t++) {
#pragma unroll
        for (int i = 0; i < WPL / 8; i++) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (active) v = *reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * K + k0 + 8 * i);
            xr[t][4 * i + 0] = v.x;
            xr[t][4 * i + 1] = v.y;
            xr[t][4 * i + 2] = v.z;
            xr[t][4 * i + 3] = v.w;
        }
    }

    const int rows_per_block = Q * kRows;
    const int64_t row_stride = K / 2;
    for (int64_t rb = blockIdx.x; rb * rows_per_block < N; rb += gridDim.x) {
        const int64_t r0 = rb * rows_per_block + static_cast<int64_t>(q) * kRows;
        uint32_t cw[kRows][WORDS];
        uint16_t sc[kRows];
#pragma unroll
        for (int j = 0; j < kRows; j++) {
            const int64_t r = r0 + j;
            const bool ok = active && r < N;
            const uint8_t* p = codes + r * row_stride + k0 / 2;
#pragma unroll
            for (int i = 0; i < WORDS / 4; i++) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (ok) v = ld_nc_v4(p + 16 * i);
                cw[j][4 * i + 0] = v.x;
                cw[j][4 * i + 1] = v.y;
                cw[j][4 * i + 2] = v.z;
                cw[j][4 * i + 3] = v.w;
            }
            sc[j] = ok ? ld_nc_u16(scales + r * G + g) : static_cast<uint16_t>(0);
        }
        float part[V];
#pragma unroll
        for (int i = 0; i < V; i++) part[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < kRows; j++) {
            const uint32_t sb = __float_as_uint(__half2float(__ushort_as_half(sc[j])));
            const uint32_t m = (sb >> 13) & 0x3FFu;
            const float pow2 = __uint_as_float(sb & 0x7F800000u);  // 2^E, or 0 for a zero scale
            const uint4 tl = ld_ca_v4(&g_vtab[2 * m]);
            const uint4 th = ld_ca_v4(&g_vtab[2 * m + 1]);
            float a0[MT], a1[MT];
#pragma unroll
            for (int t = 0; t < MT; t++) a0[t] = a1[t] = 0.0f;
#pragma unroll
            for (int wi = 0; wi < WORDS; wi++) {
                uint32_t wp[4];
                lookup8(cw[j][wi], tl, th, wp);
#pragma unroll
                for (int t = 0; t < MT; t++) {
#pragma unroll
                    for (int p = 0; p < 4; p++) fma_bf16x2(a0[t], a1[t], wp[p], xr[t][4 * wi + p]);
                }
            }
#pragma unroll
            for (int t = 0; t < MT; t++) part[j * MT + t] = (a0[t] + a1[t]) * pow2;
        }
        const float total = reduce_transposed<V>(part, lane);
        constexpr int lanes_per_value = 32 / V;
        const int idx = lane / lanes_per_value;
        const bool writer = (lane % lanes_per_value) == 0 && idx < kRows * MT;
        const int j = idx / MT, t = idx % MT;
        if (S == 1) {
            if (writer && r0 + j < N) y[static_cast<int64_t>(t) * N + r0 + j] = bf16_bits(total);
        } else {
            if (writer) red[(s * rows_per_block + q * kRows + j) * MT + t] = total;
            __syncthreads();
            for (int i = threadIdx.x; i < rows_per_block * MT; i += blockDim.x) {
                const int64_t r = rb * rows_per_block + i / MT;
                float acc = 0.0f;
                for (int ss = 0; ss < S; ss++) acc += red[ss * rows_per_block * MT + i];
                if (r < N) y[static_cast<int64_t>(i % MT) * N + r] = bf16_bits(acc);
            }
            __syncthreads();
        }
    }
}

struct TableState {
    std::mutex mu;
    bool ready[64] = {};
};
TableState g_tables;

template <int MT, int LPG>
cudaError_t launch_gemv_t(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, uint16_t* y,
                          int64_t N, int64_t K, int num_sms, cudaStream_t stream) {
    const int G = static_cast<int>(K / kGroup);
    const int gpw = 32 / LPG;
    const int S = (G + gpw - 1) / gpw;
    const int Q = S >= kMaxWarps ? 1 : kMaxWarps / S;
    const int threads = 32 * S * Q;
    const int rows_per_block = Q * kRows;
    const int64_t blocks_needed = (N + rows_per_block - 1) / rows_per_block;
    const int64_t grid = blocks_needed < num_sms ? blocks_needed : num_sms;
    const size_t smem = S > 1 ? static_cast<size_t>(S) * rows_per_block * MT * sizeof(float) : 0;
    gemv_kernel<MT, LPG><<<static_cast<int>(grid), threads, smem, stream>>>(
        x, codes, scales, y, static_cast<int>(N), static_cast<int>(K), S, Q);
    return cudaGetLastError();
}

}  // namespace

// Largest K the register-resident layout covers: kMaxWarps slices of 32 (one lane per group) or 16
// groups (two lanes per group).
int64_t gemv_max_k(int64_t M) { return static_cast<int64_t>(kMaxWarps) * (M == 1 ? 32 : 16) * kGroup; }

cudaError_t ensure_tables(int device, cudaStream_t stream) {
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_tables.mu);
    if (g_tables.ready[device]) return cudaSuccess;
    build_vtab_kernel<<<4, 256, 0, stream>>>();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // One-time wait so that later calls on any stream see the table.
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    g_tables.ready[device] = true;
    return cudaSuccess;
}

cudaError_t launch_gemv(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, uint16_t* y,
                        int64_t M, int64_t N, int64_t K, int num_sms, cudaStream_t stream) {
    switch (M) {
        case 1: return launch_gemv_t<1, 1>(x, codes, scales, y, N, K, num_sms, stream);
        case 2: return launch_gemv_t<2, 2>(x, codes, scales, y, N, K, num_sms, stream);
        case 3: return launch_gemv_t<3, 2>(x, codes, scales, y, N, K, num_sms, stream);
        case 4: return launch_gemv_t<4, 2>(x, codes, scales, y, N, K, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nf4
