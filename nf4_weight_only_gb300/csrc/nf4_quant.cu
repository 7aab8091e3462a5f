// NF4 quantize (pack) and dequantize kernels for sm_103a.
//
// Both are HBM-bound streaming kernels.  Because K is a multiple of 64, group g of row n is the
// flat group n * (K/64) + g: its 64 weights, 32 code bytes and one scale are contiguous, so both
// kernels walk a flat group index with a grid-stride loop.
#include "nf4_device.cuh"
#include "nf4_internal.h"

namespace nf4 {
namespace {

// Ordered integer key of a binary32 value (increases with the value; -0 and +0 share key 0).
__device__ __forceinline__ int32_t f32_key(float f) {
    uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? -static_cast<int32_t>(b & 0x7FFFFFFFu) : static_cast<int32_t>(b);
}

__device__ __forceinline__ float key_f32(int32_t k) {
    return __uint_as_float(k >= 0 ? static_cast<uint32_t>(k) : (0x80000000u | static_cast<uint32_t>(-k)));
}

// Decision threshold between codes i and i+1: the smallest binary32 r in [T[i], T[i+1]] that is
// strictly closer, in fp32 distance, to T[i+1] than to T[i].  Between the two table values the fp32
// distance to T[i] never decreases and the distance to T[i+1] never increases as r grows, so the
// predicate flips exactly once and bisection over the ordered bit patterns finds the flip.  The
// nearest-code rule "argmin_i |r - T[i]| in fp32, ties to the lower index" is then exactly
// code(r) = number of thresholds <= r.
__device__ float decision_threshold(int i) {
    const float t_lo = kNF4[i], t_hi = kNF4[i + 1];
    int32_t lo = f32_key(t_lo), hi = f32_key(t_hi);
    while (hi - lo > 1) {
        const int32_t mid = lo + (hi - lo) / 2;
        const float r = key_f32(mid);
        const bool upper = fabsf(__fsub_rn(r, t_hi)) < fabsf(__fsub_rn(r, t_lo));
        if (upper)
            hi = mid;
        else
            lo = mid;
    }
    return key_f32(hi);
}

// Four-step binary search over the 15 sorted thresholds.
__device__ __forceinline__ uint32_t code_of(float r, const float* thr) {
    uint32_t c = (r >= thr[7]) ? 8u : 0u;
    c += (r >= thr[c + 3]) ? 4u : 0u;
    c += (r >= thr[c + 1]) ? 2u : 0u;
    c += (r >= thr[c]) ? 1u : 0u;
    return c;
}

// Code of w / d with r = RN(w / d) as the format defines it, cheaply in almost every case.  Fast
// path: q = w * rcp, rcp an approximation of 1 / d (relative error <= 2^-23), so |q - r| <= 2^-22 |r|;
// a bucket table indexed by round(32 q + 32) gives the code c0 at the bucket's low end and the one
// threshold inside the bucket (buckets are 1/32 wide, thresholds at least 0.08 apart), so the
// candidate code is c0 + (q >= threshold).  The candidate is accepted only when q lies strictly inside
// that code's interval shrunk by 2^-20 of each bound's magnitude (bnd): then r, within 2^-22 |r| of
// q, lies inside the interval as well and has the same code.  Otherwise (a weight within about a
// millionth of a threshold, or a non-finite q from a subnormal divisor) the exact division and search
// decide.  The result never depends on the fast path: only its speed does.
__device__ __forceinline__ uint32_t fast_code(float w, float rcp, float d, const float* thr, const float2* bnd,
                                              const float2* bkt) {
    const float q = __fmul_rn(w, rcp);
    // 2^23 + 32 + 32 q rounded to an integer: its low bits are the bucket (0..64 for |q| <= 1)
    const uint32_t j = min(static_cast<uint32_t>(__float_as_int(__fmaf_rn(q, 32.0f, 8388640.0f)) - 0x4B000000), 64u);
    const float2 b = bkt[j];
    uint32_t c = __float_as_uint(b.x) + (q >= b.y ? 1u : 0u);
    const float2 lh = bnd[c];
    if (!(q > lh.x && q < lh.y)) c = code_of(__fdiv_rn(w, d), thr);
    return c;
}

// Eight lanes per group, eight weights per lane: a warp takes kQuantGroups consecutive groups per
// step, as kQuantGroups / 4 rounds of four groups (lane l: group 4 * round + l / 8 of the step,
// weights 8 (l % 8) .. 8 (l % 8) + 7 of it), and issues every round's loads before it computes any.
// A group's absmax takes three shuffle steps; a lane packs its eight codes into one 32-bit word, so
// a round's code stores are 128 contiguous bytes.  An all-zero group divides by 1 instead of by s = 0,
// which turns its weights (+0 or -0) into r = +-0, whose code is 7 (T[7] = 0) as the format requires.
constexpr int kQuantGroups = 8;
constexpr int kQuantRounds = kQuantGroups / 4;

__global__ void __launch_bounds__(256, 5) quantize_kernel(const float* __restrict__ w, int64_t groups,
                                                       uint32_t* __restrict__ codes,
                                                       uint16_t* __restrict__ scales) {
    __shared__ float thr[16];
    __shared__ float2 bnd[16];  // per code: its interval [thr[c-1], thr[c]) shrunk by 2^-20 of each bound
    __shared__ float2 bkt[65];  // per bucket: (code at its low end as integer bits, threshold inside or +inf)
    if (threadIdx.x < 15) thr[threadIdx.x] = decision_threshold(threadIdx.x);
    __syncthreads();
    if (threadIdx.x < 16) {
        const int c = threadIdx.x;
        const float lo = c == 0 ? -INFINITY : thr[c - 1], hi = c == 15 ? INFINITY : thr[c];
        bnd[c] = make_float2(c == 0 ? lo : lo + fabsf(lo) * 0x1p-20f, c == 15 ? hi : hi - fabsf(hi) * 0x1p-20f);
    } else if (threadIdx.x >= 32 && threadIdx.x < 32 + 65) {
        // bucket j holds the q with round(32 q + 32) = j: q in about [(j - 0.5) / 32 - 1, (j + 0.5) / 32 - 1]
        const int j = threadIdx.x - 32;
        const float qlo = (j - 0.5f) / 32.0f - 1.0f, qhi = (j + 0.5f) / 32.0f - 1.0f;
        const uint32_t c0 = code_of(qlo, thr);
        const float t = c0 < 15 && thr[c0] <= qhi ? thr[c0] : INFINITY;
        bkt[j] = make_float2(__uint_as_float(c0), t);
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, sub = lane >> 3, l8 = lane & 7;
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t g0 = ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * kQuantGroups;
         g0 < groups; g0 += warps * kQuantGroups) {
        float4 va[kQuantRounds], vb[kQuantRounds];
#pragma unroll
        for (int r = 0; r < kQuantRounds; r++) {
            const int64_t g = g0 + 4 * r + sub;
            const float4* src = reinterpret_cast<const float4*>(w + g * kGroup) + 2 * l8;
            va[r] = g < groups ? __ldcs(src) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            vb[r] = g < groups ? __ldcs(src + 1) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int r = 0; r < kQuantRounds; r++) {
            const float x[8] = {va[r].x, va[r].y, va[r].z, va[r].w, vb[r].x, vb[r].y, vb[r].z, vb[r].w};
            float s = fabsf(x[0]);
#pragma unroll
            for (int i = 1; i < 8; i++) s = fmaxf(s, fabsf(x[i]));
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) s = fmaxf(s, __shfl_xor_sync(0xFFFFFFFFu, s, o));
            const float d = s != 0.0f ? s : 1.0f;
            float rcp;
            asm("rcp.approx.f32 %0, %1;" : "=f"(rcp) : "f"(d));
            // outside [2^-120, 2^120] the reciprocal may leave the normal range: NaN sends every weight
            // of the group to the exact path
            if (!(d > 0x1p-120f && d < 0x1p120f)) rcp = __int_as_float(0x7FC00000);
            uint32_t word = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) word |= fast_code(x[i], rcp, d, thr, bnd, bkt) << (4 * i);
            const int64_t g = g0 + 4 * r + sub;
            if (g < groups) {
                codes[g * (kGroup / 8) + l8] = word;
                if (l8 == 0) scales[g] = __half_as_ushort(__float2half_rn(s));
            }
        }
    }
}

// Eight weights (four code bytes, one 32-bit word) -> four bf16 pairs through the half-size pair
// table at shared-window address `ptab` (lcol16 = 16 * (lane % 16)).
__device__ __forceinline__ void dequant8(uint32_t word, float s, uint32_t ptab, uint32_t lcol16, uint32_t (&out)[4]) {
#pragma unroll
    for (int b = 0; b < 4; b++) out[b] = scale_pair(lds_f2(ptab + pair_offset16(word, lcol16, b)), s);
}

// Dequant: 8-weight chunks (chunk c = weights 8c .. 8c+7 of the flat [N][K] array, group c / 8).  In
// each of kDequantUnroll rounds lane l of a warp takes chunk base + 32 * round + l, so one warp's
// 16-byte stores cover 512 contiguous bytes of w_hat; all rounds' loads are issued first.
constexpr int kDequantUnroll = 4;
constexpr int kDequantThreads = 512;

__global__ void __launch_bounds__(kDequantThreads, 2048 / kDequantThreads) dequant_kernel(const uint32_t* __restrict__ codes,
                                                                  const uint16_t* __restrict__ scales, int64_t chunks,
                                                                  uint16_t* __restrict__ w_hat) {
    __shared__ __align__(16) float2 tab[kPairTab16Bytes / 8];
    build_pair_table16(tab, threadIdx.x, blockDim.x);
    __syncthreads();
    const uint32_t ptab = smem_u32(tab);
    const int lane = threadIdx.x & 31;
    const uint32_t lcol16 = static_cast<uint32_t>(lane & 15) * 16;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t c0 = warp * 32 * kDequantUnroll; c0 < chunks; c0 += warps * 32 * kDequantUnroll) {
        uint32_t cw[kDequantUnroll];
        uint16_t sc[kDequantUnroll];
#pragma unroll
        for (int u = 0; u < kDequantUnroll; u++) {
            const int64_t c = c0 + 32 * u + lane;
            cw[u] = c < chunks ? __ldcs(codes + c) : 0u;
            sc[u] = c < chunks ? scales[c >> 3] : static_cast<uint16_t>(0);
        }
#pragma unroll
        for (int u = 0; u < kDequantUnroll; u++) {
            const int64_t c = c0 + 32 * u + lane;
            uint32_t out[4];
            dequant8(cw[u], __half2float(__ushort_as_half(sc[u])), ptab, lcol16, out);
            if (c < chunks) __stcs(reinterpret_cast<uint4*>(w_hat) + c, make_uint4(out[0], out[1], out[2], out[3]));
        }
    }
}

// Error word of nf4_embed (41: an id outside the table).
__device__ int g_embed_error;

// Packed embedding rows: thread per quarter group (16 weights) of a requested row, the same exact
// arithmetic as dequant_kernel (bf16(fp32(T[c] * scale)) per weight, from a 16-entry table: a
// launch of a few thousand rows is too short to amortise the pair table); an id outside [0, V)
// writes zeros and records 41.
__global__ void __launch_bounds__(256) embed_kernel(const int32_t* __restrict__ ids, int64_t n_ids,
                                                    const uint8_t* __restrict__ codes,
                                                    const uint16_t* __restrict__ scales, int64_t V, int64_t K,
                                                    uint16_t* __restrict__ out) {
    __shared__ float table[16];
    if (threadIdx.x < 16) table[threadIdx.x] = kNF4[threadIdx.x];
    __syncthreads();
    const int64_t qpr = K / 16;  // quarter groups per row
    const int64_t quarters = n_ids * qpr;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < quarters; q += stride) {
        const int64_t i = q / qpr, qq = q - i * qpr;
        const int64_t id = ids[i];
        uint32_t o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (id >= 0 && id < V) {
            const int64_t src = id * qpr + qq;  // quarter index inside the table
            const uint2 cw = *(reinterpret_cast<const uint2*>(codes) + src);
            const float s = __half2float(__ushort_as_half(scales[src >> 2]));
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const uint32_t byte = ((j < 4 ? cw.x : cw.y) >> (8 * (j & 3))) & 0xFFu;
                const uint32_t lo = bf16_bits(__fmul_rn(table[byte & 0xFu], s));
                const uint32_t hi = bf16_bits(__fmul_rn(table[byte >> 4], s));
                o[j] = lo | (hi << 16);
            }
        } else if (qq == 0) {
            atomicCAS(&g_embed_error, 0, 41);
        }
        uint4* dst = reinterpret_cast<uint4*>(out + q * 16);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

int grid_for(int64_t items_per_block_units, int64_t units, int num_sms, int blocks_per_sm) {
    int64_t blocks = (units + items_per_block_units - 1) / items_per_block_units;
    int64_t cap = static_cast<int64_t>(num_sms) * blocks_per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

}  // namespace

cudaError_t launch_quantize(const float* w, int64_t N, int64_t K, uint8_t* codes, uint16_t* scales,
                            int num_sms, cudaStream_t stream) {
    const int64_t groups = N * (K / kGroup);
    if (groups == 0) return cudaSuccess;
    const int grid = grid_for(8 * kQuantGroups, groups, num_sms, 5);  // 8 warps per block, 5 blocks resident
    quantize_kernel<<<grid, 256, 0, stream>>>(w, groups, reinterpret_cast<uint32_t*>(codes), scales);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                           uint16_t* w_hat, int num_sms, cudaStream_t stream) {
    const int64_t chunks = N * K / 8;
    if (chunks == 0) return cudaSuccess;
    const int grid = grid_for(static_cast<int64_t>(kDequantThreads) * kDequantUnroll, chunks, num_sms,
                              2048 / kDequantThreads);
    dequant_kernel<<<grid, kDequantThreads, 0, stream>>>(reinterpret_cast<const uint32_t*>(codes), scales, chunks,
                                                          w_hat);
    return cudaGetLastError();
}

cudaError_t launch_embed(const int32_t* ids, int64_t n_ids, const uint8_t* codes, const uint16_t* scales, int64_t V,
                         int64_t K, uint16_t* out, int num_sms, cudaStream_t stream) {
    const int64_t quarters = n_ids * (K / 16);
    if (quarters == 0) return cudaSuccess;
    const int grid = grid_for(256, quarters, num_sms, 8);
    embed_kernel<<<grid, 256, 0, stream>>>(ids, n_ids, codes, scales, V, K, out);
    return cudaGetLastError();
}

cudaError_t read_and_clear_embed_error(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_embed_error, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_embed_error, &zero, sizeof(int));
    *code = v;
    return e;
}

}  // namespace nf4
