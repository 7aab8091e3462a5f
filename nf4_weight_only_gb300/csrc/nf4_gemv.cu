// NF4 GEMV family on CUDA cores (sm_103a): y[M, N] = x[M, K] * w_hat[N, K]^T for 1 <= M <= 3.
//
// Decode is weight streaming (deep-fold README, execution-path table: the N=1 decode step runs a
// GEMV on CUDA cores and dequantizes only the current tile).  The kernel's job is to consume the
// packed codes at HBM speed, which leaves about three to four issue slots per weight on a GB300.
//
// Dequantization (helpers in nf4_device.cuh).  The GEMV computes w_hat = bf16(fp32(T[c] * scale))
// as the definition states, two weights at a time: a code byte (two codes) indexes a 256-entry
// shared-memory table whose entry is the fp32 pair {T[low nibble], T[high nibble]}; one packed
// fp32x2 multiply by the group's scale (round to nearest) and one bf16x2 conversion (round to
// nearest even) give both weights.
// The table is replicated across the 32 lanes (entry v, lane l at byte 256 v + 8 l), so a warp's
// 64-bit loads hit 32 distinct bank pairs per half-warp whatever the codes are; one byte permute
// builds that address from the code word.  Eight weights cost 4 permutes, 4 shared loads, 4 packed
// multiplies and 4 conversions before the multiply-adds: the loop is bound by shared-memory
// bandwidth (8 bytes per 2 weights), about 1.4 times the rate of a 16-entry register lookup done
// with byte permutes, which is bound by the integer pipe.  A lane sums x_k * w_hat_k in fp32 (each
// bf16 x bf16 product is exact).
//
// Work layout.  A warp owns a K-slice (32 groups at one lane per group, or 16 groups at two lanes
// per group) and keeps that slice of x in registers as bf16 pairs; it streams four rows at a time
// (128-bit loads), reduces the four row partial sums across lanes with a transposed butterfly and
// hands them to the CTA, whose warps cover all slices of the same rows; slice sums are added in a
// fixed order, so results are deterministic.  The grid is persistent: each CTA owns a contiguous
// range of rows (the rows split as evenly as the grid allows) and walks it in row blocks.
#include <mutex>

#include <cudaTypedefs.h>

#include "nf4_device.cuh"
#include "nf4_internal.h"

namespace nf4 {
namespace {

constexpr int kMaxWarps = 16;  // consumer warps per CTA (slices x row lanes)
constexpr int kHalfWarps = 8;  // consumer warps of a CTA that leaves room for a second one
constexpr int kHalfSmem = 113 * 1024;  // shared memory of such a CTA
constexpr int kMinStages = 3;          // ring stages a CTA with several K-slices keeps at least

// First stage of summing each of V values over the 32 lanes.  Recursive halving: at each of log2(V)
// steps a lane keeps the half of its values selected by one lane bit and adds its partner's copy of
// that half.  Afterwards lane l holds a partial sum of value l >> (5 - log2 V), and the 32 / V
// consecutive lanes of a value hold its whole sum between them.
template <int V>
__device__ __forceinline__ float reduce_halving(float (&v)[V], int lane) {
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

// Error word of the bounded pipeline waits of both kernels in this translation unit.
__device__ int g_tc_error;
__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_tc_error, 0, code); }

// Wall-clock limit of one pipeline wait, in nanoseconds (1 s by default: a wait that long means a
// bug, not a slow GPU).  Every wait has its own limit, so no kernel length can exhaust it.
__device__ unsigned long long g_wait_ns = 1000000000ull;

// Sleep between the tests of the producer's and the reducer's waits (mbar_wait_idle): both wait
// most of the time, and neither is on the consumers' critical path while the ring has room.
constexpr uint32_t kIdleSleepNs = 256;

// Per-row metadata the producer writes next to each row's data.
struct RowMeta {
    int problem;     // index into GemvProblems
    int local_row;   // row inside that problem
    int scale_off;   // byte offset of the row's first scale inside its 16-byte-aligned window
    int valid;       // row < total rows
};

// Launch-time layout of one ring stage (host and device agree on it).
struct GemvLayout {
    int S, Q, R;         // K-slices, row lanes per slice, rows per consumer warp per block
    int RB;              // rows per block = Q * R
    int ST;              // ring stages
    int row_code_bytes;  // K / 2: one row's codes, copied as they lie in memory
    int swin;            // bytes of one row's scale window (multiple of 16)
    int stage_bytes;     // RB * (row_code_bytes + swin) + RB * 16 (meta) + C * 128 (partials)
    int red_off;         // offset of the [C][32] halved partial sums (one float per consumer lane)
    int meta_off;
    int scales_off;
};

// Warp-specialised GEMV.  Warps 0..C-1 (C = S * Q) consume: warp c owns slice c % S and rows
// (c / S) * R .. +R of every row block, keeps its slice of x in registers and runs the lookups and
// fused multiply-adds.  Warp C produces: for each row block it waits until the ring stage is free,
// copies the block's codes (16-byte chunks, consecutive lanes on consecutive chunks, each chunk
// placed in the swizzled slot of the consumer lane that owns it), the rows' scale windows and their
// metadata, and arms the stage's `full` barrier through cp.async.mbarrier.arrive.  After a block
// each consumer warp halves its per-row sums across lanes once per value bit, leaves one float per
// lane in the stage and moves on; warp C + 1 (the reducer) adds, for every row of the block, the
// lanes and slices that hold it in a fixed order, writes y and releases the stage.  The consumers
// thus never wait on a reduction chain, and the result does not depend on the launch shape.
// Every wait is bounded; after a timeout the waiting thread records an error code and stops.
// RMAX bounds the rows a consumer warp takes per block (the launcher picks R <= RMAX).  T16 selects
// the half-size pair table (16 copies, 32 KB; one extra shift per lookup), which leaves room for
// longer rows in the ring.
template <int MT, int LPG, int RMAX, bool T16>
__global__ void __launch_bounds__((kMaxWarps + 2) * 32, 1)
    gemv_kernel(const uint16_t* __restrict__ x, const __grid_constant__ GemvProblems P, int K,
                const GemvLayout L) {
    constexpr uint32_t kTab = T16 ? kPairTab16Bytes : kPairTabBytes;  // the table, then the ring
    constexpr int WPL = kGroup / LPG;  // weights per consumer lane per row
    constexpr int CB = WPL / 2;        // code bytes per consumer lane per row
    constexpr int CHUNKS = CB / 16;
    constexpr int GPW = 32 / LPG;      // groups per slice
    constexpr int V = pow2_ceil(RMAX * MT);
    extern __shared__ __align__(16) uint8_t smem[];

    const int N = P.row0[P.count];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int C = L.S * L.Q;
    const int G = K / kGroup;
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    uint8_t* ring = smem + kTab;
    const uint32_t bars = sbase + kTab + L.ST * L.stage_bytes;  // full[ST], empty[ST], part[ST]
    // this CTA's rows: a contiguous range, the N rows split as evenly as the grid allows
    const int64_t rbeg = static_cast<int64_t>(N) * blockIdx.x / gridDim.x;
    const int64_t rend = static_cast<int64_t>(N) * (blockIdx.x + 1) / gridDim.x;
    const int64_t my_blocks = (rend - rbeg + L.RB - 1) / L.RB;

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int st = 0; st < L.ST; st++) {
            mbar_init(bars + 8 * st, 33);  // full: per producer lane after its copies, + lane 0 after the metadata
            mbar_init(bars + 8 * (L.ST + st), 1);   // empty: the reducer is done with the stage
            mbar_init(bars + 8 * (2 * L.ST + st), C);  // part: consumer partials written
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint64_t wait_ns = g_wait_ns;

    if (warp == C + 1) {
        // ------------------------------------------------------------------ reducer
        constexpr int LPV = 32 / V;  // lanes holding one value after the halving steps
        int st = 0, par = 0;
        for (int64_t t = 0; t < my_blocks; t++, st = st + 1 == L.ST ? 0 : st + 1, par ^= st == 0) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_idle(bars + 8 * (2 * L.ST + st), par, wait_ns, kIdleSleepNs))) {
                record_error(13);
                break;
            }
            const uint8_t* stg = ring + st * L.stage_bytes;
            const float* red = reinterpret_cast<const float*>(stg + L.red_off);
            for (int i = lane; i < L.RB * MT; i += 32) {
                const int j = i / MT, tt = i - j * MT;
                const RowMeta meta = *reinterpret_cast<const RowMeta*>(stg + L.meta_off + 16 * j);
                if (!meta.valid || meta.problem >= P.count) continue;
                const int q = j / L.R, v = (j - q * L.R) * MT + tt;
                float acc = 0.0f;
                for (int ss = 0; ss < L.S; ss++) {
                    const float4* src = reinterpret_cast<const float4*>(red + (q * L.S + ss) * 32 + v * LPV);
                    float sub = 0.0f;
#pragma unroll
                    for (int c = 0; c < LPV / 4; c++) {
                        // start rotated by the row (fewer bank conflicts, same order for any launch shape)
                        const float4 f = src[(c + meta.local_row) & (LPV / 4 - 1)];
                        sub += (f.x + f.y) + (f.z + f.w);
                    }
                    acc += sub;
                }
                const int np = P.row0[meta.problem + 1] - P.row0[meta.problem];
                P.y[meta.problem][static_cast<int64_t>(tt) * np + meta.local_row] = bf16_bits(acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8 * (L.ST + st));
        }
    } else if (warp == C) {
        // ------------------------------------------------------------------ producer
        // The producer moves weights only (codes, scales, row metadata into shared memory), which
        // the previous grid in the stream does not write: it starts at once, without the
        // programmatic-dependent-launch wait, so that the first blocks arrive while that grid's last
        // CTAs finish.  The consumers wait for it before they read x and write y.
        // Lane j copies rows j, j + 32, ... of the block: each row's codes with one bulk copy
        // (transaction bytes on the stage's `full` barrier) and its scale window with zero-filling
        // 16-byte copies.  Every row of the block gets its metadata (valid = 0 past the end).
        int st = 0, round = 0;  // ring stage of block t and how often the ring has wrapped
        for (int64_t t = 0; t < my_blocks; t++, st = st + 1 == L.ST ? 0 : st + 1, round += st == 0) {
            if (round > 0 && !__all_sync(0xFFFFFFFFu, mbar_wait_idle(bars + 8 * (L.ST + st), (round - 1) & 1, wait_ns, kIdleSleepNs))) {
                record_error(11);
                break;
            }
            uint8_t* stg = ring + st * L.stage_bytes;
            const int64_t r0 = rbeg + t * L.RB;
            const int64_t valid_rows = rend - r0 < L.RB ? rend - r0 : L.RB;
            if (lane == 0) mbar_expect_tx_only(bars + 8 * st, static_cast<uint32_t>(valid_rows * (K / 2)));
            __syncwarp();
            for (int j = lane; j < L.RB; j += 32) {
                const int64_t r = r0 + j;
                RowMeta meta = {0, 0, 0, 0};
                if (r < rend) {
                    const int pp = problem_of(P, r);
                    const int64_t lr = r - P.row0[pp];
                    bulk_copy_g2s(sbase + static_cast<uint32_t>(kTab + st * L.stage_bytes + j * L.row_code_bytes),
                                  P.codes[pp] + lr * (K / 2), static_cast<uint32_t>(K / 2), bars + 8 * st);
                    const int64_t sfirst = lr * G * 2;
                    const int64_t a = sfirst & ~static_cast<int64_t>(15);
                    const int64_t total = static_cast<int64_t>(P.row0[pp + 1] - P.row0[pp]) * G * 2;
                    const uint8_t* sp = reinterpret_cast<const uint8_t*>(P.scales[pp]);
                    for (int64_t c = a; c < sfirst + 2 * G; c += 16) {
                        const int64_t left = total - c;
                        cp_async16(stg + L.scales_off + j * L.swin + (c - a), sp + c,
                                   static_cast<uint32_t>(left < 16 ? left : 16));
                    }
                    meta = {pp, static_cast<int>(lr), static_cast<int>(sfirst - a), 1};
                }
                *reinterpret_cast<RowMeta*>(stg + L.meta_off + 16 * j) = meta;
            }
            // full = the bulk bytes + every lane's small copies (asynchronous arrive per lane) +
            // lane 0's release of the metadata written by the whole warp
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bars + 8 * st) : "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8 * st);
        }
        cp_async_wait<0>();
    } else {
        // ------------------------------------------------------------------ consumers
        const int s = warp % L.S, q = warp / L.S;
        const int g = s * GPW + lane / LPG;
        const bool active = g < G;
        const int k0 = s * GPW * kGroup + lane * WPL;
        // Lanes whose bit 2 is set read the two 16-byte halves of their 32 code bytes in the other
        // order (no bank conflicts for eight lanes 32 bytes apart); x is loaded in the same order.
        const int sw = LPG == 1 ? ((lane >> 2) & 1) : 0;
        // The pair table is for the consumers alone: they write it while the producer already streams
        // the first row blocks, and meet on a named barrier before the first lookup.
        if constexpr (T16)
            build_pair_table16(reinterpret_cast<float2*>(smem), threadIdx.x, 32 * C);
        else
            build_pair_table(reinterpret_cast<float2*>(smem), threadIdx.x, 32 * C);
        pdl_wait();
        uint32_t xr[MT][WPL / 2];
#pragma unroll
        for (int tt = 0; tt < MT; tt++) {
#pragma unroll
            for (int i = 0; i < WPL / 8; i++) {
                uint4 v = make_uint4(0, 0, 0, 0);
                const int isrc = i ^ (sw * (WPL / 16));  // swap the halves for swizzled lanes
                if (active) v = *reinterpret_cast<const uint4*>(x + static_cast<int64_t>(tt) * K + k0 + 8 * isrc);
                xr[tt][4 * i + 0] = v.x;
                xr[tt][4 * i + 1] = v.y;
                xr[tt][4 * i + 2] = v.z;
                xr[tt][4 * i + 3] = v.w;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(32 * C) : "memory");  // every consumer's table entries written
        // this lane's column in every table entry (twice its copy offset for the half-size table)
        const uint32_t lcol = T16 ? static_cast<uint32_t>(lane & 15) * 16 : static_cast<uint32_t>(lane) * 8;
        int st = 0, par = 0;  // ring stage of block t and the phase parity of its barriers
        for (int64_t t = 0; t < my_blocks; t++, st = st + 1 == L.ST ? 0 : st + 1, par ^= st == 0) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(bars + 8 * st, par, wait_ns))) {
                record_error(12);
                break;
            }
            // With several blocks per CTA, the upper half of the consumer warps starts about half a
            // block later: the warps of a CTA then no longer reach their latency-bound steps
            // (prologue loads, reduction, write-back) together, and the SM keeps issuing lookups.
            if (t == 0 && my_blocks >= 3 && ((warp >> 2) & 1)) __nanosleep(400u * L.R);
            const uint8_t* stg = ring + st * L.stage_bytes;
            float part[V];
#pragma unroll
            for (int i = 0; i < V; i++) part[i] = 0.0f;
            // Row prologues first (metadata -> scale is a chain of dependent shared-memory loads), for
            // all of this warp's rows of the block, so that their latencies overlap.
            float scl[RMAX];
            bool rv[RMAX];
#pragma unroll
            for (int jj = 0; jj < RMAX; jj++) {
                const int j = q * L.R + jj;
                RowMeta meta = {0, 0, 0, 0};
                if (jj < L.R) meta = *reinterpret_cast<const RowMeta*>(stg + L.meta_off + 16 * j);  // warp-uniform
                rv[jj] = meta.valid && meta.problem < P.count;
                uint32_t sc = 0;
                if (rv[jj] && active)
                    sc = *reinterpret_cast<const uint16_t*>(stg + L.scales_off + j * L.swin + meta.scale_off + 2 * g);
                scl[jj] = __half2float(__ushort_as_half(static_cast<uint16_t>(sc)));  // exact
            }
#pragma unroll
            for (int jj = 0; jj < RMAX; jj++) {
                if (!rv[jj]) continue;  // warp-uniform
                const int j = q * L.R + jj;
                float a0[MT], a1[MT];
#pragma unroll
                for (int tt = 0; tt < MT; tt++) a0[tt] = a1[tt] = 0.0f;
                // A lane past the last group reads its row's first bytes instead (its x is zero), so
                // that no read leaves the row block.
                const uint8_t* crow = stg + j * L.row_code_bytes + (active ? s * 32 * CB + lane * CB : 0);
#pragma unroll
                for (int c = 0; c < CHUNKS; c++) {
                    const uint4 cw = lds128(crow + 16 * (c ^ sw));
                    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int wi = 0; wi < 4; wi++) {
#pragma unroll
                        for (int p = 0; p < 4; p++) {
                            const uint32_t off = T16 ? pair_offset16(words[wi], lcol, p) : pair_offset(words[wi], lcol, p);
                            const uint32_t wp = scale_pair(*reinterpret_cast<const float2*>(smem + off), scl[jj]);
#pragma unroll
                            for (int tt = 0; tt < MT; tt++) fma_bf16x2(a0[tt], a1[tt], wp, xr[tt][4 * (4 * c + wi) + p]);
                        }
                    }
                }
#pragma unroll
                for (int tt = 0; tt < MT; tt++) part[jj * MT + tt] = a0[tt] + a1[tt];
            }
            // leave this warp's halved sums in the stage for the reducer
            float* red = reinterpret_cast<float*>(ring + st * L.stage_bytes + L.red_off);
            red[warp * 32 + lane] = reduce_halving<V>(part, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8 * (2 * L.ST + st));
        }
    }
}

template <int MT, int LPG, int RMAX, bool T16>
cudaError_t launch_gemv_t(const uint16_t* x, const GemvProblems& P, int64_t K, int num_sms, cudaStream_t stream) {
    constexpr int kTab = T16 ? kPairTab16Bytes : kPairTabBytes;
    constexpr int GPW = 32 / LPG;
    const int64_t N = P.row0[P.count];
    const int G = static_cast<int>(K / kGroup);
    GemvLayout L = {};
    L.S = (G + GPW - 1) / GPW;
    // Launch shape (measured on the 3B-shaped decode pass: 144 launches in one graph, chained by
    // programmatic dependent launch):
    //  - K over several slices: whole-SM CTAs, RMAX rows per warp (fewer when a block that large
    //    leaves a ring of fewer than kMinStages stages), as many row lanes as the rows need, the
    //    deepest ring that fits;
    //  - one slice and up to 2 * kMaxWarps rows per SM: row blocks sized for about 1.7 blocks per
    //    CTA (two rows per warp when a block has at most 8 rows), so that the weights of a CTA's
    //    second block arrive while its first is computed, and a two-stage ring, which leaves room on
    //    the SM for a CTA of the next launch;
    //  - one slice and more rows: two CTAs per SM of kHalfWarps warps with two rows each and half
    //    the shared memory; the two CTAs interleave their waits and tails.
    bool half = false;
    bool cap_ring = false;    // ring no deeper than the CTA's row blocks
    int64_t slots = num_sms;  // CTAs resident at once
    const int swin = ((2 * G + 15) / 16 + 1) * 16;
    const auto stage_of = [&](int q, int r) {  // bytes of one ring stage (see the layout below)
        return static_cast<int64_t>(q) * r * (K / 2 + swin + 16) + static_cast<int64_t>(L.S) * q * 32 * 4;
    };
    if (L.S > 1) {
        const int qmax = L.S >= kMaxWarps ? 1 : kMaxWarps / L.S;
        for (L.R = RMAX;; L.R--) {
            const int64_t q_needed = (N + static_cast<int64_t>(L.R) * num_sms - 1) / (static_cast<int64_t>(L.R) * num_sms);
            L.Q = static_cast<int>(q_needed < 1 ? 1 : (q_needed > qmax ? qmax : q_needed));
            if (L.R == 1 || (227 * 1024 - kTab - 256) / stage_of(L.Q, L.R) >= kMinStages) break;
        }
    } else if (N <= static_cast<int64_t>(2) * kMaxWarps * num_sms) {
        cap_ring = true;
        const int64_t rb = (N * 10 + 17LL * num_sms - 1) / (17LL * num_sms);  // rows per block
        L.R = (rb <= 8 && RMAX >= 2) ? 2 : 1;
        const int64_t q = (rb + L.R - 1) / L.R;
        L.Q = static_cast<int>(q < 1 ? 1 : (q > kMaxWarps ? kMaxWarps : q));
    } else {
        half = true;
        cap_ring = true;
        slots = 2LL * num_sms;
        L.R = RMAX < 2 ? RMAX : 2;
        L.Q = kHalfWarps;
    }
    const int64_t nblocks_all = (N + static_cast<int64_t>(L.R) * L.Q - 1) / (static_cast<int64_t>(L.R) * L.Q);
    const int64_t grid64 = nblocks_all < slots ? nblocks_all : slots;
    L.RB = L.Q * L.R;
    L.row_code_bytes = static_cast<int>(K / 2);
    L.swin = swin;
    L.scales_off = L.RB * L.row_code_bytes;
    L.meta_off = L.scales_off + L.RB * L.swin;
    L.red_off = L.meta_off + 16 * L.RB;
    L.stage_bytes = L.red_off + L.S * L.Q * 32 * 4;  // one float per consumer lane
    // ring depth: as many stages as fit next to the pair table in the CTA's share of shared memory (at
    // most 8, at least 2; see cap_ring)
    const int budget = (half ? kHalfSmem : 227 * 1024) - kTab - 3 * 8 * 8 - 64;
    const int64_t blocks_per_cta = ((N + grid64 - 1) / grid64 + L.RB - 1) / L.RB;  // of the largest row range
    L.ST = budget / L.stage_bytes;
    if (L.ST > 8) L.ST = 8;
    if (cap_ring && L.ST > blocks_per_cta) L.ST = static_cast<int>(blocks_per_cta < 2 ? 2 : blocks_per_cta);
    if (L.ST < 2) return cudaErrorInvalidValue;  // a row block does not fit twice
    const int grid = static_cast<int>(grid64);
    const size_t smem = kTab + static_cast<size_t>(L.ST) * L.stage_bytes + 3 * 8 * L.ST;
    static std::once_flag attr_once[64];  // the largest possible request, set once per device
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once[dev & 63], [&] {
        attr_err = cudaFuncSetAttribute(gemv_kernel<MT, LPG, RMAX, T16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * (L.S * L.Q + 2));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<MT, LPG, RMAX, T16>, x, P, static_cast<int>(K), L);
}

}  // namespace
}  // namespace nf4

#include "nf4_stream.cuh"
#include "nf4_narrow.cuh"

namespace nf4 {
namespace {

// cuTensorMapEncodeTiled is a driver call and needs a current context.  A host thread whose first
// CUDA work in this library is a tensor-map encode may not have one yet: the runtime binds the
// primary context to a thread lazily, at its first call that needs it.  Bind it here when the thread
// has no context at all (a context the caller made current is left alone).
cudaError_t ensure_current_context() {
    static PFN_cuCtxGetCurrent_v4000 get = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        else
            cudaGetLastError();
    });
    CUcontext c = nullptr;
    if (get && get(&c) == CUDA_SUCCESS && c != nullptr) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return cudaSetDevice(dev);
}

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

}  // namespace

namespace {

// Small-M weight streaming on the tensor cores (nf4_stream.cuh): one CTA per SM, each with a balanced
// range of rows of one problem.
template <int T>
cudaError_t launch_stream_t(const uint16_t* x, st::Params& P, int64_t M, int64_t K, cudaStream_t stream) {
    using C = st::Cfg<T>;
    auto encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    if (const cudaError_t e = ensure_current_context(); e != cudaSuccess) return e;
    // x: bf16 [M][K] viewed as [M][G][64]; a box is T tokens x S consecutive groups x 64, which lands
    // as pseudo-token rows t * S + s of 128 bytes (128-byte swizzle).  Groups past G and tokens past M
    // read as zero.
    CUtensorMap maps[2];
    const int slices[2] = {1, P.s_rem};
    for (int v = 0; v < 2; v++) {
        const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(K / 64), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(slices[v]), static_cast<cuuint32_t>(T)};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&maps[v], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(x), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // codes of each linear: uint8 [N][K/2]; full tiles load 128 rows x 128 bytes (4 groups) with the
    // 128-byte swizzle, partial tiles r_rem rows x 32 * box_span(s_rem) * s_rem bytes
    st::CodeMaps cm = {};
    const uint32_t rem_bytes = 32u * st::box_span(P.s_rem) * P.s_rem;
    for (int i = 0; i < P.count; i++) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(P.n[i])};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
        const cuuint32_t estr[2] = {1, 1};
        const cuuint32_t box_full[2] = {128, 128};
        const cuuint32_t box_rem[2] = {rem_bytes, static_cast<cuuint32_t>(P.r_rem > 0 ? P.r_rem : 1)};
        if (encode(&cm.full[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(P.codes[i]), dims, strides,
                   box_full, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
            encode(&cm.rem[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(P.codes[i]), dims, strides,
                   box_rem, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   rem_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // T <= 32: the small-M kernel (nf4_narrow.cuh); wider tiles: the GEMM form (nf4_stream.cuh)
    uint32_t kBytes;
    int kThreads;
    void (*kernel)(const CUtensorMap, const CUtensorMap, const st::CodeMaps, const st::Params);
    if constexpr (T <= 32) {
        // the narrow kernel's B tile holds T tokens x s_rem slices (its shared memory is sized for it)
        if (P.s_rem < 1 || P.s_rem > st::NCfg<T>::kSMax || 4 * (32 / P.s_rem) < P.r_rem ||
            T * P.s_rem > st::NCfg<T>::kJMax)
            return cudaErrorInvalidValue;
        kBytes = st::NCfg<T>::kBytes;
        kThreads = st::NCfg<T>::kThreads;
        kernel = st::narrow_kernel<T>;
    } else {
        kBytes = C::kBytes;
        kThreads = C::kThreads;
        kernel = st::stream_kernel<T>;
    }
    const size_t smem = kBytes + 1024;  // + slack to align the base to 1024 bytes
    static std::once_flag attr_once[64];
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once[dev & 63], [&] {
        attr_err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(P.cta0[P.count]), static_cast<unsigned>((M + T - 1) / T));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, maps[0], maps[1], cm, P);
}

}  // namespace

cudaError_t launch_stream(const uint16_t* x, int count, const uint8_t* const* codes, const uint16_t* const* scales,
                          uint16_t* const* ys, const int64_t* Ns, int64_t M, int64_t K, int num_sms,
                          cudaStream_t stream) {
    if (count < 1 || count > st::kMaxProblems || M < 1 || num_sms < 1) return cudaErrorInvalidValue;
    // Token tiles run along the grid's y dimension (at most 65535 of them): a larger M goes in
    // chunks of that many 256-token tiles, each with x and every y offset by the chunk's first
    // token (offsets of whole rows keep the 16-byte alignment the kernels rely on).
    constexpr int64_t kTokensPerLaunch = 65535LL * 256;
    if (M > kTokensPerLaunch) {
        for (int64_t m0 = 0; m0 < M; m0 += kTokensPerLaunch) {
            const int64_t mc = M - m0 < kTokensPerLaunch ? M - m0 : kTokensPerLaunch;
            uint16_t* yc[st::kMaxProblems];
            for (int i = 0; i < count; i++) yc[i] = ys[i] + m0 * Ns[i];
            const cudaError_t e = launch_stream(x + m0 * K, count, codes, scales, yc, Ns, mc, K, num_sms, stream);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    if (M > 32) {  // wide tiles of 128 rows x T tokens
        // CTAs: one per tile while every token tile's tiles fit the SMs; otherwise each token tile
        // gets num_sms / (token tiles) CTAs, shared among the problems in proportion to their tiles,
        // and each CTA walks a balanced run of consecutive tiles (see stream_kernel), unless its
        // longest run would take more tile times than waves of one-tile CTAs do (many token tiles)
        const int64_t tsel = M <= 64 ? 64 : (M <= 128 ? 128 : 256);
        const int64_t gy = (M + tsel - 1) / tsel;
        int64_t tiles[st::kMaxProblems], nc[st::kMaxProblems], total = 0;
        for (int i = 0; i < count; i++) {
            tiles[i] = (Ns[i] + 127) / 128;
            total += tiles[i];
        }
        const int64_t slots = num_sms / gy;
        if (total <= slots || slots < count) {
            for (int i = 0; i < count; i++) nc[i] = tiles[i];
        } else {
            int64_t used = 0;
            for (int i = 0; i < count; i++) {
                nc[i] = slots * tiles[i] / total;
                if (nc[i] < 1) nc[i] = 1;
                if (nc[i] > tiles[i]) nc[i] = tiles[i];
                used += nc[i];
            }
            while (used < slots) {  // the rest to the problems with the longest runs
                int best = -1;
                int64_t best_run = 0;
                for (int i = 0; i < count; i++) {
                    const int64_t run = (tiles[i] + nc[i] - 1) / nc[i];
                    if (nc[i] < tiles[i] && run > best_run) {
                        best_run = run;
                        best = i;
                    }
                }
                if (best < 0) break;
                nc[best]++;
                used++;
            }
            int64_t longest = 0;
            for (int i = 0; i < count; i++) {
                const int64_t run = (tiles[i] + nc[i] - 1) / nc[i];
                if (run > longest) longest = run;
            }
            if (longest > (total * gy + num_sms - 1) / num_sms)
                for (int i = 0; i < count; i++) nc[i] = tiles[i];
        }
        st::Params P = {};
        P.count = count;
        int64_t c = 0;
        for (int i = 0; i < count; i++) {
            P.codes[i] = codes[i];
            P.scales[i] = scales[i];
            P.y[i] = ys[i];
            P.n[i] = static_cast<int>(Ns[i]);
            P.cta0[i] = static_cast<int>(c);
            c += nc[i];
        }
        for (int i = count; i <= st::kMaxProblems; i++) P.cta0[i] = static_cast<int>(c);
        P.rstar = 128;
        P.r_rem = 0;
        P.s_rem = 1;
        P.M = static_cast<int>(M);
        P.K = static_cast<int>(K);
        P.G = static_cast<int>(K / kGroup);
        if (M <= 64) return launch_stream_t<64>(x, P, M, K, stream);
        if (M <= 128) return launch_stream_t<128>(x, P, M, K, stream);
        return launch_stream_t<256>(x, P, M, K, stream);
    }
    const int64_t G = K / kGroup;
    int64_t total = 0;
    for (int i = 0; i < count; i++) total += Ns[i];
    if (total < 1) return cudaErrorInvalidValue;
    // Rows per CTA: the smallest count that needs at most one CTA per SM (each CTA stays in one problem).
    auto ctas = [&](int64_t r) {
        int64_t c = 0;
        for (int i = 0; i < count; i++) c += (Ns[i] + r - 1) / r;
        return c;
    };
    int64_t rpc = (total + num_sms - 1) / num_sms;
    if (rpc < 1) rpc = 1;
    while (ctas(rpc) > num_sms) rpc++;
    st::Params P = {};
    P.count = count;
    int64_t c = 0;
    for (int i = 0; i < count; i++) {
        P.codes[i] = codes[i];
        P.scales[i] = scales[i];
        P.y[i] = ys[i];
        P.n[i] = static_cast<int>(Ns[i]);
        P.cta0[i] = static_cast<int>(c);
        c += (Ns[i] + rpc - 1) / rpc;
    }
    for (int i = count; i <= st::kMaxProblems; i++) P.cta0[i] = static_cast<int>(c);
    P.rstar = static_cast<int>(rpc);
    P.M = static_cast<int>(M);
    P.K = static_cast<int>(K);
    P.G = static_cast<int>(G);
    // K-slices of a partial tile: as many as fit the MMA rows (floor(32 / S) rows in each of the four
    // 32-lane quarters of tensor memory, a row's slices in consecutive lanes), the B tile's
    // pseudo-token columns (smax) and G.
    P.r_rem = static_cast<int>(rpc % 128);
    auto slices = [&](int smax) {
        int best = 1;
        for (int s = 2; s <= smax && s <= G; s++)
            if (4 * (32 / s) >= P.r_rem) best = s;
        return best;
    };
    if (M == 1) {
        P.s_rem = slices(st::NCfg<1>::kSMax);
        return launch_stream_t<1>(x, P, M, K, stream);
    }
    if (M == 2) {
        P.s_rem = slices(st::NCfg<2>::kSMax);
        return launch_stream_t<2>(x, P, M, K, stream);
    }
    if (M <= 4) {
        P.s_rem = slices(st::NCfg<4>::kSMax);
        return launch_stream_t<4>(x, P, M, K, stream);
    }
    if (M <= 8) {
        P.s_rem = slices(st::NCfg<8>::kSMax);
        return launch_stream_t<8>(x, P, M, K, stream);
    }
    if (M <= 16) {
        P.s_rem = slices(st::NCfg<16>::kSMax);
        return launch_stream_t<16>(x, P, M, K, stream);
    }
    P.s_rem = slices(st::NCfg<32>::kSMax);
    return launch_stream_t<32>(x, P, M, K, stream);
}

// One thread waits on an mbarrier that nothing arrives on, with the pipelines' bounded wait and
// error word: after `ns` nanoseconds the wait gives up and records 39 (the check of a timed-out
// wait's reporting path; no fault, no hang).
__global__ void diag_wait_kernel(uint64_t ns) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!mbar_wait(b, 0, ns)) record_error(39);
}

cudaError_t launch_diag_wait(int64_t ns, cudaStream_t stream) {
    diag_wait_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(ns));
    return cudaGetLastError();
}

// Sets the per-wait limit of every pipeline wait on the current device (ns > 0), or restores the
// default of one second (ns = 0).  Stream-ordered after the work already on `stream`.
cudaError_t set_wait_limit(int64_t ns, cudaStream_t stream) {
    const unsigned long long v = ns > 0 ? static_cast<unsigned long long>(ns) : 1000000000ull;
    return cudaMemcpyToSymbolAsync(g_wait_ns, &v, sizeof(v), 0, cudaMemcpyHostToDevice, stream);
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
    switch (M) {
        case 1: {
            // K past one slice (32 groups): four rows per warp, else up to two.  Past one slice,
            // two lanes per group (slices of 16 groups) when that leaves fewer lanes idle: K = 5120
            // is 80 groups, three slices of 32 with 16 lanes idle, or five full slices of 16.
            if (K <= 32 * kGroup) return launch_gemv_t<1, 1, 2, false>(x, P, K, num_sms, stream);
            const int64_t G = K / kGroup;
            const int64_t s1 = (G + 31) / 32, s2 = (G + 15) / 16;
            if (s2 <= kMaxWarps && 16 * s2 < 32 * s1) return launch_gemv_t<1, 2, 4, false>(x, P, K, num_sms, stream);
            // Rows so long that kMinStages blocks of four rows a warp do not fit beside the 64 KB
            // table (K past about 20000): the half-size table keeps four rows a warp (27648-wide
            // rows: 32.6 -> 29.7 us for the 5120-row linear; shorter rows lose by its extra shift).
            const int64_t swin = ((2 * G + 15) / 16 + 1) * 16;
            const int64_t stage4 = 4 * (K / 2 + swin + 16) + s1 * 32 * 4;
            if (kMinStages * stage4 > 227 * 1024 - kPairTabBytes - 256)
                return launch_gemv_t<1, 1, 4, true>(x, P, K, num_sms, stream);
            return launch_gemv_t<1, 1, 4, false>(x, P, K, num_sms, stream);
        }
        case 2: return launch_gemv_t<2, 2, 2, false>(x, P, K, num_sms, stream);
        case 3: return launch_gemv_t<3, 2, 2, false>(x, P, K, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv(const uint16_t* x, const uint8_t* codes, const uint16_t* scales, uint16_t* y,
                        int64_t M, int64_t N, int64_t K, int num_sms, cudaStream_t stream) {
    return launch_gemv_grouped(x, 1, &codes, &scales, &y, &N, M, K, num_sms, stream);
}

}  // namespace nf4
