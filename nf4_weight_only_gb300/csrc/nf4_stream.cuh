// NF4 GEMM-form weight streaming for prefill (M >= 33 positions) on the tcgen05 tensor cores,
// sm_103a: y[M, N] = x[M, K] * w_hat[N, K]^T, dequantizing only the current tile of the packed
// weights (deep-fold README, execution-path table: the prefill GEMM over packed weights).
// stream_kernel<T> is instantiated for T = 64, 128 and 256 tokens per CTA ("wide" tiles); M <= 32
// runs the small-M kernel of nf4_narrow.cuh, M <= 3 with K in range the CUDA-core GEMV.
//
//   dequant warps:  packed codes (shared memory) -> exact bf16 w_hat -> tensor memory (tcgen05.st)
//                   w_hat = bf16(fp32(T[c] * scale)) two weights at a time from the half-size fp32
//                   pair table in shared memory (pair_offset16, scale_pair in nf4_gemv.cu)
//   one warp:       tcgen05.mma, A = that w_hat tile in tensor memory, B = x tile in shared memory
//                   (TMA, 128-byte swizzle), D = fp32 accumulator in tensor memory (N = T)
//
// A CTA owns one tile of 128 rows x T tokens (grid: row tiles x token tiles).  Codes move in load
// stages of four 64-k sub-stages (one TMA box of 128 rows x 128 bytes), x per 64-k sub-tile (one box
// of T tokens), scales per 8 sub-stages (zero-filling 16-byte copies of each row's window).  The
// codes and scale rings are released by every dequant warp (each passes every fill in order), the
// x ring and the tensor-memory ring of A tiles by the MMAs, so each runs as far ahead as its own
// consumers allow.
//
// Warp roles: warp 0 streams codes and scales (lane 0 issues the TMA boxes, the warp copies
// scales), warp 1 owns tensor memory and issues the MMAs (converged, one elected lane), warps
// 2 .. 4*kSets+1 are kSets = 4 sets of four dequant warps (a set takes every fourth stage; the four
// warps of a set cover the four 32-lane quarters of tensor memory), which also run the epilogue,
// and the last warp streams x.  Weights do
// not depend on the previous kernel in the stream, so warp 0 never waits for it; only x and y do.
// (The configuration and tile arithmetic below still carry the K-slice fields of the shared tile
// description, which the wide tiles fix at one slice.)
// Every mbarrier wait is bounded; a wait that runs out records an error code, drains the copies and
// MMAs in flight (bounded again) and frees tensor memory.
#pragma once

#include <cuda.h>

namespace nf4 {
namespace st {

constexpr uint32_t kScaleSlot = 6144;           // R * (S + 2) 16-byte chunks with R * S <= 128
constexpr uint32_t kLoadBytes = 16384;          // one codes load stage: <= 128 MMA rows x 128 bytes
constexpr int kMaxProblems = 8;
constexpr uint64_t kDrainNs = 100000000ull;  // limit of each wait while draining after a timeout (0.1 s)

// Wide tiles (T = 64, 128, 256 tokens): a CTA owns one tile of 128 rows x T tokens, N = T per MMA
// (128 cycles at T = 256, so one accumulator keeps the tensor pipe busy) and no K-slices.
template <int T>
struct Cfg {
    static_assert(T >= 64, "the GEMM-form kernel runs wide tiles only (M <= 32 runs nf4_narrow.cuh)");
    static constexpr bool kWide = true;
    static constexpr int kAccN = 1;                   // accumulators
    // dequant warp sets (four warps each, one per 32-lane quarter of tensor memory); a set takes
    // every kSets-th stage, so more sets hide more of the dequantization's latency
    static constexpr int kSets = 4;
    static constexpr int kXWarp = 2 + 4 * kSets;      // the x producer, after the dequant warps
    static constexpr int kThreads = 32 * (kXWarp + 1);
    static constexpr int kTmemCols = 512;
    static constexpr int kJMax = T;                   // columns of B and of the accumulator
    static constexpr int kSMax = 1;                   // K-slices per tile
    static constexpr int kDCols = kAccN * kJMax;      // accumulator in tensor memory
    // A slots of 64 columns (two groups of K per MMA row); an even count, so that each dequant set
    // owns the same slots in every round
    static constexpr int kAStages = ((kTmemCols - kDCols) / 64 < 8 ? (kTmemCols - kDCols) / 64 : 8) & ~1;
    // release barriers of the A slots: stage q's MMAs complete on barrier q mod kARel (see the
    // dequant loop: a multiple of the sets, and two rounds of the slots)
    static constexpr int kARel = 2 * kAStages;
    static_assert(kARel % kSets == 0, "the A release barriers must be a multiple of the sets");
    // ring depths (an x box of T rows takes ~1000-1500 cycles to arrive from L2)
    static constexpr int kXStages = T == 64 ? 8 : (T == 128 ? 6 : 4);  // 64-k x sub-tiles
    static constexpr int kLoadStages = T == 64 ? 4 : 3;
    static constexpr int kScaleStages = T == 256 ? 2 : 3;
    static constexpr uint32_t kXBytes = kJMax * 128;  // one x sub-tile (multiple of 1024)
    static constexpr uint32_t kOffCodes = kXStages * kXBytes;
    static constexpr uint32_t kOffPtab = kOffCodes + kLoadStages * kLoadBytes;  // half-size pair table
    static constexpr uint32_t kOffScales = kOffPtab + kPairTab16Bytes;
    static constexpr uint32_t kOffBars = kOffScales + kScaleStages * kScaleSlot;
    static constexpr uint32_t kBytes = kOffBars + 1024;
    static_assert(kBytes + 1024 <= 227 * 1024, "shared memory budget");
    static_assert(8 * (2 * (kLoadStages + kXStages + kScaleStages) + kAStages + kARel + kSets + 2) + 4 <= 1024,
                  "barrier area");
};

// 64-k sub-stages per TMA box of codes for a tile of S slices: 128-byte rows for S = 1 and 2,
// 32 * S bytes for S >= 3.
__host__ __device__ constexpr int box_span(int s) { return s == 1 ? 4 : (s == 2 ? 2 : 1); }
// Sub-stages per codes load stage: four for S = 1, two otherwise (two boxes for S >= 3, each at its
// own 8 KB half of the slot).  A load stage thus never holds less than one whole pipeline stage,
// which keeps a dequant set's consecutive load stages at most kSets apart (see the dequant loop).
__host__ __device__ constexpr int load_span(int s) { return s == 1 ? 4 : 2; }
constexpr uint32_t kBoxStride = 8192;  // second box of a load stage (a box is <= 128 rows x 32 bytes)

struct Params {
    const uint8_t* codes[kMaxProblems];
    const uint16_t* scales[kMaxProblems];
    uint16_t* y[kMaxProblems];
    int n[kMaxProblems];            // rows of each problem
    int cta0[kMaxProblems + 1];     // first CTA of each problem; cta0[count] = grid size
    int count;
    int rstar;                      // rows per CTA (the last CTA of a problem may have fewer)
    int r_rem;                      // rows of a CTA's partial tile (rstar % 128; 0 = none)
    int s_rem;                      // its K-slices (r_rem * s_rem <= 128)
    int M, K, G;
};

// Codes of each problem, uint8 [N][K/2]: full tiles load boxes of 128 rows x 128 bytes (4 groups,
// 128-byte swizzle), partial tiles r_rem rows x 32 * load_span(s_rem) * s_rem bytes (128-byte swizzle
// when that is 128 bytes).  Rows past N and bytes past K/2 read as zero.
struct CodeMaps {
    CUtensorMap full[kMaxProblems];
    CUtensorMap rem[kMaxProblems];
};

struct Tile {
    int row0, rows, s, nt;  // first row (in the problem), rows, K-slices, 64-k sub-stages (even)
};

__device__ __forceinline__ Tile tile_of(const Params& P, int rbeg, int rows_cta, int j) {
    const int nfull = rows_cta / 128;
    Tile t;
    if (j < nfull) {
        t.row0 = rbeg + 128 * j;
        t.rows = 128;
        t.s = 1;
    } else {
        t.row0 = rbeg + 128 * nfull;
        t.rows = rows_cta - 128 * nfull;
        t.s = t.rows <= P.r_rem ? P.s_rem : 1;  // a partial tile that fits the partial box
    }
    t.nt = 2 * ((P.G + 2 * t.s - 1) / (2 * t.s));  // 64-k sub-stages, two per pipeline stage
    return t;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused for this layout)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset: next 8-row atom
    d |= static_cast<uint64_t>(1) << 46;                   // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;                   // swizzle mode: 128 bytes
    return d;
}

// 32 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}



// D[128 x N] (+)= A[128 x 16] * B[N x 16]^T with A read from tensor memory, issued by one elected
// lane of a converged warp (all 32 lanes execute the call with the same operands; see elect_one).
__device__ __forceinline__ void mma_tmem_a_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                 uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// Arrives on `bar` once every tcgen05.mma issued before by this warp's elected lane has completed.
__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}
// Arm `bar` for `bytes` of transaction and start one 2D / 3D TMA box into `dst`, from one elected
// lane of a converged warp.
__device__ __forceinline__ void expect_tx_elect(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_elect(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n\t}"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_elect(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                  uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n\t}"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// 32 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
        "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
        "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_n(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (8u << 24);
}

// Bounded wait by all 32 lanes (warp-uniform result).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, limit_ns));
}


template <int T>
__global__ void __launch_bounds__(Cfg<T>::kThreads, 1)
    stream_kernel(const __grid_constant__ CUtensorMap x_full, const __grid_constant__ CUtensorMap x_rem,
                  const __grid_constant__ CodeMaps cmaps, const __grid_constant__ Params P) {
    using C = Cfg<T>;
    static_assert(C::kWide, "stream_kernel runs the wide tiles only (T >= 64)");
    constexpr int NA = C::kAStages, NX = C::kXStages, NL = C::kLoadStages, NSS = C::kScaleStages, NR = C::kARel;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = P.G;

    // barriers
    const uint32_t b_lfull = sbase + C::kOffBars;       // [NL] codes load stage landed (tx)
    const uint32_t b_lempty = b_lfull + 8 * NL;         // [NL] codes load stage passed (every dequant warp)
    const uint32_t b_xfull = b_lempty + 8 * NL;         // [NX] x tile landed (tx)
    const uint32_t b_xempty = b_xfull + 8 * NX;         // [NX] x tile read by the MMAs (commit)
    const uint32_t b_afull = b_xempty + 8 * NX;         // [NA] A tile in tensor memory (4 warps)
    const uint32_t b_arel = b_afull + 8 * NA;           // [NR] stage q's A tile read by its MMAs (commit)
    const uint32_t b_sfull = b_arel + 8 * NR;           // [NSS] scale tile landed (32 producer lanes)
    const uint32_t b_sempty = b_sfull + 8 * NSS;        // [NSS] scale tile passed (every dequant warp)
    // accumulators complete (commit), one barrier per epilogue set: a set waits only for its own
    // tiles, one phase at a time (a parity wait more than one phase ahead would pass at once)
    const uint32_t b_dfull = b_sempty + 8 * NSS;        // [kSets]
    const uint32_t b_dfree = b_dfull + 8 * C::kSets;    // accumulators read (4 warps)
    const uint32_t b_mdone = b_dfree + 8;               // every MMA issued has completed
    uint32_t* tmem_slot =
        reinterpret_cast<uint32_t*>(smem + C::kOffBars + 8 * (2 * (NL + NX + NSS) + NA + NR + C::kSets + 2));

    // this CTA's problem and rows
    int p = 0;
    for (int i = 1; i < P.count; i++)
        if (static_cast<int>(blockIdx.x) >= P.cta0[i]) p = i;
    // a balanced run of the problem's 128-row tiles: one tile when the grid has a CTA per tile,
    // several consecutive ones otherwise (the CTA then streams a tile's weights and dequantizes its
    // first stages while the previous tile's last stages and epilogue run)
    const int nt_p = (P.n[p] + 127) / 128, nc_p = P.cta0[p + 1] - P.cta0[p];
    const int q_p = static_cast<int>(blockIdx.x) - P.cta0[p];
    const int t_beg = static_cast<int>(static_cast<int64_t>(q_p) * nt_p / nc_p);
    const int t_end = static_cast<int>(static_cast<int64_t>(q_p + 1) * nt_p / nc_p);
    const int rbeg = 128 * t_beg;
    const int rows_cta = P.n[p] - rbeg < 128 * (t_end - t_beg) ? P.n[p] - rbeg : 128 * (t_end - t_beg);
    const int ntiles = rows_cta / 128 + (rows_cta % 128 != 0);
    const int m0 = static_cast<int>(blockIdx.y) * T;  // first token of this CTA

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < NL; i++) {
            mbar_init(b_lfull + 8 * i, 1);
            mbar_init(b_lempty + 8 * i, 4 * C::kSets);  // every dequant warp, whether it reads the stage or not
        }
        for (int i = 0; i < NX; i++) {
            mbar_init(b_xfull + 8 * i, 1);
            mbar_init(b_xempty + 8 * i, 1);
        }
        for (int i = 0; i < NA; i++) mbar_init(b_afull + 8 * i, 4);
        for (int i = 0; i < NR; i++) mbar_init(b_arel + 8 * i, 1);
        for (int i = 0; i < NSS; i++) {
            mbar_init(b_sfull + 8 * i, 32);
            mbar_init(b_sempty + 8 * i, 4 * C::kSets);  // every dequant warp
        }
        for (int i = 0; i < C::kSets; i++) mbar_init(b_dfull + 8 * i, 1);
        mbar_init(b_dfree, 4 * C::kSets);  // every epilogue warp
        mbar_init(b_mdone, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t wait_ns = g_wait_ns;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        // Codes and scales only (x has its own warp): weights do not depend on the previous grid, so
        // this warp never waits for it and runs as far ahead as the codes ring allows.  Lane 0 issues
        // the TMA boxes; the warp copies scale windows.  Ring positions are counters.
        const uint8_t* sbytes = reinterpret_cast<const uint8_t*>(P.scales[p]);
        const int64_t s_total = static_cast<int64_t>(P.n[p]) * G * 2;
        const CUtensorMap* cm_full = &cmaps.full[p];
        const CUtensorMap* cm_rem = &cmaps.rem[p];
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(cm_full)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(cm_rem)) : "memory");
        }
        bool ok = true;
        int lq = 0, lslot = 0, lround = 0, sslot = 0, sround = 0;
        for (int j = 0; j < ntiles && ok; j++) {
            const Tile t = tile_of(P, rbeg, rows_cta, j);
            const int U = load_span(t.s);
            const CUtensorMap* cmap = t.s > 1 ? cm_rem : cm_full;
            const uint32_t cbytes = t.s > 1 ? 32u * U * t.s * P.r_rem : kLoadBytes;  // all boxes of a stage
            const int BS = box_span(t.s);
            const uint32_t per_row = (t.s + 2) * 16;
            for (int kb = 0, g = 0; kb < t.nt; kb++, g += t.s) {
                if ((kb & (U - 1)) == 0) {  // codes load stage: all rows x U*S groups
                    if (lround > 0 && !warp_wait(b_lempty + 8 * lslot, (lround - 1) & 1, wait_ns)) {
                        if (lane == 0) record_error(21);
                        ok = false;
                        break;
                    }
                    expect_tx_elect(b_lfull + 8 * lslot, cbytes);
                    for (int b = 0; b < U / BS; b++)
                        tma_load_2d_elect(sbase + C::kOffCodes + lslot * kLoadBytes + b * kBoxStride, cmap,
                                          (g + b * BS * t.s) * 32, t.row0, b_lfull + 8 * lslot);
                    lq++;
                    if (++lslot == NL) {
                        lslot = 0;
                        lround++;
                    }
                }
                if ((kb & 7) == 0) {  // scale tile: groups g .. g + 8S - 1 of every row
                    if (sround > 0 && !warp_wait(b_sempty + 8 * sslot, (sround - 1) & 1, wait_ns)) {
                        if (lane == 0) record_error(22);
                        ok = false;
                        break;
                    }
                    const int g1 = g + 8 * t.s < G ? g + 8 * t.s : G;
                    uint8_t* dst = smem + C::kOffScales + sslot * kScaleSlot;
                    for (int r = lane; r < t.rows; r += 32) {
                        const int64_t rb = static_cast<int64_t>(t.row0 + r) * G * 2;
                        const int64_t a = (rb + 2 * g) & ~static_cast<int64_t>(15);
                        for (int64_t c = a; c < rb + 2 * g1; c += 16) {
                            const int64_t left = s_total - c;
                            cp_async16(dst + r * per_row + (c - a), sbytes + c, static_cast<uint32_t>(left < 16 ? left : 16));
                        }
                    }
                    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(b_sfull + 8 * sslot)
                                 : "memory");
                    if (++sslot == NSS) {
                        sslot = 0;
                        sround++;
                    }
                }
                __syncwarp();
            }
        }
        cp_async_wait<0>();
        // drain: the codes of the last ring round have landed before the CTA may exit
        if (lane == 0) {
            const uint64_t dl = kDrainNs;
            for (int qq = lq - NL > 0 ? lq - NL : 0; qq < lq; qq++) mbar_wait(b_lfull + 8 * (qq % NL), (qq / NL) & 1, dl);
        }
    } else if (warp == C::kXWarp) {
        // ---------------------------------------------------------------- x producer
        // The whole warp runs the loop; one elected lane issues each TMA box (warp-uniform operands).
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&x_full)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&x_rem)) : "memory");
        }
        __syncwarp();
        pdl_wait();  // x may be written by the previous grid in the stream
        bool ok = true;
        int kq = 0, xslot = 0, xround = 0;
        for (int j = 0; j < ntiles && ok; j++) {
            const Tile t = tile_of(P, rbeg, rows_cta, j);
            const CUtensorMap* xmap = t.s > 1 ? &x_rem : &x_full;
            const uint32_t xbytes = 128u * t.s * T;
            for (int g = 0; g < t.nt * t.s; g += t.s) {  // a sub-stage: groups g .. g + S - 1
                if (xround > 0 && !warp_wait(b_xempty + 8 * xslot, (xround - 1) & 1, wait_ns)) {
                    if (lane == 0) record_error(23);
                    ok = false;
                    break;
                }
                expect_tx_elect(b_xfull + 8 * xslot, xbytes);
                tma_load_3d_elect(sbase + xslot * C::kXBytes, xmap, 0, g, m0, b_xfull + 8 * xslot);
                kq++;
                if (++xslot == NX) {
                    xslot = 0;
                    xround++;
                }
            }
        }
        // drain: the x tiles of the last ring round have landed before the CTA may exit
        for (int qq = kq - NX > 0 ? kq - NX : 0; qq < kq; qq++) mbar_wait(b_xfull + 8 * (qq % NX), (qq / NX) & 1, kDrainNs);
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // The whole warp runs the loop, so that every operand stays warp-uniform, and one elected
        // lane issues each tcgen05.mma and tcgen05.commit (a single diverged lane issuing them took
        // several times longer per instruction on this GPU).
        bool ok = true;
        int aq = 0, aslot = 0, xslot = 0;  // aq: CTA-wide stage
        uint32_t aph = 0, xph = 0;
        for (int j = 0; j < ntiles && ok; j++) {
            const Tile t = tile_of(P, rbeg, rows_cta, j);
            const int nmma = (T * t.s + 15) & ~15;
            const uint32_t idesc = idesc_n(nmma < 16 ? 16 : nmma);
            if (j > 0 && !warp_wait(b_dfree, (j - 1) & 1, wait_ns)) {
                if (lane == 0) record_error(24);
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kb = 0; kb < t.nt / 2 && ok; kb++) {
                if (!warp_wait(b_afull + 8 * aslot, aph, wait_ns)) {
                    if (lane == 0) record_error(25);
                    ok = false;
                    break;
                }
                const uint32_t a_tmem = tmem_base + C::kDCols + 64 * aslot;
                for (int h = 0; h < 2; h++) {  // two 64-k sub-stages, each with its own x sub-tile
                    if (!warp_wait(b_xfull + 8 * xslot, xph, wait_ns)) {
                        if (lane == 0) record_error(25);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = smem_desc_sw128(sbase + xslot * C::kXBytes);
#pragma unroll
                    for (int ks = 0; ks < 4; ks++) {  // K = 16 per MMA: 8 columns of A, 32 bytes of B
                        const int k8 = 4 * h + ks;
                        mma_tmem_a_elect(tmem_base + (k8 % C::kAccN) * C::kJMax, a_tmem + 8 * k8, bdesc + 2 * ks,
                                         idesc, kb > 0 || k8 >= C::kAccN);
                    }
                    mma_commit_elect(b_xempty + 8 * xslot);
                    if (++xslot == NX) {
                        xslot = 0;
                        xph ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit_elect(b_arel + 8 * (aq % NR));
                aq++;
                if (++aslot == NA) {
                    aslot = 0;
                    aph ^= 1;
                }
            }
            if (ok) mma_commit_elect(b_dfull + 8 * (j % C::kSets));
        }
        mma_commit_elect(b_mdone);  // the CTA exits only after every MMA it issued has completed
        mbar_wait(b_mdone, 0, kDrainNs);
    } else {
        // ---------------------------------------------------------------- dequant + epilogue (warps 2 .. kXWarp-1)
        const int set = (warp - 2) >> 2;
        const int quarter = warp & 3;             // tensor-memory lanes this warp may access
        const int i = quarter * 32 + lane;        // MMA row
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t ptab = sbase + C::kOffPtab;                         // shared-window addresses
        const uint32_t lcol16 = static_cast<uint32_t>(lane & 15) * 16;     // twice this lane's copy offset
        bool ok = true;
        // CTA-wide counts of the stages, codes load stages and scale tiles of the tiles before tile j:
        // ring slots and phases follow from them, so a set visits only its own stages.
        int q0 = 0, l0 = 0, s0 = 0, nst_prev = 0, nload_prev = 0, nscale_prev = 0;
        // A parity wait is sound only while the barrier is at most one phase from the awaited one:
        // the waiter must have seen the phase before it complete, and the phase after it must need
        // something the waiter has not yet done.
        //  - Codes load stages and scale tiles: every dequant warp waits for every fill in order,
        //    whether its set reads it or not, and then releases it (the empty barriers count all of
        //    them), so it always saw the slot's previous fill, and the next fill needs its own
        //    release.  A set reads at most one stage of a load stage (two stages) or a scale tile
        //    (four), its stages being kSets = 4 apart.  Every set runs every tile's epilogue, and
        //    passes the tile's remaining fills before it waits for the accumulators.
        //  - A slots: stage gq waits for the MMAs of stage gq - NA, on release barrier
        //    (gq - NA) mod NR (NR = 2 NA).  Its previous phase is stage gq - 3 NA, which this set waited
        //    for at its stage gq - 2 NA (NR is a multiple of kSets); its next is stage gq + NA, whose A
        //    tile waits for this stage's MMAs.
        int lnext = 0, snext = 0;  // the next load stage and scale tile this warp has not passed
        // The pair table is for the dequant warps alone: they write it while the producers already
        // stream the first stages, and meet on a named barrier before the first lookup.
        constexpr int kDqThreads = 32 * 4 * C::kSets;
        build_pair_table16(reinterpret_cast<float2*>(smem + C::kOffPtab), threadIdx.x - 64, kDqThreads);
        asm volatile("bar.sync 1, %0;" ::"r"(kDqThreads) : "memory");
        static_assert(!C::kWide || C::kSMax == 1, "wide tiles have one K-slice (four sub-stages per load stage)");
        for (int j = 0; j < ntiles && ok; j++) {
            q0 += nst_prev;
            l0 += nload_prev;
            s0 += nscale_prev;
            const Tile t = tile_of(P, rbeg, rows_cta, j);
            const int U = load_span(t.s), BS = box_span(t.s);
            const int nst = t.nt / 2, nload = (t.nt + U - 1) / U, nscale = (t.nt + 7) / 8;
            nst_prev = nst;
            nload_prev = nload;
            nscale_prev = nscale;
            const int r = i / t.s, sl = i - (i / t.s) * t.s;
            const bool lane_ok = r < t.rows;
            const bool warp_ok = __any_sync(0xFFFFFFFFu, lane_ok);
            // codes of row r in a box: rowb bytes, 16-byte chunks permuted by the 128-byte swizzle
            // (chunk ^ (r mod 8)) when the row is 128 bytes
            const uint32_t rowb = 32u * BS * t.s;
            const uint32_t swz = rowb == 128 ? static_cast<uint32_t>(r & 7) : 0u;
            // this lane's scale inside a scale tile: row r's window starts at the 16-byte boundary
            // below its first scale; sub-stage kb adds 2 * (kb mod 8) * S bytes
            const uint32_t soff = r * (t.s + 2) * 16 +
                                  static_cast<uint32_t>((static_cast<int64_t>(t.row0 + r) * G * 2) & 15) + 2 * sl;
            // this set's stages: CTA-wide index q0 + kb2 = set (mod kSets)
            for (int kb2 = (set - q0 % C::kSets + C::kSets) % C::kSets; kb2 < nst && ok; kb2 += C::kSets) {
                const int gq = q0 + kb2;
                const int aslot = gq % NA;
                const int kbs = 2 * kb2;                  // first of the stage's two 64-k sub-stages
                const int li = kbs / U;                   // its codes load stage, tile-relative
                const int si = kbs / 8;                   // its scale tile, tile-relative
                const int L = l0 + li, S = s0 + si;       // CTA-wide
                const int lslot = L % NL, sslot = S % NSS;
                bool good = true;
                for (; snext < S && good; snext++) {       // fills that only the other sets read
                    good = warp_wait(b_sfull + 8 * (snext % NSS), (snext / NSS) & 1, wait_ns);
                    if (good && lane == 0) mbar_arrive(b_sempty + 8 * (snext % NSS));
                }
                for (; lnext < L && good; lnext++) {
                    good = warp_wait(b_lfull + 8 * (lnext % NL), (lnext / NL) & 1, wait_ns);
                    if (good && lane == 0) mbar_arrive(b_lempty + 8 * (lnext % NL));
                }
                good = good && warp_wait(b_sfull + 8 * sslot, (S / NSS) & 1, wait_ns) &&
                       warp_wait(b_lfull + 8 * lslot, (L / NL) & 1, wait_ns);
                if (good && gq >= NA) good = warp_wait(b_arel + 8 * ((gq - NA) % NR), ((gq - NA) / NR) & 1, wait_ns);
                if (!good) {
                    record_error(26);
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int h = 0; h < 2; h++) {  // sub-stage kb: A columns 32h .. 32h + 31 of the stage's slot
                    if (!warp_ok) break;
                    const int kb = kbs + h;
                    const int u = kb & (U - 1);           // sub-stage in the load stage: box u / BS
                    uint32_t out[32];
                    const int g = kb * t.s + sl;
                    if (lane_ok && g < G) {
                        const uint8_t* crow = smem + C::kOffCodes + lslot * kLoadBytes + (u / BS) * kBoxStride + r * rowb;
                        const uint32_t ch = static_cast<uint32_t>(((u % BS) * t.s + sl) * 2);
                        const uint4 c0 = lds128(crow + 16 * (ch ^ swz)), c1 = lds128(crow + 16 * ((ch + 1) ^ swz));
                        const float sc = __half2float(__ushort_as_half(
                            lds_u16(sbase + C::kOffScales + sslot * kScaleSlot + soff + 2 * (kb & 7) * t.s)));
                        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                        for (int w = 0; w < 8; w++) {
#pragma unroll
                            for (int b = 0; b < 4; b++)
                                out[4 * w + b] = scale_pair(lds_f2(ptab + pair_offset16(words[w], lcol16, b)), sc);
                        }
                    } else {
#pragma unroll
                        for (int w = 0; w < 32; w++) out[w] = 0u;
                    }
                    tmem_st32(tmem_base + lane_addr + C::kDCols + 64 * aslot + 32 * h, out);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(b_afull + 8 * aslot);
                    mbar_arrive(b_lempty + 8 * lslot);
                    mbar_arrive(b_sempty + 8 * sslot);
                }
                lnext = L + 1;
                snext = S + 1;
            }
            // every set takes a quarter of the tile's columns in the epilogue (the sets are idle by then)
            if (!ok) continue;
            // The tile's remaining fills first: the tile's last stages may need a fill that waits for
            // this warp's release of an earlier one.
            for (; ok && snext < s0 + nscale; snext++) {
                ok = warp_wait(b_sfull + 8 * (snext % NSS), (snext / NSS) & 1, wait_ns);
                if (ok && lane == 0) mbar_arrive(b_sempty + 8 * (snext % NSS));
            }
            for (; ok && lnext < l0 + nload; lnext++) {
                ok = warp_wait(b_lfull + 8 * (lnext % NL), (lnext / NL) & 1, wait_ns);
                if (ok && lane == 0) mbar_arrive(b_lempty + 8 * (lnext % NL));
            }
            // ------------------------------------------------------------ epilogue of tile j
            if (!ok || !warp_wait(b_dfull + 8 * (j % C::kSets), (j / C::kSets) & 1, wait_ns)) {
                record_error(26);
                ok = false;
                break;
            }
            tc_fence_after();
            pdl_wait();  // y may still be read by the previous grid (returns at once by now)
            const int M = P.M - m0 < T ? P.M - m0 : T, np = P.n[p];  // tokens of this tile
            uint16_t* y = P.y[p];
            if constexpr (C::kWide) {
                // Each set writes a quarter of the tile's token columns (tokens c0 .. c0 + TC - 1)
                // straight from tensor memory: lane i holds row i, so a warp's store of one token
                // covers 64 contiguous bytes of y (the x ring may already hold the next tile's x).
                constexpr int TC = T / C::kSets;
                static_assert(TC % 16 == 0, "a set's columns are whole 16-column loads");
                const int c0 = set * TC;
                const bool row_ok = i < t.rows;
                for (int c = c0; c < c0 + TC; c += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem_base + lane_addr + c, v);
#pragma unroll
                    for (int cc = 0; cc < 16; cc++) {
                        const int tt = c + cc;
                        if (row_ok && tt < M)
                            y[static_cast<int64_t>(m0 + tt) * np + t.row0 + i] = bf16_bits(__uint_as_float(v[cc]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(b_dfree);
                continue;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(C::kTmemCols)
                     : "memory");
    }
}

}  // namespace st
}  // namespace nf4
