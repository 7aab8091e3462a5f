// Small-M NF4 weight streaming (decode and prefill up to 32 positions) on the tcgen05 tensor cores,
// sm_103a: y[M, N] = x[M, K] * w_hat[N, K]^T for 1 <= M <= 32.
//
// The deep-fold README's execution-path table runs the N = 1 decode GEMV and the prefill GEMM of up
// to 32 positions over packed weights, dequantizing only the current tile.  These shapes are bound
// by the weight stream and by the exact dequantization, so every multiply-add goes to the tensor
// cores and the CUDA cores run the dequantization alone:
//
//   dequant warps:  packed codes (shared memory) -> exact bf16 w_hat -> tensor memory (tcgen05.st)
//                   w_hat = bf16(fp32(T[c] * scale)) two weights at a time: the code byte indexes the
//                   lane-replicated fp32 pair table {T[c0], T[c1]} in shared memory, one packed fp32x2
//                   multiply by the scale, one bf16x2 conversion (see scale_pair)
//   MMA warp:       tcgen05.mma, A = that w_hat tile in tensor memory, B = x tile in shared memory
//                   (TMA, 128-byte swizzle), D = fp32 accumulators in tensor memory
//
// K-slices.  A CTA owns a contiguous range of output rows, processed as tiles
// of R rows; the 128 MMA rows of a tile are R rows x S K-slices: each 32-lane quarter of tensor memory
// holds floor(32 / S) rows, lane r' * S + s of a quarter holding slice s of its row r', that is row
// r's groups s, S + s, 2S + s, ...  The B tile holds, for token t and slice s, the x values of group
// kb*S + s as pseudo-token column t * S + s, and the epilogue adds the S partials of each (row, token)
// in a fixed order within the warp.  S need not be a power of two: a CTA with 34 rows runs three
// slices (102 MMA rows) where a power of two would allow two (68).  A CTA with a dozen rows still
// fills the MMA rows, so the grid is one CTA per SM with a balanced row range each.
//
// Pipeline stage = 128 k per MMA row (two 64-k sub-stages, 8 MMAs of K = 16).  Stage q uses A slot
// q mod 4 in tensor memory and x slot q mod 4 in shared memory (both sub-tiles of the stage), so one
// tcgen05.commit per stage frees both (on release barrier q mod 12, see the dequant loop).  Two MMA
// warps take alternate stages, each into its own pair of accumulators, so that issuing costs the
// same on two warp schedulers; an issuer waits twice per stage (x landed, A written) and commits
// once, converged, one elected lane issuing (elect_one).  The epilogue adds the four accumulators in
// a fixed order.
//
// Warp roles, one helper per warp scheduler (warp w runs on scheduler w mod 4): warp 0 streams codes
// (TMA), warps 1 and 3 issue the MMAs of even and odd stages (warp 1 also owns tensor memory), warp 2
// streams x; warps 4 .. 4*kSets+3 are kSets sets of four dequant warps (a set takes every kSets-th
// stage; the four warps of a set cover the four 32-lane quarters of tensor memory, one per
// scheduler) that also run the epilogue of every kSets-th tile.  A set's stage is done when its
// slowest warp is, so every scheduler carries the same load.  Each dequant thread reads its own
// group scales from global memory three of its stages ahead (no staging, no barrier).  Weights do not
// depend on the previous kernel in the stream, so warp 0 and the scale loads never wait for it;
// only x and y do.
// Every mbarrier wait is bounded (wall clock, per wait); a wait that runs out records an error code,
// the roles drain the copies and MMAs in flight (bounded again) and tensor memory is always freed.
#pragma once

namespace nf4 {
namespace st {

// Ring depths are powers of two (slot and phase arithmetic are masks and shifts).  K-slices are at most
// kSMax, and a row's slices sit in consecutive lanes of one warp, so the epilogue adds them with
// shuffles.
template <int T>
struct NCfg {
    static constexpr int kJMax = T <= 2 ? 16 : (T == 4 ? 32 : 64);  // columns of B and of each D
    static constexpr int kSMax = kJMax / T < 8 ? kJMax / T : 8;        // K-slices per tile
    static constexpr int kAccN = 4;                                    // two per MMA warp
    static constexpr int kDCols = kAccN * kJMax;
    static constexpr int kAStages = 4;                                 // A slots (tensor memory) = x slots
    static constexpr int kLoadStages = 4;                              // codes load stages
    static constexpr int kSets = 3;
    // release barriers of the A and x slots: stage q's MMAs complete on barrier q mod kRel, a common
    // multiple of the slots and the sets (see the dequant loop)
    static constexpr int kRel = kAStages * kSets;
    static constexpr int kThreads = 32 * (4 + 4 * kSets);             // 4 helper warps, one per scheduler
    static constexpr int kU = 4;                                       // 64-k sub-stages per codes load stage
    static constexpr uint32_t kXSub = kJMax * 128;  // one 64-k x sub-tile (multiple of 1024 bytes)
    static constexpr uint32_t kXSlot = 2 * kXSub;
    static constexpr uint32_t kOffCodes = kAStages * kXSlot;
    static constexpr uint32_t kOffPtab = kOffCodes + kLoadStages * kLoadBytes;  // pair table
    static constexpr uint32_t kOffBars = kOffPtab + kPairTabBytes;
    static constexpr uint32_t kBytes = kOffBars + 1024;
    static_assert(kBytes + 1024 <= 227 * 1024, "shared memory budget");
    static_assert(kDCols + 64 * kAStages <= 512, "tensor memory budget");
    static_assert(kAStages == 4 && kLoadStages == 4, "slot arithmetic assumes rings of four");
    static_assert(kSMax >= 1 && kSMax <= 8, "K-slices");
    static_assert(8 * (2 * kLoadStages + 2 * kAStages + kRel + kSets + 3) + 4 <= 1024, "barrier area");
};

// 32 consecutive 32-bit columns of this thread's tensor-memory lane, without waiting for the store.
__device__ __forceinline__ void tmem_st32_nowait(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
        "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
        "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// Group scale `g` of a row (bits), or 0 when g is past the row or the lane has no row.
__device__ __forceinline__ uint32_t load_scale(const uint16_t* row_scales, int g, int G, bool lane_ok) {
    return (lane_ok && g < G) ? static_cast<uint32_t>(ld_nc_u16(row_scales + g)) : 0u;
}

template <int T>
__global__ void __launch_bounds__(NCfg<T>::kThreads, 1)
    narrow_kernel(const __grid_constant__ CUtensorMap x_full, const __grid_constant__ CUtensorMap x_rem,
                  const __grid_constant__ CodeMaps cmaps, const __grid_constant__ Params P) {
    using C = NCfg<T>;
    constexpr int NA = C::kAStages, NL = C::kLoadStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = P.G;

    // barriers
    const uint32_t b_lfull = sbase + C::kOffBars;   // [NL] codes load stage landed (tx)
    const uint32_t b_lempty = b_lfull + 8 * NL;     // [NL] codes load stage passed (every dequant warp)
    const uint32_t b_xfull = b_lempty + 8 * NL;     // [NA] x slot landed (tx)
    const uint32_t b_afull = b_xfull + 8 * NA;      // [NA] A slot written (4 warps)
    const uint32_t b_rel = b_afull + 8 * NA;        // [kRel] stage q's A and x slots read by its MMAs (commit)
    const uint32_t b_dfull = b_rel + 8 * C::kRel;   // [kSets] accumulators complete (both MMA warps), per epilogue set
    const uint32_t b_dfree = b_dfull + 8 * C::kSets;  // accumulators read (4 warps)
    const uint32_t b_mdone = b_dfree + 8;           // [2] every MMA an MMA warp issued has completed
    uint32_t* tmem_slot =
        reinterpret_cast<uint32_t*>(smem + C::kOffBars + 8 * (2 * NL + 2 * NA + C::kRel + C::kSets + 3));

    // this CTA's problem and rows
    int p = 0;
    for (int i = 1; i < P.count; i++)
        if (static_cast<int>(blockIdx.x) >= P.cta0[i]) p = i;
    const int rbeg = (static_cast<int>(blockIdx.x) - P.cta0[p]) * P.rstar;
    const int rows_cta = P.n[p] - rbeg < P.rstar ? P.n[p] - rbeg : P.rstar;
    const int ntiles = rows_cta / 128 + (rows_cta % 128 != 0);
    const int m0 = static_cast<int>(blockIdx.y) * T;  // first token of this CTA

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < NL; i++) {
            mbar_init(b_lfull + 8 * i, 1);
            mbar_init(b_lempty + 8 * i, 4 * C::kSets);  // every dequant warp, whether it reads the stage or not
        }
        for (int i = 0; i < NA; i++) {
            mbar_init(b_xfull + 8 * i, 1);
            mbar_init(b_afull + 8 * i, 4);
        }
        for (int i = 0; i < C::kRel; i++) mbar_init(b_rel + 8 * i, 1);
        for (int i = 0; i < C::kSets; i++) mbar_init(b_dfull + 8 * i, 2);
        mbar_init(b_dfree, 4);
        mbar_init(b_mdone, 1);
        mbar_init(b_mdone + 8, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t wait_ns = g_wait_ns;

    if (warp == 0) {
        // ---------------------------------------------------------------- codes
        // One elected lane of the converged warp issues the TMA boxes.  A load stage is four 64-k
        // sub-stages of every row of the tile: one box of 128-byte rows (S = 1), two (S = 2) or four
        // (S >= 4, one per sub-stage), each box at its own quarter, half or whole of the slot.
        const CUtensorMap* cm_full = &cmaps.full[p];
        const CUtensorMap* cm_rem = &cmaps.rem[p];
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(cm_full)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(cm_rem)) : "memory");
        }
        __syncwarp();
        bool ok = true;
        int lq = 0;
        for (int j = 0; j < ntiles && ok; j++) {
            const Tile t = tile_of(P, rbeg, rows_cta, j);
            const CUtensorMap* cmap = t.s > 1 ? cm_rem : cm_full;
            const int BS = box_span(t.s);
            const int nbox = C::kU / BS;
            const uint32_t bstride = kLoadBytes / nbox;
            const uint32_t cbytes = t.s > 1 ? 32u * C::kU * t.s * P.r_rem : kLoadBytes;  // all boxes of a stage
            for (int kb = 0; kb < t.nt; kb += C::kU, lq++) {  // codes load stage: all rows x 4S groups
                const int lslot = lq & (NL - 1), lround = lq >> 2;
                if (lround > 0 && !warp_wait(b_lempty + 8 * lslot, (lround - 1) & 1, wait_ns)) {
                    if (lane == 0) record_error(21);
                    ok = false;
                    break;
                }
                expect_tx_elect(b_lfull + 8 * lslot, cbytes);
                for (int b = 0; b < nbox; b++)
                    tma_load_2d_elect(sbase + C::kOffCodes + lslot * kLoadBytes + b * bstride, cmap,
                                      (kb + b * BS) * t.s * 32, t.row0, b_lfull + 8 * lslot);
            }
        }
        // drain: the codes of the last ring round have landed before the CTA may exit
        for (int qq = lq - NL > 0 ? lq - NL : 0; qq < lq; qq++) mbar_wait(b_lfull + 8 * (qq & (NL - 1)), (qq >> 2) & 1, kDrainNs);
    } else if (warp == 2) {
        // ---------------------------------------------------------------- x
        // Stage q's two 64-k sub-tiles land in x slot q mod 4, counted on that slot's own barrier; the
        // slot is free once stage q - 4's MMAs have completed (release barrier (q - 4) mod kRel, whose
        // previous phase this warp saw at stage q - kRel, and whose next needs x of stage q + kRel - 4).
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&x_full)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&x_rem)) : "memory");
        }
        __syncwarp();
        pdl_wait();  // x may be written by the previous grid in the stream
        bool ok = true;
        int q = 0;
        for (int j = 0; j < ntiles && ok; j++) {
            const Tile t = tile_of(P, rbeg, rows_cta, j);
            const CUtensorMap* xmap = t.s > 1 ? &x_rem : &x_full;
            const uint32_t subbytes = 128u * t.s * T;
            for (int kb2 = 0; kb2 < t.nt / 2; kb2++, q++) {
                const int slot = q & (NA - 1);
                if (q >= NA && !warp_wait(b_rel + 8 * ((q - NA) % C::kRel), ((q - NA) / C::kRel) & 1, wait_ns)) {
                    if (lane == 0) record_error(23);
                    ok = false;
                    break;
                }
                const uint32_t dst = sbase + slot * C::kXSlot;
                expect_tx_elect(b_xfull + 8 * slot, 2 * subbytes);
                tma_load_3d_elect(dst, xmap, 0, 2 * kb2 * t.s, m0, b_xfull + 8 * slot);
                tma_load_3d_elect(dst + C::kXSub, xmap, 0, (2 * kb2 + 1) * t.s, m0, b_xfull + 8 * slot);
            }
        }
        // drain: the x slots of the last ring round have landed before the CTA may exit
        for (int qq = q - NA > 0 ? q - NA : 0; qq < q; qq++) mbar_wait(b_xfull + 8 * (qq & (NA - 1)), (qq >> 2) & 1, kDrainNs);
    } else if (warp == 1 || warp == 3) {
        // ---------------------------------------------------------------- MMA issuers
        // Warp 1 issues the stages with even CTA-wide index into accumulators 0 and 1, warp 3 the odd
        // ones into accumulators 2 and 3 (K-steps alternate between the pair).  The whole warp runs
        // the loop (every operand warp-uniform); one elected lane issues.  Both commit every tile's
        // end to the epilogue set's barrier, whether or not they had a stage in the tile.
        const int e = warp == 1 ? 0 : 1;
        const uint32_t acc0 = tmem_base + 2 * e * C::kJMax;
        bool ok = true;
        int q0 = 0;
        for (int j = 0; j < ntiles && ok; j++) {
            const Tile t = tile_of(P, rbeg, rows_cta, j);
            const int nst = t.nt / 2;
            const int nmma = (T * t.s + 15) & ~15;
            const uint32_t idesc = idesc_n(nmma < 16 ? 16 : nmma);
            if (j > 0 && !warp_wait(b_dfree, (j - 1) & 1, wait_ns)) {
                if (lane == 0) record_error(24);
                ok = false;
                break;
            }
            tc_fence_after();
            bool first = true;
            for (int kb2 = (q0 & 1) == e ? 0 : 1; kb2 < nst; kb2 += 2) {
                const int q = q0 + kb2;
                const int slot = q & (NA - 1);
                const uint32_t par = (q >> 2) & 1;
                if (!warp_wait(b_xfull + 8 * slot, par, wait_ns) || !warp_wait(b_afull + 8 * slot, par, wait_ns)) {
                    if (lane == 0) record_error(25);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_tmem = tmem_base + C::kDCols + 64 * slot;
                const uint64_t bdesc = smem_desc_sw128(sbase + slot * C::kXSlot);
#pragma unroll
                for (int k8 = 0; k8 < 8; k8++) {  // K = 16 per MMA: 8 columns of A, 32 bytes of a B row
                    const uint64_t b = bdesc + (k8 >= 4 ? (C::kXSub >> 4) : 0) + 2 * (k8 & 3);
                    mma_tmem_a_elect(acc0 + (k8 & 1) * C::kJMax, a_tmem + 8 * k8, b, idesc, !first || k8 >= 2);
                }
                mma_commit_elect(b_rel + 8 * (q % C::kRel));
                first = false;
            }
            if (!ok) break;
            mma_commit_elect(b_dfull + 8 * (j % C::kSets));
            q0 += nst;
        }
        mma_commit_elect(b_mdone + 8 * e);  // the CTA exits only after every MMA it issued has completed
        mbar_wait(b_mdone + 8 * e, 0, kDrainNs);
    } else {
        // ---------------------------------------------------------------- dequant + epilogue
        const int set = (warp - 4) >> 2;
        const int quarter = warp & 3;             // tensor-memory lanes this warp may access
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t ptab = sbase + C::kOffPtab;  // shared-window address of the pair table
        const uint32_t lcol = static_cast<uint32_t>(lane) * 8;  // this lane's column of the pair table
        bool ok = true;
        // CTA-wide counts of the stages and codes load stages of the tiles before tile j: ring slots
        // and phases follow from them, so a set visits only its own stages.
        int q0 = 0, l0 = 0;
        // A parity wait is sound only while the barrier is at most one phase from the awaited one:
        // the waiter must have seen the phase before it complete, and the phase after it must need
        // something the waiter has not yet done.
        //  - Codes load stages: every dequant warp waits for every load stage, whether its set reads
        //    it or not, and then releases it (b_lempty counts all of them), so the next fill of a
        //    slot needs its own release, and it saw the slot's previous fill: a set's consecutive
        //    stages are at most three load stages apart (the two stages between them take at most
        //    two), so when a warp waits for its own load stage L it has passed every one before the
        //    previous stage's, L - 4 among them; the load stages between are passed after L (by then
        //    they have almost always landed, so the warp does not sleep twice).  A set reads at most
        //    one stage of a load stage (its stages are kSets >= 2 apart).
        //  - A slots: stage gq waits for the MMAs of stage gq - NA, on release barrier
        //    (gq - NA) mod kRel.  That barrier's previous phase is stage gq - NA - kRel, which this set
        //    waited for at its stage gq - kRel (kRel is a multiple of kSets); its next is stage
        //    gq - NA + kRel, whose A tile waits, through the slot chain, for this stage's MMAs.  The
        //    MMA warps alternate stages, so a completed stage says nothing about the other warp's
        //    earlier ones; the wait rule above does not rely on it.
        static_assert(C::kRel % C::kSets == 0 && C::kRel % NA == 0 && C::kRel >= 2 * NA && C::kSets >= 2,
                      "release barriers must be a common multiple of the A slots and the sets");
        int lnext = 0;  // the next codes load stage this warp has not waited for and released
        // The pair table is for the dequant warps alone: they write it while the producers already
        // stream the first stages, and meet on a named barrier before the first lookup.
        constexpr int kDqThreads = 32 * 4 * C::kSets;
        build_pair_table(reinterpret_cast<float2*>(smem + C::kOffPtab), threadIdx.x - 128, kDqThreads);
        asm volatile("bar.sync 1, %0;" ::"r"(kDqThreads) : "memory");
        for (int j = 0; j < ntiles && ok; j++) {
            const Tile t = tile_of(P, rbeg, rows_cta, j);
            constexpr int lu = 2;                                 // log2 of the sub-stages per load stage
            const int BS = box_span(t.s);
            const int lbs = BS == 4 ? 2 : (BS == 2 ? 1 : 0);      // log2 BS
            const uint32_t bstride = kLoadBytes >> (lu - lbs);    // a load stage holds 4 / BS boxes
            const int S = t.s;
            const int nst = t.nt / 2, nload = (t.nt + C::kU - 1) / C::kU;
            // row r and slice sl of this lane: floor(32 / S) rows a quarter, S consecutive lanes each
            const int rq = 32 / S, rl = lane / S, sl = lane - rl * S;
            const int r = quarter * rq + rl;
            const bool lane_ok = rl < rq && r < t.rows;
            const bool warp_ok = __any_sync(0xFFFFFFFFu, lane_ok);
            // codes of row r in a box: rowb bytes, 16-byte chunks permuted by the 128-byte swizzle
            // (chunk ^ (r mod 8)) when the row is 128 bytes.  A lane past the tile's rows reads row 0
            // (its A row feeds only its own, unused, row of D).
            const int rr = lane_ok ? r : 0;
            const uint32_t rowb = 32u * BS * t.s;
            const uint32_t swz = rowb == 128 ? static_cast<uint32_t>(rr & 7) : 0u;
            const uint8_t* crow0 = smem + C::kOffCodes + rr * rowb;
            const uint16_t* row_scales = P.scales[p] + static_cast<int64_t>(t.row0 + (lane_ok ? r : 0)) * G;
            // this set's stages: CTA-wide index q0 + kb2 = set (mod kSets); scales three stages ahead
            const int kfirst = (set - q0 % C::kSets + C::kSets) % C::kSets;
            uint32_t sc_n[2], sc_n1[2], sc_n2[2], sc_n3[2];
#pragma unroll
            for (int h = 0; h < 2; h++) {
                sc_n[h] = load_scale(row_scales, (2 * kfirst + h) * S + sl, G, lane_ok);
                sc_n1[h] = load_scale(row_scales, (2 * (kfirst + C::kSets) + h) * S + sl, G, lane_ok);
                sc_n2[h] = load_scale(row_scales, (2 * (kfirst + 2 * C::kSets) + h) * S + sl, G, lane_ok);
            }
            for (int kb2 = kfirst; kb2 < nst && ok; kb2 += C::kSets) {
#pragma unroll
                for (int h = 0; h < 2; h++)
                    sc_n3[h] = load_scale(row_scales, (2 * (kb2 + 3 * C::kSets) + h) * S + sl, G, lane_ok);
                const int gq = q0 + kb2;
                const int aslot = gq & (NA - 1);
                const int kbs = 2 * kb2;                  // first of the stage's two 64-k sub-stages
                const int li = kbs >> lu;                 // its codes load stage, tile-relative
                const int L = l0 + li;                    // CTA-wide
                const int lslot = L & (NL - 1);
                bool good = warp_wait(b_lfull + 8 * lslot, (L >> 2) & 1, wait_ns);
                for (; lnext < L && good; lnext++) {       // load stages of the other sets' stages
                    good = warp_wait(b_lfull + 8 * (lnext & (NL - 1)), (lnext >> 2) & 1, wait_ns);
                    if (good && lane == 0) mbar_arrive(b_lempty + 8 * (lnext & (NL - 1)));
                }
                if (good && gq >= NA) good = warp_wait(b_rel + 8 * ((gq - NA) % C::kRel), ((gq - NA) / C::kRel) & 1, wait_ns);
                if (!good) {
                    if (lane == 0) record_error(26);
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (warp_ok) {
                    const uint8_t* crow = crow0 + lslot * kLoadBytes;
#pragma unroll
                    for (int h = 0; h < 2; h++) {  // sub-stage kb: A columns 32h .. 32h + 31 of the stage's slot
                        const int kb = kbs + h;
                        const int u = kb & (C::kU - 1);  // sub-stage in the load stage: box u / BS
                        // Every lane runs the same code: a group past K has scale 0 (its codes and its x
                        // are zero-filled), so its weights are +-0 and add nothing to the row's sums.
                        uint32_t out[32];
                        const uint8_t* cb = crow + (u >> lbs) * bstride;
                        const uint32_t ch = static_cast<uint32_t>(((u & (BS - 1)) * S + sl) * 2);
                        const uint4 c0 = lds128(cb + 16 * (ch ^ swz)), c1 = lds128(cb + 16 * ((ch + 1) ^ swz));
                        const float sc = __half2float(__ushort_as_half(static_cast<uint16_t>(h == 0 ? sc_n[0] : sc_n[1])));
                        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                        for (int w = 0; w < 8; w++) {
#pragma unroll
                            for (int b = 0; b < 4; b++)
                                out[4 * w + b] = scale_pair(lds_f2(ptab + pair_offset(words[w], lcol, b)), sc);
                        }
                        tmem_st32_nowait(tmem_base + lane_addr + C::kDCols + 64 * aslot + 32 * h, out);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(b_afull + 8 * aslot);
                    mbar_arrive(b_lempty + 8 * lslot);
                }
                lnext = L + 1;
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    sc_n[h] = sc_n1[h];
                    sc_n1[h] = sc_n2[h];
                    sc_n2[h] = sc_n3[h];
                }
            }
            // which MMA warps had a stage in this tile (the other's accumulators were not written)
            const bool has0 = nst >= 2 || (q0 & 1) == 0, has1 = nst >= 2 || (q0 & 1) == 1;
            q0 += nst;
            l0 += nload;
            if (!ok || j % C::kSets != set) continue;
            // ------------------------------------------------------------ epilogue of tile j
            if (!warp_wait(b_dfull + 8 * set, (j / C::kSets) & 1, wait_ns)) {
                if (lane == 0) record_error(26);
                ok = false;
                break;
            }
            tc_fence_after();
            pdl_wait();  // y may still be read by the previous grid (returns at once by now)
            const int M = P.M - m0 < T ? P.M - m0 : T, np = P.n[p];  // tokens of this tile
            uint16_t* y = P.y[p];
            const int J = T * S;
            int cm = 0, tt = 0;  // slice and token of column c + cc (K-sliced tiles)
            float val = 0.0f;    // this lane's slice of the current token
            for (int c = 0; c < J; c += 16) {
                // accumulators 0 + 1 (even stages), then 2 + 3 (odd stages), then their sum
                float v[16];
#pragma unroll
                for (int cc = 0; cc < 16; cc++) v[cc] = 0.0f;
#pragma unroll
                for (int pr = 0; pr < 2; pr++) {
                    if (!(pr == 0 ? has0 : has1)) continue;  // warp-uniform
                    uint32_t a[16], b[16];
                    tmem_ld16(tmem_base + lane_addr + (2 * pr) * C::kJMax + c, a);
                    tmem_ld16(tmem_base + lane_addr + (2 * pr + 1) * C::kJMax + c, b);
#pragma unroll
                    for (int cc = 0; cc < 16; cc++) v[cc] += __uint_as_float(a[cc]) + __uint_as_float(b[cc]);
                }
                if (t.s == 1) {
#pragma unroll
                    for (int cc = 0; cc < 16; cc++) {
                        const int col = c + cc;
                        if (lane_ok && col < M)
                            y[static_cast<int64_t>(m0 + col) * np + t.row0 + r] = bf16_bits(v[cc]);
                    }
                } else {
                    // column c + cc = token tt * S + slice cm: this lane keeps its own slice's value of
                    // each token, and after a token's last column the S lanes of the row add theirs
                    // with shuffles (a fixed order: the result does not depend on timing).  A token's
                    // columns may straddle two 16-column loads when S does not divide 16.
#pragma unroll
                    for (int cc = 0; cc < 16; cc++) {
                        if (cm == sl) val = v[cc];
                        if (cm == S - 1) {  // warp-uniform
                            float sum;
                            if ((S & (S - 1)) == 0) {
                                sum = val;
                                for (int off = 1; off < S; off <<= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
                            } else {  // slices 0, 1, ..., S - 1 in order (lanes past the rows read anything)
                                sum = 0.0f;
                                for (int jj = 0; jj < S; jj++) sum += __shfl_sync(0xFFFFFFFFu, val, lane - sl + jj);
                            }
                            if (sl == 0 && lane_ok && tt < M)
                                y[static_cast<int64_t>(m0 + tt) * np + t.row0 + r] = bf16_bits(sum);
                            cm = 0;
                            tt++;
                        } else {
                            cm++;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_dfree);
        }
        // the load stages after this set's last stage, which the other sets read
        for (; ok && lnext < l0; lnext++) {
            ok = warp_wait(b_lfull + 8 * (lnext & (NL - 1)), (lnext >> 2) & 1, wait_ns);
            if (!ok && lane == 0) record_error(26);
            if (ok && lane == 0) mbar_arrive(b_lempty + 8 * (lnext & (NL - 1)));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
    }
}

}  // namespace st
}  // namespace nf4
