// NF4 prefill GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// y[M, N] = x[M, K] * w_hat[N, K]^T for M >= 5 (deep-fold README, execution-path table: prefill runs
// as a GEMM on the tensor cores, dequantizing into bf16 tiles on chip; the pages stop at 32 tokens
// on Ampere mma.sync, this path serves any M).  Included into the translation unit of the GEMV so
// that both read the same per-device V table (g_vtab).
//
// Operands are swapped so that the dequantized weights fill the 128-row MMA dimension:
//   A = w_hat tile [128 rows of N][64 of K]  bf16, K-major, 128-byte swizzle (written by dequant warps)
//   B = x tile     [T tokens][64 of K]       bf16, K-major, 128-byte swizzle (TMA)
//   D = [128][T] fp32 in tensor memory (T columns), D += A * B^T over K/64 stages.
// One stage is one scale group (64 of K = one 128-byte swizzle row): its packed codes (4 KB, TMA),
// its A tile (16 KB) and its B tile (T * 128 bytes).
//
// Warp roles (320 threads): warp 0 issues the TMA loads, warp 1 owns the TMEM allocation and one
// lane issues the MMAs, warps 2-9 dequantize (256 threads, half a row each) and then run the
// epilogue (tcgen05.ld -> bf16 -> y).  Every mbarrier wait is bounded: past about a second the
// thread records an error code in g_tc_error and stops waiting; the CTA still drains its in-flight
// copies and MMAs (bounded again) and frees its tensor memory before it exits.
#pragma once

#include <cuda.h>

namespace nf4 {

namespace tc {

constexpr int kTileN = 128;   // weight rows per CTA (MMA M)
constexpr int kStages = 3;    // pipeline depth
constexpr int kDequantWarps = 8;
constexpr int kThreads = 32 * (2 + kDequantWarps);
constexpr uint32_t kABytes = kTileN * 64 * 2;    // 16 KB
constexpr uint32_t kCodeBytes = kTileN * 64 / 2;  // 4 KB
constexpr long long kDrainCycles = 200000000LL;    // ~0.1 s

template <int T>
struct Layout {
    static constexpr uint32_t kBBytes = T * 128;
    static constexpr uint32_t kStage = kABytes + kBBytes + kCodeBytes;  // multiple of 1024
    static constexpr uint32_t kVtab = kStages * kStage;
    static constexpr uint32_t kBars = kVtab + 65536;  // both halves of the V table
    static constexpr uint32_t kBytes = kBars + 256;
    static constexpr uint32_t kCols = T <= 32 ? 32 : (T <= 64 ? 64 : (T <= 128 ? 128 : 256));
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
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

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, both K-major, M = 128, N = T.
template <int T>
__device__ __forceinline__ constexpr uint32_t instr_desc() {
    return (1u << 4)                               // D format: f32
           | (1u << 7)                             // A format: bf16
           | (1u << 10)                            // B format: bf16
           | (static_cast<uint32_t>(T >> 3) << 17)  // N >> 3
           | (static_cast<uint32_t>(kTileN >> 4) << 24);  // M >> 4
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int T>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_codes,
                const uint16_t* __restrict__ scales, uint16_t* __restrict__ y, int M, int N, int K, uint32_t m1,
                uint32_t p16) {
    using L = Layout<T>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kTileN;
    const int m0 = blockIdx.y * T;
    const int KB = K / 64;
    const int G = KB;

    // barriers: loaded[s] (TMA bytes), full[s] (dequant warps), empty[s] (MMA commit), accum
    const uint32_t bar_loaded = sbase + L::kBars;
    const uint32_t bar_full = bar_loaded + 8 * kStages;
    const uint32_t bar_empty = bar_full + 8 * kStages;
    const uint32_t bar_accum = bar_empty + 8 * kStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBars + 8 * (3 * kStages + 1));
    const uint4* vtab = reinterpret_cast<const uint4*>(smem + L::kVtab);

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(bar_loaded + 8 * s, 1);
            mbar_init(bar_full + 8 * s, kDequantWarps);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_accum, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_codes)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(L::kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    for (int i = threadIdx.x; i < 4096; i += kThreads)  // all copies in flight at once
        cp_async16(smem + L::kVtab + 16 * i, &g_vtab[i]);
    cp_async_commit();
    cp_async_wait<0>();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();  // inputs may come from the previous kernel in the stream

    const long long deadline = clock64() + kWaitCycles;
    bool ok = true;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        int issued = 0;
        if (lane == 0) {
            for (int kb = 0; kb < KB && ok; kb++) {
                const int s = kb % kStages;
                const int round = kb / kStages;
                if (round > 0 && !mbar_wait(bar_empty + 8 * s, (round - 1) & 1, deadline)) {
                    record_error(1);
                    ok = false;
                    break;
                }
                const uint32_t st = sbase + s * L::kStage;
                mbar_expect_tx(bar_loaded + 8 * s, kCodeBytes + L::kBBytes);
                tma_load_2d(st + kABytes + L::kBBytes, &tmap_codes, kb * 32, n0, bar_loaded + 8 * s);
                tma_load_2d(st + kABytes, &tmap_x, kb * 64, m0, bar_loaded + 8 * s);
                issued = kb + 1;
            }
            // drain: every issued load has landed before the CTA may exit
            const long long dl = clock64() + kDrainCycles;
            for (int kb = issued - kStages > 0 ? issued - kStages : 0; kb < issued; kb++)
                mbar_wait(bar_loaded + 8 * (kb % kStages), (kb / kStages) & 1, dl);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = instr_desc<T>();
            int committed = 0;
            for (int kb = 0; kb < KB; kb++) {
                const int s = kb % kStages;
                if (!mbar_wait(bar_full + 8 * s, (kb / kStages) & 1, deadline)) {
                    record_error(2);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t st = sbase + s * L::kStage;
                const uint64_t adesc = smem_desc_sw128(st);
                const uint64_t bdesc = smem_desc_sw128(st + kABytes);
#pragma unroll
                for (int ks = 0; ks < 4; ks++)  // four K=16 steps across the 128-byte swizzle row
                    mma_bf16(tmem_base, adesc + 2 * ks, bdesc + 2 * ks, idesc, (kb | ks) != 0);
                mma_commit(bar_empty + 8 * s);
                committed = kb + 1;
            }
            mma_commit(bar_accum);  // arrives once every MMA issued above has completed
            if (!ok) {              // drain the MMAs already issued before the memory is released
                mbar_wait(bar_accum, 0, clock64() + kDrainCycles);
            }
            (void)committed;
        }
    } else {
        // ---------------- dequant (then epilogue) ----------------
        const int dt = threadIdx.x - 64;  // 0..255
        const int r = dt >> 1, h = dt & 1;
        const int64_t n = n0 + r;
        const bool valid = n < N;
        const uint16_t* srow = scales + n * G;
        // Scales of the next kScaleAhead groups are kept in flight in a register ring (indexed by
        // kb % kScaleAhead after unrolling, so it stays in registers).
        constexpr int kScaleAhead = 4;
        uint16_t ring[kScaleAhead];
#pragma unroll
        for (int u = 0; u < kScaleAhead; u++) ring[u] = (valid && u < KB) ? ld_nc_u16(srow + u) : uint16_t(0);
        for (int kb0 = 0; kb0 < KB && ok; kb0 += kScaleAhead) {
#pragma unroll
        for (int u = 0; u < kScaleAhead; u++) {
            const int kb = kb0 + u;
            if (kb >= KB) break;
            const int s = kb % kStages;
            const uint16_t sc = ring[u];
            if (valid && kb + kScaleAhead < KB) ring[u] = ld_nc_u16(srow + kb + kScaleAhead);
            const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(bar_loaded + 8 * s, (kb / kStages) & 1, deadline));
            if (!got) {
                record_error(3);
                ok = false;
                break;
            }
            uint8_t* st = smem + s * L::kStage;
            const uint4 cw = *reinterpret_cast<const uint4*>(st + kABytes + L::kBBytes + r * 32 + 16 * h);
            // The scale is sign * 2^E * (1 + m/1024).  Table row m of half p = E mod 2 holds
            // V[m][c] * 2^p; the remaining factor 2^(E - p) has an even exponent, so it only adds
            // (E - p) / 2 to the high byte (sign | exponent >> 1) of every nonzero entry.  Code 7 is
            // the one zero entry (high byte 3 of the second high-byte word) and is masked back to 0.
            const uint32_t sb = __float_as_uint(__half2float(__ushort_as_half(sc)));
            const int e = static_cast<int>((sb >> 23) & 0xFFu) - 127;
            const uint32_t par = static_cast<uint32_t>(e) & 1u;
            const uint32_t row = ((sb >> 13) & 0x3FFu) + 1024u * par;
            const uint32_t add = static_cast<uint32_t>((e - static_cast<int>(par)) >> 1) * 0x01010101u;
            const uint32_t sgn = (sb >> 31) ? 0x80808080u : 0u;
            uint4 tl = vtab[row + (row & ~7u)];
            uint4 th = vtab[row + (row & ~7u) + 8];
            th.x = (th.x + add) ^ sgn;
            th.y = ((th.y + add) & 0x00FFFFFFu) ^ sgn;
            th.z = (th.z + add) ^ sgn;
            th.w = (th.w + add) ^ sgn;
            if ((sb & 0x7FFFFFFFu) == 0u) {  // zero scale: every weight of the group is 0
                tl = make_uint4(0, 0, 0, 0);
                th = make_uint4(0, 0, 0, 0);
            }
            const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
            uint8_t* arow = st + r * 128;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                uint32_t wp[4];
                lookup8(words[i], tl, th, m1, p16, wp);
                const int chunk = (4 * h + i) ^ (r & 7);
                *reinterpret_cast<uint4*>(arow + 16 * chunk) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_full + 8 * s);
        }
        }
        // ---------------- epilogue ----------------
        if (ok && !__all_sync(0xFFFFFFFFu, mbar_wait(bar_accum, 0, deadline))) {
            record_error(4);
            ok = false;
        }
        if (ok) {
            tc_fence_after();
            const int quarter = warp & 3;  // TMEM lanes this warp may read
            const int col0 = (warp < 6) ? 0 : T / 2;
            const int ncols = (T >= 32) ? T / 2 : T;
            if (T >= 32 || warp < 6) {
                const int64_t nn = n0 + quarter * 32 + lane;
                for (int c = 0; c < ncols; c += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + col0 + c, v);
                    if (nn < N) {
#pragma unroll
                        for (int i = 0; i < 16; i++) {
                            const int64_t mm = m0 + col0 + c + i;
                            if (mm < M) y[mm * N + nn] = bf16_bits(__uint_as_float(v[i]));
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(L::kCols)
                     : "memory");
    }
}

}  // namespace tc
}  // namespace nf4
