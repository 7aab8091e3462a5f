// Device-side helpers shared by the NF4 kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace nf4 {

constexpr int kGroup = 64;  // weights per scale group (deep-fold README, format paragraph)

// The NormalFloat-4 table published with QLoRA (Dettmers et al., 2023, appendix), index 0..15.
// The published literals are the definition; each is an exact binary32 number.
__device__ __constant__ static const float kNF4[16] = {
    -1.0f,
    -0.6961928009986877f,
    -0.5250730514526367f,
    -0.39491748809814453f,
    -0.28444138169288635f,
    -0.18477343022823334f,
    -0.09105003625154495f,
    0.0f,
    0.07958029955625534f,
    0.16093020141124725f,
    0.24611230194568634f,
    0.33791524171829224f,
    0.44070982933044434f,
    0.5626170039176941f,
    0.7229568362236023f,
    1.0f,
};

// ---------------------------------------------------------------------------------------------
// Thin PTX wrappers
// ---------------------------------------------------------------------------------------------

// Byte permute: output byte i = byte sel_i of {b:a} (a = bytes 0-3, b = bytes 4-7); a selector
// nibble with bit 3 set replicates the sign bit of the addressed byte instead.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// acc + lo16(w) * lo16(x) and acc + hi16(w) * hi16(x) with bf16 operands: the product of two bf16
// numbers is exact in fp32, so each step rounds once (fp32 accumulate).
__device__ __forceinline__ void fma_bf16x2(float& acc_lo, float& acc_hi, uint32_t w, uint32_t x) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
        : "+f"(acc_lo), "+f"(acc_hi)
        : "r"(w), "r"(x));
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_ca_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_nc_u16(const uint16_t* p) {
    uint16_t v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// 16-byte asynchronous global -> shared copy; bytes past `src_bytes` (0..16) are zero-filled.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src, uint32_t src_bytes = 16) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gmem_src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch: let the next grid in the stream start launching, and wait until
// the previous grid has completed and its writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// Two floats from shared-window address `a` (8-byte aligned).
__device__ __forceinline__ float2 lds_f2(uint32_t a) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}

// 16 bits from shared-window address `a` (2-byte aligned).
__device__ __forceinline__ uint16_t lds_u16(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

// ---------------------------------------------------------------------------------------------
// Dequantization by pair table: w_hat = bf16(fp32(T[c] * scale)), two weights at a time.  A code
// byte (two codes, low nibble first) indexes a 256-entry shared-memory table whose entry is the
// fp32 pair {T[low nibble], T[high nibble]}; one packed fp32x2 multiply by the group's scale (round
// to nearest) and one bf16x2 conversion (round to nearest even) give both weights.  The table is
// replicated so that a warp's 64-bit loads never conflict, whatever the codes are.
// ---------------------------------------------------------------------------------------------
constexpr int kPairTabBytes = 256 * 32 * 8;  // 32 copies, one 8-byte column per lane (64 KB)

// Two dequantized weights from one code byte: the pair-table entry {T[c0], T[c1]} (fetched by the
// caller) times the scale in one packed fp32 multiply, then both rounded to bf16 (c0 in the low
// half).  Equals bf16(fp32(T[c] * scale)) for each code.
__device__ __forceinline__ uint32_t scale_pair(float2 t, float s) {
    uint32_t d;
    asm("{\n\t.reg .b64 t, s2, r;\n\t.reg .f32 p0, p1;\n\t"
        "mov.b64 t, {%1, %2};\n\t"
        "mov.b64 s2, {%3, %3};\n\t"
        "mul.rn.f32x2 r, t, s2;\n\t"
        "mov.b64 {p0, p1}, r;\n\t"
        "cvt.rn.bf16x2.f32 %0, p1, p0;\n\t}"
        : "=r"(d)
        : "f"(t.x), "f"(t.y), "f"(s));
    return d;
}

// Writes the pair table (kPairTabBytes at `tab`): slot e holds entry v = e / 32, the fp32 pair
// {T[v & 15], T[v >> 4]} of code byte v, for lane column e % 32.  Threads `tid` of `nthreads` (a
// multiple of 32) share the work; a warp's 32 slots belong to one entry, so the constant reads do
// not diverge.
__device__ __forceinline__ void build_pair_table(float2* tab, int tid, int nthreads) {
    for (int e = tid; e < kPairTabBytes / 8; e += nthreads) {
        const int v = e >> 5;
        tab[e] = make_float2(kNF4[v & 15], kNF4[v >> 4]);
    }
}

// Shared-memory offset of the pair-table entry of byte p (0..3) of a code word for the lane whose
// column offset is `lcol` (8 * lane): 256 * byte + lcol, built by one byte permute.
__device__ __forceinline__ uint32_t pair_offset(uint32_t word, uint32_t lcol, int p) {
    return prmt(word, lcol, 0x6504u + 16u * static_cast<uint32_t>(p));
}

// The half-size pair table (kPairTab16Bytes, for kernels whose shared memory is short): 16 copies
// side by side, slot e holding entry v = e / 16, and lane l reads copy l % 16.  A 64-bit load is
// served per half-warp, so 16 copies keep every half-warp's lanes on distinct bank pairs.
constexpr int kPairTab16Bytes = 256 * 16 * 8;
__device__ __forceinline__ void build_pair_table16(float2* tab, int tid, int nthreads) {
    for (int e = tid; e < kPairTab16Bytes / 8; e += nthreads) {
        const int v = e >> 4;
        tab[e] = make_float2(kNF4[v & 15], kNF4[v >> 4]);
    }
}
// Offset of byte p's entry in the half-size table for a lane with lcol16 = 16 * (lane % 16):
// 128 * byte + 8 * (lane % 16), a byte permute and a shift.
__device__ __forceinline__ uint32_t pair_offset16(uint32_t word, uint32_t lcol16, int p) {
    return prmt(word, lcol16, 0x6504u + 16u * static_cast<uint32_t>(p)) >> 1;
}

// Bulk (TMA-engine) copy global -> shared of `bytes` (multiple of 16, both addresses 16-byte
// aligned) whose completion is counted as transaction bytes on mbarrier `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void mbar_expect_tx_only(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// mbarrier helpers (shared-memory barrier objects in the CTA's own shared memory)
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_count(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Tests phase `parity` of `bar` (the hardware may hold the thread up to the hint, 1 us, while the
// phase is incomplete).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(1000u)
        : "memory");
    return ok != 0;
}

// Wall-clock time in nanoseconds (the GPU's global timer; the same on every SM).
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on phase `parity`: true once the phase has completed, false if it has not completed
// `limit_ns` nanoseconds of wall-clock time after this wait began.  Every wait gets its own limit
// (a long kernel with many short waits never runs out).  The first test costs no timer read; after
// that the waiting warp sleeps between tests (32 ns doubling to 256 ns), so warps that wait leave
// the issue slots and the integer pipe to the warps that work, and it reads the timer only every
// eighth test.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    uint32_t sleep_ns = 32;
    for (uint32_t n = 1;; n++) {
        __nanosleep(sleep_ns);
        if (sleep_ns < 256) sleep_ns *= 2;
        if (mbar_test(bar, parity)) return true;
        if ((n & 7) == 0 && global_ns() - t0 > limit_ns) return false;
    }
}

// Non-blocking test of phase `parity` (mbarrier.test_wait never suspends the thread).
__device__ __forceinline__ bool mbar_ready(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for a warp that spends most of its time waiting off the critical path (a producer
// whose ring is full, a reducer waiting for the consumers).  A blocking try_wait keeps the waiting
// warp issuing retries, which on this GPU takes issue slots from the warps that share its
// scheduler; this wait tests without blocking and sleeps `sleep_ns` between tests instead, at the
// cost of up to about that much wake-up latency.  Same result and limit rule as mbar_wait.
__device__ __forceinline__ bool mbar_wait_idle(uint32_t bar, uint32_t parity, uint64_t limit_ns, uint32_t sleep_ns) {
    if (mbar_ready(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t n = 1;; n++) {
        __nanosleep(sleep_ns);
        if (mbar_ready(bar, parity)) return true;
        if ((n & 7) == 0 && global_ns() - t0 > limit_ns) return false;
    }
}

// One lane of a converged warp (the same lane on every call) is true.  tcgen05.mma, tcgen05.commit
// and the TMA copies are issued by a single thread, but the warp around it runs the issue loop in
// step: its operands then stay warp-uniform, which lets each instruction issue in tens of cycles
// instead of hundreds (measured on this GPU).
__device__ __forceinline__ bool elect_one() {
    uint32_t e;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
    return e != 0;
}

__device__ __forceinline__ uint16_t bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

}  // namespace nf4
