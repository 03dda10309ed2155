// dgt_device.cuh -- device helpers shared by libdgt's kernels (sm_103a).
//
// R4 decode in registers.  A weight's BF16 bits are sign<<15 | e<<7 | mant,
// with e = table[rank] (Binade README, title paragraph).  For the 16 ranks a
// nibble can hold, the exponent is looked up with byte permutes instead of a
// memory table: e is split into its high 7 bits and its low bit; a PRMT with
// the four rank nibbles as selectors reads four entries at once.  PRMT's
// default mode uses a selector's bit 3 to replicate a byte's sign bit, which
// is exploited twice:
//   hi7: entries have bit 7 clear, so ranks 0..7 read h0:h1 directly and give
//        0 for ranks 8..15; ranks 8..15 read h2:h3 with bit 3 flipped and give
//        0 for ranks 0..7; the OR of the two is the lookup.
//   lo1: byte i of l0:l1 holds lo(i) in bit 6 and lo(i+8) in bit 7; rank i<8
//        copies the byte (bit 6 = lo(i)), rank i+8 replicates bit 7 into all
//        bits (bit 6 = lo(i+8)), so bit 6 of one PRMT is the lookup.
// Nibble 15 reads table[15] here; escapes are patched separately.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dgt.h"

#define DGT_FULL 0xFFFFFFFFu

namespace dgt {

struct R4Lut {
    uint32_t h0, h1, h2, h3, l0, l1;
};

// Built on the host from a rank table.
static inline R4Lut make_r4lut(const uint8_t *table, int n_table) {
    uint32_t hi[16], lo[16];
    for (int r = 0; r < 16; r++) {
        uint32_t e = r < n_table ? table[r] : 0u;
        hi[r] = e >> 1;
        lo[r] = e & 1u;
    }
    R4Lut L;
    L.h0 = hi[0] | hi[1] << 8 | hi[2] << 16 | hi[3] << 24;
    L.h1 = hi[4] | hi[5] << 8 | hi[6] << 16 | hi[7] << 24;
    L.h2 = hi[8] | hi[9] << 8 | hi[10] << 16 | hi[11] << 24;
    L.h3 = hi[12] | hi[13] << 8 | hi[14] << 16 | hi[15] << 24;
    uint32_t lb[8];
    for (int i = 0; i < 8; i++) lb[i] = (lo[i + 8] << 7) | (lo[i] << 6);
    L.l0 = lb[0] | lb[1] << 8 | lb[2] << 16 | lb[3] << 24;
    L.l1 = lb[4] | lb[5] << 8 | lb[6] << 16 | lb[7] << 24;
    return L;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(s));
    return r;
}

// Four weights: sel = their rank nibbles in bits 0..15, self = sel ^ 0x8888,
// smw = their four sign/mantissa bytes.  Returns two BF16 pairs
// (weight 0 in the low half of p01, weight 1 in the high half, ...).
__device__ __forceinline__ void r4_dec4(uint32_t sel, uint32_t self, uint32_t smw, const R4Lut &L,
                                        uint32_t &p01, uint32_t &p23) {
    uint32_t a = prmt(L.h0, L.h1, sel);
    uint32_t b = prmt(L.h2, L.h3, self);
    uint32_t l = prmt(L.l0, L.l1, sel);
    uint32_t b3 = a | b | (smw & 0x80808080u);               // sign | e >> 1
    uint32_t b2 = ((l << 1) & 0x80808080u) | (smw & 0x7F7F7F7Fu);  // (e & 1) << 7 | mant
    p01 = prmt(b2, b3, 0x5140u);
    p23 = prmt(b2, b3, 0x7362u);
}

// Sixteen weights: nibbles n.x (weights 0..7), n.y (8..15); sign/mantissa
// bytes s.x..s.w.  Output: eight BF16 pairs.
__device__ __forceinline__ void r4_dec16(uint2 n, uint4 s, const R4Lut &L, uint32_t p[8]) {
    uint32_t f0 = n.x ^ 0x88888888u, f1 = n.y ^ 0x88888888u;
    r4_dec4(n.x, f0, s.x, L, p[0], p[1]);
    r4_dec4(n.x >> 16, f0 >> 16, s.y, L, p[2], p[3]);
    r4_dec4(n.y, f1, s.z, L, p[4], p[5]);
    r4_dec4(n.y >> 16, f1 >> 16, s.w, L, p[6], p[7]);
}

// Bit 4j set iff nibble j of x is 15.
__device__ __forceinline__ uint32_t nib15_mask(uint32_t x) {
    uint32_t t = x & (x >> 1);
    t &= t >> 2;
    return t & 0x11111111u;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// Exclusive prefix sum over the warp; *total gets the warp sum.
__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t v, uint32_t *total) {
    const uint32_t lane = lane_id();
    uint32_t x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t y = __shfl_up_sync(DGT_FULL, x, d);
        if (lane >= (uint32_t)d) x += y;
    }
    *total = __shfl_sync(DGT_FULL, x, 31);
    return x - v;
}

// float -> bf16, nearest with ties to even; NaN -> 0x7FC0.
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

__device__ __forceinline__ void set_status(int32_t *status, int32_t code) {
    if (status) atomicCAS(status, 0, code);
}

// Streaming loads that bypass L1 allocation (each byte is read once).
__device__ __forceinline__ uint4 ldg_stream16(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_stream8(const void *p) {
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

// Patch the escaped weights of one 16-weight lane chunk, given as eight BF16
// pairs p[].  m0/m1: nib15_mask of the chunk's two nibble words (0 for an
// inactive lane); escb: the segment's escape ranks in shared memory, cnt of
// them; table_s: the rank table in shared memory.  All 32 lanes must call it.
// Returns false if the segment's 15-nibbles do not add up to cnt.
__device__ __forceinline__ bool patch_escapes(uint32_t p[8], uint32_t m0, uint32_t m1, uint32_t cnt,
                                              const uint8_t *escb, const uint8_t *table_s) {
    uint32_t tot;
    uint32_t idx = warp_excl_scan(__popc(m0) + __popc(m1), &tot);
#pragma unroll
    for (int t = 0; t < 16; t++) {
        const uint32_t m = t < 8 ? m0 : m1;
        if ((m >> (4 * (t & 7))) & 1u) {
            uint32_t e = idx < cnt ? table_s[escb[idx]] : 0u;
            idx++;
            const int sh = 16 * (t & 1);
            p[t >> 1] = (p[t >> 1] & ~(0x7F80u << sh)) | (e << (7 + sh));
        }
    }
    return tot == cnt;
}

__device__ __forceinline__ float bf16lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16hi(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

// One 32-byte streaming load (sm_100+ 256-bit vector load).
__device__ __forceinline__ void ldg_stream32(const void *p, uint4 &lo, uint4 &hi) {
    asm("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
        : "l"(p));
}

// Two fused multiply-adds in column order, the bf16 operands taken straight
// from the low and high halves of w and x: acc = fma(w.lo, x.lo, acc), then
// acc = fma(w.hi, x.hi, acc).  Each is one fp32 FMA with a single rounding.
__device__ __forceinline__ float fma2_bf16(uint32_t w, uint32_t x, float acc) {
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "mov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\t"
        "fma.rn.f32.bf16 %0, a1, b1, %0;\n\t}"
        : "+f"(acc)
        : "r"(w), "r"(x));
    return acc;
}

// Lane chunk of 16 weights (eight bf16 pairs) against x staged as bf16 pairs:
// round j, lane u -> two uint4 at [(2j + h) * 32 + u].
__device__ __forceinline__ float fma_chunk16(const uint32_t p[8], const uint4 *xs, uint32_t j, uint32_t lane,
                                             float acc) {
    const uint4 xa = xs[(2 * j) * 32 + lane];
    const uint4 xb = xs[(2 * j + 1) * 32 + lane];
    acc = fma2_bf16(p[0], xa.x, acc);
    acc = fma2_bf16(p[1], xa.y, acc);
    acc = fma2_bf16(p[2], xa.z, acc);
    acc = fma2_bf16(p[3], xa.w, acc);
    acc = fma2_bf16(p[4], xb.x, acc);
    acc = fma2_bf16(p[5], xb.y, acc);
    acc = fma2_bf16(p[6], xb.z, acc);
    acc = fma2_bf16(p[7], xb.w, acc);
    return acc;
}

// ---- mbarrier and bulk-copy (TMA, 1-D) helpers --------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order earlier generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Global -> shared bulk copy completing on the barrier (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Programmatic dependent launch: let the next kernel of the stream (launched
// with programmatic serialization) start its CTAs as this one's free their
// SMs, and, in that next kernel, wait until this grid has completed and its
// memory is visible (a no-op when nothing precedes programmatically).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking check of a barrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the barrier phase with an iteration limit (each try_wait may itself
// suspend for a while); false when the limit ran out.
constexpr uint32_t MBAR_SPIN_LIMIT = 1u << 24;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < MBAR_SPIN_LIMIT; i++)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// The same with a caller-chosen limit (0: give up at once).
__device__ __forceinline__ bool mbar_wait_n(uint32_t bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; i++)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Launch-time wait limit for waits on work in flight: the library default, or
// the short limit a caller asked for through DGT_TEST_SHORT_WAITS.
static inline uint32_t wait_limit_from_flags(unsigned flags) {
    return (flags & DGT_TEST_SHORT_WAITS) ? (flags >> 16) : MBAR_SPIN_LIMIT;
}

// Producer/consumer rings with one producer lane per consumer warp: when the
// producer lane stops (its work done, or told to abort) it publishes how many
// pieces it issued, with bit 31 set, in the ring's stop word.
__device__ __forceinline__ void ring_publish_stop(uint32_t *stop_word, uint32_t issued) {
    *(volatile uint32_t *)stop_word = issued | 0x80000000u;
}

// After a consumer gave up (a wait ran out, or the CTA aborted): wait, bounded,
// for its producer to stop, then for every piece that producer issued and the
// consumer did not take (pieces consumed..issued-1 of a ring of ns stages), so
// that no bulk copy is still writing shared memory when the CTA exits.  All
// lanes of the warp call it.
__device__ __forceinline__ void ring_drain(const uint32_t *stop_word, uint32_t full_a, uint32_t consumed,
                                           uint32_t ns) {
    uint32_t v = 0;
    for (uint32_t i = 0; i < MBAR_SPIN_LIMIT; i++) {
        v = *(const volatile uint32_t *)stop_word;
        if (v >> 31) break;
        __nanosleep(64);
    }
    if (!(v >> 31)) return;
    const uint32_t issued = v & 0x7FFFFFFFu;
    for (uint32_t q = consumed; q < issued; q++) mbar_wait(full_a + 8 * (q % ns), (q / ns) & 1u);
}

}  // namespace dgt
