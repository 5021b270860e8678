// common.cuh -- small inline-PTX helpers shared by the sm_103a kernels:
// mbarriers with bounded waits, TMA tile loads, cluster/DSMEM access,
// programmatic dependent launch, the e4m3 <-> bf16 conversions and the
// bf16 mma.sync used by the skinny-GEMM decode kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8bs {

// Error bits a kernel sets in its device error word when it gives up.
enum : uint32_t {
    ERRBIT_FULL_WAIT = 1u << 0,   // consumer gave up waiting for a TMA stage
    ERRBIT_EMPTY_WAIT = 1u << 1,  // producer gave up waiting for a free stage
    ERRBIT_MMA_WAIT = 1u << 2,    // tensor-core pipeline wait expired
    ERRBIT_TMEM = 1u << 3,        // TMEM allocation problem
    ERRBIT_INDEX = 1u << 4,       // an index argument (e.g. an expert id) was out of range
};

// Every spin on an mbarrier gives up after this much wall time (globaltimer
// nanoseconds) or this many polls, whichever comes first.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kWaitLimitPolls = 1u << 30;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// the caller must record an error) if the wait exceeded its bound.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    const uint32_t addr = smem_u32(bar);
    if (mbar_try_wait(addr, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 0; i < kWaitLimitPolls; ++i) {
        if (mbar_try_wait(addr, parity)) return true;
        if ((i & 63u) == 63u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
    return false;
}

// --------------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled TMA load of one box at element coordinates (x = inner, y = outer)
// into shared memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// 3-D tiled TMA load at element coordinates (x innermost, y, z).
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int32_t x,
                                            int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// Same, with an L2 cache-policy hint (e.g. evict-first for streamed weights).
__device__ __forceinline__ void tma_load_2d_hint(void *smem_dst, const CUtensorMap *map,
                                                 uint64_t *bar, int32_t x, int32_t y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// Untiled bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load_g2s(void *smem_dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Ask for one 2-D box to be brought into L2 (no shared memory, no
// completion).  L2 is the coherence point of device memory, so a prefetch
// can never return stale data: it is safe even while the previous kernel in
// the stream may still be writing the same addresses.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------ programmatic dep. launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------- cluster / DSMEM
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::
            : "memory");
}

__device__ __forceinline__ uint32_t dsmem_map(uint32_t local_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
    return r;
}

// Store to the shared memory of a CTA of this cluster (an address from
// dsmem_map); a later cluster barrier with release / acquire semantics makes
// it visible to that CTA.
__device__ __forceinline__ void dsmem_st_f32(uint32_t cluster_addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}

// Four consecutive floats (16-byte aligned cluster address).
__device__ __forceinline__ void dsmem_st_f32x4(uint32_t cluster_addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// Volatile keeps it after the cluster barrier; several can still be in
// flight when the caller issues them before using any result.
__device__ __forceinline__ float dsmem_ld_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}

// ------------------------------------------------------------ conversions
// Two e4m3 codes -> two exact bf16 values (packed, lower code in the lower
// half).  `sel` picks the byte pair of `word`: 0x9180 for bytes 0/1, 0xB3A2
// for bytes 2/3.  prmt places each code in the low byte of a 16-bit lane and
// replicates its sign bit through the high byte; shifting left by 4 and
// masking leaves sign | 0000 | E(4) | M(3) | 0000, which read as bf16 is the
// code's value times 2^-120 (a bf16 subnormal when E = 0, exactly as e4m3
// subnormals are); one bf16x2 multiply by 2^120 restores the value exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t word, uint32_t sel) {
    uint32_t v, out;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(v) : "r"(word), "r"(sel));
    v = (v << 4) & 0x87F087F0u;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out) : "r"(v), "r"(0x7B807B80u));
    return out;
}

// Two e4m3 codes -> the bf16 pair (dec(c0), dec(c1)) * 2^-120 * f, given
// mult = the bf16x2 pair (f, f): e4m3x2_to_bf16x2 with its final multiply
// by 2^120 replaced by one by f (f = 2^120 gives the plain decode).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_mul(uint32_t word, uint32_t sel, uint32_t mult) {
    uint32_t v, out;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(v) : "r"(word), "r"(sel));
    v = (v << 4) & 0x87F087F0u;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out) : "r"(v), "r"(mult));
    return out;
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t out;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out) : "r"(a), "r"(b));
    return out;
}

// Four e4m3 codes (one 32-bit word, byte i = code i) -> two exact f16 pairs:
// lo = (code0, code1), hi = (code2, code3), lower code in the lower half.
// Every e4m3 value is exactly representable in f16 (normal or zero).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t word, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(word));
}

// Two fp32 values -> one f16 pair (round to nearest even), `lo` in the lower half.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Two fp32 values -> two e4m3 codes (round to nearest even, saturating to
// +-448), `lo` in the low byte.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t packed) {
    return __uint_as_float(packed & 0xFFFF0000u);
}

// Exponent e of the power of two 2^e that moves a bf16 magnitude (given as
// its bits, m16 = |max| of a group of x values) into [2^14, 2^15): every
// bf16 value of the group down to 2^-31 of that maximum then converts to f16
// exactly, and nothing overflows.  Clamped to [-126, 126] so that 2^e and
// 2^-e are both normal fp32; m16 == 0 gives 0.
__device__ __forceinline__ int f16_rescale_exp(uint32_t m16) {
    if (m16 == 0) return 0;
    const int field = static_cast<int>(m16 >> 7);
    const int lg = field ? field - 127 : -133;  // floor(log2 |max|) (subnormal: below -126)
    return min(126, max(-126, 14 - lg));
}
__device__ __forceinline__ float pow2_int(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// Position of x row r of a 32-row x tile in the table of its per-row f16
// inverse factors: rows 8j+t and 8j+t+4 sit next to each other, so a GEMV
// consumer thread (which owns exactly those two rows of each 8-row group)
// reads both with one 64-bit load.
__device__ __forceinline__ int xinv_slot(int r) { return (r & ~7) | ((r & 3) << 1) | ((r >> 2) & 1); }

// Encode 8 bf16 values (one uint4) divided by s into 8 e4m3 bytes (uint2).
__device__ __forceinline__ uint2 encode8_div(const uint4 v, float s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint16_t c0 = f32x2_to_e4m3x2(bf16lo_to_f32(w[2 * h]) / s, bf16hi_to_f32(w[2 * h]) / s);
        const uint16_t c1 =
            f32x2_to_e4m3x2(bf16lo_to_f32(w[2 * h + 1]) / s, bf16hi_to_f32(w[2 * h + 1]) / s);
        out[h] = static_cast<uint32_t>(c0) | (static_cast<uint32_t>(c1) << 16);
    }
    return make_uint2(out[0], out[1]);
}


// ------------------------------------------------------------- mma.sync
// D(16x8, fp32) += A(16x16, bf16, row) * B(16x8, bf16, col).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D(16x8, fp32) += A(16x16, f16, row) * B(16x8, f16, col).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

}  // namespace fp8bs
