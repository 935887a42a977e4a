// ptx.cuh -- inline-PTX building blocks for the sm_103a NVFP4 GEMV kernels:
// mbarriers, TMA tensor loads, NVFP4/E4M3 -> f16 conversions and the f16
// tensor-core MMA.  All device-side; no host code.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace nvfp4 {

// Device error word bits (read and cleared by nvfp4_device_error()).
constexpr unsigned kDevErrTimeoutFull = 1u;    // consumer gave up waiting for a TMA stage
constexpr unsigned kDevErrTimeoutEmpty = 2u;   // producer gave up waiting for a free stage
constexpr unsigned kDevErrTimeoutDrain = 4u;   // copies still in flight at exit
constexpr unsigned kDevErrBounds = 128u;       // debug builds: an index check skipped an access

// Index checks of the kernels' computed workspace accesses (partial tiles,
// split-row counters), compiled in by -DNVFP4_DEBUG_BOUNDS: a failed check
// sets kDevErrBounds in the device error word and the caller skips the
// access (never a trap).  Release builds: always true, compiled away.
__device__ __forceinline__ bool nvfp4_in_bounds(bool ok, unsigned *err) {
#ifdef NVFP4_DEBUG_BOUNDS
    if (!ok) atomicOr(err, kDevErrBounds);
    return ok;
#else
    (void)ok;
    (void)err;
    return true;
#endif
}

// Wall-clock limit for any single wait, in nanoseconds (2 s).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch: wait for the grid ahead on the stream to
// finish (and its writes to be visible) / let the next grid start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Loads of data that the grid ahead may write (X, the global scale, the term
// scales), issued after griddep_wait().  Not the read-only path
// (ld.global.nc, __ldg): its loads presume data constant for the whole life
// of the kernel, and a kernel launched early under programmatic dependent
// launch starts before its input is final -- on GB300 such a load returned
// the value from before the grid ahead wrote it.  These are L2-coherent and
// kept after the wait by the clobber.
__device__ __forceinline__ uint4 ld_dep_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ float ld_dep_f32(const float *p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps (up to `ns` nanoseconds, or until the phase completes) instead of
// spinning, so waiting warps leave the issue slots to the working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, unsigned parity, unsigned ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// kWaitLimitNs of %globaltimer (returns false then).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ----------------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tensormap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2D tiled TMA load of box (x, y) of `tmap` into shared memory `dst`,
// completing `bytes` of transaction count on mbarrier `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ thread-block clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of shared-memory address `saddr` (this CTA's
// window) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Cluster barrier (every thread of every CTA of the cluster arrives once per
// phase): arrive with release, wait with acquire.  The warp-aligned form: the
// whole warp executes it together, converged.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Store to another CTA's shared memory (shared::cluster address).
__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// --------------------------------------------------------------- conversions
// Two E2M1 codes in one byte -> f16x2 (exact).  The low nibble lands in the
// low half.  `byte_sel` picks byte 0..3 of `w`.
template <int kByte>
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t w) {
    uint32_t d;
    static_assert(kByte >= 0 && kByte < 4, "byte index");
    if constexpr (kByte == 0) {
        asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
            " cvt.rn.f16x2.e2m1x2 %0, b0;\n}\n" : "=r"(d) : "r"(w));
    } else if constexpr (kByte == 1) {
        asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
            " cvt.rn.f16x2.e2m1x2 %0, b1;\n}\n" : "=r"(d) : "r"(w));
    } else if constexpr (kByte == 2) {
        asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
            " cvt.rn.f16x2.e2m1x2 %0, b2;\n}\n" : "=r"(d) : "r"(w));
    } else {
        asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
            " cvt.rn.f16x2.e2m1x2 %0, b3;\n}\n" : "=r"(d) : "r"(w));
    }
    return d;
}

// Runtime-indexed variant (byte = 0..3).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2_rt(uint32_t w, int byte) {
    uint32_t d;
    uint32_t v = w >> (8 * byte);
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n}\n" : "=r"(d) : "r"(v));
    return d;
}

// Two E4M3 codes (low 16 bits of `v`) -> f16x2 (exact; NaN stays NaN).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
    uint32_t d;
    asm("{\n .reg .b16 h, hh;\n mov.b32 {h, hh}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}\n"
        : "=r"(d) : "r"(v));
    return d;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// {lo, lo} and {hi, hi} from an f16x2.
__device__ __forceinline__ uint32_t dup_lo(uint32_t v) { return __byte_perm(v, v, 0x1010); }
__device__ __forceinline__ uint32_t dup_hi(uint32_t v) { return __byte_perm(v, v, 0x3232); }

// -------------------------------------------------------------------- MMA
// D[16x8] += A[16x16] * B[16x8], f16 inputs, fp32 accumulate (row.col).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp32 += f16 * f16 (mixed-precision FMA, exact product).
__device__ __forceinline__ float fma_f16_f32(uint32_t a_half_in_low, uint32_t b_half_in_low, float c) {
    float d;
    asm("{\n .reg .b16 a, b, ah, bh;\n mov.b32 {a, ah}, %1;\n mov.b32 {b, bh}, %2;\n"
        " fma.rn.f32.f16 %0, a, b, %3;\n}\n"
        : "=f"(d) : "r"(a_half_in_low), "r"(b_half_in_low), "f"(c));
    return d;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

}  // namespace nvfp4
