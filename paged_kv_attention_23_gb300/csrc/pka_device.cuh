// pka_device.cuh — inline-PTX building blocks shared by the libpka kernels
// (sm_103a): mbarriers, bulk (TMA engine) copies, per-thread async copies,
// proxy fences, exp2 and 16-byte vector conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "pka.h"

namespace pka {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// make barrier initialisation visible to the async proxy (bulk copies)
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
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

// Bounded wait: gives up after ~2^31 clock cycles (about a second) and
// returns false so the caller can record PKA_DEVCHK_TIMEOUT and leave.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > (1ll << 31)) return false;
    }
    return true;
}

// ---- programmatic dependent launch (sm_90+) ---------------------------------
// launch_dependents: the next kernel in the stream, if launched with
// programmatic stream serialization, may start its CTAs once every CTA of
// this grid has executed this (or exited).  wait: block until the grids this
// one depends on have completed and their memory writes are visible; without
// such a dependency it returns at once.
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- copies ----------------------------------------------------------------
// Bulk global -> shared copy on the TMA engine, completion counted in bytes on
// the mbarrier.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Per-thread async copies (zero-filled past src_bytes).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// The barrier receives one arrival once all of this thread's earlier
// cp.async copies have landed (the arrival is part of the init count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses to the same bytes.
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- math ------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- 16-byte vectors <-> fp32 ------------------------------------------------
template <typename T> struct Vec;

template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void to_f32(const uint4 &u, float *f)
    {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static uint4 from_f32(const float *f)
    {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

template <> struct Vec<__half> {
    static constexpr int N = 8;
    __device__ __forceinline__ static float2 w2(uint32_t x)
    {
        __half2 h = *reinterpret_cast<__half2 *>(&x);
        return __half22float2(h);
    }
    __device__ __forceinline__ static void to_f32(const uint4 &u, float *f)
    {
        float2 a = w2(u.x), b = w2(u.y), c = w2(u.z), d = w2(u.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    }
    __device__ __forceinline__ static uint32_t n2(float a, float b)
    {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static uint4 from_f32(const float *f)
    {
        return make_uint4(n2(f[0], f[1]), n2(f[2], f[3]), n2(f[4], f[5]), n2(f[6], f[7]));
    }
};

template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void to_f32(const uint4 &u, float *f)
    {
        f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xffff0000u);
        f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xffff0000u);
        f[4] = __uint_as_float(u.z << 16); f[5] = __uint_as_float(u.z & 0xffff0000u);
        f[6] = __uint_as_float(u.w << 16); f[7] = __uint_as_float(u.w & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t n2(float a, float b)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static uint4 from_f32(const float *f)
    {
        return make_uint4(n2(f[0], f[1]), n2(f[2], f[3]), n2(f[4], f[5]), n2(f[6], f[7]));
    }
};

// acc0 += q.lo * k.lo, acc1 += q.hi * k.hi for one packed pair, with the
// 16-bit operands multiplied exactly and accumulated in f32 (mixed-precision
// FMA of sm_100+): no separate widening instructions.
template <typename T> __device__ __forceinline__ void fma2_mixed(uint32_t q, uint32_t k, float &a0, float &a1);

template <> __device__ __forceinline__ void fma2_mixed<__nv_bfloat16>(uint32_t q, uint32_t k, float &a0, float &a1)
{
    asm("{\n\t.reg .b16 ql, qh, kl, kh;\n\t"
        "mov.b32 {ql, qh}, %2;\n\t"
        "mov.b32 {kl, kh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, ql, kl, %0;\n\t"
        "fma.rn.f32.bf16 %1, qh, kh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(q), "r"(k));
}

template <> __device__ __forceinline__ void fma2_mixed<__half>(uint32_t q, uint32_t k, float &a0, float &a1)
{
    asm("{\n\t.reg .b16 ql, qh, kl, kh;\n\t"
        "mov.b32 {ql, qh}, %2;\n\t"
        "mov.b32 {kl, kh}, %3;\n\t"
        "fma.rn.f32.f16 %0, ql, kl, %0;\n\t"
        "fma.rn.f32.f16 %1, qh, kh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(q), "r"(k));
}

// Relaxed increment with wrap (atomicInc semantics) at GPU scope: a counter
// that carries no data, only an index.
__device__ __forceinline__ unsigned atom_inc_relaxed(unsigned *p, unsigned wrap)
{
    unsigned old;
    asm volatile("atom.relaxed.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(wrap) : "memory");
    return old;
}

// Release-acquire increment with wrap (atomicInc semantics) at GPU scope.
__device__ __forceinline__ unsigned atom_inc_acq_rel(unsigned *p, unsigned wrap)
{
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(wrap) : "memory");
    return old;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void flag_status(int32_t *status, int bit)
{
    if (status) atomicOr(reinterpret_cast<int *>(status), bit);
}

}  // namespace pka
