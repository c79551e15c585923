// common.cuh -- device helpers shared by the NVFP4 kernels (sm_103a).
//
// Element formats (the pages name NVFP4 -- Qwen3x-Orin README, Repository map;
// FlashRT docs/qwen36_usage.md, constructor argument table -- without defining it;
// the standard definition is used): E2M1 codes s.e1e0.m with magnitudes
// {0, .5, 1, 1.5, 2, 3, 4, 6}; E4M3 (OCP E4M3FN) block scales, bias 7, max 448.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

// ---- element rounding (the quantizer's steps 2 and 3) ----------------------------

// E2M1 code of v: nearest magnitude, ties to the even code, |v| >= 6 -> 6, and the
// sign bit of v.  The magnitude comes from the hardware converter (round to nearest even
// on the E2M1 grid, saturating); the sign bit is copied from v, so a value that rounds to
// zero keeps its sign (-0.1 -> 0x8).
__device__ __forceinline__ uint32_t e2m1_encode(float v) {
    uint32_t r;
    asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}\n"
        : "=r"(r) : "f"(0.0f), "f"(fabsf(v)));
    return (r & 7u) | ((__float_as_uint(v) >> 28) & 8u);
}

// Two codes in one byte: element a in the low nibble, b in the high one (same rounding
// and sign rule as e2m1_encode).
__device__ __forceinline__ uint32_t e2m1_encode2(float a, float b) {
    uint32_t r;
    asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}\n"
        : "=r"(r) : "f"(fabsf(b)), "f"(fabsf(a)));
    return (r & 0x77u) | ((__float_as_uint(a) >> 28) & 8u) | ((__float_as_uint(b) >> 24) & 0x80u);
}

// E4M3 byte of a non-negative float: hardware round-to-nearest-even with saturation
// to the largest finite value (448, 0x7E).  The low byte of the x2 result holds the
// second source operand.
__device__ __forceinline__ uint32_t e4m3_encode_nonneg(float s) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
    return (uint32_t)r & 0xFFu;
}

// two e4m3 bytes (low 16 bits) -> f16x2, exact
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t b2) {
    uint32_t d;
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n"
        : "=r"(d) : "r"(b2));
    return d;
}

// Value of a non-negative finite E4M3 byte (0x00..0x7E), exact.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    return e ? __uint_as_float(((e + 120u) << 23) | (m << 20))
             : (float)m * 0.001953125f;  // m * 2^-9
}

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// fp32 -> bf16 bits, round to nearest even (inputs are finite).
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
    uint32_t u = __float_as_uint(f);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// Global scale from the tensor's amax: amax / (6 * 448), or 1 for an all-zero tensor.
__device__ __forceinline__ float global_scale_from_amax(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
}

// t / d rounded to nearest even, by P. Markstein's correction step ("IA-64 and Elementary
// Functions", 2000): with r = RN(1/d) and q0 = RN(t r), the residual e = t - d q0 is exact
// (one FMA) and RN(q0 + e r) is the correctly rounded quotient, provided nothing
// under- or overflows.  Only the E2M1 code of the quotient is used, so: the caller keeps
// d in [2^-100, 2^100]; a quotient that may reach 8 in magnitude is returned as +-8 (its
// code is the saturated one, 6, either way); a tiny one may lose its last bits (its code
// is zero either way); and the sign is the dividend's (d > 0), so -0 stays -0.
__device__ __forceinline__ float div_rn_by_recip(float t, float d, float r) {
    const float q0 = __fmul_rn(t, r);
    const float e = __fmaf_rn(-q0, d, t);
    const float q = fabsf(q0) < 8.0f ? fabsf(__fmaf_rn(e, r, q0)) : 8.0f;
    return copysignf(q, t);
}

// Quantize one block of 16 fp32 values with global scale g.  Returns the E4M3 scale
// byte; `lo`/`hi` get the 8 packed bytes (element 2j in the low nibble of byte j).
// Every step is one correctly rounded fp32 operation, in the reference's order:
// s_raw = bmax / (6 g), d = e4m3(s) * g, v = t / d (the quotient correctly rounded, by
// a division or by the reciprocal correction above).
__device__ __forceinline__ uint32_t quantize_block16(const float (&t)[16], float g,
                                                     uint32_t& lo, uint32_t& hi) {
    float bmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(t[i]));
    const float s_raw = __fdiv_rn(bmax, __fmul_rn(6.0f, g));
    const uint32_t s8 = e4m3_encode_nonneg(s_raw);
    const float d = __fmul_rn(e4m3_to_f32(s8), g);
    lo = 0u;
    hi = 0u;
    if (d == 0.0f) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t code = (__float_as_uint(t[i]) >> 28) & 8u;
            if (i < 8) lo |= code << (4 * i);
            else hi |= code << (4 * (i - 8));
        }
    } else if (d >= 0x1p-100f && d <= 0x1p100f) {
        const float r = __frcp_rn(d);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const uint32_t byte = e2m1_encode2(div_rn_by_recip(t[i], d, r),
                                               div_rn_by_recip(t[i + 1], d, r));
            if (i < 8) lo |= byte << (4 * i);
            else hi |= byte << (4 * (i - 8));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            // an infinite quotient (huge t, tiny d) saturates like any value >= 6
            const uint32_t byte = e2m1_encode2(copysignf(fminf(fabsf(__fdiv_rn(t[i], d)), 8.0f), t[i]),
                                               copysignf(fminf(fabsf(__fdiv_rn(t[i + 1], d)), 8.0f), t[i + 1]));
            if (i < 8) lo |= byte << (4 * i);
            else hi |= byte << (4 * (i - 8));
        }
    }
    return s8;
}

// Global scale seen by every CTA: *given_g, or amax / 2688 from the partials.
__device__ __forceinline__ float cta_global_scale(const float* __restrict__ given_g,
                                                  const float* __restrict__ partials,
                                                  int npartials) {
    __shared__ float g_sh;
    if (given_g) {
        if (threadIdx.x == 0) g_sh = *given_g;
    } else {
        float m = 0.0f;
        for (int i = threadIdx.x; i < npartials; i += blockDim.x) m = fmaxf(m, partials[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        __shared__ float red[32];
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            float r = red[0];
            for (int i = 1; i < (int)(blockDim.x / 32); ++i) r = fmaxf(r, red[i]);
            g_sh = global_scale_from_amax(r);
        }
    }
    __syncthreads();
    return g_sh;
}

// ---- swizzled scale layout ---------------------------------------------------------
// Tensor-core block-scale layout for 16-element blocks: 512-byte atoms of 128 rows x 4
// scale columns; line (r % 32) of 16 bytes holds rows r%32 + {0,32,64,96}, 4 bytes each;
// atoms advance along K first.  cp4 = number of 4-column groups = ceil(Cb / 4).
__host__ __device__ __forceinline__ int64_t swizzle_offset(int64_t r, int64_t cb,
                                                           int64_t cp4) {
    return ((r >> 7) * cp4 + (cb >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 +
           (cb & 3);
}

// ---- loads ---------------------------------------------------------------------------

// Streaming 16-byte load that bypasses L1 allocation (weights are read once).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_nc_u16(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}


// four bytes of E2M1 code pairs -> four f16x2 (exact; element 2i in the low half)
__device__ __forceinline__ void cvt8(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// ---- mbarriers, bulk copies, bounded waits (sm_90+ / sm_100 PTX) ---------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// make barrier initialisation visible to the async proxy (bulk copies, tensor cores)
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most limit_ns
// nanoseconds of wall time; false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// load with acquire semantics at GPU scope (a count another CTA advances after its writes)
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.  Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// L2 policy for data read once (streamed weights): evicted first, so that what is reused
// (activations, outputs) stays in L2
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 cache policy for the source lines
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// named barrier over `count` threads (a multiple of 32)
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// named barrier `id` over `count` threads that also ORs a predicate: every thread gets
// true when any of them passed true
__device__ __forceinline__ bool named_bar_red_or(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
        " barrier.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// L2 prefetch of a global range (16-byte aligned start, size a multiple of 16)
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch: the next kernel on the stream may be scheduled once every
// CTA of this grid has issued launch_dependents; wait_prior_grid blocks until the grid
// before this one has completed and its memory writes are visible (a no-op when the
// kernel was launched without the programmatic attribute).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// wall-time limit of every device-side wait: far beyond any legitimate wait
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Bounded-wait settings of one launch: the wall-time limit of the waits in which one
// role (or CTA) waits for another, and a test switch with which one role withholds an
// arrival, so that such a wait runs out and the error path runs (every role stops,
// copies and MMAs in flight are drained, TMEM is freed, the error word gets
// NVFP4_DEVERR_TIMEOUT).  stall is 0 in every production launch.
struct WaitCfg {
    uint64_t wait_ns = kWaitLimitNs;
    int stall = 0;
};

}  // namespace nvfp4
