// act_quant.cu -- NVFP4 activations straight from the fused gate/up projection, and the
// bf16 view of NVFP4 activations for the small-M linear.
//
// FlashRT docs/qwen36_usage.md, env-var table: FLASHRT_QWEN36_FUSE_MLP_GATE_UP (gate and
// up as one GEMM) and FLASHRT_QWEN36_FUSE_SILU_MUL_QUANT (silu(gate) * up quantized to
// NVFP4 for the down projection).  The gate/up output is bf16 [M, 2I], gate in columns
// [0, I) and up in [I, 2I).  h = (g / (1 + exp(-g))) * u is computed in fp32 registers,
// one correctly rounded operation per step, and quantized by the NVFP4 block rule without
// being stored: pass 1 writes amax partials of |h| (skipped with a static global scale),
// pass 2 recomputes h per 16-element block and writes codes and tensor-core scale atoms.
// silu(g) * u is the fixed sequence of fp32 operations of silu.cuh (its exp is not the
// library's expf), which the gate/up GEMM's fused epilogue shares.
#include <cuda_fp16.h>

#include "../../include/nvfp4.h"
#include "common.cuh"
#include "gemv_helpers.cuh"
#include "internal.h"
#include "silu.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

// the 16 values of h in block b of row m (gate at column 16 b, up at I + 16 b)
__device__ __forceinline__ void h_block(const uint16_t* __restrict__ gu, int64_t I, int64_t m,
                                        int64_t b, float (&t)[16]) {
    const uint4* gp = reinterpret_cast<const uint4*>(gu + m * 2 * I + 16 * b);
    const uint4* up = reinterpret_cast<const uint4*>(gu + m * 2 * I + I + 16 * b);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint4 gv = __ldg(gp + q), uv = __ldg(up + q);
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            t[8 * q + 2 * j] = silu_mul(bf16_to_f32(gw[j] & 0xFFFFu), bf16_to_f32(uw[j] & 0xFFFFu));
            t[8 * q + 2 * j + 1] = silu_mul(bf16_to_f32(gw[j] >> 16), bf16_to_f32(uw[j] >> 16));
        }
    }
}

// row and block of block index i (32-bit division while the indices fit)
__device__ __forceinline__ void split_index(int64_t i, int64_t per_row, int64_t& r, int64_t& b) {
    if (i <= 0xFFFFFFFFll && per_row <= 0xFFFFFFFFll) r = (uint32_t)i / (uint32_t)per_row;
    else r = i / per_row;
    b = i - r * per_row;
}

__global__ void __launch_bounds__(kThreads)
amax_silu_kernel(const uint16_t* __restrict__ gu, int64_t I, int64_t nblk,
                 float* __restrict__ partials) {
    float m = 0.0f;
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < nblk;
         i += (int64_t)gridDim.x * kThreads) {
        int64_t r, b;
        split_index(i, I >> 4, r, b);
        float t[16];
        h_block(gu, I, r, b, t);
#pragma unroll
        for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(t[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float red[kThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float r = red[0];
#pragma unroll
        for (int i = 1; i < kThreads / 32; ++i) r = fmaxf(r, red[i]);
        partials[blockIdx.x] = r;
    }
}

// One thread per 16-element block of the scale grid padded to 128 rows and 4 blocks (the
// padding gets zero scales); codes row-major [M, I/2], scales in the tensor-core atoms.
__global__ void __launch_bounds__(kThreads)
quantize_silu_kernel(const uint16_t* __restrict__ gu, int64_t M, int64_t I,
                     const float* __restrict__ partials, int npartials,
                     const float* __restrict__ given_g, uint8_t* __restrict__ packed,
                     uint8_t* __restrict__ scales, float* __restrict__ g_out) {
    const float g = cta_global_scale(given_g, partials, npartials);
    if (g_out && blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
    const int64_t cb_n = I >> 4, cp4 = (cb_n + 3) >> 2;
    const int64_t cb_iter = cp4 << 2, nblk = ((M + 127) >> 7 << 7) * cb_iter;
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < nblk;
         i += (int64_t)gridDim.x * kThreads) {
        int64_t r, cb;
        split_index(i, cb_iter, r, cb);
        if (r >= M || cb >= cb_n) {
            scales[swizzle_offset(r, cb, cp4)] = 0;
            continue;
        }
        float t[16];
        h_block(gu, I, r, cb, t);
        uint32_t lo, hi;
        const uint32_t s8 = quantize_block16(t, g, lo, hi);
        *reinterpret_cast<uint2*>(packed + r * (I >> 1) + (cb << 3)) = make_uint2(lo, hi);
        scales[swizzle_offset(r, cb, cp4)] = (uint8_t)s8;
    }
}

// NVFP4 activations -> bf16 e2m1(code) * e4m3(scale), the global scale left out (at most
// 5 significant bits, within bf16's range: exact).  One thread per 16-element block.
__global__ void __launch_bounds__(kThreads)
dequant_x_kernel(const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xs, int64_t M,
                 int64_t K, uint16_t* __restrict__ out) {
    const int64_t cb_n = K >> 4, cp4 = (cb_n + 3) >> 2, nblk = M * cb_n;
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < nblk;
         i += (int64_t)gridDim.x * kThreads) {
        int64_t r, cb;
        split_index(i, cb_n, r, cb);
        const float s = e4m3_to_f32(xs[swizzle_offset(r, cb, cp4)]);
        const uint2 c = *reinterpret_cast<const uint2*>(xq + r * (K >> 1) + (cb << 3));
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t byte = ((j < 4 ? c.x : c.y) >> (8 * (j & 3))) & 0xFFu;
            const float v0 = __fmul_rn(e2m1_to_f32(byte & 15u), s);
            const float v1 = __fmul_rn(e2m1_to_f32(byte >> 4), s);
            o[j] = (uint32_t)f32_to_bf16_rne(v0) | ((uint32_t)f32_to_bf16_rne(v1) << 16);
        }
        uint4* dst = reinterpret_cast<uint4*>(out + r * K + (cb << 4));
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

int grid_for_blocks(int64_t items, const DevInfo& dev) {
    const int64_t need = (items + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)dev.sm_count * 8;
    return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

}  // namespace

cudaError_t launch_silu_mul_quantize(const uint16_t* gate_up, int64_t M, int64_t I,
                                     uint8_t* packed, uint8_t* scales, float* g_out,
                                     const float* given_g, float* partials, int npartials,
                                     cudaStream_t stream, const DevInfo& dev) {
    if (!given_g)
        amax_silu_kernel<<<npartials, kThreads, 0, stream>>>(gate_up, I, M * (I / 16),
                                                             partials);
    const int64_t nblk = (M + 127) / 128 * 128 * ((I / 16 + 3) / 4 * 4);
    quantize_silu_kernel<<<grid_for_blocks(nblk, dev), kThreads, 0, stream>>>(
        gate_up, M, I, partials, npartials, given_g, packed, scales, g_out);
    return cudaGetLastError();
}

cudaError_t launch_dequant_x(const uint8_t* xq, const uint8_t* xs, int64_t M, int64_t K,
                             uint16_t* out, cudaStream_t stream, const DevInfo& dev) {
    dequant_x_kernel<<<grid_for_blocks(M * (K / 16), dev), kThreads, 0, stream>>>(xq, xs, M, K,
                                                                                 out);
    return cudaGetLastError();
}

}  // namespace nvfp4
