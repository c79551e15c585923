// gemv.cu -- W4A16 NVFP4 GEMV / skinny GEMM for M <= 16 (decode M = 1, MTP verify
// M = K + 1).  Qwen3x-Orin README (quick start, "--projection-backend sm87"): the
// decode projection streams every weight once per token; FlashRT
// docs/qwen36_usage.md (speculative decode argument table): verify runs K + 1 rows
// against the same weights.
//
//   y[m, n] = gw * (gx ? gx : 1) * sum_b s[n, b] * sum_{k in b} x[m, k] * e2m1(q[n, k])
//
// Design (HBM-bound: 0.5625 bytes of weight per multiply-add at M = 1):
//   - a persistent grid of CTAs_PER_SM x SMs CTAs; CTA c owns the contiguous row range
//     [N c / G, N (c+1) / G), so every CTA streams one contiguous slab of the packed
//     weights and the per-CTA work differs by at most one row;
//   - the CTA stages x (bf16, all M rows, one K chunk at a time) in shared memory,
//     split into 16-byte pieces laid out so that a warp's 32 lanes read 32
//     consecutive pieces (conflict-free);
//   - a warp takes one row at a time; lane l streams 16-byte weight chunks
//     l, l+32, ... of the row (512 contiguous bytes per warp load, four loads in
//     flight per lane), reading the two E4M3 scales of the chunk's two 16-blocks from
//     the swizzled layout (adjacent bytes);
//   - E2M1 -> fp16 by placing the 3 magnitude bits at bits 9..11 (value * 2^-14, the
//     subnormal case included) and the sign at bit 15, then fp32 FMAs with x; the
//     2^14 is folded into the block scale;
//   - per-lane fp32 partials, a warp-shuffle reduction per row, and across K chunks
//     an fp32 row accumulator in shared memory.
#include <cuda_fp16.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCtasPerSm = 4;
constexpr int kXSmemBytes = 48 * 1024;  // x staging per CTA
constexpr int kUnroll = 4;              // 16-byte weight loads in flight per lane

// 8 E2M1 codes of a word (element 2i in the low nibble of byte i) -> 8 floats, each
// equal to the code's value times 2^-14.
__device__ __forceinline__ void decode8(uint32_t w, float (&f)[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t b = (w >> (8 * i)) & 0xFFu;
        const uint32_t bits = ((b & 7u) << 9) | ((b & 8u) << 12) | ((b & 0x70u) << 21) |
                              ((b & 0x80u) << 24);
        const float2 ff = __half22float2(*reinterpret_cast<const __half2*>(&bits));
        f[2 * i] = ff.x;
        f[2 * i + 1] = ff.y;
    }
}

template <int MT>
__global__ void __launch_bounds__(kThreads)
gemv_w4a16_kernel(const uint16_t* __restrict__ x, int M, int K, const uint8_t* __restrict__ wq,
                  const uint8_t* __restrict__ wsz, const float* __restrict__ gw,
                  const float* __restrict__ gx, int N, void* __restrict__ y, int y_bf16,
                  int kc_max) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint4* xs = reinterpret_cast<uint4*>(smem);                            // [MT][4][pitch]
    float* acc_sm = reinterpret_cast<float*>(smem + (size_t)MT * kc_max * 2);  // [rows][MT]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = (int64_t)N * blockIdx.x / gridDim.x;
    const int64_t r1 = (int64_t)N * (blockIdx.x + 1) / gridDim.x;
    const int nrows = (int)(r1 - r0);
    const int64_t cp4 = ((K >> 4) + 3) >> 2;
    const int64_t row_bytes = K >> 1;
    const int pitch = kc_max >> 5;

    for (int kc0 = 0; kc0 < K; kc0 += kc_max) {
        const int kl = min(kc_max, K - kc0);
        const int nch = kl >> 5;  // 16-byte weight chunks of a row in this K chunk
        __syncthreads();
        for (int i = threadIdx.x; i < MT * 4 * nch; i += kThreads) {
            const int m = i / (4 * nch);
            const int rem = i - m * 4 * nch;
            const int c = rem >> 2, j = rem & 3;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (m < M)
                v = *reinterpret_cast<const uint4*>(x + (int64_t)m * K + kc0 + 32 * c + 8 * j);
            xs[(m * 4 + j) * pitch + c] = v;
        }
        __syncthreads();

        for (int lr = warp; lr < nrows; lr += kWarps) {
            const int64_t r = r0 + lr;
            const uint8_t* wrow = wq + r * row_bytes + (kc0 >> 1);
            float acc[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[m] = 0.0f;

            for (int cbase = 0; cbase < nch; cbase += 32 * kUnroll) {
                uint4 wv[kUnroll];
                uint32_t s01[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int c = cbase + u * 32 + lane;
                    if (c < nch) {
                        wv[u] = ld_stream_u4(wrow + 16 * (int64_t)c);
                        s01[u] = ld_nc_u16(wsz + swizzle_offset(r, (kc0 >> 4) + 2 * c, cp4));
                    } else {
                        wv[u] = make_uint4(0u, 0u, 0u, 0u);
                        s01[u] = 0u;
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int c = cbase + u * 32 + lane;
                    if (c >= nch) break;
                    const float s0 = e4m3_to_f32(s01[u] & 0xFFu) * 16384.0f;
                    const float s1 = e4m3_to_f32(s01[u] >> 8) * 16384.0f;
                    const uint32_t w[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
                    float p0[MT], p1[MT];
#pragma unroll
                    for (int m = 0; m < MT; ++m) p0[m] = p1[m] = 0.0f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float wf[8];
                        decode8(w[j], wf);
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            const uint4 xv = xs[(m * 4 + j) * pitch + c];
                            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                            float p = (j < 2) ? p0[m] : p1[m];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                p = fmaf(bf16_to_f32(xw[e] & 0xFFFFu), wf[2 * e], p);
                                p = fmaf(bf16_to_f32(xw[e] >> 16), wf[2 * e + 1], p);
                            }
                            if (j < 2) p0[m] = p; else p1[m] = p;
                        }
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) acc[m] = fmaf(s0, p0[m], fmaf(s1, p1[m], acc[m]));
                }
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
            }
            if (lane == 0) {
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    acc_sm[lr * MT + m] = (kc0 == 0 ? 0.0f : acc_sm[lr * MT + m]) + acc[m];
            }
        }
    }
    __syncthreads();
    const float scale = *gw * (gx ? *gx : 1.0f);
    for (int i = threadIdx.x; i < nrows * M; i += kThreads) {
        const int m = i / nrows, lr = i - m * nrows;
        const float v = acc_sm[lr * MT + m] * scale;
        const int64_t o = (int64_t)m * N + r0 + lr;
        if (y_bf16) static_cast<uint16_t*>(y)[o] = f32_to_bf16_rne(v);
        else static_cast<float*>(y)[o] = v;
    }
}

template <int MT>
cudaError_t launch_mt(const uint16_t* x, int M, int K, const uint8_t* wq, const uint8_t* wsz,
                      const float* gw, const float* gx, int N, void* y, bool y_bf16,
                      cudaStream_t stream, const DevInfo& dev) {
    int kc_max = (kXSmemBytes / (MT * 2)) / 32 * 32;
    if (kc_max > K) kc_max = K;
    int grid = dev.sm_count * kCtasPerSm;
    if (grid > N) grid = N;
    const int rows_max = (N + grid - 1) / grid;
    const size_t smem = (size_t)MT * kc_max * 2 + (size_t)rows_max * MT * 4;
    // opt in to the device's full dynamic shared memory once per device (not per call,
    // so that calls can be captured into CUDA graphs)
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = 1ull << (dev.device & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(gemv_w4a16_kernel<MT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)dev.smem_optin);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    if (smem > dev.smem_optin) return cudaErrorInvalidConfiguration;
    gemv_w4a16_kernel<MT><<<grid, kThreads, smem, stream>>>(x, M, K, wq, wsz, gw, gx, N, y,
                                                            y_bf16 ? 1 : 0, kc_max);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_w4a16(const uint16_t* x, int M, int K, const uint8_t* wq,
                              const uint8_t* wsz, const float* gw, const float* gx, int N,
                              void* y, bool y_bf16, cudaStream_t stream, const DevInfo& dev) {
#define NVFP4_MT(T) \
    return launch_mt<T>(x, M, K, wq, wsz, gw, gx, N, y, y_bf16, stream, dev)
    switch (M) {
        case 1: NVFP4_MT(1);
        case 2: NVFP4_MT(2);
        case 3: NVFP4_MT(3);
        case 4: NVFP4_MT(4);
        case 5: case 6: NVFP4_MT(6);
        case 7: NVFP4_MT(7);
        case 8: NVFP4_MT(8);
        case 9: case 10: case 11: case 12: NVFP4_MT(12);
        default: NVFP4_MT(16);
    }
#undef NVFP4_MT
}

}  // namespace nvfp4
