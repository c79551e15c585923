// quantize.cu -- NVFP4 quantizer (weights at load time, activations per call), the
// scale repack into the tensor-core layout, and the element-rounding diagnostic.
//
// The load-time conversion to NVFP4 and its "NVFP4 swizzle" are named by FlashRT
// docs/qwen36_usage.md (constructor paragraph; env-var table,
// FLASHRT_QWEN36_MTP_CKPT_DIR: FP8 -> BF16 -> NVFP4 at load); NVFP4 activations by
// the same table (FLASHRT_QWEN36_FUSE_SILU_MUL_QUANT).
//
// Pass 1 (amax_partial_kernel): grid-stride max |x| with 16-byte loads, one partial
// per CTA.  Pass 2 (quantize_kernel): every CTA folds the partials into the global
// scale itself (no inter-CTA counter, nothing to reset), then one thread quantizes
// one 16-element block: 64 (fp32) or 32 (bf16) contiguous bytes in, 8 packed bytes
// and one scale byte out.  Both passes are HBM-bound.
//
// FP8 checkpoints ("e4m3 block-128": E4M3 bytes with one fp32 scale per 128 x 128 tile)
// take the same two passes through their own kernels (amax_fp8_b128_kernel,
// quantize_fp8_b128_kernel): each value is bf16(e4m3 * tile scale), the chain FP8 ->
// BF16 -> NVFP4, without writing the bf16 tensor.  With 1 byte read per element these
// are bound by instruction issue rather than by HBM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "../../include/nvfp4.h"
#include "common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

template <bool kBF16>
__global__ void __launch_bounds__(kThreads)
amax_partial_kernel(const uint4* __restrict__ src, int64_t nvec, float* __restrict__ partials) {
    float m = 0.0f;
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < nvec;
         i += (int64_t)gridDim.x * kThreads) {
        const uint4 v = __ldcs(src + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (kBF16) {
                m = fmaxf(m, fabsf(bf16_to_f32(w[j] & 0xFFFFu)));
                m = fmaxf(m, fabsf(bf16_to_f32(w[j] >> 16)));
            } else {
                m = fmaxf(m, fabsf(__uint_as_float(w[j])));
            }
        }
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

template <bool kBF16, bool kSwizzled>
__global__ void __launch_bounds__(kThreads)
quantize_kernel(const void* __restrict__ src, int64_t rows, int64_t cols,
                const float* __restrict__ partials, int npartials,
                const float* __restrict__ given_g, uint8_t* __restrict__ packed,
                uint8_t* __restrict__ scales, float* __restrict__ g_out,
                uint16_t* __restrict__ deq_bf16) {
    const float g = cta_global_scale(given_g, partials, npartials);
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;

    const int64_t cb_n = cols >> 4;
    const int64_t cp4 = (cb_n + 3) >> 2;
    // with swizzled scales the grid also covers the padding (rows to 128, blocks to 4)
    const int64_t rows_iter = kSwizzled ? ((rows + 127) >> 7) << 7 : rows;
    const int64_t cb_iter = kSwizzled ? cp4 << 2 : cb_n;
    const int64_t nblk = rows_iter * cb_iter;
    for (int64_t b = blockIdx.x * (int64_t)kThreads + threadIdx.x; b < nblk;
         b += (int64_t)gridDim.x * kThreads) {
        const int64_t r = b / cb_iter, cb = b - r * cb_iter;
        if (kSwizzled && (r >= rows || cb >= cb_n)) {
            scales[swizzle_offset(r, cb, cp4)] = 0;
            continue;
        }
        const int64_t e0 = r * cols + (cb << 4);
        float t[16];
        if (kBF16) {
            const uint4* p = reinterpret_cast<const uint4*>(
                static_cast<const uint16_t*>(src) + e0);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const uint4 v = __ldcs(p + q);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    t[q * 8 + 2 * j] = bf16_to_f32(w[j] & 0xFFFFu);
                    t[q * 8 + 2 * j + 1] = bf16_to_f32(w[j] >> 16);
                }
            }
        } else {
            const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + e0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = __ldcs(p + q);
                t[4 * q] = v.x;
                t[4 * q + 1] = v.y;
                t[4 * q + 2] = v.z;
                t[4 * q + 3] = v.w;
            }
        }
        uint32_t lo, hi;
        const uint32_t s8 = quantize_block16(t, g, lo, hi);
        *reinterpret_cast<uint2*>(packed + (e0 >> 1)) = make_uint2(lo, hi);
        if (kSwizzled) scales[swizzle_offset(r, cb, cp4)] = (uint8_t)s8;
        else scales[r * cb_n + cb] = (uint8_t)s8;
        if (deq_bf16) {
            // e2m1 * e4m3 has at most 5 significant bits and lies in [2^-10, 2688]:
            // exact in bf16.
            const float s = e4m3_to_f32(s8);
            uint32_t out[8];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const uint32_t c0 = ((i < 8 ? lo : hi) >> (4 * (i & 7))) & 15u;
                const uint32_t c1 = ((i < 8 ? lo : hi) >> (4 * ((i + 1) & 7))) & 15u;
                const float m0 = (float)(c0 & 7u), m1 = (float)(c1 & 7u);
                // magnitude of code c: c < 4 ? c / 2 : (c == 4 ? 2 : c == 5 ? 3 : c == 6 ? 4 : 6)
                const float v0 = (c0 & 7u) < 4u ? 0.5f * m0 : (m0 == 7.0f ? 6.0f : m0 - 2.0f);
                const float v1 = (c1 & 7u) < 4u ? 0.5f * m1 : (m1 == 7.0f ? 6.0f : m1 - 2.0f);
                const float d0 = (c0 & 8u) ? -v0 * s : v0 * s;
                const float d1 = (c1 & 8u) ? -v1 * s : v1 * s;
                out[i / 2] = (uint32_t)f32_to_bf16_rne(d0) | ((uint32_t)f32_to_bf16_rne(d1) << 16);
            }
            uint4* dst = reinterpret_cast<uint4*>(deq_bf16 + e0);
            dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
            dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
        }
    }
}

// ---- FP8 (E4M3, one fp32 scale per 128 x 128 tile) sources --------------------------------
// A value of such a tensor, as the NVFP4 quantizer sees it: e4m3(byte) * tile scale in one
// fp32 round-to-nearest-even product, then rounded to bf16 (the checkpoint goes FP8 -> BF16
// -> NVFP4).  E4M3 values are exact in f16, so the pair conversion loses nothing.

// row and first column of 16-byte group i (cols % 16 == 0: a group lies inside one
// 128-column tile and takes one scale); 32-bit division while the indices fit
__device__ __forceinline__ float fp8_group_scale(const float* __restrict__ bs, int64_t cols,
                                                 int64_t i) {
    const int64_t gpr = cols >> 4;  // groups per row
    int64_t r;
    if (i <= 0xFFFFFFFFll && gpr <= 0xFFFFFFFFll) r = (uint32_t)i / (uint32_t)gpr;
    else r = i / gpr;
    const int64_t c = (i - r * gpr) << 4;
    return __ldg(bs + (r >> 7) * ((cols + 127) >> 7) + (c >> 7));
}

// the 16 values of a group: bytes -> f16 pairs (hardware), fp32 products, bf16 pairs (RNE)
__device__ __forceinline__ void fp8_group_values(const uint4 v, float s, float (&t)[16]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t h2 = cvt_e4m3x2_f16x2((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
        const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(f.x, s), __fmul_rn(f.y, s));
        t[2 * j] = __low2float(b);
        t[2 * j + 1] = __high2float(b);
    }
}

// Pass 1.  RN(e * s) and the bf16 rounding are monotone in |e| and odd in e, and a
// non-negative E4M3 byte orders like its value, so a group's largest |value| is
// bf16(RN(max|e| * |s|)): one byte-wise max, then one product.
__global__ void __launch_bounds__(kThreads)
amax_fp8_b128_kernel(const uint8_t* __restrict__ src, const float* __restrict__ bs,
                     int64_t cols, int64_t ngroups, float* __restrict__ partials) {
    float m = 0.0f;
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < ngroups;
         i += (int64_t)gridDim.x * kThreads) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4*>(src) + i);
        const float s = fabsf(fp8_group_scale(bs, cols, i));
        uint32_t b = __vmaxu4(__vmaxu4(v.x & 0x7F7F7F7Fu, v.y & 0x7F7F7F7Fu),
                              __vmaxu4(v.z & 0x7F7F7F7Fu, v.w & 0x7F7F7F7Fu));
        b = max(max(b & 0xFFu, (b >> 8) & 0xFFu), max((b >> 16) & 0xFFu, b >> 24));
        m = fmaxf(m, __bfloat162float(__float2bfloat16_rn(__fmul_rn(e4m3_to_f32(b), s))));
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

// One thread per 16-element block, as quantize_kernel, scales row-major.
__global__ void __launch_bounds__(kThreads)
quantize_fp8_b128_kernel(const uint8_t* __restrict__ src, const float* __restrict__ bs,
                         int64_t cols, int64_t ngroups, const float* __restrict__ partials,
                         int npartials, uint8_t* __restrict__ packed,
                         uint8_t* __restrict__ scales, float* __restrict__ g_out) {
    const float g = cta_global_scale(nullptr, partials, npartials);
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < ngroups;
         i += (int64_t)gridDim.x * kThreads) {
        float t[16];
        fp8_group_values(__ldcs(reinterpret_cast<const uint4*>(src) + i),
                         fp8_group_scale(bs, cols, i), t);
        uint32_t lo, hi;
        const uint32_t s8 = quantize_block16(t, g, lo, hi);
        reinterpret_cast<uint2*>(packed)[i] = make_uint2(lo, hi);
        scales[i] = (uint8_t)s8;
    }
}

// One thread per 16-byte line of the swizzled layout: line i of atom (rb, ka) holds
// rows rb*128 + i + {0, 32, 64, 96}, scale columns ka*4 .. ka*4+3.
__global__ void __launch_bounds__(kThreads)
repack_kernel(const uint8_t* __restrict__ s, int64_t rows, int64_t cb_n, int64_t cp4,
              uint4* __restrict__ out, int64_t nlines) {
    for (int64_t l = blockIdx.x * (int64_t)kThreads + threadIdx.x; l < nlines;
         l += (int64_t)gridDim.x * kThreads) {
        const int64_t atom = l >> 5, i = l & 31;
        const int64_t rb = atom / cp4, ka = atom - rb * cp4;
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t r = rb * 128 + j * 32 + i;
            uint32_t v = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int64_t cb = ka * 4 + c;
                if (r < rows && cb < cb_n) v |= (uint32_t)s[r * cb_n + cb] << (8 * c);
            }
            w[j] = v;
        }
        out[l] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__global__ void __launch_bounds__(kThreads)
encode_elements_kernel(const float* __restrict__ in, int64_t n, uint8_t* __restrict__ e2m1,
                       uint8_t* __restrict__ e4m3) {
    for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * kThreads) {
        const float v = in[i];
        if (e2m1) e2m1[i] = (uint8_t)e2m1_encode(v);
        if (e4m3) e4m3[i] = (uint8_t)e4m3_encode_nonneg(v > 0.0f ? v : 0.0f);
    }
}

int grid_for(int64_t items, const DevInfo& dev, int ctas_per_sm) {
    const int64_t need = (items + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)dev.sm_count * ctas_per_sm;
    return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

}  // namespace

int amax_partial_count(int64_t n_elems, int sm_count) {
    // 16-byte vectors of the smaller dtype bound the useful CTA count
    const int64_t nvec = (n_elems + 7) / 8;
    const int64_t need = (nvec + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sm_count * 8;
    return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

cudaError_t launch_quantize(const void* src, bool src_bf16, int64_t rows, int64_t cols,
                            uint8_t* packed, uint8_t* scales, bool swizzled_scales,
                            float* g_out, const float* given_g, float* partials,
                            int npartials, uint16_t* deq_bf16, cudaStream_t stream,
                            const DevInfo& dev) {
    const int64_t n = rows * cols;
    if (!given_g) {
        const int64_t nvec = n * (src_bf16 ? 2 : 4) / 16;
        if (src_bf16)
            amax_partial_kernel<true><<<npartials, kThreads, 0, stream>>>(
                static_cast<const uint4*>(src), nvec, partials);
        else
            amax_partial_kernel<false><<<npartials, kThreads, 0, stream>>>(
                static_cast<const uint4*>(src), nvec, partials);
    }
    const int64_t cb_n = cols / 16;
    const int64_t nblk = swizzled_scales ? ((rows + 127) / 128 * 128) * ((cb_n + 3) / 4 * 4)
                                         : rows * cb_n;
    const int grid = grid_for(nblk, dev, 8);
#define NVFP4_Q(B, S)                                                                   \
    quantize_kernel<B, S><<<grid, kThreads, 0, stream>>>(src, rows, cols, partials,     \
                                                         npartials, given_g, packed,    \
                                                         scales, g_out, deq_bf16)
    if (src_bf16) {
        if (swizzled_scales) NVFP4_Q(true, true); else NVFP4_Q(true, false);
    } else {
        if (swizzled_scales) NVFP4_Q(false, true); else NVFP4_Q(false, false);
    }
#undef NVFP4_Q
    return cudaGetLastError();
}

cudaError_t launch_quantize_fp8_b128(const uint8_t* src, const float* block_scales,
                                     int64_t rows, int64_t cols, uint8_t* packed,
                                     uint8_t* scales, float* g_out, float* partials,
                                     int npartials, cudaStream_t stream, const DevInfo& dev) {
    const int64_t ngroups = rows * (cols / 16);
    amax_fp8_b128_kernel<<<npartials, kThreads, 0, stream>>>(src, block_scales, cols, ngroups,
                                                             partials);
    quantize_fp8_b128_kernel<<<grid_for(ngroups, dev, 8), kThreads, 0, stream>>>(
        src, block_scales, cols, ngroups, partials, npartials, packed, scales, g_out);
    return cudaGetLastError();
}

// The row-major copy that follows the atom part: `n` scale bytes, then zero padding up to
// `padded` bytes (a multiple of 16).  Source reads stay inside the n source bytes.
__global__ void __launch_bounds__(kThreads)
rowmajor_copy_kernel(const uint8_t* __restrict__ s, int64_t n, uint4* __restrict__ out,
                     int64_t nvec) {
    for (int64_t v = blockIdx.x * (int64_t)kThreads + threadIdx.x; v < nvec;
         v += (int64_t)gridDim.x * kThreads) {
        const int64_t b = v * 16;
        uint4 r = make_uint4(0u, 0u, 0u, 0u);
        if (b + 16 <= n) {
            r = *reinterpret_cast<const uint4*>(s + b);
        } else if (b < n) {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            for (int64_t i = b; i < n; ++i) w[(i - b) >> 2] |= (uint32_t)s[i] << (8 * ((i - b) & 3));
            r = make_uint4(w[0], w[1], w[2], w[3]);
        }
        out[v] = r;
    }
}

cudaError_t launch_repack(const uint8_t* scales, int64_t rows, int64_t cols, uint8_t* out,
                          cudaStream_t stream, const DevInfo& dev) {
    const int64_t cb_n = cols / 16, cp4 = (cb_n + 3) / 4;
    const int64_t nlines = ((rows + 127) / 128) * cp4 * 32;
    repack_kernel<<<grid_for(nlines, dev, 8), kThreads, 0, stream>>>(
        scales, rows, cb_n, cp4, reinterpret_cast<uint4*>(out), nlines);
    const int64_t atom_bytes = nlines * 16;
    const int64_t n = rows * cb_n;
    const int64_t nvec = (n + 15) / 16 + 1;  // the copy, padded to 16 bytes, plus 16 bytes
    rowmajor_copy_kernel<<<grid_for(nvec, dev, 8), kThreads, 0, stream>>>(
        scales, n, reinterpret_cast<uint4*>(out + atom_bytes), nvec);
    return cudaGetLastError();
}

cudaError_t launch_encode_elements(const float* in, int64_t n, uint8_t* e2m1_out,
                                   uint8_t* e4m3_out, cudaStream_t stream,
                                   const DevInfo& dev) {
    if (n == 0) return cudaSuccess;
    encode_elements_kernel<<<grid_for(n, dev, 16), kThreads, 0, stream>>>(in, n, e2m1_out,
                                                                          e4m3_out);
    return cudaGetLastError();
}

}  // namespace nvfp4

// ---- allocation-free quantizer -----------------------------------------------------------
// Some callers cannot hand the quantizer a workspace: runtimes that plan every device
// allocation at start-up and forbid later ones, code that runs under a fixed memory
// budget with no scratch pool to lend, and latency-critical paths where cudaMalloc /
// cudaFree would stall on a device synchronization.  nvfp4_quantize_noalloc serves them
// with the same two kernels, taking the amax partials from a fixed array in device
// memory that this library owns.

namespace nvfp4 {
namespace {

// Scratch of the allocation-free quantizer: one float per pass-1 CTA.  Every GPU that
// loads the library holds these 8 KiB until the process exits.  Pass 1 writes every
// slot that pass 2 then reads, so nothing has to start at zero; calls share the array
// and keep the last call's contents.
constexpr int kNoAllocPartials = 2048;
static __device__ __align__(256) float g_noalloc_partials[kNoAllocPartials];

std::mutex g_noalloc_mu;

// cuCtxGetCurrent / cuCtxGetId, reached through the runtime so that the library needs
// no link-time dependency on the driver library.
typedef int (*CtxGetCurrentFn)(void**);
typedef int (*CtxGetIdFn)(void*, unsigned long long*);

// Identity of the calling thread's current context.  A context that a device reset
// destroyed is never given the same id again, so an address cached under an id cannot
// outlive the module load it came from.
cudaError_t current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    if (!get_current || !get_id) {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000,
                                                         cudaEnableDefault, &q1);
        if (e != cudaSuccess || q1 != cudaDriverEntryPointSuccess || !f1)
            return e != cudaSuccess ? e : cudaErrorNotSupported;
        e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
        if (e != cudaSuccess || q2 != cudaDriverEntryPointSuccess || !f2)
            return e != cudaSuccess ? e : cudaErrorNotSupported;
        get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
        get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
    void* ctx = nullptr;
    if (get_current(&ctx) != 0 || !ctx) return cudaErrorDeviceUninitialized;
    if (get_id(ctx, id) != 0) return cudaErrorDeviceUninitialized;
    return cudaSuccess;
}

struct ScratchEntry {
    unsigned long long ctx_id;
    float* ptr;
};
constexpr int kScratchEntries = 64;
ScratchEntry g_noalloc_cache[kScratchEntries] = {};
int g_noalloc_next = 0;

// Device address of g_noalloc_partials in the current context.  In host code the array's
// name only stands in for the symbol; the address a kernel can use comes from
// cudaGetSymbolAddress, looked up once per context (the first call on a device, and the
// first after a device reset or under another context made current) and cached under
// the context's id.
cudaError_t noalloc_scratch(float** out) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    unsigned long long id = 0;
    cudaError_t e = current_context_id(&id);
    if (e == cudaSuccess) {
        for (int i = 0; i < kScratchEntries; ++i)
            if (g_noalloc_cache[i].ptr && g_noalloc_cache[i].ctx_id == id) {
                *out = g_noalloc_cache[i].ptr;
                return cudaSuccess;
            }
    }
    // the lookup also makes the device's primary context current if none was yet
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_partials);
    if (e != cudaSuccess) return e;
    e = current_context_id(&id);
    if (e != cudaSuccess) return e;
    g_noalloc_cache[g_noalloc_next] = {id, static_cast<float*>(p)};
    g_noalloc_next = (g_noalloc_next + 1) % kScratchEntries;
    *out = static_cast<float*>(p);
    return cudaSuccess;
}

}  // namespace
}  // namespace nvfp4

extern "C" __attribute__((visibility("default"))) nvfp4_status nvfp4_quantize_noalloc(
    const void* src, nvfp4_dtype src_dtype, int64_t rows, int64_t cols, uint8_t* packed,
    uint8_t* scales, float* global_scale, nvfp4_stream_t stream) {
    using namespace nvfp4;
    if (!src || !packed || !scales || !global_scale) return NVFP4_ERR_NULL;
    if (src_dtype != NVFP4_F32 && src_dtype != NVFP4_BF16) return NVFP4_ERR_DTYPE;
    if (rows < 1 || cols < 16 || cols % 16 != 0 || rows > ((int64_t)1 << 30) ||
        cols > ((int64_t)1 << 30))
        return NVFP4_ERR_SHAPE;
    if (((uintptr_t)src | (uintptr_t)packed | (uintptr_t)scales) % 16 != 0 ||
        (uintptr_t)global_scale % 4 != 0)
        return NVFP4_ERR_ALIGN;
    DevInfo d;
    const nvfp4_status st = (nvfp4_status)query_device(&d);
    if (st != NVFP4_OK) return st;
    // pass 1 runs one CTA per partial, each striding over the whole input, so capping
    // the count at the array's size changes only how the work is split, as
    // nvfp4_quantize caps it at its workspace's
    int np = amax_partial_count(rows * cols, d.sm_count);
    if (np > kNoAllocPartials) np = kNoAllocPartials;
    float* partials = nullptr;
    if (noalloc_scratch(&partials) != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }
    const cudaError_t e = launch_quantize(src, src_dtype == NVFP4_BF16, rows, cols, packed,
                                          scales, false, global_scale, nullptr, partials, np,
                                          nullptr, stream, d);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}
