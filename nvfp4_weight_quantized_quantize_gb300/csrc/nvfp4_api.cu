// nvfp4_api.cu -- the C ABI (include/nvfp4.h): argument checks on the host, the
// per-device property cache, workspace layout and kernel dispatch.  Nothing here
// allocates device memory or synchronizes (except nvfp4_workspace_error, which says
// so).
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/nvfp4.h"
#include "internal.h"

#define NVFP4_API extern "C" __attribute__((visibility("default")))

namespace nvfp4 {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kHeaderBytes = 256;      // sticky error word + reserved
constexpr int kMaxPartials = 2048;        // amax partials (>= 8 per SM on any GPU here)

std::mutex g_dev_mu;
DevInfo g_dev[kMaxDevices];

nvfp4_status current_device(DevInfo* out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (g_dev[dev].device != dev) {
            DevInfo d;
            d.device = dev;
            int v = 0;
            if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) !=
                    cudaSuccess ||
                cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
                    cudaSuccess ||
                cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                    cudaSuccess ||
                cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                    cudaSuccess) {
                cudaGetLastError();
                return NVFP4_ERR_CUDA;
            }
            d.smem_optin = (size_t)v;
            g_dev[dev] = d;
        }
        *out = g_dev[dev];
    }
    if (out->cc_major != 10 || out->cc_minor != 3) return NVFP4_ERR_DEVICE;
    return NVFP4_OK;
}

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

inline nvfp4_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return NVFP4_OK;
    t_last_cuda_error = e;
    return NVFP4_ERR_CUDA;
}

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// the tensor-core atom part, then a row-major copy (padded to 16 bytes, plus 16 bytes)
size_t repack_atom_bytes(int64_t rows, int64_t cols) {
    const int64_t rp = (rows + 127) / 128 * 128;
    const int64_t cp = (cols / 16 + 3) / 4 * 4;
    return (size_t)(rp * cp);
}

size_t repack_bytes(int64_t rows, int64_t cols) {
    return repack_atom_bytes(rows, cols) + (size_t)((rows * (cols / 16) + 15) / 16 * 16) + 16;
}

// M <= 16 on the small-M kernels.  The skinny kernel takes 9 <= M <= 16 in one pass over W
// (two token tiles) where that ring fits this K; where only its 8-token ring fits, the
// call runs tokens 0..7 and then tokens 8..M-1 (the M = 1 GEMV for one): W is streamed
// twice, the second time partly from L2 and under the first launch.  Each output depends
// on its own token only, so the split changes no result.
cudaError_t small_m(const uint16_t* x, int M, int K, const uint8_t* wq, const uint8_t* wsz,
                    const float* gw, const float* gx, int N, void* y, bool ybf, uint32_t* err,
                    bool w_static, cudaStream_t stream, const DevInfo& d) {
    // up to 8 tokens, or 9..16 where the skinny kernel takes them in one pass over W (two
    // token tiles); otherwise 9..16 tokens as two skinny passes of 8 and M - 8
    if (M <= 8 || !skinny_w4a16_takes(K, d) || skinny16_w4a16_takes(K, d))
        return launch_gemv_w4a16(x, M, K, wq, wsz, gw, gx, N, y, ybf, err, w_static, stream, d);
    const cudaError_t e =
        launch_gemv_w4a16(x, 8, K, wq, wsz, gw, gx, N, y, ybf, err, w_static, stream, d);
    if (e != cudaSuccess) return e;
    return launch_gemv_w4a16(x + (int64_t)8 * K, M - 8, K, wq, wsz, gw, gx, N,
                             static_cast<uint8_t*>(y) + (int64_t)8 * N * (ybf ? 2 : 4), ybf,
                             err, w_static, stream, d);
}

int partial_count(int64_t n, const DevInfo& d) {
    int p = amax_partial_count(n, d.sm_count);
    return p > kMaxPartials ? kMaxPartials : p;
}

// W4A4 workspace: header | xq [M, K/2] | xs swizzled | gx (16 B) | partials | deq bf16
// (M <= 16) | stream-K state of the tensor-core GEMM, then the counters of its in-kernel
// quantization of x (M > 16)
struct W4A4Layout {
    size_t xq, xs, gx, partials, deq, sk, sync, total;
};

W4A4Layout w4a4_layout(int64_t M, int64_t K, int64_t N) {
    W4A4Layout L;
    L.xq = kHeaderBytes;
    L.xs = round_up(L.xq + (size_t)(M * K / 2), 256);
    L.gx = round_up(L.xs + repack_atom_bytes(M, K), 256);
    L.partials = L.gx + 256;
    L.deq = round_up(L.partials + (size_t)kMaxPartials * 4, 256);
    L.sk = round_up(L.deq + (M <= kGemvMaxM ? (size_t)(M * K * 2) : 0), 256);
    L.sync = L.sk + (M > kGemvMaxM ? gemm_w4a4_stream_k_bytes(M, K, N) : 0);
    L.total = L.sync + (M > kGemvMaxM ? gemm_w4a4_sync_bytes(M) : 0);
    return L;
}

constexpr int64_t kMaxDim = (int64_t)1 << 30;

// nvfp4_linear_silu_mul_quantize's workspace: the fused GEMM's (error word, stream-K
// counters and partial tiles, as the W4A16 GEMM's on 2I rows); otherwise the linear's own
// workspace (error word first), then gu bf16 [M, 2I]
struct SiluLayout {
    bool fused;
    size_t gu, total;
};

SiluLayout silu_layout(int64_t M, int64_t K, int64_t I) {
    SiluLayout L;
    L.fused = M > kGemvMaxM && I % 128 == 0;
    if (L.fused) {
        L.gu = 0;
        L.total = gemm_w4a16_workspace_bytes(M, K, 2 * I);
        return L;
    }
    const size_t lin = M <= kGemvMaxM ? kHeaderBytes : gemm_w4a16_workspace_bytes(M, K, 2 * I);
    L.gu = round_up(lin, 256);
    L.total = L.gu + (size_t)(M * 2 * I * 2);
    return L;
}

}  // namespace
}  // namespace nvfp4

namespace nvfp4 {
int query_device(DevInfo* out) { return (int)current_device(out); }

namespace {
thread_local bool t_expire_waits = false;
thread_local bool t_w4a4_pairs = false;
thread_local bool t_w4a4_prepass = false;
constexpr uint64_t kDebugWaitNs = 200000;  // 200 us
}  // namespace

WaitCfg current_wait_cfg() {
    WaitCfg w;
    if (t_expire_waits) {
        w.wait_ns = kDebugWaitNs;
        w.stall = 1;
    }
    return w;
}

bool w4a4_use_pairs() { return t_w4a4_pairs; }
bool w4a4_prepass_forced() { return t_w4a4_prepass; }
}  // namespace nvfp4

using namespace nvfp4;

NVFP4_API const char* nvfp4_status_str(nvfp4_status s) {
    switch (s) {
        case NVFP4_OK: return "NVFP4_OK";
        case NVFP4_ERR_NULL: return "NVFP4_ERR_NULL: a required pointer is NULL";
        case NVFP4_ERR_SHAPE: return "NVFP4_ERR_SHAPE: a size is out of range";
        case NVFP4_ERR_ALIGN: return "NVFP4_ERR_ALIGN: a pointer is misaligned";
        case NVFP4_ERR_DTYPE: return "NVFP4_ERR_DTYPE: unknown dtype or mode";
        case NVFP4_ERR_WORKSPACE: return "NVFP4_ERR_WORKSPACE: workspace missing or too small";
        case NVFP4_ERR_DEVICE: return "NVFP4_ERR_DEVICE: the current device is not sm_103";
        case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA: a CUDA call failed";
        case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT: a device-side wait ran out";
        case NVFP4_ERR_UNSUPPORTED: return "NVFP4_ERR_UNSUPPORTED: no kernel for this case";
    }
    return "unknown nvfp4_status";
}

NVFP4_API size_t nvfp4_repack_bytes(int64_t rows, int64_t cols) {
    if (rows < 1 || cols < 16 || cols % 16 != 0 || rows > kMaxDim || cols > kMaxDim) return 0;
    return repack_bytes(rows, cols);
}

NVFP4_API size_t nvfp4_workspace_bytes(int op, int64_t M, int64_t K, int64_t N,
                                       nvfp4_mode mode) {
    mode = (nvfp4_mode)(mode & ~NVFP4_STATIC_WEIGHTS);
    if (op == 0) {
        if (M < 1 || K < 16 || K % 16 != 0) return (size_t)-1;
        return kHeaderBytes + (size_t)kMaxPartials * 4;
    }
    if (op == 2) {
        if (M < 1 || K < 32 || K % 32 != 0 || N < 16 || N % 16 != 0) return (size_t)-1;
        return silu_layout(M, K, N).total;
    }
    if (op != 1 || M < 1 || K < 32 || K % 32 != 0 || N < 1) return (size_t)-1;
    if (mode == NVFP4_W4A16)
        return M <= kGemvMaxM ? kHeaderBytes : gemm_w4a16_workspace_bytes(M, K, N);
    if (mode == NVFP4_W4A4) return w4a4_layout(M, K, N).total;
    return (size_t)-1;
}

NVFP4_API nvfp4_status nvfp4_w4a4_workspace_layout(int64_t M, int64_t K, size_t* xq_offset,
                                                   size_t* xs_offset, size_t* gx_offset) {
    if (M < 1 || K < 32 || K % 32 != 0) return NVFP4_ERR_SHAPE;
    const W4A4Layout L = w4a4_layout(M, K, 1);  // these offsets do not depend on N
    if (xq_offset) *xq_offset = L.xq;
    if (xs_offset) *xs_offset = L.xs;
    if (gx_offset) *gx_offset = L.gx;
    return NVFP4_OK;
}

NVFP4_API nvfp4_status nvfp4_workspace_error(void* workspace, nvfp4_stream_t stream,
                                             uint32_t* bits) {
    if (!workspace || !bits) return NVFP4_ERR_NULL;
    uint32_t w = 0;
    cudaError_t e = cudaMemcpyAsync(&w, workspace, 4, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && w != 0) {
        e = cudaMemsetAsync(workspace, 0, 4, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    *bits = w;
    return w ? NVFP4_ERR_TIMEOUT : NVFP4_OK;
}

NVFP4_API nvfp4_status nvfp4_quantize(const void* src, nvfp4_dtype src_dtype, int64_t rows,
                                      int64_t cols, uint8_t* packed, uint8_t* scales,
                                      float* global_scale, void* workspace,
                                      size_t workspace_bytes, nvfp4_stream_t stream) {
    if (!src || !packed || !scales || !global_scale || !workspace) return NVFP4_ERR_NULL;
    if (src_dtype != NVFP4_F32 && src_dtype != NVFP4_BF16) return NVFP4_ERR_DTYPE;
    if (rows < 1 || cols < 16 || cols % 16 != 0 || rows > kMaxDim || cols > kMaxDim)
        return NVFP4_ERR_SHAPE;
    if (!aligned(src, 16) || !aligned(packed, 16) || !aligned(scales, 16) ||
        !aligned(workspace, 16) || !aligned(global_scale, 4))
        return NVFP4_ERR_ALIGN;
    if (workspace_bytes < nvfp4_workspace_bytes(0, rows, cols, 0, NVFP4_W4A16))
        return NVFP4_ERR_WORKSPACE;
    DevInfo d;
    nvfp4_status st = current_device(&d);
    if (st != NVFP4_OK) return st;
    float* partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kHeaderBytes);
    return from_cuda(launch_quantize(src, src_dtype == NVFP4_BF16, rows, cols, packed, scales,
                                     false, global_scale, nullptr, partials,
                                     partial_count(rows * cols, d), nullptr, stream, d));
}

NVFP4_API nvfp4_status nvfp4_quantize_fp8_block128(const uint8_t* src,
                                                   const float* block_scales, int64_t rows,
                                                   int64_t cols, uint8_t* packed,
                                                   uint8_t* scales, float* global_scale,
                                                   void* workspace, size_t workspace_bytes,
                                                   nvfp4_stream_t stream) {
    if (!src || !block_scales || !packed || !scales || !global_scale || !workspace)
        return NVFP4_ERR_NULL;
    if (rows < 1 || cols < 16 || cols % 16 != 0 || rows > kMaxDim || cols > kMaxDim)
        return NVFP4_ERR_SHAPE;
    if (!aligned(src, 16) || !aligned(packed, 16) || !aligned(scales, 16) ||
        !aligned(workspace, 16) || !aligned(block_scales, 4) || !aligned(global_scale, 4))
        return NVFP4_ERR_ALIGN;
    if (workspace_bytes < nvfp4_workspace_bytes(0, rows, cols, 0, NVFP4_W4A16))
        return NVFP4_ERR_WORKSPACE;
    DevInfo d;
    nvfp4_status st = current_device(&d);
    if (st != NVFP4_OK) return st;
    float* partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kHeaderBytes);
    return from_cuda(launch_quantize_fp8_b128(src, block_scales, rows, cols, packed, scales,
                                              global_scale, partials,
                                              partial_count(rows * cols, d), stream, d));
}

NVFP4_API nvfp4_status nvfp4_repack(const uint8_t* scales_rowmajor, int64_t rows, int64_t cols,
                                    uint8_t* scales_swizzled, size_t swizzled_bytes,
                                    nvfp4_stream_t stream) {
    if (!scales_rowmajor || !scales_swizzled) return NVFP4_ERR_NULL;
    if (rows < 1 || cols < 16 || cols % 16 != 0 || rows > kMaxDim || cols > kMaxDim)
        return NVFP4_ERR_SHAPE;
    if (swizzled_bytes != repack_bytes(rows, cols)) return NVFP4_ERR_SHAPE;
    if (!aligned(scales_rowmajor, 16) || !aligned(scales_swizzled, 16)) return NVFP4_ERR_ALIGN;
    DevInfo d;
    nvfp4_status st = current_device(&d);
    if (st != NVFP4_OK) return st;
    return from_cuda(launch_repack(scales_rowmajor, rows, cols, scales_swizzled, stream, d));
}

NVFP4_API nvfp4_status nvfp4_linear(const void* x, int64_t M, int64_t K,
                                    const uint8_t* w_packed, const uint8_t* w_scales_swizzled,
                                    const float* w_global_scale, int64_t N, void* y,
                                    nvfp4_dtype y_dtype, nvfp4_mode mode,
                                    const float* x_global_scale, void* workspace,
                                    size_t workspace_bytes, nvfp4_stream_t stream) {
    if (!x || !w_packed || !w_scales_swizzled || !w_global_scale || !y) return NVFP4_ERR_NULL;
    const bool w_static = (mode & NVFP4_STATIC_WEIGHTS) != 0;
    mode = (nvfp4_mode)(mode & ~NVFP4_STATIC_WEIGHTS);
    if (y_dtype != NVFP4_F32 && y_dtype != NVFP4_BF16) return NVFP4_ERR_DTYPE;
    if (mode != NVFP4_W4A16 && mode != NVFP4_W4A4) return NVFP4_ERR_DTYPE;
    if (mode == NVFP4_W4A16 && x_global_scale) return NVFP4_ERR_DTYPE;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return NVFP4_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(w_packed, 16) || !aligned(w_scales_swizzled, 16) ||
        !aligned(y, 16) || !aligned(w_global_scale, 4) ||
        (x_global_scale && !aligned(x_global_scale, 4)) || (workspace && !aligned(workspace, 16)))
        return NVFP4_ERR_ALIGN;
    const size_t need = nvfp4_workspace_bytes(1, M, K, N, mode);
    if (need > 0 && (!workspace || workspace_bytes < need)) return NVFP4_ERR_WORKSPACE;
    DevInfo d;
    nvfp4_status st = current_device(&d);
    if (st != NVFP4_OK) return st;
    const bool ybf = y_dtype == NVFP4_BF16;
    const uint16_t* xb = static_cast<const uint16_t*>(x);

    if (mode == NVFP4_W4A16) {
        if (M <= kGemvMaxM)
            return from_cuda(small_m(xb, (int)M, (int)K, w_packed, w_scales_swizzled,
                                     w_global_scale, nullptr, (int)N, y, ybf,
                                     static_cast<uint32_t*>(workspace), w_static, stream, d));
        return from_cuda(launch_gemm_w4a16(xb, (int)M, (int)K, w_packed, w_scales_swizzled,
                                           w_global_scale, (int)N, y, ybf,
                                           static_cast<uint8_t*>(workspace), stream, d));
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const W4A4Layout L = w4a4_layout(M, K, N);
    float* gx = reinterpret_cast<float*>(ws + L.gx);
    // W4A4 at M <= 8 with a static activation scale, or at M = 1 with a dynamic one: the
    // quantization of x is fused into the small-M kernels (no pre-pass; the same codes and
    // scales as below, which the dynamic M = 1 path also leaves in the workspace)
    if ((x_global_scale && M <= 8) || (!x_global_scale && M == 1 && !w4a4_prepass_forced())) {
        bool launched = false;
        const cudaError_t e = launch_gemv_w4a4_static(
            xb, (int)M, (int)K, w_packed, w_scales_swizzled, w_global_scale, x_global_scale,
            (int)N, y, ybf, static_cast<uint32_t*>(workspace), w_static, stream, d, &launched,
            ws + L.xq, ws + L.xs, gx);
        if (e != cudaSuccess || launched) return from_cuda(e);
    }
    // W4A4: quantize x into the workspace (bit-exact with nvfp4_quantize + nvfp4_repack)
    if (M > kGemvMaxM && !w4a4_prepass_forced()) {
        // one kernel: x quantized by the GEMM's own CTAs, then the block-scaled GEMM
        const cudaError_t e = launch_gemm_w4a4_quant_x(
            xb, x_global_scale, gx, reinterpret_cast<float*>(ws + L.partials),
            reinterpret_cast<uint32_t*>(ws + L.sync), ws + L.xq, ws + L.xs, (int)M, (int)K,
            w_packed, w_scales_swizzled, w_global_scale, (int)N, y, ybf,
            reinterpret_cast<uint32_t*>(ws), ws + L.sk, stream, d);
        // a device that cannot hold the whole grid at once (SMs taken by other contexts)
        // refuses the cooperative launch: quantize first, then the GEMM, as two kernels
        if (e != cudaErrorCooperativeLaunchTooLarge) return from_cuda(e);
        cudaGetLastError();
    }
    uint16_t* deq = M <= kGemvMaxM ? reinterpret_cast<uint16_t*>(ws + L.deq) : nullptr;
    cudaError_t e = launch_quantize(x, true, M, K, ws + L.xq, ws + L.xs, true, gx,
                                    x_global_scale, reinterpret_cast<float*>(ws + L.partials),
                                    partial_count(M * K, d), deq, stream, d);
    if (e != cudaSuccess) return from_cuda(e);
    if (M <= kGemvMaxM)
        return from_cuda(small_m(deq, (int)M, (int)K, w_packed, w_scales_swizzled,
                                 w_global_scale, gx, (int)N, y, ybf,
                                 reinterpret_cast<uint32_t*>(ws), w_static, stream, d));
    return from_cuda(launch_gemm_w4a4(ws + L.xq, ws + L.xs, gx, (int)M, (int)K, w_packed,
                                      w_scales_swizzled, w_global_scale, (int)N, y, ybf,
                                      reinterpret_cast<uint32_t*>(ws), ws + L.sk, stream, d));
}

NVFP4_API nvfp4_status nvfp4_silu_mul_quantize(const void* gate_up, int64_t M, int64_t I,
                                               uint8_t* packed, uint8_t* scales_swizzled,
                                               size_t scales_bytes, float* global_scale,
                                               const float* given_global_scale,
                                               void* workspace, size_t workspace_bytes,
                                               nvfp4_stream_t stream) {
    if (!gate_up || !packed || !scales_swizzled || !global_scale) return NVFP4_ERR_NULL;
    if (!given_global_scale && !workspace) return NVFP4_ERR_NULL;
    if (M < 1 || I < 16 || I % 16 != 0 || M > kMaxDim || I > kMaxDim) return NVFP4_ERR_SHAPE;
    if (scales_bytes < repack_atom_bytes(M, I)) return NVFP4_ERR_SHAPE;
    if (!aligned(gate_up, 16) || !aligned(packed, 16) || !aligned(scales_swizzled, 16) ||
        !aligned(global_scale, 4) || (given_global_scale && !aligned(given_global_scale, 4)) ||
        (workspace && !aligned(workspace, 16)))
        return NVFP4_ERR_ALIGN;
    if (!given_global_scale && workspace_bytes < nvfp4_workspace_bytes(0, M, I, 0, NVFP4_W4A16))
        return NVFP4_ERR_WORKSPACE;
    DevInfo d;
    nvfp4_status st = current_device(&d);
    if (st != NVFP4_OK) return st;
    float* partials = workspace ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                           kHeaderBytes)
                                : nullptr;
    return from_cuda(launch_silu_mul_quantize(static_cast<const uint16_t*>(gate_up), M, I,
                                              packed, scales_swizzled, global_scale,
                                              given_global_scale, partials,
                                              partial_count(M * I, d), stream, d));
}

NVFP4_API nvfp4_status nvfp4_linear_silu_mul_quantize(
    const void* x, int64_t M, int64_t K, const uint8_t* w_packed,
    const uint8_t* w_scales_swizzled, const float* w_global_scale, int64_t I,
    const float* h_global_scale, uint8_t* h_packed, uint8_t* h_scales_swizzled,
    size_t h_scales_bytes, int flags, void* workspace, size_t workspace_bytes,
    nvfp4_stream_t stream) {
    if (!x || !w_packed || !w_scales_swizzled || !w_global_scale || !h_global_scale ||
        !h_packed || !h_scales_swizzled || !workspace)
        return NVFP4_ERR_NULL;
    if (flags & ~NVFP4_STATIC_WEIGHTS) return NVFP4_ERR_DTYPE;
    if (M < 1 || K < 32 || K % 32 != 0 || I < 16 || I % 16 != 0 || M > kMaxDim ||
        K > kMaxDim || I > kMaxDim / 2)
        return NVFP4_ERR_SHAPE;
    if (h_scales_bytes < repack_atom_bytes(M, I)) return NVFP4_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(w_packed, 16) || !aligned(w_scales_swizzled, 16) ||
        !aligned(h_packed, 16) || !aligned(h_scales_swizzled, 16) || !aligned(workspace, 16) ||
        !aligned(w_global_scale, 4) || !aligned(h_global_scale, 4))
        return NVFP4_ERR_ALIGN;
    const SiluLayout L = silu_layout(M, K, I);
    if (workspace_bytes < L.total) return NVFP4_ERR_WORKSPACE;
    DevInfo d;
    nvfp4_status st = current_device(&d);
    if (st != NVFP4_OK) return st;
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (L.fused) {
        if (!gemm_w4a16_silu_takes(M, I, d)) return NVFP4_ERR_UNSUPPORTED;
        return from_cuda(launch_gemm_w4a16_silu(xb, (int)M, (int)K, w_packed, w_scales_swizzled,
                                                w_global_scale, (int)I, h_global_scale,
                                                h_packed, h_scales_swizzled, ws, stream, d));
    }
    uint16_t* gu = reinterpret_cast<uint16_t*>(ws + L.gu);
    const int N = (int)(2 * I);
    cudaError_t e = M <= kGemvMaxM
                        ? small_m(xb, (int)M, (int)K, w_packed, w_scales_swizzled,
                                  w_global_scale, nullptr, N, gu, true,
                                  reinterpret_cast<uint32_t*>(ws),
                                  (flags & NVFP4_STATIC_WEIGHTS) != 0, stream, d)
                        : launch_gemm_w4a16(xb, (int)M, (int)K, w_packed, w_scales_swizzled,
                                            w_global_scale, N, gu, true, ws, stream, d);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(launch_silu_mul_quantize(gu, M, I, h_packed, h_scales_swizzled, nullptr,
                                              h_global_scale, nullptr, 0, stream, d));
}

NVFP4_API nvfp4_status nvfp4_linear_nvfp4_x(const uint8_t* x_packed,
                                            const uint8_t* x_scales_swizzled,
                                            const float* x_global_scale, int64_t M, int64_t K,
                                            const uint8_t* w_packed,
                                            const uint8_t* w_scales_swizzled,
                                            const float* w_global_scale, int64_t N, void* y,
                                            nvfp4_dtype y_dtype, int flags, void* workspace,
                                            size_t workspace_bytes, nvfp4_stream_t stream) {
    if (!x_packed || !x_scales_swizzled || !x_global_scale || !w_packed || !w_scales_swizzled ||
        !w_global_scale || !y || !workspace)
        return NVFP4_ERR_NULL;
    if (y_dtype != NVFP4_F32 && y_dtype != NVFP4_BF16) return NVFP4_ERR_DTYPE;
    if (flags & ~NVFP4_STATIC_WEIGHTS) return NVFP4_ERR_DTYPE;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return NVFP4_ERR_SHAPE;
    if (!aligned(x_packed, 16) || !aligned(x_scales_swizzled, 16) || !aligned(w_packed, 16) ||
        !aligned(w_scales_swizzled, 16) || !aligned(y, 16) || !aligned(workspace, 16) ||
        !aligned(x_global_scale, 4) || !aligned(w_global_scale, 4))
        return NVFP4_ERR_ALIGN;
    if (workspace_bytes < nvfp4_workspace_bytes(1, M, K, N, NVFP4_W4A4))
        return NVFP4_ERR_WORKSPACE;
    DevInfo d;
    nvfp4_status st = current_device(&d);
    if (st != NVFP4_OK) return st;
    const bool ybf = y_dtype == NVFP4_BF16;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const W4A4Layout L = w4a4_layout(M, K, N);
    if (M <= kGemvMaxM) {
        uint16_t* deq = reinterpret_cast<uint16_t*>(ws + L.deq);
        cudaError_t e = launch_dequant_x(x_packed, x_scales_swizzled, M, K, deq, stream, d);
        if (e != cudaSuccess) return from_cuda(e);
        return from_cuda(small_m(deq, (int)M, (int)K, w_packed, w_scales_swizzled,
                                 w_global_scale, x_global_scale, (int)N, y, ybf,
                                 reinterpret_cast<uint32_t*>(ws),
                                 (flags & NVFP4_STATIC_WEIGHTS) != 0, stream, d));
    }
    return from_cuda(launch_gemm_w4a4(x_packed, x_scales_swizzled, x_global_scale, (int)M,
                                      (int)K, w_packed, w_scales_swizzled, w_global_scale,
                                      (int)N, y, ybf, reinterpret_cast<uint32_t*>(ws), ws + L.sk,
                                      stream, d));
}

NVFP4_API nvfp4_status nvfp4_encode_elements(const float* in, int64_t n, uint8_t* e2m1_out,
                                             uint8_t* e4m3_out, nvfp4_stream_t stream) {
    if (!in && n > 0) return NVFP4_ERR_NULL;
    if (n < 0) return NVFP4_ERR_SHAPE;
    if (!aligned(in, 4)) return NVFP4_ERR_ALIGN;
    DevInfo d;
    nvfp4_status st = current_device(&d);
    if (st != NVFP4_OK) return st;
    return from_cuda(launch_encode_elements(in, n, e2m1_out, e4m3_out, stream, d));
}

NVFP4_API void nvfp4_debug_expire_waits(int on) { t_expire_waits = on != 0; }

NVFP4_API void nvfp4_debug_w4a4_kernel(int which) {
    t_w4a4_pairs = which == 2;
    t_w4a4_prepass = which == 3;
}

NVFP4_API const char* nvfp4_last_cuda_error(void) {
    return cudaGetErrorString(t_last_cuda_error);
}
