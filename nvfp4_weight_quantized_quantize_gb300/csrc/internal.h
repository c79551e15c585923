// internal.h -- host-side launchers shared between the C-ABI layer and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace nvfp4 {

struct DevInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    size_t smem_optin = 0;  // max dynamic shared memory per block (opt-in)
};

// Number of amax partials the quantizer's first pass writes for `n_elems` inputs.
int amax_partial_count(int64_t n_elems, int sm_count);

// Quantizer: amax partials (skipped when given_g != nullptr), then one thread per
// 16-element block.  Scales go row-major [rows, cols/16] or, with swizzled_scales,
// to the swizzled layout (padding written as zero).  deq_bf16 (optional) receives
// e2m1(code) * e4m3(scale) -- the dequantized value without the global scale -- as
// bf16 [rows, cols].
cudaError_t launch_quantize(const void* src, bool src_bf16, int64_t rows, int64_t cols,
                            uint8_t* packed, uint8_t* scales, bool swizzled_scales,
                            float* g_out, const float* given_g, float* partials,
                            int npartials, uint16_t* deq_bf16, cudaStream_t stream,
                            const DevInfo& dev);

// FP8 (E4M3) source with one fp32 scale per 128 x 128 tile: each value is
// bf16(e4m3 * scale), then quantized as launch_quantize does (scales row-major).
cudaError_t launch_quantize_fp8_b128(const uint8_t* src, const float* block_scales,
                                     int64_t rows, int64_t cols, uint8_t* packed,
                                     uint8_t* scales, float* g_out, float* partials,
                                     int npartials, cudaStream_t stream, const DevInfo& dev);

// h = silu(gate) * up from bf16 gate_up [M, 2I] (gate columns [0, I)), quantized to NVFP4:
// codes [M, I/2], scales in the tensor-core atoms (rows padded to 128, blocks to 4, zero
// padding), g_out (may be null with a given scale).  Pass 1 (amax partials) only when
// given_g is null.
cudaError_t launch_silu_mul_quantize(const uint16_t* gate_up, int64_t M, int64_t I,
                                     uint8_t* packed, uint8_t* scales, float* g_out,
                                     const float* given_g, float* partials, int npartials,
                                     cudaStream_t stream, const DevInfo& dev);

// NVFP4 activations (codes [M, K/2], scale atoms) -> bf16 e2m1 * e4m3 [M, K] (exact).
cudaError_t launch_dequant_x(const uint8_t* xq, const uint8_t* xs, int64_t M, int64_t K,
                             uint16_t* out, cudaStream_t stream, const DevInfo& dev);

cudaError_t launch_repack(const uint8_t* scales, int64_t rows, int64_t cols, uint8_t* out,
                          cudaStream_t stream, const DevInfo& dev);

cudaError_t launch_encode_elements(const float* in, int64_t n, uint8_t* e2m1_out,
                                   uint8_t* e4m3_out, cudaStream_t stream,
                                   const DevInfo& dev);

// Small-M (M <= 16) W4A16 GEMV / skinny GEMM.  y = (gx ? *gx : 1) * *gw * x . W^T.
// err: the workspace's sticky error word (bounded waits OR bits into it).
// w_static: no kernel still in flight before this one writes the weights, so the M = 1
// and skinny kernels may stream them before waiting for the previous kernel on the stream
cudaError_t launch_gemv_w4a16(const uint16_t* x, int M, int K, const uint8_t* wq,
                              const uint8_t* wsz, const float* gw, const float* gx, int N,
                              void* y, bool y_bf16, uint32_t* err, bool w_static,
                              cudaStream_t stream, const DevInfo& dev);

constexpr int kGemvMaxM = 16;

// W4A4 at 1 <= M <= 8 with the quantization of x fused into the M = 1 GEMV or the skinny
// kernel (bf16 x in, no pre-pass).  With a static activation scale *gx nothing lands in
// the workspace but the error word; with gx null (M = 1 only: a dynamic scale, from x's
// own amax) the GEMV also writes x's codes, scale atoms and g_x to xq_out / xs_out /
// gx_out, as the quantizer would.  Sets *launched when a fused kernel took the call;
// otherwise nothing was enqueued and the caller quantizes x first.
cudaError_t launch_gemv_w4a4_static(const uint16_t* x, int M, int K, const uint8_t* wq,
                                    const uint8_t* wsz_all, const float* gw, const float* gx,
                                    int N, void* y, bool y_bf16, uint32_t* err, bool w_static,
                                    cudaStream_t stream, const DevInfo& dev, bool* launched,
                                    uint8_t* xq_out = nullptr, uint8_t* xs_out = nullptr,
                                    float* gx_out = nullptr);

// Whether launch_skinny_w4a16 takes calls with this K (its ring fits shared memory), for
// up to 8 tokens and for 9..16 tokens (two token tiles, one pass over W).
bool skinny_w4a16_takes(int K, const DevInfo& dev);
bool skinny16_w4a16_takes(int K, const DevInfo& dev);

// 2 <= M <= 16 W4A16 skinny GEMM streaming W through a shared-memory ring, tensor cores
// for the arithmetic (M <= 8 for the quantizing W4A4 variant).  wrm: the row-major part of the repacked scales.  Sets *launched
// when it took the call (K small enough for its ring); otherwise the caller falls back.
cudaError_t launch_skinny_w4a16(const uint16_t* x, int M, int K, const uint8_t* wq,
                                const uint8_t* wrm, const float* gw, const float* gx, int N,
                                void* y, bool y_bf16, uint32_t* err, bool w_static,
                                cudaStream_t stream, const DevInfo& dev, bool* launched,
                                bool x_quant_static = false);

// M > 16 W4A16 GEMM on the tensor cores (tcgen05, TMA).  wsz: the atom part of the
// repacked scales (offset 0 of the repacked buffer).  y = *gw * x . W^T.
// Workspace: the 256-byte header (error word) | stream-K counters, 4 per tile (zero before
// the first call; every completed call leaves them zero) | fp32 partial-tile slots.
constexpr size_t kGemmHeaderBytes = 256;
struct GemmPlan {
    int nkb = 0, ntiles_m = 0, ntiles = 0, ntiles_sk = 0, p_sk = 0, grid = 0;
    int64_t tsk = 0;
};
GemmPlan gemm_w4a16_plan(int64_t M, int64_t K, int64_t N, int sm_count);
size_t gemm_w4a16_workspace_bytes(int64_t M, int64_t K, int64_t N);
cudaError_t launch_gemm_w4a16(const uint16_t* x, int M, int K, const uint8_t* wq,
                              const uint8_t* wsz, const float* gw, int N, void* y, bool y_bf16,
                              uint8_t* workspace, cudaStream_t stream, const DevInfo& dev);

// The gate/up projection fused with the activation: W = [gate; up] stacked [2I, K] (one
// global scale gw, wsz its atom part), h = silu(bf16(x . gate^T)) * bf16(x . up^T) quantized
// to NVFP4 with the static global scale *gh in the GEMM's epilogue: codes hq [M, I/2], scale
// atoms hs (rows padded to 128 and blocks to 4, padding zero).  Taken when
// gemm_w4a16_silu_takes(M, I): M > 16 and I % 128 == 0.  err: the workspace error word.
bool gemm_w4a16_silu_takes(int64_t M, int64_t I, const DevInfo& dev);
cudaError_t launch_gemm_w4a16_silu(const uint16_t* x, int M, int K, const uint8_t* wq,
                                   const uint8_t* wsz, const float* gw, int I, const float* gh,
                                   uint8_t* hq, uint8_t* hs, uint8_t* workspace,
                                   cudaStream_t stream, const DevInfo& dev);

// M > 16 W4A4 GEMM (block-scaled tcgen05.mma, kind::mxf4nvf4).  xq [M, K/2] and xsz (scale
// atoms of x) and gx come from the quantizer; wsz: the atom part of W's repacked scales.
// y = *gx * *gw * deq(x) . deq(W)^T.  err: the workspace error word; sk_state: stream-K
// counters (zero before the first call) and partial-tile slots,
// gemm_w4a4_stream_k_bytes() of them.
size_t gemm_w4a4_stream_k_bytes(int64_t M, int64_t K, int64_t N);
// The same GEMM with x given as bf16 [M, K] and quantized inside the kernel: every CTA of
// the (cooperative, co-resident) grid quantizes a share of x into xq / xsz (the layout
// and bytes launch_quantize writes) and counts itself done in `sync`; the producers wait
// for the count to reach the grid before their first load of x.  With
// gx_static null the global scale is amax / 2688 of x: amax partials, then one grid-wide
// barrier.  gx_out receives g_x.  sync: gemm_w4a4_sync_bytes(M) bytes, zero before the
// first call and left zero by every completed call.
size_t gemm_w4a4_sync_bytes(int64_t M);
cudaError_t launch_gemm_w4a4_quant_x(const uint16_t* x, const float* gx_static, float* gx_out,
                                     float* partials, uint32_t* sync, uint8_t* xq, uint8_t* xsz,
                                     int M, int K, const uint8_t* wq, const uint8_t* wsz,
                                     const float* gw, int N, void* y, bool y_bf16, uint32_t* err,
                                     uint8_t* sk_state, cudaStream_t stream, const DevInfo& dev);
cudaError_t launch_gemm_w4a4(const uint8_t* xq, const uint8_t* xsz, const float* gx, int M,
                             int K, const uint8_t* wq, const uint8_t* wsz, const float* gw, int N,
                             void* y, bool y_bf16, uint32_t* err, uint8_t* sk_state,
                             cudaStream_t stream, const DevInfo& dev);

// True while the calling thread asks for the CTA-pair W4A4 GEMM at M > 16
// (nvfp4_debug_w4a4_kernel); by default the one-CTA kernel runs.
bool w4a4_use_pairs();
// True while the calling thread asks for the quantizer kernels ahead of the W4A4 kernels
// (at M > 16, and at M = 1 with a dynamic scale) instead of the kernels' own quantization
// of x (nvfp4_debug_w4a4_kernel).
bool w4a4_prepass_forced();

// Wait settings for the launches of the calling thread: the production limits, or (while
// nvfp4_debug_expire_waits is on) a 200 us limit and the stall switch.
WaitCfg current_wait_cfg();

// The current device's cached properties; NVFP4_ERR_DEVICE unless it is sm_103
// (the status is returned as an int holding an nvfp4_status).
int query_device(DevInfo* out);

}  // namespace nvfp4
