/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 block-scaled projection library.
 *
 * The hot path of batch-one Qwen3.x serving is the NVFP4 weight projection
 * y[M,N] = x[M,K] . W^T, run at decode (M = 1), MTP verify (M = K + 1 drafts) and on
 * prefill chunks (Qwen3x-Orin README, Functional evaluation quick start:
 * "--projection-backend sm87", "--prefill-chunk-size 512"; FlashRT
 * docs/qwen36_usage.md, generate_own_speculative_KN_nvfp4 argument table and the
 * per-step decode section).  The weights are NVFP4 ("compressed-tensors
 * nvfp4-pack-quantized", FlashRT constructor argument table): E2M1 codes packed
 * two per byte, one E4M3 scale per 16 consecutive K elements of a row, one FP32
 * global scale.  The format is named, not defined, on those pages; this library
 * uses its standard definition:
 *   value(n, k) = e2m1(q[n,k]) * e4m3(s[n, k/16]) * g,   g = amax / (6 * 448).
 *
 * Conventions shared by every call
 *   - All tensor arguments are device pointers into caller-owned memory of the
 *     current CUDA device; the library allocates nothing and keeps no state other
 *     than a per-device cache of the device's properties.
 *   - Every pointer argument must be 16-byte aligned, except `global_scale`,
 *     `w_global_scale` and `x_global_scale`, which need 4-byte alignment.
 *   - Work is enqueued on `stream` (NULL = the legacy default stream); no call
 *     synchronizes.  Calls on distinct streams are thread-safe.
 *   - Arguments are checked on the host before anything is enqueued; a failed
 *     check returns its status and enqueues nothing.  A CUDA launch error is
 *     returned as NVFP4_ERR_CUDA.
 *   - The device must be compute capability 10.3 (GB300, sm_103a); otherwise
 *     NVFP4_ERR_DEVICE.
 *   - Layouts: x [M,K] bf16 row-major; packed weights [N, K/2] bytes row-major,
 *     byte j of a row = code(2j) | code(2j+1) << 4; row-major scales [N, K/16]
 *     E4M3 bytes; y [M,N] row-major fp32 or bf16.
 *   - Workspace: a caller-owned device buffer of at least the size that
 *     nvfp4_workspace_bytes() returns.  Its first 4 bytes are a sticky error word:
 *     zero-fill the workspace once when it is allocated; kernels only OR error
 *     bits into it (never clear it), see nvfp4_workspace_error().
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvfp4_stream_t; /* the same handle as cudaStream_t */

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_NULL = 1,        /* a required pointer is NULL */
    NVFP4_ERR_SHAPE = 2,       /* a size is out of range or not a required multiple */
    NVFP4_ERR_ALIGN = 3,       /* a pointer is not aligned as required */
    NVFP4_ERR_DTYPE = 4,       /* unknown dtype or mode */
    NVFP4_ERR_WORKSPACE = 5,   /* workspace missing or too small */
    NVFP4_ERR_DEVICE = 6,      /* current device is not sm_103 */
    NVFP4_ERR_CUDA = 7,        /* a CUDA runtime call or launch failed */
    NVFP4_ERR_TIMEOUT = 8,     /* a device-side bounded wait ran out (error word) */
    NVFP4_ERR_UNSUPPORTED = 9  /* valid arguments, but no kernel for this case */
} nvfp4_status;

typedef enum { NVFP4_F32 = 0, NVFP4_BF16 = 1 } nvfp4_dtype;
typedef enum {
    NVFP4_W4A16 = 0,
    NVFP4_W4A4 = 1,
    /* Flag, OR-ed into the mode of nvfp4_linear: the caller promises that no kernel
     * enqueued earlier on the stream, and possibly still running, writes w_packed or
     * w_scales_swizzled (true of inference weights).  The decode kernels then start
     * streaming the weights before the previous kernel on the stream has finished. */
    NVFP4_STATIC_WEIGHTS = 0x10
} nvfp4_mode;

/* error-word bits (see nvfp4_workspace_error) */
#define NVFP4_DEVERR_TIMEOUT 0x1u

/*
 * nvfp4_quantize -- FP32/BF16 weights to NVFP4.
 *
 * Defines: the load-time weight conversion to NVFP4 (FlashRT docs/qwen36_usage.md,
 * constructor paragraph and env-var table FLASHRT_QWEN36_MTP_CKPT_DIR, FP8 -> BF16
 * -> NVFP4 at load).  Steps, all in fp32 round-to-nearest-even:
 *   1. amax = max |src|;  g = amax / 2688 (g = 1 when amax == 0).
 *   2. per row and 16-element block: bmax = max |src|;  s = E4M3(bmax / (6 g)),
 *      round to nearest even, saturating at 448.
 *   3. d = e4m3(s) * g; code = E2M1(src / d) (nearest of {0,.5,1,1.5,2,3,4,6},
 *      ties to the even code, |v| >= 6 -> 6, sign bit of the input kept);
 *      d == 0 gives a signed zero code.
 * Arguments:
 *   src          [rows, cols] row-major, dtype src_dtype (NVFP4_F32 or NVFP4_BF16);
 *                all values finite (non-finite input gives unspecified codes).
 *   rows, cols   rows >= 1, cols >= 16, cols % 16 == 0.
 *   packed       out [rows, cols/2] bytes.
 *   scales       out [rows, cols/16] E4M3 bytes, row-major (nvfp4_repack makes the
 *                kernel layout from it).
 *   global_scale out, one float g (device memory).
 *   workspace    >= nvfp4_workspace_bytes(0, rows, cols, 0, 0) bytes (amax
 *                partials; contents need not be initialised).
 * Two kernels are enqueued; the result is bit-exact with the CPU reference.
 */
nvfp4_status nvfp4_quantize(const void* src, nvfp4_dtype src_dtype, int64_t rows,
                            int64_t cols, uint8_t* packed, uint8_t* scales,
                            float* global_scale, void* workspace, size_t workspace_bytes,
                            nvfp4_stream_t stream);

/*
 * nvfp4_quantize_noalloc -- nvfp4_quantize for callers that cannot allocate.
 *
 * No counterpart on the pages: it exists for callers that may not allocate device
 * memory once they are running -- serving runtimes that plan every allocation at
 * start-up, code under a fixed memory budget with no scratch pool to lend, and
 * latency-critical paths where cudaMalloc/cudaFree would wait on the device.  It
 * computes exactly what nvfp4_quantize computes (same kernels, same results) but takes
 * no workspace: its scratch (one float per first-pass CTA, at most 2048 floats = 8 KiB)
 * is a fixed array in device memory owned by the library, which every GPU that loads
 * the library keeps until the process exits.  Arguments are those of nvfp4_quantize
 * without the workspace.
 *   - The first call in a CUDA context (the first on a device, and the first after a
 *     cudaDeviceReset or under another context made current) looks up the array's
 *     device address there (one cudaGetSymbolAddress) and caches it under that
 *     context's id; make that first call before any stream capture.  A reset unloads
 *     the library's device code, and the next call looks the address up again.
 *   - Every call on a device shares the one array and leaves its contents behind;
 *     nothing in it has to start at zero.  Calls whose kernels overlap on the GPU
 *     (on different streams, or from different threads) race on it: order them.
 *   - The first pass runs at most 2048 CTAs; a larger tensor is split over them (each
 *     strides over the whole input), exactly as nvfp4_quantize caps its own count.
 *   - It calls no allocating function (no cudaMalloc, no cudaFree).
 */
nvfp4_status nvfp4_quantize_noalloc(const void* src, nvfp4_dtype src_dtype, int64_t rows,
                                    int64_t cols, uint8_t* packed, uint8_t* scales,
                                    float* global_scale, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_fp8_block128 -- FP8 (E4M3, block-128 scaled) weights to NVFP4.
 *
 * Defines: the load-time conversion of an FP8 "e4m3 block-128" checkpoint (the MTP
 * head) through BF16 to NVFP4 (FlashRT docs/qwen36_usage.md, env-var table,
 * FLASHRT_QWEN36_MTP_CKPT_DIR).  The pages name the chain without its arithmetic;
 * the reading taken here is the common checkpoint convention:
 *   1. w[r][c] = e4m3(src[r][c]) * block_scales[r / 128][c / 128], one fp32
 *      round-to-nearest-even product (the scale multiplies: it is the inverse of the
 *      scale the checkpoint's quantizer divided by);
 *   2. w is rounded to bf16 (round to nearest even);
 *   3. the bf16 tensor is quantized exactly as nvfp4_quantize quantizes a
 *      NVFP4_BF16 source.
 * Arguments:
 *   src           [rows, cols] E4M3 (OCP "E4M3FN") bytes, row-major; NaN bytes (0x7F,
 *                 0xFF), non-finite scales or a product that overflows give
 *                 unspecified codes.
 *   block_scales  [ceil(rows / 128), ceil(cols / 128)] fp32, row-major (device).
 *   rows, cols    rows >= 1, cols >= 16, cols % 16 == 0 (a 16-element block never
 *                 straddles two 128-column tiles).
 *   packed, scales, global_scale, workspace: as for nvfp4_quantize (the same
 *                 workspace size, nvfp4_workspace_bytes(0, rows, cols, 0, 0)).
 *   src, packed, scales and workspace are 16-byte aligned; block_scales and
 *   global_scale 4-byte aligned.
 * Two kernels are enqueued (amax, then quantize); src is read twice and no bf16
 * copy is written.  The result is bit-exact with the CPU reference of steps 1-3.
 */
nvfp4_status nvfp4_quantize_fp8_block128(const uint8_t* src, const float* block_scales,
                                         int64_t rows, int64_t cols, uint8_t* packed,
                                         uint8_t* scales, float* global_scale,
                                         void* workspace, size_t workspace_bytes,
                                         nvfp4_stream_t stream);

/*
 * nvfp4_repack -- row-major E4M3 scales to the kernels' swizzled layout.
 *
 * Defines: the load-time "NVFP4 swizzle" (FlashRT docs/qwen36_usage.md, constructor
 * paragraph).  The buffer holds two copies of the scales:
 *   1. at byte 0, the tensor-core block-scale layout for 16-element blocks, read by the
 *      tensor-core kernels: rows padded to Rp = 128*ceil(rows/128) and blocks to
 *      Cp = 4*ceil(Cb/4) (Cb = cols/16) with zero bytes; element (r, cb) goes to byte
 *        ((r/128)*(Cp/4) + cb/4)*512 + (r%32)*16 + ((r%128)/32)*4 + cb%4;
 *   2. at byte A = Rp*Cp, the row-major scales [rows, Cb] unchanged, read by the
 *      small-M kernels (which stream a row's scales next to its codes), then zero
 *      bytes up to a multiple of 16 and 16 more.
 * Footprint: the second copy costs 1/16 byte per weight, as much as the first: with the
 * codes (1/2 byte per weight) a repacked weight takes 0.625 bytes per weight instead of
 * 0.5625, 11 % more (5.57 MB more for a 17408 x 5120 weight).  The small-M kernels need
 * the row-major copy: a CTA streams a contiguous slab of rows that does not start on a
 * 128-row block, and the atoms interleave four 32-row quarters in each 16-byte line.
 * Arguments:
 *   scales_rowmajor  [rows, cols/16] bytes.  rows >= 1, cols >= 16, cols % 16 == 0.
 *   scales_swizzled  out, exactly swizzled_bytes == nvfp4_repack_bytes(rows, cols).
 * The output must not overlap the input.
 */
nvfp4_status nvfp4_repack(const uint8_t* scales_rowmajor, int64_t rows, int64_t cols,
                          uint8_t* scales_swizzled, size_t swizzled_bytes,
                          nvfp4_stream_t stream);

/*
 * nvfp4_linear -- y[M,N] = x[M,K] . W^T with NVFP4 W.
 *
 * Defines: the NVFP4 projection at decode, MTP verify and prefill (Qwen3x-Orin
 * README, quick start; FlashRT docs/qwen36_usage.md, speculative and per-step decode
 * sections), including the fused gate/up shape with one shared global scale
 * (env-var table, FLASHRT_QWEN36_FUSE_MLP_GATE_UP) and NVFP4 activations
 * (FLASHRT_QWEN36_FUSE_SILU_MUL_QUANT).
 *   W4A16: y[m,n] = g_w * sum_b s[n,b] * sum_{k in b} x[m,k] * e2m1(q[n,k]).
 *   W4A4:  x is first quantized like nvfp4_quantize (global scale = its amax / 2688,
 *          or *x_global_scale when given) into the workspace; then
 *          y = g_x g_w * sum_b sx[m,b] sw[n,b] sum_{k in b} e2m1(qx) e2m1(qw).
 *          With a given x_global_scale and M <= 8, the M = 1 GEMV and the skinny GEMM
 *          quantize x themselves (same codes and scales, no pre-pass); x's codes are
 *          then not written to the workspace.  With a dynamic scale at M = 1 (K/32 >= 64)
 *          the GEMV also quantizes x itself: each CTA reduces x's amax over its own
 *          lanes, and the grid writes x's codes, scales and g_x to the workspace as the
 *          quantizer would.  At M > 16 the tensor-core GEMM quantizes
 *          x itself: its CTAs (one per SM, launched cooperatively so that all are
 *          resident) each quantize a share of x into the workspace -- after an amax
 *          pass and one grid-wide barrier when the scale is dynamic -- and count
 *          themselves done; the GEMM's loads of x wait for the count.  One kernel, the
 *          same bytes in the workspace.  Where the device cannot hold the whole grid at
 *          once, the call quantizes x in a kernel of its own first.
 * Accumulation is fp32.  Expected accuracy: |y - y_ref| <= 1e-3 * sum_k |x_k w_k|
 * + 2^-8 |y_ref| for bf16 y.
 * Arguments:
 *   x                  [M, K] bf16.  M >= 1, K >= 32, K % 32 == 0.
 *   w_packed           [N, K/2] bytes (nvfp4_quantize output).  N >= 1.
 *   w_scales_swizzled  nvfp4_repack_bytes(N, K) bytes (nvfp4_repack output).
 *   w_global_scale     one float (device).
 *   y                  out [M, N], dtype y_dtype (NVFP4_F32 or NVFP4_BF16).
 *   mode               NVFP4_W4A16 or NVFP4_W4A4, optionally | NVFP4_STATIC_WEIGHTS
 *                      (used by the M <= 8 kernels; the others ignore it).
 *   x_global_scale     W4A4 only: NULL = dynamic (amax of x), else one float
 *                      (device, finite, > 0).  Must be NULL for W4A16.
 *   workspace          >= nvfp4_workspace_bytes(1, M, K, N, mode) bytes (at least the
 *                      256-byte header holding the sticky error word), zero-filled once
 *                      at allocation.  Calls that share a workspace must be ordered (one
 *                      stream), since W4A4 keeps the quantized x there.  For M > 16 it
 *                      also holds the tensor-core GEMM's stream-K counters and, in
 *                      W4A4 mode, the counters of its in-kernel quantization (they must
 *                      be zero before the first call; every call that completes without
 *                      a device error leaves them zero) and fp32 partial tiles.  After a
 *                      device error (nvfp4_workspace_error != 0), zero-fill it again.
 * Kernels: M = 1 pipelined GEMV; 2 <= M <= 8 streamed skinny GEMM (mma.sync);
 * 9 <= M <= 16 the skinny GEMM with two token tiles in one pass over W where K fits its
 * warps and shared memory (else two skinny passes, tokens 0..7 and the rest, where one
 * tile fits, else an mma.sync GEMM reading W from global memory); M > 16 the tcgen05
 * GEMMs (W4A16: W dequantized to bf16 per tile; W4A4: block-scaled kind::mxf4nvf4).
 * Results are deterministic.
 */
nvfp4_status nvfp4_linear(const void* x, int64_t M, int64_t K, const uint8_t* w_packed,
                          const uint8_t* w_scales_swizzled, const float* w_global_scale,
                          int64_t N, void* y, nvfp4_dtype y_dtype, nvfp4_mode mode,
                          const float* x_global_scale, void* workspace,
                          size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_silu_mul_quantize -- NVFP4 activations of silu(gate) * up, fused.
 *
 * Defines: the activation step between the fused gate/up projection and the down
 * projection (FlashRT docs/qwen36_usage.md, env-var table: FLASHRT_QWEN36_FUSE_MLP_GATE_UP,
 * FLASHRT_QWEN36_FUSE_SILU_MUL_QUANT).  The pages name the fusion without its arithmetic;
 * the reading taken here:
 *   h[m][i] = (g / (1 + exp(-g))) * u,  g = gate_up[m][i], u = gate_up[m][I + i],
 * each step one fp32 round-to-nearest-even operation, with exp a fixed fp32 sequence
 * (Cody-Waite reduction, Taylor series to the 7th power; exp(x) = +inf above 88 and 0
 * below -87), so that the codes are reproducible bit for bit.  h stays in registers and
 * is quantized as nvfp4_quantize quantizes an fp32 source (with the given global scale
 * when there is one), the scales going straight to the tensor-core atom layout.
 * Arguments:
 *   gate_up         bf16 [M, 2I] row-major: gate in columns [0, I), up in [I, 2I).
 *   M, I            M >= 1, I >= 16, I % 16 == 0 (I % 32 == 0 to feed nvfp4_linear_nvfp4_x).
 *   packed          out [M, I/2] bytes.
 *   scales_swizzled out, the atom part of the nvfp4_repack layout for an [M, I] tensor:
 *                   ceil(M/128)*128 * ceil(I/64)*4 bytes (scales_bytes at least that);
 *                   padding rows and blocks are written as zero.
 *   global_scale    out, g (device); a copy of *given_global_scale when that is given.
 *   given_global_scale  NULL: g = amax|h| / 2688 (two kernels, h computed twice);
 *                   else a static activation scale (device, finite, > 0; one kernel).
 *   workspace       >= nvfp4_workspace_bytes(0, M, I, 0, 0) bytes when g is dynamic;
 *                   may be NULL with a given scale.
 * Alignment: gate_up, packed, scales_swizzled, workspace 16 bytes; the scales 4 bytes.
 * Non-finite gate/up values give unspecified codes.
 */
nvfp4_status nvfp4_silu_mul_quantize(const void* gate_up, int64_t M, int64_t I,
                                     uint8_t* packed, uint8_t* scales_swizzled,
                                     size_t scales_bytes, float* global_scale,
                                     const float* given_global_scale, void* workspace,
                                     size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_linear_nvfp4_x -- y = x . W^T with x already in NVFP4 (the down projection fed
 * by nvfp4_silu_mul_quantize).
 *
 *   y[m,n] = g_x * g_w * sum_k e2m1(qx[m,k]) e4m3(sx[m,k/16]) e2m1(qw[n,k]) e4m3(sw[n,k/16])
 * Arguments:
 *   x_packed           [M, K/2] codes; x_scales_swizzled the atom layout of an [M, K]
 *                      tensor (as nvfp4_silu_mul_quantize writes it); x_global_scale g_x
 *                      (device).
 *   w_*, N, y, y_dtype as for nvfp4_linear.
 *   flags              0 or NVFP4_STATIC_WEIGHTS.
 *   workspace          >= nvfp4_workspace_bytes(1, M, K, N, NVFP4_W4A4) bytes, first
 *                      4 bytes the error word.
 * M > 16 runs the block-scaled tensor-core GEMM on x's codes and scales directly;
 * M <= 16 writes x's exact bf16 value e2m1 * e4m3 into the workspace and runs the
 * small-M W4A16 kernels with g_x folded into the output scale.
 */
nvfp4_status nvfp4_linear_nvfp4_x(const uint8_t* x_packed, const uint8_t* x_scales_swizzled,
                                  const float* x_global_scale, int64_t M, int64_t K,
                                  const uint8_t* w_packed, const uint8_t* w_scales_swizzled,
                                  const float* w_global_scale, int64_t N, void* y,
                                  nvfp4_dtype y_dtype, int flags, void* workspace,
                                  size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_linear_silu_mul_quantize -- the MLP's gate/up projection with its activation
 * quantized to NVFP4 in the same pass (the epilogue of the gate/up GEMM).
 *
 * Defines: FlashRT docs/qwen36_usage.md, env-var table: FLASHRT_QWEN36_FUSE_MLP_GATE_UP
 * (gate and up as one NVFP4 GEMM, for checkpoints whose gate and up share their scales)
 * followed by FLASHRT_QWEN36_FUSE_SILU_MUL_QUANT (silu(gate) * up quantized to NVFP4 for
 * the down projection).  With gu = the bf16 output of the gate/up projection,
 *   gu = bf16(x . W^T)  [M, 2I], gate in columns [0, I), up in [I, 2I)
 * (each output rounded to bf16 once, as nvfp4_linear with a bf16 y rounds it), the call
 * writes h = silu(gate) * up quantized with the static global scale *h_global_scale --
 * exactly what nvfp4_silu_mul_quantize(gu, ..., given_global_scale = h_global_scale)
 * writes -- without writing gu to memory.
 * Arguments:
 *   x                 bf16 [M, K] row-major; M >= 1, K >= 32, K % 32 == 0.
 *   w_packed, w_scales_swizzled, w_global_scale: the stacked weight [gate; up] of 2I rows
 *                     and K columns with one global scale, as nvfp4_quantize and
 *                     nvfp4_repack produce it.
 *   I                 columns of h: I >= 16, I % 16 == 0 (I % 32 == 0 to feed
 *                     nvfp4_linear_nvfp4_x).
 *   h_global_scale    the static global scale of h (device float, finite, > 0); the down
 *                     projection takes the same pointer as its x_global_scale.
 *   h_packed          out [M, I/2] codes.
 *   h_scales_swizzled out, the tensor-core scale atoms of an [M, I] tensor (padding rows
 *                     and blocks written as zero); h_scales_bytes at least
 *                     ceil(M/128)*128 * ceil(I/64)*4.
 *   flags             0 or NVFP4_STATIC_WEIGHTS (as for nvfp4_linear).
 *   workspace         >= nvfp4_workspace_bytes(2, M, K, I, 0) bytes; first 4 bytes the
 *                     error word, then (fused path) the stream-K counters and partial
 *                     tiles of the GEMM's last partial wave, or (other shapes) the
 *                     linear's workspace and gu; zeroed once when allocated (the kernels
 *                     leave the counters at zero).
 * Alignment: x, the weights, h_packed, h_scales_swizzled, workspace 16 bytes; the global
 * scales 4 bytes.
 * Dispatch: M > 16 with I % 128 == 0 runs one tcgen05 GEMM whose tiles pair 64 gate rows
 * with the 64 matching up rows; its epilogue rounds both to bf16, forms h and quantizes it
 * (nothing but the codes and scales reaches memory).  The tiles of its last partial wave
 * are split over K across CTAs (stream-K): their fp32 partials go to the workspace and
 * the CTA that completes a tile adds them in a fixed order before the activation.  Other shapes write gu into the
 * workspace with nvfp4_linear's kernels and quantize it with nvfp4_silu_mul_quantize's.
 */
nvfp4_status nvfp4_linear_silu_mul_quantize(const void* x, int64_t M, int64_t K,
                                            const uint8_t* w_packed,
                                            const uint8_t* w_scales_swizzled,
                                            const float* w_global_scale, int64_t I,
                                            const float* h_global_scale, uint8_t* h_packed,
                                            uint8_t* h_scales_swizzled, size_t h_scales_bytes,
                                            int flags, void* workspace, size_t workspace_bytes,
                                            nvfp4_stream_t stream);

/* ---- host-only helpers: no device work ---------------------------------------- */

/* Bytes of the swizzled scale layout for a [rows, cols] tensor (0 on bad sizes). */
size_t nvfp4_repack_bytes(int64_t rows, int64_t cols);

/* Workspace bytes: op 0 = nvfp4_quantize(rows=M, cols=K), op 1 = nvfp4_linear(M, K,
 * N, mode), op 2 = nvfp4_linear_silu_mul_quantize(M, K, I = N; mode ignored).  0 when no
 * workspace is needed; (size_t)-1 on bad arguments. */
size_t nvfp4_workspace_bytes(int op, int64_t M, int64_t K, int64_t N, nvfp4_mode mode);

/* Where nvfp4_linear in W4A4 mode leaves the quantized activations inside its
 * workspace: packed codes [M, K/2] at *xq_offset, the scales in the tensor-core
 * layout (part 1 of nvfp4_repack's layout, Rp*Cp bytes) at *xs_offset and g_x (one
 * float) at *gx_offset.  They are valid once the call has completed, except after a
 * call with a given x_global_scale and M <= 8, where the small-M kernel may have
 * quantized x itself and left these areas untouched.  Returns NVFP4_OK or
 * NVFP4_ERR_SHAPE. */
nvfp4_status nvfp4_w4a4_workspace_layout(int64_t M, int64_t K, size_t* xq_offset,
                                         size_t* xs_offset, size_t* gx_offset);

/* Reads (and then clears) the sticky error word of a workspace after `stream` has
 * drained: synchronizes `stream`.  *bits gets NVFP4_DEVERR_* bits; returns
 * NVFP4_ERR_TIMEOUT if any bit was set, NVFP4_OK otherwise. */
nvfp4_status nvfp4_workspace_error(void* workspace, nvfp4_stream_t stream, uint32_t* bits);

/* Human-readable name of a status. */
const char* nvfp4_status_str(nvfp4_status status);

/* ---- diagnostics -------------------------------------------------------------- */

/* The CUDA error behind the last NVFP4_ERR_CUDA this thread got from the library
 * (cudaGetErrorString text; "no error" if there was none).  Host-only. */
const char* nvfp4_last_cuda_error(void);

/* Test switch for the failure path of the bounded device waits; never on in production.
 * While on (for calls from the calling thread), the pipelined M = 1 GEMV and the
 * tensor-core GEMMs of nvfp4_linear launch with a 200 us wait limit and one role
 * withholding an arrival: the GEMV's consumers never release a stage, the W4A16 GEMM's
 * dequantizing warps never mark a stage ready, the W4A4 GEMM's first CTA never counts its
 * share of the in-kernel quantized x.  A wait then runs out; the kernel sets
 * NVFP4_DEVERR_TIMEOUT in the workspace error word, every role stops, the copies and MMAs
 * it issued are waited for, its TMEM is freed, and it returns (y is not written in full).
 * The CUDA context stays usable: zero-fill the workspace and call again.  Host-only; the
 * switch is per thread. */
void nvfp4_debug_expire_waits(int on);

/* Test switch; never set in production.  Chooses, for calls from the calling thread, the
 * kernel of the W4A4 GEMM at M > 16 (nvfp4_linear in W4A4 mode, nvfp4_linear_nvfp4_x):
 * 0 or 1 the one-CTA tensor-core kernel (the default, the faster on this hardware); 2 CTA
 * pairs on two SMs (tcgen05 cta_group::2, 256 x 256 tiles; a device that cannot co-schedule
 * CTA pairs runs the one-CTA kernel); 3 the one-CTA kernel with bf16 x quantized by the
 * quantizer kernels ahead of it rather than inside its grid (the path of a device that
 * refuses the GEMM's cooperative launch; the same bits), and, at M = 1 with a dynamic
 * scale, the same quantizer kernels ahead of the GEMV (the same bits).  Both satisfy the same tolerance; their stream-K
 * splits differ, so outputs can differ in the last bits where a tile's K steps are summed
 * in different groups.  Host-only; the switch is per thread. */
void nvfp4_debug_w4a4_kernel(int which);

/*
 * nvfp4_encode_elements -- the device's element rounding on its own: for each of n
 * fp32 inputs, e2m1_out[i] = E2M1 code (as nvfp4_quantize step 3 rounds src/d) and
 * e4m3_out[i] = E4M3 byte of max(in[i], 0) (as step 2 rounds a block scale).  It runs
 * the same device functions the quantizer uses, so that their rounding can be
 * checked over every fp32 bit pattern.  Either output may be NULL.  n >= 0.
 */
nvfp4_status nvfp4_encode_elements(const float* in, int64_t n, uint8_t* e2m1_out,
                                   uint8_t* e4m3_out, nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H_ */
