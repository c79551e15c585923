// gemv.cu -- W4A16 NVFP4 GEMV (M = 1) and the small-M GEMM (2 <= M <= 16) fallback: the
// decode and MTP-verify projections.  Qwen3x-Orin README (quick start, "--projection-backend
// sm87"): decode streams every weight once per token; FlashRT docs/qwen36_usage.md
// (generate_own_speculative_KN_nvfp4 argument table): verify runs K + 1 rows against
// the same weights.
//
//   y[m, n] = gw * (gx ? gx : 1) * sum_b s[n, b] * sum_{k in b} x[m, k] * e2m1(q[n, k])
//
// Bound by HBM (0.5625 bytes of weight per multiply-add at M = 1) and by the issue rate
// of the dequantization, so the work per weight is kept small:
//   - E2M1 -> fp16 with the hardware converter (cvt.rn.f16x2.e2m1x2: one instruction
//     per two codes, exact);
//   - x is carried as fp16 after a power-of-two rescale that puts the largest magnitude
//     of the slice a lane (or warp) holds in [2^14, 2^15): every bf16 value within 2^31 of
//     that maximum is exact in fp16.  Should any value not be exact, an exact fp32
//     residual pass is added, so the result never depends on the rescale;
//   - fp32 mixed-precision FMAs (fma.rn.f32.f16, one per weight), the 16-block scale
//     applied once per block in fp32.
// Kernels in this file:
//   - gemv_m1_pipe_kernel (M = 1, the decode path): one CTA per SM owns a contiguous slab
//     of rows; a producer thread streams whole-row stages (codes and row-major scales, two
//     bulk copies each, behind full/empty mbarriers) into a shared-memory ring, the first
//     stage short so that it lands early; consumer warps each own a fixed group of 16-byte
//     chunks of K and keep their x in registers for the whole kernel; the lanes of a row
//     reduce by shuffles into per-(row, warp) slots that are added in a fixed order.
//     Launched as a programmatic dependent; every wait is bounded.  Its kXQ instantiation
//     is W4A4 at M = 1: each lane quantizes the x blocks it holds (a given g_x, or one
//     from x's amax reduced by every CTA, in which case the grid also writes x's codes,
//     scale atoms and g_x to the workspace, as the quantizer would) and multiplies by
//     the quantized values.
//   - gemv_m1_kernel: M = 1 where K is outside the pipelined kernel's range (K / 32 < 64
//     or > 992):
//     a grid of 2 x SMs CTAs of 8 warps, (row, K segment) units split evenly over the
//     warps, x staged in shared memory per K chunk.
//   - gemv_mma_kernel (2 <= M <= 16 where the skinny kernel does not take the K): mma.sync
//     m16n8k16 with 16 weight rows as A (block scale folded in: e2m1 * e4m3 is exact in
//     fp16) and up to 16 tokens of x as B; W read from global memory.
// All splits are deterministic (no atomics on results).
#include <cuda_fp16.h>

#include <atomic>

#include "../../include/nvfp4.h"
#include "common.cuh"
#include "gemv_helpers.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kXSmemBytes = 64 * 1024;     // fp16 x staging per CTA and K chunk, M = 1
constexpr int kXSmemBytesMma = 88 * 1024;  // the same for the mma path (K = 5120 at M <= 8)

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) r = fmaxf(r, red[i]);
    return r;
}


// ======================================================================================
// M = 1
// ======================================================================================
// smem: x' pieces [4][pitch] x 16 B (piece (q, c) = elements 32c + 8q .. +8 of the K
// chunk), then slots [rows][kWarps] floats.
constexpr int kM1Units = 8;  // 16-byte weight loads in flight per lane

__global__ void __launch_bounds__(kThreads)
gemv_m1_kernel(const uint16_t* __restrict__ x, int K, const uint8_t* __restrict__ wq,
               const uint8_t* __restrict__ wsz, const float* __restrict__ gw,
               const float* __restrict__ gx, int N, void* __restrict__ y, int y_bf16,
               int kc_max) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int pitch = kc_max >> 5;
    uint4* xs = reinterpret_cast<uint4*>(smem);
    float* slots = reinterpret_cast<float*>(smem + (size_t)4 * pitch * 16);
    __shared__ float red[kWarps];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = (int64_t)N * blockIdx.x / gridDim.x;
    const int64_t r1 = (int64_t)N * (blockIdx.x + 1) / gridDim.x;
    const int nrows = (int)(r1 - r0);
    const int64_t row_bytes = K >> 1;
    for (int i = threadIdx.x; i < nrows * kWarps; i += kThreads) slots[i] = 0.0f;

    for (int kc0 = 0; kc0 < K; kc0 += kc_max) {
        const int kl = min(kc_max, K - kc0);
        const int nch = kl >> 5;
        // ---- stage x' = x * 2^e as fp16 (e from this chunk's amax) ----
        float am = 0.0f;
        const uint32_t* xw = reinterpret_cast<const uint32_t*>(x + kc0);
        for (int i = threadIdx.x; i < (kl >> 1); i += kThreads) {
            const uint32_t v = xw[i];
            am = fmaxf(am, fmaxf(fabsf(bf16_to_f32(v & 0xFFFFu)), fabsf(bf16_to_f32(v >> 16))));
        }
        const int e = chunk_exponent(block_max(am, red));
        bool inexact = false;
        for (int p = threadIdx.x; p < 4 * nch; p += kThreads) {
            const int c = p >> 2, q = p & 3;
            const uint4 v = *reinterpret_cast<const uint4*>(x + kc0 + 32 * c + 8 * q);
            uint4 h;
            h.x = to_h2_scaled(v.x, e, inexact);
            h.y = to_h2_scaled(v.y, e, inexact);
            h.z = to_h2_scaled(v.z, e, inexact);
            h.w = to_h2_scaled(v.w, e, inexact);
            xs[q * pitch + c] = h;
        }
        const bool any_inexact = __syncthreads_or(inexact);

        // ---- (row, 32-chunk segment) units, split evenly over the warps ----
        const int nseg = (nch + 31) >> 5;
        const int units = nrows * nseg;
        const int u0 = (int)((int64_t)units * warp / kWarps);
        const int u1 = (int)((int64_t)units * (warp + 1) / kWarps);
        int row = u0 / nseg, seg = u0 - row * nseg;  // of the next unit to load
        int cur = -1;                                 // row being accumulated
        float acc = 0.0f;
        for (int u = u0; u < u1; u += kM1Units) {
            uint4 wv[kM1Units];
            uint32_t sv[kM1Units];
            int urow[kM1Units], uc[kM1Units];
            bool valid[kM1Units];
#pragma unroll
            for (int i = 0; i < kM1Units; ++i) {
                const int c = seg * 32 + lane;
                uc[i] = c;
                urow[i] = (u + i < u1) ? row : -1;
                valid[i] = (u + i < u1) && (c < nch);
                if (valid[i]) {
                    const int64_t r = r0 + row;
                    wv[i] = ld_stream_u4(wq + r * row_bytes + (kc0 >> 1) + 16 * (int64_t)c);
                    sv[i] = ld_nc_u16(wsz + r * (K >> 4) + (kc0 >> 4) + 2 * c);
                } else {
                    wv[i] = make_uint4(0u, 0u, 0u, 0u);
                    sv[i] = 0u;
                }
                if (++seg == nseg) { seg = 0; ++row; }
            }
#pragma unroll
            for (int i = 0; i < kM1Units; ++i) {
                if (urow[i] < 0) break;
                if (urow[i] != cur) {
                    if (cur >= 0) {
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                        if (lane == 0) slots[cur * kWarps + warp] += ldexpf(acc, -e);
                        acc = 0.0f;
                    }
                    cur = urow[i];
                }
                if (!valid[i]) continue;
                const int c = uc[i];
                const uint32_t w[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
                float p[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t h[4];
                    cvt8(w[j], h);
                    const uint4 xv = xs[j * pitch + c];
                    const int b = (j >> 1) * 2;
                    mfma2(p[b], p[b + 1], h[0], xv.x);
                    mfma2(p[b], p[b + 1], h[1], xv.y);
                    mfma2(p[b], p[b + 1], h[2], xv.z);
                    mfma2(p[b], p[b + 1], h[3], xv.w);
                }
                float s0 = e4m3_to_f32(sv[i] & 0xFFu), s1 = e4m3_to_f32(sv[i] >> 8);
                if (any_inexact) {
                    // exact residual of this chunk's x (slow path, rare)
                    float q0 = 0.0f, q1 = 0.0f;
                    const uint16_t* xr = x + kc0 + 32 * c;
#pragma unroll 4
                    for (int k = 0; k < 32; ++k) {
                        const uint32_t wk = k < 16 ? (k < 8 ? w[0] : w[1]) : (k < 24 ? w[2] : w[3]);
                        const uint32_t code = (wk >> (4 * (k & 7))) & 15u;
                        const float r = residual(xr[k], e) * e2m1_to_f32(code);
                        if (k < 16) q0 += r; else q1 += r;
                    }
                    acc = fmaf(s0, q0, fmaf(s1, q1, acc));
                }
                acc = fmaf(s0, p[0] + p[1], fmaf(s1, p[2] + p[3], acc));
            }
        }
        if (cur >= 0) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) slots[cur * kWarps + warp] += ldexpf(acc, -e);
        }
        __syncthreads();
    }
    const float scale = *gw * (gx ? *gx : 1.0f);
    for (int i = threadIdx.x; i < nrows; i += kThreads) {
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += slots[i * kWarps + w];
        store_y(y, r0 + i, v * scale, y_bf16);
    }
}


// ======================================================================================
// M = 1, pipelined and x-stationary
// ======================================================================================
// One CTA per SM.  The CTA's rows [r0, r1) are one contiguous slab of packed weights and,
// in the row-major part of the repacked scales, one contiguous run of scale bytes.
// Column layout: a row has C = K/32 chunks of 16 bytes (32 codes); consumer warp w owns
// the column group of chunks [w G, w G + G) and each lane one chunk of it, for the whole
// kernel, so it loads its 32 values of x once, into registers (fp16 after the rescale
// below); the G lanes of a chunk group and the 32/G rows of a step share a warp.
// Producer warp (one thread): fills a ring of `stages` stages of `rps` whole rows from the
// kernel's first instruction; a stage = the rows' packed codes and their scale bytes, two
// bulk copies gated by per-stage mbarriers (full: transaction count; empty: one arrival
// per consumer warp).  Consumers: per stage, per step, lane (row t*L + l/G, chunk
// wG + l%G) reads its 16-byte chunk and 2 scale bytes from shared memory, computes the
// 32-term dot with its registers, and the G lanes of each row reduce into the warp's slot
// for that row.  Shared memory carries only codes and scales in the main loop.  Every wait
// is bounded; on time-out the kernel sets NVFP4_DEVERR_TIMEOUT in the error word, stops,
// and lets the copies it issued land before it exits.
constexpr int kPipeMaxThreads = 1024;
constexpr int kPipeStageTarget = 80 * 1024;  // bytes of codes per stage (whole rows)
constexpr int kPipeFirstStage = 16 * 1024;   // bytes of codes of the first, short stage
constexpr int kLeanUnroll = 2;  // unroll of the predicate-free step loop

// exact x * 2^e for a bf16 value (two multiplies keep 2^e representable for any e)
__device__ __forceinline__ float pow2_scale(float v, float f1, float f2) { return v * f1 * f2; }

__host__ __device__ __forceinline__ size_t pipe_stage_bytes(int K, int rps) {
    return (((size_t)rps * (K / 2) + (size_t)rps * (K / 16) + 32) + 127) & ~(size_t)127;
}

__host__ __device__ __forceinline__ size_t pipe_slot_bytes(int rows_max, int ngroups) {
    return ((size_t)rows_max * ngroups * 4 + 15) & ~(size_t)15;
}

// Each CTA releases the next launch on the stream (programmatic dependent launch) once its
// producer has issued its last copy, so the next kernel's prologue overlaps this one's tail.
// W4A4 (kXQ): x is quantized in the kernel with g_x = *gx, or, where gx is null, with the
// g_x of x's own amax (the quantizer's rule): the CTA's consumer lanes hold all of x
// between them, so every CTA reduces the amax itself, and CTA 0 also writes x's NVFP4
// encoding (codes, scale atoms with zero padding, g_x) to xq_out / xs_out / gx_out, as the
// quantizer kernels would.
template <int G, bool kXQ>
__global__ void __launch_bounds__(kPipeMaxThreads, 1)
gemv_m1_pipe_kernel(const uint16_t* __restrict__ x, int K, const uint8_t* __restrict__ wq,
                    const uint8_t* __restrict__ wrm, const float* __restrict__ gw,
                    const float* __restrict__ gx, int N, void* __restrict__ y, int y_bf16,
                    int rows_max, int rps, int rfirst, int stages, int w_static,
                    uint32_t* __restrict__ err, WaitCfg dbg, uint8_t* __restrict__ xq_out,
                    uint8_t* __restrict__ xs_out, float* __restrict__ gx_out) {
    constexpr int L = 32 / G;              // rows per step
    extern __shared__ __align__(128) uint8_t smem[];
    const int rowchunks = K >> 5;          // 16-byte chunks per row
    const int ngroups = (rowchunks + G - 1) / G;   // = number of consumer warps
    const int nthreads_c = ngroups * 32;
    const size_t sbytes_stage = pipe_stage_bytes(K, rps);
    uint8_t* ring = smem;
    float* slots = reinterpret_cast<float*>(smem + (size_t)stages * sbytes_stage);  // [rows][ngroups]
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(slots) +
                                                 pipe_slot_bytes(rows_max, ngroups));
    uint64_t* full = bars;
    uint64_t* empty = bars + stages;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = (int64_t)N * blockIdx.x / gridDim.x;
    const int64_t r1 = (int64_t)N * (blockIdx.x + 1) / gridDim.x;
    const int nrows = (int)(r1 - r0);
    // stage 0 holds the first rfirst rows (a short stage that lands early, so that the
    // consumers start as soon as x is in registers), every later stage rps rows
    const int nst = nrows <= rfirst ? 1 : 1 + (nrows - rfirst + rps - 1) / rps;
    auto stage_beg = [&](int it) { return it == 0 ? 0 : rfirst + (it - 1) * rps; };
    auto stage_rows = [&](int it) {
        return min(it == 0 ? rfirst : rps, nrows - stage_beg(it));
    };
    const int64_t rowb = K >> 1, rows_sb = K >> 4;  // code and scale bytes per row

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], ngroups);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == ngroups) {
        // ---- producer ----
        if (lane == 0) {
            // Unless the weights are static (no kernel still in flight writes them), the
            // first ring's worth of codes only heads for L2 while the previous kernel on the
            // stream may still run (a prefetch cannot observe stale data: L2 is the point of
            // coherence), and every read that lands in shared memory comes after the wait.
            // x heads for L2 too (16-byte aligned, K * 2 bytes: a multiple of 64), so that the
            // consumers' loads of it after the wait hit L2 rather than queue behind the
            // weight stream in HBM; weight copies are marked evict-first for the same reason
            if (blockIdx.x == 0) prefetch_l2(x, (uint32_t)K * 2u);  // once for the grid
            if (!w_static) {
                for (int it = 0; it < min(nst, stages); ++it)
                    prefetch_l2(wq + (r0 + (int64_t)stage_beg(it)) * rowb,
                                (uint32_t)(stage_rows(it) * rowb));
                pdl_wait_prior_grid();
            }
            const uint64_t pol = l2_evict_first_policy();
            int issued = 0;
            for (int it = 0; it < nst; ++it) {
                const int s = it % stages;
                if (it >= stages &&
                    !mbar_wait_bounded(&empty[s], ((it / stages) - 1) & 1, dbg.wait_ns)) {
                    if (err) atomicOr(err, NVFP4_DEVERR_TIMEOUT);
                    abort_flag = 1;
                    break;
                }
                if (abort_flag) break;
                const int nr = stage_rows(it);
                const int64_t rbeg = r0 + (int64_t)stage_beg(it);
                const uint32_t wbytes = (uint32_t)(nr * rowb);
                // scale bytes of these rows, copied from a 16-byte boundary
                const int64_t s_lo = (rbeg * rows_sb) & ~(int64_t)15;
                const int64_t s_hi = ((rbeg + nr) * rows_sb + 15) & ~(int64_t)15;
                mbar_arrive_expect_tx(&full[s], wbytes + (uint32_t)(s_hi - s_lo));
                uint8_t* st = ring + (size_t)s * sbytes_stage;
                bulk_g2s_hint(st, wq + rbeg * rowb, wbytes, &full[s], pol);
                bulk_g2s_hint(st + (size_t)rps * rowb, wrm + s_lo, (uint32_t)(s_hi - s_lo),
                              &full[s], pol);
                issued = it + 1;
            }
            // every copy of this CTA is in flight: the next kernel on the stream may now
            // be scheduled (its CTAs overlap only this kernel's tail)
            pdl_launch_dependents();
            // every copy this thread issued has landed before the CTA can exit
            for (int it = max(0, issued - stages); it < issued; ++it)
                mbar_wait_bounded(&full[it % stages], (it / stages) & 1, kWaitLimitNs);
        }
        return;
    }

    // ---- consumers: this lane's 32 values of x in registers, fp16 after the lane's own
    // power-of-two rescale ----
    // A lane keeps one 32-element chunk of x for the whole kernel, so it scales the chunk
    // by its own 2^e (largest magnitude in [2^14, 2^15)) and each partial dot product back
    // by 2^-e before the row's lanes are added: no reduction over the CTA, no barrier.  A
    // bf16 value is exact in fp16 after the rescale from 2^-17 upward; a warp with any lane
    // whose smallest nonzero value falls below that takes the exact residual path.
    pdl_wait_prior_grid();
    const int c = warp * G + (lane % G);   // this lane's chunk (column), fixed
    const int rsub = lane / G;             // its row within a step
    const bool cvalid = c < rowchunks;
    uint4 xv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        xv[q] = cvalid ? *reinterpret_cast<const uint4*>(x + 32 * c + 8 * q)
                       : make_uint4(0u, 0u, 0u, 0u);
    float gq = 1.0f;  // g_x (kXQ)
    if constexpr (kXQ) {
        if (gx) {
            gq = *gx;
            quantize_chunk_static(xv, gq);
        } else {
            // dynamic g_x: the amax of all of x over the CTA's consumer warps
            __shared__ float x_amax[kPipeMaxThreads / 32];
            float am = 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t w4[4] = {xv[q].x, xv[q].y, xv[q].z, xv[q].w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    am = fmaxf(am, fmaxf(fabsf(bf16_to_f32(w4[j] & 0xFFFFu)),
                                         fabsf(bf16_to_f32(w4[j] >> 16))));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
            if (lane == 0) x_amax[warp] = am;
            named_bar_sync(2, nthreads_c);
            float a = 0.0f;
            for (int w = 0; w < ngroups; ++w) a = fmaxf(a, x_amax[w]);
            gq = global_scale_from_amax(a);
            uint32_t codes[4], s2;
            quantize_chunk_codes(xv, gq, codes, s2);
            // x's encoding, spread over the grid.  With one row, scale atom a (512 bytes)
            // holds row 0's scales of blocks 4a .. 4a + 3 in its first 4 bytes and zeros in
            // the padding rows: the lane of chunk c = 2a (blocks 4a, 4a + 1) takes the scales
            // and codes of chunk c + 1 from the next lane, and CTA a % grid writes the atom
            // and both chunks' codes
            const uint32_t s2_next = __shfl_down_sync(0xffffffffu, s2, 1);
            uint32_t codes_next[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) codes_next[q] = __shfl_down_sync(0xffffffffu, codes[q], 1);
            if (rsub == 0 && (c & 1) == 0 && c < rowchunks &&
                (unsigned)(c >> 1) % gridDim.x == blockIdx.x) {
                uint4* atom = reinterpret_cast<uint4*>(xs_out + (size_t)(c >> 1) * 512);
                atom[0] = make_uint4(s2 | (s2_next << 16), 0u, 0u, 0u);
#pragma unroll 4
                for (int i = 1; i < 32; ++i) atom[i] = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(xq_out + 16 * c) =
                    make_uint4(codes[0], codes[1], codes[2], codes[3]);
                if (c + 1 < rowchunks)
                    *reinterpret_cast<uint4*>(xq_out + 16 * (c + 1)) =
                        make_uint4(codes_next[0], codes_next[1], codes_next[2], codes_next[3]);
            }
            if (blockIdx.x == 0 && threadIdx.x == 0) *gx_out = gq;
        }
    }
    float am = 0.0f, mn = __int_as_float(0x7f800000);  // max, smallest nonzero
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t w4[4] = {xv[q].x, xv[q].y, xv[q].z, xv[q].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = fabsf(bf16_to_f32(w4[j] & 0xFFFFu)), b = fabsf(bf16_to_f32(w4[j] >> 16));
            am = fmaxf(am, fmaxf(a, b));
            if (a > 0.0f) mn = fminf(mn, a);
            if (b > 0.0f) mn = fminf(mn, b);
        }
    }
    const int e = chunk_exponent(am);
    const int e1 = e / 2, e2 = e - e / 2;
    const float f1 = __int_as_float((e1 + 127) << 23), f2 = __int_as_float((e2 + 127) << 23);
    const float u1 = __int_as_float((127 - e1) << 23), u2 = __int_as_float((127 - e2) << 23);
    // (e2m1 * e4m3 values span less than 2^22: never inexact after the rescale)
    const bool inexact = !kXQ && pow2_scale(mn, f1, f2) < 7.62939453125e-06f;
    const bool any_inexact = __any_sync(0xffffffffu, inexact);  // this warp's lanes
    uint32_t xh[16];                       // x'[32c .. 32c+32) as 16 fp16 pairs
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t w4[4] = {xv[q].x, xv[q].y, xv[q].z, xv[q].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = pow2_scale(bf16_to_f32(w4[j] & 0xFFFFu), f1, f2);
            const float b = pow2_scale(bf16_to_f32(w4[j] >> 16), f1, f2);
            const __half2 hh = __floats2half2_rn(a, b);
            xh[q * 4 + j] = *reinterpret_cast<const uint32_t*>(&hh);
        }
    }
    const bool lean = !any_inexact && ngroups * G == rowchunks;

    for (int it = 0; it < nst; ++it) {
        const int s = it % stages;
        // the wait's outcome and the abort flag are made warp-uniform before they steer
        // control flow: the reductions below are warp-collective
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (it / stages) & 1,
                                                                  dbg.wait_ns));
        if (!ok) {
            if (err && lane == 0) atomicOr(err, NVFP4_DEVERR_TIMEOUT);
            abort_flag = 1;
        }
        if (__any_sync(0xffffffffu, abort_flag != 0)) break;
        const uint8_t* st = ring + (size_t)s * sbytes_stage;
        const int nr = stage_rows(it);
        const int sbeg = stage_beg(it);
        const int64_t rbeg = r0 + (int64_t)sbeg;
        const uint8_t* sst = st + (size_t)rps * rowb + ((rbeg * rows_sb) & 15);
        // whole steps of L rows with every lane on a real chunk and no residual pass run
        // without predicates; the rest of a short last stage takes the predicated loop
        const int lean_rows = lean ? nr / L * L : 0;
        if (lean_rows > 0) {
            const uint8_t* wp = st + ((size_t)rsub * rowchunks + c) * 16;
            const uint8_t* sp = sst + (size_t)rsub * rows_sb + 2 * c;
            float* sl = slots + (size_t)(sbeg + rsub) * ngroups + warp;
            const int wstep = L * rowchunks * 16, sstep = L * rows_sb, slstep = L * ngroups;
            const int nsteps = lean_rows / L;
#pragma unroll kLeanUnroll
            for (int t = 0; t < nsteps; ++t) {
                const uint4 wv = *reinterpret_cast<const uint4*>(wp);
                const uint32_t s01 = *reinterpret_cast<const uint16_t*>(sp);
                const uint32_t s16 = cvt_e4m3x2_f16x2(s01);  // both block scales, exact
                const float2 sc = __half22float2(*reinterpret_cast<const __half2*>(&s16));
                const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
                float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t hh[4];
                    cvt8(w[j], hh);
                    const int b = (j >> 1) * 2;
                    mfma2(a[b], a[b + 1], hh[0], xh[4 * j + 0]);
                    mfma2(a[b], a[b + 1], hh[1], xh[4 * j + 1]);
                    mfma2(a[b], a[b + 1], hh[2], xh[4 * j + 2]);
                    mfma2(a[b], a[b + 1], hh[3], xh[4 * j + 3]);
                }
                float pv = fmaf(sc.x, a[0] + a[1], sc.y * (a[2] + a[3])) * u1 * u2;
#pragma unroll
                for (int o = G / 2; o > 0; o >>= 1) pv += __shfl_xor_sync(0xffffffffu, pv, o);
                // the butterfly leaves the same sum in all G lanes of the row (each pairwise
                // add is commutative), so every lane stores it: no predicate in the loop
                *sl = pv;
                wp += wstep;
                sp += sstep;
                sl += slstep;
            }
            if (lean_rows == nr) {
                __syncwarp();
                if (lane == 0 && !dbg.stall) mbar_arrive(&empty[s]);
                continue;
            }
        }
        for (int t = lean_rows; t < nr; t += L) {
            const int rl = t + rsub;       // row within the stage
            float pv = 0.0f;
            if (cvalid && rl < nr) {
                const uint4 wv = *reinterpret_cast<const uint4*>(st + ((size_t)rl * rowchunks + c) * 16);
                const uint32_t s01 = *reinterpret_cast<const uint16_t*>(sst + (size_t)rl * rows_sb + 2 * c);
                const float s0 = e4m3_to_f32(s01 & 0x7Fu), s1 = e4m3_to_f32((s01 >> 8) & 0x7Fu);
                const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
                float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t hh[4];
                    cvt8(w[j], hh);
                    const int b = (j >> 1) * 2;
                    mfma2(a[b], a[b + 1], hh[0], xh[4 * j + 0]);
                    mfma2(a[b], a[b + 1], hh[1], xh[4 * j + 1]);
                    mfma2(a[b], a[b + 1], hh[2], xh[4 * j + 2]);
                    mfma2(a[b], a[b + 1], hh[3], xh[4 * j + 3]);
                }
                pv = fmaf(s0, a[0] + a[1], s1 * (a[2] + a[3]));
                if (inexact) {
                    // exact residual of x' - fp16(x') (slow path, rare), fp16(x') formed
                    // exactly as above
                    float q0 = 0.0f, q1 = 0.0f;
                    const uint16_t* xrow = x + 32 * c;
#pragma unroll 1
                    for (int k = 0; k < 32; ++k) {
                        const uint32_t wk = k < 16 ? (k < 8 ? w[0] : w[1]) : (k < 24 ? w[2] : w[3]);
                        const uint32_t code = (wk >> (4 * (k & 7))) & 15u;
                        const float xv32 = bf16_to_f32(xrow[k]);
                        const float hi = __half2float(__float2half_rn(pow2_scale(xv32, f1, f2)));
                        const float r = (ldexpf(xv32, e) - hi) * e2m1_to_f32(code);
                        if (k < 16) q0 += r; else q1 += r;
                    }
                    pv += fmaf(s0, q0, s1 * q1);
                }
                pv = pv * u1 * u2;
            }
            // sum over the G lanes of each row of this step
#pragma unroll
            for (int o = G / 2; o > 0; o >>= 1) pv += __shfl_xor_sync(0xffffffffu, pv, o);
            if ((lane % G) == 0 && rl < nr)
                slots[(sbeg + rl) * ngroups + warp] = pv;
        }
        __syncwarp();
        if (lane == 0 && !dbg.stall) mbar_arrive(&empty[s]);
    }
    named_bar_sync(1, nthreads_c);
    if (abort_flag) return;
    const float scale = *gw * (kXQ ? gq : (gx ? *gx : 1.0f));
    for (int i = threadIdx.x; i < nrows; i += nthreads_c) {
        float v = 0.0f;
        for (int w = 0; w < ngroups; ++w) v += slots[i * ngroups + w];
        store_y(y, r0 + i, v * scale, y_bf16);
    }
}

// ======================================================================================
// 2 <= M <= 16: mma.sync m16n8k16, NT token tiles of 8
// ======================================================================================
// Fragment ownership (m16n8k16, row.col): lane = 4 g + t; A: a0 = (row g, k 2t..2t+1),
// a1 = (g+8, 2t..), a2 = (g, 2t+8..), a3 = (g+8, 2t+8..); B: b0 = (k 2t.., col g),
// b1 = (k 2t+8.., col g); D: d0/d1 = (g, cols 2t, 2t+1), d2/d3 = (g+8, ...).
// K mapping (any bijection works when A and B use the same one): thread t of a quad
// streams 16-byte chunk c = 4 kg + t of its two rows; MMA j (0..7) takes elements
// 4j .. 4j+3 of that chunk for its k-slots {2t, 2t+1, 2t+8, 2t+9}.
// x' smem layout: token row m at m * rp + 32 (m % 4) bytes, then 8-byte groups
// (4 elements) ordered (j, c): group (j, c) at ((j * pitch + c) * 8); the padding and
// the (j, c) order make the B-fragment loads of a half-warp hit 16 distinct bank pairs.
constexpr int kMmaUnits = 2;  // (16-row block, 128-element K group) units in flight

template <int NT>
__global__ void __launch_bounds__(kThreads)
gemv_mma_kernel(const uint16_t* __restrict__ x, int M, int K, const uint8_t* __restrict__ wq,
                const uint8_t* __restrict__ wsz, const float* __restrict__ gw,
                const float* __restrict__ gx, int N, void* __restrict__ y, int y_bf16,
                int kc_max, int rb_max) {
    constexpr int MT = 8 * NT;
    extern __shared__ __align__(128) uint8_t smem[];
    const int pitch = kc_max >> 5;         // chunks per token row
    const int rp = pitch * 8 * 8 + 128;    // bytes per token row (+ padding)
    uint8_t* xs = smem;
    float* acc_sm = reinterpret_cast<float*>(smem + (size_t)MT * rp);  // [rb][16][MT]
    float* slots = acc_sm + (size_t)rb_max * 16 * MT;                  // [warp][2][16][MT]
    __shared__ int piece_rb[kWarps][2];
    __shared__ int e_sh[MT];
    __shared__ float red[kWarps];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nrb_all = (N + 15) >> 4;
    const int rb0 = (int)((int64_t)nrb_all * blockIdx.x / gridDim.x);
    const int rb1 = (int)((int64_t)nrb_all * (blockIdx.x + 1) / gridDim.x);
    const int nrb = rb1 - rb0;
    const int64_t row_bytes = K >> 1;
    for (int i = threadIdx.x; i < nrb * 16 * MT; i += kThreads) acc_sm[i] = 0.0f;

    for (int kc0 = 0; kc0 < K; kc0 += kc_max) {
        const int kl = min(kc_max, K - kc0);
        const int nch = kl >> 5;
        // ---- per-token exponent for this K chunk ----
        for (int m = 0; m < MT; ++m) {
            float am = 0.0f;
            if (m < M) {
                const uint32_t* xw = reinterpret_cast<const uint32_t*>(x + (int64_t)m * K + kc0);
                for (int i = threadIdx.x; i < (kl >> 1); i += kThreads) {
                    const uint32_t v = xw[i];
                    am = fmaxf(am, fmaxf(fabsf(bf16_to_f32(v & 0xFFFFu)),
                                         fabsf(bf16_to_f32(v >> 16))));
                }
            }
            const float r = block_max(am, red);
            if (threadIdx.x == 0) e_sh[m] = chunk_exponent(r);
        }
        __syncthreads();
        bool inexact = false;
        for (int i = threadIdx.x; i < MT * nch * 8; i += kThreads) {
            const int m = i / (nch * 8);
            const int rem = i - m * nch * 8;
            const int c = rem >> 3, j = rem & 7;
            uint2 h = make_uint2(0u, 0u);
            if (m < M) {
                const uint2 v = *reinterpret_cast<const uint2*>(x + (int64_t)m * K + kc0 + 32 * c + 4 * j);
                h.x = to_h2_scaled(v.x, e_sh[m], inexact);
                h.y = to_h2_scaled(v.y, e_sh[m], inexact);
            }
            *reinterpret_cast<uint2*>(xs + (size_t)m * rp + 32 * (m & 3) +
                                      ((size_t)j * pitch + c) * 8) = h;
        }
        const bool any_inexact = __syncthreads_or(inexact);

        // ---- units: (row block, K group of 4 chunks), split evenly over warps ----
        const int nkg = (nch + 3) >> 2;
        const int units = nrb * nkg;
        const int u0 = (int)((int64_t)units * warp / kWarps);
        const int u1 = (int)((int64_t)units * (warp + 1) / kWarps);
        if (lane == 0) { piece_rb[warp][0] = -1; piece_rb[warp][1] = -1; }
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
        int cur = -1, cur_first = 0;  // row block being accumulated, its first unit
        int rb = u0 / nkg, kg = u0 - rb * nkg;

        auto flush = [&](int last_unit_excl) {
            // piece of row block `cur` covering units [cur_first, last_unit_excl)
            // a warp's only partial pieces are its first and last; interior pieces are
            // whole row blocks owned by this warp alone
            const bool full = (cur_first == cur * nkg) && (last_unit_excl == (cur + 1) * nkg);
            float* dst;
            if (full) {
                dst = acc_sm + (size_t)cur * 16 * MT;
            } else {
                const int p = (cur_first == u0) ? 0 : 1;
                if (lane == 0) piece_rb[warp][p] = cur;
                dst = slots + ((size_t)warp * 2 + p) * 16 * MT;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int m0 = 8 * nt + 2 * t;
                const float v0 = ldexpf(acc[nt][0], -e_sh[m0]);
                const float v1 = ldexpf(acc[nt][1], -e_sh[m0 + 1]);
                const float v2 = ldexpf(acc[nt][2], -e_sh[m0]);
                const float v3 = ldexpf(acc[nt][3], -e_sh[m0 + 1]);
                if (full) {
                    dst[g * MT + m0] += v0;
                    dst[g * MT + m0 + 1] += v1;
                    dst[(g + 8) * MT + m0] += v2;
                    dst[(g + 8) * MT + m0 + 1] += v3;
                } else {
                    dst[g * MT + m0] = v0;
                    dst[g * MT + m0 + 1] = v1;
                    dst[(g + 8) * MT + m0] = v2;
                    dst[(g + 8) * MT + m0 + 1] = v3;
                }
                acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
            }
        };

        for (int u = u0; u < u1; u += kMmaUnits) {
            uint4 wa[kMmaUnits], wb[kMmaUnits];
            uint32_t sa[kMmaUnits], sb[kMmaUnits];
            int urb[kMmaUnits], uc[kMmaUnits];
#pragma unroll
            for (int i = 0; i < kMmaUnits; ++i) {
                urb[i] = (u + i < u1) ? rb : -1;
                const int c = kg * 4 + t;
                uc[i] = c;
                const int64_t ra = (int64_t)(rb0 + rb) * 16 + g, rbw = ra + 8;
                const bool ok = (u + i < u1) && c < nch;
                wa[i] = wb[i] = make_uint4(0u, 0u, 0u, 0u);
                sa[i] = sb[i] = 0u;
                if (ok && ra < N) {
                    wa[i] = ld_stream_u4(wq + ra * row_bytes + (kc0 >> 1) + 16 * (int64_t)c);
                    sa[i] = ld_nc_u16(wsz + ra * (K >> 4) + (kc0 >> 4) + 2 * c);
                }
                if (ok && rbw < N) {
                    wb[i] = ld_stream_u4(wq + rbw * row_bytes + (kc0 >> 1) + 16 * (int64_t)c);
                    sb[i] = ld_nc_u16(wsz + rbw * (K >> 4) + (kc0 >> 4) + 2 * c);
                }
                if (++kg == nkg) { kg = 0; ++rb; }
            }
#pragma unroll
            for (int i = 0; i < kMmaUnits; ++i) {
                if (urb[i] < 0) break;
                if (urb[i] != cur) {
                    if (cur >= 0) flush(u + i);
                    cur = urb[i];
                    cur_first = u + i;
                }
                // every lane takes part in the warp-wide mma.sync: a chunk past the end of
                // K has zero A fragments (loaded as zero above) and reads its B fragment
                // from a valid chunk, so it adds exactly zero
                const int c = uc[i];
                const int cb = c < nch ? c : nch - 1;
                const uint32_t wA[4] = {wa[i].x, wa[i].y, wa[i].z, wa[i].w};
                const uint32_t wB[4] = {wb[i].x, wb[i].y, wb[i].z, wb[i].w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t shA = e4m3_to_h2((sa[i] >> (8 * (j >> 2))) & 0xFFu);
                    const uint32_t shB = e4m3_to_h2((sb[i] >> (8 * (j >> 2))) & 0xFFu);
                    const uint32_t byA = wA[j >> 1] >> (16 * (j & 1));
                    const uint32_t byB = wB[j >> 1] >> (16 * (j & 1));
                    const uint32_t a0 = hmul2(cvt2(byA & 0xFFu), shA);
                    const uint32_t a2 = hmul2(cvt2((byA >> 8) & 0xFFu), shA);
                    const uint32_t a1 = hmul2(cvt2(byB & 0xFFu), shB);
                    const uint32_t a3 = hmul2(cvt2((byB >> 8) & 0xFFu), shB);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int m = 8 * nt + g;
                        const uint2 b = *reinterpret_cast<const uint2*>(
                            xs + (size_t)m * rp + 32 * (m & 3) + ((size_t)j * pitch + cb) * 8);
                        asm volatile(
                            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                            : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]),
                              "+f"(acc[nt][3])
                            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
                    }
                }
                if (any_inexact) {
                    // exact residual of x' - fp16(x') for this unit (slow path, rare):
                    // plain fp32 over the thread's (row, token) outputs
                    const int64_t ra = (int64_t)(rb0 + urb[i]) * 16 + g;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int m = 8 * nt + 2 * t + (q & 1);
                            const int64_t rr = ra + ((q & 2) ? 8 : 0);
                            if (m >= M || rr >= N) continue;
                            float s = 0.0f;
                            for (int cc = 0; cc < 4; ++cc) {  // the 4 chunks of the K group
                                const int ch = (c - t) + cc;
                                if (ch >= nch) break;
                                const uint4 wv = *reinterpret_cast<const uint4*>(
                                    wq + rr * row_bytes + (kc0 >> 1) + 16 * (int64_t)ch);
                                const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
                                const uint32_t s2 = *reinterpret_cast<const uint16_t*>(
                                    wsz + rr * (K >> 4) + (kc0 >> 4) + 2 * ch);
                                const uint16_t* xr = x + (int64_t)m * K + kc0 + 32 * ch;
                                float q0 = 0.0f, q1 = 0.0f;
                                for (int k = 0; k < 32; ++k) {
                                    const uint32_t wk = k < 16 ? (k < 8 ? ww[0] : ww[1]) : (k < 24 ? ww[2] : ww[3]);
                                    const uint32_t code = (wk >> (4 * (k & 7))) & 15u;
                                    const float r = residual(xr[k], e_sh[m]) * e2m1_to_f32(code);
                                    if (k < 16) q0 += r; else q1 += r;
                                }
                                s = fmaf(e4m3_to_f32(s2 & 0xFFu), q0,
                                         fmaf(e4m3_to_f32(s2 >> 8), q1, s));
                            }
                            // this lane owns output (rr, m): it adds the residual of the
                            // whole K group (all four chunks of the quad) for it
                            acc[nt][q] += s;
                        }
                    }
                }
            }
        }
        if (cur >= 0) flush(u1);
        __syncthreads();
        // ---- add the partial pieces in warp order ----
        for (int w = 0; w < kWarps; ++w) {
            for (int p = 0; p < 2; ++p) {
                const int prb = piece_rb[w][p];
                if (prb < 0) continue;
                const float* src = slots + ((size_t)w * 2 + p) * 16 * MT;
                float* dst = acc_sm + (size_t)prb * 16 * MT;
                for (int i = threadIdx.x; i < 16 * MT; i += kThreads) dst[i] += src[i];
                __syncthreads();
            }
        }
    }
    const float scale = *gw * (gx ? *gx : 1.0f);
    for (int i = threadIdx.x; i < nrb * 16 * M; i += kThreads) {
        const int m = i / (nrb * 16), rr = i - m * nrb * 16;
        const int64_t n = (int64_t)rb0 * 16 + rr;
        if (n < N) store_y(y, (int64_t)m * N + n, acc_sm[(size_t)rr * MT + m] * scale, y_bf16);
    }
}

// ---- launch -------------------------------------------------------------------------

template <typename Kern>
cudaError_t opt_in_smem(Kern kern, const DevInfo& dev, std::atomic<uint64_t>& configured) {
    const uint64_t bit = 1ull << (dev.device & 63);
    if (configured.load(std::memory_order_acquire) & bit) return cudaSuccess;
    // dynamic + static shared memory may not exceed the opt-in limit
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(dev.smem_optin - fa.sharedSizeBytes));
    if (e == cudaSuccess) configured.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// K chunk: as large as the staging budget allows, then balanced over the chunks
int kc_for(int K, int budget, int bytes_per_k) {
    const int kc_cap = (budget / bytes_per_k) / 32 * 32;
    const int nchunks = (K + kc_cap - 1) / kc_cap;
    const int kc = ((K + nchunks - 1) / nchunks + 31) / 32 * 32;
    return kc > K ? K : kc;
}

template <int NT>
cudaError_t launch_mma(const uint16_t* x, int M, int K, const uint8_t* wq, const uint8_t* wsz,
                       const float* gw, const float* gx, int N, void* y, bool y_bf16,
                       cudaStream_t stream, const DevInfo& dev) {
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = opt_in_smem(gemv_mma_kernel<NT>, dev, configured);
    if (e != cudaSuccess) return e;
    constexpr int MT = 8 * NT;
    const int kc = kc_for(K, kXSmemBytesMma, MT * 2);
    const int nrb = (N + 15) / 16;
    int grid = dev.sm_count * 2;
    if (grid > nrb) grid = nrb;
    const int rb_max = (nrb + grid - 1) / grid;
    const int rp = (kc / 32) * 64 + 128;
    const size_t smem = (size_t)MT * rp + ((size_t)rb_max * 16 * MT + (size_t)kWarps * 2 * 16 * MT) * 4;
    if (smem + 1024 > dev.smem_optin) return cudaErrorInvalidConfiguration;
    gemv_mma_kernel<NT><<<grid, kThreads, smem, stream>>>(x, M, K, wq, wsz, gw, gx, N, y,
                                                          y_bf16 ? 1 : 0, kc, rb_max);
    return cudaGetLastError();
}

size_t pipe_smem(int K, int rows_max, int rps, int stages, int ngroups) {
    return (size_t)stages * pipe_stage_bytes(K, rps) + pipe_slot_bytes(rows_max, ngroups) +
           2 * (size_t)stages * 8;
}

template <int G, bool kXQ>
cudaError_t launch_pipe(const uint16_t* x, int K, const uint8_t* wq, const uint8_t* wrm,
                        const float* gw, const float* gx, int N, void* y, bool y_bf16,
                        uint32_t* err, bool w_static, cudaStream_t stream, const DevInfo& dev,
                        bool* launched, uint8_t* xq_out = nullptr, uint8_t* xs_out = nullptr,
                        float* gx_out = nullptr) {
    *launched = false;
    const int rowchunks = K / 32;
    const int ngroups = (rowchunks + G - 1) / G;
    int grid = dev.sm_count;
    if (grid > N) grid = N;
    const int rows_max = (N + grid - 1) / grid;
    int rps = (int)(kPipeStageTarget / (K / 2));
    if (rps < 1) rps = 1;
    if (rps > rows_max) rps = rows_max;
    // whole steps of 32/G rows per full stage (the kernel's predicate-free path)
    constexpr int L = 32 / G;
    if (rps >= L) rps = rps / L * L;
    // the deepest ring (2..8 stages) that fits one CTA per SM
    const size_t budget = dev.smem_optin - 2048;
    int stages = 8;
    while (stages > 2 && pipe_smem(K, rows_max, rps, stages, ngroups) > budget) --stages;
    // a CTA with many rows (a wide N) keeps a large slot area: shorter stages, in whole
    // steps, where two full ones do not fit beside it
    while (rps > L && pipe_smem(K, rows_max, rps, stages, ngroups) > budget) rps -= L;
    const size_t smem = pipe_smem(K, rows_max, rps, stages, ngroups);
    if (smem + 2048 > dev.smem_optin) return cudaSuccess;
    // the first stage: whole steps of L rows, about kPipeFirstStage bytes of codes
    int rfirst = (kPipeFirstStage / (K / 2) + L - 1) / L * L;
    if (rfirst < L) rfirst = L;
    if (rfirst > rps) rfirst = rps;
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = opt_in_smem(gemv_m1_pipe_kernel<G, kXQ>, dev, configured);
    if (e != cudaSuccess) return e;
    // launched as a programmatic dependent: its prologue and first L2 prefetches overlap
    // the tail of the kernel before it on the stream
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((ngroups + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemv_m1_pipe_kernel<G, kXQ>, x, K, wq, wrm, gw, gx, N,
                           y, y_bf16 ? 1 : 0, rows_max, rps, rfirst, stages,
                           w_static ? 1 : 0, err, current_wait_cfg(), xq_out, xs_out, gx_out);
    *launched = true;
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_m1(const uint16_t* x, int K, const uint8_t* wq, const uint8_t* wsz,
                      const float* gw, const float* gx, int N, void* y, bool y_bf16,
                      uint32_t* err, bool w_static, cudaStream_t stream, const DevInfo& dev) {
    // x-stationary pipelined kernel: column groups of G chunks, one consumer warp each,
    // at most 31 of them (plus the producer warp); G is the smallest of 8, 16, 32 that fits
    const int rowchunks = K / 32;
    bool launched = false;
    cudaError_t e = cudaSuccess;
    if (rowchunks >= 8 * 8 && (rowchunks + 7) / 8 <= 31)
        e = launch_pipe<8, false>(x, K, wq, wsz, gw, gx, N, y, y_bf16, err, w_static, stream, dev,
                           &launched);
    else if (rowchunks >= 8 * 16 && (rowchunks + 15) / 16 <= 31)
        e = launch_pipe<16, false>(x, K, wq, wsz, gw, gx, N, y, y_bf16, err, w_static, stream, dev,
                            &launched);
    else if (rowchunks >= 8 * 32 && (rowchunks + 31) / 32 <= 31)
        e = launch_pipe<32, false>(x, K, wq, wsz, gw, gx, N, y, y_bf16, err, w_static, stream, dev,
                            &launched);
    if (e != cudaSuccess || launched) return e;
    static std::atomic<uint64_t> configured{0};
    e = opt_in_smem(gemv_m1_kernel, dev, configured);
    if (e != cudaSuccess) return e;
    const int kc = kc_for(K, kXSmemBytes, 2);
    int grid = dev.sm_count * 2;
    if (grid > N) grid = N;
    const int rows_max = (N + grid - 1) / grid;
    const size_t smem = (size_t)kc * 2 + (size_t)rows_max * kWarps * 4;
    if (smem + 1024 > dev.smem_optin) return cudaErrorInvalidConfiguration;
    gemv_m1_kernel<<<grid, kThreads, smem, stream>>>(x, K, wq, wsz, gw, gx, N, y,
                                                     y_bf16 ? 1 : 0, kc);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_w4a4_static(const uint16_t* x, int M, int K, const uint8_t* wq,
                                    const uint8_t* wsz_all, const float* gw, const float* gx,
                                    int N, void* y, bool y_bf16, uint32_t* err, bool w_static,
                                    cudaStream_t stream, const DevInfo& dev, bool* launched,
                                    uint8_t* xq_out, uint8_t* xs_out, float* gx_out) {
    *launched = false;
    const int64_t atom = (int64_t)((N + 127) / 128 * 128) * ((K / 16 + 3) / 4 * 4);
    const uint8_t* wsz = wsz_all + atom;
    if (M >= 2) {
        // a dynamic g_x at M >= 2 takes the quantizer kernels: every skinny CTA would
        // quantize all of x again, which costs more than one pass ahead of the kernel
        if (!gx) return cudaSuccess;
        return launch_skinny_w4a16(x, M, K, wq, wsz, gw, gx, N, y, y_bf16, err, w_static,
                                   stream, dev, launched, true);
    }
    if (M != 1) return cudaSuccess;
    const int rowchunks = K / 32;
    if (rowchunks >= 8 * 8 && (rowchunks + 7) / 8 <= 31)
        return launch_pipe<8, true>(x, K, wq, wsz, gw, gx, N, y, y_bf16, err, w_static, stream,
                                    dev, launched, xq_out, xs_out, gx_out);
    if (rowchunks >= 8 * 16 && (rowchunks + 15) / 16 <= 31)
        return launch_pipe<16, true>(x, K, wq, wsz, gw, gx, N, y, y_bf16, err, w_static, stream,
                                     dev, launched, xq_out, xs_out, gx_out);
    if (rowchunks >= 8 * 32 && (rowchunks + 31) / 32 <= 31)
        return launch_pipe<32, true>(x, K, wq, wsz, gw, gx, N, y, y_bf16, err, w_static, stream,
                                     dev, launched, xq_out, xs_out, gx_out);
    return cudaSuccess;
}

cudaError_t launch_gemv_w4a16(const uint16_t* x, int M, int K, const uint8_t* wq,
                              const uint8_t* wsz_all, const float* gw, const float* gx, int N,
                              void* y, bool y_bf16, uint32_t* err, bool w_static,
                              cudaStream_t stream, const DevInfo& dev) {
    // the small-M kernels read the row-major part of the repacked scales
    const int64_t atom = (int64_t)((N + 127) / 128 * 128) * ((K / 16 + 3) / 4 * 4);
    const uint8_t* wsz = wsz_all + atom;
    if (M == 1) return launch_m1(x, K, wq, wsz, gw, gx, N, y, y_bf16, err, w_static, stream, dev);
    bool launched = false;
    const cudaError_t e = launch_skinny_w4a16(x, M, K, wq, wsz, gw, gx, N, y, y_bf16, err,
                                              w_static, stream, dev, &launched);
    if (e != cudaSuccess || launched) return e;
    if (M <= 8) return launch_mma<1>(x, M, K, wq, wsz, gw, gx, N, y, y_bf16, stream, dev);
    return launch_mma<2>(x, M, K, wq, wsz, gw, gx, N, y, y_bf16, stream, dev);
}

}  // namespace nvfp4
