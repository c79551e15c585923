/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for the NVFP4 block-scaled projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or loads
 * this file; only the tests, the smoke check and the CPU-baseline leg of the bench
 * use it.  It shares no code, table or constant generator with the CUDA path.
 *
 * What it computes, and where that is stated:
 *   - The format: "NVFP4" weights named by the Qwen3x-Orin README (Repository map:
 *     "src/quantization/  FP8 and NVFP4 format primitives") and by FlashRT
 *     docs/qwen36_usage.md (constructor argument table: "compressed-tensors
 *     nvfp4-pack-quantized safetensors"; constructor paragraph: "NVFP4 swizzle";
 *     env-var table, FLASHRT_QWEN36_MTP_CKPT_DIR: "converted FP8 -> BF16 -> NVFP4").
 *     The pages name the format without defining its arithmetic.  The definition
 *     written out here is the standard one: E2M1 values {0, .5, 1, 1.5, 2, 3, 4, 6}
 *     with a sign bit, one E4M3 (OCP FP8 "E4M3FN", bias 7, max 448) scale per 16
 *     consecutive elements of a row, and one FP32 global scale g = amax / (6 * 448).
 *   - The projection y[M,N] = x[M,K] . W^T at decode (M = 1), MTP verify (M = K + 1)
 *     and prefill chunks: Qwen3x-Orin README (Functional evaluation quick start,
 *     "--projection-backend sm87", "--prefill-chunk-size 512"); FlashRT
 *     docs/qwen36_usage.md (generate_own_speculative_KN_nvfp4 argument table:
 *     verify runs K+1 tokens at once; per-step decode section).
 *   - Fused gate/up (one GEMM, one shared global scale) and NVFP4 activations:
 *     FlashRT docs/qwen36_usage.md env-var table, FLASHRT_QWEN36_FUSE_MLP_GATE_UP
 *     and FLASHRT_QWEN36_FUSE_SILU_MUL_QUANT.
 *
 * Readings adopted where the definition leaves a step open (each is also listed in
 * the design notes):
 *   R1  amax == 0: g := 1.0f, every scale byte and every code is zero (codes keep
 *       the sign bit of a signed-zero input).
 *   R2  block scale: s_raw = bmax / (6.0f * g), two fp32 round-to-nearest-even ops
 *       in that order (product first, then the division).
 *   R3  element code: v = T / d with d = float(s8) * g, an fp32 RN division (not a
 *       reciprocal multiply); d == 0 gives a signed zero code.
 *   R4  E2M1 rounding: nearest grid value, ties to the even code, |v| >= 6 -> 6; the
 *       sign bit is the input's sign bit (so -0.1 -> code 0x8).
 *   R5  E4M3 rounding: nearest finite value, ties to the even code, saturating at
 *       448 (0x7E).  Scales are never negative.
 *   R6  packing: byte j of a row holds element 2j in its low nibble and element
 *       2j+1 in its high nibble.
 *   R7  swizzled scale layout ("NVFP4 swizzle" at load): first the 128-row x 4-block
 *       atoms of the tensor-core block scale layout, element (r, cb) at byte
 *          ((r/128)*(Cp/4) + cb/4)*512 + (r%32)*16 + ((r%128)/32)*4 + cb%4,
 *       rows padded to a multiple of 128 and blocks to a multiple of 4 with zero
 *       (A = Rp*Cp bytes); then, at byte A, the row-major scales [R, C/16] once more
 *       (for the GEMV, which streams a row's scales next to its codes), zero-padded to
 *       a multiple of 16 bytes plus 16 bytes.
 *   R8  linear: y[m,n] = sum_k x[m,k] * e2m1(q[n,k]) * e4m3(s[n,k/16]) * g_w summed
 *       in fp64; for activations quantized to NVFP4 (W4A4), x is replaced by its
 *       dequantized value.
 *   R9  non-finite inputs violate the precondition; the quantizer reports them.
 *   R10 FP8 "e4m3 block-128" source (the MTP checkpoint, FlashRT
 *       docs/qwen36_usage.md, env-var table, FLASHRT_QWEN36_MTP_CKPT_DIR: FP8 e4m3
 *       block-128, converted FP8 -> BF16 -> NVFP4): one fp32 scale per 128 x 128
 *       tile, stored [ceil(R/128), ceil(C/128)] row-major, which multiplies the E4M3
 *       value; the product is one fp32 round-to-nearest-even multiply, then rounded
 *       to bf16 (nearest even), and the bf16 tensor is quantized by R1-R9.
 *   R11 fused silu(gate) * up -> NVFP4 activations (FlashRT docs/qwen36_usage.md,
 *       env-var table, FLASHRT_QWEN36_FUSE_SILU_MUL_QUANT, after the fused gate/up GEMM
 *       of FLASHRT_QWEN36_FUSE_MLP_GATE_UP): the GEMM's bf16 output [M, 2I] holds gate
 *       in columns [0, I) and up in [I, 2I); h = (g / (1 + exp(-g))) * u in fp32, one
 *       correctly rounded operation per step, and the fp32 h goes straight to R1-R9
 *       (no bf16 copy in between: the fusion keeps h in registers).  exp is the fp32
 *       method of orc_exp_f32 below, the same steps on both sides, because the E2M1
 *       and E4M3 roundings of h hang on its last bit.
 *
 * Built with strict IEEE semantics (-O2 -ffp-contract=off, no fast-math): every
 * fp32 operation below is one correctly rounded operation.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------- */
/* Value sets                                                                */
/* ------------------------------------------------------------------------- */

/* E2M1 magnitudes for the 3 low bits of a code (sign bit is bit 3). */
static const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Decoded value of a 4-bit E2M1 code. */
ORC_EXPORT double orc_e2m1_value(uint32_t code) {
    double m = kE2M1Mag[code & 7u];
    return (code & 8u) ? -m : m;
}

/* Decoded value of an E4M3 byte (OCP "E4M3FN": bias 7, no infinities,
 * S.1111.111 is NaN).  exponent field e, mantissa m:
 *   e == 0 : m * 2^-9           (subnormal)
 *   e >= 1 : 2^(e-7) * (1 + m/8) */
ORC_EXPORT double orc_e4m3_value(uint32_t byte) {
    uint32_t e = (byte >> 3) & 15u, m = byte & 7u;
    double v;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return (byte & 0x80u) ? -v : v;
}

/* ------------------------------------------------------------------------- */
/* Rounding onto the grids (nearest value, ties to the even code)            */
/* ------------------------------------------------------------------------- */

/* R4: fp32 -> E2M1 code.  Magnitudes of 6 and above saturate to 6; below that,
 * the nearest of the 8 magnitudes by exhaustive search in fp64 (for |v| < 6 every
 * difference below is exact), ties to the even code.  The sign bit is copied from
 * the input. */
ORC_EXPORT uint32_t orc_e2m1_encode(float v) {
    double a = fabs((double)v);
    uint32_t best = 0;
    double best_d = a; /* distance to magnitude 0 */
    if (a >= 6.0) return 7u | (signbit(v) ? 8u : 0u);
    for (uint32_t c = 1; c < 8; ++c) {
        double d = fabs(a - kE2M1Mag[c]);
        if (d < best_d || (d == best_d && (c & 1u) == 0u && (best & 1u) == 1u)) {
            best = c;
            best_d = d;
        }
    }
    return best | (signbit(v) ? 8u : 0u);
}

/* R5: non-negative fp32 -> E4M3 byte in [0x00, 0x7E].  The 127 finite
 * non-negative values increase with the code, so the code whose value is the
 * largest one <= a is found by bisection; the result is whichever of it and the
 * next code is nearer, ties to the even code.  Anything above 448 is nearest
 * to 448, which is the saturating behaviour. */
ORC_EXPORT uint32_t orc_e4m3_encode(float v) {
    double a = (double)v;
    uint32_t lo = 0, hi = 126; /* invariant: value(lo) <= a when a >= 0 */
    if (!(a > 0.0)) return 0u;
    if (a >= orc_e4m3_value(126)) return 126u;
    while (hi - lo > 1u) {
        uint32_t mid = (lo + hi) / 2u;
        if (orc_e4m3_value(mid) <= a) lo = mid; else hi = mid;
    }
    /* now value(lo) <= a < value(hi), hi == lo + 1 */
    {
        double d_lo = a - orc_e4m3_value(lo);
        double d_hi = orc_e4m3_value(hi) - a;
        if (d_lo < d_hi) return lo;
        if (d_hi < d_lo) return hi;
        return (lo & 1u) ? hi : lo;
    }
}

ORC_EXPORT void orc_e2m1_encode_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e2m1_encode(v[i]);
}

ORC_EXPORT void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e4m3_encode(v[i]);
}

/* ------------------------------------------------------------------------- */
/* BF16 helpers                                                              */
/* ------------------------------------------------------------------------- */

/* BF16 is the top half of an fp32: widening is exact. */
ORC_EXPORT float orc_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp64 -> fp32 (round to nearest even) -> bf16 (round to nearest even). */
ORC_EXPORT uint16_t orc_round_bf16(double v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16); /* inf */
    {
        uint32_t lsb = (u >> 16) & 1u;
        u += 0x7FFFu + lsb;
    }
    return (uint16_t)(u >> 16);
}

ORC_EXPORT void orc_round_bf16_array(const double* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_round_bf16(v[i]);
}

/* R10: FP8 E4M3 bytes q [rows, cols] with fp32 tile scales s [ceil(rows/128),
 * ceil(cols/128)] -> bf16 bit patterns of bf16(e4m3(q) * s), the tensor that the FP8
 * -> BF16 -> NVFP4 chain hands to the quantizer.  NaN bytes stay NaN (the quantizer
 * then rejects the tensor, R9). */
ORC_EXPORT void orc_dequant_fp8_block128(const uint8_t* q, const float* s, int64_t rows,
                                         int64_t cols, uint16_t* out) {
    const int64_t tiles_per_row = (cols + 127) / 128;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            const float v = (float)orc_e4m3_value(q[r * cols + c]); /* exact */
            const float p = v * s[(r / 128) * tiles_per_row + c / 128];
            out[r * cols + c] = orc_round_bf16((double)p);          /* p is exact in fp64 */
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Quantizer                                                                 */
/* ------------------------------------------------------------------------- */

static float load_elem(const void* src, int src_is_bf16, int64_t i) {
    if (src_is_bf16) return orc_bf16_to_f32(((const uint16_t*)src)[i]);
    return ((const float*)src)[i];
}

/* Quantize T[rows, cols] (fp32 or bf16, row-major, cols % 16 == 0) to packed E2M1
 * codes [rows, cols/2], row-major E4M3 scales [rows, cols/16] and the fp32 global
 * scale.  With given_g == NULL the global scale is amax / 2688 (steps 1-2, R1);
 * otherwise *given_g (finite, > 0) is used as the global scale unchanged (a
 * static activation scale).  Returns 0, or -1 on a non-finite input, a bad given
 * scale or a bad shape (R9). */
ORC_EXPORT int orc_quantize(const void* src, int src_is_bf16, int64_t rows, int64_t cols,
                            const float* given_g, uint8_t* packed, uint8_t* scales,
                            float* g_out) {
    int64_t r, b, k;
    float g;
    if (rows < 0 || cols < 0 || cols % 16 != 0) return -1;
    /* step 1: amax over the whole tensor (|.| of an fp32 is exact) */
    {
        float amax = 0.0f;
        for (int64_t i = 0; i < rows * cols; ++i) {
            float a = fabsf(load_elem(src, src_is_bf16, i));
            if (!isfinite(a)) return -1;
            if (a > amax) amax = a;
        }
        /* step 2: global scale (R1 for an all-zero tensor) */
        if (given_g) {
            g = *given_g;
            if (!isfinite(g) || !(g > 0.0f)) return -1;
        } else if (amax == 0.0f) {
            g = 1.0f;
        } else {
            g = amax / 2688.0f; /* 6 * 448 */
        }
    }
    *g_out = g;
    for (r = 0; r < rows; ++r) {
        for (b = 0; b < cols / 16; ++b) {
            const int64_t base = r * cols + b * 16;
            float bmax = 0.0f, six_g, s_raw, d;
            uint32_t s8;
            /* step 3: block max and raw scale (R2) */
            for (k = 0; k < 16; ++k) {
                float a = fabsf(load_elem(src, src_is_bf16, base + k));
                if (a > bmax) bmax = a;
            }
            six_g = 6.0f * g;
            s_raw = bmax / six_g;
            /* step 4: E4M3 scale (R5) */
            s8 = orc_e4m3_encode(s_raw);
            scales[r * (cols / 16) + b] = (uint8_t)s8;
            /* step 5: decode scale */
            d = (float)orc_e4m3_value(s8) * g;
            /* steps 6-8: element codes (R3, R4), packing (R6) */
            for (k = 0; k < 16; k += 2) {
                uint32_t c[2];
                for (int j = 0; j < 2; ++j) {
                    float t = load_elem(src, src_is_bf16, base + k + j);
                    if (d == 0.0f) c[j] = signbit(t) ? 8u : 0u;
                    else c[j] = orc_e2m1_encode(t / d);
                }
                packed[(base + k) / 2] = (uint8_t)(c[0] | (c[1] << 4));
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Fused silu(gate) * up activations (R11)                                   */
/* ------------------------------------------------------------------------- */

/* exp(x) in fp32 by W. J. Cody and W. Waite's argument reduction ("Software Manual
 * for the Elementary Functions", 1980): n = rint(x * log2(e)), r = x - n * ln2 with ln2
 * split into a 16-bit head (so n * head is exact) and a tail, then e^r from its Taylor
 * series to r^7 (|r| <= ln2/2 + a little: the next term is below 2^-27 relative),
 * evaluated by Horner's rule with fused multiply-adds, times 2^n.  Inputs are clamped
 * first: x > 88 gives +inf and x < -87 gives 0 (n then stays in [-126, 127], so 2^n is
 * a normal float and the last multiply is one correctly rounded operation).  Every
 * step is one fp32 operation in this order; the kernels take the same steps. */
ORC_EXPORT float orc_exp_f32(float x) {
    /* fp32 constants, written as hexadecimal floats: log2(e) and ln 2 rounded to
     * nearest; the head of ln 2 keeps 16 significant bits, the tail is ln 2 - head
     * rounded to nearest; the Taylor coefficients 1/k! rounded to nearest */
    const float log2e = 0x1.715476p+0f;
    const float ln2_hi = 0x1.62e4p-1f;
    const float ln2_lo = 0x1.7f7d1cp-20f;
    float n, r, p, two_n;
    uint32_t bits;
    if (x > 88.0f) return INFINITY;
    if (x < -87.0f) return 0.0f;
    n = rintf(x * log2e);
    r = fmaf(-n, ln2_hi, x);
    r = fmaf(-n, ln2_lo, r);
    p = 0x1.a01a02p-13f;            /* 1/5040 */
    p = fmaf(p, r, 0x1.6c16c2p-10f); /* 1/720 */
    p = fmaf(p, r, 0x1.111112p-7f);  /* 1/120 */
    p = fmaf(p, r, 0x1.555556p-5f);  /* 1/24 */
    p = fmaf(p, r, 0x1.555556p-3f);  /* 1/6 */
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    bits = (uint32_t)((int32_t)n + 127) << 23;
    memcpy(&two_n, &bits, 4);
    return p * two_n;
}

/* h = silu(g) * u = (g / (1 + exp(-g))) * u, each step one fp32 RN operation. */
ORC_EXPORT float orc_silu_mul_f32(float g, float u) {
    const float e = orc_exp_f32(-g);
    const float den = 1.0f + e;
    const float sg = g / den;
    return sg * u;
}

/* R11: gate_up bf16 [M, 2I] (gate columns [0, I), up [I, 2I)) -> h fp32 [M, I]. */
ORC_EXPORT void orc_silu_mul(const uint16_t* gate_up, int64_t M, int64_t I, float* h) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t i = 0; i < I; ++i)
            h[m * I + i] = orc_silu_mul_f32(orc_bf16_to_f32(gate_up[m * 2 * I + i]),
                                            orc_bf16_to_f32(gate_up[m * 2 * I + I + i]));
}

/* ------------------------------------------------------------------------- */
/* Swizzled scale layout (R7)                                                */
/* ------------------------------------------------------------------------- */

/* bytes of the atom part of the swizzled layout */
ORC_EXPORT int64_t orc_repack_atom_bytes(int64_t rows, int64_t cols) {
    int64_t rp = (rows + 127) / 128 * 128;
    int64_t cb = cols / 16;
    int64_t cp = (cb + 3) / 4 * 4;
    return rp * cp;
}

ORC_EXPORT int64_t orc_repack_bytes(int64_t rows, int64_t cols) {
    return orc_repack_atom_bytes(rows, cols) + (rows * (cols / 16) + 15) / 16 * 16 + 16;
}

ORC_EXPORT int64_t orc_swizzle_offset(int64_t r, int64_t cb, int64_t cols) {
    int64_t cp = (cols / 16 + 3) / 4 * 4;
    return ((r / 128) * (cp / 4) + cb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 +
           cb % 4;
}

/* scales [rows, cols/16] row-major -> swizzled bytes (out_bytes must equal
 * orc_repack_bytes): the atom part, then the row-major copy; padding bytes are zero. */
ORC_EXPORT int orc_repack(const uint8_t* scales, int64_t rows, int64_t cols, uint8_t* out,
                          int64_t out_bytes) {
    if (cols % 16 != 0 || out_bytes != orc_repack_bytes(rows, cols)) return -1;
    memset(out, 0, (size_t)out_bytes);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t cb = 0; cb < cols / 16; ++cb)
            out[orc_swizzle_offset(r, cb, cols)] = scales[r * (cols / 16) + cb];
    memcpy(out + orc_repack_atom_bytes(rows, cols), scales, (size_t)(rows * (cols / 16)));
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Dequantization and the linear (R8)                                        */
/* ------------------------------------------------------------------------- */

/* Exact value of element (r, k) of a quantized tensor, without the global scale. */
static double deq_noglobal(const uint8_t* packed, const uint8_t* scales, int64_t cols,
                           int64_t r, int64_t k) {
    uint8_t byte = packed[(r * cols + k) / 2];
    uint32_t code = (k & 1) ? (uint32_t)(byte >> 4) : (uint32_t)(byte & 15u);
    return orc_e2m1_value(code) * orc_e4m3_value(scales[r * (cols / 16) + k / 16]);
}

/* out[r, k] = e2m1(code) * e4m3(scale) * g, in fp64 (exact). */
ORC_EXPORT void orc_dequantize(const uint8_t* packed, const uint8_t* scales, float g,
                               int64_t rows, int64_t cols, double* out) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < cols; ++k)
            out[r * cols + k] = deq_noglobal(packed, scales, cols, r, k) * (double)g;
}

/* One output of the W4A16 linear: y = sum_k x[m,k] * w[n,k] in fp64, plus the
 * tolerance reference sum_k |x[m,k] * w[n,k]|. */
static void dot_w4a16(const uint16_t* x, int64_t K, const uint8_t* wq, const uint8_t* ws,
                      float gw, int64_t m, int64_t n, double* y, double* absdot) {
    double acc = 0.0, aacc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = (double)orc_bf16_to_f32(x[m * K + k]) *
                   (deq_noglobal(wq, ws, K, n, k) * (double)gw);
        acc += p;
        aacc += fabs(p);
    }
    *y = acc;
    *absdot = aacc;
}

/* Full W4A16 linear: x bf16 [M,K], W quantized [N,K] (row-major scales),
 * y and absdot fp64 [M,N].  Outputs are independent; they are spread over
 * threads when OpenMP is available. */
ORC_EXPORT int orc_linear_w4a16(const uint16_t* x, int64_t M, int64_t K, const uint8_t* wq,
                                const uint8_t* ws, float gw, int64_t N, double* y,
                                double* absdot) {
    if (K % 16 != 0) return -1;
#pragma omp parallel for schedule(dynamic, 4) collapse(2)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            dot_w4a16(x, K, wq, ws, gw, m, n, &y[m * N + n], &absdot[m * N + n]);
    return 0;
}

/* The same outputs at chosen (m, n) pairs only. */
ORC_EXPORT int orc_linear_w4a16_pairs(const uint16_t* x, int64_t M, int64_t K,
                                      const uint8_t* wq, const uint8_t* ws, float gw,
                                      int64_t N, const int64_t* pm, const int64_t* pn,
                                      int64_t npairs, double* y, double* absdot) {
    if (K % 16 != 0) return -1;
    for (int64_t i = 0; i < npairs; ++i)
        if (pm[i] < 0 || pm[i] >= M || pn[i] < 0 || pn[i] >= N) return -1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < npairs; ++i)
        dot_w4a16(x, K, wq, ws, gw, pm[i], pn[i], &y[i], &absdot[i]);
    return 0;
}

/* One output of the W4A4 linear on dequantized operands. */
static void dot_w4a4(const uint8_t* xq, const uint8_t* xs, float gx, int64_t K,
                     const uint8_t* wq, const uint8_t* ws, float gw, int64_t m, int64_t n,
                     double* y, double* absdot) {
    double acc = 0.0, aacc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = (deq_noglobal(xq, xs, K, m, k) * (double)gx) *
                   (deq_noglobal(wq, ws, K, n, k) * (double)gw);
        acc += p;
        aacc += fabs(p);
    }
    *y = acc;
    *absdot = aacc;
}

/* W4A4 linear: x (bf16 [M,K]) is first quantized by orc_quantize (dynamic global
 * scale when given_gx is NULL), its codes/scales/global scale are returned in
 * xq [M,K/2], xs [M,K/16] (row-major), *gx_out, and y/absdot [M,N] are the fp64
 * products of the dequantized operands. */
ORC_EXPORT int orc_linear_w4a4(const uint16_t* x, int64_t M, int64_t K, const uint8_t* wq,
                               const uint8_t* ws, float gw, int64_t N, const float* given_gx,
                               uint8_t* xq, uint8_t* xs, float* gx_out, double* y,
                               double* absdot) {
    if (orc_quantize(x, 1, M, K, given_gx, xq, xs, gx_out) != 0) return -1;
#pragma omp parallel for schedule(dynamic, 4) collapse(2)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            dot_w4a4(xq, xs, *gx_out, K, wq, ws, gw, m, n, &y[m * N + n], &absdot[m * N + n]);
    return 0;
}

/* W4A4 outputs at chosen (m, n) pairs, from an already quantized x. */
ORC_EXPORT int orc_linear_w4a4_pairs(const uint8_t* xq, const uint8_t* xs, float gx,
                                     int64_t M, int64_t K, const uint8_t* wq,
                                     const uint8_t* ws, float gw, int64_t N,
                                     const int64_t* pm, const int64_t* pn, int64_t npairs,
                                     double* y, double* absdot) {
    if (K % 16 != 0) return -1;
    for (int64_t i = 0; i < npairs; ++i)
        if (pm[i] < 0 || pm[i] >= M || pn[i] < 0 || pn[i] >= N) return -1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < npairs; ++i)
        dot_w4a4(xq, xs, gx, K, wq, ws, gw, pm[i], pn[i], &y[i], &absdot[i]);
    return 0;
}

/* Number of threads the OpenMP loops above use (1 without OpenMP). */
ORC_EXPORT int orc_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
