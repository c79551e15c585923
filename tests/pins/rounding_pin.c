/*
 * rounding_pin.c -- an independent formulation of E2M1 and E4M3 round-to-nearest-
 * even, used only by the tests to pin the oracle's rounding functions.
 *
 * The oracle rounds by searching the value grid for the nearest value (fp64
 * distances).  This file instead works on the fp32 bit pattern with integer
 * arithmetic: it picks the quantum of the target format at the input's binade,
 * shifts the 24-bit significand down to that quantum and rounds the discarded bits
 * half-to-even, then builds the code from (exponent, quotient) and saturates.
 * The two share no code.  The sweep drivers below compare the oracle (passed in as
 * a function pointer) against this formulation over ranges of fp32 bit patterns.
 */
#include <stdint.h>
#include <string.h>

#define PIN_EXPORT __attribute__((visibility("default")))

/* Round S (24-bit significand) right by `shift` bits, half to even. */
static uint32_t rne_shift(uint32_t S, int shift) {
    uint32_t q, rem, half;
    if (shift >= 25) return 0u; /* S < 2^24 <= 2^(shift-1): below half a quantum */
    if (shift <= 0) return S << (-shift);
    q = S >> shift;
    rem = S & ((1u << shift) - 1u);
    half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return q;
}

/* E2M1: 1 mantissa bit, exponent bias 1, normals from 1.0, subnormal quantum 0.5,
 * largest value 6.  Returns the 4-bit code with the input's sign bit. */
PIN_EXPORT uint32_t pin_e2m1_from_bits(uint32_t u) {
    uint32_t sign = u >> 31, a = u & 0x7FFFFFFFu, E = a >> 23, code;
    if (E == 0u) {
        code = 0u; /* zero or fp32 subnormal: far below half of 0.5 */
    } else {
        int e = (int)E - 127;
        uint32_t S = (a & 0x7FFFFFu) | 0x800000u;
        int qe = (e > 0 ? e : 0) - 1; /* log2 of the quantum at this binade */
        uint32_t q = rne_shift(S, qe - e + 23);
        if (e < 0) code = q;                            /* q in {0, 1, 2} */
        else code = (((uint32_t)e + 1u) << 1) + q - 2u; /* q in [2, 4] */
        if (code > 7u) code = 7u;
    }
    return code | (sign << 3);
}

/* E4M3 (OCP E4M3FN): 3 mantissa bits, bias 7, normals from 2^-6, subnormal
 * quantum 2^-9, largest finite 448 = code 0x7E.  Non-positive inputs give 0. */
PIN_EXPORT uint32_t pin_e4m3_from_bits(uint32_t u) {
    uint32_t E = (u >> 23) & 0xFFu, code;
    if ((u >> 31) || E == 0u) return 0u;
    {
        int e = (int)E - 127;
        uint32_t S = (u & 0x7FFFFFu) | 0x800000u;
        int qe = (e > -6 ? e : -6) - 3;
        uint32_t q = rne_shift(S, qe - e + 23);
        if (e < -6) code = q;                             /* q in [0, 8] */
        else code = (((uint32_t)(e + 7)) << 3) + q - 8u;  /* q in [8, 16] */
        if (code > 126u) code = 126u;
    }
    return code;
}

typedef uint32_t (*enc_fn)(float);

static float bits_to_float(uint32_t u) {
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Compare oracle vs this formulation over bit patterns lo, lo+step, ... <= hi,
 * skipping NaN/Inf (outside the precondition).  Returns the mismatch count;
 * *first_bad gets the smallest mismatching pattern. */
static int64_t sweep(enc_fn oracle, uint32_t (*pin)(uint32_t), uint64_t lo, uint64_t hi,
                     uint64_t step, uint32_t* first_bad) {
    int64_t bad = 0;
    uint64_t first = UINT64_MAX;
    int64_t n = (int64_t)((hi - lo) / step) + 1;
#pragma omp parallel for schedule(static, 1 << 16) reduction(+ : bad) reduction(min : first)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t b = lo + (uint64_t)i * step;
        uint32_t u = (uint32_t)b;
        if (((u >> 23) & 0xFFu) == 0xFFu) continue;
        if (oracle(bits_to_float(u)) != pin(u)) {
            bad += 1;
            if (b < first) first = b;
        }
    }
    *first_bad = (first == UINT64_MAX) ? 0u : (uint32_t)first;
    return bad;
}

PIN_EXPORT int64_t pin_sweep_e2m1(enc_fn oracle, uint64_t lo, uint64_t hi, uint64_t step,
                                  uint32_t* first_bad) {
    return sweep(oracle, pin_e2m1_from_bits, lo, hi, step, first_bad);
}

PIN_EXPORT int64_t pin_sweep_e4m3(enc_fn oracle, uint64_t lo, uint64_t hi, uint64_t step,
                                  uint32_t* first_bad) {
    return sweep(oracle, pin_e4m3_from_bits, lo, hi, step, first_bad);
}
