// gemv_tc.cu -- W4A16 NVFP4 GEMV (M = 1) on the block-scaled tensor cores: the decode
// projection.  Qwen3x-Orin README (quick start, "--projection-backend sm87"): decode
// streams every weight once per token, so the kernel's only job is to keep HBM busy.
//
//   y[n] = gw * (gx ? gx : 1) * sum_b s[n, b] * sum_{k in b} x[k] * e2m1(q[n, k])
//
// The CUDA-core GEMV spends about one instruction per weight on dequantization and
// multiply-adds, which at the HBM rate is close to the SM's issue limit.  Here the packed
// weights and their E4M3 block scales go from HBM (TMA) straight into
// tcgen05.mma kind::mxf4nvf4, which multiplies E2M1 codes with 16-element UE4M3 block
// scales in hardware.  The bf16 vector x is not an E2M1 operand, so it is written as an
// exact sum of 16 E2M1 "digit planes", the 16 columns of the MMA's B operand:
//
//   per 16-element block b of x: E_b = floor(log2 max_b |x|) - 1 (so |x| < 4 * 2^E_b),
//   F_k = |x_k| * 2^(30 - E_b) (an integer below 2^32 when exact),
//   digit_j(k) = bits 31-2j and 30-2j of F_k, j = 0 .. 15 (values 0 .. 3),
//   x_k = sign_k * sum_j digit_j(k) * 2^(E_b - 2j).
//
// Plane j holds E2M1 codes sign | digit (the values 0, 0.5, 1, 1.5 = digit / 2) with block
// scale 2^(E_b - G) (UE4M3, exact) for a per-CTA reference exponent G, so
//
//   sum_k w_k x_k = 2^(G + 1) * sum_j 4^-j * D_j,   D_j = the MMA's column j.
//
// A bf16 value is exact in this form when its lowest significand bit is at or above
// 2^(E_b - 30), i.e. when it is within 2^-24 of its block's largest magnitude (and the
// block is within 2^-17 of the CTA's largest block).  The few elements that are not (and
// non-finite ones) are flagged; the epilogue adds their exact residual x_k - xhat_k times
// the dequantized weight from global memory, so the result never depends on the
// decomposition.
//
// Work split: unit = (128-row tile of W, 256-element K step); the units are cut evenly
// over one CTA per SM (at most kMaxGrid CTAs), each CTA a contiguous range (stream-K
// everywhere).  A CTA's range is at most two partial tiles plus whole ones; a partial
// tile's 128 results go to one of the CTA's two workspace slots and the last CTA of the
// tile (per 32-row quarter, counters that wrap back to zero) adds the slots in CTA order.
// Warp roles (10 warps):
//   warp 0      TMA producer: per unit the 128 x 128-byte code box (128-byte swizzle) and
//               the unit's 4 W scale atoms (bulk copy), kStages deep;
//   warp 1      TMEM allocation and, from one thread, 4 MMAs (128 x 16 x 64) per unit into
//               one of two 16-column fp32 accumulators;
//   warps 2-9   first the digit planes of x for the CTA's K steps (shared memory, B
//               operand layout), then
//   warps 2-5   epilogue: 16 columns -> one fp32 per row, residual fixes, y or a slot;
//   warps 6-9   scale writers: each unit's W atoms and x block scales -> TMEM.
// Every wait is bounded; on time-out the kernel sets NVFP4_DEVERR_TIMEOUT and stops.
#include <cuda.h>

#include <atomic>
#include <climits>

#include "gemv_helpers.cuh"
#include "tcgen05.cuh"

namespace nvfp4 {
namespace {

constexpr int kTerms = 16;        // digit planes of x (MMA N)
constexpr int kBN = 128;          // W rows per tile (MMA M)
constexpr int kHalf = 256;        // K of one 128-byte swizzle row of codes
constexpr int kBK = 2 * kHalf;    // K per unit
constexpr int kMmas = kBK / 64;   // MMAs per unit (K = 64 each)
constexpr int kStages = 5;
constexpr int kThreads = 10 * 32;
constexpr int kGenWarp0 = 2, kGenWarps = 8;
constexpr int kSfWarp0 = 6;
constexpr int kMaxSlots = 10;     // units' K ranges whose digit planes a CTA holds
constexpr int kMaxGrid = 160;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSf = 2 * kTerms;          // scale area after the two accumulators
constexpr uint32_t kSfColsPerStage = 8 * kMmas;   // 4 W atom columns + 4 x columns per MMA

constexpr uint32_t kBoxBytes = kBN * kHalf / 2;   // one TMA box: 128 rows x 128 bytes
constexpr uint32_t kABytes = 2 * kBoxBytes;       // 32 KB of codes per unit
constexpr uint32_t kPlaneHalfBytes = kTerms * kHalf / 2;  // 16 plane rows x 128 bytes
constexpr uint32_t kDigitBytes = 2 * kPlaneHalfBytes;     // 4 KB of x planes per slot
constexpr uint32_t kAtomBytes = 512;
constexpr uint32_t kSfaBytes = kMmas * kAtomBytes;
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffD = kOffA + kStages * kABytes;
constexpr uint32_t kOffSfa = kOffD + kMaxSlots * kDigitBytes;
constexpr uint32_t kOffSfb = kOffSfa + kStages * kSfaBytes;    // UE4M3 x block scales
constexpr uint32_t kOffEb = kOffSfb + kMaxSlots * 32;          // int8 E_b - G per block
constexpr uint32_t kOffMask = kOffEb + kMaxSlots * 32;         // inexact elements, 1 bit each
constexpr uint32_t kOffFlag = kOffMask + kMaxSlots * 64;       // a slot has inexact elements
constexpr uint32_t kOffBar = kOffFlag + kMaxSlots * 4;
constexpr uint32_t kNumBars = 3 * kStages + 4 + 1 + kMaxSlots;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment

static_assert(kTmemSf + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
static_assert(kOffD % 1024 == 0 && kOffSfa % 16 == 0 && kOffSfb % 16 == 0 &&
                  kOffBar % 8 == 0, "alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// block-scaled kind: E2M1 A and B, UE4M3 scales, dense K = 64, K-major, fp32 D, 128 x 16
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kTerms >> 3) << 17) |
                            ((uint32_t)(kBN >> 4) << 24);

// ---- the digit planes --------------------------------------------------------------------

// floor(log2 |v|) of a nonzero finite bf16 magnitude u (bits without the sign)
__device__ __forceinline__ int bf16_floor_log2(uint32_t u) {
    const uint32_t ef = u >> 7;
    return ef ? (int)ef - 127 : (31 - __clz((int)(u & 0x7Fu))) - 133;
}

// F = |x| * 2^(30 - ep), truncated; *inexact when bits were lost or x is not finite.
// Branch-free: |x| = m * 2^(e - 7) with an 8-bit significand m (7 bits for subnormals).
__device__ __forceinline__ uint32_t fixed_point(uint32_t bits, int ep, bool& inexact) {
    const uint32_t u = bits & 0x7FFFu, ef = u >> 7;
    const bool nonfinite = ef == 0xFFu;
    const uint32_t m = nonfinite ? 0u : (ef ? ((u & 0x7Fu) | 0x80u) : (u & 0x7Fu));
    const int sh = (ef ? (int)ef - 134 : -133) + 30 - ep;  // <= 24 since |x| < 2^(ep + 2)
    const int rs = min(-sh, 31);                           // m < 2^8: m >> 31 == 0
    const uint32_t F = sh >= 0 ? m << (sh & 31) : m >> rs;
    const uint32_t lost = sh >= 0 ? 0u : m & ((1u << rs) - 1u);
    inexact |= nonfinite | (lost != 0u);
    return F;
}

// 8 two-bit cells of x (bits 0..15) -> 8 four-bit cells (bits 4c, 4c + 1)
__device__ __forceinline__ uint32_t spread2to4(uint32_t x) {
    x = (x | (x << 8)) & 0x00FF00FFu;
    x = (x | (x << 4)) & 0x0F0F0F0Fu;
    x = (x | (x << 2)) & 0x33333333u;
    return x;
}

// transpose of an 8 x 8 matrix of 4-bit cells: a[i] nibble p <-> a[p] nibble i
__device__ __forceinline__ void transpose8x8_nibbles(uint32_t (&a)[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t t = ((a[i] >> 16) ^ a[i + 4]) & 0x0000FFFFu;
        a[i + 4] ^= t;
        a[i] ^= t << 16;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if ((i & 2) == 0) {
            const uint32_t t = ((a[i] >> 8) ^ a[i + 2]) & 0x00FF00FFu;
            a[i + 2] ^= t;
            a[i] ^= t << 8;
        }
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const uint32_t t = ((a[i] >> 4) ^ a[i + 1]) & 0x0F0F0F0Fu;
        a[i + 1] ^= t;
        a[i] ^= t << 4;
    }
}

// largest finite magnitude bits of 8 bf16 values (non-finite ones count as zero)
__device__ __forceinline__ uint32_t max_mag8(const uint32_t (&w)[4]) {
    uint32_t mx = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = w[i] & 0x7FFFu, hi = (w[i] >> 16) & 0x7FFFu;
        mx = max(mx, lo >= 0x7F80u ? 0u : lo);
        mx = max(mx, hi >= 0x7F80u ? 0u : hi);
    }
    return mx;
}

// E2M1 value of one code nibble times an E4M3 scale byte (exact)
__device__ __forceinline__ float wdeq(uint32_t code, uint32_t s8) {
    return e2m1_to_f32(code) * e4m3_to_f32(s8);
}

struct Range {
    int64_t u0, u1;  // units [u0, u1)
};

__device__ __forceinline__ Range cta_range(int64_t units, int c, int grid) {
    return Range{units * c / grid, units * (c + 1) / grid};
}

// the CTA whose range holds unit u
__device__ __forceinline__ int cta_of(int64_t u, int64_t units, int grid) {
    return (int)(((u + 1) * grid - 1) / units);
}

// the CTA's units as (tile, K steps [kb0, kb1)) segments
struct SegIter {
    int64_t u, u1;
    int nkb;
    __device__ bool next(int& tile, int& kb0, int& kb1) {
        if (u >= u1) return false;
        tile = (int)(u / nkb);
        kb0 = (int)(u % nkb);
        kb1 = (int)min((int64_t)nkb, kb0 + (u1 - u));
        u += kb1 - kb0;
        return true;
    }
};

// UE4M3 byte of 2^e, e in [-9, 8]
__device__ __forceinline__ uint32_t ue4m3_pow2(int e) {
    return e >= -6 ? (uint32_t)(e + 7) << 3 : 1u << (e + 9);
}

__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// atomicInc with release (this thread's and its warp's earlier stores) and acquire
// (every store released before the increments it follows) at GPU scope
__device__ __forceinline__ uint32_t atom_inc_acq_rel(uint32_t* p, uint32_t wrap) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(wrap)
                 : "memory");
    return old;
}

__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const uint16_t* __restrict__ x,
               const uint8_t* __restrict__ wq, const uint8_t* __restrict__ wsz,
               const uint8_t* __restrict__ wrm, const float* __restrict__ gw,
               const float* __restrict__ gx, void* __restrict__ y, int y_bf16, int K, int N,
               int nkb, int natoms_row, int64_t units, int w_static, uint32_t* __restrict__ err,
               uint32_t* __restrict__ counters, float* __restrict__ slots) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const uint32_t bar0 = base_s + kOffBar;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto sfull = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
    auto accfull = [&](int b) { return bar0 + 8u * (3 * kStages + b); };
    auto accempty = [&](int b) { return bar0 + 8u * (3 * kStages + 2 + b); };
    const uint32_t drain = bar0 + 8u * (3 * kStages + 4);
    auto ready = [&](int sl) { return bar0 + 8u * (3 * kStages + 5 + sl); };
    auto bar_ptr = [&](uint32_t a) { return reinterpret_cast<uint64_t*>(base + (a - base_s)); };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + kOffMisc + 4);
    int* emax = reinterpret_cast<int*>(base + kOffMisc + 8);
    uint8_t* sfb_bytes = base + kOffSfb;
    int8_t* ebt = reinterpret_cast<int8_t*>(base + kOffEb);
    uint32_t* mask = reinterpret_cast<uint32_t*>(base + kOffMask);
    volatile int* flagged = reinterpret_cast<volatile int*>(base + kOffFlag);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Range rg = cta_range(units, blockIdx.x, gridDim.x);
    // the CTA's units cover the K steps kb_first, kb_first + 1, ... (cyclically), one
    // slot of digit planes each
    const int kb_first = (int)(rg.u0 % nkb);
    const int nslots = (int)min((int64_t)nkb, rg.u1 - rg.u0);
    auto slot_of = [&](int kb) { return kb >= kb_first ? kb - kb_first : kb + nkb - kb_first; };
    auto atoms_of = [&](int kb) { return min(kMmas, natoms_row - kMmas * kb); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_ptr(full(s)), 1);
            mbar_init(bar_ptr(empty(s)), 1);
            mbar_init(bar_ptr(sfull(s)), 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_ptr(accfull(b)), 1);
            mbar_init(bar_ptr(accempty(b)), 4);
        }
        mbar_init(bar_ptr(drain), 1);
        for (int sl = 0; sl < kMaxSlots; ++sl) mbar_init(bar_ptr(ready(sl)), 1);
        *abort_flag = 0;
        *emax = INT_MIN;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < nslots * 16; i += kThreads) mask[i] = 0u;
    for (int i = threadIdx.x; i < nslots; i += kThreads) flagged[i] = 0;
    if (warp == 1) tc::tmem_alloc(base_s + kOffMisc, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            // Unless the caller declared the weights static (no kernel still in flight before
            // this one writes them), the first ring's worth of code boxes only heads for L2
            // while the previous kernel on the stream may still run (L2 is the point of
            // coherence: a prefetch cannot see stale data), and every copy into shared
            // memory comes after the wait.  Static weights stream from the start.
            if (!w_static) {
                for (int64_t u = rg.u0; u < rg.u1 && u < rg.u0 + kStages; ++u)
                    for (int h = 0; h < 2; ++h)
                        tma_prefetch_2d(&tmap_w, (int)(u % nkb) * (kBK / 2) + h * (kHalf / 2),
                                        (int)(u / nkb) * kBN);
                pdl_wait_prior_grid();
            }
            int64_t it = 0, issued = 0;
            int t = (int)(rg.u0 / nkb), kb = kb_first, s = 0;
            uint32_t ph = 0;
            for (int64_t u = rg.u0; u < rg.u1 && !*abort_flag; ++u, ++it) {
                if (it >= kStages && !tc::wait_or_abort(empty(s), ph ^ 1u, abort_flag, err)) break;
                const uint32_t sfa = (uint32_t)atoms_of(kb) * kAtomBytes;
                mbar_arrive_expect_tx(bar_ptr(full(s)), kABytes + sfa);
                const uint32_t a_s = base_s + kOffA + s * kABytes;
                tc::tma_load_2d(a_s, &tmap_w, kb * (kBK / 2), t * kBN, full(s));
                tc::tma_load_2d(a_s + kBoxBytes, &tmap_w, kb * (kBK / 2) + kHalf / 2, t * kBN,
                                full(s));
                bulk_g2s(base + kOffSfa + s * kSfaBytes,
                         wsz + ((size_t)t * natoms_row + kMmas * kb) * kAtomBytes, sfa,
                         bar_ptr(full(s)));
                issued = it + 1;
                if (++kb == nkb) { kb = 0; ++t; }
                if (++s == kStages) { s = 0; ph ^= 1u; }
            }
            // every copy of this CTA is in flight: the next kernel on the stream may launch
            pdl_launch_dependents();
            // every copy issued has landed before the CTA moves on to exit
            for (int64_t i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                mbar_wait_bounded(bar_ptr(full((int)(i % kStages))), (uint32_t)(i / kStages) & 1u,
                                  kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issue ----------------
        if (lane == 0) {
            bool ok = true;
            int s = 0, lt = 0, tile, kb0, kb1;
            uint32_t ph = 0;
            int slots_ready = 0;
            SegIter si{rg.u0, rg.u1, nkb};
            while (ok && si.next(tile, kb0, kb1)) {
                const int b = lt & 1;
                if (lt >= 2 &&
                    !tc::wait_or_abort(accempty(b), (uint32_t)((lt >> 1) - 1) & 1u, abort_flag, err))
                    break;
                tc::fence_after();
                const uint32_t d = tmem + (uint32_t)(b * kTerms);
                for (int kb = kb0; kb < kb1; ++kb) {
                    const int sl = slot_of(kb);
                    if (sl >= slots_ready) {
                        // first use of this K step's planes
                        if (!tc::wait_or_abort(ready(sl), 0, abort_flag, err)) { ok = false; break; }
                        slots_ready = sl + 1;
                    }
                    if (!tc::wait_or_abort(full(s), ph, abort_flag, err) ||
                        !tc::wait_or_abort(sfull(s), ph, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const int na = atoms_of(kb);
                    const uint32_t sf = tmem + kTmemSf + (uint32_t)s * kSfColsPerStage;
                    // descriptors advance by 32 bytes (2 in the address field) per MMA
                    // inside a 128-byte row, and by a whole box / plane tile per half
                    const uint64_t a0 = tc::sw128_desc(base_s + kOffA + s * kABytes);
                    const uint64_t b0 = tc::sw128_desc(base_s + kOffD + (uint32_t)sl * kDigitBytes);
#pragma unroll
                    for (int j = 0; j < kMmas; ++j) {
                        if (j >= na) break;
                        const uint64_t da = a0 + (uint64_t)((j >> 2) * (kBoxBytes >> 4) + 2 * (j & 3));
                        const uint64_t db =
                            b0 + (uint64_t)((j >> 2) * (kPlaneHalfBytes >> 4) + 2 * (j & 3));
                        tc::mma_mxf4nvf4(d, da, db, kIdesc, sf + 4 * j, sf + 4 * kMmas + 4 * j,
                                         (kb != kb0 || j != 0) ? 1u : 0u);
                    }
                    tc::commit(empty(s));
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc::commit(accfull(b));
                ++lt;
            }
            // MMAs in flight complete before TMEM is freed
            tc::commit(drain);
            mbar_wait_bounded(bar_ptr(drain), 0, kWaitLimitNs);
        }
    } else {
        // ---------------- warps 2-9: the digit planes of x ----------------
        const int gwarp = warp - kGenWarp0;
        pdl_wait_prior_grid();
        // lane l takes elements 8l .. 8l + 7 of a 256-element half (one 32-bit word of each
        // plane row); lanes 2i, 2i + 1 share block i
        auto load8 = [&](int sl, int h, uint32_t (&w)[4]) {
            const int kb = kb_first + sl < nkb ? kb_first + sl : kb_first + sl - nkb;
            const int64_t k0 = (int64_t)kb * kBK + h * kHalf + 8 * lane;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (k0 < K) v = *reinterpret_cast<const uint4*>(x + k0);
            w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
        };
        // pass 1: the CTA's largest block exponent; this warp's x stays in registers
        // (slots gwarp and gwarp + 8)
        static_assert(kMaxSlots <= 2 * kGenWarps, "two slots per generator warp");
        uint32_t xw[2][2][4];
        uint32_t bmax[2][2];
        int mymax = INT_MIN;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int sl = gwarp + i * kGenWarps;
                if (sl < nslots) {
                    load8(sl, h, xw[i][h]);
                } else {
                    xw[i][h][0] = xw[i][h][1] = xw[i][h][2] = xw[i][h][3] = 0u;
                }
                uint32_t mx = max_mag8(xw[i][h]);
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                bmax[i][h] = mx;
                if (mx) mymax = max(mymax, bf16_floor_log2(mx) - 1);
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mymax = max(mymax, __shfl_xor_sync(0xffffffffu, mymax, o));
        if (lane == 0 && mymax != INT_MIN) atomicMax(emax, mymax);
        named_bar_sync(1, kGenWarps * 32);
        const int G = *emax == INT_MIN ? 0 : *emax - 8;
        // pass 2: per slot, both halves, then the slot is released to the MMA
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int sl = gwarp + i * kGenWarps;
            if (sl >= nslots) break;
            bool any = false;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t (&w)[4] = xw[i][h];
                const uint32_t mx = bmax[i][h];
                const int ep = max(mx ? bf16_floor_log2(mx) - 1 : G - 9, G - 9);
                uint32_t hi[8], lo[8], sgn = 0u, p = 0u;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t bits = (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
                    bool ie = false;
                    const uint32_t F = fixed_point(bits, ep, ie);
                    p |= (uint32_t)ie << i;
                    sgn |= (bits >> 15) << (4 * i + 3);
                    hi[i] = spread2to4(F >> 16);
                    lo[i] = spread2to4(F & 0xFFFFu);
                }
                transpose8x8_nibbles(hi);
                transpose8x8_nibbles(lo);
                // plane j is row j of the half's B tile (K-major, 128-byte swizzle): this
                // lane's word is bytes 4l .. 4l + 3 of the row, in 16-byte chunk l / 4
                uint8_t* tile = base + kOffD + (size_t)sl * kDigitBytes + h * kPlaneHalfBytes;
                const uint32_t chunk = lane >> 2, within = (lane & 3) * 4;
#pragma unroll
                for (int j = 0; j < kTerms; ++j) {
                    const uint32_t r = j & 7;
                    const uint32_t word = (j < 8 ? hi[7 - j] : lo[15 - j]) | sgn;
                    *reinterpret_cast<uint32_t*>(tile + (j >> 3) * 1024 + r * 128 +
                                                 ((chunk ^ r) << 4) + within) = word;
                }
                if ((lane & 1) == 0) {
                    const int blk = sl * 32 + h * 16 + (lane >> 1);
                    ebt[blk] = (int8_t)(ep - G);
                    sfb_bytes[blk] = (uint8_t)ue4m3_pow2(ep - G);
                }
                if (p) {
                    atomicOr(&mask[sl * 16 + h * 8 + (lane >> 2)], p << (8 * (lane & 3)));
                    any = true;
                }
            }
            if (__any_sync(0xffffffffu, any) && lane == 0) flagged[sl] = 1;
            // the planes are read by the tensor cores (async proxy)
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::arrive(ready(sl));
        }

        if (warp >= kSfWarp0) {
            // ---------------- scale writers ----------------
            const int q = warp & 3;  // TMEM lane quarter this warp may access
            int s = 0, kb = kb_first, slots_ready = 0;
            uint32_t ph = 0;
            for (int64_t u = rg.u0; u < rg.u1; ++u) {
                const int sl = slot_of(kb);
                bool ok = true;
                if (sl >= slots_ready) {
                    ok = tc::wait_or_abort(ready(sl), 0, abort_flag, err);
                    slots_ready = sl + 1;
                }
                ok = ok && tc::wait_or_abort(full(s), ph, abort_flag, err);
                if (!__all_sync(0xffffffffu, ok)) break;
                // columns 4j .. 4j + 3: row (lane) of W atom j; 32 + 4j .. 32 + 4j + 3: the x
                // block scales of MMA j (the same for every plane, so every atom row and
                // every 4-byte group holds them)
                const uint8_t* sa = base + kOffSfa + s * kSfaBytes + lane * 16;
                const uint4* sb = reinterpret_cast<const uint4*>(sfb_bytes + sl * 32);
                uint32_t v[32];
#pragma unroll
                for (int j = 0; j < kMmas; ++j) {
                    const uint4 a = *reinterpret_cast<const uint4*>(sa + j * kAtomBytes);
                    v[4 * j] = a.x; v[4 * j + 1] = a.y; v[4 * j + 2] = a.z; v[4 * j + 3] = a.w;
                }
                const uint32_t col = tmem + ((uint32_t)(q * 32) << 16) + kTmemSf +
                                     (uint32_t)s * kSfColsPerStage;
                tc::tmem_st32(col, v);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint4 e4 = sb[i];
                    const uint32_t e[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        v[16 * i + 4 * j] = e[j]; v[16 * i + 4 * j + 1] = e[j];
                        v[16 * i + 4 * j + 2] = e[j]; v[16 * i + 4 * j + 3] = e[j];
                    }
                }
                tc::tmem_st32(col + 4 * kMmas, v);
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::arrive(sfull(s));
                if (++kb == nkb) kb = 0;
                if (++s == kStages) { s = 0; ph ^= 1u; }
            }
        } else {
            // ---------------- epilogue ----------------
            const int q = warp & 3;  // TMEM lane quarter this warp may access
            const int row = 32 * q + lane;
            const float g = *gw * (gx ? *gx : 1.0f);
            const int e1 = (G + 1) / 2, e2 = (G + 1) - (G + 1) / 2;  // 2^(G+1) = 2^e1 * 2^e2
            const float f1 = exp2i(e1), f2 = exp2i(e2);
            const int64_t rowb = K >> 1, rows_sb = K >> 4;
            // the slots' flags, masks and exponents, once (the MMAs wait for them anyway)
            bool tables = true;
            for (int sl = 0; sl < nslots; ++sl)
                tables = tables && tc::wait_or_abort(ready(sl), 0, abort_flag, err);
            int lt = 0, tile, kb0, kb1;
            SegIter si{rg.u0, rg.u1, nkb};
            while (si.next(tile, kb0, kb1)) {
                const int b = lt & 1;
                if (!__all_sync(0xffffffffu, tc::wait_or_abort(accfull(b), (uint32_t)(lt >> 1) & 1u,
                                                               abort_flag, err)))
                    break;
                tc::fence_after();
                uint32_t v[16];
                tc::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * kTerms), v);
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::arrive(accempty(b));
                float acc = __uint_as_float(v[kTerms - 1]);
#pragma unroll
                for (int j = kTerms - 2; j >= 0; --j) acc = fmaf(acc, 0.25f, __uint_as_float(v[j]));
                float pv = acc * f1 * f2;
                const int64_t grow = (int64_t)tile * kBN + row;
                // exact residual of the flagged elements of these K steps (rare); their slots
                // are ready: the MMAs that used them have completed
                float r_sum = 0.0f;
                for (int kb = kb0; tables && kb < kb1; ++kb) {
                    const int sl = slot_of(kb);
                    if (!flagged[sl] || grow >= N) continue;
                    for (int wd = 0; wd < 16; ++wd) {
                        uint32_t bits = mask[sl * 16 + wd];
                        while (bits) {
                            const int bpos = __ffs((int)bits) - 1;
                            bits &= bits - 1u;
                            const int kk = wd * 32 + bpos;
                            const int64_t k = (int64_t)kb * kBK + kk;
                            const uint32_t xb = x[k];
                            const int ep = G + ebt[sl * 32 + (kk >> 4)];
                            bool dummy = false;
                            float xhat = ldexpf((float)fixed_point(xb, ep, dummy), ep - 30);
                            if (xb >> 15) xhat = -xhat;
                            const float r = bf16_to_f32(xb) - xhat;
                            const uint32_t byte = wq[grow * rowb + (k >> 1)];
                            const uint32_t code = (k & 1) ? (byte >> 4) : (byte & 15u);
                            r_sum = fmaf(r, wdeq(code, wrm[grow * rows_sb + (k >> 4)]), r_sum);
                        }
                    }
                }
                pv = (pv + r_sum) * g;
                const int c_first = cta_of((int64_t)tile * nkb, units, gridDim.x);
                const int c_last = cta_of((int64_t)tile * nkb + nkb - 1, units, gridDim.x);
                if (c_first == c_last) {
                    if (grow < N) store_y(y, grow, pv, y_bf16);
                } else {
                    // slot 0: the CTA's first segment, slot 1: its last
                    const int mine = tile == (int)(rg.u0 / nkb) ? 0 : 1;
                    slots[((size_t)blockIdx.x * 2 + mine) * kBN + row] = pv;
                    // the warp's 32 stores are ordered before lane 0's release; the count
                    // wraps back to zero after the last of the tile's CTAs
                    __syncwarp();
                    const uint32_t nseg = (uint32_t)(c_last - c_first + 1);
                    uint32_t old = 0u;
                    if (lane == 0) old = atom_inc_acq_rel(&counters[(size_t)tile * 4 + q], nseg - 1u);
                    old = __shfl_sync(0xffffffffu, old, 0);
                    if (old == nseg - 1u) {
                        // the last of the tile's CTAs (lane 0 acquired every CTA's slot
                        // stores): add the slots in CTA order
                        __syncwarp();
                        float sum = 0.0f;
                        for (int c = c_first; c <= c_last; ++c) {
                            const int64_t cu0 = units * c / gridDim.x;
                            const int sl = tile == (int)(cu0 / nkb) ? 0 : 1;
                            sum += __ldcg(&slots[((size_t)c * 2 + sl) * kBN + row]);
                        }
                        if (grow < N) store_y(y, grow, sum, y_bf16);
                    }
                }
                ++lt;
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t gemv_tc_workspace_bytes(int64_t K, int64_t N) {
    (void)K;
    return kGemmHeaderBytes + tc::counters_bytes((N + kBN - 1) / kBN) +
           (size_t)kMaxGrid * 2 * kBN * sizeof(float);
}

cudaError_t launch_gemv_tc(const uint16_t* x, int K, const uint8_t* wq, const uint8_t* wsz_all,
                           const float* gw, const float* gx, int N, void* y, bool y_bf16,
                           uint8_t* workspace, bool w_static, cudaStream_t stream,
                           const DevInfo& dev, bool* launched) {
    *launched = false;
    if (!workspace || dev.smem_optin < kSmemBytes || K % 32 != 0) return cudaSuccess;
    const int nkb = (K + kBK - 1) / kBK;
    const int64_t ntiles = ((int64_t)N + kBN - 1) / kBN;
    const int64_t units = ntiles * nkb;
    int grid = dev.sm_count < kMaxGrid ? dev.sm_count : kMaxGrid;
    if (grid > units) grid = (int)units;
    // the x planes of a CTA's K steps must fit in shared memory
    const int64_t per_cta = (units + grid - 1) / grid;
    if ((per_cta < nkb ? per_cta : nkb) > kMaxSlots) return cudaSuccess;
    CUtensorMap mw;
    cudaError_t e = tc::make_map_2d(&mw, wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2,
                                    (uint64_t)N, kHalf / 2, kBN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = 1ull << (dev.device & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const int natoms_row = (K + 63) / 64;  // scale atoms per 128-row block
    // the row-major copy of the scales follows the atoms
    const uint8_t* wrm = wsz_all + (size_t)ntiles * 128 * ((K / 16 + 3) / 4 * 4);
    uint32_t* err = reinterpret_cast<uint32_t*>(workspace);
    uint32_t* counters = reinterpret_cast<uint32_t*>(workspace + kGemmHeaderBytes);
    float* slots = reinterpret_cast<float*>(workspace + kGemmHeaderBytes +
                                            tc::counters_bytes(ntiles));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemv_tc_kernel, mw, x, wq, wsz_all, wrm, gw, gx, y,
                           y_bf16 ? 1 : 0, K, N, nkb, natoms_row, units, w_static ? 1 : 0, err,
                           counters, slots);
    *launched = true;
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace nvfp4
