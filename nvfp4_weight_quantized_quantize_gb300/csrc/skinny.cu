// skinny.cu -- W4A16 NVFP4 skinny GEMM for 2 <= M <= 16 (MTP verify: drafts + 1 rows of x
// against the same weights).  FlashRT docs/qwen36_usage.md
// (generate_own_speculative_KN_nvfp4 argument table: verify runs K + 1 tokens at once).
//
//   y[m, n] = gw * sum_b s[n, b] * sum_{k in b} x[m, k] * e2m1(q[n, k])
//
// Bound by HBM (each weight is read once for all M rows of x), so the kernel streams W the
// way the M = 1 kernel does, and does the arithmetic on the tensor cores:
//   - one CTA per SM owns a contiguous run of 16-row groups; a producer warp fills a ring
//     of stages (up to four 16-row groups each: their codes and their row-major scale
//     bytes, two bulk copies, mbarrier-gated, bounded waits);
//   - consumer warp w owns the K columns [w CG, (w+1) CG) (CG = 4 U chunks of 32) for the
//     whole kernel, so its slice of x -- the B fragments of mma.sync m16n8k16, fp16 after a
//     per-token power-of-two rescale -- is built once and stays in registers;
//   - per stage and 128-element unit, a lane of quad t takes 16-byte chunk 4u + t of rows g
//     and g + 8; MMA j (0..7) takes elements 4j .. 4j+3 of those chunks for its k-slots
//     {2t, 2t+1, 2t+8, 2t+9} (any bijection works when A and B use the same one), with the
//     block scale folded into A (e2m1 * e4m3 is exact in fp16);
//   - each warp leaves its 16 x 8 partial tile of a row group in a per-stage slot; the warp
//     whose arrival completes the row group's count adds the slots in warp order
//     (deterministic) and writes the 16 rows of y.  No warp waits for another.
// x values that fp16 cannot hold exactly after the rescale (more than about 2^31 below
// the token's maximum) make every warp add the exact fp32 residual of its slice.
// 9 to 16 tokens (NT = 2) take one pass over W: each A fragment (the dequantized,
// scale-folded weights) feeds two MMAs, tokens 0..7 from registers and tokens 8..15 from
// the lane's own slots in shared memory (the register file cannot hold both tiles of x);
// at most 15 consumer warps, so that a thread may keep 128 registers.
// W4A4 with a static activation scale (the kXQ instantiations): each lane first quantizes
// its chunks of x to NVFP4 and keeps e2m1 * e4m3, which the rescale carries exactly.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "nvfp4.h"
#include "common.cuh"
#include "gemv_helpers.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kSkMaxGroups = 23;  // consumer warps, at most (plus the producer: 768 threads)
constexpr int kSkMaxThreads = (kSkMaxGroups + 1) * 32;
constexpr int kSkRows = 16;           // rows of an mma row group
constexpr int kSkMaxRgs = 4;          // row groups per stage, at most
constexpr int kSkStageTarget = 80 * 1024;  // bytes of codes per stage

// a stage: rgs row groups of codes, then their row-major scale bytes
__host__ __device__ __forceinline__ size_t sk_stage_bytes(int K, int rgs) {
    const size_t rows = (size_t)kSkRows * rgs;
    return ((rows * (K / 2) + rows * (K / 16) + 32) + 127) & ~(size_t)127;
}

// slot area of one stage: per row group, ngroups partial tiles of 16 rows x 8 NT tokens
// (fp32)
__host__ __device__ __forceinline__ size_t sk_slot_bytes(int ngroups, int rgs, int nt) {
    return (size_t)rgs * ngroups * kSkRows * 8 * nt * 4;
}

// the second token tile's B fragments (tokens 8..15), per consumer warp: U x 8 MMAs x 32
// lanes x 8 bytes
__host__ __device__ __forceinline__ size_t sk_x2_bytes(int ngroups, int u, int nt) {
    return nt == 2 ? (size_t)ngroups * u * 8 * 32 * 8 + 16 : 0;  // (+ alignment slack)
}

__host__ __device__ __forceinline__ size_t sk_smem(int K, int ngroups, int stages, int rgs,
                                                   int u, int nt) {
    return (size_t)stages * (sk_stage_bytes(K, rgs) + sk_slot_bytes(ngroups, rgs, nt)) +
           (size_t)stages * (8 + 8 + 4 * kSkMaxRgs) +  // full, empty barriers; row-group counters
           sk_x2_bytes(ngroups, u, nt);
}

// two token tiles hold twice the accumulators and read the second tile's fragments from
// shared memory: at most 16 warps, so that each thread may keep 128 registers
constexpr int kSk2MaxGroups = 15;

template <int U, bool kXQ, int NT>
__global__ void __launch_bounds__(NT == 2 ? (kSk2MaxGroups + 1) * 32 : kSkMaxThreads, 1)
skinny_pipe_kernel(const uint16_t* __restrict__ x, int M, int K, const uint8_t* __restrict__ wq,
                   const uint8_t* __restrict__ wrm, const float* __restrict__ gw,
                   const float* __restrict__ gx, int N, void* __restrict__ y, int y_bf16,
                   int stages, int rgs, int w_static, uint32_t* __restrict__ err) {
    constexpr int CG = 4 * U;  // 16-byte chunks (32 elements) of K per consumer warp
    constexpr int TT = 8 * NT;  // tokens of a partial tile
    static_assert(NT == 1 || !kXQ, "two token tiles only for bf16 x");
    extern __shared__ __align__(128) uint8_t smem[];
    const int rowchunks = K >> 5;
    const int ngroups = (rowchunks + CG - 1) / CG;
    const size_t st_bytes = sk_stage_bytes(K, rgs);
    const size_t sl_bytes = sk_slot_bytes(ngroups, rgs, NT);
    const int srows = kSkRows * rgs;  // rows of a full stage
    uint8_t* ring = smem;
    float* slots = reinterpret_cast<float*>(smem + (size_t)stages * st_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)stages * (st_bytes + sl_bytes));
    uint64_t* empty = full + stages;
    int* cnt = reinterpret_cast<int*>(empty + stages);
    // tokens 8..15 (NT = 2): each lane's B fragments, [warp][u][mma j][lane]
    uint2* x2 = reinterpret_cast<uint2*>(
        smem + (((size_t)stages * (st_bytes + sl_bytes) + (size_t)stages * (8 + 8 + 4 * kSkMaxRgs) +
                 15) & ~(size_t)15));
    __shared__ volatile int abort_flag;
    __shared__ int e_w[kSkMaxGroups][TT];    // per consumer warp and token: the exponent
    __shared__ float u_w[kSkMaxGroups][TT];  // and 2^-e

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nrg_all = (N + kSkRows - 1) / kSkRows;
    const int rg0 = (int)((int64_t)nrg_all * blockIdx.x / gridDim.x);
    const int rg1 = (int)((int64_t)nrg_all * (blockIdx.x + 1) / gridDim.x);
    const int nst = (rg1 - rg0 + rgs - 1) / rgs;
    const int64_t r_end = min((int64_t)N, (int64_t)rg1 * kSkRows);  // this CTA's rows end
    const int64_t rowb = K >> 1, rows_sb = K >> 4;  // code and scale bytes per row

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], ngroups);
            for (int r = 0; r < kSkMaxRgs; ++r) cnt[s * kSkMaxRgs + r] = 0;
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == ngroups) {
        // ---- producer ----
        if (lane == 0) {
            // the first ring's worth of codes heads for L2 while the previous kernel on the
            // stream may still run; every read that lands in shared memory comes after the
            // wait for it.  Weight copies are marked evict-first, so that x and y stay in L2.
            if (!w_static) {  // static weights stream before the wait
                for (int it = 0; it < min(nst, stages); ++it) {
                    const int64_t rbeg = (int64_t)rg0 * kSkRows + (int64_t)it * srows;
                    prefetch_l2(wq + rbeg * rowb,
                                (uint32_t)(min((int64_t)srows, r_end - rbeg) * rowb));
                }
                pdl_wait_prior_grid();
            }
            const uint64_t pol = l2_evict_first_policy();
            int issued = 0;
            for (int it = 0; it < nst; ++it) {
                const int s = it % stages;
                if (it >= stages &&
                    !mbar_wait_bounded(&empty[s], ((it / stages) - 1) & 1, kWaitLimitNs)) {
                    if (err) atomicOr(err, NVFP4_DEVERR_TIMEOUT);
                    abort_flag = 1;
                    break;
                }
                if (abort_flag) break;
                const int64_t rbeg = (int64_t)rg0 * kSkRows + (int64_t)it * srows;
                const int nr = (int)min((int64_t)srows, r_end - rbeg);
                const uint32_t wbytes = (uint32_t)(nr * rowb);
                // scale bytes of these rows, copied from a 16-byte boundary
                const int64_t s_lo = (rbeg * rows_sb) & ~(int64_t)15;
                const int64_t s_hi = ((rbeg + nr) * rows_sb + 15) & ~(int64_t)15;
                mbar_arrive_expect_tx(&full[s], wbytes + (uint32_t)(s_hi - s_lo));
                uint8_t* st = ring + (size_t)s * st_bytes;
                bulk_g2s_hint(st, wq + rbeg * rowb, wbytes, &full[s], pol);
                bulk_g2s_hint(st + (size_t)srows * rowb, wrm + s_lo, (uint32_t)(s_hi - s_lo),
                              &full[s], pol);
                issued = it + 1;
            }
            // every copy of this CTA is in flight: the next kernel on the stream may now be
            // scheduled
            pdl_launch_dependents();
            // every copy this thread issued has landed before the CTA can exit
            for (int it = max(0, issued - stages); it < issued; ++it)
                mbar_wait_bounded(&full[it % stages], (it / stages) & 1, kWaitLimitNs);
        }
        return;
    }

    // ---- consumers: this warp's slice of x in registers, an exponent per token ----
    // Every (token, chunk) pair belongs to exactly one consumer thread (token g, chunk
    // w CG + 4u + t), so one pass of loads gives the B fragments and, reduced over the four
    // threads of each token, the token's largest and smallest nonzero magnitude in this
    // warp's K slice.  The warp scales each token's slice by its own 2^e (largest magnitude
    // in [2^14, 2^15)) and each partial tile column back by 2^-e before it leaves the warp:
    // no reduction over the CTA, no barrier.  A bf16 value is exact in fp16 after the
    // rescale from 2^-17 upward; a warp with a value below that takes the residual path.
    pdl_wait_prior_grid();
    // the warp's K slice, rotated by the CTA index so that the CTAs, which all read the
    // whole of x at the same moment, start on different parts of it
    const int wk = (warp + (int)(blockIdx.x % (unsigned)ngroups)) % ngroups;
    const int cbase = wk * CG + t;  // this lane's first chunk
    // tokens 8..15 (NT = 2), first, so that their raw values are dead before the first
    // tile's fragments are built: the same steps as for the first tile below, for token
    // g + 8; the B fragments go to this lane's slots in shared memory, read back by the same
    // lane
    float ua2 = 1.0f, ub2 = 1.0f;
    bool inexact2_any = false;
    if constexpr (NT == 2) {
        uint2 raw[U][8];
        float am2 = 0.0f, mn2 = __int_as_float(0x7f800000);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = cbase + 4 * u;
            const bool ok = g + 8 < M && c < rowchunks;
            const uint4* xp = reinterpret_cast<const uint4*>(x + (int64_t)(g + 8) * K + 32 * c);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 v = ok ? xp[q] : make_uint4(0u, 0u, 0u, 0u);
                raw[u][2 * q] = make_uint2(v.x, v.y);
                raw[u][2 * q + 1] = make_uint2(v.z, v.w);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t w2[2] = {raw[u][j].x, raw[u][j].y};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float a = fabsf(bf16_to_f32(w2[h] & 0xFFFFu));
                    const float b = fabsf(bf16_to_f32(w2[h] >> 16));
                    am2 = fmaxf(am2, fmaxf(a, b));
                    if (a > 0.0f) mn2 = fminf(mn2, a);
                    if (b > 0.0f) mn2 = fminf(mn2, b);
                }
            }
        am2 = fmaxf(am2, __shfl_xor_sync(0xffffffffu, am2, 1));
        am2 = fmaxf(am2, __shfl_xor_sync(0xffffffffu, am2, 2));
        mn2 = fminf(mn2, __shfl_xor_sync(0xffffffffu, mn2, 1));
        mn2 = fminf(mn2, __shfl_xor_sync(0xffffffffu, mn2, 2));
        const int eg2 = chunk_exponent(am2);
        inexact2_any = __any_sync(0xffffffffu, times_pow2(mn2, eg2) < 7.62939453125e-06f);
        {
            const int em = __shfl_sync(0xffffffffu, eg2, 4 * (lane & 7));
            if (lane < 8) {
                e_w[warp][8 + lane] = em;
                u_w[warp][8 + lane] = times_pow2(1.0f, -em);
            }
            __syncwarp();
        }
        ua2 = u_w[warp][8 + 2 * t];
        ub2 = u_w[warp][8 + 2 * t + 1];
        bool inexact2 = false;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                x2[((warp * U + u) * 8 + j) * 32 + lane] =
                    make_uint2(to_h2_scaled(raw[u][j].x, eg2, inexact2),
                               to_h2_scaled(raw[u][j].y, eg2, inexact2));
    }
    uint2 raw[U][8];
    float am = 0.0f, mn = __int_as_float(0x7f800000);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = cbase + 4 * u;
        const bool ok = g < M && c < rowchunks;
        const uint4* xp = reinterpret_cast<const uint4*>(x + (int64_t)g * K + 32 * c);
        // the chunk's 64 bytes in four 16-byte loads (x is 16-byte aligned, K % 32 == 0)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = ok ? xp[q] : make_uint4(0u, 0u, 0u, 0u);
            raw[u][2 * q] = make_uint2(v.x, v.y);
            raw[u][2 * q + 1] = make_uint2(v.z, v.w);
        }
    }
    if constexpr (kXQ) {
        // W4A4 with a static activation scale: each chunk's two blocks quantized here
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                v[q] = make_uint4(raw[u][2 * q].x, raw[u][2 * q].y, raw[u][2 * q + 1].x,
                                  raw[u][2 * q + 1].y);
            quantize_chunk_static(v, *gx);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                raw[u][2 * q] = make_uint2(v[q].x, v[q].y);
                raw[u][2 * q + 1] = make_uint2(v[q].z, v[q].w);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t w2[2] = {raw[u][j].x, raw[u][j].y};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float a = fabsf(bf16_to_f32(w2[h] & 0xFFFFu));
                const float b = fabsf(bf16_to_f32(w2[h] >> 16));
                am = fmaxf(am, fmaxf(a, b));
                if (a > 0.0f) mn = fminf(mn, a);
                if (b > 0.0f) mn = fminf(mn, b);
            }
        }
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 2));
    const int eg = chunk_exponent(am);  // token g's exponent in this warp
    // (e2m1 * e4m3 values span less than 2^22: never inexact after the rescale)
    const bool any_inexact =
        __any_sync(0xffffffffu, !kXQ && times_pow2(mn, eg) < 7.62939453125e-06f) || inexact2_any;
    // every token's exponent and 2^-e in this warp (token m's lanes are 4m .. 4m + 3), in
    // the warp's own shared-memory row
    {
        const int em = __shfl_sync(0xffffffffu, eg, 4 * (lane & 7));
        if (lane < 8) {
            e_w[warp][lane] = em;
            u_w[warp][lane] = times_pow2(1.0f, -em);
        }
        __syncwarp();
    }
    // the columns this lane holds in the accumulator: tokens 2t and 2t + 1
    const float ua = u_w[warp][2 * t], ub = u_w[warp][2 * t + 1];

    // B fragment (unit u, mma j): b0 = token g, elements 4j, 4j+1 of chunk c; b1 = elements
    // 4j+2, 4j+3 (k-slots 2t, 2t+1 and 2t+8, 2t+9)
    uint32_t bf[U][8][2];
    bool inexact = false;  // (decided for the warp above)
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            bf[u][j][0] = to_h2_scaled(raw[u][j].x, eg, inexact);
            bf[u][j][1] = to_h2_scaled(raw[u][j].y, eg, inexact);
        }
    const float gscale = *gw * (gx ? *gx : 1.0f);

    for (int it = 0; it < nst; ++it) {
        const int s = it % stages;
        // the wait's outcome and the abort flag are made warp-uniform before they steer
        // control flow: mma.sync and the shuffles below are warp-collective
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (it / stages) & 1,
                                                                  kWaitLimitNs));
        if (!ok) {
            if (err && lane == 0) atomicOr(err, NVFP4_DEVERR_TIMEOUT);
            abort_flag = 1;
        }
        if (__any_sync(0xffffffffu, abort_flag != 0)) break;
        const uint8_t* st = ring + (size_t)s * st_bytes;
        const int64_t sbeg = (int64_t)rg0 * kSkRows + (int64_t)it * srows;
        const int snr = (int)min((int64_t)srows, r_end - sbeg);  // rows in this stage
        const uint8_t* sst = st + (size_t)srows * rowb + ((sbeg * rows_sb) & 15);
        const int nrgi = (snr + kSkRows - 1) / kSkRows;
        for (int rgi = 0; rgi < nrgi; ++rgi) {
            const int nr = min(kSkRows, snr - kSkRows * rgi);
            const uint8_t* sw = st + (size_t)(kSkRows * rgi) * rowb;
            const uint8_t* ss = sst + (size_t)(kSkRows * rgi) * rows_sb;
            const bool rga = g < nr, rgb = g + 8 < nr;  // rows past N hold stale bytes
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            float d2[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // tokens 8..15 (NT = 2)
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = cbase + 4 * u;
                const bool cv = c < rowchunks;
                const uint4 wa = (cv && rga) ? *reinterpret_cast<const uint4*>(sw + (size_t)g * rowb + 16 * c)
                                             : make_uint4(0u, 0u, 0u, 0u);
                const uint4 wb = (cv && rgb) ? *reinterpret_cast<const uint4*>(sw + (size_t)(g + 8) * rowb + 16 * c)
                                             : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t sa = (cv && rga) ? *reinterpret_cast<const uint16_t*>(ss + (size_t)g * rows_sb + 2 * c) : 0u;
                const uint32_t sb = (cv && rgb) ? *reinterpret_cast<const uint16_t*>(ss + (size_t)(g + 8) * rows_sb + 2 * c) : 0u;
                // block scales of the chunk (blocks 2c, 2c+1) as f16, each in both halves
                const uint32_t ha = cvt_e4m3x2_f16x2(sa), hb = cvt_e4m3x2_f16x2(sb);
                const uint32_t sa0 = __byte_perm(ha, 0, 0x1010), sa1 = __byte_perm(ha, 0, 0x3232);
                const uint32_t sb0 = __byte_perm(hb, 0, 0x1010), sb1 = __byte_perm(hb, 0, 0x3232);
                const uint32_t wa4[4] = {wa.x, wa.y, wa.z, wa.w};
                const uint32_t wb4[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // word q of each chunk: bytes 4q .. 4q+3 = elements 8q .. 8q+7 (block q / 2),
                    // the A registers of MMAs 2q and 2q+1
                    uint32_t ha[4], hb[4];
                    cvt8(wa4[q], ha);
                    cvt8(wb4[q], hb);
                    const uint32_t sca = q < 2 ? sa0 : sa1, scb = q < 2 ? sb0 : sb1;
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int j = 2 * q + jj;
                        const uint32_t a0 = hmul2(ha[2 * jj], sca), a2 = hmul2(ha[2 * jj + 1], sca);
                        const uint32_t a1 = hmul2(hb[2 * jj], scb), a3 = hmul2(hb[2 * jj + 1], scb);
                        asm volatile(
                            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
                            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(bf[u][j][0]), "r"(bf[u][j][1]));
                        if constexpr (NT == 2) {
                            // the same A fragment against tokens 8..15
                            const uint2 b2 = x2[((warp * U + u) * 8 + j) * 32 + lane];
                            asm volatile(
                                "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
                                "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                                : "+f"(d2[0]), "+f"(d2[1]), "+f"(d2[2]), "+f"(d2[3])
                                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b2.x), "r"(b2.y));
                        }
                    }
                }
            }
            // this warp's partial tile of the row group: slot[row][token], row g / g + 8,
            // tokens 2t, 2t+1 (and 8 + 2t, 8 + 2t + 1)
            float* tiles = slots + ((size_t)s * rgs + rgi) * ngroups * (kSkRows * TT);
            float* mine = tiles + (size_t)warp * (kSkRows * TT);
            mine[g * TT + 2 * t] = d[0] * ua;
            mine[g * TT + 2 * t + 1] = d[1] * ub;
            mine[(g + 8) * TT + 2 * t] = d[2] * ua;
            mine[(g + 8) * TT + 2 * t + 1] = d[3] * ub;
            if constexpr (NT == 2) {
                mine[g * TT + 8 + 2 * t] = d2[0] * ua2;
                mine[g * TT + 8 + 2 * t + 1] = d2[1] * ub2;
                mine[(g + 8) * TT + 8 + 2 * t] = d2[2] * ua2;
                mine[(g + 8) * TT + 8 + 2 * t + 1] = d2[3] * ub2;
            }
            if (any_inexact) {
                // exact residual x' - fp16(x') of this warp's K slice (slow path, rare): lane l
                // takes row l % 16 and tokens l / 16, l / 16 + 2, ...
                __syncwarp();
                const int r = lane & 15;
                if (r < nr) {
                    for (int m = lane >> 4; m < M; m += 2) {
                        float q = 0.0f;
                        for (int c = cbase - t; c < min(rowchunks, cbase - t + CG); ++c) {
                            const uint32_t s2 = *reinterpret_cast<const uint16_t*>(ss + (size_t)r * rows_sb + 2 * c);
                            for (int k = 0; k < 32; ++k) {
                                const uint32_t byte = sw[(size_t)r * rowb + 16 * c + (k >> 1)];
                                const uint32_t code = (k & 1) ? (byte >> 4) : (byte & 15u);
                                const float sc = e4m3_to_f32(k < 16 ? (s2 & 0xFFu) : (s2 >> 8));
                                q = fmaf(residual(x[(int64_t)m * K + 32 * c + k], e_w[warp][m]),
                                         e2m1_to_f32(code) * sc, q);
                            }
                        }
                        mine[r * TT + m] += q * u_w[warp][m];
                    }
                }
            }
            // count this warp in; the arrival that completes the row group adds its partial
            // tiles in warp order (every slot's loads in flight together) and writes its 16
            // rows of y
            __threadfence_block();
            __syncwarp();
            int* c_rg = &cnt[s * kSkMaxRgs + rgi];
            int old = 0;
            if (lane == 0) old = atomicAdd(c_rg, 1);
            if (__shfl_sync(0xffffffffu, old, 0) == ngroups - 1) {
                __threadfence_block();
                float v[4 * NT];
#pragma unroll
                for (int i = 0; i < 4 * NT; ++i) v[i] = 0.0f;
                const float* base = tiles + lane;
#pragma unroll
                for (int w = 0; w < kSkMaxGroups; ++w)
                    if (w < ngroups) {
#pragma unroll
                        for (int i = 0; i < 4 * NT; ++i)
                            v[i] += base[(size_t)w * (kSkRows * TT) + 32 * i];
                    }
                __syncwarp();
                if (lane == 0) *c_rg = 0;
                const int64_t rbeg = sbeg + kSkRows * rgi;
#pragma unroll
                for (int i = 0; i < 4 * NT; ++i) {
                    const int e = lane + 32 * i, r = e / TT, m = e % TT;
                    if (r < nr && m < M)
                        store_y(y, (int64_t)m * N + rbeg + r, v[i] * gscale, y_bf16);
                }
            }
        }
        // the stage (codes and partial tiles) is free once every warp has passed here
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

}  // namespace

namespace {

template <int U, bool kXQ, int NT>
cudaError_t launch_skinny_u(const uint16_t* x, int M, int K, const uint8_t* wq,
                            const uint8_t* wrm, const float* gw, const float* gx, int N, void* y,
                            bool y_bf16, uint32_t* err, bool w_static, cudaStream_t stream,
                            const DevInfo& dev, bool* launched) {
    *launched = false;
    const int rowchunks = K / 32;
    const int ngroups = (rowchunks + 4 * U - 1) / (4 * U);
    int grid = dev.sm_count;
    const int nrg = (N + kSkRows - 1) / kSkRows;
    if (grid > nrg) grid = nrg;
    // row groups per stage: about kSkStageTarget bytes of codes, but no fewer than four
    // stages per CTA where the CTA's rows allow, so that short slices still pipeline
    const size_t rg_bytes = (size_t)kSkRows * (K / 2);
    int rgs = (int)std::max<size_t>(1, kSkStageTarget / rg_bytes);
    rgs = std::min(rgs, std::max(1, (nrg / grid) / 4));
    rgs = std::min(rgs, kSkMaxRgs);
    // the deepest ring (2..6 stages) that fits one CTA per SM; fewer row groups per
    // stage where two stages of rgs do not fit
    int stages = 6;
    for (;;) {
        stages = 6;
        while (stages > 2 && sk_smem(K, ngroups, stages, rgs, U, NT) + 2048 > dev.smem_optin)
            --stages;
        if (sk_smem(K, ngroups, stages, rgs, U, NT) + 2048 <= dev.smem_optin || rgs == 1) break;
        --rgs;
    }
    const size_t smem = sk_smem(K, ngroups, stages, rgs, U, NT);
    if (smem + 2048 > dev.smem_optin) return cudaSuccess;
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = 1ull << (dev.device & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, skinny_pipe_kernel<U, kXQ, NT>);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(skinny_pipe_kernel<U, kXQ, NT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(dev.smem_optin - fa.sharedSizeBytes));
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, skinny_pipe_kernel<U, kXQ, NT>, x, M, K, wq, wrm, gw, gx, N,
                                       y, y_bf16 ? 1 : 0, stages, rgs, w_static ? 1 : 0,
                                       err);
    *launched = true;
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool skinny_w4a16_takes(int K, const DevInfo& dev) {
    const int rowchunks = K / 32;
    const int cg = (rowchunks + 3) / 4 <= kSkMaxGroups ? 4 : 8;  // chunks per warp (U = 1, 2)
    const int ngroups = (rowchunks + cg - 1) / cg;
    if (ngroups > kSkMaxGroups) return false;
    return sk_smem(K, ngroups, 2, 1, cg / 4, 1) + 2048 <= dev.smem_optin;  // the smallest ring
}

// chunks of K per consumer warp of the two-tile kernel: 8, 12 or 16 (at most
// kSk2MaxGroups warps); 0 when none fits
int sk2_chunks_per_warp(int K) {
    const int rowchunks = K / 32;
    for (int cg = 8; cg <= 16; cg += 4)
        if ((rowchunks + cg - 1) / cg <= kSk2MaxGroups) return cg;
    return 0;
}

bool skinny16_w4a16_takes(int K, const DevInfo& dev) {
    const int cg = sk2_chunks_per_warp(K);
    if (cg == 0) return false;
    const int ngroups = (K / 32 + cg - 1) / cg;
    return sk_smem(K, ngroups, 2, 1, cg / 4, 2) + 2048 <= dev.smem_optin;
}

cudaError_t launch_skinny_w4a16(const uint16_t* x, int M, int K, const uint8_t* wq,
                                const uint8_t* wrm, const float* gw, const float* gx, int N,
                                void* y, bool y_bf16, uint32_t* err, bool w_static,
                                cudaStream_t stream, const DevInfo& dev, bool* launched,
                                bool x_quant_static) {
    *launched = false;
    if (M < 2 || M > 16 || (x_quant_static && M > 8)) return cudaSuccess;
    const int rowchunks = K / 32;
    if (x_quant_static) {
        if ((rowchunks + 3) / 4 <= kSkMaxGroups)
            return launch_skinny_u<1, true, 1>(x, M, K, wq, wrm, gw, gx, N, y, y_bf16, err,
                                               w_static, stream, dev, launched);
        if ((rowchunks + 7) / 8 <= kSkMaxGroups)
            return launch_skinny_u<2, true, 1>(x, M, K, wq, wrm, gw, gx, N, y, y_bf16, err,
                                               w_static, stream, dev, launched);
        return cudaSuccess;
    }
    // at most kSkMaxGroups consumer warps: 4 or 8 chunks of K per warp; 9..16 tokens in two
    // token tiles over one pass of W
    if (M > 8) {
        switch (sk2_chunks_per_warp(K)) {
            case 8:
                return launch_skinny_u<2, false, 2>(x, M, K, wq, wrm, gw, gx, N, y, y_bf16, err,
                                                    w_static, stream, dev, launched);
            case 12:
                return launch_skinny_u<3, false, 2>(x, M, K, wq, wrm, gw, gx, N, y, y_bf16, err,
                                                    w_static, stream, dev, launched);
            case 16:
                return launch_skinny_u<4, false, 2>(x, M, K, wq, wrm, gw, gx, N, y, y_bf16, err,
                                                    w_static, stream, dev, launched);
            default:
                return cudaSuccess;
        }
    }
    if ((rowchunks + 3) / 4 <= kSkMaxGroups)
        return launch_skinny_u<1, false, 1>(x, M, K, wq, wrm, gw, gx, N, y, y_bf16, err,
                                            w_static, stream, dev, launched);
    if ((rowchunks + 7) / 8 <= kSkMaxGroups)
        return launch_skinny_u<2, false, 1>(x, M, K, wq, wrm, gw, gx, N, y, y_bf16, err,
                                            w_static, stream, dev, launched);
    return cudaSuccess;
}

}  // namespace nvfp4
