// gemm_w4a16.cu -- W4A16 NVFP4 GEMM for M > 16 (prefill chunks) on the 5th-generation
// tensor cores.  Qwen3x-Orin README (quick start: prefill in chunks of up to 512 tokens
// through the NVFP4 projection backend); FlashRT docs/qwen36_usage.md
// (FLASHRT_QWEN36_FUSE_MLP_GATE_UP: the gate/up projection as one NVFP4 GEMM).
//
//   y[m, n] = gw * sum_k x[m, k] * (e2m1(q[n, k]) * e4m3(s[n, k / 16]))
//
// e2m1 * e4m3 has at most 5 significant bits and lies in [2^-10, 2688], so the
// dequantized weight (without gw) is exact in bf16: the kernel dequantizes W tiles to
// bf16 in shared memory and runs bf16 x bf16 -> fp32 tcgen05.mma (kind::f16); gw is
// applied to the fp32 accumulator in the epilogue.
//
// CTA tile: 128 rows of W (the MMA's M) x 256 rows of x (the MMA's N), K in steps of 64.
// Persistent CTAs (one per SM) walk the tiles; warp roles:
//   warp 0      TMA producer: per K step one 64 x 256 bf16 box of x (128-byte swizzle),
//               one 32-byte x 128-row box of packed codes, one 512-byte scale atom
//               (the tensor-core scale layout stores one atom per 128 rows x 64 K);
//   warp 1      allocates TMEM (512 columns: two fp32 accumulators of 128 x 256) and
//               issues the MMAs from one thread (4 x 128x256x16 per K step);
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (each warp its 32 TMEM lanes),
//               x gw, store y (fp32 or bf16, rows and columns past M, N masked);
//   warps 6-13  dequantize: each thread one (W row, 32-wide K half) per step, e2m1 ->
//               f16 (hardware converter) -> f32 x scale -> bf16, written in the 128-byte
//               swizzled K-major layout the MMA descriptor names.
// Work split: tiles beyond the last full wave (all tiles when there are fewer tiles than
// SMs) go stream-K: their (tile, K step) iterations are cut into equal contiguous ranges,
// one per CTA, so every SM gets the same number of MMAs.  A range that covers a tile only
// in part leaves an fp32 partial tile in one of the CTA's two workspace slots; per quarter
// of the tile (one epilogue warp each), the warp whose arrival completes the count
// (atomicInc on a per-quarter counter, which wraps back to zero) adds the partials in
// segment order -- a fixed order, so results are deterministic -- and writes y.  No CTA
// or warp waits for another.  The remaining full waves of
// tiles are split plainly, one tile at a time.
// Ring of kStages stages (mbarriers: full = TMA bytes landed, afull = dequantized tile
// written, empty = the stage's MMAs completed); accumulators double-buffered so the
// epilogue of one tile overlaps the main loop of the next.  Out-of-range rows and K
// columns come from the TMA zero fill (and the zero-padded scale atoms).  Every wait is
// bounded in wall time: on expiry the kernel sets NVFP4_DEVERR_TIMEOUT in the error word,
// every role stops, copies and MMAs in flight are waited for, and TMEM is freed.
#include <cuda.h>
#include <cuda_fp16.h>

#include <atomic>

#include "silu.cuh"
#include "tcgen05.cuh"

namespace nvfp4 {
namespace {

constexpr int kBN = 128;   // W rows per tile (MMA M)
constexpr int kBM = 256;   // x rows per tile (MMA N)
constexpr int kBK = 64;    // K per stage (one 128-byte swizzle row of bf16)
constexpr int kStages = 4;
constexpr int kThreads = 14 * 32;
constexpr int kDequantWarp0 = 6;
constexpr int kDequantWarps = 8;
constexpr int kEpiWarp0 = 2;
constexpr int kTmemCols = 512;

constexpr uint32_t kXBytes = kBM * kBK * 2;       // 32 KB
constexpr uint32_t kABytes = kBN * kBK * 2;       // 16 KB
constexpr uint32_t kCodeBytes = kBN * kBK / 2;    // 4 KB
constexpr uint32_t kAtomBytes = 512;              // one 128 x 4 scale atom
constexpr uint32_t kFixBars = 4 * 16;             // stream-K fix-up chunk barriers, 16 per epilogue warp

// Shared-memory layout.  The fused gate/up variant takes two scale atoms per stage (the
// gate rows' and the up rows' 128-row blocks) and two exchange tiles through which the
// gate warps of the epilogue hand silu(gate) to the up warps (32 x 33 floats each).
template <bool kFuse>
struct Smem {
    static constexpr uint32_t kScaleBytes = kFuse ? 2 * kAtomBytes : kAtomBytes;
    static constexpr uint32_t kOffX = 0;
    static constexpr uint32_t kOffA = kOffX + kStages * kXBytes;
    static constexpr uint32_t kOffCode = kOffA + kStages * kABytes;
    static constexpr uint32_t kOffScale = kOffCode + kStages * kCodeBytes;
    static constexpr uint32_t kOffXch = kOffScale + kStages * kScaleBytes;
    static constexpr uint32_t kXchBytes = kFuse ? 2 * 32 * 33 * 4 : 0;
    static constexpr uint32_t kOffBar = kOffXch + kXchBytes;
    static constexpr uint32_t kNumBars = 3 * kStages + 4 + 1 + kFixBars;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kUsed = kOffMisc + 16;
    static constexpr uint32_t kBytes = kUsed + 1024;  // slack for 1024-byte alignment
};

// The stream-K fix-up of a CTA's last work item stages partials in the idle stage ring:
// a quarter of it per epilogue warp, in 4 KB chunk buffers.
constexpr uint32_t kFixupBytes = (Smem<false>::kOffBar / 4) & ~127u;
constexpr int kFixupBufs = (int)(kFixupBytes / 4096) < 16 ? (int)(kFixupBytes / 4096) : 16;
static_assert(kFixupBufs >= 2, "fix-up staging");

// Instruction descriptor, kind::f16: fp32 D, bf16 A and B, both K-major, M x N.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            ((uint32_t)(kBM >> 3) << 17) | ((uint32_t)(kBN >> 4) << 24);

// f16x2 codes times an f16 scale -> bf16x2: the products (mixed f16 x f16 -> f32 FMA with a
// zero addend) are exact in f32, and in bf16 (at most 5 significant bits, in [2^-10, 2688])
__device__ __forceinline__ uint32_t deq_bf16x2(uint32_t h2, uint32_t s16) {
    uint32_t d;
    asm("{\n .reg .f16 a0, a1, s;\n .reg .f32 p0, p1;\n mov.b32 {a0, a1}, %1;\n"
        " mov.b32 {s, _}, %2;\n fma.rn.f32.f16 p0, a0, s, 0f00000000;\n"
        " fma.rn.f32.f16 p1, a1, s, 0f00000000;\n cvt.rn.bf16x2.f32 %0, p1, p0;\n}\n"
        : "=r"(d) : "r"(h2), "r"(s16));
    return d;
}

// Arguments of the fused gate/up variant (unused by the plain GEMM).  W is the stacked
// [gate; up] weight [2I, K]; the CTA tile of work item nb takes gate rows 64 nb .. 64 nb + 63
// as its W rows 0..63 and the matching up rows I + 64 nb .. as rows 64..127, so that the
// epilogue holds gate and up of the same columns of h.
struct FuseArgs {
    int I = 0;                       // columns of h; I % 128 == 0
    const float* gh = nullptr;       // static global scale of h (device)
    uint8_t* hq = nullptr;           // h codes [M, I/2]
    uint8_t* hs = nullptr;           // h scale atoms (rows padded to 128, blocks to 4)
};

// Row pitch (floats) of the exchange tiles: 32 values plus one, so that a warp writing a
// row and a warp reading a column both touch 32 distinct banks.
constexpr int kXchPitch = 33;

// The fused gate/up epilogue for 32 accumulator columns (32 rows m of x) of a tile.  TMEM
// lanes 0..63 hold gate columns 64 nb + l of h, lanes 64..127 the up columns; warps q = 0, 1
// hold gate (their 32 lanes each), warps q = 2, 3 up, for the same 32 columns of h (q & 1).
// `a` is this warp's raw fp32 accumulator for rows c0 .. c0 + 31 (one value per row, for its
// lane's column).  Each gate/up warp pair shares an exchange tile [m][i] and splits the
// work in halves, all values first rounded to bf16 as gw * acc (the gate/up GEMM's output):
//   1. the gate warp takes silu of rows 0..15 itself and hands rows 16..31 of raw gate to
//      the up warp through the tile;
//   2. the up warp forms h = silu(g) * u for rows 16..31; the gate warp puts its silu
//      values of rows 0..15 in the tile;
//   3. the up warp multiplies rows 0..15 by their up values;
//   4. lane l of each warp quantizes one 16-element block of row m = l -- columns 0..15
//      by the gate warp, 16..31 by the up warp -- with the quantizer's one-thread block
//      rule and the static global scale: 8 bytes of codes and a scale byte each.
// Rows past M get no codes; their scale bytes inside the last 128-row block are zero.  All
// four epilogue warps call it for the same c0 (it meets at named barrier 1).
__device__ __forceinline__ void fused_rows32(const float (&a)[32], int q, int lane, int mb,
                                             int c0, int ibase, float gw, float g,
                                             const FuseArgs& fa, float* xw, int M, int m_pad,
                                             int64_t cp4) {
    const bool gate = q < 2;
    const int hb = gate ? 0 : 1;  // the 16-column block this warp quantizes
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = bf16_to_f32(f32_to_bf16_rne(a[j] * gw));
    if (gate) {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = silu_f32_nobranch(v[j]);
#pragma unroll
        for (int j = 16; j < 32; ++j) xw[j * kXchPitch + lane] = v[j];
    }
    named_bar_sync(1, 128);
    if (gate) {
#pragma unroll
        for (int j = 0; j < 16; ++j) xw[j * kXchPitch + lane] = v[j];
    } else {
#pragma unroll
        for (int j = 16; j < 32; ++j)
            xw[j * kXchPitch + lane] = __fmul_rn(silu_f32_nobranch(xw[j * kXchPitch + lane]), v[j]);
    }
    named_bar_sync(1, 128);
    if (!gate) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            xw[j * kXchPitch + lane] = __fmul_rn(xw[j * kXchPitch + lane], v[j]);
    }
    named_bar_sync(1, 128);
    const int m = mb * kBM + c0 + lane;
    if (m < m_pad) {
        float t[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) t[k] = xw[lane * kXchPitch + 16 * hb + k];
        uint32_t lo, hi;
        const uint32_t s8 = quantize_block16(t, g, lo, hi);
        // the block is scale column ibase/16 + hb of the atom
        uint8_t* sp = fa.hs + swizzle_offset(m, ibase / 16 + hb, cp4);
        if (m < M) {
            *reinterpret_cast<uint2*>(fa.hq + (int64_t)m * (fa.I / 2) + ibase / 2 + 8 * hb) =
                make_uint2(lo, hi);
            *sp = (uint8_t)s8;
        } else {
            *sp = 0;
        }
    }
    named_bar_sync(1, 128);
}

// Epilogue of one whole tile of the fused gate/up variant (see fused_rows32).
__device__ __forceinline__ void epilogue_silu_quant(uint32_t acc, int q, int lane, int tile,
                                                    int ntiles_m, float gw, const FuseArgs& fa,
                                                    float* xch, int M) {
    const int nb = tile / ntiles_m, mb = tile % ntiles_m;
    const uint32_t taddr = acc + ((uint32_t)(q * 32) << 16);
    const float g = *fa.gh;
    const int64_t cp4 = (fa.I / 16 + 3) / 4;
    const int m_pad = (M + 127) / 128 * 128;
    const int ibase = nb * 64 + (q & 1) * 32;   // this warp pair's 32 columns of h
    float* xw = xch + (q & 1) * 32 * kXchPitch;
#pragma unroll 1
    for (int c0 = 0; c0 < kBM; c0 += 32) {
        uint32_t u[32];
        tc::tmem_ld32(taddr + c0, u);
        float a[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) a[j] = __uint_as_float(u[j]);
        fused_rows32(a, q, lane, mb, c0, ibase, gw, g, fa, xw, M, m_pad, cp4);
    }
}

// Epilogue of a stream-K segment of a fused tile.  Each warp writes its quarter of the
// partial accumulator to the CTA's slot (the layout of tc::epilogue_work) and releases
// the accumulator; the four warps then count the segment once for the tile (one counter
// per tile, wrapping back to zero).  The CTA whose count completes the tile sums every
// segment's partials in segment order (a fixed order: deterministic) 32 rows at a time and
// runs the fused activation on the sums.  *last is a shared word the four warps meet on.
__device__ __forceinline__ void epilogue_silu_quant_sk(uint32_t acc, int q, int lane, int tile,
                                                       int ntiles_m, int nkb, int p_sk,
                                                       int64_t tsk, float gw,
                                                       const FuseArgs& fa, float* xch, int M,
                                                       uint32_t accempty, float* slots,
                                                       uint32_t* counters,
                                                       volatile uint32_t* last) {
    constexpr size_t kSlotFloats = (size_t)kBN * kBM;
    const uint32_t taddr = acc + ((uint32_t)(q * 32) << 16);
    const int64_t t0 = (int64_t)tile * nkb;
    const int cf = tc::sk_cta_of(t0, p_sk, tsk), cl = tc::sk_cta_of(t0 + nkb - 1, p_sk, tsk);
    float* mine = slots + (size_t)tc::sk_slot(blockIdx.x, t0, p_sk, tsk) * kSlotFloats +
                  tc::slot_chunk<kBM>(q, 0) + lane;
#pragma unroll 1
    for (int c0 = 0; c0 < kBM; c0 += 32) {
        uint32_t u[32];
        tc::tmem_ld32(taddr + c0, u);
#pragma unroll
        for (int j = 0; j < 32; ++j) mine[(size_t)(c0 + j) * 32] = __uint_as_float(u[j]);
    }
    tc::fence_before();
    __syncwarp();
    if (lane == 0) tc::arrive(accempty);
    __threadfence();
    named_bar_sync(1, 128);  // all four quarters are in the slot
    if (q == 0 && lane == 0)
        *last = atomicInc(&counters[tile * 4], (unsigned)(cl - cf)) == (unsigned)(cl - cf);
    named_bar_sync(1, 128);
    const bool is_last = *last != 0;
    named_bar_sync(1, 128);  // every warp has read the flag before it is written again
    if (!is_last) return;
    __threadfence();
    const int nb = tile / ntiles_m, mb = tile % ntiles_m;
    const float g = *fa.gh;
    const int64_t cp4 = (fa.I / 16 + 3) / 4;
    const int m_pad = (M + 127) / 128 * 128;
    const int ibase = nb * 64 + (q & 1) * 32;
    float* xw = xch + (q & 1) * 32 * kXchPitch;
#pragma unroll 1
    for (int c0 = 0; c0 < kBM; c0 += 32) {
        float a[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) a[j] = 0.0f;
#pragma unroll 1
        for (int cs = cf; cs <= cl; ++cs) {
            const float* sp = slots + (size_t)tc::sk_slot(cs, t0, p_sk, tsk) * kSlotFloats +
                              tc::slot_chunk<kBM>(q, c0) + lane;
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __ldcg(sp + (size_t)j * 32);
#pragma unroll
            for (int j = 0; j < 32; ++j) a[j] += v[j];
        }
        fused_rows32(a, q, lane, mb, c0, ibase, gw, g, fa, xw, M, m_pad, cp4);
    }
}

template <bool kFuse>
__global__ void __launch_bounds__(kThreads, 1)
gemm_w4a16_kernel(const __grid_constant__ CUtensorMap tmap_x,
                  const __grid_constant__ CUtensorMap tmap_w, const uint8_t* __restrict__ wsz,
                  const float* __restrict__ gw, void* __restrict__ y, int y_bf16, int M, int N,
                  int nkb, int ntiles_m, int ntiles, int ntiles_sk, int p_sk, int64_t tsk,
                  uint32_t* __restrict__ err, uint32_t* __restrict__ counters,
                  float* __restrict__ slots, FuseArgs fa, WaitCfg dbg) {
    using L = Smem<kFuse>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const uint32_t bar0 = base_s + L::kOffBar;
    // barrier addresses (shared space)
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto afull = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto empty = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
    auto accfull = [&](int b) { return bar0 + 8u * (3 * kStages + b); };
    auto accempty = [&](int b) { return bar0 + 8u * (3 * kStages + 2 + b); };
    const uint32_t drain = bar0 + 8u * (3 * kStages + 4);
    const uint32_t fixbar0 = bar0 + 8u * (3 * kStages + 5);  // 16 per epilogue warp
    auto bar_ptr = [&](uint32_t a) { return reinterpret_cast<uint64_t*>(base + (a - base_s)); };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + L::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_ptr(full(s)), 1);
            mbar_init(bar_ptr(afull(s)), kDequantWarps);
            mbar_init(bar_ptr(empty(s)), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_ptr(accfull(b)), 1);
            mbar_init(bar_ptr(accempty(b)), 4);
        }
        mbar_init(bar_ptr(drain), 1);
        for (uint32_t i = 0; i < kFixBars; ++i) mbar_init(bar_ptr(fixbar0 + 8u * i), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc(base_s + L::kOffMisc, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int it = 0, issued = 0;
            tc::WorkIter wi = tc::make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
            int tile, kb0, kb1;
            while (!*abort_flag && wi.next(tile, kb0, kb1)) {
                const int nb = tile / ntiles_m, mb = tile % ntiles_m;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages &&
                        !tc::wait_or_abort(empty(s), ((it / kStages) - 1) & 1, abort_flag, err, dbg.wait_ns))
                        break;
                    mbar_arrive_expect_tx(bar_ptr(full(s)),
                                          kXBytes + kCodeBytes + L::kScaleBytes);
                    tc::tma_load_2d(base_s + L::kOffX + s * kXBytes, &tmap_x, kb * kBK, mb * kBM,
                                    full(s));
                    uint8_t* sc = base + L::kOffScale + s * L::kScaleBytes;
                    if constexpr (kFuse) {
                        // 64 gate rows, then the 64 matching up rows; the scale atoms of
                        // their two 128-row blocks (I % 128 == 0)
                        const uint32_t cs = base_s + L::kOffCode + s * kCodeBytes;
                        tc::tma_load_2d(cs, &tmap_w, kb * (kBK / 2), nb * 64, full(s));
                        tc::tma_load_2d(cs + kCodeBytes / 2, &tmap_w, kb * (kBK / 2),
                                        fa.I + nb * 64, full(s));
                        bulk_g2s(sc, wsz + ((size_t)(nb >> 1) * nkb + kb) * kAtomBytes,
                                 kAtomBytes, bar_ptr(full(s)));
                        bulk_g2s(sc + kAtomBytes,
                                 wsz + ((size_t)(fa.I / 128 + (nb >> 1)) * nkb + kb) * kAtomBytes,
                                 kAtomBytes, bar_ptr(full(s)));
                    } else {
                        tc::tma_load_2d(base_s + L::kOffCode + s * kCodeBytes, &tmap_w,
                                        kb * (kBK / 2), nb * kBN, full(s));
                        bulk_g2s(sc, wsz + ((size_t)nb * nkb + kb) * kAtomBytes, kAtomBytes,
                                 bar_ptr(full(s)));
                    }
                    issued = it + 1;
                }
            }
            // every copy issued has landed before the CTA moves on to exit
            for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                mbar_wait_bounded(bar_ptr(full(i % kStages)), (i / kStages) & 1, kWaitLimitNs);
        }
        __syncwarp();  // lane 0 ran the role alone: the warp meets the block barrier converged
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int it = 0, lt = 0;
            tc::WorkIter wi = tc::make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
            int tile, kb0, kb1;
            for (; !*abort_flag && wi.next(tile, kb0, kb1); ++lt) {
                const int b = lt & 1;
                if (lt >= 2 &&
                    !tc::wait_or_abort(accempty(b), ((lt >> 1) - 1) & 1, abort_flag, err, dbg.wait_ns))
                    break;
                tc::fence_after();
                const uint32_t d = tmem + (uint32_t)(b * kBM);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!tc::wait_or_abort(full(s), ph, abort_flag, err, dbg.wait_ns) ||
                        !tc::wait_or_abort(afull(s), ph, abort_flag, err, dbg.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t a_s = base_s + L::kOffA + s * kABytes;
                    const uint32_t x_s = base_s + L::kOffX + s * kXBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc::mma_bf16(d, tc::sw128_desc(a_s + kk * 32), tc::sw128_desc(x_s + kk * 32),
                                     kIdesc, (kb != kb0 || kk != 0) ? 1u : 0u);
                    tc::commit(empty(s));
                }
                if (!ok) break;
                tc::commit(accfull(b));
            }
            // MMAs in flight complete before TMEM is freed
            tc::commit(drain);
            mbar_wait_bounded(bar_ptr(drain), 0, kWaitLimitNs);
        }
        __syncwarp();  // as in the producer warp
    } else if (warp < kEpiWarp0 + 4) {
        // ---------------- epilogue ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const float g = *gw;
        int lt = 0;
        tc::WorkIter wi = tc::make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
        int tile, kb0, kb1;
        for (; wi.next(tile, kb0, kb1); ++lt) {
            const int b = lt & 1;
            const bool ok = __all_sync(0xffffffffu,
                                       tc::wait_or_abort(accfull(b), (lt >> 1) & 1, abort_flag,
                                                         err, dbg.wait_ns));
            if constexpr (kFuse) {
                // the four warps meet at named barriers inside the tile: they leave together
                // (any warp's failed wait stops all four)
                if (named_bar_red_or(1, 128, !ok)) break;
                tc::fence_after();
                if (kb0 == 0 && kb1 == nkb) {
                    epilogue_silu_quant(tmem + (uint32_t)(b * kBM), q, lane, tile, ntiles_m, g,
                                        fa, reinterpret_cast<float*>(base + L::kOffXch), M);
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) tc::arrive(accempty(b));
                } else
                    epilogue_silu_quant_sk(tmem + (uint32_t)(b * kBM), q, lane, tile, ntiles_m,
                                           nkb, p_sk, tsk, g, fa,
                                           reinterpret_cast<float*>(base + L::kOffXch), M,
                                           accempty(b), slots, counters,
                                           reinterpret_cast<volatile uint32_t*>(
                                               base + L::kOffMisc + 8));
            } else {
                if (!ok) break;
                tc::fence_after();
                // on the CTA's last item the stage ring is idle: a quarter of it per warp
                tc::WorkIter peek = wi;
                int t_, k0_, k1_;
                uint8_t* stage = peek.next(t_, k0_, k1_) ? nullptr : base + q * kFixupBytes;
                tc::epilogue_work<kBN, kBM>(tmem + (uint32_t)(b * kBM), q, lane, tile, ntiles_m,
                                            kb0 == 0 && kb1 == nkb, nkb, p_sk, tsk, g, y, y_bf16,
                                            M, N, slots, counters, accempty(b), stage,
                                            bar_ptr(fixbar0 + 128u * q), kFixupBufs,
                                            tc::SkUnit{(int)blockIdx.x, 0, 1}, err);
            }
        }
    } else {
        // ---------------- dequantize ----------------
        const int t = threadIdx.x - kDequantWarp0 * 32;  // 0 .. 255
        const int r = t & (kBN - 1), h = t >> 7;         // W row in the tile, K half
        int it = 0;
        tc::WorkIter wi = tc::make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
        int tile, kb0, kb1;
        while (wi.next(tile, kb0, kb1)) {
            // the row's line in the scale atom(s): the fused variant's rows 0..63 are gate
            // rows of atom 0, rows 64..127 up rows of atom 1, both at row 64 (nb & 1) + r % 64
            // of their 128-row block
            int arow = r, aoff = 0;
            if constexpr (kFuse) {
                arow = (((tile / ntiles_m) & 1) << 6) | (r & 63);
                aoff = (r >> 6) * kAtomBytes;
            }
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % kStages;
                if (!__all_sync(0xffffffffu,
                                tc::wait_or_abort(full(s), (it / kStages) & 1, abort_flag, err, dbg.wait_ns))) {
                    ok = false;
                    break;
                }
                const uint4 c = *reinterpret_cast<const uint4*>(base + L::kOffCode +
                                                                s * kCodeBytes + r * 32 + h * 16);
                const uint32_t sb = *reinterpret_cast<const uint16_t*>(
                    base + L::kOffScale + s * L::kScaleBytes + aoff + (arow & 31) * 16 +
                    (arow >> 5) * 4 + 2 * h);
                // the two block scales as f16 (e4m3 is exact in f16)
                const uint32_t s01 = cvt_e4m3x2_f16x2(sb);
                const uint32_t w[4] = {c.x, c.y, c.z, c.w};
                uint8_t* arow_s = base + L::kOffA + s * kABytes + r * 128;
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                    uint32_t hh[4];
                    cvt8(w[qd], hh);
                    const uint32_t sc = qd < 2 ? (s01 & 0xFFFFu) : (s01 >> 16);
                    uint32_t o[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] = deq_bf16x2(hh[i], sc);
                    const int chunk = (4 * h + qd) ^ (r & 7);
                    *reinterpret_cast<uint4*>(arow_s + chunk * 16) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && !dbg.stall)
                    tc::arrive(afull(s));
            }
            if (!ok) break;
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kFuse>
cudaError_t configure(const DevInfo& dev) {
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = 1ull << (dev.device & 63);
    if (configured.load(std::memory_order_acquire) & bit) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(gemm_w4a16_kernel<kFuse>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)Smem<kFuse>::kBytes);
    if (e == cudaSuccess) configured.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

}  // namespace

GemmPlan gemm_w4a16_plan(int64_t M, int64_t K, int64_t N, int sm_count) {
    return tc::make_plan(M, K, N, sm_count, kBN, kBM, kBK);
}

size_t gemm_w4a16_workspace_bytes(int64_t M, int64_t K, int64_t N) {
    return kGemmHeaderBytes + tc::stream_k_bytes(M, K, N, kBN, kBM, kBK);
}

cudaError_t launch_gemm_w4a16(const uint16_t* x, int M, int K, const uint8_t* wq,
                              const uint8_t* wsz, const float* gw, int N, void* y, bool y_bf16,
                              uint8_t* workspace, cudaStream_t stream, const DevInfo& dev) {
    if (dev.smem_optin < Smem<false>::kBytes) return cudaErrorInvalidConfiguration;
    const GemmPlan p = gemm_w4a16_plan(M, K, N, dev.sm_count);
    CUtensorMap mx, mw;
    cudaError_t e = tc::make_map_2d(&mx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)K,
                                    (uint64_t)M, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    e = tc::make_map_2d(&mw, wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2, (uint64_t)N,
                        kBK / 2, kBN, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    e = configure<false>(dev);
    if (e != cudaSuccess) return e;
    uint32_t* err = reinterpret_cast<uint32_t*>(workspace);
    uint32_t* counters = reinterpret_cast<uint32_t*>(workspace + kGemmHeaderBytes);
    float* slots = reinterpret_cast<float*>(workspace + kGemmHeaderBytes +
                                            tc::counters_bytes(p.ntiles));
    gemm_w4a16_kernel<false><<<p.grid, kThreads, Smem<false>::kBytes, stream>>>(
        mx, mw, wsz, gw, y, y_bf16 ? 1 : 0, M, N, p.nkb, p.ntiles_m, p.ntiles, p.ntiles_sk, p.p_sk,
        p.tsk, err, counters, slots, FuseArgs{}, current_wait_cfg());
    return cudaGetLastError();
}

bool gemm_w4a16_silu_takes(int64_t M, int64_t I, const DevInfo& dev) {
    return M > kGemvMaxM && I % 128 == 0 && dev.smem_optin >= Smem<true>::kBytes;
}

cudaError_t launch_gemm_w4a16_silu(const uint16_t* x, int M, int K, const uint8_t* wq,
                                   const uint8_t* wsz, const float* gw, int I, const float* gh,
                                   uint8_t* hq, uint8_t* hs, uint8_t* workspace,
                                   cudaStream_t stream, const DevInfo& dev) {
    if (!gemm_w4a16_silu_takes(M, I, dev)) return cudaErrorInvalidConfiguration;
    // tiles of 64-column pairs of h (64 gate + 64 up rows of W) x 256 rows of x, persistent
    // CTAs; the last partial wave goes stream-K (the tile count and the split of the plain
    // GEMM on 2I rows)
    const GemmPlan p = gemm_w4a16_plan(M, K, 2 * (int64_t)I, dev.sm_count);
    CUtensorMap mx, mw;
    cudaError_t e = tc::make_map_2d(&mx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)K,
                                    (uint64_t)M, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    e = tc::make_map_2d(&mw, wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2,
                        (uint64_t)2 * I, kBK / 2, kBN / 2, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    e = configure<true>(dev);
    if (e != cudaSuccess) return e;
    FuseArgs fa;
    fa.I = I;
    fa.gh = gh;
    fa.hq = hq;
    fa.hs = hs;
    uint32_t* err = reinterpret_cast<uint32_t*>(workspace);
    uint32_t* counters = reinterpret_cast<uint32_t*>(workspace + kGemmHeaderBytes);
    float* slots = reinterpret_cast<float*>(workspace + kGemmHeaderBytes +
                                            tc::counters_bytes(p.ntiles));
    gemm_w4a16_kernel<true><<<p.grid, kThreads, Smem<true>::kBytes, stream>>>(
        mx, mw, wsz, gw, nullptr, 1, M, 2 * I, p.nkb, p.ntiles_m, p.ntiles, p.ntiles_sk, p.p_sk,
        p.tsk, err, counters, slots, fa, current_wait_cfg());
    return cudaGetLastError();
}

}  // namespace nvfp4
