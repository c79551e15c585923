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
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "nvfp4.h"

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
constexpr uint32_t kScaleBytes = 512;             // one 128 x 4 scale atom
constexpr uint32_t kOffX = 0;
constexpr uint32_t kOffA = kOffX + kStages * kXBytes;
constexpr uint32_t kOffCode = kOffA + kStages * kABytes;
constexpr uint32_t kOffScale = kOffCode + kStages * kCodeBytes;
constexpr uint32_t kOffBar = kOffScale + kStages * kScaleBytes;
constexpr uint32_t kNumBars = 3 * kStages + 4 + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment
constexpr int kMaxSkCtas = 160;                     // CTAs in the stream-K part, at most
constexpr size_t kSlotFloats = (size_t)kBN * kBM;   // one fp32 partial tile

// ---- tcgen05 / TMA wrappers ------------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0,
                                            int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] . B[smem desc]^T, bf16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive (once) on bar when every tcgen05 operation this thread issued so far completes
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
        "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
        "%27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle layout: rows
// of 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), the tile based at a
// 1024-byte boundary; the start address may move by 32-byte K steps inside the row.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;              // leading byte offset (unused with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset
    d |= (uint64_t)1 << 46;              // descriptor version
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp32 D, bf16 A and B, both K-major, M x N.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            ((uint32_t)(kBM >> 3) << 17) | ((uint32_t)(kBN >> 4) << 24);

// two e4m3 bytes (low 16 bits) -> f16x2, exact
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t b2) {
    uint32_t d;
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n"
        : "=r"(d) : "r"(b2));
    return d;
}

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

struct Bars {
    uint32_t full, afull, empty, accfull, accempty, drain;
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, uint32_t* err) {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bar)), parity,
                          kWaitLimitNs))
        return true;
    if (err) atomicOr(err, NVFP4_DEVERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

// The CTA's work: first its stream-K range of (tile, K step) iterations over the first
// ntiles_sk tiles, cut at tile boundaries, then whole tiles ntiles_sk + c, + grid, ...
struct WorkIter {
    int64_t i, i_end;
    int dp, ntiles, nkb, stride;
    __device__ bool next(int& tile, int& kb0, int& kb1) {
        if (i < i_end) {
            tile = (int)(i / nkb);
            kb0 = (int)(i - (int64_t)tile * nkb);
            const int64_t left = i_end - i;
            kb1 = left < (int64_t)(nkb - kb0) ? kb0 + (int)left : nkb;
            i += kb1 - kb0;
            return true;
        }
        if (dp < ntiles) {
            tile = dp;
            kb0 = 0;
            kb1 = nkb;
            dp += stride;
            return true;
        }
        return false;
    }
};

__device__ __forceinline__ WorkIter make_iter(int ntiles, int nkb, int ntiles_sk, int p_sk,
                                              int64_t tsk) {
    WorkIter w;
    const int c = blockIdx.x;
    if (c < p_sk) {
        w.i = (int64_t)c * tsk / p_sk;
        w.i_end = (int64_t)(c + 1) * tsk / p_sk;
    } else {
        w.i = w.i_end = 0;
    }
    w.dp = ntiles_sk + c;
    w.ntiles = ntiles;
    w.nkb = nkb;
    w.stride = gridDim.x;
    return w;
}

// stream-K bookkeeping: the CTA whose range holds iteration i, and the slot CTA c uses for
// its partial of the tile starting at iteration t0 (2c: its first segment, 2c + 1: its last)
__device__ __forceinline__ int sk_cta_of(int64_t i, int p_sk, int64_t tsk) {
    return (int)(((i + 1) * p_sk - 1) / tsk);
}
__device__ __forceinline__ int sk_slot(int c, int64_t t0, int p_sk, int64_t tsk) {
    return 2 * c + ((int64_t)c * tsk / p_sk < t0 ? 1 : 0);
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_w4a16_kernel(const __grid_constant__ CUtensorMap tmap_x,
                  const __grid_constant__ CUtensorMap tmap_w, const uint8_t* __restrict__ wsz,
                  const float* __restrict__ gw, void* __restrict__ y, int y_bf16, int M, int N,
                  int nkb, int ntiles_m, int ntiles, int ntiles_sk, int p_sk, int64_t tsk,
                  uint32_t* __restrict__ err, uint32_t* __restrict__ counters,
                  float* __restrict__ slots) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const uint32_t bar0 = base_s + kOffBar;
    // barrier addresses (shared space)
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto afull = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto empty = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
    auto accfull = [&](int b) { return bar0 + 8u * (3 * kStages + b); };
    auto accempty = [&](int b) { return bar0 + 8u * (3 * kStages + 2 + b); };
    const uint32_t drain = bar0 + 8u * (3 * kStages + 4);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(reinterpret_cast<uint64_t*>(base + kOffBar + 8 * s), 1);
            mbar_init(reinterpret_cast<uint64_t*>(base + kOffBar + 8 * (kStages + s)),
                      kDequantWarps);
            mbar_init(reinterpret_cast<uint64_t*>(base + kOffBar + 8 * (2 * kStages + s)), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(reinterpret_cast<uint64_t*>(base + kOffBar + 8 * (3 * kStages + b)), 1);
            mbar_init(reinterpret_cast<uint64_t*>(base + kOffBar + 8 * (3 * kStages + 2 + b)),
                      4);
        }
        mbar_init(reinterpret_cast<uint64_t*>(base + kOffBar + 8 * (3 * kStages + 4)), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(base_s + kOffMisc, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int it = 0, issued = 0;
            WorkIter wi = make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
            int tile, kb0, kb1;
            while (!*abort_flag && wi.next(tile, kb0, kb1)) {
                const int nb = tile / ntiles_m, mb = tile % ntiles_m;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages &&
                        !wait_or_abort(empty(s), ((it / kStages) - 1) & 1, abort_flag, err))
                        break;
                    mbar_arrive_expect_tx(
                        reinterpret_cast<uint64_t*>(base + kOffBar + 8 * s),
                        kXBytes + kCodeBytes + kScaleBytes);
                    tma_load_2d(base_s + kOffX + s * kXBytes, &tmap_x, kb * kBK, mb * kBM,
                                full(s));
                    tma_load_2d(base_s + kOffCode + s * kCodeBytes, &tmap_w, kb * (kBK / 2),
                                nb * kBN, full(s));
                    bulk_g2s(base + kOffScale + s * kScaleBytes,
                             wsz + ((size_t)nb * nkb + kb) * kScaleBytes, kScaleBytes,
                             reinterpret_cast<uint64_t*>(base + kOffBar + 8 * s));
                    issued = it + 1;
                }
            }
            // every copy issued has landed before the CTA moves on to exit
            for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                mbar_wait_bounded(reinterpret_cast<uint64_t*>(base + kOffBar + 8 * (i % kStages)),
                                  (i / kStages) & 1, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int it = 0, lt = 0;
            WorkIter wi = make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
            int tile, kb0, kb1;
            for (; !*abort_flag && wi.next(tile, kb0, kb1); ++lt) {
                const int b = lt & 1;
                if (lt >= 2 && !wait_or_abort(accempty(b), ((lt >> 1) - 1) & 1, abort_flag, err))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * kBM);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!wait_or_abort(full(s), ph, abort_flag, err) ||
                        !wait_or_abort(afull(s), ph, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_s = base_s + kOffA + s * kABytes;
                    const uint32_t x_s = base_s + kOffX + s * kXBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16(d, sw128_desc(a_s + kk * 32), sw128_desc(x_s + kk * 32), kIdesc,
                                 (kb != kb0 || kk != 0) ? 1u : 0u);
                    mma_commit(empty(s));
                }
                if (!ok) break;
                mma_commit(accfull(b));
            }
            // MMAs in flight complete before TMEM is freed
            mma_commit(drain);
            mbar_wait_bounded(reinterpret_cast<uint64_t*>(base + kOffBar + 8 * (3 * kStages + 4)),
                              0, kWaitLimitNs);
        }
    } else if (warp < kEpiWarp0 + 4) {
        // ---------------- epilogue ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int nl = q * 32 + lane;                   // W row of the tile (TMEM lane)
        const float g = *gw;
        int lt = 0;
        WorkIter wi = make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
        int tile, kb0, kb1;
        for (; wi.next(tile, kb0, kb1); ++lt) {
            const int b = lt & 1;
            const bool ok = __all_sync(0xffffffffu,
                                       wait_or_abort(accfull(b), (lt >> 1) & 1, abort_flag, err));
            if (!ok) break;
            tc_fence_after();
            const int nb = tile / ntiles_m, mb = tile % ntiles_m;
            const int64_t n = (int64_t)nb * kBN + nl;
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * kBM);
            const bool whole = kb0 == 0 && kb1 == nkb;
            const int64_t t0 = (int64_t)tile * nkb;
            float* mine = whole ? nullptr
                                : slots + (size_t)sk_slot(blockIdx.x, t0, p_sk, tsk) * kSlotFloats;
#pragma unroll 1
            for (int c0 = 0; c0 < kBM; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(taddr + c0, v);
                if (!whole) {
                    // partial tile: fp32 slot, [m within tile][W row within tile]
#pragma unroll
                    for (int j = 0; j < 32; ++j) mine[(c0 + j) * kBN + nl] = __uint_as_float(v[j]);
                    continue;
                }
                const int64_t m0 = (int64_t)mb * kBM + c0;
                if (n < N) {
                    if (y_bf16) {
                        uint16_t* yp = static_cast<uint16_t*>(y) + m0 * N + n;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (m0 + j < M)
                                yp[(int64_t)j * N] = f32_to_bf16_rne(__uint_as_float(v[j]) * g);
                    } else {
                        float* yp = static_cast<float*>(y) + m0 * N + n;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (m0 + j < M) yp[(int64_t)j * N] = __uint_as_float(v[j]) * g;
                    }
                }
            }
            // the accumulator is free for the tile after next
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(accempty(b))));
            if (whole) continue;
            // count this warp's quarter of the segment in (one counter per tile quarter, so
            // no epilogue warp ever waits for another); the arrival that completes the
            // quarter sums it
            const int cf = sk_cta_of(t0, p_sk, tsk), cl = sk_cta_of(t0 + nkb - 1, p_sk, tsk);
            const unsigned nseg = (unsigned)(cl - cf + 1);
            __threadfence();
            __syncwarp();
            unsigned old = 0;
            if (lane == 0) old = atomicInc(&counters[tile * 4 + q], nseg - 1);
            const bool last = __shfl_sync(0xffffffffu, old, 0) == nseg - 1;
            if (!last) continue;
            __threadfence();
            // 32 rows of the quarter at a time, every partial's 32 loads in flight together;
            // the partials are added in segment order
#pragma unroll 1
            for (int c0 = 0; c0 < kBM; c0 += 32) {
                const int64_t m0 = (int64_t)mb * kBM + c0;
                if (m0 >= M) break;
                float acc[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
#pragma unroll 1
                for (int cs = cf; cs <= cl; ++cs) {
                    const float* sp =
                        slots + (size_t)sk_slot(cs, t0, p_sk, tsk) * kSlotFloats + c0 * kBN + nl;
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __ldcg(sp + j * kBN);
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc[j] += v[j];
                }
                if (n < N) {
                    if (y_bf16) {
                        uint16_t* yp = static_cast<uint16_t*>(y) + m0 * N + n;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (m0 + j < M) yp[(int64_t)j * N] = f32_to_bf16_rne(acc[j] * g);
                    } else {
                        float* yp = static_cast<float*>(y) + m0 * N + n;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (m0 + j < M) yp[(int64_t)j * N] = acc[j] * g;
                    }
                }
            }
        }
    } else {
        // ---------------- dequantize ----------------
        const int t = threadIdx.x - kDequantWarp0 * 32;  // 0 .. 255
        const int r = t & (kBN - 1), h = t >> 7;         // W row in the tile, K half
        int it = 0;
        WorkIter wi = make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
        int tile, kb0, kb1;
        while (wi.next(tile, kb0, kb1)) {
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % kStages;
                if (!__all_sync(0xffffffffu,
                                wait_or_abort(full(s), (it / kStages) & 1, abort_flag, err))) {
                    ok = false;
                    break;
                }
                const uint4 c = *reinterpret_cast<const uint4*>(base + kOffCode + s * kCodeBytes +
                                                                r * 32 + h * 16);
                const uint32_t sb = *reinterpret_cast<const uint16_t*>(
                    base + kOffScale + s * kScaleBytes + (r & 31) * 16 + (r >> 5) * 4 + 2 * h);
                // the two block scales as f16 (e4m3 is exact in f16)
                const uint32_t s01 = cvt_e4m3x2_f16x2(sb);
                const uint32_t w[4] = {c.x, c.y, c.z, c.w};
                uint8_t* arow = base + kOffA + s * kABytes + r * 128;
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                    uint32_t hh[4];
                    cvt8(w[qd], hh);
                    const uint32_t sc = qd < 2 ? (s01 & 0xFFFFu) : (s01 >> 16);
                    uint32_t o[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] = deq_bf16x2(hh[i], sc);
                    const int chunk = (4 * h + qd) ^ (r & 7);
                    *reinterpret_cast<uint4*>(arow + chunk * 16) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(afull(s))));
            }
            if (!ok) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- host side ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D tiled map over a row-major [rows, inner] tensor
cudaError_t make_map_2d(CUtensorMap* map, const void* ptr, CUtensorMapDataType type,
                        int elem_bytes, uint64_t inner, uint64_t rows, uint32_t box_inner,
                        uint32_t box_rows, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, type, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

GemmPlan gemm_w4a16_plan(int64_t M, int64_t K, int64_t N, int sm_count) {
    GemmPlan p;
    p.nkb = (int)((K + kBK - 1) / kBK);
    p.ntiles_m = (int)((M + kBM - 1) / kBM);
    p.ntiles = (int)((N + kBN - 1) / kBN) * p.ntiles_m;
    // the tiles of the last, partial wave (all of them when fewer than the SMs) go stream-K
    int sk = p.ntiles >= sm_count ? p.ntiles % sm_count : p.ntiles;
    const int64_t tsk = (int64_t)sk * p.nkb;
    // at least 4 K steps per CTA, at most 3 CTAs' worth per tile, at most kMaxSkCtas
    int64_t psk = sm_count;
    if (psk > 3 * (int64_t)sk) psk = 3 * (int64_t)sk;
    if (psk > tsk / 4) psk = tsk / 4;
    if (psk > kMaxSkCtas) psk = kMaxSkCtas;
    if (psk < 2) {
        sk = 0;
        psk = 0;
    }
    p.ntiles_sk = sk;
    p.p_sk = (int)psk;
    p.tsk = (int64_t)sk * p.nkb;
    const int dp = p.ntiles - sk;
    int grid = dp < sm_count ? dp : sm_count;
    if (grid < p.p_sk) grid = p.p_sk;
    p.grid = grid;
    return p;
}

size_t gemm_w4a16_workspace_bytes(int64_t M, int64_t K, int64_t N) {
    // a bound over every SM count: the plan never uses more stream-K CTAs than this
    const int64_t nkb = (K + kBK - 1) / kBK;
    const int64_t ntiles = ((N + kBN - 1) / kBN) * ((M + kBM - 1) / kBM);
    int64_t psk = kMaxSkCtas;
    if (psk > 3 * ntiles) psk = 3 * ntiles;
    if (psk > ntiles * nkb / 4) psk = ntiles * nkb / 4;
    if (psk < 2) psk = 0;
    const size_t counters = ((size_t)ntiles * 16 + 255) / 256 * 256;
    return kGemmHeaderBytes + counters + (size_t)(2 * psk) * kSlotFloats * 4;
}

cudaError_t launch_gemm_w4a16(const uint16_t* x, int M, int K, const uint8_t* wq,
                              const uint8_t* wsz, const float* gw, int N, void* y, bool y_bf16,
                              uint8_t* workspace, cudaStream_t stream, const DevInfo& dev) {
    if (dev.smem_optin < kSmemBytes) return cudaErrorInvalidConfiguration;
    const GemmPlan p = gemm_w4a16_plan(M, K, N, dev.sm_count);
    CUtensorMap mx, mw;
    cudaError_t e = make_map_2d(&mx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)K,
                                (uint64_t)M, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    e = make_map_2d(&mw, wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2, (uint64_t)N,
                    kBK / 2, kBN, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = 1ull << (dev.device & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(gemm_w4a16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    uint32_t* err = reinterpret_cast<uint32_t*>(workspace);
    uint32_t* counters = reinterpret_cast<uint32_t*>(workspace + kGemmHeaderBytes);
    float* slots = reinterpret_cast<float*>(
        workspace + kGemmHeaderBytes + ((size_t)p.ntiles * 16 + 255) / 256 * 256);
    gemm_w4a16_kernel<<<p.grid, kThreads, kSmemBytes, stream>>>(
        mx, mw, wsz, gw, y, y_bf16 ? 1 : 0, M, N, p.nkb, p.ntiles_m, p.ntiles, p.ntiles_sk, p.p_sk,
        p.tsk, err, counters, slots);
    return cudaGetLastError();
}

}  // namespace nvfp4
