// gemm_w4a4.cu -- W4A4 NVFP4 GEMM for M > 16 on the 5th-generation tensor cores, block
// scaled in hardware.  FlashRT docs/qwen36_usage.md (FLASHRT_QWEN36_FUSE_SILU_MUL_QUANT:
// activations quantized to NVFP4 feed the NVFP4 GEMM).
//
//   y[m, n] = gx * gw * sum_b sx[m, b] * sw[n, b] * sum_{k in b} e2m1(qx[m, k]) * e2m1(qw[n, k])
//
// x arrives quantized (codes [M, K/2], scale atoms, gx: the NVFP4 activations of the
// down projection), or as bf16 that the kernel quantizes itself (the kQuantX variant):
// after its barriers and TMEM are set up, every CTA quantizes a share of x into the
// workspace with the quantizer's block rule -- behind an amax pass and one grid-wide
// barrier when the scale is dynamic -- and counts itself done; the TMA producer waits
// for the count to reach the grid before its first load of x.  The grid is launched
// cooperatively (one CTA per SM, all resident), every wait is bounded, and the last CTA
// to finish zeroes the counters for the next call.  tcgen05.mma kind::mxf4nvf4 with 16-element UE4M3 block scales
// (scale_vec::4X) multiplies the packed E2M1 operands straight from shared memory; the
// scales reach TMEM in the layout the block-scaled MMA reads: one 512-byte atom of the
// tensor-core scale layout (128 rows x 64 K, which is how the repacked scales are stored)
// is 32 rows of 16 bytes, and TMEM lane 32q + i, columns c .. c+3 hold row i of the atom
// for every lane quarter q.
//
// CTA tile: 128 rows of W (MMA M) x 256 rows of x (MMA N), K in steps of 256 (128 bytes of
// codes per row: one 128-byte swizzle row).  One 256-column fp32 accumulator (the rest of
// TMEM holds the scales of the stages in flight), so the MMAs of a tile start once the
// epilogue has read the previous one.  Warp roles:
//   warp 0      TMA producer: per K step the W and x scale atoms of those 256 K (bulk
//               copies, first, on a barrier of their own), then the two 128 x 128-byte
//               code boxes (128-byte swizzle);
//   warp 1      allocates TMEM (the accumulator + a scale area per stage) and, from one
//               thread, issues 4 x 128x256x64 block-scaled MMAs per stage once its codes
//               and its scales are in place;
//   warps 2-5   epilogue (shared with the W4A16 GEMM): x gx gw, y fp32 or bf16;
//   warps 6-9   scale writers: once a stage's atoms have landed (while its codes may still
//               be in flight), each thread loads row (lane) of the 12 atoms (4 of W,
//               2 x 4 of x) from shared memory and stores them to its TMEM lane (keeping
//               these copies off the MMA thread's in-order tcgen05 queue).
// Work split, stream-K fixup, bounded waits and error reporting as in the W4A16 GEMM.
//
// Further down, a CTA-pair variant of the same GEMM (tcgen05 cta_group::2, 256 x 256
// tiles), selected per thread with nvfp4_debug_w4a4_kernel: the same bits, but slower than
// the kernel above on the shapes measured (M = 2048 at K 5120, N 17408; the 512-token down
// projection at K 17408, N 5120), so not the default.
#include <cuda.h>

#include <atomic>

#include "tcgen05.cuh"

namespace nvfp4 {
namespace {

constexpr int kBN = 128;   // W rows per tile (MMA M)
constexpr int kBM = 256;   // x rows per tile (MMA N)
constexpr int kBK = 256;   // K per stage
constexpr int kStages = 4;
constexpr int kThreads = 10 * 32;
constexpr int kSfWarp0 = 6;
constexpr int kTmemCols = 512;
constexpr uint32_t kTmemSf = kBM;                 // first TMEM column of the scale area
// per stage: 4 W atoms (columns 0..15), then per MMA k-step j the x atoms of rows 0..127
// and 128..255 (columns 16 + 8j .. 16 + 8j + 7), 4 columns each
constexpr uint32_t kSfColsPerStage = 48;

constexpr uint32_t kABytes = kBN * kBK / 2;       // 16 KB of W codes
constexpr uint32_t kBBytes = kBM * kBK / 2;       // 32 KB of x codes
constexpr uint32_t kAtomBytes = 512;
constexpr uint32_t kSfaBytes = 4 * kAtomBytes;    // 4 atoms (256 K) of W
constexpr uint32_t kSfbBytes = 8 * kAtomBytes;    // 2 row blocks x 4 atoms of x
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kOffSfa = kOffB + kStages * kBBytes;
constexpr uint32_t kOffSfb = kOffSfa + kStages * kSfaBytes;
constexpr uint32_t kOffBar = kOffSfb + kStages * kSfbBytes;
constexpr uint32_t kFixBars = 4 * 16;  // stream-K fix-up chunk barriers, 16 per epilogue warp
constexpr uint32_t kNumBars = 4 * kStages + 4 + 1 + kFixBars;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment

static_assert(kTmemSf + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");

// The stream-K fix-up of a CTA's last work item stages partials in the idle stage ring:
// a quarter of it per epilogue warp, in 4 KB chunk buffers.
constexpr uint32_t kFixupBytes = (kOffBar / 4) & ~127u;
constexpr int kFixupBufs = (int)(kFixupBytes / 4096) < 16 ? (int)(kFixupBytes / 4096) : 16;
static_assert(kFixupBufs >= 2, "fix-up staging");

// Instruction descriptor, block-scaled kind: E2M1 A and B, UE4M3 scales (scale type 0),
// scale ids 0, dense K = 64 per instruction, both K-major, fp32 D, M x N.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kBM >> 3) << 17) |
                            ((uint32_t)(kBN >> 4) << 24);

// In-kernel quantization of bf16 x (the kQuantX variant): x quantized to NVFP4 by every
// CTA of the persistent grid together, before and while the GEMM starts.
struct QxArgs {
    const uint16_t* x = nullptr;      // bf16 [M, K]
    const float* gx_static = nullptr; // static global scale of x, or null: amax / 2688
    float* gx_out = nullptr;          // g_x (written by CTA 0)
    float* partials = nullptr;        // one amax partial per CTA (dynamic scale)
    uint32_t* sync = nullptr;         // [0] barrier count, [1] barrier generation,
                                      // [2] exit count, [3] CTAs whose share of x is written
    uint8_t* xq = nullptr;            // codes [M, K/2] (the GEMM's x operand)
    uint8_t* xs = nullptr;            // scale atoms of x (rows padded to 128, blocks to 4)
    int K = 0;
};

// generic-proxy writes to global memory made visible to (and ordered with) the async
// proxy: the quantized x is written with plain stores and read by TMA in other CTAs
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Spin until *p reaches `target` (acquire), at most limit_ns; false on time-out.
__device__ __forceinline__ bool wait_counter(const uint32_t* p, uint32_t target,
                                             uint64_t limit_ns) {
    if (ld_acquire_gpu(p) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ld_acquire_gpu(p) >= target) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
        __nanosleep(64);
    }
}

// Grid-wide barrier of the co-resident grid (one thread per CTA): the arrival that
// completes the count resets it and advances the generation the others wait on.
__device__ __forceinline__ bool grid_barrier(uint32_t* sync, uint64_t limit_ns) {
    volatile uint32_t* gen_p = sync + 1;
    const uint32_t gen = *gen_p;
    __threadfence();
    const uint32_t old = atomicAdd(sync, 1u);
    if (old == gridDim.x - 1) {
        atomicExch(sync, 0u);
        __threadfence();
        atomicAdd(sync + 1, 1u);
        return true;
    }
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(sync + 1) == gen) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
        __nanosleep(64);
    }
    return true;
}

// Quantize every 16-element block of x (rows padded to 128, blocks to 4): this CTA's share
// is blocks b = blockIdx.x * threads + t (+ gridDim.x * threads ...), taken kQxBatch at a
// time with all their loads in flight.  Codes go row-major, scales to the atom layout;
// padding rows and blocks get zero scales.
constexpr int kQxBatch = 4;

__device__ __forceinline__ void quantize_x_all(const QxArgs& qa, int M, float g) {
    const int K = qa.K;
    const int64_t cb_n = K >> 4, cp4 = (cb_n + 3) >> 2, cb_iter = cp4 << 2;
    const int64_t nblk = (int64_t)((M + 127) / 128 * 128) * cb_iter;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t b0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b0 < nblk;
         b0 += kQxBatch * stride) {
        uint4 v[kQxBatch][2];
        int64_t r[kQxBatch], cb[kQxBatch];
        bool real[kQxBatch];
#pragma unroll
        for (int u = 0; u < kQxBatch; ++u) {
            const int64_t b = b0 + u * stride;
            // 32-bit division while the indices fit (every realistic x)
            r[u] = nblk <= 0xFFFFFFFFll ? (int64_t)((uint32_t)b / (uint32_t)cb_iter)
                                        : b / cb_iter;
            cb[u] = b - r[u] * cb_iter;
            real[u] = b < nblk && r[u] < M && cb[u] < cb_n;
            if (real[u]) {
                const uint4* p = reinterpret_cast<const uint4*>(qa.x + r[u] * K + (cb[u] << 4));
                v[u][0] = __ldg(p);
                v[u][1] = __ldg(p + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < kQxBatch; ++u) {
            if (b0 + u * stride >= nblk) break;
            if (!real[u]) {
                qa.xs[swizzle_offset(r[u], cb[u], cp4)] = 0;
                continue;
            }
            float t[16];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const uint32_t w[4] = {v[u][q].x, v[u][q].y, v[u][q].z, v[u][q].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    t[q * 8 + 2 * j] = bf16_to_f32(w[j] & 0xFFFFu);
                    t[q * 8 + 2 * j + 1] = bf16_to_f32(w[j] >> 16);
                }
            }
            uint32_t lo, hi;
            const uint32_t s8 = quantize_block16(t, g, lo, hi);
            *reinterpret_cast<uint2*>(qa.xq + r[u] * (K >> 1) + (cb[u] << 3)) = make_uint2(lo, hi);
            qa.xs[swizzle_offset(r[u], cb[u], cp4)] = (uint8_t)s8;
        }
    }
}

// The kQuantX prologue, run by every thread of every CTA after the CTA's barriers and TMEM
// are set up: g_x (the static scale, or the amax of all of x through one grid-wide barrier,
// then amax / 2688), then this CTA's share of x quantized and counted done.  Returns g_x;
// a failed grid barrier sets abort_flag (the GEMM roles then stop at once).
template <int kNumWarps>
__device__ __forceinline__ float quantize_x_prologue(const QxArgs& qa, int M, const WaitCfg& dbg,
                                                     uint32_t* err, volatile int* abort_flag) {
    __shared__ int qx_fail;
    __shared__ float red[kNumWarps];
    __shared__ float g_sh;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) qx_fail = 0;
    float g = 1.0f;
    if (qa.gx_static) {
        g = *qa.gx_static;
    } else {
        // amax of x: a partial per CTA, a grid barrier, then every CTA folds them
        float am = 0.0f;
        const int64_t nvec = (int64_t)M * qa.K / 8;
        const int64_t stride = (int64_t)gridDim.x * blockDim.x;
        const uint4* xv = reinterpret_cast<const uint4*>(qa.x);
        for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < nvec;
             i0 += 8 * stride) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[u] = i0 + u * stride < nvec ? __ldg(xv + i0 + u * stride)
                                              : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    am = fmaxf(am, fmaxf(fabsf(bf16_to_f32(w[j] & 0xFFFFu)),
                                         fabsf(bf16_to_f32(w[j] >> 16))));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (lane == 0) red[warp] = am;
        __syncthreads();
        if (threadIdx.x == 0) {
            float r = red[0];
            for (int i = 1; i < kNumWarps; ++i) r = fmaxf(r, red[i]);
            qa.partials[blockIdx.x] = r;
            if (!grid_barrier(qa.sync, dbg.wait_ns)) {
                if (err) atomicOr(err, NVFP4_DEVERR_TIMEOUT);
                qx_fail = 1;
            }
        }
        __syncwarp();  // warp 0 converged (thread 0 spun alone) before the block barrier
        __syncthreads();
        if (!qx_fail) {
            // every CTA's partial (read from L2: other CTAs wrote them in this kernel)
            float m = 0.0f;
            for (int i = threadIdx.x; i < (int)gridDim.x; i += blockDim.x)
                m = fmaxf(m, __ldcg(qa.partials + i));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            __syncthreads();
            if (lane == 0) red[warp] = m;
            __syncthreads();
            float r = red[0];
            for (int i = 1; i < kNumWarps; ++i) r = fmaxf(r, red[i]);
            g = global_scale_from_amax(r);
        }
    }
    if (threadIdx.x == 0) {
        g_sh = g;
        if (blockIdx.x == 0) *qa.gx_out = g;
    }
    if (!qx_fail) {
        quantize_x_all(qa, M, g);
        // this CTA's share is written: publish it to the async proxy, then count it
        fence_proxy_async_global();
        __syncthreads();
        // (with the test switch on, CTA 0 withholds its count: every producer's wait for the
        // count runs out)
        if (threadIdx.x == 0 && !(dbg.stall && blockIdx.x == 0)) {
            __threadfence();
            atomicAdd(qa.sync + 3, 1u);
        }
    }
    __syncthreads();
    if (qx_fail && threadIdx.x == 0) *abort_flag = 1;
    __syncthreads();
    return g_sh;
}

template <bool kQuantX>
__global__ void __launch_bounds__(kThreads, 1)
gemm_w4a4_kernel(const __grid_constant__ CUtensorMap tmap_w,
                 const __grid_constant__ CUtensorMap tmap_x, const uint8_t* __restrict__ wsz,
                 const uint8_t* __restrict__ xsz, const float* __restrict__ gw,
                 const float* __restrict__ gx, void* __restrict__ y, int y_bf16, int M, int N,
                 int nkb, int natoms_row, int x_row_blocks, int ntiles_m, int ntiles,
                 int ntiles_sk, int p_sk,
                 int64_t tsk, uint32_t* __restrict__ err, uint32_t* __restrict__ counters,
                 float* __restrict__ slots, QxArgs qa, WaitCfg dbg) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const uint32_t bar0 = base_s + kOffBar;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto accfull = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
    auto accempty = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
    const uint32_t drain = bar0 + 8u * (2 * kStages + 4);
    auto sfull = [&](int s) { return bar0 + 8u * (2 * kStages + 5 + s); };
    auto sland = [&](int s) { return bar0 + 8u * (3 * kStages + 5 + s); };  // scales landed
    const uint32_t fixbar0 = bar0 + 8u * (4 * kStages + 5);  // 16 per epilogue warp
    auto bar_ptr = [&](uint32_t a) { return reinterpret_cast<uint64_t*>(base + (a - base_s)); };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_ptr(full(s)), 1);
            mbar_init(bar_ptr(empty(s)), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_ptr(accfull(b)), 1);
            mbar_init(bar_ptr(accempty(b)), 4);
        }
        mbar_init(bar_ptr(drain), 1);
        for (int s = 0; s < kStages; ++s) mbar_init(bar_ptr(sfull(s)), 4);
        for (int s = 0; s < kStages; ++s) mbar_init(bar_ptr(sland(s)), 1);
        for (uint32_t i = 0; i < kFixBars; ++i) mbar_init(bar_ptr(fixbar0 + 8u * i), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc(base_s + kOffMisc, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    // ---- x quantized in-kernel (kQuantX): every CTA quantizes a share of x and counts
    // itself done; the TMA producer waits for the count to reach the grid before its
    // first load of x ----
    float gx_in = 1.0f;
    if constexpr (kQuantX) gx_in = quantize_x_prologue<kThreads / 32>(qa, M, dbg, err, abort_flag);

    // scale atoms of K step kb: 4, or fewer at the end of K
    auto atoms_of = [&](int kb) { return min(4, natoms_row - 4 * kb); };

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int it = 0, issued = 0;
            tc::WorkIter wi = tc::make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
            int tile, kb0, kb1;
            if constexpr (kQuantX) {
                // every CTA's share of the quantized x is written before the first TMA read
                if (!*abort_flag && !wait_counter(qa.sync + 3, gridDim.x, dbg.wait_ns)) {
                    if (err) atomicOr(err, NVFP4_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                // the other CTAs' stores, now visible, ahead of the TMA reads below
                fence_proxy_async_global();
            }
            while (!*abort_flag && wi.next(tile, kb0, kb1)) {
                const int nb = tile / ntiles_m, mb = tile % ntiles_m;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages &&
                        !tc::wait_or_abort(empty(s), ((it / kStages) - 1) & 1, abort_flag, err, dbg.wait_ns))
                        break;
                    const uint32_t sfb = (uint32_t)atoms_of(kb) * kAtomBytes;
                    // x rows of the tile: scale row blocks 2 mb and 2 mb + 1 (the second one
                    // only when it exists; rows past M are masked in the epilogue)
                    const bool two = 2 * mb + 1 < x_row_blocks;
                    // the scale atoms first, on their own barrier: the scale writers move
                    // them into TMEM while the code boxes are still landing
                    mbar_arrive_expect_tx(bar_ptr(sland(s)), sfb * (two ? 3u : 2u));
                    bulk_g2s(base + kOffSfa + s * kSfaBytes,
                             wsz + ((size_t)nb * natoms_row + 4 * kb) * kAtomBytes, sfb,
                             bar_ptr(sland(s)));
                    bulk_g2s(base + kOffSfb + s * kSfbBytes,
                             xsz + ((size_t)(2 * mb) * natoms_row + 4 * kb) * kAtomBytes, sfb,
                             bar_ptr(sland(s)));
                    if (two)
                        bulk_g2s(base + kOffSfb + s * kSfbBytes + 4 * kAtomBytes,
                                 xsz + ((size_t)(2 * mb + 1) * natoms_row + 4 * kb) * kAtomBytes,
                                 sfb, bar_ptr(sland(s)));
                    mbar_arrive_expect_tx(bar_ptr(full(s)), kABytes + kBBytes);
                    tc::tma_load_2d(base_s + kOffA + s * kABytes, &tmap_w, kb * (kBK / 2),
                                    nb * kBN, full(s));
                    tc::tma_load_2d(base_s + kOffB + s * kBBytes, &tmap_x, kb * (kBK / 2),
                                    mb * kBM, full(s));
                    issued = it + 1;
                }
            }
            // every copy issued has landed before the CTA moves on to exit
            for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i) {
                mbar_wait_bounded(bar_ptr(sland(i % kStages)), (i / kStages) & 1, kWaitLimitNs);
                mbar_wait_bounded(bar_ptr(full(i % kStages)), (i / kStages) & 1, kWaitLimitNs);
            }
        }
        __syncwarp();  // lane 0 ran the role alone: the warp meets the block barrier converged
    } else if (warp == 1) {
        // ---------------- MMA issue ----------------
        if (lane == 0) {
            int it = 0, lt = 0;
            tc::WorkIter wi = tc::make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
            int tile, kb0, kb1;
            for (; !*abort_flag && wi.next(tile, kb0, kb1); ++lt) {
                if (lt >= 1 && !tc::wait_or_abort(accempty(0), (lt - 1) & 1, abort_flag, err, dbg.wait_ns))
                    break;
                tc::fence_after();
                const uint32_t d = tmem;
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!tc::wait_or_abort(full(s), ph, abort_flag, err, dbg.wait_ns) ||
                        !tc::wait_or_abort(sfull(s), ph, abort_flag, err, dbg.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const int na = atoms_of(kb);
                    const uint32_t sf = tmem + kTmemSf + (uint32_t)s * kSfColsPerStage;
                    const uint32_t a_s = base_s + kOffA + s * kABytes;
                    const uint32_t b_s = base_s + kOffB + s * kBBytes;
                    for (int j = 0; j < na; ++j)
                        tc::mma_mxf4nvf4(d, tc::sw128_desc(a_s + j * 32),
                                         tc::sw128_desc(b_s + j * 32), kIdesc, sf + 4 * j,
                                         sf + 16 + 8 * j, (kb != kb0 || j != 0) ? 1u : 0u);
                    tc::commit(empty(s));
                }
                if (!ok) break;
                tc::commit(accfull(0));
            }
            // MMAs in flight complete before TMEM is freed
            tc::commit(drain);
            mbar_wait_bounded(bar_ptr(drain), 0, kWaitLimitNs);
        }
        __syncwarp();  // as in the producer warp
    } else if (warp >= kSfWarp0) {
        // ---------------- scale writers ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        int it = 0;
        tc::WorkIter wi = tc::make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
        int tile, kb0, kb1;
        while (wi.next(tile, kb0, kb1)) {
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % kStages;
                if (!__all_sync(0xffffffffu,
                                tc::wait_or_abort(sland(s), (it / kStages) & 1, abort_flag, err, dbg.wait_ns))) {
                    ok = false;
                    break;
                }
                // columns 0..15: the 4 W atoms; 16 + 8j .. 16 + 8j + 7: x atom j of row blocks
                // 2 mb and 2 mb + 1 (atoms past the end of K or of M hold stale bytes that no
                // MMA reads or whose rows the epilogue masks)
                const uint8_t* sa_s = base + kOffSfa + s * kSfaBytes + lane * 16;
                const uint8_t* sb_s = base + kOffSfb + s * kSfbBytes + lane * 16;
                uint32_t v[32], u16[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 a = *reinterpret_cast<const uint4*>(sa_s + j * kAtomBytes);
                    v[4 * j] = a.x; v[4 * j + 1] = a.y; v[4 * j + 2] = a.z; v[4 * j + 3] = a.w;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 b0 = *reinterpret_cast<const uint4*>(sb_s + j * kAtomBytes);
                    const uint4 b1 = *reinterpret_cast<const uint4*>(sb_s + (4 + j) * kAtomBytes);
                    uint32_t* dst = j < 2 ? &v[16 + 8 * j] : &u16[8 * (j - 2)];
                    dst[0] = b0.x; dst[1] = b0.y; dst[2] = b0.z; dst[3] = b0.w;
                    dst[4] = b1.x; dst[5] = b1.y; dst[6] = b1.z; dst[7] = b1.w;
                }
                const uint32_t col = tmem + ((uint32_t)(q * 32) << 16) + kTmemSf +
                                     (uint32_t)s * kSfColsPerStage;
                tc::tmem_st32(col, v);
                tc::tmem_st16(col + 32, u16);
                tc::fence_before();
                __syncwarp();
                if (lane == 0 && !(dbg.stall && !kQuantX)) tc::arrive(sfull(s));
            }
            if (!ok) break;
        }
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const float g = *gw * (kQuantX ? gx_in : *gx);
        int lt = 0;
        tc::WorkIter wi = tc::make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk);
        int tile, kb0, kb1;
        for (; wi.next(tile, kb0, kb1); ++lt) {
            if (!__all_sync(0xffffffffu,
                            tc::wait_or_abort(accfull(0), lt & 1, abort_flag, err, dbg.wait_ns)))
                break;
            tc::fence_after();
            // on the CTA's last item the stage ring is idle: a quarter of it per warp
            tc::WorkIter peek = wi;
            int t_, k0_, k1_;
            uint8_t* stage = peek.next(t_, k0_, k1_) ? nullptr : base + q * kFixupBytes;
            tc::epilogue_work<kBN, kBM>(tmem, q, lane, tile, ntiles_m, kb0 == 0 && kb1 == nkb,
                                        nkb, p_sk, tsk, g, y, y_bf16, M, N, slots, counters,
                                        accempty(0), stage, bar_ptr(fixbar0 + 128u * q),
                                        kFixupBufs, tc::SkUnit{(int)blockIdx.x, 0, 1},
                                        err);
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if constexpr (kQuantX) {
        // the last CTA out (every other CTA is past all its waits) zeroes the ready counts,
        // so the workspace is ready for the next call
        if (threadIdx.x == 0) {
            __threadfence();
            if (atomicAdd(qa.sync + 2, 1u) == gridDim.x - 1) {
                atomicExch(qa.sync + 3, 0u);
                atomicExch(qa.sync, 0u);
                atomicExch(qa.sync + 2, 0u);
            }
        }
    }
}

// ---- CTA-pair kernel ---------------------------------------------------------------------
//
// A pair of CTAs on two SMs computes a 256 (W) x 256 (x) tile with M = 256 block-scaled
// MMAs (tcgen05.mma.cta_group::2): the even CTA issues the MMAs, the MMA's A is split by
// rows across the two CTAs and B by N.  CTA rank r holds W rows (2 nb + r) x 128 .. +128 of
// tile nb and half r of the tile's x rows; per K step of 256 it takes in 38 KB: 16 KB of W
// codes, 16 KB of x codes, 2 KB of W scale atoms and the 4 KB of scale atoms of all 256 x
// rows, which both CTAs' TMEM must hold.  The one-CTA kernel takes in 54 KB for the same
// MMA work.
//
// Every copy is a TMA load that lands in the issuing CTA's shared memory and completes on
// the even CTA's stage barrier, which expects both CTAs' bytes.  One thread of the even CTA
// moves the stage's scale atoms from both CTAs' shared memory into their TMEM
// (tcgen05.cp.cta_group::2, in order ahead of the MMAs that read them) and issues the four
// MMAs; its commits release the stage in both CTAs.  Each CTA's TMEM holds the fp32
// accumulator of its own 128 W rows x the tile's 256 x rows (columns 0..255) and the
// scales of the stages in flight.
//
// Warp roles per CTA:
//   warp 0      TMA producer (both CTAs, in step: both wait on their own stage barriers,
//               which the even CTA's MMA commits release together);
//   warp 1      TMEM allocation (both CTAs together), MMA issue (even CTA);
//   warps 2-9   epilogue: lane quarter (warp & 3), x-row half (warp - 2) / 4.  A whole tile
//               is read out of TMEM into registers (128 columns per warp) and the
//               accumulator released before the stores, so the next tile's MMAs overlap
//               them; a stream-K segment is written by the first half's warps (the
//               shared stream-K epilogue, per CTA half), the second half's warps release
//               at once.
namespace pairk {

constexpr int kBM = 256;   // x rows per tile (MMA N), 128 loaded by each CTA of a pair
constexpr int kBK = 256;   // K per stage
constexpr int kStages = 5;
constexpr int kThreads = 10 * 32;
constexpr int kTmemCols = 512;
constexpr uint32_t kTmemSf = kBM;
constexpr uint32_t kSfColsPerStage = 48;
constexpr uint32_t kABytes = 128 * kBK / 2;       // 16 KB: this CTA's W rows
constexpr uint32_t kBBytes = 128 * kBK / 2;       // 16 KB: this CTA's half of the x rows
constexpr uint32_t kAtomBytes = 512;
constexpr uint32_t kSfaBytes = 4 * kAtomBytes;    // W atoms of the CTA's 128 rows
constexpr uint32_t kSfbBytes = 8 * kAtomBytes;    // x atoms of both 128-row blocks [rb][j]
constexpr uint32_t kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kOffSfa = kOffB + kStages * kBBytes;
constexpr uint32_t kOffSfb = kOffSfa + kStages * kSfaBytes;
constexpr uint32_t kOffBar = kOffSfb + kStages * kSfbBytes;
constexpr uint32_t kFixBars = 4 * 16;
constexpr uint32_t kNumBars = 2 * kStages + 3 + kFixBars;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
static_assert(kTmemSf + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
constexpr uint32_t kFixupBytes = (kOffBar / 4) & ~127u;
constexpr int kFixupBufs = (int)(kFixupBytes / 4096) < 16 ? (int)(kFixupBytes / 4096) : 16;
static_assert(kFixupBufs >= 2, "fix-up staging");
// block-scaled kind, E2M1 A and B, UE4M3 scales, K-major, fp32 D, M = 256 (the pair), N = 256
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kBM >> 3) << 17) |
                            ((uint32_t)(256 >> 4) << 24);
// how long a producer waits at exit for copies it issued that no MMA consumed (after an
// abort): far longer than any copy takes to land
constexpr uint64_t kDrainNs = 1000000;

}  // namespace pairk

template <bool kQuantX>
__global__ void __launch_bounds__(pairk::kThreads, 1)
gemm_w4a4_pair_kernel(const __grid_constant__ CUtensorMap tmap_w,
                      const __grid_constant__ CUtensorMap tmap_x,
                      const __grid_constant__ CUtensorMap tmap_sw,
                      const __grid_constant__ CUtensorMap tmap_sx, const float* __restrict__ gw,
                      const float* __restrict__ gx, void* __restrict__ y, int y_bf16, int M,
                      int N, int nkb, int natoms_row, int ntiles_m, int ntiles, int ntiles_sk,
                      int p_sk, int64_t tsk, uint32_t* __restrict__ err,
                      uint32_t* __restrict__ counters, float* __restrict__ slots, QxArgs qa,
                      WaitCfg dbg) {
    // this kernel's constants (the one-CTA kernel's share the names)
    constexpr int kBM = pairk::kBM, kBK = pairk::kBK, kStages = pairk::kStages;
    constexpr int kThreads = pairk::kThreads, kTmemCols = pairk::kTmemCols;
    constexpr int kFixupBufs = pairk::kFixupBufs;
    constexpr uint32_t kTmemSf = pairk::kTmemSf, kSfColsPerStage = pairk::kSfColsPerStage;
    constexpr uint32_t kABytes = pairk::kABytes, kBBytes = pairk::kBBytes;
    constexpr uint32_t kAtomBytes = pairk::kAtomBytes, kSfaBytes = pairk::kSfaBytes;
    constexpr uint32_t kSfbBytes = pairk::kSfbBytes, kStageBytes = pairk::kStageBytes;
    constexpr uint32_t kOffA = pairk::kOffA, kOffB = pairk::kOffB, kOffSfa = pairk::kOffSfa;
    constexpr uint32_t kOffSfb = pairk::kOffSfb, kOffBar = pairk::kOffBar;
    constexpr uint32_t kOffMisc = pairk::kOffMisc, kFixBars = pairk::kFixBars;
    constexpr uint32_t kFixupBytes = pairk::kFixupBytes, kIdesc = pairk::kIdesc;
    constexpr uint64_t kDrainNs = pairk::kDrainNs;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const uint32_t bar0 = base_s + kOffBar;
    auto full = [&](int s) { return bar0 + 8u * s; };              // even CTA's is used
    auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
    const uint32_t accfull = bar0 + 8u * (2 * kStages);
    const uint32_t accempty = bar0 + 8u * (2 * kStages + 1);      // even CTA's is used
    const uint32_t drain = bar0 + 8u * (2 * kStages + 2);
    const uint32_t fixbar0 = bar0 + 8u * (2 * kStages + 3);
    auto bar_ptr = [&](uint32_t a) { return reinterpret_cast<uint64_t*>(base + (a - base_s)); };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_rank();
    const int unit = (int)(blockIdx.x >> 1), nunits = (int)(gridDim.x >> 1);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_ptr(full(s)), 1);
            mbar_init(bar_ptr(empty(s)), 1);
        }
        mbar_init(bar_ptr(accfull), 1);
        mbar_init(bar_ptr(accempty), 16);  // 8 epilogue warps in each CTA of the pair
        mbar_init(bar_ptr(drain), 1);
        for (uint32_t i = 0; i < kFixBars; ++i) mbar_init(bar_ptr(fixbar0 + 8u * i), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc_pair(base_s + kOffMisc, kTmemCols);
    tc::fence_before();
    tc::cluster_sync();  // both CTAs' barriers initialised, TMEM allocated
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    float gx_in = 1.0f;
    if constexpr (kQuantX) gx_in = quantize_x_prologue<kThreads / 32>(qa, M, dbg, err, abort_flag);

    auto atoms_of = [&](int kb) { return min(4, natoms_row - 4 * kb); };

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int it = 0, issued = 0;
            tc::WorkIter wi = tc::make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk, unit, nunits);
            int tile, kb0, kb1;
            if constexpr (kQuantX) {
                if (!*abort_flag && !wait_counter(qa.sync + 3, gridDim.x, dbg.wait_ns)) {
                    if (err) atomicOr(err, NVFP4_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                fence_proxy_async_global();
            }
            while (!*abort_flag && wi.next(tile, kb0, kb1)) {
                const int nb = tile / ntiles_m, mb = tile % ntiles_m;
                const int wrb = 2 * nb + (int)rank;  // this CTA's 128-row block of W
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages &&
                        !tc::wait_or_abort(empty(s), ((it / kStages) - 1) & 1, abort_flag, err,
                                           dbg.wait_ns))
                        break;
                    const uint32_t fb = tc::peer_addr(full(s), 0);
                    if (rank == 0) mbar_arrive_expect_tx(bar_ptr(full(s)), 2 * kStageBytes);
                    tc::tma_load_2d_pair(base_s + kOffA + s * kABytes, &tmap_w, kb * (kBK / 2),
                                         wrb * 128, fb);
                    tc::tma_load_2d_pair(base_s + kOffSfa + s * kSfaBytes, &tmap_sw, 0,
                                         wrb * natoms_row + 4 * kb, fb);
                    // x rows of the tile: half `rank` of them, 128 rows; the x scale atoms of
                    // both 128-row blocks, 4 per block (atoms past K or past the tensor's rows
                    // read as zero or as a neighbour's, which no MMA reads or whose outputs
                    // are masked)
                    const uint32_t sb_dst = base_s + kOffSfb + s * kSfbBytes;
                    tc::tma_load_2d_pair(base_s + kOffB + s * kBBytes, &tmap_x, kb * (kBK / 2),
                                         mb * kBM + (int)rank * 128, fb);
                    tc::tma_load_2d_pair(sb_dst, &tmap_sx, 0, (2 * mb) * natoms_row + 4 * kb, fb);
                    tc::tma_load_2d_pair(sb_dst + 4 * kAtomBytes, &tmap_sx, 0,
                                         (2 * mb + 1) * natoms_row + 4 * kb, fb);
                    issued = it + 1;
                }
            }
            // Before the CTA moves on to exit, the copies it issued have landed: the even
            // CTA sees its stage barriers complete, the odd CTA sees its stages released
            // (consumed); after an abort neither may come, and the wait ends after kDrainNs,
            // far longer than a copy takes.
            const uint64_t t0 = globaltimer_ns();
            for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i) {
                const uint64_t el = globaltimer_ns() - t0;
                if (el >= kDrainNs) break;
                const uint32_t b = rank == 0 ? full(i % kStages) : empty(i % kStages);
                mbar_wait_bounded(bar_ptr(b), (i / kStages) & 1, kDrainNs - el);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issue (even CTA) ----------------
        if (rank == 0 && lane == 0) {
            int it = 0, lt = 0;
            tc::WorkIter wi = tc::make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk, unit, nunits);
            int tile, kb0, kb1;
            for (; !*abort_flag && wi.next(tile, kb0, kb1); ++lt) {
                if (lt >= 1 &&
                    !tc::wait_or_abort(accempty, (lt - 1) & 1, abort_flag, err, dbg.wait_ns))
                    break;
                tc::fence_after();
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!tc::wait_or_abort(full(s), (it / kStages) & 1, abort_flag, err,
                                           dbg.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const int na = atoms_of(kb);
                    const uint32_t sf = tmem + kTmemSf + (uint32_t)s * kSfColsPerStage;
                    const uint32_t sa = base_s + kOffSfa + s * kSfaBytes;
                    const uint32_t sb = base_s + kOffSfb + s * kSfbBytes;
                    // scale atoms into both CTAs' TMEM: W atom j at columns 4j, x atom j of
                    // row block 0 / 1 at 16 + 8j / 16 + 8j + 4
                    for (int j = 0; j < na; ++j) {
                        tc::cp_atom_pair(sf + 4 * j, tc::atom_desc(sa + j * kAtomBytes));
                        tc::cp_atom_pair(sf + 16 + 8 * j, tc::atom_desc(sb + j * kAtomBytes));
                        tc::cp_atom_pair(sf + 16 + 8 * j + 4,
                                         tc::atom_desc(sb + (4 + j) * kAtomBytes));
                    }
                    const uint32_t a_s = base_s + kOffA + s * kABytes;
                    const uint32_t b_s = base_s + kOffB + s * kBBytes;
                    for (int j = 0; j < na; ++j)
                        tc::mma_mxf4nvf4_pair(tmem, tc::sw128_desc(a_s + j * 32),
                                              tc::sw128_desc(b_s + j * 32), kIdesc, sf + 4 * j,
                                              sf + 16 + 8 * j, (kb != kb0 || j != 0) ? 1u : 0u);
                    tc::commit_pair(empty(s));
                    tc::commit_pair(tc::peer_addr(empty(s), 1));
                }
                if (!ok) break;
                // (with the test switch on, the accumulator is never marked full: every
                // epilogue's wait runs out)
                if (!(dbg.stall && !kQuantX)) {
                    tc::commit_pair(accfull);
                    tc::commit_pair(tc::peer_addr(accfull, 1));
                }
            }
            // MMAs in flight complete before TMEM is freed
            tc::commit_pair(drain);
            mbar_wait_bounded(bar_ptr(drain), 0, kWaitLimitNs);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int h = (warp - 2) >> 2;   // x-row half of the tile
        const float g = *gw * (kQuantX ? gx_in : *gx);
        const tc::SkUnit u{unit, (int)rank, 2};
        const uint32_t acc_empty = rank == 0 ? accempty : tc::peer_addr(accempty, 0);
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
        int lt = 0;
        tc::WorkIter wi = tc::make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk, unit, nunits);
        int tile, kb0, kb1;
        for (; wi.next(tile, kb0, kb1); ++lt) {
            if (!__all_sync(0xffffffffu,
                            tc::wait_or_abort(accfull, lt & 1, abort_flag, err, dbg.wait_ns)))
                break;
            tc::fence_after();
            if (kb0 == 0 && kb1 == nkb) {
                const int nb = tile / ntiles_m, mb = tile % ntiles_m;
                const int64_t n = ((int64_t)nb * 2 + rank) * 128 + q * 32 + lane;
                const int64_t m0 = (int64_t)mb * kBM + h * 128;
                uint32_t v[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tc::tmem_ld32(taddr + h * 128 + c * 32, v[c]);
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::release_acc(acc_empty, u);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (m0 + c * 32 >= M) break;
                    float f[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[c][j]);
                    tc::store_rows32(y, y_bf16, M, N, m0 + c * 32, n, f, g);
                }
            } else if (h == 1) {
                __syncwarp();
                if (lane == 0) tc::release_acc(acc_empty, u);
            } else {
                // on the CTA's last item the stage ring is idle: a quarter of it per warp
                tc::WorkIter peek = wi;
                int t_, k0_, k1_;
                uint8_t* stage = peek.next(t_, k0_, k1_) ? nullptr : base + q * kFixupBytes;
                tc::epilogue_work<128, kBM>(tmem, q, lane, tile, ntiles_m, false, nkb, p_sk, tsk,
                                            g, y, y_bf16, M, N, slots, counters, acc_empty, stage,
                                            bar_ptr(fixbar0 + 128u * q), kFixupBufs, u, err);
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    tc::cluster_sync();  // no CTA of the pair exits while the other may still address it
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc_pair(tmem, kTmemCols);
    }
    if constexpr (kQuantX) {
        if (threadIdx.x == 0) {
            __threadfence();
            if (atomicAdd(qa.sync + 2, 1u) == gridDim.x - 1) {
                atomicExch(qa.sync + 3, 0u);
                atomicExch(qa.sync, 0u);
                atomicExch(qa.sync + 2, 0u);
            }
        }
    }
}

// Stream-K state of either W4A4 kernel: counters sized for the pair kernel's tiles (two
// 128-row halves per tile; at least the one-CTA kernel's count), then the larger of the two
// kernels' partial-tile slots.  Both kernels leave the counters zero.
size_t counter_region(int64_t M, int64_t N) {
    return tc::counters_bytes(2 * ((N + 255) / 256) * ((M + 255) / 256));
}

template <bool kQuantX>
cudaError_t configure(const DevInfo& dev) {
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = 1ull << (dev.device & 63);
    if (configured.load(std::memory_order_acquire) & bit) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(gemm_w4a4_kernel<kQuantX>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kSmemBytes);
    if (e == cudaSuccess) configured.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

template <bool kQuantX>
cudaError_t launch(const uint8_t* xq, const uint8_t* xsz, const float* gx, int M, int K,
                   const uint8_t* wq, const uint8_t* wsz, const float* gw, int N, void* y,
                   bool y_bf16, uint32_t* err, uint8_t* sk_state, const QxArgs& qa,
                   cudaStream_t stream, const DevInfo& dev) {
    if (dev.smem_optin < kSmemBytes) return cudaErrorInvalidConfiguration;
    const GemmPlan p = tc::make_plan(M, K, N, dev.sm_count, kBN, kBM, kBK);
    CUtensorMap mw, mx;
    cudaError_t e = tc::make_map_2d(&mw, wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2,
                                    (uint64_t)N, kBK / 2, kBN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    e = tc::make_map_2d(&mx, xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2, (uint64_t)M,
                        kBK / 2, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    e = configure<kQuantX>(dev);
    if (e != cudaSuccess) return e;
    const int natoms_row = (K + 63) / 64;  // scale atoms per 128-row block
    uint32_t* counters = reinterpret_cast<uint32_t*>(sk_state);
    float* slots = reinterpret_cast<float*>(sk_state + counter_region(M, N));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    // the in-kernel quantization has CTAs wait for one another: all of them must be
    // resident at once (one per SM), which a cooperative launch guarantees or refuses
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = kQuantX ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, gemm_w4a4_kernel<kQuantX>, mw, mx, wsz, xsz, gw, gx, y,
                           y_bf16 ? 1 : 0, M, N, p.nkb, natoms_row, (M + 127) / 128, p.ntiles_m,
                           p.ntiles, p.ntiles_sk, p.p_sk, p.tsk, err, counters, slots, qa,
                           current_wait_cfg());
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ---- pair kernel host side ----

template <bool kQuantX>
cudaError_t configure_pair(const DevInfo& dev) {
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = 1ull << (dev.device & 63);
    if (configured.load(std::memory_order_acquire) & bit) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(gemm_w4a4_pair_kernel<kQuantX>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)pairk::kSmemBytes);
    if (e == cudaSuccess) configured.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// CTA pairs the device holds at once (one CTA per SM); 0 when it cannot co-schedule them
template <bool kQuantX>
int pair_units(const DevInfo& dev) {
    static std::atomic<int> units[64];  // 0: not queried yet, else units + 1
    std::atomic<int>& slot = units[dev.device & 63];
    const int c = slot.load(std::memory_order_acquire);
    if (c) return c - 1;
    int n = 0;
    if (dev.smem_optin >= pairk::kSmemBytes && configure_pair<kQuantX>(dev) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(pairk::kThreads);
        cfg.dynamicSmemBytes = pairk::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_w4a4_pair_kernel<kQuantX>, &cfg) !=
            cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
    }
    slot.store(n + 1, std::memory_order_release);
    return n;
}

template <bool kQuantX>
cudaError_t launch_pair(int units, const uint8_t* xq, const uint8_t* xsz, const float* gx, int M,
                        int K, const uint8_t* wq, const uint8_t* wsz, const float* gw, int N,
                        void* y, bool y_bf16, uint32_t* err, uint8_t* sk_state,
                        const QxArgs& qa, cudaStream_t stream) {
    constexpr int kBM = pairk::kBM, kBK = pairk::kBK;
    constexpr int kThreads = pairk::kThreads;
    constexpr uint32_t kSmemBytes = pairk::kSmemBytes;
    const GemmPlan p = tc::make_plan(M, K, N, units, 256, kBM, kBK);
    const int natoms_row = (K + 63) / 64;
    CUtensorMap mw, mx, msw, msx;
    cudaError_t e = tc::make_map_2d(&mw, wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2,
                                    (uint64_t)N, kBK / 2, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    e = tc::make_map_2d(&mx, xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2, (uint64_t)M,
                        kBK / 2, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    // scale atoms as rows of 128 32-bit words: row (row block * natoms_row + atom), the 4
    // atoms of a K step per box
    e = tc::make_map_2d(&msw, wsz, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, 128,
                        (uint64_t)((N + 127) / 128) * natoms_row, 128, 4,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    e = tc::make_map_2d(&msx, xsz, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, 128,
                        (uint64_t)((M + 127) / 128) * natoms_row, 128, 4,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    uint32_t* counters = reinterpret_cast<uint32_t*>(sk_state);
    float* slots = reinterpret_cast<float*>(sk_state + counter_region(M, N));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = kQuantX ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, gemm_w4a4_pair_kernel<kQuantX>, mw, mx, msw, msx, gw, gx, y,
                           y_bf16 ? 1 : 0, M, N, p.nkb, natoms_row, p.ntiles_m, p.ntiles,
                           p.ntiles_sk, p.p_sk, p.tsk, err, counters, slots, qa,
                           current_wait_cfg());
    return e != cudaSuccess ? e : cudaGetLastError();
}

// The CTA-pair kernel, where the calling thread asks for it (w4a4_use_pairs); *launched
// stays false for the one-CTA kernel (the default: the faster of the two on this hardware)
// or when the device cannot co-schedule CTA pairs
template <bool kQuantX>
cudaError_t launch_pair_if_asked(const uint8_t* xq, const uint8_t* xsz, const float* gx, int M,
                                 int K, const uint8_t* wq, const uint8_t* wsz, const float* gw,
                                 int N, void* y, bool y_bf16, uint32_t* err, uint8_t* sk_state,
                                 const QxArgs& qa, cudaStream_t stream, const DevInfo& dev,
                                 bool* launched) {
    *launched = false;
    if (!w4a4_use_pairs()) return cudaSuccess;
    const int units = pair_units<kQuantX>(dev);
    if (units <= 0) return cudaSuccess;
    *launched = true;
    return launch_pair<kQuantX>(units, xq, xsz, gx, M, K, wq, wsz, gw, N, y, y_bf16, err,
                                sk_state, qa, stream);
}

}  // namespace

size_t gemm_w4a4_stream_k_bytes(int64_t M, int64_t K, int64_t N) {
    size_t slots = 0;
    for (int bn : {kBN, 256}) {
        const size_t b = tc::stream_k_bytes(M, K, N, bn, kBM, kBK) -
                         tc::counters_bytes(((N + bn - 1) / bn) * ((M + kBM - 1) / kBM));
        if (b > slots) slots = b;
    }
    return counter_region(M, N) + slots;
}

size_t gemm_w4a4_sync_bytes(int64_t) { return 256; }

cudaError_t launch_gemm_w4a4(const uint8_t* xq, const uint8_t* xsz, const float* gx, int M,
                             int K, const uint8_t* wq, const uint8_t* wsz, const float* gw, int N,
                             void* y, bool y_bf16, uint32_t* err, uint8_t* sk_state,
                             cudaStream_t stream, const DevInfo& dev) {
    bool launched = false;
    const cudaError_t e = launch_pair_if_asked<false>(xq, xsz, gx, M, K, wq, wsz, gw, N, y, y_bf16,
                                                 err, sk_state, QxArgs{}, stream, dev, &launched);
    if (launched) return e;
    return launch<false>(xq, xsz, gx, M, K, wq, wsz, gw, N, y, y_bf16, err, sk_state, QxArgs{},
                         stream, dev);
}

cudaError_t launch_gemm_w4a4_quant_x(const uint16_t* x, const float* gx_static, float* gx_out,
                                     float* partials, uint32_t* sync, uint8_t* xq, uint8_t* xsz,
                                     int M, int K, const uint8_t* wq, const uint8_t* wsz,
                                     const float* gw, int N, void* y, bool y_bf16, uint32_t* err,
                                     uint8_t* sk_state, cudaStream_t stream, const DevInfo& dev) {
    QxArgs qa;
    qa.x = x;
    qa.gx_static = gx_static;
    qa.gx_out = gx_out;
    qa.partials = partials;
    qa.sync = sync;
    qa.xq = xq;
    qa.xs = xsz;
    qa.K = K;
    bool launched = false;
    const cudaError_t e = launch_pair_if_asked<true>(xq, xsz, gx_out, M, K, wq, wsz, gw, N, y, y_bf16,
                                                err, sk_state, qa, stream, dev, &launched);
    // a device that refuses a cooperative launch of CTA pairs (or cannot hold them all)
    // takes the one-CTA kernel
    if (launched && e == cudaSuccess) return e;
    if (launched) cudaGetLastError();
    return launch<true>(xq, xsz, gx_out, M, K, wq, wsz, gw, N, y, y_bf16, err, sk_state, qa,
                        stream, dev);
}

}  // namespace nvfp4
