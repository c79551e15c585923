// tcgen05.cuh -- pieces shared by the tensor-core GEMMs (sm_100 family PTX): TMA tile loads,
// TMEM allocation and loads, MMA issue and commit, shared-memory matrix descriptors, the
// persistent work split (stream-K for the last partial wave of tiles, whole tiles for the
// rest), the stream-K epilogue, and the host-side tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "nvfp4.h"

namespace nvfp4 {
namespace tc {

// ---- TMA, TMEM, MMA wrappers -------------------------------------------------------------

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

__device__ __forceinline__ void fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
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

// D[tmem] (+)= block-scaled A . B^T: E2M1 operands (two per byte), one UE4M3 scale per 16
// elements of K for each row of A and of B, read from TMEM (sfa, sfb), fp32 accumulate
__device__ __forceinline__ void mma_mxf4nvf4(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// arrive (once) on bar when every tcgen05 operation this thread issued so far completes
__device__ __forceinline__ void commit(uint32_t bar) {
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

// 32 consecutive TMEM columns of this warp's 32 lanes <- v (each thread its own lane)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16 consecutive TMEM columns of this warp's 32 lanes <- v
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
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

// ---- CTA pairs (cta_group::2) ---------------------------------------------------------------
// A pair is a cluster of two CTAs.  TMEM is allocated by one warp in each CTA together (the
// same columns in both).  The even CTA issues M = 256 MMAs: A rows 0..127 come from its
// shared memory and 128..255 from its peer's (same offset), B's N rows are split the same
// way, and each CTA's TMEM receives its own 128 rows of D.  Scale atoms reach both CTAs'
// TMEM by tcgen05.cp from the same thread, ahead of the MMAs that read them.  TMA loads of
// either CTA land in the issuing CTA's shared memory and complete on the even CTA's
// barrier.

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %cluster_ctarank;" : "=r"(r));
    return r;
}

// every thread of both CTAs of the cluster
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

// the shared::cluster address of this CTA's shared address `saddr` in CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// TMA tile load into this CTA's shared memory, completing on the mbarrier at shared::cluster
// address cbar (the even CTA's)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0,
                                                 int c1, uint32_t cbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(cbar)
        : "memory");
}

// one 512-byte scale atom (32 rows of 16 bytes) from each CTA's shared memory into its own
// TMEM: atom row i to lane 32 q + i of every lane quarter q, four columns
__device__ __forceinline__ uint64_t atom_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128 >> 4) << 16;     // leading byte offset
    d |= (uint64_t)(128 >> 4) << 32;     // stride byte offset
    d |= (uint64_t)1 << 46;              // descriptor version
    return d;
}
__device__ __forceinline__ void cp_atom_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// block-scaled pair MMA, E2M1 operands, UE4M3 scales per 16 elements, fp32 accumulate
__device__ __forceinline__ void mma_mxf4nvf4_pair(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                                  uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                                  uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// arrive (once) on the mbarrier at shared::cluster address cbar (this CTA's or the peer's)
// when every pair operation this thread issued so far completes
__device__ __forceinline__ void commit_pair(uint32_t cbar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(cbar)
        : "memory");
}

// ---- bounded waits -----------------------------------------------------------------------

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, uint32_t* err,
                                              uint64_t limit_ns) {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bar)), parity,
                          limit_ns))
        return true;
    if (err) atomicOr(err, NVFP4_DEVERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

__device__ __forceinline__ void arrive(uint32_t bar) {
    mbar_arrive(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bar)));
}

// arrive on an mbarrier by its shared::cluster address (this CTA's or its peer's)
__device__ __forceinline__ void arrive_cluster(uint32_t cbar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}

// ---- persistent work split ---------------------------------------------------------------

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

// The work of unit c of nunits: a CTA (c = blockIdx.x), or a CTA pair sharing its tiles.
__device__ __forceinline__ WorkIter make_iter(int ntiles, int nkb, int ntiles_sk, int p_sk,
                                              int64_t tsk, int c, int nunits) {
    WorkIter w;
    if (c < p_sk) {
        w.i = (int64_t)c * tsk / p_sk;
        w.i_end = (int64_t)(c + 1) * tsk / p_sk;
    } else {
        w.i = w.i_end = 0;
    }
    w.dp = ntiles_sk + c;
    w.ntiles = ntiles;
    w.nkb = nkb;
    w.stride = nunits;
    return w;
}

__device__ __forceinline__ WorkIter make_iter(int ntiles, int nkb, int ntiles_sk, int p_sk,
                                              int64_t tsk) {
    return make_iter(ntiles, nkb, ntiles_sk, p_sk, tsk, blockIdx.x, gridDim.x);
}

// stream-K bookkeeping: the unit whose range holds iteration i, and the slot unit c uses
// for its partial of the tile starting at iteration t0 (2c: its first segment, 2c + 1: its
// last; a unit of two CTAs has a pair of slots per segment, one per CTA half)
__device__ __forceinline__ int sk_cta_of(int64_t i, int p_sk, int64_t tsk) {
    return (int)(((i + 1) * p_sk - 1) / tsk);
}
__device__ __forceinline__ int sk_slot(int c, int64_t t0, int p_sk, int64_t tsk) {
    return 2 * c + ((int64_t)c * tsk / p_sk < t0 ? 1 : 0);
}

// ---- epilogue ----------------------------------------------------------------------------

// y[m0 + j, n] = v[j] * scale for the rows inside M (fp32 or bf16 y).  A full group of 32
// rows is stored by one straight run of stores under a single warp-uniform test: a guard
// per row costs a branch and a reconvergence point per store, which made these stores
// several times slower.
__device__ __forceinline__ void store_rows32(void* y, int y_bf16, int64_t M, int64_t N,
                                             int64_t m0, int64_t n, const float (&v)[32],
                                             float scale) {
    if (n >= N) return;
    const bool full = m0 + 32 <= M;
    if (y_bf16) {
        uint16_t* yp = static_cast<uint16_t*>(y) + m0 * N + n;
        if (full) {
#pragma unroll
            for (int j = 0; j < 32; ++j) yp[(int64_t)j * N] = f32_to_bf16_rne(v[j] * scale);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (m0 + j < M) yp[(int64_t)j * N] = f32_to_bf16_rne(v[j] * scale);
        }
    } else {
        float* yp = static_cast<float*>(y) + m0 * N + n;
        if (full) {
#pragma unroll
            for (int j = 0; j < 32; ++j) yp[(int64_t)j * N] = v[j] * scale;
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (m0 + j < M) yp[(int64_t)j * N] = v[j] * scale;
        }
    }
}

// Where a CTA's stream-K state lives: its unit (the CTA itself, or the CTA pair whose two
// CTAs hold the two 128-row halves of every tile's W rows), and which half it holds.  Unit c's partial of a tile goes to slot (sk_slot(c, ...) * nhalves + half);
// the tile's counters are (tile * nhalves + half) * 4 + quarter.
struct SkUnit {
    int me = 0;
    int half = 0;
    int nhalves = 1;
};

// Release of an accumulator to the MMA issuer: a plain arrive in a one-CTA unit; from a
// pair's odd CTA an arrive on its even CTA's barrier (its TMEM reads, ordered by the
// caller's tcgen05 fence, come before the issuer's next MMAs into it)
__device__ __forceinline__ void release_acc(uint32_t accempty, const SkUnit& u) {
    if (u.nhalves >= 2 && (u.half & 1))
        arrive_cluster(accempty);
    else
        arrive(accempty);
}

// How long the first segment of a stream-K tile waits, on its CTA's last item, for the
// tile's other segments before it writes its own partial like them
constexpr uint64_t kOwnerWaitNs = 20000;

// A stream-K slot holds a partial tile as [lane quarter q][x row c][W row within the
// quarter]: the quarter's 32 x rows from c0 on are one contiguous 4 KB chunk, written by the
// warp of that quarter with one 128-byte line per store.
template <int BM>
__device__ __forceinline__ size_t slot_chunk(int q, int c0) {
    return ((size_t)q * BM + c0) * 32;
}

// The fix-up of one tile quarter through shared memory.  The partials of the tile's other
// segments stream into `nbuf` 4 KB chunk buffers at `stage` by bulk copies, each buffer with
// its own mbarrier (`bars`, initialised with the kernel's barriers), up to nbuf chunks in
// flight; for every 32 x rows the partials are added in segment order (the CTA's own from
// TMEM when own_tmem), then stored to y.  Only for the CTA's last work item, when every MMA
// of the CTA has completed and the stage ring is idle.
template <int BN, int BM>
__device__ __forceinline__ void fixup_staged(uint32_t taddr, bool own_tmem, int q, int lane,
                                             int mb, int cf, int cl, int64_t t0, int p_sk,
                                             int64_t tsk, const float* slots, uint8_t* stage,
                                             uint64_t* bars, int nbuf, float scale, void* y,
                                             int y_bf16, int M, int N, int64_t n, SkUnit u,
                                             uint32_t* err) {
    constexpr size_t kSlotFloats = (size_t)BN * BM;
    const int me = u.me;
    const int64_t rows_left = (int64_t)M - (int64_t)mb * BM;
    const int nrow = rows_left >= BM ? BM / 32 : (int)((rows_left + 31) / 32);
    const int nother = cl - cf + 1 - (own_tmem ? 1 : 0);
    const int total = nrow * nother;
    float* bufs = reinterpret_cast<float*>(stage);
    // this quarter's part of segment cs's slot: the tile's first segment may be its CTA's
    // second slot; every later segment starts its CTA's range (the first slot)
    const float* q_base = slots + (size_t)q * BM * 32;
    const float* first_seg =
        q_base + ((size_t)sk_slot(cf, t0, p_sk, tsk) * u.nhalves + u.half) * kSlotFloats;
    auto seg_src = [&](int cs) {
        return cs == cf ? first_seg
                        : q_base + ((size_t)(2 * cs) * u.nhalves + u.half) * kSlotFloats;
    };
    // the chunk stream, in the order it is read: x rows 32 ci .. of every other segment
    int is_ci = 0, is_cs = (own_tmem && cf == me) ? cf + 1 : cf, is_b = 0, issued = 0;
    auto issue_next = [&]() {
        if (lane == 0) {
            mbar_arrive_expect_tx(bars + is_b, 4096);
            bulk_g2s(bufs + (size_t)is_b * 1024, seg_src(is_cs) + (size_t)is_ci * 32 * 32, 4096,
                     bars + is_b);
        }
        ++issued;
        if (++is_b == nbuf) is_b = 0;
        if (++is_cs == me && own_tmem) ++is_cs;
        if (is_cs > cl) {
            ++is_ci;
            is_cs = (own_tmem && cf == me) ? cf + 1 : cf;
        }
    };
    const int pre = total < nbuf ? total : nbuf;
#pragma unroll 1
    for (int k = 0; k < pre; ++k) issue_next();
    int rb = 0, nread = 0;
    uint32_t rph = 0;
    bool ok = true;
#pragma unroll 1
    for (int ci = 0; ci < nrow && ok; ++ci) {
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
#pragma unroll 1
        for (int cs = cf; cs <= cl; ++cs) {
            float v[32];
            if (own_tmem && cs == me) {
                uint32_t u[32];
                tmem_ld32(taddr + (uint32_t)(ci * 32), u);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(u[j]);
            } else {
                bool landed = mbar_try_wait(bars + rb, rph);
                if (!__all_sync(0xffffffffu, landed))
                    landed = mbar_wait_bounded(bars + rb, rph, kWaitLimitNs);
                if (!__all_sync(0xffffffffu, landed)) {
                    ok = false;
                    break;
                }
                const float* src = bufs + (size_t)rb * 1024 + lane;
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = src[j * 32];
                if (issued < total) {
                    // the buffer is read before the copy that refills it is issued
                    __syncwarp();
                    fence_proxy_async_smem();
                    issue_next();
                }
                ++nread;
                if (++rb == nbuf) {
                    rb = 0;
                    rph ^= 1u;
                }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] += v[j];
        }
        if (ok) store_rows32(y, y_bf16, M, N, (int64_t)mb * BM + ci * 32, n, acc, scale);
    }
    if (!ok) {
        if (lane == 0 && err) atomicOr(err, NVFP4_DEVERR_TIMEOUT);
        // the copies in flight land before the CTA moves on to exit: the unread ones, from
        // buffer rb on
        int b = rb;
        uint32_t ph = rph;
        for (int i = nread; i < issued; ++i) {
            mbar_wait_bounded(bars + b, ph, kWaitLimitNs);
            if (++b == nbuf) {
                b = 0;
                ph ^= 1u;
            }
        }
    }
}

// One work item's epilogue for one epilogue warp: TMEM lane quarter q holds W rows
// q*32 .. q*32+31 of the CTA's BN rows of the tile (the half u.half of a pair's 2 BN rows),
// columns 0 .. BM-1 the tile's x rows.  `accempty` is the mbarrier that releases the
// accumulator: this CTA's, or for a pair's odd CTA the even CTA's (a shared::cluster
// address).  A whole tile goes to y.
// A stream-K segment goes to this CTA's fp32 slot, and the arrival that completes the
// quarter's count (one counter per tile quarter, wrapping back to zero) adds the quarter's
// partials in segment order and writes y.  On the CTA's last work item (`stage` not null:
// this warp's share of the idle stage ring, nbuf chunk buffers with their mbarriers at
// `fixbars`) a segment that finds every other segment of its tile already counted (the
// tile's first segment waits up to kOwnerWaitNs for that) skips its slot: it keeps its
// partial in TMEM and adds it in its place in the order, the other partials streamed in
// through shared memory.  The order of the additions is the same on every path, so results are
// deterministic.  The accumulator is released (accempty) as soon as it has been read.
template <int BN, int BM>
__device__ __forceinline__ void epilogue_work(uint32_t acc, int q, int lane, int tile,
                                              int ntiles_m, bool whole, int nkb, int p_sk,
                                              int64_t tsk, float scale, void* y, int y_bf16,
                                              int M, int N, float* slots, uint32_t* counters,
                                              uint32_t accempty, uint8_t* stage,
                                              uint64_t* fixbars, int nbuf, SkUnit u,
                                              uint32_t* err) {
    static_assert(BN == 128, "four lane quarters of 32 W rows");
    constexpr size_t kSlotFloats = (size_t)BN * BM;
    const int nb = tile / ntiles_m, mb = tile % ntiles_m;
    const int nl = q * 32 + lane;
    const int64_t n = ((int64_t)nb * u.nhalves + u.half) * BN + nl;
    const uint32_t taddr = acc + ((uint32_t)(q * 32) << 16);
    const int64_t t0 = (int64_t)tile * nkb;
    int cf = 0, cl = 0;
    unsigned nseg = 1;
    if (!whole) {
        cf = sk_cta_of(t0, p_sk, tsk);
        cl = sk_cta_of(t0 + nkb - 1, p_sk, tsk);
        nseg = (unsigned)(cl - cf + 1);
        if (stage) {
            unsigned seen = 0;
            if (lane == 0) {
                const uint32_t* cnt = &counters[(tile * u.nhalves + u.half) * 4 + q];
                seen = ld_acquire_gpu(cnt);
                // The tile's first segment waits a little for the others to be counted
                // rather than writing its own slot: on a CTA's last item the others end at
                // about the same time (the stream-K ranges are balanced).  The wait is
                // bounded; when it runs out the segment takes the ordinary path below.
                if (seen != nseg - 1 && u.me == cf) {
                    const uint64_t w0 = globaltimer_ns();
                    while (seen != nseg - 1 && globaltimer_ns() - w0 < kOwnerWaitNs) {
                        __nanosleep(64);
                        seen = ld_acquire_gpu(cnt);
                    }
                }
            }
            if (__shfl_sync(0xffffffffu, seen, 0) == nseg - 1) {
                // every other partial is in its slot; the count goes back to zero for the
                // next call (no other segment touches it again)
                if (lane == 0) counters[(tile * u.nhalves + u.half) * 4 + q] = 0u;
                fixup_staged<BN, BM>(taddr, true, q, lane, mb, cf, cl, t0, p_sk, tsk, slots,
                                     stage, fixbars, nbuf, scale, y, y_bf16, M, N, n, u, err);
                fence_before();
                __syncwarp();
                if (lane == 0) release_acc(accempty, u);
                return;
            }
        }
    }
    float* mine = whole ? nullptr
                        : slots + ((size_t)sk_slot(u.me, t0, p_sk, tsk) * u.nhalves + u.half) *
                                      kSlotFloats +
                              slot_chunk<BM>(q, 0) + lane;
#pragma unroll 1
    for (int c0 = 0; c0 < BM; c0 += 32) {
        uint32_t u[32];
        tmem_ld32(taddr + c0, u);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(u[j]);
        if (whole) {
            store_rows32(y, y_bf16, M, N, (int64_t)mb * BM + c0, n, v, scale);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) mine[(size_t)(c0 + j) * 32] = v[j];
        }
    }
    fence_before();
    __syncwarp();
    if (lane == 0) release_acc(accempty, u);
    if (whole) return;
    __threadfence();
    __syncwarp();
    unsigned old = 0;
    if (lane == 0) old = atomicInc(&counters[(tile * u.nhalves + u.half) * 4 + q], nseg - 1);
    if (__shfl_sync(0xffffffffu, old, 0) != nseg - 1) return;
    __threadfence();
    if (stage) {
        fixup_staged<BN, BM>(taddr, false, q, lane, mb, cf, cl, t0, p_sk, tsk, slots, stage,
                             fixbars, nbuf, scale, y, y_bf16, M, N, n, u, err);
        return;
    }
    // 32 rows of the quarter at a time, every partial's 32 loads in flight together; the
    // partials are added in segment order
#pragma unroll 1
    for (int c0 = 0; c0 < BM; c0 += 32) {
        const int64_t m0 = (int64_t)mb * BM + c0;
        if (m0 >= M) break;
        float accv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) accv[j] = 0.0f;
#pragma unroll 1
        for (int cs = cf; cs <= cl; ++cs) {
            const float* sp = slots + ((size_t)sk_slot(cs, t0, p_sk, tsk) * u.nhalves + u.half) *
                                          kSlotFloats +
                              slot_chunk<BM>(q, c0) + lane;
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __ldcg(sp + (size_t)j * 32);
#pragma unroll
            for (int j = 0; j < 32; ++j) accv[j] += v[j];
        }
        store_rows32(y, y_bf16, M, N, m0, n, accv, scale);
    }
}

// ---- host side ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
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

// 2-D tiled map over a row-major [rows, inner] tensor, zero fill outside it
inline cudaError_t make_map_2d(CUtensorMap* map, const void* ptr, CUtensorMapDataType type,
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

constexpr int kMaxSkCtas = 160;  // CTAs in the stream-K part, at most

// Tiles of BN W rows x BM x rows, nkb K steps each.  The tiles of the last, partial wave
// (all of them when there are fewer than the SMs) go stream-K over p_sk CTAs: at least 4 K
// steps per CTA, at most 3 CTAs' worth per tile, at most kMaxSkCtas.
inline GemmPlan make_plan(int64_t M, int64_t K, int64_t N, int sm_count, int bn, int bm,
                          int bk) {
    GemmPlan p;
    p.nkb = (int)((K + bk - 1) / bk);
    p.ntiles_m = (int)((M + bm - 1) / bm);
    p.ntiles = (int)((N + bn - 1) / bn) * p.ntiles_m;
    int sk = p.ntiles >= sm_count ? p.ntiles % sm_count : p.ntiles;
    const int64_t tsk = (int64_t)sk * p.nkb;
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

// Stream-K state after a 256-byte header: counters (4 per tile, 256-byte padded), then two
// fp32 partial-tile slots per stream-K CTA.  A bound over every SM count.
inline size_t counters_bytes(int64_t ntiles) { return ((size_t)ntiles * 16 + 255) / 256 * 256; }
inline size_t stream_k_bytes(int64_t M, int64_t K, int64_t N, int bn, int bm, int bk) {
    const int64_t nkb = (K + bk - 1) / bk;
    const int64_t ntiles = ((N + bn - 1) / bn) * ((M + bm - 1) / bm);
    int64_t psk = kMaxSkCtas;
    if (psk > 3 * ntiles) psk = 3 * ntiles;
    if (psk > ntiles * nkb / 4) psk = ntiles * nkb / 4;
    if (psk < 2) psk = 0;
    return counters_bytes(ntiles) + (size_t)(2 * psk) * (size_t)bn * bm * 4;
}

}  // namespace tc
}  // namespace nvfp4
