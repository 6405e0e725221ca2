// tc_grouped_sm103.cu -- bf16 NHWC/KYXC dgrad for narrow groups (C/G = K/G in
// {8, 16, 32}) on the tcgen05 tensor cores, e.g. the grouped 3x3 layers of
// ResNeXt-style networks (a workload named on page "[igemm_dynamic] v4r1 bwd
// dynamic kernel").
//
// With 8 channels per group the layer does ~14 FLOP per byte: it is bound by
// HBM (dy read once, dx written once), not by the tensor cores.  So the
// groups of one 64-channel block (64 / Cg of them) are folded into a single
// 64 x 64 GEMM whose B operand is block-diagonal:
//   B_tap[k, c] = w[gb*64 + k, y, x, c mod Cg]  if k / Cg == c / Cg, else 0
// which spends 64/Cg times the useful multiply-adds on the tensor cores --
// affordable far below the ridge -- and turns the layer into the same
// residue-class implicit GEMM as the wide layers (the v4r1 backward-data
// split of pages "Backward data" and "[igemm_dynamic] v4r1 bwd dynamic
// kernel"): per class (ty, tx) and group block gb,
//   D[m, c] = sum over taps (j, i) of sum over k < 64 of A[m, k] * B_tap[k, c]
//   A[m, k] = dy[n, ht - j*DH, wt - i*DW, gb*64 + k]      (zero outside dy)
//   dx[n, ht*sh + ty*dh - ph, wt*sw + tx*dw - pw, gb*64 + c] = bf16_rne(D[m, c]).
//
// Each CTA owns one group block for the whole launch, so its block-diagonal B
// (one 8 KB 128-byte-swizzled tile per filter tap, built from w by the CTA's
// threads at start) stays resident in shared memory; only A streams in, one
// TMA im2col load of 128 rows x 64 channels per tap (one map per class, as in
// the wide kernels).  Roles:
//   warps 0-7   epilogue, two groups of four: group e drains the tiles whose
//               TMEM accumulator is buffer e (tiles t with t % 2 == e), so two
//               tiles' stores are in flight while the MMAs run ahead;
//   warp 8      A producer (one lane issues the TMA loads);
//   warp 9      TMEM allocation and the single-thread tcgen05.mma issue
//               (M = 128, N = 64, K = 16, bf16 x bf16 -> fp32).
// Every barrier wait is bounded; on a timeout the kernel records the status
// word, lets its copies land and returns.
//
// Where it runs: the planner sends C/G = 32 here (no other kernel covers it)
// and keeps C/G in {8, 16} on the warp-level MMA kernel (grouped.cu), which
// stages each dy row once per item and reuses it for every tap.  This kernel
// loads A once per tap (9 im2col loads per dy pixel on a 3x3 layer, served by
// L2) and measured 78 us against 51 us on the ResNeXt layer
// (64x56x56x256, G = 32); CONVBWD_DEBUG_GROUPED=tc selects it there.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "device_util.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace cbd {

struct TgCfg {
    static constexpr int BM = 128;
    static constexpr int BN = 64;           // one block of 64 channels
    static constexpr int STAGES = 6;
    static constexpr int A_BYTES = BM * 64 * 2;
    static constexpr int B_TAP_BYTES = 64 * 64 * 2;
    static constexpr int STAGE_OUT_BYTES = 8 * 32 * 128;  // epilogue staging: 8 warps x 32 rows x 128 B
    static constexpr int BAR_BYTES = 256;
    static constexpr int EPI_WARPS = 8;
    static constexpr int PROD_WARP = 8;
    static constexpr int MMA_WARP = 9;
    static constexpr int THREADS = 32 * 10;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int FIXED_SMEM = 1024 + STAGES * A_BYTES + STAGE_OUT_BYTES + BAR_BYTES;
};

size_t tc_grouped_smem_bytes(int taps) { return (size_t)TgCfg::FIXED_SMEM + (size_t)taps * TgCfg::B_TAP_BYTES; }

// u-th tile of a group block: class and m-block.  When every class has the
// same number of m-blocks the classes are interleaved (u = mb * classes + ci),
// so that the CTAs of a group block work on one region of dy with all its
// taps at once and the re-reads of dy hit L2; otherwise class after class
// (cls[i].tile_begin = first tile of class i within one group block).
__device__ __forceinline__ void tg_tile(const TcParams &p, int u, int &ci, int &mb) {
    if (p.interleave) {
        mb = u / p.num_classes;
        ci = u - mb * p.num_classes;
        return;
    }
    ci = 0;
    for (int i = 1; i < p.num_classes; ++i)
        if (u >= p.cls[i].tile_begin) ci = i;
    mb = u - p.cls[ci].tile_begin;
}

__global__ void __launch_bounds__(TgCfg::THREADS, 1) tc_grouped_dgrad_kernel(const __grid_constant__ TcParams p) {
    using Cfg = TgCfg;
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const Geom &g = p.g;  // folded geometry: G = group blocks, Cg = Kg = 64
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // [A stages | B tiles (taps x 8 KB) | epilogue staging | barriers], all 1024-aligned
    uint8_t *sA = smem;
    uint8_t *sB = sA + S * Cfg::A_BYTES;
    uint8_t *stage = sB + g.Y * g.X * Cfg::B_TAP_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(stage + Cfg::STAGE_OUT_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 4);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);

    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 2);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int gblocks = g.G;
    const int gb = blockIdx.x % gblocks;            // this CTA's group block
    const int local = blockIdx.x / gblocks, nlocal = gridDim.x / gblocks;
    const int units = p.total_tiles / gblocks;     // tiles of one group block
    if (threadIdx.x == 0) CBD_PHASE(p, kPhEntry);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 128);  // the 128 threads of epilogue group b
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == Cfg::MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tc_fence_before();
    }
    if (warp == Cfg::PROD_WARP && lane == 0)
        for (int ci = 0; ci < p.num_classes; ++ci)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_a[ci])) : "memory");

    // Block-diagonal B of this group block, one 64 (k) x 64 (c) tile per filter
    // tap, laid out as a 128-byte-swizzled MN-major operand (row k = 128 bytes
    // of c; 16-byte chunk q of row k at chunk q ^ (k % 8)).  Chunk q of row k
    // holds channels 8q..8q+7, nonzero only inside k's own group.
    {
        // One thread per (tap, k) row, four rows in flight per thread: the row's
        // cg / 8 nonzero chunks are loaded first (16-byte loads: cg and the
        // chunk offsets are multiples of 8), then all 8 chunks are written.
        const int cg = p.bd_cg, nzc = cg / 8;
        const int ntap = g.Y * g.X, rows = ntap * 64;
        const uint16_t *w = static_cast<const uint16_t *>(p.w);
        const int64_t rowlen = (int64_t)ntap * cg;  // bf16 per filter row k (KYXC, C/G channels)
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int r0 = threadIdx.x; r0 < rows; r0 += 4 * Cfg::THREADS) {
            uint4 v[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = r0 + u * Cfg::THREADS;
                const int tap = r >> 6, k = r & 63;
                const uint16_t *src = w + ((int64_t)gb * 64 + k) * rowlen + (int64_t)tap * cg;
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    v[u][h] = (r < rows && h < nzc) ? *reinterpret_cast<const uint4 *>(src + 8 * h) : z;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = r0 + u * Cfg::THREADS;
                if (r >= rows) break;
                const int tap = r >> 6, k = r & 63;
                const int first = (k / cg) * nzc;  // chunk of channel (k / cg) * cg
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    uint4 val = z;
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        if (h < nzc && q == first + h) val = v[u][h];
                    *reinterpret_cast<uint4 *>(sB + tap * Cfg::B_TAP_BYTES + k * 128 + ((q ^ (k & 7)) << 4)) = val;
                }
            }
        }
        fence_proxy_async_smem();  // generic-proxy writes, read by the tensor cores
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) CBD_PHASE(p, kPhSetup);

    if (warp == Cfg::PROD_WARP) {
        // ------------------------------------------------------------ A producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true, issued = false;
            for (int u = local; u < units && ok; u += nlocal) {
                int ci, mb;
                tg_tile(p, u, ci, mb);
                const ClassDesc &c = p.cls[ci];
                const int HTWT = c.HT * c.WT;
                const int m0 = mb * 128;
                const int n0 = m0 / HTWT, rem = m0 - n0 * HTWT;
                const int bh = c.ht_lo + rem / c.WT - (c.taps_y - 1) * g.DH;
                const int bw = c.wt_lo + rem % c.WT - (c.taps_x - 1) * g.DW;
                const CUtensorMap *amap = &p.tmap_a[ci];
                for (int j = 0; j < c.taps_y && ok; ++j)
                    for (int i = 0; i < c.taps_x; ++i, ++it) {
                        const uint32_t s = it % S, ph = (it / S) & 1;
                        if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, p.wait_budget, abort_flag, p.status,
                                               kDevTimeoutProducer)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full0 + 8 * s, (uint32_t)Cfg::A_BYTES);
                        tma_load_im2col(smem_u32(sA + s * Cfg::A_BYTES), amap, full0 + 8 * s, gb * 64, bw, bh, n0,
                                        (uint16_t)((c.taps_x - 1 - i) * g.DW), (uint16_t)((c.taps_y - 1 - j) * g.DH));
                        if (it == 0) CBD_PHASE(p, kPhFirstIssue);
                        issued = true;
                    }
            }
            if (issued) CBD_PHASE(p, kPhLastIssue);
            if (!ok && issued) {
                for (int q = 0; q < 100; ++q) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else if (warp == Cfg::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16<Cfg::BN>();
            const uint32_t b_base = smem_u32(sB);
            uint32_t it = 0, tc = 0;
            bool ok = true, issued = false;
            for (int u = local; u < units && ok; u += nlocal, ++tc) {
                int ci, mb;
                tg_tile(p, u, ci, mb);
                const ClassDesc &c = p.cls[ci];
                const uint32_t b = tc & 1, tph = (tc >> 1) & 1;
                if (!mbar_wait_bounded(tempty0 + 8 * b, tph ^ 1, p.wait_budget, abort_flag, p.status,
                                       kDevTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (tc == 1) CBD_PHASE(p, kPhMma1Start);
                const uint32_t d_tmem = tmem_base + b * Cfg::BN;
                bool first = true;
                for (int j = 0; j < c.taps_y && ok; ++j)
                    for (int i = 0; i < c.taps_x; ++i, ++it) {
                        const uint32_t s = it % S, ph = (it / S) & 1;
                        if (!mbar_wait_bounded(full0 + 8 * s, ph, p.wait_budget, abort_flag, p.status,
                                               kDevTimeoutMma)) {
                            ok = false;
                            break;
                        }
                        if (it == 0) CBD_PHASE(p, kPhFirstFull);
                        tc_fence_after();
                        const int tap = (c.ty + g.YT * j) * g.X + c.tx + g.XT * i;
                        const uint32_t a_addr = smem_u32(sA + s * Cfg::A_BYTES);
                        const uint32_t b_addr = b_base + (uint32_t)tap * Cfg::B_TAP_BYTES;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = smem_desc_sw128(a_addr + kk * 32, 16, 1024);
                            const uint64_t bd = smem_desc_sw128(b_addr + kk * 2048, 8192, 1024);
                            tc_mma(d_tmem, ad, bd, idesc, (!first || kk != 0) ? 1u : 0u);
                        }
                        first = false;
                        issued = true;
                        tc_commit(empty0 + 8 * s);
                    }
                if (!ok) break;
                tc_commit(tfull0 + 8 * b);
                if (tc == 0) CBD_PHASE(p, kPhMma0Done);
                CBD_PHASE(p, kPhMmaLast);
            }
            if (!ok && issued) {
                for (int q = 0; q < 100; ++q) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (two groups)
        const int e = warp >> 2;                  // group: TMEM buffer e, tiles tc % 2 == e
        const int row = (warp & 3) * 32 + lane;   // TMEM lane = tile row
        __nv_bfloat16 *dx = static_cast<__nv_bfloat16 *>(p.dx);
        if (p.fill) fill_uncovered(p, threadIdx.x, 32 * Cfg::EPI_WARPS);
        if (threadIdx.x == 0) CBD_PHASE(p, kPhFillDone);
        uint32_t tc = 0;
        for (int u = local; u < units; u += nlocal, ++tc) {
            if ((int)(tc & 1) != e) continue;
            int ci, mb;
            tg_tile(p, u, ci, mb);
            const ClassDesc &c = p.cls[ci];
            const uint32_t tph = (tc >> 1) & 1;
            bool ok = mbar_wait_bounded(tfull0 + 8 * e, tph, p.wait_budget, abort_flag, p.status, kDevTimeoutEpilogue);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            if (threadIdx.x == 0 && tc == 0) CBD_PHASE(p, kPhEpi0Start);
            const int m = mb * 128 + row;
            const bool rvalid = m < c.M;
            int64_t off = 0;
            if (rvalid) {
                const int HTWT = c.HT * c.WT;
                const int n = m / HTWT;
                const int rem = m - n * HTWT;
                const int hi = (c.ht_lo + rem / c.WT) * g.sh + c.ty * g.dh - g.ph;
                const int wi = (c.wt_lo + rem % c.WT) * g.sw + c.tx * g.dw - g.pw;
                off = (((int64_t)n * g.Hi + hi) * g.Wi + wi) * g.C + (int64_t)gb * 64;
            }
            const uint32_t tbase = tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)e * Cfg::BN;
            epilogue_rows<Cfg::BN>(tbase, stage + warp * 4096, lane, rvalid, off, 0, 64, dx);
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * e);
            if (threadIdx.x == 0 && tc == 0) CBD_PHASE(p, kPhEpi0Done);
            if (lane == 0 && (warp & 3) == 0) CBD_PHASE(p, kPhEpiLast);
        }
    }

    __syncthreads();
    if (threadIdx.x == 0) CBD_PHASE(p, kPhExit);
    if (warp == Cfg::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

cudaError_t launch_tc_grouped(const TcParams &p, int grid, cudaStream_t s) {
    if (grid <= 0 || p.total_tiles <= 0) return cudaSuccess;
    const size_t smem = tc_grouped_smem_bytes(p.g.Y * p.g.X);
    cudaError_t e = cudaFuncSetAttribute(tc_grouped_dgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    tc_grouped_dgrad_kernel<<<grid, TgCfg::THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace cbd
